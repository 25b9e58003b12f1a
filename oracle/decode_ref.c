/*
 * ORACLE (test infrastructure only; never part of the product path).
 *
 * Plain fp64 CPU paged GQA decode attention, written from its definition.
 * Only tests/, the smoke check and the bench's CPU-baseline leg may load it.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * What it computes (one query token per sequence):
 *   for sequence b, query head j, kv head h = floor(j / G), G = H_q / H_kv,
 *   N = seq_lens[b]:
 *     token t < N lives in physical block block_table[b][t / 64], slot t % 64
 *       ("Using HPC-Ops Backends in vLLM": --block-size 64);
 *     s_t   = softmax_scale * sum_d q[b][j][d] * k_t[d]
 *     m     = max_t s_t
 *     l     = sum_t exp(s_t - m)
 *     out   = sum_t exp(s_t - m) * v_t / l
 *     lse   = m + ln(l)                       (natural log)
 *   N == 0 gives out = 0 and lse = -inf.
 * GQA shape (64 query heads sharing 8 KV heads, head_dim 128) follows the
 * Hy3 paragraph of the 24-ai.news page; the fp8_e4m3 KV cache follows
 * "Using HPC-Ops Backends in vLLM" (--kv-cache-dtype fp8_e4m3). FP8 values
 * are decoded from the OCP E4M3 format definition and multiplied by the
 * per-tensor fp32 scale of K or V.
 *
 * All arithmetic is fp64; bf16 and e4m3 values widen to fp64 exactly.
 * Work is split over (sequence, kv head) pairs on POSIX threads; every
 * output element is computed by exactly one thread, in plain loop order.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_BLOCK 64

/* bf16 is the top 16 bits of an IEEE binary32. */
double oracle_bf16_to_f64(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP 8-bit E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
 * Exponent field 0 is subnormal (2^-6 * m/8); S.1111.111 is NaN; there are
 * no infinities. */
double oracle_e4m3_to_f64(uint8_t byte) {
  int sign = (byte >> 7) & 1;
  int e = (byte >> 3) & 0xF;
  int m = byte & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

typedef struct {
  int32_t num_seqs, num_q_heads, num_kv_heads, head_dim;
  const uint16_t* q;
  const void* k_cache;
  const void* v_cache;
  int32_t kv_is_fp8;
  double k_scale, v_scale;
  const int32_t* block_table;
  int32_t max_blocks;
  const int32_t* seq_lens;
  double softmax_scale;
  double* out;
  double* lse;
  long next_task; /* protected by mu */
  pthread_mutex_t mu;
  int status;
} oracle_job;

/* Element d of K or V for (physical block, kv head, slot). */
static double kv_value(const oracle_job* J, const void* cache, double scale, long blk,
                       int h, int slot, int d) {
  long idx = (((blk * J->num_kv_heads + h) * (long)ORACLE_BLOCK + slot) * J->head_dim) + d;
  if (J->kv_is_fp8) return oracle_e4m3_to_f64(((const uint8_t*)cache)[idx]) * scale;
  return oracle_bf16_to_f64(((const uint16_t*)cache)[idx]);
}

static void run_task(oracle_job* J, long task, double* s) {
  int b = (int)(task / J->num_kv_heads);
  int h = (int)(task % J->num_kv_heads);
  int G = J->num_q_heads / J->num_kv_heads;
  int D = J->head_dim;
  int N = J->seq_lens[b];
  for (int g = 0; g < G; ++g) {
    int j = h * G + g;
    double* o = J->out + ((long)b * J->num_q_heads + j) * D;
    const uint16_t* qv = J->q + ((long)b * J->num_q_heads + j) * D;
    if (N == 0) {
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      J->lse[(long)b * J->num_q_heads + j] = -INFINITY;
      continue;
    }
    /* scores */
    for (int t = 0; t < N; ++t) {
      long blk = J->block_table[(long)b * J->max_blocks + t / ORACLE_BLOCK];
      int slot = t % ORACLE_BLOCK;
      double acc = 0.0;
      for (int d = 0; d < D; ++d)
        acc += oracle_bf16_to_f64(qv[d]) * kv_value(J, J->k_cache, J->k_scale, blk, h, slot, d);
      s[t] = J->softmax_scale * acc;
    }
    /* softmax with the max subtracted, then the weighted sum of V rows */
    double m = s[0];
    for (int t = 1; t < N; ++t)
      if (s[t] > m) m = s[t];
    double l = 0.0;
    for (int t = 0; t < N; ++t) l += exp(s[t] - m);
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int t = 0; t < N; ++t) {
      long blk = J->block_table[(long)b * J->max_blocks + t / ORACLE_BLOCK];
      int slot = t % ORACLE_BLOCK;
      double p = exp(s[t] - m);
      for (int d = 0; d < D; ++d) o[d] += p * kv_value(J, J->v_cache, J->v_scale, blk, h, slot, d);
    }
    for (int d = 0; d < D; ++d) o[d] /= l;
    J->lse[(long)b * J->num_q_heads + j] = m + log(l);
  }
}

static void* worker(void* arg) {
  oracle_job* J = (oracle_job*)arg;
  long max_len = 1;
  for (int b = 0; b < J->num_seqs; ++b)
    if (J->seq_lens[b] > max_len) max_len = J->seq_lens[b];
  double* s = (double*)malloc(sizeof(double) * (size_t)max_len);
  if (!s) {
    pthread_mutex_lock(&J->mu);
    J->status = 3;
    pthread_mutex_unlock(&J->mu);
    return NULL;
  }
  long total = (long)J->num_seqs * J->num_kv_heads;
  for (;;) {
    pthread_mutex_lock(&J->mu);
    long task = J->next_task++;
    pthread_mutex_unlock(&J->mu);
    if (task >= total) break;
    run_task(J, task, s);
  }
  free(s);
  return NULL;
}

int oracle_num_cpus(void) {
  long n = sysconf(_SC_NPROCESSORS_ONLN);
  return n > 0 ? (int)n : 1;
}

/*
 * Returns 0 on success, 1 on invalid arguments, 2 if a thread could not be
 * started, 3 on allocation failure. Layouts (row-major, contiguous):
 *   q           uint16 (bf16 bits) [num_seqs][num_q_heads][head_dim]
 *   k/v_cache   bf16 bits or e4m3 bytes [num_blocks][num_kv_heads][64][head_dim]
 *   block_table int32 [num_seqs][max_blocks]
 *   out         double [num_seqs][num_q_heads][head_dim]
 *   lse         double [num_seqs][num_q_heads]
 * num_threads <= 0 uses every online CPU.
 */
int oracle_paged_decode(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                        int32_t head_dim, const uint16_t* q, const void* k_cache,
                        const void* v_cache, int32_t kv_is_fp8, double k_scale,
                        double v_scale, const int32_t* block_table, int32_t max_blocks,
                        const int32_t* seq_lens, double softmax_scale, double* out,
                        double* lse, int32_t num_threads) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 1;
  if (num_q_heads % num_kv_heads != 0) return 1;
  for (int b = 0; b < num_seqs; ++b) {
    if (seq_lens[b] < 0) return 1;
    if ((seq_lens[b] + ORACLE_BLOCK - 1) / ORACLE_BLOCK > max_blocks) return 1;
  }
  oracle_job J;
  memset(&J, 0, sizeof J);
  J.num_seqs = num_seqs;
  J.num_q_heads = num_q_heads;
  J.num_kv_heads = num_kv_heads;
  J.head_dim = head_dim;
  J.q = q;
  J.k_cache = k_cache;
  J.v_cache = v_cache;
  J.kv_is_fp8 = kv_is_fp8;
  J.k_scale = kv_is_fp8 ? k_scale : 1.0;
  J.v_scale = kv_is_fp8 ? v_scale : 1.0;
  J.block_table = block_table;
  J.max_blocks = max_blocks;
  J.seq_lens = seq_lens;
  J.softmax_scale = softmax_scale;
  J.out = out;
  J.lse = lse;
  pthread_mutex_init(&J.mu, NULL);
  int nt = num_threads > 0 ? num_threads : oracle_num_cpus();
  if (nt > 256) nt = 256;
  pthread_t th[256];
  int started = 0;
  for (int i = 0; i < nt; ++i) {
    if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
    ++started;
  }
  if (started == 0) {
    pthread_mutex_destroy(&J.mu);
    return 2;
  }
  for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
  pthread_mutex_destroy(&J.mu);
  return J.status;
}
