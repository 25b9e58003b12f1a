// Prefill / extend attention over the paged KV cache on the 5th-generation
// tensor cores (tcgen05), for sm_103a.
//
// The pages benchmark one attention kernel across prefill, extend and decode
// shapes ("vLLM x HPC-Ops", section "Attention Across Prefill, Extend and
// Decode Shapes": q512 prefill, "8q1s1k" decode) without describing it. What
// it computes here: sequence b has L_b positions in its paged cache, the
// last n_b of which are its new tokens (already written); new token i
// attends causally to the positions before L_b - n_b + 1 + i. Prefill is
// n_b = L_b. GQA with 8 query heads per KV head, head_dim 128, 64-token
// blocks, BF16 or FP8-e4m3 cache with per-tensor scales.
//
// GB300 design. Unlike decode (8 FLOP per byte, HBM-bound, mma.sync), a
// tile of 16 new tokens x 8 query heads = 128 query rows shares every K / V
// tile, so the work is a dense contraction and runs on tcgen05:
//  * CTA = (KV head, QT tiles of 16 new tokens of one sequence), QT = 1 or 2.
//    Warps: 4 softmax warps per query tile (thread = query row = TMEM lane),
//    4 e4m3 -> f16 converter warps (FP8 caches only), 1 TMA producer warp,
//    1 MMA warp per query tile (the tiles' pipelines never wait on each other).
//  * TMA loads Q once (3-D map over [token][head][128], box 16 x 8 x 64,
//    128-byte swizzle: row t*8+g of the tile is query head g of token t) and
//    the K / V tiles of the sequence's blocks into a shared-memory ring (for
//    FP8, into an e4m3 ring that the converters widen into the 16-bit ring).
//  * FP8 caches run the MMAs in fp16: every e4m3 value is an f16 value (one
//    conversion per pair), each softmax thread converts its own Q row in
//    place to f16 with a power-of-two scale putting the row's max |q| in
//    [2^14, 2^15) (exact for every bf16 value that lands in f16's normal
//    range) and takes the scale back out of its logit scale, and P is packed
//    as f16 (P < 256). BF16 caches run everything in bf16.
//  * S_j = Q K_j^T (M 128, N 64, K 128, both operands K-major in shared
//    memory) into tensor memory; S is single-buffered and S_{j+1} is issued
//    as soon as the softmax warps have copied S_j out.
//  * Online softmax in the log2 domain, one row per thread, no shuffles, with
//    paired f32 math. The running maximum is only moved (and O rescaled in
//    tensor memory) when a row's maximum grows by more than 8 (a factor 256):
//    P = 2^(s - m) then stays below 256, and the final O / l uses one
//    consistent m per row.
//  * P (16-bit pairs) goes back to tensor memory (double-buffered) and
//    O += P V_j (M 128, N 128, K 64) reads A = P from tensor memory and V as
//    the MN-major operand of its tile; O accumulates in tensor memory.
//  * Epilogue: O * v_scale / l -> bf16 rows of out, lse = ln 2 (m + log2 l).
//    A full 16-token tile is staged in its (then free) Q buffer and written
//    by one TMA store per 64-column half; a partial tile row by row.
//  * Every wait is bounded (globaltimer); a timeout sets the error bit, all
//    roles stop issuing, and the CTA drains its copies and MMAs and frees its
//    tensor memory before leaving. No trap, no assert.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "hpc_decode.h"
#include "hpc_internal.h"
#include "prefill.h"
#include "tc05.cuh"

namespace hpc {

namespace {

using namespace tc05;

constexpr int kRows = 128;          // query rows of one MMA tile (16 tokens x 8 heads)
constexpr int kGroupRows = 8;      // query heads per KV head
constexpr uint32_t kQBytes = kRows * 128 * 2;         // 32 KB: two 16 KB column halves
constexpr uint32_t kKVTileBytes = 64 * 128 * 2;       // 16 KB: two 8 KB column halves
constexpr uint32_t kStageBytes = 2 * kKVTileBytes;    // K + V
constexpr uint32_t kKVTileBytes8 = 64 * 128;          // 8 KB: one e4m3 K or V tile
constexpr uint32_t kStageBytes8 = 2 * kKVTileBytes8;  // e4m3 K + V
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// QT query tiles of 128 rows per CTA (QT = 1 or 2). Warps 0 .. 4*QT-1 are
// the softmax warpgroups (warpgroup g owns tile g: rows = TMEM lanes of its
// own S and O columns), then one TMA producer warp and one MMA warp per query
// tile, so the two tiles' S -> softmax -> P*V chains never wait on each other.
template <int QT, bool FP8>
struct Layout {
  // FP8 caches: 4 converter warps widen each e4m3 K / V tile to bf16 in place
  // of the TMA writing bf16 directly
  static constexpr int kConvWarps = FP8 ? 4 : 0;
  static constexpr int kConvWarp0 = 4 * QT;
  static constexpr int kProducerWarp = 4 * QT + kConvWarps, kMmaWarp0 = kProducerWarp + 1;
  static constexpr int kThreads = 32 * (kMmaWarp0 + QT);
  static constexpr int kStages = FP8 ? 4 : (QT == 1 ? 6 : 5);            // 16-bit K+V ring
  static constexpr int kStages8 = FP8 ? (QT == 1 ? 4 : 2) : 0;           // e4m3 K+V ring
  static constexpr uint32_t kOffQ = 0;                                   // QT x 32 KB
  static constexpr uint32_t kOffKV = QT * kQBytes;                       // stages x 32 KB
  static constexpr uint32_t kOffKV8 = kOffKV + kStages * kStageBytes;    // stages8 x 16 KB
  static constexpr uint32_t kOffBar = kOffKV8 + kStages8 * kStageBytes8;
  // q_full, kv_full[S], kv_empty[S], kv8_full[S8], kv8_empty[S8],
  // per tile: s_full, s_free, p_full[2], pv_done[2], drain, q_ready (FP8)
  static constexpr int kNumBars = 1 + 2 * kStages + 2 * kStages8 + 8 * QT;
  static constexpr uint32_t kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr uint32_t kSmemBytes = kOffMisc + 64 + 1024;  // + slack to align to 1024
  // tensor memory per query tile: S (64 columns) | P0, P1 (32 each, bf16 pairs) | O (128)
  static constexpr uint32_t kTmemCols = 256 * QT;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};
constexpr uint32_t kColS = 0, kColP = 64, kColO = 128;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Packed pairs of f32 (sm_100+ paired FMA / add): one instruction, two lanes.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Two e4m3 bytes (low byte -> low half) to f16x2, exactly: every e4m3 value
// is an f16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t x) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(x));
  return h;
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Bounded wait on an mbarrier phase; false when the CTA aborts or the limit
// passes (then the abort flag and the error bit are set).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int32_t* err, unsigned long long limit_ns,
                                         bool honour_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (honour_abort && *abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) {
        if (err) atomicOr(err, HPC_DEVCHK_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct TileInfo {
  int valid;   // 0: no tile for this CTA
  int b;       // sequence
  int t0;      // first new token of the tile (within the sequence)
  int n;       // new tokens of the sequence
  int L;       // positions of the sequence
  int q0;      // row of the sequence's first new token in q / out
  int n_kv;    // KV tiles this CTA reads
};

// Warp-cooperative: map tile index y (heaviest first) to (sequence, tile).
// Every sequence contributes ceil(n_b / tile_tokens) tiles; tiles are numbered in
// sequence order and y counts from the last one, so the CTAs launched first
// take the tiles that see the most keys. Each lane loads its sequence's row
// offset, new-token count and length together (independent loads), so up to
// 32 sequences cost one memory round trip and the found sequence's values
// come from a shuffle, not from a second, dependent load.
__device__ TileInfo find_tile(const ExtendParams& p, int y, int lane, int tile_tokens) {
  TileInfo ti;
  ti.valid = 0;
  const int B = p.num_seqs;
  int q0 = 0, n = 0, L = 0;
  auto lane_seq = [&](int c) -> int {  // tiles of sequence c + lane
    const int b = c + lane;
    q0 = n = L = 0;
    if (b < B) {
      q0 = p.cu_q_lens[b];
      n = p.cu_q_lens[b + 1] - q0;
      L = p.seq_lens[b];
    }
    return n > 0 ? (n + tile_tokens - 1) / tile_tokens : 0;
  };
  int total = 0;
  if (B > 32)  // several chunks: the total first (one chunk: its own sum)
    for (int c = 0; c < B; c += 32) total += warp_sum_i(lane_seq(c));
  int base = 0;
  for (int c = 0; c < B; c += 32) {
    const int nt = lane_seq(c);
    int incl = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int chunk = __shfl_sync(0xffffffffu, incl, 31);
    if (B <= 32) total = chunk;
    if (y >= total) return ti;
    const int gx = total - 1 - y;
    if (gx < base + chunk) {
      const unsigned hit = __ballot_sync(0xffffffffu, gx < base + incl);
      const int f = __ffs(hit) - 1;
      const int incl_f = __shfl_sync(0xffffffffu, incl, f);
      const int nt_f = __shfl_sync(0xffffffffu, nt, f);
      ti.b = c + f;
      ti.t0 = (gx - (base + incl_f - nt_f)) * tile_tokens;
      ti.q0 = __shfl_sync(0xffffffffu, q0, f);
      ti.n = __shfl_sync(0xffffffffu, n, f);
      ti.L = __shfl_sync(0xffffffffu, L, f);
      ti.valid = 1;
      break;
    }
    base += chunk;
  }
  if (!ti.valid) return ti;
  if (ti.L < ti.n) {  // more new tokens than positions
    if (lane == 0 && p.err) atomicOr(p.err, HPC_DEVCHK_BAD_LENGTH);
    ti.valid = 0;
    return ti;
  }
  ti.n_kv = 0;  // per query tile, see tile_kv()
  return ti;
}

// KV tiles read by query tile g of a CTA (16 tokens from t0 + 16 g): the keys
// its last row sees (rows past n clamp to L); 0 when the tile has no row.
__device__ __forceinline__ int tile_kv(int L, int n, int t0g) {
  if (t0g >= n) return 0;
  int kv_len = L - n + t0g + kExtendTileTokens;
  if (kv_len > L) kv_len = L;
  return (kv_len + 63) / 64;
}

}  // namespace

namespace {

template <int QT, bool FP8>
__global__ void __launch_bounds__(Layout<QT, FP8>::kThreads, 1)
    extend_kernel(const __grid_constant__ ExtendParams p, const __grid_constant__ CUtensorMap tmq,
                  const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const __grid_constant__ CUtensorMap tmo) {
  using Lt = Layout<QT, FP8>;
  constexpr int S = Lt::kStages, S8 = Lt::kStages8;
  constexpr int S8n = S8 > 0 ? S8 : 1;  // e4m3 ring positions (the ring exists for FP8 only)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1024-B alignment
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base + Lt::kOffQ, sKV = base + Lt::kOffKV, sKV8 = base + Lt::kOffKV8;
  const uint32_t bars = base + Lt::kOffBar;
  const uint32_t bar_q = bars;
  auto kv_full = [&](int s) { return bars + 8u * (1 + s); };
  auto kv_empty = [&](int s) { return bars + 8u * (1 + S + s); };
  auto kv8_full = [&](int s) { return bars + 8u * (1 + 2 * S + s); };
  auto kv8_empty = [&](int s) { return bars + 8u * (1 + 2 * S + S8 + s); };
  auto gbar = [&](int g, int k) { return bars + 8u * (1 + 2 * S + 2 * S8 + 8 * g + k); };
  auto s_full = [&](int g) { return gbar(g, 0); };
  auto s_free = [&](int g) { return gbar(g, 1); };
  auto p_full = [&](int g, int i) { return gbar(g, 2 + i); };
  auto pv_done = [&](int g, int i) { return gbar(g, 4 + i); };
  auto drain = [&](int g) { return gbar(g, 6); };
  auto q_ready = [&](int g) { return gbar(g, 7); };  // FP8: Q tile g converted to f16
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + Lt::kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + Lt::kOffMisc + 4);
  int* s_info = reinterpret_cast<int*>(smem + Lt::kOffMisc + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const unsigned long long lim_ns = p.timeout_ns;

  if (warp == 0) {
    const TileInfo ti = find_tile(p, blockIdx.y, lane, kExtendTileTokens * QT);
    if (lane == 0) {
      s_info[0] = ti.valid;
      s_info[1] = ti.b;
      s_info[2] = ti.t0;
      s_info[3] = ti.n;
      s_info[4] = ti.L;
      s_info[5] = ti.q0;
    }
  } else if (warp == Lt::kProducerWarp) {
    if (lane == 0) {
      mbar_init(bar_q, 1);
      for (int s = 0; s < S; ++s) {
        // bf16 tile landed: the TMA's transaction count, or the converter threads
        mbar_init(kv_full(s), FP8 ? 32 * Lt::kConvWarps : 1);
        mbar_init(kv_empty(s), QT);  // one arrival per query tile's MMA warp
      }
      for (int s = 0; s < S8; ++s) {
        mbar_init(kv8_full(s), 1);
        mbar_init(kv8_empty(s), 32 * Lt::kConvWarps);
      }
      for (int g = 0; g < QT; ++g) {
        mbar_init(s_full(g), 1);
        mbar_init(s_free(g), kRows);
        for (int i = 0; i < 2; ++i) {
          mbar_init(p_full(g, i), kRows);
          mbar_init(pv_done(g, i), 1);
        }
        mbar_init(drain(g), 1);
        mbar_init(q_ready(g), kRows);
      }
      *s_abort = 0;
      fence_barrier_init();
      prefetch_map(&tmq);
      prefetch_map(&tmk);
      prefetch_map(&tmv);
      prefetch_map(&tmo);
    }
  } else if (warp == Lt::kMmaWarp0) {
    tmem_alloc(smem_u32(s_tmem), Lt::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int valid = s_info[0], b = s_info[1], t0 = s_info[2], n = s_info[3], L = s_info[4],
            q0 = s_info[5];
  int nkv[QT];
  int n_kv = 0;
#pragma unroll
  for (int g = 0; g < QT; ++g) {
    nkv[g] = valid ? tile_kv(L, n, t0 + kExtendTileTokens * g) : 0;
    n_kv = nkv[g] > n_kv ? nkv[g] : n_kv;
  }
  const uint32_t tmem = *s_tmem;
  int32_t* err = p.err;

  if (warp == Lt::kProducerWarp) {
    // ------------------------------------------------------------ producer
    int issued = 0;  // K/V tiles whose copies were issued (in order)
    if (n_kv > 0 && !p.withhold_copies) {  // failure-path test: nothing is issued
      if (lane == 0) {
        mbar_expect_tx(bar_q, QT * kQBytes);
#pragma unroll
        for (int g = 0; g < QT; ++g) {
          const int row = q0 + t0 + kExtendTileTokens * g;
          tma_load_3d(sQ + g * kQBytes, &tmq, bar_q, 0, kGroupRows * h, row);
          tma_load_3d(sQ + g * kQBytes + kQBytes / 2, &tmq, bar_q, 64, kGroupRows * h, row);
        }
      }
      const int c1 = p.kv_swap ? h : 0, c2 = p.kv_swap ? 0 : h;
      int stop = 0;
      for (int j0 = 0; j0 < n_kv && !stop; j0 += 32) {
        const int jj = j0 + lane;
        int blk = -1;
        if (jj < n_kv) {
          if (jj < p.max_blocks) {
            blk = p.block_table[(int64_t)b * p.bt_sb + jj];
            if ((blk < 0 || blk >= p.num_blocks) && err) atomicOr(err, HPC_DEVCHK_BAD_BLOCK);
          } else if (err) {
            atomicOr(err, HPC_DEVCHK_TABLE_TOO_SHORT);
          }
        }
        const int cnt = n_kv - j0 < 32 ? n_kv - j0 : 32;
        for (int u = 0; u < cnt; ++u) {
          const int bk = __shfl_sync(0xffffffffu, blk, u);
          if (lane == 0) {
            const int j = j0 + u;
            if (FP8) {
              // e4m3 tiles (64 rows x 128 bytes, one box each) for the converters
              const int slot = j % S8n, round = j / S8n;
              const bool ok = round == 0 ||
                              wait_bar(kv8_empty(slot), (round - 1) & 1, s_abort, err, lim_ns);
              if (ok) {
                const uint32_t fb = kv8_full(slot);
                const uint32_t dk = sKV8 + slot * kStageBytes8, dv = dk + kKVTileBytes8;
                mbar_expect_tx(fb, kStageBytes8);
                tma_load_4d(dk, &tmk, fb, 0, c1, c2, bk);
                tma_load_4d(dv, &tmv, fb, 0, c1, c2, bk);
                issued = j + 1;
              } else {
                stop = 1;
              }
            } else {
              const int slot = j % S, round = j / S;
              const bool ok =
                  round == 0 || wait_bar(kv_empty(slot), (round - 1) & 1, s_abort, err, lim_ns);
              if (ok) {
                const uint32_t fb = kv_full(slot);
                const uint32_t dk = sKV + slot * kStageBytes, dv = dk + kKVTileBytes;
                mbar_expect_tx(fb, kStageBytes);
                tma_load_4d(dk, &tmk, fb, 0, c1, c2, bk);
                tma_load_4d(dk + kKVTileBytes / 2, &tmk, fb, 64, c1, c2, bk);
                tma_load_4d(dv, &tmv, fb, 0, c1, c2, bk);
                tma_load_4d(dv + kKVTileBytes / 2, &tmv, fb, 64, c1, c2, bk);
                issued = j + 1;
              } else {
                stop = 1;
              }
            }
          }
          stop = __shfl_sync(0xffffffffu, stop, 0);
          if (stop) break;
        }
      }
    }
    named_bar_sync(1, Lt::kThreads);
    // drain: the last copy issued into each slot has landed
    if (lane == 0) {
      constexpr int SR = FP8 ? S8n : S;  // the ring the copies went to
      for (int s = 0; s < SR && s < issued; ++s) {
        const int rounds = (issued - s + SR - 1) / SR;
        wait_bar(FP8 ? kv8_full(s) : kv_full(s), (rounds - 1) & 1, s_abort, err, lim_ns, false);
      }
    }
  } else if (FP8 && warp >= Lt::kConvWarp0 && warp < Lt::kProducerWarp) {
    // -------------------------------------------- e4m3 -> f16 converters
    // Each e4m3 tile (64 token rows x 128 bytes, 128-byte swizzle: 16-byte
    // chunk c of row t at c ^ (t % 8)) is widened exactly (e4m3 values are
    // f16 values) into the f16 tile the MMAs read: two 64-column halves,
    // 8-element chunk c' of row t at c' ^ (t % 8). The scales stay out:
    // k_scale is in the logit scale, v_scale in the epilogue.
    constexpr int kNT = FP8 ? 32 * Lt::kConvWarps : 128;  // (no converters with a bf16 cache)
    static_assert(kNT == 64 || kNT == 128, "2 or 4 converter warps");
    constexpr int kRowSteps = 1024 / kNT / 2;  // items per matrix: rows t in kRowSteps bands
    const int ct = threadIdx.x - 32 * Lt::kConvWarp0;  // 0 .. kNT - 1
    // Work item it of thread ct: matrix it / kRowSteps, row t, 16-byte chunk
    // c. A 16-byte shared access is served 8 threads at a time; each such
    // group takes four chunks of one row and the other four of a row of the
    // opposite swizzle parity, so its e4m3 loads and both of its bf16 stores
    // (chunks 2(c % 4) and 2(c % 4) + 1 of a half, the halves 8 KB apart on
    // the same banks) each cover all 8 bank groups: no bank conflict, and no
    // extra instruction in the loop.
    const int cq = ct & 15, c = cq & 7, cr = ((cq >> 2) & 1) ^ (cq >> 3);
    bool ok = n_kv > 0;
    for (int j = 0; ok && j < n_kv; ++j) {
      const int s8 = j % S8n, sb = j % S;
      ok = __all_sync(0xffffffffu, wait_bar(kv8_full(s8), (j / S8n) & 1, s_abort, err, lim_ns));
      if (ok && j >= S)
        ok = __all_sync(0xffffffffu,
                        wait_bar(kv_empty(sb), ((j / S) - 1) & 1, s_abort, err, lim_ns));
      if (!ok) break;
      const uint32_t e8 = sKV8 + s8 * kStageBytes8, kb = sKV + sb * kStageBytes;
#pragma unroll 2
      for (int it = 0; it < 2 * kRowSteps; ++it) {
        const int mat = it / kRowSteps;
        const int t = (it % kRowSteps) * (64 / kRowSteps) + (ct >> 4) * 2 + cr;
        uint32_t x0, x1, x2, x3;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                     : "r"(e8 + mat * kKVTileBytes8 + t * 128 + ((uint32_t)(c ^ (t & 7)) << 4)));
        uint32_t w[8];
        const uint32_t xs[4] = {x0, x1, x2, x3};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          w[2 * q] = e4m3x2_to_f16x2((uint16_t)(xs[q] & 0xFFFFu));
          w[2 * q + 1] = e4m3x2_to_f16x2((uint16_t)(xs[q] >> 16));
        }
        // elements 16c .. 16c+15 -> half c / 4, 8-element chunks 2(c % 4) and 2(c % 4) + 1
        const int cc = (c & 3) * 2;
        const uint32_t row = kb + mat * kKVTileBytes + (c >> 2) * (kKVTileBytes / 2) + t * 128;
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                         row + ((uint32_t)(cc ^ (t & 7)) << 4)),
                     "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                     : "memory");
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                         row + ((uint32_t)((cc + 1) ^ (t & 7)) << 4)),
                     "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                     : "memory");
      }
      fence_async_shared();  // the MMAs read the bf16 tile through the async proxy
      mbar_arrive(kv8_empty(s8));
      mbar_arrive(kv_full(sb));
    }
    named_bar_sync(1, Lt::kThreads);
  } else if (warp >= Lt::kMmaWarp0) {
    // ---------------------------------------------- MMA issue for tile g
    // The whole warp runs the schedule (waits, descriptor arithmetic) so its
    // values stay warp-uniform; one elected lane issues the MMAs and commits.
    // Descriptors are formed once; per K step only immediates are added to
    // the start-address field (bits 0..13, bytes >> 4).
    const int g = warp - Lt::kMmaWarp0;
    const int nkg = g == 0 ? nkv[0] : nkv[QT - 1];
    const bool leader = elect_one() != 0;
    bool issued_any = false;
    if (n_kv > 0) {
      constexpr uint32_t kIdS =
          FP8 ? idesc_f16_f32(kRows, 64, false, false) : idesc_bf16_f32(kRows, 64, false, false);
      constexpr uint32_t kIdPV =
          FP8 ? idesc_f16_f32(kRows, 128, false, true) : idesc_bf16_f32(kRows, 128, false, true);
      const uint64_t qd = smem_desc_sw128(sQ + g * kQBytes, 16, 1024);
      const uint64_t kd0 = smem_desc_sw128(sKV, 16, 1024);
      // V: MN-major; 64-column halves 8 KB apart, 8-token row groups 1 KB apart
      const uint64_t vd0 = smem_desc_sw128(sKV + kKVTileBytes, kKVTileBytes / 2, 1024);
      const uint32_t dS = tmem + 256u * g + kColS, od = tmem + 256u * g + kColO;
      // O_g += P_g V_i, P from tensor memory (16 keys = 8 columns per step);
      // the K/V slot of tile i is released once this tile's MMAs on it are done
      auto issue_pv = [&](int i) -> bool {
        if (!__all_sync(0xffffffffu,
                        wait_bar(p_full(g, i & 1), (i >> 1) & 1, s_abort, err, lim_ns)))
          return false;
        tc_fence_after();
        const uint64_t vd = vd0 + (uint64_t)((i % S) * (kStageBytes >> 4));
        const uint32_t pa = tmem + 256u * g + kColP + 32u * (uint32_t)(i & 1);
        if (leader) {
          mma_f16_ts(od, pa, vd, kIdPV, i > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 1; kk < 4; ++kk)
            mma_f16_ts(od, pa + 8 * kk, vd + kk * (2048 >> 4), kIdPV, 1u);
          mma_commit(pv_done(g, i & 1));
          mma_commit(kv_empty(i % S));
        }
        __syncwarp();
        return true;
      };
      // S_g(j) = Q_g K_j^T; S is single-buffered, so S(j) waits until the
      // softmax warps have copied S(j-1) out (early in their tile j-1)
      auto issue_s = [&](int j) -> bool {
        const int slot = j % S;
        if (!__all_sync(0xffffffffu,
                        wait_bar(kv_full(slot), (j / S) & 1, s_abort, err, lim_ns)))
          return false;
        if (j >= 1 && !__all_sync(0xffffffffu,
                                  wait_bar(s_free(g), (j - 1) & 1, s_abort, err, lim_ns)))
          return false;
        tc_fence_after();
        const uint64_t kd = kd0 + (uint64_t)(slot * (kStageBytes >> 4));
        if (leader) {
          // Q and K: K-major; 64-column halves (16 KB / 8 KB apart), 16 columns = 32 bytes
          mma_f16_ss(dS, qd, kd, kIdS, 0u);
#pragma unroll
          for (int kk = 1; kk < 8; ++kk)
            mma_f16_ss(dS, qd + (kk >> 2) * ((kQBytes / 2) >> 4) + (kk & 3) * 2,
                       kd + (kk >> 2) * ((kKVTileBytes / 2) >> 4) + (kk & 3) * 2, kIdS, 1u);
          mma_commit(s_full(g));
        }
        __syncwarp();
        return true;
      };
      // software pipeline: S(j+1) runs on the tensor cores while the softmax
      // warps work on tile j; P(j) V_j follows once P(j) is written
      // Q in shared memory: as landed (BF16), or once the softmax warps have
      // converted it to f16 (FP8)
      bool ok = __all_sync(0xffffffffu, wait_bar(FP8 ? q_ready(g) : bar_q, 0, s_abort, err, lim_ns));
      if (ok && nkg > 0) {
        ok = issue_s(0);
        issued_any = true;
      }
      for (int j = 0; ok && j < nkg; ++j) {
        if (j + 1 < nkg) ok = issue_s(j + 1);
        if (ok) ok = issue_pv(j);
      }
      // K/V tiles this query tile does not read still get its arrival, in the
      // right round: once the tile has landed, the slot's previous round is over
      for (int j = nkg; ok && j < n_kv; ++j) {
        ok = __all_sync(0xffffffffu, wait_bar(kv_full(j % S), (j / S) & 1, s_abort, err, lim_ns));
        if (ok && leader) mbar_arrive(kv_empty(j % S));
        __syncwarp();
      }
    }
    if (leader && issued_any) {
      mma_commit(drain(g));  // every MMA this lane issued has completed
      wait_bar(drain(g), 0, s_abort, err, lim_ns, false);
    }
    __syncwarp();
    tc_fence_before();
    named_bar_sync(1, Lt::kThreads);
    tc_fence_after();
    if (warp == Lt::kMmaWarp0) tmem_dealloc(tmem, Lt::kTmemCols);
  } else {
    // ------------------------------------------------ softmax warpgroup g
    const int g = warp >> 2;
    const int r = threadIdx.x - kRows * g;  // query row = TMEM lane
    const int tok = t0 + kExtendTileTokens * g + (r >> 3), head = kGroupRows * h + (r & 7);
    const bool row_ok = valid && tok < n;
    int lim = L - n + 1 + tok;  // keys visible to this row: positions < lim
    if (lim > L) lim = L;
    const int nk = g == 0 ? nkv[0] : nkv[QT - 1];
    // the tile leaves by TMA when all its 16 tokens are new tokens of this
    // sequence (see the epilogue); uniform over the warpgroup
    const bool full = valid && nk > 0 && t0 + kExtendTileTokens * (g + 1) <= n;
    const uint32_t trow = tmem + 256u * g + ((uint32_t)((warp & 3) * 32) << 16);
    bool ok = nk > 0;
    float qinv = 1.f;  // FP8: 2^-e, the scale this row's Q was converted with
    if constexpr (FP8) {
      // Q row r of this tile, both 64-column halves, converted in place from
      // bf16 to f16 with 2^e putting the row's max |q| in [2^14, 2^15): f16
      // holds every bf16 value of that range exactly. Elementwise in place,
      // so the swizzled chunk order of the row does not matter. Every thread
      // arrives on q_ready, with or without work, so the MMA warp's wait ends.
      if (ok) ok = __all_sync(0xffffffffu, wait_bar(bar_q, 0, s_abort, err, lim_ns));
      if (ok) {
        const uint32_t qrow = sQ + g * kQBytes + r * 128;
        // the 16 chunks of the row (2 halves x 8): read for the max, then
        // read again, converted and written back (registers stay free). Row r
        // takes its chunks in the order i ^ (r % 8), so the 8 rows served by
        // one shared-memory wavefront hit 8 different bank groups.
        auto chunk = [&](int i) {
          return qrow + (i >> 3) * (kQBytes / 2) + ((uint32_t)((i & 7) ^ (r & 7)) << 4);
        };
        // max |q| of the row on packed pairs: max.xorsign.abs gives the larger
        // magnitude of each half (its sign is dropped below)
        uint32_t m2[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          uint32_t x[4];
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3])
                       : "r"(chunk(i)));
#pragma unroll
          for (int e = 0; e < 4; ++e)
            asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m2[e]) : "r"(m2[e]), "r"(x[e]));
        }
        float mx = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          mx = fmax3(mx, fabsf(__uint_as_float(m2[e] << 16)),
                     fabsf(__uint_as_float(m2[e] & 0xFFFF0000u)));
        int e2 = 0;
        if (mx > 0.f) {
          e2 = 14 - ((int)((__float_as_uint(mx) >> 23) & 0xFF) - 127);
          e2 = e2 < -100 ? -100 : (e2 > 100 ? 100 : e2);
        }
        const float qs = __uint_as_float((uint32_t)(127 + e2) << 23);
        qinv = __uint_as_float((uint32_t)(127 - e2) << 23);
#pragma unroll 4
        for (int i = 0; i < 16; ++i) {
          uint32_t x[4], y[4];
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3])
                       : "r"(chunk(i)));
#pragma unroll
          for (int e = 0; e < 4; ++e)
            y[e] = pack_f16(__uint_as_float(x[e] << 16) * qs,
                            __uint_as_float(x[e] & 0xFFFF0000u) * qs);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(chunk(i)), "r"(y[0]),
                       "r"(y[1]), "r"(y[2]), "r"(y[3])
                       : "memory");
        }
        fence_async_shared();  // the S MMAs read Q through the async proxy
      }
      mbar_arrive(q_ready(g));
    }
    const float sc = p.score_scale_log2 * qinv;
    float m = -INFINITY, l = 0.f;
    for (int j = 0; ok && j < nk; ++j) {
      ok = __all_sync(0xffffffffu, wait_bar(s_full(g), j & 1, s_abort, err, lim_ns));
      if (!ok) break;
      tc_fence_after();
      float s[64];
      tmem_ld32(trow + kColS, *reinterpret_cast<float(*)[32]>(&s[0]));
      tmem_ld32(trow + kColS + 32, *reinterpret_cast<float(*)[32]>(&s[32]));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(s_free(g));
      const int kv0 = j * 64;
      if (kv0 + 64 > lim) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (kv0 + c >= lim) s[c] = -INFINITY;
      }
      // row maximum: eight independent chains of three-input max
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = s[i];
#pragma unroll
      for (int c = 8; c + 16 <= 64; c += 16)  // columns 8 .. 55
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], s[c + i], s[c + 8 + i]);
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], s[56 + i]);  // columns 56 .. 63
      const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]),
                             fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
      const float m_new = fmaxf(m, mx * sc);
      // move the row maximum only when it grew by more than the threshold
      const bool need = j > 0 && m_new > m + kRescaleThreshold;
      const float m_use = (j == 0 || need) ? m_new : m;
      const float alpha = need ? ex2(m - m_new) : 1.f;
      // exponents s*sc - m in packed pairs; row sum in four packed accumulators
      uint32_t pk[32];
      const uint64_t sc2 = pack2(sc, sc), nm2 = pack2(-m_use, -m_use);
      uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        float x0, x1;
        unpack2(ffma2(pack2(s[2 * c], s[2 * c + 1]), sc2, nm2), x0, x1);
        const float p0 = ex2(x0), p1 = ex2(x1);
        acc2[c & 3] = fadd2(acc2[c & 3], pack2(p0, p1));
        pk[c] = FP8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);  // keys 2c (low half) and 2c + 1
      }
      float r0, r1;
      unpack2(fadd2(fadd2(acc2[0], acc2[1]), fadd2(acc2[2], acc2[3])), r0, r1);
      l = l * alpha + (r0 + r1);
      m = m_use;
      // The P buffer of this tile was last read by P(j-2) V_{j-2}. This query
      // tile's MMA warp issued that MMA before S(j), and the commit behind
      // s_full fires only when every MMA the thread issued earlier has
      // completed: the s_full(j) wait above (and its fence) already ordered it.
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // O is stable once the PV of tile j - 1 is done
        ok = __all_sync(0xffffffffu, wait_bar(pv_done(g, (j - 1) & 1), ((j - 1) >> 1) & 1,
                                              s_abort, err, lim_ns));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float o[32];
          tmem_ld32(trow + kColO + q * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(trow + kColO + q * 32, o);
        }
      }
      // P (bf16 pairs) into this tile's tensor-memory buffer: row = lane
      tmem_st32(trow + kColP + 32u * (uint32_t)(j & 1), pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(p_full(g, j & 1));
    }
    if (ok) {
      ok = __all_sync(0xffffffffu, wait_bar(pv_done(g, (nk - 1) & 1), ((nk - 1) >> 1) & 1,
                                            s_abort, err, lim_ns));
    }
    // A full 16-token tile leaves through shared memory: its Q buffer is free
    // once the tile's last P V is done (every S MMA of the tile came before
    // it), the rows go there in the layout of the Q / out tensor maps
    // (row t*8 + head, 128-byte swizzle), and one thread stores each 64-column
    // half with TMA. A partial tile's box would cover rows of the next
    // sequence, so it is stored row by row. `full` is uniform over the
    // warpgroup, so every thread reaches the staging barrier even when some
    // warp stopped early.
    const uint32_t sQg = sQ + g * kQBytes;
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? p.v_scale / l : 0.f;
      __nv_bfloat16* orow = p.out + (int64_t)(q0 + tok) * p.o_st + (int64_t)head * p.o_sh;
      // O in two rounds of 64 columns: two tensor-memory loads in flight per wait
#pragma unroll
      for (int q = 0; q < 4; q += 2) {
        float o[64];
        tmem_ld32(trow + kColO + q * 32, *reinterpret_cast<float(*)[32]>(&o[0]));
        tmem_ld32(trow + kColO + q * 32 + 32, *reinterpret_cast<float(*)[32]>(&o[32]));
        tmem_wait_ld();
        const uint32_t srow = sQg + (q >> 1) * (kQBytes / 2) + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4 v;
          v.x = pack_bf16(o[8 * c + 0] * inv, o[8 * c + 1] * inv);
          v.y = pack_bf16(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
          v.z = pack_bf16(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
          v.w = pack_bf16(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
          if (full) {
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                             srow + ((uint32_t)(c ^ (r & 7)) << 4)),
                         "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                         : "memory");
          } else if (row_ok) {
            *reinterpret_cast<uint4*>(orow + q * 32 + c * 8) = v;
          }
        }
      }
      if (row_ok && p.lse)
        p.lse[(int64_t)(q0 + tok) * p.l_st + (int64_t)head * p.l_sh] =
            l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
    }
    if (full) {
      fence_async_shared();  // the TMA store reads the rows through the async proxy
      if (g == 0) named_bar_sync(2, kRows); else named_bar_sync(3, kRows);
      if (r == 0 && !*s_abort) {
        // the tile's first row, re-read here rather than held through the loop
        const volatile int* si = s_info;
        const int row = si[5] + si[2] + kExtendTileTokens * g;
        tma_store_3d(&tmo, sQg, 0, kGroupRows * h, row);
        tma_store_3d(&tmo, sQg + kQBytes / 2, 64, kGroupRows * h, row);
        bulk_commit_and_wait_read();  // the buffer is read before the CTA retires
      }
    }
    tc_fence_before();
    named_bar_sync(1, Lt::kThreads);
  }
}

template <int QT, bool FP8>
cudaError_t launch_qt(const ExtendParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                      const CUtensorMap& tv, const CUtensorMap& to, int tiles,
                      cudaStream_t stream) {
  using Lt = Layout<QT, FP8>;
  static std::atomic<uint64_t> configured{0};  // devices whose copy is configured
  const cudaError_t e = once_per_device(configured, [] {
    return cudaFuncSetAttribute(extend_kernel<QT, FP8>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)Lt::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  extend_kernel<QT, FP8><<<dim3(p.num_kv_heads, tiles), Lt::kThreads, Lt::kSmemBytes, stream>>>(
      p, tq, tk, tv, to);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_extend(const ExtendParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& to, int tiles,
                          int tiles_per_cta, cudaStream_t stream) {
  if (tiles <= 0 || p.num_kv_heads <= 0) return cudaSuccess;
  if (p.kv_fp8) {
    if (tiles_per_cta == 2) return launch_qt<2, true>(p, tq, tk, tv, to, tiles, stream);
    return launch_qt<1, true>(p, tq, tk, tv, to, tiles, stream);
  }
  if (tiles_per_cta == 2) return launch_qt<2, false>(p, tq, tk, tv, to, tiles, stream);
  return launch_qt<1, false>(p, tq, tk, tv, to, tiles, stream);
}

}  // namespace hpc
