// One decode step with one query token per sequence, planned, computed and
// merged by a single persistent kernel (hpc_decode_step's path for q
// [B][H_q][128]).
//
// The method ("vLLM x HPC-Ops", section "Attention Backend: Dynamic
// Load-Balanced Scheduling"): every sequence's KV cache is cut into uniform
// 64-token tiles, the tiles are spread over the CTAs of a persistent grid by
// actual work, each CTA computes split-KV attention over its share and
// partial softmax states are merged by log-sum-exp rescaling. This kernel
// takes the unit of work one step finer and orders it so that a CTA's share
// holds whole (sequence, KV head) pairs where it can:
//  * sequence b has n_b * H_kv units, unit u being tile u % n_b of KV head
//    u / n_b; units are flattened in sequence order (T in all);
//  * the first S = T - floor(T / 8) units are split into P = min(G,
//    ceil(S / 8)) balanced contiguous parts (part p = [floor(pS/P),
//    floor((p+1)S/P))), one per CTA; the rest is a pool of chunks of
//    C = max(8, ceil(S / (12 P)), ceil(W / (4 G))) units that CTAs take with
//    an atomic counter as they run out of work, so SMs that stream faster
//    than others take more of it;
//  * a piece is an owner's range (a part or a chunk) intersected with one
//    pair; the 8 consumer warps share a piece's tiles round-robin, then each
//    deposits its state (o = acc / l as 16-bit pairs, (m, l) in fp32) in
//    shared memory and goes on, and an epilogue warp combines the 8 states;
//  * a pair held by one piece is final and written as bf16 out + lse; the k
//    pieces of a split pair each leave a partial state in slot 2*owner (the
//    owner's first piece) or 2*owner + 1 (its last) and count themselves in
//    the pair's arrival counter; the CTA that brings the counter to k merges
//    the k states (M = max m_i, l = sum l_i 2^(m_i - M), out = sum o_i
//    2^(m_i - M) / l) and resets the counter to zero. No merge kernel runs.
//    An owner's pieces run split ones first (its first piece, then its last
//    when that pair continues past the range), whole pairs last, so merges
//    overlap the streaming instead of following it;
//  * every CTA plans the step itself from the device lengths (a prefix scan
//    in shared memory), and CTAs with no static part start on the pool.
//
// Roles: 1 producer warp (pieces, block-table reads, TMA copies of each
// (tile, KV head) K and V tile into a STAGES-deep ring), 8 consumer warps
// (the unit math of decode_common.cuh: S^T = K Q^T and O^T += V^T P^T on
// mma.sync with the online softmax in registers) and 2 epilogue warps taking
// alternate pieces (combine, final or partial writes, arrival counts and
// merges, whose global round trips would otherwise queue behind each other
// at the end of the step). Every wait is bounded; on a
// timeout the CTA keeps walking and publishing its pieces without copies, so
// the arrival counters and the pool still return to zero.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode_common.cuh"
#include "hpc_internal.h"
#include "ptx.cuh"

namespace hpc {
namespace {

constexpr int kSNC = 8;                           // consumer warps
constexpr int kEpilogueWarps = 2;                 // epilogue warps, taking pieces in turn
constexpr int kProducerWarp = kSNC, kEpilogueWarp0 = kSNC + 1;
constexpr int kSThreads = (kSNC + 1 + kEpilogueWarps) * 32;
constexpr int kPieceQ = 4;                        // piece descriptors in flight
// A queue slot always serves the same epilogue warp, so the epilogue warps'
// waits on descriptors are exact like the consumers'.
static_assert(kPieceQ % kEpilogueWarps == 0, "queue slots per epilogue warp");
constexpr int kDescInts = 8;
// A consumer warp's deposit, per lane: its normalised output o = acc / l at
// its 32 positions as 16-bit pairs (4 x 16 bytes) and (m, m, l, l) in fp32.
// With an e4m3 cache |o| <= 448 and the pairs are fp16 (2^-11 rounding); with
// a bf16 cache |o| is bounded only by the cache's values and the pairs are
// bf16, whose range is fp32's. The accumulation itself stays fp32 throughout.
constexpr int kDepSlices = kSNC + 1;              // 8 accumulator slices + (m, l) (partials)
constexpr int kDepVec = 5;                        // 16-byte words per lane in a deposit
constexpr int kDepBytes = kSNC * kDepVec * 32 * 16;  // one state per consumer warp
// Waits on the descriptor queue and the deposits give up only this many data
// waits later: once a data wait has timed out every role runs on without
// copies, and this bookkeeping must then still finish, so that the arrival
// counters and the pool return to zero.
constexpr unsigned long long kBookkeepingWaits = 8;
constexpr int kClaimAhead = 2;                    // units left to issue when the next chunk is asked for
constexpr int kFlagEnd = 1, kFlagWhole = 2;

template <bool FP8, int STAGES>
struct StepCfg {
  static constexpr int kTile = Geom<FP8>::kTileBytes;
  static constexpr int kStage = Geom<FP8>::kStageBytes;
  static constexpr int kDepOff = STAGES * kStage;
  // full, empty, piece full, piece free, deposit full (one per epilogue
  // warp), deposit free
  static constexpr int kNumBars = 2 * STAGES + 2 * kPieceQ + kEpilogueWarps + 1;
  static constexpr int kBarOff = kDepOff + kDepBytes;
  static constexpr int kIssuedOff = kBarOff + 8 * kNumBars;
  static constexpr int kDescOff = kIssuedOff + ((4 * STAGES + 15) / 16) * 16;
  static constexpr int kMiscOff = kDescOff + 4 * kDescInts * kPieceQ;
  static constexpr int kPlanOff = kMiscOff + 256;  // abort flag, flags, scan scratch
  static constexpr int kSmemBytes = 1024 /* alignment slack */ + kPlanOff;
  static constexpr int kSmemBytesMax = kSmemBytes + 4 * (kStepMaxSeqs + 1);
};

// atomicAdd with acquire-release semantics at device scope: the writes that
// happen before it (this thread's, and the warp's through a warp barrier)
// are visible before the addition, and reads after it see what the earlier
// releasers wrote.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int32_t* p, int v) {
  int prev;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(prev) : "l"(p), "r"(v)
               : "memory");
  return prev;
}

template <bool FP8>
__device__ __forceinline__ uint32_t pack_dep(float lo, float hi) {
  return FP8 ? pack_f16(lo, hi) : pack_bf16(lo, hi);
}
template <bool FP8>
__device__ __forceinline__ float2 unpack_dep(uint32_t v) {
  if constexpr (FP8) {
    return __half22float2(*reinterpret_cast<const __half2*>(&v));
  } else {
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
  }
}

// Owner arithmetic of the step plan: parts [0, P) over the first S units,
// then chunks of C units up to T. Every unit index is below T <= INT32_MAX,
// so the arithmetic is 32-bit (short, fast code on a path that runs cold once
// per step); the part formulas take 64 bits only when S * P does not fit.
struct StepMath {
  uint32_t T, S, P, C, chunks;
  bool small;  // (S + 1) * (P + 1) < 2^32
  __device__ __forceinline__ uint32_t part_start(uint32_t o) const {
    return small ? o * S / P : (uint32_t)((uint64_t)o * S / P);
  }
  __device__ __forceinline__ uint32_t start(uint32_t o) const {
    return o < P ? part_start(o) : S + (o - P) * C;
  }
  __device__ __forceinline__ uint32_t end(uint32_t o) const {
    if (o < P) return o + 1 < P ? part_start(o + 1) : S;
    const uint32_t e = S + (o - P + 1) * C;
    return e < T ? e : T;
  }
  __device__ __forceinline__ uint32_t owner_of(uint32_t x) const {
    if (x < S) return small ? ((x + 1) * P - 1) / S : (uint32_t)(((uint64_t)(x + 1) * P - 1) / S);
    return P + (x - S) / C;
  }
};

// Output dims held by a lane in accumulator slice dm (see acc_d).
template <bool FP8>
__device__ __forceinline__ void slice_dims(int dm, int g, int& d0, int& d1) {
  d0 = acc_d<FP8>(dm, 0, g);
  d1 = acc_d<FP8>(dm, 1, g);
}

// Writes this lane's share of a final result: query heads j0, j0 + 1 of
// sequence b at dims d0, d1; o = (j0 d0, j0+1 d0, j0 d1, j0+1 d1).
__device__ __forceinline__ void write_final(const StepParams& p, int b, int j0, int d0, int d1,
                                            float4 o, float inv0, float inv1) {
  __nv_bfloat16* r0 = p.out + (int64_t)b * p.o_sb + (int64_t)j0 * p.o_sh;
  __nv_bfloat16* r1 = r0 + p.o_sh;
  r0[d0] = __float2bfloat16_rn(o.x * inv0);
  r1[d0] = __float2bfloat16_rn(o.y * inv1);
  r0[d1] = __float2bfloat16_rn(o.z * inv0);
  r1[d1] = __float2bfloat16_rn(o.w * inv1);
}

__device__ __forceinline__ float lse_of(float m, float l) {
  return l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
}

// A partial state is stored in the lanes' own layout: [slot][slice][lane]
// float4, slices 0..7 the accumulator (query heads 2c, 2c + 1 at the lane's two
// dims of slice dm), slice 8 the lane's (m, m, l, l) of its two query heads.
constexpr int kPartFloat4 = kDepSlices * 32;

// The warp that counts the last piece of a split pair merges the pair's k
// partial states in owner order (M = max m_i, l = sum l_i 2^(m_i - M),
// out = sum o_i 2^(m_i - M) / l). They were written by other CTAs, which
// released them with their count, and are read from L2 (.cg), never L1.
template <bool FP8>
__device__ __forceinline__ void merge_pair(const StepParams& p, const StepMath& M,
                                           const int32_t* cu, int b, int h, int lane) {
  const int g = lane >> 2, c = lane & 3;
  const uint32_t nb = (uint32_t)(cu[b + 1] - cu[b]) / (uint32_t)p.num_kv_heads;
  const uint32_t A = (uint32_t)cu[b] + (uint32_t)h * nb;
  const uint32_t first = M.owner_of(A), last = M.owner_of(A + nb - 1);
  const float4* part = reinterpret_cast<const float4*>(p.ws_part);
  float M0 = -INFINITY, M1 = -INFINITY, L0 = 0.f, L1 = 0.f;
  float acc[8][4];
#pragma unroll
  for (int dm = 0; dm < 8; ++dm) acc[dm][0] = acc[dm][1] = acc[dm][2] = acc[dm][3] = 0.f;
  constexpr int kBatch = 2;
  for (uint32_t o0 = first; o0 <= last; o0 += kBatch) {
    float4 st[kBatch][kDepSlices];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const uint32_t ow = o0 + u;
      if (ow <= last) {
        const int64_t s = 2 * (int64_t)ow + (A <= M.start(ow) ? 0 : 1);
        const float4* src = part + s * kPartFloat4 + lane;
#pragma unroll
        for (int k = 0; k < kDepSlices; ++k) st[u][k] = __ldcg(src + k * 32);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) st[u][k] = make_float4(0.f, 0.f, 0.f, 0.f);
        st[u][8] = make_float4(-INFINITY, -INFINITY, 0.f, 0.f);
      }
    }
    float N0 = M0, N1 = M1;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      N0 = fmaxf(N0, st[u][8].x);
      N1 = fmaxf(N1, st[u][8].y);
    }
    const float s0 = (M0 == -INFINITY) ? 0.f : ex2(M0 - N0);
    const float s1 = (M1 == -INFINITY) ? 0.f : ex2(M1 - N1);
    L0 *= s0;
    L1 *= s1;
#pragma unroll
    for (int dm = 0; dm < 8; ++dm) {
      acc[dm][0] *= s0; acc[dm][2] *= s0;
      acc[dm][1] *= s1; acc[dm][3] *= s1;
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const float w0 = (st[u][8].x == -INFINITY) ? 0.f : ex2(st[u][8].x - N0);
      const float w1 = (st[u][8].y == -INFINITY) ? 0.f : ex2(st[u][8].y - N1);
      L0 += st[u][8].z * w0;
      L1 += st[u][8].w * w1;
#pragma unroll
      for (int dm = 0; dm < 8; ++dm) {
        acc[dm][0] += st[u][dm].x * w0; acc[dm][2] += st[u][dm].z * w0;
        acc[dm][1] += st[u][dm].y * w1; acc[dm][3] += st[u][dm].w * w1;
      }
    }
    M0 = N0;
    M1 = N1;
  }
  const int j0 = h * kGroup + 2 * c;
  const float inv0 = L0 > 0.f ? 1.f / L0 : 0.f, inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
#pragma unroll
  for (int dm = 0; dm < 8; ++dm) {
    int d0, d1;
    slice_dims<FP8>(dm, g, d0, d1);
    write_final(p, b, j0, d0, d1, make_float4(acc[dm][0], acc[dm][1], acc[dm][2], acc[dm][3]),
                inv0, inv1);
  }
  if (g == 0 && p.lse) {
    float* lr = p.lse + (int64_t)b * p.l_sb + (int64_t)j0 * p.l_sh;
    lr[0] = lse_of(M0, L0);
    lr[p.l_sh] = lse_of(M1, L1);
  }
}

template <bool FP8, int STAGES>
__global__ void __launch_bounds__(kSThreads, 1)
    step_kernel(const __grid_constant__ StepParams p, const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmv) {
  using Cfg = StepCfg<FP8, STAGES>;
  constexpr int kTile = Cfg::kTile;
  constexpr int kStage = Cfg::kStage;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_full = smem_base + Cfg::kBarOff;
  const uint32_t bar_empty = bar_full + 8 * STAGES;
  const uint32_t bar_pfull = bar_empty + 8 * STAGES;
  const uint32_t bar_pfree = bar_pfull + 8 * kPieceQ;
  const uint32_t bar_dfull = bar_pfree + 8 * kPieceQ;  // + 8 * (piece % kEpilogueWarps)
  const uint32_t bar_dfree = bar_dfull + 8 * kEpilogueWarps;
  const uint32_t issued_word = smem_base + Cfg::kIssuedOff;
  int* desc = reinterpret_cast<int*>(smem + Cfg::kDescOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kMiscOff);
  int* s_bad = reinterpret_cast<int*>(smem + Cfg::kMiscOff + 8);
  const unsigned long long book_ns = p.timeout_ns * kBookkeepingWaits;
  int32_t* warp_tot = reinterpret_cast<int32_t*>(smem + Cfg::kMiscOff + 128);
  int32_t* cu = reinterpret_cast<int32_t*>(smem + Cfg::kPlanOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
  const int B = p.num_seqs, H = p.num_kv_heads, G = (int)gridDim.x;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);  // one consumer warp per unit
      reinterpret_cast<volatile uint32_t*>(smem + Cfg::kIssuedOff)[s] = 0xFFFFFFFFu;
    }
    for (int s = 0; s < kPieceQ; ++s) {
      mbar_init(bar_pfull + 8 * s, 1);
      mbar_init(bar_pfree + 8 * s, kSNC + 1);  // the consumer warps and the piece's epilogue warp
    }
    // every consumer warp has deposited its state of the piece; piece j on
    // barrier j % kEpilogueWarps, so each barrier serves one epilogue warp
    // and its phase k is that warp's k-th piece
    for (int e = 0; e < kEpilogueWarps; ++e) mbar_init(bar_dfull + 8 * e, kSNC);
    mbar_init(bar_dfree, 1);     // the epilogue warp has read the deposits
    *abort_flag = 0;
    *s_bad = 0;
    cu[0] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == kProducerWarp && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
  }
  griddep_wait();
  griddep_launch_dependents();
  __syncthreads();

  // ---- plan: units per sequence, prefix in shared memory
  int64_t carry = 0;
  for (int base = 0; base < B; base += kSThreads) {
    const int b = base + tid;
    int32_t n = 0;
    if (b < B) {
      const int32_t len = p.seq_lens[b];
      // a sequence of more units than INT32_MAX / kSThreads is reported, so
      // that no partial sum of a scan pass (kSThreads sequences) wraps
      const int64_t units = len > 0 ? ((int64_t)len + kBlockTokens - 1) / kBlockTokens * H : 0;
      if (len < 0 || units > (int64_t)(INT32_MAX / kSThreads)) *s_bad = 1;
      else n = (int32_t)units;
    }
    int32_t tot;
    const int32_t incl = cta_inclusive_scan(n, warp_tot, &tot);
    if (b < B) cu[b + 1] = (int32_t)(carry + incl);
    carry += tot;
  }
  __syncthreads();
  const bool bad = *s_bad != 0 || carry > INT32_MAX;
  StepMath M;
  M.T = bad ? 0u : (uint32_t)carry;
  const uint32_t W = M.T / kStepPoolDiv;
  M.S = M.T - W;
  {
    const uint32_t want = (M.S + kStepMinPartDiv - 1) / kStepMinPartDiv;  // a unit per consumer warp
    M.P = want < (uint32_t)G ? want : (uint32_t)G;
    // a twelfth of a static part, at least one unit per consumer warp, at
    // most kStepChunksPerCta chunks per CTA
    const uint32_t per = (uint32_t)kStepChunksPerCta * (uint32_t)G;
    uint32_t c = (W + per - 1) / per;
    const uint32_t frac = (uint32_t)kStepPartChunks * M.P;
    const uint32_t twelfth = M.P > 0 ? (M.S + frac - 1) / frac : 0;
    c = c > twelfth ? c : twelfth;
    M.C = c > (uint32_t)kStepMinChunk ? c : (uint32_t)kStepMinChunk;
  }
  M.chunks = (W + M.C - 1) / M.C;
  M.small = (uint64_t)(M.S + 1) * (M.P + 1) < (uint64_t)UINT32_MAX;
  if (blockIdx.x == 0 && tid == 0) {
    if (bad) atomicOr(p.err, HPC_DEVCHK_BAD_LENGTH);
    if (p.words) {
      p.words[kMagic] = kPlanMagic; p.words[kKind] = HPC_PLAN_STEP; p.words[kNumSeqs] = B;
      p.words[kNumParts] = (int32_t)M.P; p.words[kNumTiles] = (int32_t)M.T;
      p.words[kNumSegs] = (int32_t)M.chunks; p.words[kNumSms] = G; p.words[kSplits] = H;
    }
  }
  // sequences without tiles (or a bad step): out = 0, lse = -inf
  for (uint32_t r = blockIdx.x * kSThreads + tid; r < (uint32_t)B * (uint32_t)p.num_q_heads;
       r += (uint32_t)G * kSThreads) {
    const int b = (int)(r / (uint32_t)p.num_q_heads);
    const int j = (int)(r - (uint32_t)b * (uint32_t)p.num_q_heads);
    if (bad || cu[b + 1] == cu[b]) {
      uint4* o = reinterpret_cast<uint4*>(p.out + (int64_t)b * p.o_sb + (int64_t)j * p.o_sh);
#pragma unroll
      for (int i = 0; i < kHeadDim / 8; ++i) o[i] = make_uint4(0u, 0u, 0u, 0u);
      if (p.lse) p.lse[(int64_t)b * p.l_sb + (int64_t)j * p.l_sh] = -INFINITY;
    }
  }

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = evict_first_policy();
    bool stop = p.withhold_copies != 0;  // failure-path test: no copy is issued
    bool lost = false;                   // the consumers stopped taking pieces
    uint32_t g = 0, issued = 0;
    int j = 0;
    // ask the pool for a chunk: the atomic's result is consumed only when
    // the current owner is done, so its latency hides behind the copies
    int pend = 0;
    bool asked = false;
    auto ask = [&]() {
      if (lane == 0) pend = atomicAdd(p.pool, 1);
      asked = true;
    };
    auto resolve = [&]() -> int {
      const int c = __shfl_sync(0xffffffffu, pend, 0);
      asked = false;
      return (uint32_t)c < M.chunks ? (int)(M.P + (uint32_t)c) : -1;
    };
    auto publish = [&](int b, int h, int t0, int t1, int flags, int slot) {
      if (lane == 0 && !lost) {
        const int qs = j % kPieceQ;
        if (!wait_phase(bar_pfree + 8 * qs, ((j / kPieceQ) & 1u) ^ 1u, abort_flag, p.err,
                        book_ns, false)) {
          lost = true;
        } else {
          int* d = desc + qs * kDescInts;
          d[0] = b; d[1] = h; d[2] = t0; d[3] = t1;
          d[4] = flags; d[5] = slot; d[6] = (int)g; d[7] = 0;
          mbar_arrive(bar_pfull + 8 * qs);  // release: the descriptor is visible to its waiters
        }
      }
      ++j;
    };
    int owner;
    if (blockIdx.x < M.P) {
      owner = blockIdx.x;
    } else {
      ask();
      owner = resolve();
    }
    // the sequence holding unit x (cu[b] <= x < cu[b + 1])
    auto seq_at = [&](uint32_t x) -> int {
      int l0 = 0, h0 = B;  // last b with cu[b] <= x, then past empty sequences
      while (h0 - l0 > 1) {
        const int mid = (l0 + h0) >> 1;
        if ((uint32_t)cu[mid] <= x) l0 = mid; else h0 = mid;
      }
      while ((uint32_t)cu[l0 + 1] <= x) ++l0;
      return l0;
    };
    while (owner >= 0) {
      const uint32_t lo = M.start(owner), hi = M.end(owner);
      int npieces = 0;
      // The owner's unit ranges, walked in this order: its first piece; then
      // its last piece when that is the head of a pair continuing past hi;
      // then the whole pairs between them. Both sides of a part boundary are
      // then computed early, so the arrival counts and merges of the pairs
      // that boundaries split overlap the streaming of the rest, and a part
      // ends on a whole pair (a final write). Pieces, slots and every result
      // bit are those of the unit order.
      uint32_t ra = lo, rb = hi;         // the range being walked
      uint32_t rest_a = hi, rest_b = hi;  // whole pairs left for after it
      bool first = false;                 // walking the first of several pieces
      int b = seq_at(lo);
      {
        const uint32_t nb0 = (uint32_t)(cu[b + 1] - cu[b]) / (uint32_t)H;
        const uint32_t e0 = (uint32_t)cu[b] + ((lo - (uint32_t)cu[b]) / nb0 + 1) * nb0;
        if (e0 < hi) {
          rb = e0;
          first = true;
        }
      }
      uint32_t left = hi - lo;  // units of this owner from the current one on
      for (;;) {
        for (uint32_t u = ra; u < rb;) {
          while ((uint32_t)cu[b + 1] <= u) ++b;
          const uint32_t nb = (uint32_t)(cu[b + 1] - cu[b]) / (uint32_t)H;
          const uint32_t rel = u - (uint32_t)cu[b];
          const uint32_t hu = rel / nb;
          const int h = (int)hu, t0 = (int)(rel - hu * nb);
          const uint32_t pair_lo = (uint32_t)cu[b] + hu * nb, pair_hi = pair_lo + nb;
          const uint32_t e = rb < pair_hi ? rb : pair_hi;
          const int t1 = t0 + (int)(e - u);
          const bool whole = t0 == 0 && t1 == (int)nb;
          const int slot = whole ? -1 : (u == lo ? 2 * owner : 2 * owner + 1);
          const int k = whole ? 1 : (int)(M.owner_of(pair_hi - 1) - M.owner_of(pair_lo) + 1);
          publish(b, h, t0, t1, (whole ? kFlagWhole : 0) | (k << 8), slot);
          ++npieces;
          const int32_t* btrow = p.block_table + (int64_t)b * p.bt_sb;
          const int n = t1 - t0;
          const int c1 = p.kv_swap ? h : 0, c2 = p.kv_swap ? 0 : h;
          for (int i0 = 0; i0 < n; i0 += 32) {
            const int i = i0 + lane;
            int blk = p.num_blocks;  // out of range: TMA fills zeros
            if (i < n) {
              const int t = t0 + i;
              if (t < p.max_blocks) {
                const int v = __ldg(btrow + t);
                if (v >= 0 && v < p.num_blocks) blk = v;
                else atomicOr(p.err, HPC_DEVCHK_BAD_BLOCK);
              } else {
                atomicOr(p.err, HPC_DEVCHK_TABLE_TOO_SHORT);
              }
            }
            const int cnt = n - i0 < 32 ? n - i0 : 32;
            for (int ii = 0; ii < cnt; ++ii, ++g, --left) {
              const int bk = __shfl_sync(0xffffffffu, blk, ii);
              if (!asked && left <= (uint32_t)kClaimAhead) ask();
              if (lane != 0 || stop) continue;
              const uint32_t slot_r = g % STAGES;
              if (!wait_phase(bar_empty + 8 * slot_r, ((g / STAGES) & 1u) ^ 1u, abort_flag, p.err,
                              p.timeout_ns)) {
                stop = true;
                continue;
              }
              const uint32_t fb = bar_full + 8 * slot_r;
              const uint32_t dk = smem_base + slot_r * kStage;
              const uint32_t dv = dk + kTile;
              mbar_arrive_expect_tx(fb, kStage);
              if constexpr (FP8) {
                tma_load_4d(dk, &tmk, fb, 0, c1, c2, bk, policy);
                tma_load_4d(dv, &tmv, fb, 0, c1, c2, bk, policy);
              } else {
                tma_load_4d(dk, &tmk, fb, 0, c1, c2, bk, policy);
                tma_load_4d(dk + 8192, &tmk, fb, 64, c1, c2, bk, policy);
                tma_load_4d(dv, &tmv, fb, 0, c1, c2, bk, policy);
                tma_load_4d(dv + 8192, &tmv, fb, 64, c1, c2, bk, policy);
              }
              st_release_shared(issued_word + 4 * slot_r, g);
              issued = g + 1;
            }
          }
          u = e;
        }
        if (first) {  // then the last piece, if split, ahead of the whole pairs
          first = false;
          const uint32_t e0 = rb;
          const int b1 = seq_at(hi - 1);
          const uint32_t nb1 = (uint32_t)(cu[b1 + 1] - cu[b1]) / (uint32_t)H;
          const uint32_t s1 = (uint32_t)cu[b1] + ((hi - 1 - (uint32_t)cu[b1]) / nb1) * nb1;
          if (s1 + nb1 > hi && s1 > e0) {
            rest_a = e0;
            rest_b = s1;
            ra = s1;
            b = b1;
          } else {
            ra = e0;
          }
          rb = hi;
          continue;
        }
        if (rest_a < rest_b) {
          ra = rest_a;
          rb = rest_b;
          rest_a = rest_b;
          b = seq_at(ra);
          continue;
        }
        break;
      }
      if (lane == 0 && p.rec) {
        int32_t* r = p.rec + 4 * owner;
        r[0] = (int32_t)lo;
        r[1] = (int32_t)hi;
        r[2] = npieces;
        atomicAdd(r + 3, 1);
      }
      if (!asked) ask();
      owner = resolve();
    }
    // This CTA's failed request ended its work; the last CTA to get there
    // resets the pool for the next step (every CTA asked for the last time).
    if (lane == 0 && atomicAdd(p.pool + 1, 1) == G - 1) {
      p.pool[0] = 0;
      p.pool[1] = 0;
    }
    // one end marker per epilogue warp (they take alternate pieces; the
    // consumer warps stop at the first)
    for (int e = 0; e < kEpilogueWarps; ++e) publish(0, 0, 0, 0, kFlagEnd, -1);
    named_bar_sync(3, kSThreads);
    if (lane == 0 && *abort_flag) {  // copies may still be landing: wait for the last ones
      for (uint32_t u = issued > (uint32_t)STAGES ? issued - STAGES : 0; u < issued; ++u)
        wait_phase(bar_full + 8 * (u % STAGES), (u / STAGES) & 1u, abort_flag, p.err,
                   1000000000ull, false);
    }
    return;
  }

  float4* dep = reinterpret_cast<float4*>(smem + Cfg::kDepOff);  // [warp][slice][lane]
  if (warp >= kEpilogueWarp0) {
    // ------------------------------------------------------------ epilogue
    // For every piece: combine the consumer warps' 8 states (in warp order,
    // from shared memory), hand the deposit buffer back, then write the
    // result -- final bf16 out + lse for a whole pair, else the piece's
    // partial state and the pair's arrival count, and for the last arriving
    // piece the merge of the pair. The global writes, fences and atomics of
    // this latency-heavy part never hold up the consumer warps.
    const int g8 = lane >> 2, c4 = lane & 3;
    for (int j = warp - kEpilogueWarp0;; j += kEpilogueWarps) {
      const int qs = j % kPieceQ;
      if (!wait_phase(bar_pfull + 8 * qs, (j / kPieceQ) & 1u, abort_flag, p.err, book_ns, false))
        break;
      const int* d = desc + qs * kDescInts;
      const int b = d[0], h = d[1], fl = d[4], slot = d[5];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pfree + 8 * qs);
      if (fl & kFlagEnd) break;
      // the deposits of piece j complete phase j / kEpilogueWarps of this
      // warp's barrier; its next phase needs this warp's read first, so the
      // barrier is at most one phase ahead of the wait and the parity is exact
      if (!wait_phase(bar_dfull + 8 * (j % kEpilogueWarps), (j / kEpilogueWarps) & 1u, abort_flag,
                      p.err, book_ns, false))
        break;
      // the 8 warps' states, combined in warp order
      // acc = sum_v o_v l_v 2^(m_v - M): the unnormalised sum of the 8 states
      const uint4* dep4 = reinterpret_cast<const uint4*>(dep);
      float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
      for (int v = 0; v < kSNC; ++v) {
        const float2 mv =
            *reinterpret_cast<const float2*>(dep4 + (v * kDepVec + 4) * 32 + lane);
        M0 = fmaxf(M0, mv.x);
        M1 = fmaxf(M1, mv.y);
      }
      float L0 = 0.f, L1 = 0.f;
      float acc[8][4];
#pragma unroll
      for (int dm = 0; dm < 8; ++dm) acc[dm][0] = acc[dm][1] = acc[dm][2] = acc[dm][3] = 0.f;
      // a rolled loop: this code runs once per piece and often cold (its
      // instructions fetched from DRAM), so it is kept short
#pragma unroll 1
      for (int v = 0; v < kSNC; ++v) {
        const float4 ml = *reinterpret_cast<const float4*>(dep4 + (v * kDepVec + 4) * 32 + lane);
        const float w0 = ml.x == -INFINITY ? 0.f : ml.z * ex2(ml.x - M0);
        const float w1 = ml.y == -INFINITY ? 0.f : ml.w * ex2(ml.y - M1);
        L0 += w0;
        L1 += w1;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 h4 = dep4[(v * kDepVec + k) * 32 + lane];
          const float2 a = unpack_dep<FP8>(h4.x), b2 = unpack_dep<FP8>(h4.y);
          const float2 c2 = unpack_dep<FP8>(h4.z), d2 = unpack_dep<FP8>(h4.w);
          acc[2 * k][0] += a.x * w0;  acc[2 * k][1] += a.y * w1;
          acc[2 * k][2] += b2.x * w0; acc[2 * k][3] += b2.y * w1;
          acc[2 * k + 1][0] += c2.x * w0; acc[2 * k + 1][1] += c2.y * w1;
          acc[2 * k + 1][2] += d2.x * w0; acc[2 * k + 1][3] += d2.y * w1;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_dfree);  // the consumers may deposit the next piece
      if (fl & kFlagWhole) {
        const int j0 = h * kGroup + 2 * c4;
        const float inv0 = L0 > 0.f ? p.v_scale / L0 : 0.f, inv1 = L1 > 0.f ? p.v_scale / L1 : 0.f;
#pragma unroll
        for (int dm = 0; dm < 8; ++dm) {
          int d0, d1;
          slice_dims<FP8>(dm, g8, d0, d1);
          write_final(p, b, j0, d0, d1,
                      make_float4(acc[dm][0], acc[dm][1], acc[dm][2], acc[dm][3]), inv0, inv1);
        }
        if (g8 == 0 && p.lse) {
          float* lr = p.lse + (int64_t)b * p.l_sb + (int64_t)j0 * p.l_sh;
          lr[0] = lse_of(M0, L0);
          lr[p.l_sh] = lse_of(M1, L1);
        }
        continue;
      }
      // a piece of a split pair: its partial state, then the pair's count
      float4* pd = reinterpret_cast<float4*>(p.ws_part) + (int64_t)slot * kPartFloat4 + lane;
#pragma unroll
      for (int dm = 0; dm < 8; ++dm)
        pd[dm * 32] = make_float4(acc[dm][0] * p.v_scale, acc[dm][1] * p.v_scale,
                                  acc[dm][2] * p.v_scale, acc[dm][3] * p.v_scale);
      pd[8 * 32] = make_float4(M0, M1, L0, L1);
      // One acquire-release atomic by lane 0 counts the piece: its release
      // covers the whole warp's partial writes (ordered before it by the
      // warp barrier), its acquire the other pieces' partials, which the
      // warp's merge reads after the second warp barrier.
      __syncwarp();
      int last = 0;
      if (lane == 0) {
        int32_t* cnt = p.pair_cnt + (int64_t)b * H + h;
        last = atom_add_acq_rel_gpu(cnt, 1) == (fl >> 8) - 1;
        if (last) *cnt = 0;  // every piece of the pair has arrived: ready for the next step
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      __syncwarp();
      if (last) merge_pair<FP8>(p, M, cu, b, h, lane);
    }
    named_bar_sync(3, kSThreads);
    return;
  }

  // -------------------------------------------------------------- consumers
  // The consumer warps take a piece's units round-robin and deposit their
  // states; they never wait for each other, only for the deposit buffer to
  // be handed back by the epilogue warp.
  const int w = warp;
  bool dead = false;
  for (int j = 0;; ++j) {
    const int qs = j % kPieceQ;
    if (!wait_phase(bar_pfull + 8 * qs, (j / kPieceQ) & 1u, abort_flag, p.err, book_ns, false))
      break;  // no descriptor arrived: the producer is gone
    const int* d = desc + qs * kDescInts;
    const int b = d[0], h = d[1], t0 = d[2], t1 = d[3], fl = d[4], g0 = d[6];
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_pfree + 8 * qs);  // this warp has read the descriptor
    if (fl & kFlagEnd) break;
    const int n = t1 - t0;
    // tile t of pair (b, h) goes to warp (t + b * H_kv + h) % 8: a function of
    // the piece alone, so a piece gives the same bits whichever CTA runs it
    const int rot = (int)(((int64_t)t0 + (int64_t)b * H + h) & (kSNC - 1));
    const int i0 = (w - rot + kSNC) & (kSNC - 1);  // this warp's first unit
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float acc[8][4];
#pragma unroll
    for (int dm = 0; dm < 8; ++dm) acc[dm][0] = acc[dm][1] = acc[dm][2] = acc[dm][3] = 0.f;
    if (i0 < n) {
      const int len = __ldg(p.seq_lens + b);
      uint32_t qf[8][2];
      const float qinv = load_q<FP8>(p.q + (int64_t)b * p.q_sb + (int64_t)(h * kGroup) * p.q_sh,
                                     p.q_sh, lane, qf);
      const float sl2 = p.score_scale_log2 * qinv;
      for (int i = i0; i < n; i += kSNC) {
        const uint32_t gu = (uint32_t)(g0 + i);
        const uint32_t s = gu % STAGES;
        if (dead) continue;
        const bool ok = wait_issued(issued_word + 4 * s, gu, abort_flag, p.err, p.timeout_ns) &&
                        wait_phase(bar_full + 8 * s, (gu / STAGES) & 1u, abort_flag, p.err,
                                   p.timeout_ns);
        if (!__all_sync(0xffffffffu, ok)) {  // warp-uniform decision
          dead = true;
          continue;
        }
        const int valid = len - (t0 + i) * kBlockTokens;
        if (valid > 0) {
          const uint32_t kb = smem_base + s * kStage;
          compute_unit<FP8>(kb, kb + kTile, qf, valid, sl2, m, l, acc, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
      }
    }
    // row sums over the 8 lanes sharing a query-head pair
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], o);
      l[1] += __shfl_xor_sync(0xffffffffu, l[1], o);
    }
    // deposit once the epilogue warp has read the previous piece's states
    wait_phase(bar_dfree, (j & 1u) ^ 1u, abort_flag, p.err, book_ns, false);
    {
      // approximate reciprocals: the result is rounded to 16 bits right after
      const float i0 = l[0] > 0.f ? __fdividef(1.f, l[0]) : 0.f;
      const float i1 = l[1] > 0.f ? __fdividef(1.f, l[1]) : 0.f;
      uint4* dw = reinterpret_cast<uint4*>(dep) + (w * kDepVec) * 32 + lane;
#pragma unroll
      for (int k = 0; k < 4; ++k)  // slices 2k, 2k + 1
        dw[k * 32] = make_uint4(pack_dep<FP8>(acc[2 * k][0] * i0, acc[2 * k][1] * i1),
                                pack_dep<FP8>(acc[2 * k][2] * i0, acc[2 * k][3] * i1),
                                pack_dep<FP8>(acc[2 * k + 1][0] * i0, acc[2 * k + 1][1] * i1),
                                pack_dep<FP8>(acc[2 * k + 1][2] * i0, acc[2 * k + 1][3] * i1));
      reinterpret_cast<float4*>(dw)[4 * 32] = make_float4(m[0], m[1], l[0], l[1]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_dfull + 8 * (j % kEpilogueWarps));  // release to the epilogue
  }
  named_bar_sync(3, kSThreads);  // see the producer's exit
}

template <bool FP8, int STAGES>
cudaError_t launch_step_cfg(const StepParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                            int grid, cudaStream_t stream) {
  using Cfg = StepCfg<FP8, STAGES>;
  auto kern = step_kernel<FP8, STAGES>;
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = once_per_device(configured, [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg::kSmemBytesMax);
  });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kSThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes + 4 * ((size_t)p.num_seqs + 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, tk, tv);
}

}  // namespace

cudaError_t launch_step(const StepParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                        bool fp8, int grid, cudaStream_t stream) {
  if (p.num_seqs > kStepMaxSeqs) return cudaErrorInvalidValue;
  return fp8 ? launch_step_cfg<true, 12>(p, tk, tv, grid, stream)
             : launch_step_cfg<false, 6>(p, tk, tv, grid, stream);
}

}  // namespace hpc
