// Multi-token split-KV decode on the 5th-generation tensor cores (tcgen05),
// for sm_103a.
//
// The method is the decode path of "vLLM x HPC-Ops" (section "Attention
// Backend: Dynamic Load-Balanced Scheduling"): the per-step planner cuts
// every sequence's KV cache into 64-token tiles and gives each part of the
// persistent grid an equal share; partial softmax states of a sequence
// spread over several parts are combined by the log-sum-exp merge. With
// q_len new tokens per sequence (speculative or multi-token decode), the
// q_len x 8 query rows of one KV head share every K / V tile, so the tile
// products are small dense contractions: here they run on tcgen05 with the
// accumulators in tensor memory instead of in the registers of one warp per
// query token.
//
// Design (the extend kernel's pipeline, made persistent over segments):
//  * CTA = (KV head h, plan part y); it walks the part's segments (sequence
//    b, tiles [tb, te)) in order. Warps: 4 softmax warps (thread = query row
//    = TMEM lane; row 8t + g is token t, query head g), 8 e4m3 -> f16
//    converter warps (FP8 caches only: 8 warps widen a tile in half the time
//    of 4), 1 TMA producer warp, 1 MMA warp.
//  * FP8 caches run the MMAs in fp16: every e4m3 value is an f16 value (one
//    conversion per pair); at the start of each segment every softmax thread
//    converts its own Q row in place to f16 with a power-of-two scale putting
//    the row's max |q| in [2^14, 2^15) and keeps the inverse for its logit
//    scale; P is packed as f16. The MMA warp starts a segment's S MMAs once
//    every softmax thread has arrived on q_ready.
//  * Q of a segment: one TMA per 64-column half (box 64 x 8 heads x q_len
//    tokens, 128-byte swizzle) into one of two 16 KB Q slots, so the next
//    segment's Q loads while this one finishes. Rows past 8 q_len are never
//    written; their S and O rows are not read.
//  * K / V tiles stream through a shared-memory ring (for FP8 an e4m3 ring
//    the converters widen into the bf16 ring). Ring slots and the S / P
//    barrier phases count tiles over the whole CTA, across segments.
//  * S_j = Q K_j^T (M 128, N 64, K 128) into tensor memory; online softmax in
//    the log2 domain with the running maximum moved only when it grows by
//    more than 8 (P = 2^(s - m) < 256); P (16-bit) back to tensor memory;
//    O += P V_j (M 128, N 128, K 64) with A = P from tensor memory and V as
//    the MN-major operand. The first P V of a segment (accumulate off)
//    overwrites O: it waits for P of the segment's first tile, which the
//    softmax warps write only after their epilogue of the previous segment
//    has read O out, so no barrier of its own is needed.
//  * Epilogue per segment: a sequence held whole by this segment gets its
//    bf16 rows (O v_scale / l) and lse; otherwise the unnormalised partial
//    (O v_scale, m, l) goes to the workspace row (segment, token, head) that
//    the merge kernel reads. A row with no visible key leaves m = -inf,
//    l = 0.
//  * Every wait is bounded (globaltimer); a timeout sets the error bit, all
//    roles stop issuing, and the CTA drains its copies and MMAs and frees its
//    tensor memory before leaving. No trap, no assert.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode_tc.h"
#include "hpc_decode.h"
#include "hpc_internal.h"
#include "ptx.cuh"
#include "tc05.cuh"

namespace hpc {

namespace {

using namespace tc05;

constexpr int kRows = 128;                      // MMA rows (query rows 8t + g, t < q_len)
constexpr int kGroupRows = 8;                   // query heads per KV head
constexpr uint32_t kQSlotBytes = 16384;         // one Q slot: two 8 KB column halves
constexpr uint32_t kQHalfBytes = 8192;          // 64 rows x 128 bytes
constexpr uint32_t kKVTileBytes = 64 * 128 * 2;     // 16 KB: two 8 KB column halves
constexpr uint32_t kStageBytes = 2 * kKVTileBytes;  // K + V
constexpr uint32_t kKVTileBytes8 = 64 * 128;        // 8 KB: one e4m3 K or V tile
constexpr uint32_t kStageBytes8 = 2 * kKVTileBytes8;
constexpr uint32_t kColS = 0, kColP = 64, kColO = 128, kTmemCols = 256;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <bool FP8>
struct TcLayout {
  static constexpr int kConvWarps = FP8 ? 8 : 0;
  static constexpr int kConvWarp0 = 4;
  static constexpr int kProducerWarp = 4 + kConvWarps, kMmaWarp = kProducerWarp + 1;
  static constexpr int kThreads = 32 * (kMmaWarp + 1);
  static constexpr int kStages = FP8 ? 4 : 6;   // bf16 K+V ring
  static constexpr int kStages8 = FP8 ? 4 : 0;  // e4m3 K+V ring
  static constexpr uint32_t kOffQ = 0;          // 2 Q slots
  static constexpr uint32_t kOffKV = 2 * kQSlotBytes;
  static constexpr uint32_t kOffKV8 = kOffKV + kStages * kStageBytes;
  static constexpr uint32_t kOffBar = kOffKV8 + kStages8 * kStageBytes8;
  // q_full[2], q_empty[2], kv_full[S], kv_empty[S], kv8_full[S8], kv8_empty[S8],
  // s_full, s_free, p_full[2], pv_done[2], drain, q_ready[2]
  static constexpr int kNumBars = 4 + 2 * kStages + 2 * kStages8 + 9;
  static constexpr uint32_t kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;  // + slack to align to 1024
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

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
// Two e4m3 bytes (low byte -> low half) to bf16x2, exactly.
// Two e4m3 bytes (low byte -> low half) to f16x2, exactly.
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

// One segment record of the plan: sequence b, tiles [tb, te), whole flag.
struct Seg {
  int b, tb, te;
  bool whole;
};
__device__ __forceinline__ Seg read_seg(const DecodeTcParams& p, int sg) {
  const int4 rec = *reinterpret_cast<const int4*>(p.plan + p.seg_off + 4 * (int64_t)sg);
  Seg s;
  s.b = rec.x;
  s.tb = rec.y;
  s.te = rec.z;
  s.whole = (rec.w & HPC_SEG_WHOLE) != 0;
  return s;
}

template <bool FP8>
__global__ void __launch_bounds__(TcLayout<FP8>::kThreads, 1)
    decode_tc_kernel(const __grid_constant__ DecodeTcParams p,
                     const __grid_constant__ CUtensorMap tmq,
                     const __grid_constant__ CUtensorMap tmk,
                     const __grid_constant__ CUtensorMap tmv) {
  using Lt = TcLayout<FP8>;
  constexpr int S = Lt::kStages, S8 = Lt::kStages8;
  constexpr int S8n = S8 > 0 ? S8 : 1;  // e4m3 ring positions (the ring exists for FP8 only)
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1024-B alignment
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base + Lt::kOffQ, sKV = base + Lt::kOffKV, sKV8 = base + Lt::kOffKV8;
  const uint32_t bars = base + Lt::kOffBar;
  auto q_full = [&](int i) { return bars + 8u * i; };
  auto q_empty = [&](int i) { return bars + 8u * (2 + i); };
  auto kv_full = [&](int s) { return bars + 8u * (4 + s); };
  auto kv_empty = [&](int s) { return bars + 8u * (4 + S + s); };
  auto kv8_full = [&](int s) { return bars + 8u * (4 + 2 * S + s); };
  auto kv8_empty = [&](int s) { return bars + 8u * (4 + 2 * S + S8 + s); };
  const uint32_t bar1 = bars + 8u * (4 + 2 * S + 2 * S8);
  const uint32_t s_full = bar1, s_free = bar1 + 8;
  auto p_full = [&](int i) { return bar1 + 16u + 8u * i; };
  auto pv_done = [&](int i) { return bar1 + 32u + 8u * i; };
  const uint32_t drain = bar1 + 48;
  auto q_ready = [&](int i) { return bar1 + 56u + 8u * i; };  // FP8: Q slot i converted
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + Lt::kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + Lt::kOffMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x, part = blockIdx.y;
  const int T = p.q_len;
  const unsigned long long lim_ns = p.timeout_ns;
  int32_t* err = p.err;

  if (warp == Lt::kProducerWarp) {
    if (lane == 0) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(q_full(i), 1);
        mbar_init(q_empty(i), 1);  // the MMA warp's commit after a segment's last S
      }
      for (int s = 0; s < S; ++s) {
        mbar_init(kv_full(s), FP8 ? 32 * Lt::kConvWarps : 1);
        mbar_init(kv_empty(s), 1);
      }
      for (int s = 0; s < S8; ++s) {
        mbar_init(kv8_full(s), 1);
        mbar_init(kv8_empty(s), 32 * Lt::kConvWarps);
      }
      mbar_init(s_full, 1);
      mbar_init(s_free, kRows);
      for (int i = 0; i < 2; ++i) {
        mbar_init(p_full(i), kRows);
        mbar_init(pv_done(i), 1);
      }
      mbar_init(drain, 1);
      for (int i = 0; i < 2; ++i) mbar_init(q_ready(i), kRows);
      *s_abort = 0;
      fence_barrier_init();
      prefetch_map(&tmq);
      prefetch_map(&tmk);
      prefetch_map(&tmv);
    }
  } else if (warp == Lt::kMmaWarp) {
    tmem_alloc(smem_u32(s_tmem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  griddep_wait();  // the plan (and inputs) of the preceding kernels are visible
  griddep_launch_dependents();

  // this CTA's segments (every role walks the same list)
  int sg0 = 0, sg1 = 0;
  if (part < p.plan[kNumParts]) {
    sg0 = p.plan[p.part_off + part];
    sg1 = p.plan[p.part_off + part + 1];
  }
  const uint32_t tmem = *s_tmem;

  if (warp == Lt::kProducerWarp) {
    // ------------------------------------------------------------ producer
    int issued = 0, q_issued = 0;  // K/V tiles and Q loads issued (in order)
    int stop = p.withhold_copies != 0 ? 1 : 0;  // failure-path test: nothing is issued
    const int c1 = p.kv_swap ? h : 0, c2 = p.kv_swap ? 0 : h;
    int G = 0, k = 0;  // tiles and segments before this one
    for (int sg = sg0; sg < sg1 && !stop; ++sg) {
      const Seg sgm = read_seg(p, sg);
      const int n = sgm.te - sgm.tb;
      if (n <= 0) continue;
      if (lane == 0) {
        const int L = p.seq_lens[sgm.b];
        const int nt = L > 0 ? (L + 63) / 64 : 0;
        if (sgm.te > nt || (sgm.whole && (sgm.tb != 0 || sgm.te != nt)))
          atomicOr(err, HPC_DEVCHK_BAD_LENGTH);
        // Q slot k % 2 is free once the S MMAs of segment k - 2 are done
        const bool ok = k < 2 || wait_bar(q_empty(k & 1), ((k >> 1) - 1) & 1, s_abort, err, lim_ns);
        if (ok) {
          const uint32_t dq = sQ + (uint32_t)(k & 1) * kQSlotBytes;
          mbar_expect_tx(q_full(k & 1), 2u * kQHalfBytes / 8u * (uint32_t)T);
          tma_load_4d(dq, &tmq, q_full(k & 1), 0, kGroupRows * h, 0, sgm.b);
          tma_load_4d(dq + kQHalfBytes, &tmq, q_full(k & 1), 64, kGroupRows * h, 0, sgm.b);
          q_issued = k + 1;
        } else {
          stop = 1;
        }
      }
      stop = __shfl_sync(0xffffffffu, stop, 0);
      const int32_t* btrow = p.block_table + (int64_t)sgm.b * p.bt_sb;
      for (int j0 = 0; j0 < n && !stop; j0 += 32) {
        const int jj = sgm.tb + j0 + lane;  // tile of the sequence
        int blk = -1;                       // out of range: TMA fills zeros
        if (j0 + lane < n) {
          if (jj < p.max_blocks) {
            const int v = __ldg(btrow + jj);
            if (v >= 0 && v < p.num_blocks) blk = v;
            else atomicOr(err, HPC_DEVCHK_BAD_BLOCK);
          } else {
            atomicOr(err, HPC_DEVCHK_TABLE_TOO_SHORT);
          }
        }
        const int cnt = n - j0 < 32 ? n - j0 : 32;
        for (int u = 0; u < cnt; ++u) {
          const int bk = __shfl_sync(0xffffffffu, blk, u);
          if (lane == 0) {
            const int g = G + j0 + u;  // position in the CTA's tile stream
            if (FP8) {
              const int slot = g % S8n, round = g / S8n;
              const bool ok = round == 0 ||
                              wait_bar(kv8_empty(slot), (round - 1) & 1, s_abort, err, lim_ns);
              if (ok) {
                const uint32_t fb = kv8_full(slot);
                const uint32_t dk = sKV8 + slot * kStageBytes8, dv = dk + kKVTileBytes8;
                mbar_expect_tx(fb, kStageBytes8);
                tma_load_4d(dk, &tmk, fb, 0, c1, c2, bk);
                tma_load_4d(dv, &tmv, fb, 0, c1, c2, bk);
                issued = g + 1;
              } else {
                stop = 1;
              }
            } else {
              const int slot = g % S, round = g / S;
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
                issued = g + 1;
              } else {
                stop = 1;
              }
            }
          }
          stop = __shfl_sync(0xffffffffu, stop, 0);
          if (stop) break;
        }
      }
      G += n;
      ++k;
    }
    named_bar_sync(1, Lt::kThreads);
    // drain: the last copy issued into each ring slot and each Q slot has landed
    if (lane == 0) {
      constexpr int SR = FP8 ? S8n : S;  // the ring the copies went to
      for (int s = 0; s < SR && s < issued; ++s) {
        const int rounds = (issued - s + SR - 1) / SR;
        wait_bar(FP8 ? kv8_full(s) : kv_full(s), (rounds - 1) & 1, s_abort, err, lim_ns, false);
      }
      for (int i = 0; i < 2 && i < q_issued; ++i) {
        const int uses = (q_issued - i + 1) / 2;
        wait_bar(q_full(i), (uses - 1) & 1, s_abort, err, lim_ns, false);
      }
    }
  } else if (FP8 && warp >= Lt::kConvWarp0 && warp < Lt::kProducerWarp) {
    // -------------------------------------------- e4m3 -> f16 converters
    // Each e4m3 tile (64 token rows x 128 bytes, 128-byte swizzle: 16-byte
    // chunk c of row t at c ^ (t % 8)) is widened exactly into the f16 tile
    // the MMAs read (two 64-column halves, 8-element chunk c' of row t at
    // c' ^ (t % 8)). With 8 warps threads 0..127 widen K and 128..255 V; with
    // 4 warps each thread takes a K item, then a V item. Thread-to-chunk map:
    // each group of 8 threads serving one 16-byte access covers all 8 bank
    // groups on the load and both stores.
    constexpr int kNT = FP8 ? 32 * Lt::kConvWarps : 256;  // (no converters with a bf16 cache)
    static_assert(kNT == 128 || kNT == 256, "4 or 8 converter warps");
    const int ct = threadIdx.x - 32 * Lt::kConvWarp0;  // 0 .. kNT - 1
    const int ctl = ct & 127;
    const int cq = ctl & 15, c = cq & 7, cr = ((cq >> 2) & 1) ^ (cq >> 3);
    bool ok = true;
    int G = 0;
    for (int sg = sg0; sg < sg1 && ok; ++sg) {
      const Seg sgm = read_seg(p, sg);
      const int n = sgm.te - sgm.tb;
      if (n <= 0) continue;
      for (int j = 0; ok && j < n; ++j) {
        const int g = G + j;
        const int s8 = g % S8n, sb = g % S;
        ok = __all_sync(0xffffffffu, wait_bar(kv8_full(s8), (g / S8n) & 1, s_abort, err, lim_ns));
        if (ok && g >= S)
          ok = __all_sync(0xffffffffu,
                          wait_bar(kv_empty(sb), ((g / S) - 1) & 1, s_abort, err, lim_ns));
        if (!ok) break;
        const uint32_t e8 = sKV8 + s8 * kStageBytes8, kb = sKV + sb * kStageBytes;
#pragma unroll 4
        for (int it = 0; it < 1024 / kNT; ++it) {
          const int mat = kNT == 256 ? ct >> 7 : it >> 2;
          const int t = (it & 3) * 16 + (ctl >> 4) * 2 + cr;
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
        fence_async_shared();  // the MMAs read the f16 tile through the async proxy
        mbar_arrive(kv8_empty(s8));
        mbar_arrive(kv_full(sb));
      }
      G += n;
    }
    named_bar_sync(1, Lt::kThreads);
  } else if (warp == Lt::kMmaWarp) {
    // ---------------------------------------------------------- MMA issue
    // The whole warp runs the schedule so its values stay warp-uniform; one
    // elected lane issues the MMAs and commits.
    const bool leader = elect_one() != 0;
    bool issued_any = false;
    constexpr uint32_t kIdS =
        FP8 ? idesc_f16_f32(kRows, 64, false, false) : idesc_bf16_f32(kRows, 64, false, false);
    constexpr uint32_t kIdPV =
        FP8 ? idesc_f16_f32(kRows, 128, false, true) : idesc_bf16_f32(kRows, 128, false, true);
    const uint64_t kd0 = smem_desc_sw128(sKV, 16, 1024);
    // V: MN-major; 64-column halves 8 KB apart, 8-token row groups 1 KB apart
    const uint64_t vd0 = smem_desc_sw128(sKV + kKVTileBytes, kKVTileBytes / 2, 1024);
    const uint32_t dS = tmem + kColS, od = tmem + kColO;
    // O += P(g) V_g, P from tensor memory (16 keys = 8 columns per step); the
    // ring slot of tile g is released once the MMAs on it are done
    auto issue_pv = [&](int g, bool acc) -> bool {
      if (!__all_sync(0xffffffffu, wait_bar(p_full(g & 1), (g >> 1) & 1, s_abort, err, lim_ns)))
        return false;
      tc_fence_after();
      const uint64_t vd = vd0 + (uint64_t)((g % S) * (kStageBytes >> 4));
      const uint32_t pa = tmem + kColP + 32u * (uint32_t)(g & 1);
      if (leader) {
        mma_f16_ts(od, pa, vd, kIdPV, acc ? 1u : 0u);
#pragma unroll
        for (int kk = 1; kk < 4; ++kk) mma_f16_ts(od, pa + 8 * kk, vd + kk * (2048 >> 4), kIdPV, 1u);
        mma_commit(pv_done(g & 1));
        mma_commit(kv_empty(g % S));
      }
      __syncwarp();
      return true;
    };
    // S(g) = Q K_g^T into the single S buffer, once the softmax warps have
    // copied S(g - 1) out; after a segment's last S its Q slot is released
    auto issue_s = [&](int g, uint64_t qd, int q_release) -> bool {
      const int slot = g % S;
      if (!__all_sync(0xffffffffu, wait_bar(kv_full(slot), (g / S) & 1, s_abort, err, lim_ns)))
        return false;
      if (g >= 1 &&
          !__all_sync(0xffffffffu, wait_bar(s_free, (g - 1) & 1, s_abort, err, lim_ns)))
        return false;
      tc_fence_after();
      const uint64_t kd = kd0 + (uint64_t)(slot * (kStageBytes >> 4));
      if (leader) {
        // Q and K: K-major; 64-column halves (8 KB apart), 16 columns = 32 bytes
        mma_f16_ss(dS, qd, kd, kIdS, 0u);
#pragma unroll
        for (int kk = 1; kk < 8; ++kk)
          mma_f16_ss(dS, qd + (kk >> 2) * (kQHalfBytes >> 4) + (kk & 3) * 2,
                     kd + (kk >> 2) * ((kKVTileBytes / 2) >> 4) + (kk & 3) * 2, kIdS, 1u);
        mma_commit(s_full);
        if (q_release >= 0) mma_commit(q_empty(q_release));
      }
      __syncwarp();
      return true;
    };
    bool ok = true;
    int G = 0, k = 0;
    for (int sg = sg0; sg < sg1 && ok; ++sg) {
      const Seg sgm = read_seg(p, sg);
      const int n = sgm.te - sgm.tb;
      if (n <= 0) continue;
      // Q of the segment: as landed (BF16), or converted to f16 (FP8)
      ok = __all_sync(0xffffffffu, wait_bar(FP8 ? q_ready(k & 1) : q_full(k & 1), (k >> 1) & 1,
                                            s_abort, err, lim_ns));
      if (!ok) break;
      const uint64_t qd = smem_desc_sw128(sQ + (uint32_t)(k & 1) * kQSlotBytes, 16, 1024);
      // software pipeline: S(g+1) runs while the softmax warps work on tile g;
      // P(g) V_g follows once P(g) is written
      ok = issue_s(G, qd, n == 1 ? (k & 1) : -1);
      issued_any = true;
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) ok = issue_s(G + j + 1, qd, j + 2 == n ? (k & 1) : -1);
        if (ok) ok = issue_pv(G + j, j > 0);
      }
      G += n;
      ++k;
    }
    if (leader && issued_any) {
      mma_commit(drain);  // every MMA this lane issued has completed
      wait_bar(drain, 0, s_abort, err, lim_ns, false);
    }
    __syncwarp();
    tc_fence_before();
    named_bar_sync(1, Lt::kThreads);
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  } else if (warp < 4) {
    // ---------------------------------------------------- softmax warpgroup
    const int r = threadIdx.x;  // query row = TMEM lane
    const int t = r >> 3, head = kGroupRows * h + (r & 7);
    const bool row_ok = t < T;
    // warps whose 32 rows are all past the q_len tokens only keep the
    // barrier counts (their S, P and O rows are never read)
    const bool live = 32 * warp < kGroupRows * T;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    const float sc0 = p.score_scale_log2;
    bool ok = true;
    int G = 0, k = 0;
    for (int sg = sg0; sg < sg1 && ok; ++sg) {
      const Seg sgm = read_seg(p, sg);
      const int n = sgm.te - sgm.tb;
      if (n <= 0) continue;
      const int L = p.seq_lens[sgm.b];
      // keys visible to this row: positions < lim (the q_len new tokens are
      // the last q_len positions of the sequence). Rows past the q_len tokens
      // are not masked (their values are never read) so that a warp holding
      // some of them does not run the masking loop on every tile.
      const int lim = row_ok ? L - (T - 1 - t) : 0x7FFFFFFF;
      float sc = sc0;
      if constexpr (FP8) {
        // this segment's Q row, both 64-column halves, converted in place from
        // bf16 to f16 with 2^e putting the row's max |q| in [2^14, 2^15) (f16
        // holds every bf16 value of that range exactly); chunk i of row r in
        // the order i ^ (r % 8), so one shared-memory wavefront's 8 rows hit 8
        // bank groups. Every thread arrives on q_ready, with a row or not.
        ok = __all_sync(0xffffffffu, wait_bar(q_full(k & 1), (k >> 1) & 1, s_abort, err, lim_ns));
        if (ok && row_ok) {
          const uint32_t qrow = sQ + (uint32_t)(k & 1) * kQSlotBytes + (uint32_t)r * 128;
          auto chunk = [&](int i) {
            return qrow + (i >> 3) * kQHalfBytes + ((uint32_t)((i & 7) ^ (r & 7)) << 4);
          };
          uint32_t m2[4] = {0u, 0u, 0u, 0u};  // larger magnitude per half (sign dropped below)
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
          float mq = 0.f;
#pragma unroll
          for (int e = 0; e < 4; ++e)
            mq = fmax3(mq, fabsf(__uint_as_float(m2[e] << 16)),
                       fabsf(__uint_as_float(m2[e] & 0xFFFF0000u)));
          int e2 = 0;
          if (mq > 0.f) {
            e2 = 14 - ((int)((__float_as_uint(mq) >> 23) & 0xFF) - 127);
            e2 = e2 < -100 ? -100 : (e2 > 100 ? 100 : e2);
          }
          const float qs = __uint_as_float((uint32_t)(127 + e2) << 23);
          sc = sc0 * __uint_as_float((uint32_t)(127 - e2) << 23);
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
        mbar_arrive(q_ready(k & 1));
        if (!ok) break;
      }
      float m = -INFINITY, l = 0.f;
      for (int j = 0; ok && j < n; ++j) {
        const int g = G + j;
        ok = __all_sync(0xffffffffu, wait_bar(s_full, g & 1, s_abort, err, lim_ns));
        if (!ok) break;
        tc_fence_after();
        if (!live) {
          tc_fence_before();
          mbar_arrive(s_free);
        } else {
          float s[64];
          tmem_ld32(trow + kColS, *reinterpret_cast<float(*)[32]>(&s[0]));
          tmem_ld32(trow + kColS + 32, *reinterpret_cast<float(*)[32]>(&s[32]));
          tmem_wait_ld();
          tc_fence_before();
          mbar_arrive(s_free);
          const int kv0 = (sgm.tb + j) * 64;
          if (kv0 + 64 > lim) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (kv0 + c >= lim) s[c] = -INFINITY;
          }
          float mx8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx8[i] = s[i];
#pragma unroll
          for (int c = 8; c + 16 <= 64; c += 16)
#pragma unroll
            for (int i = 0; i < 8; ++i) mx8[i] = fmax3(mx8[i], s[c + i], s[c + 8 + i]);
#pragma unroll
          for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], s[56 + i]);
          const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]),
                                 fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7]));
          const float m_new = fmaxf(m, mx * sc);
          // move the row maximum only when it grew by more than the threshold
          const bool need = row_ok && j > 0 && m_new > m + kRescaleThreshold;
          const float m_use = (j == 0 || need) ? m_new : m;
          const float alpha = need ? ex2(m - m_new) : 1.f;
          // a row with no visible key so far keeps m = -inf and P = 0
          const float m_ref = m_use == -INFINITY ? 0.f : m_use;
          uint32_t pk[32];
          const uint64_t sc2 = pack2(sc, sc), nm2 = pack2(-m_ref, -m_ref);
          uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            float x0, x1;
            unpack2(ffma2(pack2(s[2 * c], s[2 * c + 1]), sc2, nm2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            acc2[c & 3] = fadd2(acc2[c & 3], pack2(p0, p1));
            pk[c] = FP8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);  // keys 2c (low) and 2c + 1
          }
          float r0, r1;
          unpack2(fadd2(fadd2(acc2[0], acc2[1]), fadd2(acc2[2], acc2[3])), r0, r1);
          l = l * alpha + (r0 + r1);
          m = m_use;
          // The P buffer of tile g was last read by P(g-2) V_{g-2}, which the
          // MMA warp issued before S(g); the commit behind s_full(g) fires
          // only when every earlier MMA of that thread has completed.
          if (j > 0 && __any_sync(0xffffffffu, need)) {
            // O is stable once the P V of tile g - 1 is done
            ok = __all_sync(0xffffffffu, wait_bar(pv_done((g - 1) & 1), ((g - 1) >> 1) & 1,
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
          tmem_st32(trow + kColP + 32u * (uint32_t)(g & 1), pk);
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(p_full(g & 1));
      }
      if (!ok) break;
      // ---- epilogue of the segment
      const int gl = G + n - 1;
      ok = __all_sync(0xffffffffu, wait_bar(pv_done(gl & 1), (gl >> 1) & 1, s_abort, err, lim_ns));
      if (!ok) break;
      tc_fence_after();
      if (live) {
        const int64_t hv = (int64_t)T * p.num_q_heads;
        const int64_t jv = (int64_t)t * p.num_q_heads + head;
        const float inv = l > 0.f ? p.v_scale / l : 0.f;
        __nv_bfloat16* orow =
            p.out + (int64_t)sgm.b * p.o_sb + (int64_t)t * p.o_st + (int64_t)head * p.o_sh;
        float* wrow = p.ws_o + ((int64_t)sg * hv + jv) * 128;
#pragma unroll
        for (int q = 0; q < 4; q += 2) {
          float o[64];
          tmem_ld32(trow + kColO + q * 32, *reinterpret_cast<float(*)[32]>(&o[0]));
          tmem_ld32(trow + kColO + q * 32 + 32, *reinterpret_cast<float(*)[32]>(&o[32]));
          tmem_wait_ld();
          if (row_ok) {
            if (sgm.whole) {
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                uint4 v;
                v.x = pack_bf16(o[8 * c + 0] * inv, o[8 * c + 1] * inv);
                v.y = pack_bf16(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
                v.z = pack_bf16(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
                v.w = pack_bf16(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
                *reinterpret_cast<uint4*>(orow + q * 32 + c * 8) = v;
              }
            } else {
#pragma unroll
              for (int c = 0; c < 16; ++c)
                *reinterpret_cast<float4*>(wrow + q * 32 + 4 * c) =
                    make_float4(o[4 * c] * p.v_scale, o[4 * c + 1] * p.v_scale,
                                o[4 * c + 2] * p.v_scale, o[4 * c + 3] * p.v_scale);
            }
          }
        }
        if (row_ok) {
          if (sgm.whole) {
            if (p.lse)
              p.lse[(int64_t)sgm.b * p.l_sb + (int64_t)t * p.l_st + (int64_t)head * p.l_sh] =
                  l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
          } else {
            p.ws_m[(int64_t)sg * hv + jv] = l > 0.f ? m : -INFINITY;
            p.ws_l[(int64_t)sg * hv + jv] = l;
          }
        }
      }
      G += n;
      ++k;
    }
    named_bar_sync(1, Lt::kThreads);
  } else {
    named_bar_sync(1, Lt::kThreads);  // no such warp in this layout
  }
}

template <bool FP8>
cudaError_t launch_tc(const DecodeTcParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                      const CUtensorMap& tv, int num_parts, cudaStream_t stream) {
  using Lt = TcLayout<FP8>;
  static std::atomic<uint64_t> configured{0};  // devices whose copy is configured
  const cudaError_t e = once_per_device(configured, [] {
    return cudaFuncSetAttribute(decode_tc_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)Lt::kSmemBytes);
  });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)p.num_kv_heads, (unsigned)num_parts);
  cfg.blockDim = dim3(Lt::kThreads);
  cfg.dynamicSmemBytes = Lt::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel<FP8>, p, tq, tk, tv);
}

}  // namespace

cudaError_t launch_decode_tc(const DecodeTcParams& p, const CUtensorMap& tq,
                             const CUtensorMap& tk, const CUtensorMap& tv, bool fp8,
                             int num_parts, cudaStream_t stream) {
  if (num_parts <= 0 || p.num_kv_heads <= 0) return cudaSuccess;
  return fp8 ? launch_tc<true>(p, tq, tk, tv, num_parts, stream)
             : launch_tc<false>(p, tq, tk, tv, num_parts, stream);
}

}  // namespace hpc
