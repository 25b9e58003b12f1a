// Split-KV paged GQA decode attention for sm_103a (the merge pass is in merge_kernel.cu).
//
// The method ("vLLM x HPC-Ops", section "Attention Backend: Dynamic
// Load-Balanced Scheduling"): a persistent grid whose CTAs each walk a list
// of 64-token KV tiles chosen by the per-step planner; each CTA computes
// split-KV attention of one query token per sequence over its tiles and
// leaves a partial softmax state where a sequence spans several CTAs; a merge
// pass combines the partial states. Paged 64-token blocks and the fp8_e4m3
// cache come from section "Using HPC-Ops Backends in vLLM"; the GQA shape
// (8 query heads per KV head, head_dim 128) from the 24-ai.news Hy3 paragraph.
//
// GB300 design (the pages' Hopper kernel is not described beyond the above):
//  * One CTA per SM: 1 producer warp + NC consumer warps.
//  * Work unit = (tile, kv head): one 64x128 K tile and one V tile, 16 KB
//    each in BF16 (8 KB in FP8), fetched by TMA (4-D tensor map over
//    [blocks][kv heads][64 slots][128], 128-byte swizzle, L2 evict-first)
//    into a STAGES-deep shared-memory ring guarded by mbarriers.
//  * Consumer warp math on the tensor cores with mma.sync m16n8k16, in the
//    transposed orientation so no row is padded: S^T = K Q^T (M = 16 tokens,
//    N = the 8 query heads of the group, K = head dim), online softmax in
//    registers, then O^T = V^T P^T (M = head dim, N = 8 heads, K = tokens).
//    P^T reaches the B-operand layout with movmatrix (no shared memory).
//  * FP8 e4m3 tiles are widened in registers with cvt.f16x2.e4m3x2 (exact)
//    and multiplied in f16; Q is given a power-of-two scale into f16 range;
//    k_scale folds into the softmax scale, v_scale into the epilogue.
//  * Every wait is bounded (globaltimer); a timeout sets an error bit and the
//    CTA drains its own in-flight copies before leaving. No trap, no assert.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "decode_common.cuh"
#include "hpc_internal.h"
#include "ptx.cuh"

namespace hpc {

namespace {

constexpr int kCombineFloats = 36;  // per lane: acc[32], m[2], l[2]

template <bool FP8, int STAGES, int NC, bool COMBINE>
struct KernelCfg {
  static constexpr int kThreads = (NC + 1) * 32;
  static constexpr int kBarOff = STAGES * Geom<FP8>::kStageBytes;
  static constexpr int kAbortOff = kBarOff + 2 * STAGES * 8;
  static constexpr int kIssuedOff = kAbortOff + 16;  // u32 per slot: last unit issued
  static constexpr int kCombOff = kIssuedOff + ((4 * STAGES + 15) / 16) * 16;
  static constexpr int kPlanOff = kCombOff + (COMBINE ? NC * 32 * kCombineFloats * 4 : 0);
  static constexpr int kSmemBytes = 1024 /* alignment slack */ + kPlanOff;
  // with a fused plan: + 2 * (B + 1) int32 prefix arrays
  static constexpr int kSmemBytesFused = kSmemBytes + 8 * (kFusedPlanMaxSeqs + 1);
};

// The segments of one CTA, read from a plan in global memory or derived from
// the prefix arrays (tiles cu[], segments so[]) of a plan built in the CTA.
struct SegCursor {
  bool fused;
  // plan in global memory
  const int32_t* recs;
  int seg, seg_end;
  // plan built in the CTA
  const int32_t* cu;
  const int32_t* so;
  PartMath pm;
  int part, cur, B;
  int32_t s_lo, s_hi;

  __device__ __forceinline__ bool next(int& b, int& tb, int& te, bool& whole, int& slot) {
    if (!fused) {
      if (seg >= seg_end) return false;
      const int4 rec = *reinterpret_cast<const int4*>(recs + 4 * seg);
      b = rec.x;
      tb = rec.y;
      te = rec.z;
      whole = (rec.w & HPC_SEG_WHOLE) != 0;
      slot = seg++;
      return true;
    }
    while (cur < B) {
      const int32_t lo_b = cu[cur], hi_b = cu[cur + 1];
      if (lo_b >= s_hi) return false;
      const int bb = cur++;
      if (hi_b <= s_lo || hi_b == lo_b) continue;
      b = bb;
      tb = (lo_b > s_lo ? lo_b : s_lo) - lo_b;
      te = (hi_b < s_hi ? hi_b : s_hi) - lo_b;
      whole = so[bb + 1] - so[bb] == 1;
      slot = so[bb] + (int)(part - pm.of(lo_b));
      return true;
    }
    return false;
  }
};

// Final output (whole sequence in this CTA) or a partial state.
template <bool FP8>
__device__ __forceinline__ void write_result(const AttnParams& p, bool whole, int b, int t, int h,
                                             int seg,
                                             const float (&m)[2], const float (&l)[2],
                                             const float (&acc)[8][4], int lane) {
  const int g = lane >> 2, c = lane & 3;
  if (whole) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int j = h * kGroup + 2 * c + e;
      const float inv = l[e] > 0.f ? p.v_scale / l[e] : 0.f;
      __nv_bfloat16* orow = p.out + (int64_t)b * p.o_sb + (int64_t)t * p.o_st + (int64_t)j * p.o_sh;
      if constexpr (FP8) {
#pragma unroll
        for (int dm = 0; dm < 8; ++dm)
          *reinterpret_cast<__nv_bfloat162*>(orow + acc_d<true>(dm, 0, g)) =
              __floats2bfloat162_rn(acc[dm][e] * inv, acc[dm][2 + e] * inv);
      } else {
#pragma unroll
        for (int dm = 0; dm < 8; ++dm) {
          orow[acc_d<false>(dm, 0, g)] = __float2bfloat16_rn(acc[dm][e] * inv);
          orow[acc_d<false>(dm, 1, g)] = __float2bfloat16_rn(acc[dm][2 + e] * inv);
        }
      }
      if (p.lse && g == 0)
        p.lse[(int64_t)b * p.l_sb + (int64_t)t * p.l_st + (int64_t)j * p.l_sh] =
            l[e] > 0.f ? (m[e] + __log2f(l[e])) * kLn2 : -INFINITY;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int j = h * kGroup + 2 * c + e;
      // partial rows are indexed by (segment, query token, query head)
      const int64_t hv = (int64_t)p.q_len * p.num_q_heads;
      const int64_t jv = (int64_t)t * p.num_q_heads + j;
      float* o = p.ws_o + ((int64_t)seg * hv + jv) * kHeadDim;
#pragma unroll
      for (int dm = 0; dm < 8; ++dm) {
        if constexpr (FP8) {
          *reinterpret_cast<float2*>(o + acc_d<true>(dm, 0, g)) =
              make_float2(acc[dm][e] * p.v_scale, acc[dm][2 + e] * p.v_scale);
        } else {
          o[acc_d<false>(dm, 0, g)] = acc[dm][e];
          o[acc_d<false>(dm, 1, g)] = acc[dm][2 + e];
        }
      }
      if (g == 0) {
        p.ws_m[(int64_t)seg * hv + jv] = m[e];
        p.ws_l[(int64_t)seg * hv + jv] = l[e];
      }
    }
  }
}

template <bool FP8, int STAGES, int NC, bool COMBINE>
__global__ void __launch_bounds__((NC + 1) * 32, 1)
    attn_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tmk,
                const __grid_constant__ CUtensorMap tmv) {
  using Cfg = KernelCfg<FP8, STAGES, NC, COMBINE>;
  constexpr int kTile = Geom<FP8>::kTileBytes;
  constexpr int kStage = Geom<FP8>::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar_full = smem_base + Cfg::kBarOff;
  const uint32_t bar_empty = bar_full + STAGES * 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kAbortOff);
  const uint32_t issued_word = smem_base + Cfg::kIssuedOff;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Prologue that needs nothing from the preceding kernel: it overlaps that
  // kernel's tail when launched with programmatic stream serialization.
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, p.q_len);  // one consumer warp per query token
    }
    *abort_flag = 0;
    for (int s = 0; s < STAGES; ++s)
      reinterpret_cast<volatile uint32_t*>(smem + Cfg::kIssuedOff)[s] = 0xFFFFFFFFu;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == NC && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
  }
  griddep_wait();  // the plan (and inputs) of the preceding kernels are visible
  griddep_launch_dependents();

  SegCursor cur0;
  cur0.fused = false;
  cur0.recs = p.plan + p.seg_off;
  int h_begin, h_count;
  if (p.static_mode) {
    cur0.seg = blockIdx.x;
    cur0.seg_end = cur0.seg + 1;
    h_begin = blockIdx.y;
    h_count = 1;
  } else if (!p.fused_plan) {
    if ((int)blockIdx.x >= p.plan[kNumParts]) return;  // fewer parts than CTAs
    cur0.seg = p.plan[p.part_off + blockIdx.x];
    cur0.seg_end = p.plan[p.part_off + blockIdx.x + 1];
    h_begin = 0;
    h_count = p.num_kv_heads;
  } else {
    // ---- plan this step inside the CTA (same closed forms as the planners)
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t s_bad;
    int32_t* cu = reinterpret_cast<int32_t*>(smem + Cfg::kPlanOff);
    int32_t* so = cu + (p.num_seqs + 1);
    const int B = p.num_seqs, nt = blockDim.x, tid = threadIdx.x;
    if (tid == 0) {
      s_bad = 0;
      cu[0] = 0;
      so[0] = 0;
    }
    __syncthreads();
    int64_t carry = 0;
    for (int base = 0; base < B; base += nt) {
      const int b = base + tid;
      int32_t n = 0;
      if (b < B) {
        const int32_t len = p.seq_lens[b];
        if (len < 0) s_bad = 1;
        n = len > 0 ? (int32_t)((len + kBlockTokens - 1) / kBlockTokens) * p.plan_units : 0;
      }
      int32_t tot;
      const int32_t incl = cta_inclusive_scan(n, warp_tot, &tot);
      if (b < B) cu[b + 1] = (int32_t)(carry + incl);
      carry += tot;
    }
    __syncthreads();
    const bool bad = s_bad || carry > INT32_MAX;
    const int64_t T = bad ? 0 : carry;
    const int64_t P = T < p.plan_num_sms ? T : p.plan_num_sms;
    PartMath pm{T, P, (T + 1) * (P + 1) < (int64_t)UINT32_MAX};
    int64_t gcarry = 0;
    for (int base = 0; base < B; base += nt) {
      const int b = base + tid;
      int32_t cnt = 0;
      if (b < B && !bad && cu[b + 1] > cu[b]) cnt = (int32_t)(pm.of(cu[b + 1] - 1) - pm.of(cu[b]) + 1);
      int32_t tot;
      const int32_t incl = cta_inclusive_scan(cnt, warp_tot, &tot);
      if (b < B) so[b + 1] = (int32_t)(gcarry + incl);
      gcarry += tot;
    }
    __syncthreads();
    // this CTA's share of the plan words (read later by the merge and export)
    int32_t* w = p.plan_out;
    for (int b = blockIdx.x + gridDim.x * tid; b < B; b += gridDim.x * nt) {
      w[p.cu_off + b + 1] = bad ? 0 : cu[b + 1];
      w[p.seq_off + b + 1] = bad ? 0 : so[b + 1];
    }
    const int part = blockIdx.x;
    if (!bad && part < P && tid == 0) {
      const int32_t s0 = (int32_t)pm.start(part);
      int lo = 0, hi = B;  // last b with cu[b] <= s0 (a non-empty sequence)
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cu[mid] <= s0) lo = mid; else hi = mid;
      }
      w[p.part_off + part] = so[lo] + (int32_t)(part - pm.of(cu[lo]));
    }
    if (blockIdx.x == 0 && tid == 0) {
      if (bad) atomicOr(p.err, HPC_DEVCHK_BAD_LENGTH);
      w[kMagic] = kPlanMagic; w[kKind] = HPC_PLAN_DYNAMIC; w[kNumSeqs] = B;
      w[kNumParts] = (int32_t)P; w[kNumTiles] = (int32_t)T; w[kNumSegs] = (int32_t)gcarry;
      w[kNumSms] = p.plan_num_sms; w[kSplits] = p.plan_units > 1 ? p.plan_units : 0;
      w[p.cu_off] = 0; w[p.seq_off] = 0; w[p.part_off + P] = (int32_t)gcarry;
    }
    if (part >= P) return;  // uniform over the CTA
    cur0.fused = true;
    cur0.cu = cu;
    cur0.so = so;
    cur0.pm = pm;
    cur0.part = part;
    cur0.B = B;
    cur0.s_lo = (int32_t)pm.start(part);
    cur0.s_hi = (int32_t)pm.start(part + 1);
    int lo = 0, hi = B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (cu[mid] <= cur0.s_lo) lo = mid; else hi = mid;
    }
    cur0.cur = lo;
    h_begin = 0;
    h_count = p.num_kv_heads;
  }
  // KV heads processed together per pass; each (tile, head) unit is read by
  // q_len consumer warps (one per query token), and tph warps per (head,
  // token) split the tiles when warps are left over.
  const WarpLayout wl = warp_layout(h_count, p.q_len, NC);
  const int hpass = wl.hpass, npass = wl.npass, tph = wl.tph;
  __syncthreads();

  if (warp == NC) {
    // ------------------------------------------------------------ producer
    const uint64_t policy = evict_first_policy();
    uint32_t g = 0, issued = 0;
    bool stop = p.withhold_copies != 0;  // failure-path test: no copy is issued
    SegCursor sc = cur0;
    int b, tb, te, slot;
    bool whole;
    const int U = p.plan_units;  // 1: segments hold tiles; U > 1: (tile, head) units
    while (sc.next(b, tb, te, whole, slot)) {
      // tiles [t0, t0 + n) touched by the segment; with U > 1 only the heads of
      // units in [tb, te) are loaded at the first and last tile
      const int t0 = tb / U;
      const int n = (te - 1) / U + 1 - t0;
      if (sc.fused && lane == 0) {  // this part's segment records of the plan
        int4 rec;
        rec.x = b;
        rec.y = tb;
        rec.z = te;
        rec.w = whole ? HPC_SEG_WHOLE : 0;
        *reinterpret_cast<int4*>(p.plan_out + p.seg_off + 4 * (int64_t)slot) = rec;
      }
      const int32_t* btrow = p.block_table + (int64_t)b * p.bt_sb;
      for (int pass = 0; pass < npass; ++pass) {
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
          for (int ii = 0; ii < cnt; ++ii) {
            const int bk = __shfl_sync(0xffffffffu, blk, ii);
            const int ta = t0 + i0 + ii;  // absolute tile
            const int hlo = U > 1 && ta * U < tb ? tb - ta * U : 0;
            const int hhi = U > 1 && (ta + 1) * U > te ? te - ta * U : hpass;
            for (int hl = hlo; hl < hhi; ++hl, ++g) {
              if (lane != 0 || stop) continue;
              const int h = h_begin + pass * hpass + hl;
              const uint32_t slot = g % STAGES;
              const uint32_t par = ((g / STAGES) & 1u) ^ 1u;
              if (!wait_phase(bar_empty + 8 * slot, par, abort_flag, p.err, p.timeout_ns)) {
                stop = true;
                continue;
              }
              const uint32_t fb = bar_full + 8 * slot;
              const uint32_t dk = smem_base + slot * kStage;
              const uint32_t dv = dk + kTile;
              const int c1 = p.kv_swap ? h : 0, c2 = p.kv_swap ? 0 : h;
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
              st_release_shared(issued_word + 4 * slot, g);
              issued = g + 1;
            }
          }
        }
      }
    }
    // Every warp of the CTA meets here before any thread leaves. If a wait gave
    // up anywhere (producer or consumer, before or after the producer finished
    // issuing), copies may still be landing in shared memory: wait (bounded)
    // for the last issued ones, so the CTA never exits with a copy in flight.
    named_bar_sync(3, (NC + 1) * 32);
    if (lane == 0 && *abort_flag) {
      for (uint32_t u = issued > (uint32_t)STAGES ? issued - STAGES : 0; u < issued; ++u)
        wait_phase(bar_full + 8 * (u % STAGES), (u / STAGES) & 1u, abort_flag, p.err,
                   1000000000ull, false);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  float* comb = reinterpret_cast<float*>(smem + Cfg::kCombOff);
  const int hl = warp % hpass;                     // kv head (within the pass)
  const int tok = (warp / hpass) % p.q_len;        // query token of this warp
  const int tphase = (warp / hpass) / p.q_len;     // tiles i = tphase (mod tph)
  const bool active = tphase < tph;                // idle when warps are left over
  const int c = lane & 3;
  uint32_t gbase = 0;
  bool dead = false;
  SegCursor sc = cur0;
  int b, tb, te, seg;
  bool whole;
  const int U = p.plan_units;
  while (sc.next(b, tb, te, whole, seg)) {
    const int t0 = tb / U;
    const int n = (te - 1) / U + 1 - t0;  // tiles touched by the segment
    const int len = p.seq_lens[b];
    // this warp's tiles [i_lo, i_hi) (relative to t0): all of them in tile
    // plans; with U > 1 the tiles t whose unit t * U + h lies in [tb, te)
    int i_lo = 0, i_hi = n;
    if (U > 1) {
      i_lo = (tb + (U - 1 - hl)) / U - t0;
      i_hi = (te - 1 - hl >= 0 ? (te - 1 - hl) / U + 1 : 0) - t0;
    }
    if (!sc.fused && warp == 0 && lane == 0) {
      const int n_plan = p.plan[p.cu_off + b + 1] - p.plan[p.cu_off + b];
      const int n_dev = (len > 0 ? (len + kBlockTokens - 1) / kBlockTokens : 0) * U;
      if (n_plan != n_dev) atomicOr(p.err, HPC_DEVCHK_BAD_LENGTH);
    }
    for (int pass = 0; pass < npass; ++pass) {
      const int h = h_begin + pass * hpass + hl;
      float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
      float acc[8][4];
#pragma unroll
      for (int dm = 0; dm < 8; ++dm) acc[dm][0] = acc[dm][1] = acc[dm][2] = acc[dm][3] = 0.f;
      // causal limit of this warp's query token: the q_len new tokens are the
      // last q_len positions of the sequence
      const int len_t = len - (p.q_len - 1 - tok);
      if (active && i_lo + tphase < i_hi) {
        uint32_t qf[8][2];
        const float qinv = load_q<FP8>(p.q + (int64_t)b * p.q_sb + (int64_t)tok * p.q_st +
                                           (int64_t)(h * kGroup) * p.q_sh,
                                       p.q_sh, lane, qf);
        const float sl2 = p.score_scale_log2 * qinv;
        for (int i = i_lo + tphase; i < i_hi; i += tph) {
          // position of unit (tile t0 + i, head hl) in the order of issue
          const uint32_t gu = U > 1 ? gbase + (uint32_t)((t0 + i) * U + hl - tb)
                                    : gbase + (uint32_t)(i * hpass + hl);
          const uint32_t slot = gu % STAGES;
          if (dead) continue;
          const bool ok =
              wait_issued(issued_word + 4 * slot, gu, abort_flag, p.err, p.timeout_ns) &&
              wait_phase(bar_full + 8 * slot, (gu / STAGES) & 1u, abort_flag, p.err,
                         p.timeout_ns);
          if (!__all_sync(0xffffffffu, ok)) {  // warp-uniform decision
            dead = true;
            continue;
          }
          const int valid = len_t - (t0 + i) * kBlockTokens;
          if (valid > 0) {
            const uint32_t kb = smem_base + slot * kStage;
            compute_unit<FP8>(kb, kb + kTile, qf, valid, sl2, m, l, acc, lane);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
        }
      }
      gbase += U > 1 ? (uint32_t)(te - tb) : (uint32_t)(n * hpass);
      // reduce the row sums over the 8 lanes sharing a column pair
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        l[0] += __shfl_xor_sync(0xffffffffu, l[0], o);
        l[1] += __shfl_xor_sync(0xffffffffu, l[1], o);
      }
      if (!COMBINE || tph == 1) {
        if (!dead && active) write_result<FP8>(p, whole, b, tok, h, seg, m, l, acc, lane);
      } else {
        // warps of one (head, token): hl + hpass * (tok + q_len * k), k < tph
        const int wstep = hpass * p.q_len;
        if (active && tphase > 0) {
          float* cw = comb + (warp * 32 + lane) * kCombineFloats;
#pragma unroll
          for (int dm = 0; dm < 8; ++dm)
            *reinterpret_cast<float4*>(cw + 4 * dm) =
                make_float4(acc[dm][0], acc[dm][1], acc[dm][2], acc[dm][3]);
          *reinterpret_cast<float4*>(cw + 32) = make_float4(m[0], m[1], l[0], l[1]);
        }
        named_bar_sync(1, NC * 32);
        if (active && tphase == 0) {
          float M0 = m[0], M1 = m[1];
          for (int k = 1; k < tph; ++k) {
            const float4 ml =
                *reinterpret_cast<const float4*>(comb + ((warp + k * wstep) * 32 + lane) *
                                                            kCombineFloats + 32);
            M0 = fmaxf(M0, ml.x);
            M1 = fmaxf(M1, ml.y);
          }
          const float f0 = m[0] == -INFINITY ? 0.f : ex2(m[0] - M0);
          const float f1 = m[1] == -INFINITY ? 0.f : ex2(m[1] - M1);
          l[0] *= f0;
          l[1] *= f1;
#pragma unroll
          for (int dm = 0; dm < 8; ++dm) {
            acc[dm][0] *= f0;
            acc[dm][1] *= f1;
            acc[dm][2] *= f0;
            acc[dm][3] *= f1;
          }
          for (int k = 1; k < tph; ++k) {
            const float* cw = comb + ((warp + k * wstep) * 32 + lane) * kCombineFloats;
            const float4 ml = *reinterpret_cast<const float4*>(cw + 32);
            const float k0 = ml.x == -INFINITY ? 0.f : ex2(ml.x - M0);
            const float k1 = ml.y == -INFINITY ? 0.f : ex2(ml.y - M1);
            l[0] += ml.z * k0;
            l[1] += ml.w * k1;
#pragma unroll
            for (int dm = 0; dm < 8; ++dm) {
              const float4 a = *reinterpret_cast<const float4*>(cw + 4 * dm);
              acc[dm][0] += a.x * k0;
              acc[dm][1] += a.y * k1;
              acc[dm][2] += a.z * k0;
              acc[dm][3] += a.w * k1;
            }
          }
          m[0] = M0;
          m[1] = M1;
          if (!*abort_flag) write_result<FP8>(p, whole, b, tok, h, seg, m, l, acc, lane);
        }
        named_bar_sync(1, NC * 32);
      }
    }
  }
  named_bar_sync(3, (NC + 1) * 32);  // see the producer's exit
  (void)c;
}

template <bool FP8, int STAGES, int NC, bool COMBINE>
cudaError_t launch_cfg(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int gx,
                       int gy, cudaStream_t stream) {
  using Cfg = KernelCfg<FP8, STAGES, NC, COMBINE>;
  auto kern = attn_kernel<FP8, STAGES, NC, COMBINE>;
  static std::atomic<uint64_t> configured{0};  // devices whose copy is configured
  cudaError_t e = once_per_device(configured, [&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg::kSmemBytesFused);
  });
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(gx, gy);
  cfg.blockDim = dim3(Cfg::kThreads);
  cfg.dynamicSmemBytes =
      Cfg::kSmemBytes + (p.fused_plan ? 8 * ((size_t)p.num_seqs + 1) : 0);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, tk, tv);
}

}  // namespace

cudaError_t launch_attention(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                             bool fp8, int gx, int gy, cudaStream_t stream) {
  const int hc = p.static_mode ? 1 : p.num_kv_heads;
  const bool combine = warp_layout(hc, p.q_len, 8).tph > 1;
  if (fp8) {
    return combine ? launch_cfg<true, 10, 8, true>(p, tk, tv, gx, gy, stream)
                   : launch_cfg<true, 12, 8, false>(p, tk, tv, gx, gy, stream);
  }
  return combine ? launch_cfg<false, 5, 8, true>(p, tk, tv, gx, gy, stream)
                 : launch_cfg<false, 6, 8, false>(p, tk, tv, gx, gy, stream);
}

}  // namespace hpc
