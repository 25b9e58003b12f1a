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

#include "hpc_internal.h"
#include "ptx.cuh"

namespace hpc {

namespace {

constexpr float kLn2 = 0.6931471805599453f;

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          bar),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t movm_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// lo -> bits 0..15, hi -> bits 16..31
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Two e4m3 bytes (low byte -> low half) to f16x2; exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t x16) {
  uint32_t r;
  const uint16_t h = (uint16_t)(x16 & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
  return r;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, 0, %2;" : "=r"(r) : "r"(a), "r"(sel));
  return r;
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void st_release_shared(uint32_t addr, uint32_t v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_shared(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// Bounded wait until the producer has issued unit `unit` into its slot. A
// slot's successive rounds are consumed by different warps, so a warp may ask
// for round r while the slot's barrier has completed only round r-2; the
// mbarrier parity cannot tell those apart. Once the slot's issued word equals
// the unit, rounds < r have completed and round r+1 cannot start before this
// warp releases the slot, so the parity wait that follows is exact.
__device__ __forceinline__ bool wait_issued(uint32_t word, uint32_t unit, volatile int* abort_flag,
                                            int32_t* err, unsigned long long limit_ns) {
  if (ld_acquire_shared(word) == unit) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (ld_acquire_shared(word) == unit) return true;
    if ((it & 63u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) {
        atomicOr(err, HPC_DEVCHK_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// Bounded wait on an mbarrier phase. Returns false when the CTA is aborting
// or the time limit passed (then the abort flag and the error bit are set).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           int32_t* err, unsigned long long limit_ns,
                                           bool honour_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (honour_abort && *abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) {
        atomicOr(err, HPC_DEVCHK_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

template <bool FP8>
struct Geom {
  static constexpr int kTileBytes = FP8 ? 8192 : 16384;  // one 64 x 128 tile
  static constexpr int kStageBytes = 2 * kTileBytes;     // K + V
};

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

// Part arithmetic of the balanced plan: part start floor(p*T/P) and the part
// owning tile x, floor(((x+1)*P - 1)/T); 32-bit division when products fit.
struct PartMath {
  int64_t T, P;
  bool small;
  __device__ __forceinline__ int64_t start(int64_t q) const {
    return small ? (int64_t)((uint32_t)(q * T) / (uint32_t)P) : (q * T) / P;
  }
  __device__ __forceinline__ int64_t of(int64_t x) const {
    return small ? (int64_t)((uint32_t)((x + 1) * P - 1) / (uint32_t)T) : ((x + 1) * P - 1) / T;
  }
};

// Inclusive scan of one value per thread over the whole CTA (any size <= 1024).
__device__ __forceinline__ int32_t cta_inclusive_scan(int32_t v, int32_t* warp_tot,
                                                      int32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int32_t t = lane < nwarps ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t u = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += u;
    }
    warp_tot[lane] = t;
  }
  __syncthreads();
  const int32_t res = v + (warp > 0 ? warp_tot[warp - 1] : 0);
  *total = warp_tot[nwarps - 1];
  __syncthreads();
  return res;
}

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

// Output coordinate of accumulator element (dm, r): BF16 rows are d = 16dm+g
// (+8); the FP8 V path permutes rows so a thread owns d = 16dm+2g (+1).
template <bool FP8>
__device__ __forceinline__ int acc_d(int dm, int r, int g) {
  return FP8 ? (16 * dm + 2 * g + r) : (16 * dm + g + 8 * r);
}

// Q of one (sequence, kv head) as mma B fragments (B[k = d][n = q head]).
template <bool FP8>
__device__ __forceinline__ float load_q(const AttnParams& p, int b, int t, int h, int lane,
                                        uint32_t (&qf)[8][2]) {
  const int g = lane >> 2, c = lane & 3;
  const __nv_bfloat16* qrow = p.q + (int64_t)b * p.q_sb + (int64_t)t * p.q_st +
                              (int64_t)(h * kGroup + g) * p.q_sh;
  if constexpr (!FP8) {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qf[ks][0] = __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c));
      qf[ks][1] = __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c + 8));
    }
    return 1.0f;
  } else {
    // Logical k (2c, 2c+1 | 2c+8, 2c+9) of k-step ks maps to d = 16ks + 4c + (0,1 | 2,3),
    // matching the byte order ldmatrix gives the FP8 K tile.
    float v[8][4];
    float amax = 0.f;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint2 u = __ldg(reinterpret_cast<const uint2*>(qrow + 16 * ks + 4 * c));
      v[ks][0] = __uint_as_float(u.x << 16);
      v[ks][1] = __uint_as_float(u.x & 0xFFFF0000u);
      v[ks][2] = __uint_as_float(u.y << 16);
      v[ks][3] = __uint_as_float(u.y & 0xFFFF0000u);
#pragma unroll
      for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(v[ks][e]));
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    // Power-of-two scale putting max|q| in [2^14, 2^15): f16 holds every
    // bf16 value of that range exactly.
    int e = 0;
    if (amax > 0.f) {
      const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
      e = 14 - ex;
      e = e < -60 ? -60 : (e > 60 ? 60 : e);
    }
    const float sc = __uint_as_float((uint32_t)(e + 127) << 23);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qf[ks][0] = pack_f16(v[ks][0] * sc, v[ks][1] * sc);
      qf[ks][1] = pack_f16(v[ks][2] * sc, v[ks][3] * sc);
    }
    return __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e
  }
}

// One (tile, kv head) unit: scores, online softmax update, P.V accumulate.
template <bool FP8>
__device__ __forceinline__ void compute_unit(uint32_t kbase, uint32_t vbase,
                                             const uint32_t (&qf)[8][2], int valid, float sl2,
                                             float (&m)[2], float (&l)[2], float (&acc)[8][4],
                                             int lane) {
  const int r8 = lane & 7;
  const int mi = lane >> 3;
  const int g = lane >> 2;
  float s[4][4];
#pragma unroll
  for (int mt = 0; mt < 4; ++mt) s[mt][0] = s[mt][1] = s[mt][2] = s[mt][3] = 0.f;

  // ---- S^T = K Q^T
  const uint32_t k_lane = kbase + (uint32_t)((r8 + (mi & 1) * 8) * 128);
  if constexpr (!FP8) {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const uint32_t off = (uint32_t)((ks >> 2) * 8192 + ((((2 * ks) & 7) + (mi >> 1)) ^ r8) * 16);
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(k_lane + mt * 2048 + off, a0, a1, a2, a3);
        mma_bf16(s[mt], a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
      }
    }
  } else {
#pragma unroll
    for (int kp = 0; kp < 4; ++kp) {
      const uint32_t off = (uint32_t)((((2 * kp) + (mi >> 1)) ^ r8) * 16);
#pragma unroll
      for (int mt = 0; mt < 4; ++mt) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4(k_lane + mt * 2048 + off, r0, r1, r2, r3);
        mma_f16(s[mt], e4m3x2_to_f16x2(r0), e4m3x2_to_f16x2(r1), e4m3x2_to_f16x2(r0 >> 16),
                e4m3x2_to_f16x2(r1 >> 16), qf[2 * kp][0], qf[2 * kp][1]);
        mma_f16(s[mt], e4m3x2_to_f16x2(r2), e4m3x2_to_f16x2(r3), e4m3x2_to_f16x2(r2 >> 16),
                e4m3x2_to_f16x2(r3 >> 16), qf[2 * kp + 1][0], qf[2 * kp + 1][1]);
      }
    }
  }

  // ---- online softmax (log2 domain); columns 2c (e=0) and 2c+1 (e=1)
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int tok = mt * 16 + g + 8 * r;
      float x0 = s[mt][2 * r] * sl2, x1 = s[mt][2 * r + 1] * sl2;
      if (tok >= valid) x0 = x1 = -INFINITY;
      s[mt][2 * r] = x0;
      s[mt][2 * r + 1] = x1;
      mx0 = fmaxf(mx0, x0);
      mx1 = fmaxf(mx1, x1);
    }
  }
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
  }
  const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
  const float al0 = ex2(m[0] - mn0), al1 = ex2(m[1] - mn1);
  m[0] = mn0;
  m[1] = mn1;
  float ps0 = 0.f, ps1 = 0.f;
  uint32_t pb[4][2];
#pragma unroll
  for (int mt = 0; mt < 4; ++mt) {
    const float p0 = ex2(s[mt][0] - mn0), p1 = ex2(s[mt][1] - mn1);
    const float p2 = ex2(s[mt][2] - mn0), p3 = ex2(s[mt][3] - mn1);
    ps0 += p0 + p2;
    ps1 += p1 + p3;
    if constexpr (!FP8) {
      pb[mt][0] = movm_trans(pack_bf16(p0, p1));
      pb[mt][1] = movm_trans(pack_bf16(p2, p3));
    } else {
      pb[mt][0] = movm_trans(pack_f16(p0, p1));
      pb[mt][1] = movm_trans(pack_f16(p2, p3));
    }
  }
  l[0] = l[0] * al0 + ps0;
  l[1] = l[1] * al1 + ps1;
#pragma unroll
  for (int dm = 0; dm < 8; ++dm) {
    acc[dm][0] *= al0;
    acc[dm][1] *= al1;
    acc[dm][2] *= al0;
    acc[dm][3] *= al1;
  }

  // ---- O^T += V^T P^T
  if constexpr (!FP8) {
    const uint32_t v_lane = vbase + (uint32_t)(((r8) + ((mi >> 1) << 3)) * 128);
#pragma unroll
    for (int dm = 0; dm < 8; ++dm) {
      const uint32_t off = (uint32_t)((dm >> 2) * 8192 + ((((2 * dm) & 7) + (mi & 1)) ^ r8) * 16);
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(v_lane + kt * 2048 + off, a0, a1, a2, a3);
        mma_bf16(acc[dm], a0, a1, a2, a3, pb[kt][0], pb[kt][1]);
      }
    }
  } else {
    const uint32_t v_lane = vbase + (uint32_t)((r8 + ((mi & 1) << 3)) * 128);
#pragma unroll
    for (int dp = 0; dp < 4; ++dp) {
      const uint32_t off = (uint32_t)((((2 * dp) + (mi >> 1)) ^ r8) * 16);
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
        uint32_t r0, r1, r2, r3;
        ldsm_x4_t(v_lane + kt * 2048 + off, r0, r1, r2, r3);
        // bytes {0,2} = (token 2c, 2c+1) at even d; bytes {1,3} at odd d
        const uint32_t x0 = prmt(r0, 0x3120), x1 = prmt(r1, 0x3120);
        const uint32_t x2 = prmt(r2, 0x3120), x3 = prmt(r3, 0x3120);
        mma_f16(acc[2 * dp], e4m3x2_to_f16x2(x0), e4m3x2_to_f16x2(x0 >> 16), e4m3x2_to_f16x2(x1),
                e4m3x2_to_f16x2(x1 >> 16), pb[kt][0], pb[kt][1]);
        mma_f16(acc[2 * dp + 1], e4m3x2_to_f16x2(x2), e4m3x2_to_f16x2(x2 >> 16),
                e4m3x2_to_f16x2(x3), e4m3x2_to_f16x2(x3 >> 16), pb[kt][0], pb[kt][1]);
      }
    }
  }
}

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
        const float qinv = load_q<FP8>(p, b, tok, h, lane, qf);
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
