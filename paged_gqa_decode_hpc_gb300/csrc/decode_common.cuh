// Device pieces shared by the decode kernels (attn_kernel.cu, step_kernel.cu):
// inline-PTX shims for mbarriers, TMA and the legacy tensor-core MMA, the
// bounded waits, and the math of one (tile, KV head) unit -- scores
// S^T = K Q^T of the 8 query heads of a KV head against a 64-token tile,
// the online-softmax update and O^T += V^T P^T -- on a K/V tile pair that
// TMA left in shared memory with 128-byte swizzle.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "hpc_internal.h"

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



// Output coordinate of accumulator element (dm, r): BF16 rows are d = 16dm+g
// (+8); the FP8 V path permutes rows so a thread owns d = 16dm+2g (+1).
template <bool FP8>
__device__ __forceinline__ int acc_d(int dm, int r, int g) {
  return FP8 ? (16 * dm + 2 * g + r) : (16 * dm + g + 8 * r);
}

// Q of one (sequence, kv head) as mma B fragments (B[k = d][n = q head]).
// q0 points at the first query head of the KV head's group, q_sh is the
// stride between query heads (elements).
template <bool FP8>
__device__ __forceinline__ float load_q(const __nv_bfloat16* q0, int64_t q_sh, int lane,
                                        uint32_t (&qf)[8][2]) {
  const int g = lane >> 2, c = lane & 3;
  const __nv_bfloat16* qrow = q0 + (int64_t)g * q_sh;
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

}  // namespace
}  // namespace hpc
