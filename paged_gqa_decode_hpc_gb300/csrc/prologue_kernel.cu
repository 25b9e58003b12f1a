// Fused decode prologue: QK-Norm + RoPE on the new token's q and k, the paged
// KV-cache write of k and v, and optionally an FP8 copy of q, in one kernel
// ("vLLM x HPC-Ops", section "Attention Backend: Dynamic Load-Balanced
// Scheduling", paragraph on HpcRopeNorm; the 24-ai.news page names RoPE,
// QK-Norm and the KV write). The pages give no formulas; this kernel takes
// RMSNorm over head_dim with one weight vector for q and one for k, then
// rotate-half RoPE with angle pos * base^(-2i/D), pos = seq_len - 1.
//
// One warp per row (a query head, a key head or a value head of one
// sequence); lane l holds elements [4l, 4l + 4), so the RoPE partner
// (i <-> i + 64) is lane l ^ 16. Positions reach 2^18 and beyond, where an
// fp32 product pos * f is off by ~1e-2 rad; the angle is therefore carried as
// a float-float sum (exact FMA product terms, host-made double-precision
// frequencies split in two floats) and reduced modulo 2*pi before the sine.
// Everything runs in fp32 (GB300's fp64 rate is a small fraction of it).
#include <cuda_bf16.h>

#include "hpc_internal.h"
#include "ptx.cuh"

namespace hpc {

namespace {

constexpr int kRowsPerCta = 8;

__device__ __forceinline__ float4 load4(const void* base, int32_t dtype, int64_t off) {
  if (dtype == HPC_F32) return *reinterpret_cast<const float4*>((const float*)base + off);
  const uint2 u = *reinterpret_cast<const uint2*>((const __nv_bfloat16*)base + off);
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}

__device__ __forceinline__ uint2 to_bf16x4(float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  const __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

// Four values to e4m3 (round to nearest even, saturating), element 0 in the
// lowest byte.
__device__ __forceinline__ uint32_t to_e4m3x4(float4 v) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(v.y), "f"(v.x));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(v.w), "f"(v.z));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// x / s rounded to odd in fp32: the quotient truncated toward zero, with its
// lowest mantissa bit set when the division was inexact (the FMA remainder of
// a faithfully rounded quotient is exact). A value rounded to odd with 24
// significant bits and then rounded to nearest-even at e4m3's 4 bits equals
// the nearest-even e4m3 of the exact quotient (Boldo and Melquiond, "When
// double rounding is odd", 2005: a p-bit odd rounding followed by a
// nearest rounding to at most p - 2 bits is a single correct rounding).
__device__ __forceinline__ float div_round_odd(float x, float s) {
  const float q = __fdiv_rz(x, s);
  const float r = fmaf(-q, s, x);
  return r != 0.f ? __uint_as_float(__float_as_uint(q) | 1u) : q;
}

// e4m3(v / s) of four values, each correctly rounded from the exact quotient.
__device__ __forceinline__ uint32_t quantise_e4m3x4(float4 v, float s) {
  return to_e4m3x4(make_float4(div_round_odd(v.x, s), div_round_odd(v.y, s),
                               div_round_odd(v.z, s), div_round_odd(v.w, s)));
}

__global__ void __launch_bounds__(kRowsPerCta * 32) prologue_kernel(const PrologueParams p) {
  griddep_wait();
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  const int per_seq = p.num_q_heads + 2 * p.num_kv_heads;
  if (row >= (int64_t)p.num_seqs * per_seq) return;
  const int b = (int)(row / per_seq);
  const int r = (int)(row % per_seq);
  const int32_t len = p.seq_lens[b];
  if (len <= 0) return;  // no new token for an empty sequence
  const int32_t pos = len - 1;
  const int kind = r < p.num_q_heads ? 0 : (r < p.num_q_heads + p.num_kv_heads ? 1 : 2);
  const int h = kind == 0 ? r : (kind == 1 ? r - p.num_q_heads : r - p.num_q_heads - p.num_kv_heads);
  const int d0 = 4 * lane;

  float4 x;
  if (kind == 0) x = load4(p.q_in, HPC_BF16, (int64_t)b * p.qi_sb + (int64_t)h * p.qi_sh + d0);
  else if (kind == 1) x = load4(p.k_in, HPC_BF16, (int64_t)b * p.ki_sb + (int64_t)h * p.ki_sh + d0);
  else x = load4(p.v_in, HPC_BF16, (int64_t)b * p.vi_sb + (int64_t)h * p.vi_sh + d0);

  if (kind != 2) {
    // RMSNorm over the 128 elements of the row
    float ss = x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = rsqrtf(ss * (1.0f / kHeadDim) + p.eps);
    const float4 w = load4(kind == 0 ? p.wq : p.wk, kind == 0 ? p.wq_dtype : p.wk_dtype, d0);
    x.x *= inv * w.x; x.y *= inv * w.y; x.z *= inv * w.z; x.w *= inv * w.w;
    // rotate-half RoPE: lanes 0-15 hold i < 64, lanes 16-31 hold i + 64
    const float4 y = make_float4(__shfl_xor_sync(0xffffffffu, x.x, 16),
                                 __shfl_xor_sync(0xffffffffu, x.y, 16),
                                 __shfl_xor_sync(0xffffffffu, x.z, 16),
                                 __shfl_xor_sync(0xffffffffu, x.w, 16));
    const float sgn = lane < 16 ? -1.f : 1.f;
    float c[4], s[4];
    const float fpos = (float)pos;  // exact below 2^24
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = 4 * (lane & 15) + j;
      // angle = pos * f with f = f_hi + f_lo: pos * f_hi exactly as a_hi + a_err
      const float a_hi = fpos * p.inv_freq_hi[i];
      const float a_err = fmaf(fpos, p.inv_freq_hi[i], -a_hi);
      const float a_lo = fmaf(fpos, p.inv_freq_lo[i], a_err);
      // reduce modulo 2*pi (= two_pi_hi + two_pi_lo) into [-pi, pi]
      const float k = rintf(a_hi * (1.0f / p.two_pi_hi));
      float r = fmaf(-k, p.two_pi_hi, a_hi);
      r = fmaf(-k, p.two_pi_lo, r) + a_lo;
      __sincosf(r, &s[j], &c[j]);  // |r| <= pi: absolute error ~5e-7
    }
    x = make_float4(x.x * c[0] + sgn * y.x * s[0], x.y * c[1] + sgn * y.y * s[1],
                    x.z * c[2] + sgn * y.z * s[2], x.w * c[3] + sgn * y.w * s[3]);
  }

  if (kind == 0) {
    *reinterpret_cast<uint2*>(p.q_out + (int64_t)b * p.qo_sb + (int64_t)h * p.qo_sh + d0) =
        to_bf16x4(x);
    if (p.q_fp8) {
      *reinterpret_cast<uint32_t*>(p.q_fp8 + (int64_t)b * p.qf_sb + (int64_t)h * p.qf_sh + d0) =
          quantise_e4m3x4(x, p.q_fp8_scale);
    }
    return;
  }
  // KV-cache slot of the new token
  const int t = pos / kBlockTokens;
  if (t >= p.max_blocks) {
    if (lane == 0 && p.err) atomicOr(p.err, HPC_DEVCHK_TABLE_TOO_SHORT);
    return;
  }
  const int blk = p.block_table[(int64_t)b * p.bt_sb + t];
  if (blk < 0 || blk >= p.num_blocks) {
    if (lane == 0 && p.err) atomicOr(p.err, HPC_DEVCHK_BAD_BLOCK);
    return;
  }
  const int64_t off = (int64_t)blk * p.c_sblk + (int64_t)h * p.c_shead +
                      (int64_t)(pos % kBlockTokens) * p.c_sslot + d0;
  void* cache = kind == 1 ? p.k_cache : p.v_cache;
  if (p.cache_fp8) {
    *reinterpret_cast<uint32_t*>((uint8_t*)cache + off) =
        quantise_e4m3x4(x, kind == 1 ? p.k_scale : p.v_scale);
  } else {
    *reinterpret_cast<uint2*>((__nv_bfloat16*)cache + off) = to_bf16x4(x);
  }
}

}  // namespace

cudaError_t launch_prologue(const PrologueParams& p, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.num_seqs * (p.num_q_heads + 2 * p.num_kv_heads);
  if (rows == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((rows + kRowsPerCta - 1) / kRowsPerCta));
  cfg.blockDim = dim3(kRowsPerCta * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prologue_kernel, p);
}

}  // namespace hpc
