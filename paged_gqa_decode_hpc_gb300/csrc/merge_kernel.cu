// Log-sum-exp merge of split-KV partial states.
//
// A sequence whose tiles were spread over several CTAs leaves one partial
// state per segment: m (largest scaled score, log2 units), l (sum of
// 2^(s - m)) and o (sum of 2^(s - m) v, unnormalised). They combine exactly:
//   M = max_i m_i,  l = sum_i l_i 2^(m_i - M),  out = sum_i o_i 2^(m_i - M) / l,
//   lse = ln 2 * (M + log2 l).
// The pages describe split-KV partial work ("vLLM x HPC-Ops", section
// "Attention Backend: Dynamic Load-Balanced Scheduling") but print no merge;
// this is the standard identity that makes the split softmax exact.
//
// One CTA per (sequence, query head): 8 warps take the sequence's partials
// round-robin, each lane owns 4 of the 128 output columns; every warp keeps a
// running (M, l, o) and prefetches its next partials, and the warps' states
// are combined in shared memory. A sequence with no tiles gets out = 0 and
// lse = -inf here; a sequence finished inside one CTA is skipped.
#include <cuda_bf16.h>

#include "hpc_internal.h"
#include "ptx.cuh"

namespace hpc {

namespace {

constexpr int kMergeWarps = 8;
constexpr float kLn2f = 0.6931471805599453f;

struct State {
  float m, l;
  float4 o;
};

__device__ __forceinline__ void absorb(State& st, float mi, float li, const float4& oi) {
  if (mi == -INFINITY) return;  // empty partial
  const float mn = fmaxf(st.m, mi);
  const float a = st.m == -INFINITY ? 0.f : ptx_ex2(st.m - mn);
  const float b = ptx_ex2(mi - mn);
  st.m = mn;
  st.l = st.l * a + li * b;
  st.o.x = st.o.x * a + oi.x * b;
  st.o.y = st.o.y * a + oi.y * b;
  st.o.z = st.o.z * a + oi.z * b;
  st.o.w = st.o.w * a + oi.w * b;
}

__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const MergeParams p) {
  __shared__ float4 s_o[kMergeWarps][32];
  __shared__ float s_m[kMergeWarps], s_l[kMergeWarps];
  griddep_wait();  // partials come from the attention kernel
  const int b = blockIdx.x, j = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s0 = p.plan[p.seq_off + b], s1 = p.plan[p.seq_off + b + 1];
  const int ns = s1 - s0;
  if (ns == 1) return;  // written by the attention kernel
  __nv_bfloat16* o = p.out + (int64_t)b * p.o_sb + (int64_t)j * p.o_sh + 4 * lane;
  float* lse = p.lse ? p.lse + (int64_t)b * p.l_sb + (int64_t)j * p.l_sh : nullptr;
  if (ns == 0) {
    if (warp == 0) {
      *reinterpret_cast<uint2*>(o) = make_uint2(0u, 0u);
      if (lse && lane == 0) *lse = -INFINITY;
    }
    return;
  }
  State st{-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
  constexpr int U = 4;
  int s = s0 + warp;
  for (; s + (U - 1) * kMergeWarps < s1; s += U * kMergeWarps) {
    float mm[U], ll[U];
    float4 oo[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t r = (int64_t)(s + u * kMergeWarps) * p.num_q_heads + j;
      mm[u] = p.ws_m[r];
      ll[u] = p.ws_l[r];
      oo[u] = *reinterpret_cast<const float4*>(p.ws_o + r * kHeadDim + 4 * lane);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) absorb(st, mm[u], ll[u], oo[u]);
  }
  for (; s < s1; s += kMergeWarps) {
    const int64_t r = (int64_t)s * p.num_q_heads + j;
    absorb(st, p.ws_m[r], p.ws_l[r], *reinterpret_cast<const float4*>(p.ws_o + r * kHeadDim + 4 * lane));
  }
  s_o[warp][lane] = st.o;
  if (lane == 0) {
    s_m[warp] = st.m;
    s_l[warp] = st.l;
  }
  __syncthreads();
  if (warp != 0) return;
  State t{-INFINITY, 0.f, make_float4(0.f, 0.f, 0.f, 0.f)};
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) absorb(t, s_m[w], s_l[w], s_o[w][lane]);
  const float inv = t.l > 0.f ? 1.f / t.l : 0.f;
  const __nv_bfloat162 lo = __floats2bfloat162_rn(t.o.x * inv, t.o.y * inv);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(t.o.z * inv, t.o.w * inv);
  *reinterpret_cast<uint2*>(o) =
      make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
  if (lse && lane == 0) *lse = t.l > 0.f ? (t.m + __log2f(t.l)) * kLn2f : -INFINITY;
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, int32_t /*num_kv_heads*/, cudaStream_t stream) {
  if (p.num_seqs == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_seqs, p.num_q_heads);
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge_kernel, p);
}

}  // namespace hpc
