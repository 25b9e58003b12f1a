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
// One CTA of 4 warps per (sequence, query head), the heads of a sequence
// adjacent in the launch order. A sequence with at most 8 partials is merged
// by one warp per head, four heads per CTA. Otherwise a warp takes every 4th
// partial; per round of up to 32 partials each lane loads one partial's
// (m, l) while the first 8 o rows are fetched alongside (each lane owns 4 of
// the 128 columns), so a round of up to 8 partials costs one memory round
// trip. At 64 registers, 8 CTAs fit on an SM: batches with many short split
// sequences (thousands of CTAs) take fewer waves. The warps'
// running (M, l, o) states are combined in shared memory. A sequence with no
// tiles gets out = 0 and lse = -inf here; a sequence finished inside one CTA
// is skipped.
#include <cuda_bf16.h>

#include "hpc_internal.h"
#include "ptx.cuh"

namespace hpc {

namespace {

constexpr int kMergeWarps = 4;
constexpr int kWarpMerge = 8;  // at most this many partials: one warp per (token, head)
constexpr float kLn2f = 0.6931471805599453f;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__global__ void __launch_bounds__(kMergeWarps * 32, 8) merge_kernel(const MergeParams p) {
  __shared__ float4 s_o[kMergeWarps][32];
  __shared__ float s_m[kMergeWarps], s_l[kMergeWarps];
  griddep_wait();  // partials come from the attention kernel
  // CTA = (sequence b, jv = t * H_q + j: query token t, query head j), jv
  // fastest: the CTAs of one sequence launch together, so a long sequence's
  // many-partial merges start in the first wave instead of being spread over
  // the launch order
  const int b = (int)(blockIdx.y + blockIdx.z * gridDim.y), jv = (int)blockIdx.x;
  if (b >= p.num_seqs) return;  // past the last sequence (batches of more than 65535)
  const int t = jv / p.num_q_heads, j = jv % p.num_q_heads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s0 = p.plan[p.seq_off + b], s1 = p.plan[p.seq_off + b + 1];
  const int ns = s1 - s0;
  if (ns == 1) return;  // written by the attention kernel
  __nv_bfloat16* o = p.out + (int64_t)b * p.o_sb + (int64_t)t * p.o_st + (int64_t)j * p.o_sh +
                     4 * lane;
  float* lse = p.lse ? p.lse + (int64_t)b * p.l_sb + (int64_t)t * p.l_st + (int64_t)j * p.l_sh
                     : nullptr;
  if (ns == 0) {
    if (warp == 0) {
      *reinterpret_cast<uint2*>(o) = make_uint2(0u, 0u);
      if (lse && lane == 0) *lse = -INFINITY;
    }
    return;
  }
  const int64_t hq = (int64_t)p.q_len * p.num_q_heads;  // partial rows per segment
  if (ns <= kWarpMerge) {
    // Few partials (every head of the sequence has the same count): one warp
    // merges one (token, head) alone in one memory round trip, four per CTA
    // (jv .. jv+3 share the token: H_q is a multiple of 4), and the CTAs of
    // the other three heads have nothing to do. A batch of short split
    // sequences then needs a quarter of the merge warps.
    if ((jv & 3) != 0) return;
    const int jw = jv + warp, tw = jw / p.num_q_heads, hw = jw % p.num_q_heads;
    __nv_bfloat16* ow = p.out + (int64_t)b * p.o_sb + (int64_t)tw * p.o_st +
                        (int64_t)hw * p.o_sh + 4 * lane;
    const float* ob = p.ws_o + (int64_t)jw * kHeadDim + 4 * lane;
    float mk = -INFINITY, lk = 0.f;
    if (lane < ns) {
      mk = p.ws_m[(s0 + lane) * hq + jw];
      lk = p.ws_l[(s0 + lane) * hq + jw];
    }
    float4 v[kWarpMerge];
#pragma unroll
    for (int u = 0; u < kWarpMerge; ++u)
      v[u] = u < ns ? *reinterpret_cast<const float4*>(ob + (s0 + u) * hq * kHeadDim)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
    const float M = warp_max(mk);
    const float wk = (M == -INFINITY || mk == -INFINITY) ? 0.f : ptx_ex2(mk - M);
    const float L = warp_sum(lk * wk);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < kWarpMerge; ++u) {
      const float w = __shfl_sync(0xffffffffu, wk, u);
      acc.x += w * v[u].x; acc.y += w * v[u].y; acc.z += w * v[u].z; acc.w += w * v[u].w;
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(ow) = make_uint2(*reinterpret_cast<const uint32_t*>(&lo),
                                               *reinterpret_cast<const uint32_t*>(&hi));
    if (p.lse && lane == 0)
      p.lse[(int64_t)b * p.l_sb + (int64_t)tw * p.l_st + (int64_t)hw * p.l_sh] =
          L > 0.f ? (M + __log2f(L)) * kLn2f : -INFINITY;
    return;
  }
  const float* obase = p.ws_o + (int64_t)jv * kHeadDim + 4 * lane;
  float M = -INFINITY, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  // this warp's partials: s0 + warp + kMergeWarps * t, t = 0, 1, ...
  const int mine = (ns - warp + kMergeWarps - 1) / kMergeWarps;
  constexpr int kBatch = 8;  // partial rows in flight per lane
  for (int r0 = 0; r0 < mine; r0 += 32) {
    const int cnt = mine - r0 < 32 ? mine - r0 : 32;
    const int64_t my_s = s0 + warp + (int64_t)kMergeWarps * (r0 + lane);
    float mk = -INFINITY, lk = 0.f;
    if (lane < cnt) {
      mk = p.ws_m[my_s * hq + jv];
      lk = p.ws_l[my_s * hq + jv];
    }
    // the first rows do not depend on the weights: fetch them with (m, l)
    float4 v[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int64_t sr = s0 + warp + (int64_t)kMergeWarps * (r0 + u);
      v[u] = u < cnt ? *reinterpret_cast<const float4*>(obase + sr * hq * kHeadDim)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const float Mn = fmaxf(M, warp_max(mk));
    if (Mn == -INFINITY) continue;  // only empty partials so far
    const float scale = M == -INFINITY ? 0.f : ptx_ex2(M - Mn);
    const float wk = mk == -INFINITY ? 0.f : ptx_ex2(mk - Mn);
    L = L * scale + warp_sum(lk * wk);
    acc.x *= scale; acc.y *= scale; acc.z *= scale; acc.w *= scale;
    M = Mn;
    for (int k0 = 0; k0 < cnt; k0 += kBatch) {
      if (k0 > 0) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int64_t sr = s0 + warp + (int64_t)kMergeWarps * (r0 + k0 + u);
          v[u] = k0 + u < cnt ? *reinterpret_cast<const float4*>(obase + sr * hq * kHeadDim)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const float w = __shfl_sync(0xffffffffu, wk, (k0 + u) & 31);
        acc.x += w * v[u].x; acc.y += w * v[u].y; acc.z += w * v[u].z; acc.w += w * v[u].w;
      }
    }
  }
  s_o[warp][lane] = acc;
  if (lane == 0) {
    s_m[warp] = M;
    s_l[warp] = L;
  }
  __syncthreads();
  if (warp != 0) return;
  float Mt = -INFINITY;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) Mt = fmaxf(Mt, s_m[w]);
  float Lt = 0.f;
  float4 tot = make_float4(0.f, 0.f, 0.f, 0.f);
  if (Mt != -INFINITY) {
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) {
      const float f = s_m[w] == -INFINITY ? 0.f : ptx_ex2(s_m[w] - Mt);
      Lt += s_l[w] * f;
      tot.x += s_o[w][lane].x * f; tot.y += s_o[w][lane].y * f;
      tot.z += s_o[w][lane].z * f; tot.w += s_o[w][lane].w * f;
    }
  }
  const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
  const __nv_bfloat162 lo = __floats2bfloat162_rn(tot.x * inv, tot.y * inv);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(tot.z * inv, tot.w * inv);
  *reinterpret_cast<uint2*>(o) =
      make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
  if (lse && lane == 0) *lse = Lt > 0.f ? (Mt + __log2f(Lt)) * kLn2f : -INFINITY;
}

}  // namespace

cudaError_t launch_merge(const MergeParams& p, int32_t /*num_kv_heads*/, cudaStream_t stream) {
  if (p.num_seqs == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  // x = query token x head (fastest in the launch order), y (and z beyond
  // 65535 sequences) = sequence
  const unsigned gy = p.num_seqs < 65535 ? (unsigned)p.num_seqs : 65535u;
  cfg.gridDim = dim3((unsigned)(p.q_len * p.num_q_heads), gy, (p.num_seqs + gy - 1) / gy);
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
