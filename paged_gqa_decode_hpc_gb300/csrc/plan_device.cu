// Device tile planner: the per-step load-balanced plan computed on the GPU
// from device lengths, with no host round trip ("vLLM x HPC-Ops", section
// "Attention Backend: Dynamic Load-Balanced Scheduling": a per-step
// scheduler). It writes the same words as the host planner (plan_host.cu):
// both evaluate the same closed forms
//   part start  s_p = floor(p*T/P),   part of tile x = floor(((x+1)*P - 1)/T),
// so the results agree bit for bit.
//
// One CTA of 1024 threads: two block-wide scans (tile counts, then segments
// per sequence), then one thread per segment and one per part, each locating
// its sequence by binary search. The prefix arrays are kept in shared memory
// when they fit, so the searches never wait on global memory.
#include "hpc_internal.h"
#include "ptx.cuh"

namespace hpc {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kSmemSeqs = 6000;  // 2 * (6000 + 1) int32 fit the default 48 KB

// floor(p*T/P) and the part owning tile x; 32-bit division when products fit.
struct PartMath {
  int64_t T, P;
  bool small;
  __device__ __forceinline__ int64_t start(int64_t p) const {
    return small ? (int64_t)((uint32_t)(p * T) / (uint32_t)P) : (p * T) / P;
  }
  __device__ __forceinline__ int64_t of(int64_t x) const {
    return small ? (int64_t)((uint32_t)((x + 1) * P - 1) / (uint32_t)T) : ((x + 1) * P - 1) / T;
  }
};

// Inclusive block scan of one int per thread; returns the block total too.
__device__ __forceinline__ int32_t block_inclusive_scan(int32_t v, int32_t* warp_tot,
                                                        int32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int32_t u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  if (lane == 31) warp_tot[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int32_t t = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t u = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += u;
    }
    warp_tot[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  const int32_t res = v + (warp > 0 ? warp_tot[warp - 1] : 0);
  *total = warp_tot[31];
  __syncthreads();  // warp_tot is reused by the next call
  return res;
}

__global__ void __launch_bounds__(kPlanThreads) plan_device_kernel(
    const int32_t* __restrict__ seq_lens, int32_t B, int32_t num_sms, int32_t* __restrict__ w,
    PlanLayout L, int32_t* __restrict__ err, int32_t units) {
  extern __shared__ int32_t dsm[];
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t bad;
  griddep_wait();  // seq_lens may come from the preceding kernel
  griddep_launch_dependents();
  const bool staged = B <= kSmemSeqs;
  int32_t* cu_g = w + L.cu_off();
  int32_t* so_g = w + L.seq_off();
  int32_t* cu = staged ? dsm : cu_g;              // read copies
  int32_t* so = staged ? dsm + (B + 1) : so_g;
  int32_t* part_off = w + L.part_off();
  int32_t* segs = w + L.seg_off();
  const int tid = threadIdx.x;
  if (tid == 0) {
    bad = 0;
    cu[0] = 0;
    cu_g[0] = 0;
  }
  __syncthreads();

  // 1. tile counts and their prefix sum cu[0..B]
  int64_t carry = 0;
  for (int32_t base = 0; base < B; base += kPlanThreads) {
    const int32_t b = base + tid;
    int32_t n = 0;
    if (b < B) {
      const int32_t len = seq_lens[b];
      if (len < 0) bad = 1;  // benign race: every writer stores 1
      n = len > 0 ? (int32_t)((len + kBlockTokens - 1) / kBlockTokens) * units : 0;
    }
    int32_t chunk_total;
    const int32_t incl = block_inclusive_scan(n, warp_tot, &chunk_total);
    if (b < B) {
      const int64_t v = carry + incl;
      if (v > INT32_MAX) bad = 1;
      cu[b + 1] = (int32_t)v;
      if (staged) cu_g[b + 1] = (int32_t)v;
    }
    carry += chunk_total;
  }
  __syncthreads();
  if (bad || carry > INT32_MAX) {
    // Empty plan; the attention kernel then does nothing for this step.
    if (tid == 0) {
      atomicOr(err, HPC_DEVCHK_BAD_LENGTH);
      w[kMagic] = kPlanMagic; w[kKind] = HPC_PLAN_DYNAMIC; w[kNumSeqs] = B;
      w[kNumParts] = 0; w[kNumTiles] = 0; w[kNumSegs] = 0; w[kNumSms] = num_sms;
      w[kSplits] = units > 1 ? units : 0; part_off[0] = 0;
    }
    for (int32_t b = tid; b <= B; b += kPlanThreads) so_g[b] = 0;
    return;
  }
  const int64_t T = carry;
  const int64_t P = T < num_sms ? T : num_sms;
  PartMath pm{T, P, (T + 1) * (P + 1) < (int64_t)UINT32_MAX};

  // 2. segments per sequence -> seq_seg_off
  if (tid == 0) {
    so[0] = 0;
    so_g[0] = 0;
  }
  int64_t gcarry = 0;
  for (int32_t base = 0; base < B; base += kPlanThreads) {
    const int32_t b = base + tid;
    int32_t cnt = 0;
    if (b < B) {
      const int64_t lo_b = cu[b], hi_b = cu[b + 1];
      if (hi_b > lo_b) cnt = (int32_t)(pm.of(hi_b - 1) - pm.of(lo_b) + 1);
    }
    int32_t chunk_total;
    const int32_t incl = block_inclusive_scan(cnt, warp_tot, &chunk_total);
    if (b < B) {
      so[b + 1] = (int32_t)(gcarry + incl);
      if (staged) so_g[b + 1] = (int32_t)(gcarry + incl);
    }
    gcarry += chunk_total;
  }
  __syncthreads();
  const int32_t S = (int32_t)gcarry;

  // 3. the segments, one thread each: sequence = last b with so[b] <= g
  for (int32_t g = tid; g < S; g += kPlanThreads) {
    int32_t lo = 0, hi = B;
    while (hi - lo > 1) {
      const int32_t mid = (lo + hi) >> 1;
      if (so[mid] <= g) lo = mid; else hi = mid;
    }
    const int32_t b = lo, j = g - so[b];
    const int64_t lo_b = cu[b], hi_b = cu[b + 1];
    const int32_t cnt = so[b + 1] - so[b];
    const int64_t p = pm.of(lo_b) + j;
    const int64_t s0 = pm.start(p), s1 = pm.start(p + 1);
    int4 rec;
    rec.x = b;
    rec.y = (int32_t)((lo_b > s0 ? lo_b : s0) - lo_b);
    rec.z = (int32_t)((hi_b < s1 ? hi_b : s1) - lo_b);
    rec.w = cnt == 1 ? HPC_SEG_WHOLE : 0;
    *reinterpret_cast<int4*>(segs + 4 * (int64_t)g) = rec;
  }

  // 4. first segment of each part
  for (int64_t p = tid; p < P; p += kPlanThreads) {
    const int32_t s = (int32_t)pm.start(p);
    int32_t lo = 0, hi = B;  // the last b with cu[b] <= s (a non-empty sequence)
    while (hi - lo > 1) {
      const int32_t mid = (lo + hi) >> 1;
      if (cu[mid] <= s) lo = mid; else hi = mid;
    }
    part_off[p] = so[lo] + (int32_t)(p - pm.of(cu[lo]));
  }
  if (tid == 0) {
    part_off[P] = (int32_t)gcarry;
    w[kMagic] = kPlanMagic;
    w[kKind] = HPC_PLAN_DYNAMIC;
    w[kNumSeqs] = B;
    w[kNumParts] = (int32_t)P;
    w[kNumTiles] = (int32_t)T;
    w[kNumSegs] = (int32_t)gcarry;
    w[kNumSms] = num_sms;
    w[kSplits] = units > 1 ? units : 0;
  }
}

}  // namespace

cudaError_t launch_plan_device(const int32_t* seq_lens, int32_t num_seqs, int32_t num_sms,
                               int32_t* words, const PlanLayout& L, int32_t* err,
                               cudaStream_t stream, int32_t units_per_tile) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(kPlanThreads);
  cfg.dynamicSmemBytes =
      num_seqs <= kSmemSeqs ? (size_t)2 * (num_seqs + 1) * sizeof(int32_t) : 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, plan_device_kernel, seq_lens, num_seqs, num_sms, words, L, err,
                            units_per_tile);
}

}  // namespace hpc
