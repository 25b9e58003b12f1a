// Device tile planner: the per-step load-balanced plan computed on the GPU
// from device lengths, with no host round trip ("vLLM x HPC-Ops", section
// "Attention Backend: Dynamic Load-Balanced Scheduling": a per-step
// scheduler). It writes the same words as the host planner (plan_host.cu):
// both evaluate the same closed forms
//   part start  s_p = floor(p*T/P),   part of tile x = floor(((x+1)*P - 1)/T),
// so the results agree bit for bit.
//
// One CTA of 1024 threads walks the sequences in chunks of 1024 with two
// block-wide scans (tile counts, then segments per sequence). The prefix
// arrays are kept in shared memory when they fit, so the per-part searches
// never wait on global memory.
#include "hpc_internal.h"
#include "ptx.cuh"

namespace hpc {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kSmemSeqs = 6000;  // 2 * (6000 + 1) int32 fit the default 48 KB

__device__ __forceinline__ int64_t dpart_start(int64_t p, int64_t T, int64_t P) {
  return (p * T) / P;
}
__device__ __forceinline__ int64_t dpart_of(int64_t x, int64_t T, int64_t P) {
  return ((x + 1) * P - 1) / T;
}

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
    PlanLayout L, int32_t* __restrict__ err) {
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
      n = len > 0 ? (int32_t)((len + kBlockTokens - 1) / kBlockTokens) : 0;
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
      w[kSplits] = 0; part_off[0] = 0;
    }
    for (int32_t b = tid; b <= B; b += kPlanThreads) so_g[b] = 0;
    return;
  }
  const int64_t T = carry;
  const int64_t P = T < num_sms ? T : num_sms;

  // 2. segments per sequence -> seq_seg_off, and 3. the segments themselves
  if (tid == 0) {
    so[0] = 0;
    so_g[0] = 0;
  }
  int64_t gcarry = 0;
  for (int32_t base = 0; base < B; base += kPlanThreads) {
    const int32_t b = base + tid;
    int32_t cnt = 0;
    int64_t pf = 0, lo_b = 0, hi_b = 0;
    if (b < B) {
      lo_b = cu[b];
      hi_b = cu[b + 1];
      if (hi_b > lo_b) {
        pf = dpart_of(lo_b, T, P);
        cnt = (int32_t)(dpart_of(hi_b - 1, T, P) - pf + 1);
      }
    }
    int32_t chunk_total;
    const int32_t incl = block_inclusive_scan(cnt, warp_tot, &chunk_total);
    if (b < B) {
      const int64_t first = gcarry + incl - cnt;
      so[b + 1] = (int32_t)(first + cnt);
      if (staged) so_g[b + 1] = (int32_t)(first + cnt);
      for (int32_t j = 0; j < cnt; ++j) {
        const int64_t p = pf + j;
        const int64_t s0 = dpart_start(p, T, P), s1 = dpart_start(p + 1, T, P);
        int4 rec;
        rec.x = b;
        rec.y = (int32_t)((lo_b > s0 ? lo_b : s0) - lo_b);
        rec.z = (int32_t)((hi_b < s1 ? hi_b : s1) - lo_b);
        rec.w = cnt == 1 ? HPC_SEG_WHOLE : 0;
        *reinterpret_cast<int4*>(segs + 4 * (first + j)) = rec;
      }
    }
    gcarry += chunk_total;
  }
  __syncthreads();

  // 4. first segment of each part
  for (int64_t p = tid; p < P; p += kPlanThreads) {
    const int32_t s = (int32_t)dpart_start(p, T, P);
    int32_t lo = 0, hi = B;  // the last b with cu[b] <= s (a non-empty sequence)
    while (hi - lo > 1) {
      const int32_t mid = (lo + hi) >> 1;
      if (cu[mid] <= s) lo = mid; else hi = mid;
    }
    part_off[p] = so[lo] + (int32_t)(p - dpart_of(cu[lo], T, P));
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
    w[kSplits] = 0;
  }
}

}  // namespace

cudaError_t launch_plan_device(const int32_t* seq_lens, int32_t num_seqs, int32_t num_sms,
                               int32_t* words, const PlanLayout& L, int32_t* err,
                               cudaStream_t stream) {
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
  return cudaLaunchKernelEx(&cfg, plan_device_kernel, seq_lens, num_seqs, num_sms, words, L, err);
}

}  // namespace hpc
