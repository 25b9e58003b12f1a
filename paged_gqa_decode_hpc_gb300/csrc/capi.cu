// C ABI of libhpc_decode.so: argument checks, plan objects, TMA descriptors
// and launches. See include/hpc_decode.h for the contract of every call.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "decode_tc.h"
#include "hpc_internal.h"
#include "prefill.h"

namespace hpc {

namespace {
thread_local std::string g_last_error;

hpc_status fail(hpc_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

#define HPC_CUDA_TRY(expr)                                                                  \
  do {                                                                                      \
    cudaError_t e__ = (expr);                                                               \
    if (e__ != cudaSuccess) {                                                               \
      return fail(e__ == cudaErrorMemoryAllocation ? HPC_ERR_OOM : HPC_ERR_CUDA,            \
                  std::string(#expr) + ": " + cudaGetErrorString(e__));                     \
    }                                                                                       \
  } while (0)

unsigned long long wait_limit_ns() {
  static unsigned long long v = [] {
    const char* s = std::getenv("HPC_DECODE_WAIT_LIMIT_MS");
    long long ms = s ? std::atoll(s) : 2000;
    if (ms < 0) ms = 2000;
    return (unsigned long long)ms * 1000000ull;
  }();
  return v;
}

// Failure-path test switch: with HPC_DECODE_TEST_WITHHOLD_COPIES=1 the
// producers of the attention and extend kernels issue no copies, so every
// consumer wait runs out (bounded by HPC_DECODE_WAIT_LIMIT_MS) and the call
// must come back with HPC_DEVCHK_TIMEOUT and a usable context. Read at every
// call, so a test can follow a failed step with a normal one on the same plan.
bool withhold_copies() {
  const char* s = std::getenv("HPC_DECODE_TEST_WITHHOLD_COPIES");
  return s && s[0] == '1';
}

// Smallest q_len (new tokens per sequence) that hpc_decode_attn* and
// hpc_decode_step run on the tensor-core decode kernel (decode_tc_kernel.cu)
// instead of the one-warp-per-token kernel (attn_kernel.cu); values above
// kMaxQueryTokens turn the tensor-core path off. 0 selects the measured
// crossover of each cache dtype: on the skewed 1 x 128K + 31 x 4K batch the
// tensor-core kernel is faster from q_len 4 with a bf16 cache (170 vs
// 173 us) and from q_len 3 with an e4m3 cache (159 vs 171 us).
std::atomic<int32_t> g_tc_min_q_len{0};
int32_t tc_min_q_len(bool fp8) {
  const int32_t v = g_tc_min_q_len.load(std::memory_order_relaxed);
  return v > 0 ? v : (fp8 ? 3 : 4);
}

// Parts of the tile plan hpc_decode_step builds for a step of this shape on
// num_sms SMs: max(1, num_sms / H_kv) when q_len reaches the tensor-core
// threshold (one CTA per (KV head, part)), else num_sms. Sets *tensor_core
// accordingly.
int32_t decode_plan_parts(const hpc_tensor* q, const hpc_tensor* k_cache, int32_t num_sms,
                          bool* tensor_core) {
  const int64_t T = (q && q->ndim == 4) ? q->shape[1] : 1;
  const bool fp8 = k_cache && k_cache->dtype == HPC_FP8_E4M3;
  const bool tc = q && q->ndim == 4 && T >= tc_min_q_len(fp8) && T <= kMaxQueryTokens;
  if (tensor_core) *tensor_core = tc;
  if (!tc) return num_sms;
  const int64_t hkv =
      (k_cache && k_cache->ndim == 4 && k_cache->shape[1] > 0) ? k_cache->shape[1] : 1;
  return (int32_t)std::max<int64_t>(1, num_sms / hkv);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

void free_plan(hpc_plan_s* pl) {
  if (!pl) return;
  if (pl->d_words) cudaFree(pl->d_words);
  if (pl->d_err) cudaFree(pl->d_err);
  if (pl->d_ws) cudaFree(pl->d_ws);
  if (pl->d_step) cudaFree(pl->d_step);
  if (pl->d_stage) cudaFree(pl->d_stage);
  if (pl->h_pinned) cudaFreeHost(pl->h_pinned);
  if (pl->copy_done) cudaEventDestroy(pl->copy_done);
  delete pl;
}

// Allocate the plan buffer + error word for layout L on the current device.
hpc_status alloc_plan_buffers(hpc_plan_s* pl) {
  HPC_CUDA_TRY(cudaGetDevice(&pl->device));
  HPC_CUDA_TRY(cudaMalloc(&pl->d_words, (size_t)pl->layout.words() * sizeof(int32_t)));
  HPC_CUDA_TRY(cudaMalloc(&pl->d_err, sizeof(int32_t)));
  HPC_CUDA_TRY(cudaMemset(pl->d_err, 0, sizeof(int32_t)));
  return HPC_OK;
}

hpc_status ensure_workspace(hpc_plan_s* pl, int64_t num_q_heads, bool may_allocate) {
  if (pl->d_ws && pl->ws_heads >= num_q_heads) return HPC_OK;
  if (!may_allocate)
    return fail(HPC_ERR_INVALID_ARG,
                "plan workspace was sized for fewer query heads; create the plan with "
                "num_q_heads >= " + std::to_string(num_q_heads));
  if (pl->d_ws) {
    HPC_CUDA_TRY(cudaDeviceSynchronize());
    cudaFree(pl->d_ws);
    pl->d_ws = nullptr;
  }
  size_t floats = (size_t)std::max<int64_t>(pl->layout.cap_segs, 1) * num_q_heads *
                  (kHeadDim + 2);
  if (pl->d_step)  // a one-token step's partial states
    floats = std::max(floats, (size_t)step_ws_floats(pl->layout.cap_parts));
  HPC_CUDA_TRY(cudaMalloc(&pl->d_ws, floats * sizeof(float)));
  pl->ws_heads = num_q_heads;
  pl->ws_floats = (int64_t)floats;
  return HPC_OK;
}

int elt_bytes(int32_t dt) {
  switch (dt) {
    case HPC_BF16: return 2;
    case HPC_FP8_E4M3: return 1;
    case HPC_F32: case HPC_I32: return 4;
    default: return 0;
  }
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

hpc_status check_tensor(const hpc_tensor* t, const char* name, int ndim, bool nullable = false) {
  if (!t || !t->data) {
    if (nullable && (!t || !t->data)) return HPC_OK;
    return fail(HPC_ERR_INVALID_ARG, std::string(name) + " is null");
  }
  if (t->ndim != ndim)
    return fail(HPC_ERR_INVALID_ARG, std::string(name) + " must have " + std::to_string(ndim) +
                                         " dimensions");
  for (int i = 0; i < ndim; ++i)
    if (t->shape[i] < 0 || t->stride[i] < 0)
      return fail(HPC_ERR_INVALID_ARG, std::string(name) + " has a negative shape or stride");
  if (elt_bytes(t->dtype) == 0) return fail(HPC_ERR_INVALID_ARG, std::string(name) + ": bad dtype");
  return HPC_OK;
}

// 4-D TMA descriptor over a [blocks][kv heads][64][128] cache (any strides
// that are multiples of 16 bytes). The two middle dimensions are ordered by
// stride so that either cache layout maps onto a monotone tensor.
hpc_status make_kv_map(const hpc_tensor* t, bool fp8, bool swap, CUtensorMap* map) {
  auto enc = encode_fn();
  if (!enc) return fail(HPC_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const int64_t e = fp8 ? 1 : 2;
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
  dims[0] = kHeadDim;
  box[0] = fp8 ? 128 : 64;
  if (!swap) {
    dims[1] = kBlockTokens; dims[2] = (cuuint64_t)t->shape[1];
    strides[0] = t->stride[2] * e; strides[1] = t->stride[1] * e;
    box[1] = kBlockTokens; box[2] = 1;
  } else {
    dims[1] = (cuuint64_t)t->shape[1]; dims[2] = kBlockTokens;
    strides[0] = t->stride[1] * e; strides[1] = t->stride[2] * e;
    box[1] = 1; box[2] = kBlockTokens;
  }
  dims[3] = (cuuint64_t)t->shape[0];
  strides[2] = t->stride[0] * e;
  box[3] = 1;
  CUresult r = enc(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                   t->data, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(HPC_ERR_INVALID_ARG, "cuTensorMapEncodeTiled rejected the KV cache (error " +
                                         std::to_string((int)r) + ")");
  return HPC_OK;
}

// Copy a capacity-layout word array into the canonical export layout.
hpc_status write_canonical(const int32_t* w, const PlanLayout& L, int32_t* buf, int64_t cap,
                           int64_t* len) {
  const int32_t B = w[kNumSeqs], P = w[kNumParts], S = w[kNumSegs];
  if (w[kMagic] != kPlanMagic || B < 0 || B > L.cap_seqs || P < 0 || P > L.cap_parts || S < 0 ||
      S > L.cap_segs)
    return fail(HPC_ERR_DEVICE_CHECK, "plan buffer is inconsistent");
  const int64_t n = kHeaderWords + (P + 1) + (B + 1) + 4LL * S;
  *len = n;
  if (cap == 0 && !buf) return HPC_OK;
  if (!buf || cap < n) return fail(HPC_ERR_INVALID_ARG, "export buffer too small");
  int64_t o = 0;
  for (int i = 0; i < kHeaderWords; ++i) buf[o++] = w[i];
  for (int i = 0; i <= P; ++i) buf[o++] = w[L.part_off() + i];
  for (int i = 0; i <= B; ++i) buf[o++] = w[L.seq_off() + i];
  for (int64_t i = 0; i < 4LL * S; ++i) buf[o++] = w[L.seg_off() + i];
  return HPC_OK;
}

hpc_status new_host_plan(const int32_t* words, const PlanLayout& L, int32_t kind,
                         int32_t num_sms, int32_t num_seqs, int32_t parts, int32_t segs,
                         int32_t kv_heads, hpc_plan_t* out) {
  hpc_plan_s* pl = new (std::nothrow) hpc_plan_s();
  if (!pl) return fail(HPC_ERR_OOM, "host allocation failed");
  pl->kind = kind;
  pl->layout = L;
  pl->num_sms = num_sms;
  pl->max_seqs = num_seqs;
  pl->num_seqs = num_seqs;
  pl->host_num_parts = parts;
  pl->host_num_segs = segs;
  pl->static_kv_heads = kv_heads;
  hpc_status st = alloc_plan_buffers(pl);
  if (st == HPC_OK) {
    cudaError_t e = cudaMemcpy(pl->d_words, words, (size_t)L.words() * sizeof(int32_t),
                               cudaMemcpyHostToDevice);
    if (e != cudaSuccess) st = fail(HPC_ERR_CUDA, std::string("plan upload: ") +
                                                      cudaGetErrorString(e));
  }
  if (st != HPC_OK) {
    free_plan(pl);
    return st;
  }
  *out = pl;
  return HPC_OK;
}

}  // namespace

void set_error(const std::string& msg) { g_last_error = msg; }


}  // namespace hpc

using namespace hpc;

extern "C" {

const char* hpc_last_error(void) { return g_last_error.c_str(); }

hpc_status hpc_device_sm_count(int32_t* num_sms) {
  if (!num_sms) return fail(HPC_ERR_INVALID_ARG, "num_sms is null");
  int dev = 0, n = 0;
  HPC_CUDA_TRY(cudaGetDevice(&dev));
  HPC_CUDA_TRY(cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev));
  *num_sms = n;
  return HPC_OK;
}

hpc_status hpc_decode_plan(const int32_t* seq_lens, int32_t num_seqs, int32_t num_sms,
                           hpc_plan_t* plan_out) {
  return hpc_decode_plan_ex(seq_lens, num_seqs, num_sms, 1, plan_out);
}

hpc_status hpc_decode_plan_ex(const int32_t* seq_lens, int32_t num_seqs, int32_t num_sms,
                              int32_t units_per_tile, hpc_plan_t* plan_out) {
  if (!plan_out) return fail(HPC_ERR_INVALID_ARG, "plan_out is null");
  *plan_out = nullptr;
  if (num_seqs < 0 || (num_seqs > 0 && !seq_lens))
    return fail(HPC_ERR_INVALID_ARG, "seq_lens is null or num_seqs < 0");
  if (num_sms <= 0) return fail(HPC_ERR_INVALID_ARG, "num_sms must be positive");
  if (units_per_tile <= 0) return fail(HPC_ERR_INVALID_ARG, "units_per_tile must be positive");
  int64_t T = 0;
  for (int32_t b = 0; b < num_seqs; ++b) {
    if (seq_lens[b] < 0)
      return fail(HPC_ERR_INVALID_ARG, "negative sequence length at index " + std::to_string(b));
    T += (seq_lens[b] + (int64_t)kBlockTokens - 1) / kBlockTokens * units_per_tile;
  }
  PlanLayout L;
  L.cap_seqs = num_seqs;
  L.cap_parts = (int32_t)std::min<int64_t>(num_sms, T);
  L.cap_segs = (int32_t)dynamic_max_segs(num_seqs, L.cap_parts);
  std::vector<int32_t> w((size_t)L.words(), 0);
  std::string err;
  hpc_status st = plan_dynamic_host(seq_lens, num_seqs, num_sms, w.data(), L, &err,
                                    units_per_tile);
  if (st != HPC_OK) return fail(st, err);
  st = new_host_plan(w.data(), L, HPC_PLAN_DYNAMIC, num_sms, num_seqs, w[kNumParts],
                     w[kNumSegs], 0, plan_out);
  if (st == HPC_OK) (*plan_out)->units = units_per_tile;
  return st;
}

hpc_status hpc_decode_plan_static(const int32_t* seq_lens, int32_t num_seqs, int32_t num_sms,
                                  int32_t num_kv_heads, int32_t num_splits,
                                  hpc_plan_t* plan_out) {
  if (!plan_out) return fail(HPC_ERR_INVALID_ARG, "plan_out is null");
  *plan_out = nullptr;
  int32_t* w = nullptr;
  PlanLayout L;
  std::string err;
  hpc_status st =
      plan_static_host(seq_lens, num_seqs, num_sms, num_kv_heads, num_splits, &w, &L, &err);
  if (st != HPC_OK) return fail(st, err);
  st = new_host_plan(w, L, HPC_PLAN_STATIC, num_sms, num_seqs, w[kNumParts], w[kNumSegs],
                     num_kv_heads, plan_out);
  free(w);
  return st;
}

hpc_status hpc_decode_plan_create(int32_t max_seqs, int32_t num_sms, int32_t num_q_heads,
                                  hpc_plan_t* plan_out) {
  if (!plan_out) return fail(HPC_ERR_INVALID_ARG, "plan_out is null");
  *plan_out = nullptr;
  if (max_seqs < 0 || num_sms <= 0 || num_q_heads <= 0)
    return fail(HPC_ERR_INVALID_ARG, "max_seqs >= 0, num_sms > 0 and num_q_heads > 0 required");
  hpc_plan_s* pl = new (std::nothrow) hpc_plan_s();
  if (!pl) return fail(HPC_ERR_OOM, "host allocation failed");
  pl->kind = HPC_PLAN_DYNAMIC;
  pl->layout.cap_seqs = max_seqs;
  pl->layout.cap_parts = num_sms;
  pl->layout.cap_segs = (int32_t)dynamic_max_segs(max_seqs, num_sms);
  pl->num_sms = num_sms;
  pl->max_seqs = max_seqs;
  pl->num_seqs = 0;
  pl->host_num_parts = 0;
  pl->host_num_segs = 0;
  auto cleanup = [&](hpc_status st) {
    free_plan(pl);
    return st;
  };
  hpc_status st = alloc_plan_buffers(pl);
  if (st != HPC_OK) return cleanup(st);
  pl->step_kv_heads = std::max(1, num_q_heads / kGroup);
  {
    const size_t sb = (size_t)step_words(num_sms, max_seqs, pl->step_kv_heads) * sizeof(int32_t);
    if (cudaMalloc(&pl->d_step, sb) != cudaSuccess || cudaMemset(pl->d_step, 0, sb) != cudaSuccess)
      return cleanup(fail(HPC_ERR_OOM, "step counters allocation failed"));
  }
  st = ensure_workspace(pl, num_q_heads, true);
  if (st != HPC_OK) return cleanup(st);
  const size_t bytes = (size_t)pl->layout.words() * sizeof(int32_t);
  if (cudaMallocHost(&pl->h_pinned, bytes) != cudaSuccess ||
      cudaEventCreateWithFlags(&pl->copy_done, cudaEventDisableTiming) != cudaSuccess)
    return cleanup(fail(HPC_ERR_OOM, "pinned host allocation failed"));
  // an empty step: zero sequences
  std::memset(pl->h_pinned, 0, bytes);
  std::string err;
  st = plan_dynamic_host(nullptr, 0, num_sms, pl->h_pinned, pl->layout, &err);
  if (st != HPC_OK) return cleanup(fail(st, err));
  if (cudaMemcpy(pl->d_words, pl->h_pinned, bytes, cudaMemcpyHostToDevice) != cudaSuccess)
    return cleanup(fail(HPC_ERR_CUDA, "plan upload failed"));
  *plan_out = pl;
  return HPC_OK;
}

hpc_status hpc_decode_plan_device(const int32_t* seq_lens_dev, int32_t num_seqs, int32_t num_sms,
                                  hpc_plan_t plan, void* stream) {
  if (!plan || plan->kind != HPC_PLAN_DYNAMIC || !plan->h_pinned)
    return fail(HPC_ERR_INVALID_ARG, "plan must come from hpc_decode_plan_create");
  if (num_seqs < 0 || (num_seqs > 0 && !seq_lens_dev))
    return fail(HPC_ERR_INVALID_ARG, "seq_lens_dev is null or num_seqs < 0");
  if (num_seqs > plan->layout.cap_seqs)
    return fail(HPC_ERR_INVALID_ARG, "num_seqs exceeds the plan's max_seqs");
  if (num_sms <= 0 || num_sms > plan->layout.cap_parts)
    return fail(HPC_ERR_INVALID_ARG, "num_sms must be in [1, plan num_sms]");
  cudaError_t e = launch_plan_device(seq_lens_dev, num_seqs, num_sms, plan->d_words, plan->layout,
                                     plan->d_err, (cudaStream_t)stream);
  if (e != cudaSuccess)
    return fail(HPC_ERR_CUDA, std::string("device planner launch: ") + cudaGetErrorString(e));
  plan->num_seqs = num_seqs;
  plan->num_sms = num_sms;
  plan->host_num_parts = -1;
  plan->host_num_segs = -1;
  plan->units = 1;
  return HPC_OK;
}

hpc_status hpc_decode_plan_update(const int32_t* seq_lens, int32_t num_seqs, int32_t num_sms,
                                  hpc_plan_t plan, void* stream) {
  if (!plan || plan->kind != HPC_PLAN_DYNAMIC || !plan->h_pinned)
    return fail(HPC_ERR_INVALID_ARG, "plan must come from hpc_decode_plan_create");
  if (num_sms <= 0 || num_sms > plan->layout.cap_parts)
    return fail(HPC_ERR_INVALID_ARG, "num_sms must be in [1, plan num_sms]");
  // the staging buffer may still feed the previous upload
  HPC_CUDA_TRY(cudaEventSynchronize(plan->copy_done));
  std::string err;
  hpc_status st = plan_dynamic_host(seq_lens, num_seqs, num_sms, plan->h_pinned, plan->layout,
                                    &err);
  if (st != HPC_OK) return fail(st, err);
  HPC_CUDA_TRY(cudaMemcpyAsync(plan->d_words, plan->h_pinned,
                               (size_t)plan->layout.words() * sizeof(int32_t),
                               cudaMemcpyHostToDevice, (cudaStream_t)stream));
  HPC_CUDA_TRY(cudaEventRecord(plan->copy_done, (cudaStream_t)stream));
  plan->num_seqs = num_seqs;
  plan->num_sms = num_sms;
  plan->host_num_parts = plan->h_pinned[kNumParts];
  plan->host_num_segs = plan->h_pinned[kNumSegs];
  plan->units = 1;
  return HPC_OK;
}

hpc_status hpc_decode_plan_export(hpc_plan_t plan, int32_t* buf, int64_t cap, int64_t* len) {
  if (!plan || !len) return fail(HPC_ERR_INVALID_ARG, "plan or len is null");
  const PlanLayout& L = plan->layout;
  std::vector<int32_t> w((size_t)L.words());
  HPC_CUDA_TRY(cudaDeviceSynchronize());
  HPC_CUDA_TRY(cudaMemcpy(w.data(), plan->d_words, w.size() * sizeof(int32_t),
                          cudaMemcpyDeviceToHost));
  if (w[kMagic] == kPlanMagic && w[kKind] == HPC_PLAN_STEP) {
    // header, then one record per owner (parts, then pool chunks):
    // first unit, end unit, pieces, executions since the plan was created
    const int64_t owners = (int64_t)w[kNumParts] + w[kNumSegs];
    if (!plan->d_step || owners < 0 || owners > (1 + kStepChunksPerCta) * (int64_t)L.cap_parts)
      return fail(HPC_ERR_DEVICE_CHECK, "plan buffer is inconsistent");
    const int64_t n = kHeaderWords + 4 * owners;
    *len = n;
    if (cap == 0 && !buf) return HPC_OK;
    if (!buf || cap < n) return fail(HPC_ERR_INVALID_ARG, "export buffer too small");
    for (int i = 0; i < kHeaderWords; ++i) buf[i] = w[i];
    if (owners > 0)
      HPC_CUDA_TRY(cudaMemcpy(buf + kHeaderWords, plan->d_step + step_rec_off(),
                              (size_t)(4 * owners) * sizeof(int32_t), cudaMemcpyDeviceToHost));
    return HPC_OK;
  }
  return write_canonical(w.data(), L, buf, cap, len);
}

hpc_status hpc_decode_plan_compute(const int32_t* seq_lens, int32_t num_seqs, int32_t num_sms,
                                   int32_t* buf, int64_t cap, int64_t* len) {
  return hpc_decode_plan_compute_ex(seq_lens, num_seqs, num_sms, 1, buf, cap, len);
}

hpc_status hpc_decode_plan_compute_ex(const int32_t* seq_lens, int32_t num_seqs, int32_t num_sms,
                                      int32_t units_per_tile, int32_t* buf, int64_t cap,
                                      int64_t* len) {
  if (!len) return fail(HPC_ERR_INVALID_ARG, "len is null");
  if (num_seqs < 0 || (num_seqs > 0 && !seq_lens))
    return fail(HPC_ERR_INVALID_ARG, "seq_lens is null or num_seqs < 0");
  if (num_sms <= 0) return fail(HPC_ERR_INVALID_ARG, "num_sms must be positive");
  PlanLayout L;
  L.cap_seqs = num_seqs;
  L.cap_parts = num_sms;
  L.cap_segs = (int32_t)dynamic_max_segs(num_seqs, num_sms);
  std::vector<int32_t> w((size_t)L.words(), 0);
  std::string err;
  hpc_status st = plan_dynamic_host(seq_lens, num_seqs, num_sms, w.data(), L, &err,
                                    units_per_tile);
  if (st != HPC_OK) return fail(st, err);
  return write_canonical(w.data(), L, buf, cap, len);
}

hpc_status hpc_decode_plan_static_compute(const int32_t* seq_lens, int32_t num_seqs,
                                          int32_t num_sms, int32_t num_kv_heads,
                                          int32_t num_splits, int32_t* buf, int64_t cap,
                                          int64_t* len) {
  if (!len) return fail(HPC_ERR_INVALID_ARG, "len is null");
  int32_t* w = nullptr;
  PlanLayout L;
  std::string err;
  hpc_status st =
      plan_static_host(seq_lens, num_seqs, num_sms, num_kv_heads, num_splits, &w, &L, &err);
  if (st != HPC_OK) return fail(st, err);
  st = write_canonical(w, L, buf, cap, len);
  free(w);
  return st;
}

hpc_status hpc_decode_plan_status(hpc_plan_t plan, int32_t* device_error) {
  if (!plan || !device_error) return fail(HPC_ERR_INVALID_ARG, "plan or device_error is null");
  HPC_CUDA_TRY(cudaDeviceSynchronize());
  int32_t v = 0;
  HPC_CUDA_TRY(cudaMemcpy(&v, plan->d_err, sizeof v, cudaMemcpyDeviceToHost));
  HPC_CUDA_TRY(cudaMemset(plan->d_err, 0, sizeof v));
  *device_error = v;
  if (v != 0)
    return fail(HPC_ERR_DEVICE_CHECK, "device check fired (bits " + std::to_string(v) + ")");
  return HPC_OK;
}

void hpc_decode_plan_destroy(hpc_plan_t plan) {
  if (!plan) return;
  cudaDeviceSynchronize();
  free_plan(plan);
}

}  // extern "C"

namespace hpc {
namespace {
// 4-D TMA descriptor over q [B][q_len][H_q][128] for the tensor-core decode
// kernel: box (64 columns, 8 heads, q_len tokens, 1 sequence), 128-byte
// swizzle. False when the strides do not form such a tensor (the caller then
// keeps the one-warp-per-token kernel).
bool make_decode_q_map(const hpc_tensor* q, CUtensorMap* map) {
  auto enc = encode_fn();
  if (!enc || q->ndim != 4) return false;
  cuuint64_t dims[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)q->shape[2], (cuuint64_t)q->shape[1],
                        (cuuint64_t)q->shape[0]};
  cuuint64_t strides[3] = {(cuuint64_t)q->stride[2] * 2, (cuuint64_t)q->stride[1] * 2,
                           (cuuint64_t)q->stride[0] * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)kGroup, (cuuint32_t)q->shape[1], 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, q->data, dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Attention + merge. fused_num_sms > 0: the attention kernel plans the step
// itself (P = min(fused_num_sms, T)) and writes the plan words into `plan`.
hpc_status attn_impl(const hpc_tensor* q, const hpc_tensor* k_cache, const hpc_tensor* v_cache,
                     const hpc_tensor* block_table, const hpc_tensor* seq_lens, hpc_plan_t plan,
                     hpc_tensor* out, hpc_tensor* lse, float softmax_scale, void* stream,
                     int32_t fused_num_sms, bool check_only, int32_t step_grid = 0) {
  hpc_status st;
  // q/out are [B][H_q][128] (one query token per sequence) or
  // [B][q_len][H_q][128] (q_len new tokens; lse then [B][q_len][H_q]).
  const int qnd = q ? q->ndim : 0;
  if (qnd != 3 && qnd != 4) return fail(HPC_ERR_INVALID_ARG, "q must be [B][H_q][128] or [B][q_len][H_q][128]");
  if ((st = check_tensor(q, "q", qnd)) != HPC_OK) return st;
  if ((st = check_tensor(k_cache, "k_cache", 4)) != HPC_OK) return st;
  if ((st = check_tensor(v_cache, "v_cache", 4)) != HPC_OK) return st;
  if ((st = check_tensor(block_table, "block_table", 2)) != HPC_OK) return st;
  if ((st = check_tensor(seq_lens, "seq_lens", 1)) != HPC_OK) return st;
  if ((st = check_tensor(out, "out", qnd)) != HPC_OK) return st;
  if ((st = check_tensor(lse, "lse", qnd - 1, true)) != HPC_OK) return st;
  if (!plan) return fail(HPC_ERR_INVALID_ARG, "plan is null");
  const bool has_lse = lse && lse->data;
  const bool multi = qnd == 4;
  const int64_t B = q->shape[0], T = multi ? q->shape[1] : 1;
  const int64_t Hq = q->shape[qnd - 2], D = q->shape[qnd - 1];
  const int64_t q_st = multi ? q->stride[1] : 0, q_sh = q->stride[qnd - 2];
  const int64_t o_st = multi ? out->stride[1] : 0, o_sh = out->stride[qnd - 2];
  const int64_t l_st = (has_lse && multi) ? lse->stride[1] : 0;
  const int64_t l_sh = has_lse ? lse->stride[qnd - 2] : 0;
  const int64_t NB = k_cache->shape[0], Hkv = k_cache->shape[1];
  if (q->dtype != HPC_BF16) return fail(HPC_ERR_INVALID_ARG, "q must be bf16");
  if (out->dtype != HPC_BF16) return fail(HPC_ERR_INVALID_ARG, "out must be bf16");
  if (k_cache->dtype != v_cache->dtype ||
      (k_cache->dtype != HPC_BF16 && k_cache->dtype != HPC_FP8_E4M3))
    return fail(HPC_ERR_INVALID_ARG, "k_cache/v_cache must both be bf16 or both fp8_e4m3");
  const bool fp8 = k_cache->dtype == HPC_FP8_E4M3;
  for (int i = 0; i < 4; ++i)
    if (k_cache->shape[i] != v_cache->shape[i] || k_cache->stride[i] != v_cache->stride[i])
      return fail(HPC_ERR_INVALID_ARG, "k_cache and v_cache must have the same shape and strides");
  if (D != kHeadDim || k_cache->shape[3] != kHeadDim)
    return fail(HPC_ERR_UNSUPPORTED, "head_dim must be 128");
  if (k_cache->shape[2] != kBlockTokens)
    return fail(HPC_ERR_UNSUPPORTED, "KV blocks must hold 64 tokens");
  if (Hkv <= 0 || Hq != kGroup * Hkv)
    return fail(HPC_ERR_UNSUPPORTED, "num_q_heads must be 8 * num_kv_heads");
  if (!(Hkv == 1 || Hkv == 2 || Hkv == 4 || (Hkv % 8 == 0 && Hkv <= 64)))
    return fail(HPC_ERR_UNSUPPORTED, "num_kv_heads must be 1, 2, 4, 8, 16, 32 or 64");
  if (T < 1 || T > kMaxQueryTokens)
    return fail(HPC_ERR_UNSUPPORTED, "q_len must be between 1 and 8");
  for (int i = 0; i < qnd; ++i)
    if (out->shape[i] != q->shape[i])
      return fail(HPC_ERR_INVALID_ARG, "out must have q's shape");
  if (has_lse) {
    if (lse->dtype != HPC_F32) return fail(HPC_ERR_INVALID_ARG, "lse must be f32");
    for (int i = 0; i < qnd - 1; ++i)
      if (lse->shape[i] != q->shape[i])
        return fail(HPC_ERR_INVALID_ARG, "lse must be [B][H_q] or [B][q_len][H_q]");
  }
  if (block_table->dtype != HPC_I32 || block_table->shape[0] != B || block_table->stride[1] != 1)
    return fail(HPC_ERR_INVALID_ARG, "block_table must be int32 [B][max_blocks], row-contiguous");
  if (seq_lens->dtype != HPC_I32 || seq_lens->shape[0] != B || (B > 1 && seq_lens->stride[0] != 1))
    return fail(HPC_ERR_INVALID_ARG, "seq_lens must be contiguous int32 [B]");
  if (q->stride[qnd - 1] != 1 || out->stride[qnd - 1] != 1 || k_cache->stride[3] != 1)
    return fail(HPC_ERR_INVALID_ARG, "innermost stride of q, out and the caches must be 1");
  if (q->stride[0] % 8 || q_st % 8 || q_sh % 8 || out->stride[0] % 8 || o_st % 8 || o_sh % 8 ||
      !aligned(q->data, 16) || !aligned(out->data, 16))
    return fail(HPC_ERR_INVALID_ARG, "q/out must be 16-byte aligned with strides of 8 elements");
  const int64_t e = fp8 ? 1 : 2;
  for (int i = 0; i < 3; ++i)
    if ((k_cache->stride[i] * e) % 16)
      return fail(HPC_ERR_INVALID_ARG, "cache strides must be multiples of 16 bytes");
  if (!aligned(k_cache->data, 16) || !aligned(v_cache->data, 16))
    return fail(HPC_ERR_INVALID_ARG, "cache base addresses must be 16-byte aligned");
  // slot/head strides: either [.., H_kv, 64, 128] or [.., 64, H_kv, 128], non-overlapping
  const int64_t s_head = k_cache->stride[1], s_slot = k_cache->stride[2],
                s_blk = k_cache->stride[0];
  bool swap;
  if (s_slot >= kHeadDim && s_head >= kBlockTokens * s_slot && s_blk >= Hkv * s_head)
    swap = false;
  else if (s_head >= kHeadDim && s_slot >= Hkv * s_head && s_blk >= kBlockTokens * s_slot)
    swap = true;
  else
    return fail(HPC_ERR_UNSUPPORTED, "cache strides must describe a [blocks][kv heads][64][128] "
                                     "or [blocks][64][kv heads][128] layout");
  if (plan->num_seqs != B)
    return fail(HPC_ERR_INVALID_ARG, "plan was built for " + std::to_string(plan->num_seqs) +
                                         " sequences, q has " + std::to_string(B));
  if (plan->kind == HPC_PLAN_STATIC && plan->static_kv_heads != Hkv)
    return fail(HPC_ERR_INVALID_ARG, "static plan was built for another number of kv heads");
  if (plan->units > 1) {
    const WarpLayout wl = warp_layout((int)Hkv, (int)T, 8);
    if (plan->units != Hkv || wl.npass != 1 || wl.tph != 1)
      return fail(HPC_ERR_UNSUPPORTED, "a plan with " + std::to_string(plan->units) +
                                           " units per tile needs num_kv_heads == units and "
                                           "num_kv_heads * q_len <= 8");
  }
  if (fp8 && (!std::isfinite(k_cache->scale) || !std::isfinite(v_cache->scale)))
    return fail(HPC_ERR_INVALID_ARG, "FP8 scales must be finite");
  if (check_only) return HPC_OK;
  if (B == 0) return HPC_OK;
  if (B > INT32_MAX || block_table->shape[1] > INT32_MAX || NB > INT32_MAX)
    return fail(HPC_ERR_INVALID_ARG, "sizes exceed int32");

  // grid
  int gx, gy = 1;
  if (fused_num_sms > 0) {
    gx = fused_num_sms;
  } else if (plan->kind == HPC_PLAN_STATIC) {
    gx = plan->host_num_segs;
    gy = (int)Hkv;
  } else {
    gx = plan->host_num_parts >= 0 ? plan->host_num_parts : plan->num_sms;
  }
  st = ensure_workspace(plan, T * Hq, plan->h_pinned == nullptr);
  if (st != HPC_OK) return st;

  const PlanLayout& L = plan->layout;
  cudaStream_t s = (cudaStream_t)stream;
  if (step_grid > 0) {
    // one-token step: planned, computed and merged by the step kernel alone
    if (!plan->d_step || Hkv > plan->step_kv_heads || step_grid > L.cap_parts ||
        B > L.cap_seqs || plan->ws_floats < step_ws_floats(step_grid))
      return fail(HPC_ERR_INVALID_ARG, "plan is too small for this step");
    if (NB == 0) return fail(HPC_ERR_INVALID_ARG, "k_cache has no blocks");
    CUtensorMap tk, tv;
    if ((st = make_kv_map(k_cache, fp8, swap, &tk)) != HPC_OK) return st;
    if ((st = make_kv_map(v_cache, fp8, swap, &tv)) != HPC_OK) return st;
    StepParams sp;
    std::memset(&sp, 0, sizeof sp);
    sp.q = (const __nv_bfloat16*)q->data;
    sp.q_sb = q->stride[0];
    sp.q_sh = q->stride[1];
    sp.out = (__nv_bfloat16*)out->data;
    sp.o_sb = out->stride[0];
    sp.o_sh = out->stride[1];
    sp.lse = has_lse ? (float*)lse->data : nullptr;
    sp.l_sb = has_lse ? lse->stride[0] : 0;
    sp.l_sh = has_lse ? lse->stride[1] : 0;
    sp.block_table = (const int32_t*)block_table->data;
    sp.bt_sb = block_table->stride[0];
    sp.max_blocks = (int32_t)block_table->shape[1];
    sp.seq_lens = (const int32_t*)seq_lens->data;
    sp.num_seqs = (int32_t)B;
    sp.num_q_heads = (int32_t)Hq;
    sp.num_kv_heads = (int32_t)Hkv;
    sp.num_blocks = (int32_t)NB;
    sp.kv_swap = swap;
    const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)kHeadDim);
    sp.score_scale_log2 = scale * 1.4426950408889634f * (fp8 ? k_cache->scale : 1.0f);
    sp.v_scale = fp8 ? v_cache->scale : 1.0f;
    sp.ws_part = plan->d_ws;
    sp.pool = plan->d_step;
    sp.rec = plan->d_step + step_rec_off();
    sp.pair_cnt = plan->d_step + step_pair_off(L.cap_parts);
    sp.words = plan->d_words;
    sp.err = plan->d_err;
    sp.timeout_ns = wait_limit_ns();
    sp.withhold_copies = withhold_copies();
    if (plan->ev_start) HPC_CUDA_TRY(cudaEventRecord(plan->ev_start, s));
    cudaError_t ce = launch_step(sp, tk, tv, fp8, step_grid, s);
    if (ce != cudaSuccess)
      return fail(HPC_ERR_CUDA, std::string("step kernel launch: ") + cudaGetErrorString(ce));
    if (plan->ev_mid) HPC_CUDA_TRY(cudaEventRecord(plan->ev_mid, s));
    if (plan->ev_end) HPC_CUDA_TRY(cudaEventRecord(plan->ev_end, s));
    return HPC_OK;
  }
  if (gx > 0) {
    if (NB == 0) return fail(HPC_ERR_INVALID_ARG, "k_cache has no blocks");
    CUtensorMap tk, tv;
    if ((st = make_kv_map(k_cache, fp8, swap, &tk)) != HPC_OK) return st;
    if ((st = make_kv_map(v_cache, fp8, swap, &tv)) != HPC_OK) return st;
    AttnParams p;
    std::memset(&p, 0, sizeof p);
    p.q = (const __nv_bfloat16*)q->data;
    p.q_sb = q->stride[0];
    p.q_st = q_st;
    p.q_sh = q_sh;
    p.out = (__nv_bfloat16*)out->data;
    p.o_sb = out->stride[0];
    p.o_st = o_st;
    p.o_sh = o_sh;
    p.lse = has_lse ? (float*)lse->data : nullptr;
    p.l_sb = has_lse ? lse->stride[0] : 0;
    p.l_st = l_st;
    p.l_sh = l_sh;
    p.q_len = (int32_t)T;
    p.block_table = (const int32_t*)block_table->data;
    p.bt_sb = block_table->stride[0];
    p.max_blocks = (int32_t)block_table->shape[1];
    p.seq_lens = (const int32_t*)seq_lens->data;
    p.plan = plan->d_words;
    p.seq_off = (int32_t)L.seq_off();
    p.seg_off = (int32_t)L.seg_off();
    p.part_off = (int32_t)L.part_off();
    p.cu_off = (int32_t)L.cu_off();
    p.num_seqs = (int32_t)B;
    p.num_q_heads = (int32_t)Hq;
    p.num_kv_heads = (int32_t)Hkv;
    p.num_blocks = (int32_t)NB;
    p.static_mode = plan->kind == HPC_PLAN_STATIC;
    p.kv_swap = swap;
    p.fused_plan = fused_num_sms > 0;
    p.plan_num_sms = fused_num_sms;
    p.plan_units = plan->kind == HPC_PLAN_STATIC ? 1 : plan->units;
    p.plan_out = plan->d_words;
    const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)kHeadDim);
    p.score_scale_log2 = scale * 1.4426950408889634f * (fp8 ? k_cache->scale : 1.0f);
    p.v_scale = fp8 ? v_cache->scale : 1.0f;
    const int64_t cs = std::max<int64_t>(L.cap_segs, 1);
    p.ws_o = plan->d_ws;
    p.ws_m = plan->d_ws + cs * T * Hq * kHeadDim;
    p.ws_l = p.ws_m + cs * T * Hq;
    p.err = plan->d_err;
    p.timeout_ns = wait_limit_ns();
    p.withhold_copies = withhold_copies();
    // q_len >= the tensor-core threshold with a tile plan: the q_len x 8 query
    // rows of a KV head go through tcgen05 (decode_tc_kernel.cu)
    CUtensorMap tq;
    const bool tc = multi && T >= tc_min_q_len(fp8) &&
                    plan->kind == HPC_PLAN_DYNAMIC && plan->units == 1 && fused_num_sms == 0 &&
                    make_decode_q_map(q, &tq);
    if (plan->ev_start) HPC_CUDA_TRY(cudaEventRecord(plan->ev_start, s));
    cudaError_t ce;
    if (tc) {
      DecodeTcParams tp;
      std::memset(&tp, 0, sizeof tp);
      tp.block_table = p.block_table;
      tp.bt_sb = p.bt_sb;
      tp.max_blocks = p.max_blocks;
      tp.seq_lens = p.seq_lens;
      tp.plan = plan->d_words;
      tp.part_off = p.part_off;
      tp.seg_off = p.seg_off;
      tp.num_seqs = p.num_seqs;
      tp.num_q_heads = p.num_q_heads;
      tp.num_kv_heads = p.num_kv_heads;
      tp.num_blocks = p.num_blocks;
      tp.q_len = p.q_len;
      tp.kv_swap = p.kv_swap;
      tp.out = p.out;
      tp.o_sb = p.o_sb;
      tp.o_st = p.o_st;
      tp.o_sh = p.o_sh;
      tp.lse = p.lse;
      tp.l_sb = p.l_sb;
      tp.l_st = p.l_st;
      tp.l_sh = p.l_sh;
      tp.ws_o = p.ws_o;
      tp.ws_m = p.ws_m;
      tp.ws_l = p.ws_l;
      tp.score_scale_log2 = p.score_scale_log2;
      tp.v_scale = p.v_scale;
      tp.err = p.err;
      tp.timeout_ns = p.timeout_ns;
      tp.withhold_copies = p.withhold_copies;
      ce = launch_decode_tc(tp, tq, tk, tv, fp8, gx, s);
    } else {
      ce = launch_attention(p, tk, tv, fp8, gx, gy, s);
    }
    if (ce != cudaSuccess)
      return fail(HPC_ERR_CUDA, std::string("attention launch: ") + cudaGetErrorString(ce));
  }
  if (plan->ev_mid) HPC_CUDA_TRY(cudaEventRecord(plan->ev_mid, s));
  MergeParams mp;
  std::memset(&mp, 0, sizeof mp);
  mp.out = (__nv_bfloat16*)out->data;
  mp.o_sb = out->stride[0];
  mp.o_st = o_st;
  mp.o_sh = o_sh;
  mp.lse = has_lse ? (float*)lse->data : nullptr;
  mp.l_sb = has_lse ? lse->stride[0] : 0;
  mp.l_st = l_st;
  mp.l_sh = l_sh;
  mp.q_len = (int32_t)T;
  mp.plan = plan->d_words;
  mp.seq_off = (int32_t)L.seq_off();
  mp.seg_off = (int32_t)L.seg_off();
  mp.num_seqs = (int32_t)B;
  mp.num_q_heads = (int32_t)Hq;
  const int64_t cs = std::max<int64_t>(L.cap_segs, 1);
  mp.ws_o = plan->d_ws;
  mp.ws_m = plan->d_ws + cs * T * Hq * kHeadDim;
  mp.ws_l = mp.ws_m + cs * T * Hq;
  cudaError_t ce = launch_merge(mp, (int32_t)Hkv, s);
  if (ce != cudaSuccess)
    return fail(HPC_ERR_CUDA, std::string("merge launch: ") + cudaGetErrorString(ce));
  if (plan->ev_end) HPC_CUDA_TRY(cudaEventRecord(plan->ev_end, s));
  return HPC_OK;
}


}  // namespace

hpc_status check_decode_args(const hpc_tensor* q, const hpc_tensor* k_cache,
                             const hpc_tensor* v_cache, const hpc_tensor* block_table,
                             const hpc_tensor* seq_lens, hpc_plan_t plan, hpc_tensor* out,
                             hpc_tensor* lse) {
  return attn_impl(q, k_cache, v_cache, block_table, seq_lens, plan, out, lse, -1.0f, nullptr, 0,
                   true);
}

}  // namespace hpc

extern "C" {

hpc_status hpc_decode_attn_ex(const hpc_tensor* q, const hpc_tensor* k_cache,
                              const hpc_tensor* v_cache, const hpc_tensor* block_table,
                              const hpc_tensor* seq_lens, hpc_plan_t plan, hpc_tensor* out,
                              hpc_tensor* lse, float softmax_scale, void* stream) {
  return attn_impl(q, k_cache, v_cache, block_table, seq_lens, plan, out, lse, softmax_scale,
                   stream, 0, false);
}

hpc_status hpc_decode_step(const hpc_tensor* q, const hpc_tensor* k_cache,
                           const hpc_tensor* v_cache, const hpc_tensor* block_table,
                           const hpc_tensor* seq_lens, hpc_plan_t plan, int32_t num_sms,
                           hpc_tensor* out, hpc_tensor* lse, void* stream) {
  if (!plan || plan->kind != HPC_PLAN_DYNAMIC || !plan->h_pinned)
    return fail(HPC_ERR_INVALID_ARG, "plan must come from hpc_decode_plan_create");
  if (!q || !q->data || (q->ndim != 3 && q->ndim != 4))
    return fail(HPC_ERR_INVALID_ARG, "q must be [B][H_q][128] or [B][q_len][H_q][128]");
  if (!seq_lens || !seq_lens->data || seq_lens->ndim != 1 || seq_lens->dtype != HPC_I32 ||
      seq_lens->shape[0] != q->shape[0] || (q->shape[0] > 1 && seq_lens->stride[0] != 1))
    return fail(HPC_ERR_INVALID_ARG, "seq_lens must be contiguous device int32 [B]");
  const int64_t B = q->shape[0];
  if (B > plan->layout.cap_seqs)
    return fail(HPC_ERR_INVALID_ARG, "num_seqs exceeds the plan's max_seqs");
  if (num_sms <= 0 || num_sms > plan->layout.cap_parts)
    return fail(HPC_ERR_INVALID_ARG, "num_sms must be in [1, plan num_sms]");
  // q_len at or above the tensor-core threshold: a tile plan of
  // num_sms / H_kv parts, one CTA per (KV head, part), built by the planner
  // kernel.
  bool tensor_core = false;
  const int32_t parts = decode_plan_parts(q, k_cache, num_sms, &tensor_core);
  if (tensor_core) {
    cudaError_t e = launch_plan_device((const int32_t*)seq_lens->data, (int32_t)B, parts,
                                       plan->d_words, plan->layout, plan->d_err,
                                       (cudaStream_t)stream, 1);
    if (e != cudaSuccess)
      return fail(HPC_ERR_CUDA, std::string("device planner launch: ") + cudaGetErrorString(e));
    plan->num_seqs = (int32_t)B;
    plan->num_sms = parts;
    plan->host_num_parts = -1;
    plan->host_num_segs = -1;
    plan->units = 1;
    return attn_impl(q, k_cache, v_cache, block_table, seq_lens, plan, out, lse, -1.0f, stream,
                     0, false);
  }
  // One query token per sequence: the step kernel plans, computes and merges
  // the step alone (step_kernel.cu).
  if (q->ndim == 3 && B <= kStepMaxSeqs && plan->d_step) {
    plan->units = 1;
    plan->num_seqs = (int32_t)B;
    plan->num_sms = num_sms;
    plan->host_num_parts = -1;
    plan->host_num_segs = -1;
    return attn_impl(q, k_cache, v_cache, block_table, seq_lens, plan, out, lse, -1.0f, stream,
                     0, false, num_sms);
  }
  // One unit per (tile, KV head) when the kernel's warp layout takes all KV
  // heads in one pass with one warp per (head, token): an 8x finer partition.
  int32_t units = 1;
  if (k_cache && k_cache->ndim == 4) {
    const int64_t hkv = k_cache->shape[1], T = q->ndim == 4 ? q->shape[1] : 1;
    if (hkv > 1 && hkv <= 64 && T >= 1 && T <= kMaxQueryTokens) {
      const WarpLayout wl = warp_layout((int)hkv, (int)T, 8);
      if (wl.npass == 1 && wl.tph == 1) units = (int32_t)hkv;
    }
  }
  if (B > kFusedPlanMaxSeqs || B == 0) {  // separate planner kernel
    cudaError_t e = launch_plan_device((const int32_t*)seq_lens->data, (int32_t)B, num_sms,
                                       plan->d_words, plan->layout, plan->d_err,
                                       (cudaStream_t)stream, units);
    if (e != cudaSuccess)
      return fail(HPC_ERR_CUDA, std::string("device planner launch: ") + cudaGetErrorString(e));
    plan->num_seqs = (int32_t)B;
    plan->num_sms = num_sms;
    plan->host_num_parts = -1;
    plan->host_num_segs = -1;
    plan->units = units;
    return attn_impl(q, k_cache, v_cache, block_table, seq_lens, plan, out, lse, -1.0f, stream,
                     0, false);
  }
  plan->units = units;
  plan->num_seqs = (int32_t)B;
  plan->num_sms = num_sms;
  plan->host_num_parts = -1;
  plan->host_num_segs = -1;
  return attn_impl(q, k_cache, v_cache, block_table, seq_lens, plan, out, lse, -1.0f, stream,
                   num_sms, false);
}

// A host tensor of the step's batch: present, 1 to 4 dims, dense (outermost
// first), so one copy moves it; its size in bytes.
static bool host_dense(const hpc_tensor* t, size_t* bytes) {
  if (!t || !t->data || t->ndim < 1 || t->ndim > 4) return false;
  const size_t eb = t->dtype == HPC_BF16 ? 2 : t->dtype == HPC_FP8_E4M3 ? 1 : 4;
  int64_t n = 1;
  for (int i = t->ndim - 1; i >= 0; --i) {
    if (t->shape[i] < 0) return false;
    if (t->shape[i] > 1 && t->stride[i] != n) return false;
    n *= t->shape[i];
  }
  *bytes = (size_t)n * eb;
  return true;
}

hpc_status hpc_decode_step_host(const hpc_tensor* q, const hpc_tensor* k_cache,
                                const hpc_tensor* v_cache, const hpc_tensor* block_table,
                                const hpc_tensor* seq_lens, hpc_plan_t plan, int32_t num_sms,
                                hpc_tensor* out, hpc_tensor* lse, void* stream) {
  if (!plan) return fail(HPC_ERR_INVALID_ARG, "plan is null");
  const hpc_tensor* host[5] = {q, block_table, seq_lens, out, lse};
  const char* names[5] = {"q", "block_table", "seq_lens", "out", "lse"};
  size_t bytes[5] = {0, 0, 0, 0, 0}, off[6] = {0, 0, 0, 0, 0, 0};
  for (int i = 0; i < 5; ++i) {
    if (i == 4 && !lse) {
      off[i + 1] = off[i];
      continue;
    }
    if (!host_dense(host[i], &bytes[i]))
      return fail(HPC_ERR_INVALID_ARG,
                  std::string(names[i]) + " must be a dense host tensor of 1 to 4 dims");
    off[i + 1] = off[i] + (bytes[i] + 255) / 256 * 256;
  }
  const size_t need = off[5] > 256 ? off[5] : 256;
  if (plan->stage_bytes < need) {
    if (plan->d_stage) {
      HPC_CUDA_TRY(cudaStreamSynchronize((cudaStream_t)stream));  // the old area's last use
      cudaFree(plan->d_stage);
      plan->d_stage = nullptr;
      plan->stage_bytes = 0;
    }
    HPC_CUDA_TRY(cudaMalloc(&plan->d_stage, need));
    plan->stage_bytes = need;
  }
  hpc_tensor dev[5];
  for (int i = 0; i < 5; ++i) {
    if (!host[i]) continue;
    dev[i] = *host[i];
    dev[i].data = static_cast<uint8_t*>(plan->d_stage) + off[i];
  }
  const cudaStream_t s = (cudaStream_t)stream;
  for (int i = 0; i < 3; ++i)  // q, block table, lengths up
    if (bytes[i]) HPC_CUDA_TRY(cudaMemcpyAsync(dev[i].data, host[i]->data, bytes[i],
                                               cudaMemcpyHostToDevice, s));
  const hpc_status st = hpc_decode_step(&dev[0], k_cache, v_cache, &dev[1], &dev[2], plan, num_sms,
                                        &dev[3], lse ? &dev[4] : nullptr, stream);
  if (st != HPC_OK) return st;
  for (int i = 3; i < 5; ++i)  // out and lse down
    if (host[i] && bytes[i])
      HPC_CUDA_TRY(cudaMemcpyAsync(host[i]->data, dev[i].data, bytes[i], cudaMemcpyDeviceToHost,
                                   s));
  return HPC_OK;
}

hpc_status hpc_decode_tc_min_q_len(int32_t q_len, int32_t* previous) {
  if (previous) *previous = g_tc_min_q_len.load(std::memory_order_relaxed);
  if (q_len < 0) return HPC_OK;
  if (q_len == 1) return fail(HPC_ERR_INVALID_ARG, "the tensor-core path needs q_len >= 2");
  g_tc_min_q_len.store(q_len, std::memory_order_relaxed);
  return HPC_OK;
}

hpc_status hpc_decode_plan_set_timing_events(hpc_plan_t plan, void* ev_start, void* ev_attn_done,
                                             void* ev_end) {
  if (!plan) return fail(HPC_ERR_INVALID_ARG, "plan is null");
  plan->ev_start = (cudaEvent_t)ev_start;
  plan->ev_mid = (cudaEvent_t)ev_attn_done;
  plan->ev_end = (cudaEvent_t)ev_end;
  return HPC_OK;
}

hpc_status hpc_rope_norm_kv_write(const hpc_tensor* q_in, const hpc_tensor* k_in,
                                  const hpc_tensor* v_in, const hpc_tensor* seq_lens,
                                  const hpc_tensor* block_table, const hpc_tensor* q_norm_weight,
                                  const hpc_tensor* k_norm_weight, float eps, float rope_base,
                                  hpc_tensor* q_out, hpc_tensor* q_out_fp8, hpc_tensor* k_cache,
                                  hpc_tensor* v_cache, int32_t* device_error, void* stream) {
  hpc_status st;
  if ((st = check_tensor(q_in, "q_in", 3)) != HPC_OK) return st;
  if ((st = check_tensor(k_in, "k_in", 3)) != HPC_OK) return st;
  if ((st = check_tensor(v_in, "v_in", 3)) != HPC_OK) return st;
  if ((st = check_tensor(seq_lens, "seq_lens", 1)) != HPC_OK) return st;
  if ((st = check_tensor(block_table, "block_table", 2)) != HPC_OK) return st;
  if ((st = check_tensor(q_norm_weight, "q_norm_weight", 1)) != HPC_OK) return st;
  if ((st = check_tensor(k_norm_weight, "k_norm_weight", 1)) != HPC_OK) return st;
  if ((st = check_tensor(q_out, "q_out", 3)) != HPC_OK) return st;
  if ((st = check_tensor(q_out_fp8, "q_out_fp8", 3, true)) != HPC_OK) return st;
  if ((st = check_tensor(k_cache, "k_cache", 4)) != HPC_OK) return st;
  if ((st = check_tensor(v_cache, "v_cache", 4)) != HPC_OK) return st;
  const bool has_qf = q_out_fp8 && q_out_fp8->data;
  const int64_t B = q_in->shape[0], Hq = q_in->shape[1], Hkv = k_in->shape[1];
  if (q_in->dtype != HPC_BF16 || k_in->dtype != HPC_BF16 || v_in->dtype != HPC_BF16 ||
      q_out->dtype != HPC_BF16)
    return fail(HPC_ERR_INVALID_ARG, "q_in, k_in, v_in and q_out must be bf16");
  if (q_in->shape[2] != kHeadDim || k_in->shape[2] != kHeadDim || v_in->shape[2] != kHeadDim ||
      k_cache->shape[3] != kHeadDim)
    return fail(HPC_ERR_UNSUPPORTED, "head_dim must be 128");
  if (k_cache->shape[2] != kBlockTokens)
    return fail(HPC_ERR_UNSUPPORTED, "KV blocks must hold 64 tokens");
  if (k_in->shape[0] != B || v_in->shape[0] != B || v_in->shape[1] != Hkv ||
      q_out->shape[0] != B || q_out->shape[1] != Hq || q_out->shape[2] != kHeadDim ||
      k_cache->shape[1] != Hkv || Hkv <= 0 || Hq % Hkv != 0)
    return fail(HPC_ERR_INVALID_ARG, "inconsistent q/k/v/out/cache shapes");
  if (has_qf && (q_out_fp8->dtype != HPC_FP8_E4M3 || q_out_fp8->shape[0] != B ||
                 q_out_fp8->shape[1] != Hq || q_out_fp8->shape[2] != kHeadDim ||
                 q_out_fp8->stride[2] != 1 || q_out_fp8->stride[0] % 4 ||
                 q_out_fp8->stride[1] % 4 || !aligned(q_out_fp8->data, 4) ||
                 !(q_out_fp8->scale > 0.f) || !std::isfinite(q_out_fp8->scale)))
    return fail(HPC_ERR_INVALID_ARG, "q_out_fp8 must be e4m3 [B][H_q][128] with a positive scale");
  for (const hpc_tensor* t : {q_in, k_in, v_in, (const hpc_tensor*)q_out})
    if (t->stride[2] != 1 || t->stride[0] % 4 || t->stride[1] % 4 || !aligned(t->data, 8))
      return fail(HPC_ERR_INVALID_ARG, "q/k/v/out rows must be contiguous and 8-byte aligned");
  if (seq_lens->dtype != HPC_I32 || seq_lens->shape[0] != B || (B > 1 && seq_lens->stride[0] != 1))
    return fail(HPC_ERR_INVALID_ARG, "seq_lens must be contiguous int32 [B]");
  if (block_table->dtype != HPC_I32 || block_table->shape[0] != B || block_table->stride[1] != 1)
    return fail(HPC_ERR_INVALID_ARG, "block_table must be int32 [B][max_blocks]");
  for (const hpc_tensor* w : {q_norm_weight, k_norm_weight})
    if ((w->dtype != HPC_BF16 && w->dtype != HPC_F32) || w->shape[0] != kHeadDim ||
        w->stride[0] != 1 || !aligned(w->data, 16))
      return fail(HPC_ERR_INVALID_ARG, "norm weights must be contiguous bf16/f32 [128], 16-B aligned");
  if (k_cache->dtype != v_cache->dtype ||
      (k_cache->dtype != HPC_BF16 && k_cache->dtype != HPC_FP8_E4M3))
    return fail(HPC_ERR_INVALID_ARG, "k_cache/v_cache must both be bf16 or both fp8_e4m3");
  const bool fp8 = k_cache->dtype == HPC_FP8_E4M3;
  for (int i = 0; i < 4; ++i)
    if (k_cache->shape[i] != v_cache->shape[i] || k_cache->stride[i] != v_cache->stride[i])
      return fail(HPC_ERR_INVALID_ARG, "k_cache and v_cache must have the same shape and strides");
  if (k_cache->stride[3] != 1 || k_cache->stride[0] % 4 || k_cache->stride[1] % 4 ||
      k_cache->stride[2] % 4 || !aligned(k_cache->data, 8) || !aligned(v_cache->data, 8))
    return fail(HPC_ERR_INVALID_ARG, "cache rows must be contiguous and 8-byte aligned");
  if (fp8 && (!(k_cache->scale > 0.f) || !(v_cache->scale > 0.f) ||
              !std::isfinite(k_cache->scale) || !std::isfinite(v_cache->scale)))
    return fail(HPC_ERR_INVALID_ARG, "FP8 caches need positive finite scales");
  if (!(eps >= 0.f) || !(rope_base > 1.f) || !std::isfinite(rope_base))
    return fail(HPC_ERR_INVALID_ARG, "eps must be >= 0 and rope_base > 1");
  if (B == 0) return HPC_OK;
  PrologueParams p;
  std::memset(&p, 0, sizeof p);
  p.q_in = (const __nv_bfloat16*)q_in->data; p.qi_sb = q_in->stride[0]; p.qi_sh = q_in->stride[1];
  p.k_in = (const __nv_bfloat16*)k_in->data; p.ki_sb = k_in->stride[0]; p.ki_sh = k_in->stride[1];
  p.v_in = (const __nv_bfloat16*)v_in->data; p.vi_sb = v_in->stride[0]; p.vi_sh = v_in->stride[1];
  p.seq_lens = (const int32_t*)seq_lens->data;
  p.block_table = (const int32_t*)block_table->data;
  p.bt_sb = block_table->stride[0];
  p.max_blocks = (int32_t)block_table->shape[1];
  p.wq = q_norm_weight->data; p.wq_dtype = q_norm_weight->dtype;
  p.wk = k_norm_weight->data; p.wk_dtype = k_norm_weight->dtype;
  p.eps = eps;
  for (int i = 0; i < kHeadDim / 2; ++i) {
    const double f = std::pow((double)rope_base, -2.0 * i / kHeadDim);
    p.inv_freq_hi[i] = (float)f;
    p.inv_freq_lo[i] = (float)(f - (double)p.inv_freq_hi[i]);
  }
  const double two_pi = 2.0 * 3.14159265358979323846;
  p.two_pi_hi = (float)two_pi;
  p.two_pi_lo = (float)(two_pi - (double)p.two_pi_hi);
  p.q_out = (__nv_bfloat16*)q_out->data; p.qo_sb = q_out->stride[0]; p.qo_sh = q_out->stride[1];
  if (has_qf) {
    p.q_fp8 = (uint8_t*)q_out_fp8->data;
    p.qf_sb = q_out_fp8->stride[0];
    p.qf_sh = q_out_fp8->stride[1];
    p.q_fp8_scale = q_out_fp8->scale;
  }
  p.k_cache = k_cache->data;
  p.v_cache = v_cache->data;
  p.c_sblk = k_cache->stride[0]; p.c_shead = k_cache->stride[1]; p.c_sslot = k_cache->stride[2];
  p.cache_fp8 = fp8;
  p.k_scale = fp8 ? k_cache->scale : 1.f;
  p.v_scale = fp8 ? v_cache->scale : 1.f;
  p.num_blocks = (int32_t)std::min<int64_t>(k_cache->shape[0], INT32_MAX);
  p.num_seqs = (int32_t)B;
  p.num_q_heads = (int32_t)Hq;
  p.num_kv_heads = (int32_t)Hkv;
  p.err = device_error;
  cudaError_t e = launch_prologue(p, (cudaStream_t)stream);
  if (e != cudaSuccess)
    return fail(HPC_ERR_CUDA, std::string("prologue launch: ") + cudaGetErrorString(e));
  return HPC_OK;
}

hpc_status hpc_decode_attn(const hpc_tensor* q, const hpc_tensor* k_cache,
                           const hpc_tensor* v_cache, const hpc_tensor* block_table,
                           const hpc_tensor* seq_lens, hpc_plan_t plan, hpc_tensor* out,
                           hpc_tensor* lse, void* stream) {
  return hpc_decode_attn_ex(q, k_cache, v_cache, block_table, seq_lens, plan, out, lse, -1.0f,
                            stream);
}

}  // extern "C"

// ------------------------------------------------------------------------
// Prefill / extend attention (prefill_kernel.cu).
namespace hpc {
namespace {

// 3-D TMA descriptor over q or out [total_q][H_q][128] bf16: box = 16 tokens
// x 8 heads x 64 columns, 128-byte swizzle (one 16 KB half of a 128-row tile).
hpc_status make_q_map(const hpc_tensor* q, CUtensorMap* map, const char* what = "q") {
  auto enc = encode_fn();
  if (!enc) return fail(HPC_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)q->shape[1], (cuuint64_t)q->shape[0]};
  cuuint64_t strides[2] = {(cuuint64_t)q->stride[1] * 2, (cuuint64_t)q->stride[0] * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)kGroup, (cuuint32_t)kExtendTileTokens};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q->data, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(HPC_ERR_INVALID_ARG, std::string("cuTensorMapEncodeTiled rejected ") + what +
                                         " (error " + std::to_string((int)r) + ")");
  return HPC_OK;
}

}  // namespace
}  // namespace hpc

extern "C" hpc_status hpc_extend_attn_ex(const hpc_tensor* q, const hpc_tensor* k_cache,
                                         const hpc_tensor* v_cache, const hpc_tensor* block_table,
                                         const hpc_tensor* seq_lens, const hpc_tensor* cu_q_lens,
                                         hpc_tensor* out, hpc_tensor* lse, float softmax_scale,
                                         int32_t tiles_per_cta, int32_t* device_error,
                                         void* stream) {
  using namespace hpc;
  if (tiles_per_cta < 0 || tiles_per_cta > 2)
    return fail(HPC_ERR_INVALID_ARG, "tiles_per_cta must be 0 (automatic), 1 or 2");
  hpc_status st;
  if ((st = check_tensor(q, "q", 3)) != HPC_OK) return st;
  if ((st = check_tensor(k_cache, "k_cache", 4)) != HPC_OK) return st;
  if ((st = check_tensor(v_cache, "v_cache", 4)) != HPC_OK) return st;
  if ((st = check_tensor(block_table, "block_table", 2)) != HPC_OK) return st;
  if ((st = check_tensor(seq_lens, "seq_lens", 1)) != HPC_OK) return st;
  if ((st = check_tensor(cu_q_lens, "cu_q_lens", 1)) != HPC_OK) return st;
  if ((st = check_tensor(out, "out", 3)) != HPC_OK) return st;
  if ((st = check_tensor(lse, "lse", 2, true)) != HPC_OK) return st;
  const bool has_lse = lse && lse->data;
  const int64_t total_q = q->shape[0], Hq = q->shape[1], D = q->shape[2];
  const int64_t B = seq_lens->shape[0];
  const int64_t NB = k_cache->shape[0], Hkv = k_cache->shape[1];
  if (q->dtype != HPC_BF16 || out->dtype != HPC_BF16)
    return fail(HPC_ERR_INVALID_ARG, "q and out must be bf16");
  if (k_cache->dtype != v_cache->dtype ||
      (k_cache->dtype != HPC_BF16 && k_cache->dtype != HPC_FP8_E4M3))
    return fail(HPC_ERR_INVALID_ARG, "k_cache/v_cache must both be bf16 or both fp8_e4m3");
  const bool fp8 = k_cache->dtype == HPC_FP8_E4M3;
  if (fp8 && (!std::isfinite(k_cache->scale) || !std::isfinite(v_cache->scale)))
    return fail(HPC_ERR_INVALID_ARG, "FP8 scales must be finite");
  for (int i = 0; i < 4; ++i)
    if (k_cache->shape[i] != v_cache->shape[i] || k_cache->stride[i] != v_cache->stride[i])
      return fail(HPC_ERR_INVALID_ARG, "k_cache and v_cache must have the same shape and strides");
  if (D != kHeadDim || k_cache->shape[3] != kHeadDim)
    return fail(HPC_ERR_UNSUPPORTED, "head_dim must be 128");
  if (k_cache->shape[2] != kBlockTokens)
    return fail(HPC_ERR_UNSUPPORTED, "KV blocks must hold 64 tokens");
  if (Hkv <= 0 || Hq != kGroup * Hkv)
    return fail(HPC_ERR_UNSUPPORTED, "num_q_heads must be 8 * num_kv_heads");
  for (int i = 0; i < 3; ++i)
    if (out->shape[i] != q->shape[i]) return fail(HPC_ERR_INVALID_ARG, "out must have q's shape");
  if (has_lse && (lse->dtype != HPC_F32 || lse->shape[0] != total_q || lse->shape[1] != Hq))
    return fail(HPC_ERR_INVALID_ARG, "lse must be f32 [total_q][H_q]");
  if (block_table->dtype != HPC_I32 || block_table->shape[0] != B || block_table->stride[1] != 1)
    return fail(HPC_ERR_INVALID_ARG, "block_table must be int32 [B][max_blocks], row-contiguous");
  if (seq_lens->dtype != HPC_I32 || (B > 1 && seq_lens->stride[0] != 1))
    return fail(HPC_ERR_INVALID_ARG, "seq_lens must be contiguous int32 [B]");
  if (cu_q_lens->dtype != HPC_I32 || cu_q_lens->shape[0] != B + 1 || cu_q_lens->stride[0] != 1)
    return fail(HPC_ERR_INVALID_ARG, "cu_q_lens must be contiguous int32 [B+1]");
  if (q->stride[2] != 1 || out->stride[2] != 1 || k_cache->stride[3] != 1)
    return fail(HPC_ERR_INVALID_ARG, "innermost stride of q, out and the caches must be 1");
  if (q->stride[0] % 8 || q->stride[1] % 8 || out->stride[0] % 8 || out->stride[1] % 8 ||
      !aligned(q->data, 16) || !aligned(out->data, 16))
    return fail(HPC_ERR_INVALID_ARG, "q/out must be 16-byte aligned with strides of 8 elements");
  const int64_t ce = fp8 ? 1 : 2;
  for (int i = 0; i < 3; ++i)
    if ((k_cache->stride[i] * ce) % 16)
      return fail(HPC_ERR_INVALID_ARG, "cache strides must be multiples of 16 bytes");
  if (!aligned(k_cache->data, 16) || !aligned(v_cache->data, 16))
    return fail(HPC_ERR_INVALID_ARG, "cache base addresses must be 16-byte aligned");
  const int64_t s_head = k_cache->stride[1], s_slot = k_cache->stride[2],
                s_blk = k_cache->stride[0];
  bool swap;
  if (s_slot >= kHeadDim && s_head >= kBlockTokens * s_slot && s_blk >= Hkv * s_head)
    swap = false;
  else if (s_head >= kHeadDim && s_slot >= Hkv * s_head && s_blk >= kBlockTokens * s_slot)
    swap = true;
  else
    return fail(HPC_ERR_UNSUPPORTED, "cache strides must describe a [blocks][kv heads][64][128] "
                                     "or [blocks][64][kv heads][128] layout");
  if (B == 0 || total_q == 0) return HPC_OK;
  if (NB == 0) return fail(HPC_ERR_INVALID_ARG, "k_cache has no blocks");
  if (B > INT32_MAX || total_q > INT32_MAX || NB > INT32_MAX || block_table->shape[1] > INT32_MAX)
    return fail(HPC_ERR_INVALID_ARG, "sizes exceed int32");
  if (tiles_per_cta == 0) {
    // two 128-row query tiles per CTA (measured as fast or faster from q512
    // prefill up) unless that leaves more than half of the SMs idle
    int dev = 0, sms = 0;
    HPC_CUDA_TRY(cudaGetDevice(&dev));
    HPC_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const int64_t pairs = (total_q + 2 * kExtendTileTokens - 1) / (2 * kExtendTileTokens);
    tiles_per_cta = 2 * pairs * Hkv >= sms ? 2 : 1;
  }
  // CTA tiles of T = 16 * tiles_per_cta tokens: sum_b ceil(n_b / T) <= total_q / T + B
  const int64_t tt = (int64_t)kExtendTileTokens * tiles_per_cta;
  const int64_t tiles = (total_q + tt - 1) / tt + B;
  if (tiles > 65535)
    return fail(HPC_ERR_UNSUPPORTED, "too many query tiles in one call (split the batch)");
  CUtensorMap tq, tk, tv, to;
  if ((st = make_q_map(q, &tq)) != HPC_OK) return st;
  if ((st = make_q_map(out, &to, "out")) != HPC_OK) return st;  // full tiles leave by TMA
  if ((st = make_kv_map(k_cache, fp8, swap, &tk)) != HPC_OK) return st;
  if ((st = make_kv_map(v_cache, fp8, swap, &tv)) != HPC_OK) return st;
  ExtendParams p;
  std::memset(&p, 0, sizeof p);
  p.block_table = (const int32_t*)block_table->data;
  p.bt_sb = block_table->stride[0];
  p.max_blocks = (int32_t)block_table->shape[1];
  p.seq_lens = (const int32_t*)seq_lens->data;
  p.cu_q_lens = (const int32_t*)cu_q_lens->data;
  p.num_seqs = (int32_t)B;
  p.num_q_heads = (int32_t)Hq;
  p.num_kv_heads = (int32_t)Hkv;
  p.num_blocks = (int32_t)NB;
  p.kv_swap = swap;
  p.out = (__nv_bfloat16*)out->data;
  p.o_st = out->stride[0];
  p.o_sh = out->stride[1];
  p.lse = has_lse ? (float*)lse->data : nullptr;
  p.l_st = has_lse ? lse->stride[0] : 0;
  p.l_sh = has_lse ? lse->stride[1] : 0;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt((float)kHeadDim);
  p.kv_fp8 = fp8;
  p.score_scale_log2 = scale * 1.4426950408889634f * (fp8 ? k_cache->scale : 1.0f);
  p.v_scale = fp8 ? v_cache->scale : 1.0f;
  p.err = device_error;
  p.timeout_ns = wait_limit_ns();
  p.withhold_copies = withhold_copies();
  cudaError_t e =
      launch_extend(p, tq, tk, tv, to, (int)tiles, tiles_per_cta, (cudaStream_t)stream);
  if (e != cudaSuccess)
    return fail(HPC_ERR_CUDA, std::string("extend launch: ") + cudaGetErrorString(e));
  return HPC_OK;
}

extern "C" hpc_status hpc_extend_attn(const hpc_tensor* q, const hpc_tensor* k_cache,
                                      const hpc_tensor* v_cache, const hpc_tensor* block_table,
                                      const hpc_tensor* seq_lens, const hpc_tensor* cu_q_lens,
                                      hpc_tensor* out, hpc_tensor* lse, float softmax_scale,
                                      int32_t* device_error, void* stream) {
  return hpc_extend_attn_ex(q, k_cache, v_cache, block_table, seq_lens, cu_q_lens, out, lse,
                            softmax_scale, 0, device_error, stream);
}
