// hpc_decode_attn_noalloc: one decode step with no allocation anywhere. The
// work list, the partial softmax states and the error word live in a
// file-scope device array; host code obtains that array's device address per
// device with cudaGetSymbolAddress and hands it to the ordinary planner and
// attention launches.
#include <mutex>
#include <string>
#include <utility>

#include "hpc_internal.h"

namespace hpc {
namespace {

constexpr int32_t kNaMaxSeqs = HPC_NOALLOC_MAX_SEQS;
constexpr int32_t kNaMaxCtas = HPC_NOALLOC_MAX_CTAS;
constexpr int32_t kNaMaxHeads = HPC_NOALLOC_MAX_Q_HEADS;

constexpr PlanLayout na_layout() {
  PlanLayout L;
  L.cap_seqs = kNaMaxSeqs;
  L.cap_parts = kNaMaxCtas;
  L.cap_segs = kNaMaxSeqs + kNaMaxCtas;
  return L;
}
constexpr size_t round256(size_t x) { return (x + 255) & ~size_t(255); }
constexpr size_t kPlanBytes = round256(
    (size_t)(((kHeaderWords + kNaMaxCtas + 1 + 2 * (kNaMaxSeqs + 1)) + 3) / 4 * 4 +
             4 * (kNaMaxSeqs + kNaMaxCtas)) * sizeof(int32_t));
constexpr size_t kErrOff = kPlanBytes;
constexpr size_t kWsOff = kErrOff + 256;
constexpr size_t kWsBytes =
    (size_t)(kNaMaxSeqs + kNaMaxCtas) * kNaMaxHeads * (kHeadDim + 2) * sizeof(float);
constexpr size_t kScratchBytes = kWsOff + kWsBytes;

// The scratch of every hpc_decode_attn_noalloc call on this device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};  // context the address belongs to

// Unique id of the calling thread's current CUDA context (ids are never
// reused, so a context created after a device reset has a new one). False
// when the driver offers no such call or no context is current.
bool current_context_id(unsigned long long* id) {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static const std::pair<GetCurrent, GetId> fns = [] {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault, &qa) !=
            cudaSuccess || qa != cudaDriverEntryPointSuccess)
      a = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) !=
            cudaSuccess || qb != cudaDriverEntryPointSuccess)
      b = nullptr;
    return std::make_pair(reinterpret_cast<GetCurrent>(a), reinterpret_cast<GetId>(b));
  }();
  if (!fns.first || !fns.second) return false;
  CUcontext ctx = nullptr;
  if (fns.first(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return fns.second(ctx, id) == CUDA_SUCCESS;
}

hpc_status na_fail(hpc_status st, const std::string& msg) {
  set_error(msg);
  return st;
}

}  // namespace
}  // namespace hpc

using namespace hpc;

extern "C" hpc_status hpc_decode_attn_noalloc(const hpc_tensor* q, const hpc_tensor* k_cache,
                                              const hpc_tensor* v_cache,
                                              const hpc_tensor* block_table,
                                              const hpc_tensor* seq_lens, int32_t num_sms,
                                              hpc_tensor* out, hpc_tensor* lse,
                                              int32_t* device_error, void* stream) {
  if (!q || !q->data || q->ndim != 3)
    return na_fail(HPC_ERR_INVALID_ARG,
                   "hpc_decode_attn_noalloc takes one query token per sequence: q must be "
                   "[B][H_q][128]");
  if (!seq_lens || !seq_lens->data || seq_lens->ndim != 1 || seq_lens->dtype != HPC_I32 ||
      seq_lens->shape[0] != q->shape[0])
    return na_fail(HPC_ERR_INVALID_ARG, "seq_lens must be device int32 [B]");
  const int64_t B = q->shape[0], Hq = q->shape[1];
  if (B > kNaMaxSeqs)
    return na_fail(HPC_ERR_INVALID_ARG,
                   "hpc_decode_attn_noalloc: num_seqs " + std::to_string(B) +
                       " exceeds its fixed scratch limit of " + std::to_string(kNaMaxSeqs));
  if (Hq > kNaMaxHeads)
    return na_fail(HPC_ERR_INVALID_ARG,
                   "hpc_decode_attn_noalloc: num_q_heads " + std::to_string(Hq) +
                       " exceeds its fixed scratch limit of " + std::to_string(kNaMaxHeads));
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return na_fail(HPC_ERR_CUDA, "hpc_decode_attn_noalloc: no usable current device");
  if (num_sms <= 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return na_fail(HPC_ERR_CUDA, "hpc_decode_attn_noalloc: cannot read the SM count");
    num_sms = n;
  }
  if (num_sms > kNaMaxCtas)
    return na_fail(HPC_ERR_INVALID_ARG,
                   "hpc_decode_attn_noalloc: " + std::to_string(num_sms) +
                       " CTAs exceed its fixed scratch limit of " + std::to_string(kNaMaxCtas));
  // Device address of the scratch array on this device: looked up once per
  // device (again only if the device's context was replaced, e.g. after a
  // cudaDeviceReset, where the module and its array may have moved).
  unsigned char* base = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    unsigned long long ctx_id = 0;
    const bool have_id = current_context_id(&ctx_id);
    if (!g_scratch_ptr[dev] || !have_id || g_scratch_ctx[dev] != ctx_id) {
      void* ptr = nullptr;
      cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess || !ptr)
        return na_fail(HPC_ERR_CUDA, std::string("cudaGetSymbolAddress(scratch): ") +
                                         cudaGetErrorString(e));
      g_scratch_ptr[dev] = ptr;
      g_scratch_ctx[dev] = current_context_id(&ctx_id) ? ctx_id : 0;
    }
    base = static_cast<unsigned char*>(g_scratch_ptr[dev]);
  }
  // A plan object that only points into the scratch array.
  hpc_plan_s plan;
  plan.kind = HPC_PLAN_DYNAMIC;
  plan.device = dev;
  plan.layout = na_layout();
  plan.num_sms = num_sms;
  plan.max_seqs = kNaMaxSeqs;
  plan.num_seqs = (int32_t)B;
  plan.host_num_parts = -1;
  plan.host_num_segs = -1;
  plan.d_words = reinterpret_cast<int32_t*>(base);
  plan.d_err = reinterpret_cast<int32_t*>(base + kErrOff);
  plan.d_ws = reinterpret_cast<float*>(base + kWsOff);
  plan.ws_heads = kNaMaxHeads;
  if ((size_t)plan.layout.words() * sizeof(int32_t) > kPlanBytes)
    return na_fail(HPC_ERR_UNSUPPORTED, "hpc_decode_attn_noalloc: internal scratch layout error");
  // Every argument check of the attention call first: a rejected call
  // enqueues nothing and leaves the scratch array and the error word as they were.
  hpc_status st = check_decode_args(q, k_cache, v_cache, block_table, seq_lens, &plan, out, lse);
  if (st != HPC_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  int32_t* err = device_error;
  if (!err) {
    err = plan.d_err;
    if (cudaMemsetAsync(err, 0, sizeof(int32_t), s) != cudaSuccess)
      return na_fail(HPC_ERR_CUDA, "hpc_decode_attn_noalloc: clearing the error word failed");
  }
  plan.d_err = err;
  if (B > 0) {
    cudaError_t e = launch_plan_device((const int32_t*)seq_lens->data, (int32_t)B, num_sms,
                                       plan.d_words, plan.layout, err, s);
    if (e != cudaSuccess)
      return na_fail(HPC_ERR_CUDA, std::string("device planner launch: ") + cudaGetErrorString(e));
  }
  return hpc_decode_attn_ex(q, k_cache, v_cache, block_table, seq_lens, &plan, out, lse, -1.0f,
                            stream);
}
