// Internal declarations of libhpc_decode.so (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include <string>

#include "hpc_decode.h"

namespace hpc {

constexpr int kBlockTokens = 64;   // paged block = one tile of 64 tokens
constexpr int kHeadDim = 128;
constexpr int kGroup = 8;          // query heads per KV head
constexpr int32_t kPlanMagic = 0x48504344;

// Plan buffer words (device). Offsets of the variable arrays depend on the
// plan's capacity, not on the step, so a device-built plan can be refilled
// without moving anything:
//   [0..7]            header (see hpc_decode_plan_export)
//   part_seg_off      cap_parts + 1
//   seq_seg_off       cap_seqs + 1
//   cu_tiles          cap_seqs + 1   (device planner scratch; not exported)
//   segs              4 * cap_segs
enum HeaderWord { kMagic = 0, kKind, kNumSeqs, kNumParts, kNumTiles, kNumSegs, kNumSms,
                  kSplits, kHeaderWords };

struct PlanLayout {
  int32_t cap_seqs = 0, cap_parts = 0, cap_segs = 0;
  __host__ __device__ int64_t part_off() const { return kHeaderWords; }
  __host__ __device__ int64_t seq_off() const { return part_off() + cap_parts + 1; }
  __host__ __device__ int64_t cu_off() const { return seq_off() + cap_seqs + 1; }
  __host__ __device__ int64_t seg_off() const { return (cu_off() + cap_seqs + 1 + 3) & ~int64_t(3); }  // 16-B aligned
  __host__ __device__ int64_t words() const { return seg_off() + 4LL * cap_segs; }
};

}  // namespace hpc

struct hpc_plan_s {
  int32_t kind = HPC_PLAN_DYNAMIC;
  int32_t device = 0;
  hpc::PlanLayout layout;
  int32_t num_sms = 0;        // CTAs the plan was sized for (dynamic grid)
  int32_t max_seqs = 0;
  // Host-side knowledge of the current step (always known: the caller passes
  // num_seqs; the part/segment counts are known for host-built plans).
  int32_t num_seqs = 0;
  int32_t host_num_parts = -1;   // -1: only the device knows (device planner)
  int32_t host_num_segs = -1;
  int32_t static_kv_heads = 0;   // static plans: grid.y
  int32_t units = 1;             // units per tile of the current work list
  int32_t* d_words = nullptr;    // plan buffer
  int32_t* h_pinned = nullptr;   // staging for hpc_decode_plan_update
  cudaEvent_t copy_done = nullptr;  // last upload from h_pinned
  int32_t* d_err = nullptr;      // device error word
  float* d_ws = nullptr;         // partial workspace: o [cap_segs][H_q][128], m, l
  int64_t ws_heads = 0;          // H_q the workspace was sized for
  cudaEvent_t ev_start = nullptr, ev_mid = nullptr, ev_end = nullptr;  // optional timing
  // One-token step path (step_kernel.cu): pool counters, per-owner records and
  // per-(sequence, KV head) arrival counters, zeroed at creation and left at
  // zero by every step; sized for step_kv_heads KV heads.
  int32_t* d_step = nullptr;
  int32_t step_kv_heads = 0;
  // hpc_decode_step_host: device staging for the step's host-side buffers
  void* d_stage = nullptr;
  size_t stage_bytes = 0;
  int64_t ws_floats = 0;         // floats allocated at d_ws
};

namespace hpc {

// Kernel parameter block of the attention kernel (passed by value).
struct AttnParams {
  const __nv_bfloat16* q;
  int64_t q_sb, q_st, q_sh;     // strides (elements) of q over b, query token, head
  __nv_bfloat16* out;
  int64_t o_sb, o_st, o_sh;
  float* lse;                   // may be null
  int64_t l_sb, l_st, l_sh;
  int32_t q_len;                // query tokens per sequence (1 = plain decode)
  const int32_t* block_table;
  int64_t bt_sb;
  int32_t max_blocks;
  const int32_t* seq_lens;
  const int32_t* plan;          // plan buffer words
  int32_t seq_off, seg_off, part_off, cu_off;  // word offsets in the plan buffer
  int32_t num_seqs, num_q_heads, num_kv_heads, num_blocks;
  int32_t static_mode;          // 1: blockIdx.x = segment, blockIdx.y = kv head
  int32_t fused_plan;           // 1: each CTA plans its own part from seq_lens and
                                //    the CTAs write the plan words (plan_out)
  int32_t plan_num_sms;         // fused: parts cap (P = min(plan_num_sms, T))
  int32_t plan_units;           // units per tile of the plan (1: tiles; H_kv: (tile, head))
  int32_t* plan_out;            // fused: plan buffer written by the kernel
  int32_t kv_swap;              // tensor map dims are (d, head, slot, block)
  float score_scale_log2;       // softmax_scale * log2(e) (* k_scale for FP8)
  float v_scale;                // FP8 V scale (1 for BF16)
  float* ws_o;                  // [cap_segs][H_q][128]
  float* ws_m;                  // [cap_segs][H_q]  (log2 domain)
  float* ws_l;                  // [cap_segs][H_q]
  int32_t* err;
  unsigned long long timeout_ns;
  int32_t withhold_copies;      // failure-path test: the producer issues nothing
};

struct MergeParams {
  __nv_bfloat16* out;
  int64_t o_sb, o_st, o_sh;
  float* lse;
  int64_t l_sb, l_st, l_sh;
  int32_t q_len;
  const int32_t* plan;
  int32_t seq_off, seg_off;
  int32_t num_seqs, num_q_heads;  // num_q_heads per query token
  const float* ws_o;
  const float* ws_m;
  const float* ws_l;
};

// Parameter block of the one-token step kernel (step_kernel.cu).
struct StepParams {
  const __nv_bfloat16* q;
  int64_t q_sb, q_sh;
  __nv_bfloat16* out;
  int64_t o_sb, o_sh;
  float* lse;                   // may be null
  int64_t l_sb, l_sh;
  const int32_t* block_table;
  int64_t bt_sb;
  int32_t max_blocks;
  const int32_t* seq_lens;
  int32_t num_seqs, num_q_heads, num_kv_heads, num_blocks;
  int32_t kv_swap;
  float score_scale_log2;
  float v_scale;
  float* ws_part;               // [slots][9][32] float4: partial states of split pairs
                                //   in the consumer lanes' layout (step_kernel.cu)
  int32_t* pool;                // [2]: next pool chunk, CTAs done claiming
  int32_t* rec;                 // [owners][4]: first unit, end unit, pieces, runs
  int32_t* pair_cnt;            // [num_seqs * num_kv_heads] arrival counters
  int32_t* words;               // plan header words
  int32_t* err;
  unsigned long long timeout_ns;
  int32_t withhold_copies;
};
// Step plan constants (the oracle's step_plan uses the same values).
constexpr int32_t kStepPoolDiv = 8;      // pool = floor(T / 8) units
constexpr int32_t kStepMinChunk = 8;     // smallest pool chunk, units
constexpr int32_t kStepChunksPerCta = 4; // at most this many chunks per CTA
constexpr int32_t kStepMaxSeqs = 3072;   // prefix array in shared memory
constexpr int32_t kStepMinPartDiv = 8;   // P = min(G, ceil(S / 8)) static parts
constexpr int32_t kStepPartChunks = 12;  // a pool chunk is at least 1/12 of a static part
// d_step layout (int32 words): pool[2] | records[5 * cap_parts][4] | pair counters
inline int64_t step_rec_off() { return 2; }
inline int64_t step_pair_off(int32_t cap_parts) { return 2 + 4LL * (1 + kStepChunksPerCta) * cap_parts; }
inline int64_t step_words(int32_t cap_parts, int32_t cap_seqs, int32_t kv_heads) {
  return step_pair_off(cap_parts) + (int64_t)cap_seqs * kv_heads;
}
// Partial slots of a step on G CTAs: two per owner, owners <= G + 4 G; each
// slot holds 9 x 32 float4 (8 accumulator slices and (m, l) per lane).
inline int64_t step_slots(int32_t grid) { return 2LL * (1 + kStepChunksPerCta) * grid; }
inline int64_t step_ws_floats(int32_t grid) { return step_slots(grid) * 9 * 32 * 4; }
cudaError_t launch_step(const StepParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                        bool fp8, int grid, cudaStream_t stream);

// Parameter block of the fused prologue kernel (prologue_kernel.cu).
struct PrologueParams {
  const __nv_bfloat16* q_in;
  int64_t qi_sb, qi_sh;
  const __nv_bfloat16* k_in;
  int64_t ki_sb, ki_sh;
  const __nv_bfloat16* v_in;
  int64_t vi_sb, vi_sh;
  const int32_t* seq_lens;
  const int32_t* block_table;
  int64_t bt_sb;
  int32_t max_blocks;
  const void* wq;
  const void* wk;
  int32_t wq_dtype, wk_dtype;  // HPC_BF16 or HPC_F32
  float eps;
  // RoPE inverse frequencies base^(-2i/128) as float-float pairs, and 2*pi
  // split the same way (both formed on the host in double precision)
  float inv_freq_hi[64], inv_freq_lo[64];
  float two_pi_hi, two_pi_lo;
  __nv_bfloat16* q_out;
  int64_t qo_sb, qo_sh;
  uint8_t* q_fp8;  // may be null
  int64_t qf_sb, qf_sh;
  float q_fp8_scale;
  void* k_cache;
  void* v_cache;
  int64_t c_sblk, c_shead, c_sslot;  // element strides (same for K and V)
  int32_t cache_fp8;
  float k_scale, v_scale;
  int32_t num_blocks, num_seqs, num_q_heads, num_kv_heads;
  int32_t* err;  // may be null
};
cudaError_t launch_prologue(const PrologueParams& p, cudaStream_t stream);

// Host planners (plan_host.cu). Fill `words` (canonical layout sized by the
// returned length) or report an error message.
// units_per_tile = U > 1: every (tile, KV head) pair is one unit of the
// partition (head-granular plan); header word kSplits then holds U.
hpc_status plan_dynamic_host(const int32_t* seq_lens, int32_t num_seqs, int32_t num_sms,
                             int32_t* words, const PlanLayout& L, std::string* err,
                             int32_t units_per_tile = 1);
hpc_status plan_static_host(const int32_t* seq_lens, int32_t num_seqs, int32_t num_sms,
                            int32_t num_kv_heads, int32_t num_splits,
                            int32_t** words_out, PlanLayout* L_out, std::string* err);
int64_t dynamic_max_segs(int32_t num_seqs, int32_t num_parts);

// Launchers (kernels .cu files).
cudaError_t launch_plan_device(const int32_t* seq_lens, int32_t num_seqs, int32_t num_sms,
                               int32_t* words, const PlanLayout& L, int32_t* err,
                               cudaStream_t stream, int32_t units_per_tile = 1);
cudaError_t launch_attention(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                             bool fp8, int grid_x, int grid_y, cudaStream_t stream);
// Query tokens per sequence the attention kernel supports (one consumer warp
// per token and KV head).
constexpr int32_t kMaxQueryTokens = 8;
// Consumer-warp layout shared by the kernel and its launcher: KV heads taken
// together per pass, and tile phases (warps splitting one head's tiles).
struct WarpLayout {
  int hpass, npass, tph;
};
__host__ __device__ inline WarpLayout warp_layout(int h_count, int q_len, int nc) {
  int hpass = nc / q_len;
  if (hpass < 1) hpass = 1;
  if (hpass > h_count) hpass = h_count;
  while (h_count % hpass) --hpass;
  WarpLayout wl;
  wl.hpass = hpass;
  wl.npass = h_count / hpass;
  wl.tph = (nc / hpass) / q_len;
  return wl;
}
// Largest batch the attention kernel can plan by itself (prefix arrays in
// shared memory next to the K/V ring).
constexpr int32_t kFusedPlanMaxSeqs = 3072;
cudaError_t launch_merge(const MergeParams& p, int32_t num_kv_heads, cudaStream_t stream);

void set_error(const std::string& msg);

// Every argument check hpc_decode_attn makes, with no launch and no
// allocation (capi.cu).
hpc_status check_decode_args(const hpc_tensor* q, const hpc_tensor* k_cache,
                             const hpc_tensor* v_cache, const hpc_tensor* block_table,
                             const hpc_tensor* seq_lens, hpc_plan_t plan, hpc_tensor* out,
                             hpc_tensor* lse);

// Runs `set` (a cudaFuncSetAttribute call) once per device for one kernel:
// kernel attributes belong to each device's copy of the function, so a
// process that launches on several devices configures each of them. `done`
// holds one bit per device id (ids >= 64 are configured on every call).
template <typename F>
cudaError_t once_per_device(std::atomic<uint64_t>& done, F set) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = set();
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

}  // namespace hpc
