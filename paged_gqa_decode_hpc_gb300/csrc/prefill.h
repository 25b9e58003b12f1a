// Internal declarations of the prefill / extend attention kernel
// (prefill_kernel.cu); not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace hpc {

// New tokens of one sequence per CTA tile: 16 tokens x 8 query heads of one
// KV head fill the 128 rows of one tcgen05.mma (M = 128).
constexpr int kExtendTileTokens = 16;

struct ExtendParams {
  const int32_t* block_table;
  int64_t bt_sb;
  int32_t max_blocks;
  const int32_t* seq_lens;      // [B] positions per sequence, new tokens included
  const int32_t* cu_q_lens;     // [B+1] new-token offsets into q / out
  int32_t num_seqs, num_q_heads, num_kv_heads, num_blocks;
  int32_t kv_swap;              // KV tensor map dims are (d, head, slot, block)
  __nv_bfloat16* out;           // [total_q][H_q][128]
  int64_t o_st, o_sh;           // element strides over token, head
  float* lse;                   // [total_q][H_q] or null
  int64_t l_st, l_sh;
  int32_t kv_fp8;               // cache bytes are e4m3 (else bf16)
  float score_scale_log2;       // softmax_scale * log2(e) (* k_scale for e4m3)
  float v_scale;                // e4m3 V scale (1 for bf16)
  int32_t* err;                 // device flag word (HPC_DEVCHK_*) or null
  unsigned long long timeout_ns;
  int32_t withhold_copies;      // failure-path test: the producer issues no copy
};

// grid = (H_kv, tiles): tiles >= the number of (16 * tiles_per_cta)-token
// tiles of the batch; tiles_per_cta = 1 or 2 query tiles of 128 rows per CTA.
cudaError_t launch_extend(const ExtendParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& to, int tiles,
                          int tiles_per_cta, cudaStream_t stream);

}  // namespace hpc
