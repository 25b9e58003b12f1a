// Internal declarations of the tensor-core multi-token decode kernel
// (decode_tc_kernel.cu); not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace hpc {

// q_len new tokens per sequence: a query tile holds rows 8t + g (token t,
// query head g of the KV head), q_len * 8 <= 64 of the MMA's 128 rows.
struct DecodeTcParams {
  const int32_t* block_table;
  int64_t bt_sb;
  int32_t max_blocks;
  const int32_t* seq_lens;      // [B] positions per sequence, the q_len new tokens included
  const int32_t* plan;          // dynamic tile plan (one unit per tile)
  int32_t part_off, seg_off;    // word offsets of its part and segment arrays
  int32_t num_seqs, num_q_heads, num_kv_heads, num_blocks, q_len;
  int32_t kv_swap;              // KV tensor map dims are (d, head, slot, block)
  __nv_bfloat16* out;           // [B][q_len][H_q][128] (element strides below)
  int64_t o_sb, o_st, o_sh;
  float* lse;                   // [B][q_len][H_q] or null
  int64_t l_sb, l_st, l_sh;
  float* ws_o;                  // partial rows [segment][q_len][H_q][128]
  float* ws_m;                  // [segment][q_len][H_q]
  float* ws_l;
  float score_scale_log2;       // softmax_scale * log2(e) (* k_scale for e4m3)
  float v_scale;                // e4m3 V scale (1 for bf16)
  int32_t* err;                 // device flag word (HPC_DEVCHK_*)
  unsigned long long timeout_ns;
  int32_t withhold_copies;      // failure-path test: the producer issues no copy
};

// grid = (H_kv, num_parts): CTA (h, y) runs the segments of part y for KV
// head h. tq is a 4-D map over q [B][q_len][H_q][128] with box
// (64, 8, q_len, 1) and 128-byte swizzle.
cudaError_t launch_decode_tc(const DecodeTcParams& p, const CUtensorMap& tq,
                             const CUtensorMap& tk, const CUtensorMap& tv, bool fp8,
                             int num_parts, cudaStream_t stream);

}  // namespace hpc
