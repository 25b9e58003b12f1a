/*
 * hpc_decode.h -- C ABI of libhpc_decode.so: mixed-length paged GQA decode
 * attention for NVIDIA GB300 (sm_103a), one GPU per process.
 *
 * The operation ("vLLM x HPC-Ops: High-Performance Attention and MoE
 * Backends", section "Attention Backend: Dynamic Load-Balanced Scheduling"):
 * each decode step, every sequence's KV cache is cut into uniform 64-token
 * tiles, the tiles are spread by actual work over the CTAs of a persistent
 * grid, each CTA runs split-KV attention of one query token per sequence over
 * its tiles, and a merge pass combines the partial softmax states. The KV
 * cache is paged in 64-token blocks and may be fp8_e4m3 (section "Using
 * HPC-Ops Backends in vLLM": --block-size 64, --kv-cache-dtype fp8_e4m3).
 * The model shape is GQA with 8 query heads per KV head and head_dim 128
 * (24-ai.news page, Hy3 paragraph: 64 query heads, 8 KV heads, head dim 128).
 *
 * For sequence b, query head j (kv head h = j / 8), N = seq_lens[b]:
 *   s_t = softmax_scale * q[b][j] . k_t,     t < N
 *   out[b][j] = sum_t exp(s_t - m) v_t / sum_t exp(s_t - m),  m = max_t s_t
 *   lse[b][j] = m + ln(sum_t exp(s_t - m))                    (natural log)
 * Token t of sequence b is slot t % 64 of physical block block_table[b][t/64].
 * A sequence of length 0 yields out = 0 and lse = -inf.
 *
 * Conventions for every call:
 *   - Return value: an hpc_status. Nothing throws across the ABI. On failure
 *     hpc_last_error() returns a message for the calling thread.
 *   - Device pointers are CUDA device (or managed) memory of the current
 *     device; "host" pointers are ordinary CPU memory.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls
 *     that take a stream only enqueue work and never synchronise it, unless
 *     stated otherwise.
 *   - The caller owns every tensor. A plan owns its device work list, its
 *     partial-result workspace and its device error word; destroy frees them.
 *   - There is no CPU fallback: without a usable CUDA device the calls
 *     return HPC_ERR_CUDA.
 */
#ifndef HPC_DECODE_H
#define HPC_DECODE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  HPC_OK = 0,
  HPC_ERR_INVALID_ARG = 1,   /* null pointer, bad shape/stride/dtype, bad length */
  HPC_ERR_UNSUPPORTED = 2,   /* valid request this build does not implement */
  HPC_ERR_CUDA = 3,          /* a CUDA runtime/driver call or a launch failed */
  HPC_ERR_OOM = 4,           /* device or host allocation failed */
  HPC_ERR_DEVICE_CHECK = 5   /* a kernel's own bounds/consistency check fired */
} hpc_status;

typedef enum {
  HPC_BF16 = 0,
  HPC_FP8_E4M3 = 1,
  HPC_F32 = 2,
  HPC_I32 = 3
} hpc_dtype;

/*
 * Strided tensor descriptor. `shape`/`stride` hold `ndim` entries (outermost
 * first); strides are in elements. `scale` is the per-tensor dequantisation
 * scale of an FP8 K or V cache (value = e4m3(byte) * scale); it is ignored for
 * every other tensor.
 */
typedef struct {
  void* data;
  int32_t dtype; /* hpc_dtype */
  int32_t ndim;
  int64_t shape[4];
  int64_t stride[4];
  float scale;
} hpc_tensor;

/* Opaque plan handle: the tile -> CTA work list of one decode step. */
typedef struct hpc_plan_s* hpc_plan_t;

/* Plan kinds reported in word 1 of an exported plan. */
#define HPC_PLAN_DYNAMIC 0
#define HPC_PLAN_STATIC 1
/* The work list a one-token hpc_decode_step ran (see hpc_decode_step). */
#define HPC_PLAN_STEP 2

/* Segment flag: the segment covers every tile of its sequence. */
#define HPC_SEG_WHOLE 1

/*
 * hpc_decode_plan -- the per-step load-balanced tile scheduler (section
 * "Attention Backend: Dynamic Load-Balanced Scheduling": uniform 64-token
 * tiles, assigned to CTAs by actual work; the 24-ai.news page: tiles spread
 * in proportion to each sequence's current length).
 *
 * Rule (every tile costs one unit; no sorting): sequence b has
 * n_b = ceil(seq_lens[b] / 64) tiles; tiles are flattened in sequence order,
 * T = sum n_b, P = min(num_sms, T) parts; part p owns flattened tiles
 * [floor(p*T/P), floor((p+1)*T/P)). A segment is the part's intersection with
 * one sequence, listed by part then sequence; its partial-result slot is its
 * index in that list. One part runs on one CTA of the persistent grid.
 *
 *   seq_lens  host int32 [num_seqs], each >= 0 (else HPC_ERR_INVALID_ARG)
 *   num_seqs  >= 0
 *   num_sms   > 0: CTAs of the persistent grid (normally the SM count)
 *   plan_out  receives a new plan; the caller destroys it
 * The work list is uploaded to the current device before returning
 * (synchronous). The plan's capacity is exactly this step's size.
 */
hpc_status hpc_decode_plan(const int32_t* seq_lens, int32_t num_seqs, int32_t num_sms,
                           hpc_plan_t* plan_out);

/*
 * hpc_decode_plan_ex -- hpc_decode_plan with a finer unit of work: with
 * units_per_tile = U > 1 every (64-token tile, KV head) pair is one unit
 * (U must then equal the cache's number of KV heads), sequence b has n_b * U
 * units (unit u = head u % U of tile u / U), and the same partition is taken
 * over the units; segments then hold unit ranges and word 7 of the exported
 * plan is U. Batches with few tiles per CTA balance U times more finely.
 * hpc_decode_attn accepts such a plan when num_kv_heads * q_len <= 8
 * (otherwise HPC_ERR_UNSUPPORTED). U = 1 is hpc_decode_plan.
 */
hpc_status hpc_decode_plan_ex(const int32_t* seq_lens, int32_t num_seqs, int32_t num_sms,
                              int32_t units_per_tile, hpc_plan_t* plan_out);

/*
 * hpc_decode_plan_create -- an empty dynamic plan able to hold any step with
 * at most `max_seqs` sequences on `num_sms` CTAs; fill it with
 * hpc_decode_plan_device (or hpc_decode_plan_update) every step. All device
 * memory, including the partial workspace for `num_q_heads` query heads of
 * head_dim 128, is allocated here, so later calls allocate nothing and may be
 * captured in a CUDA graph.
 */
hpc_status hpc_decode_plan_create(int32_t max_seqs, int32_t num_sms, int32_t num_q_heads,
                                  hpc_plan_t* plan_out);

/*
 * hpc_decode_plan_device -- the same rule as hpc_decode_plan, computed on the
 * GPU from device lengths, into a plan from hpc_decode_plan_create. No host
 * synchronisation; the result is bit-identical to the host plan of the same
 * lengths (see hpc_decode_plan_export).
 *   seq_lens_dev  device int32 [num_seqs]; a negative length makes the device
 *                 check fire (reported by hpc_decode_plan_status), and the
 *                 plan is then empty.
 *   num_seqs      <= the plan's max_seqs;   num_sms <= the plan's num_sms.
 */
hpc_status hpc_decode_plan_device(const int32_t* seq_lens_dev, int32_t num_seqs,
                                  int32_t num_sms, hpc_plan_t plan, void* stream);

/*
 * hpc_decode_plan_update -- the host planner into an existing plan (same
 * capacity rules as hpc_decode_plan_device); the upload is enqueued on
 * `stream` from a plan-owned pinned buffer, so the previous step's kernels
 * must not still read it (they are ordered on the same stream).
 */
hpc_status hpc_decode_plan_update(const int32_t* seq_lens, int32_t num_seqs, int32_t num_sms,
                                  hpc_plan_t plan, void* stream);

/*
 * hpc_decode_plan_static -- the static even split-KV schedule, the baseline
 * the pages compare against (same section: "static split-KV"; the 24-ai.news
 * page: it assumes uniform lengths). Sequence b is cut into S splits
 * [floor(i*n_b/S), floor((i+1)*n_b/S)), empty splits dropped; each split runs
 * on one CTA per KV head (grid = splits x num_kv_heads, not persistent).
 * num_splits > 0 fixes S; num_splits <= 0 uses
 * S = clamp(ceil(2*num_sms / (num_seqs*num_kv_heads)), 1, max_b n_b).
 * S is always clamped to [1, max_b n_b]. Upload is synchronous.
 */
hpc_status hpc_decode_plan_static(const int32_t* seq_lens, int32_t num_seqs, int32_t num_sms,
                                  int32_t num_kv_heads, int32_t num_splits,
                                  hpc_plan_t* plan_out);

/*
 * hpc_decode_plan_export -- copy a plan to host memory (synchronises the
 * device) in this canonical int32 layout:
 *   [0] 0x48504344  [1] kind  [2] num_seqs B  [3] num_parts P  [4] num_tiles T
 *   [5] num_segs S  [6] num_sms  [7] static split count (0 for dynamic)
 *   part_seg_off[P + 1], seq_seg_off[B + 1],
 *   segs[S][4] = {seq, tile_begin, tile_end, flags}   (tiles relative to seq)
 * For a static plan part p is segment p (part_seg_off = 0..S).
 *   buf  host int32 [cap] (may be NULL when cap == 0: only *len is written)
 *   len  receives the number of words; HPC_ERR_INVALID_ARG if cap < *len.
 */
hpc_status hpc_decode_plan_export(hpc_plan_t plan, int32_t* buf, int64_t cap, int64_t* len);

/*
 * hpc_decode_plan_compute / _compute_ex / hpc_decode_plan_static_compute --
 * the host planners alone: the same plans as hpc_decode_plan / _ex / _static,
 * written in the canonical layout of hpc_decode_plan_export into host memory.
 * No device is touched (usable on machines without a GPU).
 *   buf  host int32 [cap] (may be NULL when cap == 0: only *len is written)
 *   len  receives the number of words; HPC_ERR_INVALID_ARG if cap < *len.
 */
hpc_status hpc_decode_plan_compute(const int32_t* seq_lens, int32_t num_seqs, int32_t num_sms,
                                   int32_t* buf, int64_t cap, int64_t* len);
hpc_status hpc_decode_plan_compute_ex(const int32_t* seq_lens, int32_t num_seqs, int32_t num_sms,
                                      int32_t units_per_tile, int32_t* buf, int64_t cap,
                                      int64_t* len);
hpc_status hpc_decode_plan_static_compute(const int32_t* seq_lens, int32_t num_seqs,
                                          int32_t num_sms, int32_t num_kv_heads,
                                          int32_t num_splits, int32_t* buf, int64_t cap,
                                          int64_t* len);

/*
 * hpc_decode_plan_status -- synchronise the device and read (then clear) the
 * plan's device error word. *device_error = 0 when no kernel check fired;
 * otherwise a bit set of HPC_DEVCHK_* values. Returns HPC_ERR_DEVICE_CHECK
 * when the word was non-zero.
 */
#define HPC_DEVCHK_BAD_LENGTH 1       /* negative length, or lengths != plan */
#define HPC_DEVCHK_BAD_BLOCK 2        /* block id outside [0, num_blocks) */
#define HPC_DEVCHK_TABLE_TOO_SHORT 4  /* a sequence needs more than max_blocks */
#define HPC_DEVCHK_TIMEOUT 8          /* a bounded wait gave up */
#define HPC_DEVCHK_CAPACITY 16        /* a step larger than the plan's capacity */
hpc_status hpc_decode_plan_status(hpc_plan_t plan, int32_t* device_error);

/* hpc_decode_plan_destroy -- free a plan (NULL is a no-op). Synchronises the
 * device first so that no enqueued kernel still reads it. */
void hpc_decode_plan_destroy(hpc_plan_t plan);

/*
 * hpc_decode_attn -- run decode attention for one step with a plan built from
 * the same lengths: the persistent split-KV kernel (dynamic plan) or the
 * per-split kernel (static plan), then the log-sum-exp merge of split
 * sequences. Softmax scale 1/sqrt(head_dim).
 *
 *   q            device bf16 [B][H_q][128], or [B][q_len][H_q][128] for q_len
 *                (1..8) new tokens per sequence, innermost stride 1. The
 *                q_len tokens are the last q_len positions of the sequence:
 *                token t sees positions < seq_lens[b] - (q_len - 1 - t)
 *   k_cache      device bf16 or fp8_e4m3 [num_blocks][H_kv][64][128],
 *   v_cache      innermost stride 1, other strides multiples of 16 bytes, base
 *                16-byte aligned (a [num_blocks][64][H_kv][128] cache passes as
 *                a permuted view). Both must have the same dtype; FP8 caches
 *                carry their per-tensor scale in `scale`.
 *   block_table  device int32 [B][max_blocks], innermost stride 1; entry
 *                [b][i] for i < ceil(seq_lens[b]/64) is a physical block id
 *   seq_lens     device int32 [B]: the lengths the plan was built from
 *   plan         from any hpc_decode_plan* call with num_seqs == B
 *   out          device bf16, q's shape, innermost stride 1 (written)
 *   lse          device f32 [B][H_q] (or [B][q_len][H_q]) natural-log LSE
 *                (written), or NULL
 * With q_len >= the threshold of hpc_decode_tc_min_q_len (by default 4 for
 * a bf16 cache, 3 for fp8_e4m3) and a
 * dynamic tile plan, the tile products run on the tcgen05 tensor cores, one
 * CTA per (KV head, plan part): such a plan is best built with
 * num_sms / H_kv parts. Otherwise one warp per (token, KV head) runs them.
 * Requirements: H_q == 8 * H_kv and H_kv in {1, 2, 4, 8, 16, 32, 64};
 * head_dim 128; 64-token blocks -- else HPC_ERR_UNSUPPORTED.
 * The first call on a plan from hpc_decode_plan / _static allocates its
 * partial workspace (plans from hpc_decode_plan_create already have it).
 * Bad block ids read zeros and set HPC_DEVCHK_BAD_BLOCK; see
 * hpc_decode_plan_status.
 */
hpc_status hpc_decode_attn(const hpc_tensor* q, const hpc_tensor* k_cache,
                           const hpc_tensor* v_cache, const hpc_tensor* block_table,
                           const hpc_tensor* seq_lens, hpc_plan_t plan, hpc_tensor* out,
                           hpc_tensor* lse, void* stream);

/*
 * hpc_decode_step -- one whole decode step on the device, planned from the
 * device lengths inside the step (section "Attention Backend: Dynamic
 * Load-Balanced Scheduling": tiles spread over a persistent grid by actual
 * work, partial states merged by log-sum-exp). Three routes:
 *  - one query token per sequence (q [B][H_q][128]) and B <= 3072: one
 *    launch of the step kernel, which plans the step (units = (tile, KV
 *    head) pairs; balanced static parts plus a pool of chunks the CTAs take
 *    at run time), computes it and merges every split (sequence, KV head)
 *    pair in the kernel. Afterwards `plan` holds the step's work list as
 *    HPC_PLAN_STEP records (hpc_decode_plan_export);
 *  - q_len at or above the tensor-core threshold (hpc_decode_tc_min_q_len):
 *    the planner kernel builds a tile plan of max(1, num_sms / H_kv) parts,
 *    the tensor-core kernel runs one CTA per (KV head, part), then the merge
 *    kernel;
 *  - otherwise (multi-token q below the threshold, or B > 3072): the balanced
 *    plan of hpc_decode_plan_device (folded into the attention kernel's
 *    start up to 3072 sequences, else the planner kernel first), attention
 *    and merge; `plan` then holds that plan's words, word for word the host
 *    planner's for the same lengths (hpc_decode_plan_compute_ex): one unit
 *    per (tile, KV head) when num_kv_heads * q_len <= 8 and num_kv_heads > 1,
 *    else tiles.
 * Allocates nothing; may be captured in a CUDA graph after a first call
 * outside the capture.
 *   q, k_cache, v_cache, block_table, out, lse: as hpc_decode_attn
 *   seq_lens  device int32 [B], contiguous; on the one-token route a negative
 *             length, a sequence of more than INT32_MAX / 352 (tile, KV head)
 *             units, or more than INT32_MAX units in all set
 *             HPC_DEVCHK_BAD_LENGTH and the step writes out = 0, lse = -inf
 *             for every sequence
 *   plan      from hpc_decode_plan_create with max_seqs >= B
 *   num_sms   CTAs of the persistent grid, <= the plan's num_sms
 */
hpc_status hpc_decode_step(const hpc_tensor* q, const hpc_tensor* k_cache,
                           const hpc_tensor* v_cache, const hpc_tensor* block_table,
                           const hpc_tensor* seq_lens, hpc_plan_t plan, int32_t num_sms,
                           hpc_tensor* out, hpc_tensor* lse, void* stream);

/*
 * hpc_decode_step_host -- hpc_decode_step with the step's inputs and results
 * in HOST memory: the copies in, the step and the copies out are enqueued on
 * `stream` by the library (one cudaMemcpyAsync per buffer), so a caller
 * whose batch lives on the host makes one call per step. The caches stay on
 * the device.
 *   q, block_table, seq_lens  host tensors, contiguous (dense, outermost
 *                             first), same shapes and dtypes as for
 *                             hpc_decode_step; read by the copies, which
 *                             are asynchronous only for page-locked memory
 *   out, lse                  host tensors, contiguous, written when the
 *                             stream reaches the copies out (lse may be NULL)
 *   k_cache, v_cache, plan, num_sms, stream: as hpc_decode_step
 * The plan owns a device staging area for the five buffers; the first call
 * (or one with a larger batch) allocates it, later calls reuse it. Host
 * buffers must stay valid and unchanged until the stream has passed the
 * copies; two calls on one plan must not overlap on different streams.
 * Errors: HPC_ERR_INVALID_ARG for a null or non-contiguous host tensor (no
 * copy enqueued), HPC_ERR_OOM if the staging area cannot be allocated,
 * otherwise hpc_decode_step's.
 */
hpc_status hpc_decode_step_host(const hpc_tensor* q, const hpc_tensor* k_cache,
                                const hpc_tensor* v_cache, const hpc_tensor* block_table,
                                const hpc_tensor* seq_lens, hpc_plan_t plan, int32_t num_sms,
                                hpc_tensor* out, hpc_tensor* lse, void* stream);

/* hpc_decode_attn_ex -- hpc_decode_attn with an explicit softmax scale
 * (> 0; a value <= 0 selects 1/sqrt(head_dim)). */
hpc_status hpc_decode_attn_ex(const hpc_tensor* q, const hpc_tensor* k_cache,
                              const hpc_tensor* v_cache, const hpc_tensor* block_table,
                              const hpc_tensor* seq_lens, hpc_plan_t plan, hpc_tensor* out,
                              hpc_tensor* lse, float softmax_scale, void* stream);

/*
 * hpc_decode_tc_min_q_len -- the smallest q_len for which hpc_decode_attn*
 * and hpc_decode_step use the tensor-core kernel (process-wide setting).
 *   q_len     >= 2: the new threshold for both cache dtypes (above 8: the
 *             path is never used); 0: the defaults (4 with a bf16 cache, 3
 *             with fp8_e4m3, the measured crossovers); < 0: no change
 *             (query only); 1: HPC_ERR_INVALID_ARG
 *   previous  host int32 receiving the setting before the call (0 for the
 *             defaults), or NULL
 * Both kernels compute the same attention; the setting moves only the
 * choice of kernel (tests and benchmarks pin one with it).
 */
hpc_status hpc_decode_tc_min_q_len(int32_t q_len, int32_t* previous);

/*
 * hpc_decode_plan_set_timing_events -- instrumentation: while set, each
 * hpc_decode_attn on this plan records `ev_start` just before the attention
 * kernel, `ev_attn_done` between the attention and merge kernels, and
 * `ev_end` after the merge kernel, all on the call's stream. Each argument is
 * a cudaEvent_t owned by the caller, or NULL (not recorded).
 */
hpc_status hpc_decode_plan_set_timing_events(hpc_plan_t plan, void* ev_start, void* ev_attn_done,
                                             void* ev_end);

/*
 * hpc_decode_attn_noalloc -- one decode step (device planner, attention,
 * merge) that allocates no memory at all. The pages have no counterpart of
 * this call; it exists for callers that cannot call cudaMalloc/cudaFree:
 * code running inside an engine's enqueue step or a plugin whose contract
 * forbids allocation there, and code whose device memory is all owned by a
 * caching allocator, where a direct cudaMalloc/cudaFree would synchronise the
 * device or fail under memory pressure.
 *
 * Its work list, partial results and error word live in one file-scope
 * device array of about 13.9 MB that every GPU loading this library holds
 * until the process exits. Limits (HPC_ERR_INVALID_ARG beyond them, with a
 * message): num_seqs <= HPC_NOALLOC_MAX_SEQS, CTAs <= HPC_NOALLOC_MAX_CTAS,
 * num_q_heads <= HPC_NOALLOC_MAX_Q_HEADS.
 *
 *   q, out      bf16 [B][H_q][128]: one query token per sequence only (the
 *               multi-token [B][q_len][H_q][128] form of hpc_decode_attn is
 *               refused with HPC_ERR_INVALID_ARG: its partial states would
 *               need q_len times the scratch)
 *   k_cache, v_cache, block_table, seq_lens, lse: as hpc_decode_attn
 *               (seq_lens on the device; the plan is built from them here)
 *   num_sms     CTAs of the persistent grid; <= 0 uses the device's SM count
 *   device_error  device int32 receiving HPC_DEVCHK_* bits by atomic OR (the
 *               caller zeroes it), or NULL to discard them
 * Every argument check is made before anything is enqueued: a call that
 * returns an error has launched nothing and left the array as it was. The
 * first call on each device looks up the array's device address for that
 * device (cudaGetSymbolAddress) with the device current; make that first call
 * before any stream capture. The lookup is repeated only when the device's
 * context has been replaced (after cudaDeviceReset the module, and with it the
 * array, may sit elsewhere). Every call uses the same array and it keeps the
 * last call's contents, so calls whose work overlaps on the GPU (other
 * streams, other threads) race with each other: order them on one stream.
 */
#define HPC_NOALLOC_MAX_SEQS 256
#define HPC_NOALLOC_MAX_CTAS 160
#define HPC_NOALLOC_MAX_Q_HEADS 64
hpc_status hpc_decode_attn_noalloc(const hpc_tensor* q, const hpc_tensor* k_cache,
                                   const hpc_tensor* v_cache, const hpc_tensor* block_table,
                                   const hpc_tensor* seq_lens, int32_t num_sms, hpc_tensor* out,
                                   hpc_tensor* lse, int32_t* device_error, void* stream);

/*
 * hpc_rope_norm_kv_write -- the fused decode prologue that feeds the path
 * ("vLLM x HPC-Ops", section "Attention Backend: Dynamic Load-Balanced
 * Scheduling", the HpcRopeNorm paragraph: QK-Norm, RoPE, KV-cache write and,
 * in FP8, query quantisation in one kernel). For the new token of every
 * sequence (position pos = seq_lens[b] - 1; sequences with seq_lens <= 0 are
 * skipped):
 *   q' = RoPE(RMSNorm(q) * q_norm_weight), k' = RoPE(RMSNorm(k) * k_norm_weight)
 *   RMSNorm(x) = x / sqrt(mean(x^2) + eps) over head_dim, per head;
 *   RoPE rotates pairs (i, i + 64) by pos * rope_base^(-2i/128);
 * then writes q' to q_out (bf16; may alias q_in), optionally e4m3(q' / scale)
 * to q_out_fp8 (scale in its descriptor), and k', v into the cache at slot
 * pos % 64 of block block_table[b][pos / 64] (bf16, or e4m3(x / scale) with
 * the cache's per-tensor scale, round to nearest even, saturating at 448).
 *   q_in [B][H_q][128], k_in / v_in [B][H_kv][128]: device bf16, rows contiguous
 *   seq_lens device int32 [B] (lengths including the new token)
 *   block_table device int32 [B][max_blocks]
 *   q_norm_weight, k_norm_weight: device bf16 or f32 [128], 16-byte aligned
 *   k_cache, v_cache: as hpc_decode_attn (written in place)
 *   device_error: optional device int32 receiving HPC_DEVCHK_* bits (a block
 *   id out of range or a table too short skips that row's write)
 * The readings where the pages are silent (RMSNorm, norm before RoPE, the
 * rotate-half pairing) are stated above; rope_base > 1, eps >= 0.
 */
hpc_status hpc_rope_norm_kv_write(const hpc_tensor* q_in, const hpc_tensor* k_in,
                                  const hpc_tensor* v_in, const hpc_tensor* seq_lens,
                                  const hpc_tensor* block_table, const hpc_tensor* q_norm_weight,
                                  const hpc_tensor* k_norm_weight, float eps, float rope_base,
                                  hpc_tensor* q_out, hpc_tensor* q_out_fp8, hpc_tensor* k_cache,
                                  hpc_tensor* v_cache, int32_t* device_error, void* stream);

/*
 * hpc_extend_attn -- prefill / extend attention over the paged cache ("vLLM x
 * HPC-Ops", section "Attention Across Prefill, Extend and Decode Shapes",
 * which benchmarks q512 prefill with the decode kernel's shapes). Sequence b
 * has n_b = cu_q_lens[b+1] - cu_q_lens[b] new tokens whose K and V are
 * already in its cache as its last n_b positions of L_b = seq_lens[b]; new
 * token i attends to positions 0 .. L_b - n_b + i (causal). Prefill is
 * n_b = L_b, decode n_b = 1. Runs on the tcgen05 tensor cores, one CTA per
 * (KV head, 16 or 32 new tokens of one sequence; see hpc_extend_attn_ex).
 *   q           device bf16 [total_q][H_q][128], ragged: the rows of sequence
 *               b start at cu_q_lens[b]; innermost stride 1, other strides
 *               multiples of 8 elements, base 16-byte aligned
 *   k_cache, v_cache, block_table: as hpc_decode_attn (bf16, or fp8_e4m3
 *               with per-tensor scales in the descriptors; e4m3 tiles are
 *               widened exactly to bf16 on the chip before the MMAs)
 *   seq_lens    device int32 [B], L_b >= n_b (else HPC_DEVCHK_BAD_LENGTH and
 *               that sequence's rows are not written)
 *   cu_q_lens   device int32 [B+1], non-decreasing, cu_q_lens[0] = 0,
 *               cu_q_lens[B] = total_q
 *   out         device bf16 [total_q][H_q][128] (written), q's layout rules
 *   lse         device f32 [total_q][H_q] natural-log LSE (written), or NULL
 *   softmax_scale  > 0, or <= 0 for 1/sqrt(128)
 *   device_error   optional device int32 receiving HPC_DEVCHK_* bits
 * Requirements: H_q == 8 * H_kv, head_dim 128, 64-token blocks, and
 * ceil(total_q / T) + B <= 65535 with T = 16 or 32 the CTA's new tokens
 * (else HPC_ERR_UNSUPPORTED). Allocates nothing; never synchronises the
 * stream.
 */
hpc_status hpc_extend_attn(const hpc_tensor* q, const hpc_tensor* k_cache,
                           const hpc_tensor* v_cache, const hpc_tensor* block_table,
                           const hpc_tensor* seq_lens, const hpc_tensor* cu_q_lens,
                           hpc_tensor* out, hpc_tensor* lse, float softmax_scale,
                           int32_t* device_error, void* stream);

/* hpc_extend_attn_ex -- hpc_extend_attn with the CTA shape chosen by the
 * caller: tiles_per_cta = 1 (one 128-row query tile of 16 tokens x 8 heads
 * per CTA) or 2 (two tiles, 32 tokens, sharing every K / V tile; the
 * choice for batches that fill the GPU), or 0 for the automatic choice of
 * hpc_extend_attn (2 when ceil(total_q / 32) * H_kv >= SMs / 2). Results
 * are identical either way. Other values give HPC_ERR_INVALID_ARG. */
hpc_status hpc_extend_attn_ex(const hpc_tensor* q, const hpc_tensor* k_cache,
                              const hpc_tensor* v_cache, const hpc_tensor* block_table,
                              const hpc_tensor* seq_lens, const hpc_tensor* cu_q_lens,
                              hpc_tensor* out, hpc_tensor* lse, float softmax_scale,
                              int32_t tiles_per_cta, int32_t* device_error, void* stream);

/* hpc_device_sm_count -- streaming multiprocessors of the current device. */
hpc_status hpc_device_sm_count(int32_t* num_sms);

/* hpc_last_error -- message of the calling thread's last failure ("" if none). */
const char* hpc_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* HPC_DECODE_H */
