// Prefill / extend attention over the paged KV cache on the 5th-generation
// tensor cores (tcgen05), for sm_103a.
//
// The pages benchmark one attention kernel across prefill, extend and decode
// shapes ("vLLM x HPC-Ops", section "Attention Across Prefill, Extend and
// Decode Shapes": q512 prefill, "8q1s1k" decode) without describing it. What
// it computes here: sequence b has L_b positions in its paged cache, the
// last n_b of which are its new tokens (already written); new token i
// attends causally to the positions before L_b - n_b + 1 + i. Prefill is
// n_b = L_b. GQA with 8 query heads per KV head, head_dim 128, 64-token
// blocks, BF16 cache.
//
// GB300 design. Unlike decode (8 FLOP per byte, HBM-bound, mma.sync), a
// tile of 16 new tokens x 8 query heads = 128 query rows shares every K / V
// tile, so the work is a dense contraction and runs on tcgen05:
//  * CTA = (KV head, 16-token tile of one sequence); 6 warps: 4 softmax
//    warps (thread = query row = TMEM lane), 1 TMA producer warp, 1 MMA warp.
//  * TMA loads Q once (3-D map over [token][head][128], box 16 x 8 x 64,
//    128-byte swizzle: row t*8+g of the tile is query head g of token t) and
//    the K / V tiles of the sequence's blocks into a 4-stage ring.
//  * S_j = Q K_j^T (M 128, N 64, K 128) into tensor memory, two buffers so
//    the MMA of tile j+1 runs while the softmax warps work on tile j.
//  * Online softmax in the log2 domain, one row per thread, no shuffles. The
//    running maximum is only moved (and O rescaled in tensor memory) when a
//    row's maximum grows by more than 8 (a factor 256): P = 2^(s - m) then
//    stays below 256, and the final O / l uses one consistent m per row.
//  * P (bf16) is written to shared memory in the K-major 128-byte-swizzled
//    layout and O += P V_j (M 128, N 128, K 64) accumulates in tensor memory
//    (V is the MN-major operand straight from its TMA tile).
//  * Epilogue: O / l -> bf16 rows of out, lse = ln 2 * (m + log2 l).
//  * Every wait is bounded (globaltimer); a timeout sets the error bit, all
//    roles stop issuing, and the CTA drains its copies and MMAs and frees its
//    tensor memory before leaving. No trap, no assert.
#include <cuda_bf16.h>

#include "hpc_decode.h"
#include "prefill.h"
#include "tc05.cuh"

namespace hpc {

namespace {

using namespace tc05;

constexpr int kRows = 128;
constexpr int kGroupRows = 8;  // query heads per KV head
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr uint32_t kQBytes = kRows * 128 * 2;         // 32 KB: two 16 KB column halves
constexpr uint32_t kKVTileBytes = 64 * 128 * 2;       // 16 KB: two 8 KB column halves
constexpr uint32_t kStageBytes = 2 * kKVTileBytes;    // K + V
constexpr uint32_t kPBytes = kRows * 64 * 2;          // 16 KB: 128 rows x 64 tokens
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kOffQ + kQBytes;
constexpr uint32_t kOffP = kOffKV + kStages * kStageBytes;
constexpr uint32_t kOffBar = kOffP + 2 * kPBytes;
// barriers: q_full, kv_full[S], kv_empty[S], s_full[2], s_free[2], p_full[2], pv_done[2], drain
constexpr int kNumBars = 1 + 2 * kStages + 8 + 1;
constexpr uint32_t kOffMisc = kOffBar + 8 * kNumBars;
constexpr uint32_t kSmemBytes = kOffMisc + 64 + 1024;  // + slack to align the base to 1024
constexpr uint32_t kTmemCols = 256;  // S0 | S1 | O
constexpr uint32_t kColS = 0, kColO = 128;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Bounded wait on an mbarrier phase; false when the CTA aborts or the limit
// passes (then the abort flag and the error bit are set).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int32_t* err, unsigned long long limit_ns,
                                         bool honour_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (honour_abort && *abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) {
        if (err) atomicOr(err, HPC_DEVCHK_TIMEOUT);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct TileInfo {
  int valid;   // 0: no tile for this CTA
  int b;       // sequence
  int t0;      // first new token of the tile (within the sequence)
  int n;       // new tokens of the sequence
  int L;       // positions of the sequence
  int q0;      // row of the sequence's first new token in q / out
  int n_kv;    // KV tiles this CTA reads
};

// Warp-cooperative: map tile index y (heaviest first) to (sequence, tile).
// Every sequence contributes ceil(n_b / 16) tiles; tiles are numbered in
// sequence order and y counts from the last one, so the CTAs launched first
// take the tiles that see the most keys.
__device__ TileInfo find_tile(const ExtendParams& p, int y, int lane) {
  TileInfo ti;
  ti.valid = 0;
  const int B = p.num_seqs;
  int total = 0;
  for (int c = 0; c < B; c += 32) {
    const int b = c + lane;
    int nt = 0;
    if (b < B) {
      const int n = p.cu_q_lens[b + 1] - p.cu_q_lens[b];
      nt = n > 0 ? (n + kExtendTileTokens - 1) / kExtendTileTokens : 0;
    }
    total += warp_sum_i(nt);
  }
  if (y >= total) return ti;
  const int gx = total - 1 - y;
  int base = 0;
  for (int c = 0; c < B; c += 32) {
    const int b = c + lane;
    int nt = 0;
    if (b < B) {
      const int n = p.cu_q_lens[b + 1] - p.cu_q_lens[b];
      nt = n > 0 ? (n + kExtendTileTokens - 1) / kExtendTileTokens : 0;
    }
    int incl = nt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    const int chunk = __shfl_sync(0xffffffffu, incl, 31);
    if (gx < base + chunk) {
      const unsigned hit = __ballot_sync(0xffffffffu, gx < base + incl);
      const int f = __ffs(hit) - 1;
      const int incl_f = __shfl_sync(0xffffffffu, incl, f);
      const int nt_f = __shfl_sync(0xffffffffu, nt, f);
      ti.b = c + f;
      ti.t0 = (gx - (base + incl_f - nt_f)) * kExtendTileTokens;
      ti.valid = 1;
      break;
    }
    base += chunk;
  }
  if (!ti.valid) return ti;
  ti.q0 = p.cu_q_lens[ti.b];
  ti.n = p.cu_q_lens[ti.b + 1] - ti.q0;
  ti.L = p.seq_lens[ti.b];
  if (ti.L < ti.n) {  // more new tokens than positions
    if (lane == 0 && p.err) atomicOr(p.err, HPC_DEVCHK_BAD_LENGTH);
    ti.valid = 0;
    return ti;
  }
  // keys seen by the tile's last token (padding rows past n clamp to L)
  int kv_len = ti.L - ti.n + ti.t0 + kExtendTileTokens;
  if (kv_len > ti.L) kv_len = ti.L;
  ti.n_kv = (kv_len + 63) / 64;
  return ti;
}

}  // namespace

namespace {

__global__ void __launch_bounds__(kThreads, 1)
    extend_kernel(const __grid_constant__ ExtendParams p, const __grid_constant__ CUtensorMap tmq,
                  const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1024-B alignment
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t sQ = base + kOffQ, sKV = base + kOffKV, sP = base + kOffP;
  const uint32_t bars = base + kOffBar;
  const uint32_t bar_q = bars;
  auto kv_full = [&](int s) { return bars + 8u * (1 + s); };
  auto kv_empty = [&](int s) { return bars + 8u * (1 + kStages + s); };
  auto s_full = [&](int i) { return bars + 8u * (1 + 2 * kStages + i); };
  auto s_free = [&](int i) { return bars + 8u * (3 + 2 * kStages + i); };
  auto p_full = [&](int i) { return bars + 8u * (5 + 2 * kStages + i); };
  auto pv_done = [&](int i) { return bars + 8u * (7 + 2 * kStages + i); };
  const uint32_t bar_drain = bars + 8u * (9 + 2 * kStages);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int* s_info = reinterpret_cast<int*>(smem + kOffMisc + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const unsigned long long lim_ns = p.timeout_ns;

  if (warp == 0) {
    const TileInfo ti = find_tile(p, blockIdx.y, lane);
    if (lane == 0) {
      s_info[0] = ti.valid;
      s_info[1] = ti.b;
      s_info[2] = ti.t0;
      s_info[3] = ti.n;
      s_info[4] = ti.L;
      s_info[5] = ti.q0;
      s_info[6] = ti.valid ? ti.n_kv : 0;
    }
  } else if (warp == kProducerWarp) {
    if (lane == 0) {
      mbar_init(bar_q, 1);
      for (int s = 0; s < kStages; ++s) {
        mbar_init(kv_full(s), 1);
        mbar_init(kv_empty(s), 1);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(s_full(i), 1);
        mbar_init(s_free(i), kRows);
        mbar_init(p_full(i), kRows);
        mbar_init(pv_done(i), 1);
      }
      mbar_init(bar_drain, 1);
      *s_abort = 0;
      fence_barrier_init();
      prefetch_map(&tmq);
      prefetch_map(&tmk);
      prefetch_map(&tmv);
    }
  } else if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(s_tmem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const int valid = s_info[0], b = s_info[1], t0 = s_info[2], n = s_info[3], L = s_info[4],
            q0 = s_info[5], n_kv = s_info[6];
  const uint32_t tmem = *s_tmem;
  int32_t* err = p.err;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    int issued = 0;  // K/V tiles whose copies were issued (in order)
    if (valid && n_kv > 0) {
      if (lane == 0) {
        mbar_expect_tx(bar_q, kQBytes);
        tma_load_3d(sQ, &tmq, bar_q, 0, kGroupRows * h, q0 + t0);
        tma_load_3d(sQ + kQBytes / 2, &tmq, bar_q, 64, kGroupRows * h, q0 + t0);
      }
      const int c1 = p.kv_swap ? h : 0, c2 = p.kv_swap ? 0 : h;
      int stop = 0;
      for (int j0 = 0; j0 < n_kv && !stop; j0 += 32) {
        const int jj = j0 + lane;
        int blk = -1;
        if (jj < n_kv) {
          if (jj < p.max_blocks) {
            blk = p.block_table[(int64_t)b * p.bt_sb + jj];
            if ((blk < 0 || blk >= p.num_blocks) && err) atomicOr(err, HPC_DEVCHK_BAD_BLOCK);
          } else if (err) {
            atomicOr(err, HPC_DEVCHK_TABLE_TOO_SHORT);
          }
        }
        const int cnt = n_kv - j0 < 32 ? n_kv - j0 : 32;
        for (int u = 0; u < cnt; ++u) {
          const int bk = __shfl_sync(0xffffffffu, blk, u);
          if (lane == 0) {
            const int j = j0 + u, slot = j % kStages, round = j / kStages;
            bool ok = round == 0 ||
                      wait_bar(kv_empty(slot), (round - 1) & 1, s_abort, err, lim_ns);
            if (ok) {
              const uint32_t fb = kv_full(slot);
              const uint32_t dk = sKV + slot * kStageBytes, dv = dk + kKVTileBytes;
              mbar_expect_tx(fb, kStageBytes);
              tma_load_4d(dk, &tmk, fb, 0, c1, c2, bk);
              tma_load_4d(dk + kKVTileBytes / 2, &tmk, fb, 64, c1, c2, bk);
              tma_load_4d(dv, &tmv, fb, 0, c1, c2, bk);
              tma_load_4d(dv + kKVTileBytes / 2, &tmv, fb, 64, c1, c2, bk);
              issued = j + 1;
            } else {
              stop = 1;
            }
          }
          stop = __shfl_sync(0xffffffffu, stop, 0);
          if (stop) break;
        }
      }
    }
    named_bar_sync(1, kThreads);
    // drain: the last copy issued into each slot has landed
    if (lane == 0) {
      for (int s = 0; s < kStages && s < issued; ++s) {
        const int rounds = (issued - s + kStages - 1) / kStages;
        wait_bar(kv_full(s), (rounds - 1) & 1, s_abort, err, lim_ns, false);
      }
    }
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------- MMA issue
    bool issued_any = false;
    if (valid && n_kv > 0 && lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16_f32(kRows, 64, false, false);
      constexpr uint32_t kIdPV = idesc_bf16_f32(kRows, 128, false, true);
      auto issue_pv = [&](int i) -> bool {
        if (!wait_bar(p_full(i & 1), (i >> 1) & 1, s_abort, err, lim_ns)) return false;
        tc_fence_after();
        const uint32_t vb = sKV + (i % kStages) * kStageBytes + kKVTileBytes;
        const uint32_t pb = sP + (i & 1) * kPBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          // P: K-major, 16 tokens = 32 bytes along the swizzled row
          const uint64_t a = smem_desc_sw128(pb + kk * 32, 16, 1024);
          // V: MN-major; 64-column halves 8 KB apart, 8-token row groups 1 KB apart
          const uint64_t bd = smem_desc_sw128(vb + kk * 2048, kKVTileBytes / 2, 1024);
          mma_f16_ss(tmem + kColO, a, bd, kIdPV, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(pv_done(i & 1));
        mma_commit(kv_empty(i % kStages));
        return true;
      };
      bool ok = wait_bar(bar_q, 0, s_abort, err, lim_ns);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int slot = j % kStages;
        ok = wait_bar(kv_full(slot), (j / kStages) & 1, s_abort, err, lim_ns);
        if (ok && j >= 2) ok = wait_bar(s_free(j & 1), ((j - 2) >> 1) & 1, s_abort, err, lim_ns);
        if (!ok) break;
        tc_fence_after();
        const uint32_t kb = sKV + slot * kStageBytes;
        const uint32_t dS = tmem + kColS + (uint32_t)(j & 1) * 64;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // Q and K: K-major; 64-column halves (16 KB / 8 KB apart), 16 columns = 32 bytes
          const uint64_t a = smem_desc_sw128(sQ + (kk >> 2) * (kQBytes / 2) + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(kb + (kk >> 2) * (kKVTileBytes / 2) + (kk & 3) * 32, 16, 1024);
          mma_f16_ss(dS, a, bd, kIdS, kk > 0 ? 1u : 0u);
        }
        issued_any = true;
        mma_commit(s_full(j & 1));
        if (j >= 1) ok = issue_pv(j - 1);
      }
      if (ok) issue_pv(n_kv - 1);
    }
    named_bar_sync(1, kThreads);
    if (lane == 0 && issued_any) {
      mma_commit(bar_drain);  // every MMA of this CTA has completed
      wait_bar(bar_drain, 0, s_abort, err, lim_ns, false);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  } else if (warp < 4) {
    // ------------------------------------------------------------- softmax
    const int r = threadIdx.x;  // query row = TMEM lane
    const int g = r & 7, tok = t0 + (r >> 3);
    const bool row_ok = valid && tok < n;
    int lim = L - n + 1 + tok;  // keys visible to this row: positions < lim
    if (lim > L) lim = L;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    const float sc = p.score_scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = valid && n_kv > 0;
    for (int j = 0; ok && j < n_kv; ++j) {
      ok = __all_sync(0xffffffffu, wait_bar(s_full(j & 1), (j >> 1) & 1, s_abort, err, lim_ns));
      if (!ok) break;
      tc_fence_after();
      float s[64];
      tmem_ld32(trow + kColS + (uint32_t)(j & 1) * 64, *reinterpret_cast<float(*)[32]>(&s[0]));
      tmem_ld32(trow + kColS + (uint32_t)(j & 1) * 64 + 32,
                *reinterpret_cast<float(*)[32]>(&s[32]));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(s_free(j & 1));
      const int kv0 = j * 64;
      if (kv0 + 64 > lim) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (kv0 + c >= lim) s[c] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < 64; ++c) mx = fmaxf(mx, s[c]);
      const float m_new = fmaxf(m, mx * sc);
      const bool need = m_new > m + kRescaleThreshold;
      if (j == 0) {
        m = m_new;
      } else if (__any_sync(0xffffffffu, need)) {
        ok = __all_sync(0xffffffffu,
                        wait_bar(pv_done((j - 1) & 1), ((j - 1) >> 1) & 1, s_abort, err, lim_ns));
        if (!ok) break;
        tc_fence_after();
        const float alpha = need ? ex2(m - m_new) : 1.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float o[32];
          tmem_ld32(trow + kColO + q * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(trow + kColO + q * 32, o);
        }
        tmem_wait_st();
        if (need) {
          l *= alpha;
          m = m_new;
        }
      }
      uint32_t pk[32];
      float rs = 0.f;
      const float nm = -m;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float p0 = ex2(fmaf(s[2 * c], sc, nm));
        const float p1 = ex2(fmaf(s[2 * c + 1], sc, nm));
        rs += p0 + p1;
        pk[c] = pack_bf16(p0, p1);
      }
      l += rs;
      if (j >= 2) {
        ok = __all_sync(0xffffffffu,
                        wait_bar(pv_done(j & 1), ((j - 2) >> 1) & 1, s_abort, err, lim_ns));
        if (!ok) break;
      }
      // row r of the K-major 128-byte-swizzled P tile: 16-byte chunk c -> c ^ (r % 8)
      const uint32_t prow = sP + (uint32_t)(j & 1) * kPBytes + (uint32_t)r * 128;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                         prow + ((uint32_t)(ch ^ (r & 7)) << 4)),
                     "r"(pk[4 * ch]), "r"(pk[4 * ch + 1]), "r"(pk[4 * ch + 2]),
                     "r"(pk[4 * ch + 3])
                     : "memory");
      }
      fence_async_shared();
      tc_fence_before();
      mbar_arrive(p_full(j & 1));
    }
    if (ok) {
      ok = __all_sync(0xffffffffu, wait_bar(pv_done((n_kv - 1) & 1), ((n_kv - 1) >> 1) & 1,
                                            s_abort, err, lim_ns));
    }
    if (ok) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow =
          p.out + (int64_t)(q0 + tok) * p.o_st + (int64_t)(kGroupRows * h + g) * p.o_sh;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float o[32];
        tmem_ld32(trow + kColO + q * 32, o);
        tmem_wait_ld();
        if (row_ok) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint4 v;
            v.x = pack_bf16(o[8 * c + 0] * inv, o[8 * c + 1] * inv);
            v.y = pack_bf16(o[8 * c + 2] * inv, o[8 * c + 3] * inv);
            v.z = pack_bf16(o[8 * c + 4] * inv, o[8 * c + 5] * inv);
            v.w = pack_bf16(o[8 * c + 6] * inv, o[8 * c + 7] * inv);
            *reinterpret_cast<uint4*>(orow + q * 32 + c * 8) = v;
          }
        }
      }
      if (row_ok && p.lse)
        p.lse[(int64_t)(q0 + tok) * p.l_st + (int64_t)(kGroupRows * h + g) * p.l_sh] =
            l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
    }
    tc_fence_before();
    named_bar_sync(1, kThreads);
  }
}

}  // namespace

cudaError_t launch_extend(const ExtendParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, int tiles, cudaStream_t stream) {
  if (tiles <= 0 || p.num_kv_heads <= 0) return cudaSuccess;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(extend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  extend_kernel<<<dim3(p.num_kv_heads, tiles), kThreads, kSmemBytes, stream>>>(p, tq, tk, tv);
  return cudaGetLastError();
}

}  // namespace hpc
