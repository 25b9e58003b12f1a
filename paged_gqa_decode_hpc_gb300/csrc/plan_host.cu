// Host tile planners: the per-step load-balanced plan and the static
// even split-KV plan ("vLLM x HPC-Ops", section "Attention Backend: Dynamic
// Load-Balanced Scheduling"). The device planner (plan_device.cu) computes
// the same words from the same closed forms.
#include <algorithm>
#include <cstring>
#include <vector>

#include "hpc_internal.h"

namespace hpc {

namespace {

inline int64_t part_start(int64_t p, int64_t T, int64_t P) { return (p * T) / P; }
// Part owning flattened tile x: the largest p with floor(p*T/P) <= x.
inline int64_t part_of(int64_t x, int64_t T, int64_t P) { return ((x + 1) * P - 1) / T; }

}  // namespace

int64_t dynamic_max_segs(int32_t num_seqs, int32_t num_parts) {
  // A segment starts at a part start or at a sequence start.
  return (int64_t)num_seqs + num_parts;
}

hpc_status plan_dynamic_host(const int32_t* seq_lens, int32_t B, int32_t num_sms, int32_t* w,
                             const PlanLayout& L, std::string* err, int32_t units_per_tile) {
  if (units_per_tile <= 0) {
    *err = "units_per_tile must be positive";
    return HPC_ERR_INVALID_ARG;
  }
  if (B < 0 || (B > 0 && !seq_lens)) {
    *err = "seq_lens is null or num_seqs < 0";
    return HPC_ERR_INVALID_ARG;
  }
  if (num_sms <= 0) {
    *err = "num_sms must be positive";
    return HPC_ERR_INVALID_ARG;
  }
  if (B > L.cap_seqs) {
    *err = "num_seqs exceeds the plan's capacity";
    return HPC_ERR_INVALID_ARG;
  }
  int32_t* cu = w + L.cu_off();
  cu[0] = 0;
  int64_t total = 0;
  for (int32_t b = 0; b < B; ++b) {
    if (seq_lens[b] < 0) {
      *err = "negative sequence length at index " + std::to_string(b);
      return HPC_ERR_INVALID_ARG;
    }
    total += (seq_lens[b] + (int64_t)kBlockTokens - 1) / kBlockTokens * units_per_tile;
    if (total > INT32_MAX) {
      *err = "total tile count exceeds 2^31-1";
      return HPC_ERR_INVALID_ARG;
    }
    cu[b + 1] = (int32_t)total;
  }
  const int64_t T = total;
  const int64_t P = std::min<int64_t>(num_sms, T);
  if (P > L.cap_parts || (int64_t)B + P > L.cap_segs) {
    *err = "step exceeds the plan's capacity (parts)";
    return HPC_ERR_INVALID_ARG;
  }
  int32_t* seq_off = w + L.seq_off();
  int32_t* part_off = w + L.part_off();
  int32_t* segs = w + L.seg_off();
  seq_off[0] = 0;
  int64_t g = 0;
  for (int32_t b = 0; b < B; ++b) {
    const int64_t lo_b = cu[b], hi_b = cu[b + 1];
    int64_t cnt = 0;
    if (hi_b > lo_b) {
      const int64_t pf = part_of(lo_b, T, P), pl = part_of(hi_b - 1, T, P);
      cnt = pl - pf + 1;
      for (int64_t j = 0; j < cnt; ++j) {
        const int64_t p = pf + j;
        const int64_t lo = std::max(lo_b, part_start(p, T, P));
        const int64_t hi = std::min(hi_b, part_start(p + 1, T, P));
        int32_t* s = segs + 4 * (g + j);
        s[0] = b;
        s[1] = (int32_t)(lo - lo_b);
        s[2] = (int32_t)(hi - lo_b);
        s[3] = cnt == 1 ? HPC_SEG_WHOLE : 0;
      }
    }
    g += cnt;
    seq_off[b + 1] = (int32_t)g;
  }
  if (g > L.cap_segs) {
    *err = "internal: segment capacity exceeded";
    return HPC_ERR_INVALID_ARG;
  }
  for (int64_t p = 0; p < P; ++p) {
    const int64_t s = part_start(p, T, P);
    // sequence holding tile s: last b with cu[b] <= s (it is non-empty)
    const int32_t b = (int32_t)(std::upper_bound(cu, cu + B + 1, (int32_t)s) - cu) - 1;
    part_off[p] = seq_off[b] + (int32_t)(p - part_of(cu[b], T, P));
  }
  part_off[P] = (int32_t)g;
  w[kMagic] = kPlanMagic;
  w[kKind] = HPC_PLAN_DYNAMIC;
  w[kNumSeqs] = B;
  w[kNumParts] = (int32_t)P;
  w[kNumTiles] = (int32_t)T;
  w[kNumSegs] = (int32_t)g;
  w[kNumSms] = num_sms;
  w[kSplits] = units_per_tile > 1 ? units_per_tile : 0;
  return HPC_OK;
}

hpc_status plan_static_host(const int32_t* seq_lens, int32_t B, int32_t num_sms,
                            int32_t num_kv_heads, int32_t num_splits, int32_t** words_out,
                            PlanLayout* L_out, std::string* err) {
  *words_out = nullptr;
  if (B < 0 || (B > 0 && !seq_lens) || num_sms <= 0 || num_kv_heads <= 0) {
    *err = "invalid static plan arguments";
    return HPC_ERR_INVALID_ARG;
  }
  std::vector<int64_t> n(B);
  int64_t total = 0, max_n = 1;
  for (int32_t b = 0; b < B; ++b) {
    if (seq_lens[b] < 0) {
      *err = "negative sequence length at index " + std::to_string(b);
      return HPC_ERR_INVALID_ARG;
    }
    n[b] = (seq_lens[b] + (int64_t)kBlockTokens - 1) / kBlockTokens;
    total += n[b];
    max_n = std::max(max_n, n[b]);
  }
  if (total > INT32_MAX) {
    *err = "total tile count exceeds 2^31-1";
    return HPC_ERR_INVALID_ARG;
  }
  int64_t S;
  if (num_splits > 0) {
    S = num_splits;
  } else {
    const int64_t denom = (int64_t)B * num_kv_heads;
    S = denom > 0 ? (2LL * num_sms + denom - 1) / denom : 1;
  }
  S = std::max<int64_t>(1, std::min(S, max_n));
  std::vector<int32_t> segs;
  std::vector<int32_t> seq_off(B + 1, 0);
  for (int32_t b = 0; b < B; ++b) {
    int64_t nonempty = 0;
    for (int64_t i = 0; i < S; ++i) nonempty += ((i + 1) * n[b]) / S > (i * n[b]) / S;
    for (int64_t i = 0; i < S; ++i) {
      const int64_t lo = (i * n[b]) / S, hi = ((i + 1) * n[b]) / S;
      if (lo < hi) {
        segs.push_back(b);
        segs.push_back((int32_t)lo);
        segs.push_back((int32_t)hi);
        segs.push_back(nonempty == 1 ? HPC_SEG_WHOLE : 0);
      }
    }
    seq_off[b + 1] = (int32_t)(segs.size() / 4);
  }
  const int32_t nseg = (int32_t)(segs.size() / 4);
  PlanLayout L;
  L.cap_seqs = B;
  L.cap_parts = nseg;
  L.cap_segs = nseg;
  int32_t* w = (int32_t*)calloc((size_t)L.words(), sizeof(int32_t));
  if (!w) {
    *err = "host allocation failed";
    return HPC_ERR_OOM;
  }
  w[kMagic] = kPlanMagic;
  w[kKind] = HPC_PLAN_STATIC;
  w[kNumSeqs] = B;
  w[kNumParts] = nseg;
  w[kNumTiles] = (int32_t)total;
  w[kNumSegs] = nseg;
  w[kNumSms] = num_sms;
  w[kSplits] = (int32_t)S;
  for (int32_t p = 0; p <= nseg; ++p) w[L.part_off() + p] = p;
  std::copy(seq_off.begin(), seq_off.end(), w + L.seq_off());
  int32_t* cu = w + L.cu_off();
  cu[0] = 0;
  for (int32_t b = 0; b < B; ++b) cu[b + 1] = cu[b] + (int32_t)n[b];
  if (!segs.empty()) std::memcpy(w + L.seg_off(), segs.data(), segs.size() * sizeof(int32_t));
  *words_out = w;
  *L_out = L;
  return HPC_OK;
}

}  // namespace hpc
