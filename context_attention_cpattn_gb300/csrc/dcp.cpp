// Dynamic context-parallel scheduler (host): per-micro-batch CP size and
// packing of variable-length samples ("Speeding up Variable-Length Training
// with Dynamic Context Parallelism and NVIDIA Megatron Core", data-scheduling
// section, Eq. 1-3, and the runtime section on the solver's small grid
// search).
//
//   workload(S) = attn_coef * S(S+1)/2 + lin_coef * S   (O(S^2) + O(S))
//   memory(S)   = S tokens                              (O(S))
//
// Quota per micro-batch Q = ceil(total / n_micro) (Eq. 2-3 with the same
// micro-batch count on every DP rank).  A sample takes the smallest power of
// two c <= max_cp with workload <= c*Q and S <= c*cap (else max_cp).  The
// n_micro lowest-workload samples open one micro-batch each (memory first);
// every other sample, by descending workload, goes to the micro-batch whose
// per-GPU load after the placement, workload * max_cp / cp, is least among
// those that keep tokens <= cp * cap (else the least-loaded one).  A
// micro-batch's CP size is the largest of its samples'.  Ties go to the lower
// index.  All decisions are in exact integer arithmetic.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <string>
#include <vector>

#include "../../include/cpattn.h"

namespace cpattn {
cpattn_status_t set_error(cpattn_status_t s, const std::string& msg);
}

namespace {

using i128 = __int128;
constexpr int64_t kI64Max = INT64_MAX;

struct Schedule {
  std::vector<int32_t> sample_micro, sample_cp, micro_cp;
  std::vector<int64_t> micro_work, micro_tokens;
};

cpattn_status_t check_config(const cpattn_dcp_config_t* cfg) {
  if (!cfg) return cpattn::set_error(CPATTN_INVALID_ARG, "dcp: config is NULL");
  const int32_t c = cfg->max_cp;
  if (c < 1 || c > 1024 || (c & (c - 1)) != 0)
    return cpattn::set_error(CPATTN_INVALID_ARG, "dcp: max_cp must be a power of two in [1, 1024]");
  if (cfg->cap_tokens < 1) return cpattn::set_error(CPATTN_INVALID_ARG, "dcp: cap_tokens must be >= 1");
  if (cfg->attn_coef < 0 || cfg->lin_coef < 0)
    return cpattn::set_error(CPATTN_INVALID_ARG, "dcp: workload coefficients must be >= 0");
  return CPATTN_OK;
}

// Per-sample workloads; rejects lengths < 1 and totals whose per-GPU load
// (total * max_cp) leaves int64.
cpattn_status_t workloads(const int64_t* seqlens, int64_t n, const cpattn_dcp_config_t* cfg,
                          std::vector<int64_t>* w, int64_t* total) {
  if (n < 0 || (n > 0 && !seqlens)) return cpattn::set_error(CPATTN_INVALID_ARG, "dcp: bad sample list");
  w->resize((size_t)n);
  i128 sum = 0;
  for (int64_t s = 0; s < n; ++s) {
    const int64_t S = seqlens[s];
    if (S < 1 || S > (int64_t(1) << 40)) return cpattn::set_error(CPATTN_INVALID_ARG, "dcp: sample length out of range");
    const i128 x = (i128)cfg->attn_coef * ((i128)S * (S + 1) / 2) + (i128)cfg->lin_coef * S;
    sum += x;
    if (sum * cfg->max_cp > (i128)kI64Max)
      return cpattn::set_error(CPATTN_INVALID_ARG, "dcp: total workload * max_cp exceeds int64");
    (*w)[(size_t)s] = (int64_t)x;
  }
  *total = (int64_t)sum;
  return CPATTN_OK;
}

void schedule(const int64_t* S, const std::vector<int64_t>& w, int64_t total, const cpattn_dcp_config_t* cfg,
              int32_t n_micro, Schedule* out) {
  const int64_t n = (int64_t)w.size();
  const int32_t max_cp = cfg->max_cp;
  const i128 cap = cfg->cap_tokens;
  const int64_t quota = (total + n_micro - 1) / n_micro;

  out->sample_micro.assign((size_t)n, -1);
  out->sample_cp.resize((size_t)n);
  out->micro_cp.assign((size_t)n_micro, 1);
  out->micro_work.assign((size_t)n_micro, 0);
  out->micro_tokens.assign((size_t)n_micro, 0);
  for (int64_t s = 0; s < n; ++s) {
    int32_t c = max_cp;
    for (int32_t t = 1; t <= max_cp; t *= 2)
      if ((i128)w[s] <= (i128)t * quota && (i128)S[s] <= (i128)t * cap) {
        c = t;
        break;
      }
    out->sample_cp[(size_t)s] = c;
  }

  std::vector<int64_t> order((size_t)n);
  for (int64_t s = 0; s < n; ++s) order[(size_t)s] = s;
  std::sort(order.begin(), order.end(), [&](int64_t a, int64_t b) { return w[a] != w[b] ? w[a] < w[b] : a < b; });

  auto place = [&](int32_t b, int64_t s) {
    out->sample_micro[(size_t)s] = b;
    out->micro_work[b] += w[s];
    out->micro_tokens[b] += S[s];
    out->micro_cp[b] = std::max(out->micro_cp[b], out->sample_cp[(size_t)s]);
  };
  const int64_t seeds = std::min<int64_t>(n, n_micro);
  for (int64_t i = 0; i < seeds; ++i) place((int32_t)i, order[(size_t)i]);

  std::sort(order.begin() + seeds, order.end(),
            [&](int64_t a, int64_t b) { return w[a] != w[b] ? w[a] > w[b] : a < b; });
  for (int64_t i = seeds; i < n; ++i) {
    const int64_t s = order[(size_t)i];
    int32_t best = -1, fall = -1;
    i128 best_load = 0, fall_load = 0;
    for (int32_t b = 0; b < n_micro; ++b) {
      const int32_t c = std::max(out->micro_cp[b], out->sample_cp[(size_t)s]);
      const i128 ld = (i128)(out->micro_work[b] + w[s]) * (max_cp / c);
      if (fall < 0 || ld < fall_load) {
        fall = b;
        fall_load = ld;
      }
      if ((i128)out->micro_tokens[b] + S[s] <= (i128)c * cap && (best < 0 || ld < best_load)) {
        best = b;
        best_load = ld;
      }
    }
    place(best >= 0 ? best : fall, s);
  }
}

int64_t max_load(const Schedule& sc, int32_t max_cp) {
  int64_t m = 0;
  for (size_t b = 0; b < sc.micro_work.size(); ++b)
    m = std::max(m, sc.micro_work[b] * (max_cp / sc.micro_cp[b]));
  return m;
}

template <typename T>
void copy_out(const std::vector<T>& v, T* dst) {
  if (dst) std::copy(v.begin(), v.end(), dst);
}

}  // namespace

extern "C" {

cpattn_status_t cpattn_dcp_quotas(const int32_t* m, int32_t dp, int32_t vpp, int32_t pp, double total, double* w_out) {
  if (!m || !w_out || dp < 1 || vpp < 1 || pp < 1 || !std::isfinite(total) || total < 0)
    return cpattn::set_error(CPATTN_INVALID_ARG, "dcp_quotas: bad arguments");
  // Eq. 1: W_i (m_i V + p - 1) = K on every rank; Eq. 3: sum_i W_i m_i = total.
  double denom = 0.0;
  for (int32_t i = 0; i < dp; ++i) {
    if (m[i] < 1) return cpattn::set_error(CPATTN_INVALID_ARG, "dcp_quotas: micro-batch counts must be >= 1");
    denom += (double)m[i] / ((double)m[i] * vpp + pp - 1);
  }
  const double K = total / denom;
  for (int32_t i = 0; i < dp; ++i) w_out[i] = K / ((double)m[i] * vpp + pp - 1);
  return CPATTN_OK;
}

cpattn_status_t cpattn_dcp_schedule(const int64_t* seqlens, int64_t n, const cpattn_dcp_config_t* cfg,
                                    int32_t n_micro, int32_t* sample_micro, int32_t* sample_cp, int32_t* micro_cp,
                                    int64_t* micro_work, int64_t* micro_tokens) {
  if (cpattn_status_t st = check_config(cfg)) return st;
  if (n_micro < 1) return cpattn::set_error(CPATTN_INVALID_ARG, "dcp_schedule: n_micro must be >= 1");
  std::vector<int64_t> w;
  int64_t total = 0;
  if (cpattn_status_t st = workloads(seqlens, n, cfg, &w, &total)) return st;
  Schedule sc;
  schedule(seqlens, w, total, cfg, n_micro, &sc);
  copy_out(sc.sample_micro, sample_micro);
  copy_out(sc.sample_cp, sample_cp);
  copy_out(sc.micro_cp, micro_cp);
  copy_out(sc.micro_work, micro_work);
  copy_out(sc.micro_tokens, micro_tokens);
  return CPATTN_OK;
}

cpattn_status_t cpattn_dcp_sweep(const int64_t* seqlens, int64_t n, const cpattn_dcp_config_t* cfg, int32_t dp,
                                 int32_t pp, int32_t vpp, int32_t mult, int64_t* budgets, int32_t* knee_m,
                                 int32_t* best_m) {
  if (cpattn_status_t st = check_config(cfg)) return st;
  if (dp < 1 || pp < 1 || vpp < 1 || mult < 1 || (int64_t)dp * mult * pp > (1 << 20))
    return cpattn::set_error(CPATTN_INVALID_ARG, "dcp_sweep: need dp, pp, vpp, mult >= 1 and dp*mult*pp <= 2^20");
  std::vector<int64_t> w;
  int64_t total = 0;
  if (cpattn_status_t st = workloads(seqlens, n, cfg, &w, &total)) return st;
  const int32_t g = (mult - 1) * pp + 1;  // m = pp .. mult*pp
  std::vector<int64_t> bud((size_t)g);
  Schedule sc;
  for (int32_t i = 0; i < g; ++i) {
    schedule(seqlens, w, total, cfg, dp * (pp + i), &sc);
    bud[(size_t)i] = max_load(sc, cfg->max_cp);
  }
  // knee: the point farthest below the chord of the [0,1]-scaled curve
  const i128 X = g - 1, Y = (i128)bud[0] - bud[(size_t)g - 1];
  int32_t k = 0;
  if (X > 0 && Y > 0) {
    i128 best = 0;
    for (int32_t i = 0; i < g; ++i) {
      const i128 score = (i128)i * Y + ((i128)bud[(size_t)i] - bud[(size_t)g - 1]) * X;
      if (i == 0 || score < best) {
        best = score;
        k = i;
      }
    }
  }
  // neighbourhood of the knee, scored by the Eq. 1 step time budget * (mV + p - 1)
  int32_t pick = -1;
  i128 pick_t = 0;
  for (int32_t i = k - 1; i <= k + 1; ++i) {
    if (i < 0 || i >= g) continue;
    const i128 t = (i128)bud[(size_t)i] * ((i128)(pp + i) * vpp + pp - 1);
    if (pick < 0 || t < pick_t) {
      pick = i;
      pick_t = t;
    }
  }
  copy_out(bud, budgets);
  if (knee_m) *knee_m = pp + k;
  if (best_m) *best_m = pp + pick;
  return CPATTN_OK;
}

}  // extern "C"
