// Host-side DP partition planner behind the cz_plan_* entry points.
//
// Canzona summary page (paper-graph-ui), section 3.4: Eq. 1 (start-index
// ownership), the objectives J_DP / J_Comm, and Algorithm 1 (alpha-Balanced
// Greedy LPT).  Compiled with -ffp-contract=off and without fast-math so that
// every double operation rounds exactly as written; the operation order below
// is the one the reference planner uses, which makes the two bit-exact.

#include "cz_internal.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <new>
#include <numeric>
#include <vector>

using cz::Plan;

namespace cz {
uint64_t next_uid() {
  static std::atomic<uint64_t> counter{1};
  return counter.fetch_add(1);
}
}  // namespace cz

namespace {

int check_inputs(const int64_t* numels, int64_t n_params, const int64_t* bucket_sizes,
                 int64_t n_buckets, int32_t R, const int64_t* costs = nullptr) {
  if (!numels || !bucket_sizes || n_params <= 0 || n_buckets <= 0 || R < 1) return CZ_ERR_INVALID;
  int64_t sum = 0;
  for (int64_t i = 0; i < n_params; ++i)
    if (numels[i] <= 0 || (costs && costs[i] <= 0)) return CZ_ERR_INVALID;
  for (int64_t i = 0; i < n_buckets; ++i) {
    if (bucket_sizes[i] <= 0) return CZ_ERR_INVALID;
    sum += bucket_sizes[i];
    if (sum > n_params) return CZ_ERR_INVALID;
  }
  return sum == n_params ? CZ_OK : CZ_ERR_INVALID;
}

// Per-bucket prefixes, u = 0..n_i, in flat arrays: elements (phi) and cost units (cphi).
void build_prefix(Plan& p) {
  p.bucket_first.resize(p.n_buckets + 1);
  p.phi_first.resize(p.n_buckets + 1);
  p.phi.clear();
  p.cphi.clear();
  int64_t pos = 0;
  for (int64_t i = 0; i < p.n_buckets; ++i) {
    p.bucket_first[i] = pos;
    p.phi_first[i] = (int64_t)p.phi.size();
    int64_t acc = 0, cacc = 0;
    p.phi.push_back(0);
    p.cphi.push_back(0);
    for (int64_t u = 0; u < p.bucket_sizes[i]; ++u) {
      acc += p.numels[pos + u];
      cacc += p.costs[pos + u];
      p.phi.push_back(acc);
      p.cphi.push_back(cacc);
    }
    pos += p.bucket_sizes[i];
  }
  p.bucket_first[p.n_buckets] = pos;
  p.phi_first[p.n_buckets] = (int64_t)p.phi.size();
}

// Owner per parameter, rank loads, elem cuts and metrics from param_cuts.
void finish(Plan& p) {
  const int32_t R = p.R;
  p.owner.assign(p.n_params, 0);
  p.rank_load.assign(R, 0);
  p.rank_elems.assign(R, 0);
  p.elem_cuts.assign(p.n_buckets * (R + 1), 0);
  for (int64_t i = 0; i < p.n_buckets; ++i) {
    const int64_t* s = &p.param_cuts[i * (R + 1)];
    const int64_t* phi = &p.phi[p.phi_first[i]];
    const int64_t base = p.bucket_first[i];
    for (int32_t r = 0; r < R; ++r) {
      for (int64_t u = s[r]; u < s[r + 1]; ++u) {
        p.owner[base + u] = r;
        p.rank_load[r] += p.costs[base + u];
        p.rank_elems[r] += p.numels[base + u];
      }
    }
    for (int32_t r = 0; r <= R; ++r) p.elem_cuts[i * (R + 1) + r] = phi[s[r]];
  }
  // metrics, in the reference planner's order
  int64_t total = 0;
  for (int32_t r = 0; r < R; ++r) total += p.rank_load[r];
  const double mu = (double)total / (double)R;
  int64_t mx = 0;
  for (int32_t r = 0; r < R; ++r) mx = std::max(mx, p.rank_load[r]);
  p.r_lb = total > 0 ? (double)mx / mu : 1.0;
  double jdp = 0.0;
  for (int32_t r = 0; r < R; ++r) jdp = std::max(jdp, std::fabs((double)p.rank_load[r] - mu));
  p.j_dp = jdp;
  double jc = 0.0;
  for (int64_t i = 0; i < p.n_buckets; ++i) {
    const int64_t* ec = &p.elem_cuts[i * (R + 1)];
    const int64_t size = ec[R];
    for (int32_t r = 0; r < R; ++r)
      jc += std::fabs((double)(ec[r + 1] - ec[r]) - (double)size / (double)R);
  }
  p.j_comm = jc;
}

Plan* new_plan(const int64_t* numels, int64_t n_params, const int64_t* bucket_sizes,
               int64_t n_buckets, int32_t R, const int64_t* costs = nullptr) {
  Plan* p = new (std::nothrow) Plan();
  if (!p) return nullptr;
  p->R = R;
  p->n_params = n_params;
  p->n_buckets = n_buckets;
  p->numels.assign(numels, numels + n_params);
  if (costs) p->costs.assign(costs, costs + n_params);
  else p->costs = p->numels;
  p->bucket_sizes.assign(bucket_sizes, bucket_sizes + n_buckets);
  build_prefix(*p);
  p->param_cuts.assign(n_buckets * (R + 1), 0);
  return p;
}

}  // namespace

extern "C" {

int cz_make_buckets(const int64_t* numels, int64_t n_params, int64_t cap_elems,
                    int64_t* counts_out, int64_t* n_buckets_out) {
  if (!numels || !counts_out || !n_buckets_out || n_params <= 0 || cap_elems <= 0)
    return CZ_ERR_INVALID;
  int64_t nb = 0, cur_n = 0, cur_el = 0;
  for (int64_t i = 0; i < n_params; ++i) {
    if (numels[i] <= 0) return CZ_ERR_INVALID;
    cur_n += 1;
    cur_el += numels[i];
    if (cur_el >= cap_elems) {
      counts_out[nb++] = cur_n;
      cur_n = 0;
      cur_el = 0;
    }
  }
  if (cur_n) counts_out[nb++] = cur_n;
  *n_buckets_out = nb;
  return CZ_OK;
}

int cz_plan_naive(const int64_t* numels, int64_t n_params, const int64_t* bucket_sizes,
                  int64_t n_buckets, int32_t R, cz_plan** out) {
  if (!out) return CZ_ERR_INVALID;
  *out = nullptr;
  cz::NvtxRange range("cz/plan_naive");
  int st = check_inputs(numels, n_params, bucket_sizes, n_buckets, R);
  if (st != CZ_OK) return st;
  Plan* p = new_plan(numels, n_params, bucket_sizes, n_buckets, R);
  if (!p) return CZ_ERR_NOMEM;
  p->kind = 1;
  p->alpha = 0.0;
  for (int64_t i = 0; i < n_buckets; ++i) {
    const int64_t nb = bucket_sizes[i];
    const int64_t* phi = &p->phi[p->phi_first[i]];
    const int64_t size = phi[nb];
    int64_t* s = &p->param_cuts[i * (R + 1)];
    // owner(u) = floor(phi[u] * R / size) is non-decreasing in u; s_r = first u with owner >= r.
    // phi[u] * R stays exact: both fit in int64 for any buffer below 2^63 / R elements.
    int64_t u = 0;
    s[0] = 0;
    for (int32_t r = 1; r < R; ++r) {
      while (u < nb && (phi[u] * (int64_t)R) / size < r) ++u;
      s[r] = u;
    }
    s[R] = nb;
  }
  finish(*p);
  *out = p;
  return CZ_OK;
}

int cz_plan_partition(const int64_t* numels, int64_t n_params, const int64_t* bucket_sizes,
                      int64_t n_buckets, int32_t R, double alpha, cz_plan** out) {
  return cz_plan_partition_cost(numels, nullptr, n_params, bucket_sizes, n_buckets, R, alpha, out);
}

int cz_plan_partition_cost(const int64_t* numels, const int64_t* costs, int64_t n_params,
                           const int64_t* bucket_sizes, int64_t n_buckets, int32_t R, double alpha,
                           cz_plan** out) {
  if (!out) return CZ_ERR_INVALID;
  *out = nullptr;
  cz::NvtxRange range("cz/plan_partition");
  int st = check_inputs(numels, n_params, bucket_sizes, n_buckets, R, costs);
  if (st != CZ_OK) return st;
  if (!(alpha >= 0.0 && alpha <= 1.0)) return CZ_ERR_INVALID;
  Plan* p = new_plan(numels, n_params, bucket_sizes, n_buckets, R, costs);
  if (!p) return CZ_ERR_NOMEM;
  p->kind = 0;
  p->alpha = alpha;

  std::vector<int64_t> Wb(n_buckets);
  int64_t total = 0;
  for (int64_t i = 0; i < n_buckets; ++i) {
    Wb[i] = p->cphi[p->phi_first[i] + bucket_sizes[i]];
    total += Wb[i];
  }
  const double mu = (double)total / (double)R;
  std::vector<int64_t> order(n_buckets);
  std::iota(order.begin(), order.end(), 0);
  std::sort(order.begin(), order.end(), [&](int64_t x, int64_t y) {
    if (Wb[x] != Wb[y]) return Wb[x] > Wb[y];
    return x < y;
  });

  std::vector<double> L(R, 0.0), d(R), t(R);
  for (int64_t k : order) {
    const int64_t nk = bucket_sizes[k];
    const int64_t* phi = &p->cphi[p->phi_first[k]];   // Phi_k(u) in cost units
    // step 1: deficits at the start of this bucket
    double D = 0.0;
    for (int32_t r = 0; r < R; ++r) {
      d[r] = std::max(0.0, mu - L[r]);
    }
    for (int32_t r = 0; r < R; ++r) D += d[r];
    // steps 2-3: blended target
    const double Wk = (double)Wb[k];
    for (int32_t r = 0; r < R; ++r) {
      double v;
      if (D > 0.0) {
        v = (1.0 - alpha) * (1.0 / (double)R) + alpha * (d[r] / D);
      } else {
        v = 1.0 / (double)R;
      }
      t[r] = Wk * v;
    }
    // step 4: atomic discretisation.  |Phi(u) - C| is non-increasing while
    // Phi(u) < C and non-decreasing once Phi(u) >= C (Phi strictly increasing),
    // so the first u with Phi(u) >= C ends the scan; a strict '<' keeps the
    // smaller u on ties.  Each scan starts at the previous cut: O(n_k + R).
    int64_t* s = &p->param_cuts[k * (R + 1)];
    s[0] = 0;
    double C = 0.0;
    for (int32_t r = 0; r + 1 < R; ++r) {
      C += t[r];
      int64_t best_u = s[r];
      double best = std::fabs((double)phi[best_u] - C);
      if ((double)phi[best_u] < C) {
        for (int64_t u = s[r] + 1; u <= nk; ++u) {
          const double dist = std::fabs((double)phi[u] - C);
          if (dist < best) {
            best = dist;
            best_u = u;
          }
          if ((double)phi[u] >= C) break;
        }
      }
      s[r + 1] = best_u;
      L[r] += (double)(phi[s[r + 1]] - phi[s[r]]);
    }
    s[R] = nk;
    L[R - 1] += (double)(phi[s[R]] - phi[s[R - 1]]);
  }
  finish(*p);
  *out = p;
  return CZ_OK;
}

void cz_plan_free(cz_plan* plan) { delete static_cast<Plan*>(plan); }

int cz_plan_info(const cz_plan* plan, int64_t* n_params, int64_t* n_buckets, int32_t* R) {
  if (!plan) return CZ_ERR_INVALID;
  const Plan* p = static_cast<const Plan*>(plan);
  if (n_params) *n_params = p->n_params;
  if (n_buckets) *n_buckets = p->n_buckets;
  if (R) *R = p->R;
  return CZ_OK;
}

int cz_plan_owner(const cz_plan* plan, int32_t* owner_out) {
  if (!plan || !owner_out) return CZ_ERR_INVALID;
  const Plan* p = static_cast<const Plan*>(plan);
  std::copy(p->owner.begin(), p->owner.end(), owner_out);
  return CZ_OK;
}

int cz_plan_cuts(const cz_plan* plan, int64_t* param_cuts, int64_t* elem_cuts) {
  if (!plan) return CZ_ERR_INVALID;
  const Plan* p = static_cast<const Plan*>(plan);
  if (param_cuts) std::copy(p->param_cuts.begin(), p->param_cuts.end(), param_cuts);
  if (elem_cuts) std::copy(p->elem_cuts.begin(), p->elem_cuts.end(), elem_cuts);
  return CZ_OK;
}

int cz_plan_rank_load(const cz_plan* plan, int64_t* load_out) {
  if (!plan || !load_out) return CZ_ERR_INVALID;
  const Plan* p = static_cast<const Plan*>(plan);
  std::copy(p->rank_load.begin(), p->rank_load.end(), load_out);
  return CZ_OK;
}

int cz_plan_rank_elems(const cz_plan* plan, int64_t* elems_out) {
  if (!plan || !elems_out) return CZ_ERR_INVALID;
  const Plan* p = static_cast<const Plan*>(plan);
  std::copy(p->rank_elems.begin(), p->rank_elems.end(), elems_out);
  return CZ_OK;
}

int cz_plan_metrics(const cz_plan* plan, double* r_lb, double* j_dp, double* j_comm) {
  if (!plan) return CZ_ERR_INVALID;
  const Plan* p = static_cast<const Plan*>(plan);
  if (r_lb) *r_lb = p->r_lb;
  if (j_dp) *j_dp = p->j_dp;
  if (j_comm) *j_comm = p->j_comm;
  return CZ_OK;
}

}  // extern "C"
