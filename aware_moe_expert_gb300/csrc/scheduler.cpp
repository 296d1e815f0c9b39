// Quality-tiered batching of requests with per-request routing budgets, on
// the host.  "MoE-Prism: Model and System Support for Request-Level Compute
// Elasticity in MoE Serving" (arXiv 2510.19366), §III-C2 "Temporal Separation
// via Quality-Tiered Batching", Eq. (5).
//
// A dispatch that runs every request of a batch at one budget (the batch
// maximum) over-serves its low-budget requests.  The queue is sorted by
// (k, arrival) and scanned tier by tier; batches are filled in FIFO order up
// to a token budget M.  When a tier leaves a residual batch (n_cur tokens at
// budget k), the next tier's leading requests that still fit contribute
// n_next tokens, and the residual is promoted to that tier's budget k_next and
// merged iff
//     (n_cur + n_next) / T(n_cur + n_next, k_next) >= n_cur / T(n_cur, k),
// T(n, k) being the layer time profiled at token and budget buckets and
// interpolated between them.  Otherwise the residual is dispatched at k.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "../../include/moe.h"

namespace {

// Piecewise-linear interpolation of y over the increasing points xs, with the
// end segments extended linearly; a single point scales proportionally.
double interp(const int32_t* xs, const double* ys, int n, double x) {
  if (n == 1) return xs[0] != 0 ? ys[0] * x / xs[0] : ys[0];
  int i = 0;
  while (i + 2 < n && x > xs[i + 1]) ++i;
  const double x0 = xs[i], x1 = xs[i + 1];
  const double f = (x - x0) / (x1 - x0);
  return ys[i] + f * (ys[i + 1] - ys[i]);
}

bool table_ok(const moe_cost_table* t) {
  if (t == nullptr || t->n_count < 1 || t->k_count < 1 || t->n_points == nullptr ||
      t->k_points == nullptr || t->t_us == nullptr)
    return false;
  for (int i = 0; i + 1 < t->n_count; ++i)
    if (t->n_points[i] >= t->n_points[i + 1]) return false;
  for (int i = 0; i + 1 < t->k_count; ++i)
    if (t->k_points[i] >= t->k_points[i + 1]) return false;
  for (int i = 0; i < t->n_count * t->k_count; ++i)
    if (!(t->t_us[i] > 0.0)) return false;   // times are positive (NaN fails too)
  return true;
}

struct Batch {
  std::vector<int32_t> reqs;   // original request indices, in dispatch order
  long long tokens = 0;
  int32_t k = 0;
};

}  // namespace

extern "C" {

double moe_cost_lookup(const moe_cost_table* t, double n, double k) {
  if (!table_ok(t)) return -1.0;
  // clamp k into the profiled budgets; interpolate in k between the two
  // neighbouring rows, each interpolated in n
  const double kk = std::min<double>(std::max<double>(k, t->k_points[0]),
                                     t->k_points[t->k_count - 1]);
  int j = 0;
  while (j + 1 < t->k_count && kk > t->k_points[j + 1]) ++j;
  const double y0 = interp(t->n_points, t->t_us + static_cast<size_t>(j) * t->n_count,
                           t->n_count, n);
  if (j + 1 >= t->k_count || kk == t->k_points[j]) return y0;
  const double y1 = interp(t->n_points, t->t_us + static_cast<size_t>(j + 1) * t->n_count,
                           t->n_count, n);
  const double f = (kk - t->k_points[j]) / (t->k_points[j + 1] - t->k_points[j]);
  return y0 + f * (y1 - y0);
}

int32_t moe_tier_schedule(const moe_tier_request* reqs, int32_t n_req, int32_t M,
                          const moe_cost_table* table, int32_t* batch_of, int32_t* batch_k,
                          int32_t* batch_tokens, int32_t max_batches) {
  if (n_req < 0 || M < 1 || !table_ok(table) || (n_req > 0 && (reqs == nullptr ||
                                                              batch_of == nullptr)))
    return -1;
  for (int i = 0; i < n_req; ++i)
    if (reqs[i].n_tokens < 1) return -1;
  std::vector<int32_t> order(static_cast<size_t>(n_req));
  for (int i = 0; i < n_req; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [reqs](int32_t a, int32_t b) {
    if (reqs[a].k != reqs[b].k) return reqs[a].k < reqs[b].k;
    return reqs[a].arrival < reqs[b].arrival;
  });
  std::vector<Batch> out;
  Batch cur;                 // the open batch (residual between tiers)
  bool open = false;
  size_t i = 0;
  while (i < order.size()) {
    const int32_t k = reqs[order[i]].k;
    size_t end = i;
    while (end < order.size() && reqs[order[end]].k == k) ++end;   // this tier: [i, end)
    if (open) {
      // residual of the previous tier: promote to k and merge, or dispatch
      long long n_next = 0;
      size_t take = i;
      while (take < end && cur.tokens + n_next + reqs[order[take]].n_tokens <= M) {
        n_next += reqs[order[take]].n_tokens;
        ++take;
      }
      const double n_cur = static_cast<double>(cur.tokens);
      const double lhs = (n_cur + n_next) / moe_cost_lookup(table, n_cur + n_next, k);
      const double rhs = n_cur / moe_cost_lookup(table, n_cur, cur.k);
      if (take > i && lhs >= rhs) {
        cur.k = k;
        for (size_t q = i; q < take; ++q) {
          cur.reqs.push_back(order[q]);
          cur.tokens += reqs[order[q]].n_tokens;
        }
        i = take;
      } else {
        out.push_back(cur);
        cur = Batch();
        open = false;
      }
    }
    // fill batches of this tier in FIFO order
    for (; i < end; ++i) {
      const int32_t r = order[i];
      if (open && cur.tokens + reqs[r].n_tokens > M) {
        out.push_back(cur);
        cur = Batch();
        open = false;
      }
      if (!open) {
        cur.k = k;
        open = true;
      }
      cur.reqs.push_back(r);
      cur.tokens += reqs[r].n_tokens;
    }
  }
  if (open) out.push_back(cur);
  if (static_cast<int32_t>(out.size()) > max_batches) return -2;
  for (size_t b = 0; b < out.size(); ++b) {
    for (int32_t r : out[b].reqs) batch_of[r] = static_cast<int32_t>(b);
    if (batch_k != nullptr) batch_k[b] = out[b].k;
    if (batch_tokens != nullptr) batch_tokens[b] = static_cast<int32_t>(out[b].tokens);
  }
  return static_cast<int32_t>(out.size());
}

}  // extern "C"
