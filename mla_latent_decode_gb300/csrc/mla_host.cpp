// mla_host.cpp -- host side of the MLA decode C ABI: error state, the split
// planners, the page-table check and the argument checks shared by the
// launches.  Page citations use the tags defined in include/mla_decode.h.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <functional>
#include <queue>
#include <vector>

#include "mla_internal.h"

namespace mla {

std::string& last_error() {
  static thread_local std::string msg;
  return msg;
}

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  last_error() = buf;
  return code;
}

int check_decode_args(const DecodeArgs& a) {
  if (!a.q_nope || !a.q_rope || !a.kv || !a.req_to_token || !a.seq_lens ||
      !a.O_part || !a.LSE_part)
    return fail(MLA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (a.B < 1 || a.q_len < 1 || a.H < 1 || a.num_shards < 1 ||
      a.num_splits < 1)
    return fail(MLA_ERR_INVALID_ARG,
                "B=%d q_len=%d H=%d num_shards=%d num_splits=%d must be >= 1",
                a.B, a.q_len, a.H, a.num_shards, a.num_splits);
  if (a.num_splits > 4096 || a.num_shards > 64)
    return fail(MLA_ERR_INVALID_ARG, "num_splits %d > 4096 or num_shards %d > 64",
                a.num_splits, a.num_shards);
  const int64_t rows = (int64_t)a.B * a.q_len * a.H;
  if (rows * a.num_shards * a.num_splits > (int64_t)1 << 31)
    return fail(MLA_ERR_INVALID_ARG, "too many output rows");
  if (a.page_size != MLA_PAGE_SIZE)
    return fail(MLA_ERR_UNSUPPORTED, "page_size %d: only %d is built",
                a.page_size, MLA_PAGE_SIZE);
  if (a.kv_dtype != MLA_KV_BF16 && a.kv_dtype != MLA_KV_FP8_E4M3)
    return fail(MLA_ERR_INVALID_ARG, "unknown kv_dtype %d", (int)a.kv_dtype);
  if (a.kv_dtype == MLA_KV_FP8_E4M3 && !a.kv_scale)
    return fail(MLA_ERR_INVALID_ARG, "FP8 KV needs kv_scale");
  if (a.num_slots < a.page_size || a.num_slots > ((int64_t)1 << 31) - 1)
    return fail(MLA_ERR_INVALID_ARG, "num_slots %lld out of range",
                (long long)a.num_slots);
  if (a.r2t_stride < 1)
    return fail(MLA_ERR_INVALID_ARG, "r2t_stride %lld < 1",
                (long long)a.r2t_stride);
  if (!std::isfinite(a.sm_scale) || !(a.sm_scale > 0.f))
    return fail(MLA_ERR_INVALID_ARG, "sm_scale %g is not a positive number",
                (double)a.sm_scale);
  if (!aligned(a.q_nope, 16) || !aligned(a.q_rope, 16) || !aligned(a.kv, 16) ||
      !aligned(a.O_part, 16) || !aligned(a.LSE_part, 4) ||
      !aligned(a.req_to_token, 4) || !aligned(a.seq_lens, 4) ||
      (a.kv_limit && !aligned(a.kv_limit, 4)) ||
      (a.kv_scale && !aligned(a.kv_scale, 16)) ||
      (a.status && !aligned(a.status, 4)) ||
      (a.split_pages && !aligned(a.split_pages, 4)))
    return fail(MLA_ERR_MISALIGNED,
                "q/kv/kv_scale/O_part need 16-B alignment, the other arrays 4-B");
  return MLA_OK;
}

int check_work(const DecodeArgs& a) {
  if (!a.work) {
    if (a.num_work != 0)
      return fail(MLA_ERR_INVALID_ARG, "num_work %d without a work list", a.num_work);
    return MLA_OK;
  }
  const int R = a.kv_dtype == MLA_KV_FP8_E4M3 ? MLA_ROWS_PER_UNIT / 2
                                             : MLA_ROWS_PER_UNIT;
  const int64_t U = ((int64_t)a.q_len * a.H + R - 1) / R;
  const int64_t n = (int64_t)a.B * a.num_shards * a.num_splits * U;
  if (a.num_work != n)
    return fail(MLA_ERR_INVALID_ARG, "num_work %d: the launch has %lld work units",
                a.num_work, (long long)n);
  if (!aligned(a.work, 4))
    return fail(MLA_ERR_MISALIGNED, "work needs 4-B alignment");
  return MLA_OK;
}

// Default cost constants of the planners, in units of one page of one work
// unit (about 0.9 us on a GB300): a work unit's fixed cost (launch, Q load,
// pipeline fill and drain, O_part write, wave hand-over) and the price of one
// more split per 1024 query rows (partial outputs written and re-read by the
// combine).  The split price and the FP8 unit cost were fitted to the
// kernels' measured times over B = 1..24 requests x {100k, 400k} tokens x
// {1, 2, 3, 4, 6, 9, 18} splits; the BF16 unit cost was refitted once its
// query load and epilogue shrank (a unit's fixed time fell from about 20 to
// about 8 us): every value from 8 to 24 then gives the fastest measured plan
// on the sweep at 100k, dp16 and DCP, and 16 sits in the middle.
constexpr double kPlanUnitCostBf16 = 16.0;
constexpr double kPlanUnitCostFp8 = 32.0;
constexpr double kPlanSplitCost = 1.0;

static double plan_unit_cost(mla_kv_dtype kv_dtype) {
  return kv_dtype == MLA_KV_FP8_E4M3 ? kPlanUnitCostFp8 : kPlanUnitCostBf16;
}

// The planners score each candidate plan by its list-scheduling makespan
// plus a price per split, and keep the first candidate that beats the best
// score so far by more than 1e-9.  A candidate whose makespan is known to
// reach `cutoff` = best score - its split price (+ a relative margin far above
// rounding) cannot win, so its schedule stops there: the chosen plan is the
// one the full search gives.  A list schedule on m slots never ends before
// max(total cost / m, largest unit cost), which prunes most candidates before
// any scheduling.
static double prune_cutoff(bool have_best, double best_score, double price) {
  if (!have_best) return INFINITY;
  return best_score - price + 1e-7 * std::max(1.0, std::fabs(best_score));
}

// List-scheduling makespan of units in launch order on `slots` slots, or
// INFINITY once it is known to reach `cutoff`.
static double makespan(const std::vector<double>& costs, int slots,
                       double cutoff) {
  if (costs.empty()) return 0.0;
  std::priority_queue<double, std::vector<double>, std::greater<double>> heap;
  const size_t n = std::min<size_t>((size_t)slots, costs.size());
  for (size_t k = 0; k < n; ++k) heap.push(0.0);
  double end = 0.0;
  for (double c : costs) {
    double t = heap.top() + c;
    heap.pop();
    end = std::max(end, t);
    if (end >= cutoff) return INFINITY;
    heap.push(t);
  }
  return end;
}

}  // namespace mla

using namespace mla;

extern "C" {

const char* mla_last_error_string(void) { return last_error().c_str(); }

int mla_num_sms(int device) {
  int n = 0;
  cudaError_t e =
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
  return n;
}

// [K3-MLA]: split = min(148 // B // (q_len * 2), 32), floored at 1.
int mla_plan_heuristic(int B, int q_len) {
  if (B < 1 || q_len < 1)
    return fail(MLA_ERR_INVALID_ARG, "B and q_len must be >= 1");
  return std::max(1, std::min(148 / B / (q_len * 2), 32));
}

int mla_plan_ex(int V, int q_len, int H, int rows_per_unit,
                const int32_t* seq_lens_host, int slots, int s_max, double c0,
                double lam, int* num_splits_out, float* wave_eff_out,
                double* makespan_out) {
  if (V < 1 || q_len < 1 || H < 1 || !seq_lens_host || !num_splits_out)
    return fail(MLA_ERR_INVALID_ARG, "bad planner arguments");
  if (rows_per_unit < 1 || slots < 1 || s_max < 1 || s_max > 1024 ||
      !(c0 >= 0) || !(lam >= 0))
    return fail(MLA_ERR_INVALID_ARG,
                "rows_per_unit/slots/s_max/c0/lam out of range");
  const int G = (H * q_len + rows_per_unit - 1) / rows_per_unit;
  const double rows = (double)V * q_len * H;
  double bestJ = 0, bestEff = 0, bestMs = 0;
  int bestS = 0;
  int64_t sumP = 0, maxP = 0;
  for (int v = 0; v < V; ++v) {
    const int64_t L = std::max<int32_t>(seq_lens_host[v], 0);
    const int64_t P = (L + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE;
    sumP += P;
    maxP = std::max(maxP, P);
  }
  std::vector<double> costs;
  for (int S = 1; S <= s_max; ++S) {
    const double price = lam * S * rows / 1024.0;
    const double cutoff = prune_cutoff(bestS != 0, bestJ, price);
    // Every part costs its pages + c0 and a request's parts hold all its
    // pages, the largest ceil(P / S): the bound needs no cost list.
    const double total_lb = (double)G * ((double)sumP + (double)V * S * c0);
    const double cmax_lb = (double)((maxP + S - 1) / S) + c0;
    if (std::max(total_lb / slots, cmax_lb) >= cutoff) continue;
    costs.clear();
    double total = 0, cmax = 0;
    for (int s = 0; s < S; ++s) {
      for (int v = 0; v < V; ++v) {
        const int64_t L = std::max<int32_t>(seq_lens_host[v], 0);
        const int64_t P = (L + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE;
        const double c = (double)((s + 1) * P / S - s * P / S) + c0;
        cmax = std::max(cmax, c);
        for (int g = 0; g < G; ++g) {
          costs.push_back(c);
          total += c;
        }
      }
    }
    if (std::max(total / slots, cmax) >= cutoff) continue;
    const double ms = makespan(costs, slots, cutoff);
    if (ms == INFINITY) continue;
    const double J = ms + price;
    if (bestS == 0 || J < bestJ - 1e-9) {
      bestJ = J;
      bestS = S;
      bestMs = ms;
      bestEff = ms > 0 ? total / ((double)slots * ms) : 1.0;
    }
  }
  *num_splits_out = bestS;
  if (wave_eff_out) *wave_eff_out = (float)bestEff;
  if (makespan_out) *makespan_out = bestMs;
  return MLA_OK;
}

int mla_plan(int B, int q_len, int H, int num_shards, mla_kv_dtype kv_dtype,
             const int32_t* seq_lens_host, int num_sms, int* num_splits_out,
             float* wave_eff_out) {
  if (B < 1 || num_shards < 1)
    return fail(MLA_ERR_INVALID_ARG, "B and num_shards must be >= 1");
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3)
    return fail(MLA_ERR_INVALID_ARG, "unknown kv_dtype %d", (int)kv_dtype);
  // BF16: 256 query rows per 4-CTA cluster; E4M3: 128 rows per 2-CTA cluster.
  const bool fp8 = kv_dtype == MLA_KV_FP8_E4M3;
  const int ctas = fp8 ? 2 : 4;
  int slots;
  if (num_sms > 0) {
    slots = std::max(1, num_sms / ctas);
  } else {
    slots = fp8 ? pair_slots_fp8() : mla_cluster_slots();
    if (slots < 0) return slots;
    if (slots == 0) return fail(MLA_ERR_CUDA, "no decode cluster fits on this device");
  }
  return mla_plan_ex(B * num_shards, q_len, H,
                     fp8 ? MLA_ROWS_PER_UNIT / 2 : MLA_ROWS_PER_UNIT,
                     seq_lens_host, slots, 64, plan_unit_cost(kv_dtype), kPlanSplitCost,
                     num_splits_out, wave_eff_out, nullptr);
}

// One split schedule (boundaries bnd[v * (S + 1) + k]): its work units, each
// (part s, request v, row unit u) costing its pages + c0 (an empty one
// c_empty), are list-scheduled on `slots` in launch order, which is by
// increasing id (s * V + v) * U + u (part-major), or with `lpt` longest first
// (equal costs by increasing id).  Returns the makespan, adds the unit costs
// to *total and, when `order` is given, stores the ids in launch order.
// Returns INFINITY (and no order) once the makespan is known to reach
// `cutoff`.
static double schedule_makespan(const std::vector<int64_t>& P, int U, int S,
                                const std::vector<int64_t>& bnd, int slots,
                                double c0, double c_empty, bool lpt,
                                double* total, std::vector<int32_t>* order,
                                double cutoff = INFINITY) {
  const size_t V = P.size();
  // the U units of one (s, v) share its cost and have consecutive ids
  std::vector<std::pair<double, int64_t>> groups;
  groups.reserve(V * (size_t)S);
  double lower = 0, cmax = 0;
  for (int s = 0; s < S; ++s)
    for (size_t v = 0; v < V; ++v) {
      const int64_t pages = bnd[v * (S + 1) + s + 1] - bnd[v * (S + 1) + s];
      const double c = pages > 0 ? (double)pages + c0 : c_empty;
      groups.emplace_back(c, (int64_t)s * (int64_t)V + (int64_t)v);
      lower += c * U;
      cmax = std::max(cmax, c);
    }
  if (std::max(lower / slots, cmax) >= cutoff) return INFINITY;
  if (lpt)
    std::stable_sort(groups.begin(), groups.end(),
                     [](const std::pair<double, int64_t>& a,
                        const std::pair<double, int64_t>& b) {
                       return a.first > b.first;
                     });
  std::priority_queue<double, std::vector<double>, std::greater<double>> heap;
  const size_t n = std::min<size_t>((size_t)slots, V * (size_t)S * (size_t)U);
  for (size_t k = 0; k < n; ++k) heap.push(0.0);
  double end = 0.0, tot = 0.0;
  if (order) order->clear();
  for (const auto& g : groups)
    for (int u = 0; u < U; ++u) {
      const double t = heap.top() + g.first;
      heap.pop();
      end = std::max(end, t);
      if (end >= cutoff) return INFINITY;
      heap.push(t);
      tot += g.first;
      if (order) order->push_back((int32_t)(g.second * U + u));
    }
  *total = tot;
  return end;
}

// The candidate families of the parts planner (uniform deals, capped first
// part, equal chunks), scored by the schedule's makespan + lam * S * rows /
// 1024 in launch order or longest first; the first of equal scores wins.
struct PartsPlan {
  int S = 0;
  std::vector<int64_t> bnd;
  double makespan = 0, total = 0;
};

static int plan_parts_impl(int V, int q_len, int H, int rows_per_unit,
                           const int32_t* seq_lens_host, int slots, int s_max,
                           int max_parts, double c0, double lam, bool lpt,
                           PartsPlan* best_out) {
  if (V < 1 || q_len < 1 || H < 1 || !seq_lens_host)
    return fail(MLA_ERR_INVALID_ARG, "bad planner arguments");
  if (rows_per_unit < 1 || slots < 1 || s_max < 1 || s_max > 1024 ||
      max_parts < 1 || max_parts > s_max || !(c0 >= 0) || !(lam >= 0))
    return fail(MLA_ERR_INVALID_ARG,
                "rows_per_unit/slots/s_max/max_parts/c0/lam out of range");
  const int U = (H * q_len + rows_per_unit - 1) / rows_per_unit;
  const double rows = (double)V * q_len * H;
  std::vector<int64_t> P(V);
  int64_t Pmax = 0;
  for (int v = 0; v < V; ++v) {
    const int64_t L = std::max<int32_t>(seq_lens_host[v], 0);
    P[v] = (L + MLA_PAGE_SIZE - 1) / MLA_PAGE_SIZE;
    Pmax = std::max(Pmax, P[v]);
  }
  constexpr int kCaps = 32;
  constexpr double kEmpty = 1.0;
  double bestJ = 0;
  PartsPlan& best = *best_out;
  best = PartsPlan();
  std::vector<int64_t> bnd;
  auto consider = [&](int S) {
    double tot = 0;
    const double price = lam * S * rows / 1024.0;
    const double ms =
        schedule_makespan(P, U, S, bnd, slots, c0, kEmpty, lpt, &tot, nullptr,
                          prune_cutoff(best.S != 0, bestJ, price));
    if (ms == INFINITY) return;
    const double J = ms + price;
    if (best.S == 0 || J < bestJ - 1e-9) {
      bestJ = J;
      best.S = S;
      best.makespan = ms;
      best.total = tot;
      best.bnd = bnd;
    }
  };
  // Uniform deals.  Request v's S parts hold its P pages, min(P, S) of them
  // non-empty and none above ceil(P / S): the schedule's lower bound comes
  // before any boundary is written.
  for (int S = 1; S <= s_max; ++S) {
    if (best.S != 0) {
      double lower = 0, cmax = 0;
      for (int v = 0; v < V; ++v) {
        const int64_t full = std::min<int64_t>(P[v], S);
        lower += (double)P[v] + c0 * full + kEmpty * (S - full);
        if (P[v] > 0) cmax = std::max(cmax, (double)((P[v] + S - 1) / S) + c0);
        if (full < S) cmax = std::max(cmax, kEmpty);
      }
      lower *= U;
      if (std::max(lower / slots, cmax) >=
          prune_cutoff(true, bestJ, lam * S * rows / 1024.0))
        continue;
    }
    bnd.assign((size_t)V * (S + 1), 0);
    for (int v = 0; v < V; ++v)
      for (int k = 0; k <= S; ++k) bnd[(size_t)v * (S + 1) + k] = k * P[v] / S;
    consider(S);
  }
  // First part capped at b pages, the rest dealt over S - 1 parts.
  for (int S = 2; S <= max_parts; ++S) {
    int64_t prev = -1;
    for (int k = 1; k <= kCaps; ++k) {
      const int64_t b = (Pmax * k + kCaps - 1) / kCaps;
      if (b == prev || b < 1) continue;
      prev = b;
      if (best.S != 0) {
        // The first part holds min(P, b) pages, the other S - 1 parts the
        // rest, min(rest, S - 1) of them non-empty, none above
        // ceil(rest / (S - 1)).
        double lower = 0, cmax = 0;
        for (int v = 0; v < V; ++v) {
          const int64_t first = std::min(P[v], b), rest = P[v] - first;
          const int64_t full = std::min<int64_t>(rest, S - 1);
          lower += (double)P[v] + c0 * ((first > 0) + full) +
                   kEmpty * ((first == 0) + (S - 1 - full));
          cmax = std::max(cmax, first > 0 ? (double)first + c0 : kEmpty);
          if (rest > 0)
            cmax = std::max(cmax, (double)((rest + S - 2) / (S - 1)) + c0);
          if (full < S - 1) cmax = std::max(cmax, kEmpty);
        }
        lower *= U;
        if (std::max(lower / slots, cmax) >=
            prune_cutoff(true, bestJ, lam * S * rows / 1024.0))
          continue;
      }
      bnd.assign((size_t)V * (S + 1), 0);
      for (int v = 0; v < V; ++v) {
        const int64_t first = std::min(P[v], b), rest = P[v] - first;
        int64_t* row = &bnd[(size_t)v * (S + 1)];
        row[0] = 0;
        for (int m = 1; m <= S; ++m) row[m] = first + (m - 1) * rest / (S - 1);
      }
      consider(S);
    }
  }
  // Equal chunks: parts of u = ceil(Pmax / S) pages in token order, so the
  // longest request has S full parts and a shorter one fewer (the rest
  // empty): every non-empty unit but a request's last carries u pages.
  for (int S = 2; S <= max_parts; ++S) {
    const int64_t u = (Pmax + S - 1) / S;
    if (u < 1) continue;
    bnd.assign((size_t)V * (S + 1), 0);
    for (int v = 0; v < V; ++v) {
      int64_t* row = &bnd[(size_t)v * (S + 1)];
      for (int m = 0; m <= S; ++m) row[m] = std::min(P[v], (int64_t)m * u);
    }
    consider(S);
  }
  return MLA_OK;
}

// Cluster slots of the kernel that serves kv_dtype (num_sms > 0: that many
// SMs divided by the cluster size instead of asking the device).
static int decode_slots(mla_kv_dtype kv_dtype, int num_sms) {
  const bool fp8 = kv_dtype == MLA_KV_FP8_E4M3;
  const int ctas = fp8 ? 2 : 4;
  if (num_sms > 0) return std::max(1, num_sms / ctas);
  const int slots = fp8 ? pair_slots_fp8() : mla_cluster_slots();
  if (slots == 0) return fail(MLA_ERR_CUDA, "no decode cluster fits on this device");
  return slots;
}

int mla_plan_parts_ex(int V, int q_len, int H, int rows_per_unit,
                      const int32_t* seq_lens_host, int slots, int s_max,
                      int max_parts, double c0, double lam,
                      int32_t* split_pages_out, int* num_parts_out,
                      float* wave_eff_out, double* makespan_out) {
  if (!split_pages_out || !num_parts_out)
    return fail(MLA_ERR_INVALID_ARG, "bad planner arguments");
  PartsPlan best;
  const int rc = plan_parts_impl(V, q_len, H, rows_per_unit, seq_lens_host,
                                 slots, s_max, max_parts, c0, lam, false, &best);
  if (rc != MLA_OK) return rc;
  for (size_t i = 0; i < best.bnd.size(); ++i)
    split_pages_out[i] = (int32_t)best.bnd[i];
  *num_parts_out = best.S;
  if (wave_eff_out)
    *wave_eff_out = best.makespan > 0
                        ? (float)(best.total / ((double)slots * best.makespan))
                        : 1.f;
  if (makespan_out) *makespan_out = best.makespan;
  return MLA_OK;
}

int mla_plan_sched_ex(int V, int q_len, int H, int rows_per_unit,
                      const int32_t* seq_lens_host, int slots, int s_max,
                      int max_parts, double c0, double lam,
                      int32_t* split_pages_out, int* num_parts_out,
                      int32_t* work_out, int64_t work_capacity,
                      int64_t* num_work_out, float* wave_eff_out,
                      double* makespan_out) {
  if (!split_pages_out || !num_parts_out || !work_out || !num_work_out)
    return fail(MLA_ERR_INVALID_ARG, "bad scheduler arguments");
  PartsPlan best;
  int rc = plan_parts_impl(V, q_len, H, rows_per_unit, seq_lens_host, slots,
                           s_max, max_parts, c0, lam, true, &best);
  if (rc != MLA_OK) return rc;
  const int U = (H * q_len + rows_per_unit - 1) / rows_per_unit;
  const int64_t n = (int64_t)V * best.S * U;
  if (n > work_capacity || n > 0x7fffffff)
    return fail(MLA_ERR_INVALID_ARG, "work list needs %lld entries, capacity %lld",
                (long long)n, (long long)work_capacity);
  std::vector<int64_t> P(V);
  for (int v = 0; v < V; ++v)
    P[v] = ((int64_t)std::max<int32_t>(seq_lens_host[v], 0) + MLA_PAGE_SIZE - 1) /
           MLA_PAGE_SIZE;
  std::vector<int32_t> order;
  double tot = 0;
  schedule_makespan(P, U, best.S, best.bnd, slots, c0, 1.0, true, &tot, &order);
  for (size_t i = 0; i < best.bnd.size(); ++i)
    split_pages_out[i] = (int32_t)best.bnd[i];
  for (int64_t i = 0; i < n; ++i) work_out[i] = order[(size_t)i];
  *num_parts_out = best.S;
  *num_work_out = n;
  if (wave_eff_out)
    *wave_eff_out = best.makespan > 0
                        ? (float)(best.total / ((double)slots * best.makespan))
                        : 1.f;
  if (makespan_out) *makespan_out = best.makespan;
  return MLA_OK;
}

int mla_plan_parts(int B, int q_len, int H, int num_shards,
                   mla_kv_dtype kv_dtype, const int32_t* seq_lens_host,
                   int num_sms, int max_parts, int32_t* split_pages_out,
                   int* num_parts_out, float* wave_eff_out) {
  if (B < 1 || num_shards < 1)
    return fail(MLA_ERR_INVALID_ARG, "B and num_shards must be >= 1");
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3)
    return fail(MLA_ERR_INVALID_ARG, "unknown kv_dtype %d", (int)kv_dtype);
  const int slots = decode_slots(kv_dtype, num_sms);
  if (slots < 0) return slots;
  return mla_plan_parts_ex(B * num_shards, q_len, H,
                           kv_dtype == MLA_KV_FP8_E4M3 ? MLA_ROWS_PER_UNIT / 2
                                                       : MLA_ROWS_PER_UNIT,
                           seq_lens_host, slots, 64, max_parts, plan_unit_cost(kv_dtype),
                           kPlanSplitCost, split_pages_out, num_parts_out,
                           wave_eff_out, nullptr);
}

int mla_plan_sched(int B, int q_len, int H, int num_shards,
                   mla_kv_dtype kv_dtype, const int32_t* seq_lens_host,
                   int num_sms, int max_parts, int32_t* split_pages_out,
                   int* num_parts_out, int32_t* work_out,
                   int64_t work_capacity, int64_t* num_work_out,
                   float* wave_eff_out) {
  if (B < 1 || num_shards < 1)
    return fail(MLA_ERR_INVALID_ARG, "B and num_shards must be >= 1");
  if (kv_dtype != MLA_KV_BF16 && kv_dtype != MLA_KV_FP8_E4M3)
    return fail(MLA_ERR_INVALID_ARG, "unknown kv_dtype %d", (int)kv_dtype);
  const int slots = decode_slots(kv_dtype, num_sms);
  if (slots < 0) return slots;
  return mla_plan_sched_ex(B * num_shards, q_len, H,
                           kv_dtype == MLA_KV_FP8_E4M3 ? MLA_ROWS_PER_UNIT / 2
                                                       : MLA_ROWS_PER_UNIT,
                           seq_lens_host, slots, 64, max_parts, plan_unit_cost(kv_dtype),
                           kPlanSplitCost, split_pages_out, num_parts_out,
                           work_out, work_capacity, num_work_out, wave_eff_out,
                           nullptr);
}

int mla_check_page_table(const int32_t* r2t, int64_t stride,
                         const int32_t* seq_lens, const int32_t* kv_limit,
                         int V, int q_len, int page_size, int64_t num_slots) {
  if (!r2t || !seq_lens || V < 1 || q_len < 1 || stride < 1 ||
      page_size < 1 || num_slots < 1)
    return fail(MLA_ERR_INVALID_ARG, "bad page-table check arguments");
  for (int v = 0; v < V; ++v) {
    const int64_t L = seq_lens[v];
    if (L < 0 || L > stride)
      return fail(MLA_ERR_PAGE_TABLE, "seq_lens[%d] = %lld outside [0, %lld]",
                  v, (long long)L, (long long)stride);
    if (!kv_limit && L < q_len)
      return fail(MLA_ERR_PAGE_TABLE, "seq_lens[%d] = %lld < q_len %d", v,
                  (long long)L, q_len);
    if (kv_limit)
      for (int i = 0; i < q_len; ++i) {
        const int32_t k = kv_limit[(int64_t)v * q_len + i];
        if (k < 0 || k > L)
          return fail(MLA_ERR_PAGE_TABLE, "kv_limit[%d,%d] = %d outside [0, %lld]",
                      v, i, k, (long long)L);
      }
    const int32_t* row = r2t + (int64_t)v * stride;
    for (int64_t t = 0; t < L; ++t) {
      const int64_t first = row[t - t % page_size];
      if (first % page_size != 0)
        return fail(MLA_ERR_PAGE_TABLE, "page of token %lld of request %d starts "
                    "at slot %lld, not a multiple of %d", (long long)t, v,
                    (long long)first, page_size);
      if (row[t] != first + t % page_size)
        return fail(MLA_ERR_PAGE_TABLE, "token %lld of request %d: slot %d is not "
                    "page-contiguous", (long long)t, v, row[t]);
      if (row[t] < 0 || row[t] >= num_slots)
        return fail(MLA_ERR_PAGE_TABLE, "token %lld of request %d: slot %d outside "
                    "[0, %lld)", (long long)t, v, row[t], (long long)num_slots);
    }
  }
  return MLA_OK;
}

int mla_decode_partial(const void* q_nope_absorbed, const void* q_rope,
                       const void* kv_pages, const float* kv_scale,
                       mla_kv_dtype kv_dtype, int64_t num_slots,
                       const int32_t* req_to_token, int64_t r2t_stride,
                       const int32_t* seq_lens, const int32_t* kv_limit, int B,
                       int q_len, int H, int num_shards, int page_size,
                       float sm_scale, int num_splits,
                       const int32_t* split_pages, const int32_t* work,
                       int num_work, float* O_part, float* LSE_part,
                       int* status, mla_stream_t stream) {
  DecodeArgs a{q_nope_absorbed, q_rope,    kv_pages, kv_scale,  kv_dtype,
               num_slots,       req_to_token, r2t_stride, seq_lens, kv_limit,
               B,               q_len,     H,        num_shards, page_size,
               sm_scale,        num_splits, split_pages, O_part,  LSE_part,  status,
               (cudaStream_t)stream};
  a.work = work;
  a.num_work = num_work;
  int rc = check_decode_args(a);
  if (rc != MLA_OK) return rc;
  rc = check_work(a);
  if (rc != MLA_OK) return rc;
  return launch_tc(a);
}

int mla_decode_partial_bf16_parts(
    const void* q_nope_absorbed, const void* q_rope, const void* kv_pages,
    const float* kv_scale, mla_kv_dtype kv_dtype, int64_t num_slots,
    const int32_t* req_to_token, int64_t r2t_stride, const int32_t* seq_lens,
    const int32_t* kv_limit, int B, int q_len, int H, int num_shards,
    int page_size, float sm_scale, int num_splits, const int32_t* split_pages,
    const int32_t* work, int num_work, void* O_part, float* LSE_part,
    int* status, mla_stream_t stream) {
  DecodeArgs a{q_nope_absorbed, q_rope,    kv_pages, kv_scale,  kv_dtype,
               num_slots,       req_to_token, r2t_stride, seq_lens, kv_limit,
               B,               q_len,     H,        num_shards, page_size,
               sm_scale,        num_splits, split_pages,
               static_cast<float*>(O_part), LSE_part, status,
               (cudaStream_t)stream};
  a.work = work;
  a.num_work = num_work;
  a.o_bf16 = 1;
  int rc = check_decode_args(a);
  if (rc != MLA_OK) return rc;
  rc = check_work(a);
  if (rc != MLA_OK) return rc;
  return launch_tc(a);
}

int mla_decode(const void* q_nope_absorbed, const void* q_rope,
               const void* kv_pages, const float* kv_scale,
               mla_kv_dtype kv_dtype, int64_t num_slots,
               const int32_t* req_to_token, int64_t r2t_stride,
               const int32_t* seq_lens, const int32_t* kv_limit, int B,
               int q_len, int H, int num_shards, int page_size, float sm_scale,
               int num_splits, const int32_t* split_pages,
               const int32_t* work, int num_work, float* O_part,
               float* LSE_part, int32_t* counters, void* out, float* lse_out,
               int* status, mla_stream_t stream) {
  DecodeArgs a{q_nope_absorbed, q_rope,    kv_pages, kv_scale,  kv_dtype,
               num_slots,       req_to_token, r2t_stride, seq_lens, kv_limit,
               B,               q_len,     H,        num_shards, page_size,
               sm_scale,        num_splits, split_pages, O_part,  LSE_part,  status,
               (cudaStream_t)stream};
  a.work = work;
  a.num_work = num_work;
  int rc = check_decode_args(a);
  if (rc != MLA_OK) return rc;
  rc = check_work(a);
  if (rc != MLA_OK) return rc;
  if (!counters || !out)
    return fail(MLA_ERR_INVALID_ARG, "counters and out are required");
  if (!aligned(counters, 4) || !aligned(out, 16) || (lse_out && !aligned(lse_out, 4)))
    return fail(MLA_ERR_MISALIGNED, "out needs 16-B alignment, counters and lse_out 4-B");
  a.out = out;
  a.lse_out = lse_out;
  a.counters = counters;
  return launch_tc(a);
}

int mla_decode_partial_simt(const void* q_nope_absorbed, const void* q_rope,
                            const void* kv_pages, const float* kv_scale,
                            mla_kv_dtype kv_dtype, int64_t num_slots,
                            const int32_t* req_to_token, int64_t r2t_stride,
                            const int32_t* seq_lens, const int32_t* kv_limit,
                            int B, int q_len, int H, int num_shards,
                            int page_size, float sm_scale, int num_splits,
                            const int32_t* split_pages,
                            float* O_part, float* LSE_part, int* status,
                            mla_stream_t stream) {
  DecodeArgs a{q_nope_absorbed, q_rope,    kv_pages, kv_scale,  kv_dtype,
               num_slots,       req_to_token, r2t_stride, seq_lens, kv_limit,
               B,               q_len,     H,        num_shards, page_size,
               sm_scale,        num_splits, split_pages, O_part,  LSE_part,  status,
               (cudaStream_t)stream};
  int rc = check_decode_args(a);
  if (rc != MLA_OK) return rc;
  return launch_simt(a);
}

}  // extern "C"
