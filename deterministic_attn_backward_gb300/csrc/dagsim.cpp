// dagsim.cpp -- DAG model of the deterministic attention backward schedules.
//
// DASH (technical summary section 2.1) models the backward pass as a DAG whose
// nodes are compute phases (one per processed (KV tile, Q tile) pair) and
// reduction phases, and whose edges are data dependences plus the mandatory
// dQ accumulation order; a schedule is judged by the length of the critical
// path.  This file builds that DAG for the schedules of sched.h and measures
// it, with a finite number of CTAs that take units in the order the main
// kernel dispatches them.  Host-only; used by tests and for schedule design.
//
// Nodes, for step t of unit U (global unit index over all heads):
//   C(U,t) compute, weight wc;  R(U,t) reduction of dQ_j, weight wr.
// Edges:
//   C(U,t-1) -> C(U,t)                       (the CTA computes in order)
//   R(U,t-1) -> C(U,t)      reducer_depth 0   (reduction inside the chain)
//   R(U,t-1-k) -> C(U,t)    reducer_depth k   (k reductions may trail)
//   C(U,t) -> R(U,t),  R(U,t-1) -> R(U,t)     (one reducer per CTA)
//   R(rank-w contributor of dQ_j) -> R(U,t)   (fixed reduction order; with
//                                             w interleaved accumulation
//                                             buffers, rank r follows r - w)
//   last C / R of the previous unit on the same CTA -> first C / R of U.
#include <algorithm>
#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "tile_sched.h"

namespace {

struct Problem {
  int sched, mask, N, heads, ctas, reducer_depth;
  double wc, wr;
  int ways = 1;                   // interleaved accumulation buffers
  int uph = 0;                    // units per head
  int total = 0;                  // units overall
  std::vector<int> step_off;      // node offset of unit U's first step
  std::vector<int> steps;         // steps of unit U
  std::vector<int> node_q;        // Q tile of each step node
  std::vector<int> node_rank;     // rank of each step node (-1 atomic)
  std::vector<int> node_head;
  int nodes = 0;
  // rank_node[(head * N + j) * N + rank] = step node holding that contribution
  std::vector<int> rank_node;
};

bool build(Problem& P) {
  if (P.N <= 0 || P.heads <= 0 || P.ctas <= 0 || P.reducer_depth < 0) return false;
  if (P.sched == dab::kSchedShift && P.mask == dab::kMaskCausal && (P.N % 2) != 0) return false;
  P.uph = dab::units_per_head(P.sched, P.mask, P.N);
  P.total = P.uph * P.heads;
  P.step_off.resize(P.total + 1);
  P.steps.resize(P.total);
  int off = 0;
  for (int U = 0; U < P.total; ++U) {
    P.step_off[U] = off;
    P.steps[U] = dab::unit_steps(P.sched, P.mask, P.N, U % P.uph);
    off += P.steps[U];
  }
  P.step_off[P.total] = off;
  P.nodes = off;
  P.node_q.resize(off);
  P.node_rank.resize(off);
  P.node_head.resize(off);
  P.rank_node.assign((size_t)P.heads * P.N * P.N, -1);
  for (int U = 0; U < P.total; ++U) {
    const int h = U / P.uph, u = U % P.uph;
    for (int t = 0; t < P.steps[U]; ++t) {
      const dab::Step s = dab::step(P.sched, P.mask, P.N, u, t);
      const int n = P.step_off[U] + t;
      P.node_q[n] = s.q;
      P.node_head[n] = h;
      const int r = dab::rank(P.sched, P.mask, P.N, s.kv, s.q);
      P.node_rank[n] = r;
      if (r >= 0) {
        if (r >= P.N) return false;
        int& slot = P.rank_node[((size_t)h * P.N + s.q) * P.N + r];
        if (slot != -1) return false;  // two contributions with one rank
        slot = n;
      }
    }
  }
  return true;
}

int rank_pred(const Problem& P, int n) {
  const int r = P.node_rank[n];
  if (r < P.ways) return -1;
  return P.rank_node[((size_t)P.node_head[n] * P.N + P.node_q[n]) * P.N + (r - P.ways)];
}

// Static placement (unit U on CTA U mod ctas, ascending U): longest paths
// by Kahn's algorithm.  Returns false on a cycle (deadlock).
bool run_static(const Problem& P, double* makespan) {
  const int n2 = 2 * P.nodes;  // node x: C = 2x, R = 2x + 1
  std::vector<std::vector<int>> out(n2);
  std::vector<int> indeg(n2, 0);
  auto edge = [&](int a, int b) { out[a].push_back(b); indeg[b]++; };
  std::vector<int> prev_unit(P.ctas, -1);
  for (int U = 0; U < P.total; ++U) {
    const int cta = U % P.ctas;
    const int base = P.step_off[U];
    const int T = P.steps[U];
    for (int t = 0; t < T; ++t) {
      const int n = base + t;
      if (t > 0) {
        edge(2 * (n - 1), 2 * n);
        edge(2 * (n - 1) + 1, 2 * n + 1);
        const int k = P.reducer_depth + 1;  // C(t) waits for R(t - 1 - depth)
        if (t - k >= 0) edge(2 * (n - k) + 1, 2 * n);
      }
      edge(2 * n, 2 * n + 1);
      const int rp = rank_pred(P, n);
      if (rp >= 0) edge(2 * rp + 1, 2 * n + 1);
    }
    const int pu = prev_unit[cta];
    if (pu >= 0) {
      const int last = P.step_off[pu] + P.steps[pu] - 1;
      edge(2 * last, 2 * base);
      edge(2 * last + 1, 2 * base + 1);
      if (P.reducer_depth == 0) edge(2 * last + 1, 2 * base);
    }
    prev_unit[cta] = U;
  }
  std::vector<double> start(n2, 0.0), fin(n2, 0.0);
  std::vector<int> queue;
  queue.reserve(n2);
  for (int x = 0; x < n2; ++x)
    if (indeg[x] == 0) queue.push_back(x);
  size_t head = 0;
  double mk = 0.0;
  while (head < queue.size()) {
    const int x = queue[head++];
    fin[x] = start[x] + ((x & 1) ? P.wr : P.wc);
    mk = std::max(mk, fin[x]);
    for (int y : out[x]) {
      start[y] = std::max(start[y], fin[x]);
      if (--indeg[y] == 0) queue.push_back(y);
    }
  }
  if ((int)queue.size() != n2) return false;
  *makespan = mk;
  return true;
}

// Dynamic dispatch (ascending units to the CTA whose compute frees first).
// Every dependence points to a lower unit, so units are timed in order.
bool run_dynamic(const Problem& P, double* makespan) {
  std::vector<double> c_free(P.ctas, 0.0), r_free(P.ctas, 0.0);
  std::vector<double> r_fin(P.nodes, -1.0), c_fin(P.nodes, 0.0);
  double mk = 0.0;
  for (int U = 0; U < P.total; ++U) {
    int cta = 0;
    for (int c = 1; c < P.ctas; ++c)
      if (c_free[c] < c_free[cta]) cta = c;
    double cprev = c_free[cta], rprev = r_free[cta];
    if (P.reducer_depth == 0) cprev = std::max(cprev, rprev);
    const int base = P.step_off[U];
    for (int t = 0; t < P.steps[U]; ++t) {
      const int n = base + t;
      double cs = cprev;
      if (t > 0) {
        const int k = P.reducer_depth + 1;
        if (t - k >= 0) cs = std::max(cs, r_fin[n - k]);
      }
      c_fin[n] = cs + P.wc;
      cprev = c_fin[n];
      double rs = std::max(c_fin[n], rprev);
      const int rp = rank_pred(P, n);
      if (rp >= 0) {
        if (r_fin[rp] < 0) return false;  // depends on a later unit
        rs = std::max(rs, r_fin[rp]);
      }
      r_fin[n] = rs + P.wr;
      rprev = r_fin[n];
      mk = std::max(mk, r_fin[n]);
    }
    c_free[cta] = (P.reducer_depth == 0) ? rprev : cprev;
    r_free[cta] = rprev;
  }
  *makespan = mk;
  return true;
}

}  // namespace

extern "C" int dab_dag_simulate_ways(int sched, int mask, int N, int heads, int ctas,
                                     double wc, double wr, int reducer_depth, int ways,
                                     double* makespan, double* busy_fraction) {
  if (sched < 0 || sched > 3 || mask < 0 || mask > 1 || wc < 0 || wr < 0 || ways < 1) return -1;
  Problem P{sched, mask, N, heads, ctas, reducer_depth, wc, wr};
  P.ways = ways;
  if (!build(P)) return -1;
  double mk = 0.0;
  bool ok;
  if (dab::static_dispatch(sched)) {
    ok = run_static(P, &mk);
  } else {
    ok = run_dynamic(P, &mk);
  }
  if (!ok) return -2;
  if (makespan) *makespan = mk;
  if (busy_fraction) {
    const double work = (double)P.nodes * wc;
    *busy_fraction = mk > 0 ? work / ((double)ctas * mk) : 0.0;
  }
  return 0;
}

extern "C" int dab_dag_simulate(int sched, int mask, int N, int heads, int ctas,
                                double wc, double wr, int reducer_depth,
                                double* makespan, double* busy_fraction) {
  return dab_dag_simulate_ways(sched, mask, N, heads, ctas, wc, wr, reducer_depth, 1, makespan,
                               busy_fraction);
}

extern "C" double dab_dag_critical_path(int sched, int mask, int N, double wc, double wr,
                                        int reducer_depth) {
  Problem P{sched, mask, N, 1, 1, reducer_depth, wc, wr};
  if (!build(P)) return -1.0;
  P.ctas = P.total;  // one processor per unit
  double mk = 0.0;
  if (!run_static(P, &mk)) return -2.0;
  return mk;
}

// Schedule selection (the "palette" of DASH, technical summary section 4:
// the best schedule depends on the mask and the problem shape).  The DAG
// model above, with the weights that match the GB300 measurements of this
// library (reduction phase as long as a compute phase, one reduction
// trailing the compute, four interleaved accumulation buffers), picks the
// deterministic schedule with the smallest predicted makespan.  On the GB300
// sweep (29 shapes, d 64 and 128, S 1024 to 32768, both masks) its pick is
// the measured fastest deterministic schedule in 27; the summed loss against
// the measured best is 1.4 %, the largest 1.1 % (B4 H16 S8192 d128, full
// mask, where SHIFT ran faster than predicted).  An extra penalty on SHIFT's
// prediction (its statically placed rings run in lock step) helped an
// earlier kernel whose reduction was slower; with this kernel any penalty
// above 1 % loses more than it gains, so there is none.  Ties go to
// DESCENDING_Q, then SERIAL, then SHIFT.  Results are cached.
extern "C" int dab_sched_select(int mask, int B, int H, int S, int ctas) {
  if (mask < 0 || mask > 1 || B < 1 || H < 1 || S < 128 || (S % 128) != 0 || ctas < 1) return -1;
  const int N = S / 128;
  const long long bh = (long long)B * H;
  static std::mutex mu;
  static std::map<std::tuple<int, long long, int, int>, int> cache;
  const auto key = std::make_tuple(mask, bh, N, ctas);
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  constexpr double kWc = 1.0, kWr = 1.0;
  constexpr int kDepth = 1, kWays = 4;
  const int order[3] = {dab::kSchedDescending, dab::kSchedSerial, dab::kSchedShift};
  int best = dab::kSchedDescending;
  double best_mk = -1.0;
  for (int sched : order) {
    if (sched == dab::kSchedShift && mask == dab::kMaskCausal && (N % 2) != 0) continue;
    if (dab::gang_size(sched, mask, N) > ctas) continue;
    const int uph = dab::units_per_head(sched, mask, N);
    // All heads up to a budget of ~1.5M DAG nodes (the placement of units
    // on CTAs repeats only after many heads, and it decides whether a shift
    // gang is split between rounds), but at least enough to fill the CTAs
    // twice.
    const long long fill = (2LL * ctas + uph - 1) / uph;
    const long long budget = 1500000LL / ((long long)N * N);
    const int heads = (int)std::min<long long>(bh, std::max<long long>({1LL, fill, budget}));
    double mk = 0.0;
    if (dab_dag_simulate_ways(sched, mask, N, heads, ctas, kWc, kWr, kDepth, kWays, &mk, nullptr) != 0)
      continue;
    if (best_mk < 0.0 || mk < best_mk * (1.0 - 1e-9)) {
      best = sched;
      best_mk = mk;
    }
  }
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = best;
  return best;
}

