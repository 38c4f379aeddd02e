// Host-side balanced schedule of the causal forward's work units.
//
// A causal forward unit (two query tiles 2p, 2p+1 of one head) costs about
// 2 (2p+1) + 2 (2p+2) tensor-core products plus a fixed cost per unit (the
// pipeline fill at its start and the output epilogue at its end).  Measured on
// GB300 with the kernel's timestamps, a CTA's finishing time fits
// 0.55 us x products + 8.7 us x units (residual 1.4 us) on both causal d = 128
// workloads: the fixed part is worth about 16 products.
// Handing the units out longest first (greedy list scheduling, the order of
// "CMU 11-868 L21" notes, slides 27-46) leaves the CTAs finishing up to one
// small unit apart; here the longest-first assignment is computed once on the
// host and then improved by moving and swapping units out of the most loaded
// CTA while that lowers the largest load.  Each CTA then runs its units longest
// first.  The result depends only on the shape and the grid, so it is cached.
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "fa_kernels.h"

namespace fa {
namespace {

using Key = std::tuple<int, int, int, int, int, int>;  // B, Hq, Nq, d, fp8, grid
std::map<Key, FwdSched> g_cache;
std::mutex g_mu;

// Cost of forward unit u in tensor-core products (one 128 x 128 x d product = 1).
double unit_cost(const Dims& s, int u, double per_unit) {
  int b, h, p;
  fwd_unit(s, u, b, h, p);
  const int nq = q_tiles(s);
  double steps = 0;
  for (int t = 0; t < 2; ++t) {
    const int qt = 2 * p + t;
    if (qt < nq) steps += qt + 1;  // key tiles 0 .. qt
  }
  return 2.0 * steps + per_unit;
}

void build(const Dims& s, int d, bool fp8, int grid, FwdSched* out) {
  const int n = fwd_units(s);
  // the fixed cost per unit relative to one product: products take half as long at
  // d = 64 and with one-byte operands, the fixed part does not
  const double per_unit = 16.0 * (128.0 / d) * (fp8 ? 2.0 : 1.0);
  std::vector<double> cost(n);
  for (int u = 0; u < n; ++u) cost[u] = unit_cost(s, u, per_unit);
  std::vector<int> order(n);
  for (int u = 0; u < n; ++u) order[u] = u;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return cost[a] > cost[b]; });

  // longest first onto the least loaded CTA
  std::vector<std::vector<int>> bins(grid);
  std::vector<double> load(grid, 0.0);
  for (int u : order) {
    const int c = static_cast<int>(std::min_element(load.begin(), load.end()) - load.begin());
    bins[c].push_back(u);
    load[c] += cost[u];
  }
  // improve: move or swap a unit out of the most loaded CTA while the largest load drops
  for (int iter = 0; iter < 8 * n; ++iter) {
    const int m = static_cast<int>(std::max_element(load.begin(), load.end()) - load.begin());
    double best = load[m];
    int bi = -1, bc = -1, bj = -1;  // unit index in bins[m], other CTA, unit index there (-1: a move)
    for (int i = 0; i < static_cast<int>(bins[m].size()); ++i) {
      const double cx = cost[bins[m][i]];
      for (int c = 0; c < grid; ++c) {
        if (c == m) continue;
        const double mv = std::max(load[m] - cx, load[c] + cx);
        if (mv < best - 1e-9) {
          best = mv;
          bi = i, bc = c, bj = -1;
        }
        for (int j = 0; j < static_cast<int>(bins[c].size()); ++j) {
          const double cy = cost[bins[c][j]];
          if (cy >= cx) continue;
          const double sw = std::max(load[m] - cx + cy, load[c] - cy + cx);
          if (sw < best - 1e-9) {
            best = sw;
            bi = i, bc = c, bj = j;
          }
        }
      }
    }
    if (bi < 0) break;
    const int x = bins[m][bi];
    if (bj < 0) {
      bins[m].erase(bins[m].begin() + bi);
      bins[bc].push_back(x);
      load[m] -= cost[x];
      load[bc] += cost[x];
    } else {
      const int y = bins[bc][bj];
      bins[m][bi] = y;
      bins[bc][bj] = x;
      load[m] += cost[y] - cost[x];
      load[bc] += cost[x] - cost[y];
    }
  }
  out->on = 1;
  out->grid = grid;
  int k = 0;
  for (int c = 0; c < grid; ++c) {
    std::stable_sort(bins[c].begin(), bins[c].end(), [&](int a, int b) { return cost[a] > cost[b]; });
    out->start[c] = static_cast<uint16_t>(k);
    for (int u : bins[c]) out->ord[k++] = static_cast<uint16_t>(u);
  }
  out->start[grid] = static_cast<uint16_t>(k);
}

}  // namespace

// Key-split plan of an unmasked forward.  Its units all cost the same, so with U
// units on `sms` SMs the last wave holds R = U mod sms of them (all U when U <
// sms) and the launch lasts ceil(U / sms) units while the SMs average U / sms.
// Splitting those R units along the keys into f = floor(sms / R) parts (at most
// 4, each of at least two key tiles) lets the last wave fill the SMs: it then
// lasts 1/f of a unit.  The parts' outputs are merged by LSE afterwards.
FwdSplit fwd_split_plan(const Dims& s, int sms) {
  const int U = fwd_units(s), nk = k_tiles(s);
  FwdSplit r{U, 1};
  if (mask_kind(s) != MASK_NONE || s.cu_q != nullptr || sms < 2 || U < 1) return r;
  const int R = U >= sms ? U % sms : U;
  if (R == 0) return r;
  const int f = std::min(std::min(sms / R, 4), nk / 2);
  if (f < 2) return r;
  r.split0 = U - R;
  r.nsplit = f;
  return r;
}

const FwdSched* causal_schedule(const Dims& s, int d, bool fp8, int grid) {
  if (mask_kind(s) != MASK_CAUSAL || s.cu_q != nullptr) return nullptr;
  const int n = fwd_units(s);
  if (n > SCHED_MAX_UNITS || grid < 1 || grid > SCHED_MAX_CTAS || grid > n) return nullptr;
  const Key key{s.B, s.Hq, s.Nq, d, fp8 ? 1 : 0, grid};
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_cache.find(key);
  if (it == g_cache.end()) {
    FwdSched sc{};
    build(s, d, fp8, grid, &sc);
    it = g_cache.emplace(key, sc).first;
  }
  return &it->second;
}

}  // namespace fa
