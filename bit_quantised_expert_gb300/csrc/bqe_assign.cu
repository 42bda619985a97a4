// bqe_assign.cu — byte-budgeted per-expert format assignment (host code).
//
// Strata 4090 post, section 5, first paragraph (quantisation): each routed
// expert takes ternary PTQ1_0, Q2_0 or Q3_K; the byte budget is what the same
// experts take as all-Q2_0; the assignment is a Lagrangian relaxation with a
// bisection on the multiplier followed by a greedy pass over the bytes left;
// an expert's cost for a format is its held-out error over the routed output
// energy of its layer (the first two and last three layers counted twice);
// at most half of a layer's experts are ternary, and an expert seen by fewer
// than 8 held-out tokens stays Q2_0.  Where the post is silent (ties, the
// bisection's length, the greedy order) the choices are stated at each step
// below.  All arithmetic is IEEE double in a fixed order, with floating-point
// contraction off, so the result is the same on every host.
#include <stdint.h>

#include <algorithm>
#include <vector>

#include "../../include/bqe.h"

#define BQE_NOCONTRACT __attribute__((optimize("fp-contract=off")))

namespace {

struct Problem {
  int L, E;
  std::vector<double> cost;     // [l][e][f], f = 0 ternary, 1 Q2_0, 2 Q3_K
  std::vector<uint8_t> locked;  // [l][e]
  std::vector<int> cap;         // ternary experts allowed per layer
  double nbytes[3];
};

// The relaxed problem at multiplier lam: every unlocked expert takes the
// format of least cost + lam * bytes (ties: fewer bytes); when more than the
// layer's cap take ternary, those that lose most by giving it up keep it (ties:
// lower expert index) and the rest take their best other format — the exact
// minimum of the layer's relaxed problem under the cap.
BQE_NOCONTRACT void relaxed(const Problem& p, double lam, std::vector<uint8_t>& pick) {
  pick.assign((size_t)p.L * p.E, 1);
  std::vector<uint8_t> alt((size_t)p.E);
  std::vector<std::pair<double, int>> keen;
  for (int l = 0; l < p.L; ++l) {
    keen.clear();
    for (int e = 0; e < p.E; ++e) {
      const size_t ie = (size_t)l * p.E + e;
      if (p.locked[ie]) continue;
      const double* c = &p.cost[ie * 3];
      double s[3];
      for (int f = 0; f < 3; ++f) {
        const double t = lam * p.nbytes[f];
        s[f] = c[f] + t;
      }
      int best = 0;
      for (int f = 1; f < 3; ++f)
        if (s[f] < s[best]) best = f;
      const int other = s[1] <= s[2] ? 1 : 2;
      pick[ie] = (uint8_t)best;
      alt[e] = (uint8_t)other;
      if (best == 0) keen.emplace_back(s[other] - s[0], e);
    }
    if ((int)keen.size() > p.cap[l]) {
      std::sort(keen.begin(), keen.end(), [](const std::pair<double, int>& a, const std::pair<double, int>& b) {
        return a.first != b.first ? a.first > b.first : a.second < b.second;
      });
      for (size_t k = (size_t)p.cap[l]; k < keen.size(); ++k) pick[(size_t)l * p.E + keen[k].second] = alt[keen[k].second];
    }
  }
}

uint64_t total_bytes(const Problem& p, const std::vector<uint8_t>& pick, const uint64_t* nb) {
  uint64_t t = 0;
  for (uint8_t f : pick) t += nb[f];
  return t;
}

}  // namespace

extern "C" BQE_NOCONTRACT int bqe_assign_formats(int32_t n_layers, int32_t n_experts, const double* err,
                                                 const double* energy, const double* layer_weight,
                                                 const int32_t* heldout_tokens, int32_t min_tokens,
                                                 double tq1_cap_frac, const uint64_t* fmt_bytes, uint64_t budget,
                                                 int32_t* fmt_out, double* lambda_out, uint64_t* bytes_out,
                                                 double* cost_out) {
  if (n_layers <= 0 || n_experts <= 0 || !err || !energy || !layer_weight || !fmt_bytes || !fmt_out)
    return BQE_EINVAL;
  if (!(tq1_cap_frac >= 0.0 && tq1_cap_frac <= 1.0)) return BQE_EINVAL;
  if (!(fmt_bytes[0] < fmt_bytes[1] && fmt_bytes[1] < fmt_bytes[2])) return BQE_EINVAL;
  Problem p;
  p.L = n_layers;
  p.E = n_experts;
  const size_t n = (size_t)n_layers * n_experts;
  p.cost.resize(n * 3);
  p.locked.resize(n);
  p.cap.resize(n_layers);
  for (int f = 0; f < 3; ++f) p.nbytes[f] = (double)fmt_bytes[f];
  double spread = 0.0;
  for (int l = 0; l < n_layers; ++l) {
    if (!(energy[l] > 0.0) || !(layer_weight[l] >= 0.0)) return BQE_EINVAL;
    p.cap[l] = (int)(tq1_cap_frac * (double)n_experts);
    for (int e = 0; e < n_experts; ++e) {
      const size_t ie = (size_t)l * n_experts + e;
      double mx = 0.0, mn = 0.0;
      for (int f = 0; f < 3; ++f) {
        const double v = err[ie * 3 + f];
        if (!(v >= 0.0) || v > 1e300) return BQE_EINVAL;
        const double c = layer_weight[l] * v / energy[l];  // the layer's weight times error over energy
        p.cost[ie * 3 + f] = c;
        if (f == 0 || c > mx) mx = c;
        if (f == 0 || c < mn) mn = c;
      }
      spread = std::max(spread, mx - mn);
      p.locked[ie] = heldout_tokens && heldout_tokens[ie] < min_tokens;
    }
  }
  const double gap = std::min(p.nbytes[1] - p.nbytes[0], p.nbytes[2] - p.nbytes[1]);
  const double lam_max = 2.0 * spread / gap + 1.0;
  std::vector<uint8_t> pick;
  relaxed(p, lam_max, pick);
  if (total_bytes(p, pick, fmt_bytes) > budget) return BQE_EINVAL;  // below what the guard rails allow
  // the multiplier: 0 if that already fits, else 100 halvings of [0, lam_max]
  // keeping the upper end (the least multiplier found that fits)
  double lam = 0.0;
  relaxed(p, 0.0, pick);
  if (total_bytes(p, pick, fmt_bytes) > budget) {
    double lo = 0.0, hi = lam_max;
    for (int it = 0; it < 100; ++it) {
      const double mid = 0.5 * (lo + hi);
      relaxed(p, mid, pick);
      if (total_bytes(p, pick, fmt_bytes) <= budget)
        hi = mid;
      else
        lo = mid;
    }
    lam = hi;
    relaxed(p, hi, pick);
  }
  // greedy: the upgrade of largest cost decrease per byte that fits the bytes
  // left (ties: lower layer, expert, format), until none fits
  uint64_t left = budget - total_bytes(p, pick, fmt_bytes);
  while (true) {
    double br = 0.0;
    int bl = -1, be = -1, bg = -1;
    for (int l = 0; l < n_layers; ++l)
      for (int e = 0; e < n_experts; ++e) {
        const size_t ie = (size_t)l * n_experts + e;
        if (p.locked[ie]) continue;
        const int f = pick[ie];
        for (int g = f + 1; g < 3; ++g) {
          const uint64_t db = fmt_bytes[g] - fmt_bytes[f];
          const double dc = p.cost[ie * 3 + g] - p.cost[ie * 3 + f];
          if (dc < 0.0 && db <= left) {
            const double r = dc / (double)db;
            if (bl < 0 || r < br) {
              br = r;
              bl = l;
              be = e;
              bg = g;
            }
          }
        }
      }
    if (bl < 0) break;
    const size_t ie = (size_t)bl * n_experts + be;
    left -= fmt_bytes[bg] - fmt_bytes[pick[ie]];
    pick[ie] = (uint8_t)bg;
  }
  double total = 0.0;
  for (size_t ie = 0; ie < n; ++ie) {
    total += p.cost[ie * 3 + pick[ie]];
    fmt_out[ie] = pick[ie] == 0 ? BQE_FMT_TQ1 : pick[ie] == 1 ? BQE_FMT_Q2_0 : BQE_FMT_Q3_K;
  }
  if (lambda_out) *lambda_out = lam;
  if (bytes_out) *bytes_out = total_bytes(p, pick, fmt_bytes);
  if (cost_out) *cost_out = total;
  return BQE_OK;
}
