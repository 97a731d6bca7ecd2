// spec_budget_plan: the hardware-aware budget controller of BASTION
// ("Metodologia", sections 1-3), on the host.
//
// Path score (section 1): a node at depth d reached through candidates
// c_1..c_d scores rho = prod_k q_k(c_k), q_k the drafter's marginal at position
// k. Acceptance surrogate and growth (section 2): A(T) = sum of rho over the
// tree, grown best-first - the frontier node with the largest rho joins next,
// ties to the one that entered the frontier first, and its children (the
// candidates of the next position, in candidate order) enter the frontier.
// Controller (section 3): T_verify(N) is a roofline estimate corrected by the
// measured latencies, a T_roof(N) + c with (a, c) the least-squares fit to the
// calibration samples; S(N) = A(T_N) L_AR / (T_draft + T_verify(N)); the tree
// grows one node at a time and the chosen size is the last one before S first
// decreases.
//
// The frontier is a binary heap, so growing N nodes costs O(N C log(N C)).
#include <cmath>
#include <cstdint>
#include <queue>
#include <vector>

#include "../../include/specverify.h"

namespace {

struct Candidate {
    double rho;
    int64_t order;  // entry order into the frontier (the tie-break)
    int32_t parent, depth, cand;
};

// std::priority_queue pops the largest element under this "less": larger rho
// first, then the earlier entry.
struct Later {
    bool operator()(const Candidate &a, const Candidate &b) const {
        if (a.rho != b.rho) return a.rho < b.rho;
        return a.order > b.order;
    }
};

bool is_finite_value(double x) { return std::isfinite(x); }

}  // namespace

extern "C" spec_status_t spec_budget_plan(const double *marginals, int K, int C, int n_max, double t_draft,
                                          double l_ar, double bytes0, double bytes_per_node, double flops_per_node,
                                          double bw, double peak, const double *cal_n, const double *cal_t,
                                          int n_cal, int32_t *parents, int32_t *depth, int32_t *cand, double *rho,
                                          double *speedup, double *calib, int32_t *n_chosen, int32_t *n_eval) {
    if (!marginals || !cal_n || !cal_t || !parents || !depth || !cand || !rho || !speedup || !calib || !n_chosen ||
        !n_eval)
        return SPEC_ERR_INVALID_ARG;
    if (K < 1 || C < 1 || n_max < 1 || n_cal < 1) return SPEC_ERR_INVALID_ARG;
    const double scalars[] = {bw, peak, t_draft, l_ar, bytes0, bytes_per_node, flops_per_node};
    for (const double v : scalars)
        if (!is_finite_value(v)) return SPEC_ERR_INVALID_ARG;
    if (!(bw > 0) || !(peak > 0)) return SPEC_ERR_INVALID_ARG;
    for (int64_t i = 0; i < (int64_t)K * C; ++i)
        if (!(marginals[i] >= 0.0 && marginals[i] <= 1.0)) return SPEC_ERR_INVALID_ARG;
    for (int j = 0; j < n_cal; ++j)
        if (!is_finite_value(cal_n[j]) || !is_finite_value(cal_t[j])) return SPEC_ERR_INVALID_ARG;

    auto t_roof = [&](double n) {
        const double tb = (bytes0 + bytes_per_node * n) / bw, tf = flops_per_node * n / peak;
        return tb > tf ? tb : tf;
    };
    // calibration: least squares of t on x = T_roof(n); with fewer than two distinct x the
    // ratio of the means, without offset
    std::vector<double> x(n_cal);
    bool distinct = false;
    double xs = 0.0, ts = 0.0;
    for (int j = 0; j < n_cal; ++j) {
        x[j] = t_roof(cal_n[j]);
        distinct |= x[j] != x[0];
        xs += x[j];
        ts += cal_t[j];
    }
    const double xm = xs / n_cal, tm = ts / n_cal;
    double a, c;
    if (!distinct) {
        a = tm / xm;
        c = 0.0;
    } else {
        double sxt = 0.0, sxx = 0.0;
        for (int j = 0; j < n_cal; ++j) {
            sxt += (x[j] - xm) * (cal_t[j] - tm);
            sxx += (x[j] - xm) * (x[j] - xm);
        }
        a = sxt / sxx;
        c = tm - a * xm;
    }
    if (!is_finite_value(a) || !is_finite_value(c)) return SPEC_ERR_INVALID_ARG;
    calib[0] = a;
    calib[1] = c;

    std::priority_queue<Candidate, std::vector<Candidate>, Later> frontier;
    int64_t order = 0;
    for (int cc = 0; cc < C; ++cc) frontier.push({marginals[cc], order++, -1, 1, cc});
    double surrogate = 0.0;
    int grown = 0, chosen = 0;
    while (grown < n_max && !frontier.empty()) {
        const Candidate top = frontier.top();
        frontier.pop();
        const int node = grown++;
        parents[node] = top.parent;
        depth[node] = top.depth;
        cand[node] = top.cand;
        rho[node] = top.rho;
        if (top.depth < K)
            for (int c2 = 0; c2 < C; ++c2)
                frontier.push({top.rho * marginals[(int64_t)top.depth * C + c2], order++, node, top.depth + 1, c2});
        surrogate += top.rho;
        const int n = node + 1;
        const double cost = t_draft + (a * t_roof((double)n) + c);
        if (!(cost > 0)) return SPEC_ERR_INVALID_ARG;
        speedup[node] = surrogate * l_ar / cost;
        if (n >= 2 && speedup[node] < speedup[node - 1]) {
            chosen = n - 1;
            break;
        }
        chosen = n;
    }
    *n_chosen = chosen;
    *n_eval = grown;
    return SPEC_OK;
}
