// Per-operation offload ratios ("DAK: Direct-Access-Enabled GPU Memory Offloading with
// Optimal Efficiency for LLM Inference", section 4.2 and Appendix A).
//
// Each operation i reads C_i bytes; with b_i of them offloaded its time under the
// effective-bandwidth model (section 4.2.1) is
//     T_i(b) = max(T_comp,i, (C_i - b) / B_hbm, b / B_host).
// T_i falls with slope -1/B_hbm up to b_dec,i (the peak for a memory-bound operation,
// x* = B_h / (B_h + B_g), or the point where the HBM time meets T_comp), stays flat up to
// b_flat,i (the threshold x* = B_h / B_i of a compute-bound operation, B_i = C_i / T_comp,i)
// and then rises with slope +1/B_host. The slopes are the same for every operation, so the
// greedy of section 4.2.2 is optimal: phase 1 fills the falling segments, phase 2 the flat
// ones, phase 3 the rising ones. Within a phase every allocation is optimal (Theorems 1-3);
// this one gives every operation the same fraction of its segment.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <limits>
#include <numeric>
#include <vector>

#include "../../include/dak.h"

namespace {

struct Seg {
    double dec, flat;  // end of the falling and of the flat segment, bytes
};

double op_time(double C, double tc, double b, double bh, double bg) {
    return std::max(tc, std::max((C - b) / bg, b / bh));
}

Seg segments(double C, double tc, double bh, double bg) {
    Seg s;
    s.dec = std::min(C - bg * tc, C * bh / (bh + bg));
    s.dec = std::min(std::max(s.dec, 0.0), C);
    s.flat = std::min(std::max(std::max(s.dec, bh * tc), 0.0), C);
    return s;
}

dak_status plan_continuous(const dak_op* ops, int n, double bh, double bg, double D, bool equality, double* ratios,
                           double* tmodel) {
    std::vector<Seg> seg(n);
    double cap1 = 0, cap2 = 0, cap3 = 0;
    for (int i = 0; i < n; ++i) {
        seg[i] = segments(ops[i].bytes, ops[i].t_comp, bh, bg);
        cap1 += seg[i].dec;
        cap2 += seg[i].flat - seg[i].dec;
        cap3 += ops[i].bytes - seg[i].flat;
    }
    // phase 1 is free gain: under ">=" it is taken whole even past the budget
    const double total = equality ? D : std::max(D, cap1);
    double a1 = std::min(total, cap1);
    double a2 = std::min(total - a1, cap2);
    double a3 = std::min(total - a1 - a2, cap3);
    const double f1 = cap1 > 0 ? a1 / cap1 : 0.0;
    const double f2 = cap2 > 0 ? a2 / cap2 : 0.0;
    const double f3 = cap3 > 0 ? a3 / cap3 : 0.0;
    double t = 0;
    for (int i = 0; i < n; ++i) {
        const double C = ops[i].bytes;
        double b = f1 * seg[i].dec + f2 * (seg[i].flat - seg[i].dec) + f3 * (C - seg[i].flat);
        b = std::min(std::max(b, 0.0), C);
        ratios[i] = C > 0 ? b / C : 0.0;
        t += op_time(C, ops[i].t_comp, b, bh, bg);
    }
    if (tmodel) *tmodel = t;
    return DAK_OK;
}

// Exact optimum over whole tiles for sum_i b_i >= D: dynamic programme over operations,
// state = offloaded bytes in units of the gcd of the tile sizes, capped at the budget.
dak_status plan_tiles(const dak_op* ops, int n, double bh, double bg, double D, double* ratios, double* tmodel) {
    std::vector<int64_t> tile(n), C(n), nt(n);
    int64_t g = 0;
    for (int i = 0; i < n; ++i) {
        C[i] = static_cast<int64_t>(std::llround(ops[i].bytes));
        tile[i] = static_cast<int64_t>(std::llround(ops[i].tile_bytes));
        if (tile[i] <= 0 || C[i] < 0) return DAK_ERR_INVALID;
        nt[i] = (C[i] + tile[i] - 1) / tile[i];
        g = std::gcd(g, tile[i]);
        if (C[i] % tile[i]) g = std::gcd(g, C[i] % tile[i]);
    }
    if (g <= 0) return DAK_ERR_INVALID;
    const int64_t UD = D <= 0 ? 0 : static_cast<int64_t>(std::ceil(D / static_cast<double>(g) - 1e-9));
    double work = 0;
    for (int i = 0; i < n; ++i) work += static_cast<double>(nt[i] + 1) * static_cast<double>(UD + 1);
    if (work > 4e9) return DAK_ERR_UNSUPPORTED;
    if (static_cast<double>(n + 1) * static_cast<double>(UD + 1) > 1e8) return DAK_ERR_UNSUPPORTED;
    const double INF = std::numeric_limits<double>::infinity();
    // layers[i][u]: least time of ops 0..i-1 with min(offloaded units, UD) == u
    std::vector<std::vector<double>> layers(n + 1, std::vector<double>(UD + 1, INF));
    layers[0][0] = 0;
    for (int i = 0; i < n; ++i) {
        for (int64_t k = 0; k <= nt[i]; ++k) {
            const int64_t b = std::min(k * tile[i], C[i]);
            const int64_t w = b / g;
            const double cost = op_time(static_cast<double>(C[i]), ops[i].t_comp, static_cast<double>(b), bh, bg);
            for (int64_t u = 0; u <= UD; ++u) {
                if (layers[i][u] == INF) continue;
                const int64_t v = std::min(UD, u + w);
                layers[i + 1][v] = std::min(layers[i + 1][v], layers[i][u] + cost);
            }
        }
    }
    if (layers[n][UD] == INF) return DAK_ERR_INVALID;
    int64_t v = UD;
    for (int i = n - 1; i >= 0; --i) {
        bool found = false;
        for (int64_t k = 0; k <= nt[i] && !found; ++k) {
            const int64_t b = std::min(k * tile[i], C[i]);
            const int64_t w = b / g;
            const double cost = op_time(static_cast<double>(C[i]), ops[i].t_comp, static_cast<double>(b), bh, bg);
            // predecessors: exact u = v - w, or (when v == UD) any u with u + w >= UD
            const int64_t lo = v == UD ? std::max<int64_t>(0, UD - w) : v - w;
            const int64_t hi = v == UD ? UD : v - w;
            for (int64_t u = lo; u <= hi && u >= 0; ++u) {
                if (layers[i][u] == INF) continue;
                if (layers[i][u] + cost == layers[i + 1][v]) {
                    ratios[i] = C[i] > 0 ? static_cast<double>(b) / static_cast<double>(C[i]) : 0.0;
                    v = u;
                    found = true;
                    break;
                }
            }
        }
        if (!found) return DAK_ERR_INVALID;
    }
    if (tmodel) *tmodel = layers[n][UD];
    return DAK_OK;
}

}  // namespace

extern "C" dak_status dak_plan_ratios(const dak_op* ops, int n, double b_host, double b_hbm,
                                      double min_offload_bytes, int mode, double* ratios_out, double* model_time_out) {
    if (n < 0 || (n > 0 && (!ops || !ratios_out)) || !(b_host > 0) || !(b_hbm > 0)) return DAK_ERR_INVALID;
    if (mode < 0 || mode > 2 || !(min_offload_bytes >= 0) || std::isinf(min_offload_bytes)) return DAK_ERR_INVALID;
    double total = 0;
    for (int i = 0; i < n; ++i) {
        if (!(ops[i].bytes >= 0) || !(ops[i].t_comp >= 0) || std::isinf(ops[i].bytes)) return DAK_ERR_INVALID;
        total += ops[i].bytes;
    }
    if (min_offload_bytes > total * (1 + 1e-12)) return DAK_ERR_INVALID;
    if (n == 0) {
        if (model_time_out) *model_time_out = 0;
        return DAK_OK;
    }
    if (mode == 2) return plan_tiles(ops, n, b_host, b_hbm, min_offload_bytes, ratios_out, model_time_out);
    return plan_continuous(ops, n, b_host, b_hbm, std::min(min_offload_bytes, total), mode == 1, ratios_out,
                           model_time_out);
}

// Whole-unit placement for any number of operations: the greedy ratios floored to whole
// units, then one unit at a time added where the model time grows least (to the
// picosecond; ties go to the operation whose ratio stays lowest) until the budget is met.
extern "C" dak_status dak_plan_units(const dak_op* ops, int n, double b_host, double b_hbm, double min_offload_bytes,
                                     int64_t* host_units_out, double* model_time_out) {
    if (n < 0 || (n > 0 && (!ops || !host_units_out)) || !(b_host > 0) || !(b_hbm > 0)) return DAK_ERR_INVALID;
    if (!(min_offload_bytes >= 0) || std::isinf(min_offload_bytes)) return DAK_ERR_INVALID;
    double total = 0;
    std::vector<int64_t> units(n), cnt(n);
    for (int i = 0; i < n; ++i) {
        if (!(ops[i].bytes >= 0) || !(ops[i].t_comp >= 0) || std::isinf(ops[i].bytes) || !(ops[i].tile_bytes > 0))
            return DAK_ERR_INVALID;
        total += ops[i].bytes;
        units[i] = static_cast<int64_t>(std::ceil(ops[i].bytes / ops[i].tile_bytes - 1e-9));
    }
    if (min_offload_bytes > total * (1 + 1e-12)) return DAK_ERR_INVALID;
    if (n == 0) {
        if (model_time_out) *model_time_out = 0;
        return DAK_OK;
    }
    std::vector<double> ratios(n);
    dak_status st = plan_continuous(ops, n, b_host, b_hbm, std::min(min_offload_bytes, total), false, ratios.data(), nullptr);
    if (st != DAK_OK) return st;
    auto bytes_of = [&](int i, int64_t k) { return std::min(ops[i].bytes, static_cast<double>(k) * ops[i].tile_bytes); };
    auto t_of = [&](int i, int64_t k) { return op_time(ops[i].bytes, ops[i].t_comp, bytes_of(i, k), b_host, b_hbm); };
    double host = 0;
    for (int i = 0; i < n; ++i) {
        cnt[i] = std::min(units[i], static_cast<int64_t>(std::floor(ratios[i] * ops[i].bytes / ops[i].tile_bytes + 1e-9)));
        host += bytes_of(i, cnt[i]);
    }
    const double D = std::min(min_offload_bytes, total);
    while (host < D * (1 - 1e-12)) {
        int best = -1;
        long long best_dt = 0;
        double best_r = 0;
        for (int i = 0; i < n; ++i) {
            if (cnt[i] >= units[i]) continue;
            const long long dt = std::llround((t_of(i, cnt[i] + 1) - t_of(i, cnt[i])) * 1e12);
            const double r = static_cast<double>(cnt[i] + 1) / static_cast<double>(units[i]);
            if (best < 0 || dt < best_dt || (dt == best_dt && r < best_r)) {
                best = i;
                best_dt = dt;
                best_r = r;
            }
        }
        if (best < 0) break;
        host += bytes_of(best, cnt[best] + 1) - bytes_of(best, cnt[best]);
        ++cnt[best];
    }
    double t = 0;
    for (int i = 0; i < n; ++i) {
        host_units_out[i] = cnt[i];
        t += t_of(i, cnt[i]);
    }
    if (model_time_out) *model_time_out = t;
    return DAK_OK;
}
