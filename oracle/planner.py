"""Per-operation offload ratios -- oracle by exhaustive search.

The problem ([DAK] section 4.2.2 "Problem Formulation" and Appendix A eq. (1)): given
operations i with data size C_i (bytes of weights or KV) and pure compute time
T_comp,i, choose offloaded bytes b_i = x_i C_i in [0, C_i] to minimise the end-to-end
time sum_i C_i / EB_i(x_i), where ([DAK] section 4.2.1; [DAK-explainer] section on the
mathematical model of the offload ratio)

    T_i(b) = C_i / EB_i = max(T_comp,i, (C_i - b) / B_g, b / B_h)

with B_g the GPU-memory bandwidth and B_h the host-link bandwidth, subject to the global
budget sum_i b_i = D (the paper's eq. (1), ``mode="eq"``) or sum_i b_i >= D (the capacity
reading x_global >= max(0, (M - H)/M), ``mode="ge"``).

The oracle solves it by plain enumeration, not by the paper's greedy phases:

* ``exhaustive_continuous``: each T_i is convex and piecewise linear with its kinks among
  {0, C_i, C_i - B_g T_comp,i, B_h T_comp,i, C_i B_h / (B_h + B_g)}. A linear programme
  over the segments has an optimal basic solution in which at most one operation is off
  those points, so the optimum is found by trying every choice of free operation and
  every assignment of candidate points to the others (size ~5^(n-1) * n; small n only).
* ``exhaustive_tiles``: every vector of whole tile counts (b_i = min(k_i * tile_i, C_i)),
  for the tile-granular variant; tiny cases only.

Parity pins (tests/test_oracle_planner.py): hand-worked values of EB(x) for a
memory-bound and a compute-bound operation; a hand-worked two-operation whole-tile case
whose optimum puts an operation (one with a ragged last tile) wholly on the host; the
single-operation turning points
x* = B_h/(B_h+B_g) (memory-bound) and x* = B_h/B_i with B_i = C_i/T_comp,i
(compute-bound) from [DAK] section 4.2.1 / Fig. 6; the worked GH200 value
x* = 0.9/(4.0+0.9) ~ 18.4% from [DAK-explainer]; the optimal objective values that
Appendix A's Theorems 1-3 give in closed form in their three regimes; and agreement of
the continuous optimum with the tile enumeration when tiles are fine.
"""
import itertools
import math

INF = float("inf")


def op_time(C: float, t_comp: float, b: float, b_host: float, b_gpu: float) -> float:
    """T_i(b) = max(T_comp, (C - b)/B_g, b/B_h)."""
    return max(t_comp, (C - b) / b_gpu, b / b_host)


def effective_bandwidth(C: float, t_comp: float, x: float, b_host: float, b_gpu: float) -> float:
    """EB(x) = C / max(T_comp, T_mem), T_mem = max(T_h, T_g)  ([DAK] section 4.2.1)."""
    t = op_time(C, t_comp, x * C, b_host, b_gpu)
    return C / t if t > 0 else INF


def objective(ops, b, b_host, b_gpu) -> float:
    return sum(op_time(C, tc, bi, b_host, b_gpu) for (C, tc), bi in zip(ops, b))


def candidate_points(C: float, t_comp: float, b_host: float, b_gpu: float):
    pts = {0.0, float(C), C - b_gpu * t_comp, b_host * t_comp, C * b_host / (b_host + b_gpu)}
    return sorted({min(max(p, 0.0), float(C)) for p in pts})


def _close(a, b, rel=1e-12):
    return abs(a - b) <= rel * max(1.0, abs(a), abs(b))


def exhaustive_continuous(ops, b_host, b_gpu, D, mode="ge"):
    """Minimum of sum_i T_i(b_i) over the feasible set; returns (objective, b vector).

    ops: list of (C_i, T_comp_i). Returns (inf, None) when sum C_i < D."""
    n = len(ops)
    total = sum(C for C, _ in ops)
    if D > total * (1 + 1e-12):
        return INF, None
    cands = [candidate_points(C, tc, b_host, b_gpu) for C, tc in ops]
    best, best_b = INF, None
    # budget met with equality
    for free in range(n):
        others = [j for j in range(n) if j != free]
        Cf = ops[free][0]
        for combo in itertools.product(*[cands[j] for j in others]):
            rest = D - sum(combo)
            tol = 1e-12 * max(1.0, total)
            if rest < -tol or rest > Cf + tol:
                continue
            b = [0.0] * n
            for j, v in zip(others, combo):
                b[j] = v
            b[free] = min(max(rest, 0.0), Cf)
            val = objective(ops, b, b_host, b_gpu)
            if val < best:
                best, best_b = val, b
    if mode == "ge":
        # unconstrained optimum: every op at a minimiser; feasible if the largest
        # minimisers together reach the budget
        b = []
        for (C, tc), cs in zip(ops, cands):
            ts = [op_time(C, tc, p, b_host, b_gpu) for p in cs]
            tmin = min(ts)
            b.append(max(p for p, t in zip(cs, ts) if _close(t, tmin)))
        if sum(b) >= D - 1e-12 * max(1.0, total):
            val = objective(ops, b, b_host, b_gpu)
            if val < best or _close(val, best):
                best, best_b = val, b
    elif mode != "eq":
        raise ValueError(mode)
    return best, best_b


def exhaustive_tiles(ops, tile_bytes, b_host, b_gpu, D):
    """Brute force over whole-tile allocations with sum_i b_i >= D.

    ops: list of (C_i, T_comp_i); tile_bytes[i]: granularity of op i; b_i(k) = min(k tile, C)."""
    grids = []
    for (C, _), t in zip(ops, tile_bytes):
        nt = math.ceil(C / t) if C > 0 else 0  # the last tile may be ragged: b = C there
        grids.append([min(k * t, C) for k in range(nt + 1)])
    best, best_b = INF, None
    for combo in itertools.product(*grids):
        if sum(combo) < D - 1e-9:
            continue
        val = objective(ops, combo, b_host, b_gpu)
        if val < best:
            best, best_b = val, list(combo)
    return best, best_b


def turning_point_memory_bound(b_host: float, b_gpu: float) -> float:
    """x* = B_h / (B_h + B_g): transfer times balance ([DAK] section 4.2.1, Fig. 6)."""
    return b_host / (b_host + b_gpu)


def turning_point_compute_bound(C: float, t_comp: float, b_host: float) -> float:
    """x* = B_h / B_i with B_i = C / T_comp: host time reaches compute time."""
    return b_host * t_comp / C


def uniform_plan(ops, ratio):
    """The uniform policy compared against in [DAK] section 4.2.1: x_i = OR for all i."""
    return [ratio * C for C, _ in ops]
