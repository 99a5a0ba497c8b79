"""Pins for the planner and placement oracles: the pages' closed forms and printed values."""
import math

import pytest

import synth
from conftest import read_golden
from oracle import placement as opl
from oracle import planner as op

pytestmark = pytest.mark.cpu

GB = 1e9


def test_worked_gh200_turning_point():
    (bg, bh, pct), = read_golden("gh200_turning_point.txt")
    x = op.turning_point_memory_bound(float(bh), float(bg))
    assert round(100 * x, 1) == float(pct)


@pytest.mark.parametrize("bh,bg", [(0.9e12, 4.0e12), (0.35e12, 6.7e12), (64e9, 1.8e12)])
def test_single_memory_bound_op_peaks_at_balance(bh, bg):
    C = 1e9
    obj, b = op.exhaustive_continuous([(C, 0.0)], bh, bg, 0.0, mode="ge")
    assert b[0] / C == pytest.approx(bh / (bh + bg), rel=1e-12)
    # the peak effective bandwidth is B_h + B_g
    assert C / obj == pytest.approx(bh + bg, rel=1e-12)


def test_single_compute_bound_threshold():
    bh, bg = 0.9e12, 4.0e12
    C, tc = 1e9, 1e9 / 1.0e12  # B_i = 1 TB/s < B_g: compute-bound
    xt = op.turning_point_compute_bound(C, tc, bh)
    assert xt == pytest.approx(bh / (C / tc))
    # flat up to the threshold ...
    for x in (0.0, 0.3 * xt, xt):
        obj, _ = op.exhaustive_continuous([(C, tc)], bh, bg, x * C, mode="eq")
        assert obj == pytest.approx(tc, rel=1e-12)
    # ... then slope 1/B_h
    obj, _ = op.exhaustive_continuous([(C, tc)], bh, bg, (xt + 0.1) * C, mode="eq")
    assert obj == pytest.approx((xt + 0.1) * C / bh, rel=1e-12)


def _ops(seed, n):
    u = synth.uniform_f64(seed, 0, 2 * n)
    ops = []
    for i in range(n):
        C = (0.2 + u[2 * i]) * GB
        # half the ops compute-bound (B_i = C/T_comp in [1, 3.5] TB/s, below B_g = 4 TB/s,
        # so that x* = B_h/B_i < 1), half memory-bound
        tc = C / (1e12 * (1.0 + 2.5 * u[2 * i + 1])) if i % 2 else 0.2 * C / 4e12 * u[2 * i + 1]
        ops.append((C, tc))
    return ops


@pytest.mark.parametrize("seed", range(6))
def test_appendix_a_theorem_regimes(seed):
    """Closed-form optimal times of Theorems 1-3 (Appendix A) in their regimes."""
    bh, bg = 0.9e12, 4.0e12
    ops = _ops(seed, 4)
    mem = [(C, tc) for C, tc in ops if tc < C / bg]
    comp = [(C, tc) for C, tc in ops if tc >= C / bg]
    # paper's x*: memory-bound B_h/(B_h+B_g) (valid when T_comp is below the balanced time)
    assert all(tc <= C / (bh + bg) for C, tc in mem)
    xm = bh / (bh + bg)
    mem_budget = sum(C * xm for C, _ in mem)
    comp_budget = sum(bh * tc for C, tc in comp)
    total = sum(C for C, _ in ops)
    # Theorem 1 regime: budget below the memory-bound ops' peaks; the time is
    # sum_mem (C - b)/B_g with all budget on memory-bound ops, plus T_comp of the others
    D1 = 0.5 * mem_budget
    obj1, _ = op.exhaustive_continuous(ops, bh, bg, D1, mode="eq")
    t1 = (sum(C for C, _ in mem) - D1) / bg + sum(tc for _, tc in comp)
    assert obj1 == pytest.approx(t1, rel=1e-10)
    # Theorem 2 regime: sum_mem C/(B_h+B_g) + sum_comp C/B_i  (C/B_i = T_comp)
    D2 = mem_budget + 0.5 * comp_budget
    obj2, _ = op.exhaustive_continuous(ops, bh, bg, D2, mode="eq")
    t2 = sum(C / (bh + bg) for C, _ in mem) + sum(tc for _, tc in comp)
    assert obj2 == pytest.approx(t2, rel=1e-10)
    # Theorem 3 regime: every op past its turning point, time = D / B_h
    D3 = mem_budget + comp_budget + 0.3 * (total - mem_budget - comp_budget)
    obj3, _ = op.exhaustive_continuous(ops, bh, bg, D3, mode="eq")
    assert obj3 == pytest.approx(D3 / bh, rel=1e-10)


def test_ge_mode_takes_free_gains():
    bh, bg = 0.9e12, 4.0e12
    ops = [(1e9, 0.0), (2e9, 0.0)]
    obj, b = op.exhaustive_continuous(ops, bh, bg, 0.0, mode="ge")
    assert obj == pytest.approx(3e9 / (bh + bg), rel=1e-12)
    obj_eq, _ = op.exhaustive_continuous(ops, bh, bg, 0.0, mode="eq")
    assert obj_eq == pytest.approx(3e9 / bg)


def test_infeasible_budget():
    obj, b = op.exhaustive_continuous([(1e9, 0.0)], 1e11, 1e12, 2e9)
    assert obj == math.inf and b is None


def test_tiles_converge_to_continuous_with_fine_tiles():
    bh, bg = 0.9e12, 4.0e12
    ops = [(1.6e9, 0.0), (0.8e9, 1e-3)]
    D = 0.45e9
    cont, _ = op.exhaustive_continuous(ops, bh, bg, D, mode="ge")
    tiles, _ = op.exhaustive_tiles(ops, [0.1e9, 0.05e9], bh, bg, D)
    assert tiles >= cont - 1e-15
    assert tiles == pytest.approx(cont, rel=0.05)


def test_uniform_is_never_better():
    bh, bg = 0.9e12, 4.0e12
    for seed in range(4):
        ops = _ops(seed + 10, 4)
        for r in (0.05, 0.2, 0.5):
            D = r * sum(C for C, _ in ops)
            best, _ = op.exhaustive_continuous(ops, bh, bg, D, mode="eq")
            uni = op.objective(ops, op.uniform_plan(ops, r), bh, bg)
            assert best <= uni * (1 + 1e-12)


# ------------------------------ placement ------------------------------------------------

@pytest.mark.parametrize("fixture", ["fig10_global_ratio.txt", "fig14_global_ratio.txt"])
def test_global_ratio_matches_printed_tables(fixture):
    H = 96.0  # GB, GH200 (section 6, Testbed)
    for _, _, w, kv, pct in read_golden(fixture):
        x = opl.global_ratio(float(w) + float(kv), H)
        assert abs(100 * x - float(pct)) <= 1.5, (w, kv, pct, 100 * x)


def test_table1_host_traffic():
    host = 7168 * 7168 * 2
    for n, val, unit, amp in read_golden("table1_host_traffic.txt"):
        t = opl.host_link_traffic(host, int(n), 256)
        scale = 1e6 if unit == "MB" else 1e9
        printed = float(val)
        digits = len(val.split(".")[1])
        assert abs(t / scale - printed) <= 0.5 * 10 ** -digits + 1e-12
        assert abs(t / 1e6 / 98 - float(amp)) <= 0.005 + 1e-12


def test_tile_counts():
    assert opl.n_tiles(1024, 64) == 16
    assert opl.n_host_tiles(0.25, 1024, 64) == 4
    assert opl.n_host_tiles(0.0, 1024, 64) == 0
    assert opl.n_host_tiles(1.0, 1024, 64) == 16
    assert opl.n_host_tiles(0.05, 6144, 64) == 5  # ceil(4.8)
    assert opl.n_tiles(130, 64) == 3
    assert opl.n_host_requests(0.125, 32) == 4


def test_tier_roofline_limits():
    C = 1e9
    assert opl.tier_roofline(C, 0.0, 1e11, 7e12) == pytest.approx(7e12)
    xb = 1e11 / (1e11 + 7e12)
    assert opl.tier_roofline(C, xb, 1e11, 7e12) == pytest.approx(7.1e12)
    assert opl.tier_roofline(C, 0.5, 1e11, 7e12) == pytest.approx(2e11)


# ------------------------------ effective bandwidth and whole-tile search, hand values ------

def test_effective_bandwidth_memory_bound_hand_values():
    """EB(x) of a memory-bound op ([DAK] section 4.2.1, Fig. 6) at C = 1 GB, B_h = 100 GB/s,
    B_g = 400 GB/s, worked by hand: all in HBM 400; at x* = 0.2 the two transfers take
    2 ms each, EB = 500 = B_h + B_g; at x = 0.5 the host half takes 5 ms, EB = 200; all on
    the host 100."""
    C, bh, bg = 1e9, 100e9, 400e9
    for x, eb in ((0.0, 400e9), (0.2, 500e9), (0.5, 200e9), (1.0, 100e9), (0.1, 1e9 / 2.25e-3)):
        assert op.effective_bandwidth(C, 0.0, x, bh, bg) == pytest.approx(eb, rel=1e-12), x


def test_effective_bandwidth_compute_bound_hand_values():
    """A compute-bound op (T_comp = 4 ms > C / B_g = 2.5 ms): EB stays at C / T_comp = 250 GB/s
    until the host part takes 4 ms (x = 0.4), then falls as C / (x C / B_h): 1/6 TB/s at 0.6."""
    C, tc, bh, bg = 1e9, 4e-3, 100e9, 400e9
    for x, eb in ((0.0, 250e9), (0.25, 250e9), (0.4, 250e9), (0.6, 1e9 / 6e-3), (1.0, 100e9)):
        assert op.effective_bandwidth(C, tc, x, bh, bg) == pytest.approx(eb, rel=1e-12), x


def test_exhaustive_tiles_hand_case_fully_offloaded_op():
    """Two ops, three whole tiles (unit bandwidths B_h = B_g = 1). Op 0: C = 2.5 in tiles of 1
    (grid 0, 1, 2, 2.5: the last tile ragged), no compute; op 1: C = 1 in one tile,
    T_comp = 0.9. Worked by hand over every grid point:
      D = 2:   (1, 1) -> max(1.5, 1) + max(0.9, 0, 1) = 2.5   (best; op 1 at b = C)
               (2, 0) -> 2 + 1 = 3, (2, 1) -> 3, (2.5, 0) -> 3.5, (2.5, 1) -> 3.5
      D = 3.5: only (2.5, 1) -> 2.5 + 1 = 3.5                   (both ops at b = C)
    A search that dropped the last grid point of an op, or put op 0's last point at 3,
    would miss these optima."""
    ops = [(2.5, 0.0), (1.0, 0.9)]
    obj, b = op.exhaustive_tiles(ops, [1.0, 1.0], 1.0, 1.0, 2.0)
    assert obj == pytest.approx(2.5, abs=1e-12)
    assert b == [1.0, 1.0]
    obj, b = op.exhaustive_tiles(ops, [1.0, 1.0], 1.0, 1.0, 3.5)
    assert obj == pytest.approx(3.5, abs=1e-12)
    assert b == [2.5, 1.0]
    obj, b = op.exhaustive_tiles(ops, [1.0, 1.0], 1.0, 1.0, 4.0)  # more than both ops hold
    assert obj == math.inf and b is None
