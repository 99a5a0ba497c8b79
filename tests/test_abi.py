"""The C ABI without a GPU: the library loads, exports every declared symbol, validates
arguments, and its host-only planner matches the oracle's exhaustive search."""
import ctypes
import os
import re

import pytest

import synth
from conftest import ROOT
from oracle import planner as op

pytestmark = pytest.mark.cpu


@pytest.fixture(scope="module")
def dak():
    import __graft_entry__
    __graft_entry__.build()
    import direct_host_memory_gb300 as m
    return m


def _declared():
    src = open(os.path.join(ROOT, "include", "dak.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dak_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(dak):
    names = _declared()
    assert len(names) >= 15
    lib = ctypes.CDLL(dak._lib.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(dak.EXPORTS)


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++11")])
def test_header_compiles_standalone(lang, std, tmp_path):
    """include/dak.h is plain C: it compiles on its own as C99 (pedantic) and as C++."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("t.c" if lang == "c" else "t.cpp")
    src.write_text('#include "dak.h"\nint main(void) { dak_gemm_plan_info i; dak_tuning t; (void)i; (void)t;'
                   ' return 0; }\n')
    inc = os.path.join(ROOT, "include")
    r = subprocess.run([cc, std, "-Wall", "-Wextra", "-pedantic", "-Werror", "-fsyntax-only", "-I", inc, str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_status_strings(dak):
    assert dak.lib.dak_status_string(0) == b"ok"
    assert dak.lib.dak_status_string(6) == b"kernel wait timed out"


def test_link_begin_rejects_bad_slots(dak):
    """Handoff sequences are slots 1..8; any other slot is refused before any CUDA call."""
    for slot in (0, -1, 9, 1 << 20):
        assert dak.lib.dak_link_begin(slot, None) == 1  # DAK_ERR_INVALID


def test_planner_rejects_bad_arguments(dak):
    with pytest.raises(dak.DakError):
        dak.dak_plan_ratios([(1e9, 0.0)], 1e11, 1e12, 2e9)  # budget above the total
    with pytest.raises(dak.DakError):
        dak.dak_plan_ratios([(1e9, 0.0)], -1.0, 1e12, 0.0)
    with pytest.raises(dak.DakError):
        dak.dak_plan_ratios([(1e9, 0.0)], 1e11, 1e12, 0.0, mode=7)
    r, t = dak.dak_plan_ratios([], 1e11, 1e12, 0.0)
    assert t == 0.0


def _ops(seed, n, tiles=False):
    u = synth.uniform_f64(seed, 5, 3 * n)
    ops = []
    for i in range(n):
        C = float(int((0.1 + u[3 * i]) * 16)) * 64e6  # whole 64 MB tiles
        kind = u[3 * i + 1]
        if kind < 0.4:
            tc = 0.0
        elif kind < 0.7:
            tc = C / (1e12 * (1.0 + 2.5 * u[3 * i + 2]))  # compute-bound
        else:
            tc = C / 6e12 * u[3 * i + 2]  # memory-bound with some compute
        ops.append((C, tc, 64e6) if tiles else (C, tc))
    return ops


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("mode", [0, 1])
def test_planner_continuous_matches_exhaustive(dak, seed, mode):
    bh, bg = 0.35e12, 6.7e12
    ops = _ops(seed, 4)
    total = sum(C for C, _ in ops)
    u = synth.uniform_f64(seed, 6, 1)[0]
    D = u * 0.7 * total
    ratios, t = dak.dak_plan_ratios(ops, bh, bg, D, mode=mode)
    ref, _ = op.exhaustive_continuous(ops, bh, bg, D, mode="eq" if mode == 1 else "ge")
    assert t == pytest.approx(ref, rel=1e-9, abs=1e-15)
    b = [r * C for r, (C, _) in zip(ratios, ops)]
    assert op.objective(ops, b, bh, bg) == pytest.approx(t, rel=1e-12)
    if mode == 1:
        assert sum(b) == pytest.approx(D, rel=1e-9, abs=1.0)
    else:
        assert sum(b) >= D * (1 - 1e-9) - 1.0


@pytest.mark.parametrize("seed", range(8))
def test_planner_tiles_matches_brute_force(dak, seed):
    bh, bg = 0.35e12, 6.7e12
    ops = [(C, tc, t) for C, tc, t in _ops(100 + seed, 3, tiles=True)]
    total = sum(o[0] for o in ops)
    D = synth.uniform_f64(seed, 7, 1)[0] * 0.6 * total
    ratios, t = dak.dak_plan_ratios(ops, bh, bg, D, mode=2)
    ref, _ = op.exhaustive_tiles([(C, tc) for C, tc, _ in ops], [o[2] for o in ops], bh, bg, D)
    assert t == pytest.approx(ref, rel=1e-12)
    b = [r * o[0] for r, o in zip(ratios, ops)]
    assert sum(b) >= D - 1.0
    for bi, o in zip(b, ops):
        assert abs(bi / o[2] - round(bi / o[2])) < 1e-9 or abs(bi - o[0]) < 1.0


def test_planner_single_op_turning_points(dak):
    bh, bg = 0.9e12, 4.0e12
    r, _ = dak.dak_plan_ratios([(1e9, 0.0)], bh, bg, 0.0, mode=0)
    assert r[0] == pytest.approx(op.turning_point_memory_bound(bh, bg), rel=1e-12)
    # compute-bound: the capacity budget lands on the flat segment at no cost
    C, tc = 1e9, 1e-3
    xt = op.turning_point_compute_bound(C, tc, bh)
    r, t = dak.dak_plan_ratios([(C, tc)], bh, bg, 0.5 * xt * C, mode=1)
    assert t == pytest.approx(tc) and r[0] == pytest.approx(0.5 * xt)


@pytest.mark.parametrize("seed", range(8))
def test_plan_units_near_exhaustive_optimum(dak, seed):
    """Whole-unit placement: meets the budget, never beats the exhaustive whole-tile optimum
    and stays within one unit's host time per operation of it."""
    bh, bg = 0.35e12, 6.7e12
    ops = [(C, tc, t) for C, tc, t in _ops(200 + seed, 3, tiles=True)]
    total = sum(o[0] for o in ops)
    D = synth.uniform_f64(seed, 8, 1)[0] * 0.6 * total
    units, t = dak.dak_plan_units(ops, bh, bg, D)
    b = [min(o[0], u * o[2]) for u, o in zip(units, ops)]
    assert sum(b) >= D * (1 - 1e-12)
    assert op.objective([(C, tc) for C, tc, _ in ops], b, bh, bg) == pytest.approx(t, rel=1e-12)
    ref, _ = op.exhaustive_tiles([(C, tc) for C, tc, _ in ops], [o[2] for o in ops], bh, bg, D)
    assert t >= ref * (1 - 1e-12)
    assert t <= ref + sum(o[2] for o in ops) / bh


def test_plan_units_memory_bound_ops_stay_uniform(dak):
    """All operations memory-bound and host-bound at the budget (one decode layer's shapes):
    the model time is the host bytes over B_host, the budget is overshot by less than the
    smallest unit, and operations with the same unit size end at the same ratio to within
    one unit (the top-up goes to the cheapest units, lowest ratio first)."""
    bh, bg = 211e9, 7.3e12
    M = 1 << 20
    ops = [(48 * M, 0.0, M // 2), (32 * M, 0.0, M // 2), (224 * M, 0.0, M // 2), (112 * M, 0.0, 7 * M // 4),
           (256 * M, 0.0, 16 * M)]
    total = sum(o[0] for o in ops)
    units, t = dak.dak_plan_units(ops, bh, bg, 0.3 * total)
    host = sum(min(o[0], u * o[2]) for u, o in zip(units, ops))
    assert 0.3 * total <= host < 0.3 * total + M // 2
    assert t == pytest.approx(host / bh, rel=1e-12)
    small = [u / -(-o[0] // o[2]) for u, o in zip(units, ops) if o[2] == M // 2]
    assert max(small) - min(small) <= 1.0 / 64 + 1e-12


def test_plan_units_rejects_bad_arguments(dak):
    with pytest.raises(dak.DakError):
        dak.dak_plan_units([(1e9, 0.0, 0.0)], 1e11, 1e12, 0.0)  # no unit size
    with pytest.raises(dak.DakError):
        dak.dak_plan_units([(1e9, 0.0, 1e6)], 1e11, 1e12, 2e9)  # budget above the bytes
