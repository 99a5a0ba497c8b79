"""The arithmetic bench.py reports with, on the CPU: the tier-aggregate roofline and the
decode step's planner view (bytes, compute times and placement units per operation)."""
import math

import pytest

import bench
import synth

pytestmark = pytest.mark.cpu


def test_tier_roofline_special_points():
    C, bh, bg = 1.5e9, 211e9, 7.3e12
    assert bench.tier_roofline(C, 0.0, bh, bg) == pytest.approx(bg)  # all in HBM
    assert bench.tier_roofline(C, 1.0, bh, bg) == pytest.approx(bh)  # all on the host
    xs = bh / (bh + bg)  # both tiers finish together: the two bandwidths add
    assert bench.tier_roofline(C, xs, bh, bg) == pytest.approx(bh + bg)
    # on either side of x* one tier bounds the time
    for x in (0.5 * xs, 2 * xs, 0.25, 0.5):
        t = max(x * C / bh, (1 - x) * C / bg)
        assert bench.tier_roofline(C, x, bh, bg) == pytest.approx(C / t)
        assert bench.tier_roofline(C, x, bh, bg) <= bh + bg


def test_decode_ops_bytes_and_units():
    cfg = dict(synth.DECODER_8B)
    ops, meta = bench.decode_ops(cfg, peak_flops=1.7e15)
    names = [k for k, _ in meta]
    assert names == ["qkv", "o", "gate_up", "down", "kv_heads"]
    nl, B, L = cfg["n_layers"], cfg["batch"], cfg["context"]
    d, f, D = cfg["hidden"], cfg["ffn"], cfg["head_dim"]
    qkv_rows = (cfg["n_heads"] + 2 * cfg["n_kv_heads"]) * D
    want = {"qkv": qkv_rows * d, "o": d * cfg["n_heads"] * D, "gate_up": 2 * f * d, "down": d * f}
    for (C, tc, tile), (k, units) in zip(ops, meta):
        if k == "kv_heads":
            per_slab = 2 * L * D * 2  # K and V of one (request, kv head)
            Hkv = cfg["n_kv_heads"]
            assert C == nl * B * Hkv * per_slab and tile == per_slab and units == B * Hkv
        else:
            assert C == nl * want[k] * 2
            M = want[k] // (d if k != "down" else f)
            assert units == math.ceil(M / 64)
            assert tile == 64 * (C // (nl * 2 * M)) * 2  # one 64-row tile row of K columns
            assert tc == pytest.approx(nl * 2.0 * want[k] * B / 1.7e15)
    # one step of the 8B shape: 22.5 GB of weights and KV
    assert sum(o[0] for o in ops) == pytest.approx(22.55e9, rel=2e-3)


def test_ratio_to_units_matches_the_oracle():
    """The package's caller-side rounding of a ratio to host units (tile rows, requests,
    (request, kv head) slabs) is the oracle's ceil(x * units)."""
    import __graft_entry__
    __graft_entry__.build()
    import direct_host_memory_gb300 as dak
    from oracle import placement as opl
    for x in (0.0, 0.01, 0.03, 0.05, 0.1, 0.125, 0.25, 1 / 3, 0.5, 0.99, 1.0):
        for M in (64, 1000, 6144, 28672):
            assert dak.host_tiles_for_ratio(x, M) == opl.n_host_tiles(x, M, 64)
            assert dak.host_tiles_for_ratio(x, M, 128) == opl.n_host_tiles(x, M, 128)
        for B, Hkv in ((1, 8), (16, 8), (32, 8), (5, 2)):
            assert dak.host_requests_for_ratio(x, B) == opl.n_host_requests(x, B)
            assert dak.host_heads_for_ratio(x, B, Hkv) == opl.n_host_requests(x, B * Hkv)
