"""dak_gemm_plan: the launch decisions of dak_gemm (pieces per tile row, ring layout, CTAs of
each role) from host arithmetic alone, checked on the CPU.

The piece rule and the chunk rule were fitted to measurements on a 152-SM GB300; the
tables below pin the choices they make for the decode linears of the 8B- and 70B-shaped
models, so that a change to the rule shows up here. The invariants hold for any shape:
every unit has a CTA, no tail wave is partial, and the pieces (hence the order of every
fp32 sum) do not depend on how many tile rows sit in host memory.
"""
import itertools
import random

import pytest

import direct_host_memory_gb300 as dak

SMS = 152
LINEARS_8B = {"qkv": (6144, 4096), "o": (4096, 4096), "gate_up": (28672, 4096), "down": (4096, 14336)}
LINEARS_70B = {"qkv": (10240, 8192), "o": (8192, 8192), "gate_up": (57344, 8192), "down": (8192, 28672)}


def plan(M, K, h, N, **kw):
    return dak.dak_gemm_plan(M, K, h, N, sm_count=kw.pop("sms", SMS), **kw)


@pytest.mark.parametrize("N,expect", [(16, {"qkv": 3, "o": 2, "gate_up": 1, "down": 7}),
                                      (32, {"qkv": 1, "o": 2, "gate_up": 1, "down": 2})])
def test_pieces_8b(N, expect):
    assert {k: plan(M, K, 0, N)["pieces"] for k, (M, K) in LINEARS_8B.items()} == expect


def test_pieces_70b():
    got = {k: plan(M, K, 0, 16)["pieces"] for k, (M, K) in LINEARS_70B.items()}
    assert got == {"qkv": 3, "o": 1, "gate_up": 1, "down": 7}


@pytest.mark.parametrize("N,n_pad,chunk", [(1, 8, 512), (2, 8, 512), (7, 8, 512), (8, 8, 512), (16, 16, 512),
                                           (40, 40, 512), (64, 64, 384), (128, 128, 256), (256, 256, 128)])
def test_chunk_rule(N, n_pad, chunk):
    p = plan(4096, 4096, 0, N)
    assert p["tensor_cores"] == (1 if N >= 2 else 0)
    assert p["n_pad"] == n_pad
    assert p["chunk_k"] == chunk
    assert p["hbm_stages"] >= 2
    assert p["piece_step"] == (64 if N >= 2 else 256)
    assert p["smem_bytes"] <= 216 * 1024 + 1024


def test_no_automatic_pieces_at_256_rows():
    # at 256 rows a tile row is tensor work, not bytes: pieces only when asked for
    M, K = LINEARS_8B["down"]
    assert plan(M, K, 0, 256)["pieces"] == 1
    assert plan(M, K, 0, 256, tuning={"split_k": 3})["pieces"] == 3


def test_split_k_fixes_pieces():
    M, K = LINEARS_8B["down"]
    for sk, want in ((1, 1), (2, 2), (5, 5), (8, 8), (12, 8)):
        assert plan(M, K, 5, 16, tuning={"split_k": sk})["pieces"] == want
    # a piece is at least one piece step: K = 128 leaves two steps of 64 columns
    assert plan(4096, 128, 0, 16, tuning={"split_k": 8})["pieces"] == 2
    assert plan(4096, 128, 0, 1, tuning={"split_k": 8})["pieces"] == 1


def test_caller_workspace_bounds_pieces():
    M, K = LINEARS_8B["down"]
    full = plan(M, K, 0, 16)
    assert full["pieces"] == 7
    # the partials of 7 pieces: room for T + 2 = 66 tile rows of 64 x 16 fp32 each
    assert plan(M, K, 0, 16, ws_bytes=(256 << 10) + 66 * 64 * 16 * 4 * 7)["pieces"] == 7
    # room for fewer partial tiles than 7 pieces of 64 tile rows need: fewer pieces
    small = plan(M, K, 0, 16, ws_bytes=(256 << 10) + 66 * 64 * 16 * 4 * 3)
    assert 1 <= small["pieces"] <= 3


def test_wide_b_clusters_and_launches():
    M, K = LINEARS_8B["o"]
    p = plan(M, K, 8, 512)
    # HBM tile rows: every rank streams them in the unified ring (128-column chunks at 256
    # rows); host tile rows: rank 0 fetches 256-column A-only chunks and forwards them
    assert (p["cluster"], p["n_pad"], p["launches"], p["pieces"], p["chunk_k"]) == (2, 256, 1, 1, 128)
    assert p["host_chunk_k"] == 256
    assert p["host_ctas"] % 2 == 0 and p["hbm_ctas"] % 2 == 0
    assert plan(M, K, 8, 1024)["cluster"] == 4
    assert plan(M, K, 8, 1500)["launches"] == 2
    cb = plan(M, K, 8, 1024, tuning={"column_blocks": 1})
    assert (cb["launches"], cb["cluster"]) == (4, 1)


def test_host_part_one_wave():
    # 61 host tile rows of gate+up at 16 rows (one piece each): one wave of 61 CTAs rather
    # than two waves under the cap of 48 (per-CTA timestamps on the GPU show the same split)
    M, K = LINEARS_8B["gate_up"]
    p = plan(M, K, 61, 16)
    assert (p["pieces"], p["host_ctas"], p["hbm_ctas"]) == (1, 61, 78)


def test_trace_matches_for_qkv():
    # 33 of 96 QKV tile rows on the host at 16 rows: 3 pieces, 33 host CTAs with 3 units
    # each, 95 HBM CTAs with 2 each
    M, K = LINEARS_8B["qkv"]
    p = plan(M, K, 33, 16)
    assert (p["pieces"], p["host_ctas"], p["hbm_ctas"]) == (3, 33, 95)


def _waves(units, ctas):
    return -(-units // ctas)


def _check_invariants(M, K, h, N, sms, tuning=None, tile_m=64):
    p = plan(M, K, h, N, sms=sms, tuning=tuning, tile_m=tile_m)
    assert p["tile_m"] == tile_m
    T = -(-M // tile_m)
    P, cl = p["pieces"], p["cluster"]
    # a unit is a piece of one tile (64 or 128 rows)
    hu, mu = h * P, (T - h) * P
    assert (p["host_ctas"] > 0) == (hu > 0)
    assert (p["hbm_ctas"] > 0) == (mu > 0)
    assert p["host_ctas"] + p["hbm_ctas"] <= sms
    assert p["host_ctas"] // cl <= max(hu, 0) and p["hbm_ctas"] // cl <= max(mu, 0)
    if not (tuning and tuning.get("no_wave_align")):
        # whole waves: with w waves a role has exactly ceil(units / w) CTAs
        for units, ctas in ((hu, p["host_ctas"] // cl), (mu, p["hbm_ctas"] // cl)):
            if units:
                assert ctas == -(-units // _waves(units, ctas))
    assert 1 <= p["host_window"] <= p["host_stages"]
    assert 1 <= p["hbm_window"] <= p["hbm_stages"]
    assert 1 <= P <= 8
    assert p["chunk_k"] % 64 == 0 and p["host_chunk_k"] % 64 == 0
    return p


def test_invariants_random_shapes():
    rng = random.Random(7)
    for _ in range(400):
        M = rng.choice([64, 100, 1000, 4096, 6144, 14336, 28672]) * rng.choice([1, 1, 2])
        K = 8 * rng.randint(1, 4096)
        N = rng.choice([1, 2, 5, 8, 16, 24, 32, 48, 64, 96, 128, 200, 256, 300, 512, 1024])
        tile_m = rng.choice([64, 64, 128])
        T = -(-M // tile_m)
        h = rng.randint(0, T)
        sms = rng.choice([132, 148, 152, 160])
        tun = rng.choice([None, {"no_wave_align": 1}, {"host_ctas": 16}, {"split_k": rng.randint(1, 8)}])
        _check_invariants(M, K, h, N, sms, tun, tile_m)


@pytest.mark.parametrize("tile_m", [64, 128])
@pytest.mark.parametrize("N", [1, 8, 16, 32, 64, 128, 256])
def test_pieces_do_not_depend_on_placement(N, tile_m):
    # the pieces, and so the order of every tile row's fp32 sum, come from the shape and the
    # SM count alone: the result is bit-identical at every offload ratio
    for (M, K) in itertools.chain(LINEARS_8B.values(), [(1000, 1032), (64, 8), (640, 20000)]):
        T = -(-M // tile_m)
        ps = {(plan(M, K, h, N, tile_m=tile_m)["pieces"], plan(M, K, h, N, tile_m=tile_m)["n_pad"])
              for h in sorted({0, 1, T // 3, T // 2, T - 1, T})}
        assert len(ps) == 1, (M, K, N, ps)


def test_errors():
    for args in ((0, 4096, 0, 16), (4096, 12, 0, 16), (4096, 0, 0, 16), (4096, 4096, 65, 16),
                 (4096, 4096, -1, 16), (4096, 4096, 0, 0)):
        with pytest.raises(dak.DakError):
            plan(*args)
    with pytest.raises(dak.DakError):
        plan(4096, 4096, 0, 16, sms=0)
    with pytest.raises(dak.DakError):
        plan(4096, 4096, 0, 16, ws_bytes=1000)
    with pytest.raises(dak.DakError):
        plan(4096, 4096, 0, 16, tuning={"chunk_k": 100})


def test_cluster_slots_bound_the_schedule():
    # a cluster launch schedules at most cluster_slots clusters (the count the GPU holds at
    # once; the plan API's default is sm_count / cluster)
    M, K = LINEARS_8B["gate_up"]
    for tile_m, h in ((64, 112), (128, 56)):
        for cs in (0, 36, 20, 7):
            p = plan(M, K, h, 1024, tile_m=tile_m, tuning={"cluster_slots": cs} if cs else None)
            assert p["cluster"] == 4
            assert p["cluster_slots"] == (cs or SMS // 4)
            assert (p["host_ctas"] + p["hbm_ctas"]) // 4 <= p["cluster_slots"]
            assert p["host_ctas"] > 0 and p["hbm_ctas"] > 0
    # one CTA per tile: cluster_slots counts CTAs and is not capped
    assert plan(4096, 4096, 0, 16)["cluster_slots"] == SMS


# ------------------------------------------------------------------ chains: dealing by size

FIXED_BYTES = 32 * 1024  # a unit's fixed cost in the dealing's work measure


def _chain_units(shapes, N, tile_ms):
    """Each operation's units (work, operation, unit) and its CTAs, re-derived from
    dak_gemm_plan's pieces, piece step and CTA counts (tensor cores at every N of a chain)."""
    units, ctas = [], []
    for j, ((M, K), tm) in enumerate(zip(shapes, tile_ms)):
        p = plan(M, K, 0, max(N, 2), tile_m=tm)
        blocks = -(-M // tm)
        P, step = p["pieces"], p["piece_step"]
        K_pad = -(-K // 16) * 16
        steps = -(-K_pad // step)
        for u in range(blocks * P):
            i = u % P
            k0 = (i * steps // P) * step
            k1 = min(((i + 1) * steps // P) * step, K_pad)
            units.append(((k1 - k0) * 128 * (tm // 64) + FIXED_BYTES, j, u))
        ctas.append((p["host_ctas"], p["hbm_ctas"]))
    return units, ctas


def _deal(units, ctas):
    """The busiest CTA's work over the mean (x 1000, floored) dealt per operation (unit u of
    operation j on CTA host_ctas + u mod hbm_ctas, counted from where the previous operation's
    CTAs ended) and dealt by size (longest first to the least loaded, ties to the lower CTA)."""
    grid = max(h + g for h, g in ctas)
    rot, r = [], 0
    for h, g in ctas:
        rot.append(r)
        r = (r + h + g) % grid
    per_op = [0] * grid
    for w, j, u in units:
        per_op[(ctas[j][0] + u % ctas[j][1] + rot[j]) % grid] += w
    by_size = [0] * grid
    for w, j, u in sorted(units, key=lambda x: -x[0]):
        c = min(range(grid), key=lambda i: (by_size[i], i))
        by_size[c] += w
    total = sum(per_op)
    return grid, max(per_op) * 1000 * grid // total, max(by_size) * 1000 * grid // total, max(by_size), max(per_op)


@pytest.mark.parametrize("N", [2, 8, 16, 32, 64, 128])
def test_chain_dealing_8b_linears(N):
    shapes = list(LINEARS_8B.values())
    got = dak.dak_gemm_chain_plan(shapes, N, sm_count=SMS)
    units, ctas = _chain_units(shapes, N, [64] * 4)
    grid, per_op, by_size, smax, rmax = _deal(units, ctas)
    assert got == {"grid": grid, "units": len(units), "by_size": int(smax * 100 <= rmax * 97),
                   "busiest_per_op": per_op, "busiest_by_size": by_size}
    # the pieces of a tile row at N >= 32 are few and uneven in size (896 KiB down rows beside
    # 512 and 256 KiB ones): dealt per operation the busiest CTA carries 13% over the mean
    assert got["by_size"] == (N >= 32)
    if N >= 32:
        assert (got["busiest_per_op"], got["busiest_by_size"]) == (1126, 1041)
    assert dak.dak_gemm_chain_plan(shapes, N, sm_count=SMS, tuning=dict(chain_rr=1))["by_size"] == 0


def test_chain_dealing_one_row_is_eight():
    shapes = list(LINEARS_8B.values())
    assert dak.dak_gemm_chain_plan(shapes, 1, sm_count=SMS) == dak.dak_gemm_chain_plan(shapes, 8, sm_count=SMS)


def test_chain_dealing_random_shapes():
    rng = random.Random(7)
    for case in range(12):
        n = rng.randint(1, 8)
        tms = [rng.choice([64, 128])] * n  # one ring layout (tile height) per chain
        shapes = [(rng.randint(1, 9000), 8 * rng.randint(1, 2048)) for _ in range(n)]
        N = rng.choice([2, 8, 24, 40, 64, 96])
        try:
            got = dak.dak_gemm_chain_plan(shapes, N, tile_m=tms, sm_count=SMS)
        except dak.DakError as e:
            assert e.status == 7  # operations whose launches stream with different rings
            continue
        units, ctas = _chain_units(shapes, N, tms)
        assert got["units"] == len(units), case
        if len(units) > 4096:
            assert got["by_size"] == 0 and got["busiest_per_op"] == 0, case
            continue
        grid, per_op, by_size, smax, rmax = _deal(units, ctas)
        assert got == {"grid": grid, "units": len(units), "by_size": int(smax * 100 <= rmax * 97),
                       "busiest_per_op": per_op, "busiest_by_size": by_size}, case


def test_chain_dealing_applies_only_all_hbm_and_independent():
    shapes = list(LINEARS_8B.values())
    for kw in (dict(n_host_tiles=[1, 0, 0, 0]), dict(after_prev=[0, 1, 0, 0])):
        got = dak.dak_gemm_chain_plan(shapes, 32, sm_count=SMS, **kw)
        assert (got["by_size"], got["busiest_per_op"], got["busiest_by_size"]) == (0, 0, 0), kw
        assert got["units"] == 800
    with pytest.raises(dak.DakError):
        dak.dak_gemm_chain_plan(shapes, 129, sm_count=SMS)
    with pytest.raises(dak.DakError):
        dak.dak_gemm_chain_plan([(64, 12)], 8, sm_count=SMS)  # K not a multiple of 8
