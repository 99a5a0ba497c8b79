"""SplitK_GEMM over placements of 128-row tiles (tile_m = 128), through the C ABI, against the
CPU oracle. A 128-row tile is one unit of work and one M = 128 tcgen05 MMA per K step (one
FMA block of 128 rows on the CUDA cores); the host / HBM split moves in whole 128-row tiles
(section 4.1's T = ceil(M / m) with m = 128). The product is the same matrix product, so
every parity bound of the 64-row placement applies unchanged."""
import numpy as np
import pytest

import synth
from gpu_util import FP32_OUT_TOL, REL_TOL, bits_of, check_errors, to_dev, to_np
from oracle import bf16 as obf
from oracle import gemm as og
from oracle import placement as opl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dak(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    import direct_host_memory_gb300 as m
    return m


def _run(dak, A, B, h, fp32=True, tuning=None, tile_m=128):
    import torch
    p = dak.dak_place_matrix(A, h, tile_m=tile_m)
    C = dak.dak_gemm(p, to_dev(B), c_fp32=fp32, tuning=tuning)
    st, info = dak.dak_last_error()
    assert st == 0, f"device status {st} info {info:#x}"
    p.free()
    torch.cuda.synchronize()
    return C


def test_placement_counts_128_row_tiles(dak):
    A, _ = synth.gemm_inputs(320, 256, 1, seed=1)
    p = dak.dak_place_matrix(A, 1, tile_m=128)
    info = dak.dak_placement_info(p)
    assert (info["units"], info["host_units"]) == (3, 1)  # ceil(320 / 128) tiles, one on the host
    assert info["host_bytes"] == 128 * 256 * 2
    p.free()
    with pytest.raises(dak.DakError):
        dak.dak_place_matrix(A, 4, tile_m=128)  # more host tiles than tiles
    with pytest.raises(dak.DakError):
        dak.dak_place_matrix(A, 0, tile_m=96)  # 64 and 128 only


@pytest.mark.parametrize("N", [1, 2, 8, 16, 24, 64, 128, 136, 200, 256])
def test_widths(dak, N):
    M, K = 320, 1280  # 2.5 tiles of 128: the last tile's second half lies past M
    A, B = synth.gemm_inputs(M, K, N, seed=N)
    ref = og.gemm_ref(A, B)
    for h in (0, 1, 3):
        check_errors(to_np(_run(dak, A, B, h)), ref, FP32_OUT_TOL, f"gemm tile128 N={N} h={h}")
    check_errors(to_np(_run(dak, A, B, 2, fp32=False)), ref, REL_TOL, f"gemm tile128 bf16 N={N}")


@pytest.mark.parametrize("M,K", [(200, 520), (64, 8), (130, 1000), (1, 16), (65, 4104), (1000, 24), (384, 64)])
@pytest.mark.parametrize("N", [1, 13, 130])
def test_ragged_shapes(dak, M, K, N):
    A, B = synth.gemm_inputs(M, K, N, seed=M + K)
    T = opl.n_tiles(M, 128)
    ref = og.gemm_ref(A, B)
    for h in sorted({0, T // 2, T}):
        assert og.rel_err(to_np(_run(dak, A, B, h)), ref) <= FP32_OUT_TOL, (h,)


@pytest.mark.parametrize("N", [1, 64, 128, 256])
def test_integer_inputs_bit_exact(dak, N):
    """Integer-valued bf16 inputs in [-8, 8]: every partial sum is exact in fp32."""
    M, K = 384, 4096
    A, B = synth.gemm_inputs(M, K, N, seed=7, integer=True)
    ref = og.gemm_ref(A, B)
    assert np.array_equal(to_np(_run(dak, A, B, 1)), ref)
    assert np.array_equal(bits_of(_run(dak, A, B, 1, fp32=False)), obf.round_f64_to_bf16(ref))


@pytest.mark.parametrize("N", [1, 16, 64, 128, 200, 256])
def test_bit_identical_across_offload_ratio(dak, N):
    M, K = 640, 2048  # 5 tiles of 128
    A, B = synth.gemm_inputs(M, K, N, seed=3)
    base = bits_of(_run(dak, A, B, 0))
    for h in range(1, 6):
        assert np.array_equal(bits_of(_run(dak, A, B, h)), base), h


@pytest.mark.parametrize("N", [1, 16, 128, 256])
def test_same_bits_as_64_row_tiles(dak, N):
    """One piece per tile and the same K order: a row's fp32 sum is the same whether its
    tile is a 64-row (M = 64) or a 128-row (M = 128) unit."""
    M, K = 640, 2048
    A, B = synth.gemm_inputs(M, K, N, seed=5)
    tun = dict(split_k=1)
    a = bits_of(_run(dak, A, B, 0, tuning=tun, tile_m=64))
    b = bits_of(_run(dak, A, B, 0, tuning=tun, tile_m=128))
    assert np.array_equal(a, b)


@pytest.mark.parametrize("N", [1, 32, 128])
@pytest.mark.parametrize("S", [2, 3, 4, 8])
def test_split_pieces(dak, N, S):
    """A tile's K range cut into S pieces; the CTA finishing the last piece adds the 128-row
    partials in piece order: matches the oracle and is identical for every offload ratio."""
    M, K = 384 + 64, 3072  # 4 tiles of 128, the last half past M
    A, B = synth.gemm_inputs(M, K, N, seed=S * 100 + N)
    ref = og.gemm_ref(A, B)
    tun = dict(split_k=S)
    base = _run(dak, A, B, 0, tuning=tun)
    assert og.rel_err(to_np(base), ref) <= FP32_OUT_TOL
    for h in (1, 2, 4):
        assert np.array_equal(bits_of(_run(dak, A, B, h, tuning=tun)), bits_of(base)), h


@pytest.mark.parametrize("N", [300, 512, 1024])
def test_large_n_clusters(dak, N):
    """N > 256: clusters sharing each 128-row tile (rank 0 forwards host tiles)."""
    M, K = 320, 1280
    A, B = synth.gemm_inputs(M, K, N, seed=N + 1)
    ref = og.gemm_ref(A, B)
    base = _run(dak, A, B, 0)
    assert og.rel_err(to_np(base), ref) <= FP32_OUT_TOL
    for h in (1, 3):
        assert np.array_equal(bits_of(_run(dak, A, B, h)), bits_of(base)), h


@pytest.mark.parametrize("N", [1, 16, 130])
def test_glu_placement(dak, N):
    from oracle import decoder as od
    f, K = 288, 640  # 2f = 576 rows: 4.5 tiles of 128
    A, B = synth.gemm_inputs(2 * f, K, N, seed=500 + N)
    ref = od.swiglu(og.gemm_ref(A, B), f)
    outs = []
    for h in (0, 2, 5):
        p = dak.dak_place_matrix_glu(A, h, tile_m=128)
        C = dak.dak_gemm(p, to_dev(B), c_fp32=True)
        C3 = dak.dak_gemm(p, to_dev(B), c_fp32=True, tuning=dict(split_k=3))
        assert dak.dak_last_error()[0] == 0
        assert og.rel_err(to_np(C), ref) <= FP32_OUT_TOL, h
        assert og.rel_err(to_np(C3), ref) <= FP32_OUT_TOL, h
        outs.append(bits_of(C))
        p.free()
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


@pytest.mark.parametrize("N", [16, 128])
def test_chain_of_128_row_placements(dak, N):
    """A chain over 128-row placements equals the separate launches bit for bit; a chain
    mixing tile heights is refused."""
    shapes = [(640, 1024), (1000, 520), (384, 4096)]
    mats = [synth.gemm_inputs(M, K, N, seed=40 + i)[0] for i, (M, K) in enumerate(shapes)]
    Bbits = [synth.normal_bf16(50 + i, 2, N * K).reshape(N, K) for i, (M, K) in enumerate(shapes)]
    Bs = [to_dev(b) for b in Bbits]
    pls = [dak.dak_place_matrix(A, 1, tile_m=128) for A in mats]
    ops = [dict(A=p, B=B, c_fp32=True) for p, B in zip(pls, Bs)]
    got = dak.dak_gemm_chain(ops)
    assert dak.dak_last_error()[0] == 0
    for g, o, A, B in zip(got, ops, mats, Bbits):
        sep = dak.dak_gemm(o["A"], o["B"], c_fp32=True)
        assert np.array_equal(bits_of(g), bits_of(sep))
        assert og.rel_err(to_np(g), og.gemm_ref(A, B)) <= FP32_OUT_TOL
    p64 = dak.dak_place_matrix(mats[0], 1)
    with pytest.raises(dak.DakError):
        dak.dak_gemm_chain([dict(A=p64, B=Bs[0]), ops[1]])
    for p in pls + [p64]:
        p.free()


@pytest.mark.parametrize("N", [1, 128])
def test_chain_of_128_row_8b_linears_dealt_by_size(dak, N):
    """The four 8B-shaped linears in 128-row tiles, all in HBM, as one chain: at N = 128 the
    chain deals its pair blocks by size (the busiest CTA 20% over the mean dealt per
    operation), at N = 1 per operation; either way the same bits as the other dealing and
    (N = 128) as the separate launches."""
    import torch
    shapes = list(synth.LINEARS_8B.values())
    plan = dak.dak_gemm_chain_plan(shapes, N, tile_m=[128] * 4)
    assert plan["by_size"] == (1 if N == 128 else 0)  # on a 152-SM GB300
    lin = [synth.gemm_inputs(M, K, N, seed=190 + i, tensor_index=i) for i, (M, K) in enumerate(shapes)]
    pls = [dak.dak_place_matrix(A, 0, tile_m=128) for A, _ in lin]
    Bs = [to_dev(B) for _, B in lin]
    ops = [dict(A=p, B=B, c_fp32=True) for p, B in zip(pls, Bs)]
    outs = {}
    for rr in (0, 1):
        Cs = [torch.full((N, A.shape[0]), float("nan"), device="cuda") for A, _ in lin]
        dak.dak_gemm_chain([dict(o, C=C) for o, C in zip(ops, Cs)], tuning=dict(pdl=1, chain_rr=rr))
        st, info = dak.dak_last_error()
        assert st == 0, f"device status {st} info {info:#x}"
        outs[rr] = [bits_of(C) for C in Cs]
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a, b)
    if N > 1:
        for o, a in zip(ops, outs[0]):
            assert np.array_equal(bits_of(dak.dak_gemm(o["A"], o["B"], c_fp32=True)), a)
    rows = np.arange(0, shapes[3][0], 257)
    ref = og.gemm_ref(lin[3][0][rows], lin[3][1])
    assert og.rel_err(outs[0][3].view(np.float32)[:, rows], ref) <= FP32_OUT_TOL
    for p in pls:
        p.free()


@pytest.mark.slow
@pytest.mark.parametrize("N", [128, 256, 512])
def test_gate_up_full_size_sampled(dak, N):
    """The 8B gate+up weight (28672 x 4096) in 128-row tiles at x = 0.25, sampled rows of C
    against the oracle's row-by-row product."""
    import torch
    M, K = synth.LINEARS_8B["gate_up"]
    A, _ = synth.gemm_inputs(M, K, 1, seed=0, tensor_index=2)
    B = synth.normal_bf16(900 + N, 2, N * K).reshape(N, K)
    p = dak.dak_place_matrix(to_dev(A), dak.host_tiles_for_ratio(0.25, M, 128), tile_m=128)
    C = dak.dak_gemm(p, to_dev(B), c_fp32=True)
    assert dak.dak_last_error()[0] == 0
    rows = np.random.default_rng(N).choice(M, 256, replace=False)
    got = C.cpu().numpy()[:, rows]
    ref = og.gemm_ref(A[rows], B)
    check_errors(got, ref, FP32_OUT_TOL, f"gate_up tile128 N={N} sampled")
    p.free()
    torch.cuda.synchronize()


@pytest.mark.parametrize("tile_m", [64, 128])
def test_cluster_slots_keep_results(dak, tile_m):
    """Cluster launches (N > 256) size their persistent grid to the clusters the GPU holds at
    once; the launch plan reports the count it uses, and scheduling for fewer clusters moves
    work between CTAs without changing a bit of the result."""
    M, K, N = 640, 1024, 600
    A, B = synth.gemm_inputs(M, K, N, seed=11)
    p = dak.dak_place_matrix(A, 2, tile_m=tile_m)
    lp = dak.dak_gemm_launch_plan(p, N)
    assert lp["cluster"] == 3 and lp["tile_m"] == tile_m
    assert 1 <= lp["cluster_slots"] <= dak.dak_sm_count() // 3
    assert (lp["host_ctas"] + lp["hbm_ctas"]) // 3 <= lp["cluster_slots"]
    Bd = to_dev(B)
    base = bits_of(dak.dak_gemm(p, Bd, c_fp32=True))
    for cs in (2, 5, lp["cluster_slots"]):
        tun = dict(cluster_slots=cs)
        assert dak.dak_gemm_launch_plan(p, N, tuning=tun)["cluster_slots"] == cs
        assert np.array_equal(bits_of(dak.dak_gemm(p, Bd, c_fp32=True, tuning=tun)), base), cs
    assert dak.dak_last_error()[0] == 0
    assert og.rel_err(to_np(dak.dak_gemm(p, Bd, c_fp32=True)), og.gemm_ref(A, B)) <= FP32_OUT_TOL
    p.free()
