"""SplitK_GEMM on the GPU against the CPU oracle, through the C ABI."""
import numpy as np
import pytest

import synth
from gpu_util import FP32_OUT_TOL, REL_TOL, bits_of, to_dev, to_np
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


def _run(dak, A, B, h, fp32=True, tuning=None, device_src=False):
    import torch
    src = to_dev(A) if device_src else A
    p = dak.dak_place_matrix(src, h)
    C = dak.dak_gemm(p, to_dev(B), c_fp32=fp32, tuning=tuning)
    st, info = dak.dak_last_error()
    assert st == 0, f"device status {st} info {info:#x}"
    p.free()
    torch.cuda.synchronize()
    return C


def test_gemv_decode_1024(dak):
    """A 1024x1024 ~N(0,0.02), B 1x1024 ~N(0,1), m = 64, x = 0.25 (4 of 16 tile rows on the host)."""
    A, B = synth.gemm_inputs(1024, 1024, 1, seed=0)
    h = opl.n_host_tiles(0.25, 1024, 64)
    assert h == 4
    ref = og.gemm_ref(A, B)
    C32 = _run(dak, A, B, h, fp32=True)
    assert og.rel_err(to_np(C32), ref) <= FP32_OUT_TOL
    C16 = _run(dak, A, B, h, fp32=False)
    assert og.rel_err(to_np(C16), ref) <= REL_TOL
    # bf16 output is the fp32 result rounded to nearest even
    assert np.array_equal(bits_of(C16), obf.round_f32_to_bf16(C32.cpu().numpy()))


@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 7, 8, 16, 24, 32, 64, 72, 128, 256])
def test_widths(dak, N):
    M, K = 320, 1280  # 5 tile rows, 5 chunks of 256 (and 20 of 64)
    A, B = synth.gemm_inputs(M, K, N, seed=N)
    ref = og.gemm_ref(A, B)
    C = _run(dak, A, B, 2)
    assert og.rel_err(to_np(C), ref) <= FP32_OUT_TOL
    C16 = _run(dak, A, B, 2, fp32=False)
    assert og.rel_err(to_np(C16), ref) <= REL_TOL


@pytest.mark.parametrize("M,K", [(200, 520), (64, 8), (130, 1000), (1, 16), (65, 4104), (1000, 24)])
@pytest.mark.parametrize("N", [1, 8, 13])
def test_ragged_shapes(dak, M, K, N):
    A, B = synth.gemm_inputs(M, K, N, seed=M + K)
    T = opl.n_tiles(M, 64)
    ref = og.gemm_ref(A, B)
    for h in sorted({0, T // 2, T}):
        C = _run(dak, A, B, h)
        assert og.rel_err(to_np(C), ref) <= FP32_OUT_TOL, (h,)


@pytest.mark.parametrize("N", [1, 8, 64])
def test_integer_inputs_bit_exact(dak, N):
    """Integer-valued bf16 inputs in [-8, 8]: every partial sum is exact in fp32."""
    M, K = 256, 4096
    A, B = synth.gemm_inputs(M, K, N, seed=7, integer=True)
    ref = og.gemm_ref(A, B)
    C = _run(dak, A, B, 1)
    assert np.array_equal(to_np(C), ref)
    C16 = _run(dak, A, B, 1, fp32=False)
    assert np.array_equal(bits_of(C16), obf.round_f64_to_bf16(ref))


@pytest.mark.parametrize("N", [1, 4, 16, 64, 200, 256])
def test_bit_identical_across_offload_ratio(dak, N):
    M, K = 640, 2048
    A, B = synth.gemm_inputs(M, K, N, seed=3)
    base = bits_of(_run(dak, A, B, 0))
    for h in range(1, 11):
        assert np.array_equal(bits_of(_run(dak, A, B, h)), base), h


@pytest.mark.parametrize("N", [1, 16])
def test_bit_identical_across_tuning(dak, N):
    """Knobs that only move work between CTAs (host CTA count, windows, HBM CTA cap) leave
    every bit of the result unchanged; chunk width and split count change the summation
    order and are checked against the oracle instead."""
    M, K = 640, 2048
    A, B = synth.gemm_inputs(M, K, N, seed=4)
    base = bits_of(_run(dak, A, B, 4))
    for tun in [dict(host_ctas=1), dict(host_ctas=3, window=1), dict(window=2, hbm_window=2), dict(hbm_ctas=3)]:
        assert np.array_equal(bits_of(_run(dak, A, B, 4, tuning=tun)), base), tun
    ref = og.gemm_ref(A, B)
    chunks = [dict(chunk_k=256), dict(chunk_k=512)] if N == 1 else \
        [dict(chunk_k=64), dict(chunk_k=128, split_k=1), dict(chunk_k=256, split_k=2)]
    for tun in chunks:
        assert og.rel_err(to_np(_run(dak, A, B, 4, tuning=tun)), ref) <= FP32_OUT_TOL, tun


@pytest.mark.parametrize("N", [1, 8, 32, 64])
@pytest.mark.parametrize("S", [1, 2, 3, 4, 8])
def test_split_pieces(dak, N, S):
    """Each tile row's K range cut into S pieces that any CTA may take; the CTA finishing a
    tile row's last piece adds the partials in piece order: matches the oracle and is
    identical for every offload ratio."""
    M, K = 384, 3072  # 6 tile rows
    A, B = synth.gemm_inputs(M, K, N, seed=S * 100 + N)
    ref = og.gemm_ref(A, B)
    tun = dict(split_k=S)
    base = _run(dak, A, B, 0, tuning=tun)
    assert og.rel_err(to_np(base), ref) <= FP32_OUT_TOL
    for h in (1, 3, 6):
        assert np.array_equal(bits_of(_run(dak, A, B, h, tuning=tun)), bits_of(base)), h


@pytest.mark.parametrize("N", [2, 3, 5, 7])
def test_small_n_on_tensor_cores(dak, N):
    """N = 2..7 runs on the tensor cores with B padded to 8 rows (zero-filled by the tensor
    map): matches the oracle, writes only the N real rows of C, and keeps its bits across
    offload ratios; ragged M and K."""
    import torch
    M, K = 328, 1000
    A, B = synth.gemm_inputs(M, K, N, seed=60 + N)
    ref = og.gemm_ref(A, B)
    base = _run(dak, A, B, 0)
    assert base.shape == (N, M)
    assert og.rel_err(to_np(base), ref) <= FP32_OUT_TOL
    for h in (1, 3, 6):
        assert np.array_equal(bits_of(_run(dak, A, B, h)), bits_of(base)), h
    C = torch.full((N + 1, M), 7.0, device="cuda")  # one guard row past the N rows of C
    p = dak.dak_place_matrix(A, 2)
    dak.dak_gemm(p, to_dev(B), C[:N], c_fp32=True)
    assert dak.dak_last_error()[0] == 0
    assert torch.all(C[N] == 7.0)
    assert og.rel_err(to_np(C[:N]), ref) <= FP32_OUT_TOL
    p.free()


@pytest.mark.parametrize("N", [1, 24])
@pytest.mark.parametrize("K", [1000, 1040, 4096 + 16])
def test_split_pieces_ragged_k(dak, K, N):
    """Pieces end at multiples of 64 columns except the last, which ends at K rounded up to 16;
    few CTAs (hbm_ctas, host_ctas) so that one CTA takes several pieces of one tile row (on
    the CUDA-core path, more units per CTA than the finisher's lag of four)."""
    M = 200
    A, B = synth.gemm_inputs(M, K, N, seed=K)
    ref = og.gemm_ref(A, B)
    for S in (2, 5, 8):
        for tun in (dict(split_k=S), dict(split_k=S, hbm_ctas=3, host_ctas=2)):
            C = _run(dak, A, B, 1, tuning=tun)
            assert og.rel_err(to_np(C), ref) <= FP32_OUT_TOL, tun


def test_gemm_caller_workspace(dak):
    """dak_gemm_ws: the split workspace of the caller's gives the same bits as the library's own;
    launches on two streams with workspaces of their own may overlap; a workspace that is too
    small or misaligned is refused."""
    import torch
    A1, B1 = synth.gemm_inputs(4096, 4096, 16, seed=71)
    A2, B2 = synth.gemm_inputs(6144, 1024, 16, seed=72)
    p1, p2 = dak.dak_place_matrix(A1, 5), dak.dak_place_matrix(A2, 0)
    b1, b2 = to_dev(B1), to_dev(B2)
    base1 = dak.dak_gemm(p1, b1, c_fp32=True, tuning=dict(split_k=3))
    base2 = dak.dak_gemm(p2, b2, c_fp32=True, tuning=dict(split_k=5))
    n1, n2 = dak.dak_gemm_workspace_bytes(p1, 16), dak.dak_gemm_workspace_bytes(p2, 16)
    assert n1 >= 256 * 1024 + 64 * 8 * 64 * 16 * 4 and n2 > 0
    w1 = torch.zeros(n1 // 4 + 64, dtype=torch.float32, device="cuda")
    w2 = torch.zeros(n2 // 4 + 64, dtype=torch.float32, device="cuda")
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(4):
        with torch.cuda.stream(s1):
            c1 = dak.dak_gemm(p1, b1, c_fp32=True, tuning=dict(split_k=3), workspace=w1, stream=s1)
        with torch.cuda.stream(s2):
            c2 = dak.dak_gemm(p2, b2, c_fp32=True, tuning=dict(split_k=5), workspace=w2, stream=s2)
        outs.append((c1, c2))
    torch.cuda.synchronize()
    assert dak.dak_last_error()[0] == 0
    for c1, c2 in outs:
        assert np.array_equal(bits_of(c1), bits_of(base1))
        assert np.array_equal(bits_of(c2), bits_of(base2))
    assert og.rel_err(to_np(base1), og.gemm_ref(A1, B1)) <= FP32_OUT_TOL
    # one workspace for both matrices, in turn on one stream: the counters are shared by tile row
    for _ in range(3):
        c1 = dak.dak_gemm(p1, b1, c_fp32=True, tuning=dict(split_k=3), workspace=w1)
        c2 = dak.dak_gemm(p2, b2, c_fp32=True, tuning=dict(split_k=5), workspace=w1)
    assert np.array_equal(bits_of(c1), bits_of(base1)) and np.array_equal(bits_of(c2), bits_of(base2))
    with pytest.raises(dak.DakError):
        dak.dak_gemm(p1, b1, c_fp32=True, workspace=torch.zeros(1024, device="cuda"))
    with pytest.raises(dak.DakError):
        dak.dak_gemm(p1, b1, c_fp32=True, workspace=w1[1:])  # 4-byte offset: not 256-byte aligned
    for pl in (p1, p2):
        pl.free()


def test_split_pieces_graph_replay(dak):
    """The per-tile-row piece counters return to zero after every launch: a CUDA graph of three
    split GEMMs (two sharing tile-row indices) replayed many times gives the same bits."""
    import torch
    A1, B = synth.gemm_inputs(640, 2048, 16, seed=41)
    A2, _ = synth.gemm_inputs(320, 640, 16, seed=42)
    p1, p2 = dak.dak_place_matrix(A1, 2), dak.dak_place_matrix(A2, 0)
    Bt = to_dev(B)
    C1 = torch.empty(16, 640, device="cuda", dtype=torch.float32)
    C2 = torch.empty(16, 320, device="cuda", dtype=torch.float32)
    C3 = torch.empty(16, 640, device="cuda", dtype=torch.float32)

    def step():
        dak.dak_gemm(p1, Bt, C1, c_fp32=True, tuning=dict(split_k=3, pdl=1))
        dak.dak_gemm(p2, C1.to(torch.bfloat16), C2, c_fp32=True, tuning=dict(split_k=5, pdl=1))
        dak.dak_gemm(p1, Bt, C3, c_fp32=True, tuning=dict(split_k=7, pdl=1))

    step()
    torch.cuda.synchronize()
    ref = [bits_of(x) for x in (C1, C2, C3)]
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    for _ in range(25):
        g.replay()
    torch.cuda.synchronize()
    assert dak.dak_last_error()[0] == 0
    for r, x in zip(ref, (C1, C2, C3)):
        assert np.array_equal(bits_of(x), r)
    assert og.rel_err(to_np(C1), og.gemm_ref(A1, B)) <= FP32_OUT_TOL
    for pl in (p1, p2):
        pl.free()


def test_split_k_integer_exact(dak):
    M, K, N = 256, 4096, 32
    A, B = synth.gemm_inputs(M, K, N, seed=17, integer=True)
    for S in (2, 4, 8):
        C = _run(dak, A, B, 1, tuning=dict(split_k=S))
        assert np.array_equal(to_np(C), og.gemm_ref(A, B)), S


def test_device_source_placement(dak):
    A, B = synth.gemm_inputs(384, 512, 8, seed=5)
    a = bits_of(_run(dak, A, B, 3))
    b = bits_of(_run(dak, A, B, 3, device_src=True))
    assert np.array_equal(a, b)


def test_prefetch_staged_equals_direct(dak):
    import torch
    A, B = synth.gemm_inputs(512, 1024, 8, seed=6)
    p = dak.dak_place_matrix(A, 5)
    Bt = to_dev(B)
    direct = dak.dak_gemm(p, Bt, c_fp32=True)
    staging = torch.empty(p.host_bytes, dtype=torch.uint8, device="cuda")
    dak.dak_prefetch(p, staging)
    staged = dak.dak_gemm_staged(p, staging, Bt, c_fp32=True)
    assert dak.dak_last_error()[0] == 0
    assert torch.equal(direct, staged)
    p.free()


def test_empty_and_errors(dak):
    import torch
    A = np.zeros((0, 64), dtype=np.uint16)
    p = dak.dak_place_matrix(A, 0)
    assert p.units == 0
    C = torch.empty((1, 0), dtype=torch.bfloat16, device="cuda")
    dak.dak_gemm(p, torch.zeros((1, 64), dtype=torch.bfloat16, device="cuda"), C)
    p.free()
    A2, _ = synth.gemm_inputs(64, 64, 1)
    with pytest.raises(dak.DakError):
        dak.dak_place_matrix(A2, 2)  # more host tiles than tiles
    with pytest.raises(dak.DakError):
        dak.dak_place_matrix(np.zeros((64, 60), dtype=np.uint16), 0)  # K % 8 != 0
    p = dak.dak_place_matrix(A2, 1)
    with pytest.raises(dak.DakError):
        dak.dak_gemm(p, torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda"),
                     torch.zeros((1, 64), dtype=torch.bfloat16, device="cuda"))  # N = 0
    p.free()


@pytest.mark.slow
@pytest.mark.parametrize("name", list(synth.LINEARS_8B))
@pytest.mark.parametrize("N", [1, 8, 16, 32, 64])
def test_8b_linears_full_size_sampled(dak, name, N):
    """Full-size 8B-shaped linear at x = 0.25 (N = 32: the bench's launch configuration;
    16: the decode step's batch); 96 sampled output rows (all N columns) against the
    oracle computed row by row."""
    M, K = synth.LINEARS_8B[name]
    A, B = synth.gemm_inputs(M, K, N, seed=0, tensor_index=list(synth.LINEARS_8B).index(name))
    h = opl.n_host_tiles(0.25, M, 64)
    C = to_np(_run(dak, A, B, h, fp32=False))
    rows = np.unique(np.concatenate([
        (synth.uniform_f64(1, 9, 80) * M).astype(int),
        [0, 63, 64, h * 64 - 1, h * 64, M - 1]]))
    rows = rows[(rows >= 0) & (rows < M)]
    ref = og.gemm_ref(A[rows], B)
    assert og.rel_err(C[:, rows], ref) <= REL_TOL


def test_programmatic_launch_chain(dak):
    """pdl = 1 lets a kernel start while the previous one runs; the hidden states (and Q)
    are read only after it finishes. Chain: C1 = A1.B, C2 = A2.C1, attention over Q = C1;
    every result must equal the plainly launched one bit for bit."""
    import torch
    A1, B = synth.gemm_inputs(1024, 512, 16, seed=31)
    A2, _ = synth.gemm_inputs(256, 1024, 16, seed=32)
    _, k, v = synth.attn_inputs(16, 16, 4, 64, 300, seed=33)
    p1, p2 = dak.dak_place_matrix(A1, 3), dak.dak_place_matrix(A2, 1)
    kv = dak.dak_place_kv(k, v, 5)
    Bt = to_dev(B)
    outs = []
    for pdl in (0, 1):
        tun = dict(pdl=pdl)
        C1 = dak.dak_gemm(p1, Bt, tuning=tun)
        C2 = dak.dak_gemm(p2, C1, tuning=tun)
        O = dak.dak_attn(C1.view(16, 16, 64), kv, tuning=tun)
        C3 = dak.dak_gemm(p2, C1, tuning=dict(pdl=pdl, split_k=4))
        assert dak.dak_last_error()[0] == 0
        outs.append([bits_of(x) for x in (C1, C2, O, C3)])
    for a, b in zip(*outs):
        assert np.array_equal(a, b)
    assert og.rel_err(to_np(torch.from_numpy(outs[0][1].view(np.int16)).view(torch.bfloat16)),
                      og.gemm_ref(A2, outs[0][0])) <= REL_TOL
    for p in (p1, p2, kv):
        p.free()


@pytest.mark.parametrize("cols", [0, 1])
@pytest.mark.parametrize("N", [257, 300, 512, 777, 1024, 2100])
def test_large_n(dak, N, cols):
    """N > 256, as cluster launches of up to 1024 rows in which rank 0 fetches every A chunk
    and forwards it to the other CTAs through distributed shared memory (default), or as
    column blocks of 256 rows (column_blocks = 1); matches the oracle and stays identical
    across offload ratios."""
    M, K = 320, 1280
    A, B = synth.gemm_inputs(M, K, N, seed=N + 1)
    ref = og.gemm_ref(A, B)
    tun = dict(column_blocks=cols)
    base = _run(dak, A, B, 0, tuning=tun)
    assert og.rel_err(to_np(base), ref) <= FP32_OUT_TOL
    for h in (2, 5):
        assert np.array_equal(bits_of(_run(dak, A, B, h, tuning=tun)), bits_of(base)), h
    C16 = _run(dak, A, B, 3, fp32=False, tuning=tun)
    assert og.rel_err(to_np(C16), ref) <= REL_TOL


def test_large_n_integer_exact(dak):
    M, K, N = 192, 2048, 520
    A, B = synth.gemm_inputs(M, K, N, seed=9, integer=True)
    for cols in (0, 1):
        C = _run(dak, A, B, 1, tuning=dict(pdl=1, column_blocks=cols))
        assert np.array_equal(to_np(C), og.gemm_ref(A, B)), cols


@pytest.mark.parametrize("cols", [0, 1])
def test_large_n_ragged_k_and_tuning(dak, cols):
    """K not a multiple of 64 (2-D B boxes), tuning knobs that only move work."""
    M, K, N = 200, 520, 600
    A, B = synth.gemm_inputs(M, K, N, seed=77)
    ref = og.gemm_ref(A, B)
    base = _run(dak, A, B, 1, tuning=dict(column_blocks=cols))
    assert og.rel_err(to_np(base), ref) <= FP32_OUT_TOL
    for tun in (dict(host_ctas=1, window=2), dict(no_wave_align=1), dict(pdl=1)):
        tun["column_blocks"] = cols
        assert np.array_equal(bits_of(_run(dak, A, B, 2, tuning=tun)), bits_of(base)), tun


@pytest.mark.parametrize("N", [1, 5, 16, 64, 300])
def test_glu_placement_fused_swiglu(dak, N):
    """Gate/up interleaved placement: dak_gemm returns silu(gate) * up straight from its
    accumulators; matches the oracle's swiglu of the plain product, identical across
    offload ratios."""
    from oracle import decoder as od
    f, K = 256, 640  # 2f = 512 rows = 8 tile rows
    A, B = synth.gemm_inputs(2 * f, K, N, seed=500 + N)
    ref = od.swiglu(og.gemm_ref(A, B), f)
    outs = []
    for h in (0, 3, 8):
        p = dak.dak_place_matrix_glu(A, h)
        C = dak.dak_gemm(p, to_dev(B), c_fp32=True)
        C16 = dak.dak_gemm(p, to_dev(B), c_fp32=False)
        C3 = dak.dak_gemm(p, to_dev(B), c_fp32=True, tuning=dict(split_k=3))  # summed by the last piece
        assert dak.dak_last_error()[0] == 0
        assert tuple(C.shape) == (N, f)
        assert og.rel_err(to_np(C), ref) <= FP32_OUT_TOL, h
        assert og.rel_err(to_np(C16), ref) <= REL_TOL, h
        assert og.rel_err(to_np(C3), ref) <= FP32_OUT_TOL, h
        outs.append(bits_of(C))
        p.free()
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])


def test_glu_placement_rejects_bad_shapes(dak):
    A = np.zeros((96, 64), dtype=np.uint16)  # 2f = 96: not whole tiles of 32 gate/up pairs
    with pytest.raises(dak.DakError):
        dak.dak_place_matrix_glu(A, 0)
