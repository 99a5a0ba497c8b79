"""dak_gemm_chain: several GEMMs in one persistent launch, through the C ABI. Every result
must equal the separate dak_gemm launch bit for bit (same tiering, dealing and pieces), at
every offload ratio, with and without dependencies between the operations, over repeated
launches on one workspace; and the chain must match the fp64 oracle."""
import numpy as np
import pytest

import synth
from gpu_util import FP32_OUT_TOL, REL_TOL, bits_of, to_dev, to_np
from oracle import gemm as og

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dak(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    import direct_host_memory_gb300 as m
    return m


def _separate(dak, ops, tuning=None):
    outs = []
    for o in ops:
        outs.append(dak.dak_gemm(o["A"], o["B"], c_fp32=o.get("c_fp32", False), tuning=tuning))
    assert dak.dak_last_error()[0] == 0
    return outs


SHAPES = [(640, 1024), (4096, 4096), (320, 4104), (6144, 4096), (1000, 520)]


@pytest.mark.parametrize("N", [2, 8, 16, 32, 64, 128])
def test_independent_chain_equals_separate_launches(dak, N):
    mats = [synth.gemm_inputs(M, K, N, seed=40 + i)[0] for i, (M, K) in enumerate(SHAPES)]
    Bs = [synth.normal_bf16(50 + i, 2, N * K).reshape(N, K) for i, (M, K) in enumerate(SHAPES)]
    for frac in (0.0, 0.3, 1.0):
        pls = [dak.dak_place_matrix(A, int(np.ceil(frac * -(-A.shape[0] // 64)))) for A in mats]
        ops = [dict(A=p, B=to_dev(B), c_fp32=(i % 2 == 0)) for i, (p, B) in enumerate(zip(pls, Bs))]
        got = dak.dak_gemm_chain(ops)
        st, info = dak.dak_last_error()
        assert st == 0, f"device status {st} info {info:#x}"
        ref = _separate(dak, ops)
        for g, r in zip(got, ref):
            assert np.array_equal(bits_of(g), bits_of(r))
        for g, A, B, o in zip(got, mats, Bs, ops):
            tol = FP32_OUT_TOL if o["c_fp32"] else REL_TOL
            assert og.rel_err(to_np(g), og.gemm_ref(A, B)) <= tol
        for p in pls:
            p.free()


@pytest.mark.parametrize("N", [1, 8, 32, 64])
def test_size_dealing_same_bits(dak, N):
    """An independent chain all in HBM deals its units by size over the CTAs (chain_rr = 0);
    every unit is computed once and lands where the per-operation dealing (chain_rr = 1)
    and the separate launches put it (N >= 2; at N = 1 dak_gemm runs the CUDA cores): the
    same bits, eagerly (a new chain, then the same one again) and replayed from a CUDA
    graph."""
    import torch
    lin = [synth.gemm_inputs(M, K, N, seed=170 + i, tensor_index=i) for i, (M, K) in
           enumerate(list(synth.LINEARS_8B.values()) + [(1000, 520)])]
    pls = [dak.dak_place_matrix(A, 0) for A, _ in lin]
    Bs = [to_dev(B) for _, B in lin]

    def ops(cs=None):
        return [dict(A=p, B=B, c_fp32=(i % 2 == 1), C=None if cs is None else cs[i])
                for i, (p, B) in enumerate(zip(pls, Bs))]

    def nan_outs():
        return [torch.full((N, A.shape[0]), float("nan"), device="cuda",
                           dtype=torch.float32 if i % 2 == 1 else torch.bfloat16) for i, (A, _) in enumerate(lin)]

    if N > 1:
        sep = [bits_of(c) for c in _separate(dak, ops())]
    else:
        sep = [bits_of(c) for c in dak.dak_gemm_chain(ops(), tuning=dict(pdl=1, chain_rr=1))]
    for rr in (0, 1, 0):
        outs = nan_outs()
        dak.dak_gemm_chain(ops(outs), tuning=dict(pdl=1, chain_rr=rr))
        st, info = dak.dak_last_error()
        assert st == 0, f"device status {st} info {info:#x}"
        for c, r in zip(outs, sep):
            assert np.array_equal(bits_of(c), r), rr
    outs = nan_outs()
    o = ops(outs)
    ws = torch.zeros(dak.dak_gemm_chain_workspace_bytes(o, N), dtype=torch.uint8, device="cuda")
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dak.dak_gemm_chain(o, workspace=ws, tuning=dict(pdl=1))
        with torch.cuda.graph(g, stream=s):
            dak.dak_gemm_chain(o, workspace=ws, tuning=dict(pdl=1))
    for c in outs:
        c.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert dak.dak_last_error()[0] == 0
    for c, r, (A, B) in zip(outs, sep, lin):
        assert np.array_equal(bits_of(c), r)
    for p in pls:
        p.free()


def test_one_row_chain(dak):
    """N = 1: the chain runs the tensor cores with B padded to 8 rows, where dak_gemm runs the
    CUDA cores. The same bits at every offload ratio, the oracle's values, and dak_gemm's to
    fp32 rounding (the same products summed in another order)."""
    mats = [synth.gemm_inputs(M, K, 1, seed=140 + i)[0] for i, (M, K) in enumerate(SHAPES)]
    Bs = [synth.normal_bf16(150 + i, 2, K).reshape(1, K) for i, (M, K) in enumerate(SHAPES)]
    base = None
    for frac in (0.0, 0.3, 1.0):
        pls = [dak.dak_place_matrix(A, int(np.ceil(frac * -(-A.shape[0] // 64)))) for A in mats]
        ops = [dict(A=p, B=to_dev(B), c_fp32=True) for p, B in zip(pls, Bs)]
        got = [bits_of(c) for c in dak.dak_gemm_chain(ops, tuning=dict(pdl=1))]
        st, info = dak.dak_last_error()
        assert st == 0, f"device status {st} info {info:#x}"
        if base is None:
            base = got
        for g, b in zip(got, base):
            assert np.array_equal(g, b), frac
        sep = _separate(dak, ops)
        for g, s, A, B in zip(got, sep, mats, Bs):
            ref = og.gemm_ref(A, B)
            assert og.rel_err(g.view(np.float32), ref) <= FP32_OUT_TOL
            assert og.rel_err(g.view(np.float32), to_np(s)) <= FP32_OUT_TOL
        for p in pls:
            p.free()


@pytest.mark.parametrize("N", [1, 4, 16, 64])
def test_dependent_chain(dak, N):
    """C1 = A1 . B, C2 = A2 . C1, C3 = A3 . C2, C4 = A4 . C3 (bf16 between the operations),
    one launch with after_prev, against the four launches one after the other."""
    import torch
    dims = [1024, 2048, 512, 1536, 768]
    mats = [synth.gemm_inputs(dims[i + 1], dims[i], N, seed=60 + i)[0] for i in range(4)]
    B0 = to_dev(synth.normal_bf16(70, 2, N * dims[0]).reshape(N, dims[0]))
    pls = [dak.dak_place_matrix(A, i + 1) for i, A in enumerate(mats)]
    Cs = [torch.empty((N, dims[i + 1]), dtype=torch.bfloat16, device="cuda") for i in range(4)]
    ops = [dict(A=pls[0], B=B0, C=Cs[0])] + [dict(A=pls[i], B=Cs[i - 1], C=Cs[i], after_prev=True)
                                           for i in range(1, 4)]
    ws = torch.zeros(dak.dak_gemm_chain_workspace_bytes(ops, N), dtype=torch.uint8, device="cuda")
    seq, seq_t = [], []
    x = B0
    for p in pls:
        x = dak.dak_gemm(p, x)
        seq.append(bits_of(x))
        seq_t.append(x)
    first = None
    for rep in range(3):  # the counters are back at zero after every launch
        for c in Cs:
            c.fill_(float("nan"))
        dak.dak_gemm_chain(ops, workspace=ws, tuning=dict(pdl=rep % 2))
        st, info = dak.dak_last_error()
        assert st == 0, f"device status {st} info {info:#x}"
        got = [bits_of(c) for c in Cs]
        first = first or got
        for c, g, f, s, st_ in zip(Cs, got, first, seq, seq_t):
            assert np.array_equal(g, f), rep
            if N > 1:
                assert np.array_equal(g, s), rep
            else:  # dak_gemm on the CUDA cores: the same products in another order
                assert og.rel_err(to_np(c), to_np(st_)) <= REL_TOL, rep
    assert int(ws[:256].view(torch.int32).abs().sum()) == 0
    ref = og.gemm_ref(mats[1], bits_of(Cs[0]))
    assert og.rel_err(to_np(Cs[1]), ref) <= REL_TOL
    for p in pls:
        p.free()


def test_8b_linears_chain_bit_identical_across_offload(dak):
    """The four 8B-shaped linears (their pieces per tile row at 16 rows: QKV 3, O 2, down 7) as
    one independent chain at x = 0, 0.1 and 0.3: bit-identical to separate launches."""
    N = 16
    lin = {k: synth.gemm_inputs(M, K, N, seed=i, tensor_index=i) for i, (k, (M, K)) in
           enumerate(synth.LINEARS_8B.items())}
    base = None
    for x in (0.0, 0.1, 0.3):
        pls = {k: dak.dak_place_matrix(A, int(np.ceil(x * A.shape[0] / 64))) for k, (A, _) in lin.items()}
        ops = [dict(A=pls[k], B=to_dev(B)) for k, (_, B) in lin.items()]
        got = [bits_of(c) for c in dak.dak_gemm_chain(ops)]
        assert dak.dak_last_error()[0] == 0
        ref = [bits_of(c) for c in _separate(dak, ops)]
        for g, r in zip(got, ref):
            assert np.array_equal(g, r)
        if base is None:
            base = got
        for g, b in zip(got, base):
            assert np.array_equal(g, b)
        for p in pls.values():
            p.free()


def test_glu_placement_in_chain(dak):
    import torch
    N = 16
    A, B = synth.gemm_inputs(1024, 512, N, seed=81)
    A2, _ = synth.gemm_inputs(256, 512, N, seed=82)
    pg = dak.dak_place_matrix_glu(A, 3)
    p2 = dak.dak_place_matrix(A2, 1)
    Bt = to_dev(B)
    act = torch.empty((N, 512), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((N, 256), dtype=torch.float32, device="cuda")
    dak.dak_gemm_chain([dict(A=pg, B=Bt, C=act), dict(A=p2, B=act, C=out, c_fp32=True, after_prev=True)])
    assert dak.dak_last_error()[0] == 0
    a_ref = dak.dak_gemm(pg, Bt)
    o_ref = dak.dak_gemm(p2, a_ref, c_fp32=True)
    assert torch.equal(act, a_ref) and torch.equal(out, o_ref)
    pg.free()
    p2.free()


def test_chain_errors(dak):
    import torch
    A, B = synth.gemm_inputs(256, 512, 16, seed=90)
    p = dak.dak_place_matrix(A, 1)
    Bt = to_dev(B)
    one = [dict(A=p, B=Bt)]
    need = dak.dak_gemm_chain_workspace_bytes(one, 16)
    assert need >= 256
    small = torch.zeros(need - 256 if need > 256 else 0, dtype=torch.uint8, device="cuda")
    if small.numel():
        with pytest.raises(dak.DakError) as e:
            dak.dak_gemm_chain(one, workspace=small)
        assert e.value.status == 1
    with pytest.raises(dak.DakError) as e:  # one CTA per tile row holds at most 128 rows
        dak.dak_gemm_chain([dict(A=p, B=torch.zeros((129, 512), dtype=torch.bfloat16, device="cuda"))])
    assert e.value.status == 7
    with pytest.raises(dak.DakError) as e:
        dak.dak_gemm_chain([dict(A=p, B=Bt)] * 9)
    assert e.value.status == 1
    assert dak.dak_last_error()[0] == 0
    p.free()
