"""Host-link handoff sequences (dak_link_begin, tuning link) through the C ABI: launches that
join a sequence start streaming their host tiles / requests only after the earlier launches
have issued all of theirs. The handoff paces loads and nothing else, so every output must
equal the launch without it bit for bit, eagerly and in a captured CUDA graph, for the
GEMM on CUDA cores (one hidden-state row), on tensor cores, with 128-row tiles, with
clusters sharing tile rows (N > 256) and for the attention."""
import numpy as np
import pytest

import synth
from gpu_util import FP32_OUT_TOL, bits_of, to_dev, to_np
from oracle import gemm as og

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dak(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    import direct_host_memory_gb300 as m
    return m


SHAPES = [(640, 1024), (1000, 520), (384, 4096), (2048, 2048)]


def _ops(dak, N, frac, tile_m=64, seed=0):
    ops = []
    for i, (M, K) in enumerate(SHAPES):
        A, B = synth.gemm_inputs(M, K, N, seed=seed + 10 * i)
        T = -(-M // tile_m)
        p = dak.dak_place_matrix(A, int(np.ceil(frac * T)), tile_m=tile_m)
        ops.append((p, to_dev(B), A, B))
    return ops


def _run(dak, ops, tuning, begin=None):
    if begin:
        dak.dak_link_begin(begin)
    return [dak.dak_gemm(p, Bd, c_fp32=True, tuning=tuning) for p, Bd, _, _ in ops]


@pytest.mark.parametrize("N,tile_m", [(1, 64), (16, 64), (128, 64), (64, 128), (300, 64)])
def test_gemm_sequence_same_bits(dak, N, tile_m):
    import torch
    dak.dak_link_timeouts()  # start from zero
    for frac in (0.0, 0.3, 1.0):
        ops = _ops(dak, N, frac, tile_m, seed=N)
        base = [bits_of(c) for c in _run(dak, ops, dict(pdl=1))]
        for slot in (1, 8):
            got = _run(dak, ops, dict(pdl=1, link=slot), begin=slot)
            assert dak.dak_last_error()[0] == 0
            for g, b in zip(got, base):
                assert np.array_equal(bits_of(g), b), (frac, slot)
        # a sequence captured in a graph and replayed: the begin call's zeroing is part of it
        outs = [torch.empty((N, p.meta["M"]), dtype=torch.float32, device="cuda") for p, _, _, _ in ops]

        def seq():
            dak.dak_link_begin(3)
            for (p, Bd, _, _), C in zip(ops, outs):
                dak.dak_gemm(p, Bd, C, c_fp32=True, tuning=dict(pdl=1, link=3))

        seq()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                seq()
        for _ in range(3):
            for C in outs:
                C.zero_()
            g.replay()
        torch.cuda.synchronize()
        assert dak.dak_last_error()[0] == 0
        for C, b, (_, _, A, B) in zip(outs, base, ops):
            assert np.array_equal(bits_of(C), b), frac
            assert og.rel_err(to_np(C), og.gemm_ref(A, B)) <= FP32_OUT_TOL
        assert dak.dak_link_timeouts() == 0  # every launch found its predecessors in time
        for p, _, _, _ in ops:
            p.free()


def test_attention_and_gemms_in_one_sequence(dak):
    """QKV-like GEMM -> attention over a cache with a third of the requests on the host ->
    O-like GEMM, all joining one sequence."""
    import torch
    B, Hq, Hkv, D, L = 12, 8, 2, 128, 700
    q, k, v = synth.attn_inputs(B, Hq, Hkv, D, L, seed=5)
    kv = dak.dak_place_kv(k, v, 4)
    Q = torch.from_numpy(q.view("int16")).view(torch.bfloat16).cuda()
    ops = _ops(dak, 16, 0.3, seed=77)
    ns = dak.dak_attn_default_split(kv)
    ws = torch.empty(max(1, dak.dak_attn_workspace_bytes(B, Hq, D, ns) // 4), dtype=torch.float32, device="cuda")

    def seq(link):
        t = dict(pdl=1, link=link)
        if link:
            dak.dak_link_begin(link)
        c0 = dak.dak_gemm(ops[0][0], ops[0][1], c_fp32=True, tuning=t)
        O = dak.dak_attn(Q, kv, workspace=ws, tuning=dict(t, n_split=ns))
        c1 = dak.dak_gemm(ops[1][0], ops[1][1], c_fp32=True, tuning=t)
        return [bits_of(c0), bits_of(O), bits_of(c1)]

    base = seq(0)
    dak.dak_link_timeouts()
    for _ in range(2):
        got = seq(2)
        assert dak.dak_last_error()[0] == 0
        for g, b in zip(got, base):
            assert np.array_equal(g, b)
    assert dak.dak_link_timeouts() == 0
    kv.free()
    for p, _, _, _ in ops:
        p.free()


def test_join_without_begin_and_tuner_ignore_link(dak):
    """Launches that join a slot nobody began still run (the count starts at zero with the
    module); the tuner drops the field from its base."""
    ops = _ops(dak, 8, 0.5, seed=9)
    base = [bits_of(c) for c in _run(dak, ops, dict(pdl=1))]
    got = [bits_of(c) for c in _run(dak, ops, dict(pdl=1, link=6))]
    assert dak.dak_last_error()[0] == 0
    for g, b in zip(got, base):
        assert np.array_equal(g, b)
    p, Bd, _, _ = ops[0]
    import torch
    C = torch.empty((8, p.meta["M"]), dtype=torch.bfloat16, device="cuda")
    r = dak.dak_tune_gemm(p, Bd, C, reps=2, base=dict(pdl=1, link=6))
    assert r["best"].get("link", 0) == 0
    for p, _, _, _ in ops:
        p.free()


def test_random_sequences(dak):
    """Random sequences of GEMM launches (N from 1 to 300, 64- and 128-row tiles, any number of
    host tile rows) and attention launches (any number of host requests), joined in one
    sequence, eager and captured: the same bits as without the handoff, and no wait gives up."""
    import torch
    rng = np.random.default_rng(2024)
    dak.dak_link_timeouts()
    for case in range(8):
        launches = []
        for j in range(int(rng.integers(3, 7))):
            if rng.random() < 0.7:
                tm = int(rng.choice([64, 128]))
                M, K = int(rng.integers(1, 1500)), int(rng.choice([64, 520, 1024, 4096]))
                N = int(rng.choice([1, 2, 16, 64, 200, 300]))
                A, B = synth.gemm_inputs(M, K, N, seed=1000 * case + j)
                T = -(-M // tm)
                p = dak.dak_place_matrix(A, int(rng.integers(0, T + 1)), tile_m=tm)
                launches.append(("gemm", p, to_dev(B)))
            else:
                Bq, Hkv, G, L = int(rng.integers(1, 20)), int(rng.choice([1, 2, 8])), int(rng.choice([1, 4])), \
                    int(rng.integers(1, 900))
                q, k, v = synth.attn_inputs(Bq, Hkv * G, Hkv, 128, L, seed=1000 * case + j)
                kv = dak.dak_place_kv(k, v, int(rng.integers(0, Bq + 1)))
                Qd = torch.from_numpy(q.view("int16")).view(torch.bfloat16).cuda()
                ns = dak.dak_attn_default_split(kv)
                ws = torch.empty(max(1, dak.dak_attn_workspace_bytes(Bq, Hkv * G, 128, ns) // 4),
                                 dtype=torch.float32, device="cuda")
                launches.append(("attn", kv, Qd, ws, ns))

        def run(link):
            outs = []
            if link:
                dak.dak_link_begin(5)
            for ln in launches:
                t = dict(pdl=1, link=link)
                if ln[0] == "gemm":
                    outs.append(dak.dak_gemm(ln[1], ln[2], c_fp32=True, tuning=t))
                else:
                    outs.append(dak.dak_attn(ln[2], ln[1], workspace=ln[3], tuning=dict(t, n_split=ln[4])))
            return outs

        base = [bits_of(o) for o in run(0)]
        for link in (5, 5):
            got = run(link)
            assert dak.dak_last_error()[0] == 0
            for g, b in zip(got, base):
                assert np.array_equal(bits_of(g), b), case
        assert dak.dak_link_timeouts() == 0, case
        for ln in launches:
            ln[1].free()
