"""Seeded random shapes, placements and launch knobs for dak_gemm and dak_attn against the
CPU oracle (combinations the structured tests do not enumerate)."""
import math

import numpy as np
import pytest

import synth
from gpu_util import FP32_OUT_TOL, REL_TOL, to_dev, to_np
from oracle import attention as oa
from oracle import gemm as og

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dak(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    import direct_host_memory_gb300 as m
    return m


def _pick(u, choices):
    return choices[min(len(choices) - 1, int(u * len(choices)))]


@pytest.mark.parametrize("case", range(24))
def test_gemm_random(dak, case):
    u = synth.uniform_f64(900, case, 8)
    M = 1 + int(u[0] * 900)
    K = 8 * (1 + int(u[1] * 400))
    N = _pick(u[2], [1, 3, 7, 8, 12, 31, 64, 100, 129, 256, 300, 513])
    T = math.ceil(M / 64)
    h = int(u[3] * (T + 1))
    tun = {}
    if u[4] < 0.3:
        tun["host_ctas"] = 1 + int(u[5] * 40)
    if u[6] < 0.3:
        tun["window"] = 1 + int(u[7] * 6)
    if u[4] > 0.7:
        tun["pdl"] = 1
    A, B = synth.gemm_inputs(M, K, N, seed=1000 + case)
    p = dak.dak_place_matrix(A, h)
    C = dak.dak_gemm(p, to_dev(B), c_fp32=True, tuning=tun or None)
    st, info = dak.dak_last_error()
    p.free()
    assert st == 0, (M, K, N, h, tun, hex(info))
    assert og.rel_err(to_np(C), og.gemm_ref(A, B)) <= FP32_OUT_TOL, (M, K, N, h, tun)


@pytest.mark.parametrize("case", range(24))
def test_gemm_random_pieces(dak, case):
    """Random shapes with an explicit piece count, few CTAs (so that a CTA takes several
    pieces, also of one tile row) and, half of the time, the gate/up interleaved placement:
    matches the oracle, and the fp32 result does not depend on the placement."""
    from oracle import decoder as od
    u = synth.uniform_f64(903, case, 8)
    glu = u[0] < 0.5
    M = 64 * (1 + int(u[1] * 14)) if glu else 1 + int(u[1] * 900)  # glu: f a multiple of 32
    K = 8 * (1 + int(u[2] * 600))
    N = _pick(u[3], [1, 2, 5, 8, 16, 40, 64, 128])
    T = math.ceil(M / 64)
    P = _pick(u[4], [2, 3, 4, 5, 7, 8])
    tun = dict(split_k=P)
    if u[5] < 0.5:
        tun["hbm_ctas"] = 1 + int(u[6] * 6)
        tun["host_ctas"] = 1 + int(u[7] * 3)
    A, B = synth.gemm_inputs(M, K, N, seed=3000 + case)
    ref = og.gemm_ref(A, B)
    if glu:
        ref = od.swiglu(ref, M // 2)
    outs = []
    for h in sorted({0, T // 3, T}):
        p = dak.dak_place_matrix_glu(A, h) if glu else dak.dak_place_matrix(A, h)
        C = dak.dak_gemm(p, to_dev(B), c_fp32=True, tuning=tun)
        st, info = dak.dak_last_error()
        p.free()
        assert st == 0, (M, K, N, h, tun, glu, hex(info))
        assert og.rel_err(to_np(C), ref) <= FP32_OUT_TOL, (M, K, N, h, tun, glu)
        outs.append(to_np(C))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0]), (M, K, N, tun, glu)


@pytest.mark.parametrize("case", range(16))
def test_attn_random(dak, case):
    import torch
    u = synth.uniform_f64(901, case, 8)
    B = 1 + int(u[0] * 12)
    Hkv = _pick(u[1], [1, 2, 4, 8])
    G = _pick(u[2], [1, 2, 4, 8, 16])
    D = _pick(u[3], [64, 128])
    L = 1 + int(u[4] * 1500)
    h_r = int(u[5] * (B + 1))
    n_split = _pick(u[6], [0, 1, 2, 3, 7])
    q, k, v = synth.attn_inputs(B, Hkv * G, Hkv, D, L, seed=2000 + case)
    lens = [1 + int(x * L) for x in synth.uniform_f64(902, case, B)] if u[7] < 0.5 else None
    p = dak.dak_place_kv(k, v, h_r)
    sl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    O = dak.dak_attn(to_dev(q), p, seq_lens=sl, tuning=dict(n_split=n_split) if n_split else None)
    st, info = dak.dak_last_error()
    p.free()
    assert st == 0, (B, Hkv, G, D, L, h_r, n_split, hex(info))
    ref = oa.decode_attention_ref(q, k, v, seq_lens=lens)
    assert og.rel_err(to_np(O), ref) <= REL_TOL, (B, Hkv, G, D, L, h_r, n_split)
