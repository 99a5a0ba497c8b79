"""Pins for the attention oracle: closed forms of softmax attention on structured inputs."""
import math

import numpy as np
import pytest

import synth
from oracle import attention as oa
from oracle import bf16 as obf
from oracle import gemm as og

pytestmark = pytest.mark.cpu


def _bits(x):
    return obf.round_f64_to_bf16(np.asarray(x, dtype=np.float64))


def _inputs(B=2, Hq=8, Hkv=2, L=24, D=16, seed=0):
    q, k, v = synth.attn_inputs(B, Hq, Hkv, D, L, seed=seed)
    return q, k, v


def test_constant_keys_give_mean_of_values():
    q, k, v = _inputs()
    k_const = np.broadcast_to(k[:, :, :1, :], k.shape).copy()
    o = oa.decode_attention_ref(q, k_const, v)
    mean_v = obf.to_f64(v).mean(axis=2)  # [B][Hkv][D]
    G = q.shape[1] // k.shape[1]
    for h in range(q.shape[1]):
        assert np.allclose(o[:, h], mean_v[:, h // G], rtol=0, atol=1e-12)


def test_constant_values_give_that_value():
    q, k, v = _inputs()
    v_const = np.broadcast_to(v[:, :, 3:4, :], v.shape).copy()
    o = oa.decode_attention_ref(q, k, v_const)
    G = q.shape[1] // k.shape[1]
    vf = obf.to_f64(v)
    for h in range(q.shape[1]):
        assert np.allclose(o[:, h], vf[:, h // G, 3], rtol=0, atol=1e-12)


def test_single_token_returns_v0():
    q, k, v = _inputs(L=1)
    o = oa.decode_attention_ref(q, k, v)
    G = q.shape[1] // k.shape[1]
    vf = obf.to_f64(v)
    for h in range(q.shape[1]):
        assert np.array_equal(o[:, h], vf[:, h // G, 0])


def test_head_mapping_is_grouped():
    # values constant per kv head, with distinct constants: o[b,h] must equal the constant
    # of kv head h // (Hq/Hkv) (a modulo mapping would fail)
    B, Hq, Hkv, L, D = 1, 8, 4, 5, 8
    q, k, _ = _inputs(B, Hq, Hkv, L, D)
    v = np.zeros((B, Hkv, L, D))
    for g in range(Hkv):
        v[:, g] = g + 1
    o = oa.decode_attention_ref(q, k, _bits(v))
    for h in range(Hq):
        assert np.allclose(o[0, h], h // 2 + 1, rtol=0, atol=1e-12)


def test_two_keys_logistic_closed_form():
    D = 4
    q = np.zeros((1, 1, D)); q[0, 0, 0] = 2.0
    k = np.zeros((1, 1, 2, D)); k[0, 0, 0, 0] = 1.0; k[0, 0, 1, 0] = -0.5
    v = np.zeros((1, 1, 2, D)); v[0, 0, 0, :] = 3.0; v[0, 0, 1, :] = -1.0
    scale = 1.0 / math.sqrt(D)
    o = oa.decode_attention_ref(_bits(q), _bits(k), _bits(v))
    s0, s1 = scale * 2.0 * 1.0, scale * 2.0 * -0.5
    p0 = 1.0 / (1.0 + math.exp(s1 - s0))
    assert np.allclose(o[0, 0], p0 * 3.0 + (1 - p0) * -1.0, rtol=1e-14, atol=0)


def test_dominant_key_selects_its_value():
    B, Hq, Hkv, L, D = 1, 4, 1, 16, 8
    q = np.zeros((B, Hq, D)); q[:, :, 0] = 8.0
    k = np.zeros((B, Hkv, L, D)); k[0, 0, 5, 0] = 8.0
    _, _, v = _inputs(B, Hq, Hkv, L, D)
    o = oa.decode_attention_ref(_bits(q), _bits(k), v, scale=1.0)
    # p_5 = e^64 / (e^64 + 15): other weights ~ 1e-27
    assert np.allclose(o[0, :], obf.to_f64(v)[0, 0, 5], rtol=0, atol=1e-20)


def test_token_permutation_invariance():
    q, k, v = _inputs(L=20)
    perm = np.argsort(synth.uniform_f64(3, 0, 20))
    o1 = oa.decode_attention_ref(q, k, v)
    o2 = oa.decode_attention_ref(q, k[:, :, perm], v[:, :, perm])
    assert np.allclose(o1, o2, rtol=1e-13, atol=1e-13)


def test_seq_lens_truncate():
    q, k, v = _inputs(B=2, L=24)
    lens = [10, 24]
    o = oa.decode_attention_ref(q, k, v, seq_lens=lens)
    o_short = oa.decode_attention_ref(q[:1], k[:1, :, :10], v[:1, :, :10])
    assert np.array_equal(o[0], o_short[0])


def test_one_row_helper_matches_full():
    q, k, v = _inputs(B=2, Hq=8, Hkv=2, L=33, D=16)
    o = oa.decode_attention_ref(q, k, v)
    for b, h in [(0, 0), (1, 7), (1, 3)]:
        assert np.allclose(oa.decode_attention_one(q, k, v, b, h), o[b, h], rtol=1e-14, atol=0)


def test_fp32_tolerance_sees_a_dropped_or_doubled_token():
    """The fp32-output parity mode's 1e-4 bound (of max |ref|) sees one token dropped or
    counted twice at the full context of 8192, wherever it sits; the mistakes are planted in
    the oracle's input, on the CPU."""
    from gpu_util import ATTN_FP32_TOL
    L = 8192
    q, k, v = synth.attn_inputs(1, 4, 1, 128, L, seed=3)
    ref = oa.decode_attention_ref(q, k, v)
    for j in (0, 63, 64, 4095, L - 1):
        keep = np.delete(np.arange(L), j)
        dropped = oa.decode_attention_ref(q, k[:, :, keep], v[:, :, keep])
        assert og.rel_err(dropped, ref) > 2 * ATTN_FP32_TOL, j
        twice = np.concatenate([np.arange(L), [j]])
        doubled = oa.decode_attention_ref(q, k[:, :, twice], v[:, :, twice])
        assert og.rel_err(doubled, ref) > 2 * ATTN_FP32_TOL, j
