"""Pins for the decode-step oracle: closed forms of each piece and an independent
full-sequence formulation of the whole step."""
import math

import numpy as np
import pytest
from scipy.special import expit

import synth
from oracle import bf16 as obf
from oracle import decoder as od

pytestmark = pytest.mark.cpu

TINY = dict(n_layers=2, hidden=32, n_heads=4, n_kv_heads=2, head_dim=8, ffn=48, rms_eps=1e-5,
            rope_theta=10000.0)


def _cfg(d):
    return od.Config(d["n_layers"], d["hidden"], d["n_heads"], d["n_kv_heads"], d["head_dim"],
                     d["ffn"], d["rms_eps"], d["rope_theta"])


def _bits(x):
    return obf.round_f64_to_bf16(np.asarray(x, dtype=np.float64))


def test_rmsnorm_constant_rows_and_scale():
    g = obf.to_f64(synth.normal_bf16(0, 1, 16, 1.0, 0.1))
    for c in (-3.0, 0.25, 7.0):
        out = od.rmsnorm(np.full((2, 16), c), g, 1e-5)
        assert np.allclose(out, g * c / math.sqrt(c * c + 1e-5), rtol=1e-14, atol=0)
    x = obf.to_f64(synth.normal_bf16(0, 2, 3 * 64)).reshape(3, 64)
    one = np.ones(64)
    # eps = 0: invariant to the row's scale, output rms exactly 1
    assert np.allclose(od.rmsnorm(5.5 * x, one, 0.0), od.rmsnorm(x, one, 0.0), rtol=1e-13, atol=1e-14)
    assert np.allclose(np.mean(od.rmsnorm(x, one, 0.0) ** 2, axis=-1), 1.0, rtol=1e-13)


def test_rope_is_complex_rotation():
    D, theta = 16, 500000.0
    v = obf.to_f64(synth.normal_bf16(1, 3, 5 * D)).reshape(5, D)
    pos = np.array([0, 1, 7, 4095, 123456])
    z = v[:, : D // 2] + 1j * v[:, D // 2:]
    freq = np.array([theta ** (-(2 * i) / D) for i in range(D // 2)])
    r = z * np.exp(1j * pos[:, None] * freq[None, :])
    out = od.rope(v, pos[:, None][:, 0], theta)
    assert np.allclose(out[:, : D // 2], r.real, rtol=0, atol=1e-12)
    assert np.allclose(out[:, D // 2:], r.imag, rtol=0, atol=1e-12)
    assert np.array_equal(od.rope(v[:1], np.array([0]), theta), v[:1])  # position 0: identity


def test_rope_hand_value():
    # D = 4, theta = 100: pair 1 = (element 1, element 3) turns by pos * 100^(-1/2) = 0.1 at pos 1
    out = od.rope(np.array([[0.0, 1.0, 0.0, 0.0]]), np.array([1]), 100.0)
    assert np.allclose(out, [[0.0, 0.9950041652780258, 0.0, 0.09983341664682815]], rtol=0, atol=1e-15)
    # pair 0 (elements 0 and 2) turns by 1 radian
    out = od.rope(np.array([[1.0, 0.0, 0.0, 0.0]]), np.array([1]), 100.0)
    assert np.allclose(out, [[0.5403023058681398, 0.0, 0.8414709848078965, 0.0]], rtol=0, atol=1e-15)


def test_rope_relative_position_and_norm():
    D, theta = 32, 10000.0
    q = obf.to_f64(synth.normal_bf16(2, 4, D))
    k = obf.to_f64(synth.normal_bf16(2, 5, D))
    dots = []
    for shift in (0, 5, 1000):
        rq = od.rope(q[None], np.array([17 + shift]), theta)[0]
        rk = od.rope(k[None], np.array([3 + shift]), theta)[0]
        dots.append(rq @ rk)
        assert math.isclose(np.linalg.norm(rq), np.linalg.norm(q), rel_tol=1e-13)
    assert np.allclose(dots, dots[0], rtol=1e-11)
    # and the dot product does change with the distance
    rq = od.rope(q[None], np.array([18]), theta)[0]
    rk = od.rope(k[None], np.array([3]), theta)[0]
    assert abs(rq @ rk - dots[0]) > 1e-6


def test_silu_and_swiglu():
    z = np.linspace(-30, 30, 301)
    assert np.allclose(od.silu(z), z * expit(z), rtol=1e-13, atol=1e-300)
    assert od.silu(np.array([0.0]))[0] == 0.0
    gu = np.concatenate([z[None], 2.0 * np.ones((1, 301))], axis=1)
    assert np.allclose(od.swiglu(gu, 301), 2.0 * z * expit(z), rtol=1e-13, atol=1e-300)


def _tiny_model(seed=0, cfg=TINY):
    layers = [synth.decoder_layer(cfg, l, seed) for l in range(cfg["n_layers"])]
    return layers, synth.decoder_final_norm(cfg, seed)


def test_zero_output_projections_give_identity_layer():
    cfg = _cfg(TINY)
    layers, _ = _tiny_model()
    w = dict(layers[0])
    w["o"] = np.zeros_like(w["o"])
    w["down"] = np.zeros_like(w["down"])
    B, L = 3, 10
    k, v = synth.decoder_kv(TINY, 0, B, L, seed=1)
    kc, vc = obf.to_f64(k), obf.to_f64(v)
    x = obf.to_f64(synth.decoder_x0(TINY, B, seed=1))
    pos = np.array([0, 4, 9])
    x1 = od.decode_layer(cfg, x, w, kc, vc, pos)
    assert np.array_equal(x1, x)
    # the new key was appended after rotation, the new value as is
    h = od.rmsnorm(x, w["attn_norm"], cfg.rms_eps)
    qkv = h @ obf.to_f64(w["qkv"]).T
    Hq, Hkv, D = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    for b in range(B):
        knew = qkv[b, Hq * D:(Hq + Hkv) * D].reshape(Hkv, D)
        vnew = qkv[b, (Hq + Hkv) * D:].reshape(Hkv, D)
        assert np.allclose(kc[b, :, pos[b]], od.rope(knew, np.full(Hkv, pos[b]), cfg.rope_theta), atol=1e-14)
        assert np.allclose(vc[b, :, pos[b]], vnew, atol=1e-14)


def test_zero_query_weights_attend_uniformly():
    """q = 0 -> every cached position gets the same weight, so the attention output of
    query head h is the mean of kv head h // G's values over positions 0..pos (the new value
    included). With Wo = identity and the MLP off, x' = x + that mean."""
    cfg = _cfg(TINY)
    layers, _ = _tiny_model()
    Hq, Hkv, D, d = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.hidden
    assert d == Hq * D
    w = dict(layers[1])
    qkv = w["qkv"].copy()
    qkv[: Hq * D] = 0
    w["qkv"] = qkv
    w["o"] = _bits(np.eye(d))
    w["down"] = np.zeros_like(w["down"])
    B, L = 2, 12
    k, v = synth.decoder_kv(TINY, 1, B, L, seed=2)
    kc, vc = obf.to_f64(k), obf.to_f64(v)
    v_before = vc.copy()
    x = obf.to_f64(synth.decoder_x0(TINY, B, seed=2))
    pos = np.array([11, 3])
    x1 = od.decode_layer(cfg, x, w, kc, vc, pos)
    h = od.rmsnorm(x, w["attn_norm"], cfg.rms_eps)
    vproj = (h @ obf.to_f64(w["qkv"]).T)[:, (Hq + Hkv) * D:].reshape(B, Hkv, D)
    G = Hq // Hkv
    for b in range(B):
        vals = np.concatenate([v_before[b, :, : pos[b]], vproj[b][:, None, :]], axis=1)
        mean = vals.mean(axis=1)  # [Hkv][D]
        expect = x[b] + np.concatenate([mean[hq // G] for hq in range(Hq)])
        assert np.allclose(x1[b], expect, rtol=0, atol=1e-12)


def _causal_forward(cfg, X, layers, final_norm):
    """Full-sequence forward of T tokens of one request, attention as a masked matrix."""
    T = X.shape[0]
    Hq, Hkv, D, f = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn
    G = Hq // Hkv
    pos = np.arange(T)
    mask = np.triu(np.full((T, T), -np.inf), k=1)
    x = X.copy()
    for w in layers:
        h = od.rmsnorm(x, w["attn_norm"], cfg.rms_eps)
        qkv = h @ obf.to_f64(w["qkv"]).T
        Q = od.rope(qkv[:, : Hq * D].reshape(T, Hq, D), pos[:, None], cfg.rope_theta)
        K = od.rope(qkv[:, Hq * D:(Hq + Hkv) * D].reshape(T, Hkv, D), pos[:, None], cfg.rope_theta)
        V = qkv[:, (Hq + Hkv) * D:].reshape(T, Hkv, D)
        A = np.zeros((T, Hq, D))
        for hq in range(Hq):
            S = Q[:, hq] @ K[:, hq // G].T / math.sqrt(D) + mask
            P = np.exp(S - S.max(axis=1, keepdims=True))
            P /= P.sum(axis=1, keepdims=True)
            A[:, hq] = P @ V[:, hq // G]
        x = x + A.reshape(T, Hq * D) @ obf.to_f64(w["o"]).T
        h = od.rmsnorm(x, w["mlp_norm"], cfg.rms_eps)
        gu = h @ obf.to_f64(w["gate_up"]).T
        x = x + (od.silu(gu[:, :f]) * gu[:, f:]) @ obf.to_f64(w["down"]).T
    return od.rmsnorm(x, final_norm, cfg.rms_eps)


def test_decode_steps_equal_causal_forward():
    cfg = _cfg(TINY)
    layers, fnorm = _tiny_model(seed=3)
    T = 7
    X = obf.to_f64(synth.normal_bf16(3, 5, T * cfg.hidden)).reshape(T, cfg.hidden)
    ref = _causal_forward(cfg, X, layers, fnorm)
    # caches start as garbage past the current position: the step must not read them
    caches = [tuple(obf.to_f64(a) for a in synth.decoder_kv(TINY, l, 1, T, seed=4))
              for l in range(cfg.n_layers)]
    for t in range(T):
        out, caches = od.decode_step(cfg, X[t:t + 1], layers, caches, np.array([t]), fnorm)
        assert np.allclose(out[0], ref[t], rtol=0, atol=1e-10), t


def test_batched_step_equals_per_request_steps():
    cfg = _cfg(TINY)
    layers, fnorm = _tiny_model(seed=5)
    B, L = 3, 9
    x0 = synth.decoder_x0(TINY, B, seed=5)
    caches = [synth.decoder_kv(TINY, l, B, L, seed=5) for l in range(cfg.n_layers)]
    pos = np.array([8, 0, 5])
    out, _ = od.decode_step(cfg, x0, layers, caches, pos, fnorm)
    for b in range(B):
        cb = [(k[b:b + 1], v[b:b + 1]) for k, v in caches]
        ob, _ = od.decode_step(cfg, x0[b:b + 1], layers, cb, pos[b:b + 1], fnorm)
        assert np.allclose(out[b], ob[0], rtol=0, atol=1e-12)


def test_zero_layers_is_final_norm():
    cfg = _cfg(dict(TINY, n_layers=0))
    x0 = synth.decoder_x0(TINY, 2, seed=6)
    fnorm = synth.decoder_final_norm(TINY, seed=6)
    out, _ = od.decode_step(cfg, x0, [], [], np.array([0, 0]), fnorm)
    x = obf.to_f64(x0)
    g = obf.to_f64(fnorm)
    expect = x / np.sqrt((x * x).mean(axis=1, keepdims=True) + 1e-5) * g
    assert np.allclose(out, expect, rtol=1e-14, atol=0)
