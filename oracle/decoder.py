"""One decode step of a Llama-shaped transformer -- oracle (fp64). TEST INFRASTRUCTURE ONLY.

[DAK] section 3 and section 6.1 measure the method inside the decode step of OPT and Llama
models (time per output token), and section 5 swaps each nn.Linear for SplitK_GEMM and the
attention for SplitK_FlashAttn without touching the rest of the model. The pages do not
spell the layer out; this oracle takes the plainest reading of an 8B/70B Llama-shaped
decoder layer with RMSNorm and RoPE (pre-norm, residual stream, grouped-query attention,
SwiGLU MLP):

    h    = rmsnorm(x) * g_attn
    q,k,v = split(h . Wqkv^T)               rows of Wqkv: Hq*D query, Hkv*D key, Hkv*D value
    q, k = rope(q, pos), rope(k, pos)
    cache[b, :, pos_b] = (k[b], v[b])       append the new token, then attend over
    a    = attention(q, cache, L_b = pos_b + 1)  positions 0 .. pos_b (oracle.attention)
    x    = x + a . Wo^T
    h    = rmsnorm(x) * g_mlp
    gu   = h . Wgu^T                        rows of Wgu: f gate rows, then f up rows
    x    = x + (silu(gate) * up) . Wdown^T
    out  = rmsnorm(x_final) * g_final       (embedding and LM head are not part of the step)

rmsnorm(x) = x / sqrt(mean(x^2) + eps). RoPE pairs element i with element i + D/2 of a
head (the rotate-half convention) and turns the pair by pos * theta^(-2i/D), i < D/2.
silu(z) = z / (1 + e^-z). Everything is computed in fp64 from the bf16 weights, inputs and
cache as given; nothing is rounded in between.

Parity pins (tests/test_oracle_decoder.py): rmsnorm on constant rows and its scale
invariance; RoPE against complex multiplication by e^(i*angle), position 0, norm
preservation and the relative-position property of q.k; silu against the logistic
function; a layer whose output projections are zero is the identity; a layer with zero
query weights attends uniformly (closed form through the mean of the values, checking the
head mapping, the append and the value path); and a decode step with the cache built by
earlier decode steps equals the last position of a causal full-sequence forward written
with a masked attention matrix.
"""
import math

import numpy as np

from .attention import decode_attention_ref
from .bf16 import to_f64


def _f64(a):
    a = np.asarray(a)
    return to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


def rmsnorm(x, g, eps):
    """x [..., d] -> x / sqrt(mean(x^2) + eps) * g."""
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * _f64(g)


def rope_angles(pos, D, theta):
    """angles [..., D/2] = pos * theta^(-2i/D)."""
    i = np.arange(D // 2, dtype=np.float64)
    inv_freq = float(theta) ** (-2.0 * i / D)
    return np.asarray(pos, dtype=np.float64)[..., None] * inv_freq


def rope(v, pos, theta):
    """Rotate the pairs (i, i + D/2) of the last axis of v by the angles of position pos
    (pos broadcasts against v's leading axes)."""
    v = _f64(v)
    D = v.shape[-1]
    a = rope_angles(pos, D, theta)
    c, s = np.cos(a), np.sin(a)
    x1, x2 = v[..., : D // 2], v[..., D // 2:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(z):
    z = _f64(z)
    return z / (1.0 + np.exp(-z))


def swiglu(gu, f):
    """gu [..., 2f] (gate then up) -> silu(gate) * up [..., f]."""
    gu = _f64(gu)
    return silu(gu[..., :f]) * gu[..., f:]


class Config:
    """Shape of the decoder: n_layers, hidden d, Hq / Hkv heads of dim D, FFN width f."""

    def __init__(self, n_layers, hidden, n_heads, n_kv_heads, head_dim, ffn, rms_eps=1e-5,
                 rope_theta=500000.0):
        self.n_layers, self.hidden, self.n_heads = n_layers, hidden, n_heads
        self.n_kv_heads, self.head_dim, self.ffn = n_kv_heads, head_dim, ffn
        self.rms_eps, self.rope_theta = rms_eps, rope_theta


def decode_layer(cfg, x, w, k_cache, v_cache, positions):
    """One layer for B tokens. x [B][d] fp64; w: dict with 'qkv', 'o', 'gate_up', 'down'
    (bf16 bits [out][in]), 'attn_norm', 'mlp_norm' (bf16 bits [d]); k_cache / v_cache
    [B][Hkv][L][D] fp64, updated in place at positions. Returns the new x."""
    B = x.shape[0]
    Hq, Hkv, D, f = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.ffn
    pos = np.asarray(positions, dtype=np.int64)
    h = rmsnorm(x, w["attn_norm"], cfg.rms_eps)
    qkv = h @ _f64(w["qkv"]).T
    q = qkv[:, : Hq * D].reshape(B, Hq, D)
    k = qkv[:, Hq * D: (Hq + Hkv) * D].reshape(B, Hkv, D)
    v = qkv[:, (Hq + Hkv) * D:].reshape(B, Hkv, D)
    q = rope(q, pos[:, None], cfg.rope_theta)
    k = rope(k, pos[:, None], cfg.rope_theta)
    for b in range(B):
        k_cache[b, :, pos[b]] = k[b]
        v_cache[b, :, pos[b]] = v[b]
    a = decode_attention_ref(q, k_cache, v_cache, seq_lens=pos + 1, scale=1.0 / math.sqrt(D))
    x = x + a.reshape(B, Hq * D) @ _f64(w["o"]).T
    h = rmsnorm(x, w["mlp_norm"], cfg.rms_eps)
    x = x + swiglu(h @ _f64(w["gate_up"]).T, f) @ _f64(w["down"]).T
    return x


def decode_step(cfg, x0, layers, caches, positions, final_norm):
    """x0 [B][d] (bf16 bits or floats); layers: one weight dict per layer; caches: one
    (K, V) pair per layer, [B][Hkv][L][D] (bf16 bits or floats; copied, not modified).
    Returns (out [B][d] fp64, the updated caches as fp64)."""
    x = _f64(x0)
    new_caches = []
    for w, (kc, vc) in zip(layers, caches):
        kc, vc = _f64(kc).copy(), _f64(vc).copy()
        x = decode_layer(cfg, x, w, kc, vc, positions)
        new_caches.append((kc, vc))
    return rmsnorm(x, final_norm, cfg.rms_eps), new_caches
