"""Single-query (decode) GQA attention over a request-partitioned KV cache -- oracle (fp64).

[DAK] section 5 "Supporting FlashAttention": the attention kernel keeps the interface of
PyTorch's scaled dot-product attention and splits the KV cache along the batch dimension,
so each request's keys and values sit wholly in host memory or wholly in GPU memory and
the result is exact attention ([DAK-explainer], section on how a matrix lives in both
HBM and host memory: the split introduces no approximation). The oracle is therefore the
plain definition of SDPA for one query token per request, with no mask:

    for request b, query head h, kv head g = floor(h / (Hq / Hkv)):
        s_j = scale * <q[b,h], k[b,g,j]>      for j < L_b
        p   = softmax(s)                      (max-subtracted, fp64)
        o[b,h] = sum_j p_j v[b,g,j]

The kv-head mapping is the grouped-query convention of SDPA's ``enable_gqa`` (query heads
h*G .. h*G+G-1 share kv head h, G = Hq/Hkv); ``scale`` defaults to 1/sqrt(D).

Parity pins (tests/test_oracle_attention.py): constant keys (o = mean of values),
constant values (o = v), L = 1 (o = v_0), a dominant key (o -> v_j), the two-key closed
form through the logistic function, per-kv-head constant values (checks the head
mapping), token-permutation invariance and seq_lens truncation.
"""
import math

import numpy as np

from .bf16 import to_f64


def decode_attention_ref(q_bits, k_bits, v_bits, seq_lens=None, scale=None) -> np.ndarray:
    """q [B][Hq][D], k/v [B][Hkv][L][D] (bf16 bits or float arrays) -> o [B][Hq][D] fp64."""
    q = to_f64(q_bits) if np.asarray(q_bits).dtype == np.uint16 else np.asarray(q_bits, np.float64)
    k = to_f64(k_bits) if np.asarray(k_bits).dtype == np.uint16 else np.asarray(k_bits, np.float64)
    v = to_f64(v_bits) if np.asarray(v_bits).dtype == np.uint16 else np.asarray(v_bits, np.float64)
    B, Hq, D = q.shape
    _, Hkv, L, _ = k.shape
    assert Hq % Hkv == 0
    G = Hq // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = np.zeros((B, Hq, D))
    for b in range(B):
        Lb = L if seq_lens is None else int(seq_lens[b])
        if Lb <= 0:
            continue
        for h in range(Hq):
            g = h // G
            s = scale * (k[b, g, :Lb] @ q[b, h])
            s = s - s.max()
            p = np.exp(s)
            p = p / p.sum()
            out[b, h] = p @ v[b, g, :Lb]
    return out


def decode_attention_one(q_bits, k_bits, v_bits, b: int, h: int, L: int = None, scale=None):
    """One output row o[b, h] (D,) from the full arrays; for sampled checks at full size."""
    q = to_f64(q_bits[b, h])
    Hq = q_bits.shape[1]
    Hkv = k_bits.shape[1]
    g = h // (Hq // Hkv)
    k = to_f64(k_bits[b, g, :L])
    v = to_f64(v_bits[b, g, :L])
    D = q.shape[0]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    s = scale * (k @ q)
    s = s - s.max()
    p = np.exp(s)
    p = p / p.sum()
    return p @ v
