"""SplitK_FlashAttn in its fp32-output parity mode (dak_attn_f32) against the fp64 oracle,
through the C ABI: a tolerance of 1e-4 of max |ref| that a dropped or doubled token would
exceed, dominant keys placed at chunk and split boundaries (o = v_j in closed form), the
per-element error report, and the bf16 output of dak_attn from the same inputs."""
import numpy as np
import pytest

import synth
from gpu_util import ATTN_FP32_TOL, REL_TOL, bits_of, check_errors, to_dev, to_np
from oracle import attention as oa
from oracle import bf16 as obf
from oracle import placement as opl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dak(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    import direct_host_memory_gb300 as m
    return m


def _run32(dak, q, k, v, h_r, seq_lens=None, n_split=0):
    import torch
    p = dak.dak_place_kv(k, v, h_r)
    lens = None if seq_lens is None else torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    tun = dict(n_split=n_split) if n_split else None
    O32 = dak.dak_attn_f32(to_dev(q), p, seq_lens=lens, tuning=tun)
    O16 = dak.dak_attn(to_dev(q), p, seq_lens=lens, tuning=tun)
    st, info = dak.dak_last_error()
    assert st == 0, f"device status {st} info {info:#x}"
    p.free()
    torch.cuda.synchronize()
    # each output is checked against the oracle by the caller: the bf16 one at the method's
    # 2e-2, the fp32 one at 1e-4
    return to_np(O32), to_np(O16)


@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 129, 1000, 4096])
@pytest.mark.parametrize("n_split", [1, 2, 4, 8])
def test_fp32_context_lengths_and_splits(dak, L, n_split):
    q, k, v = synth.attn_inputs(3, 8, 2, 128, L, seed=100 + L)
    ref = oa.decode_attention_ref(q, k, v)
    o32, o16 = _run32(dak, q, k, v, 1, n_split=n_split)
    check_errors(o32, ref, ATTN_FP32_TOL, "fp32")
    check_errors(o16, ref, REL_TOL, "bf16")


@pytest.mark.parametrize("hq,hkv,D", [(4, 4, 128), (16, 4, 128), (64, 4, 128), (16, 1, 128), (16, 4, 64),
                                      (8, 8, 64)])
def test_fp32_groups_and_head_dims(dak, hq, hkv, D):
    q, k, v = synth.attn_inputs(3, hq, hkv, D, 700, seed=hq + D)
    ref = oa.decode_attention_ref(q, k, v)
    for n_split in (1, 4):
        o32, _ = _run32(dak, q, k, v, 1, n_split=n_split)
        check_errors(o32, ref, ATTN_FP32_TOL, "fp32")


def test_fp32_seq_lens(dak):
    lens = [1, 64, 100, 513, 700, 7, 65, 640]
    q, k, v = synth.attn_inputs(8, 8, 2, 128, 700, seed=105)
    ref = oa.decode_attention_ref(q, k, v, seq_lens=lens)
    for n_split in (1, 4, 16):
        o32, _ = _run32(dak, q, k, v, 3, seq_lens=lens, n_split=n_split)
        check_errors(o32, ref, ATTN_FP32_TOL, "fp32")


def _dominant(q, k, G, b, g, j):
    """Make token j of (request b, kv head g) dominant for every query head of the group: the
    group's queries all become u = q[b, g G] and k[b, g, j] = 8 u (exact in bf16), so its
    score is 8 |u|^2 / sqrt(D) (about 90 at D = 128, 64 at D = 64) against about N(0, 1) for
    the others."""
    u = q[b, g * G].copy()
    q[b, g * G:(g + 1) * G] = u
    k[b, g, j] = obf.round_f64_to_bf16(8.0 * obf.to_f64(u))


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("n_split", [1, 4, 16])
def test_dominant_key_at_boundaries(dak, D, n_split):
    """o = v_j when one key dominates. The dominant token sits at chunk and split boundaries:
    tokens 0, 63, 64, 127, the last token of a request (L_b - 1, with and without seq_lens)
    and both sides of every split boundary (splits of 256 tokens at 4 splits, 64 at 16); a
    token dropped at any of them would give about the mean of V instead."""
    B, Hq, Hkv, L = 8, 16, 8, 1000
    G = Hq // Hkv
    q, k, v = synth.attn_inputs(B, Hq, Hkv, D, L, seed=200 + D)
    lens = [L, L, 700, 65, L, 321, L, L]
    split_len = -(-(-(-L // n_split)) // 64) * 64  # the library's split: whole 64-token chunks
    bounds = sorted({t for s in range(1, n_split) for t in (s * split_len - 1, s * split_len) if t < L})
    spots = [0, 63, 64, 127, L - 1] + bounds
    picks = {}
    i = 0
    for b in range(B):
        for g in range(Hkv):
            if lens[b] < L:  # a shorter request: its newest token, or a token inside it
                j = lens[b] - 1 if g == 0 else (64 * g - 1) % lens[b]
            else:  # full-length requests (40 kv heads) take the spots in turn
                j = spots[i % len(spots)]
                i += 1
            picks[(b, g)] = j
            _dominant(q, k, G, b, g, j)
    assert set(spots) <= set(picks.values())
    ref = oa.decode_attention_ref(q, k, v, seq_lens=lens)
    o32, _ = _run32(dak, q, k, v, 2, seq_lens=lens, n_split=n_split)
    check_errors(o32, ref, ATTN_FP32_TOL, "fp32")
    vf = obf.to_f64(v)
    for (b, g), j in picks.items():
        for h in range(g * G, (g + 1) * G):
            assert np.max(np.abs(o32[b, h] - vf[b, g, j])) <= 1e-6 * np.max(np.abs(vf[b, g, j])), (b, g, j, h)


@pytest.mark.slow
def test_decode_gqa_full_size_fp32_sampled(dak):
    """32 requests, 32/8 heads, D 128, context 8192, 8 requests on the host (x = 0.25), in the
    bench's launch configuration, fp32 output: 48 sampled (request, head) rows at 1e-4."""
    cfg = synth.ATTN_DECODE
    q, k, v = synth.attn_inputs(cfg["batch"], cfg["h_q"], cfg["h_kv"], cfg["head_dim"], cfg["context"], seed=0)
    h_r = opl.n_host_requests(0.25, cfg["batch"])
    p = dak.dak_place_kv(k, v, h_r)
    O = to_np(dak.dak_attn_f32(to_dev(q), p))
    assert dak.dak_last_error()[0] == 0
    p.free()
    u = synth.uniform_f64(3, 9, 96)
    picks = {(int(u[2 * i] * cfg["batch"]), int(u[2 * i + 1] * cfg["h_q"])) for i in range(48)}
    picks |= {(0, 0), (h_r - 1, 31), (h_r, 0), (31, 31)}
    got = np.stack([O[b, h] for b, h in sorted(picks)])
    ref = np.stack([oa.decode_attention_one(q, k, v, b, h) for b, h in sorted(picks)])
    check_errors(got, ref, ATTN_FP32_TOL, "fp32")
