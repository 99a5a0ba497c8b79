"""SplitK_FlashAttn on the GPU against the CPU oracle, through the C ABI."""
import numpy as np
import pytest

import synth
from gpu_util import REL_TOL, bits_of, to_dev, to_np
from oracle import attention as oa
from oracle import gemm as og
from oracle import placement as opl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dak(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    import direct_host_memory_gb300 as m
    return m


def _run(dak, q, k, v, h_r, seq_lens=None, n_split=0, device_src=False, scale=0.0):
    import torch
    src_k, src_v = (to_dev(k), to_dev(v)) if device_src else (k, v)
    p = dak.dak_place_kv(src_k, src_v, h_r)
    lens = None if seq_lens is None else torch.tensor(seq_lens, dtype=torch.int32, device="cuda")
    O = dak.dak_attn(to_dev(q), p, seq_lens=lens, scale=scale, tuning=dict(n_split=n_split) if n_split else None)
    st, info = dak.dak_last_error()
    assert st == 0, f"device status {st} info {info:#x}"
    p.free()
    torch.cuda.synchronize()
    return O


@pytest.mark.parametrize("h_r", [0, 1, 2, 4])
def test_small_parity(dak, h_r):
    q, k, v = synth.attn_inputs(4, 8, 2, 128, 300, seed=1)
    ref = oa.decode_attention_ref(q, k, v)
    assert og.rel_err(to_np(_run(dak, q, k, v, h_r)), ref) <= REL_TOL


@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 129, 1000])
@pytest.mark.parametrize("n_split", [1, 2, 4, 8])
def test_context_lengths_and_splits(dak, L, n_split):
    q, k, v = synth.attn_inputs(3, 8, 2, 128, L, seed=L)
    ref = oa.decode_attention_ref(q, k, v)
    assert og.rel_err(to_np(_run(dak, q, k, v, 1, n_split=n_split)), ref) <= REL_TOL


@pytest.mark.parametrize("D,L,n_split", [(128, 4096, 16), (128, 4096, 32), (128, 1000, 64), (64, 2000, 300),
                                         (128, 700, 1024)])
def test_many_splits_one_request(dak, D, L, n_split):
    """One request: the context cut into many splits (some empty when the splits outnumber
    the 64-token chunks), merged by the combine's split groups."""
    q, k, v = synth.attn_inputs(1, 32, 8, D, L, seed=n_split)
    ref = oa.decode_attention_ref(q, k, v)
    assert og.rel_err(to_np(_run(dak, q, k, v, 0, n_split=n_split)), ref) <= REL_TOL
    assert og.rel_err(to_np(_run(dak, q, k, v, 1, n_split=n_split)), ref) <= REL_TOL


def test_workspace_alignment(dak):
    import torch
    q, k, v = synth.attn_inputs(2, 8, 2, 128, 300, seed=5)
    p = dak.dak_place_kv(k, v, 1)
    Q = to_dev(q)
    need = dak.dak_attn_workspace_bytes(2, 8, 128, 4)
    buf = torch.zeros(need + 64, dtype=torch.uint8, device="cuda")
    with pytest.raises(dak.DakError) as e:
        dak.dak_attn(Q, p, workspace=buf[4:4 + need], tuning=dict(n_split=4))
    assert e.value.status == 2  # DAK_ERR_ALIGN: the merge reads the partials as float2
    O8 = dak.dak_attn(Q, p, workspace=buf[8:8 + need], tuning=dict(n_split=4))
    O0 = dak.dak_attn(Q, p, tuning=dict(n_split=4))
    assert dak.dak_last_error()[0] == 0
    assert torch.equal(O8, O0)
    p.free()


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 4), (16, 4), (32, 4), (64, 4), (16, 1)])
def test_group_sizes(dak, hq, hkv):
    q, k, v = synth.attn_inputs(2, hq, hkv, 128, 200, seed=hq)
    ref = oa.decode_attention_ref(q, k, v)
    assert og.rel_err(to_np(_run(dak, q, k, v, 1)), ref) <= REL_TOL


def test_head_dim_64(dak):
    q, k, v = synth.attn_inputs(4, 16, 4, 64, 333, seed=4)
    ref = oa.decode_attention_ref(q, k, v)
    assert og.rel_err(to_np(_run(dak, q, k, v, 2)), ref) <= REL_TOL


def test_seq_lens(dak):
    lens = [1, 64, 100, 513, 700, 7]
    q, k, v = synth.attn_inputs(6, 8, 2, 128, 700, seed=5)
    ref = oa.decode_attention_ref(q, k, v, seq_lens=lens)
    for n_split in (1, 4):
        assert og.rel_err(to_np(_run(dak, q, k, v, 3, seq_lens=lens, n_split=n_split)), ref) <= REL_TOL


def test_explicit_scale(dak):
    q, k, v = synth.attn_inputs(2, 8, 2, 128, 90, seed=6)
    ref = oa.decode_attention_ref(q, k, v, scale=0.3)
    assert og.rel_err(to_np(_run(dak, q, k, v, 1, scale=0.3)), ref) <= REL_TOL


def test_bit_identical_across_offload_ratio(dak):
    q, k, v = synth.attn_inputs(8, 8, 2, 128, 500, seed=7)
    base = bits_of(_run(dak, q, k, v, 0, n_split=4))
    for h_r in range(1, 9):
        assert np.array_equal(bits_of(_run(dak, q, k, v, h_r, n_split=4)), base), h_r


def test_device_source_and_staged(dak):
    import torch
    q, k, v = synth.attn_inputs(4, 8, 2, 128, 256, seed=8)
    a = bits_of(_run(dak, q, k, v, 2))
    b = bits_of(_run(dak, q, k, v, 2, device_src=True))
    assert np.array_equal(a, b)
    p = dak.dak_place_kv(k, v, 2)
    qt = to_dev(q)
    direct = dak.dak_attn(qt, p)
    staging = torch.empty(p.host_bytes, dtype=torch.uint8, device="cuda")
    dak.dak_prefetch(p, staging)
    staged = dak.dak_attn_staged(qt, p, staging)
    assert dak.dak_last_error()[0] == 0
    assert torch.equal(direct, staged)
    p.free()


def test_errors(dak):
    q, k, v = synth.attn_inputs(2, 8, 2, 128, 16, seed=9)
    with pytest.raises(dak.DakError):
        dak.dak_place_kv(k, v, 3)  # more host requests than requests
    k96 = np.zeros((1, 1, 4, 96), dtype=np.uint16)
    with pytest.raises(dak.DakError):
        dak.dak_place_kv(k96, k96, 0)  # head dim 96 not supported


@pytest.mark.slow
def test_decode_gqa_full_size_sampled(dak):
    """32 requests, 32/8 heads, D 128, context 8192, 8 requests on the host (x = 0.25), in
    the bench's launch configuration; 48 sampled (request, head) rows against the oracle."""
    cfg = synth.ATTN_DECODE
    q, k, v = synth.attn_inputs(cfg["batch"], cfg["h_q"], cfg["h_kv"], cfg["head_dim"], cfg["context"], seed=0)
    h_r = opl.n_host_requests(0.25, cfg["batch"])
    O = to_np(_run(dak, q, k, v, h_r))
    u = synth.uniform_f64(2, 9, 96)
    picks = {(int(u[2 * i] * cfg["batch"]), int(u[2 * i + 1] * cfg["h_q"])) for i in range(48)}
    picks |= {(0, 0), (h_r - 1, 31), (h_r, 0), (31, 31)}
    got = np.stack([O[b, h] for b, h in sorted(picks)])
    ref = np.stack([oa.decode_attention_one(q, k, v, b, h) for b, h in sorted(picks)])
    assert og.rel_err(got, ref) <= REL_TOL


@pytest.mark.parametrize("D", [64, 128])
def test_head_granular_placement(dak, D):
    """dak_place_kv_heads: the first h (request, kv head) slabs on the host, so a request may
    have heads in both tiers. Every slab attends within its tier: the output is the same bit
    for bit for every h (device and host sources, eager and staged), matches the oracle, and
    the placement reports slabs."""
    import torch
    B, Hq, Hkv, L = 5, 8, 2, 300
    q, k, v = synth.attn_inputs(B, Hq, Hkv, D, L, seed=31 + D)
    ref = oa.decode_attention_ref(q, k, v)
    qt = to_dev(q)
    base = None
    slab = -(-L // 64) * 2 * 64 * D * 2
    for h in range(B * Hkv + 1):
        src = (to_dev(k), to_dev(v)) if h % 2 else (k, v)
        p = dak.dak_place_kv_heads(src[0], src[1], h)
        info = dak.dak_placement_info(p)
        assert (info["units"], info["host_units"], info["host_bytes"]) == (B * Hkv, h, h * slab)
        O = dak.dak_attn(qt, p, tuning=dict(n_split=2))
        assert dak.dak_last_error()[0] == 0
        if base is None:
            base = bits_of(O)
            assert og.rel_err(to_np(O), ref) <= REL_TOL
        assert np.array_equal(bits_of(O), base), h
        if h in (3, 7):
            staging = torch.empty(max(16, p.host_bytes), dtype=torch.uint8, device="cuda")
            dak.dak_prefetch(p, staging)
            staged = dak.dak_attn_staged(qt, p, staging, tuning=dict(n_split=2))
            assert dak.dak_last_error()[0] == 0
            assert np.array_equal(bits_of(staged), base), h
        p.free()
    # whole requests through either entry point: the same placement
    a = dak.dak_place_kv(k, v, 2)
    b = dak.dak_place_kv_heads(k, v, 2 * Hkv)
    assert dak.dak_placement_info(a) == dak.dak_placement_info(b)
    a.free()
    b.free()
    with pytest.raises(dak.DakError):
        dak.dak_place_kv_heads(k, v, B * Hkv + 1)
    with pytest.raises(dak.DakError):
        dak.dak_place_kv_heads(k, v, -1)
