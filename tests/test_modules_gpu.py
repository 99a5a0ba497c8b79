"""The drop-in modules (SplitK_GEMM for a bias-free nn.Linear, SplitK_FlashAttn for decode
attention over a placed static cache) and the cache append, through the C ABI: the same bits
as the library calls they wrap, at every offload ratio, and the oracle's values."""
import numpy as np
import pytest

import synth
from gpu_util import ATTN_FP32_TOL, FP32_OUT_TOL, REL_TOL, bits_of, to_dev, to_np
from oracle import attention as oa
from oracle import gemm as og

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dak(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    import direct_host_memory_gb300 as m
    return m


@pytest.mark.parametrize("tile_m", [64, 128])
def test_splitk_gemm_from_linear(dak, tile_m):
    import torch
    M, K = 640, 1024
    A, B = synth.gemm_inputs(M, K, 6, seed=71)
    lin = torch.nn.Linear(K, M, bias=False, device="cuda", dtype=torch.bfloat16)
    with torch.no_grad():
        lin.weight.copy_(to_dev(A))
    x = to_dev(B).view(2, 3, K)
    ref = og.gemm_ref(A, B)
    base = None
    for ratio in (0.0, 0.3, 1.0):
        mod = dak.SplitK_GEMM.from_linear(lin, offload_ratio=ratio, tile_m=tile_m, fp32_out=True)
        y = mod(x)
        assert dak.dak_last_error()[0] == 0
        assert tuple(y.shape) == (2, 3, M) and y.dtype == torch.float32
        assert og.rel_err(to_np(y.reshape(6, M)), ref) <= FP32_OUT_TOL
        direct = dak.dak_gemm(mod.placement, x.reshape(6, K), c_fp32=True)
        assert np.array_equal(bits_of(y.reshape(6, M)), bits_of(direct))
        if base is None:
            base = bits_of(y)
        assert np.array_equal(bits_of(y), base), ratio  # the split never changes a bit
        assert mod.host_bytes == mod.placement.host_bytes
    y16 = dak.SplitK_GEMM(lin.weight, offload_ratio=0.25, tile_m=tile_m)(x)
    assert y16.dtype == torch.bfloat16
    assert og.rel_err(to_np(y16.reshape(6, M)), ref) <= REL_TOL
    with pytest.raises(ValueError):
        dak.SplitK_GEMM.from_linear(torch.nn.Linear(K, M, bias=True))
    with pytest.raises(ValueError):
        dak.SplitK_GEMM(lin.weight)(torch.zeros(2, K + 8, dtype=torch.bfloat16, device="cuda"))


def test_splitk_gemm_in_a_cuda_graph(dak):
    import torch
    M, K, N = 384, 512, 16
    A, B = synth.gemm_inputs(M, K, N, seed=72)
    mod = dak.SplitK_GEMM(to_dev(A), offload_ratio=0.5)
    x = to_dev(B)
    eager = mod(x).clone()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        mod(x)
        with torch.cuda.graph(g, stream=s):
            y = mod(x)
    g.replay()
    torch.cuda.synchronize()
    assert dak.dak_last_error()[0] == 0
    assert torch.equal(y, eager)


@pytest.mark.parametrize("D", [64, 128])
def test_splitk_flash_attn(dak, D):
    import torch
    B, Hq, Hkv, L = 5, 8, 2, 300
    q, k, v = synth.attn_inputs(B, Hq, Hkv, D, L, seed=73 + D)
    ref = oa.decode_attention_ref(q, k, v)
    qd = to_dev(q)
    base = None
    for ratio in (0.0, 0.3, 1.0):
        attn = dak.SplitK_FlashAttn(to_dev(k), to_dev(v), offload_ratio=ratio, fp32_out=True)
        o = attn(qd)
        assert dak.dak_last_error()[0] == 0
        assert o.dtype == torch.float32 and tuple(o.shape) == (B, Hq, D)
        assert og.rel_err(to_np(o), ref) <= ATTN_FP32_TOL
        if base is None:
            base = bits_of(o)
        assert np.array_equal(bits_of(o), base), ratio
        o4 = attn(qd.view(B, Hq, 1, D))
        assert tuple(o4.shape) == (B, Hq, 1, D) and torch.equal(o4.view(B, Hq, D), o)
    o16 = dak.SplitK_FlashAttn(to_dev(k), to_dev(v), offload_ratio=0.5)(qd, scale=0.2)
    assert og.rel_err(to_np(o16), oa.decode_attention_ref(q, k, v, scale=0.2)) <= REL_TOL


def test_kv_append_then_attention(dak):
    """Two steps of a static cache: each request's new key and value appended at its position
    (requests split between the tiers, a request's kv heads too), then attention over positions
    0..pos; against the oracle over the cache with those rows replaced."""
    import torch
    B, Hq, Hkv, D, L = 6, 8, 2, 128, 200
    q, k, v = synth.attn_inputs(B, Hq, Hkv, D, L, seed=74)
    k = k.copy()
    v = v.copy()
    attn = dak.SplitK_FlashAttn(to_dev(k), to_dev(v), n_host_heads=5, fp32_out=True)  # request 2 split
    pos = np.array([0, 63, 64, 130, 199, 100], dtype=np.int32)
    for step in range(2):
        p = np.minimum(pos + step, L - 1).astype(np.int32)
        kn = synth.normal_bf16(75, 2 * step, B * Hkv * D).reshape(B, Hkv, D)
        vn = synth.normal_bf16(75, 2 * step + 1, B * Hkv * D).reshape(B, Hkv, D)
        pt = torch.tensor(p, dtype=torch.int32, device="cuda")
        attn.append(to_dev(kn), to_dev(vn), pt)
        for b in range(B):
            k[b, :, p[b]] = kn[b]
            v[b, :, p[b]] = vn[b]
        o = attn(to_dev(q), seq_lens=pt + 1)
        assert dak.dak_last_error()[0] == 0
        ref = oa.decode_attention_ref(q, k, v, seq_lens=p + 1)
        assert og.rel_err(to_np(o), ref) <= ATTN_FP32_TOL, step
    # a position outside the cache is skipped and reported
    bad = torch.tensor([0, 1, L, 2, 3, 4], dtype=torch.int32, device="cuda")
    attn.append(to_dev(kn), to_dev(vn), bad)
    st, info = dak.dak_last_error()
    assert st == 8  # DAK_ERR_BOUNDS
    with pytest.raises(ValueError):
        attn.append(to_dev(kn)[:, :1], to_dev(vn), pt)
