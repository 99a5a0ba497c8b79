"""The 70B-shaped decode step's operations at full size (hidden 8192, GQA 64/8, head dim 128,
FFN 28672, 16 requests, context 16384), every one about 30% offloaded as the planner does at
x_global = 0.3: each linear and the attention on sampled rows against the oracle computed
row by row, and one full decoder layer at that width against the fp64 oracle step."""
import math

import numpy as np
import pytest

import synth
from gpu_util import ATTN_FP32_TOL, FP32_OUT_TOL, REL_TOL, check_errors, to_dev, to_np
from oracle import attention as oa
from oracle import decoder as od
from oracle import gemm as og

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

CFG = dict(synth.DECODER_70B)
X = 0.3


@pytest.fixture(scope="module")
def dak(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    import direct_host_memory_gb300 as m
    return m


@pytest.mark.parametrize("name", ["qkv", "o", "gate_up", "down"])
def test_70b_linear_sampled(dak, name):
    """QKV 10240x8192, O 8192x8192, gate+up 57344x8192, down 8192x28672 (the down projection
    cuts its tile rows into pieces at 16 rows) at N = 16 and x = 0.3: 96 sampled output rows
    (all 16 columns), fp32 and bf16 outputs."""
    M, K = synth.decoder_shapes(CFG)[name]
    A = synth.decoder_tensor(CFG, 0, name)
    N = CFG["batch"]
    B = synth.normal_bf16(77, 2, N * K).reshape(N, K)
    T = -(-M // 64)
    h = math.ceil(X * T)
    p = dak.dak_place_matrix(A, h)
    Bt = to_dev(B)
    C32 = to_np(dak.dak_gemm(p, Bt, c_fp32=True))
    C16 = to_np(dak.dak_gemm(p, Bt, c_fp32=False))
    assert dak.dak_last_error()[0] == 0
    p.free()
    rows = np.unique(np.concatenate([(synth.uniform_f64(5, 9, 90) * M).astype(int),
                                     [0, 63, 64, h * 64 - 1, h * 64, M - 1]]))
    rows = rows[(rows >= 0) & (rows < M)]
    ref = og.gemm_ref(A[rows], B)
    check_errors(C32[:, rows], ref, FP32_OUT_TOL, "fp32")
    check_errors(C16[:, rows], ref, REL_TOL, "bf16")


def test_70b_attention_sampled(dak):
    """16 requests x 64/8 heads over a context of 16384, 5 requests on the host, fp32 output:
    48 sampled (request, head) rows at 1e-4, plus the bf16 output of the same launch."""
    B, Hq, Hkv, D, L = CFG["batch"], CFG["n_heads"], CFG["n_kv_heads"], CFG["head_dim"], CFG["context"]
    q, k, v = synth.attn_inputs(B, Hq, Hkv, D, L, seed=70)
    h_r = math.ceil(X * B)
    p = dak.dak_place_kv(k, v, h_r)
    O32 = to_np(dak.dak_attn_f32(to_dev(q), p))
    O16 = to_np(dak.dak_attn(to_dev(q), p))
    assert dak.dak_last_error()[0] == 0
    p.free()
    u = synth.uniform_f64(6, 9, 96)
    picks = {(int(u[2 * i] * B), int(u[2 * i + 1] * Hq)) for i in range(48)}
    picks |= {(0, 0), (h_r - 1, Hq - 1), (h_r, 0), (B - 1, Hq - 1)}
    picks = sorted(picks)
    ref = np.stack([oa.decode_attention_one(q, k, v, b, h) for b, h in picks])
    check_errors(np.stack([O32[b, h] for b, h in picks]), ref, ATTN_FP32_TOL, "fp32")
    check_errors(np.stack([O16[b, h] for b, h in picks]), ref, REL_TOL, "bf16")


def test_decoder_70b_width_one_layer(dak):
    """One decoder layer at the 70B width (hidden 8192, GQA 64/8, FFN 28672), 16 requests with
    contexts up to 16384, every operation offloaded about 30%, in the benchmark's launch
    configuration (graph, programmatic launch, folded RMSNorms), against the fp64 step."""
    import torch
    cfg = dict(CFG, n_layers=1)
    Bq, L = cfg["batch"], cfg["context"]
    pos = np.array([L - 1 - 997 * b for b in range(Bq)])
    w = synth.decoder_layer(cfg, 0, 0)
    kv = synth.decoder_kv(cfg, 0, Bq, L, 0)
    fnorm, x0 = synth.decoder_final_norm(cfg, 0), synth.decoder_x0(cfg, Bq, 0)
    sh = synth.decoder_shapes(cfg)
    units = {k_: math.ceil(X * math.ceil(sh[k_][0] / 64)) for k_ in ("qkv", "o", "gate_up", "down")}
    units["kv"] = math.ceil(X * Bq)
    layer = dak.place_decoder_layer(w, kv, units)
    dec = dak.Decoder(cfg, [layer], to_dev(fnorm))
    xin, out = to_dev(x0), torch.empty(Bq, cfg["hidden"], dtype=torch.bfloat16, device="cuda")
    posd = torch.tensor(pos, dtype=torch.int32, device="cuda")
    dec.capture(xin, posd, out)
    dec.replay()
    st, info = dak.dak_last_error()
    assert st == 0, f"device status {st} info {info:#x}"
    got = to_np(out)
    dec.free()
    ocfg = od.Config(1, cfg["hidden"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["ffn"],
                     cfg["rms_eps"], cfg["rope_theta"])
    ref, _ = od.decode_step(ocfg, x0, [w], [kv], pos, fnorm)
    check_errors(got, ref, REL_TOL, "step")
