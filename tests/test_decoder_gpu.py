"""Decode step (RMSNorm, QKV, RoPE + KV append, attention, O, SwiGLU MLP) on the GPU against
the CPU oracle, through the C ABI."""
import numpy as np
import pytest

import synth
from gpu_util import REL_TOL, bits_of, to_np
from oracle import decoder as od
from oracle import gemm as og

pytestmark = pytest.mark.gpu

# hidden = H_q * D as in Llama; capacities and positions cut across 64-token chunks
SMALL64 = dict(n_layers=3, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn=512, rms_eps=1e-5,
               rope_theta=10000.0)
SMALL128 = dict(n_layers=2, hidden=512, n_heads=4, n_kv_heads=1, head_dim=128, ffn=1024, rms_eps=1e-5,
                rope_theta=500000.0)


@pytest.fixture(scope="module")
def dak(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    import direct_host_memory_gb300 as m
    return m


def _ocfg(c):
    return od.Config(c["n_layers"], c["hidden"], c["n_heads"], c["n_kv_heads"], c["head_dim"], c["ffn"],
                     c["rms_eps"], c["rope_theta"])


def _inputs(cfg, B, L, seed):
    layers = [synth.decoder_layer(cfg, l, seed) for l in range(cfg["n_layers"])]
    caches = [synth.decoder_kv(cfg, l, B, L, seed) for l in range(cfg["n_layers"])]
    return layers, caches, synth.decoder_final_norm(cfg, seed), synth.decoder_x0(cfg, B, seed)


def _host_units(cfg, B, frac):
    """Host tile rows / requests for offload fraction frac of every operation."""
    import math
    sh = synth.decoder_shapes(cfg)
    u = {k: math.ceil(frac * math.ceil(sh[k][0] / 64)) for k in ("qkv", "o", "gate_up", "down")}
    u["kv"] = math.ceil(frac * B)
    return u


def _build(dak, cfg, layers, caches, fnorm, units, glu=True, **kw):
    import torch
    placed = []
    for l, (w, kv) in enumerate(zip(layers, caches)):
        u = units[l] if isinstance(units, list) else units
        placed.append(dak.place_decoder_layer(w, kv, u, glu=glu))
    g = torch.from_numpy(fnorm.view(np.int16)).view(torch.bfloat16).cuda()
    return dak.Decoder(cfg, placed, g, **kw)


def _dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()


def _pos(p):
    import torch
    return torch.tensor(np.asarray(p, dtype=np.int32), device="cuda")


def _run(dak, dec, x0, pos, mode=0, graph=False):
    import torch
    x = _dev(x0)
    p = _pos(pos)
    out = torch.empty_like(x)
    if graph:
        dec.capture(x, p, out, mode)
        dec.replay()
    else:
        dec.step(x, p, out, mode)
    st, info = dak.dak_last_error()
    assert st == 0, f"device status {st} info {info:#x}"
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("B", [24, 100])
def test_decoder_folded_norms_wide_batch(dak, B):
    """Batches above 16 rows (the folded norm reads the residual in its store instead of
    preloading it) and up to the 128-row limit, against the oracle."""
    cfg, L = SMALL128, 96
    pos = [(11 * b + 3) % L for b in range(B)]
    layers, caches, fnorm, x0 = _inputs(cfg, B, L, seed=22)
    ref, _ = od.decode_step(_ocfg(cfg), x0, layers, caches, np.array(pos), fnorm)
    dec = _build(dak, cfg, layers, caches, fnorm, _host_units(cfg, B, 0.3))
    out = _run(dak, dec, x0, pos)
    assert og.rel_err(to_np(out), ref) <= REL_TOL
    dec.free()


@pytest.mark.parametrize("B,knobs", [(5, {"split_k": 3}), (24, {"split_k": 3}), (16, {"ctas_per_sm": 2})])
def test_decoder_folded_norms_split_tile_rows(dak, B, knobs):
    """Every projection with its tile rows cut into pieces (split_k = 3): the folded norm
    runs in the epilogue that adds the pieces, with and without the residual preload; and
    rings sized for two CTAs per SM."""
    cfg, L = SMALL128, 96
    pos = [(13 * b + 5) % L for b in range(B)]
    layers, caches, fnorm, x0 = _inputs(cfg, B, L, seed=23)
    ref, _ = od.decode_step(_ocfg(cfg), x0, layers, caches, np.array(pos), fnorm)
    tun = {k: dict(knobs) for k in ("qkv", "o", "gate_up", "down")}
    dec = _build(dak, cfg, layers, caches, fnorm, _host_units(cfg, B, 0.3), op_tuning=tun)
    out = _run(dak, dec, x0, pos)
    assert og.rel_err(to_np(out), ref) <= REL_TOL
    dec.free()


def test_decoder_large_batch_separate_norms(dak):
    """More requests than the GEMMs' folded RMSNorm takes (128): the step keeps its separate
    RMSNorm kernels, with the same results against the oracle."""
    cfg, B, L = SMALL64, 130, 80
    pos = [(7 * b) % L for b in range(B)]
    layers, caches, fnorm, x0 = _inputs(cfg, B, L, seed=21)
    ref, _ = od.decode_step(_ocfg(cfg), x0, layers, caches, np.array(pos), fnorm)
    dec = _build(dak, cfg, layers, caches, fnorm, _host_units(cfg, B, 0.3))
    combine = 1 if dak.dak_attn_default_split(dec.layers[0]["kv"]) > 1 else 0
    assert dec.launches() == 1 + cfg["n_layers"] * (8 + combine)
    out = _run(dak, dec, x0, pos)
    assert og.rel_err(to_np(out), ref) <= REL_TOL
    dec.free()


@pytest.mark.parametrize("cfg,B,L,pos", [
    (SMALL64, 5, 200, [0, 63, 64, 130, 199]),
    (SMALL128, 3, 300, [299, 0, 128]),
    (SMALL64, 1, 200, [130]),        # batch 1: the linears run on the CUDA-core GEMV path
    (SMALL128, 2, 300, [5, 299]),    # batch 2: tensor cores with B padded to 8 rows
])
@pytest.mark.parametrize("frac", [0.0, 0.3, 1.0])
def test_decoder_small_parity(dak, cfg, B, L, pos, frac):
    layers, caches, fnorm, x0 = _inputs(cfg, B, L, seed=11)
    ref, _ = od.decode_step(_ocfg(cfg), x0, layers, caches, np.array(pos), fnorm)
    dec = _build(dak, cfg, layers, caches, fnorm, _host_units(cfg, B, frac))
    out = _run(dak, dec, x0, pos)
    assert og.rel_err(to_np(out), ref) <= REL_TOL
    dec.free()


def test_decoder_bit_identical_across_placement_modes_and_launches(dak):
    """Offload ratio, prefetch baselines, CUDA graph, plain launches and the host-link handoff
    change where bytes come from and when kernels start, never the result."""
    cfg, B, L, pos = SMALL64, 5, 200, [0, 63, 64, 130, 199]
    layers, caches, fnorm, x0 = _inputs(cfg, B, L, seed=12)
    base = None
    mixed = [_host_units(cfg, B, f) for f in (0.1, 0.5, 0.9)]
    for units in (_host_units(cfg, B, 0.0), mixed, _host_units(cfg, B, 1.0)):
        for plain, handoff in ((False, True), (False, False), (True, True)):
            dec = _build(dak, cfg, layers, caches, fnorm, units, plain_launch=plain, link_handoff=handoff)
            for mode in (0, 1, 2):
                for graph in (False, True):
                    b = bits_of(_run(dak, dec, x0, pos, mode, graph))
                    if base is None:
                        base = b
                    assert np.array_equal(b, base), (units, plain, handoff, mode, graph)
            dec.free()


@pytest.mark.slow
def test_decoder_link_handoff_8b_width(dak):
    """The host-link handoff at 8B widths (QKV 6144, O 4096, gate+up 28672, down 14336 rows /
    columns; 16 requests, a third of every operation on the host): each kernel's host tiles
    start after the previous kernels' host loads are issued; the results are those of the
    step without it, bit for bit, in one step and over consecutive graph replays."""
    import torch
    cfg = dict(synth.DECODER_8B, n_layers=2)
    B, L = 16, 320
    layers = [synth.decoder_layer(cfg, l, 21) for l in range(2)]
    caches = [synth.decoder_kv(cfg, l, B, L, 21) for l in range(2)]
    fnorm, x0 = synth.decoder_final_norm(cfg, 21), synth.decoder_x0(cfg, B, 21)
    units = _host_units(cfg, B, 0.3)
    pos = [L - 1 - 7 * i for i in range(B)]
    outs = []
    for handoff in (True, False):
        dec = _build(dak, cfg, layers, caches, fnorm, units, link_handoff=handoff)
        x, p = _dev(x0), _pos(pos)
        out = torch.empty_like(x)
        dec.capture(x, p, out, 0)
        dak.dak_link_timeouts()
        for _ in range(3):
            dec.replay()
        torch.cuda.synchronize()
        assert dak.dak_last_error()[0] == 0
        assert dak.dak_link_timeouts() == 0  # every kernel found its predecessors in time
        outs.append(bits_of(out))
        dec.free()
    assert np.array_equal(outs[0], outs[1])


def test_decoder_kv_head_granular_placement(dak):
    """KV caches placed by (request, kv head) slab, with a request split between the tiers
    (its first kv head on the host, its second in HBM): three consecutive steps append each
    new key and value into the right tier and match the oracle, and equal the all-HBM
    decoder bit for bit, in every mode."""
    cfg, B, L = SMALL64, 3, 150
    layers, caches, fnorm, _ = _inputs(cfg, B, L, seed=17)
    units = dict(_host_units(cfg, B, 0.3))
    del units["kv"]
    outs = {}
    for name, kvh in (("split", 3), ("hbm", 0)):
        u = dict(units, kv_heads=kvh) if name == "split" else dict(_host_units(cfg, B, 0.0))
        ocfg = _ocfg(cfg)
        dec = _build(dak, cfg, layers, caches, fnorm, u)
        ocaches = caches
        pos = np.array([5, 70, 130])
        res = []
        for t in range(3):
            x = synth.normal_bf16(17, 600 + t, B * cfg["hidden"]).reshape(B, cfg["hidden"])
            ref, ocaches = od.decode_step(ocfg, x, layers, ocaches, pos + t, fnorm)
            out = _run(dak, dec, x, pos + t, graph=(t == 2))
            assert og.rel_err(to_np(out), ref) <= REL_TOL, (name, t)
            res.append(bits_of(out))
        outs[name] = res
        dec.free()
    for a, b in zip(outs["split"], outs["hbm"]):
        assert np.array_equal(a, b)


def test_decoder_fused_swiglu_matches_separate_kernel(dak):
    """SwiGLU in the gate/up GEMM's epilogue (interleaved placement) against the separate
    SwiGLU kernel: same expression on the same fp32 accumulators, identical outputs."""
    cfg, B, L, pos = SMALL128, 3, 300, [299, 0, 128]
    layers, caches, fnorm, x0 = _inputs(cfg, B, L, seed=16)
    outs = []
    for glu in (True, False):
        dec = _build(dak, cfg, layers, caches, fnorm, _host_units(cfg, B, 0.3), glu=glu)
        outs.append(bits_of(_run(dak, dec, x0, pos)))
        combine = 1 if dak.dak_attn_default_split(dec.layers[0]["kv"]) > 1 else 0
        # the first RMSNorm, per layer QKV, RoPE + append, attention (+ merge), O, gate+up
        # (+ SwiGLU), down; the mid-layer norms are folded into the GEMMs, the last one stays
        assert dec.launches() == 1 + cfg["n_layers"] * (6 + combine + (0 if glu else 1)) + 1
        dec.free()
    assert np.array_equal(outs[0], outs[1])


def test_decoder_consecutive_steps(dak):
    """Three steps in a row: each step's key and value stay in the cache for the next."""
    cfg, B, L = SMALL64, 4, 150
    layers, caches, fnorm, _ = _inputs(cfg, B, L, seed=13)
    dec = _build(dak, cfg, layers, caches, fnorm, _host_units(cfg, B, 0.5))
    ocfg = _ocfg(cfg)
    pos = np.array([10, 70, 0, 140])
    ocaches = caches
    for t in range(3):
        x = synth.normal_bf16(13, 500 + t, B * cfg["hidden"]).reshape(B, cfg["hidden"])
        ref, ocaches = od.decode_step(ocfg, x, layers, ocaches, pos + t, fnorm)
        out = _run(dak, dec, x, pos + t, graph=(t == 2))
        assert og.rel_err(to_np(out), ref) <= REL_TOL, t
    dec.free()


def test_decoder_many_requests(dak):
    """300 requests per step: the projections run with more than 256 hidden-state rows
    (clusters sharing each tile row) and the cache spans tiers."""
    cfg, B, L = dict(SMALL64, n_layers=2), 300, 70
    layers, caches, fnorm, x0 = _inputs(cfg, B, L, seed=17)
    pos = np.array([(37 * b) % L for b in range(B)])
    ref, _ = od.decode_step(_ocfg(cfg), x0, layers, caches, pos, fnorm)
    dec = _build(dak, cfg, layers, caches, fnorm, _host_units(cfg, B, 0.3))
    out = _run(dak, dec, x0, pos, graph=True)
    assert og.rel_err(to_np(out), ref) <= REL_TOL
    dec.free()


def test_decoder_position_out_of_range_reported(dak):
    import torch
    cfg, B, L = SMALL64, 2, 64
    layers, caches, fnorm, x0 = _inputs(cfg, B, L, seed=14)
    dec = _build(dak, cfg, layers, caches, fnorm, _host_units(cfg, B, 0.0))
    x = _dev(x0)
    out = torch.empty_like(x)
    dec.step(x, _pos([3, 64]), out)
    st, info = dak.dak_last_error()
    assert st == 8  # DAK_ERR_BOUNDS, request 1
    assert info & 0xFFFFFFFF == 1
    # the context is still usable
    dec.step(x, _pos([3, 5]), out)
    assert dak.dak_last_error()[0] == 0
    dec.free()


def test_decoder_errors(dak):
    import torch
    cfg, B, L = SMALL64, 2, 64
    layers, caches, fnorm, _ = _inputs(cfg, B, L, seed=15)
    bad = dict(cfg, hidden=cfg["hidden"] + 8)
    with pytest.raises(dak.DakError):
        _build(dak, bad, layers, caches, fnorm, _host_units(cfg, B, 0.0))
    dec = _build(dak, cfg, layers, caches, fnorm, _host_units(cfg, B, 0.0))
    x = torch.zeros((B, cfg["hidden"]), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dak.DakError):
        dec.replay()  # nothing captured
    assert dak.lib.dak_decoder_step(dec.handle, None, None, None, 0, None) == 1
    with pytest.raises(dak.DakError):
        dec.step(x, _pos([0, 0]), torch.empty_like(x), mode=3)
    dec.free()


@pytest.mark.slow
@pytest.mark.parametrize("B", [16, 1])
def test_decoder_8b_width_two_layers(dak, B):
    """Two layers at the 8B shape (hidden 4096, GQA 32/8, FFN 14336), 16 requests (or one)
    with contexts up to 4096, every operation offloaded about 30% as the planner does at
    x_global = 0.3, in the launch configuration the benchmark times. At this width the O and
    down projections split their tile rows into pieces, so the folded RMSNorms run in the
    epilogues that add the pieces (tensor cores at 16 requests, the GEMV's finisher at one)."""
    cfg = dict(synth.DECODER_8B, n_layers=2, batch=B)
    L = cfg["context"]
    pos = np.array([L - 1 - 97 * b for b in range(B)])
    layers, caches, fnorm, x0 = _inputs(cfg, B, L, seed=0)
    dec = _build(dak, cfg, layers, caches, fnorm, _host_units(cfg, B, 0.3))
    out = _run(dak, dec, x0, pos, graph=True)
    dec.free()
    ref, _ = od.decode_step(_ocfg(cfg), x0, layers, caches, pos, fnorm)
    assert og.rel_err(to_np(out), ref) <= REL_TOL
