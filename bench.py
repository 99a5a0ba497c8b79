"""Benchmark: one decode layer of an 8B-shaped model over a host/HBM tiered placement.

Step = the whole direct-access hot path once: the four decode linears of an 8B-shaped
layer (QKV 6144x4096, O 4096x4096, gate+up 28672x4096, down 4096x14336; bf16 weights)
at batch N through dak_gemm, and decode GQA attention (32 requests, 32/8 heads, head dim
128, context 8192, bf16 KV) through dak_attn, with a fraction x of every weight matrix's
tile rows and of the requests' KV in pinned host memory (default x = 0.25, N = 32).

Metric: effective bandwidth (bytes of weights + KV per step / step time) and decode
tokens/s, against the tier-aggregate roofline R(x) = C / max(x C / B_host, (1-x) C / B_hbm)
with B_host and B_hbm measured in the same run by read-stream kernels over each tier.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--x 0.25] [--batch 32]
  python bench.py --impl reference ...   (the CPU oracle on a bounded sample of the step)
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective GB/s & decode tok/s vs tier-aggregate roofline, per offload ratio x"
LAYERS_8B = 32


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="dak", choices=["dak", "reference"])
    ap.add_argument("--x", type=float, default=0.25)
    ap.add_argument("--batch", type=int, default=32)
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--decode", default="8b,70b",
                    help="also time full decode steps of these models (comma list of 8b, 70b; none = off): the "
                         "8B step with the launch tuner, the x_global sweep and the one-request step, the 70B step "
                         "at --decode-x and all in HBM")
    ap.add_argument("--decode-x", type=float, default=0.3, help="x_global of the decode step's HBM cap")
    ap.add_argument("--decode-steps", type=int, default=20)
    ap.add_argument("--decode-sweep", default="0.03,0.05,0.1,0.2,0.5",
                    help="further x_global values for the decode step (comma list, empty = none)")
    ap.add_argument("--no-planner-check", action="store_true",
                    help="skip the compute-bound / greedy-vs-uniform planner measurement")
    ap.add_argument("--decode-batch", type=int, default=None,
                    help="--profile decode: batch of the step (default: the model configuration's)")
    ap.add_argument("--plain-launch", action="store_true",
                    help="--profile decode: eager steps with ordinary launches (no graph, no programmatic launch)")
    ap.add_argument("--tile-m", type=int, default=64, choices=[64, 128],
                    help="--profile of one linear: tile height of its placement")
    ap.add_argument("--profile", default=None, choices=["attn", "qkv", "o", "gate_up", "down", "decode", "chain"],
                    help="place one operation of the step at --x and launch it --steps times (for ncu); chain: the "
                         "four 8B linears as one grouped dak_gemm_chain launch")
    return ap.parse_args()


# ------------------------------------------------------------------------------ workload

def workload_bytes(batch):
    import synth
    w = sum(M * K * 2 for M, K in synth.LINEARS_8B.values())
    c = synth.ATTN_DECODE
    kv = 2 * c["batch"] * c["h_kv"] * c["context"] * c["head_dim"] * 2
    return w, kv


def gen_inputs(batch, seed=0):
    import synth
    lin = {}
    for i, (name, (M, K)) in enumerate(synth.LINEARS_8B.items()):
        lin[name] = synth.gemm_inputs(M, K, batch, seed=seed, tensor_index=i)
    c = synth.ATTN_DECODE
    attn = synth.attn_inputs(c["batch"], c["h_q"], c["h_kv"], c["head_dim"], c["context"], seed=seed,
                             tensor_index=len(lin))
    return lin, attn


class Step:
    """The placed workload at one offload ratio plus device buffers for one step."""

    def __init__(self, dak, lin, attn, x, dev):
        import torch
        self.dak = dak
        self.x = x
        self.pl, self.B, self.C = {}, {}, {}
        q, k, v = attn
        # the step's inputs (every B, then Q) and outputs (every C, then O) are views of one
        # device buffer each, so that the end-to-end step moves them in one copy each way
        n_in = sum(B.size for _, B in lin.values()) + q.size
        n_out = sum(B.shape[0] * A.shape[0] for A, B in lin.values()) + q.size
        self.inbuf = torch.empty(n_in, dtype=torch.bfloat16, device=dev)
        self.outbuf = torch.empty(n_out, dtype=torch.bfloat16, device=dev)
        oi = oo = 0
        for name, (A, B) in lin.items():
            M = A.shape[0]
            self.pl[name] = dak.dak_place_matrix(A, dak.host_tiles_for_ratio(x, M))
            self.B[name] = self.inbuf[oi:oi + B.size].view(B.shape)
            self.B[name].copy_(torch.from_numpy(B.view("int16")).view(torch.bfloat16))
            self.C[name] = self.outbuf[oo:oo + B.shape[0] * M].view(B.shape[0], M)
            oi += B.size
            oo += B.shape[0] * M
        self.kv = dak.dak_place_kv(k, v, dak.host_requests_for_ratio(x, k.shape[0]))
        self.Q = self.inbuf[oi:].view(q.shape)
        self.Q.copy_(torch.from_numpy(q.view("int16")).view(torch.bfloat16))
        self.O = self.outbuf[oo:].view(q.shape)
        self.n_split = dak.dak_attn_default_split(self.kv)
        ws = dak.dak_attn_workspace_bytes(q.shape[0], q.shape[1], q.shape[2], self.n_split)
        self.ws = torch.empty(max(1, ws // 4), dtype=torch.float32, device=dev)
        # programmatic launch: no op of the step writes the weights or KV cache another op streams;
        # the direct-access launches join host-link handoff sequence 1 (begun here, on the
        # stream every run() uses; eager launches keep the count in step from run to run)
        self.tun = dict(n_split=self.n_split, pdl=1, link=1)
        self.gtun = dict(pdl=1, link=1)
        self.stun = dict(n_split=self.n_split, pdl=1)  # the prefetch baselines' staged launches
        self.sgtun = dict(pdl=1)
        dak.dak_link_begin(1)
        self.host_bytes = sum(p.host_bytes for p in self.pl.values()) + self.kv.host_bytes
        self.total_bytes = sum(p.host_bytes + p.hbm_bytes for p in self.pl.values()) + \
            self.kv.host_bytes + self.kv.hbm_bytes
        self.launches = len(self.pl) + (2 if self.n_split > 1 else 1)

    def run(self, ev=None):
        d = self.dak
        for name, p in self.pl.items():
            d.dak_gemm(p, self.B[name], self.C[name], tuning=self.gtun)
        if ev is not None:
            ev[0].record()
        d.dak_attn(self.Q, self.kv, O=self.O, workspace=self.ws, tuning=self.tun)
        if ev is not None:
            ev[1].record()

    # prefetch baseline: copy every host-resident part into HBM staging, then the all-HBM kernels
    def alloc_staging(self, dev):
        import torch
        self.stage = {n: torch.empty(max(16, p.host_bytes), dtype=torch.uint8, device=dev) for n, p in self.pl.items()}
        self.stage_kv = torch.empty(max(16, self.kv.host_bytes), dtype=torch.uint8, device=dev)

    def run_prefetch_serial(self):
        d = self.dak
        for name, p in self.pl.items():
            d.dak_prefetch(p, self.stage[name])
        d.dak_prefetch(self.kv, self.stage_kv)
        for name, p in self.pl.items():
            d.dak_gemm_staged(p, self.stage[name], self.B[name], self.C[name], tuning=self.sgtun)
        d.dak_attn_staged(self.Q, self.kv, self.stage_kv, O=self.O, workspace=self.ws, tuning=self.stun)

    def run_prefetch_overlap(self, copy_stream, events):
        """FlexGen-style: copies of the host parts run on a side stream in op order and each
        op waits only for its own copy (best case: staging for every op)."""
        import torch
        d = self.dak
        cur = torch.cuda.current_stream()
        copy_stream.wait_stream(cur)
        names = list(self.pl)
        with torch.cuda.stream(copy_stream):
            for i, name in enumerate(names):
                d.dak_prefetch(self.pl[name], self.stage[name], stream=copy_stream)
                events[i].record(copy_stream)
            d.dak_prefetch(self.kv, self.stage_kv, stream=copy_stream)
            events[len(names)].record(copy_stream)
        for i, name in enumerate(names):
            cur.wait_event(events[i])
            d.dak_gemm_staged(self.pl[name], self.stage[name], self.B[name], self.C[name], tuning=self.sgtun)
        cur.wait_event(events[len(names)])
        d.dak_attn_staged(self.Q, self.kv, self.stage_kv, O=self.O, workspace=self.ws, tuning=self.stun)

    def free(self):
        for p in self.pl.values():
            p.free()
        self.kv.free()


# ------------------------------------------------------------------------------ decode step

def decode_ops(cfg, peak_flops):
    """The planner's view of one decode step, one entry per operation type (every layer is
    alike, so each type gets one ratio for all layers): the four weight products and the
    attention over the KV cache, with their bytes and compute time over all layers at
    peak_flops, and their placement unit (a 64-row tile row, or one (request, kv head) slab
    of the KV cache: dak_place_kv_heads)."""
    import synth
    sh = synth.decoder_shapes(cfg)
    nl, B, L, D = cfg["n_layers"], cfg["batch"], cfg["context"], cfg["head_dim"]
    kv_req = 2 * cfg["n_kv_heads"] * L * D * 2
    ops, meta = [], []
    for k in ("qkv", "o", "gate_up", "down"):
        M, K = sh[k]
        ops.append((nl * M * K * 2, nl * 2.0 * M * K * B / peak_flops, 64 * K * 2))
        meta.append((k, -(-M // 64)))
    ops.append((nl * B * kv_req, nl * 4.0 * B * cfg["n_heads"] * L * D / peak_flops, kv_req // cfg["n_kv_heads"]))
    meta.append(("kv_heads", B * cfg["n_kv_heads"]))
    return ops, meta


def decode_plan(dak, cfg, b_host, b_hbm, x_global, peak_flops):
    """Host units per operation type (tile rows or KV slabs, the same in every layer) for an
    HBM cap of (1 - x_global) of all bytes, from the library's whole-unit planner
    (dak_plan_units: the greedy ratios floored to whole units and topped up where the model
    time grows least). x_global = 0: no offload."""
    ops, meta = decode_ops(cfg, peak_flops)
    nl = cfg["n_layers"]
    if x_global <= 0:
        return [{k: 0 for k, _ in meta} for _ in range(nl)], sum(o[0] for o in ops) / b_hbm
    total = sum(o[0] for o in ops)
    # one unit of an operation type = that unit in every layer
    units, tmodel = dak.dak_plan_units([(C, tc, tile * nl) for C, tc, tile in ops], b_host, b_hbm,
                                       x_global * total)
    return [{k: int(u) for (k, _), u in zip(meta, units)} for _ in range(nl)], tmodel


def build_decoder(dak, cfg, units, seed=0, plain_launch=False):
    """Random-init bf16 weights and KV cache drawn on the GPU, placed layer by layer."""
    import synth
    layers = []
    for l in range(cfg["n_layers"]):
        w = {k: synth.decoder_tensor_dev(cfg, l, k, seed) for k in synth.decoder_shapes(cfg)}
        kv = synth.decoder_kv_dev(cfg, l, cfg["batch"], cfg["context"], seed)
        layers.append(dak.place_decoder_layer(w, kv, units[l]))
        del w, kv
    fn = synth.dev_normal_bf16(seed, 999, cfg["hidden"], 1.0, synth.NORM_STD)
    return dak.Decoder(cfg, layers, fn, plain_launch=plain_launch)


def tune_decoder_ops(dak, cfg, dec, dev):
    """dak_tune_gemm / dak_tune_attn on layer 0 of a placed decoder (same shapes and
    placement in every layer); returns the per-operation results and the tuning table."""
    import torch
    import synth
    B = cfg["batch"]
    L0 = dec.layers[0]
    sh = synth.decoder_shapes(cfg)
    res, table = {}, {}
    for k in ("qkv", "o", "gate_up", "down"):
        M, K = sh[k]
        Bt = torch.randn(B, K, device=dev).to(torch.bfloat16)
        Ct = torch.empty(B, M, device=dev, dtype=torch.float32)
        r = dak.dak_tune_gemm(L0[k], Bt, Ct, c_fp32=True, reps=5, base=dict(pdl=1))
        res[k] = r
        table[k] = {f: v for f, v in r["best"].items() if f != "pdl"}
    Q = torch.randn(B, cfg["n_heads"], cfg["head_dim"], device=dev).to(torch.bfloat16)
    O = torch.empty_like(Q)
    r = dak.dak_tune_attn(Q, L0["kv"], O, reps=5, base=dict(pdl=1))
    res["attn"] = r
    table["attn"] = {f: v for f, v in r["best"].items() if f != "pdl"}
    return res, table


def run_decode(dak, args, b_host, b_hbm, dev, sync_all, local, model="8b", full=True):
    """Full decode step: planner-chosen per-op ratios at x_global, one CUDA graph per mode.
    full: also the launch tuner, the x_global sweep and the one-request step."""
    import torch
    import synth
    cfg = dict(synth.DECODER_8B if model == "8b" else synth.DECODER_70B)
    pk, _ = peaks()
    peak_flops = pk.get("bf16_tflops_sustained", 1700.0) * 1e12
    B, d, L = cfg["batch"], cfg["hidden"], cfg["context"]
    x_in = torch.from_numpy(synth.decoder_x0(cfg, B).view("int16")).view(torch.bfloat16).to(dev)
    pos = torch.full((B,), L - 1, dtype=torch.int32, device=dev)  # context L: L - 1 cached + the new token
    out = torch.empty_like(x_in)
    res = {"workload": f"{cfg['n_layers']}-layer {model.upper()}-shaped decode step (hidden {d}, GQA "
                       f"{cfg['n_heads']}/{cfg['n_kv_heads']}, head dim {cfg['head_dim']}, FFN {cfg['ffn']}, "
                       f"RMSNorm, RoPE, SwiGLU), random-init bf16, batch {B}, context {L}",
           "batch": B, "context": L, "x_global_target": args.decode_x}
    for xg, key in ((args.decode_x, None), (0.0, "hbm_only")):
        t0 = time.time()
        units, tmodel = decode_plan(dak, cfg, b_host, b_hbm, xg, peak_flops)
        dec = build_decoder(dak, cfg, units)
        build_s = time.time() - t0
        C = sum(L_[k].host_bytes + L_[k].hbm_bytes for L_ in dec.layers for k in dak.DECODER_OPS)
        H = dec.host_bytes()
        dec.capture(x_in, pos, out, dak.MODE_DIRECT)
        for _ in range(3):
            dec.replay()
        torch.cuda.synchronize()
        st0 = dak.dak_last_error()[0]
        dak.dak_link_timeouts()  # count the handoff waits of the timed steps only
        sampler = ClockSampler(local)
        sampler.start()
        time.sleep(0.2)
        tw0 = time.time()
        t = time_steps(dec.replay, args.decode_steps, 2, sync_all)
        tw1 = time.time()
        time.sleep(0.2)
        sampler.stop()
        roof = tier_roofline(C, H / C, b_host, b_hbm)
        timeouts = dak.dak_link_timeouts()
        rec = {"x_effective": H / C, "bytes_per_step": C, "host_bytes_per_step": H, "ms_per_step": t * 1e3,
               "tok_s": B / t, "eff_gbps": C / t / 1e9, "roofline_gbps": roof / 1e9, "frac": (C / t) / roof,
               "planner_model_ms": tmodel * 1e3, "host_units_per_layer": units[0] if units else {},
               "build_s": build_s,
               "launches_per_step": dec.launches(), "clocks": sampler.summary(tw0, tw1),
               "link_timeouts": timeouts}
        if xg > 0 and full:
            # launch tuner per operation type on layer 0's placements, then the step with its choices
            tuned, table = tune_decoder_ops(dak, cfg, dec, dev)
            rec["tuner"] = tuned
            dec_t = dak.Decoder(cfg, dec.layers, dec.final_norm, op_tuning=table)
            dec_t.capture(x_in, pos, out, dak.MODE_DIRECT)
            tt = time_steps(dec_t.replay, args.decode_steps, 2, sync_all)
            rec["tuned_tok_s"] = B / tt
            rec["tuned_frac"] = (C / tt) / roof
            dec_t.free(placements=False)
        if xg > 0:
            # ablation: the same step without the host-link handoff between its kernels
            dec_n = dak.Decoder(cfg, dec.layers, dec.final_norm, link_handoff=False)
            dec_n.capture(x_in, pos, out, dak.MODE_DIRECT)
            tn = time_steps(dec_n.replay, max(5, args.decode_steps // 2), 2, sync_all)
            rec["no_link_handoff_tok_s"] = B / tn
            dec_n.free(placements=False)
            for mode, name in ((dak.MODE_PREFETCH_SERIAL, "prefetch_serial"), (dak.MODE_PREFETCH_OVERLAP,
                                                                                 "prefetch_overlap")):
                dec.capture(x_in, pos, out, mode)
                tp = time_steps(dec.replay, max(5, args.decode_steps // 2), 2, sync_all)
                rec[name + "_tok_s"] = B / tp
            rec["vs_prefetch_best"] = rec["tok_s"] / max(rec["prefetch_serial_tok_s"], rec["prefetch_overlap_tok_s"])
            # end to end: the step's hidden states and positions copied in from pinned host
            # memory and its output copied back, every step
            dec.capture(x_in, pos, out, dak.MODE_DIRECT)
            hx, hp = x_in.cpu().pin_memory(), pos.cpu().pin_memory()
            ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()

            def e2e():
                x_in.copy_(hx, non_blocking=True)
                pos.copy_(hp, non_blocking=True)
                dec.replay()
                ho.copy_(out, non_blocking=True)

            te = time_steps(e2e, max(5, args.decode_steps // 2), 2, sync_all)
            rec["e2e"] = {"tok_s": B / te, "eff_gbps": C / te / 1e9, "h2d_bytes_per_step": hx.numel() * 2 + B * 4,
                          "d2h_bytes_per_step": ho.numel() * 2}
        rec["status"] = [st0, dak.dak_last_error()[0]]
        dec.free()
        del dec
        torch.cuda.empty_cache()
        if key:
            res[key] = rec
        else:
            res.update(rec)
    # per-x sweep of the step with both prefetch baselines (planner ratios at each x_global)
    sweep = []
    for xs in [float(v) for v in args.decode_sweep.split(",") if v.strip() and full]:
        units, tmodel = decode_plan(dak, cfg, b_host, b_hbm, xs, peak_flops)
        dec = build_decoder(dak, cfg, units)
        C = sum(L_[k].host_bytes + L_[k].hbm_bytes for L_ in dec.layers for k in dak.DECODER_OPS)
        H = dec.host_bytes()
        roof = tier_roofline(C, H / C, b_host, b_hbm)
        rec = {"x_global": xs, "x_effective": H / C}
        for mode, name in ((dak.MODE_DIRECT, "dak"), (dak.MODE_PREFETCH_SERIAL, "prefetch_serial"),
                           (dak.MODE_PREFETCH_OVERLAP, "prefetch_overlap")):
            dec.capture(x_in, pos, out, mode)
            t = time_steps(dec.replay, max(4, args.decode_steps // 4), 2, sync_all)
            rec[name + "_tok_s"] = B / t
            if mode == dak.MODE_DIRECT:
                rec["frac"] = (C / t) / roof
                rec["eff_gbps"] = C / t / 1e9
        rec["vs_prefetch_best"] = rec["dak_tok_s"] / max(rec["prefetch_serial_tok_s"], rec["prefetch_overlap_tok_s"])
        rec["planner_model_ms"] = tmodel * 1e3
        rec["status"] = dak.dak_last_error()[0]
        sweep.append(rec)
        dec.free()
        del dec
        torch.cuda.empty_cache()
    if full:
        res["per_x"] = sweep
    if full and not args.no_sweep:
        res["batch1"] = run_decode_batch1(dak, args, cfg, b_host, b_hbm, dev, sync_all, peak_flops)
    return res


def run_decode_batch1(dak, args, cfg, b_host, b_hbm, dev, sync_all, peak_flops):
    """The same decode step at batch 1 (every linear a GEMV on CUDA cores), all in HBM and at
    the target x_global, against both prefetch baselines."""
    import torch
    import synth
    cfg = dict(cfg, batch=1)
    L = cfg["context"]
    x_in = torch.from_numpy(synth.decoder_x0(cfg, 1).view("int16")).view(torch.bfloat16).to(dev)
    pos = torch.full((1,), L - 1, dtype=torch.int32, device=dev)
    out = torch.empty_like(x_in)
    recs = []
    for xg in (0.0, args.decode_x):
        units, tmodel = decode_plan(dak, cfg, b_host, b_hbm, xg, peak_flops)
        dec = build_decoder(dak, cfg, units)
        C = sum(L_[k].host_bytes + L_[k].hbm_bytes for L_ in dec.layers for k in dak.DECODER_OPS)
        H = dec.host_bytes()
        roof = tier_roofline(C, H / C, b_host, b_hbm)
        rec = {"x_global": xg, "x_effective": H / C, "bytes_per_step": C}
        modes = [(dak.MODE_DIRECT, "dak")]
        if xg > 0:
            modes += [(dak.MODE_PREFETCH_SERIAL, "prefetch_serial"), (dak.MODE_PREFETCH_OVERLAP, "prefetch_overlap")]
        for mode, name in modes:
            dec.capture(x_in, pos, out, mode)
            t = time_steps(dec.replay, max(4, args.decode_steps // 2), 2, sync_all)
            rec[name + "_tok_s"] = 1 / t
            if mode == dak.MODE_DIRECT:
                rec["ms_per_step"] = t * 1e3
                rec["frac"] = (C / t) / roof
                rec["eff_gbps"] = C / t / 1e9
        if xg > 0:
            rec["vs_prefetch_best"] = rec["dak_tok_s"] / max(rec["prefetch_serial_tok_s"],
                                                             rec["prefetch_overlap_tok_s"])
        rec["planner_model_ms"] = tmodel * 1e3
        rec["status"] = dak.dak_last_error()[0]
        recs.append(rec)
        dec.free()
        del dec
        torch.cuda.empty_cache()
    return recs


# ------------------------------------------------------------------------------ planner check

PLANNER_N = 256  # batch at which the 8B-shaped linears become tensor-bound


def _time_fn(fn, reps=20, warmup=3):
    return time_steps(fn, reps, warmup)


def run_planner_check(dak, lin, attn, b_host, b_hbm, dev, x_global=0.1):
    """The planner outside the all-memory-bound regime ([DAK] section 4.2, Fig. 6 and 11):
    (1) t(x) of the 8B gate+up linear at N = 256 against the model max(T_c, (1-x)C/B_hbm,
    xC/B_host) with T_c its measured all-HBM time, in 128-row tiles (and 64-row ones); (2)
    one step of the four linears at N = 256 (each in the tile height that runs it faster all
    in HBM) plus the 32-request attention, placed by the greedy planner and uniformly at the
    same x_global, both timed. Launches run back to back with programmatic launch in one
    host-link handoff sequence."""
    import math
    import numpy as np
    import torch
    import synth
    N = PLANNER_N
    res = {"batch": N, "x_global": x_global}
    Bs, Cs = {}, {}
    for i, (name, (A, _)) in enumerate(lin.items()):
        K = A.shape[1]
        Bs[name] = torch.from_numpy(synth.normal_bf16(0 + i, 2, N * K).view("int16")).view(torch.bfloat16) \
            .to(dev).view(N, K)
        Cs[name] = torch.empty((N, A.shape[0]), dtype=torch.bfloat16, device=dev)
    # back-to-back launches with programmatic launch, joined in one host-link handoff sequence
    gt = dict(pdl=1, link=5)
    dak.dak_link_begin(5)

    # (1) flat segment of a tensor-bound operation, in 128-row tiles (M = 128 MMAs, the
    # placement for tensor-bound N) and, for comparison, in 64-row tiles
    A = lin["gate_up"][0]
    M, K = A.shape
    C = M * K * 2

    def curve_of(tile_m):
        curve, t0 = [], None
        for x in (0.0, 0.02, 0.04, 0.06, 0.08, 0.12, 0.2):
            p = dak.dak_place_matrix(A, dak.host_tiles_for_ratio(x, M, tile_m), tile_m=tile_m)
            t = _time_fn(lambda: dak.dak_gemm(p, Bs["gate_up"], Cs["gate_up"], tuning=gt))
            xe = p.host_bytes / C
            if t0 is None:
                t0 = t
            model = max(t0, (1 - xe) * C / b_hbm, xe * C / b_host)
            curve.append({"x": xe, "us": t * 1e6, "model_us": 1e6 * model, "vs_model": t / model})
            p.free()
        return curve, t0

    curve, t0 = curve_of(128)
    res["gate_up_tile_m"] = 128
    res["gate_up_curve"] = curve
    res["gate_up_t_comp_us"] = t0 * 1e6
    res["gate_up_memory_us"] = C / b_hbm * 1e6
    res["gate_up_flat_until_x"] = t0 * b_host / C
    curve64, t064 = curve_of(64)
    res["gate_up_curve_tile64"] = curve64
    res["gate_up_t_comp_us_tile64"] = t064 * 1e6

    # (2) greedy vs uniform on a mixed step
    q, k, v = attn
    Q = torch.from_numpy(q.view("int16")).view(torch.bfloat16).to(dev)
    O = torch.empty_like(Q)
    kv_req = 2 * k.shape[1] * k.shape[2] * k.shape[3] * 2
    names = list(lin) + ["attn"]
    # T_c per operation: the measured all-HBM time where it is clearly above the memory time
    # (tensor-bound), else the FLOP count at the sustained tensor rate
    pk, _ = peaks()
    P = pk.get("bf16_tflops_sustained", 1700.0) * 1e12
    ops, units = [], []
    pl0 = {}
    tile_ms = {}
    for name in names:
        if name == "attn":
            pl0[name] = dak.dak_place_kv(k, v, 0)
            nb = k.shape[0] * kv_req
            ws = torch.empty(max(1, dak.dak_attn_workspace_bytes(q.shape[0], q.shape[1], q.shape[2],
                                                               dak.dak_attn_default_split(pl0[name])) // 4),
                             dtype=torch.float32, device=dev)
            t = _time_fn(lambda: dak.dak_attn(Q, pl0["attn"], O=O, workspace=ws, tuning=dict(pdl=1, link=5)))
            flops = 4.0 * q.shape[0] * q.shape[1] * k.shape[2] * k.shape[3]
            ops.append((nb, t if t > 1.15 * nb / b_hbm else flops / P, kv_req))
            units.append(k.shape[0])
        else:
            # each linear in the tile height that runs it faster all in HBM (128-row tiles
            # when it is tensor-bound with many tiles, else 64)
            A = lin[name][0]
            best = None
            for tm in (64, 128):
                pt = dak.dak_place_matrix(A, 0, tile_m=tm)
                t = _time_fn(lambda: dak.dak_gemm(pt, Bs[name], Cs[name], tuning=gt))
                if best is None or t < best[1]:
                    if best is not None:
                        best[2].free()
                    best = (tm, t, pt)
                else:
                    pt.free()
            tm, t, pl0[name] = best
            tile_ms[name] = tm
            nb = A.shape[0] * A.shape[1] * 2
            flops = 2.0 * A.shape[0] * A.shape[1] * N
            ops.append((nb, t if t > 1.15 * nb / b_hbm else flops / P, tm * A.shape[1] * 2))
            units.append(-(-A.shape[0] // tm))
        res.setdefault("t_comp_us", {})[name] = ops[-1][1] * 1e6
    for p in pl0.values():
        p.free()
    total = sum(o[0] for o in ops)
    budget = x_global * total
    r_greedy, t_greedy_model = dak.dak_plan_ratios(ops, b_host, b_hbm, budget, 0)
    plans = {"greedy": [min(u, math.ceil(r * u - 1e-9)) for r, u in zip(r_greedy, units)],
             "uniform": [min(u, math.ceil(x_global * u - 1e-9)) for u in units]}

    def model(counts):
        t = 0.0
        for (c, tc, _), h, u in zip(ops, counts, units):
            b = c * h / u
            t += max(tc, (c - b) / b_hbm, b / b_host)
        return t

    for pname, counts in plans.items():
        pl = {}
        for name, h in zip(names, counts):
            pl[name] = dak.dak_place_kv(k, v, h) if name == "attn" else \
                dak.dak_place_matrix(lin[name][0], h, tile_m=tile_ms[name])

        def step():
            for name in lin:
                dak.dak_gemm(pl[name], Bs[name], Cs[name], tuning=gt)
            dak.dak_attn(Q, pl["attn"], O=O, workspace=ws, tuning=dict(pdl=1, link=5))

        t = _time_fn(step, 10, 2)
        host = sum(pl[n].host_bytes for n in names)
        res[pname] = {"host_units": dict(zip(names, counts)), "x_effective": host / total, "ms": t * 1e3,
                      "model_ms": model(counts) * 1e3}
        for p in pl.values():
            p.free()
    res["greedy_vs_uniform"] = res["uniform"]["ms"] / res["greedy"]["ms"]
    res["tile_m"] = tile_ms
    res["status"] = dak.dak_last_error()[0]
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------------------ large N

def run_large_n(dak, lin, b_host, b_hbm, dev, x=0.25, tile_m=128):
    """dak_gemm beyond one CTA's 256 hidden-state rows: the 8B gate+up linear at x in tiles
    of tile_m rows, N in {256, 512, 1024, 2048}, both ways: shared tiles (the default: a
    cluster of ceil(N/256) CTAs, at most 4, rank 0 forwarding every A chunk through
    distributed shared memory, host bytes read once per launch of up to 1024 rows) and
    column blocks of 256 rows (host bytes read once per block, as [DAK] Table 1 counts traffic
    without multicast), against both traffic models. t_comp_us: the same launch all in HBM;
    frac_single_read: the single-read host-link bound over the shared-tile time. Launches run
    back to back with programmatic launch in one host-link handoff sequence."""
    import torch
    import synth
    A = lin["gate_up"][0]
    M, K = A.shape
    p = dak.dak_place_matrix(A, dak.host_tiles_for_ratio(x, M, tile_m), tile_m=tile_m)
    p0 = dak.dak_place_matrix(A, 0, tile_m=tile_m)
    rows = []
    for N in (256, 512, 1024, 2048):
        B = torch.from_numpy(synth.normal_bf16(7, 2, N * K).view("int16")).view(torch.bfloat16).to(dev).view(N, K)
        C = torch.empty((N, M), dtype=torch.bfloat16, device=dev)
        blocks = -(-N // 256)
        launches = -(-N // 1024)
        rec = {"N": N,
               "model_per_256_rows_us": 1e6 * blocks * max(p.host_bytes / b_host, p.hbm_bytes / b_hbm),
               "model_single_read_us": 1e6 * launches * max(p.host_bytes / b_host, p.hbm_bytes / b_hbm),
               "t_comp_us": 1e6 * time_steps(lambda: dak.dak_gemm(p0, B, C, tuning=dict(pdl=1)), 5, 1),
               "plan": {k: v for k, v in dak.dak_gemm_launch_plan(p, N, tuning=dict(pdl=1)).items()
                        if k in ("cluster", "cluster_slots", "host_ctas", "hbm_ctas")}}
        for cols, key in ((1, "column_blocks"), (0, "shared_tiles")):
            dak.dak_link_begin(6)  # back-to-back launches in one host-link handoff sequence
            t = time_steps(lambda: dak.dak_gemm(p, B, C, tuning=dict(pdl=1, column_blocks=cols, link=6)), 5, 1)
            link = p.host_bytes * (blocks if cols else launches)
            rec[key] = {"us": t * 1e6, "host_link_bytes": link, "host_link_gbps": link / t / 1e9}
        rec["frac_single_read"] = rec["model_single_read_us"] / rec["shared_tiles"]["us"]
        rows.append(rec)
    p.free()
    p0.free()
    return {"op": "gate_up 28672x4096", "x": x, "tile_m": tile_m, "host_bytes": p.host_bytes, "rows": rows,
            "status": dak.dak_last_error()[0]}


# ------------------------------------------------------------------------------ hidden-state rows

def run_linears_n(dak, lin, b_host, b_hbm, dev, xs=(0.0, 0.25), ns=(1, 8, 32, 64)):
    """The four 8B linears (QKV, O, gate+up, down: 436 MB, more than L2) as one graph of four
    dak_gemm launches (programmatic launch, one host-link handoff sequence), at each offload
    ratio in xs and each hidden-state row count N in ns (decode batch sizes from one request
    to 64): time per pass, effective GB/s and the fraction of the tier roofline."""
    import torch
    import synth
    rows = []
    for x in xs:
        pls = {n: dak.dak_place_matrix(A, dak.host_tiles_for_ratio(x, A.shape[0])) for n, (A, _) in lin.items()}
        C_bytes = sum(p.host_bytes + p.hbm_bytes for p in pls.values())
        H = sum(p.host_bytes for p in pls.values())
        for N in ns:
            Bs = {n: torch.from_numpy(synth.normal_bf16(11, i, N * A.shape[1]).view("int16")).view(torch.bfloat16)
                  .to(dev).view(N, A.shape[1]) for i, (n, (A, _)) in enumerate(lin.items())}
            Cs = {n: torch.empty((N, A.shape[0]), dtype=torch.bfloat16, device=dev) for n, (A, _) in lin.items()}

            def one_pass():
                if H:  # (all in HBM there is nothing to hand on)
                    dak.dak_link_begin(7)
                for n, p in pls.items():
                    dak.dak_gemm(p, Bs[n], Cs[n], tuning=dict(pdl=1, link=7 if H else 0))
            one_pass()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                with torch.cuda.graph(g, stream=s):
                    one_pass()
            t = time_steps(g.replay, 20, 3)
            roof = tier_roofline(C_bytes, H / C_bytes, b_host, b_hbm)
            row = {"N": N, "x": x, "us": t * 1e6, "gbps": C_bytes / t / 1e9, "frac": (C_bytes / t) / roof}
            del g
            # the same four GEMMs as one grouped launch (dak_gemm_chain, no dependencies;
            # tensor cores at every N, B padded to 8 rows at N = 1)
            ops = [dict(A=p, B=Bs[n], C=Cs[n]) for n, p in pls.items()]
            ws = torch.zeros(dak.dak_gemm_chain_workspace_bytes(ops, N), dtype=torch.uint8, device=dev)
            g = _capture(lambda: dak.dak_gemm_chain(ops, workspace=ws, tuning=dict(pdl=1)))
            tc = time_steps(g.replay, 20, 3)
            row.update(chain_us=tc * 1e6, chain_gbps=C_bytes / tc / 1e9, chain_frac=(C_bytes / tc) / roof)
            cplan = dak.dak_gemm_chain_plan([A.shape for A, _ in lin.values()], N, n_host_tiles=[
                dak.host_tiles_for_ratio(x, A.shape[0]) for A, _ in lin.values()])
            row["chain_dealing"] = "by size" if cplan["by_size"] else "per operation"
            del g, ws
            rows.append(row)
        for p in pls.values():
            p.free()
    return {"ops": "8B QKV, O, gate+up, down: one graph of four dak_gemm launches (us, frac), and one grouped "
                   "dak_gemm_chain launch of the four (chain_us, chain_frac; chain_dealing: how its units were dealt to its CTAs)", "rows": rows,
            "status": dak.dak_last_error()[0]}


# ------------------------------------------------------------------------------ per operation, per x

def _capture(fn):
    """A CUDA graph of fn's launches (captured on a side stream)."""
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    return g


def run_per_op_x(dak, lin, attn, b_host, b_hbm, dev, ns=(1, 8, 32, 64)):
    """Each operation of the step alone, against its tier roofline at every offload ratio:
    the four 8B linears at x = 0, 0.05, ..., 0.5 for N in ns, the 32-request attention at
    x in {0, 0.125, 0.25, 0.5}, and the 1024x1024 GEMV at x = 0.25. Two timings per point:
    `single`, one launch after a write of twice the L2 size (cold L2, launch latency
    included; CUDA events around the launch), and `chain`, a CUDA graph of launches with
    programmatic launch and the host-link handoff (dak_link_begin) over enough copies of
    the placement that they stream more than twice the L2 size (the rate of the operation
    repeated back to back, as in a model's layers); for the linears also
    `grouped`, up to 8 of those copies in one dak_gemm_chain launch. Bytes are the
    operation's weights (or KV cache)."""
    import math
    import torch
    import synth
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device=dev)
    xs = [round(0.05 * i, 2) for i in range(11)]

    def single(fn, reps=5):
        ts = []
        for _ in range(reps):
            flush.fill_(1.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) / 1e3)
        return statistics.median(ts)

    def point(C_bytes, H, t1, tc):
        roof = tier_roofline(C_bytes, H / C_bytes, b_host, b_hbm)
        return {"x_effective": H / C_bytes, "single_us": t1 * 1e6, "chain_us": tc * 1e6,
                "single_gbps": C_bytes / t1 / 1e9, "chain_gbps": C_bytes / tc / 1e9, "roofline_gbps": roof / 1e9,
                "single_frac": (C_bytes / t1) / roof, "chain_frac": (C_bytes / tc) / roof}

    res = {"linears": [], "l2_bytes": l2}
    pdl = dict(pdl=1)
    linked = dict(pdl=1, link=2)

    def seq(launches, begin=True):
        if begin:  # (all in HBM there is nothing to hand on)
            dak.dak_link_begin(2)
        for f in launches:
            f()
    for i, (name, (A, _)) in enumerate(lin.items()):
        M, K = A.shape
        Ad = torch.from_numpy(A.view("int16")).view(torch.bfloat16).to(dev)
        copies = max(2, math.ceil(2 * l2 / (M * K * 2)))
        Bs = {N: torch.from_numpy(synth.normal_bf16(13, i, N * K).view("int16")).view(torch.bfloat16).to(dev)
              .view(N, K) for N in ns}
        Cs = {N: torch.empty((N, M), dtype=torch.bfloat16, device=dev) for N in ns}
        rows = []
        for x in xs:
            pls = [dak.dak_place_matrix(Ad, dak.host_tiles_for_ratio(x, M)) for _ in range(copies)]
            C_bytes, H = pls[0].host_bytes + pls[0].hbm_bytes, pls[0].host_bytes
            for N in ns:
                t1 = single(lambda: dak.dak_gemm(pls[0], Bs[N], Cs[N]))
                tun = linked if H else pdl
                g = _capture(lambda: seq([lambda p=p: dak.dak_gemm(p, Bs[N], Cs[N], tuning=tun) for p in pls], H > 0))
                tc = time_steps(g.replay, 10, 3) / copies
                del g
                rec = dict(x=x, N=N, **point(C_bytes, H, t1, tc))
                # the copies as one grouped launch (dak_gemm_chain: up to 8 operations)
                ops = [dict(A=p, B=Bs[N], C=Cs[N]) for p in pls[:8]]
                ws = torch.zeros(dak.dak_gemm_chain_workspace_bytes(ops, N), dtype=torch.uint8, device=dev)
                g = _capture(lambda: dak.dak_gemm_chain(ops, workspace=ws, tuning=pdl))
                tg = time_steps(g.replay, 10, 3) / len(ops)
                del g, ws
                roof = tier_roofline(C_bytes, H / C_bytes, b_host, b_hbm)
                rec.update(grouped_us=tg * 1e6, grouped_frac=(C_bytes / tg) / roof)
                rows.append(rec)
            for p in pls:
                p.free()
        del Ad
        res["linears"].append({"op": f"{name} {M}x{K}", "copies_in_chain": copies, "rows": rows})
        torch.cuda.empty_cache()
    # the attention (1 GiB of KV: launches back to back already stream more than twice the L2)
    q, k, v = attn
    Q = torch.from_numpy(q.view("int16")).view(torch.bfloat16).to(dev)
    O = torch.empty_like(Q)
    arows = []
    for x in (0.0, 0.125, 0.25, 0.5):
        p = dak.dak_place_kv(k, v, dak.host_requests_for_ratio(x, k.shape[0]))
        ns_ = dak.dak_attn_default_split(p)
        ws = torch.empty(max(1, dak.dak_attn_workspace_bytes(q.shape[0], q.shape[1], q.shape[2], ns_) // 4),
                         dtype=torch.float32, device=dev)
        t1 = single(lambda: dak.dak_attn(Q, p, O=O, workspace=ws, tuning=dict(n_split=ns_)))
        dak.dak_link_begin(3)  # eager launches back to back, each joining the sequence
        tc = time_steps(lambda: dak.dak_attn(Q, p, O=O, workspace=ws, tuning=dict(pdl=1, n_split=ns_, link=3)),
                        10, 3)
        C_bytes, H = p.host_bytes + p.hbm_bytes, p.host_bytes
        arows.append(dict(x=x, n_split=ns_, **point(C_bytes, H, t1, tc)))
        p.free()
    res["attention"] = {"op": "GQA decode attention, 32 requests, 32/8 heads, D 128, context 8192",
                        "rows": arows}
    # the single decode GEMV (2 MiB: the chain cycles over enough copies to leave L2)
    A1, B1 = synth.gemm_inputs(1024, 1024, 1, seed=0)
    A1d = torch.from_numpy(A1.view("int16")).view(torch.bfloat16).to(dev)
    B1d = torch.from_numpy(B1.view("int16")).view(torch.bfloat16).to(dev)
    C1 = torch.empty((1, 1024), dtype=torch.bfloat16, device=dev)
    copies = math.ceil(2 * l2 / (1024 * 1024 * 2))
    pls = [dak.dak_place_matrix(A1d, dak.host_tiles_for_ratio(0.25, 1024)) for _ in range(copies)]
    t1 = single(lambda: dak.dak_gemm(pls[0], B1d, C1))
    g = _capture(lambda: seq([lambda p=p: dak.dak_gemm(p, B1d, C1, tuning=linked) for p in pls]))
    tc = time_steps(g.replay, 10, 3) / copies
    del g
    res["gemv"] = dict(op="GEMV 1024x1024, N = 1, x = 0.25 (4 of 16 tile rows on the host)", copies_in_chain=copies,
                       **point(pls[0].host_bytes + pls[0].hbm_bytes, pls[0].host_bytes, t1, tc))
    for p in pls:
        p.free()
    res["status"] = dak.dak_last_error()[0]
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [s.strip() for s in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        inside = [r for t, r in self.rows if t0 <= t <= t1]
        where = "timed region"
        if not inside:
            inside = [r for t, r in self.rows]
            where = "around the timed region (region shorter than the sampling period)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm = [float(r[1]) for r in inside if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in inside if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in inside for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside), "sampled": where,
                "power_w_max": max((float(r[3]) for r in inside if r[3].replace(".", "").isdigit()), default=None)}


# ------------------------------------------------------------------------------ measurement

def measure_tiers(dak):
    """B_host and B_hbm: best read-stream bandwidth of each tier (GB/s), plus the
    concurrent split at the kernels' default host CTA count."""
    G = 1 << 30
    best_h, best_g = 0.0, 0.0
    for m, c, w in ((0, 16, 4), (0, 32, 4), (2, 16, 4)):
        try:
            g, ok = dak.dak_probe_read_bw(0, G, m, c, w, 32768, 3)
            if ok:
                best_h = max(best_h, g)
        except dak.DakError:
            pass
    for c in (dak.dak_sm_count(), 100):
        g, ok = dak.dak_probe_read_bw(1, 4 * G, 0, c, 4, 32768, 3)
        if ok:
            best_g = max(best_g, g)
    hc = 16
    ch, cg = dak.dak_probe_concurrent(G, 4 * G, hc, 4, dak.dak_sm_count() - hc, 4, 32768, 3)
    return best_h * 1e9, best_g * 1e9, {"host_ctas": hc, "host_gbps": ch, "hbm_gbps": cg,
                                        "h2d_copy_gbps": h2d_copy_gbps()}


def h2d_copy_gbps(nbytes=1 << 30, reps=3):
    """cudaMemcpy host-to-device rate from pinned memory (the copy engine's path), recorded
    beside the SM read probes for comparison."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d.copy_(h, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        d.copy_(h, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    gbps = reps * nbytes / (e0.elapsed_time(e1) / 1e3) / 1e9
    del h, d
    return gbps


def time_steps(fn, steps, warmup, sync_all=None):
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if sync_all:
        sync_all()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    if sync_all:
        sync_all()
    return e0.elapsed_time(e1) / 1e3 / steps


def aggregate_replicas(t_step, bytes_per_step, dist=None):
    """Replicas: every rank runs the same step on its own GPU. The job time is the slowest
    rank's; the job moves world x bytes_per_step per step. Returns (GB/s, max step time)."""
    world = 1
    if dist is not None and dist.is_initialized():
        import torch
        world = dist.get_world_size()
        dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
        tt = torch.tensor([float(t_step)], dtype=torch.float64, device=dev)
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        t_step = float(tt.item())
    return world * bytes_per_step / t_step / 1e9, t_step


def step_config(args, world):
    """The workload both arms report (identical for --impl dak and --impl reference)."""
    return {"workload": f"8B-shaped decode layer at batch {args.batch}: linears QKV 6144x4096, O 4096x4096, "
                        f"gate+up 28672x4096, down 4096x14336 + GQA decode attention over 32 requests, 32/8 heads, "
                        f"D 128, context 8192; bf16 weights/KV, fp32 accumulate",
            "x": args.x, "batch": args.batch, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (1.51 GB of weights and KV per step)"}


def tier_roofline(C, x, bh, bg):
    t = max(x * C / bh, (1 - x) * C / bg)
    return C / t


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


# ------------------------------------------------------------------------------ CPU oracle

def cpu_oracle_sample(lin, attn, frac_rows=1 / 32, offset=0):
    """Time the CPU oracle (as it stands) on a bounded sample of one step: every 32nd tile
    row of each linear (from tile row `offset` mod 32) and one request in 32 of the
    attention (the offset-th). Returns (GB/s, sample, s)."""
    import numpy as np
    from oracle import attention as oa
    from oracle import gemm as og
    f = int(1 / frac_rows)
    t0 = time.perf_counter()
    nbytes = 0
    for A, B in lin.values():
        rows = np.concatenate([np.arange(t * 64, t * 64 + 64) for t in range(offset % f, A.shape[0] // 64, f)])
        og.gemm_ref(A[rows], B)
        nbytes += rows.size * A.shape[1] * 2
    q, k, v = attn
    nreq = max(1, int(q.shape[0] * frac_rows))
    r0 = (offset * nreq) % q.shape[0]
    oa.decode_attention_ref(q[r0:r0 + nreq], k[r0:r0 + nreq], v[r0:r0 + nreq])
    nbytes += 2 * k[r0:r0 + nreq].size * 2
    dt = time.perf_counter() - t0
    return nbytes / dt / 1e9, f"1/{int(1 / frac_rows)} of the step: one 64-row tile in {int(1 / frac_rows)} of each " \
                              f"linear and {nreq} of {q.shape[0]} attention requests ({nbytes / 1e6:.0f} MB)", dt


def cpu_oracle_timed(lin, attn, target_s=10.0):
    """The oracle over successive 1/32 slices of the step (offsets 0, 1, 2, ..., every 32 a
    whole step) until about target_s seconds have passed. Returns (GB/s, sample)."""
    t0 = time.perf_counter()
    nbytes, n = 0.0, 0
    while True:
        g, _, dt = cpu_oracle_sample(lin, attn, offset=n)
        nbytes += g * dt * 1e9
        n += 1
        el = time.perf_counter() - t0
        if el >= target_s:
            break
    return nbytes / el / 1e9, (f"{n} slices of 1/32 of the step (every 32nd tile row of each linear from "
                               f"offsets 0..{n - 1} mod 32, one attention request each; {nbytes / 1e9:.1f} GB, "
                               f"{el:.1f} s)")


def cpu_oracle_sample_sliced(batch=32, frac=32):
    """cpu_oracle_sample on the same sampled tile rows and requests, drawing only those
    slices of the inputs (the generator is counter-based, so any slice regenerates alone)."""
    import numpy as np
    import synth
    from oracle import attention as oa
    from oracle import gemm as og
    parts = []
    for i, (name, (M, K)) in enumerate(synth.LINEARS_8B.items()):
        s = 0 + i
        rows = [synth.normal_bf16(s, 1, 64 * K, 0.0, synth.WEIGHT_STD, offset=t * 64 * K).reshape(64, K)
                for t in range(0, M // 64, frac)]
        B = synth.normal_bf16(s, 2, batch * K).reshape(batch, K)
        parts.append((np.concatenate(rows), B))
    c = synth.ATTN_DECODE
    nreq = max(1, c["batch"] // frac)
    ti = len(synth.LINEARS_8B)
    q = synth.normal_bf16(ti, 11, nreq * c["h_q"] * c["head_dim"]).reshape(nreq, c["h_q"], c["head_dim"])
    kv = [synth.attn_kv_request(b, c["h_kv"], c["head_dim"], c["context"], seed=0, tensor_index=ti)
          for b in range(nreq)]
    k = np.stack([a for a, _ in kv])
    v = np.stack([b for _, b in kv])
    t0 = time.perf_counter()
    nbytes = 0
    for A, B in parts:
        og.gemm_ref(A, B)
        nbytes += A.size * 2
    oa.decode_attention_ref(q, k, v)
    nbytes += 2 * k.size * 2
    dt = time.perf_counter() - t0
    return nbytes / dt / 1e9, dt


def cpu_oracle_one_core(timeout_s=300):
    """The same oracle sample in a child process limited to one BLAS / OpenMP thread (the
    thread count is fixed when numpy loads, so it has to be a fresh process)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1")
    code = ("import json, sys; sys.path.insert(0, %r); import bench; "
            "g, dt = bench.cpu_oracle_sample_sliced(); print(json.dumps({'value': g, 'seconds': dt}))" % ROOT)
    try:
        out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                             timeout=timeout_s, check=True).stdout.strip().splitlines()[-1]
        r = json.loads(out)
        return {"value": r["value"], "unit": "GB/s", "cores": 1, "seconds": r["seconds"]}
    except Exception as e:  # a failed reference measurement must not fail the benchmark
        return {"unavailable": f"{type(e).__name__}"}


def cpu_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        if info:
            return max(i.get("num_threads", 1) for i in info)
    except Exception:
        pass
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------------------ main

def run_reference(args, rank, world):
    if rank != 0:
        return
    w_bytes, kv_bytes = workload_bytes(args.batch)
    lin, attn = gen_inputs(args.batch)
    for i in range(args.warmup):
        cpu_oracle_sample(lin, attn, offset=i)
    vals, dts = [], []
    for i in range(args.steps):  # successive 1/32 slices of the step
        gbps, sample, dt = cpu_oracle_sample(lin, attn, offset=args.warmup + i)
        vals.append(gbps)
        dts.append(dt)
    v = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(dts),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": step_config(args, world),
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = _args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "dak" else "gloo")
    if args.profile:
        run_profile(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        if dist:
            dist.barrier()
            dist.destroy_process_group()
        return

    import torch
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import direct_host_memory_gb300 as dak

    def sync_all():
        if dist:
            dist.barrier()

    b_host, b_hbm, conc = measure_tiers(dak)
    lin, attn = gen_inputs(args.batch)
    w_bytes, kv_bytes = workload_bytes(args.batch)

    st = Step(dak, lin, attn, args.x, dev)
    C = st.total_bytes
    # the attention launch is the step's dominant kernel: time it with events on its stream
    att_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    for _ in range(args.warmup):
        st.run()
    torch.cuda.synchronize()
    status = dak.dak_last_error()
    sync_all()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    t_wall0 = time.time()
    e0.record()
    step_ev[0].record()
    for i in range(args.steps):
        st.run(att_ev[i])
        step_ev[i + 1].record()
    e1.record()
    torch.cuda.synchronize()
    t_wall1 = time.time()
    per_step = sorted(step_ev[i].elapsed_time(step_ev[i + 1]) for i in range(args.steps))

    def pct(q):
        return per_step[min(len(per_step) - 1, int(q * (len(per_step) - 1) + 0.5))]
    sync_all()
    value, t_step = aggregate_replicas(e0.elapsed_time(e1) / 1e3 / args.steps, st.total_bytes, dist)
    att_ms = statistics.mean(a.elapsed_time(b) for a, b in att_ev)
    time.sleep(0.3)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    status2 = dak.dak_last_error()

    # end to end through the public API with host buffers: hidden states / queries copied in
    # from pinned memory and outputs copied back every step
    # (every B and Q in one pinned buffer and one copy in; every C and O in one copy out)
    host_in = st.inbuf.cpu().pin_memory()
    host_out = torch.empty(st.outbuf.shape, dtype=st.outbuf.dtype).pin_memory()
    h2d = host_in.numel() * 2
    d2h = host_out.numel() * 2

    def e2e_step():
        st.inbuf.copy_(host_in, non_blocking=True)
        st.run()
        host_out.copy_(st.outbuf, non_blocking=True)

    e2e_value, t_e2e = aggregate_replicas(time_steps(e2e_step, max(10, args.steps // 3), 3, sync_all), C, dist)

    # per-x sweep with the prefetch baselines
    per_x = []
    if not args.no_sweep:
        cs = torch.cuda.Stream()
        evs = [torch.cuda.Event() for _ in range(len(lin) + 1)]
        for x in (0.0, 0.05, 0.1, 0.125, 0.25, 0.5):
            s = st if abs(x - args.x) < 1e-12 else Step(dak, lin, attn, x, dev)
            t = time_steps(s.run, 30, 3)
            rec = {"x": x, "host_bytes": s.host_bytes, "gbps": s.total_bytes / t / 1e9,
                   "tok_s": args.batch / (t * LAYERS_8B), "ms": t * 1e3,
                   "roofline_gbps": tier_roofline(s.total_bytes, s.host_bytes / s.total_bytes, b_host, b_hbm) / 1e9}
            rec["frac"] = rec["gbps"] / rec["roofline_gbps"]
            if x > 0:
                s.alloc_staging(dev)
                tp = time_steps(s.run_prefetch_serial, 10, 2)
                to = time_steps(lambda: s.run_prefetch_overlap(cs, evs), 10, 2)
                rec["prefetch_serial_gbps"] = s.total_bytes / tp / 1e9
                rec["prefetch_overlap_gbps"] = s.total_bytes / to / 1e9
                rec["vs_prefetch_best"] = rec["gbps"] / max(rec["prefetch_serial_gbps"], rec["prefetch_overlap_gbps"])
                del s.stage, s.stage_kv
            per_x.append(rec)
            if s is not st:
                s.free()
            torch.cuda.empty_cache()
    status3 = dak.dak_last_error()

    pk, pk_src = peaks()
    att_bytes = kv_bytes + 2 * st.Q.numel() * 2
    x_eff = st.host_bytes / C
    att_host = st.kv.host_bytes
    att_roof = tier_roofline(att_bytes, att_host / att_bytes, b_host, b_hbm)
    achieved = att_bytes / (att_ms / 1e3)
    traffic = read_ncu_traffic()

    models = [m.strip() for m in args.decode.split(",") if m.strip() in ("8b", "70b")]
    decode = {m: run_decode(dak, args, b_host, b_hbm, dev, sync_all, local, model=m, full=(m == "8b"))
              for m in models}
    planner_check = None
    if not args.no_planner_check:
        pc_sampler = ClockSampler(local)
        pc_sampler.start()
        tw0 = time.time()
        planner_check = run_planner_check(dak, lin, attn, b_host, b_hbm, dev)
        tw1 = time.time()
        pc_sampler.stop()
        planner_check["clocks"] = pc_sampler.summary(tw0, tw1)  # tensor-bound timings follow the SM clock
    large_n = None if args.no_planner_check else run_large_n(dak, lin, b_host, b_hbm, dev)
    per_n = None if args.no_sweep else run_linears_n(dak, lin, b_host, b_hbm, dev)
    per_op = None if args.no_sweep else run_per_op_x(dak, lin, attn, b_host, b_hbm, dev)

    cpu = None
    if rank == 0 and not args.no_cpu:
        gbps, sample = cpu_oracle_timed(lin, attn)
        cpu = {"value": gbps, "unit": "GB/s", "cores": cpu_threads(), "kind": "oracle", "sample": sample,
               "one_core": cpu_oracle_one_core()}

    n = world
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": step_config(args, world),
        "ms_per_step_p10_p50_p90": [pct(0.1), pct(0.5), pct(0.9)],
        "step": {"x_effective": x_eff, "bytes_per_step": C, "host_bytes_per_step": st.host_bytes,
                 "kernels": "dak_gemm x4 (tcgen05 for N >= 2) + dak_attn (+ split combine)"},
        "decode_tok_s": n * args.batch / (t_step * LAYERS_8B),
        "tier_roofline_gbps": tier_roofline(C, x_eff, b_host, b_hbm) / 1e9,
        "tier_roofline_frac": (C / t_step) / tier_roofline(C, x_eff, b_host, b_hbm),
        "b_host_gbps": b_host / 1e9, "b_hbm_gbps": b_hbm / 1e9, "concurrent_probe": conc,
        "roofline": {"bound": "hbm", "kernel": "attn_kernel<128> + split combine (dak_attn)",
                     "achieved": achieved / 1e9, "peak": att_roof / 1e9, "unit": "GB/s",
                     "frac": achieved / att_roof, "traffic": traffic,
                     "peak_kind": "tier-aggregate C/max(xC/B_host,(1-x)C/B_hbm), B_host/B_hbm measured in this run",
                     "hbm_peak_gbs": pk.get("hbm_gbs"), "hbm_peak_source": pk_src,
                     "algorithmic_bytes_per_launch": att_bytes, "launch_ms": att_ms},
        "per_x": per_x,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": st.launches * args.steps,
        "clocks": clocks,
        "status": [status[0], status2[0], status3[0]],
    }
    if "8b" in decode:
        line["decode_step"] = decode["8b"]
    if "70b" in decode:
        line["decode_step_70b"] = decode["70b"]
    if per_op:
        line["per_op_x"] = per_op
    if planner_check:
        line["planner_check"] = planner_check
    if large_n:
        line["large_n"] = large_n
    if per_n:
        line["per_n"] = per_n
    if cpu:
        line["cpu_baseline"] = cpu
    st.free()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


KERNEL_SOURCES = ["direct_host_memory_gb300/csrc/dak_attn.cu", "direct_host_memory_gb300/csrc/dak_device.cuh"]


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_ncu_traffic():
    """DRAM bytes per launch of the attention kernel at this workload from the committed ncu
    summary, or None when there is none or the kernel source changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            t = json.load(f)
        if t.get("source_hash") != kernel_source_hash():
            return None
        return t.get("attn_kernel_dram_bytes_per_launch")
    except Exception:
        return None


def run_profile(args):
    """One operation of the step, placed at --x, launched --warmup + --steps times."""
    import torch
    import direct_host_memory_gb300 as dak
    import synth
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    if args.profile == "decode":
        # the 8B-shaped decode step at x_global = --x (planner ratios), one graph replay per step
        cfg = dict(synth.DECODER_8B)
        if args.decode_batch:
            cfg["batch"] = args.decode_batch
        b_host, b_hbm, _ = measure_tiers(dak) if args.x > 0 else (211e9, 7.3e12, None)
        pk, _ = peaks()
        units, _ = decode_plan(dak, cfg, b_host, b_hbm, args.x, pk.get("bf16_tflops_sustained", 1700.0) * 1e12)
        dec = build_decoder(dak, cfg, units, plain_launch=args.plain_launch)
        x_in = torch.from_numpy(synth.decoder_x0(cfg, cfg["batch"]).view("int16")).view(torch.bfloat16).to(dev)
        pos = torch.full((cfg["batch"],), cfg["context"] - 1, dtype=torch.int32, device=dev)
        out = torch.empty_like(x_in)
        if args.plain_launch:
            t = time_steps(lambda: dec.step(x_in, pos, out), args.steps, args.warmup)
        else:
            dec.capture(x_in, pos, out, dak.MODE_DIRECT)
            t = time_steps(dec.replay, args.steps, args.warmup)
        st = dak.dak_last_error()
        print(json.dumps({"profile": "decode", "x_global": args.x, "ms_per_step": t * 1e3,
                          "tok_s": cfg["batch"] / t, "launches_per_step": dec.launches(), "status": st[0],
                          "host_units_per_layer": units[0]}))
        dec.free()
        return
    if args.profile == "chain":
        pls, ops = [], []
        for i, (name, (M, K)) in enumerate(synth.LINEARS_8B.items()):
            A, B = synth.gemm_inputs(M, K, args.batch, seed=0, tensor_index=i)
            pls.append(dak.dak_place_matrix(A, dak.host_tiles_for_ratio(args.x, M)))
            ops.append(dict(A=pls[-1], B=torch.from_numpy(B.view("int16")).view(torch.bfloat16).to(dev)))
        ws = torch.zeros(dak.dak_gemm_chain_workspace_bytes(ops, args.batch), dtype=torch.uint8, device=dev)
        outs = [torch.empty((args.batch, p.meta["M"]), dtype=torch.bfloat16, device=dev) for p in pls]
        for o, c in zip(ops, outs):
            o["C"] = c
        t = time_steps(lambda: dak.dak_gemm_chain(ops, workspace=ws), args.steps, args.warmup)
        nbytes = sum(p.host_bytes + p.hbm_bytes for p in pls)
        print(json.dumps({"profile": "chain", "x": args.x, "batch": args.batch, "us_per_launch": t * 1e6,
                          "gbps": nbytes / t / 1e9, "status": dak.dak_last_error()[0]}))
        for p in pls:
            p.free()
        return
    if args.profile == "attn":
        c = synth.ATTN_DECODE
        q, k, v = synth.attn_inputs(c["batch"], c["h_q"], c["h_kv"], c["head_dim"], c["context"], seed=0,
                                    tensor_index=len(synth.LINEARS_8B))
        p = dak.dak_place_kv(k, v, dak.host_requests_for_ratio(args.x, c["batch"]))
        Q = torch.from_numpy(q.view("int16")).view(torch.bfloat16).to(dev)
        O = torch.empty_like(Q)
        fn = lambda: dak.dak_attn(Q, p, O=O)  # noqa: E731
        nbytes = k.nbytes * 2
    else:
        M, K = synth.LINEARS_8B[args.profile]
        A, B = synth.gemm_inputs(M, K, args.batch, seed=0, tensor_index=list(synth.LINEARS_8B).index(args.profile))
        p = dak.dak_place_matrix(A, dak.host_tiles_for_ratio(args.x, M, args.tile_m), tile_m=args.tile_m)
        Bt = torch.from_numpy(B.view("int16")).view(torch.bfloat16).to(dev)
        C = torch.empty((args.batch, M), dtype=torch.bfloat16, device=dev)
        fn = lambda: dak.dak_gemm(p, Bt, C)  # noqa: E731
        nbytes = A.nbytes
    t = time_steps(fn, args.steps, args.warmup)
    st = dak.dak_last_error()
    print(json.dumps({"profile": args.profile, "x": args.x, "batch": args.batch, "tile_m": args.tile_m,
                      "us_per_launch": t * 1e6,
                      "gbps": nbytes / t / 1e9, "host_bytes": p.host_bytes, "status": st[0],
                      "source_hash": kernel_source_hash()}))
    p.free()


if __name__ == "__main__":
    main()
