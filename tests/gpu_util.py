"""Helpers for the GPU tests: bf16 bit arrays <-> torch tensors, tolerances."""
import numpy as np

# rel-err bound for bf16 inputs with fp32 accumulation, max |gpu - ref| / max |ref| against the
# fp64 oracle: the 2e-2 the direct-access kernels are held to for bf16 outputs
REL_TOL = 2e-2
# the kernels accumulate in fp32; against the fp64 oracle the error is far below REL_TOL
FP32_OUT_TOL = 1e-5
# fp32-output attention (dak_attn_f32): scores, probabilities and the online-softmax rescaling
# run in fp32 (P enters P.V as bf16(P) + bf16(P - bf16(P)), 2^-17 relative); over up to
# 8192 tokens the rescaling steps and sums leave about 1e-5 of max |ref|, so 1e-4 catches a
# dropped or doubled token (about 1/L of an output, a few 1e-3 of max |ref| at L = 8192)
ATTN_FP32_TOL = 1e-4
# Per-element error with a floor of 1e-3 rms(ref): |got - ref| / max(|ref|, 1e-3 rms(ref)).
# It is reported, not bounded: elements near zero carry the absolute error of the fp32 path
# (or of a decode step's bf16 intermediates) over the floor, so its maximum says little about
# the arithmetic; the bounds are the max-normalised ones above. check_errors records every
# check here and conftest.py prints the table at the end of the session.
REPORT = []


def elem_err(got, ref, floor_frac=1e-3):
    """(max, 99.9th percentile, median) of |got - ref| / max(|ref|, floor_frac * rms(ref))."""
    got = np.asarray(got, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    if ref.size == 0:
        return 0.0, 0.0, 0.0
    rms = float(np.sqrt(np.mean(ref * ref)))
    den = np.maximum(np.abs(ref), floor_frac * rms)
    den[den == 0.0] = 1.0
    e = np.abs(got - ref) / den
    return float(e.max()), float(np.quantile(e, 0.999)), float(np.median(e))


def check_errors(got, ref, rel_tol, kind):
    """Assert the max-normalised error against rel_tol and record it with the per-element
    report (kind names the output: bf16, fp32 or a decode step's)."""
    import os
    from oracle import gemm as og
    rel = og.rel_err(got, ref)
    emax, ep, emed = elem_err(got, ref)
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    REPORT.append((test, kind, rel, rel_tol, emax, ep, emed))
    assert rel <= rel_tol, f"max-normalised error {rel:.3e} > {rel_tol:.1e}"
    return rel, emax, ep


def to_dev(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_np(t) -> np.ndarray:
    return t.detach().double().cpu().numpy()


def bits_of(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)
    return t.detach().cpu().view(torch.int32).numpy().view(np.uint32)
