"""Helpers for the GPU tests: bf16 bit arrays <-> torch tensors, tolerances."""
import numpy as np

# rel-err bound for bf16 inputs with fp32 accumulation, max |gpu - ref| / max |ref| against the
# fp64 oracle: the 2e-2 the direct-access kernels are held to for bf16 outputs
REL_TOL = 2e-2
# the kernels accumulate in fp32; against the fp64 oracle the error is far below REL_TOL
FP32_OUT_TOL = 1e-5


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
