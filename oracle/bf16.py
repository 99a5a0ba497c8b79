"""bf16 helpers for the oracle (its own copy; the CUDA path does its own conversions).

bf16 is the upper 16 bits of an IEEE-754 binary32 value. Decoding is exact; encoding
rounds to nearest, ties to even. Pinned by tests: exact round-trip of every bf16 value,
known rounding cases (ties to even, overflow to inf).
"""
import numpy as np


def to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def round_f32_to_bf16(x) -> np.ndarray:
    """float32 values -> bf16 bits, round to nearest even (NaN kept quiet)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    nan = np.isnan(f)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    r[nan] = ((u[nan] >> np.uint64(16)) | np.uint64(0x40)).astype(np.uint16)
    return r


def round_f64_to_bf16(x) -> np.ndarray:
    """float64 -> bf16 bits via float32 (exact for values already representable in fp32)."""
    return round_f32_to_bf16(np.asarray(x, dtype=np.float64).astype(np.float32))
