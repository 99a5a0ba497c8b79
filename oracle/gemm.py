"""Decode GEMM over a tile-row partitioned weight matrix -- oracle (fp64).

[DAK] section 4.1 "Data Partition" and Fig. 5a: C = A x B where A (weights, M x K) is
cut along M into tile rows of m x K; some tile rows sit in host memory and the rest in
GPU memory, and every tile row yields an independent block of output rows. Where a tile
row is stored changes only where its bytes are read from, never the product, so the
oracle is the plain definition of the product:

    C[n][r] = sum_k A[r][k] * B[n][k]          (A: [M][K], B: [N][K], C: [N][M])

evaluated in fp64 from the exact bf16 inputs. ``tile_rows_product`` evaluates the same
thing one tile row at a time, reading each row block from the tier the placement puts it
in, to state the partition explicitly; the tests check that it equals ``gemm_ref``.

Parity pins (tests/test_oracle_gemm.py): identity and selection matrices (C = B, and
C[n][r] = B[n][k_r] on non-square shapes, which catches a transposed operand), all-ones
A (row sums), integer inputs against exact Python-integer sums, and linearity.
"""
import numpy as np

from .bf16 import to_f64


def gemm_ref(A_bits, B_bits) -> np.ndarray:
    """fp64 C [N][M] = B [N][K] . A[M][K]^T from bf16 bit arrays."""
    A = to_f64(A_bits)
    B = to_f64(B_bits)
    assert A.ndim == 2 and B.ndim == 2 and A.shape[1] == B.shape[1]
    return B @ A.T


def tile_rows_product(A_host_bits, A_hbm_bits, B_bits, tile_m: int) -> np.ndarray:
    """The product assembled tile row by tile row from the two tiers.

    ``A_host_bits`` holds tile rows 0 .. h-1 (the rows placed in host memory) and
    ``A_hbm_bits`` the remaining rows, in order ([DAK] Fig. 5a puts tile row 0 on the host).
    """
    B = to_f64(B_bits)
    parts = []
    for tier in (A_host_bits, A_hbm_bits):
        A = to_f64(tier)
        for r0 in range(0, A.shape[0], tile_m):
            blk = A[r0:r0 + tile_m]
            out = np.zeros((B.shape[0], blk.shape[0]))
            for n in range(B.shape[0]):
                out[n] = blk @ B[n]
            parts.append(out)
    if not parts:
        return np.zeros((B.shape[0], 0))
    return np.concatenate(parts, axis=1)


def rel_err(got, ref) -> float:
    """max |got - ref| / max |ref| (0 when both are all zero)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref)) if ref.size else 0.0
    num = np.max(np.abs(got - ref)) if ref.size else 0.0
    if den == 0.0:
        return float(num)
    return float(num / den)
