"""Pins for the GEMM oracle: structured inputs with known products, exact integer sums."""
import numpy as np
import pytest

import synth
from oracle import bf16 as obf
from oracle import gemm as og

pytestmark = pytest.mark.cpu


def _bits(x):
    return obf.round_f64_to_bf16(np.asarray(x, dtype=np.float64))


def test_bf16_roundtrip_and_rounding():
    allbits = np.arange(1 << 16, dtype=np.uint16)
    f = obf.to_f32(allbits)
    finite = np.isfinite(f)
    assert np.array_equal(obf.round_f32_to_bf16(f[finite]), allbits[finite])
    # ties to even: 1 + 2^-8 sits halfway between 1 and 1 + 2^-7 -> rounds to 1
    assert obf.round_f32_to_bf16(np.float32(1 + 2 ** -8)) == 0x3F80
    # 1 + 3*2^-8 is halfway between 1+2^-7 and 1+2^-6 -> rounds to the even one (1+2^-6)
    assert obf.round_f32_to_bf16(np.float32(1 + 3 * 2 ** -8)) == 0x3F82
    assert obf.round_f32_to_bf16(np.float32(3.4e38)) == 0x7F80  # overflow -> inf


def test_identity_gives_B():
    K = 48
    A = _bits(np.eye(K))
    _, B = synth.gemm_inputs(K, K, 3, seed=5)
    C = og.gemm_ref(A, B)
    assert np.array_equal(C, obf.to_f64(B))


def test_selection_matrix_nonsquare_catches_transpose():
    M, K, N = 40, 72, 5
    rng = synth.uniform_f64(7, 0, M)
    cols = (rng * K).astype(int)
    A = np.zeros((M, K))
    A[np.arange(M), cols] = 1.0
    _, B = synth.gemm_inputs(M, K, N, seed=3)
    C = og.gemm_ref(_bits(A), B)
    Bf = obf.to_f64(B)
    assert C.shape == (N, M)
    assert np.array_equal(C, Bf[:, cols])


def test_all_ones_gives_row_sums():
    M, K, N = 16, 100, 4
    _, B = synth.gemm_inputs(M, K, N, seed=9)
    C = og.gemm_ref(_bits(np.ones((M, K))), B)
    rs = obf.to_f64(B).sum(axis=1)
    assert np.allclose(C, rs[:, None], rtol=0, atol=1e-12)


def test_integer_inputs_exact_against_python_ints():
    M, K, N = 24, 37, 3
    A, B = synth.gemm_inputs(M, K, N, seed=11, integer=True)
    Ai = obf.to_f64(A).astype(int).tolist()
    Bi = obf.to_f64(B).astype(int).tolist()
    C = og.gemm_ref(A, B)
    for n in range(N):
        for r in range(M):
            exact = sum(Ai[r][k] * Bi[n][k] for k in range(K))
            assert C[n, r] == exact


def test_linearity_in_A():
    M, K, N = 8, 64, 2
    A1, B = synth.gemm_inputs(M, K, N, seed=1, integer=True)
    A2, _ = synth.gemm_inputs(M, K, N, seed=2, integer=True)
    S = _bits(obf.to_f64(A1) + obf.to_f64(A2))  # small integers: exact in bf16
    assert np.array_equal(og.gemm_ref(S, B), og.gemm_ref(A1, B) + og.gemm_ref(A2, B))


@pytest.mark.parametrize("M,tile_m,h", [(256, 64, 1), (200, 64, 2), (64, 64, 0), (130, 64, 3)])
def test_tile_row_partition_equals_product(M, tile_m, h):
    K, N = 96, 3
    A, B = synth.gemm_inputs(M, K, N, seed=4)
    cut = min(M, h * tile_m)
    C = og.tile_rows_product(A[:cut], A[cut:], B, tile_m)
    assert np.allclose(C, og.gemm_ref(A, B), rtol=1e-13, atol=1e-13)


def test_rel_err_metric():
    ref = np.array([1.0, -4.0, 2.0])
    assert og.rel_err(ref + np.array([0.0, 0.04, 0.0]), ref) == pytest.approx(0.01)
    assert og.rel_err(np.zeros(3), np.zeros(3)) == 0.0
