"""Failure detection on the GPU without a fault: a bounded wait runs out, the status word
reports it, and the context keeps working."""
import numpy as np
import pytest

import synth
from gpu_util import FP32_OUT_TOL, to_dev, to_np
from oracle import gemm as og

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dak(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    import direct_host_memory_gb300 as m
    return m


def test_bounded_wait_times_out_and_context_survives(dak):
    assert dak.dak_last_error()[0] == 0
    dak.dak_selftest_wait()
    st, info = dak.dak_last_error()
    assert st == 6  # DAK_ERR_TIMEOUT
    assert (info >> 32) == 0x5E1F
    assert dak.dak_last_error()[0] == 0  # read clears it
    A, B = synth.gemm_inputs(128, 256, 8, seed=12)
    p = dak.dak_place_matrix(A, 1)
    C = dak.dak_gemm(p, to_dev(B), c_fp32=True)
    assert dak.dak_last_error()[0] == 0
    assert og.rel_err(to_np(C), og.gemm_ref(A, B)) <= FP32_OUT_TOL
    p.free()


def test_handoff_wait_gives_up_without_error(dak):
    """The host-link handoff's wait only paces loads: one that nothing releases gives up
    after its bound, is counted, and raises no error."""
    dak.dak_link_timeouts()  # start from zero
    dak.dak_selftest_link()
    assert dak.dak_link_timeouts() == 1
    assert dak.dak_link_timeouts() == 0  # read clears it
    assert dak.dak_last_error()[0] == 0
