"""Host-side fault injection without a GPU: the switch's API, its environment variable and
the live-allocation counters (the GPU half, tests/test_fault_injection_gpu.py, makes the
injected failures happen inside placements, decoders and GEMM launches)."""
import os
import subprocess
import sys

import pytest

from conftest import ROOT

pytestmark = pytest.mark.cpu


@pytest.fixture(scope="module")
def dak():
    import __graft_entry__
    __graft_entry__.build()
    import direct_host_memory_gb300 as m
    return m


def test_switch_round_trip(dak):
    for kind in (dak.FAULT_HOST_ALLOC, dak.FAULT_DEVICE_ALLOC, dak.FAULT_TENSOR_MAP):
        dak.dak_inject_fault(kind, count=3, skip=2)
        assert dak.dak_fault_pending(kind) == 3
        dak.dak_inject_fault(kind, count=-1)
        assert dak.dak_fault_pending(kind) == -1
        dak.dak_inject_fault(kind, count=0)
        assert dak.dak_fault_pending(kind) == 0
    assert dak.dak_fault_pending(0) == 0 and dak.dak_fault_pending(4) == 0


@pytest.mark.parametrize("kind,skip,count", [(0, 0, 1), (4, 0, 1), (1, -1, 1), (1, 0, -2)])
def test_switch_rejects_bad_arguments(dak, kind, skip, count):
    with pytest.raises(dak.DakError) as e:
        dak.dak_inject_fault(kind, count=count, skip=skip)
    assert e.value.status == 1


def test_environment_variable_sets_the_switch():
    code = ("import sys; sys.path.insert(0, %r); import direct_host_memory_gb300 as d; "
            "print(d.dak_fault_pending(1), d.dak_fault_pending(2), d.dak_fault_pending(3))" % ROOT)
    env = dict(os.environ, DAK_FAULT_INJECT="host_alloc=2:3,device_alloc=-1,tensor_map=1,bogus=4")
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, check=True)
    assert out.stdout.split() == ["3", "-1", "1"]


def test_counts_start_at_zero_and_failed_calls_hold_nothing(dak):
    import numpy as np
    h0, d0 = dak.dak_alloc_counts()
    assert h0 >= 0 and d0 >= 0
    A = np.zeros((64, 64), dtype=np.uint16)
    dak.dak_inject_fault(dak.FAULT_HOST_ALLOC, count=1)
    with pytest.raises(dak.DakError):
        dak.dak_place_matrix(A, 1)  # fails here (no device) or at the injected host allocation
    dak.dak_inject_fault(dak.FAULT_HOST_ALLOC, count=0)
    assert dak.dak_alloc_counts() == (h0, d0)
