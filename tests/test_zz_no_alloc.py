"""dak_attn_noalloc: decode attention for callers that cannot allocate device memory.

Such callers (an engine whose own pools already hold the device's memory, code without
access to the process's allocator, a loop where an allocation would synchronise the
device) get the split workspace from a fixed array inside the library. These checks call
the entry point through the C ABI twice in a row, with different inputs so that the
second call runs over the first call's leftovers in the shared array, and compare each
result with dak_attn given its own workspace. The file is named to be collected last.
"""
import numpy as np
import pytest

import synth
from gpu_util import REL_TOL, to_dev, to_np
from oracle import gemm as og

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dak(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    import direct_host_memory_gb300 as m
    return m


def test_noalloc_matches_dak_attn_on_two_calls(dak):
    import torch
    q1, k, v = synth.attn_inputs(8, 32, 8, 128, 1000, seed=21)
    q2 = synth.normal_bf16(22, 11, q1.size).reshape(q1.shape)
    p = dak.dak_place_kv(k, v, 3)
    lens = torch.tensor([1000, 999, 640, 1, 65, 1000, 300, 128], dtype=torch.int32, device="cuda")
    n_split = dak.dak_attn_default_split(p)
    assert n_split > 1  # the workspace is really used
    assert dak.dak_attn_workspace_bytes(8, 32, 128, n_split) <= dak.NOALLOC_SCRATCH_BYTES
    for q in (q1, q2):
        qt = to_dev(q)
        ref = dak.dak_attn(qt, p, seq_lens=lens)
        out = torch.empty_like(qt)
        dak.dak_attn_noalloc(qt, p, out, seq_lens=lens)
        st, info = dak.dak_last_error()
        assert st == 0, f"device status {st} info {info:#x}"
        # the same kernels with the same split and merge order: only the workspace differs
        assert torch.equal(out, ref)
        assert og.rel_err(to_np(out), to_np(ref)) <= REL_TOL
    p.free()


def test_noalloc_rejects_calls_beyond_its_array(dak):
    import torch
    _, k, v = synth.attn_inputs(64, 8, 8, 128, 64, seed=23)
    p = dak.dak_place_kv(k, v, 0)
    q = to_dev(synth.normal_bf16(24, 11, 64 * 128 * 128).reshape(64, 128, 128))
    out = torch.empty_like(q)
    # 64 requests x 128 heads x 64 splits x 130 floats is far above the array
    assert dak.dak_attn_workspace_bytes(64, 128, 128, 64) > dak.NOALLOC_SCRATCH_BYTES
    with pytest.raises(dak.DakError):
        dak.dak_attn_noalloc(q, p, out, tuning=dict(n_split=64))
    # the library's own check, called through the C ABI past the Python wrapper's
    import ctypes
    t = dak.dak_tuning(n_split=64)
    st = dak.lib.dak_attn_noalloc(ctypes.c_void_p(q.data_ptr()), p.handle, None, 128, ctypes.c_float(0.0),
                                  ctypes.c_void_p(out.data_ptr()), ctypes.byref(t),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 1  # DAK_ERR_INVALID
    assert dak.dak_last_error()[0] == 0  # nothing was launched
    p.free()
