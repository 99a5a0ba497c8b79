"""Host-side fault injection on the GPU: every injected failure of a pinned host allocation,
a device allocation or the tensor-map encode comes back as its typed status, frees whatever
the call had allocated (the library's live-allocation counts and the device's free memory
are unchanged after 100 failed calls), and leaves the library usable."""
import numpy as np
import pytest

import synth
from gpu_util import FP32_OUT_TOL, to_dev, to_np
from oracle import gemm as og

pytestmark = pytest.mark.gpu

HOST_ALLOC, DEVICE_ALLOC, CUDA = 3, 4, 5


@pytest.fixture(scope="module")
def dak(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    import direct_host_memory_gb300 as m
    yield m
    for k in (m.FAULT_HOST_ALLOC, m.FAULT_DEVICE_ALLOC, m.FAULT_TENSOR_MAP):
        m.dak_inject_fault(k, count=0)


def _expect(dak, status, fn):
    with pytest.raises(dak.DakError) as e:
        fn()
    assert e.value.status == status, (e.value.status, status)


def test_hundred_failed_placements_leak_nothing(dak):
    import torch
    A, _ = synth.gemm_inputs(640, 1024, 1, seed=31)
    Ad = to_dev(A)
    q, k, v = synth.attn_inputs(4, 8, 2, 128, 200, seed=32)
    torch.cuda.synchronize()
    counts0 = dak.dak_alloc_counts()
    free0, _ = torch.cuda.mem_get_info()
    cases = [
        # (kind, skip, call, status): host part; HBM part; packing buffer of a host source (the
        # second device allocation); KV host part; KV HBM part; KV packing buffer
        (dak.FAULT_HOST_ALLOC, 0, lambda: dak.dak_place_matrix(A, 3), HOST_ALLOC),
        (dak.FAULT_DEVICE_ALLOC, 0, lambda: dak.dak_place_matrix(A, 3), DEVICE_ALLOC),
        (dak.FAULT_DEVICE_ALLOC, 1, lambda: dak.dak_place_matrix(A, 3), DEVICE_ALLOC),
        (dak.FAULT_DEVICE_ALLOC, 0, lambda: dak.dak_place_matrix(Ad, 0), DEVICE_ALLOC),
        (dak.FAULT_HOST_ALLOC, 0, lambda: dak.dak_place_kv(k, v, 2), HOST_ALLOC),
        (dak.FAULT_DEVICE_ALLOC, 0, lambda: dak.dak_place_kv(k, v, 2), DEVICE_ALLOC),
        (dak.FAULT_DEVICE_ALLOC, 1, lambda: dak.dak_place_kv(k, v, 2), DEVICE_ALLOC),
        (dak.FAULT_HOST_ALLOC, 0, lambda: dak.dak_place_matrix_glu(A, 2), HOST_ALLOC),
    ]
    for i in range(100):
        kind, skip, call, status = cases[i % len(cases)]
        dak.dak_inject_fault(kind, count=1, skip=skip)
        _expect(dak, status, call)
        assert dak.dak_fault_pending(kind) == 0, i  # the failure was consumed by this call
        assert dak.dak_alloc_counts() == counts0, i
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 >= free0 - (4 << 20)
    # the library still works: the same placement succeeds and computes the right product
    p = dak.dak_place_matrix(A, 3)
    B = synth.normal_bf16(33, 2, 8 * 1024).reshape(8, 1024)
    C = dak.dak_gemm(p, to_dev(B), c_fp32=True)
    assert dak.dak_last_error()[0] == 0
    assert og.rel_err(to_np(C), og.gemm_ref(A, B)) <= FP32_OUT_TOL
    p.free()
    assert dak.dak_alloc_counts() == counts0


def test_tensor_map_failure_launches_nothing(dak):
    import torch
    A, B = synth.gemm_inputs(256, 512, 16, seed=34)
    p = dak.dak_place_matrix(A, 1)
    Bt = to_dev(B)
    C = torch.full((16, 256), 7.0, dtype=torch.float32, device="cuda")
    dak.dak_inject_fault(dak.FAULT_TENSOR_MAP, count=1)
    _expect(dak, CUDA, lambda: dak.dak_gemm(p, Bt, C, c_fp32=True))
    torch.cuda.synchronize()
    assert bool((C == 7.0).all())  # nothing ran
    assert dak.dak_fault_pending(dak.FAULT_TENSOR_MAP) == 0
    dak.dak_gemm(p, Bt, C, c_fp32=True)
    assert dak.dak_last_error()[0] == 0
    assert og.rel_err(to_np(C), og.gemm_ref(A, B)) <= FP32_OUT_TOL
    p.free()


def test_decoder_allocation_failures(dak):
    """A decoder's activations (dak_decoder_create) and its prefetch staging buffers (first
    prefetch-mode step) fail at each of their device allocations in turn."""
    import torch
    cfg = dict(n_layers=1, hidden=256, n_heads=4, n_kv_heads=2, head_dim=64, ffn=512, rms_eps=1e-5,
               rope_theta=10000.0)
    w = synth.decoder_layer(cfg, 0, 3)
    kv = synth.decoder_kv(cfg, 0, 3, 100, 3)
    L = dak.place_decoder_layer(w, kv, dict(qkv=1, o=1, gate_up=1, down=1, kv=1))
    fn = to_dev(synth.decoder_final_norm(cfg, 3))
    counts0 = dak.dak_alloc_counts()
    for skip in range(24):
        dak.dak_inject_fault(dak.FAULT_DEVICE_ALLOC, count=1, skip=skip)
        try:
            dec = dak.Decoder(cfg, [L], fn)
        except dak.DakError as e:
            assert e.status == DEVICE_ALLOC
            assert dak.dak_alloc_counts() == counts0, skip
            continue
        # every allocation of create succeeded: the injected one is still pending
        dak.dak_inject_fault(dak.FAULT_DEVICE_ALLOC, count=0)
        dec.free(placements=False)
        assert skip >= 10
        break
    else:
        pytest.fail("decoder create never completed")
    dec = dak.Decoder(cfg, [L], fn)
    x0 = to_dev(synth.decoder_x0(cfg, 3, 3))
    pos = torch.tensor([99, 0, 64], dtype=torch.int32, device="cuda")
    ref = dec.step(x0, pos)
    counts1 = dak.dak_alloc_counts()
    for skip in (0, 1):  # first or second staging buffer
        dak.dak_inject_fault(dak.FAULT_DEVICE_ALLOC, count=1, skip=skip)
        _expect(dak, DEVICE_ALLOC, lambda: dec.step(x0, pos, mode=dak.MODE_PREFETCH_SERIAL))
        assert dak.dak_alloc_counts() == counts1
    out = dec.step(x0, pos, mode=dak.MODE_PREFETCH_SERIAL)  # staging allocated now, all of it
    assert dak.dak_last_error()[0] == 0
    assert torch.equal(out, ref)
    dec.free()


def test_probe_host_buffer_failure(dak):
    dak.dak_inject_fault(dak.FAULT_HOST_ALLOC, count=1)
    counts0 = dak.dak_alloc_counts()
    _expect(dak, HOST_ALLOC, lambda: dak.dak_probe_read_bw(0, 1 << 20, 0, 4, 2, 32768, 1))
    assert dak.dak_alloc_counts() == counts0
