"""The launch tuner's persisted tables (host side) and, on the GPU, the tuner itself."""
import json
import os

import numpy as np
import pytest

import synth
from oracle import gemm as og


def test_tuning_table_round_trip(tmp_path):
    import direct_host_memory_gb300 as dak
    table = {"qkv": {"host_ctas": 8, "window": 3}, "attn": {"host_ctas": 12, "window": 4, "n_split": 4}}
    p = os.path.join(tmp_path, "t.json")
    dak.save_tuning(p, table, meta={"gpu": "test"})
    assert dak.load_tuning(p) == table
    with open(p) as f:
        doc = json.load(f)
    doc["tuning"]["qkv"]["bogus"] = 1
    with open(p, "w") as f:
        json.dump(doc, f)
    with pytest.raises(ValueError):
        dak.load_tuning(p)


def test_tuning_struct_fields_match_header():
    """dak_tuning's fields, in order, as include/dak.h declares them."""
    import re
    import direct_host_memory_gb300 as dak
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "dak.h")).read()
    body = re.search(r"typedef struct \{([^}]*)\} dak_tuning;", hdr).group(1)
    fields = re.findall(r"int (\w+);", body)
    assert fields == dak.TUNING_FIELDS


@pytest.fixture(scope="module")
def dakg(cuda_ok):
    import __graft_entry__
    __graft_entry__.build()
    import direct_host_memory_gb300 as m
    return m


def _dev(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()


@pytest.mark.gpu
def test_tune_gemm_choices_keep_results(dakg):
    dak = dakg
    import torch
    M, K, N = 2048, 4096, 16
    A, B = synth.gemm_inputs(M, K, N, seed=41)
    p = dak.dak_place_matrix(A, 9)
    Bt = _dev(B)
    C = torch.empty((N, M), dtype=torch.float32, device="cuda")
    r = dak.dak_tune_gemm(p, Bt, C, c_fp32=True, reps=3)
    assert dak.dak_last_error()[0] == 0
    assert r["candidates"] > 0 and 0 < r["best_us"] <= r["default_us"]
    assert r["cc_off_us"] > 0 and r["no_align_us"] > 0
    base = dak.dak_gemm(p, Bt, c_fp32=True)
    moves_only = [dict(host_ctas=32, window=8), dict(no_wave_align=1), dict(host_ctas=1 << 20, window=8),
                  {k: v for k, v in r["best"].items() if k not in ("chunk_k", "split_k")}]
    for t in moves_only:
        assert torch.equal(dak.dak_gemm(p, Bt, c_fp32=True, tuning=t), base), t
    best = dak.dak_gemm(p, Bt, c_fp32=True, tuning=r["best"])
    assert og.rel_err(best.double().cpu().numpy(), og.gemm_ref(A, B)) <= 1e-5
    assert dak.dak_last_error()[0] == 0
    p.free()


@pytest.mark.gpu
def test_tune_attn_choices_keep_results(dakg):
    dak = dakg
    import torch
    q, k, v = synth.attn_inputs(8, 32, 8, 128, 1000, seed=42)
    kv = dak.dak_place_kv(k, v, 3)
    Q = _dev(q)
    O = torch.empty_like(Q)
    r = dak.dak_tune_attn(Q, kv, O, reps=3)
    assert dak.dak_last_error()[0] == 0
    assert r["candidates"] > 0 and 0 < r["best_us"] <= r["default_us"]
    base = dak.dak_attn(Q, kv)
    for t in (r["best"], dict(no_wave_align=1), dict(host_ctas=1 << 20, window=8)):
        assert torch.equal(dak.dak_attn(Q, kv, tuning=t), base), t
    assert dak.dak_last_error()[0] == 0
    kv.free()
