"""ctypes binding of libdak.so: argument marshalling only, every step runs in the library.

Names match the C ABI in include/dak.h. Tensors are torch tensors (device memory and
streams come from PyTorch); host-side sources may also be numpy arrays of bf16 bits.
A missing library raises at import time: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdak.so")

DAK_OK = 0
STATUS_NAMES = {
    0: "DAK_OK", 1: "DAK_ERR_INVALID", 2: "DAK_ERR_ALIGN", 3: "DAK_ERR_HOST_ALLOC",
    4: "DAK_ERR_DEVICE_ALLOC", 5: "DAK_ERR_CUDA", 6: "DAK_ERR_TIMEOUT", 7: "DAK_ERR_UNSUPPORTED",
    8: "DAK_ERR_BOUNDS",
}

# every symbol include/dak.h declares
EXPORTS = [
    "dak_status_string", "dak_place_matrix", "dak_place_kv", "dak_free", "dak_placement_info",
    "dak_gemm", "dak_attn_workspace_bytes", "dak_attn", "dak_attn_default_split", "dak_plan_ratios",
    "dak_last_error", "dak_sm_count", "dak_probe_read_bw", "dak_probe_concurrent", "dak_prefetch",
    "dak_gemm_staged", "dak_attn_staged", "dak_attn_noalloc", "dak_selftest_wait",
    "dak_decoder_create", "dak_decoder_batch", "dak_decoder_step", "dak_decoder_capture",
    "dak_decoder_replay", "dak_decoder_launches", "dak_decoder_free", "dak_tune_gemm", "dak_tune_attn",
    "dak_place_matrix_glu", "dak_plan_units", "dak_gemm_workspace_bytes", "dak_gemm_ws", "dak_gemm_plan", "dak_gemm_launch_plan",
    "dak_attn_f32", "dak_inject_fault", "dak_fault_pending", "dak_alloc_counts", "dak_gemm_chain",
    "dak_gemm_chain_workspace_bytes", "dak_link_begin", "dak_link_timeouts", "dak_selftest_link",
    "dak_place_kv_heads", "dak_kv_append", "dak_gemm_chain_plan",
]

# host-side fault injection kinds (DAK_FAULT_* in dak.h)
FAULT_HOST_ALLOC, FAULT_DEVICE_ALLOC, FAULT_TENSOR_MAP = 1, 2, 3

# size of the fixed device array dak_attn_noalloc uses (DAK_NOALLOC_SCRATCH_BYTES in dak.h)
NOALLOC_SCRATCH_BYTES = 4 << 20


class DakError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}")


class dak_tuning(ctypes.Structure):
    _fields_ = [("host_ctas", ctypes.c_int), ("window", ctypes.c_int), ("hbm_window", ctypes.c_int),
                ("chunk_k", ctypes.c_int), ("n_split", ctypes.c_int), ("hbm_ctas", ctypes.c_int),
                ("split_k", ctypes.c_int), ("pdl", ctypes.c_int), ("ctas_per_sm", ctypes.c_int),
                ("no_wave_align", ctypes.c_int), ("column_blocks", ctypes.c_int), ("cluster_slots", ctypes.c_int),
                ("link", ctypes.c_int), ("chain_rr", ctypes.c_int)]


class dak_gemm_op(ctypes.Structure):
    _fields_ = [("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("C", ctypes.c_void_p), ("c_fp32", ctypes.c_int),
                ("after_prev", ctypes.c_int)]


class dak_op(ctypes.Structure):
    _fields_ = [("bytes", ctypes.c_double), ("t_comp", ctypes.c_double), ("tile_bytes", ctypes.c_double)]


class dak_tune_result(ctypes.Structure):
    _fields_ = [("best", dak_tuning), ("best_us", ctypes.c_double), ("default_us", ctypes.c_double),
                ("cc_off_us", ctypes.c_double), ("no_align_us", ctypes.c_double), ("candidates", ctypes.c_int)]


class dak_gemm_chain_plan_info(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int) for f in ("grid", "units", "by_size", "busiest_per_op", "busiest_by_size")]


class dak_gemm_plan_info(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int) for f in (
        "tensor_cores", "launches", "cluster", "n_pad", "pieces", "piece_step", "chunk_k", "host_chunk_k",
        "hbm_stages", "host_stages", "host_ctas", "hbm_ctas", "host_window", "hbm_window", "smem_bytes",
        "tile_m", "cluster_slots")]


class dak_decoder_config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float), ("plain_launch", ctypes.c_int),
                ("op_tuning", dak_tuning * 5), ("no_link_handoff", ctypes.c_int)]


class dak_decoder_layer(ctypes.Structure):
    _fields_ = [("qkv", ctypes.c_void_p), ("o", ctypes.c_void_p), ("gate_up", ctypes.c_void_p),
                ("down", ctypes.c_void_p), ("kv", ctypes.c_void_p), ("attn_norm", ctypes.c_void_p),
                ("mlp_norm", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built (run __graft_entry__.build()); "
                          "the direct-access path has no fallback")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, i64, dbl, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_size_t
    P = ctypes.POINTER
    sig = {
        "dak_status_string": (ctypes.c_char_p, [i32]),
        "dak_place_matrix": (i32, [vp, i32, i64, i64, i64, i32, i32, P(vp)]),
        "dak_place_kv": (i32, [vp, vp, i32, i32, i32, i32, i32, i32, P(vp)]),
        "dak_place_kv_heads": (i32, [vp, vp, i32, i32, i32, i32, i32, i32, P(vp)]),
        "dak_kv_append": (i32, [vp, vp, vp, vp, vp]),
        "dak_place_matrix_glu": (i32, [vp, i32, i64, i64, i64, i32, i32, P(vp)]),
        "dak_free": (i32, [vp]),
        "dak_placement_info": (i32, [vp, P(i64), P(i64), P(i64), P(i64)]),
        "dak_gemm": (i32, [vp, vp, vp, i32, i32, P(dak_tuning), vp]),
        "dak_gemm_staged": (i32, [vp, vp, vp, vp, i32, i32, P(dak_tuning), vp]),
        "dak_gemm_workspace_bytes": (sz, [vp, i32]),
        "dak_gemm_ws": (i32, [vp, vp, vp, i32, i32, P(dak_tuning), vp, sz, vp]),
        "dak_gemm_plan": (i32, [i64, i64, i32, i32, i32, i32, P(dak_tuning), sz, P(dak_gemm_plan_info)]),
        "dak_gemm_launch_plan": (i32, [vp, i32, P(dak_tuning), sz, P(dak_gemm_plan_info)]),
        "dak_gemm_chain_workspace_bytes": (sz, [P(dak_gemm_op), i32, i32, P(dak_tuning)]),
        "dak_gemm_chain": (i32, [P(dak_gemm_op), i32, i32, P(dak_tuning), vp, sz, vp]),
        "dak_gemm_chain_plan": (i32, [P(i64), P(i64), P(i32), P(i32), P(i32), i32, i32, i32, P(dak_tuning),
                                      P(dak_gemm_chain_plan_info)]),
        "dak_attn_workspace_bytes": (sz, [i32, i32, i32, i32]),
        "dak_attn": (i32, [vp, vp, vp, i32, ctypes.c_float, vp, vp, sz, P(dak_tuning), vp]),
        "dak_attn_staged": (i32, [vp, vp, vp, vp, i32, ctypes.c_float, vp, vp, sz, P(dak_tuning), vp]),
        "dak_attn_f32": (i32, [vp, vp, vp, i32, ctypes.c_float, vp, vp, sz, P(dak_tuning), vp]),
        "dak_attn_default_split": (i32, [vp]),
        "dak_plan_ratios": (i32, [P(dak_op), i32, dbl, dbl, dbl, i32, P(dbl), P(dbl)]),
        "dak_plan_units": (i32, [P(dak_op), i32, dbl, dbl, dbl, P(i64), P(dbl)]),
        "dak_last_error": (i32, [vp, P(ctypes.c_uint64)]),
        "dak_sm_count": (i32, []),
        "dak_probe_read_bw": (i32, [i32, i64, i32, i32, i32, i32, i32, P(dbl), P(i32)]),
        "dak_probe_concurrent": (i32, [i64, i64, i32, i32, i32, i32, i32, i32, P(dbl), P(dbl)]),
        "dak_prefetch": (i32, [vp, vp, vp]),
        "dak_link_begin": (i32, [i32, vp]),
        "dak_link_timeouts": (i32, [vp, P(ctypes.c_uint32)]),
        "dak_selftest_link": (i32, [vp]),
        "dak_attn_noalloc": (i32, [vp, vp, vp, i32, ctypes.c_float, vp, P(dak_tuning), vp]),
        "dak_selftest_wait": (i32, [vp]),
        "dak_inject_fault": (i32, [i32, i32, i32]),
        "dak_fault_pending": (i32, [i32]),
        "dak_alloc_counts": (i32, [P(i64), P(i64)]),
        "dak_decoder_create": (i32, [P(dak_decoder_config), P(dak_decoder_layer), vp, P(vp)]),
        "dak_decoder_batch": (i32, [vp]),
        "dak_decoder_step": (i32, [vp, vp, vp, vp, i32, vp]),
        "dak_decoder_capture": (i32, [vp, vp, vp, vp, i32]),
        "dak_decoder_replay": (i32, [vp, vp]),
        "dak_decoder_launches": (i32, [vp, i32]),
        "dak_decoder_free": (i32, [vp]),
        "dak_tune_gemm": (i32, [vp, vp, vp, i32, i32, i32, P(dak_tuning), P(dak_tune_result)]),
        "dak_tune_attn": (i32, [vp, vp, vp, i32, vp, vp, sz, i32, P(dak_tuning), P(dak_tune_result)]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = _load()


def _check(status: int, where: str):
    if status != DAK_OK:
        raise DakError(status, where)


def _stream_ptr(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _tuning(t):
    if t is None:
        return None
    if isinstance(t, dak_tuning):
        return ctypes.byref(t)
    tt = dak_tuning(**{k: int(v) for k, v in dict(t).items()})
    return ctypes.byref(tt)


def _ptr(x):
    """Data pointer of a torch tensor or numpy array."""
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        if not x.flags["C_CONTIGUOUS"]:
            raise ValueError("numpy source must be C-contiguous")
        return ctypes.c_void_p(x.ctypes.data)
    return ctypes.c_void_p(x.data_ptr())


def _on_device(x) -> int:
    return 0 if isinstance(x, np.ndarray) else int(x.is_cuda)


class Placement:
    """A library-owned placement (dak_placement*). Free with .free() or by dropping it."""

    def __init__(self, handle: ctypes.c_void_p, kind: str, **meta):
        self._h = handle
        self.kind = kind
        self.meta = meta
        hb, gb, u, hu = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(lib.dak_placement_info(handle, ctypes.byref(hb), ctypes.byref(gb), ctypes.byref(u),
                                      ctypes.byref(hu)), "dak_placement_info")
        self.host_bytes, self.hbm_bytes = hb.value, gb.value
        self.units, self.host_units = u.value, hu.value

    @property
    def handle(self):
        if self._h is None:
            raise ValueError("placement already freed")
        return self._h

    def free(self):
        if self._h is not None:
            lib.dak_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


# ------------------------------------------------------------------------------- placement

def host_tiles_for_ratio(x: float, M: int, tile_m: int = 64) -> int:
    """Tile rows to place on the host for offload ratio x: ceil(x * T), T = ceil(M / tile_m),
    so that at least the fraction x of the rows leaves HBM."""
    import math
    T = -(-int(M) // int(tile_m))
    return max(0, min(T, math.ceil(float(x) * T - 1e-12)))


def host_requests_for_ratio(x: float, batch: int) -> int:
    """Requests whose KV goes to the host for offload ratio x: ceil(x * B)."""
    import math
    return max(0, min(int(batch), math.ceil(float(x) * int(batch) - 1e-12)))


def host_heads_for_ratio(x: float, batch: int, h_kv: int) -> int:
    """(request, kv head) slabs whose KV goes to the host for offload ratio x: ceil(x * B * H_kv)."""
    return host_requests_for_ratio(x, int(batch) * int(h_kv))


def dak_place_matrix(A, n_host_tiles: int, tile_m: int = 64) -> Placement:
    """Place weights A [M][K] (bf16: torch tensor on host or device, or numpy uint16 bits)."""
    if A.ndim != 2:
        raise ValueError("A must be 2-D [M][K]")
    M, K = int(A.shape[0]), int(A.shape[1])
    out = ctypes.c_void_p()
    _check(lib.dak_place_matrix(_ptr(A), _on_device(A), M, K, K, tile_m, int(n_host_tiles),
                                ctypes.byref(out)), "dak_place_matrix")
    return Placement(out, "matrix", M=M, K=K, tile_m=tile_m)


def dak_place_matrix_glu(A, n_host_tiles: int, tile_m: int = 64) -> Placement:
    """Place a SwiGLU weight A [2f][K] (f gate rows, then f up rows) interleaved, so that
    dak_gemm over it returns silu(gate) * up [N][f]."""
    if A.ndim != 2 or int(A.shape[0]) % 2:
        raise ValueError("A must be 2-D [2f][K]")
    M, K = int(A.shape[0]), int(A.shape[1])
    out = ctypes.c_void_p()
    _check(lib.dak_place_matrix_glu(_ptr(A), _on_device(A), M // 2, K, K, tile_m, int(n_host_tiles),
                                    ctypes.byref(out)), "dak_place_matrix_glu")
    return Placement(out, "matrix", M=M, K=K, tile_m=tile_m, glu=True)


def dak_place_kv(K, V, n_host_requests: int) -> Placement:
    """Place a KV cache, K and V [B][H_kv][L][D] bf16 (torch or numpy uint16 bits)."""
    if K.shape != V.shape or K.ndim != 4:
        raise ValueError("K and V must both be [B][H_kv][L][D]")
    B, Hkv, L, D = (int(s) for s in K.shape)
    out = ctypes.c_void_p()
    _check(lib.dak_place_kv(_ptr(K), _ptr(V), _on_device(K), B, Hkv, L, D, int(n_host_requests),
                            ctypes.byref(out)), "dak_place_kv")
    return Placement(out, "kv", B=B, H_kv=Hkv, L=L, D=D)


def dak_place_kv_heads(K, V, n_host_heads: int) -> Placement:
    """dak_place_kv by (request, kv head) slab: the first n_host_heads slabs in request-major
    order (request b, head g is slab b * H_kv + g) go to the host."""
    if K.shape != V.shape or K.ndim != 4:
        raise ValueError("K and V must both be [B][H_kv][L][D]")
    B, Hkv, L, D = (int(s) for s in K.shape)
    out = ctypes.c_void_p()
    _check(lib.dak_place_kv_heads(_ptr(K), _ptr(V), _on_device(K), B, Hkv, L, D, int(n_host_heads),
                                  ctypes.byref(out)), "dak_place_kv_heads")
    return Placement(out, "kv", B=B, H_kv=Hkv, L=L, D=D)


def dak_kv_append(KV: Placement, k_new, v_new, positions, stream=None):
    """Write one new token per (request, kv head) into a placed cache: k_new and v_new bf16
    CUDA [B][H_kv][D], positions int32 CUDA [B] (the row each request's token goes to)."""
    import torch
    _check_bf16_cuda(k_new, "k_new")
    _check_bf16_cuda(v_new, "v_new")
    shape = (KV.meta["B"], KV.meta["H_kv"], KV.meta["D"])
    if tuple(k_new.shape) != shape or tuple(v_new.shape) != shape:
        raise ValueError(f"k_new / v_new must be {list(shape)}")
    if positions.dtype != torch.int32 or not positions.is_cuda or positions.numel() != shape[0]:
        raise ValueError("positions must be int32 CUDA [B]")
    _check(lib.dak_kv_append(KV.handle, _ptr(k_new), _ptr(v_new), _ptr(positions), _stream_ptr(stream)),
           "dak_kv_append")


def dak_free(p: Placement):
    p.free()


def dak_placement_info(p: Placement):
    return dict(host_bytes=p.host_bytes, hbm_bytes=p.hbm_bytes, units=p.units, host_units=p.host_units)


# ------------------------------------------------------------------------------- hot path

def _check_bf16_cuda(t, name):
    import torch
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")


def dak_gemm(A: Placement, B, C=None, c_fp32: bool = False, tuning=None, stream=None, workspace=None):
    """C [N][M] = B [N][K] . A^T over the tiered placement A (returns C). workspace: an optional
    split workspace of the caller's (a zeroed device tensor of dak_gemm_workspace_bytes(A, N)
    bytes or more), for launches that may overlap others on different streams."""
    import torch
    _check_bf16_cuda(B, "B")
    N = int(B.shape[0])
    if B.ndim != 2 or int(B.shape[1]) != A.meta["K"]:
        raise ValueError("B must be [N][K]")
    if C is None:
        cols = A.meta["M"] // 2 if A.meta.get("glu") else A.meta["M"]
        C = torch.empty((N, cols), dtype=torch.float32 if c_fp32 else torch.bfloat16, device=B.device)
    if workspace is None:
        _check(lib.dak_gemm(A.handle, _ptr(B), _ptr(C), N, int(bool(c_fp32)), _tuning(tuning), _stream_ptr(stream)),
               "dak_gemm")
    else:
        nbytes = workspace.numel() * workspace.element_size()
        _check(lib.dak_gemm_ws(A.handle, _ptr(B), _ptr(C), N, int(bool(c_fp32)), _tuning(tuning), _ptr(workspace),
                               ctypes.c_size_t(nbytes), _stream_ptr(stream)), "dak_gemm_ws")
    return C


def _chain_ops(ops):
    arr = (dak_gemm_op * len(ops))()
    for j, o in enumerate(ops):
        arr[j].A = o["A"].handle
        arr[j].B = o["B"].data_ptr() if o.get("B") is not None else None
        arr[j].C = o["C"].data_ptr() if o.get("C") is not None else None
        arr[j].c_fp32 = int(bool(o.get("c_fp32", False)))
        arr[j].after_prev = int(bool(o.get("after_prev", False)))
    return arr


def dak_gemm_chain_workspace_bytes(ops, N: int, tuning=None) -> int:
    """Bytes of the workspace dak_gemm_chain needs (ops: dicts with at least 'A')."""
    return int(lib.dak_gemm_chain_workspace_bytes(_chain_ops(ops), len(ops), int(N), _tuning(tuning)))


def dak_gemm_chain(ops, tuning=None, workspace=None, stream=None):
    """Several GEMMs in one persistent launch. ops: list of dicts with 'A' (Placement), 'B'
    (bf16 [N][K] CUDA tensor), optional 'C', 'c_fp32' and 'after_prev' (B comes from an
    earlier operation of the chain). workspace: a zeroed CUDA tensor of
    dak_gemm_chain_workspace_bytes bytes (allocated and zeroed here when None). Returns the
    list of C tensors."""
    import torch
    if not ops:
        raise ValueError("empty chain")
    N = int(ops[0]["B"].shape[0])
    ops = [dict(o) for o in ops]
    for o in ops:
        _check_bf16_cuda(o["B"], "B")
        if int(o["B"].shape[0]) != N or int(o["B"].shape[1]) != o["A"].meta["K"]:
            raise ValueError("every B must be [N][K] with the same N")
        if o.get("C") is None:
            cols = o["A"].meta["M"] // 2 if o["A"].meta.get("glu") else o["A"].meta["M"]
            o["C"] = torch.empty((N, cols), dtype=torch.float32 if o.get("c_fp32") else torch.bfloat16,
                                 device=o["B"].device)
    if workspace is None:
        nbytes = dak_gemm_chain_workspace_bytes(ops, N, tuning) if len(ops) <= 8 else 0
        if nbytes == 0:  # a chain the library rejects: let it say why
            _check(lib.dak_gemm_chain(_chain_ops(ops), len(ops), N, _tuning(tuning), None, 0, _stream_ptr(stream)),
                   "dak_gemm_chain")
        workspace = torch.zeros(nbytes, dtype=torch.uint8, device=ops[0]["B"].device)
    _check(lib.dak_gemm_chain(_chain_ops(ops), len(ops), N, _tuning(tuning), _ptr(workspace),
                              ctypes.c_size_t(workspace.numel() * workspace.element_size()), _stream_ptr(stream)),
           "dak_gemm_chain")
    return [o["C"] for o in ops]


def dak_gemm_chain_plan(shapes, N: int, n_host_tiles=None, tile_m=None, after_prev=None, sm_count: int = None,
                        tuning=None) -> dict:
    """How dak_gemm_chain would deal a chain's units over its CTAs, from host arithmetic alone:
    shapes [(M, K), ...], per operation n_host_tiles, tile_m (64 or 128) and after_prev;
    sm_count None = this process's GPU."""
    n = len(shapes)
    if sm_count is None:
        sm_count = dak_sm_count()

    def arr(t, vals):
        return (t * n)(*[int(v) for v in vals])
    out = dak_gemm_chain_plan_info()
    _check(lib.dak_gemm_chain_plan(arr(ctypes.c_int64, [m for m, _ in shapes]), arr(ctypes.c_int64, [k for _, k in shapes]),
                                   arr(ctypes.c_int, tile_m or [64] * n), arr(ctypes.c_int, n_host_tiles or [0] * n),
                                   arr(ctypes.c_int, after_prev or [0] * n), n, int(N), int(sm_count), _tuning(tuning),
                                   ctypes.byref(out)), "dak_gemm_chain_plan")
    return {f: int(getattr(out, f)) for f, _ in dak_gemm_chain_plan_info._fields_}


def dak_gemm_workspace_bytes(A: Placement, N: int) -> int:
    """Bytes of a caller's split workspace for dak_gemm over A with N hidden-state rows."""
    return int(lib.dak_gemm_workspace_bytes(A.handle, int(N)))


def dak_gemm_plan(M: int, K: int, n_host_tiles: int, N: int, sm_count: int = None, tuning=None,
                  ws_bytes: int = 0, tile_m: int = 64) -> dict:
    """The launch dak_gemm would make for an M x K matrix placed in tiles of tile_m rows with
    n_host_tiles of them on the host and N hidden-state rows (pieces, rings, CTAs of each
    role), from host arithmetic alone; sm_count None = this process's GPU."""
    if sm_count is None:
        sm_count = dak_sm_count()
    out = dak_gemm_plan_info()
    _check(lib.dak_gemm_plan(int(M), int(K), int(tile_m), int(n_host_tiles), int(N), int(sm_count), _tuning(tuning),
                             ctypes.c_size_t(int(ws_bytes)), ctypes.byref(out)), "dak_gemm_plan")
    return {f: int(getattr(out, f)) for f, _ in dak_gemm_plan_info._fields_}


def dak_gemm_launch_plan(A: Placement, N: int, tuning=None, ws_bytes: int = 0) -> dict:
    """The plan dak_gemm would use for placement A and N rows on this process's GPU."""
    out = dak_gemm_plan_info()
    _check(lib.dak_gemm_launch_plan(A.handle, int(N), _tuning(tuning), ctypes.c_size_t(int(ws_bytes)),
                                    ctypes.byref(out)), "dak_gemm_launch_plan")
    return {f: int(getattr(out, f)) for f, _ in dak_gemm_plan_info._fields_}


def dak_gemm_staged(A: Placement, staging, B, C=None, c_fp32: bool = False, tuning=None, stream=None):
    import torch
    _check_bf16_cuda(B, "B")
    N = int(B.shape[0])
    if C is None:
        C = torch.empty((N, A.meta["M"]), dtype=torch.float32 if c_fp32 else torch.bfloat16, device=B.device)
    _check(lib.dak_gemm_staged(A.handle, _ptr(staging), _ptr(B), _ptr(C), N, int(bool(c_fp32)), _tuning(tuning),
                               _stream_ptr(stream)), "dak_gemm_staged")
    return C


def dak_attn_workspace_bytes(B: int, H_q: int, D: int, n_split: int) -> int:
    return int(lib.dak_attn_workspace_bytes(B, H_q, D, n_split))


def dak_attn_default_split(KV: Placement) -> int:
    return int(lib.dak_attn_default_split(KV.handle))


def _attn_common(Q, KV, O, workspace, tuning):
    import torch
    _check_bf16_cuda(Q, "Q")
    B, Hq, D = (int(s) for s in Q.shape)
    if B != KV.meta["B"] or D != KV.meta["D"]:
        raise ValueError("Q does not match the KV placement")
    n_split = int(dict(tuning or {}).get("n_split", 0) or 0) if not isinstance(tuning, dak_tuning) else tuning.n_split
    if n_split <= 0:
        n_split = dak_attn_default_split(KV)
    ws_bytes = dak_attn_workspace_bytes(B, Hq, D, n_split)
    if workspace is None and ws_bytes:
        workspace = torch.empty(ws_bytes // 4, dtype=torch.float32, device=Q.device)
    if O is None:
        O = torch.empty_like(Q)
    tun = dict(tuning or {}) if not isinstance(tuning, dak_tuning) else tuning
    if not isinstance(tun, dak_tuning):
        tun["n_split"] = n_split
    ws_len = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return Hq, O, workspace, ws_len, tun


def dak_attn(Q, KV: Placement, seq_lens=None, scale: float = 0.0, O=None, workspace=None, tuning=None, stream=None):
    """Decode attention o [B][Hq][D] over the request-partitioned KV placement (returns O)."""
    Hq, O, workspace, ws_len, tun = _attn_common(Q, KV, O, workspace, tuning)
    _check(lib.dak_attn(_ptr(Q), KV.handle, _ptr(seq_lens), Hq, float(scale), _ptr(O), _ptr(workspace), ws_len,
                        _tuning(tun), _stream_ptr(stream)), "dak_attn")
    return O


def dak_attn_f32(Q, KV: Placement, seq_lens=None, scale: float = 0.0, O=None, workspace=None, tuning=None,
                 stream=None):
    """dak_attn with an fp32 output o [B][Hq][D] (the parity mode; returns O)."""
    import torch
    if O is None:
        O = torch.empty(tuple(Q.shape), dtype=torch.float32, device=Q.device)
    if not (O.dtype == torch.float32 and O.is_cuda and O.is_contiguous() and tuple(O.shape) == tuple(Q.shape)):
        raise ValueError("O must be a contiguous fp32 CUDA tensor shaped like Q")
    Hq, O, workspace, ws_len, tun = _attn_common(Q, KV, O, workspace, tuning)
    _check(lib.dak_attn_f32(_ptr(Q), KV.handle, _ptr(seq_lens), Hq, float(scale), _ptr(O), _ptr(workspace), ws_len,
                            _tuning(tun), _stream_ptr(stream)), "dak_attn_f32")
    return O


def dak_attn_staged(Q, KV: Placement, staging, seq_lens=None, scale: float = 0.0, O=None, workspace=None,
                    tuning=None, stream=None):
    Hq, O, workspace, ws_len, tun = _attn_common(Q, KV, O, workspace, tuning)
    _check(lib.dak_attn_staged(_ptr(Q), KV.handle, _ptr(staging), _ptr(seq_lens), Hq, float(scale), _ptr(O),
                               _ptr(workspace), ws_len, _tuning(tun), _stream_ptr(stream)), "dak_attn_staged")
    return O


def dak_attn_noalloc(Q, KV: Placement, O, seq_lens=None, scale: float = 0.0, tuning=None, stream=None):
    """dak_attn without a workspace argument, for callers that cannot allocate device memory
    (an engine whose pools already hold the device's memory, code without access to the
    process's allocator, a loop where an allocation would synchronise the device). The
    library takes the split workspace from its fixed NOALLOC_SCRATCH_BYTES device array,
    shared by all calls: calls that overlap on the GPU race on it. O must be preallocated."""
    _check_bf16_cuda(Q, "Q")
    _check_bf16_cuda(O, "O")
    B, Hq, D = (int(s) for s in Q.shape)
    if B != KV.meta["B"] or D != KV.meta["D"] or tuple(O.shape) != tuple(Q.shape):
        raise ValueError("Q / O do not match the KV placement")
    tun = tuning if isinstance(tuning, dak_tuning) else dict(tuning or {})
    n_split = tun.n_split if isinstance(tun, dak_tuning) else int(tun.get("n_split", 0) or 0)
    if n_split <= 0:
        n_split = dak_attn_default_split(KV)
    need = dak_attn_workspace_bytes(B, Hq, D, n_split)
    if need > NOALLOC_SCRATCH_BYTES:
        raise DakError(1, f"dak_attn_noalloc: needs {need} bytes of workspace, more than the fixed "
                          f"{NOALLOC_SCRATCH_BYTES}-byte array; use dak_attn with a workspace")
    _check(lib.dak_attn_noalloc(_ptr(Q), KV.handle, _ptr(seq_lens), Hq, float(scale), _ptr(O), _tuning(tuning),
                                _stream_ptr(stream)), "dak_attn_noalloc")
    return O


def dak_link_begin(slot: int, stream=None):
    """Start host-link handoff sequence `slot` (1..8) on `stream`: later dak_gemm / dak_attn
    calls with tuning link=slot stream their host tiles / requests only once the sequence's
    earlier launches have issued all of their host loads (paces the loads; results are
    unchanged)."""
    _check(lib.dak_link_begin(int(slot), _stream_ptr(stream)), "dak_link_begin")


def dak_link_timeouts(stream=None) -> int:
    """Handoff waits that gave up at their bound since the last call (0 when every launch of
    every sequence found its predecessors in time); the count restarts at zero."""
    c = ctypes.c_uint32()
    _check(lib.dak_link_timeouts(_stream_ptr(stream), ctypes.byref(c)), "dak_link_timeouts")
    return int(c.value)


def dak_selftest_link(stream=None):
    """One pacing wait that must give up (see dak_link_timeouts)."""
    _check(lib.dak_selftest_link(_stream_ptr(stream)), "dak_selftest_link")


def dak_prefetch(p: Placement, staging, stream=None):
    _check(lib.dak_prefetch(p.handle, _ptr(staging), _stream_ptr(stream)), "dak_prefetch")


# ------------------------------------------------------------------------------- planner

def dak_plan_ratios(ops, b_host: float, b_hbm: float, min_offload_bytes: float, mode: int = 0):
    """ops: iterable of (bytes, t_comp[, tile_bytes]). Returns (ratios ndarray, model time s)."""
    ops = list(ops)
    arr = (dak_op * max(1, len(ops)))()
    for i, o in enumerate(ops):
        arr[i].bytes = float(o[0])
        arr[i].t_comp = float(o[1])
        arr[i].tile_bytes = float(o[2]) if len(o) > 2 else 0.0
    ratios = (ctypes.c_double * max(1, len(ops)))()
    t = ctypes.c_double()
    _check(lib.dak_plan_ratios(arr, len(ops), float(b_host), float(b_hbm), float(min_offload_bytes), int(mode),
                               ratios, ctypes.byref(t)), "dak_plan_ratios")
    return np.array(ratios[:len(ops)], dtype=np.float64), t.value


def dak_plan_units(ops, b_host: float, b_hbm: float, min_offload_bytes: float):
    """ops: iterable of (bytes, t_comp, unit_bytes). Returns (host units ndarray int64, model time s)."""
    ops = list(ops)
    arr = (dak_op * max(1, len(ops)))()
    for i, o in enumerate(ops):
        arr[i].bytes, arr[i].t_comp, arr[i].tile_bytes = float(o[0]), float(o[1]), float(o[2])
    out = (ctypes.c_int64 * max(1, len(ops)))()
    t = ctypes.c_double()
    _check(lib.dak_plan_units(arr, len(ops), float(b_host), float(b_hbm), float(min_offload_bytes), out,
                              ctypes.byref(t)), "dak_plan_units")
    return np.array(out[:len(ops)], dtype=np.int64), t.value


# ------------------------------------------------------------------------------- errors / probes

def dak_last_error(stream=None):
    """Synchronise and return (status, info) of the device status word (cleared)."""
    info = ctypes.c_uint64()
    st = lib.dak_last_error(_stream_ptr(stream), ctypes.byref(info))
    return int(st), int(info.value)


def dak_selftest_wait(stream=None):
    """Launch the bounded-wait self-test kernel (its wait must time out after ~2 s)."""
    _check(lib.dak_selftest_wait(_stream_ptr(stream)), "dak_selftest_wait")


def dak_inject_fault(kind: int, count: int = 1, skip: int = 0):
    """Make the library's next `count` calls of this kind (FAULT_*) fail after `skip` more
    succeed (count -1: every call; count 0 clears). Host side only."""
    _check(lib.dak_inject_fault(int(kind), int(skip), int(count)), "dak_inject_fault")


def dak_fault_pending(kind: int) -> int:
    return int(lib.dak_fault_pending(int(kind)))


def dak_alloc_counts():
    """(pinned host buffers, device buffers) the library holds right now."""
    h, d = ctypes.c_int64(), ctypes.c_int64()
    _check(lib.dak_alloc_counts(ctypes.byref(h), ctypes.byref(d)), "dak_alloc_counts")
    return int(h.value), int(d.value)


def dak_sm_count() -> int:
    return int(lib.dak_sm_count())


def dak_probe_read_bw(tier: int, nbytes: int, method: int = 0, ctas: int = 16, window: int = 4,
                      chunk_bytes: int = 32768, iters: int = 5):
    g = ctypes.c_double()
    ok = ctypes.c_int()
    _check(lib.dak_probe_read_bw(tier, nbytes, method, ctas, window, chunk_bytes, iters, ctypes.byref(g),
                                 ctypes.byref(ok)), "dak_probe_read_bw")
    return g.value, bool(ok.value)


def dak_probe_concurrent(host_bytes: int, hbm_bytes: int, host_ctas: int, host_window: int, hbm_ctas: int,
                         hbm_window: int, chunk_bytes: int = 32768, iters: int = 5):
    h, g = ctypes.c_double(), ctypes.c_double()
    _check(lib.dak_probe_concurrent(host_bytes, hbm_bytes, host_ctas, host_window, hbm_ctas, hbm_window, chunk_bytes,
                                    iters, ctypes.byref(h), ctypes.byref(g)), "dak_probe_concurrent")
    return h.value, g.value


# ------------------------------------------------------------------------------- decode step

DECODER_OPS = ("qkv", "o", "gate_up", "down", "kv")
MODE_DIRECT, MODE_PREFETCH_SERIAL, MODE_PREFETCH_OVERLAP = 0, 1, 2


class Decoder:
    """A dak_decoder over placed layers. `layers` is a list of dicts with the placements
    'qkv', 'o', 'gate_up', 'down', 'kv' and the bf16 CUDA gains 'attn_norm', 'mlp_norm';
    the decoder keeps references to them (and frees the placements in .free())."""

    def __init__(self, cfg: dict, layers, final_norm, n_split: int = 0, plain_launch: bool = False,
                 op_tuning=None, link_handoff: bool = True):
        """op_tuning: optional dict mapping 'qkv', 'o', 'gate_up', 'down', 'attn' to dak_tuning
        fields (dicts); n_split sets the attention's context splits (0 = library default);
        link_handoff=False turns off the host-link handoff between the step's kernels."""
        c = dak_decoder_config(n_layers=len(layers), hidden=int(cfg["hidden"]), n_heads=int(cfg["n_heads"]),
                               n_kv_heads=int(cfg["n_kv_heads"]), head_dim=int(cfg["head_dim"]),
                               ffn=int(cfg["ffn"]), rms_eps=float(cfg.get("rms_eps", 1e-5)),
                               rope_theta=float(cfg.get("rope_theta", 500000.0)),
                               plain_launch=int(bool(plain_launch)), no_link_handoff=int(not link_handoff))
        for i, name in enumerate(("qkv", "o", "gate_up", "down", "attn")):
            for k, v in dict((op_tuning or {}).get(name, {})).items():
                setattr(c.op_tuning[i], k, int(v))
        if n_split:
            c.op_tuning[4].n_split = int(n_split)
        for L in layers:
            _check_bf16_cuda(L["attn_norm"], "attn_norm")
            _check_bf16_cuda(L["mlp_norm"], "mlp_norm")
        _check_bf16_cuda(final_norm, "final_norm")
        arr = (dak_decoder_layer * max(1, len(layers)))()
        for i, L in enumerate(layers):
            arr[i] = dak_decoder_layer(L["qkv"].handle, L["o"].handle, L["gate_up"].handle, L["down"].handle,
                                       L["kv"].handle, L["attn_norm"].data_ptr(), L["mlp_norm"].data_ptr())
        out = ctypes.c_void_p()
        _check(lib.dak_decoder_create(ctypes.byref(c), arr, _ptr(final_norm), ctypes.byref(out)),
               "dak_decoder_create")
        self._h = out
        self.cfg = dict(cfg)
        self.layers = list(layers)
        self.final_norm = final_norm
        self.batch = int(lib.dak_decoder_batch(out))

    @property
    def handle(self):
        if self._h is None:
            raise ValueError("decoder already freed")
        return self._h

    def launches(self, mode: int = MODE_DIRECT) -> int:
        return int(lib.dak_decoder_launches(self.handle, int(mode)))

    def host_bytes(self) -> int:
        return sum(L[k].host_bytes for L in self.layers for k in DECODER_OPS)

    def step(self, x_in, positions, out=None, mode: int = MODE_DIRECT, stream=None):
        """One decode step: x_in bf16 [B][d], positions int32 [B] (CUDA) -> out bf16 [B][d]."""
        import torch
        _check_bf16_cuda(x_in, "x_in")
        if out is None:
            out = torch.empty_like(x_in)
        _check(lib.dak_decoder_step(self.handle, _ptr(x_in), _ptr(positions), _ptr(out), int(mode),
                                    _stream_ptr(stream)), "dak_decoder_step")
        return out

    def capture(self, x_in, positions, out, mode: int = MODE_DIRECT):
        """Capture one step with these buffers into the decoder's CUDA graph."""
        _check(lib.dak_decoder_capture(self.handle, _ptr(x_in), _ptr(positions), _ptr(out), int(mode)),
               "dak_decoder_capture")

    def replay(self, stream=None):
        _check(lib.dak_decoder_replay(self.handle, _stream_ptr(stream)), "dak_decoder_replay")

    def free(self, placements: bool = True):
        if self._h is not None:
            lib.dak_decoder_free(self._h)
            self._h = None
        if placements:
            for L in self.layers:
                for k in DECODER_OPS:
                    L[k].free()

    def __del__(self):
        try:
            self.free(placements=False)
        except Exception:
            pass


def place_decoder_layer(weights: dict, kv, host_units: dict, device=None, glu: bool = True) -> dict:
    """Place one layer: weights maps 'qkv', 'o', 'gate_up', 'down' to [out][in] bf16 sources
    (numpy bits or torch) and 'attn_norm', 'mlp_norm' to [d] gains; kv = (K, V) sources
    [B][H_kv][L][D]; host_units maps 'qkv', 'o', 'gate_up', 'down' to their host tile rows
    and either 'kv' to host requests or 'kv_heads' to host (request, kv head) slabs.
    glu places gate_up interleaved so that the SwiGLU runs in the GEMM's epilogue."""
    import torch
    dev = device or torch.device("cuda")
    L = {}
    for k in ("qkv", "o", "gate_up", "down"):
        if k == "gate_up" and glu:
            L[k] = dak_place_matrix_glu(weights[k], int(host_units[k]))
        else:
            L[k] = dak_place_matrix(weights[k], int(host_units[k]))
    if "kv_heads" in host_units:
        L["kv"] = dak_place_kv_heads(kv[0], kv[1], int(host_units["kv_heads"]))
    else:
        L["kv"] = dak_place_kv(kv[0], kv[1], int(host_units["kv"]))
    for k in ("attn_norm", "mlp_norm"):
        g = weights[k]
        if isinstance(g, np.ndarray):
            g = torch.from_numpy(g.view(np.int16)).view(torch.bfloat16)
        L[k] = g.to(dev).contiguous()
    return L


# ------------------------------------------------------------------------------- launch tuner

TUNING_FIELDS = [f for f, _ in dak_tuning._fields_]


def tuning_to_dict(t: dak_tuning, keep_zero: bool = False) -> dict:
    return {f: int(getattr(t, f)) for f in TUNING_FIELDS if keep_zero or getattr(t, f)}


def _tune_result(r: dak_tune_result) -> dict:
    return {"best": tuning_to_dict(r.best), "best_us": r.best_us, "default_us": r.default_us,
            "cc_off_us": r.cc_off_us, "no_align_us": r.no_align_us, "candidates": r.candidates}


def dak_tune_gemm(A: Placement, B, C, c_fp32: bool = False, reps: int = 5, base=None) -> dict:
    """Time dak_gemm over the tuner's candidates (host CTAs x window x chunk) and the
    congestion-control and wave-alignment ablations; returns the fastest tuning and times."""
    _check_bf16_cuda(B, "B")
    r = dak_tune_result()
    _check(lib.dak_tune_gemm(A.handle, _ptr(B), _ptr(C), int(B.shape[0]), int(bool(c_fp32)), int(reps),
                             _tuning(base), ctypes.byref(r)), "dak_tune_gemm")
    return _tune_result(r)


def dak_tune_attn(Q, KV: Placement, O, workspace=None, seq_lens=None, reps: int = 5, base=None) -> dict:
    """dak_tune_gemm for dak_attn (host CTAs x window; n_split from base or the default)."""
    Hq, O, workspace, ws_len, tun = _attn_common(Q, KV, O, workspace, base)
    r = dak_tune_result()
    _check(lib.dak_tune_attn(_ptr(Q), KV.handle, _ptr(seq_lens), Hq, _ptr(O), _ptr(workspace), ws_len, int(reps),
                             _tuning(tun), ctypes.byref(r)), "dak_tune_attn")
    return _tune_result(r)


def save_tuning(path: str, table: dict, meta: dict = None):
    """Persist a table {operation name: tuning fields} (e.g. the tuner's choices) as JSON."""
    import json
    doc = {"tuning": {k: {f: int(v) for f, v in dict(t).items() if f in TUNING_FIELDS} for k, t in table.items()}}
    if meta:
        doc["meta"] = meta
    with open(path, "w") as f:
        json.dump(doc, f, indent=1, sort_keys=True)


def load_tuning(path: str) -> dict:
    """Read a table written by save_tuning; unknown fields are rejected."""
    import json
    with open(path) as f:
        doc = json.load(f)
    table = {}
    for k, t in doc.get("tuning", {}).items():
        bad = set(t) - set(TUNING_FIELDS)
        if bad:
            raise ValueError(f"{path}: unknown tuning fields {sorted(bad)} for {k}")
        table[k] = {f: int(v) for f, v in t.items()}
    return table
