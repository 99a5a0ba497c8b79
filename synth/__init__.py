"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the CPU oracle.

Nothing here computes any part of the offloading method: the module only produces bf16
bit patterns (numpy ``uint16``) from a counter-based generator (SplitMix64 hash +
Box-Muller, see ``gen.c``), plus the shapes and distributions of the workloads the
direct-access kernels are measured on:

* decode GEMV: A 1024x1024 ~N(0, 0.02), B 1x1024 ~N(0, 1), tile rows of 64;
* 8B-shaped decode linears: QKV 6144x4096, O 4096x4096, gate+up 28672x4096,
  down 4096x14336, weights ~N(0, 0.02), hidden states N x K ~N(0, 1);
* decode GQA attention: 32 requests, 32 query / 8 KV heads, head dim 128, context
  8192, q/K/V ~N(0, 1).

Every tensor gets its own stream number so that any slice of it can be regenerated
independently (element i of a stream never depends on how many elements were drawn).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = os.path.join(_HERE, "_gen.so")
_DEV_SRC = os.path.join(_HERE, "gen_dev.cu")
_lock = threading.Lock()
_lib = None
_dev_lib = None


def build(force: bool = False) -> str:
    """Compile gen.c into _gen.so (plain gcc + OpenMP); returns the library path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _dev_lib_path() -> str:
    import platform
    return os.path.join(_HERE, f"_gen_dev_{platform.machine()}.so")


def build_dev(force: bool = False) -> str:
    """Compile gen_dev.cu (the device twin of the generator) with nvcc for sm_103a."""
    lib = _dev_lib_path()
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(_DEV_SRC):
        import shutil
        nvcc = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
                               "-Xcompiler", "-fPIC", "-o", tmp, _DEV_SRC])
        os.replace(tmp, lib)
    return lib


def _load_dev():
    global _dev_lib
    with _lock:
        if _dev_lib is None:
            lib = ctypes.CDLL(build_dev())
            u64, dbl, vp = ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p
            lib.synth_dev_normal_bf16.argtypes = [u64, u64, dbl, dbl, u64, u64, vp, vp]
            lib.synth_dev_normal_bf16.restype = ctypes.c_int
            _dev_lib = lib
    return _dev_lib


def dev_normal_bf16(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0, offset: int = 0,
                    out=None, cuda_stream=None):
    """The values of normal_bf16, drawn on the GPU into a bf16 torch tensor (or `out`)."""
    import torch
    if out is None:
        out = torch.empty(int(n), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream if cuda_stream is None else cuda_stream
    err = _load_dev().synth_dev_normal_bf16(seed, stream, float(mean), float(std), int(offset), int(n),
                                             out.data_ptr(), s)
    if err:
        raise RuntimeError(f"synth_dev_normal_bf16: CUDA error {err}")
    return out


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, dbl, i32 = ctypes.c_uint64, ctypes.c_double, ctypes.c_int
            vp = ctypes.c_void_p
            lib.synth_normal_bf16.argtypes = [u64, u64, dbl, dbl, u64, u64, vp]
            lib.synth_int_bf16.argtypes = [u64, u64, i32, i32, u64, u64, vp]
            lib.synth_uniform_f64.argtypes = [u64, u64, u64, u64, vp]
            lib.synth_threads.restype = i32
            _lib = lib
    return _lib


def normal_bf16(seed: int, stream: int, n: int, mean: float = 0.0, std: float = 1.0,
                offset: int = 0) -> np.ndarray:
    """n bf16 values (as uint16 bits) ~ N(mean, std^2), elements offset..offset+n-1 of the stream."""
    out = np.empty(int(n), dtype=np.uint16)
    if n:
        _load().synth_normal_bf16(seed, stream, float(mean), float(std), int(offset), int(n),
                                  out.ctypes.data)
    return out


def int_bf16(seed: int, stream: int, n: int, lo: int, hi: int, offset: int = 0) -> np.ndarray:
    """n bf16 values (uint16 bits) holding integers drawn uniformly from [lo, hi]."""
    out = np.empty(int(n), dtype=np.uint16)
    if n:
        _load().synth_int_bf16(seed, stream, int(lo), int(hi), int(offset), int(n), out.ctypes.data)
    return out


def uniform_f64(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(int(n), dtype=np.float64)
    if n:
        _load().synth_uniform_f64(seed, stream, int(offset), int(n), out.ctypes.data)
    return out


def threads() -> int:
    return int(_load().synth_threads())


# ----------------------------------------------------------------------------------------
# Workload recipes (shapes, distributions, seeds). Stream numbers are fixed per tensor.
# ----------------------------------------------------------------------------------------

WEIGHT_STD = 0.02

# 8B-shaped decode linear layers: name -> (M = out features, K = in features)
LINEARS_8B = {
    "qkv": (6144, 4096),
    "o": (4096, 4096),
    "gate_up": (28672, 4096),
    "down": (4096, 14336),
}

ATTN_DECODE = dict(batch=32, h_q=32, h_kv=8, head_dim=128, context=8192)


def gemm_inputs(M: int, K: int, N: int, seed: int = 0, tensor_index: int = 0,
                integer: bool = False):
    """Weights A [M][K] ~N(0, 0.02) and hidden states B [N][K] ~N(0, 1) as bf16 bits.

    ``integer=True`` draws both from the integers [-8, 8] instead (exact fp32 sums)."""
    s = seed + tensor_index
    if integer:
        A = int_bf16(s, 1, M * K, -8, 8).reshape(M, K)
        B = int_bf16(s, 2, N * K, -8, 8).reshape(N, K)
    else:
        A = normal_bf16(s, 1, M * K, 0.0, WEIGHT_STD).reshape(M, K)
        B = normal_bf16(s, 2, N * K, 0.0, 1.0).reshape(N, K)
    return A, B


def attn_inputs(batch: int, h_q: int, h_kv: int, head_dim: int, context: int, seed: int = 0,
                tensor_index: int = 0):
    """q [B][Hq][D], K and V [B][Hkv][L][D], all ~N(0, 1), as bf16 bits."""
    s = seed + tensor_index
    q = normal_bf16(s, 11, batch * h_q * head_dim).reshape(batch, h_q, head_dim)
    n_kv = batch * h_kv * context * head_dim
    k = normal_bf16(s, 12, n_kv).reshape(batch, h_kv, context, head_dim)
    v = normal_bf16(s, 13, n_kv).reshape(batch, h_kv, context, head_dim)
    return q, k, v


def attn_kv_request(b: int, h_kv: int, head_dim: int, context: int, seed: int = 0,
                    tensor_index: int = 0):
    """K and V of request b alone ([Hkv][L][D] each), identical to the slice of attn_inputs."""
    s = seed + tensor_index
    per = h_kv * context * head_dim
    k = normal_bf16(s, 12, per, offset=b * per).reshape(h_kv, context, head_dim)
    v = normal_bf16(s, 13, per, offset=b * per).reshape(h_kv, context, head_dim)
    return k, v


# Decode step of a Llama-shaped transformer. Weights ~N(0, 0.02); RMSNorm gains ~N(1, 0.1)
# (not all ones, so that a dropped gain shows); hidden states and the cached keys and values
# ~N(0, 1). Tensor t of layer l uses stream 1000 + 16 l + t.
DECODER_8B = dict(n_layers=32, hidden=4096, n_heads=32, n_kv_heads=8, head_dim=128, ffn=14336,
                  batch=16, context=4096, rms_eps=1e-5, rope_theta=500000.0)
DECODER_70B = dict(n_layers=80, hidden=8192, n_heads=64, n_kv_heads=8, head_dim=128, ffn=28672,
                   batch=16, context=16384, rms_eps=1e-5, rope_theta=500000.0)
NORM_STD = 0.1

_DEC_TENSORS = ("qkv", "o", "gate_up", "down", "attn_norm", "mlp_norm", "k_cache", "v_cache")


def decoder_shapes(cfg: dict) -> dict:
    """[out][in] shape of each weight of one layer, and [d] of each norm gain."""
    d, Hq, Hkv, D, f = (cfg["hidden"], cfg["n_heads"], cfg["n_kv_heads"], cfg["head_dim"],
                        cfg["ffn"])
    return {"qkv": ((Hq + 2 * Hkv) * D, d), "o": (d, Hq * D), "gate_up": (2 * f, d),
            "down": (d, f), "attn_norm": (d,), "mlp_norm": (d,)}


def decoder_stream(layer: int, name: str) -> int:
    return 1000 + 16 * layer + _DEC_TENSORS.index(name)


def decoder_tensor(cfg: dict, layer: int, name: str, seed: int = 0) -> np.ndarray:
    """One weight ([out][in]) or norm gain ([d]) of layer `layer`, as bf16 bits."""
    shape = decoder_shapes(cfg)[name]
    n = int(np.prod(shape))
    if name.endswith("_norm"):
        return normal_bf16(seed, decoder_stream(layer, name), n, 1.0, NORM_STD).reshape(shape)
    return normal_bf16(seed, decoder_stream(layer, name), n, 0.0, WEIGHT_STD).reshape(shape)


def decoder_layer(cfg: dict, layer: int, seed: int = 0) -> dict:
    return {name: decoder_tensor(cfg, layer, name, seed) for name in decoder_shapes(cfg)}


def decoder_final_norm(cfg: dict, seed: int = 0) -> np.ndarray:
    return normal_bf16(seed, 999, cfg["hidden"], 1.0, NORM_STD)


def decoder_x0(cfg: dict, batch: int, seed: int = 0) -> np.ndarray:
    """Hidden states entering layer 0 (the embedding output), [batch][d]."""
    return normal_bf16(seed, 998, batch * cfg["hidden"]).reshape(batch, cfg["hidden"])


def decoder_kv(cfg: dict, layer: int, batch: int, capacity: int, seed: int = 0):
    """Cached keys and values of layer `layer`, [batch][Hkv][capacity][D] each ~N(0, 1)."""
    n = batch * cfg["n_kv_heads"] * capacity * cfg["head_dim"]
    shape = (batch, cfg["n_kv_heads"], capacity, cfg["head_dim"])
    k = normal_bf16(seed, decoder_stream(layer, "k_cache"), n).reshape(shape)
    v = normal_bf16(seed, decoder_stream(layer, "v_cache"), n).reshape(shape)
    return k, v


def decoder_tensor_dev(cfg: dict, layer: int, name: str, seed: int = 0):
    """decoder_tensor drawn on the GPU (bf16 torch tensor of the same shape)."""
    shape = decoder_shapes(cfg)[name]
    n = int(np.prod(shape))
    mean, std = (1.0, NORM_STD) if name.endswith("_norm") else (0.0, WEIGHT_STD)
    return dev_normal_bf16(seed, decoder_stream(layer, name), n, mean, std).view(*shape)


def decoder_kv_dev(cfg: dict, layer: int, batch: int, capacity: int, seed: int = 0):
    """decoder_kv drawn on the GPU (bf16 torch tensors)."""
    n = batch * cfg["n_kv_heads"] * capacity * cfg["head_dim"]
    shape = (batch, cfg["n_kv_heads"], capacity, cfg["head_dim"])
    k = dev_normal_bf16(seed, decoder_stream(layer, "k_cache"), n).view(*shape)
    v = dev_normal_bf16(seed, decoder_stream(layer, "v_cache"), n).view(*shape)
    return k, v
