"""PyTorch drop-in modules over the C ABI, named as in "DAK: Direct-Access-Enabled GPU Memory
Offloading with Optimal Efficiency for LLM Inference", section 5: SplitK_GEMM replaces a
model's nn.Linear and SplitK_FlashAttn its decode attention over a pre-allocated (static)
KV cache. Each module owns a placement of its operand across pinned host memory and HBM
and calls the library's kernels; the modules only reshape and check arguments, every
arithmetic step runs in libdak.so. They hold no trainable parameters (inference only)."""
import torch

from . import _lib


class SplitK_GEMM(torch.nn.Module):
    """y = x . W^T for a bf16 weight W [out_features][in_features] split by tile rows between
    host memory (the first n_host_tiles) and HBM ([DAK] section 4.1). x is any bf16 CUDA
    tensor [..., in_features] (contiguous); the leading dimensions are the GEMM's N rows.
    Bias-free like the Llama-family linears: every step of the product runs in the
    library's kernels, and a bias add would not. fp32_out returns the fp32 accumulators
    instead of bf16 (round to nearest even)."""

    def __init__(self, weight, offload_ratio: float = 0.0, n_host_tiles: int = None, tile_m: int = 64,
                 fp32_out: bool = False, tuning=None):
        super().__init__()
        if weight.ndim != 2:
            raise ValueError("weight must be [out_features][in_features]")
        self.out_features, self.in_features = int(weight.shape[0]), int(weight.shape[1])
        if n_host_tiles is None:
            n_host_tiles = _lib.host_tiles_for_ratio(offload_ratio, self.out_features, tile_m)
        w = weight.detach() if isinstance(weight, torch.Tensor) else weight
        if isinstance(w, torch.Tensor) and w.dtype != torch.bfloat16:
            raise ValueError("weight must be bf16")
        self.placement = _lib.dak_place_matrix(w.contiguous() if isinstance(w, torch.Tensor) else w,
                                               int(n_host_tiles), tile_m=tile_m)
        self.fp32_out = bool(fp32_out)
        self.tuning = tuning

    @classmethod
    def from_linear(cls, linear: torch.nn.Linear, offload_ratio: float = 0.0, **kw) -> "SplitK_GEMM":
        """The placed counterpart of a bias-free nn.Linear (its bf16 weight)."""
        if linear.bias is not None:
            raise ValueError("SplitK_GEMM replaces bias-free linears")
        return cls(linear.weight.to(torch.bfloat16), offload_ratio=offload_ratio, **kw)

    @property
    def host_bytes(self) -> int:
        return self.placement.host_bytes

    def forward(self, x):
        if x.shape[-1] != self.in_features:
            raise ValueError(f"last dimension {x.shape[-1]} != in_features {self.in_features}")
        lead = x.shape[:-1]
        y = _lib.dak_gemm(self.placement, x.reshape(-1, self.in_features), c_fp32=self.fp32_out,
                          tuning=self.tuning)
        return y.view(*lead, self.out_features)

    def extra_repr(self):
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"host_bytes={self.placement.host_bytes}, hbm_bytes={self.placement.hbm_bytes}")


class SplitK_FlashAttn(torch.nn.Module):
    """Decode attention with the semantics of torch's scaled_dot_product_attention for one
    new query token per request (grouped-query: query head h reads kv head h // (H_q / H_kv),
    scale 1/sqrt(D) unless given, positions past seq_lens[b] masked), over a static KV cache
    K, V [B][H_kv][L][D] bf16 placed across host memory and HBM ([DAK] section 5): the first
    n_host_heads (request, kv head) slabs on the host. The cache is copied into the placement
    at construction; append(k, v, positions) writes each step's new token into it.
    forward(query [B][H_q][D] or [B][H_q][1][D], seq_lens int32 [B]) returns the same shape,
    bf16 (or fp32 with fp32_out)."""

    def __init__(self, k_cache, v_cache, offload_ratio: float = 0.0, n_host_heads: int = None,
                 n_split: int = 0, fp32_out: bool = False, tuning=None):
        super().__init__()
        if k_cache.shape != v_cache.shape or k_cache.ndim != 4:
            raise ValueError("k_cache and v_cache must both be [B][H_kv][L][D]")
        B, Hkv, L, D = (int(s) for s in k_cache.shape)
        if n_host_heads is None:
            n_host_heads = _lib.host_heads_for_ratio(offload_ratio, B, Hkv)
        self.placement = _lib.dak_place_kv_heads(k_cache, v_cache, int(n_host_heads))
        self.batch, self.n_kv_heads, self.capacity, self.head_dim = B, Hkv, L, D
        self.n_split = int(n_split) or _lib.dak_attn_default_split(self.placement)
        self.fp32_out = bool(fp32_out)
        self.tuning = dict(tuning or {})
        self._ws = None

    @property
    def host_bytes(self) -> int:
        return self.placement.host_bytes

    def append(self, k_new, v_new, positions):
        """Write one token per request: k_new, v_new bf16 CUDA [B][H_kv][D] (or [B][H_kv][1][D]),
        positions int32 CUDA [B]."""
        shape = (self.batch, self.n_kv_heads, self.head_dim)
        n = self.batch * self.n_kv_heads * self.head_dim
        if k_new.numel() != n or v_new.numel() != n:
            raise ValueError(f"k_new / v_new must hold {list(shape)}")
        _lib.dak_kv_append(self.placement, k_new.reshape(shape), v_new.reshape(shape), positions)

    def forward(self, query, seq_lens=None, scale: float = None):
        squeeze = query.ndim == 4
        if squeeze:
            if query.shape[2] != 1:
                raise ValueError("one query token per request (decode)")
            q = query.reshape(query.shape[0], query.shape[1], query.shape[3])
        else:
            q = query
        Hq = int(q.shape[1])
        need = _lib.dak_attn_workspace_bytes(self.batch, Hq, self.head_dim, self.n_split)
        if need and (self._ws is None or self._ws.numel() * 4 < need or self._ws.device != q.device):
            self._ws = torch.empty((need + 3) // 4, dtype=torch.float32, device=q.device)
        tun = dict(self.tuning, n_split=self.n_split)
        fn = _lib.dak_attn_f32 if self.fp32_out else _lib.dak_attn
        o = fn(q, self.placement, seq_lens=seq_lens, scale=float(scale or 0.0), workspace=self._ws, tuning=tun)
        return o.view(query.shape) if squeeze else o

    def extra_repr(self):
        return (f"batch={self.batch}, n_kv_heads={self.n_kv_heads}, capacity={self.capacity}, "
                f"head_dim={self.head_dim}, n_split={self.n_split}, host_bytes={self.placement.host_bytes}")
