"""Direct-access tiered-memory decode kernels for GB300 (sm_103a).

A weight matrix (or KV cache) is split between pinned, device-mapped host memory and HBM;
CTAs read each tier straight into shared memory and compute a decode GEMM or a decode
attention from it, with no staging copy in HBM. The work is done by libdak.so (CUDA C++
built in-tree); this package only marshals arguments to its C ABI.
"""
from ._lib import (  # noqa: F401
    DAK_OK, DECODER_OPS, EXPORTS, FAULT_DEVICE_ALLOC, FAULT_HOST_ALLOC, FAULT_TENSOR_MAP, MODE_DIRECT,
    MODE_PREFETCH_OVERLAP, MODE_PREFETCH_SERIAL, NOALLOC_SCRATCH_BYTES, TUNING_FIELDS, DakError,
    Decoder, Placement, dak_alloc_counts, dak_attn, dak_attn_default_split, dak_attn_f32,
    dak_attn_noalloc, dak_attn_staged, dak_attn_workspace_bytes, dak_fault_pending, dak_free, dak_gemm,
    dak_gemm_chain, dak_gemm_chain_plan, dak_gemm_chain_workspace_bytes, dak_gemm_launch_plan, dak_gemm_op, dak_gemm_plan,
    dak_gemm_staged, dak_gemm_workspace_bytes, dak_inject_fault, dak_kv_append, dak_last_error,
    dak_link_begin, dak_link_timeouts, dak_op, dak_place_kv, dak_place_kv_heads, dak_place_matrix,
    dak_place_matrix_glu, dak_placement_info, dak_plan_ratios, dak_plan_units, dak_prefetch,
    dak_probe_concurrent, dak_probe_read_bw, dak_selftest_link, dak_selftest_wait, dak_sm_count,
    dak_tune_attn, dak_tune_gemm, dak_tuning, host_requests_for_ratio, host_heads_for_ratio,
    host_tiles_for_ratio, lib, load_tuning, place_decoder_layer, save_tuning, tuning_to_dict,
)
from .modules import SplitK_FlashAttn, SplitK_GEMM  # noqa: F401,E402
