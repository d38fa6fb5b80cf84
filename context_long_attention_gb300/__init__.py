"""Context-parallel attention on one GB300 (sm_103a): Python binding.

A thin ctypes layer over ``libcpattn.so`` (declared in ``include/cpattn.h``).
It only marshals arguments: PyTorch provides device memory and the current
stream, and every step of the computation runs in the library's CUDA kernels.
The functions keep the C names:

    cp_shard_plan, cp_prefill_attn, cp_decode_plan, cp_decode_plan_ex,
    cp_kv_shard_pack, cp_decode_attn, cp_lse_merge, cp_lse_fold,
    cp_device_error_check

There is no CPU fallback: importing the package loads the library, and
raises if it has not been built (``__graft_entry__.build()``).
"""

from ._binding import (  # noqa: F401
    CP_BF16,
    CP_DCP_CONTIGUOUS,
    CP_DCP_ROUND_ROBIN,
    CP_DCP_SELECTED,
    CP_DECODE_GQA,
    CP_DECODE_MLA,
    CP_FP8_E4M3,
    CP_FP32,
    CP_INTERLEAVE,
    CP_ZIGZAG,
    CpError,
    DecodePlan,
    PageTable,
    PrefillPlan,
    cp_decode_attn,
    cp_decode_attn_merged,
    cp_decode_attn_noalloc,
    cp_decode_attn_paged,
    cp_decode_plan,
    cp_decode_plan_ex,
    cp_decode_merged_workspace_size,
    cp_decode_workspace_size,
    cp_device_error_check,
    cp_kv_shard_pack,
    cp_kv_shard_pack_paged,
    cp_lse_fold,
    cp_lse_merge,
    cp_plan_size,
    cp_prefill_attn,
    cp_shard_plan,
    cp_sparse_decode_attn,
    cp_sparse_decode_attn_merged,
    cp_sparse_gather,
    cp_sparse_plan,
    cp_sparse_topk,
    cp_sparse_workspace_size,
    lib,
    lib_path,
    sparse_slot_rows,
)
