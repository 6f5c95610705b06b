"""gemv_dg_bf16_gb300 -- Python binding of libdecodegemm (decode-time skinny linears on GB300).

The functions carry the C ABI's names and only marshal arguments: every step of
the computation runs in the library's CUDA kernels.  Importing this package does
not load the library; the first call does, and it raises if the library is
missing (there is no CPU fallback).
"""
from ._binding import (  # noqa: F401
    DG_OP_GATE_UP_SILU, DG_OP_GEMV_BF16, DG_OP_HEAD_FP8_ARGMAX, DG_OP_MOE_W1, DG_OP_MOE_W2, DG_OP_GEMV_A8W8,
    dg_gemv_a8w8_blockscale, dg_quant_a8_blockscale,
    DG_VAR_CC_BULK, DG_VAR_CC_WARP, DG_VAR_DEFAULT, DG_VAR_MMA, DG_VAR_TC, DGError,
    DG_OK, DG_ERR_INVALID_ARG, DG_ERR_ALIGNMENT, DG_ERR_UNSUPPORTED_SHAPE, DG_ERR_WORKSPACE_TOO_SMALL, DG_ERR_CUDA,
    DG_ERR_TABLE_REFUSED, DG_ERR_NO_DEVICE, DG_ERR_BAD_VARIANT, DG_DEVERR_BAD_TOPK_ID, DG_DEVERR_WAIT_TIMEOUT, ROWS_BUCKETS, Choice,
    dg_build_id, dg_device_status, dg_device_status_clear, dg_gate_up_silu, dg_gemv_bf16, dg_head_fp8_argmax,
    dg_head_fp8_argmax_noalloc, dg_head_fp8_argmax_noalloc_status, dg_head_fp8_argmax_noalloc_scratch,
    dg_init, dg_launch_flags, dg_moe_w1_silu, dg_set_launch_flags, DG_LAUNCH_PDL,
    dg_set_numerics, dg_numerics, DG_NUMERICS_FASTEST, DG_NUMERICS_BATCH_INVARIANT, dg_moe_w2, dg_select,
    dg_selection_space, dg_selftest_wait_timeout, dg_moe_route_debug, DG_ROUTE_DEBUG_INTS, dg_status_str,
    dg_sweep,
    dg_table_check, dg_table_clear, dg_table_entries, dg_table_load, dg_workspace_bytes, lib,
    library_path, workspace,
)
