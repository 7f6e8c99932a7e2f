"""Weight-streaming batch-1 decode on GB300 (sm_103a).

The compute path is libwsg.so (CUDA kernels behind the C ABI of
include/wsg.h); this package holds its build script, the ctypes binding with
the same function names, and a small Decoder wrapper that owns the device
workspace. Nothing here computes on the CPU.
"""
from .binding import (  # noqa: F401
    DEC_BF16,
    DEC_F32,
    DEC_Q4G64,
    DEC_SKIP_LOGITS,
    EXPORTED,
    WsgError,
    dec_config,
    dec_create,
    dec_destroy,
    dec_device_errors,
    dec_generate,
    dec_get_kv,
    dec_last_error,
    dec_layer_weights,
    dec_load_weights,
    dec_position,
    dec_prefill_chunk,
    dec_reset,
    dec_rewind,
    dec_set_trace,
    dec_set_wait_limit,
    dec_step,
    dec_trace_bytes,
    dec_verify2,
    dec_weights,
    dec_workspace_bytes,
    gemm_bf16,
    gemv,
    gemv_device_errors,
    gemv_q4,
    gemv_q4_rows_per_warp,
    greedy_head_noalloc,
    library,
    pack_bf16_exact,
)
