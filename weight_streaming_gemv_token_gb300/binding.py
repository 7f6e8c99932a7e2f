"""ctypes binding of libwsg.so: the same names as the C ABI in include/wsg.h.

Argument marshalling only. Device pointers may be given as ints or as torch
tensors (their data_ptr() is passed); streams as ints (cudaStream_t), torch
streams, or None for the legacy default stream. Every non-zero dec_status
raises WsgError carrying the library's message. There is no fallback: if the
library is missing the import of a function raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

c_int32, c_uint32, c_float, c_size_t, c_void_p = ctypes.c_int32, ctypes.c_uint32, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

DEC_OK, DEC_EINVAL, DEC_ESTATE, DEC_ECAPACITY, DEC_ENOMEM, DEC_ECUDA, DEC_EDEVICE = range(7)
STATUS_NAMES = {0: "DEC_OK", 1: "DEC_EINVAL", 2: "DEC_ESTATE", 3: "DEC_ECAPACITY", 4: "DEC_ENOMEM", 5: "DEC_ECUDA", 6: "DEC_EDEVICE"}
DEC_F32, DEC_BF16, DEC_Q4G64 = 0, 1, 2
DEC_SKIP_LOGITS = 0x1
DEC_ENGINE_PERSISTENT, DEC_ENGINE_STAGED = 0, 1
DEC_DEVERR_WAIT_TIMEOUT, DEC_DEVERR_ARGMAX_NAN, DEC_DEVERR_BAD_TOKEN = 0x1, 0x2, 0x4
DEC_DEVERR_BAD_POSITION, DEC_DEVERR_EXCHANGE_TIMEOUT, DEC_DEVERR_GEMM_TIMEOUT, DEC_DEVERR_BARRIER_TIMEOUT = (
    0x8, 0x10, 0x20, 0x40)

# Every symbol include/wsg.h declares.
EXPORTED = (
    "dec_workspace_bytes", "dec_create", "dec_load_weights", "dec_reset", "dec_rewind", "dec_step", "dec_prefill_chunk",
    "dec_generate", "dec_get_kv", "dec_position", "dec_trace_bytes", "dec_set_trace", "dec_device_errors",
    "dec_destroy", "dec_last_error",
    "gemv", "gemv_q4", "gemv_q4_rows_per_warp", "gemv_device_errors", "greedy_head_noalloc", "gemm_bf16",
    "pack_bf16_exact", "dec_verify2", "dec_set_wait_limit",
)


class WsgError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class dec_config(ctypes.Structure):
    _fields_ = [
        ("layers", c_int32), ("hidden", c_int32), ("inter", c_int32), ("n_q", c_int32), ("n_kv", c_int32),
        ("head_dim", c_int32), ("vocab", c_int32), ("eps", c_float), ("rope_theta", c_float),
        ("wdtype", c_int32), ("kvdtype", c_int32), ("max_seq", c_int32), ("chunk_cap", c_int32),
        ("engine", c_int32),
    ]


class dec_layer_weights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in
                ("w_q", "w_k", "w_v", "w_o", "w_gate", "w_up", "w_down", "g_in", "g_post", "g_q", "g_k")]


class dec_weights(ctypes.Structure):
    _fields_ = [("embed", c_void_p), ("g_final", c_void_p), ("layers", ctypes.POINTER(dec_layer_weights))]


_lib = None


def library() -> ctypes.CDLL:
    """The loaded libwsg.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"{_build.LIB} is missing: build it with weight_streaming_gemv_token_gb300.build.build()")
        lib = ctypes.CDLL(_build.LIB)
        P = ctypes.POINTER
        sig = {
            "dec_workspace_bytes": (c_size_t, [P(dec_config)]),
            "dec_create": (c_int32, [P(dec_config), c_void_p, c_size_t, c_void_p, P(c_void_p)]),
            "dec_load_weights": (c_int32, [c_void_p, P(dec_weights)]),
            "dec_reset": (c_int32, [c_void_p]),
            "dec_rewind": (c_int32, [c_void_p, c_int32]),
            "dec_verify2": (c_int32, [c_void_p, P(c_int32), c_void_p, P(c_int32)]),
            "dec_step": (c_int32, [c_void_p, c_int32, c_uint32, c_void_p, P(c_int32)]),
            "dec_prefill_chunk": (c_int32, [c_void_p, P(c_int32), c_int32, c_int32, c_void_p, P(c_int32)]),
            "dec_generate": (c_int32, [c_void_p, c_int32, c_int32, c_void_p]),
            "dec_get_kv": (c_int32, [c_void_p, c_int32, P(c_void_p), P(c_void_p), P(c_int32)]),
            "dec_position": (c_int32, [c_void_p]),
            "dec_trace_bytes": (c_size_t, [c_void_p]),
            "dec_set_trace": (c_int32, [c_void_p, c_void_p, c_size_t]),
            "dec_set_wait_limit": (c_int32, [c_void_p, ctypes.c_uint64]),
            "dec_device_errors": (c_int32, [c_void_p, c_int32, P(c_uint32)]),
            "dec_destroy": (None, [c_void_p]),
            "dec_last_error": (ctypes.c_char_p, [c_void_p]),
            "gemv": (c_int32, [c_int32, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_void_p]),
            "gemv_q4": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_void_p]),
            "gemv_q4_rows_per_warp": (c_int32, [c_int32, c_int32]),
            "gemv_device_errors": (c_int32, [c_int32, P(c_uint32)]),
            "pack_bf16_exact": (c_int32, [c_void_p, c_void_p, ctypes.c_int64, c_void_p, P(ctypes.c_int64)]),
            "gemm_bf16": (c_int32, [c_void_p, c_void_p, c_void_p, c_int32, c_int32, c_int32, c_int32, c_int32, c_void_p]),
            "greedy_head_noalloc": (c_int32, [c_int32, c_void_p, c_void_p, c_void_p, c_float, c_int32, c_int32,
                                              c_void_p, c_void_p, c_void_p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"expected a device pointer (int or tensor), got {type(x)}")


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, ctx=None):
    if status != DEC_OK:
        msg = library().dec_last_error(ctx)
        raise WsgError(status, msg.decode() if msg else "")


# ---- C ABI, one Python function per symbol ----

def dec_workspace_bytes(cfg: dec_config) -> int:
    return library().dec_workspace_bytes(ctypes.byref(cfg))


def dec_create(cfg: dec_config, workspace, workspace_bytes: int, stream=None) -> int:
    h = c_void_p()
    _check(library().dec_create(ctypes.byref(cfg), _ptr(workspace), workspace_bytes, _stream(stream), ctypes.byref(h)))
    return h.value


def dec_load_weights(ctx: int, weights: dec_weights):
    _check(library().dec_load_weights(ctx, ctypes.byref(weights)), ctx)


def dec_reset(ctx: int):
    _check(library().dec_reset(ctx), ctx)


def dec_rewind(ctx: int, pos: int):
    _check(library().dec_rewind(ctx, int(pos)), ctx)


def dec_step(ctx: int, token: int, flags: int = 0, d_logits=None, want_next: bool = True) -> int | None:
    nxt = c_int32(-1)
    _check(library().dec_step(ctx, token, flags, _ptr(d_logits), ctypes.byref(nxt) if want_next else None), ctx)
    return nxt.value if want_next else None


def dec_verify2(ctx: int, tokens, d_logits=None, want_next: bool = True) -> tuple[int, int] | None:
    if len(tokens) != 2:
        raise ValueError("dec_verify2 takes two tokens")
    arr = (c_int32 * 2)(int(tokens[0]), int(tokens[1]))
    nxt = (c_int32 * 2)(-1, -1)
    _check(library().dec_verify2(ctx, arr, _ptr(d_logits), nxt if want_next else None), ctx)
    return (nxt[0], nxt[1]) if want_next else None


def dec_prefill_chunk(ctx: int, tokens, is_last: bool, d_logits=None, want_next: bool = True) -> int | None:
    arr = (c_int32 * len(tokens))(*[int(t) for t in tokens])
    nxt = c_int32(-1)
    want = want_next and is_last
    _check(library().dec_prefill_chunk(ctx, arr, len(tokens), int(bool(is_last)), _ptr(d_logits),
                                       ctypes.byref(nxt) if want else None), ctx)
    return nxt.value if want else None


def dec_generate(ctx: int, token: int, n: int, d_tokens_out):
    _check(library().dec_generate(ctx, token, n, _ptr(d_tokens_out)), ctx)


def dec_get_kv(ctx: int, layer: int) -> tuple[int, int, int]:
    k, v, n = c_void_p(), c_void_p(), c_int32()
    _check(library().dec_get_kv(ctx, layer, ctypes.byref(k), ctypes.byref(v), ctypes.byref(n)), ctx)
    return k.value, v.value, n.value


def dec_position(ctx: int) -> int:
    return library().dec_position(ctx)


def dec_trace_bytes(ctx: int) -> int:
    return library().dec_trace_bytes(ctx)


def dec_set_trace(ctx: int, d_trace, nbytes: int):
    _check(library().dec_set_trace(ctx, _ptr(d_trace), nbytes), ctx)


def dec_set_wait_limit(ctx: int, ns: int):
    _check(library().dec_set_wait_limit(ctx, int(ns)), ctx)


def dec_device_errors(ctx: int, clear: bool = True) -> int:
    bits = c_uint32()
    _check(library().dec_device_errors(ctx, int(clear), ctypes.byref(bits)), ctx)
    return bits.value


def dec_destroy(ctx: int):
    library().dec_destroy(ctx)


def dec_last_error(ctx=None) -> str:
    m = library().dec_last_error(ctx)
    return m.decode() if m else ""


def gemv(wdtype: int, W, x, y, out: int, inp: int, stream=None):
    _check(library().gemv(wdtype, _ptr(W), _ptr(x), _ptr(y), out, inp, _stream(stream)))


def gemv_q4(codes, scale, bias, x, y, out: int, inp: int, ntok: int, stream=None):
    _check(library().gemv_q4(_ptr(codes), _ptr(scale), _ptr(bias), _ptr(x), _ptr(y), out, inp, ntok, _stream(stream)))


def gemv_q4_rows_per_warp(ntok: int, r: int = 0) -> int:
    v = library().gemv_q4_rows_per_warp(ntok, r)
    if v < 0:
        raise WsgError(DEC_EINVAL, f"gemv_q4_rows_per_warp({ntok}, {r})")
    return v


def pack_bf16_exact(src, dst, n: int, stream=None) -> int:
    """dst = high halves of the float32 src; returns how many elements that storage does not hold exactly."""
    bad = ctypes.c_int64()
    _check(library().pack_bf16_exact(_ptr(src), _ptr(dst), n, _stream(stream), ctypes.byref(bad)))
    return bad.value


def gemv_device_errors(clear: bool = True) -> int:
    bits = c_uint32()
    _check(library().gemv_device_errors(int(clear), ctypes.byref(bits)))
    return bits.value


def greedy_head_noalloc(wdtype: int, embed, h, gain, eps: float, vocab: int, hidden: int, logits, token, stream=None):
    """Final RMSNorm, tied vocabulary GEMV and greedy argmax with no device allocation (library-held scratch)."""
    _check(library().greedy_head_noalloc(wdtype, _ptr(embed), _ptr(h), _ptr(gain), eps, vocab, hidden, _ptr(logits),
                                         _ptr(token), _stream(stream)))


def gemm_bf16(A, W, C, M: int, N: int, K: int, ldc: int | None = None, accumulate: bool = False, stream=None):
    """C[M][N] (=, or += with accumulate) A[M][K] . W[N][K]^T, bfloat16 operands, FP32 accumulation (tensor cores)."""
    _check(library().gemm_bf16(_ptr(A), _ptr(W), _ptr(C), M, N, K, N if ldc is None else ldc, int(bool(accumulate)),
                               _stream(stream)))
