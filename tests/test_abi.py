"""The C-ABI library builds, loads and exports every symbol include/wsg.h declares.

CPU only: no call here reaches a kernel. Argument validation that happens on
the host (before any device query) is exercised too.
"""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wsg.h")


@pytest.fixture(scope="module")
def lib():
    from weight_streaming_gemv_token_gb300 import build as bld

    bld.build()
    import weight_streaming_gemv_token_gb300 as W

    return W.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "sizeof")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("dec_create", "dec_load_weights", "dec_reset", "dec_prefill_chunk", "dec_step", "gemv", "gemv_q4"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    import weight_streaming_gemv_token_gb300 as W

    names = declared_functions()
    assert sorted(W.EXPORTED) == names
    for n in names:
        assert getattr(lib, n) is not None
    from weight_streaming_gemv_token_gb300 import build as bld

    out = subprocess.run(["nm", "-D", "--defined-only", bld.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    assert set(names) <= exported


def test_library_targets_sm103a_only():
    from weight_streaming_gemv_token_gb300 import build as bld

    assert bld.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_workspace_size_host_logic(lib):
    import workloads as Wl
    from weight_streaming_gemv_token_gb300 import binding as B

    s = Wl.QWEN3_06B
    cfg = B.dec_config(layers=s.layers, hidden=s.hidden, inter=s.inter, n_q=s.n_q, n_kv=s.n_kv, head_dim=s.head_dim,
                       vocab=s.vocab, eps=1e-6, rope_theta=1e6, wdtype=B.DEC_BF16, kvdtype=B.DEC_BF16,
                       max_seq=5120, chunk_cap=0)
    n = B.dec_workspace_bytes(cfg)
    kv = 2 * s.layers * s.n_kv * 5120 * s.head_dim * 2
    assert kv <= n < kv + 64 * 2**20
    cfg.kvdtype = B.DEC_F32
    assert B.dec_workspace_bytes(cfg) >= 2 * kv
    # invalid configurations give 0
    for field, bad in [("n_kv", 3), ("head_dim", 130), ("hidden", 0), ("wdtype", 7), ("max_seq", 0), ("head_dim", 6)]:
        c2 = B.dec_config.from_buffer_copy(cfg)
        setattr(c2, field, bad)
        assert B.dec_workspace_bytes(c2) == 0, field


def test_q4_configuration_rules(lib):
    """The 4-bit configuration: either engine, tokenwise prompts, widths multiples of 512; its
    workspace holds two rows of activations and logits for the verify step."""
    import workloads as Wl
    from weight_streaming_gemv_token_gb300 import binding as B

    s = Wl.QWEN3_06B
    cfg = B.dec_config(layers=s.layers, hidden=s.hidden, inter=s.inter, n_q=s.n_q, n_kv=s.n_kv, head_dim=s.head_dim,
                       vocab=s.vocab, eps=1e-6, rope_theta=1e6, wdtype=B.DEC_BF16, kvdtype=B.DEC_F32,
                       max_seq=512, chunk_cap=0, engine=B.DEC_ENGINE_STAGED)
    n_bf16 = B.dec_workspace_bytes(cfg)
    cfg.wdtype = B.DEC_Q4G64
    n_q4 = B.dec_workspace_bytes(cfg)
    assert n_q4 >= n_bf16 + 4 * s.vocab  # a second logit row
    c3 = B.dec_config.from_buffer_copy(cfg)
    c3.engine = B.DEC_ENGINE_PERSISTENT
    assert B.dec_workspace_bytes(c3) == n_q4
    for field, bad in [("chunk_cap", 128), ("hidden", 1024 + 64),
                       ("inter", 3072 + 256), ("n_q", 12)]:
        c2 = B.dec_config.from_buffer_copy(cfg)
        setattr(c2, field, bad)
        assert B.dec_workspace_bytes(c2) == 0, field
    assert lib.dec_verify2(None, None, None, None) == B.DEC_EINVAL


def test_host_side_argument_errors(lib):
    from weight_streaming_gemv_token_gb300 import binding as B

    # Each of these is rejected before any CUDA call.
    assert lib.gemv(7, None, None, None, 4, 4, None) == B.DEC_EINVAL
    assert lib.gemv(B.DEC_F32, None, None, None, -1, 4, None) == B.DEC_EINVAL
    assert lib.gemv(B.DEC_F32, None, None, None, 0, 4, None) == B.DEC_OK        # empty: no work
    assert lib.gemv(B.DEC_F32, None, None, None, 4, 4, None) == B.DEC_EINVAL    # NULL pointers
    assert "NULL" in B.dec_last_error(None)
    assert lib.gemv_q4(None, None, None, None, None, 4, 100, 1, None) == B.DEC_EINVAL  # in % 64
    assert lib.gemv_q4(None, None, None, None, None, 4, 128, 3, None) == B.DEC_EINVAL  # ntok
    assert lib.gemv_q4(None, None, None, None, None, 0, 128, 1, None) == B.DEC_OK
    assert lib.gemv_q4_rows_per_warp(1, 3) == -1
    assert lib.gemv_q4_rows_per_warp(3, 1) == -1
    assert lib.gemv_q4_rows_per_warp(1, -2) == -1
    # the setting is host state: set, read back, and return to the automatic choice
    assert lib.gemv_q4_rows_per_warp(2, 4) == 4
    assert lib.gemv_q4_rows_per_warp(2, 0) == 4
    assert lib.gemv_q4_rows_per_warp(2, -1) == 0
    assert lib.gemv_q4_rows_per_warp(2, 0) == 0
    h = ctypes.c_void_p()
    cfg = B.dec_config(layers=1, hidden=64, inter=64, n_q=2, n_kv=1, head_dim=16, vocab=10, eps=1e-6,
                       rope_theta=1e4, wdtype=0, kvdtype=0, max_seq=8, chunk_cap=0)
    assert lib.dec_create(ctypes.byref(cfg), None, 0, None, ctypes.byref(h)) == B.DEC_EINVAL
    assert lib.dec_create(ctypes.byref(cfg), ctypes.c_void_p(256), 16, None, ctypes.byref(h)) == B.DEC_ENOMEM
    assert lib.dec_create(ctypes.byref(cfg), ctypes.c_void_p(258), 1 << 30, None, ctypes.byref(h)) == B.DEC_EINVAL
    assert lib.dec_step(None, 0, 0, None, None) == B.DEC_EINVAL
    assert lib.dec_position(None) == -1
    assert lib.dec_reset(None) == B.DEC_EINVAL
    assert lib.dec_rewind(None, 0) == B.DEC_EINVAL
    bad = ctypes.c_int64(7)
    assert lib.pack_bf16_exact(None, None, -1, None, ctypes.byref(bad)) == B.DEC_EINVAL
    assert lib.pack_bf16_exact(None, None, 4, None, ctypes.byref(bad)) == B.DEC_EINVAL
    assert lib.pack_bf16_exact(None, None, 0, None, None) == B.DEC_EINVAL
    assert lib.pack_bf16_exact(None, None, 0, None, ctypes.byref(bad)) == B.DEC_OK and bad.value == 0


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    from weight_streaming_gemv_token_gb300 import binding as B
    from weight_streaming_gemv_token_gb300 import build as bld

    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(bld, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        B.library()


def test_device_error_bits_are_documented_once():
    """Every error bit a kernel can set has its own value and is declared in the header (and the binding)."""
    import glob

    from weight_streaming_gemv_token_gb300 import binding as B

    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    header = open(os.path.join(root, "include", "wsg.h")).read()
    public = {n: int(v, 16) for n, v in re.findall(r"#define (DEC_DEVERR_\w+) (0x[0-9a-fA-F]+)u", header)}
    internal = {}
    for f in glob.glob(os.path.join(root, "weight_streaming_gemv_token_gb300", "csrc", "*.cu*")):
        for n, k in re.findall(r"\b(ERR_\w+) = 1u << (\d+)", open(f).read()):
            internal[n] = 1 << int(k)
    assert len(set(internal.values())) == len(internal), internal
    assert sorted(internal.values()) == sorted(public.values()), (internal, public)
    for n, v in public.items():
        assert getattr(B, n) == v
