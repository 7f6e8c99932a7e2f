"""Parity of gemv (float32 / bfloat16) and gemv_q4 with the oracle, through the C ABI."""
import numpy as np
import pytest

import oracle as O
import workloads as Wl

from gpu_util import FP32_TOL, LOW_TOL, accumulation_bound, close, dev, lib

pytestmark = pytest.mark.gpu

SMALL = [(1, 4), (7, 12), (153, 1028), (1000, 64), (33, 4100), (5, 3076), (300, 2048)]
UNALIGNED = [(9, 7), (17, 1023), (3, 1)]


def run_gemv(W, dtype, Wm, x):
    import torch

    out, inp = Wm.shape
    y = torch.full((out,), float("nan"), dtype=torch.float32, device="cuda")
    W.gemv(W.DEC_F32 if dtype == "f32" else W.DEC_BF16, dev(Wm), dev(x), y, out, inp, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert W.gemv_device_errors() == 0
    return y.cpu().numpy()


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SMALL + UNALIGNED)
def test_gemv_small_and_ragged(dtype, shape):
    W = lib()
    out, inp = shape
    Wm = Wl.gemv_matrix(out, inp, seed=out * 7 + inp, dtype=dtype)
    x = Wl.gemv_vector(inp, seed=inp + 1, dtype=dtype)
    y = run_gemv(W, dtype, Wm, x)
    ref = O.gemv(Wm, x)
    close(y, ref, FP32_TOL if dtype == "f32" else LOW_TOL, f"gemv {dtype} {shape}")
    assert np.all(np.abs(y - ref) <= accumulation_bound(Wm, x, inp))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", Wl.GEMV_SHAPES)
def test_gemv_full_shapes(dtype, shape):
    W = lib()
    out, inp = shape
    Wm = Wl.gemv_matrix(out, inp, seed=11, dtype=dtype)
    x = Wl.gemv_vector(inp, seed=12, dtype=dtype)
    y = run_gemv(W, dtype, Wm, x)
    ref = O.gemv(Wm, x)
    close(y, ref, FP32_TOL if dtype == "f32" else LOW_TOL, f"gemv {dtype} {shape}")
    assert np.all(np.abs(y - ref) <= accumulation_bound(Wm, x, inp))


# Shapes of the bulk-copy kernel (at least 16 rows and 96 KB of W per SM): ragged row
# counts per CTA and stage, a partial last pass of the row, 1, 2 and 4 rows per warp.
BULK = [("f32", (5000, 1000)), ("f32", (20003, 264)), ("bf16", (9000, 1000)), ("bf16", (60001, 256))]


@pytest.mark.parametrize("dtype,shape", BULK)
def test_gemv_bulk_shapes(dtype, shape):
    W = lib()
    out, inp = shape
    Wm = Wl.gemv_matrix(out, inp, seed=out + inp, dtype=dtype)
    x = Wl.gemv_vector(inp, seed=inp + 3, dtype=dtype)
    y = run_gemv(W, dtype, Wm, x)
    ref = O.gemv(Wm, x)
    close(y, ref, FP32_TOL if dtype == "f32" else LOW_TOL, f"gemv {dtype} {shape}")
    assert np.all(np.abs(y - ref) <= accumulation_bound(Wm, x, inp))


def test_gemv_edge_cases():
    import torch

    W = lib()
    # in == 0: y = 0
    y = torch.full((5,), 7.0, device="cuda")
    W.gemv(W.DEC_F32, 0, 0, y, 5, 0, None)
    torch.cuda.synchronize()
    assert torch.all(y == 0)
    # out == 0: nothing written, no error
    W.gemv(W.DEC_F32, 0, 0, y, 0, 16, None)
    # misaligned weight pointer takes the element-load path and stays exact to the bound
    Wm = Wl.gemv_matrix(40, 64, seed=3)
    x = Wl.gemv_vector(64, seed=4)
    buf = torch.zeros(40 * 64 + 1, dtype=torch.float32, device="cuda")
    buf[1:] = torch.from_numpy(Wm.ravel()).cuda()
    y = torch.empty(40, device="cuda")
    W.gemv(W.DEC_F32, buf.data_ptr() + 4, dev(x), y, 40, 64, None)
    torch.cuda.synchronize()
    close(y.cpu().numpy(), O.gemv(Wm, x), FP32_TOL, "misaligned")
    # bad dtype
    with pytest.raises(W.WsgError):
        W.gemv(5, buf, buf, y, 4, 4, None)


def test_gemv_is_deterministic_and_round_robin():
    """Back-to-back launches over distinct matrices (the cold-benchmark pattern) give each right answer, bit-stably."""
    import torch

    W = lib()
    out, inp = 4096, 1024
    mats = [Wl.gemv_matrix(out, inp, seed=100 + i) for i in range(4)]
    x = Wl.gemv_vector(inp, seed=5)
    dW = [dev(m) for m in mats]
    dx = dev(x)
    ys = [torch.empty(out, device="cuda") for _ in mats]
    for _ in range(3):
        for m, y in zip(dW, ys):
            W.gemv(W.DEC_F32, m, dx, y, out, inp, torch.cuda.current_stream())
    torch.cuda.synchronize()
    first = [y.clone() for y in ys]
    for m, y in zip(dW, ys):
        W.gemv(W.DEC_F32, m, dx, y, out, inp, torch.cuda.current_stream())
    torch.cuda.synchronize()
    for m, y, f in zip(mats, ys, first):
        close(y.cpu().numpy(), O.gemv(m, x), FP32_TOL, "round robin")
        assert torch.equal(y, f)


# ---- 4-bit groupwise affine ----

def run_q4(W, m, x, ntok):
    import torch

    out, inp = m["codes"].shape
    y = torch.full((ntok, out), float("nan"), dtype=torch.float32, device="cuda")
    W.gemv_q4(dev(m["packed"]), dev(m["scale"].view(np.uint16)), dev(m["bias"].view(np.uint16)),
              dev(x), y, out, inp, ntok, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert W.gemv_device_errors() == 0
    return y.cpu().numpy()


def q4_ref(m, x):
    return O.gemv_q4(m["packed"], m["scale"], m["bias"], x)


@pytest.mark.parametrize("ntok", [1, 2])
@pytest.mark.parametrize("shape", [(1, 64), (7, 128), (300, 192), (37, 1024), (1024, 3072), (999, 2048)])
@pytest.mark.parametrize("rows", [1, 2, 4, 8])
def test_gemv_q4_small(ntok, shape, rows):
    W = lib()
    prev = W.gemv_q4_rows_per_warp(ntok)
    W.gemv_q4_rows_per_warp(ntok, rows)
    try:
        out, inp = shape
        m = Wl.q4_matrix(out, inp, seed=out + inp)
        x = Wl.q4_activations(inp, ntok, seed=inp)
        y = run_q4(W, m, x, ntok)
        ref = q4_ref(m, x)
        close(y, ref, LOW_TOL, f"q4 {shape} ntok={ntok} R={rows}")
        # much tighter than the stated tolerance: the float32 error of a length-in dot
        wabs = np.abs(O.q4_dequant(m["packed"], m["scale"], m["bias"]))
        bound = 2e-5 * (np.abs(O.widen(x)) @ wabs.T) + 1e-6
        assert np.all(np.abs(y - ref) <= bound)
    finally:
        W.gemv_q4_rows_per_warp(ntok, prev if prev > 0 else -1)


@pytest.mark.parametrize("ntok", [1, 2])
@pytest.mark.parametrize("shape", Wl.GEMV_SHAPES)
def test_gemv_q4_full_shapes(ntok, shape):
    W = lib()
    out, inp = shape
    m = Wl.q4_matrix(out, inp, seed=21)
    x = Wl.q4_activations(inp, ntok, seed=22)
    y = run_q4(W, m, x, ntok)
    if out > 20000:  # sampled rows: the oracle dequantises only those
        rows = np.unique(np.concatenate([np.arange(64), np.random.default_rng(0).integers(0, out, 512), [out - 1]]))
        sub = {k: v[rows] for k, v in m.items()}
        close(y[:, rows], q4_ref(sub, x), LOW_TOL, f"q4 {shape} sampled")
    else:
        close(y, q4_ref(m, x), LOW_TOL, f"q4 {shape}")
