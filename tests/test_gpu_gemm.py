"""Parity of the tensor-core projection GEMM (gemm_bf16) with the oracle's
chunk projection, through the C ABI: ragged and full tiles, accumulate mode,
the Qwen3-0.6B chunked-prefill shapes."""
import numpy as np
import pytest

import oracle as O
import workloads as Wl

from gpu_util import dev, lib

pytestmark = pytest.mark.gpu

# (M, N, K): single elements, ragged M/N/K, several tiles, and the projections of
# a 512-row chunk of the Qwen3-0.6B shape (QKV, O, gate/up, down). The tile
# width is planned per launch: the small products run 64-column tiles, the
# 512-row QKV shape 128-column ones, and the last three 256-column tiles (the
# gate/up product of a 1024-row chunk, then ragged M, N and K twice).
SHAPES = [(1, 1, 8), (3, 5, 16), (128, 128, 64), (129, 130, 72), (200, 300, 96), (257, 64, 1024),
          (512, 4096, 1024), (512, 1024, 2048), (300, 3072, 1024), (384, 1024, 3072),
          (1024, 6144, 1024), (1100, 2500, 200), (1900, 3000, 264)]


def bf16_matrix(rows, cols, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return Wl.f32_to_bf16_bits((scale * rng.standard_normal((rows, cols))).astype(np.float32))


def bound(A, W, K):
    """FP32 accumulation of K exact products: 2 K u sum |a w| (u = 2^-24)."""
    return 2.0 * K * 2.0 ** -24 * (np.abs(O.widen(A)) @ np.abs(O.widen(W)).T) + 1e-30


def run(W_, A, Wm, M, N, K, ldc=None, init=None, accumulate=False):
    import torch

    ldc = ldc or N
    C = torch.full((M, ldc), float("nan"), dtype=torch.float32, device="cuda") if init is None else dev(init)
    W_.gemm_bf16(dev(A), dev(Wm), C, M, N, K, ldc=ldc, accumulate=accumulate, stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert W_.gemv_device_errors() == 0
    return C.cpu().numpy()


@pytest.mark.parametrize("shape", SHAPES)
def test_gemm_matches_oracle(shape):
    W_ = lib()
    M, N, K = shape
    A = bf16_matrix(M, K, 11, 1.0)
    Wm = bf16_matrix(N, K, 12, 0.02)
    got = run(W_, A, Wm, M, N, K)
    ref = O.project_rows(A, Wm)
    err = np.abs(got - ref)
    assert np.all(err <= bound(A, Wm, K)), (shape, float(err.max()))


def test_gemm_accumulate_and_column_stride():
    """accumulate adds onto C; only columns < N of rows < M are written."""
    W_ = lib()
    M, N, K, ldc = 150, 200, 128, 256
    A = bf16_matrix(M, K, 21)
    Wm = bf16_matrix(N, K, 22, 0.02)
    rng = np.random.default_rng(23)
    init = rng.standard_normal((M, ldc)).astype(np.float32)
    got = run(W_, A, Wm, M, N, K, ldc=ldc, init=init, accumulate=True)
    ref = init[:, :N].astype(np.float64) + O.project_rows(A, Wm)
    assert np.all(np.abs(got[:, :N] - ref) <= bound(A, Wm, K) + 2.0 ** -23 * np.abs(ref))
    np.testing.assert_array_equal(got[:, N:], init[:, N:])


def test_gemm_accumulate_wide_tiles():
    """accumulate with 256-column tiles (1100 x 2500 x 200) and a row stride past N."""
    W_ = lib()
    M, N, K, ldc = 1100, 2500, 200, 2504
    A = bf16_matrix(M, K, 31)
    Wm = bf16_matrix(N, K, 32, 0.02)
    rng = np.random.default_rng(33)
    init = rng.standard_normal((M, ldc)).astype(np.float32)
    got = run(W_, A, Wm, M, N, K, ldc=ldc, init=init, accumulate=True)
    ref = init[:, :N].astype(np.float64) + O.project_rows(A, Wm)
    assert np.all(np.abs(got[:, :N] - ref) <= bound(A, Wm, K) + 2.0 ** -23 * np.abs(ref))
    np.testing.assert_array_equal(got[:, N:], init[:, N:])


def test_gemm_rejects_bad_arguments():
    import torch

    W_ = lib()
    A = torch.zeros((4, 8), dtype=torch.int16, device="cuda")
    C = torch.zeros((4, 4), dtype=torch.float32, device="cuda")
    for args in [(4, 4, 7), (0, 4, 8), (4, 4, 8, 3)]:
        with pytest.raises(W_.WsgError):
            M, N, K = args[:3]
            W_.gemm_bf16(A, A, C, M, N, K, ldc=args[3] if len(args) > 3 else None)
