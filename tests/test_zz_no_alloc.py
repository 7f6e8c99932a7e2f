"""greedy_head_noalloc: the greedy head with library-held scratch, for callers that cannot allocate.

Some callers cannot call cudaMalloc: code inside a host framework that owns every
device allocation, or a generation loop that must not risk the device
synchronisation an allocation can cause. This entry point keeps its scratch in a
fixed array inside the library. Checked here through the C ABI:

* against the oracle (x = RMSNorm(h) * gain, logits = E x in float64) on two
  calls in a row with different inputs, which also checks that the shared
  scratch is reset between calls; and against the existing gemv entry point;
* that a call changes the device's free memory by nothing;
* the lowest-ID argmax rule on planted ties, signed zeros and NaN rows, and
  that an all-NaN head returns token 0 and sets DEC_DEVERR_ARGMAX_NAN in the
  error word gemv_device_errors reads.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest

import oracle as O
import workloads as Wl

import argmax_cases as AC
from gpu_util import FP32_TOL, close, dev, lib

pytestmark = pytest.mark.gpu

DEVERR_ARGMAX_NAN = 0x2


def _call(W, code, dE, h, gain, vocab, hidden, logits, token):
    import torch

    W.greedy_head_noalloc(code, dE, dev(h), dev(gain), 1e-6, vocab, hidden, logits, token,
                          torch.cuda.current_stream())
    torch.cuda.synchronize()
    return logits.cpu().numpy(), int(token.item())


@pytest.mark.parametrize("dtype,vocab,hidden", [("f32", 151936, 1024), ("bf16", 151936, 1024), ("f32", 777, 96)])
def test_greedy_head_noalloc_matches_oracle(dtype, vocab, hidden):
    import torch

    W = lib()
    code = W.DEC_F32 if dtype == "f32" else W.DEC_BF16
    E = Wl.gemv_matrix(vocab, hidden, seed=vocab + hidden, dtype=dtype)
    dE = dev(E)
    W.gemv_device_errors(True)
    for call in range(2):
        h = Wl.gemv_vector(hidden, seed=100 + call, scale=1.0)
        gain = (1.0 + 0.1 * np.random.default_rng(200 + call).standard_normal(hidden)).astype(np.float32)
        logits = torch.full((vocab,), float("nan"), device="cuda")
        token = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        got, t = _call(W, code, dE, h, gain, vocab, hidden, logits, token)
        # the oracle: float64 RMSNorm and product on the same stored values
        want = O.gemv(E, O.rmsnorm(h, gain, 1e-6))
        close(got, want, FP32_TOL, f"logits vs oracle, call {call}")
        assert t == O.argmax_lowest(got)[0], "token is not the argmax of the call's own logits"
        srt = np.sort(want)[::-1]
        if srt[0] - srt[1] > 2 * (FP32_TOL + FP32_TOL * abs(srt[0])):
            assert t == O.argmax_lowest(want)[0], f"call {call}: token {t} vs oracle {O.argmax_lowest(want)[0]}"
        # the existing entry point on the same x (float32 weights widened exactly from bf16)
        x = O.rmsnorm(h, gain, 1e-6).astype(np.float32)
        ref = torch.empty(vocab, device="cuda")
        Ef = E if dtype == "f32" else Wl.bf16_bits_to_f32(E)
        W.gemv(W.DEC_F32, dev(Ef), dev(x), ref, vocab, hidden, None)
        torch.cuda.synchronize()
        close(got, ref.cpu().numpy(), FP32_TOL, f"logits vs gemv, call {call}")
    assert W.gemv_device_errors(True) == 0


def test_greedy_head_noalloc_allocates_nothing():
    import torch

    W = lib()
    vocab, hidden = 151936, 1024
    dE = dev(Wl.gemv_matrix(vocab, hidden, seed=5))
    h = dev(Wl.gemv_vector(hidden, seed=6, scale=1.0))
    gain = dev(np.ones(hidden, dtype=np.float32))
    logits = torch.empty(vocab, device="cuda")
    token = torch.empty(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    W.greedy_head_noalloc(W.DEC_F32, dE, h, gain, 1e-6, vocab, hidden, logits, token, stream)  # set-up call
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        W.greedy_head_noalloc(W.DEC_F32, dE, h, gain, 1e-6, vocab, hidden, logits, token, stream)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "free device memory changed across calls"


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_greedy_head_noalloc_argmax_rule(dtype):
    import torch

    W = lib()
    code = W.DEC_F32 if dtype == "f32" else W.DEC_BF16
    vocab, hidden = AC.VOCAB, 512
    E = AC.plant_float(Wl.gemv_matrix(vocab, hidden, seed=7))
    dE = dev(E if dtype == "f32" else Wl.f32_to_bf16_bits(E))
    h = Wl.gemv_vector(hidden, seed=8, scale=1.0)
    logits = torch.empty(vocab, device="cuda")
    token = torch.empty(1, dtype=torch.int32, device="cuda")
    W.gemv_device_errors(True)
    for name, col, kind, rows in AC.CASES:
        gain = AC.gain_for(col, hidden, float(h[col]), kind)
        logits.fill_(-1.0)
        got, t = _call(W, code, dE, h, gain, vocab, hidden, logits, token)
        errs = W.gemv_device_errors(True)
        exp, all_nan = AC.expected(kind, rows)
        assert t == exp, f"{name}: token {t}, the rule gives {exp}"
        assert O.argmax_lowest(got)[0] == t
        if all_nan:
            assert np.isnan(got).all() and errs & DEVERR_ARGMAX_NAN, f"{name}: errors {errs:#x}"
        else:
            assert errs == 0, f"{name}: device errors {errs:#x}"
            assert np.isnan(got[list(AC.NAN_ROWS)]).all()
            assert (got[list(rows)] == np.nanmax(got)).all()


def test_greedy_head_noalloc_rejects_bad_sizes():
    import torch

    W = lib()
    from weight_streaming_gemv_token_gb300 import binding as B

    buf = torch.zeros(64, device="cuda")
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(W.WsgError) as e:
        B.greedy_head_noalloc(W.DEC_F32, buf, buf, buf, 1e-6, 10, 3, None, tok)  # rows of 12 bytes
    assert e.value.status == B.DEC_EINVAL
    with pytest.raises(W.WsgError):
        B.greedy_head_noalloc(W.DEC_F32, buf, buf, buf, 1e-6, 0, 16, None, tok)
    with pytest.raises(W.WsgError) as e:
        B.greedy_head_noalloc(W.DEC_F32, buf, buf, buf, 1e-6, 4, 1 << 20, None, tok)  # staging too large
    assert e.value.status == B.DEC_EINVAL
