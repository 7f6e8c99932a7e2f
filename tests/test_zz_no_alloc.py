"""greedy_head_noalloc: the greedy head with library-held scratch, for callers that cannot allocate.

Checked against the existing gemv entry point on the same inputs: logits =
gemv(E, RMSNorm(h) * gain) within the float32 tolerance, and the token equal
to the lowest-ID argmax of those logits (unless the top two are within the
tolerance band). Two calls in a row, with different inputs, check that the
shared scratch is reset between calls. This file is collected last on purpose.
"""
import numpy as np
import pytest

import oracle as O
import workloads as Wl

from gpu_util import FP32_TOL, LOW_TOL, close, dev, lib

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,vocab,hidden", [("f32", 151936, 1024), ("bf16", 151936, 1024), ("f32", 777, 96)])
def test_greedy_head_noalloc_matches_gemv(dtype, vocab, hidden):
    import torch

    W = lib()
    code = W.DEC_F32 if dtype == "f32" else W.DEC_BF16
    tol = FP32_TOL if dtype == "f32" else LOW_TOL
    E = Wl.gemv_matrix(vocab, hidden, seed=vocab + hidden, dtype=dtype)
    dE = dev(E)
    for call in range(2):
        h = Wl.gemv_vector(hidden, seed=100 + call, scale=1.0)
        gain = (1.0 + 0.1 * np.random.default_rng(200 + call).standard_normal(hidden)).astype(np.float32)
        logits = torch.full((vocab,), float("nan"), device="cuda")
        token = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        W.greedy_head_noalloc(code, dE, dev(h), dev(gain), 1e-6, vocab, hidden, logits, token,
                              torch.cuda.current_stream())
        # the same head through the existing entry point: x on the host, logits by gemv
        x = O.rmsnorm(h, gain, 1e-6).astype(np.float32)
        ref = torch.empty(vocab, device="cuda")
        # gemv's bf16 form takes bf16 x, so the bf16 head (float32 x) is compared with
        # gemv on float32 weights widened exactly from the same bf16 values
        Ef = E if dtype == "f32" else Wl.bf16_bits_to_f32(E)
        W.gemv(W.DEC_F32, dev(Ef), dev(x), ref, vocab, hidden, None)
        torch.cuda.synchronize()
        got, want = logits.cpu().numpy(), ref.cpu().numpy()
        close(got, want, tol, f"logits, call {call}")
        t = int(token.item())
        assert t == O.argmax_lowest(got)[0], "token is not the argmax of the call's own logits"
        srt = np.sort(want.astype(np.float64))[::-1]
        if srt[0] - srt[1] > 2 * (tol + tol * abs(srt[0])):
            assert t == O.argmax_lowest(want)[0], f"call {call}: token {t} vs gemv argmax {O.argmax_lowest(want)[0]}"


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
    with pytest.raises(W.WsgError):
        B.greedy_head_noalloc(W.DEC_F32, buf, buf, buf, 1e-6, 4, 1 << 20, None, tok)  # staging too large
