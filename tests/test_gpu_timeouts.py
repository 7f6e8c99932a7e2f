"""The give-up path of the persistent engines' bounded waits, on the GPU.

Every wait of a persistent kernel on another CTA's results is bounded; when one
runs out the kernel records the cause in the device error word, waits for its
own copies in flight and returns, so the context stays usable. Here the limit is
set to 1 ns (dec_set_wait_limit), so any wait that is not already satisfied
gives up at once: the forward must end, the error bit must be set, dec_reset
must clear it, and after the default limit is restored the same context must
reproduce, bit for bit, what a fresh context computes.
"""
import numpy as np
import pytest

import workloads as Wl

from gpu_util import lib

pytestmark = pytest.mark.gpu

DEVERR_EXCHANGE_TIMEOUT = 0x10
DEVERR_BARRIER_TIMEOUT = 0x40


def _run(dec, prompt, n, vocab):
    import torch

    logits = torch.empty(vocab, dtype=torch.float32, device="cuda")
    dec.reset()
    tok = dec.prefill(prompt, is_last=True, logits=logits)
    out, rows = [tok], [logits.cpu().numpy().copy()]
    for _ in range(n):
        tok = dec.step(tok, logits=logits)
        out.append(tok)
        rows.append(logits.cpu().numpy().copy())
    return out, rows


@pytest.mark.parametrize("wd", ["f32", "q4"])
def test_persistent_wait_gives_up_and_context_recovers(wd):
    lib()
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    if wd == "q4":
        shape, w, bit = Wl.Q4_SMALL, Wl.decoder_weights_q4(Wl.Q4_SMALL, seed=1), DEVERR_BARRIER_TIMEOUT
    else:
        shape, w, bit = Wl.TINY, Wl.decoder_weights(Wl.TINY, seed=1), DEVERR_EXCHANGE_TIMEOUT
    prompt = [int(t) for t in Wl.prompt_uniform(6, shape.vocab, seed=4)]
    ref = Decoder(shape, w, max_seq=32, engine="persistent")
    want_tok, want_logits = _run(ref, prompt, 4, shape.vocab)
    assert ref.device_errors() == 0
    ref.close()

    dec = Decoder(shape, w, max_seq=32, engine="persistent")
    dec.prefill(prompt[:-1], is_last=False)
    assert dec.device_errors() == 0
    dec.set_wait_limit(1)
    dec.step(prompt[-1])  # returns once the launch has given up; its token is undefined
    errs = dec.device_errors(clear=False)
    assert errs & bit, f"device errors {errs:#x}: the timeout bit {bit:#x} is not set"
    dec.set_wait_limit(0)
    dec.reset()
    assert dec.device_errors(clear=False) == 0, "dec_reset did not clear the device error word"
    got_tok, got_logits = _run(dec, prompt, 4, shape.vocab)
    assert got_tok == want_tok
    for j, (a, b) in enumerate(zip(got_logits, want_logits)):
        assert np.array_equal(a, b), f"logits of output {j} differ from a fresh context's"
    assert dec.device_errors() == 0
    dec.close()
