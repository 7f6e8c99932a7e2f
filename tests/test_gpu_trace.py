"""Stage tracing of the persistent engines (dec_trace_bytes / dec_set_trace).

The trace holds, for the first forward of a launch, one %globaltimer stamp per
CTA, layer and stage event. Checked: every CTA stamps every layer's QKV stage
entry, the stage's later events follow its entry, layers follow each other, the
head comes after the last layer; a buffer that is too small and the staged
engine are refused; with tracing off nothing is written.
"""
import numpy as np
import pytest

import workloads as Wl

from gpu_util import lib

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wd", ["f32", "q4"])
def test_persistent_stage_trace(wd):
    import torch

    W = lib()
    from weight_streaming_gemv_token_gb300 import binding as B
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    if wd == "q4":
        shape, w = Wl.Q4_SMALL, Wl.decoder_weights_q4(Wl.Q4_SMALL, seed=1)
    else:
        shape, w = Wl.TINY, Wl.decoder_weights(Wl.TINY, seed=1)
    dec = Decoder(shape, w, max_seq=32, engine="persistent")
    tok = dec.prefill([int(t) for t in Wl.prompt_uniform(5, shape.vocab, seed=2)], is_last=True)
    nb = W.dec_trace_bytes(dec.ctx)
    G = torch.cuda.get_device_properties(0).multi_processor_count
    L = shape.layers
    n_stage = G * (L + 1) * 5 * 4
    assert nb >= n_stage * 8
    with pytest.raises(W.WsgError) as e:
        W.dec_set_trace(dec.ctx, torch.zeros(8, dtype=torch.int64, device="cuda"), 64)
    assert e.value.status == B.DEC_EINVAL
    buf = torch.zeros(nb // 8, dtype=torch.int64, device="cuda")
    W.dec_set_trace(dec.ctx, buf, nb)
    out = dec.generate(tok, 2)
    torch.cuda.synchronize()
    tr = buf.cpu().numpy()[:n_stage].reshape(G, L + 1, 5, 4).astype(np.int64)
    entry = tr[:, :L, 0, 0]
    assert (entry > 0).all(), "a CTA did not stamp a layer's QKV stage entry"
    # within a CTA: layers in order, and a layer's QKV inputs staged and its outputs published (or,
    # in the 4-bit engine, its products done) after the stage's entry
    assert (np.diff(entry, axis=1) > 0).all()
    qkv = tr[:, :L, 0, :]
    later = qkv[..., 1:3]
    assert ((later == 0) | (later >= qkv[..., :1])).all()
    # the head's vocabulary stage entry comes after the CTA's last layer
    head = tr[:, L, 0, 0]
    assert (head > entry[:, -1]).all()
    # tracing off: a new launch writes nothing
    W.dec_set_trace(dec.ctx, None, 0)
    buf.zero_()
    dec.generate(int(out[-1].item()), 2)
    torch.cuda.synchronize()
    assert int(buf.abs().sum().item()) == 0
    assert dec.device_errors() == 0
    dec.close()


def test_staged_engine_has_no_trace():
    import torch

    W = lib()
    from weight_streaming_gemv_token_gb300 import binding as B
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    dec = Decoder(Wl.TINY, Wl.decoder_weights(Wl.TINY, seed=1), max_seq=16, engine="staged")
    assert W.dec_trace_bytes(dec.ctx) == 0
    with pytest.raises(W.WsgError) as e:
        W.dec_set_trace(dec.ctx, torch.zeros(1024, dtype=torch.int64, device="cuda"), 8192)
    assert e.value.status == B.DEC_EINVAL
    dec.close()
