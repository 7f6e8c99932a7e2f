"""Lossless bfloat16 storage of float32 weights ("Megakernels", "Lossless decode-weight storage"),
through the C ABI: the packing check, and the packed decoder against the float32 oracle."""
import numpy as np
import pytest

import oracle as O
import workloads as Wl

from gpu_util import FP32_TOL, close, lib

pytestmark = pytest.mark.gpu


def test_pack_counts_inexact_values():
    import torch

    W = lib()
    vals = np.array([0.0, -0.0, 1.0, -2.5, 3.0517578125e-05, 1.0 + 2.0**-10, 0.1, np.inf, -np.inf, np.nan, 1e-40,
                     2.0**-133], dtype=np.float32)
    exact = (vals.view(np.uint32) & 0xFFFF) == 0
    exact &= np.isfinite(vals)
    src = torch.from_numpy(vals).cuda()
    dst = torch.empty(len(vals), dtype=torch.bfloat16, device="cuda")
    bad = W.pack_bf16_exact(src, dst, len(vals), torch.cuda.current_stream())
    assert bad == int((~exact).sum())
    hi = (vals.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(dst.view(torch.int16).cpu().numpy().view(np.uint16), hi)
    # a large exact array (many CTAs): zero inexact, bit-exact halves
    big = Wl.bf16_bits_to_f32(Wl.f32_to_bf16_bits(np.random.default_rng(3).standard_normal(1 << 20).astype(np.float32)))
    src = torch.from_numpy(big).cuda()
    dst = torch.empty(big.size, dtype=torch.bfloat16, device="cuda")
    assert W.pack_bf16_exact(src, dst, big.size, None) == 0
    assert torch.equal(dst.float(), src)


@pytest.mark.parametrize("engine", ["persistent", "staged"])
def test_packed_decoder_matches_the_float32_oracle(engine):
    import torch

    from weight_streaming_gemv_token_gb300.decoder import Decoder

    s = Wl.TINY
    w = Wl.decoder_weights(s, seed=1, wdtype="f32_from_bf16")
    prompt = [int(t) for t in Wl.prompt_uniform(8, s.vocab, seed=0)]
    dec = Decoder(s, w, kv_dtype="f32", max_seq=24, engine=engine, lossless=True)
    assert dec.lossless and dec.dev["embed"].dtype == torch.bfloat16
    ora = O.OracleDecoder(s, w, kv_dtype="f32", max_seq=24)
    logits = torch.empty(s.vocab, device="cuda")
    for t in prompt[:-1]:
        dec.step(t, skip_logits=True)
        ora.body(t)
    cur = prompt[-1]
    for j in range(8):
        nxt = dec.step(cur, logits=logits)
        ref = ora.step(cur)
        got = logits.cpu().numpy()
        close(got, ref, FP32_TOL, f"packed logits step {j}")
        assert nxt == O.argmax_lowest(got)[0]
        cur = nxt
    for l in range(s.layers):
        K, V, n = dec.kv(l)
        rk, rv = ora.kv(l)
        close(K[:, :n].cpu().numpy(), rk, FP32_TOL, f"K layer {l}")
        close(V[:, :n].cpu().numpy(), rv, FP32_TOL, f"V layer {l}")
    assert dec.device_errors() == 0
    dec.close()


def test_inexact_weights_stay_float32():
    import torch

    from weight_streaming_gemv_token_gb300.decoder import Decoder

    s = Wl.TINY
    w = Wl.decoder_weights(s, seed=1, wdtype="f32")
    dec = Decoder(s, w, kv_dtype="f32", max_seq=8, lossless=True)
    assert not dec.lossless and dec.dev["embed"].dtype == torch.float32
    ora = O.OracleDecoder(s, w, kv_dtype="f32", max_seq=8)
    logits = torch.empty(s.vocab, device="cuda")
    dec.step(5, logits=logits)
    close(logits.cpu().numpy(), ora.step(5), FP32_TOL, "unpacked")
    dec.close()
