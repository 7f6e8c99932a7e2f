"""The greedy argmax rule on the GPU, through every decoder head.

"Megakernels", "GPU-wide end-to-end generation": the GPU argmax picks the lowest
token ID among equal maxima. The design notes add: NaN never wins, -0 == +0,
and an all-NaN logit vector returns token 0 and sets DEC_DEVERR_ARGMAX_NAN.

Random logits never tie, so the decoder tests elsewhere cannot see this rule.
Here the tied embedding carries planted columns (tests/argmax_cases.py): with
the final-norm gain zero except in one column, each logit is exactly one
product, so equal planted entries tie bit for bit in any summation order. The
model is 2 layers wide 512 with the full 151,936-token vocabulary, so the head
spans every CTA of the GPU. Each case rewinds to the last prompt position and
repeats its forward with that case's gain; the expected token comes from the
planted pattern and the oracle's sign of the final residual in that column.
"""
import numpy as np
import pytest

import oracle as O
import workloads as Wl

import argmax_cases as AC
from gpu_util import lib

pytestmark = pytest.mark.gpu

SHAPE = Wl.DecoderShape(layers=2, hidden=512, inter=1024, n_q=4, n_kv=2, head_dim=128, vocab=AC.VOCAB)
PROMPT = [11, 12345, 54321, 777]
DEVERR_ARGMAX_NAN = 0x2


def _dequantised(w):
    deq = lambda m: O.q4_dequant(m["packed"], m["scale"], m["bias"])  # noqa: E731
    return {"embed": deq(w["embed"]), "g_final": w["g_final"],
            "layers": [{k: (v if k.startswith("g_") else deq(v)) for k, v in lw.items()} for lw in w["layers"]]}


def planted_model(wd):
    """(weights with the planted embedding, the oracle's final residual after the prompt)."""
    if wd == "q4":
        w = Wl.decoder_weights_q4(SHAPE, seed=1)
        w["embed"] = AC.plant_q4(w["embed"])
        ow = _dequantised(w)
    else:
        w = Wl.decoder_weights(SHAPE, seed=1, wdtype=wd)
        E = AC.plant_float(w["embed"] if wd == "f32" else Wl.bf16_bits_to_f32(w["embed"]))
        w["embed"] = E if wd == "f32" else Wl.f32_to_bf16_bits(E)
        ow = w
    assert not AC.fed_rows() & set(PROMPT)
    ora = O.OracleDecoder(SHAPE, ow, max_seq=8)
    for t in PROMPT:
        h = ora.body(t)
    return w, h


@pytest.fixture(scope="module", params=["f32", "bf16", "q4"])
def planted(request):
    return request.param, planted_model(request.param)


def check_case(got, tok, errs, kind, rows, what):
    exp, all_nan = AC.expected(kind, rows)
    assert tok == exp, f"{what}: token {tok}, the rule gives {exp}"
    own, ok = O.argmax_lowest(got)
    assert own == tok and ok == (not all_nan), f"{what}: token {tok} vs argmax of its own logits {own}"
    if all_nan:
        assert np.isnan(got).all(), f"{what}: not every logit is NaN"
        assert errs & DEVERR_ARGMAX_NAN, f"{what}: all-NaN logits did not set DEC_DEVERR_ARGMAX_NAN"
        return
    assert errs == 0, f"{what}: device errors {errs:#x}"
    assert np.isnan(got[list(AC.NAN_ROWS)]).all(), f"{what}: NaN rows are not NaN"
    top = np.nanmax(got)
    vals = got[list(rows)]
    if kind == "tie":
        assert (vals == top).all(), f"{what}: planted rows {vals} are not all the maximum {top}"
    else:  # signed zeros: the planted rows hold the maximum, zero (either sign)
        assert top == 0.0 and (vals == 0.0).all(), f"{what}: planted zero rows {vals}, maximum {top}"


@pytest.mark.parametrize("engine", ["persistent", "staged"])
def test_decoder_head_argmax_rule(planted, engine):
    import torch

    lib()
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    wd, (w, h) = planted
    rms = float(np.sqrt(np.mean(h ** 2)))
    dec = Decoder(SHAPE, w, max_seq=8, engine=engine)
    for t in PROMPT[:-1]:
        dec.step(t, skip_logits=True)
    logits = torch.empty(SHAPE.vocab, dtype=torch.float32, device="cuda")
    for name, col, kind, rows in AC.CASES:
        assert abs(h[col]) > 0.1 * rms, f"{name}: the oracle's residual in column {col} is too small to sign"
        dec.dev["g_final"].copy_(torch.from_numpy(AC.gain_for(col, SHAPE.hidden, h[col], kind)))
        dec.rewind(len(PROMPT) - 1)
        logits.fill_(-1.0)
        tok = dec.step(PROMPT[-1], logits=logits)
        got = logits.cpu().numpy()
        errs = dec.device_errors(clear=True)
        check_case(got, tok, errs, kind, rows, f"{wd} {engine} {name}")
    dec.close()
