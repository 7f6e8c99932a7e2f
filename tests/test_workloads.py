"""Seeded inputs: the float32 model converted from bfloat16 (lossless-storage workload)."""
import numpy as np

import workloads as Wl


def test_f32_from_bf16_is_the_bf16_model_widened():
    a = Wl.decoder_weights(Wl.TINY, seed=1, wdtype="f32_from_bf16")
    b = Wl.decoder_weights(Wl.TINY, seed=1, wdtype="bf16")
    assert a["wdtype"] == "f32" and a["embed"].dtype == np.float32
    assert np.array_equal(Wl.bf16_bits_to_f32(b["embed"]), a["embed"])
    for la, lb in zip(a["layers"], b["layers"]):
        for k in Wl.LAYER_TENSORS:
            if k.startswith("g_"):
                assert np.array_equal(la[k], lb[k])  # gains stay float32 draws
            else:
                assert np.array_equal(Wl.bf16_bits_to_f32(lb[k]), la[k])
                assert np.all((la[k].view(np.uint32) & 0xFFFF) == 0)
    # the plain float32 draws are not bfloat16 values
    c = Wl.decoder_weights(Wl.TINY, seed=1, wdtype="f32")
    assert np.any((c["embed"].view(np.uint32) & 0xFFFF) != 0)


def test_q4_decoder_weights_layout_and_spread():
    import workloads as Wl

    s = Wl.Q4_SMALL
    a = Wl.decoder_weights_q4(s, seed=1)
    b = Wl.decoder_weights_q4(s, seed=1)
    assert a["wdtype"] == "q4"
    shp = Wl.tensor_shapes(s)
    for name, m in [("embed", a["embed"])] + [(k, v) for k, v in a["layers"][0].items()]:
        if name.startswith("g_"):
            assert m.dtype == np.float32 and m.shape == shp[name]
            continue
        out, inp = shp[name]
        assert m["packed"].dtype == np.uint32 and m["packed"].shape == (out, inp // 8)
        assert m["scale"].dtype == np.float16 and m["scale"].shape == (out, inp // 64)
        assert m["bias"].dtype == np.float16 and m["bias"].shape == (out, inp // 64)
    np.testing.assert_array_equal(a["layers"][1]["w_down"]["packed"], b["layers"][1]["w_down"]["packed"])
    # w = s q + b: centred near zero, spread near that of the 0.02 N(0, 1) float draws
    from oracle import q4_dequant

    m = a["layers"][0]["w_gate"]
    wq = q4_dequant(m["packed"], m["scale"], m["bias"])
    assert abs(wq.mean()) < 2e-3 and 0.015 < wq.std() < 0.035


def test_q4_weight_buffer_layout_matches_the_abi():
    """A 4-bit matrix buffer is its codes [out][in/8] (uint32, code j of word w at bits 4j..4j+3 for
    column 8w+j), then the scales and then the biases [out][in/64] (fp16), back to back."""
    pytest = __import__("pytest")
    pytest.importorskip("torch")
    import workloads as Wl
    from weight_streaming_gemv_token_gb300.decoder import q4_blob

    out, inp = 24, 512
    m = Wl.decoder_weights_q4(Wl.DecoderShape(layers=1, hidden=inp, inter=inp, n_q=4, n_kv=2, head_dim=128,
                                              vocab=out), seed=3)["embed"]
    b = q4_blob(m, device="cpu").numpy()
    cb, sb = out * inp // 2, out * (inp // 64) * 2
    assert b.dtype == np.uint8 and b.size == cb + 2 * sb
    words = b[:cb].view(np.uint32).reshape(out, inp // 8)
    np.testing.assert_array_equal(words, m["packed"])
    np.testing.assert_array_equal(b[cb:cb + sb].view(np.float16).reshape(out, inp // 64), m["scale"])
    np.testing.assert_array_equal(b[cb + sb:].view(np.float16).reshape(out, inp // 64), m["bias"])
    # code j of word w is column 8w + j (low nibble first)
    from oracle import q4_unpack

    codes = q4_unpack(words)
    assert int(codes[0, 9]) == (int(words[0, 1]) >> 4) & 0xF
    # every section starts on a 16-byte boundary (bulk copies need it) when in % 512 == 0
    assert cb % 16 == 0 and sb % 16 == 0
