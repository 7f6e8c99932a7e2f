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
