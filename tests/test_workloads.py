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
