"""Derivation of the full-size tolerance of the 4-bit decoder tests (run by hand, not by pytest).

The 4-bit configuration rounds each projection's input vector to bfloat16. Whether an element
rounds up or down depends on its last bits, so two correct evaluations of the same forward that
differ only in the rounding of their float arithmetic can take different bfloat16 decisions, and
over 28 layers those decisions compound. This script measures that spread on the oracle alone:
the oracle against itself, with the activations perturbed by a relative amount `eps` (the size of
float32 arithmetic, or of the 4-bit kernel's 16-bit fixed-point x) before each rounding, at the
Qwen3-0.6B geometry with the seeded 4-bit weights of the tests.

    python tests/q4_tolerance_derivation.py 1e-7 1e-6 3e-5

prints, per eps, the largest and the rms logit difference and how many logits leave 2e-2. About
5 GB of host memory and a minute per eps.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle as O  # noqa: E402
import workloads as Wl  # noqa: E402


def dequantised(w):
    deq = lambda m: O.q4_dequant(m["packed"], m["scale"], m["bias"])  # noqa: E731
    return {"embed": deq(w["embed"]), "g_final": w["g_final"],
            "layers": [{k: (v if k.startswith("g_") else deq(v)) for k, v in lw.items()} for lw in w["layers"]]}


def main(eps_list):
    s = Wl.QWEN3_06B
    w = dequantised(Wl.decoder_weights_q4(s, seed=1))
    prompt = [int(t) for t in Wl.prompt_uniform(4, s.vocab, seed=0)]
    exact = O.OracleDecoder(s, w, max_seq=16, act_round="bf16")
    for t in prompt[:-1]:
        exact.body(t)
    ref = exact.step(prompt[-1])
    for eps in eps_list:
        rng = np.random.default_rng(0)
        pert = O.OracleDecoder(s, w, max_seq=16, act_round="bf16")
        # the same reading, each rounding decision taken on a slightly perturbed value
        pert._act = lambda x: O.round_to_bf16(np.asarray(x) * (1 + eps * rng.standard_normal(np.shape(x))))
        for t in prompt[:-1]:
            pert.body(t)
        got = pert.step(prompt[-1])
        d = np.abs(got - ref)
        print(f"eps {eps:g}: logit scale {ref.std():.3f}, max diff {d.max():.4f}, rms {np.sqrt(np.mean(d ** 2)):.4f}, "
              f"outside 2e-2: {int((d > 0.02 + 0.02 * np.abs(ref)).sum())}", flush=True)


if __name__ == "__main__":
    main([float(a) for a in sys.argv[1:]] or [1e-7, 1e-6, 3e-5])
