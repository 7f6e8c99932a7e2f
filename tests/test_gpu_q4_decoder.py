"""The 4-bit configuration: every projection and the tied head on the 4-bit
matrix-vector product, and its two-token verify step, against the oracle.

The oracle is the float64 forward on the exact dequantised weights s * q + b;
the decoder's activations stay float32 (the 4-bit products take them in 16-bit
fixed point per 32 columns, not rounded to a 16-bit float). Tolerance: the
4-bit one, rtol = atol = 2e-2, at every size; tokens by the same near-tie rule
as the float decoders.
"""
import numpy as np
import pytest

import oracle as O
import workloads as Wl

from gpu_util import LOW_TOL, close, lib
from test_gpu_decoder import kv_to_np, run_and_compare


pytestmark = pytest.mark.gpu


def dequantised(w):
    """The oracle's view of a 4-bit model: float64 matrices s * q + b."""
    deq = lambda m: O.q4_dequant(m["packed"], m["scale"], m["bias"])  # noqa: E731
    return {"embed": deq(w["embed"]), "g_final": w["g_final"],
            "layers": [{k: (v if k.startswith("g_") else deq(v)) for k, v in lw.items()} for lw in w["layers"]]}


@pytest.fixture(scope="module")
def small_q4():
    w = Wl.decoder_weights_q4(Wl.Q4_SMALL, seed=1)
    return w, dequantised(w)


ENGINES = ["staged", "persistent"]


@pytest.mark.parametrize("engine", ENGINES)
@pytest.mark.parametrize("kv", ["f32", "bf16"])
def test_small_q4_every_logit_and_kv(small_q4, kv, engine):
    w, deq = small_q4
    prompt = Wl.prompt_uniform(9, Wl.Q4_SMALL.vocab, seed=3)
    run_and_compare(Wl.Q4_SMALL, w, prompt, 12, kv, LOW_TOL, engine=engine, oracle_weights=deq)


@pytest.mark.parametrize("engine", ENGINES)
def test_q4_generate_and_prefill_match_steps(small_q4, engine):
    """One call running many forwards (dec_generate, a tokenwise prompt) gives the tokens, logits and
    cache of the same forwards run one dec_step each, bit for bit."""
    import torch

    lib()
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    w, _ = small_q4
    s = Wl.Q4_SMALL
    prompt = [int(t) for t in Wl.prompt_uniform(7, s.vocab, seed=9)]
    a = Decoder(s, w, max_seq=40, engine=engine)
    b = Decoder(s, w, max_seq=40, engine=engine)
    first = a.prefill(prompt, is_last=True)
    for t in prompt[:-1]:
        b.step(t, skip_logits=True)
    assert b.step(prompt[-1]) == first
    out = a.generate(first, 9).cpu().tolist()
    cur, ref = first, []
    for _ in range(9):
        cur = b.step(cur)
        ref.append(cur)
    assert out == ref
    la = torch.empty(s.vocab, device="cuda")
    lb = torch.empty(s.vocab, device="cuda")
    a.step(out[-1], logits=la)
    b.step(out[-1], logits=lb)
    assert torch.equal(la, lb)
    for l in range(s.layers):
        ka, va, na = a.kv(l)
        kb, vb, nb = b.kv(l)
        assert na == nb and torch.equal(ka[:, :na], kb[:, :nb]) and torch.equal(va[:, :na], vb[:, :nb])
    assert a.device_errors() == 0 and b.device_errors() == 0
    a.close()
    b.close()


def check_verify(shape, w, deq, prompt, drafts, kv="f32", tol=LOW_TOL, engine="staged"):
    """Prompt tokenwise, then verify steps of (current token, draft) pairs; every row's logits
    against the oracle's forward of the same rows, the cache after each, and the token rule."""
    import torch

    lib()
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    max_seq = len(prompt) + 2 * len(drafts) + 4
    dec = Decoder(shape, w, kv_dtype=kv, max_seq=max_seq, engine=engine)
    ora = O.OracleDecoder(shape, deq, kv_dtype=kv, max_seq=max_seq)
    for t in prompt[:-1]:
        dec.step(int(t), skip_logits=True)
        ora.body(int(t))
    cur = int(prompt[-1])
    logits = torch.empty((2, shape.vocab), dtype=torch.float32, device="cuda")
    for j, draft in enumerate(drafts):
        p = dec.position
        n0, n1 = dec.verify2([cur, int(draft)], logits)
        assert dec.position == p + 2
        refs = [ora.step(cur), ora.step(int(draft))]
        got = logits.cpu().numpy()
        for r in range(2):
            close(got[r], refs[r], tol, f"verify {j} row {r}")
            own, ok = O.argmax_lowest(got[r])
            assert ok and (n0, n1)[r] == own, f"verify {j} row {r}: token is not the argmax of its own logits"
            srt = np.sort(refs[r])[::-1]
            if srt[0] - srt[1] > 2 * (tol + tol * abs(srt[0])):
                assert (n0, n1)[r] == O.argmax_lowest(refs[r])[0]
        for l in range(shape.layers):
            K, V, n = dec.kv(l)
            assert n == ora.pos
            rk, rv = ora.kv(l)
            close(kv_to_np(K[:, :n]), rk, tol, f"K layer {l} verify {j}")
            close(kv_to_np(V[:, :n]), rv, tol, f"V layer {l} verify {j}")
        cur = n1
    assert dec.device_errors() == 0
    dec.close()


@pytest.mark.parametrize("engine", ENGINES)
def test_small_q4_verify_two_rows(small_q4, engine):
    """Verify steps between single steps of either engine (the prompt goes through that engine)."""
    w, deq = small_q4
    prompt = Wl.prompt_uniform(6, Wl.Q4_SMALL.vocab, seed=5)
    drafts = Wl.prompt_uniform(5, Wl.Q4_SMALL.vocab, seed=6)
    check_verify(Wl.Q4_SMALL, w, deq, prompt, drafts, engine=engine)


def test_verify_accepts_and_rewinds_like_single_steps(small_q4):
    """A verify whose draft is the greedy token continues exactly like two single steps would (same
    tokens); a rejected draft is undone by rewinding to p + 1 and stepping the verified token."""
    import torch

    lib()
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    w, _ = small_q4
    s = Wl.Q4_SMALL
    prompt = [int(t) for t in Wl.prompt_uniform(5, s.vocab, seed=8)]
    a = Decoder(s, w, max_seq=32, engine="staged")
    b = Decoder(s, w, max_seq=32, engine="staged")
    a.prefill(prompt[:-1], is_last=False)
    b.prefill(prompt[:-1], is_last=False)
    t1 = a.step(prompt[-1])
    t2 = a.step(t1)
    t3 = a.step(t2)
    # b verifies (last prompt token, t1): an accepted draft
    v0, v1 = b.verify2([prompt[-1], t1])
    assert v0 == t1 and v1 == t2
    assert b.step(v1) == t3
    # a rejected draft: wrong token at p + 1, then rewind and step the verified token
    c = Decoder(s, w, max_seq=32, engine="staged")
    c.prefill(prompt[:-1], is_last=False)
    wrong = (t1 + 1) % s.vocab
    r0, _ = c.verify2([prompt[-1], wrong])
    assert r0 == t1
    c.rewind(len(prompt))
    assert c.step(r0) == t2
    ka, va, na = a.kv(1)
    kc, vc, nc = c.kv(1)
    assert na == nc + 1
    torch.testing.assert_close(kc[:, :nc], ka[:, :nc], rtol=LOW_TOL, atol=LOW_TOL)
    for d in (a, b, c):
        assert d.device_errors() == 0
        d.close()


def test_q4_config_errors(small_q4):
    W = lib()
    from weight_streaming_gemv_token_gb300 import binding as B
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    w, _ = small_q4
    with pytest.raises(W.WsgError):
        Decoder(Wl.Q4_SMALL, w, chunk_cap=128, engine="staged")
    d = Decoder(Wl.Q4_SMALL, w, max_seq=3, engine="staged")
    with pytest.raises(W.WsgError) as e:
        d.verify2([1, Wl.Q4_SMALL.vocab])
    assert e.value.status == B.DEC_EINVAL
    d.step(1, skip_logits=True)
    d.step(2, skip_logits=True)
    with pytest.raises(W.WsgError) as e:
        d.verify2([3, 4])  # positions 2 and 3 with max_seq 3
    assert e.value.status == B.DEC_ECAPACITY
    d.close()
    f = Decoder(Wl.TINY, Wl.decoder_weights(Wl.TINY, seed=1), engine="staged")
    with pytest.raises(W.WsgError) as e:
        f.verify2([1, 2])
    assert e.value.status == B.DEC_EINVAL
    f.close()


@pytest.fixture(scope="module")
def qwen_q4():
    w = Wl.decoder_weights_q4(Wl.QWEN3_06B, seed=1)
    return w, dequantised(w)


def test_qwen3_q4_generation_and_verify(qwen_q4):
    """Qwen3-0.6B geometry in the 4-bit configuration: a short generation and two verify steps,
    every logit and cache entry against the oracle."""
    w, deq = qwen_q4
    s = Wl.QWEN3_06B
    prompt = Wl.prompt_uniform(4, s.vocab, seed=0)
    for engine in ENGINES:
        run_and_compare(s, w, prompt, 3, "f32", LOW_TOL, check_kv_every=2, engine=engine, oracle_weights=deq)
    for engine in ENGINES:
        check_verify(s, w, deq, Wl.prompt_uniform(3, s.vocab, seed=2), Wl.prompt_uniform(2, s.vocab, seed=4),
                     engine=engine)


@pytest.mark.parametrize("engine", ENGINES)
def test_qwen3_q4_bench_launch_configuration(qwen_q4, engine):
    """The launch sequence bench.py times for the 4-bit configuration on each engine: the 32-token
    prompt, 4 warm-up steps in one call, then 256 steps in one call (positions 36-291), in a cache
    sized as the bench sizes it. Every token against the oracle on the dequantised weights,
    teacher-forced on the GPU's tokens (equal wherever the oracle's top-2 gap exceeds twice the
    tolerance), then every layer's whole cache (292 positions) at 2e-2."""
    lib()
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    w, deq = qwen_q4
    s = Wl.QWEN3_06B
    prompt = Wl.prompt_uniform(32, s.vocab, seed=0)
    dec = Decoder(s, w, kv_dtype="f32", max_seq=32 + 8 + 256 + 2 * (64 + 4) + 8, engine=engine)
    first = dec.prefill(prompt, is_last=True)
    warm = dec.generate(first, 4).cpu().tolist()
    timed = dec.generate(warm[-1], 256).cpu().tolist()
    toks = [first] + warm + timed
    assert dec.position == 32 + 4 + 256 and dec.device_errors() == 0
    ora = O.OracleDecoder(s, deq, max_seq=300)
    ref = O.generate(ora, prompt, len(toks), forced=toks)
    for j, (got, lg) in enumerate(zip(toks, ref["logits"])):
        srt = np.sort(lg)[::-1]
        if srt[0] - srt[1] > 2 * (LOW_TOL + LOW_TOL * abs(srt[0])):
            assert got == O.argmax_lowest(lg)[0], f"token {j}: GPU {got}, oracle {O.argmax_lowest(lg)[0]}"
    assert ora.pos == dec.position
    for l in range(s.layers):
        K, V, n = dec.kv(l)
        rk, rv = ora.kv(l)
        assert n == ora.pos
        close(kv_to_np(K[:, :n]), rk, LOW_TOL, f"K layer {l}")
        close(kv_to_np(V[:, :n]), rv, LOW_TOL, f"V layer {l}")
    dec.close()
