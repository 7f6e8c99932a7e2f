"""Long-context decode against the oracle: the key-parallel attention's merge of
many splits, and the held-out size of the long-document workload.

Decode attention splits the p + 1 cached keys of each key/value head into
nsplit = min(ceil((p + 1) / 64), min(64, SMs / n_kv)) ranges. Split 0 merges the
others' partials eight at a time on the persistent engine, so past 9 splits the
merge runs over several polling rounds; the staged engine's last CTA merges
them all. Each test asserts the split count its positions reach.

"Benchmark methodology", "Long-document chunked prefill": validation checks the
entire valid K/V prefix of every layer at each chunk boundary, then every
generated step's full logits, exact token and newly written K/V slot, and the
whole prefix again at the final output. The held-out workload is a 4,096-token
prompt (Zipf(1.1) draws from seed 2 stand in for the document) with BF16
weights and cache, in 1,024- and 2,048-row chunks; the oracle is the float64 forward,
batched over the rows of each chunk and continued on the GPU's tokens.
"""
import math

import numpy as np
import pytest

import oracle as O
import workloads as Wl

from gpu_util import FP32_TOL, LOW_TOL, close, lib
from test_gpu_decoder import kv_to_np

pytestmark = pytest.mark.gpu


def nsplit_at(shape, pos):
    """Split count of decode attention at position pos (its rule, documented in include/wsg.h)."""
    import torch

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = pos + 1
    ns = min(math.ceil(n / 64), max(1, min(64, sms // shape.n_kv)))
    per = math.ceil(n / ns)
    return math.ceil(n / per)


def check_token(got, ref, tok, tol, what):
    own, ok = O.argmax_lowest(got)
    assert ok and tok == own, f"{what}: GPU token {tok} is not the argmax {own} of its own logits"
    srt = np.sort(ref)[::-1]
    if srt[0] - srt[1] > 2 * (tol + tol * abs(srt[0])):
        assert tok == O.argmax_lowest(ref)[0], f"{what}: GPU {tok} vs oracle {O.argmax_lowest(ref)[0]}"


def check_prefix(dec, ora, shape, n, tol, what, layers=None):
    for l in layers if layers is not None else range(shape.layers):
        K, V, nv = dec.kv(l)
        assert nv == n == ora.pos
        rk, rv = ora.kv(l)
        close(kv_to_np(K[:, :n]), rk, tol, f"K layer {l} {what}")
        close(kv_to_np(V[:, :n]), rv, tol, f"V layer {l} {what}")


def check_slot(dec, ora, shape, p, tol, what):
    """The K/V slot at position p of every layer."""
    for l in range(shape.layers):
        K, V, _ = dec.kv(l)
        rk, rv = ora.kv(l)
        close(kv_to_np(K[:, p]), rk[:, p], tol, f"K layer {l} slot {p} {what}")
        close(kv_to_np(V[:, p]), rv[:, p], tol, f"V layer {l} slot {p} {what}")


def decode_and_check(dec, ora, shape, first, n_out, tol):
    """n_out decode steps from token `first`; logits, token and new slot at each, prefix at the end."""
    import torch

    logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    cur = first
    for j in range(n_out):
        p = dec.position
        tok = dec.step(cur, logits=logits)
        ref = ora.step(cur)
        got = logits.cpu().numpy()
        close(got, ref, tol, f"decode step {j} (position {p}) logits")
        check_token(got, ref, tok, tol, f"decode step {j}")
        check_slot(dec, ora, shape, p, tol, f"decode step {j}")
        cur = tok
    check_prefix(dec, ora, shape, dec.position, tol, "after decode")
    assert dec.device_errors() == 0


def run_long(shape, w, kv, engine, P, n_out=3, seed=0):
    import torch

    lib()
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    tol = FP32_TOL if (kv == "f32" and w.get("wdtype", "f32") == "f32") else LOW_TOL
    prompt = [int(t) for t in Wl.prompt_uniform(P, shape.vocab, seed=seed)]
    max_seq = P + n_out + 2
    assert nsplit_at(shape, P + n_out - 1) > 9, "too few splits for a merge over several rounds"
    dec = Decoder(shape, w, kv_dtype=kv, max_seq=max_seq, engine=engine)
    ora = O.OracleDecoder(shape, w, kv_dtype=kv, max_seq=max_seq)
    logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    tok = dec.prefill(prompt, is_last=True, logits=logits)
    ref = ora.prefill(prompt)["logits"][P - 1]
    got = logits.cpu().numpy()
    close(got, ref, tol, "first output logits")
    check_token(got, ref, tok, tol, "first output")
    check_prefix(dec, ora, shape, P, tol, "after the prompt")
    decode_and_check(dec, ora, shape, tok, n_out, tol)
    dec.close()


@pytest.mark.parametrize("engine", ["persistent", "staged"])
@pytest.mark.parametrize("kv", ["f32", "bf16"])
@pytest.mark.parametrize("P", [1100, 4700])
def test_tiny_long_context(engine, kv, P):
    """Tiny model: 18 splits (3 merge rounds) at ~1,100 positions, 64 (8 rounds) at ~4,700."""
    run_long(Wl.TINY, Wl.decoder_weights(Wl.TINY, seed=1), kv, engine, P)


@pytest.mark.parametrize("engine", ["persistent", "staged"])
def test_ragged_geometry_long_context(engine):
    """4 query heads per key/value head, head_dim 32, widths that are not multiples of the tiles."""
    shape = Wl.DecoderShape(layers=3, hidden=96, inter=200, n_q=8, n_kv=2, head_dim=32, vocab=777)
    run_long(shape, Wl.decoder_weights(shape, seed=9), "bf16", engine, 1100, seed=3)


@pytest.mark.slow
@pytest.mark.parametrize("C", [1024, 2048])
def test_qwen3_bf16_held_out_size_against_oracle(C):
    """The held-out size of the long-document workload on the Qwen3-0.6B shape: the 4,096-token
    prompt in chunks of C rows (tensor-core projections; 2,048 is the chunk bench.py's tuning
    picks and times, with 256-column tiles for Q/K/V and gate/up), every layer's whole K/V prefix
    at each chunk boundary and the first output's logits against the oracle, the tokenwise path's
    first output too (once), then decode steps at positions 4,096 and up (19 splits per
    key/value head, merged over 3 polling rounds) with their logits, tokens and new slots, and the
    prefix at the end."""
    import torch

    lib()
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    s = Wl.QWEN3_06B
    P, n_out = 4096, 3
    w = Wl.decoder_weights(s, seed=1, wdtype="bf16")
    prompt = [int(t) for t in Wl.prompt_zipf(P, s.vocab, seed=2)]
    max_seq = P + n_out + 1
    assert nsplit_at(s, P) > 9
    dec = Decoder(s, w, kv_dtype="bf16", max_seq=max_seq, chunk_cap=C)
    ora = O.OracleDecoder(s, w, kv_dtype="bf16", max_seq=max_seq)
    logits = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
    for c0 in range(0, P, C):
        last = c0 + C >= P
        tok = dec.prefill(prompt[c0:c0 + C], is_last=last, logits=logits if last else None)
        out = ora.prefill(prompt[c0:c0 + C], logit_rows=[C - 1] if last else [])
        check_prefix(dec, ora, s, c0 + C, LOW_TOL, f"at the chunk boundary {c0 + C}")
    ref = out["logits"][C - 1]
    got = logits.cpu().numpy()
    close(got, ref, LOW_TOL, "first output logits (chunked)")
    check_token(got, ref, tok, LOW_TOL, "first output (chunked)")
    if C == 1024:  # the tokenwise path of the same prompt: first output
        tw = Decoder(s, w, kv_dtype="bf16", max_seq=max_seq)
        lt = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
        ttok = tw.prefill(prompt, is_last=True, logits=lt)
        gt = lt.cpu().numpy()
        close(gt, ref, LOW_TOL, "first output logits (tokenwise)")
        check_token(gt, ref, ttok, LOW_TOL, "first output (tokenwise)")
        assert tw.device_errors() == 0
        tw.close()
    decode_and_check(dec, ora, s, tok, n_out, LOW_TOL)
    dec.close()


@pytest.mark.slow
def test_qwen3_bf16_held_out_generation_as_benched():
    """The held-out generation exactly as bench.py runs it: the 4,096-token prompt in 2,048-row
    chunks into a 5,128-row cache, then the remaining 1,023 outputs in one launch (positions
    4,096-5,118, 19 splits per key/value head). The oracle prefills the same chunks and follows the
    GPU's tokens (one batched forward over them, the same mathematics as stepping): every token
    equal to the oracle's wherever its top-2 gap exceeds twice the tolerance, and every layer's
    whole cache (5,119 positions) at the end."""
    lib()
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    s = Wl.QWEN3_06B
    P, C, N = 4096, 2048, 1024
    w = Wl.decoder_weights(s, seed=1, wdtype="bf16")
    prompt = [int(t) for t in Wl.prompt_zipf(P, s.vocab, seed=2)]
    dec = Decoder(s, w, kv_dtype="bf16", max_seq=P + N + 8, chunk_cap=C)
    for c0 in range(0, P, C):
        first = dec.prefill(prompt[c0:c0 + C], is_last=c0 + C >= P)
    toks = [first] + dec.generate(first, N - 1).cpu().tolist()
    assert dec.position == P + N - 1 and dec.device_errors() == 0
    ora = O.OracleDecoder(s, w, kv_dtype="bf16", max_seq=P + N)
    for c0 in range(0, P, C):
        out = ora.prefill(prompt[c0:c0 + C], logit_rows=[C - 1] if c0 + C >= P else [])
    forced = ora.prefill(toks[:-1], logit_rows=list(range(N - 1)))["logits"]
    refs = [out["logits"][C - 1]] + [forced[r] for r in range(N - 1)]
    for j, (got, lg) in enumerate(zip(toks, refs)):
        srt = np.sort(lg)[::-1]
        if srt[0] - srt[1] > 2 * (LOW_TOL + LOW_TOL * abs(srt[0])):
            assert got == O.argmax_lowest(lg)[0], f"output {j}: GPU {got}, oracle {O.argmax_lowest(lg)[0]}"
    check_prefix(dec, ora, s, P + N - 1, LOW_TOL, "after 1,024 outputs")
    dec.close()
