"""Chunked prefill (tensor-core projections, causal attention over cache + chunk)
against the oracle's tokenwise forward, through the C ABI.

The chunked path computes the same forward as tokenwise prefill ("Megakernels",
"Chunked prefill for long prompts"): its projections are BF16 tensor-core
products whose activation operand is a bfloat16 value plus remainder pair, so
the rows keep float32 precision and the oracle is the plain forward (batched
over the prompt rows). Checked: the first output's logits and token, every KV
entry of every layer after the prompt, and a few decode steps after it (which
read the cache the chunks wrote), with BF16 weights and KV.
"""
import numpy as np
import pytest

import oracle as O
import workloads as Wl

from gpu_util import LOW_TOL, close, lib
from test_gpu_decoder import kv_to_np

pytestmark = pytest.mark.gpu


def check_token(got_logits, ref_logits, tok, tol, what):
    own, ok = O.argmax_lowest(got_logits)
    assert ok and tok == own, f"{what}: GPU token {tok} is not the argmax {own} of its own logits"
    srt = np.sort(ref_logits)[::-1]
    ref_tok, _ = O.argmax_lowest(ref_logits)
    if srt[0] - srt[1] > 2 * (tol + tol * abs(srt[0])):
        assert tok == ref_tok, f"{what}: GPU {tok} vs oracle {ref_tok}"


def run_chunked(shape, weights, prompt, chunk, n_out, engine, kv_every=1, kv_dtype="bf16"):
    import torch

    lib()
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    max_seq = len(prompt) + n_out + 4
    dec = Decoder(shape, weights, kv_dtype=kv_dtype, max_seq=max_seq, chunk_cap=chunk, engine=engine)
    ora = O.OracleDecoder(shape, weights, kv_dtype=kv_dtype, max_seq=max_seq)
    logits = torch.empty(shape.vocab, dtype=torch.float32, device="cuda")
    # GPU: the prompt in chunks of `chunk` rows; oracle: token by token
    for c0 in range(0, len(prompt), chunk):
        part = [int(t) for t in prompt[c0:c0 + chunk]]
        last = c0 + chunk >= len(prompt)
        nxt = dec.prefill(part, is_last=last, logits=logits if last else None)
    ref = ora.prefill(prompt)["logits"][len(prompt) - 1]
    got = logits.cpu().numpy()
    close(got, ref, LOW_TOL, "first output logits")
    check_token(got, ref, nxt, LOW_TOL, "first output")
    assert dec.position == len(prompt)
    for l in range(shape.layers):
        K, V, n = dec.kv(l)
        assert n == len(prompt)
        rk, rv = ora.kv(l)
        close(kv_to_np(K[:, :n]), rk, LOW_TOL, f"K layer {l} after the prompt")
        close(kv_to_np(V[:, :n]), rv, LOW_TOL, f"V layer {l} after the prompt")
    # decode after the chunks: the oracle continues on the GPU's tokens
    cur = nxt
    for j in range(n_out):
        tok = dec.step(cur, logits=logits)
        ref = ora.step(cur)
        got = logits.cpu().numpy()
        close(got, ref, LOW_TOL, f"decode step {j} logits")
        check_token(got, ref, tok, LOW_TOL, f"decode step {j}")
        cur = tok
    if n_out:
        for l in range(0, shape.layers, kv_every):
            K, V, n = dec.kv(l)
            rk, rv = ora.kv(l)
            close(kv_to_np(K[:, :n]), rk, LOW_TOL, f"K layer {l} after decode")
            close(kv_to_np(V[:, :n]), rv, LOW_TOL, f"V layer {l} after decode")
    assert dec.device_errors() == 0
    dec.close()


@pytest.fixture(scope="module")
def tiny_bf16():
    return Wl.decoder_weights(Wl.TINY, seed=1, wdtype="bf16")


@pytest.mark.parametrize("engine", ["persistent", "staged"])
@pytest.mark.parametrize("chunk", [64, 128])
def test_tiny_chunked_prefill(tiny_bf16, engine, chunk):
    """150 prompt rows in chunks of 64 (64 + 64 + 22) or of 128 (128 + 22); then decode
    steps that read the cache the chunks wrote."""
    prompt = Wl.prompt_uniform(150, Wl.TINY.vocab, seed=0)
    run_chunked(Wl.TINY, tiny_bf16, prompt, chunk, 4, engine)


def test_ragged_geometry_chunked_prefill():
    """4 query heads per KV head, head_dim 32, widths that are not multiples of the tiles."""
    shape = Wl.DecoderShape(layers=3, hidden=96, inter=200, n_q=8, n_kv=2, head_dim=32, vocab=777)
    w = Wl.decoder_weights(shape, seed=9, wdtype="bf16")
    prompt = Wl.prompt_zipf(77, shape.vocab, seed=0)
    run_chunked(shape, w, prompt, 32, 3, "persistent")


def test_fused_projection_launches_ragged_k():
    """Q, K, V (and gate, up) widths that are whole 128-column tiles share one GEMM launch per
    group; hidden 200 leaves a ragged K, 150 rows in chunks of 64 ragged row tiles."""
    shape = Wl.DecoderShape(layers=2, hidden=200, inter=256, n_q=4, n_kv=2, head_dim=64, vocab=500)
    w = Wl.decoder_weights(shape, seed=5, wdtype="bf16")
    prompt = Wl.prompt_zipf(150, shape.vocab, seed=1)
    run_chunked(shape, w, prompt, 64, 3, "persistent")


@pytest.mark.parametrize("kv_dtype", ["bf16", "f32"])
def test_head_dim_128_both_cache_types(kv_dtype):
    """head_dim 128 (the Qwen3 head) with a bfloat16 cache (tensor-core attention) and a float32
    cache (the CUDA-core attention kernel); 200 rows in chunks of 64 (ragged)."""
    shape = Wl.DecoderShape(layers=2, hidden=256, inter=512, n_q=4, n_kv=2, head_dim=128, vocab=500)
    w = Wl.decoder_weights(shape, seed=6, wdtype="bf16")
    prompt = Wl.prompt_zipf(200, shape.vocab, seed=3)
    run_chunked(shape, w, prompt, 64, 3, "persistent", kv_dtype=kv_dtype)


@pytest.mark.parametrize("n_q,n_kv", [(2, 2), (4, 2), (8, 2), (8, 1)])
def test_head_dim_128_query_groups(n_q, n_kv):
    """head_dim 128 with a bfloat16 cache (the tcgen05 attention: 128 query vectors per CTA, 128 /
    group rows) for groups of 1, 2, 4 and 8 query heads per key/value head; 300 rows in chunks of
    128 (128 + 128 + 44), so the later chunks walk two and three key tiles of 128 and the last
    tile and row block are ragged."""
    shape = Wl.DecoderShape(layers=2, hidden=256, inter=512, n_q=n_q, n_kv=n_kv, head_dim=128, vocab=500)
    w = Wl.decoder_weights(shape, seed=11, wdtype="bf16")
    prompt = Wl.prompt_zipf(300, shape.vocab, seed=4)
    run_chunked(shape, w, prompt, 128, 2, "persistent")


def test_head_dim_128_peaked_scores():
    """Q and K norm gains scaled by 3 (scores of standard deviation ~9): in layer 0 of the float64
    forward, 45 of the 688 (row, query head) pairs with more than 128 keys meet a later key tile of
    128 whose maximum passes the reference maximum by more than 2^8 (log2 units), so the attention
    rescales its output accumulator mid-walk.
    (At a gain of 6 the forward itself is ill-conditioned: the float64 forward with only the
    value + remainder operand roundings applied already moves layer-1 keys past the tolerance.)"""
    shape = Wl.DecoderShape(layers=2, hidden=256, inter=512, n_q=4, n_kv=2, head_dim=128, vocab=500)
    w = Wl.decoder_weights(shape, seed=12, wdtype="bf16")
    for lw in w["layers"]:
        lw["g_q"] = (lw["g_q"] * 3).astype(np.float32)
        lw["g_k"] = (lw["g_k"] * 3).astype(np.float32)
    prompt = Wl.prompt_zipf(300, shape.vocab, seed=5)
    run_chunked(shape, w, prompt, 128, 2, "staged")


def qwen3_widths_one_chunk(rows, reps):
    """Three layers of the Qwen3-0.6B widths, one chunk of `rows` rows, `reps` times on fresh
    decoders; every layer's K/V after each run against the oracle."""
    import dataclasses

    import torch

    lib()
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    s = dataclasses.replace(Wl.QWEN3_06B, layers=3)
    w = Wl.decoder_weights(s, seed=1, wdtype="bf16")
    prompt = [int(t) for t in Wl.prompt_zipf(rows, s.vocab, seed=2)]
    ora = O.OracleDecoder(s, w, kv_dtype="bf16", max_seq=rows + 8)
    ora.prefill(prompt, logit_rows=[])
    for rep in range(reps):
        dec = Decoder(s, w, kv_dtype="bf16", max_seq=rows + 8, chunk_cap=rows)
        dec.prefill(prompt, is_last=False)
        torch.cuda.synchronize()
        for l in range(s.layers):
            K, V, n = dec.kv(l)
            rk, rv = ora.kv(l)
            close(kv_to_np(K[:, :n]), rk, LOW_TOL, f"run {rep}: K layer {l}")
            close(kv_to_np(V[:, :n]), rv, LOW_TOL, f"run {rep}: V layer {l}")
        assert dec.device_errors() == 0
        dec.close()


def test_qwen3_widths_1024_row_chunk_repeated():
    """A 1024-row chunk three times: the attention's CTAs walk one to eight key tiles of 128
    (rows 128-255 two), so the waits on the output accumulator of the last tile run against
    products still in flight."""
    qwen3_widths_one_chunk(1024, 3)


def test_qwen3_widths_2048_row_chunk():
    """A 2048-row chunk: the Q/K/V and gate/up products take 256-column tiles (the SwiGLU
    epilogue pairing 128 gate and 128 up outputs), O and down 128-column ones."""
    qwen3_widths_one_chunk(2048, 1)


def test_single_row_chunks():
    """Chunks of one row: the causal attention sees only the cache."""
    w = Wl.decoder_weights(Wl.TINY, seed=2, wdtype="bf16")
    prompt = Wl.prompt_uniform(5, Wl.TINY.vocab, seed=1)
    run_chunked(Wl.TINY, w, prompt, 1, 2, "persistent")


@pytest.mark.slow
def test_qwen3_bf16_chunked_prefill():
    """The Qwen3-0.6B shape (BF16 weights and KV), a 300-token Zipf prompt in chunks of 128."""
    w = Wl.decoder_weights(Wl.QWEN3_06B, seed=1, wdtype="bf16")
    prompt = Wl.prompt_zipf(300, Wl.QWEN3_06B.vocab, seed=0)
    run_chunked(Wl.QWEN3_06B, w, prompt, 128, 2, "persistent", kv_every=7)


def test_chunked_prefill_needs_bf16_weights():
    lib()
    import weight_streaming_gemv_token_gb300 as W
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    w = Wl.decoder_weights(Wl.TINY, seed=1)
    with pytest.raises(W.WsgError):
        Decoder(Wl.TINY, w, kv_dtype="f32", max_seq=64, chunk_cap=64)
