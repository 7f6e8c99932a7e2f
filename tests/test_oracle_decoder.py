"""Whole-model pins for the oracle decoder (tiny configuration, CPU only).

The model is the composition of the primitives pinned in
test_oracle_primitives.py. Here the composition itself is pinned by the
structural counts the pages print, by two independent formulations of the
same forward (token by token versus batched rows), and by invariants that a
wrongly wired layer would break.
"""
import copy
import dataclasses
import os

import numpy as np
import pytest

import oracle as O
import workloads as W


def _geometry(golden_dir):
    vals = {}
    with open(os.path.join(golden_dir, "qwen3_geometry.txt")) as f:
        for line in f:
            line = line.split("#")[0].split("|")[0].strip()
            if line:
                k, v = line.split("=")
                vals[k.strip()] = int(v)
    return vals


def test_geometry_matches_printed_values(golden_dir):
    g = _geometry(golden_dir)
    s = W.QWEN3_06B
    assert (s.layers, s.hidden, s.inter, s.n_q, s.n_kv, s.head_dim, s.vocab) == (
        g["layers"], g["hidden"], g["inter"], g["n_q"], g["n_kv"], g["head_dim"], g["vocab"])
    assert s.q_width == g["q_width"]
    shapes = W.tensor_shapes(s)
    assert shapes["w_q"] == (g["q_width"], g["hidden"])
    assert shapes["w_o"] == (g["hidden"], g["q_width"])
    # eight stages per layer plus embedding, final norm and vocabulary projection
    assert g["stages_per_layer"] * g["layers"] + 3 == g["dispatches_per_forward"]
    # one 32-lane group per vocabulary row, 256 threads = 8 rows per threadgroup
    assert g["vocab"] // (256 // 32) == g["vocab_threadgroups"]
    # P + N - 1 cache entries after generation; N - 1 advancing forwards
    assert g["held_out_prompt"] + g["held_out_outputs"] - 1 == g["held_out_cache_entries"]
    assert g["held_out_outputs"] - 1 == g["advancing_forwards"]


@pytest.fixture(scope="module")
def tiny_weights():
    return W.decoder_weights(W.TINY, seed=1)


def test_generation_protocol_cache_length(tiny_weights):
    m = O.OracleDecoder(W.TINY, tiny_weights, max_seq=64)
    prompt = W.prompt_uniform(8, W.TINY.vocab, seed=0)
    out = O.generate(m, prompt, 8)
    assert len(out["tokens"]) == 8
    assert m.pos == 8 + 8 - 1
    # every output is the argmax of its own logits
    for t, lg in zip(out["tokens"], out["logits"]):
        assert t == O.argmax_lowest(lg)[0]


def test_teacher_forcing_with_own_tokens_is_free_running(tiny_weights):
    prompt = W.prompt_uniform(5, W.TINY.vocab, seed=0)
    a = O.generate(O.OracleDecoder(W.TINY, tiny_weights, max_seq=32), prompt, 6)
    b = O.generate(O.OracleDecoder(W.TINY, tiny_weights, max_seq=32), prompt, 6, forced=a["tokens"])
    assert a["tokens"] == b["tokens"]
    for x, y in zip(a["logits"], b["logits"]):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("kv", ["f32", "bf16"])
def test_tokenwise_equals_batched_rows(tiny_weights, kv):
    prompt = W.prompt_uniform(11, W.TINY.vocab, seed=0)
    a = O.OracleDecoder(W.TINY, tiny_weights, kv_dtype=kv, max_seq=32)
    for t in prompt[:-1]:
        a.body(t)
    la = a.step(prompt[-1])
    b = O.OracleDecoder(W.TINY, tiny_weights, kv_dtype=kv, max_seq=32)
    # two chunks, the second continuing the causal prefix of the first
    b.prefill(prompt[:4], logit_rows=[])
    lb = b.prefill(prompt[4:])["logits"][len(prompt) - 5]
    assert a.pos == b.pos == len(prompt)
    for l in range(W.TINY.layers):
        tol = dict(rtol=1e-12, atol=1e-13) if kv == "f32" else dict(rtol=2.0 ** -7, atol=1e-12)
        np.testing.assert_allclose(a.kv(l)[0], b.kv(l)[0], **tol)
        np.testing.assert_allclose(a.kv(l)[1], b.kv(l)[1], **tol)
    np.testing.assert_allclose(la, lb, rtol=1e-10 if kv == "f32" else 1e-2, atol=1e-12 if kv == "f32" else 1e-3)


def test_batched_continuation_logits_equal_steps(tiny_weights):
    """Teacher forcing in one call: after a chunked prompt, a batched forward over forced tokens
    with logits on every row gives each row the logits that stepping through the same tokens gives
    (the long-context GPU tests follow the GPU's tokens this way)."""
    prompt = W.prompt_zipf(40, W.TINY.vocab, seed=2)
    forced = W.prompt_uniform(12, W.TINY.vocab, seed=5)
    a = O.OracleDecoder(W.TINY, tiny_weights, kv_dtype="bf16", max_seq=64)
    b = O.OracleDecoder(W.TINY, tiny_weights, kv_dtype="bf16", max_seq=64)
    for m in (a, b):
        m.prefill(prompt[:16], logit_rows=[])
        m.prefill(prompt[16:], logit_rows=[])
    rows = a.prefill(forced, logit_rows=list(range(len(forced))))["logits"]
    for r, t in enumerate(forced):
        np.testing.assert_allclose(rows[r], b.step(int(t)), rtol=1e-12, atol=1e-12)
    assert a.pos == b.pos == 52
    for l in range(W.TINY.layers):
        np.testing.assert_array_equal(a.kv(l)[0], b.kv(l)[0])
        np.testing.assert_array_equal(a.kv(l)[1], b.kv(l)[1])


def test_bf16_cache_holds_bf16_values(tiny_weights):
    m = O.OracleDecoder(W.TINY, tiny_weights, kv_dtype="bf16", max_seq=16)
    for t in W.prompt_uniform(4, W.TINY.vocab, seed=0):
        m.body(t)
    for l in range(W.TINY.layers):
        K, V = m.kv(l)
        np.testing.assert_array_equal(O.round_to_bf16(K), K)
        np.testing.assert_array_equal(O.round_to_bf16(V), V)


def test_zero_output_projections_pass_embedding_through(tiny_weights):
    w = copy.deepcopy(tiny_weights)
    for lw in w["layers"]:
        lw["w_o"] = np.zeros_like(lw["w_o"])
        lw["w_down"] = np.zeros_like(lw["w_down"])
    m = O.OracleDecoder(W.TINY, w, max_seq=8)
    tok = 123
    E = w["embed"].astype(np.float64)
    x = E[tok] / np.sqrt(np.mean(E[tok] ** 2) + W.TINY.eps) * w["g_final"].astype(np.float64)
    np.testing.assert_allclose(m.step(tok), E @ x, rtol=1e-13, atol=1e-15)


def test_cache_is_causal(tiny_weights):
    p1 = W.prompt_uniform(6, W.TINY.vocab, seed=0)
    p2 = p1.copy()
    p2[4] = (p2[4] + 1) % W.TINY.vocab
    a = O.OracleDecoder(W.TINY, tiny_weights, max_seq=8)
    b = O.OracleDecoder(W.TINY, tiny_weights, max_seq=8)
    for t in p1:
        a.body(t)
    for t in p2:
        b.body(t)
    for l in range(W.TINY.layers):
        np.testing.assert_array_equal(a.kv(l)[0][:, :4], b.kv(l)[0][:, :4])
        assert not np.allclose(a.kv(l)[0][:, 4:], b.kv(l)[0][:, 4:])


def test_cached_key_is_normed_and_rotated(tiny_weights):
    s = W.TINY
    m = O.OracleDecoder(s, tiny_weights, max_seq=8)
    tok = 42
    m.body(7)
    m.body(tok)      # position 1
    lw = tiny_weights["layers"][0]
    E = tiny_weights["embed"].astype(np.float64)
    x = O.rmsnorm(E[tok], lw["g_in"], s.eps)
    k = (lw["w_k"].astype(np.float64) @ x).reshape(s.n_kv, s.head_dim)
    v = (lw["w_v"].astype(np.float64) @ x).reshape(s.n_kv, s.head_dim)
    k = O.rope(O.rmsnorm(k, lw["g_k"], s.eps), 1, s.rope_theta)
    np.testing.assert_allclose(m.kv(0)[0][:, 1], k, rtol=1e-13)
    np.testing.assert_allclose(m.kv(0)[1][:, 1], v, rtol=1e-13)


def test_regression_golden_tokens(tiny_weights, golden_dir):
    """Frozen oracle output (written by tests/golden/make_golden.py); guards against drift."""
    path = os.path.join(golden_dir, "tiny_fp32_8x8.txt")
    ref = {}
    with open(path) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, v = line.split("=")
                ref[k.strip()] = [float(t) for t in v.split()]
    m = O.OracleDecoder(W.TINY, tiny_weights, max_seq=32)
    out = O.generate(m, W.prompt_uniform(8, W.TINY.vocab, seed=0), 8)
    assert out["tokens"] == [int(t) for t in ref["tokens"]]
    np.testing.assert_allclose(out["logits"][0][:16], ref["logits0_head"], rtol=1e-12)


# -- rescaling invariants -----------------------------------------------------------
# Each pair of weight changes below leaves the forward unchanged under the model's
# definition and changes it under a plausible miswiring (the norm named in the
# test id missing or given the wrong gain, gate and up swapped, a normalised
# value path, a wrong query-to-key/value-head grouping). Factors are powers of
# two, so the float32 weights change exactly; the invariants are exact as the
# RMSNorm eps goes to 0 (at 1e-6 against mean squares of q of ~0.025 they move
# the logits by ~4e-5), so these forwards run the tiny shape with eps = 1e-12.
TINY_SMALL_EPS = dataclasses.replace(W.TINY, eps=1e-12)


def _logits_and_cache(weights, prompt, kv="f32"):
    m = O.OracleDecoder(TINY_SMALL_EPS, weights, kv_dtype=kv, max_seq=16)
    for t in prompt[:-1]:
        m.body(t)
    return m.step(prompt[-1]), m


def _scaled(weights, **factors):
    w = copy.deepcopy(weights)
    for lw in w["layers"]:
        for name, f in factors.items():
            lw[name] = (lw[name] * np.float32(f)).astype(np.float32)
    return w


INVARIANT_PROMPT = [5, 300, 17, 17, 411, 2]


def _assert_same_forward(a, b):
    np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-9 * np.abs(a).max())


def _assert_other_forward(a, b):
    assert np.abs(a - b).max() > 1e-3 * np.abs(a).max()


@pytest.mark.parametrize("name,factors", [
    ("q_norm", dict(w_q=4.0)),                           # q is normalised per head
    ("q_k_norms", dict(w_q=4.0, w_k=0.25)),              # and so is k
    ("input_norm_gain", dict(g_in=4.0, w_q=0.25, w_k=0.25, w_v=0.25)),
    ("post_attention_norm_gain", dict(g_post=4.0, w_gate=0.25, w_up=0.25)),
    ("value_path_linear", dict(w_v=4.0, w_o=0.25)),      # v is not normalised
    ("up_linear", dict(w_up=-1.0, w_down=-1.0)),         # silu(gate) * up: odd in up
])
def test_forward_invariant_under_rescaling(tiny_weights, name, factors):
    ref, _ = _logits_and_cache(tiny_weights, INVARIANT_PROMPT)
    got, _ = _logits_and_cache(_scaled(tiny_weights, **factors), INVARIANT_PROMPT)
    _assert_same_forward(ref, got)


@pytest.mark.parametrize("factors", [
    dict(w_gate=-1.0, w_down=-1.0),   # the gate is not odd: silu(-z) != -silu(z)
    dict(g_post=4.0),                 # the MLP sees the post-attention gain
    dict(g_in=4.0),                   # and the value path the input gain
])
def test_forward_changes_under_an_uncompensated_rescaling(tiny_weights, factors):
    """Counterparts of the invariants: these changes are not undone, and each moves
    the logits by far more than the invariants' tolerance."""
    ref, _ = _logits_and_cache(tiny_weights, INVARIANT_PROMPT)
    got, _ = _logits_and_cache(_scaled(tiny_weights, **factors), INVARIANT_PROMPT)
    _assert_other_forward(ref, got)


def test_cached_values_scale_with_the_value_projection(tiny_weights):
    """The cache holds raw values: scaling w_v by 4 scales every cached value by
    exactly 4 in layer 0 (whose input does not depend on w_v) and leaves the keys
    alone."""
    _, a = _logits_and_cache(tiny_weights, INVARIANT_PROMPT)
    _, b = _logits_and_cache(_scaled(tiny_weights, w_v=4.0), INVARIANT_PROMPT)
    np.testing.assert_array_equal(b.kv(0)[1], 4.0 * a.kv(0)[1])
    np.testing.assert_array_equal(b.kv(0)[0], a.kv(0)[0])


def test_key_value_head_permutation(tiny_weights):
    """Swapping the two key/value heads together with the query heads that read
    them (query head h reads key/value head h // group) and with the matching
    columns of w_o leaves the logits unchanged; swapping only the key/value heads
    does not."""
    s = W.TINY
    d, group = s.head_dim, s.n_q // s.n_kv
    perm_kv = [1, 0]
    perm_q = [perm_kv[h // group] * group + h % group for h in range(s.n_q)]

    def rows(m, perm):
        return np.concatenate([m[p * d:(p + 1) * d] for p in perm], axis=0)

    w = copy.deepcopy(tiny_weights)
    only_kv = copy.deepcopy(tiny_weights)
    for lw, lo in zip(w["layers"], only_kv["layers"]):
        for m in (lw, lo):
            m["w_k"] = rows(m["w_k"], perm_kv)
            m["w_v"] = rows(m["w_v"], perm_kv)
        lw["w_q"] = rows(lw["w_q"], perm_q)
        lw["w_o"] = rows(lw["w_o"].T, perm_q).T.copy()
    ref, _ = _logits_and_cache(tiny_weights, INVARIANT_PROMPT)
    got, _ = _logits_and_cache(w, INVARIANT_PROMPT)
    _assert_same_forward(ref, got)
    bad, _ = _logits_and_cache(only_kv, INVARIANT_PROMPT)
    _assert_other_forward(ref, bad)
