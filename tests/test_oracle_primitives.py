"""Pins for the oracle's primitives: closed forms, invariants, special cases, brute force.

Each test is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign or index, a transposed operand, a wrong pairing) fails it.
"""
import math
import os

import numpy as np
import pytest

import oracle as O
import workloads as W


def _golden(golden_dir, name):
    vals = {}
    with open(os.path.join(golden_dir, name)) as f:
        for line in f:
            line = line.split("#")[0].split("|")[0].strip()
            if not line:
                continue
            k, v = line.split("=")
            vals[k.strip()] = np.array([float(t) for t in v.split()])
    return vals


# -- RMSNorm -------------------------------------------------------------------

def test_rmsnorm_hand_example(golden_dir):
    g = _golden(golden_dir, "closed_forms.txt")
    y = O.rmsnorm(np.array([3.0, 4.0]), np.ones(2), 0.0)
    np.testing.assert_allclose(y, g["rmsnorm_34"], rtol=1e-15)


def test_rmsnorm_constant_vector_maps_to_gain():
    c, eps = 2.5, 1e-6
    gain = np.linspace(0.5, 1.5, 16)
    y = O.rmsnorm(np.full(16, c), gain, eps)
    np.testing.assert_allclose(y, gain * c / math.sqrt(c * c + eps), rtol=1e-15)


def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(5)
    x = rng.standard_normal(1024)
    eps = 1e-6
    y = O.rmsnorm(x, np.ones(1024), eps)
    ms = np.mean(x * x)
    assert abs(math.sqrt(np.mean(y * y)) - math.sqrt(ms / (ms + eps))) < 1e-14
    np.testing.assert_allclose(O.rmsnorm(7.0 * x, np.ones(1024), 0.0), O.rmsnorm(x, np.ones(1024), 0.0), rtol=1e-13)


def test_rmsnorm_rows_are_independent():
    rng = np.random.default_rng(6)
    X = rng.standard_normal((5, 32))
    g = rng.standard_normal(32)
    Y = O.rmsnorm(X, g, 1e-6)
    for i in range(5):
        np.testing.assert_allclose(Y[i], O.rmsnorm(X[i], g, 1e-6), rtol=1e-15)


# -- RoPE -----------------------------------------------------------------------

def test_rope_hand_examples(golden_dir):
    g = _golden(golden_dir, "closed_forms.txt")
    e = np.eye(4)
    np.testing.assert_allclose(O.rope(e[0], 1, 100.0), g["rope_e0_pos1"], atol=1e-15)
    np.testing.assert_allclose(O.rope(e[1], 2, 100.0), g["rope_e1_pos2"], atol=1e-15)
    np.testing.assert_allclose(O.rope(e[2], 1, 100.0), g["rope_e2_pos1"], atol=1e-15)


def test_rope_position_zero_is_identity():
    x = np.random.default_rng(1).standard_normal((3, 128))
    np.testing.assert_array_equal(O.rope(x, 0, 1e6), x)


def test_rope_preserves_pair_norms():
    x = np.random.default_rng(2).standard_normal(128)
    y = O.rope(x, 37, 1e6)
    np.testing.assert_allclose(x[:64] ** 2 + x[64:] ** 2, y[:64] ** 2 + y[64:] ** 2, rtol=1e-13)


def test_rope_relative_position_property():
    rng = np.random.default_rng(3)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    for m, n in [(5, 2), (100, 37), (4095, 17)]:
        lhs = O.rope(q, m, 1e6) @ O.rope(k, n, 1e6)
        rhs = O.rope(q, m - n, 1e6) @ k
        assert abs(lhs - rhs) < 1e-9 * (1 + abs(rhs))


def test_rope_vectorised_positions_match_scalar():
    x = np.random.default_rng(4).standard_normal((6, 2, 16))
    pos = np.arange(10, 16)
    Y = O.rope(x, pos[:, None], 1e6)
    for i, p in enumerate(pos):
        np.testing.assert_allclose(Y[i], O.rope(x[i], p, 1e6), rtol=1e-15)


# -- SiLU / SwiGLU ---------------------------------------------------------------

def test_silu_values(golden_dir):
    g = _golden(golden_dir, "closed_forms.txt")
    assert O.silu(np.array([0.0]))[0] == 0.0
    assert abs(O.silu(np.array([1.0]))[0] - g["silu_1"][0]) < 1e-16
    assert abs(O.silu(np.array([40.0]))[0] - 40.0) < 1e-12
    assert abs(O.silu(np.array([-40.0]))[0]) < 1e-15
    z = np.random.default_rng(7).standard_normal(50)
    u = np.random.default_rng(8).standard_normal(50)
    np.testing.assert_allclose(O.swiglu(z, u), z / (1 + np.exp(-z)) * u, rtol=1e-15)
    # swiglu is not symmetric in its operands
    assert not np.allclose(O.swiglu(z, u), O.swiglu(u, z))


# -- softmax / attention -----------------------------------------------------------

def test_attention_single_key_returns_its_value():
    rng = np.random.default_rng(9)
    q = rng.standard_normal((4, 16))
    K = rng.standard_normal((2, 1, 16))
    V = rng.standard_normal((2, 1, 16))
    o = O.gqa_decode_attention(q, K, V)
    for h in range(4):
        np.testing.assert_array_equal(o[h], V[h // 2, 0])


def test_attention_equal_keys_average_values():
    rng = np.random.default_rng(10)
    q = rng.standard_normal((2, 8))
    K = np.repeat(rng.standard_normal((1, 1, 8)), 5, axis=1)
    V = rng.standard_normal((1, 5, 8))
    o = O.gqa_decode_attention(q, K, V)
    np.testing.assert_allclose(o, np.repeat(V[0].mean(0)[None], 2, 0), rtol=1e-14)


def test_attention_two_keys_closed_form():
    rng = np.random.default_rng(11)
    d = 16
    q = rng.standard_normal((1, d))
    K = rng.standard_normal((1, 2, d))
    V = rng.standard_normal((1, 2, d))
    s0, s1 = K[0, 0] @ q[0] / math.sqrt(d), K[0, 1] @ q[0] / math.sqrt(d)
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    expect = w0 * V[0, 0] + (1 - w0) * V[0, 1]
    np.testing.assert_allclose(O.gqa_decode_attention(q, K, V)[0], expect, rtol=1e-13)


def test_attention_gqa_grouping():
    n_q, n_kv, T, d = 16, 8, 3, 4
    rng = np.random.default_rng(12)
    q = rng.standard_normal((n_q, d))
    K = rng.standard_normal((n_kv, T, d))
    V = np.zeros((n_kv, T, d))
    for g in range(n_kv):
        V[g] = g + 1.0
    o = O.gqa_decode_attention(q, K, V)
    for h in range(n_q):
        np.testing.assert_allclose(o[h], h // 2 + 1.0, rtol=1e-14)


def test_attention_large_gap_selects_key():
    d = 4
    q = np.array([[10.0, 0, 0, 0]])
    K = np.array([[[0.0, 0, 0, 0], [30.0, 0, 0, 0], [1.0, 0, 0, 0]]])
    V = np.array([[[1.0, 1, 1, 1], [2.0, 3, 4, 5], [9.0, 9, 9, 9]]])
    np.testing.assert_allclose(O.gqa_decode_attention(q, K, V)[0], [2, 3, 4, 5], rtol=1e-12)


def test_causal_prefill_matches_per_row_decode_and_ignores_future():
    rng = np.random.default_rng(13)
    n_q, n_kv, d, p0, T = 4, 2, 8, 3, 5
    Q = rng.standard_normal((T, n_q, d))
    K = rng.standard_normal((n_kv, p0 + T, d))
    V = rng.standard_normal((n_kv, p0 + T, d))
    out = O.causal_prefill_attention(Q, K, V, p0)
    for i in range(T):
        ref = O.gqa_decode_attention(Q[i], K[:, : p0 + i + 1], V[:, : p0 + i + 1])
        np.testing.assert_allclose(out[i], ref, rtol=1e-13)
    K2, V2 = K.copy(), V.copy()
    K2[:, -1] += 100.0
    V2[:, -1] -= 100.0
    out2 = O.causal_prefill_attention(Q, K2, V2, p0)
    np.testing.assert_array_equal(out[:-1], out2[:-1])
    assert not np.allclose(out[-1], out2[-1])


# -- GEMV ----------------------------------------------------------------------------

def test_gemv_structure_and_orientation():
    out, inp = 3, 5
    Wm = np.array([[10 * i + j for j in range(inp)] for i in range(out)], dtype=np.float32)
    for j in range(inp):
        np.testing.assert_array_equal(O.gemv(Wm, np.eye(inp, dtype=np.float32)[j]), Wm[:, j])
    np.testing.assert_array_equal(O.gemv(np.eye(4, dtype=np.float32), np.arange(4, dtype=np.float32)), np.arange(4))


def test_gemv_brute_force_exact_sum():
    rng = np.random.default_rng(14)
    Wm = rng.standard_normal((7, 33)).astype(np.float32)
    x = rng.standard_normal(33).astype(np.float32)
    y = O.gemv(Wm, x)
    for i in range(7):
        exact = math.fsum(float(Wm[i, j]) * float(x[j]) for j in range(33))
        assert abs(y[i] - exact) <= 1e-14 * (1 + abs(exact))


def test_gemv_bf16_bits_widen_exactly():
    Wf = W.gemv_matrix(9, 16, seed=3)
    Wb = W.f32_to_bf16_bits(Wf)
    widened = O.widen(Wb)
    np.testing.assert_array_equal(widened, W.bf16_bits_to_f32(Wb).astype(np.float64))
    assert np.max(np.abs(widened - Wf) / np.abs(Wf)) <= 2.0 ** -8


# -- bf16 rounding ----------------------------------------------------------------------

def test_round_to_bf16_ties_and_agreement():
    one = 1.0
    assert O.round_to_bf16(one + 2.0 ** -8) == 1.0                 # tie -> even (1.0)
    assert O.round_to_bf16(one + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6  # tie -> even (1 + 2^-6)
    assert O.round_to_bf16(one + 2.0 ** -8 + 2.0 ** -20) == 1.0 + 2.0 ** -7
    assert O.round_to_bf16(-3.0) == -3.0
    x = np.random.default_rng(15).standard_normal(10000).astype(np.float32)
    bits_gen = W.f32_to_bf16_bits(x)
    np.testing.assert_array_equal(O.bf16_bits_of(O.round_to_bf16(x.astype(np.float64))), bits_gen)


# -- 4-bit groupwise affine ----------------------------------------------------------------

def test_q4_bit_layout():
    words = np.array([[0x76543210, 0xFEDCBA98]], dtype=np.uint32)
    np.testing.assert_array_equal(O.q4_unpack(words)[0], np.arange(16))


def test_q4_pack_roundtrip():
    m = W.q4_matrix(8, 128, seed=4)
    np.testing.assert_array_equal(O.q4_unpack(m["packed"]), m["codes"])


def test_q4_dequant_groups():
    out, inp = 2, 128
    codes = np.zeros((out, inp), dtype=np.uint8)
    codes[:, :64] = 3
    codes[:, 64:] = np.arange(64) % 16
    s = np.array([[0.5, 0.0], [0.25, 2.0]], dtype=np.float16)
    b = np.array([[-1.0, 1.0], [0.0, -0.5]], dtype=np.float16)
    w = O.q4_dequant(W.pack_q4(codes), s, b)
    np.testing.assert_array_equal(w[0, :64], 0.5)       # 0.5 * 3 - 1
    np.testing.assert_array_equal(w[0, 64:], 1.0)       # 0 * q + 1
    np.testing.assert_array_equal(w[1, :64], 0.75)      # 0.25 * 3 + 0
    np.testing.assert_array_equal(w[1, 64:], 2.0 * (np.arange(64) % 16) - 0.5)


def test_q4_gemv_closed_form():
    m = W.q4_matrix(5, 192, seed=6)
    x = W.q4_activations(192, 2, seed=7)
    y = O.gemv_q4(m["packed"], m["scale"], m["bias"], x)
    xf = O.widen(x)
    for t in range(2):
        for i in range(5):
            acc = 0.0
            for g in range(3):
                sl = slice(64 * g, 64 * g + 64)
                acc += float(m["scale"][i, g]) * float(m["codes"][i, sl].astype(np.float64) @ xf[t, sl])
                acc += float(m["bias"][i, g]) * float(xf[t, sl].sum())
            assert abs(y[t, i] - acc) <= 1e-12 * (1 + abs(acc))
    np.testing.assert_allclose(O.gemv_q4(m["packed"], m["scale"], m["bias"], x[0]), y[0], rtol=1e-15)


# -- argmax -------------------------------------------------------------------------------------

def test_argmax_ties_nan_and_signed_zero():
    assert O.argmax_lowest([1.0, 3.0, 2.0, 3.0]) == (1, True)
    assert O.argmax_lowest([np.nan, 1.0, 5.0, np.nan, 5.0]) == (2, True)
    assert O.argmax_lowest([-1.0, -0.0, 0.0, -2.0]) == (1, True)
    assert O.argmax_lowest([-2.0, 0.0, -0.0]) == (1, True)
    assert O.argmax_lowest([-np.inf, -np.inf]) == (0, True)
    assert O.argmax_lowest([np.nan, np.nan]) == (0, False)
    v = np.zeros(151936, dtype=np.float32)
    v[151935] = 1.0
    v[77] = 1.0
    assert O.argmax_lowest(v) == (77, True)


# -- input generators ------------------------------------------------------------------------------

def test_zipf_prompt_distribution():
    p = W.prompt_zipf(20000, 151936, seed=0)
    assert p.min() >= 0 and p.max() < 151936
    # P(id = 0) = 1 / H(1.1, V); about 0.095 for V = 151936
    k = np.arange(1, 151937, dtype=np.float64)
    p0 = 1.0 / np.sum(k ** -1.1)
    assert abs(np.mean(p == 0) - p0) < 0.01
    assert np.mean(p == 1) < np.mean(p == 0)


def test_weights_draw_order_is_stable():
    a = W.decoder_weights(W.TINY, seed=1)
    b = W.decoder_weights(W.TINY, seed=1)
    np.testing.assert_array_equal(a["layers"][1]["w_down"], b["layers"][1]["w_down"])
    assert a["embed"].shape == (512, 64)
    g = a["layers"][0]["g_in"]
    assert abs(g.mean() - 1.0) < 0.05 and 0.05 < g.std() < 0.15


def test_project_rows_is_a_gemv_per_row_and_brute_force():
    """The chunk projection is the GEMV applied to every row (the definition),
    and on a tiny case equals the explicit triple loop."""
    rng = np.random.default_rng(5)
    A = rng.standard_normal((7, 13)).astype(np.float32)
    W = rng.standard_normal((5, 13)).astype(np.float32)
    C = O.project_rows(A, W)
    assert C.shape == (7, 5)
    for m in range(7):  # same sums, float64 summation order aside
        np.testing.assert_allclose(C[m], O.gemv(W, A[m]), rtol=1e-13, atol=1e-13)
    brute = np.zeros((7, 5))
    for m in range(7):
        for n in range(5):
            brute[m, n] = sum(float(A[m, k]) * float(W[n, k]) for k in range(13))
    np.testing.assert_allclose(C, brute, rtol=1e-12, atol=1e-12)
    # orientation: a unit row of A picks a column of W
    e = np.zeros((1, 13), np.float32)
    e[0, 4] = 1.0
    np.testing.assert_array_equal(O.project_rows(e, W)[0], W[:, 4].astype(np.float64))
