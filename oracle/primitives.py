"""Oracle primitives: plain float64 restatements of each step of the decode path.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline leg use this package; the product path never imports it and shares
no code with it.

Every function computes its step's plain mathematical definition in float64.
Inputs arrive as float32 arrays or as bfloat16 bit patterns (uint16) and are
widened exactly. Citations name the page and section that define the step.
"""
from __future__ import annotations

import numpy as np


def widen(a) -> np.ndarray:
    """Exact float64 copy of a float32 array or of bfloat16 bits (uint16)."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def round_to_bf16(x) -> np.ndarray:
    """Nearest bfloat16 value (ties to even) of float64 values, returned as float64.

    bfloat16 keeps 8 significant bits. Used where the BF16 configuration stores
    a value (the KV cache: "Weights, cached keys/values ... use the selected
    dtype", Megakernels, "What runs in the DSL").
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                       # x = m * 2**e with 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)


def bf16_bits_of(x) -> np.ndarray:
    """bfloat16 bit patterns of values already representable in bfloat16."""
    return (np.asarray(x, dtype=np.float64).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def rmsnorm(x, g, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * g.

    Megakernels, "What runs in the DSL": the RMSNorm stages before attention,
    before the MLP and before the vocabulary projection, and the per-head Q/K
    RMSNorm. The gain multiplies the normalised vector directly.
    """
    x = widen(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * widen(g)


def rope(x, pos, theta: float) -> np.ndarray:
    """Rotary position embedding, rotate-half pairing, applied over the last axis.

    Megakernels, "What runs in the DSL" (RoPE after the per-head Q/K RMSNorm).
    Pair (i, i + d/2) for i < d/2 is rotated by the angle pos * theta**(-2i/d):
    (a, b) -> (a cos - b sin, a sin + b cos). ``pos`` is the absolute 0-based
    position; it may be an array broadcasting against x's leading axes.
    """
    x = widen(x)
    d = x.shape[-1]
    half = d // 2
    inv_freq = float(theta) ** (-2.0 * np.arange(half, dtype=np.float64) / d)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def silu(z) -> np.ndarray:
    """SiLU activation z * sigmoid(z) = z / (1 + exp(-z))."""
    z = widen(z)
    return z / (1.0 + np.exp(-z))


def swiglu(gate, up) -> np.ndarray:
    """SwiGLU: silu(gate) * up (Megakernels, "What runs in the DSL": gate/up projections -> SwiGLU)."""
    return silu(gate) * widen(up)


def softmax(s) -> np.ndarray:
    """Softmax over the last axis, maximum subtracted first. -inf entries get weight 0."""
    s = widen(s)
    m = np.max(s, axis=-1, keepdims=True)
    w = np.exp(s - m)
    return w / np.sum(w, axis=-1, keepdims=True)


def gqa_decode_attention(q, K, V) -> np.ndarray:
    """Grouped-query attention of one token over its cached keys and values.

    Megakernels, "What runs in the DSL" (grouped-query attention + KV update)
    and "GPU-wide end-to-end generation" (attention distributed over heads).
    q: [n_q, d]; K, V: [n_kv, T, d] holding positions 0..T-1 (the current
    token's entry included). Query head h reads key/value head h // (n_q/n_kv).
    Scores are q.k / sqrt(d) ("scaling happens after the QK product",
    "Matrix-tiled attention"). Returns o: [n_q, d].
    """
    q, K, V = widen(q), widen(K), widen(V)
    n_q, d = q.shape
    n_kv = K.shape[0]
    group = n_q // n_kv
    o = np.empty((n_q, d))
    for h in range(n_q):
        g = h // group
        w = softmax((K[g] @ q[h]) / np.sqrt(d))
        o[h] = w @ V[g]
    return o


def causal_prefill_attention(Q, K, V, p0: int) -> np.ndarray:
    """Attention of T consecutive rows at positions p0..p0+T-1 over the cache.

    Megakernels, "Chunked prefill for long prompts": each row attends to its
    whole causal prefix, earlier chunks included. Q: [T, n_q, d]; K, V:
    [n_kv, p0+T, d]. Row i sees keys 0..p0+i. Returns [T, n_q, d].
    """
    Q, K, V = widen(Q), widen(K), widen(V)
    T, n_q, d = Q.shape
    n_kv = K.shape[0]
    group = n_q // n_kv
    n = K.shape[1]
    assert n == p0 + T
    future = np.arange(n)[None, :] > (p0 + np.arange(T))[:, None]
    out = np.empty((T, n_q, d))
    for h in range(n_q):
        g = h // group
        s = (Q[:, h, :] @ K[g].T) / np.sqrt(d)
        s[future] = -np.inf
        out[:, h, :] = softmax(s) @ V[g]
    return out


def gemv(W, x) -> np.ndarray:
    """y = W x with W [out, in] row-major, accumulated in float64.

    "Our Kernel Benchmark Was Measuring the System Cache" (Summary): the
    matrix-vector product whose weight stream the benchmark measures.
    """
    return widen(W) @ widen(x)


def project_rows(A, W) -> np.ndarray:
    """Rows of a prompt chunk through one projection: C[m] = W A[m] for every
    row, i.e. C = A W^T with A [rows, in] and W [out, in], accumulated in
    float64 ("Megakernels", "Chunked prefill for long prompts": the chunk's
    rows go through each projection together).
    """
    return widen(A) @ widen(W).T


def q4_unpack(packed) -> np.ndarray:
    """uint4 codes [out, in] from words [out, in/8]; code j of word w is bits [4j, 4j+4), column 8w+j."""
    packed = np.asarray(packed, dtype=np.uint32)
    out, nw = packed.shape
    codes = np.empty((out, nw, 8), dtype=np.uint8)
    for j in range(8):
        codes[:, :, j] = (packed >> np.uint32(4 * j)) & np.uint32(0xF)
    return codes.reshape(out, nw * 8)


def q4_dequant(packed, scale, bias, group: int = 64) -> np.ndarray:
    """Groupwise-affine 4-bit weights: w = s * q + b, one fp16 (s, b) per 64 consecutive columns.

    "Our Kernel Benchmark Was Measuring the System Cache" (Summary: the 4-bit
    matrix-vector kernel). Evaluated exactly in float64.
    """
    q = q4_unpack(packed).astype(np.float64)
    s = np.repeat(np.asarray(scale, dtype=np.float64), group, axis=1)
    b = np.repeat(np.asarray(bias, dtype=np.float64), group, axis=1)
    return s * q + b


def gemv_q4(packed, scale, bias, x, group: int = 64) -> np.ndarray:
    """y[t] = W x[t] for the dequantised 4-bit W and each token row t of x [ntok, in]."""
    W = q4_dequant(packed, scale, bias, group)
    x = widen(x)
    if x.ndim == 1:
        return W @ x
    return x @ W.T


def argmax_lowest(v) -> tuple[int, bool]:
    """Greedy token: the lowest index reaching the maximum.

    Megakernels, "GPU-wide end-to-end generation": the argmax breaks ties by
    lowest token ID. NaN never wins; -0 and +0 compare equal. Returns
    (index, ok); an all-NaN vector gives (0, False).
    """
    v = np.asarray(v, dtype=np.float64)
    finite_or_inf = ~np.isnan(v)
    if not finite_or_inf.any():
        return 0, False
    m = np.max(v[finite_or_inf])
    return int(np.flatnonzero(v == m)[0]), True
