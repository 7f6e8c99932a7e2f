"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module only draws numbers and lays them out in the storage formats the
decoder and the GEMV entry points accept. It contains none of the method's
arithmetic: no norm, projection, rotary, attention or argmax step lives here.

Workloads follow the Qwen3-0.6B geometry of the "Megakernels" page (section
"What runs in the DSL": 28 layers, hidden 1024, intermediate 3072, 16 query
heads, 8 key/value heads, head dim 128, tied 151936-token vocabulary) and a
tiny decoder of the same structure. Real checkpoints and document prompts are
not available, so weights are N(0, 0.02), norm gains 1 + N(0, 0.1), and
prompts are uniform or bounded-Zipf token draws.

Storage formats produced here:
  * f32 arrays: numpy float32.
  * bf16 arrays: numpy uint16 holding the upper 16 bits of the float32 value
    after round-to-nearest-even.
  * 4-bit groupwise-affine matrices: codes packed 8 per uint32 (code j of
    word w sits at bits [4j, 4j+4) and belongs to input column 8w+j), fp16
    scale and bias per group of 64 consecutive input columns, each stored
    row-major as [out][in/8] and [out][in/64].
"""
from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass(frozen=True)
class DecoderShape:
    layers: int
    hidden: int
    inter: int
    n_q: int
    n_kv: int
    head_dim: int
    vocab: int
    eps: float = 1e-6
    rope_theta: float = 1e6

    @property
    def q_width(self) -> int:
        return self.n_q * self.head_dim

    @property
    def kv_width(self) -> int:
        return self.n_kv * self.head_dim


# Tiny decoder with the Qwen3 structure (2 layers, hidden 64, ...).
TINY = DecoderShape(layers=2, hidden=64, inter=192, n_q=4, n_kv=2, head_dim=16, vocab=512)
# The smallest decoder the 4-bit configuration takes (widths multiples of 512).
Q4_SMALL = DecoderShape(layers=2, hidden=512, inter=1024, n_q=4, n_kv=2, head_dim=128, vocab=1024)
# Qwen3-0.6B geometry ("Megakernels", "What runs in the DSL").
QWEN3_06B = DecoderShape(layers=28, hidden=1024, inter=3072, n_q=16, n_kv=8, head_dim=128, vocab=151936)

# Per-layer tensors, in the order they are drawn from the weight generator.
LAYER_TENSORS = ("w_q", "w_k", "w_v", "w_o", "w_gate", "w_up", "w_down", "g_in", "g_post", "g_q", "g_k")

# The five GEMV shapes (out x in) of one Qwen3-0.6B layer and the vocabulary head.
GEMV_SHAPES = ((4096, 1024), (1024, 2048), (6144, 1024), (1024, 3072), (151936, 1024))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def tensor_shapes(s: DecoderShape) -> dict:
    """Row-major shapes of every decoder tensor (out x in for projections)."""
    H, I, d = s.hidden, s.inter, s.head_dim
    return {
        "embed": (s.vocab, H),
        "w_q": (s.q_width, H),
        "w_k": (s.kv_width, H),
        "w_v": (s.kv_width, H),
        "w_o": (H, s.q_width),
        "w_gate": (I, H),
        "w_up": (I, H),
        "w_down": (H, I),
        "g_in": (H,),
        "g_post": (H,),
        "g_q": (d,),
        "g_k": (d,),
        "g_final": (H,),
    }


def decoder_weights(s: DecoderShape, seed: int = 1, wdtype: str = "f32") -> dict:
    """Random decoder weights.

    Draw order from ``numpy.random.default_rng(seed)``: embed, then for each
    layer the tensors of LAYER_TENSORS in that order, then g_final.
    Projections and the tied embedding are 0.02 * N(0, 1); RMSNorm gains are
    1 + 0.1 * N(0, 1). Gains stay float32 in every configuration; with
    ``wdtype == "bf16"`` the projection and embedding draws are rounded to
    bfloat16 and returned as uint16 bit arrays.

    ``wdtype == "f32_from_bf16"`` gives the float32 model converted from the
    bfloat16 one: the same rounded draws widened back to float32 (their low 16
    bits are zero), tagged "f32".

    Returns {"embed", "g_final", "layers": [dict per layer]}.
    """
    if wdtype not in ("f32", "bf16", "f32_from_bf16"):
        raise ValueError(wdtype)
    rng = np.random.default_rng(seed)
    shapes = tensor_shapes(s)

    def draw(name):
        shp = shapes[name]
        n = int(np.prod(shp))
        z = rng.standard_normal(n, dtype=np.float32).reshape(shp)
        if name.startswith("g_"):
            return (np.float32(1.0) + np.float32(0.1) * z).astype(np.float32)
        w = (np.float32(0.02) * z).astype(np.float32)
        if wdtype == "bf16":
            return f32_to_bf16_bits(w)
        if wdtype == "f32_from_bf16":
            return bf16_bits_to_f32(f32_to_bf16_bits(w))
        return w

    out = {"embed": draw("embed"), "layers": []}
    for _ in range(s.layers):
        out["layers"].append({name: draw(name) for name in LAYER_TENSORS})
    out["g_final"] = draw("g_final")
    out["wdtype"] = "f32" if wdtype == "f32_from_bf16" else wdtype
    return out


def prompt_uniform(n: int, vocab: int, seed: int = 0) -> np.ndarray:
    """n token IDs uniform over [0, vocab)."""
    return np.random.default_rng(seed).integers(0, vocab, n).astype(np.int32)


def prompt_zipf(n: int, vocab: int, s: float = 1.1, seed: int = 0) -> np.ndarray:
    """n token IDs from a Zipf(s) law bounded to the vocabulary.

    P(id = k - 1) is proportional to k**-s for k = 1..vocab; drawn by inverse
    CDF from ``default_rng(seed).random(n)``. Stands in for the document
    prompts of the long-document benchmark, which are not available.
    """
    k = np.arange(1, vocab + 1, dtype=np.float64)
    cdf = np.cumsum(k ** -s)
    cdf /= cdf[-1]
    u = np.random.default_rng(seed).random(n)
    return np.minimum(np.searchsorted(cdf, u, side="right"), vocab - 1).astype(np.int32)


def gemv_matrix(out: int, inp: int, seed: int, dtype: str = "f32") -> np.ndarray:
    """W ~ 0.02 * N(0, 1) of shape [out, in] (float32, or bf16 bits)."""
    w = (np.float32(0.02) * np.random.default_rng(seed).standard_normal(out * inp, dtype=np.float32)).reshape(out, inp)
    return f32_to_bf16_bits(w) if dtype == "bf16" else w


def gemv_vector(n: int, seed: int, dtype: str = "f32", scale: float = 0.02) -> np.ndarray:
    """x ~ scale * N(0, 1) (float32, or bf16 bits)."""
    x = (np.float32(scale) * np.random.default_rng(seed).standard_normal(n, dtype=np.float32)).astype(np.float32)
    return f32_to_bf16_bits(x) if dtype == "bf16" else x


def pack_q4(codes: np.ndarray) -> np.ndarray:
    """Pack uint4 codes [out, in] (values 0..15) 8 per uint32, low nibble first."""
    out, inp = codes.shape
    if inp % 8:
        raise ValueError("in must be a multiple of 8")
    c = codes.astype(np.uint32).reshape(out, inp // 8, 8)
    word = np.zeros((out, inp // 8), dtype=np.uint32)
    for j in range(8):
        word |= c[:, :, j] << np.uint32(4 * j)
    return word


def q4_matrix(out: int, inp: int, seed: int, group: int = 64) -> dict:
    """4-bit groupwise-affine matrix: codes U{0..15}, s ~ U(0.001, 0.01), b ~ 0.02 * N(0, 1).

    Returns {"codes": uint8 [out, in], "packed": uint32 [out, in/8],
    "scale": float16 [out, in/64], "bias": float16 [out, in/64]}.
    """
    if inp % group:
        raise ValueError("in must be a multiple of the group size")
    rng = np.random.default_rng(seed)
    codes = rng.integers(0, 16, size=(out, inp), dtype=np.uint8)
    scale = rng.uniform(0.001, 0.01, size=(out, inp // group)).astype(np.float16)
    bias = (0.02 * rng.standard_normal((out, inp // group))).astype(np.float16)
    return {"codes": codes, "packed": pack_q4(codes), "scale": scale, "bias": bias}


def q4_activations(inp: int, ntok: int, seed: int) -> np.ndarray:
    """x ~ N(0, 1) rounded to bf16, shape [ntok, in] as bf16 bits."""
    x = np.random.default_rng(seed).standard_normal((ntok, inp), dtype=np.float32)
    return f32_to_bf16_bits(x)


def decoder_weights_q4(s: DecoderShape, seed: int = 1, group: int = 64) -> dict:
    """Random 4-bit decoder: every projection and the tied embedding groupwise-affine.

    Draw order from ``numpy.random.default_rng(seed)`` as in decoder_weights
    (embed, each layer's LAYER_TENSORS, g_final). A matrix draws its codes
    U{0..15}, then s ~ U(0.004, 0.008) and b = -7.5 s + 0.002 N(0, 1) per
    64-column group (fp16), so w = s q + b is centred near zero with a spread
    close to the 0.02 N(0, 1) float draws. Gains are 1 + 0.1 N(0, 1), float32.

    Matrices are {"packed": uint32 [out, in/8], "scale", "bias": float16
    [out, in/64]}. Returns {"embed", "g_final", "layers", "wdtype": "q4"}.
    """
    rng = np.random.default_rng(seed)
    shapes = tensor_shapes(s)

    def draw(name):
        shp = shapes[name]
        if name.startswith("g_"):
            z = rng.standard_normal(int(np.prod(shp)), dtype=np.float32).reshape(shp)
            return (np.float32(1.0) + np.float32(0.1) * z).astype(np.float32)
        out, inp = shp
        if inp % group:
            raise ValueError("in must be a multiple of the group size")
        codes = rng.integers(0, 16, size=(out, inp), dtype=np.uint8)
        sc = rng.uniform(0.004, 0.008, size=(out, inp // group)).astype(np.float16)
        bi = (-7.5 * sc.astype(np.float64) + 0.002 * rng.standard_normal((out, inp // group))).astype(np.float16)
        return {"packed": pack_q4(codes), "scale": sc, "bias": bi}

    out = {"embed": draw("embed"), "layers": []}
    for _ in range(s.layers):
        out["layers"].append({name: draw(name) for name in LAYER_TENSORS})
    out["g_final"] = draw("g_final")
    out["wdtype"] = "q4"
    return out
