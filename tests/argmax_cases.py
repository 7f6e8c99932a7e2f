"""Planted logit patterns for GPU tests of the greedy argmax rule.

The rule ("Megakernels", "GPU-wide end-to-end generation"): the greedy token is
the lowest token ID among the largest logits. With the readings of the design
notes: NaN never wins, -0 and +0 are equal (so they tie), and an all-NaN vector
gives token 0 with the DEC_DEVERR_ARGMAX_NAN bit.

How the patterns reach a head. The head computes logits = E x with
x = RMSNorm(h) * g. With a gain g that is zero in every column but k, every
x_j (j != k) is a signed zero, so every logit is E[i, k] * x_k plus signed
zeros: the same value whatever order a kernel sums in. Equal entries of
column k therefore give bit-equal logits (exact ties), a zero entry gives a
zero logit, and one NaN anywhere in a row makes that row's logit NaN for
every k (NaN * 0 is NaN). Each case uses its own column (and, for the 4-bit
format, its own 64-column group), so one matrix holds every case and a test
selects a case by its gain.

The expected tokens follow from the pattern alone (and from the sign of x_k,
which the caller makes positive); no kernel output is used to build them.
"""
from __future__ import annotations

import numpy as np

VOCAB = 151936

# Rows whose logit is NaN in every case (a NaN in column NAN_COL).
NAN_ROWS = (0, 2, 64, 70000, 151900)
NAN_COL = 330

# name, column, kind, planted rows. Rows span one warp (adjacent rows), several
# warps and 256-row chunks of one CTA, and CTAs far apart (152 CTAs cover the
# vocabulary in ranges of about 1000 rows).
CASES = (
    ("tie_near", 4, "tie", (70001, 70002, 70017, 70300, 71999, 151935)),
    ("tie_far", 68, "tie", (151935, 99001, 99000, 5)),
    ("signed_zeros", 133, "zero", (120000, 4001, 4000, 150001)),
    ("single_max_after_nans", 196, "tie", (151934,)),
    ("all_nan", 260, "all_nan", ()),
)

TIE_VALUE = 1.0  # column-k value of tied rows: far above 0.02 N(0, 1) draws


def expected(kind: str, rows) -> tuple[int, bool]:
    """(token, all_nan) the rule gives for a planted case."""
    if kind == "all_nan":
        return 0, True
    return min(rows), False


def fed_rows() -> set:
    """Rows a test must not feed as tokens (their embeddings carry the patterns)."""
    s = set(NAN_ROWS)
    for _, _, _, rows in CASES:
        s.update(rows)
    return s


def plant_float(E: np.ndarray) -> np.ndarray:
    """Plant every case into a float32 [V, H] matrix (a modified copy)."""
    E = np.array(E, dtype=np.float32, copy=True)
    assert E.shape[0] == VOCAB and E.shape[1] > NAN_COL
    for _, col, kind, rows in CASES:
        if kind == "tie":
            E[list(rows), col] = TIE_VALUE
        elif kind == "zero":
            E[:, col] = -(np.abs(E[:, col]) + np.float32(1e-3))
            E[list(rows), col] = 0.0
    E[list(NAN_ROWS), NAN_COL] = np.nan
    return E


def _set_code(packed: np.ndarray, rows, col: int, q: int):
    w, j = col // 8, col % 8
    mask = np.uint32(0xF << (4 * j))
    packed[rows, w] = (packed[rows, w] & ~mask) | np.uint32(q << (4 * j))


def plant_q4(m: dict, group: int = 64) -> dict:
    """Plant every case into a 4-bit matrix {"packed", "scale", "bias"} (modified copies).

    Tied rows: code 15, scale and bias 0.01 in the case's group, so
    w = 0.16 there (other rows' w = s q + b stays within about +-0.07).
    Signed zeros: code 0 in the column for every row, bias -(|b| + 1e-3) in
    the group, bias 0 for the planted rows, so the logits are b * x_k: zero for
    the planted rows, negative for the rest. NaN rows: a NaN scale.
    """
    packed = m["packed"].copy()
    scale = m["scale"].copy()
    bias = m["bias"].copy()
    groups = [NAN_COL // group] + [c // group for _, c, _, _ in CASES]
    assert len(set(groups)) == len(groups), "each case needs its own group"
    for _, col, kind, rows in CASES:
        g = col // group
        if kind == "tie":
            r = list(rows)
            _set_code(packed, r, col, 15)
            scale[r, g] = np.float16(0.01)
            bias[r, g] = np.float16(0.01)
        elif kind == "zero":
            _set_code(packed, slice(None), col, 0)
            bias[:, g] = (-(np.abs(bias[:, g].astype(np.float32)) + np.float32(1e-3))).astype(np.float16)
            bias[list(rows), g] = np.float16(0.0)
    scale[list(NAN_ROWS), NAN_COL // group] = np.float16(np.nan)
    return {"packed": packed, "scale": scale, "bias": bias}


def gain_for(col: int, hidden: int, sign: float, kind: str) -> np.ndarray:
    """Gain selecting column col with x_col of the given sign (NaN for the all-NaN case)."""
    g = np.zeros(hidden, dtype=np.float32)
    g[col] = np.float32(np.nan) if kind == "all_nan" else np.float32(1.0 if sign >= 0 else -1.0)
    return g
