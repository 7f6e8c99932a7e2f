"""Oracle decoder: the batch-1 Qwen3-shaped token-to-logits forward in float64.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline leg use this module; the product path never imports it.

It writes out the forward of the "Megakernels" page, section "What runs in the
DSL":

    token ID -> embedding
    per layer: RMSNorm -> Q/K/V projections -> per-head Q/K RMSNorm -> RoPE
               -> grouped-query attention + KV update -> output projection
               -> residual add -> RMSNorm -> gate/up projections -> SwiGLU
               -> down projection -> residual add
    final RMSNorm -> tied vocabulary projection -> logits

and the generation protocol of "GPU-wide end-to-end generation": the first
output comes from the final prompt row, every later output is the forward of
the previous output at the next position, so P prompt tokens and N outputs
leave P + N - 1 cache entries.

Arithmetic is float64 throughout. The only rounding is the storage format of
the KV cache in the BF16 configuration, where cached keys and values are
bfloat16 ("Weights, cached keys/values ... use the selected dtype").

Readings of points the pages leave open (each also listed in the design notes):
  * gains multiply the normalised vector (y = x_hat * g); one g_q and one g_k
    of length head_dim per layer, shared by all heads; values are not normed;
  * RoPE pairs (i, i + d/2), angle = pos * theta^(-2i/d), absolute position;
  * query head h uses key/value head h // (n_q / n_kv);
  * cached keys are post-norm, post-RoPE; cached values are the raw projection;
  * no biases anywhere; the embedding matrix doubles as the vocabulary head;
  * the 4-bit configuration is this same forward on the exact dequantised
    weights s * q + b of the 4-bit groupwise-affine format ("Our Kernel
    Benchmark Was Measuring the System Cache", Summary): the pages fix the
    weight format, not the precision of the activations inside the decoder,
    so the activations stay those of the float forward.
"""
from __future__ import annotations

import numpy as np

from . import primitives as P


class OracleDecoder:
    """Plain float64 decoder with its own KV cache.

    ``weights`` is the dict produced by the seeded generator: "embed" [V, H],
    "g_final" [H] and "layers", a list of dicts with w_q [n_q*d, H],
    w_k/w_v [n_kv*d, H], w_o [H, n_q*d], w_gate/w_up [I, H], w_down [H, I],
    g_in/g_post [H], g_q/g_k [d]. Arrays may be float32 or bf16 bit patterns.
    """

    def __init__(self, shape, weights: dict, kv_dtype: str = "f32", max_seq: int = 4096):
        if kv_dtype not in ("f32", "bf16"):
            raise ValueError(kv_dtype)
        self.s = shape
        self.kv_dtype = kv_dtype
        self.max_seq = int(max_seq)
        self.E = P.widen(weights["embed"])
        self.g_final = P.widen(weights["g_final"])
        self.layers = [{k: P.widen(v) for k, v in lw.items()} for lw in weights["layers"]]
        self.reset()

    # -- state -------------------------------------------------------------
    def reset(self):
        s = self.s
        self.pos = 0
        self.K = np.zeros((s.layers, s.n_kv, self.max_seq, s.head_dim))
        self.V = np.zeros((s.layers, s.n_kv, self.max_seq, s.head_dim))

    def _store(self, x):
        return P.round_to_bf16(x) if self.kv_dtype == "bf16" else x

    def kv(self, layer: int):
        """(K, V) cache of one layer, [n_kv, n_valid, d], as stored."""
        return self.K[layer, :, : self.pos], self.V[layer, :, : self.pos]

    # -- one token -----------------------------------------------------------
    def body(self, token: int) -> np.ndarray:
        """Decoder body for one token at the current position; writes the cache, advances pos.

        Returns the final residual stream h [H] (before the final RMSNorm).
        """
        s = self.s
        p = self.pos
        if p >= self.max_seq:
            raise IndexError("KV cache full")
        d, eps = s.head_dim, s.eps
        h = self.E[int(token)].copy()
        for l, w in enumerate(self.layers):
            x = P.rmsnorm(h, w["g_in"], eps)
            q = (w["w_q"] @ x).reshape(s.n_q, d)
            k = (w["w_k"] @ x).reshape(s.n_kv, d)
            v = (w["w_v"] @ x).reshape(s.n_kv, d)
            q = P.rope(P.rmsnorm(q, w["g_q"], eps), p, s.rope_theta)
            k = P.rope(P.rmsnorm(k, w["g_k"], eps), p, s.rope_theta)
            self.K[l, :, p] = self._store(k)
            self.V[l, :, p] = self._store(v)
            o = P.gqa_decode_attention(q, self.K[l, :, : p + 1], self.V[l, :, : p + 1])
            h = h + w["w_o"] @ o.reshape(-1)
            x = P.rmsnorm(h, w["g_post"], eps)
            h = h + w["w_down"] @ P.swiglu(w["w_gate"] @ x, w["w_up"] @ x)
        self.pos = p + 1
        return h

    def head(self, h) -> np.ndarray:
        """Final RMSNorm and tied vocabulary projection: logits [V]."""
        return self.E @ P.rmsnorm(h, self.g_final, self.s.eps)

    def step(self, token: int) -> np.ndarray:
        """Full token-to-logits forward at the current position."""
        return self.head(self.body(token))

    # -- many rows at once -------------------------------------------------------
    def prefill(self, tokens, logit_rows=None) -> dict:
        """Forward of consecutive prompt rows at positions pos..pos+T-1, batched.

        Megakernels, "Chunked prefill for long prompts": rows of one request,
        each attending to its whole causal prefix. The same mathematics as T
        calls of ``body``, written with matrix products over the rows.
        Returns {"logits": {row: logits}} for the requested rows (default:
        the last row only).
        """
        s = self.s
        tokens = np.asarray(tokens, dtype=np.int64)
        T = len(tokens)
        p0 = self.pos
        if p0 + T > self.max_seq:
            raise IndexError("KV cache full")
        if logit_rows is None:
            logit_rows = [T - 1]
        d, eps = s.head_dim, s.eps
        pos = p0 + np.arange(T)
        Hs = self.E[tokens]
        for l, w in enumerate(self.layers):
            X = P.rmsnorm(Hs, w["g_in"], eps)
            Q = (X @ w["w_q"].T).reshape(T, s.n_q, d)
            K = (X @ w["w_k"].T).reshape(T, s.n_kv, d)
            V = (X @ w["w_v"].T).reshape(T, s.n_kv, d)
            Q = P.rope(P.rmsnorm(Q, w["g_q"], eps), pos[:, None], s.rope_theta)
            K = P.rope(P.rmsnorm(K, w["g_k"], eps), pos[:, None], s.rope_theta)
            self.K[l, :, p0 : p0 + T] = self._store(K).transpose(1, 0, 2)
            self.V[l, :, p0 : p0 + T] = self._store(V).transpose(1, 0, 2)
            O = P.causal_prefill_attention(Q, self.K[l, :, : p0 + T], self.V[l, :, : p0 + T], p0)
            Hs = Hs + O.reshape(T, -1) @ w["w_o"].T
            X = P.rmsnorm(Hs, w["g_post"], eps)
            Hs = Hs + P.swiglu(X @ w["w_gate"].T, X @ w["w_up"].T) @ w["w_down"].T
        self.pos = p0 + T
        return {"logits": {int(r): self.head(Hs[r]) for r in logit_rows}}


def generate(model: OracleDecoder, prompt, n_out: int, forced=None, keep_logits=True) -> dict:
    """Greedy generation with the pages' protocol (EOS ignored).

    Prompt tokens run one at a time through the body; the final prompt row
    gives the first output. Output j >= 2 is the forward of output j-1. With
    ``forced`` (a token sequence from another implementation), the oracle
    feeds those tokens instead of its own choices (teacher forcing) while
    still reporting its own argmax and logits at every step.

    Returns {"tokens": own argmax per output, "logits": list of [V] arrays}.
    """
    prompt = [int(t) for t in prompt]
    for t in prompt[:-1]:
        model.body(t)
    logits_all, toks = [], []
    cur = prompt[-1]
    for j in range(n_out):
        lg = model.step(cur)
        nxt, _ = P.argmax_lowest(lg)
        toks.append(nxt)
        if keep_logits:
            logits_all.append(lg)
        if j + 1 < n_out:
            cur = int(forced[j]) if forced is not None else nxt
    return {"tokens": toks, "logits": logits_all}
