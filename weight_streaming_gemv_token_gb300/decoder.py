"""Decoder: owns a workspace tensor and a dec_ctx, and marshals weights to the C ABI.

PyTorch provides device memory and the stream; every step of the forward
runs in libwsg.so's kernels.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import binding as B

_LAYER_KEYS = ("w_q", "w_k", "w_v", "w_o", "w_gate", "w_up", "w_down", "g_in", "g_post", "g_q", "g_k")


def q4_blob(m: dict, device="cuda") -> torch.Tensor:
    """One device buffer holding a 4-bit matrix as the C ABI takes it: codes, then scales, then biases."""
    parts = [np.ascontiguousarray(m[k]).view(np.uint8).reshape(-1) for k in ("packed", "scale", "bias")]
    return torch.from_numpy(np.concatenate(parts)).to(device)


def to_device(a, device="cuda") -> torch.Tensor:
    """numpy array -> device tensor; uint16 arrays are taken as bfloat16 bit patterns."""
    if isinstance(a, torch.Tensor):
        return a.to(device).contiguous()
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


class Decoder:
    """Batch-1 decoder on the current CUDA device.

    shape: an object with layers, hidden, inter, n_q, n_kv, head_dim, vocab,
    eps, rope_theta. weights: dict as made by workloads.decoder_weights
    (numpy) or the same layout of device tensors. lossless: with float32
    weights, store them as bfloat16 when every value is one (self.lossless
    tells whether that happened).
    """

    def __init__(self, shape, weights: dict, kv_dtype: str = "f32", max_seq: int = 4096, chunk_cap: int = 0,
                 stream: torch.cuda.Stream | None = None, engine: str = "persistent", lossless: bool = False):
        wd = weights.get("wdtype", "f32")
        self.shape = shape
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        # device copies of the weights; kept alive as long as the context
        up = q4_blob if wd == "q4" else to_device
        self.dev = {"embed": up(weights["embed"]), "g_final": to_device(weights["g_final"]),
                    "layers": [{k: (to_device if k.startswith("g_") else up)(lw[k]) for k in _LAYER_KEYS}
                               for lw in weights["layers"]]}
        # Lossless storage ("Megakernels", "Lossless decode-weight storage"): float32 projections
        # and embedding whose values are all bfloat16 values are kept as their bfloat16 halves and
        # run on the bfloat16-weight kernels; any inexact tensor keeps the whole model in float32.
        self.lossless = False
        if lossless and wd == "f32":
            self.stream.wait_stream(torch.cuda.current_stream())  # the uploads above
            packed, bad = {}, 0
            names = [("embed", None)] + [(k, i) for i in range(shape.layers) for k in _LAYER_KEYS
                                         if not k.startswith("g_")]
            for k, i in names:
                src = self.dev[k] if i is None else self.dev["layers"][i][k]
                dst = torch.empty(src.shape, dtype=torch.bfloat16, device="cuda")
                bad += B.pack_bf16_exact(src, dst, src.numel(), self.stream)
                packed[(k, i)] = dst
            if bad == 0:
                for (k, i), t in packed.items():
                    if i is None:
                        self.dev[k] = t
                    else:
                        self.dev["layers"][i][k] = t
                wd, self.lossless = "bf16", True
            del packed
        self.cfg = B.dec_config(
            layers=shape.layers, hidden=shape.hidden, inter=shape.inter, n_q=shape.n_q, n_kv=shape.n_kv,
            head_dim=shape.head_dim, vocab=shape.vocab, eps=shape.eps, rope_theta=shape.rope_theta,
            wdtype={"f32": B.DEC_F32, "bf16": B.DEC_BF16, "q4": B.DEC_Q4G64}[wd],
            kvdtype=B.DEC_F32 if kv_dtype == "f32" else B.DEC_BF16,
            max_seq=max_seq, chunk_cap=chunk_cap,
            engine=B.DEC_ENGINE_PERSISTENT if engine == "persistent" else B.DEC_ENGINE_STAGED)
        self.kv_dtype = kv_dtype
        nbytes = B.dec_workspace_bytes(self.cfg)
        if nbytes == 0:
            raise B.WsgError(B.DEC_EINVAL, "invalid decoder configuration")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        self.ctx = B.dec_create(self.cfg, self.workspace, nbytes, self.stream)
        arr = (B.dec_layer_weights * shape.layers)()
        for i, lw in enumerate(self.dev["layers"]):
            for k in _LAYER_KEYS:
                setattr(arr[i], k, lw[k].data_ptr())
        self._layer_arr = arr
        w = B.dec_weights(embed=self.dev["embed"].data_ptr(), g_final=self.dev["g_final"].data_ptr(),
                          layers=ctypes.cast(arr, ctypes.POINTER(B.dec_layer_weights)))
        B.dec_load_weights(self.ctx, w)

    def close(self):
        if getattr(self, "ctx", None):
            B.dec_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- calls ---------------------------------------------------------------
    def reset(self):
        B.dec_reset(self.ctx)

    def rewind(self, pos: int):
        """Back to position pos (<= the current one); the next forward overwrites cache slot pos."""
        B.dec_rewind(self.ctx, pos)

    @property
    def position(self) -> int:
        return B.dec_position(self.ctx)

    def step(self, token: int, logits: torch.Tensor | None = None, skip_logits: bool = False):
        if skip_logits:
            return B.dec_step(self.ctx, int(token), B.DEC_SKIP_LOGITS, None, want_next=False)
        return B.dec_step(self.ctx, int(token), 0, logits, want_next=True)

    def verify2(self, tokens, logits: torch.Tensor | None = None) -> tuple[int, int]:
        """Two-token verify step (4-bit configuration): rows at p and p+1; the greedy token after each."""
        return B.dec_verify2(self.ctx, tokens, logits)

    def prefill(self, tokens, is_last: bool = True, logits: torch.Tensor | None = None):
        return B.dec_prefill_chunk(self.ctx, tokens, is_last, logits if is_last else None, want_next=is_last)

    def generate(self, token: int, n: int, out: torch.Tensor | None = None) -> torch.Tensor:
        if out is None:
            out = torch.empty(n, dtype=torch.int32, device="cuda")
        B.dec_generate(self.ctx, int(token), n, out)
        return out

    def kv(self, layer: int) -> tuple[torch.Tensor, torch.Tensor, int]:
        """(K, V, n_valid): views of the cache, each [n_kv, max_seq, head_dim]."""
        k, v, n = B.dec_get_kv(self.ctx, layer)
        base = self.workspace.data_ptr()
        s = self.shape
        elem = 4 if self.kv_dtype == "f32" else 2
        count = s.n_kv * self.cfg.max_seq * s.head_dim
        dt = torch.float32 if self.kv_dtype == "f32" else torch.bfloat16

        def view(p):
            off = p - base
            return self.workspace[off: off + count * elem].view(dt).view(s.n_kv, self.cfg.max_seq, s.head_dim)

        return view(k), view(v), n

    def set_wait_limit(self, ns: int):
        """Limit of the persistent engines' waits on other CTAs (0: the 2 s default)."""
        B.dec_set_wait_limit(self.ctx, ns)

    def device_errors(self, clear: bool = True) -> int:
        return B.dec_device_errors(self.ctx, clear)
