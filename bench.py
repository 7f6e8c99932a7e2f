"""Benchmark: batch-1 decode tokens/s of the Qwen3-0.6B-shaped decoder, plus cold GEMV GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one token-to-logits forward with greedy argmax (the whole decode
hot path: embedding, 28 layers, final norm, tied vocabulary projection,
argmax). Steps run back to back through dec_generate, each reading the
previous step's token on the device. The FP32 weights stream 2.4 GB per step,
far beyond the 129 MB L2, so every step is cold by construction.

Beside the headline line the JSON carries:
  e2e         the same metric through dec_step with host token in / host token
              out every step (4 B each way, host synchronisation included);
  roofline    the dominant kernel (the GEMV streaming engine at the gate/up
              shape) against the measured HBM copy bandwidth;
  gemv_cold   cold GB/s of gemv / gemv_q4 on the five layer shapes, each
              cycling >= 1 GiB of distinct matrices;
  cpu_baseline the float64 oracle's decode rate on the host cores;
  q4_decoder  the same decoder with 4-bit weights (staged engine): decode
              rate against its own step roofline, and the two-token verify step.

--impl reference times the oracle (the CPU restatement of the same forward)
on a bounded sample of the same workload, on the host cores.

N > 1: independent replicas, one per GPU (the batch-1 step does not shard);
value is the total tokens/s over all ranks, timed by the slowest rank.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as Wl  # noqa: E402

METRIC = "batch-1 decode tokens/s + cold GEMV HBM GB/s (% of GB300 peak), 1 GPU"

# DRAM traffic of the persistent decode kernel per algorithmic byte, from an ncu capture of a
# 4-layer / 32768-vocabulary case of the same widths. The last capture, (387,498,496 read +
# 2,787,584 written) / 387,186,688 algorithmic bytes = 1.008, predates the decode attention's
# change to request each warp's next key and value chunks later in its loop (the same rows, read
# once each), so the figure is not reported until it is measured again.
MK_TRAFFIC_PER_ALG_BYTE = None
# DRAM bytes (read + written) per launch of the standalone gemv bulk-copy kernel at 151936x1024 f32
# (the tied vocabulary shape), from an ncu capture: 622,377,984 B read + 3,492,352 B written; None
# until measured for the current kernel.
GEMV_TRAFFIC = 622377984 + 3492352
GEMV_ROOF_SHAPE = (151936, 1024)
PROMPT = 32


def measured_bf16_tflops():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if "bf16_tflops" in d:
            return float(d["bf16_tflops"])
    return 1900.0


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class Clocks:
    """Samples SM clocks and throttle reasons with nvidia-smi while a region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def dist_setup():
    import torch
    import torch.distributed as dist

    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return ws, rank, local


def barrier_max(value: float, ws: int) -> float:
    """The largest value over the ranks (the slowest rank's time); NCCL reduces on the GPU, gloo on the CPU."""
    if ws == 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


# ---------------------------------------------------------------- GPU arm ----

def bytes_per_step(s, pos):
    """Algorithmic bytes of one FP32 decode step at position pos: every weight once plus the KV read."""
    H, I, d = s.hidden, s.inter, s.head_dim
    per_layer = (s.q_width + 2 * s.kv_width) * H + H * s.q_width + 2 * I * H + H * I
    weights = s.layers * per_layer + s.vocab * H
    kv = s.layers * 2 * s.kv_width * (pos + 1)
    return 4 * (weights + kv) + 4 * s.vocab  # plus the logits write


def time_gemv_cold(W, torch, dtype, out, inp, stream, rounds=5, min_bytes=1 << 30, ntok=1, gen=None):
    """Cold GB/s: cycle >= 1 GiB of distinct matrices; returns (GB/s, bytes per launch, avg launch s, launches)."""
    if dtype == "q4":
        per = out * inp // 2 + out * (inp // 64) * 4
    else:
        per = out * inp * (4 if dtype == "f32" else 2)
    count = max(2, -(-min_bytes // per))
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    if dtype == "q4":
        codes = [torch.randint(-2**31, 2**31 - 1, (out, inp // 8), dtype=torch.int32, device="cuda", generator=gen)
                 for _ in range(count)]
        sc = [torch.empty((out, inp // 64), dtype=torch.float16, device="cuda").uniform_(0.001, 0.01, generator=gen)
              for _ in range(count)]
        bi = [torch.empty((out, inp // 64), dtype=torch.float16, device="cuda").normal_(0, 0.02, generator=gen)
              for _ in range(count)]
        x = torch.randn((ntok, inp), device="cuda", generator=gen).to(torch.bfloat16)
        y = torch.empty((ntok, out), device="cuda")

        def call(i, st):
            W.gemv_q4(codes[i], sc[i], bi[i], x, y, out, inp, ntok, st)
        per_launch = per + ntok * (inp * 2 + out * 4)
    else:
        mats = [(0.02 * torch.randn((out, inp), device="cuda", generator=gen)).to(tdt) for _ in range(count)]
        x = (0.02 * torch.randn(inp, device="cuda", generator=gen)).to(tdt)
        y = torch.empty(out, device="cuda")
        code = W.DEC_F32 if dtype == "f32" else W.DEC_BF16

        def call(i, st):
            W.gemv(code, mats[i], x, y, out, inp, st)
        per_launch = per + inp * (4 if dtype == "f32" else 2) + out * 4
    # One graph launches every matrix once (back to back, with the launch
    # edges the library sets); replaying it removes host launch overhead.
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        for i in range(count):  # warm-up outside capture: lazy set-up happens here
            call(i, cap)
    cap.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=cap):
        for i in range(count):
            call(i, cap)
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = rounds * count
    e0.record(stream)
    for r in range(rounds):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / 1e3
    avg = sec / n
    del graph
    if dtype == "q4":
        del codes, sc, bi
    else:
        del mats
    torch.cuda.empty_cache()
    return per_launch / avg / 1e9, per_launch, avg, n


def lossless_config(W, torch, stream, headline_embed, hbm, K=200):
    """Lossless bfloat16 storage of float32 weights ("Megakernels", "Lossless decode-weight
    storage"): the float32 Qwen3-0.6B-shaped model converted from bfloat16 (every weight has zero
    low 16 bits) decodes from float32 storage and from its packed bfloat16 halves (same values);
    the headline model's random float32 weights are checked for eligibility too."""
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    s = Wl.QWEN3_06B
    emb = torch.from_numpy(headline_embed).cuda()
    tmp = torch.empty(emb.shape, dtype=torch.bfloat16, device="cuda")
    bad = W.pack_bf16_exact(emb, tmp, emb.numel(), stream)
    del emb, tmp
    w = Wl.decoder_weights(s, seed=1, wdtype="f32_from_bf16")
    prompt = Wl.prompt_uniform(PROMPT, s.vocab, seed=0)
    res = {"workload": "Qwen3-0.6B-shaped decoder, float32 weights converted from bfloat16, float32 KV, "
                       f"{K} greedy steps after a {PROMPT}-token prompt",
           "headline_weights_eligible": bad == 0, "headline_embedding_inexact_values": int(bad)}
    toks = {}
    for packed in (False, True):
        dec = Decoder(s, w, kv_dtype="f32", max_seq=PROMPT + K + 32, stream=stream, lossless=packed)
        assert dec.lossless == packed
        first = dec.prefill(prompt, is_last=True)
        warm = dec.generate(first, 8)
        torch.cuda.synchronize()
        out = torch.empty(K, dtype=torch.int32, device="cuda")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dec.generate(int(warm[-1].item()), K, out)
        e1.record(stream)
        torch.cuda.synchronize()
        assert dec.device_errors() == 0
        toks[packed] = out.cpu()
        sec = e0.elapsed_time(e1) / 1e3
        elem = 2 if packed else 4
        shp = Wl.tensor_shapes(s)
        per_layer = sum(int(np.prod(shp[k])) for k in Wl.LAYER_TENSORS if not k.startswith("g_"))
        wbytes = elem * (int(np.prod(shp["embed"])) + s.layers * per_layer)
        res["packed" if packed else "float32"] = {
            "tokens_per_s": round(K / sec, 1), "ms_per_step": round(sec / K * 1e3, 4),
            "weight_bytes_per_step": wbytes, "weight_GB/s": round(wbytes * K / sec / 1e9, 1)}
        dec.close()
        del dec
    res["same_tokens"] = bool(torch.equal(toks[False], toks[True]))
    torch.cuda.empty_cache()
    return res


def fixed_context_latency(dec, torch, s, stream, contexts=(0, 16, 64), trials=9, warm=3):
    """Decode-forward latency at a fixed cache slot ("Megakernels", "Fixed-context methodology"):
    after `ctx` prompt tokens, each trial rewinds to slot ctx and runs one full forward of the same
    token (host token in, greedy token read back); median over the trials, wall clock and CUDA events."""
    toks = [int(t) for t in Wl.prompt_uniform(max(contexts) + 1, s.vocab, seed=0)]
    res = {}
    for ctx in contexts:
        dec.reset()
        if ctx:
            dec.prefill(toks[:ctx], is_last=False)
        walls, devs, outs = [], [], set()
        for i in range(warm + trials):
            dec.rewind(ctx)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            e0.record(stream)
            nxt = dec.step(toks[ctx])
            e1.record(stream)
            torch.cuda.synchronize()
            wall = time.perf_counter() - t0
            outs.add(nxt)
            if i >= warm:
                walls.append(wall * 1e3)
                devs.append(e0.elapsed_time(e1))
        assert len(outs) == 1, "a repeated forward at one slot changed its token"
        res[str(ctx)] = {"median_ms": round(statistics.median(walls), 4), "device_median_ms": round(statistics.median(devs), 4),
                         "trials": trials}
    return res


def generation_timings(dec, torch, s, pairs=((8, 8), (8, 16), (32, 8), (32, 16)), warm=2, trials=5):
    """Greedy generation timed the pages' way ("Megakernels", "GPU-wide end-to-end generation";
    "Benchmark methodology", "Median of paired per-trial ratios"): from before the cache reset to
    the final token ID on the host, with the host reading every token (dec_step). TTFT ends when
    the first output (from the final prompt row) is on the host; the decode rate uses the N - 1
    forwards after it. Two warm-up generations, then the median of five trials, each of which must
    reproduce the warm-up's token IDs."""
    res = {}
    for P, N in pairs:
        prompt = [int(t) for t in Wl.prompt_uniform(P, s.vocab, seed=0)]
        ref, tt, tot, rate = None, [], [], []
        for i in range(warm + trials):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            dec.reset()
            cur = dec.prefill(prompt, is_last=True)
            t1 = time.perf_counter()
            toks = [cur]
            for _ in range(N - 1):
                cur = dec.step(cur)
                toks.append(cur)
            t2 = time.perf_counter()
            if ref is None:
                ref = toks
            assert toks == ref, f"generation {P}/{N}: a trial changed its token IDs"
            if i >= warm:
                tt.append((t1 - t0) * 1e3)
                tot.append((t2 - t0) * 1e3)
                rate.append((N - 1) / (t2 - t1))
        res[f"{P}/{N}"] = {"ttft_ms": round(statistics.median(tt), 3), "total_ms": round(statistics.median(tot), 3),
                           "decode_tokens_per_s": round(statistics.median(rate), 1), "trials": trials,
                           "outputs": len(ref)}
    return res


def time_q4_cold_rows(W, torch, out, inp, stream, ntok, rows_options, rounds=5, min_bytes=1 << 30, gen=None):
    """Cold GB/s of gemv_q4 for each rows-per-warp setting on one set of >= 1 GiB of distinct
    packed matrices (each setting captured in its own graph); {R: (GB/s, bytes per launch, avg s)}."""
    per = out * inp // 2 + out * (inp // 64) * 4
    count = max(2, -(-min_bytes // per))
    codes = [torch.randint(-2**31, 2**31 - 1, (out, inp // 8), dtype=torch.int32, device="cuda", generator=gen)
             for _ in range(count)]
    sc = [torch.empty((out, inp // 64), dtype=torch.float16, device="cuda").uniform_(0.001, 0.01, generator=gen)
          for _ in range(count)]
    bi = [torch.empty((out, inp // 64), dtype=torch.float16, device="cuda").normal_(0, 0.02, generator=gen)
          for _ in range(count)]
    x = torch.randn((ntok, inp), device="cuda", generator=gen).to(torch.bfloat16)
    y = torch.empty((ntok, out), device="cuda")
    per_launch = per + ntok * (inp * 2 + out * 4)
    res = {}
    prev = W.gemv_q4_rows_per_warp(ntok)
    try:
        for r in rows_options:
            W.gemv_q4_rows_per_warp(ntok, r)
            cap = torch.cuda.Stream()
            cap.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(cap):
                for i in range(count):
                    W.gemv_q4(codes[i], sc[i], bi[i], x, y, out, inp, ntok, cap)
            cap.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=cap):
                for i in range(count):
                    W.gemv_q4(codes[i], sc[i], bi[i], x, y, out, inp, ntok, cap)
            graph.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(rounds):
                graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            avg = e0.elapsed_time(e1) / 1e3 / (rounds * count)
            res[r] = (per_launch / avg / 1e9, per_launch, avg)
            del graph
    finally:
        W.gemv_q4_rows_per_warp(ntok, prev if prev > 0 else -1)
    del codes, sc, bi
    torch.cuda.empty_cache()
    return res


def prefill_config(W, torch, hbm, tflops_peak):
    """BF16 Qwen3-0.6B shape with chunked prefill (tensor-core projections): the
    chunk size is tuned on a 2048-token Zipf(1.1) prompt with 8 outputs, then a
    held-out 4096-token prompt (a different seed) decodes 1024 outputs at that
    chunk size. TTFT = prompt rows in + first token read back (wall clock)."""
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    s = Wl.QWEN3_06B
    w = Wl.decoder_weights(s, seed=1, wdtype="bf16")

    def ttft(dec, prompt, chunk):
        dec.reset()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for c0 in range(0, len(prompt), chunk):
            last = c0 + chunk >= len(prompt)
            nxt = dec.prefill([int(t) for t in prompt[c0:c0 + chunk]], is_last=last)
        return time.perf_counter() - t0, nxt

    tuning = {}
    prompt = Wl.prompt_zipf(2048, s.vocab, seed=0)
    for chunk in (128, 256, 512, 1024, 2048):
        dec = Decoder(s, w, kv_dtype="bf16", max_seq=2048 + 16, chunk_cap=chunk)
        ttft(dec, prompt, chunk)  # warm-up (lazy set-up)
        runs = [ttft(dec, prompt, chunk)[0] for _ in range(3)]
        dec.generate(ttft(dec, prompt, chunk)[1], 7)
        torch.cuda.synchronize()
        assert dec.device_errors() == 0
        tuning[chunk] = round(statistics.median(runs) * 1e3, 2)
        dec.close()
    best = min(tuning, key=lambda c: (tuning[c], c))  # exact ties go to the smaller chunk
    P, N = 4096, 1024
    prompt = Wl.prompt_zipf(P, s.vocab, seed=2)
    dec = Decoder(s, w, kv_dtype="bf16", max_seq=P + N + 8, chunk_cap=best)
    ttft(dec, prompt[:best], best)
    t_first, first = ttft(dec, prompt, best)
    out = torch.empty(N - 1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    dec.generate(first, N - 1, out)
    torch.cuda.synchronize()
    t_dec = time.perf_counter() - t0
    assert dec.device_errors() == 0
    dec.close()
    H, I, d = s.hidden, s.inter, s.head_dim
    per_layer = (s.q_width + 2 * s.kv_width) * H + H * s.q_width + 2 * I * H + H * I
    proj_flops = 2.0 * s.layers * per_layer * P
    attn_flops = 2.0 * 2 * s.layers * s.n_q * d * (P * (P + 1) / 2)
    mid = P + N // 2
    dec_bytes = 2 * (s.layers * per_layer + s.vocab * H) + 2 * s.layers * 2 * s.kv_width * (mid + 1) + 4 * s.vocab
    rate = (N - 1) / t_dec
    # the projection GEMM alone on one chunk of the chosen size (gate/up shape), timed on the device
    A = (torch.randn((best, H), device="cuda") * 0.5).to(torch.bfloat16)
    Wg = (0.02 * torch.randn((2 * I, H), device="cuda")).to(torch.bfloat16)
    C = torch.empty((best, 2 * I), device="cuda")
    st = torch.cuda.current_stream()
    for _ in range(3):
        W.gemm_bf16(A, Wg, C, best, 2 * I, H, stream=st)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(50):
        W.gemm_bf16(A, Wg, C, best, 2 * I, H, stream=st)
    e1.record(st)
    torch.cuda.synchronize()
    g_sec = e0.elapsed_time(e1) / 1e3 / 50
    g_tflops = 2.0 * best * 2 * I * H / g_sec / 1e12
    return {
        "workload": "Qwen3-0.6B-shaped decoder, BF16 weights and KV cache, chunked prefill (tcgen05 projections), "
                    "Zipf(1.1) prompts: chunk tuned on 2048 tokens / 8 outputs, held-out 4096 tokens / 1024 outputs",
        "tuning_ttft_ms": tuning, "chunk": best,
        "held_out": {"prompt": P, "outputs": N, "ttft_ms": round(t_first * 1e3, 2),
                     "decode_tokens_per_s": round(rate, 1), "total_s": round(t_first + t_dec, 3),
                     "decode_step_roofline_frac": round(dec_bytes * rate / 1e9 / hbm, 4),
                     "prefill_tflops_algorithmic": round((proj_flops + attn_flops) / t_first / 1e12, 2)},
        "gemm": {"shape": f"{best}x{2 * I}x{H} (chunk rows x gate/up rows x hidden)", "us": round(g_sec * 1e6, 2),
                 "tflops_algorithmic": round(g_tflops, 1), "peak": tflops_peak, "frac": round(g_tflops / tflops_peak, 4),
                 "note": "activation operand as bfloat16 value + remainder: 2 MMAs per product"},
    }


def q4_bytes_per_token(s, pos):
    """Algorithmic bytes of one 4-bit forward at position pos: every 4-bit matrix once (codes
    half a byte per weight, an fp16 scale and bias per 64 weights), the float32 K/V rows 0..pos
    of every layer, the cache row written, the logits written."""
    per_w = 0.5 + 4.0 / 64
    per_layer = (s.q_width + 2 * s.kv_width) * s.hidden + s.hidden * s.q_width + 2 * s.inter * s.hidden + \
        s.hidden * s.inter
    weights = (s.layers * per_layer + s.vocab * s.hidden) * per_w
    kv = s.layers * 2 * s.kv_width * 4 * (pos + 1)
    return int(weights + kv + 4 * s.vocab)


def q4_config(W, torch, stream, hbm, steps=256, verifies=64):
    """Qwen3-0.6B shape in the 4-bit configuration: greedy decode rate after a 32-token prompt on
    the persistent engine (one cooperative launch for all steps) and on the staged engine (a CUDA
    graph per step), and the two-token verify step back to back."""
    w = Wl.decoder_weights_q4(Wl.QWEN3_06B, seed=1)
    res = q4_engine(W, torch, stream, hbm, w, "staged", steps, verifies)
    pers = q4_engine(W, torch, stream, hbm, w, "persistent", steps, verifies)
    res["persistent_engine"] = {k: pers[k] for k in ("decode_tokens_per_s", "ms_per_step", "frac", "gpu_launches_per_step")}
    return res


def q4_engine(W, torch, stream, hbm, w, engine, steps, verifies):
    from weight_streaming_gemv_token_gb300 import binding as B
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    s = Wl.QWEN3_06B
    prompt = Wl.prompt_uniform(PROMPT, s.vocab, seed=0)
    dec = Decoder(s, w, kv_dtype="f32", max_seq=PROMPT + 8 + steps + 2 * (verifies + 4) + 8, stream=stream,
                  engine=engine)
    first = dec.prefill(prompt, is_last=True)
    out = torch.empty(steps + 4, dtype=torch.int32, device="cuda")
    dec.generate(first, 4, out[:4])
    torch.cuda.synchronize()
    tok = int(out[3].item())
    pos0 = dec.position
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    dec.generate(tok, steps, out[4:])
    e1.record(stream)
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / 1e3
    rate = steps / sec
    bpt = q4_bytes_per_token(s, pos0 + steps // 2)
    # verify steps back to back (no read-back), then one with the tokens read back
    pair = [int(out[steps + 3].item()), int(out[steps + 2].item())]
    for _ in range(3):
        B.dec_verify2(dec.ctx, pair, None, want_next=False)
    torch.cuda.synchronize()
    vpos = dec.position
    e0.record(stream)
    for _ in range(verifies):
        B.dec_verify2(dec.ctx, pair, None, want_next=False)
    e1.record(stream)
    torch.cuda.synchronize()
    vsec = e0.elapsed_time(e1) / 1e3 / verifies
    vb = q4_bytes_per_token(s, vpos + verifies) + s.layers * 2 * s.kv_width * 4 * (vpos + verifies + 2) + 4 * s.vocab
    assert dec.device_errors() == 0
    dec.close()
    return {
        "workload": "Qwen3-0.6B-shaped decoder, 4-bit groupwise-affine weights (all projections and the tied head), "
                    f"FP32 KV, {engine} engine, greedy decode after a {PROMPT}-token prompt",
        "decode_tokens_per_s": round(rate, 1), "ms_per_step": round(sec / steps * 1e3, 4),
        "bytes_per_token": bpt, "achieved_GB/s": round(bpt * rate / 1e9, 1), "peak": hbm,
        "frac": round(bpt * rate / 1e9 / hbm, 4), "roofline_tokens_per_s": round(hbm * 1e9 / bpt, 1),
        "gpu_launches_per_step": round(1 / steps, 4) if engine == "persistent" else 5 * s.layers + 3,
        "verify2": {"ms_per_call": round(vsec * 1e3, 4), "rows_per_s": round(2 / vsec, 1),
                    "vs_two_steps": round(2 * sec / steps / vsec, 3), "bytes_per_call": vb,
                    "frac": round(vb / vsec / 1e9 / hbm, 4)},
    }


def summary(line):
    """The line's figures in a few hundred characters: fractions of the measured peak per GEMV
    shape (in the order of workloads.GEMV_SHAPES), the generation timings (TTFT ms, total ms,
    decode tokens/s), the 4-bit and chunked-prefill configurations and the oracle on the CPU."""
    def r3(v):
        return None if v is None else round(v, 3)

    out = {"tok_s": line["value"], "step_frac": line["step_roofline"]["frac"], "e2e_tok_s": line["e2e"]["value"]}
    g = line.get("gemv_cold")
    if g:
        for dt, key in (("f32", "f32"), ("bf16", "bf16"), ("q4 ntok=1", "q4n1"), ("q4 ntok=2", "q4n2")):
            out[f"gemv_frac_{key}"] = [r3(g.get(f"{dt} {o}x{i}", {}).get("frac")) for (o, i) in Wl.GEMV_SHAPES]
    gen = line.get("generation")
    if gen:
        out["gen_ttft_total_rate"] = {k: [v["ttft_ms"], v["total_ms"], v["decode_tokens_per_s"]] for k, v in gen.items()}
    q = line.get("q4_decoder")
    if q:
        pe = q.get("persistent_engine", {})
        out["q4"] = {"staged_tok_s": q["decode_tokens_per_s"], "staged_frac": q["frac"],
                     "persistent_tok_s": pe.get("decode_tokens_per_s"), "persistent_frac": pe.get("frac"),
                     "verify2_ms": q["verify2"]["ms_per_call"]}
    p = line.get("prefill")
    if p:
        h = p["held_out"]
        out["prefill"] = {"chunk": p["chunk"], "ttft_ms": h["ttft_ms"], "decode_tok_s": h["decode_tokens_per_s"],
                          "decode_frac": h["decode_step_roofline_frac"], "tflops": h["prefill_tflops_algorithmic"]}
    c = line.get("cpu_baseline")
    if c:
        one = c.get("one_core") or {}
        out["cpu"] = {"tok_s": c["value"], "tok_s_1core": one.get("decode_tokens_per_s"), "cores": c["cores"]}
    return out


def gpu_arm(args):
    import torch

    ws, rank, local = dist_setup()
    torch.cuda.set_device(local)
    from weight_streaming_gemv_token_gb300 import build

    build.build()
    import weight_streaming_gemv_token_gb300 as W
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    s = Wl.QWEN3_06B
    weights = Wl.decoder_weights(s, seed=1)
    prompt = Wl.prompt_uniform(PROMPT, s.vocab, seed=0)
    K, Wm = args.steps, args.warmup
    max_seq = PROMPT + 1 + Wm + K + 1 + 2 * args.e2e_steps + 8
    stream = torch.cuda.current_stream()
    dec = Decoder(s, weights, kv_dtype="f32", max_seq=max_seq, stream=stream, engine=args.engine)
    dec.reset()
    first = dec.prefill(prompt, is_last=True)
    out_buf = torch.empty(max(Wm, 1) + K, dtype=torch.int32, device="cuda")
    # warm-up steps (untimed)
    dec.generate(first, Wm, out_buf[:Wm]) if Wm > 0 else None
    torch.cuda.synchronize()
    tok = int(out_buf[Wm - 1].item()) if Wm > 0 else first
    pos0 = dec.position
    hbm, peak_kind = measured_peaks()

    # ---- timed region: K decode steps on the device ----
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize()
    with Clocks(local) as clk:
        e0.record(stream)
        dec.generate(tok, K, out_buf[Wm:Wm + K])
        e1.record(stream)
        torch.cuda.synchronize()
    barrier(ws)
    sec = barrier_max(e0.elapsed_time(e1) / 1e3, ws)
    value = ws * K / sec
    assert dec.device_errors() == 0, "device error during the timed region"
    mid_pos = pos0 + K // 2
    step_bytes = bytes_per_step(s, mid_pos)

    # ---- e2e: host token in, host token out, every step ----
    tok = int(out_buf[Wm + K - 1].item())
    n_e2e = args.e2e_steps
    for _ in range(3):
        tok = dec.step(tok)
    barrier(ws)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(n_e2e):
        tok = dec.step(tok)          # H2D of the token, graph, D2H of the next token, sync
    f1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    e2e_sec = barrier_max(max(wall, f0.elapsed_time(f1) / 1e3), ws)
    e2e_value = ws * n_e2e / e2e_sec
    fixed = fixed_context_latency(dec, torch, s, stream)
    generation = generation_timings(dec, torch, s)
    dec.close()
    del dec
    torch.cuda.empty_cache()

    extra = {}
    if rank == 0:
        gen = torch.Generator(device="cuda")
        gen.manual_seed(1234)
        if args.engine == "persistent":
            # the dominant (only) kernel of the timed region: one persistent launch for all K steps
            achieved = step_bytes * K / sec / 1e9
            extra["roofline"] = {
                "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4),
                "traffic": (round(MK_TRAFFIC_PER_ALG_BYTE * step_bytes * K) if MK_TRAFFIC_PER_ALG_BYTE else None),
                "peak_kind": peak_kind, "kernel": "decode_megakernel<float,float,2> (one cooperative launch, K steps)",
                "bytes_per_launch": step_bytes * K, "launch_us": round(sec * 1e6, 1), "launches": 1,
                "traffic_source": ("ncu dram bytes of a 4-layer/32768-vocab case of the same widths, scaled by "
                                   "algorithmic bytes" if MK_TRAFFIC_PER_ALG_BYTE else
                                   "not measured for the current kernel (last capture, before a change of the "
                                   "attention's load order: 1.008 of algorithmic bytes)")}
        # the standalone GEMV alone at the tied-vocabulary shape (the step's largest product), cold
        o, i = GEMV_ROOF_SHAPE
        gbs, per_launch, avg, launches = time_gemv_cold(W, torch, "f32", o, i, stream, gen=gen)
        extra["roofline" if args.engine != "persistent" else "gemv_roofline"] = {
            "bound": "hbm", "achieved": round(gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 4),
            # ncu dram__bytes_read+write per launch of this kernel on this shape; None until measured
            # for the current kernel
            "traffic": GEMV_TRAFFIC, "peak_kind": peak_kind,
            "kernel": f"gemv_bulk_kernel<float,1> {o}x{i} (tied vocabulary shape), standalone gemv entry, "
                      "cold round-robin",
            "bytes_per_launch": per_launch, "avg_launch_us": round(avg * 1e6, 3), "launches": launches}
        if not args.no_sweep:
            sweep = {}
            for dt in ("f32", "bf16"):
                for (o, i) in Wl.GEMV_SHAPES:
                    g, _, a, _ = time_gemv_cold(W, torch, dt, o, i, stream, gen=gen)
                    sweep[f"{dt} {o}x{i}"] = {"GB/s": round(g, 1), "frac": round(g / hbm, 4), "us": round(a * 1e6, 3)}
            # rows per warp tuned per shape on the cold number ("Our Kernel Benchmark Was Measuring
            # the System Cache"); "auto" is the library's default choice
            for ntok in (1, 2):
                for (o, i) in Wl.GEMV_SHAPES:
                    res = time_q4_cold_rows(W, torch, o, i, stream, ntok, (-1, 1, 2, 4, 8), gen=gen)
                    best = max((r for r in res if r > 0), key=lambda r: res[r][0])
                    g, _, a = res[best]
                    sweep[f"q4 ntok={ntok} {o}x{i}"] = {
                        "GB/s": round(g, 1), "frac": round(g / hbm, 4), "us": round(a * 1e6, 3), "rows_per_warp": best,
                        "auto_GB/s": round(res[-1][0], 1),
                        "by_rows_GB/s": {str(r): round(res[r][0], 1) for r in res if r > 0}}
            extra["gemv_cold"] = sweep
        if not args.no_prefill:
            extra["prefill"] = prefill_config(W, torch, hbm, measured_bf16_tflops())
        if not args.no_lossless:
            extra["lossless_storage"] = lossless_config(W, torch, stream, weights["embed"], hbm)
        if not args.no_q4:
            extra["q4_decoder"] = q4_config(W, torch, stream, hbm)

    if rank == 0:
        cpu = None if args.no_cpu else cpu_baseline_sample(weights, prompt, budget_s=args.cpu_seconds)
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": ws, "steps": K, "warmup": Wm,
            "ms_per_step": round(sec / K * 1e3, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded N(0,0.02) weights, uniform prompt)",
            "config": {
                "workload": "Qwen3-0.6B-shaped decoder, FP32 weights/activations/KV, batch-1 greedy decode "
                            f"after a {PROMPT}-token prompt (positions {pos0}..{pos0 + K - 1})",
                "layers": s.layers, "hidden": s.hidden, "inter": s.inter, "heads": f"{s.n_q}q/{s.n_kv}kv",
                "head_dim": s.head_dim, "vocab": s.vocab, "global_batch": 1, "seq_len": pos0 + K,
                "parallelism": "replicas" if ws > 1 else "single GPU", "engine": args.engine,
                "l2": "inputs larger than L2 (2.38 GB of weights streamed per step)",
            },
            "step_roofline": {"bytes_per_step": step_bytes, "achieved_GB/s": round(step_bytes * K / sec / 1e9, 1),
                              "peak": hbm, "frac": round(step_bytes * K / sec / 1e9 / hbm, 4),
                              "roofline_tokens_per_s": round(hbm * 1e9 / step_bytes, 1)},
            "e2e": {"value": round(e2e_value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 4,
                    "d2h_bytes_per_step": 4, "steps": n_e2e},
            "fixed_context": fixed,
            "generation": generation,
            "gpu_launches": 1 if args.engine == "persistent" else K * (5 * s.layers + 1),
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
        }
        line.update(extra)
        line["summary"] = summary(line)  # last, so that a tail of the line keeps it
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


# ---------------------------------------------------------------- CPU side ----

def oracle_decode_rate(weights, prompt, budget_s, min_tokens=3, max_tokens=200):
    """The oracle's greedy decode rate (tokens/s) after the prompt, for about budget_s seconds."""
    import oracle as O

    s = Wl.QWEN3_06B
    m = O.OracleDecoder(s, weights, kv_dtype="f32", max_seq=len(prompt) + max_tokens + 8)
    for t in prompt[:-1]:
        m.body(int(t))
    cur = int(prompt[-1])
    n = 0
    t0 = time.perf_counter()
    while n < min_tokens or (time.perf_counter() - t0 < budget_s and n < max_tokens):
        cur, _ = O.argmax_lowest(m.step(cur))
        n += 1
    return n, n / (time.perf_counter() - t0)


def oracle_gemv_rates(shapes, dtypes):
    """The oracle's GEMV (float64 product of the widened or dequantised matrix) in GB/s of the
    same algorithmic bytes the GPU sweep counts: one call per shape, as the oracle stands."""
    import oracle as O

    res = {}
    for dt in dtypes:
        for (o, i) in shapes:
            if dt.startswith("q4"):
                ntok = 2 if dt == "q4 ntok=2" else 1
                m = Wl.q4_matrix(o, i, seed=o + i)
                x = Wl.q4_activations(i, ntok, seed=7)
                if ntok == 1:
                    x = x[0]
                fn = lambda: O.gemv_q4(m["packed"], m["scale"], m["bias"], x)  # noqa: E731
                nbytes = o * i // 2 + o * (i // 64) * 4 + ntok * (2 * i + 4 * o)
            else:
                Wm = Wl.gemv_matrix(o, i, seed=o + i, dtype=dt)
                x = Wl.gemv_vector(i, seed=7, dtype=dt)
                fn = lambda: O.gemv(Wm, x)  # noqa: E731
                e = 4 if dt == "f32" else 2
                nbytes = o * i * e + i * e + 4 * o
            t0 = time.perf_counter()
            fn()
            res[f"{dt} {o}x{i}"] = round(nbytes / (time.perf_counter() - t0) / 1e9, 3)
    return res


def cpu_one_core_worker():
    """Run in a child process whose BLAS is limited to one thread: oracle decode rate and f32 GEMV GB/s."""
    s = Wl.QWEN3_06B
    weights = Wl.decoder_weights(s, seed=1)
    prompt = Wl.prompt_uniform(PROMPT, s.vocab, seed=0)
    n, rate = oracle_decode_rate(weights, prompt, budget_s=6.0, min_tokens=2)
    del weights
    gemv = oracle_gemv_rates(Wl.GEMV_SHAPES, ("f32",))
    print(json.dumps({"decode_tokens_per_s": round(rate, 4), "decode_tokens": n, "gemv_GB/s": gemv}), flush=True)


def cpu_baseline_sample(weights, prompt, budget_s=10.0):
    """The oracle on the host cores: decode rate on all cores (the line's value), the same on one
    core (a child process with one BLAS thread), and its GEMV GB/s on the five layer shapes in
    float32, bfloat16 and 4-bit (one and two tokens) on all cores, float32 on one core."""
    n, rate = oracle_decode_rate(weights, prompt, budget_s)
    gemv = oracle_gemv_rates(Wl.GEMV_SHAPES, ("f32", "bf16", "q4 ntok=1", "q4 ntok=2"))
    one = None
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-worker"], env=env, capture_output=True,
                           text=True, timeout=300)
        if r.returncode == 0 and r.stdout.strip():
            one = json.loads(r.stdout.strip().splitlines()[-1])
        else:
            one = {"error": (r.stderr or "no output").strip().splitlines()[-1][:200]}
    except (subprocess.TimeoutExpired, OSError, ValueError) as e:
        one = {"error": str(e)[:200]}
    return {"value": round(rate, 4), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} greedy decode forwards of the FP32 Qwen3-0.6B-shaped decoder after the {len(prompt)}-token "
                      f"prompt (float64 numpy oracle, BLAS threads = host cores)",
            "one_core": one, "gemv_GB/s": gemv}


def reference_arm(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle as O

    s = Wl.QWEN3_06B
    weights = Wl.decoder_weights(s, seed=1)
    prompt = Wl.prompt_uniform(PROMPT, s.vocab, seed=0)
    m = O.OracleDecoder(s, weights, kv_dtype="f32", max_seq=PROMPT + args.warmup + args.steps + 4)
    for t in prompt[:-1]:
        m.body(int(t))
    cur = int(prompt[-1])
    for _ in range(args.warmup):
        cur, _ = O.argmax_lowest(m.step(cur))
    t0 = time.perf_counter()
    for _ in range(args.steps):
        cur, _ = O.argmax_lowest(m.step(cur))
    sec = time.perf_counter() - t0
    value = args.steps / sec
    sample = f"{args.steps} greedy decode forwards (after {args.warmup} warm-up) of the FP32 Qwen3-0.6B-shaped decoder"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "Qwen3-0.6B-shaped decoder, FP32 weights, batch-1 greedy decode after a "
                               f"{PROMPT}-token prompt, run by the float64 CPU oracle"},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-sweep", action="store_true", help="skip the cold GEMV sweep")
    ap.add_argument("--engine", default="persistent", choices=["persistent", "staged"])
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--no-prefill", action="store_true", help="skip the BF16 chunked-prefill configuration")
    ap.add_argument("--no-lossless", action="store_true", help="skip the lossless bfloat16 storage comparison")
    ap.add_argument("--no-q4", action="store_true", help="skip the 4-bit decoder configuration")
    ap.add_argument("--cpu-worker", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_worker:
        cpu_one_core_worker()
        return
    if args.impl == "reference":
        args.steps = args.steps if args.steps is not None else 5
        args.warmup = args.warmup if args.warmup is not None else 1
        # each reference step is one oracle forward (~0.1-1 s); keep the run to a few minutes
        args.steps = min(args.steps, 60)
        args.warmup = min(args.warmup, 5)
        reference_arm(args)
        return
    args.steps = args.steps if args.steps is not None else 500
    args.warmup = max(3, args.warmup if args.warmup is not None else 20)
    gpu_arm(args)


if __name__ == "__main__":
    main()
