"""Profiling driver: runs a region of interest between cudaProfilerStart/Stop.

Use under ncu with --profile-from-start off, e.g.

  ncu --profile-from-start off --metrics gpu__time_duration.sum --clock-control none --csv \\
      python profile_step.py decode --steps 1
  ncu --profile-from-start off --set full --clock-control none -k regex:gemv_stream -c 3 -o prof \\
      python profile_step.py gemv --out 6144 --in 1024 --count 8

decode: Qwen3-0.6B-shaped decoder (optionally fewer layers / a smaller
        vocabulary, for captures that must stay small; --dtype q4 with
        --engine staged for the 4-bit configuration) with seeded random
        weights, a uniform prompt, warm-up steps, then --steps decode steps
        inside the region.
gemv:   --count distinct matrices of one shape (sized past L2 by default),
        one warm-up pass, then one launch per matrix inside the region.
q4:     the same for gemv_q4 (4-bit codes, fp16 scales and biases, bf16 x).
prefill: BF16 Qwen3-0.6B-shaped decoder (optionally fewer layers) with chunked
        prefill: a --prompt-token Zipf(1.1) prompt in chunks of --chunk rows,
        one untimed pass, then the whole prompt again inside the region.
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def decode(args):
    import workloads as Wl

    from weight_streaming_gemv_token_gb300 import build
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    build.build()
    s = Wl.QWEN3_06B
    if args.layers or args.vocab:
        import dataclasses

        s = dataclasses.replace(s, layers=args.layers or s.layers, vocab=args.vocab or s.vocab)
    w = Wl.decoder_weights_q4(s, seed=1) if args.dtype == "q4" else Wl.decoder_weights(s, seed=1, wdtype=args.dtype)
    prompt = Wl.prompt_uniform(args.prompt, s.vocab, seed=0)
    dec = Decoder(s, w, kv_dtype=args.kv, max_seq=args.prompt + args.warmup + args.steps + 4, engine=args.engine,
                  chunk_cap=args.chunk)
    if args.chunk:
        for c0 in range(0, args.prompt - args.chunk, args.chunk):
            dec.prefill([int(t) for t in prompt[c0:c0 + args.chunk]], is_last=False)
        c0 = (args.prompt - 1) // args.chunk * args.chunk
        first = dec.prefill([int(t) for t in prompt[c0:]], is_last=True)
    else:
        first = dec.prefill(prompt, is_last=True)
    out = dec.generate(first, args.warmup)
    torch.cuda.synchronize()
    tok = int(out[-1].item())
    torch.cuda.profiler.start()
    dec.generate(tok, args.steps)
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    assert dec.device_errors() == 0


def gemv(args):
    from weight_streaming_gemv_token_gb300 import binding as B
    from weight_streaming_gemv_token_gb300 import build

    build.build()
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    tdt = torch.float32 if args.dtype == "f32" else torch.bfloat16
    per = args.out * args.inp * (4 if args.dtype == "f32" else 2)
    count = args.count or max(2, -(-(256 << 20) // per))
    mats = [(0.02 * torch.randn((args.out, args.inp), device="cuda", generator=g)).to(tdt) for _ in range(count)]
    x = (0.02 * torch.randn(args.inp, device="cuda", generator=g)).to(tdt)
    y = torch.empty(args.out, device="cuda")
    code = B.DEC_F32 if args.dtype == "f32" else B.DEC_BF16
    for m in mats:
        B.gemv(code, m, x, y, args.out, args.inp, None)
    torch.cuda.synchronize()
    torch.cuda.profiler.start()
    for m in mats:
        B.gemv(code, m, x, y, args.out, args.inp, None)
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()


def q4(args):
    from weight_streaming_gemv_token_gb300 import binding as B
    from weight_streaming_gemv_token_gb300 import build

    build.build()
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    out, inp, ntok = args.out, args.inp, args.ntok
    per = out * inp // 2 + out * (inp // 64) * 4
    count = args.count or max(2, -(-(256 << 20) // per))
    codes = [torch.randint(-2**31, 2**31 - 1, (out, inp // 8), dtype=torch.int32, device="cuda", generator=g)
             for _ in range(count)]
    sc = [torch.empty((out, inp // 64), dtype=torch.float16, device="cuda").uniform_(0.001, 0.01, generator=g)
          for _ in range(count)]
    bi = [torch.empty((out, inp // 64), dtype=torch.float16, device="cuda").normal_(0, 0.02, generator=g)
          for _ in range(count)]
    x = torch.randn((ntok, inp), device="cuda", generator=g).to(torch.bfloat16)
    y = torch.empty((ntok, out), device="cuda")
    if args.rows:
        B.gemv_q4_rows_per_warp(ntok, args.rows)
    for i in range(count):
        B.gemv_q4(codes[i], sc[i], bi[i], x, y, out, inp, ntok, None)
    torch.cuda.synchronize()
    torch.cuda.profiler.start()
    for i in range(count):
        B.gemv_q4(codes[i], sc[i], bi[i], x, y, out, inp, ntok, None)
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    assert B.gemv_device_errors() == 0


def prefill(args):
    import dataclasses

    import workloads as Wl

    from weight_streaming_gemv_token_gb300 import build
    from weight_streaming_gemv_token_gb300.decoder import Decoder

    build.build()
    s = Wl.QWEN3_06B
    if args.layers:
        s = dataclasses.replace(s, layers=args.layers)
    w = Wl.decoder_weights(s, seed=1, wdtype="bf16")
    prompt = Wl.prompt_zipf(args.prompt, s.vocab, seed=0)
    dec = Decoder(s, w, kv_dtype="bf16", max_seq=args.prompt + 8, chunk_cap=args.chunk)

    def run():
        dec.reset()
        for c0 in range(0, args.prompt, args.chunk):
            last = c0 + args.chunk >= args.prompt
            dec.prefill([int(t) for t in prompt[c0:c0 + args.chunk]], is_last=last)

    run()
    torch.cuda.synchronize()
    torch.cuda.profiler.start()
    run()
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    assert dec.device_errors() == 0


def main():
    ap = argparse.ArgumentParser()
    sub = ap.add_subparsers(dest="mode", required=True)
    d = sub.add_parser("decode")
    d.add_argument("--dtype", default="f32", choices=["f32", "bf16", "q4"], help="q4: the 4-bit configuration (staged)")
    d.add_argument("--kv", default="f32", choices=["f32", "bf16"])
    d.add_argument("--prompt", type=int, default=32)
    d.add_argument("--warmup", type=int, default=3)
    d.add_argument("--steps", type=int, default=1)
    d.add_argument("--layers", type=int, default=0, help="fewer layers than the Qwen3-0.6B shape (0: 28)")
    d.add_argument("--vocab", type=int, default=0, help="smaller vocabulary (0: 151936)")
    d.add_argument("--engine", default="persistent", choices=["persistent", "staged"])
    d.add_argument("--chunk", type=int, default=0, help="prefill the prompt in chunks of this many rows (bf16 only)")
    gm = sub.add_parser("gemv")
    gm.add_argument("--out", type=int, default=6144)
    gm.add_argument("--in", dest="inp", type=int, default=1024)
    gm.add_argument("--dtype", default="f32", choices=["f32", "bf16"])
    gm.add_argument("--count", type=int, default=0)
    qm = sub.add_parser("q4")
    qm.add_argument("--out", type=int, default=151936)
    qm.add_argument("--in", dest="inp", type=int, default=1024)
    qm.add_argument("--ntok", type=int, default=1, choices=[1, 2])
    qm.add_argument("--rows", type=int, default=0, help="rows per warp (0: the library default)")
    qm.add_argument("--count", type=int, default=0)
    pf = sub.add_parser("prefill")
    pf.add_argument("--prompt", type=int, default=4096)
    pf.add_argument("--chunk", type=int, default=1024)
    pf.add_argument("--layers", type=int, default=0, help="fewer layers than the Qwen3-0.6B shape (0: 28)")
    args = ap.parse_args()
    {"decode": decode, "gemv": gemv, "q4": q4, "prefill": prefill}[args.mode](args)


if __name__ == "__main__":
    main()
