"""Kernel micro-benchmark: one layer-template kernel at a given shape, timed with CUDA events.

  python -m host_memory_streamed_stream_gb300.microbench gemm --M 8192 --N 4096 --K 4096 --layout fwd [--split]
  python -m host_memory_streamed_stream_gb300.microbench attn --B 2 --s 4096 --nh 32 --nkv 32 --hd 128
  python -m host_memory_streamed_stream_gb300.microbench rmsnorm --T 8192 --h 4096

GEMM layouts: fwd (y = x W^T), dgrad (dx = dy W), wgrad (dW = dy^T x), and the fused
epilogues qkv_rope, swiglu (N = f) and swiglu_bwd (N = f). Prints one JSON line
with the mean launch time and TFLOP/s (causal-half FLOPs for attention). Inputs are random
bf16 on the current device; nothing here is used by the training step itself.
"""
from __future__ import annotations

import argparse
import json

import torch

from . import kernels as K


def _time(fn, iters: int, warmup: int) -> float:
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(iters):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def bench_gemm(M: int, N: int, K_: int, layout: str, iters: int, warmup: int) -> dict:
    g = torch.Generator(device="cuda").manual_seed(0)
    bf = torch.bfloat16
    if layout == "fwd":  # A [M][K], B [N][K]
        A = torch.randn(M, K_, device="cuda", generator=g).to(bf)
        B = torch.randn(N, K_, device="cuda", generator=g).to(bf)
        a_mn, b_mn = 0, 0
    elif layout == "dgrad":  # A [M][K], B [K][N]
        A = torch.randn(M, K_, device="cuda", generator=g).to(bf)
        B = torch.randn(K_, N, device="cuda", generator=g).to(bf)
        a_mn, b_mn = 0, 1
    else:  # wgrad: A [K][M], B [K][N]
        A = torch.randn(K_, M, device="cuda", generator=g).to(bf)
        B = torch.randn(K_, N, device="cuda", generator=g).to(bf)
        a_mn, b_mn = 1, 1
    out = torch.empty(M, N, dtype=bf, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ms = _time(lambda: K.gemm(A, a_mn, B, b_mn, M, N, K_, out=out, err=err), iters, warmup)
    return {"kernel": "gemm", "layout": layout, "M": M, "N": N, "K": K_, "ms": ms,
            "tflops": 2.0 * M * N * K_ / (ms / 1e3) / 1e12, "err_flag": int(err.item())}


def bench_fused(kind: str, M: int, N: int, K_: int, iters: int, warmup: int) -> dict:
    """Fused-epilogue GEMMs of the layer template. N is the output width: (nh+2nkv)*128 for
    qkv_rope (heads of 128, q = k = v head counts), f for swiglu (gate and up: 2f columns of
    work) and swiglu_bwd (dact = dy Wd)."""
    g = torch.Generator(device="cuda").manual_seed(0)
    bf = torch.bfloat16
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if kind == "qkv_rope":
        hd, heads = 128, N // 128
        a = torch.randn(M, K_, device="cuda", generator=g).to(bf)
        w = torch.randn(N, K_, device="cuda", generator=g).to(bf)
        cs = torch.randn(M, hd // 2, 2, device="cuda", generator=g)
        fn = lambda: K.gemm_qkv_rope(a, w, cs, M, heads // 3, heads // 3, hd, err=err)  # noqa: E731
        work = N
    elif kind == "swiglu":
        b = torch.randn(M, K_, device="cuda", generator=g).to(bf)
        w = torch.randn(2 * N, K_, device="cuda", generator=g).to(bf)
        fn = lambda: K.gemm_swiglu(b, w, N, keep_gu=True, err=err)  # noqa: E731
        work = 2 * N
    else:
        dy = torch.randn(M, K_, device="cuda", generator=g).to(bf)
        wd = torch.randn(K_, N, device="cuda", generator=g).to(bf)
        gu = torch.randn(M, 2 * N, device="cuda", generator=g).to(bf)
        fn = lambda: K.gemm_swiglu_bwd(dy, wd, gu, N, err=err)  # noqa: E731
        work = N
    ms = _time(fn, iters, warmup)
    return {"kernel": "gemm_" + kind, "M": M, "N": N, "K": K_, "ms": ms,
            "tflops": 2.0 * M * work * K_ / (ms / 1e3) / 1e12, "err_flag": int(err.item())}


def bench_attn(B: int, s: int, nh: int, nkv: int, hd: int, iters: int, warmup: int, rope: bool = False) -> dict:
    g = torch.Generator(device="cuda").manual_seed(0)
    qkv = torch.randn(B * s, (nh + 2 * nkv) * hd, device="cuda", generator=g).to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = K.attn_fwd(qkv, B, s, nh, nkv, hd, err=err)
    dout = torch.randn_like(o)
    cs = torch.rand(s, hd // 2, 2, device="cuda", generator=g) if rope else None
    fwd = _time(lambda: K.attn_fwd(qkv, B, s, nh, nkv, hd, err=err), iters, warmup)
    bwd = _time(lambda: K.attn_bwd(qkv, o, lse, dout, B, s, nh, nkv, hd, err=err, cos_sin=cs), iters, warmup)
    f = 2.0 * B * s * s * nh * hd  # causal half of QK^T and PV
    return {"kernel": "attention", "B": B, "s": s, "nh": nh, "nkv": nkv, "hd": hd, "rope_bwd": rope,
            "fwd_ms": fwd, "bwd_ms": bwd,
            "fwd_tflops": f / (fwd / 1e3) / 1e12, "bwd_tflops": 2.5 * f / (bwd / 1e3) / 1e12,
            "err_flag": int(err.item())}


def bench_rmsnorm(T: int, h: int, iters: int, warmup: int) -> dict:
    """RMSNorm forward (fp32 in, bf16 out) and backward (+ residual gradient, fp32 and bf16 out,
    two-stage gain gradient): achieved GB/s from the bytes each must move."""
    g = torch.Generator(device="cuda").manual_seed(0)
    x = torch.randn(T, h, device="cuda", generator=g)
    gamma = torch.ones(h, device="cuda").to(torch.bfloat16)
    dy = torch.randn(T, h, device="cuda", generator=g)
    dres = torch.randn(T, h, device="cuda", generator=g)
    _, rstd = K.rmsnorm_fwd(x, gamma)
    fwd = _time(lambda: K.rmsnorm_fwd(x, gamma), iters, warmup)
    bwd = _time(lambda: K.rmsnorm_bwd(dy, x, gamma, rstd, dres), iters, warmup)
    fwd_bytes = T * h * (4 + 2)               # x in, y out
    bwd_bytes = T * h * (4 + 4 + 4 + 4 + 2)   # dy, x, dres in; dx fp32 and bf16 out
    return {"kernel": "rmsnorm", "T": T, "h": h, "fwd_ms": fwd, "bwd_ms": bwd,
            "fwd_gbs": fwd_bytes / (fwd / 1e3) / 1e9, "bwd_gbs": bwd_bytes / (bwd / 1e3) / 1e9}


def main():
    ap = argparse.ArgumentParser()
    sub = ap.add_subparsers(dest="kind", required=True)
    pg = sub.add_parser("gemm")
    pg.add_argument("--M", type=int, default=8192)
    pg.add_argument("--N", type=int, default=4096)
    pg.add_argument("--K", type=int, default=4096)
    pg.add_argument("--layout", choices=["fwd", "dgrad", "wgrad", "qkv_rope", "swiglu", "swiglu_bwd"], default="fwd")
    pr = sub.add_parser("rmsnorm")
    pr.add_argument("--T", type=int, default=8192)
    pr.add_argument("--h", type=int, default=4096)
    pa = sub.add_parser("attn")
    pa.add_argument("--B", type=int, default=2)
    pa.add_argument("--s", type=int, default=4096)
    pa.add_argument("--nh", type=int, default=32)
    pa.add_argument("--nkv", type=int, default=32)
    pa.add_argument("--hd", type=int, default=128)
    pa.add_argument("--rope", action="store_true", help="backward with the RoPE backward fused into dq/dk")
    pg.add_argument("--split", action="store_true",
                    help="give the GEMM a workspace, so that its last partial wave is split over K")
    for p in (pg, pa, pr):
        p.add_argument("--iters", type=int, default=20)
        p.add_argument("--warmup", type=int, default=3)
    args = ap.parse_args()
    ws = K.gemm_use_workspace("cuda") if args.kind == "gemm" and args.split else None  # noqa: F841
    if args.kind == "gemm" and args.layout in ("qkv_rope", "swiglu", "swiglu_bwd"):
        r = bench_fused(args.layout, args.M, args.N, args.K, args.iters, args.warmup)
    elif args.kind == "gemm":
        r = bench_gemm(args.M, args.N, args.K, args.layout, args.iters, args.warmup)
    elif args.kind == "rmsnorm":
        r = bench_rmsnorm(args.T, args.h, args.iters, args.warmup)
    else:
        r = bench_attn(args.B, args.s, args.nh, args.nkv, args.hd, args.iters, args.warmup, args.rope)
    if args.kind == "gemm":
        r["split"] = bool(args.split)
    print(json.dumps(r), flush=True)


if __name__ == "__main__":
    main()
