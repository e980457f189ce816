"""Timing of single kernels of the inner loop through the kernel-level C entry
points (include/ttt_kernels.h), for profiling one kernel in isolation.

    python -m long_context_lm_ttt_b300.microbench gemm --M 1024 --N 16384 --K 3072
    python -m long_context_lm_ttt_b300.microbench gemm --M 1024 --N 16384 --K 3072 --dual 1   # + A B2^T
    python -m long_context_lm_ttt_b300.microbench gemm-sgd --M 3072 --N 8192 --K 1024
    python -m long_context_lm_ttt_b300.microbench attn-fwd --n 1024 --H 24 --Hkv 8 --hd 128 --W 8192
    python -m long_context_lm_ttt_b300.microbench attn-bwd --n 1024 --H 24 --Hkv 8 --hd 128 --W 8192
    python -m long_context_lm_ttt_b300.microbench attn-fwd --n 1 --impl 4 --pos0 9000   # a decode step
    python -m long_context_lm_ttt_b300.microbench gemm --M 1 --N 16384 --K 3072          # a one-row product

Inputs are seeded random bf16 tensors on cuda:0.  Prints one JSON line with
the mean time of `--iters` launches (CUDA events, after `--warmup`) and the
algorithmic TFLOP/s (2 per multiply-add; attention counts unmasked pairs).
"""
from __future__ import annotations

import argparse
import json

import torch

from . import ttt as T


def _events(fn, warmup, iters):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(iters):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / iters


def gemm(args):
    g = torch.Generator(device="cuda").manual_seed(0)
    M, N, K = args.M, args.N, args.K
    A = (torch.randn((K, M) if args.a_mn else (M, K), device="cuda", generator=g)).to(torch.bfloat16)
    B = (torch.randn((K, N) if args.b_mn else (N, K), device="cuda", generator=g)).to(torch.bfloat16)
    # --dual: a second B of the same layout added into the same output (the
    # forward's fast-weight products read the weights as a bf16 hi/lo pair)
    B2 = (torch.randn(B.shape, device="cuda", generator=g)).to(torch.bfloat16) if args.dual else None
    C = torch.empty((M, N), device="cuda", dtype=torch.float32)
    lda = M if args.a_mn else K
    ldb = N if args.b_mn else K

    def run():
        T.ttt_kernel_gemm(M, N, K, A, lda, args.a_mn, B, ldb, args.b_mn, B2, C, N, args.impl)

    ms = _events(run, args.warmup, args.iters)
    assert T.ttt_kernel_error() == 0
    mult = 2.0 if args.dual else 1.0
    return {"kernel": "gemm", "M": M, "N": N, "K": K, "a_mn": args.a_mn, "b_mn": args.b_mn, "dual": args.dual,
            "ms": ms, "tflops": mult * 2.0 * M * N * K / (ms / 1e3) / 1e12}


def gemm_sgd(args):
    g = torch.Generator(device="cuda").manual_seed(0)
    M, N, K = args.M, args.N, args.K
    A = torch.randn((K, M), device="cuda", generator=g).to(torch.bfloat16)
    B = torch.randn((K, N), device="cuda", generator=g).to(torch.bfloat16)
    w32 = torch.randn((M, N), device="cuda", generator=g) * 0.02
    hi = torch.empty((M, N), device="cuda", dtype=torch.bfloat16)
    lo = torch.empty((M, N), device="cuda", dtype=torch.bfloat16)

    def run():
        T.ttt_kernel_gemm_sgd(M, N, K, A, M, 1, B, N, 1, w32, hi, lo, N, 1e-6, args.impl)

    ms = _events(run, args.warmup, args.iters)
    assert T.ttt_kernel_error() == 0
    nbytes = 12.0 * M * N + 2.0 * K * (M + N)
    return {"kernel": "gemm_sgd", "M": M, "N": N, "K": K, "ms": ms,
            "tflops": 2.0 * M * N * K / (ms / 1e3) / 1e12, "gbs": nbytes / (ms / 1e3) / 1e9}


def _attn_inputs(args):
    n, H, Hkv, hd, W = args.n, args.H, args.Hkv, args.hd, args.W
    R = ((W + n - 1 + 127) // 128) * 128
    g = torch.Generator(device="cuda").manual_seed(1)
    q = torch.randn((n, H * hd), device="cuda", generator=g).to(torch.bfloat16)
    kr = torch.randn((Hkv, R, hd), device="cuda", generator=g).to(torch.bfloat16)
    vr = torch.randn((Hkv, R, hd), device="cuda", generator=g).to(torch.bfloat16)
    o = torch.empty((n, H * hd), device="cuda", dtype=torch.bfloat16)
    lse = torch.empty((H, n), device="cuda", dtype=torch.float32)
    pairs = sum(min(args.pos0 + r + 1, W) for r in range(n))
    local = sum(min(r + 1, W) for r in range(n))
    return n, H, Hkv, hd, W, R, q, kr, vr, o, lse, pairs, local


def attn_fwd(args):
    n, H, Hkv, hd, W, R, q, kr, vr, o, lse, pairs, _ = _attn_inputs(args)
    lib = T.load()

    def run():
        rc = lib.ttt_kernel_attn_fwd(args.impl, n, H, Hkv, hd, W, R, args.pos0, q.data_ptr(), kr.data_ptr(),
                                     vr.data_ptr(), o.data_ptr(), lse.data_ptr(), n, None)
        assert rc == 0, rc

    ms = _events(run, args.warmup, args.iters)
    assert T.ttt_kernel_error() == 0
    return {"kernel": "attn_fwd", "n": n, "H": H, "Hkv": Hkv, "hd": hd, "W": W, "pos0": args.pos0, "ms": ms,
            "tflops": 4.0 * H * hd * pairs / (ms / 1e3) / 1e12}


def attn_bwd(args):
    n, H, Hkv, hd, W, R, q, kr, vr, o, lse, pairs, local = _attn_inputs(args)
    lib = T.load()
    assert lib.ttt_kernel_attn_fwd(0, n, H, Hkv, hd, W, R, args.pos0, q.data_ptr(), kr.data_ptr(), vr.data_ptr(),
                                   o.data_ptr(), lse.data_ptr(), n, None) == 0
    g = torch.Generator(device="cuda").manual_seed(2)
    dout = torch.randn((n, H * hd), device="cuda", generator=g).to(torch.bfloat16)
    dsum = torch.empty((H, n), device="cuda", dtype=torch.float32)
    dqkv = torch.empty((n, (H + 2 * Hkv) * hd), device="cuda", dtype=torch.bfloat16)

    def run():
        rc = lib.ttt_kernel_attn_bwd(args.impl, n, H, Hkv, hd, W, R, args.pos0, q.data_ptr(), kr.data_ptr(),
                                     vr.data_ptr(), o.data_ptr(), lse.data_ptr(), n, dout.data_ptr(),
                                     dsum.data_ptr(), dqkv.data_ptr(), None)
        assert rc == 0, rc

    ms = _events(run, args.warmup, args.iters)
    assert T.ttt_kernel_error() == 0
    return {"kernel": "attn_bwd", "n": n, "H": H, "Hkv": Hkv, "hd": hd, "W": W, "pos0": args.pos0, "ms": ms,
            "tflops": (6.0 * H * hd * pairs + 4.0 * H * hd * local) / (ms / 1e3) / 1e12}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    sub = ap.add_subparsers(dest="what", required=True)
    g = sub.add_parser("gemm")
    g.add_argument("--M", type=int, default=1024)
    g.add_argument("--N", type=int, default=16384)
    g.add_argument("--K", type=int, default=3072)
    g.add_argument("--a-mn", type=int, default=0)
    g.add_argument("--b-mn", type=int, default=0)
    g.add_argument("--dual", type=int, default=0, help="1: add A B2^T, B2 a second B (counted in TFLOP/s)")
    gs = sub.add_parser("gemm-sgd")
    gs.add_argument("--M", type=int, default=3072)
    gs.add_argument("--N", type=int, default=8192)
    gs.add_argument("--K", type=int, default=1024)
    for name in ("attn-fwd", "attn-bwd"):
        a = sub.add_parser(name)
        a.add_argument("--n", type=int, default=1024)
        a.add_argument("--H", type=int, default=24)
        a.add_argument("--Hkv", type=int, default=8)
        a.add_argument("--hd", type=int, default=128)
        a.add_argument("--W", type=int, default=8192)
        a.add_argument("--pos0", type=int, default=40960)
    for p in sub.choices.values():
        p.add_argument("--impl", type=int, default=0,
                       help="as the C entry point's impl: 0 tensor cores, 1 SIMT; gemm 3/4 and gemm-sgd 2/3 "
                            "force single-CTA / CTA-pair tiles")
        p.add_argument("--warmup", type=int, default=3)
        p.add_argument("--iters", type=int, default=10)
    args = ap.parse_args()
    torch.cuda.set_device(0)
    T.load()
    out = {"gemm": gemm, "gemm-sgd": gemm_sgd, "attn-fwd": attn_fwd, "attn-bwd": attn_bwd}[args.what](args)
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
