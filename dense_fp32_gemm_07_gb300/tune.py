"""Per-plan timing sweep behind the shape-keyed tune table (csrc/tune_table.h).

    python -m dense_fp32_gemm_07_gb300.tune [--once] [--cold] [--plans REGEX] MxNxK[xALPHAxBETA] ...
    python -m dense_fp32_gemm_07_gb300.tune --tf32x3 [--once] MxNxK[xALPHAxBETA] ...

Times every compiled plan that accepts the operands on each shape (CUDA events
on the launching stream, after warm-up, operands uniform[-1, 1) made by
torch), prints TFLOP/s per plan and marks the one the table picks.  Plans
that read A stored K x M (tmaT_*) get a transposed copy of A.  With --once
every plan runs exactly one launch per shape and nothing is timed: that is the
form to run under ncu to compare plans' counters.  --plans keeps only the
plans whose name matches REGEX (re.search); the table's plan is always kept.
--cold rotates the calls through as many copies of the operands as it takes
to pass twice the 129 MB L2 between two uses of a copy (at most 8), as the
bench's skinny measurement does, and adds the algorithmic bytes' rate
(4(MK + KN + MN(1 + [beta != 0])) per call) to each line.
--tf32x3 times the 3xTF32 tensor-core path instead, each kernel variant
(0: one CTA per 128 x 128 tile, 1 and 2: a CTA pair per 256 x 128 or 256 x 256
tile), split kernels included; --variants picks which.
"""
from __future__ import annotations

import argparse
import re
import sys

import dense_fp32_gemm_07_gb300 as b2g


def parse_shape(s: str):
    f = s.split("x")
    M, N, K = int(f[0]), int(f[1]), int(f[2])
    alpha = float(f[3]) if len(f) > 3 else 1.0
    beta = float(f[4]) if len(f) > 4 else 0.0
    return M, N, K, alpha, beta


L2_BYTES = 129e6


def sweep(shapes, once=False, out=sys.stdout, pattern=None, cold=False):
    import torch

    from dense_fp32_gemm_07_gb300 import build

    build.build()
    names = b2g.plans()
    for M, N, K, alpha, beta in shapes:
        nbytes = 4.0 * (M * K + K * N + M * N * (2 if beta != 0 else 1))
        copies = 1
        if cold:
            copies = max(1, min(8, -(-int(2 * L2_BYTES) // int(nbytes))))
        sets = []
        for _ in range(copies):
            A = torch.rand(M, K, device="cuda") * 2 - 1
            B = torch.rand(K, N, device="cuda") * 2 - 1
            C = torch.rand(M, N, device="cuda") * 2 - 1
            sets.append((A, B, C, A.t().contiguous()))
        A, B, C, At = sets[0]
        flops = 2.0 * M * N * K
        iters = max(3, min(50, int(2e11 / flops)))
        if cold:
            iters = max(iters, 50 * copies)
        sel = b2g.b2g_sgemm_select_plan(0, 0, M, N, K, alpha, A.data_ptr(), K, B.data_ptr(), N,
                                        C.data_ptr(), N)
        for pi, name in enumerate(names):
            if pattern and pi != sel and not re.search(pattern, name):
                continue
            trans = name.startswith("tmaT")
            turn = [0]

            def call():
                a_, b_, c_, at_ = sets[turn[0] % copies]
                turn[0] += 1
                b2g.sgemm(at_ if trans else a_, b_, c_, alpha, beta, transA=trans, plan=pi)

            try:
                call()
            except b2g.B2GError:
                continue  # the plan cannot take these operands
            torch.cuda.synchronize()
            if once:
                print(f"{M}x{N}x{K} {name}", file=out, flush=True)
                continue
            for _ in range(2 * copies):
                call()
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)
            ev0.record()
            for _ in range(iters):
                call()
            ev1.record()
            torch.cuda.synchronize()
            ms = ev0.elapsed_time(ev1) / iters
            mark = "  <- table" if pi == sel else ""
            rate = f" {nbytes / ms / 1e9:7.2f} TB/s ({copies} copies)" if cold else ""
            print(f"{M}x{N}x{K} {name:26s} {ms:9.4f} ms {flops / ms / 1e9:8.2f} TFLOP/s{rate}{mark}",
                  file=out, flush=True)


def sweep_tf32x3(shapes, once=False, out=sys.stdout, variants=(0, 1, 2)):
    import torch

    from dense_fp32_gemm_07_gb300 import build

    build.build()
    for M, N, K, alpha, beta in shapes:
        A = torch.rand(M, K, device="cuda") * 2 - 1
        B = torch.rand(K, N, device="cuda") * 2 - 1
        C = torch.rand(M, N, device="cuda") * 2 - 1
        flops = 2.0 * M * N * K
        iters = max(3, min(50, int(2e12 / flops)))
        for variant in variants:
            def call():
                b2g.sgemm_3xtf32(A, B, C, alpha, beta, variant=variant)

            call()
            torch.cuda.synchronize()
            if once:
                print(f"{M}x{N}x{K} tf32x3 variant {variant}", file=out, flush=True)
                continue
            for _ in range(2):
                call()
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)
            ev0.record()
            for _ in range(iters):
                call()
            ev1.record()
            torch.cuda.synchronize()
            ms = ev0.elapsed_time(ev1) / iters
            print(f"{M}x{N}x{K} tf32x3 variant {variant}  {ms:9.4f} ms {flops / ms / 1e9:8.2f} "
                  f"TFLOP/s ({3 * flops / ms / 1e9:7.1f} TF32 TFLOP/s)", file=out, flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("shapes", nargs="*", default=["4096x4096x4096x1x0.5"])
    ap.add_argument("--once", action="store_true")
    ap.add_argument("--plans", default=None, help="regex: time only the matching plans")
    ap.add_argument("--tf32x3", action="store_true", help="time the 3xTF32 kernel variants")
    ap.add_argument("--variants", default="0,1,2",
                    help="3xTF32 kernel variants to run, comma-separated (with --tf32x3)")
    ap.add_argument("--cold", action="store_true",
                    help="rotate operand copies so that every call reads them from HBM")
    args = ap.parse_args()
    shapes = [parse_shape(s) for s in args.shapes]
    if args.tf32x3:
        sweep_tf32x3(shapes, once=args.once,
                     variants=tuple(int(v) for v in args.variants.split(",")))
    else:
        sweep(shapes, once=args.once, pattern=args.plans, cold=args.cold)


if __name__ == "__main__":
    main()
