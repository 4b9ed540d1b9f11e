"""Run one operation of the library on one synthetic shape, a few times.

Meant for profilers (e.g. ``ncu -k regex:gemm_reduce_kernel -c 1``): it does
nothing but allocate random inputs on the device, create a workspace and call
the operation ``--iters`` times.  It makes no timing claims.

    python -m all_reduce_epilogue_gb300.profile_case gemm_rs --R 4 --M 8192 --N 4096 --K 2048
    python -m all_reduce_epilogue_gb300.profile_case allreduce_rmsnorm --R 8 --M 4096 --N 7168
"""
from __future__ import annotations

import argparse
import sys


def main(argv=None) -> int:
    import torch

    import all_reduce_epilogue_gb300 as are

    ap = argparse.ArgumentParser()
    ap.add_argument("op", choices=["gemm_rs", "gemm_ar", "allreduce_rmsnorm"])
    ap.add_argument("--R", type=int, default=8)
    ap.add_argument("--M", type=int, default=4096)
    ap.add_argument("--N", type=int, default=7168)
    ap.add_argument("--K", type=int, default=2048)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--views", type=int, default=0, help="gemm_ar: distinct output views (default R)")
    ap.add_argument("--path", choices=["default", "oneshot", "lamport"], default="default",
                    help="allreduce_rmsnorm: force a kernel")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--order", default="", help="gemm: group_m,block_pairs,rank_group (0 = default)")
    ap.add_argument("--chunks", type=int, default=0, help="gemm_rs: chunks per owner segment (rotated order)")
    a = ap.parse_args(argv)
    torch.manual_seed(a.seed)
    dev = torch.device("cuda", 0)

    def bf(*shape, scale=1.0):
        return (torch.randn(*shape, device=dev) * scale).to(torch.bfloat16)

    if a.op == "allreduce_rmsnorm":
        parts = [bf(a.M, a.N) for _ in range(a.R)]
        res = bf(a.M, a.N)
        gamma = 1 + 0.1 * torch.randn(a.N, device=dev)
        out = torch.empty_like(res)
        with are.Workspace(R_max=a.R, M_max=a.M, N_max=a.N) as ws:
            ws.set_debug({"default": 0, "oneshot": are.DEBUG_AR_ONESHOT, "lamport": are.DEBUG_AR_LAMPORT}[a.path])
            for _ in range(a.iters):
                are.allreduce_rmsnorm(parts, res, gamma, 1e-6, out, ws)
            st = ws.device_status()
    else:
        s = a.K ** -0.5
        A = [bf(a.M, a.K, scale=s) for _ in range(a.R)]
        B = [bf(a.K, a.N, scale=s) for _ in range(a.R)]
        with are.Workspace(R_max=a.R, M_max=a.M, N_max=a.N, K_max=a.K) as ws:
            if a.order:
                ws.set_gemm_order(*[int(v) for v in a.order.split(",")])
            if a.chunks:
                ws.set_chunks(a.chunks, 0)
            if a.op == "gemm_rs":
                out = torch.empty(a.M, a.N, dtype=torch.bfloat16, device=dev)
                for _ in range(a.iters):
                    are.gemm_rs(A, B, out, ws)
            else:
                nv = a.views if a.views > 0 else a.R
                distinct = [torch.empty(a.M, a.N, dtype=torch.bfloat16, device=dev) for _ in range(nv)]
                views = [distinct[r % nv] for r in range(a.R)]
                for _ in range(a.iters):
                    are.gemm_ar(A, B, views, ws)
            st = ws.device_status()
    torch.cuda.synchronize()
    if st["code"] != 0:
        print(f"device status: {st}", file=sys.stderr)
        return 1
    print(f"{a.op} R={a.R} M={a.M} N={a.N} K={a.K} x{a.iters}: ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())
