"""Run one kernel of the block on a small seeded case (for ncu captures).

    python -m memory_bounded_video_gb300.profile_case gemm --mode swiglu \\
        --int8 --M 2048 --N 8192 --K 3072 --reps 3
    python -m memory_bounded_video_gb300.profile_case attention --Tq 2048 \\
        --T 8192 --heads 4 --head-dim 128 --reps 3 [--no-split]
    python -m memory_bounded_video_gb300.profile_case modln --M 8192 --D 3072
    python -m memory_bounded_video_gb300.profile_case final --M 8192 --D 3072 [--int8]
    python -m memory_bounded_video_gb300.profile_case expand --M 8192 --D 3072

``gemm --scaled`` runs the bf16 main loop on int8 values with per-row scales
(the weight-scratch path); ``expand`` the int8 -> bf16 expansion of an
[M, D] int8 matrix.

Every launch goes through the C ABI; the inputs are random device tensors of
the requested shapes (sized to exceed L2 where the case allows), the outputs
are discarded.  Prints the mean CUDA-event time per launch.
"""

from __future__ import annotations

import argparse
import sys

import torch

from . import build as dbuild
from . import ditstream as ds

MODES = {"store_bf16": ds.EPI_STORE_BF16, "store_f32": ds.EPI_STORE_F32,
         "kv": ds.EPI_KV, "resid": ds.EPI_RESID, "swiglu": ds.EPI_SWIGLU,
         "down": ds.EPI_DOWN}


def gemm_case(a):
    g = torch.Generator(device="cuda").manual_seed(0)
    M, N, K = a.M, a.N, a.K
    A = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    if a.int8:
        B0 = torch.randint(-127, 128, (N, K), device="cuda", generator=g,
                           dtype=torch.int8)
        B1 = torch.randint(-127, 128, (N, K), device="cuda", generator=g,
                           dtype=torch.int8)
        s0 = torch.full((N,), 0.02 / 127, device="cuda")
        s1 = s0.clone()
    elif a.scaled:
        B0 = torch.randint(-127, 128, (N, K), device="cuda", generator=g,
                           dtype=torch.int8).to(torch.bfloat16)
        B1 = torch.randint(-127, 128, (N, K), device="cuda", generator=g,
                           dtype=torch.int8).to(torch.bfloat16)
        s0 = torch.full((N,), 0.02 / 127, device="cuda")
        s1 = s0.clone()
    else:
        B0 = (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        B1 = (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        s0 = s1 = None
    mode = MODES[a.mode]
    out = torch.empty(M, N, device="cuda", dtype=torch.float32)
    Vt = torch.empty(N, M, device="cuda", dtype=torch.bfloat16)
    x = torch.zeros(M, N, device="cuda")
    gate = torch.rand(N, device="cuda", generator=g)
    args = ds.GemmArgs(mode=mode, M=M, N=N, K=K, a=ds.ptr(A), lda=K, b0=ds.ptr(B0),
                       b1=ds.ptr(B1), ldb=K,
                       b_dtype=ds.W_INT8 if a.int8 else ds.W_BF16,
                       b0_scale=ds.ptr(s0), b1_scale=ds.ptr(s1), out=ds.ptr(out),
                       ldo=N, out2=ds.ptr(Vt), ldo2=M, row_offset=0,
                       split_n=N // 2, x=ds.ptr(x), ldx=N, gate=ds.ptr(gate),
                       acc=ds.ptr(out), ldacc=N, acc_load=0, acc_final=1)
    keep = (A, B0, B1, s0, s1, out, Vt, x, gate)
    flops = (4 if mode == ds.EPI_SWIGLU else 2) * M * N * K
    return (lambda: ds.gemm(args)), flops, keep


def attention_case(a):
    g = torch.Generator(device="cuda").manual_seed(0)
    D = a.heads * a.head_dim
    q = torch.randn(a.Tq, D, device="cuda", generator=g).to(torch.bfloat16)
    k = torch.randn(a.T, D, device="cuda", generator=g).to(torch.bfloat16)
    ldvt = (a.T + 127) // 128 * 128
    vt = torch.randn(D, ldvt, device="cuda", generator=g).to(torch.bfloat16)
    o = torch.empty(a.Tq, D, device="cuda", dtype=torch.bfloat16)
    flops = 4 * a.Tq * a.T * D
    if a.no_split:  # whole units only, one after another per CTA
        keep = (q, k, vt, o)
        return (lambda: ds.attention(q, a.Tq, D, k, D, vt, ldvt, a.T, a.heads,
                                     a.head_dim, o, D)), flops, keep
    # the block forward's launch: the last wave's units cut into key ranges
    nb = ds.attention_split_bytes(a.head_dim, 160)
    ws = torch.zeros(nb, dtype=torch.uint8, device="cuda")
    keep = (q, k, vt, o, ws)
    return (lambda: ds.attention_ex(q, a.Tq, D, k, D, vt, ldvt, a.T, a.heads, a.head_dim,
                                    o, D, split_ws=ws, split_bytes=nb)), flops, keep


def modln_case(a):
    x = torch.randn(a.M, a.D, device="cuda")
    sh = torch.randn(a.D, device="cuda") * 0.1
    sc = torch.randn(a.D, device="cuda") * 0.1
    out = torch.empty(a.M, a.D, device="cuda", dtype=torch.bfloat16)
    keep = (x, sh, sc, out)
    return (lambda: ds.modln_cast(x, a.M, a.D, sh, sc, out)), 6 * a.M * a.D, keep


def final_case(a):
    x = torch.randn(a.M, a.D, device="cuda")
    if a.int8:  # int8 W_f with one fp32 scale per output row
        wf = torch.randint(-127, 128, (64, a.D), device="cuda", dtype=torch.int8)
        ws = torch.full((64,), 0.02 / 127, device="cuda")
    else:
        wf = torch.randn(64, a.D, device="cuda") * 0.02
        ws = None
    mod_f = torch.randn(2, a.D, device="cuda") * 0.1
    out = torch.empty(a.M, 64, device="cuda")
    plan = ds.block_plan(a.M, a.D, a.D // 128, 128, 0, 0)
    keep = (x, wf, ws, mod_f, out, plan)
    return (lambda: plan.final_forward(x, wf, ws, mod_f, out)), 4 * a.M * a.D, keep


def expand_case(a):
    q = torch.randint(-127, 128, (a.M, a.D), device="cuda", dtype=torch.int8)
    out = torch.empty(a.M, a.D, device="cuda", dtype=torch.bfloat16)
    keep = (q, out)
    return (lambda: ds.int8_to_bf16(q, a.M * a.D, out)), 3 * a.M * a.D, keep


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("kernel", choices=("gemm", "attention", "modln", "final", "expand"))
    ap.add_argument("--mode", default="store_bf16", choices=sorted(MODES))
    ap.add_argument("--int8", action="store_true")
    ap.add_argument("--scaled", action="store_true")
    ap.add_argument("--M", type=int, default=2048)
    ap.add_argument("--N", type=int, default=3072)
    ap.add_argument("--K", type=int, default=3072)
    ap.add_argument("--D", type=int, default=3072)
    ap.add_argument("--Tq", type=int, default=2048)
    ap.add_argument("--T", type=int, default=8192)
    ap.add_argument("--heads", type=int, default=4)
    ap.add_argument("--head-dim", type=int, default=128)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--no-split", action="store_true",
                    help="attention: no key-range split of the last wave's units")
    a = ap.parse_args(argv)
    dbuild.build()
    ds.load()
    fn, work, keep = {"gemm": gemm_case, "attention": attention_case,
                      "modln": modln_case, "final": final_case,
                      "expand": expand_case}[a.kernel](a)
    fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / a.reps
    unit = "GB/s" if a.kernel in ("modln", "final", "expand") else "TFLOP/s"
    rate = work / (ms / 1e3) / (1e9 if unit == "GB/s" else 1e12)
    print(f"{a.kernel}: {ms:.4f} ms per launch, {rate:.1f} {unit}")
    del keep
    return 0


if __name__ == "__main__":
    sys.exit(main())
