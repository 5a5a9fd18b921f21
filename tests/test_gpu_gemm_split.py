"""The GEMM's work split on the GPU: cutting the last wave's output tiles
into K ranges handed from CTA to CTA must not change a bit.

Every epilogue (Q store with and without the Q/K transform, K/V store,
gated residual, SwiGLU, the down projection with and without its carried
accumulator) runs with bf16 and int8 weights (in both tile shapes: without
and with LoRA K-steps), once whole tiles only (dit_gemm)
and twice with the split (dit_gemm_ex with a CTA cap that makes small cases
cut tiles), on the same inputs; the outputs must be equal bit for bit.
Launches without LoRA run on cluster pairs of CTAs (256-row tiles), those
with LoRA on one-CTA tiles.  The
unsplit results are checked against the oracle in test_gpu_kernels.py and
test_gpu_lora.py."""

import pytest
import torch

from memory_bounded_video_gb300 import build as dbuild
from memory_bounded_video_gb300 import ditstream as ds

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    dbuild.build()
    return ds.load()


def gemm_units(M, N, two_b, pair):
    bm = 256 if pair else 128
    bn = 128 if two_b else 256
    return -(-M // bm) * -(-N // bn)


def bf(g, *shape, std=1.0):
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16).cuda()


class Case:
    """Inputs and output buffers of one GEMM launch; run() resets the
    outputs (x is read-modify-written) and returns copies of them."""

    def __init__(self, mode, M, N, K, int8, seed, qk=False, lora=0, acc_load=0,
                 acc_final=1):
        g = torch.Generator().manual_seed(seed)
        self.mode, self.M, self.N, self.K = mode, M, N, K
        two_b = mode == ds.EPI_SWIGLU
        self.keep = []
        a = bf(g, M, K)
        args = ds.GemmArgs(mode=mode, M=M, N=N, K=K, a=ds.ptr(a), lda=K, ldb=K)
        self.keep.append(a)
        bs = []
        for _ in range(2 if two_b else 1):
            if int8:
                q = torch.randint(-127, 128, (N, K), generator=g, dtype=torch.int16)
                b = q.to(torch.int8).cuda()
                s = (0.02 / 127 * (0.5 + torch.rand(N, generator=g))).cuda()
            else:
                b, s = bf(g, N, K, std=0.05), None
            bs.append((b, s))
            self.keep += [b, s]
        args.b_dtype = ds.W_INT8 if int8 else ds.W_BF16
        args.b0, args.b0_scale = ds.ptr(bs[0][0]), ds.ptr(bs[0][1])
        if two_b:
            args.b1, args.b1_scale = ds.ptr(bs[1][0]), ds.ptr(bs[1][1])
        self.outs = {}

        def out(name, shape, dtype):
            t = torch.zeros(*shape, dtype=dtype, device="cuda")
            self.outs[name] = t
            return t

        if mode in (ds.EPI_STORE_BF16, ds.EPI_SWIGLU):
            args.out, args.ldo = ds.ptr(out("out", (M, N), torch.bfloat16)), N
        elif mode == ds.EPI_KV:
            split = N // 2
            args.split_n, args.row_offset = split, 100
            args.out, args.ldo = ds.ptr(out("k", (M + 100, split), torch.bfloat16)), split
            ldo2 = (M + 100 + 7) // 8 * 8
            args.out2, args.ldo2 = ds.ptr(out("vt", (N - split, ldo2), torch.bfloat16)), ldo2
        if mode in (ds.EPI_RESID, ds.EPI_DOWN):
            self.x0 = torch.randn(M, N, generator=g).cuda()
            gate = torch.rand(N, generator=g).cuda()
            self.keep += [self.x0, gate]
            args.x, args.ldx, args.gate = ds.ptr(out("x", (M, N), torch.float32)), N, ds.ptr(gate)
        if mode == ds.EPI_DOWN:
            args.acc_load, args.acc_final = acc_load, acc_final
            self.acc0 = torch.randn(M, N, generator=g).cuda() * 0.1
            self.keep.append(self.acc0)
            args.acc, args.ldacc = ds.ptr(out("acc", (M, N), torch.float32)), N
        if qk:
            hd = 128
            qn = (1 + 0.1 * torch.randn(hd, generator=g)).cuda()
            ang = torch.rand(M + 100, hd // 2, generator=g, dtype=torch.float64) * 6.28
            cos, sin = ang.cos().float().cuda(), ang.sin().float().cuda()
            self.keep += [qn, cos, sin]
            args.qk_norm, args.rope_cos, args.rope_sin = ds.ptr(qn), ds.ptr(cos), ds.ptr(sin)
            args.head_dim, args.qk_eps, args.rope_pos0 = hd, 1e-6, 37
        if lora:
            u, l = bf(g, M, lora), bf(g, N, lora, std=0.05)
            self.keep += [u, l]
            args.lora_u0, args.lora_ldu0 = ds.ptr(u), lora
            args.lora_l0, args.lora_ldl0, args.lora_rank0 = ds.ptr(l), lora, lora
        self.args = args
        # launches without LoRA run on cluster pairs (256-row tiles, one
        # worker per two CTAs, two hand-off slots per cut tile)
        self.pair = not lora
        self.tiles = gemm_units(M, N, two_b, self.pair)
        self.num_k = K // 64

    def run(self, split_ws=None, split_bytes=0, max_ctas=0):
        for name, t in self.outs.items():
            if name == "x":
                t.copy_(self.x0)
            elif name == "acc":
                t.copy_(self.acc0)
            else:
                t.zero_()
        st = torch.zeros(4, dtype=torch.int32, device="cuda")
        if split_ws is None:
            ds.gemm_ex(self.args, max_ctas=max_ctas, dev_status=st)
        else:
            ds.gemm_ex(self.args, split_ws, split_bytes, max_ctas, dev_status=st)
        torch.cuda.synchronize()
        assert int(st[0].item()) == 0
        return {k: v.clone() for k, v in self.outs.items()}


CASES = [
    # (name, mode, M, N, K, int8, CTA cap, extra)
    ("q_bf16", ds.EPI_STORE_BF16, 1000, 1024, 512, False, 10, {}),
    ("q_int8", ds.EPI_STORE_BF16, 1000, 1024, 512, True, 10, {}),
    ("q_qk_bf16", ds.EPI_STORE_BF16, 700, 768, 256, False, 8, {"qk": True}),
    ("q_qk_int8", ds.EPI_STORE_BF16, 700, 768, 256, True, 8, {"qk": True}),
    ("kv_bf16", ds.EPI_KV, 600, 1024, 512, False, 10, {}),
    ("kv_qk_int8", ds.EPI_KV, 600, 1024, 512, True, 10, {"qk": True}),
    ("resid_int8", ds.EPI_RESID, 900, 768, 1024, True, 10, {}),
    ("swiglu_int8", ds.EPI_SWIGLU, 520, 640, 512, True, 8, {}),
    ("swiglu_bf16", ds.EPI_SWIGLU, 520, 640, 512, False, 8, {}),
    ("down_carry_int8", ds.EPI_DOWN, 700, 512, 1024, True, 8, {"acc_load": 1, "acc_final": 1}),
    ("down_partial_bf16", ds.EPI_DOWN, 700, 512, 1024, False, 10, {"acc_load": 0, "acc_final": 0}),
    ("down_mid_int8", ds.EPI_DOWN, 700, 512, 1024, True, 8, {"acc_load": 1, "acc_final": 0}),
    ("q_lora_int8", ds.EPI_STORE_BF16, 600, 512, 512, True, 4, {"lora": 64}),
    ("swiglu_lora_bf16", ds.EPI_SWIGLU, 600, 512, 512, False, 6, {"lora": 64}),
    # the bench's launch sizes on every SM
    ("q_int8_8192", ds.EPI_STORE_BF16, 8192, 3072, 3072, True, 0, {}),
    ("down_int8_8192", ds.EPI_DOWN, 8192, 3072, 8192, True, 0, {"acc_load": 0, "acc_final": 1}),
]


@pytest.mark.parametrize("name,mode,M,N,K,int8,cap,extra", CASES, ids=[c[0] for c in CASES])
def test_split_gemm_is_bit_identical_to_unsplit(name, mode, M, N, K, int8, cap, extra):
    case = Case(mode, M, N, K, int8, seed=M + N + K, **extra)
    ctas = cap or torch.cuda.get_device_properties(0).multi_processor_count
    if case.pair:
        _, n_split, _ = ds.attention_schedule(case.tiles, case.num_k, max(ctas // 2, 1), 32)
    else:
        _, n_split, _ = ds.attention_schedule(case.tiles, case.num_k, ctas, 64)
    assert n_split > 0, "the case must cut tiles"
    ref = case.run(max_ctas=cap)
    nbytes = ds.gemm_split_bytes(64)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    for _ in range(2):  # the second call reuses the hand-off space as left
        got = case.run(ws, nbytes, cap)
        for k in ref:
            a, b = ref[k], got[k]
            if a.dtype == torch.bfloat16:
                a, b = a.view(torch.int16), b.view(torch.int16)
            else:
                a, b = a.view(torch.int32), b.view(torch.int32)
            assert torch.equal(a, b), f"{name}: {k} differs"
        assert int(ws[:1024].count_nonzero().item()) == 0, "hand-off flags left set"


def test_bf16_residual_launch_is_not_split():
    # its epilogue bounds it: the split would only add work (all whole tiles)
    case = Case(ds.EPI_RESID, 900, 768, 1024, False, seed=5)
    ref = case.run(max_ctas=5)
    nbytes = ds.gemm_split_bytes(64)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    got = case.run(ws, nbytes, 5)
    assert torch.equal(ref["x"].view(torch.int32), got["x"].view(torch.int32))


def test_unsplit_cta_cap_does_not_change_the_result():
    case = Case(ds.EPI_RESID, 900, 768, 1024, True, seed=3)
    outs = [case.run(max_ctas=c)["x"] for c in (0, 1, 7)]
    for o in outs[1:]:
        assert torch.equal(outs[0].view(torch.int32), o.view(torch.int32))


CHILD = """
import sys, torch
sys.path.insert(0, {root!r})
from memory_bounded_video_gb300 import runner, synth
inp = synth.make_inputs(8192, 1024, 16, 2816, seed=11, int8=True, jitter=True)
dev = runner.upload(inp)
stack = runner.DitStack(8192, 1024, 16, 2816, 2048, 2048)
x = dev.x.clone()
stack.forward(x, dev)
stack.check()
torch.save(x.cpu(), {out!r})
"""


def test_block_without_gemm_split_gives_the_same_bits(tmp_path):
    """DITSTREAM_GEMM_SPLIT=0 (read once per process) makes every GEMM of the
    block run whole tiles without a cooperative launch; the block's output
    must keep its bits.  Both runs happen in child processes so that each
    reads the variable afresh."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    outs = []
    for flag in ("1", "0"):
        out = str(tmp_path / f"x_{flag}.pt")
        env = dict(os.environ, DITSTREAM_GEMM_SPLIT=flag)
        subprocess.run([sys.executable, "-c", CHILD.format(root=root, out=out)],
                       env=env, check=True, timeout=600)
        outs.append(torch.load(out))
    assert torch.equal(outs[0].view(torch.int32), outs[1].view(torch.int32))
