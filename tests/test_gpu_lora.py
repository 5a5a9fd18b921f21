"""Activation-space LoRA in the tensor-core GEMM and the block forward,
against the float64 oracle (``oracle.block.lora_delta``).

"ComfyUI-StaticPipeline", section "Activation-space LoRA (bypass mode)":
y = W x + alpha B (A x) with W left packed; "Four levels of chunking": the
delta is added chunk by chunk, in place.  Here the delta's K-steps join W's
accumulation, so the output stays bit-identical across chunk settings and
FFN slice widths."""

import numpy as np
import pytest
import torch

from memory_bounded_video_gb300 import build as dbuild
from memory_bounded_video_gb300 import ditstream as ds
from memory_bounded_video_gb300 import runner, synth
from oracle import block as ob

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
MAX_ABS = 5e-2
BRANCH_REL_L2 = 2e-2


@pytest.fixture(scope="module", autouse=True)
def lib():
    dbuild.build()
    return ds.load()


def f64(t):
    return t.double().cpu().numpy()


class Gemm:
    """GemmArgs plus the device tensors it points at."""

    def __init__(self, **kw):
        self.keep = []
        self.args = ds.GemmArgs()
        for k, v in kw.items():
            if isinstance(v, torch.Tensor):
                self.keep.append(v)
                v = ds.ptr(v)
            setattr(self.args, k, v)

    def run(self):
        st = torch.zeros(4, dtype=torch.int32, device="cuda")
        ds.gemm(self.args, st)
        torch.cuda.synchronize()
        assert int(st[0]) == 0


def bf(g, *shape, std=1.0):
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


# ---------------------------------------------------------------- prepare

@pytest.mark.parametrize("with_scale", [False, True])
def test_lora_prepare_is_exact(with_scale):
    g = torch.Generator().manual_seed(1)
    rows, rank = 777, 64
    b = bf(g, rows, rank, std=0.02)
    s = (0.02 / 127 * (0.5 + torch.rand(rows, generator=g))) if with_scale else None
    out = torch.empty(rows, rank, dtype=torch.bfloat16, device="cuda")
    ds.lora_prepare(b.cuda(), rows, rank, rank, 0.75, None if s is None else s.cuda(),
                    out, rank)
    torch.cuda.synchronize()
    ref = 0.75 * b.float()
    if s is not None:
        ref = ref / s[:, None]
    assert torch.equal(out.cpu(), ref.to(torch.bfloat16))


# ---------------------------------------------------------------- GEMM

@pytest.mark.parametrize("M,N,K,r", [(300, 384, 256, 32), (129, 512, 128, 96),
                                     (1000, 256, 512, 200), (64, 640, 64, 8)])
def test_gemm_lora_store_f32(M, N, K, r):
    g = torch.Generator().manual_seed(M + r)
    a, b = bf(g, M, K), bf(g, N, K, std=0.05)
    u, l = bf(g, M, r), bf(g, N, r, std=0.05)
    out = torch.full((M, N), float("nan"), device="cuda")
    Gemm(mode=ds.EPI_STORE_F32, M=M, N=N, K=K, a=a.cuda(), lda=K, b0=b.cuda(), ldb=K,
         b_dtype=ds.W_BF16, out=out, ldo=N, lora_u0=u.cuda(), lora_ldu0=r,
         lora_l0=l.cuda(), lora_ldl0=r, lora_rank0=r).run()
    ref = f64(a) @ f64(b).T + f64(u) @ f64(l).T
    err = np.abs(f64(out) - ref).max() / np.abs(ref).max()
    assert err < 2e-5 * max(1.0, (K + r) / 256), err


@pytest.mark.parametrize("int8,halves", [(False, (1, 1)), (False, (1, 0)), (False, (0, 1)),
                                         (True, (1, 1))])
def test_gemm_lora_swiglu(int8, halves):
    g = torch.Generator().manual_seed(7 + int8)
    M, N, K, r0, r1 = 300, 384, 256, 64, 32
    a = bf(g, M, K)
    if int8:
        qg = torch.randint(-127, 128, (N, K), generator=g, dtype=torch.int16).to(torch.int8)
        qu = torch.randint(-127, 128, (N, K), generator=g, dtype=torch.int16).to(torch.int8)
        sg = 0.02 / 127 * (0.5 + torch.rand(N, generator=g))
        su = 0.02 / 127 * (0.5 + torch.rand(N, generator=g))
        wg, wu = ob.dequant_int8(qg.numpy(), sg.numpy()), ob.dequant_int8(qu.numpy(), su.numpy())
        extra = dict(b0=qg.cuda(), b1=qu.cuda(), b_dtype=ds.W_INT8, b0_scale=sg.cuda(),
                     b1_scale=su.cuda())
    else:
        bg, bu = bf(g, N, K, std=0.05), bf(g, N, K, std=0.05)
        wg, wu = f64(bg), f64(bu)
        extra = dict(b0=bg.cuda(), b1=bu.cuda(), b_dtype=ds.W_BF16)
    ug, lg = bf(g, M, r0), bf(g, N, r0, std=0.05)
    uu, lu = bf(g, M, r1), bf(g, N, r1, std=0.05)
    # with int8 weights L carries 1 / row scale (the epilogue multiplies by it)
    lg_dev, lu_dev = lg.cuda(), lu.cuda()
    if int8:
        lg_dev, lu_dev = torch.empty_like(lg_dev), torch.empty_like(lu_dev)
        ds.lora_prepare(lg.cuda(), N, r0, r0, 1.0, sg.cuda(), lg_dev, r0)
        ds.lora_prepare(lu.cuda(), N, r1, r1, 1.0, su.cuda(), lu_dev, r1)
    kw = {}
    if halves[0]:
        kw.update(lora_u0=ug.cuda(), lora_ldu0=r0, lora_l0=lg_dev, lora_ldl0=r0, lora_rank0=r0)
    if halves[1]:
        kw.update(lora_u1=uu.cuda(), lora_ldu1=r1, lora_l1=lu_dev, lora_ldl1=r1, lora_rank1=r1)
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    Gemm(mode=ds.EPI_SWIGLU, M=M, N=N, K=K, a=a.cuda(), lda=K, ldb=K, out=out, ldo=N,
         **extra, **kw).run()
    # the GEMM's own inputs: with int8 weights L enters as the prepared
    # bf16(L / s) times s (that rounding has its own exact test above)
    lg64, lu64 = f64(lg), f64(lu)
    if int8:
        lg64 = f64(lg_dev) * sg.double().numpy()[:, None]
        lu64 = f64(lu_dev) * su.double().numpy()[:, None]
    gate = f64(a) @ wg.T + (f64(ug) @ lg64.T if halves[0] else 0)
    up = f64(a) @ wu.T + (f64(uu) @ lu64.T if halves[1] else 0)
    ref = ob.silu(gate) * up
    err = np.abs(f64(out) - ref) / np.maximum(np.abs(ref), 1e-2)
    assert err.max() <= 2.0 ** -7, err.max()


def test_store_bf16_starts_from_the_fp32_carry():
    g = torch.Generator().manual_seed(3)
    M, N, K = 333, 96, 128
    a, b = bf(g, M, K), bf(g, N, K, std=0.05)
    carry = torch.randn(M, N, generator=g)
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    Gemm(mode=ds.EPI_STORE_BF16, M=M, N=N, K=K, a=a.cuda(), lda=K, b0=b.cuda(), ldb=K,
         b_dtype=ds.W_BF16, out=out, ldo=N, acc=carry.cuda(), ldacc=N, acc_load=1).run()
    ref = f64(carry) + f64(a) @ f64(b).T
    err = np.abs(f64(out) - ref) / np.maximum(np.abs(ref), 1e-2)
    assert err.max() <= 2.0 ** -8 + 1e-4


# ---------------------------------------------------------------- block

def weights64(bw):
    if bw.int8:
        return ob.DitWeights(**{k: ob.dequant_int8(v.numpy(), bw.scales[k].numpy())
                                for k, v in bw.named().items()})
    return ob.DitWeights(**{k: v.double().numpy() for k, v in bw.named().items()})


def lora64(lora):
    return {k: (f64(A), f64(B), al) for k, (A, B, al) in lora.items()}


def run_block(inp, cm, ca, fs=0, lora=None, rank=0, qk=None):
    T, D = inp.x.shape
    dev = runner.upload(inp)
    stack = runner.DitStack(T, D, inp.meta["heads"], inp.meta["F"], cm, ca, fs,
                            lora_rank=rank)
    dl = None if lora is None else [runner.upload_lora(lora, dev.blocks[0])]
    x = dev.x.clone()
    stack.forward(x, dev, lora=dl, qk=None if qk is None else runner.upload_qk(qk))
    stack.check()
    return x


def compare(got, ref, x_in):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    mx = np.abs(got - ref).max()
    br = np.linalg.norm(got - ref) / np.linalg.norm(ref - x_in)
    return rel, mx, br


@pytest.mark.parametrize("T,D,heads,F,int8,rank", [
    (512, 256, 4, 704, False, 32),
    (1000, 1024, 8, 1024, False, 64),    # ragged T, d = 128
    (640, 1024, 8, 1024, True, 96),      # int8 weights, rank not a multiple of 64
])
def test_block_with_lora_matches_oracle_and_is_chunk_invariant(T, D, heads, F, int8, rank):
    inp = synth.make_inputs(T, D, heads, F, seed=T + rank, int8=int8, jitter=int8)
    lora = synth.make_lora(D, F, rank, seed=rank, alpha=0.5)
    outs = [run_block(inp, cm, ca, fs, lora, rank)
            for cm, ca, fs in [(0, 0, 0), (128, 128, 64), (256, 384, 256)]]
    for x in outs[1:]:
        assert torch.equal(x, outs[0])
    x_in = inp.x.double().numpy()
    ref = ob.dit_block(x_in, weights64(inp.blocks[0]), inp.mods[0].double().numpy(),
                       heads, lora=lora64(lora))
    rel, mx, br = compare(outs[0].cpu().numpy(), ref, x_in)
    assert rel <= REL_L2 and mx <= MAX_ABS and br <= BRANCH_REL_L2, (rel, mx, br)
    # the adapters change the result, and the oracle without them is far off
    plain = run_block(inp, 128, 128)
    assert not torch.equal(plain, outs[0])
    ref0 = ob.dit_block(x_in, weights64(inp.blocks[0]), inp.mods[0].double().numpy(), heads)
    assert compare(outs[0].cpu().numpy(), ref0, x_in)[2] > 3 * BRANCH_REL_L2


@pytest.mark.parametrize("names", [("qkv",), ("o",), ("gate",), ("up",), ("down",)])
def test_each_adapter_alone(names):
    inp = synth.make_inputs(512, 256, 4, 704, seed=21)
    lora = synth.make_lora(256, 704, 32, seed=5, names=names, alpha=1.0)
    x = run_block(inp, 128, 256, 64, lora, 32)
    x_in = inp.x.double().numpy()
    ref = ob.dit_block(x_in, weights64(inp.blocks[0]), inp.mods[0].double().numpy(), 4,
                       lora=lora64(lora))
    rel, mx, br = compare(x.cpu().numpy(), ref, x_in)
    assert rel <= REL_L2 and mx <= MAX_ABS and br <= BRANCH_REL_L2, (names, rel, mx, br)


def test_no_adapters_is_the_plain_forward():
    inp = synth.make_workload("dit_T512_D256", seed=8)
    a = run_block(inp, 128, 128, 0, {}, 64)
    assert torch.equal(a, run_block(inp, 128, 128))


def test_lora_with_qk_transform():
    inp = synth.make_inputs(768, 1024, 8, 1024, seed=4)
    lora = synth.make_lora(1024, 1024, 64, seed=2)
    qk = synth.make_qk(768, 128, seed=3, angles="axial")
    x = run_block(inp, 256, 256, 512, lora, 64, qk)
    x_in = inp.x.double().numpy()
    qk64 = {k: (v.double().numpy() if isinstance(v, torch.Tensor) else v)
            for k, v in qk.items()}
    ref = ob.dit_block(x_in, weights64(inp.blocks[0]), inp.mods[0].double().numpy(), 8,
                       qk=qk64, lora=lora64(lora))
    rel, mx, br = compare(x.cpu().numpy(), ref, x_in)
    assert rel <= REL_L2 and mx <= MAX_ABS and br <= BRANCH_REL_L2, (rel, mx, br)


def test_block_T16384_D3072_int8_lora_sampled_rows():
    inp = synth.make_inputs(16384, 3072, 24, 8192, seed=11, int8=True, jitter=True)
    lora = synth.make_lora(3072, 8192, 64, seed=11)
    x = run_block(inp, 8192, 8192, 4096, lora, 64)
    T = 16384
    rng = np.random.default_rng(2)
    rows = np.array(sorted(set(range(32)) | set(range(T - 32, T))
                           | set(rng.choice(T, 96, replace=False).tolist())))
    ref, _ = ob.dit_block_rows(inp.x.double().numpy(), weights64(inp.blocks[0]),
                               inp.mods[0].double().numpy(), 24, rows, lora=lora64(lora))
    rel, mx, br = compare(x.cpu().numpy()[rows], ref, inp.x.double().numpy()[rows])
    assert rel <= REL_L2 and mx <= MAX_ABS and br <= BRANCH_REL_L2, (rel, mx, br)
