"""Q/K RMSNorm + rotary embedding fused into the Q and K projection
epilogues, against the float64 oracle (``oracle.block.qk_transform``).

"Proposal: Generic memory-aware streaming execution for transformer models",
attention section: the model's Q normalisation and positional transform run
on each bounded Q region; K gets the same in pass one.  The transform is
row-local and uses each token's global position, so the block output stays
bit-identical across chunk settings."""

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
    return None if t is None else t.double().cpu().numpy()


def dev(t):
    return None if t is None else t.cuda().contiguous()


def weights64(bw):
    if bw.int8:
        return ob.DitWeights(**{k: ob.dequant_int8(v.numpy(), bw.scales[k].numpy())
                                for k, v in bw.named().items()})
    return ob.DitWeights(**{k: v.double().numpy() for k, v in bw.named().items()})


def qk64(qk):
    return dict(q_norm=f64(qk["q_norm"]), k_norm=f64(qk["k_norm"]),
                cos=f64(qk["cos"]), sin=f64(qk["sin"]), eps=qk["eps"])


def close_bf16(got, ref, what):
    # one bf16 rounding (2^-8 relative) of a value with fp32 error
    err = np.abs(got - ref) / np.maximum(np.abs(ref), 0.05)
    assert err.max() <= 2.0 ** -8 + 2e-3, f"{what}: {err.max()}"


# ---------------------------------------------------------------- GEMM stage

CASES = [  # (head_dim, angles, norm, int8)
    (128, "axial", True, False), (64, "random", True, False),
    (128, "random", False, False), (64, None, True, False),
    (128, "random", True, True), (64, "axial", False, True),
]


@pytest.mark.parametrize("d,angles,norm,int8", CASES)
def test_q_projection_with_transform(d, angles, norm, int8):
    g = torch.Generator().manual_seed(d + 3 * int(norm) + 7 * int(int8))
    M, D, T, off = 300, 512, 700, 257  # ragged M; positions 257..556
    a = (torch.randn(M, D, generator=g)).to(torch.bfloat16)
    if int8:
        q = torch.randint(-127, 128, (D, D), generator=g, dtype=torch.int16).to(torch.int8)
        s = 0.02 / 127 * (0.5 + torch.rand(D, generator=g))
        w64 = ob.dequant_int8(q.numpy(), s.numpy())
        b, extra = q, dict(b_dtype=ds.W_INT8, b0_scale=dev(s))
    else:
        b = (torch.randn(D, D, generator=g) * 0.05).to(torch.bfloat16)
        w64, extra = f64(b), {}
    qk = synth.make_qk(T, d, seed=d, angles=angles, norm=norm)
    keep = [dev(a), dev(b), dev(qk["q_norm"]), dev(qk["cos"]), dev(qk["sin"])]
    out = torch.full((M, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    args = ds.GemmArgs(mode=ds.EPI_STORE_BF16, M=M, N=D, K=D, a=ds.ptr(keep[0]), lda=D,
                       b0=ds.ptr(keep[1]), ldb=D, b_dtype=ds.W_BF16, out=ds.ptr(out),
                       ldo=D, rope_pos0=off, qk_norm=ds.ptr(keep[2]),
                       rope_cos=ds.ptr(keep[3]), rope_sin=ds.ptr(keep[4]), head_dim=d,
                       qk_eps=1e-6)
    for k, v in extra.items():
        keep.append(v)
        setattr(args, k, ds.ptr(v) if isinstance(v, torch.Tensor) else v)
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    ds.gemm(args, st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    rows = np.arange(off, off + M)
    cos = None if qk["cos"] is None else f64(qk["cos"])[rows]
    sin = None if qk["sin"] is None else f64(qk["sin"])[rows]
    ref = ob.qk_transform(f64(a) @ w64.T, D // d, f64(qk["q_norm"]), cos, sin)
    close_bf16(f64(out), ref, "Q")


@pytest.mark.parametrize("d,int8", [(128, False), (64, True)])
def test_kv_projection_transforms_k_only(d, int8):
    g = torch.Generator().manual_seed(40 + d)
    M, D, T, off, T_pad = 200, 384, 640, 300, 640  # D = 3 x 128: a tile straddles K|V
    a = torch.randn(M, D, generator=g).to(torch.bfloat16)
    if int8:
        q = torch.randint(-127, 128, (2 * D, D), generator=g, dtype=torch.int16).to(torch.int8)
        s = 0.02 / 127 * (0.5 + torch.rand(2 * D, generator=g))
        w64 = ob.dequant_int8(q.numpy(), s.numpy())
        b, extra = q, dict(b_dtype=ds.W_INT8, b0_scale=dev(s))
    else:
        b = (torch.randn(2 * D, D, generator=g) * 0.05).to(torch.bfloat16)
        w64, extra = f64(b), {}
    qk = synth.make_qk(T, d, seed=5, angles="random")
    keep = [dev(a), dev(b), dev(qk["k_norm"]), dev(qk["cos"]), dev(qk["sin"])]
    K = torch.zeros(T_pad, D, dtype=torch.bfloat16, device="cuda")
    Vt = torch.zeros(D, T_pad, dtype=torch.bfloat16, device="cuda")
    args = ds.GemmArgs(mode=ds.EPI_KV, M=M, N=2 * D, K=D, a=ds.ptr(keep[0]), lda=D,
                       b0=ds.ptr(keep[1]), ldb=D, b_dtype=ds.W_BF16, out=ds.ptr(K), ldo=D,
                       out2=ds.ptr(Vt), ldo2=T_pad, row_offset=off, rope_pos0=off, split_n=D,
                       qk_norm=ds.ptr(keep[2]), rope_cos=ds.ptr(keep[3]),
                       rope_sin=ds.ptr(keep[4]), head_dim=d, qk_eps=1e-6)
    for k, v in extra.items():
        keep.append(v)
        setattr(args, k, ds.ptr(v) if isinstance(v, torch.Tensor) else v)
    ds.gemm(args)
    torch.cuda.synchronize()
    acc = f64(a) @ w64.T
    rows = np.arange(off, off + M)
    ref_k = ob.qk_transform(acc[:, :D], D // d, f64(qk["k_norm"]),
                            f64(qk["cos"])[rows], f64(qk["sin"])[rows])
    close_bf16(f64(K[off:off + M]), ref_k, "K")
    close_bf16(f64(Vt[:, off:off + M]).T, acc[:, D:], "V")
    # rows outside [off, off + M) untouched
    assert not K[:off].any() and not K[off + M:].any()


# ---------------------------------------------------------------- whole block

def run_block(inp, cm, ca, fs=0, qk=None):
    T, D = inp.x.shape
    d_in = runner.upload(inp)
    stack = runner.DitStack(T, D, inp.meta["heads"], inp.meta["F"], cm, ca, fs)
    x = d_in.x.clone()
    stack.forward(x, d_in, qk=None if qk is None else runner.upload_qk(qk))
    stack.check()
    return x


def compare(got, ref, x_in):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    mx = np.abs(got - ref).max()
    br = np.linalg.norm(got - ref) / np.linalg.norm(ref - x_in)
    return rel, mx, br


@pytest.mark.parametrize("T,D,heads,F,int8,angles", [
    (512, 256, 4, 704, False, "axial"),     # d = 64
    (1000, 1024, 8, 704, False, "random"),  # d = 128, ragged T
    (640, 1024, 8, 1024, True, "axial"),    # int8 weights
])
def test_block_with_qk_matches_oracle_and_is_chunk_invariant(T, D, heads, F, int8, angles):
    inp = synth.make_inputs(T, D, heads, F, seed=T + D, int8=int8, jitter=int8)
    qk = synth.make_qk(T, D // heads, seed=T, angles=angles)
    outs = [run_block(inp, cm, ca, fs, qk)
            for cm, ca, fs in [(0, 0, 0), (128, 128, 0), (256, 384, 256)]]
    for x in outs[1:]:
        assert torch.equal(x, outs[0])
    x_in = inp.x.double().numpy()
    ref = ob.dit_block(x_in, weights64(inp.blocks[0]), inp.mods[0].double().numpy(),
                       heads, qk=qk64(qk))
    rel, mx, br = compare(outs[0].cpu().numpy(), ref, x_in)
    assert rel <= REL_L2 and mx <= MAX_ABS and br <= BRANCH_REL_L2, (rel, mx, br)
    # the transform changes the result (it is not silently skipped)
    plain = run_block(inp, 128, 128)
    assert not torch.equal(plain, outs[0])


def test_empty_transform_is_the_plain_forward():
    inp = synth.make_workload("dit_T512_D256", seed=9)
    qk = synth.make_qk(512, 64, angles=None, norm=False)
    assert torch.equal(run_block(inp, 128, 256, qk=qk), run_block(inp, 128, 256))


def test_zero_angles_and_unit_norm_weights_is_norm_only():
    # cos = 1, sin = 0 turns the rotation into the identity: the result must
    # equal the norm-only transform bit for bit
    inp = synth.make_workload("dit_T512_D256", seed=10)
    qk = synth.make_qk(512, 64, angles="random")
    ident = dict(qk, cos=torch.ones_like(qk["cos"]), sin=torch.zeros_like(qk["sin"]))
    norm_only = dict(qk, cos=None, sin=None)
    assert torch.equal(run_block(inp, 128, 128, qk=ident),
                       run_block(inp, 128, 128, qk=norm_only))


def test_block_T16384_D3072_with_qk_sampled_rows():
    name = "dit_T16384_D3072"
    inp = synth.make_workload(name, seed=3)
    T = inp.x.shape[0]
    qk = synth.make_qk(T, 128, seed=1, angles="axial")
    x = run_block(inp, 8192, 8192, qk=qk)
    rng = np.random.default_rng(1)
    rows = np.array(sorted(set(range(64)) | set(range(T - 64, T))
                           | set(rng.choice(T, 128, replace=False).tolist())))
    ref, _ = ob.dit_block_rows(inp.x.double().numpy(), weights64(inp.blocks[0]),
                               inp.mods[0].double().numpy(), 24, rows, qk=qk64(qk))
    rel, mx, br = compare(x.cpu().numpy()[rows], ref, inp.x.double().numpy()[rows])
    assert rel <= REL_L2 and mx <= MAX_ABS and br <= BRANCH_REL_L2, (rel, mx, br)
