"""Per-kernel parity of the CUDA path (through the C ABI) against the oracle.

Inputs are seeded CPU draws (bf16 where the kernel takes bf16); the expected
values are the float64 oracle / the plain definition on exactly those inputs.
Sizes span several tiles and a ragged tail."""

import numpy as np
import pytest
import torch

from memory_bounded_video_gb300 import build as dbuild
from memory_bounded_video_gb300 import ditstream as ds
from oracle import block as ob

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    dbuild.build()
    return ds.load()


def gen(seed):
    g = torch.Generator().manual_seed(seed)
    return g


def randn(g, *shape, std=1.0):
    return torch.randn(*shape, generator=g) * std


def f64(t):
    return t.double().cpu().numpy()


def status_buf():
    return torch.zeros(4, dtype=torch.int32, device="cuda")


def assert_status_ok(st):
    torch.cuda.synchronize()
    assert int(st[0].item()) == 0, "device status word set"


# ---------------------------------------------------------------- modln_cast

@pytest.mark.parametrize("rows,D", [(1, 256), (300, 256), (129, 1024), (70, 3072)])
def test_modln_cast_matches_oracle(rows, D):
    g = gen(rows + D)
    x = randn(g, rows, D) * 2 + 0.5
    shift = randn(g, D, std=0.1)
    scale = randn(g, D, std=0.1)
    out = torch.empty(rows, D, dtype=torch.bfloat16, device="cuda")
    xd, shd, scd = x.cuda(), shift.cuda(), scale.cuda()
    ds.modln_cast(xd, rows, D, shd, scd, out)
    torch.cuda.synchronize()
    ref = ob.ln_modulate(f64(x), f64(shift), f64(scale))
    got = f64(out)
    # one bf16 rounding of a value with fp32 error: within 2^-8 relative
    err = np.abs(got - ref) / np.maximum(np.abs(ref), 1e-3)
    assert err.max() <= 2.0 ** -8 + 1e-4


def test_modln_cast_is_row_local():
    g = gen(3)
    x = randn(g, 256, 1024)
    sh, sc = randn(g, 1024, std=0.1).cuda(), randn(g, 1024, std=0.1).cuda()
    full = torch.empty(256, 1024, dtype=torch.bfloat16, device="cuda")
    part = torch.empty(56, 1024, dtype=torch.bfloat16, device="cuda")
    xd = x.cuda()
    ds.modln_cast(xd, 256, 1024, sh, sc, full)
    ds.modln_cast(xd[200:], 56, 1024, sh, sc, part)
    torch.cuda.synchronize()
    assert torch.equal(full[200:].view(torch.int16), part.view(torch.int16))


# ---------------------------------------------------------------- GEMM

class Gemm:
    """GemmArgs plus references to every device tensor it points at (the
    tensors must outlive the launch)."""

    def __init__(self, mode, a, b, **kw):
        M, K = a.shape
        N = b.shape[0]
        self.keep = [a, b]
        self.args = ds.GemmArgs(mode=mode, M=M, N=N, K=K, a=ds.ptr(a),
                                lda=a.stride(0), b0=ds.ptr(b),
                                ldb=b.stride(0), b_dtype=ds.W_BF16)
        for k, v in kw.items():
            if isinstance(v, torch.Tensor):
                self.keep.append(v)
                v = ds.ptr(v)
            setattr(self.args, k, v)

    def run(self, st=None):
        ds.gemm(self.args, st)


def gemm_args(mode, a, b, **kw):
    return Gemm(mode, a, b, **kw)


def bf16_pair(g, M, N, K, std_a=1.0, std_b=0.05):
    a = randn(g, M, K, std=std_a).to(torch.bfloat16)
    b = randn(g, N, K, std=std_b).to(torch.bfloat16)
    return a, b


def check_close(got, ref, K, what):
    # fp32 accumulation of K bf16 products: error ~ sqrt(K) * 2^-24 * scale
    scale = np.abs(ref).max() + 1e-6
    err = np.abs(got - ref).max() / scale
    assert err < 2e-5 * max(1.0, K / 256), f"{what}: rel err {err}"


@pytest.mark.parametrize("M,N,K", [(1, 32, 64), (300, 288, 320), (128, 256, 64),
                                   (4096, 2048, 256), (777, 800, 1024)])
def test_gemm_store_f32(M, N, K):
    g = gen(M * 7 + N)
    a, b = bf16_pair(g, M, N, K)
    out = torch.full((M, N), float("nan"), device="cuda")
    st = status_buf()
    gemm_args(ds.EPI_STORE_F32, a.cuda(), b.cuda(), out=out, ldo=N).run(st)
    assert_status_ok(st)
    check_close(f64(out), f64(a) @ f64(b).T, K, "store_f32")


def test_gemm_store_bf16_and_row_locality():
    g = gen(11)
    M, N, K = 1000, 512, 512
    a, b = bf16_pair(g, M, N, K)
    ad, bd = a.cuda(), b.cuda()
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    gemm_args(ds.EPI_STORE_BF16, ad, bd, out=out, ldo=N).run()
    part = torch.empty(M - 300, N, dtype=torch.bfloat16, device="cuda")
    gemm_args(ds.EPI_STORE_BF16, ad[300:], bd, out=part, ldo=N).run()
    torch.cuda.synchronize()
    ref = f64(a) @ f64(b).T
    err = np.abs(f64(out) - ref) / np.maximum(np.abs(ref), 1e-2)
    assert err.max() <= 2.0 ** -8 + 1e-3
    assert torch.equal(out[300:].view(torch.int16), part.view(torch.int16))


def test_gemm_kv_epilogue_writes_k_and_transposed_v():
    g = gen(5)
    M, D, row_off, T_pad = 200, 256, 128, 512
    a, b = bf16_pair(g, M, 2 * D, D)
    K = torch.zeros(T_pad, D, dtype=torch.bfloat16, device="cuda")
    Vt = torch.zeros(D, T_pad, dtype=torch.bfloat16, device="cuda")
    gemm_args(ds.EPI_KV, a.cuda(), b.cuda(), out=K, ldo=D, out2=Vt,
              ldo2=T_pad, row_offset=row_off, split_n=D).run()
    torch.cuda.synchronize()
    ref = f64(a) @ f64(b).T
    k_got = f64(K[row_off:row_off + M])
    v_got = f64(Vt[:, row_off:row_off + M]).T
    for got, r in ((k_got, ref[:, :D]), (v_got, ref[:, D:])):
        err = np.abs(got - r) / np.maximum(np.abs(r), 1e-2)
        assert err.max() <= 2.0 ** -8 + 1e-3
    # nothing outside the slab's rows was written
    assert torch.count_nonzero(K[:row_off]) == 0
    assert torch.count_nonzero(Vt[:, row_off + M:]) == 0


def test_gemm_resid_epilogue():
    g = gen(6)
    M, N, K = 333, 1024, 1024
    a, b = bf16_pair(g, M, N, K)
    x = randn(g, M, N)
    gate = torch.rand(N, generator=g)
    xd = x.cuda()
    gemm_args(ds.EPI_RESID, a.cuda(), b.cuda(), x=xd, ldx=N,
              gate=gate.cuda()).run()
    torch.cuda.synchronize()
    ref = f64(x) + f64(gate) * (f64(a) @ f64(b).T)
    assert np.abs(f64(xd) - ref).max() < 1e-4


def test_gemm_swiglu_epilogue():
    g = gen(7)
    M, N, K = 300, 704, 256
    a = randn(g, M, K).to(torch.bfloat16)
    wg = randn(g, N, K, std=0.1).to(torch.bfloat16)
    wu = randn(g, N, K, std=0.1).to(torch.bfloat16)
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    gemm_args(ds.EPI_SWIGLU, a.cuda(), wg.cuda(), b1=wu.cuda(), out=out,
              ldo=N).run()
    torch.cuda.synchronize()
    gv, uv = f64(a) @ f64(wg).T, f64(a) @ f64(wu).T
    ref = ob.silu(gv) * uv
    err = np.abs(f64(out) - ref) / np.maximum(np.abs(ref), 1e-2)
    assert err.max() <= 2.0 ** -7


@pytest.mark.parametrize("fs", [64, 256, 512])
def test_gemm_down_carry_is_bit_identical_to_unsliced(fs):
    g = gen(8 + fs)
    M, D, F = 300, 512, 512
    h = randn(g, M, F).to(torch.bfloat16).cuda()
    wd = randn(g, D, F, std=0.05).to(torch.bfloat16).cuda()
    x = randn(g, M, D)
    gate = torch.rand(D, generator=g).cuda()
    x_ref = x.cuda()
    gemm_args(ds.EPI_DOWN, h, wd, x=x_ref, ldx=D, gate=gate, acc_load=0,
              acc_final=1).run()
    x_sl = x.cuda()
    acc = torch.empty(M, D, device="cuda")
    for f in range(0, F, fs):
        gemm_args(ds.EPI_DOWN, h[:, f:f + fs], wd[:, f:f + fs], x=x_sl,
                  ldx=D, gate=gate, acc=acc, ldacc=D, acc_load=int(f > 0),
                  acc_final=int(f + fs >= F)).run()
    torch.cuda.synchronize()
    ref = f64(x) + f64(gate) * (f64(h) @ f64(wd).T)
    assert np.abs(f64(x_ref) - ref).max() < 1e-4
    assert torch.equal(x_ref, x_sl)


# ---------------------------------------------------------------- attention

def run_attention(q, k, v, heads, hd):
    Tq, T = q.shape[0], k.shape[0]
    D = heads * hd
    ldvt = (T + 127) // 128 * 128
    vt = torch.zeros(D, ldvt, dtype=torch.bfloat16, device="cuda")
    vt[:, :T] = v.cuda().T
    o = torch.empty(Tq, D, dtype=torch.bfloat16, device="cuda")
    st = status_buf()
    qd, kd = q.cuda(), k.cuda()
    ds.attention(qd, Tq, D, kd, D, vt, ldvt, T, heads, hd, o, D, st)
    assert_status_ok(st)
    return o


@pytest.mark.parametrize("Tq,T,H,hd,sharp", [
    (128, 128, 1, 64, 1.0), (200, 300, 2, 64, 1.0), (130, 1000, 2, 128, 1.0),
    (256, 2048, 3, 128, 1.0), (100, 777, 2, 128, 6.0), (64, 5, 2, 64, 4.0)])
def test_attention_matches_oracle(Tq, T, H, hd, sharp):
    g = gen(Tq + T + H)
    D = H * hd
    q = (randn(g, Tq, D) * sharp).to(torch.bfloat16)
    k = randn(g, T, D).to(torch.bfloat16)
    v = randn(g, T, D).to(torch.bfloat16)
    o = run_attention(q, k, v, H, hd)
    ref = ob.mha_attention(f64(q), f64(k), f64(v), H)
    got = f64(o)
    rel_l2 = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel_l2 < 1e-2, rel_l2
    assert np.abs(got - ref).max() < 2e-2 * max(1.0, np.abs(ref).max())


# The running reference max moves only when a row's score exceeds it by more
# than 8 (log2 units).  The kernel computes P against the current max first
# and takes the tile max only for warps where some row's probabilities sum to
# more than 2^8: a later key tile whose scores sit 7.48 above the first
# tile's max (sum far above 2^8, max not moved) and one 8.66 above (max
# moved, O and l rescaled, P redone).  Every query row scores key j as
# q . k_j / sqrt(d) = b_j with q = (sqrt(d), 0, ...) and k_j = (b_j, 0, ...).
@pytest.mark.parametrize("hd", [64, 128])
@pytest.mark.parametrize("b1", [9.1875, 10.0], ids=["sum_over_256_max_kept", "max_moved"])
def test_attention_later_tile_above_the_reference_max(b1, hd):
    H, Tq, T = 1, 256, 3 * 128 + 17
    g = gen(23)
    q = torch.zeros(Tq, hd)
    q[:, 0] = hd ** 0.5  # q . k / sqrt(hd) = k[0]
    k = torch.zeros(T, hd)
    k[0, 0] = 4.0              # first tile: max score 4, the others 0
    k[128:256, 0] = b1         # second tile: every score b1
    k[256:, 0] = -2.0          # third tile and the ragged tail: small
    q, k = q.to(torch.bfloat16), k.to(torch.bfloat16)
    v = randn(g, T, hd).to(torch.bfloat16)
    o = run_attention(q, k, v, H, hd)
    ref = ob.mha_attention(f64(q), f64(k), f64(v), H)
    got = f64(o)
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 1e-2
    assert np.abs(got - ref).max() < 2e-2


# Random scores with single keys planted in a later tile that score far above
# every earlier key for a few rows of a warp only: those rows move their max,
# the warp's other rows keep theirs (multiplied by exactly 1).
@pytest.mark.parametrize("hd", [64, 128])
def test_attention_max_moves_for_some_rows_of_a_warp(hd):
    H, Tq, T = 2, 256, 1000
    D = H * hd
    g = gen(24)
    q = randn(g, Tq, D).to(torch.bfloat16)
    k = randn(g, T, D)
    rows = [3, 17, 40, 130, 255]
    for i, r in enumerate(rows):
        for h in range(H):
            k[3 * 128 + 5 + i, h * hd:(h + 1) * hd] = 2.5 * q[r, h * hd:(h + 1) * hd].float()
    k = k.to(torch.bfloat16)
    v = randn(g, T, D).to(torch.bfloat16)
    o = run_attention(q, k, v, H, hd)
    ref = ob.mha_attention(f64(q), f64(k), f64(v), H)
    got = f64(o)
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 1e-2
    assert np.abs(got - ref).max() < 2e-2 * max(1.0, np.abs(ref).max())
    # the case does what it is for: every planted row's planted score is more
    # than 8 (log2 units) above every score of the first key tile
    qf, kf = f64(q), f64(k)
    for i, r in enumerate(rows):
        for h in range(H):
            sc = kf[:, h * hd:(h + 1) * hd] @ qf[r, h * hd:(h + 1) * hd] / np.sqrt(hd) * np.log2(np.e)
            assert sc[3 * 128 + 5 + i] > sc[:128].max() + 8


def test_attention_rows_do_not_depend_on_slab():
    g = gen(21)
    H, hd, T = 2, 128, 700
    D = H * hd
    q = randn(g, 400, D).to(torch.bfloat16)
    k = randn(g, T, D).to(torch.bfloat16)
    v = randn(g, T, D).to(torch.bfloat16)
    full = run_attention(q, k, v, H, hd)
    part = run_attention(q[256:], k, v, H, hd)
    assert torch.equal(full[256:].view(torch.int16), part.view(torch.int16))


def test_attention_equal_values_return_that_row():
    g = gen(22)
    H, hd, T = 2, 64, 333
    D = H * hd
    q = (randn(g, 150, D) * 3).to(torch.bfloat16)
    k = (randn(g, T, D) * 3).to(torch.bfloat16)
    row = randn(g, D).to(torch.bfloat16)
    v = row.expand(T, D).contiguous()
    o = run_attention(q, k, v, H, hd)
    # sum of bf16-rounded probabilities is within 2^-8 of one
    np.testing.assert_allclose(f64(o), np.tile(f64(row), (150, 1)), rtol=1e-2,
                               atol=1e-2)


# ---------------------------------------------------------------- int8 weights

def int8_weight(g, N, K, jitter=True):
    q = torch.randint(-127, 128, (N, K), generator=g, dtype=torch.int16).to(torch.int8)
    s = torch.full((N,), 0.02 / 127)
    if jitter:
        s = s * (0.5 + torch.rand(N, generator=g))
    return q, s


def deq(q, s):
    return ob.dequant_int8(q.numpy(), s.numpy())


@pytest.mark.parametrize("M,N,K", [(1, 32, 64), (300, 288, 320), (1000, 512, 1024)])
def test_gemm_int8_store_f32(M, N, K):
    g = gen(100 + M)
    a = randn(g, M, K).to(torch.bfloat16)
    q, s = int8_weight(g, N, K)
    out = torch.full((M, N), float("nan"), device="cuda")
    st = status_buf()
    gemm_args(ds.EPI_STORE_F32, a.cuda(), q.cuda(), out=out, ldo=N,
              b_dtype=ds.W_INT8, b0_scale=s.cuda()).run(st)
    assert_status_ok(st)
    check_close(f64(out), f64(a) @ deq(q, s).T, K, "int8 store_f32")


def test_gemm_int8_swiglu_and_kv():
    g = gen(101)
    M, N, K = 300, 704, 256
    a = randn(g, M, K).to(torch.bfloat16)
    qg, sg = int8_weight(g, N, K)
    qu, su = int8_weight(g, N, K)
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    gemm_args(ds.EPI_SWIGLU, a.cuda(), qg.cuda(), b1=qu.cuda(), out=out, ldo=N,
              b_dtype=ds.W_INT8, b0_scale=sg.cuda(), b1_scale=su.cuda()).run()
    torch.cuda.synchronize()
    ref = ob.silu(f64(a) @ deq(qg, sg).T) * (f64(a) @ deq(qu, su).T)
    err = np.abs(f64(out) - ref) / np.maximum(np.abs(ref), 1e-2)
    assert err.max() <= 2.0 ** -7
    # K/V store with int8 weights
    D, row_off, T_pad = 256, 64, 512
    qkv, skv = int8_weight(g, 2 * D, D)
    a2 = randn(g, 200, D).to(torch.bfloat16)
    Kb = torch.zeros(T_pad, D, dtype=torch.bfloat16, device="cuda")
    Vt = torch.zeros(D, T_pad, dtype=torch.bfloat16, device="cuda")
    gemm_args(ds.EPI_KV, a2.cuda(), qkv.cuda(), out=Kb, ldo=D, out2=Vt, ldo2=T_pad,
              row_offset=row_off, split_n=D, b_dtype=ds.W_INT8,
              b0_scale=skv.cuda()).run()
    torch.cuda.synchronize()
    ref = f64(a2) @ deq(qkv, skv).T
    for got, r in ((f64(Kb[row_off:row_off + 200]), ref[:, :D]),
                   (f64(Vt[:, row_off:row_off + 200]).T, ref[:, D:])):
        e = np.abs(got - r) / np.maximum(np.abs(r), 1e-2)
        assert e.max() <= 2.0 ** -8 + 1e-3


@pytest.mark.parametrize("fs", [64, 256])
def test_gemm_int8_down_carry_bit_identical(fs):
    g = gen(102 + fs)
    M, D, F = 300, 512, 512
    h = randn(g, M, F).to(torch.bfloat16).cuda()
    q, s = int8_weight(g, D, F)
    qd, sd = q.cuda(), s.cuda()
    x = randn(g, M, D)
    gate = torch.rand(D, generator=g).cuda()
    x_ref = x.cuda()
    gemm_args(ds.EPI_DOWN, h, qd, x=x_ref, ldx=D, gate=gate, acc_load=0,
              acc_final=1, b_dtype=ds.W_INT8, b0_scale=sd).run()
    x_sl = x.cuda()
    acc = torch.empty(M, D, device="cuda")
    for f in range(0, F, fs):
        gemm_args(ds.EPI_DOWN, h[:, f:f + fs], qd[:, f:f + fs], x=x_sl, ldx=D,
                  gate=gate, acc=acc, ldacc=D, acc_load=int(f > 0),
                  acc_final=int(f + fs >= F), b_dtype=ds.W_INT8, b0_scale=sd).run()
    torch.cuda.synchronize()
    ref = f64(x) + f64(gate) * (f64(h) @ deq(q, s).T)
    assert np.abs(f64(x_ref) - ref).max() < 1e-4
    assert torch.equal(x_ref, x_sl)


def test_attention_probabilities_elementwise():
    # With V = I (T = d keys) the output row is the probability row itself,
    # so every exponential is checked element by element: bf16 rounding of P
    # and of the output (up to 2^-8 relative each) bound the relative error;
    # an error of 1% in the exponential for any subset of keys exceeds it.
    g = gen(23)
    hd, T, Tq = 128, 128, 256
    q = (randn(g, Tq, hd) * 2).to(torch.bfloat16)
    k = (randn(g, T, hd) * 2).to(torch.bfloat16)
    v = torch.eye(T, hd).to(torch.bfloat16)
    o = run_attention(q, k, v, 1, hd)
    ref = ob.mha_attention(f64(q), f64(k), f64(v), 1)
    got = f64(o)
    big = ref > 1e-3
    rel = np.abs(got - ref)[big] / ref[big]
    assert rel.max() < 2 * 2.0 ** -8 + 1e-4, rel.max()
    np.testing.assert_allclose(got.sum(axis=1), 1.0, atol=2e-2)
