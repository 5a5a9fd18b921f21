"""The GEMM's cluster-pair tiles against its one-CTA tiles, bit for bit.

Launches without LoRA run on pairs of CTAs (256 x 256 output tiles, M = 256
MMAs issued by one CTA for both); launches with LoRA K-steps keep one-CTA
128-row tiles.  A LoRA adapter whose L factor is all zeros adds exact zeros
after W's K-steps, so the one-CTA launch with it and the pair launch without
it must agree in every bit, for every epilogue, with bf16 and int8 weights,
at ragged sizes (rows, columns and K not multiples of the tiles).  Agreement
with the oracle is checked in test_gpu_kernels.py."""

import pytest
import torch

from memory_bounded_video_gb300 import build as dbuild
from memory_bounded_video_gb300 import ditstream as ds
from test_gpu_gemm_split import Case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    dbuild.build()
    return ds.load()


CASES = [
    # (name, mode, M, N, K, int8, extra)
    ("store_bf16", ds.EPI_STORE_BF16, 700, 768, 320, False, {}),
    ("store_bf16_int8", ds.EPI_STORE_BF16, 700, 768, 320, True, {}),
    ("store_qk_int8", ds.EPI_STORE_BF16, 300, 512, 256, True, {"qk": True}),
    ("kv_bf16", ds.EPI_KV, 333, 1024, 256, False, {}),
    ("kv_qk_int8", ds.EPI_KV, 333, 1024, 256, True, {"qk": True}),
    ("resid_bf16", ds.EPI_RESID, 520, 384, 512, False, {}),
    ("resid_int8", ds.EPI_RESID, 520, 384, 512, True, {}),
    ("swiglu_bf16", ds.EPI_SWIGLU, 400, 640, 256, False, {}),
    ("swiglu_int8", ds.EPI_SWIGLU, 400, 640, 256, True, {}),
    ("down_carry_int8", ds.EPI_DOWN, 257, 512, 512, True, {"acc_load": 1, "acc_final": 1}),
    ("down_partial_bf16", ds.EPI_DOWN, 257, 512, 512, False, {"acc_load": 0, "acc_final": 0}),
    ("store_f32_tiny", ds.EPI_STORE_F32, 1, 32, 64, False, {}),
    # fewer K-steps than converter groups and than ring stages
    ("store_int8_k64", ds.EPI_STORE_BF16, 300, 512, 64, True, {}),
    ("swiglu_int8_k192", ds.EPI_SWIGLU, 200, 384, 192, True, {}),
    ("down_int8_k128", ds.EPI_DOWN, 300, 256, 128, True, {"acc_load": 1, "acc_final": 1}),
]


def store_f32_case(M, N, K, seed, lora):
    g = torch.Generator().manual_seed(seed)
    a = (torch.randn(M, K, generator=g)).to(torch.bfloat16).cuda()
    b = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16).cuda()
    out = torch.zeros(M, N, device="cuda")
    args = ds.GemmArgs(mode=ds.EPI_STORE_F32, M=M, N=N, K=K, a=ds.ptr(a), lda=K,
                       b0=ds.ptr(b), ldb=K, b_dtype=ds.W_BF16, out=ds.ptr(out), ldo=N)
    keep = [a, b, out]
    if lora:
        u = torch.randn(M, lora, generator=g).to(torch.bfloat16).cuda()
        z = torch.zeros(N, lora, dtype=torch.bfloat16, device="cuda")
        keep += [u, z]
        args.lora_u0, args.lora_ldu0 = ds.ptr(u), lora
        args.lora_l0, args.lora_ldl0, args.lora_rank0 = ds.ptr(z), lora, lora
    ds.gemm(args)
    torch.cuda.synchronize()
    return out.clone(), keep


@pytest.mark.parametrize("name,mode,M,N,K,int8,extra", CASES, ids=[c[0] for c in CASES])
def test_pair_tiles_match_one_cta_tiles(name, mode, M, N, K, int8, extra):
    seed = 1000 + M + N
    if mode == ds.EPI_STORE_F32:
        got, _k1 = store_f32_case(M, N, K, seed, 0)
        ref, _k2 = store_f32_case(M, N, K, seed, 64)
        assert torch.equal(got.view(torch.int32), ref.view(torch.int32))
        return
    pair = Case(mode, M, N, K, int8, seed, **extra)
    one = Case(mode, M, N, K, int8, seed, lora=64, **extra)
    assert pair.pair and not one.pair
    # the same draws up to the adapter; its L factor zeroed
    z = torch.zeros(N, 64, dtype=torch.bfloat16, device="cuda")
    one.keep.append(z)
    one.args.lora_l0 = ds.ptr(z)
    got, ref = pair.run(), one.run()
    for k in ref:
        a, b = ref[k], got[k]
        a = a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32)
        b = b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32)
        assert torch.equal(a, b), f"{name}: {k} differs"
