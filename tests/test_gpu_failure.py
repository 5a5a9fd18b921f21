"""Failure detection on the GPU without a fault: a bounded device wait that
runs out is reported as DIT_ERR_TIMEOUT and the context stays usable.

The GEMM's test hook makes CTA 0's producer withhold one copy (a transaction
that nothing completes).  The MMA warp's wait gives up after its limit, the
kernel records the status, drains what it issued, frees its tensor memory and
returns.  No trap, no bad address, no endless loop."""

import numpy as np
import pytest
import torch

from memory_bounded_video_gb300 import build as dbuild
from memory_bounded_video_gb300 import ditstream as ds

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    dbuild.build()
    return ds.load()


def gemm_f32(a, b, out, flags=0, status=None, scale=None):
    M, K = a.shape
    N = b.shape[0]
    args = ds.GemmArgs(mode=ds.EPI_STORE_F32, M=M, N=N, K=K, a=ds.ptr(a), lda=K,
                       b0=ds.ptr(b), ldb=K,
                       b_dtype=ds.W_INT8 if scale is not None else ds.W_BF16,
                       b0_scale=ds.ptr(scale), out=ds.ptr(out), ldo=N, flags=flags)
    ds.gemm(args, status)


# bf16: the cluster pair's copies complete on the leading CTA's barrier; int8:
# the pair whose converter warps fill the B operand (CTA 0's A copy withheld,
# so its stage never completes while the converters and the peer go on)
@pytest.mark.parametrize("int8", [False, True], ids=["bf16_pair", "int8_pair"])
def test_withheld_copy_times_out_and_context_survives(int8):
    g = torch.Generator().manual_seed(31)
    M, N, K = 256, 256, 256
    a = torch.randn(M, K, generator=g).to(torch.bfloat16).cuda()
    if int8:
        q = torch.randint(-127, 128, (N, K), generator=g, dtype=torch.int16).to(torch.int8)
        s = 0.02 / 127 * (0.5 + torch.rand(N, generator=g))
        b, scale = q.cuda(), s.float().cuda()
        w = q.double().numpy() * s.double().numpy()[:, None]
    else:
        b = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16).cuda()
        scale, w = None, None
    out = torch.zeros(M, N, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    gemm_f32(a, b, out, flags=ds.GEMM_FLAG_INJECT_STALL, status=status, scale=scale)
    torch.cuda.synchronize()  # returns after the bounded waits run out
    assert int(status[0].item()) == ds.ERR_TIMEOUT
    # the context is intact: the same GEMM without the hook is correct
    status.zero_()
    gemm_f32(a, b, out, status=status, scale=scale)
    torch.cuda.synchronize()
    assert int(status[0].item()) == 0
    if w is None:
        w = b.double().cpu().numpy()
    ref = a.double().cpu().numpy() @ w.T
    assert np.abs(out.cpu().numpy() - ref).max() < 1e-3


def test_unknown_flags_are_rejected_on_the_host():
    a = torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(128, 64, device="cuda")
    with pytest.raises(ds.DitError) as e:
        gemm_f32(a, b, out, flags=4)
    assert e.value.status == ds.ERR_INVALID_ARG
