"""The persistent attention's work split on the GPU: cutting the last wave's
units into key ranges handed from CTA to CTA must not change a bit.

Each case caps the CTA count so that, at sizes that run in milliseconds, the
remainder units are cut into chains of several ranges (ranges aligned to the
units and ranges that straddle two of them; in the extended split, ranges
longer than a unit, one of them holding a whole unit between two pieces),
including a ragged last key tile and peaked softmax rows whose reference max
moves across a hand-off.
The split result is compared bit for bit with the unsplit launch (one whole
unit per CTA turn), whose agreement with the float64 oracle is checked in
test_gpu_kernels.py, and once more here against the oracle directly."""

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


def inputs(Tq, T, H, hd, seed, sharp):
    g = torch.Generator().manual_seed(seed)
    D = H * hd
    q = (torch.randn(Tq, D, generator=g) * sharp).to(torch.bfloat16)
    k = torch.randn(T, D, generator=g).to(torch.bfloat16)
    v = torch.randn(T, D, generator=g).to(torch.bfloat16)
    ldvt = (T + 127) // 128 * 128
    vt = torch.zeros(D, ldvt, dtype=torch.bfloat16, device="cuda")
    vt[:, :T] = v.cuda().T
    return q, k, v, q.cuda(), k.cuda(), vt, ldvt


def sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


# (Tq, T, heads, head_dim, CTA cap (0: one per SM), softmax sharpness)
CASES = [
    (2048, 1000, 3, 128, 7, 1.0),    # ranges straddling units; ragged keys
    (2048, 1000, 3, 128, 7, 6.0),    # peaked rows: the max moves after a hand-off
    (1500, 3000, 4, 64, 9, 1.0),     # ragged queries and keys, d = 64
    (4096, 4096, 2, 128, 10, 1.0),   # four aligned ranges per cut unit
    (512, 1500, 6, 64, 5, 6.0),      # extended split: a CTA's range holds a unit's
    (512, 1500, 6, 128, 5, 1.0),     #   end, a whole unit and another's start
    (256, 2000, 9, 128, 7, 1.0),     # extended split with one whole unit per CTA
    (8192, 8192, 6, 128, 0, 1.0),    # all SMs: one whole unit each + a cut remainder
    (8192, 32768, 24, 128, 0, 1.0),  # the 32k-token slab of the default workload
]


@pytest.mark.parametrize("Tq,T,H,hd,ctas,sharp", CASES)
def test_split_attention_is_bit_identical_to_unsplit(Tq, T, H, hd, ctas, sharp):
    units, n_kv = -(-Tq // 256) * H, -(-T // 128)
    cap = ctas or sms()
    n_cta, n_split, items = ds.attention_schedule(units, n_kv, cap, 160)
    assert n_split > 0, "the case must cut units"
    q, k, v, qd, kd, vt, ldvt = inputs(Tq, T, H, hd, Tq + T + H, sharp)
    D = H * hd
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    plain = torch.empty(Tq, D, dtype=torch.bfloat16, device="cuda")
    ds.attention_ex(qd, Tq, D, kd, D, vt, ldvt, T, H, hd, plain, D, max_ctas=ctas,
                    dev_status=st)
    nbytes = ds.attention_split_bytes(hd, 160)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    for _ in range(2):  # the second call reuses the hand-off space as left
        split = torch.full((Tq, D), 7.0, dtype=torch.bfloat16, device="cuda")
        ds.attention_ex(qd, Tq, D, kd, D, vt, ldvt, T, H, hd, split, D, split_ws=ws,
                        split_bytes=nbytes, max_ctas=ctas, dev_status=st)
        torch.cuda.synchronize()
        assert int(st[0].item()) == 0
        assert torch.equal(plain.view(torch.int16), split.view(torch.int16))
        assert int(ws[:1024].count_nonzero().item()) == 0, "hand-off flags left set"
    if Tq * T <= 2048 * 4096:
        ref = ob.mha_attention(q.double().numpy(), k.double().numpy(),
                               v.double().numpy(), H)
        got = split.double().cpu().numpy()
        assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 1e-2


def test_unsplit_cta_cap_does_not_change_the_result():
    # round robin over fewer CTAs runs the same units in a different order
    Tq, T, H, hd = 1000, 700, 3, 64
    q, k, v, qd, kd, vt, ldvt = inputs(Tq, T, H, hd, 5, 2.0)
    D = H * hd
    outs = []
    for ctas in (0, 1, 5):
        o = torch.empty(Tq, D, dtype=torch.bfloat16, device="cuda")
        ds.attention_ex(qd, Tq, D, kd, D, vt, ldvt, T, H, hd, o, D, max_ctas=ctas)
        outs.append(o)
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(outs[0].view(torch.int16), o.view(torch.int16))
