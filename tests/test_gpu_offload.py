"""K/V offload below the K/V floor.

"LayerStream: H3 Chunking" ("Where people get burned"): K and V of the whole
sequence stay resident, so activation memory has a floor of 4*T*D bytes that
chunking cannot go under; only K/V offload can.  Here K and V^T of all tokens
live in pinned host memory, pass two streams them back in key blocks, and
the attention carries its softmax state between blocks: the output bits must
equal the resident schedule's, and the device workspace must not grow with T.
"""

import numpy as np
import pytest
import torch

from memory_bounded_video_gb300 import build as dbuild
from memory_bounded_video_gb300 import ditstream as ds
from memory_bounded_video_gb300 import runner, synth
from oracle import block as ob

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    dbuild.build()
    return ds.load()


@pytest.mark.parametrize("Tq,T,H,hd,kb,sharp", [
    (1000, 3000, 4, 128, 1024, 4.0),   # ragged T: last block 952 keys
    (777, 2500, 8, 64, 512, 4.0),
    (256, 4096, 2, 128, 128, 8.0),     # one tile per block
    (300, 1000, 4, 64, 2048, 1.0),     # one block (first = last)
])
def test_attention_over_key_blocks_equals_one_launch(Tq, T, H, hd, kb, sharp):
    g = torch.Generator().manual_seed(Tq + T)
    D = H * hd
    q = (torch.randn(Tq, D, generator=g) * sharp).to(torch.bfloat16).cuda()
    k = torch.randn(T, D, generator=g).to(torch.bfloat16).cuda()
    ldvt = (T + 127) // 128 * 128
    vt = torch.randn(D, ldvt, generator=g).to(torch.bfloat16).cuda()
    ref = torch.empty(Tq, D, dtype=torch.bfloat16, device="cuda")
    ds.attention(q, Tq, D, k, D, vt, ldvt, T, H, hd, ref, D)
    o = torch.full((Tq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    o_st = torch.empty(Tq, D, device="cuda")
    m_st = torch.empty(Tq, H, device="cuda")
    l_st = torch.empty(Tq, H, device="cuda")
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    nb = (T + kb - 1) // kb
    for b in range(nb):
        k0 = b * kb
        n = min(kb, T - k0)
        vt_blk = vt[:, k0:k0 + kb].contiguous() if n == kb else \
            torch.nn.functional.pad(vt[:, k0:k0 + n], (0, (n + 7) // 8 * 8 - n)).contiguous()
        ds.attention_part(q, Tq, D, k[k0:], D, vt_blk, vt_blk.shape[1], n, H, hd, o, D,
                          o_st, m_st, l_st, D, b == 0, b == nb - 1, st)
    torch.cuda.synchronize()
    assert int(st[0]) == 0
    assert torch.equal(o.view(torch.int16), ref.view(torch.int16))


def run(inp, cm, ca, fs=0, kv_offload=0, lora=None, rank=0, qk=None, scratch=False):
    T, D = inp.x.shape
    dev = runner.upload(inp)
    stack = runner.DitStack(T, D, inp.meta["heads"], inp.meta["F"], cm, ca, fs,
                            lora_rank=rank, kv_offload=kv_offload, weight_scratch=scratch)
    dl = None if lora is None else [runner.upload_lora(lo, b) for lo, b in zip(lora, dev.blocks)]
    x = dev.x.clone()
    out = stack.forward(x, dev, lora=dl, qk=None if qk is None else runner.upload_qk(qk))
    stack.check()
    return x, out, stack


@pytest.mark.parametrize("cm,ca,kvb", [(128, 384, 256), (0, 0, 384), (256, 128, 1024)])
def test_offloaded_block_equals_resident(cm, ca, kvb):
    inp = synth.make_inputs(1000, 256, 4, 704, seed=41)
    x0, _, _ = run(inp, cm, ca)
    x1, _, _ = run(inp, cm, ca, kv_offload=kvb)
    assert torch.equal(x0, x1)


def test_offloaded_int8_stack_with_lora_qk_equals_resident():
    inp = synth.make_inputs(768, 1024, 8, 1024, seed=42, int8=True, jitter=True, blocks=2,
                            final=True)
    lora = [synth.make_lora(1024, 1024, 32, seed=i) for i in range(2)]
    qk = synth.make_qk(768, 128, seed=5, angles="axial")
    x0, o0, _ = run(inp, 256, 256, 512, 0, lora, 32, qk, True)
    x1, o1, _ = run(inp, 256, 256, 512, 256, lora, 32, qk, True)
    assert torch.equal(x0, x1) and torch.equal(o0, o1)


def test_offload_T16384_D3072_matches_oracle_rows_and_resident():
    inp = synth.make_workload("dit_T16384_D3072", seed=4)
    T = inp.x.shape[0]
    x0, _, _ = run(inp, 8192, 4096)
    # small chunks and key blocks: the whole workspace is below what the
    # resident K and V alone take (and the bits do not depend on the chunks)
    x1, _, st = run(inp, 2048, 4096, 2048, kv_offload=2048)
    assert torch.equal(x0, x1)
    assert st.plan.workspace_bytes() < 4 * T * 3072
    rows = np.array([0, 1, 4095, 4096, 9999, T - 1])
    w = ob.DitWeights(**{k: v.double().numpy() for k, v in inp.blocks[0].named().items()})
    ref, _ = ob.dit_block_rows(inp.x.double().numpy(), w, inp.mods[0].double().numpy(), 24,
                               rows)
    got = x1.cpu().double().numpy()[rows]
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) <= 1e-2


def test_offloaded_forward_allocates_no_device_memory():
    inp = synth.make_inputs(2048, 1024, 8, 2816, seed=43)
    T, D = inp.x.shape
    dev = runner.upload(inp)
    stack = runner.DitStack(T, D, 8, 2816, 512, 512, 0, kv_offload=512)
    x = dev.x.clone()
    stack.forward(x, dev)  # loads every kernel's module
    stack.check()
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    x2 = dev.x.clone()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    stack.forward(x2, dev)
    stack.check()
    assert torch.cuda.memory_allocated() == alloc0 + x2.numel() * 4
    assert torch.cuda.mem_get_info()[0] == free1
    assert torch.equal(x, x2)
