"""Long video (T = 65536) with the FFN sliced 4 x 2048, and the memory bound.

"LayerStream: H3 Chunking" ("Where people get burned"): K and V of the whole
sequence stay resident, so the activation floor grows with T; everything else
is bounded by the chunk sizes.  The library allocates no device memory: the
caller's workspace is all it uses."""

import ctypes

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


def weights64(bw):
    return ob.DitWeights(**{k: v.double().numpy() for k, v in bw.named().items()})


def mem_free():
    free, _ = torch.cuda.mem_get_info()
    return free


def test_long_video_T65536_ffn_sliced():
    name = "dit_T65536_D3072"
    cfg = synth.WORKLOADS[name]
    inp = synth.make_workload(name, seed=0)
    T, D = inp.x.shape
    dev = runner.upload(inp)
    stream = torch.cuda.current_stream()

    stack = runner.DitStack(T, D, 24, 8192, cfg["mlp_chunk"], cfg["attn_chunk"],
                            cfg["ffn_slice"])
    assert stack.plan.info()["ffn_slice"] == 2048
    x = dev.x.clone()
    stack.forward(x, dev, stream)  # also loads every kernel's module
    stack.check(stream)
    # a second forward allocates nothing, neither through torch nor by the
    # library itself (device free memory unchanged)
    x_again = dev.x.clone()
    torch.cuda.synchronize()
    free0 = mem_free()
    alloc0 = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    stack.forward(x_again, dev, stream)
    stack.check(stream)
    assert torch.cuda.max_memory_allocated() == alloc0
    assert mem_free() == free0
    assert torch.equal(x_again, x)
    del x_again

    # sampled rows against the oracle (K/V of all 65536 tokens in float64)
    rng = np.random.default_rng(5)
    rows = np.array(sorted(set(range(32)) | set(range(T - 32, T))
                           | set(rng.choice(T, 96, replace=False).tolist())))
    ref, _ = ob.dit_block_rows(inp.x.double().numpy(), weights64(inp.blocks[0]),
                               inp.mods[0].double().numpy(), 24, rows)
    got = x.cpu().double().numpy()[rows]
    x_in = inp.x.double().numpy()[rows]
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= 1e-2 and np.abs(got - ref).max() <= 5e-2
    br = np.linalg.norm(got - ref) / np.linalg.norm(ref - x_in)
    assert br <= 2e-2, br

    # the FFN slicing and the chunk sizes do not change a bit
    for cm, ca, fs in [(8192, 4096, 0), (4096, 8192, 4096)]:
        st = runner.DitStack(T, D, 24, 8192, cm, ca, fs)
        x2 = dev.x.clone()
        st.forward(x2, dev, stream)
        st.check(stream)
        assert torch.equal(x2, x), (cm, ca, fs)
        del st, x2


def test_activation_beyond_kv_floor_does_not_grow_with_T():
    D, F, C, FS = 3072, 8192, 4096, 2048
    rest = []
    for T in (8192, 16384, 32768, 65536):
        p = ds.block_plan(T, D, 24, F, C, C, FS)
        rest.append(p.workspace_bytes() - 4 * T * D)
    assert max(rest) - min(rest) <= 4096
    # and it is the chunk-sized part: about 88 MiB at 4096-token chunks
    assert rest[0] < 100 * 2**20
