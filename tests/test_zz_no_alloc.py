"""dit_block_forward_static: the block forward that allocates nothing.

Callers that cannot allocate device memory (code running under an allocator
that owns every device byte, or where allocation is not allowed) use this
entry point instead of binding a workspace; the library's fixed device
scratch takes the workspace's place.  Its output must equal the ordinary
entry point's bit for bit (the tolerance the chunk-sweep tests use), on two
calls in a row, since the second call starts from the first call's leftover
scratch contents.  This file is collected last so that a failure here
leaves every other test already run."""

import pytest
import torch

from memory_bounded_video_gb300 import build as dbuild
from memory_bounded_video_gb300 import ditstream as ds
from memory_bounded_video_gb300 import runner, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    dbuild.build()
    return ds.load()


@pytest.mark.parametrize("T,D,H,F,cm,ca,fs", [
    (512, 256, 4, 704, 128, 128, 0),
    (1000, 256, 4, 704, 256, 384, 64),
    (4096, 1024, 16, 2816, 512, 512, 0),
])
def test_static_scratch_forward_equals_workspace_forward(T, D, H, F, cm, ca, fs):
    inp = synth.make_inputs(T, D, H, F, seed=11)
    dev = runner.upload(inp)
    stream = torch.cuda.current_stream()

    stack = runner.DitStack(T, D, H, F, cm, ca, fs)
    x_ref = dev.x.clone()
    stack.forward(x_ref, dev, stream)
    stack.check(stream)

    plan = ds.block_plan(T, D, H, F, cm, ca, fs)  # no workspace bound
    assert plan.workspace_bytes() <= ds.STATIC_SCRATCH_BYTES
    for _ in range(2):
        x = dev.x.clone()
        for b in dev.blocks:
            plan.forward_static(x, b.struct, b.mod, stream)
        torch.cuda.synchronize()
        assert torch.equal(x, x_ref)


def test_static_scratch_rejects_plans_larger_than_the_scratch():
    inp = synth.make_inputs(512, 256, 4, 704, seed=12)
    dev = runner.upload(inp)
    big = ds.block_plan(32768, 3072, 24, 8192, 8192, 8192)
    assert big.workspace_bytes() > ds.STATIC_SCRATCH_BYTES
    with pytest.raises(ds.DitError) as e:
        big.forward_static(dev.x, dev.blocks[0].struct, dev.blocks[0].mod)
    assert e.value.status == ds.ERR_WORKSPACE_TOO_SMALL
