"""dit_block_forward_static: the block forward that allocates nothing.

Callers that cannot allocate device memory (code running under an allocator
that owns every device byte, or where allocation is not allowed) use this
entry point instead of binding a workspace; the library's fixed device
scratch takes the workspace's place.  Its output must equal the ordinary
entry point's bit for bit (the tolerance the chunk-sweep tests use), on two
calls in a row, since the second call starts from the first call's leftover
scratch contents; after the first call on the device (which may make the
driver reserve the scratch array) no call may change the device's free
memory; and the status word must read clean after every call.  This file is
collected last so that a failure here leaves every other test already
run."""

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


def _static_stack(plan, x, dev, stream):
    for b in dev.blocks:
        plan.forward_static(x, b.struct, b.mod, stream)


@pytest.mark.parametrize("T,D,H,F,cm,ca,fs,int8", [
    (512, 256, 4, 704, 128, 128, 0, False),
    (1000, 256, 4, 704, 256, 384, 64, False),
    (4096, 1024, 16, 2816, 512, 512, 0, False),
    (1000, 1024, 16, 2816, 256, 512, 1024, True),
])
def test_static_scratch_forward_equals_workspace_forward(T, D, H, F, cm, ca, fs, int8):
    inp = synth.make_inputs(T, D, H, F, seed=11, int8=int8, jitter=int8)
    dev = runner.upload(inp)
    stream = torch.cuda.current_stream()

    stack = runner.DitStack(T, D, H, F, cm, ca, fs)
    x_ref = dev.x.clone()
    stack.forward(x_ref, dev, stream)
    stack.check(stream)

    plan = ds.block_plan(T, D, H, F, cm, ca, fs)  # no workspace bound
    assert plan.workspace_bytes() <= ds.STATIC_SCRATCH_BYTES
    x = torch.empty_like(dev.x)
    free = []
    for _ in range(3):
        x.copy_(dev.x)
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
        _static_stack(plan, x, dev, stream)
        assert plan.sync_status(stream) == ds.OK
        assert torch.equal(x, x_ref)
    # the first call may have made the driver reserve the scratch; from
    # then on nothing on the device is allocated
    torch.cuda.synchronize()
    free.append(torch.cuda.mem_get_info()[0])
    assert free[1] == free[2] == free[3]


def test_static_forward_leaves_a_bound_workspace_in_use():
    # a plan with its own workspace: a static call in between ordinary
    # calls neither uses nor disturbs that workspace
    T, D, H, F = 1000, 256, 4, 704
    inp = synth.make_inputs(T, D, H, F, seed=13)
    dev = runner.upload(inp)
    stream = torch.cuda.current_stream()
    stack = runner.DitStack(T, D, H, F, 256, 256)
    x_ref = dev.x.clone()
    stack.forward(x_ref, dev, stream)
    stack.check(stream)

    x = dev.x.clone()
    _static_stack(stack.plan, x, dev, stream)
    assert stack.plan.sync_status(stream) == ds.OK
    assert torch.equal(x, x_ref)
    x2 = dev.x.clone()
    stack.forward(x2, dev, stream)
    stack.check(stream)
    assert torch.equal(x2, x_ref)


def test_static_scratch_rejects_plans_larger_than_the_scratch():
    inp = synth.make_inputs(512, 256, 4, 704, seed=12)
    dev = runner.upload(inp)
    big = ds.block_plan(32768, 3072, 24, 8192, 8192, 8192)
    assert big.workspace_bytes() > ds.STATIC_SCRATCH_BYTES
    with pytest.raises(ds.DitError) as e:
        big.forward_static(dev.x, dev.blocks[0].struct, dev.blocks[0].mod)
    assert e.value.status == ds.ERR_WORKSPACE_TOO_SMALL
