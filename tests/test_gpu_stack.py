"""int8-weight blocks, the fp32 final layer and the 4-block stack.

int8 weights are W = s_row * q ("MiniMax-H3-Comfy-NPU", section 2.2: one
weight_scale per output row); the oracle dequantises them in float64.  The
parity cases use per-row scales 0.02/127 * U(0.5, 1.5) so that a row/column
mix-up of the scales shows."""

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


def weights64(bw):
    if bw.int8:
        return ob.DitWeights(**{k: ob.dequant_int8(v.numpy(), bw.scales[k].numpy())
                                for k, v in bw.named().items()})
    return ob.DitWeights(**{k: v.double().numpy() for k, v in bw.named().items()})


def final64(inp):
    if inp.wf_scale is not None:
        return ob.dequant_int8(inp.wf.numpy(), inp.wf_scale.numpy())
    return inp.wf.double().numpy()


def compare(got, ref, x_in):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    mx = np.abs(got - ref).max()
    br = np.linalg.norm(got - ref) / max(np.linalg.norm(ref - x_in), 1e-30)
    return rel, mx, br


def run_stack(inp, cm, ca, fs=0):
    T, D = inp.x.shape
    dev = runner.upload(inp)
    stack = runner.DitStack(T, D, inp.meta["heads"], inp.meta["F"], cm, ca, fs)
    x = dev.x.clone()
    out = stack.forward(x, dev)
    stack.check()
    return x, out


def test_int8_block_matches_oracle_and_is_chunk_invariant():
    inp = synth.make_inputs(1000, 256, 4, 704, seed=6, int8=True, jitter=True)
    outs = [run_stack(inp, cm, ca, fs)[0]
            for cm, ca, fs in [(0, 0, 0), (128, 256, 64), (384, 128, 0)]]
    for x in outs[1:]:
        assert torch.equal(x, outs[0])
    x_in = inp.x.double().numpy()
    ref = ob.dit_block(x_in, weights64(inp.blocks[0]), inp.mods[0].double().numpy(), 4)
    rel, mx, br = compare(outs[0].cpu().numpy(), ref, x_in)
    assert rel <= REL_L2 and mx <= MAX_ABS and br <= BRANCH_REL_L2, (rel, mx, br)


@pytest.mark.parametrize("int8", [False, True])
def test_final_layer_matches_oracle(int8):
    T, D = 1000, 256
    inp = synth.make_inputs(T, D, 4, 704, seed=7, int8=int8, final=True, jitter=True)
    dev = runner.upload(inp)
    plan = ds.block_plan(T, D, 4, 704, 0, 0)
    out = torch.full((T, 64), float("nan"), device="cuda")
    plan.final_forward(dev.x, dev.wf, dev.wf_scale, dev.mod_f, out)
    torch.cuda.synchronize()
    ref = ob.final_layer(inp.x.double().numpy(), final64(inp), inp.mod_f.double().numpy())
    got = out.cpu().double().numpy()
    # fp32-level arithmetic over D terms (an fp32 FMA loop and the split
    # tf32 tensor-core products with fp32 partial sums both land near 2e-6)
    assert np.abs(got - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())


def test_final_layer_rows_are_independent_of_T():
    T, D = 1000, 256
    inp = synth.make_inputs(T, D, 4, 704, seed=8, final=True)
    dev = runner.upload(inp)
    outs = []
    for t in (T, 333):
        plan = ds.block_plan(t, D, 4, 704, 0, 0)
        out = torch.empty(t, 64, device="cuda")
        plan.final_forward(dev.x, dev.wf, None, dev.mod_f, out)
        outs.append(out)
    torch.cuda.synchronize()
    assert torch.equal(outs[0][:333], outs[1])


def test_stack_of_four_int8_blocks_and_final_layer_full_oracle():
    # the 32k workload's model (D=3072, 24x128 heads, FFN 8192, 4 int8
    # blocks + final layer) at a length the float64 oracle finishes quickly
    T = 640
    inp = synth.make_inputs(T, 3072, 24, 8192, seed=9, blocks=4, int8=True,
                            final=True, jitter=True)
    x, out = run_stack(inp, 256, 384)
    xr = inp.x.double().numpy()
    for bw, mod in zip(inp.blocks, inp.mods):
        xr = ob.dit_block(xr, weights64(bw), mod.double().numpy(), 24)
    yr = ob.final_layer(xr, final64(inp), inp.mod_f.double().numpy())
    rel, mx, _ = compare(x.cpu().numpy(), xr, inp.x.double().numpy())
    assert rel <= REL_L2 and mx <= MAX_ABS, (rel, mx)
    got = out.cpu().double().numpy()
    rel_y = np.linalg.norm(got - yr) / np.linalg.norm(yr)
    assert rel_y <= REL_L2, rel_y


def sampled_rows(T, n, seed=0):
    rng = np.random.default_rng(seed)
    rows = set(range(64)) | set(range(T - 64, T))
    rows |= set(rng.choice(T, size=n, replace=False).tolist())
    return np.array(sorted(rows))


def test_headline_stack_T32768_full_size():
    """The 4-block int8 + final workload at its full size, in the launch
    configuration the benchmark times (chunks 8192): block one against the
    oracle on sampled rows (K/V of all tokens computed by the oracle), and
    the whole stack bit-identical across chunk settings."""
    name = "dit4_int8_final_T32768_D3072"
    cfg = synth.WORKLOADS[name]
    inp = synth.make_workload(name, seed=0)
    T, D = inp.x.shape
    dev = runner.upload(inp)
    stream = torch.cuda.current_stream()

    # block one alone vs the oracle on sampled rows
    stack = runner.DitStack(T, D, 24, 8192, cfg["mlp_chunk"], cfg["attn_chunk"])
    x1 = dev.x.clone()
    stack.plan.forward(x1, dev.blocks[0].struct, dev.blocks[0].mod, stream)
    stack.check()
    rows = sampled_rows(T, 192)
    ref, _ = ob.dit_block_rows(inp.x.double().numpy(), weights64(inp.blocks[0]),
                               inp.mods[0].double().numpy(), 24, rows)
    rel, mx, br = compare(x1.cpu().numpy()[rows], ref, inp.x.double().numpy()[rows])
    assert rel <= REL_L2 and mx <= MAX_ABS and br <= BRANCH_REL_L2, (rel, mx, br)
    del x1

    # the stack: bit-identical for every chunk setting tried
    results = []
    for cm, ca in [(8192, 8192), (2048, 4096), (0, 0)]:
        st = runner.DitStack(T, D, 24, 8192, cm, ca)
        x = dev.x.clone()
        out = st.forward(x, dev, stream)
        st.check()
        assert torch.isfinite(out).all()
        results.append((x, out))
        del st
    for x, out in results[1:]:
        assert torch.equal(x, results[0][0])
        assert torch.equal(out, results[0][1])


def test_headline_stack_chunk_sweep_T32768_is_bit_identical():
    """The 32k int8 stack's chunk sweep: mlp and attention chunks of every
    power of two from 256 to 32768 tokens (and two unequal pairs) give the
    same residual and final-layer bits."""
    name = "dit4_int8_final_T32768_D3072"
    inp = synth.make_workload(name, seed=1)
    T, D = inp.x.shape
    dev = runner.upload(inp)
    stream = torch.cuda.current_stream()
    ref = None
    for cm, ca in [(c, c) for c in (256, 512, 1024, 2048, 4096, 8192, 16384, 32768)] + \
                  [(256, 32768), (32768, 512)]:
        st = runner.DitStack(T, D, 24, 8192, cm, ca)
        x = dev.x.clone()
        out = st.forward(x, dev, stream)
        st.check()
        if ref is None:
            assert torch.isfinite(out).all()
            ref = (x, out)
        else:
            assert torch.equal(x, ref[0]), (cm, ca)
            assert torch.equal(out, ref[1]), (cm, ca)
        del st


# ---------------------------------------------------------------- weight scratch

def test_int8_to_bf16_is_exact():
    q = torch.arange(-128, 128, dtype=torch.int16).to(torch.int8).repeat(64)
    out = torch.empty(q.numel(), dtype=torch.bfloat16, device="cuda")
    ds.int8_to_bf16(q.cuda(), q.numel(), out)
    torch.cuda.synchronize()
    assert torch.equal(out.cpu().float(), q.float())


def run_scratch(inp, cm, ca, fs, scratch, lora=None, rank=0, qk=None):
    T, D = inp.x.shape
    dev = runner.upload(inp)
    stack = runner.DitStack(T, D, inp.meta["heads"], inp.meta["F"], cm, ca, fs,
                            lora_rank=rank, weight_scratch=scratch)
    dl = None if lora is None else [runner.upload_lora(lo, b)
                                    for lo, b in zip(lora, dev.blocks)]
    x = dev.x.clone()
    out = stack.forward(x, dev, lora=dl, qk=None if qk is None else runner.upload_qk(qk))
    stack.check()
    return x, out


@pytest.mark.parametrize("cm,ca,fs", [(0, 0, 0), (128, 256, 64), (384, 128, 0)])
def test_weight_scratch_gives_the_same_bits(cm, ca, fs):
    # int8 weights expanded to bf16 ahead of the GEMMs: same MMA operands,
    # order and epilogue scale as the in-kernel conversion
    inp = synth.make_inputs(1000, 256, 4, 704, seed=31, int8=True, jitter=True, blocks=2,
                            final=True)
    x0, o0 = run_scratch(inp, cm, ca, fs, False)
    x1, o1 = run_scratch(inp, cm, ca, fs, True)
    assert torch.equal(x0, x1) and torch.equal(o0, o1)


def test_weight_scratch_with_lora_and_qk_gives_the_same_bits():
    inp = synth.make_inputs(768, 1024, 8, 1024, seed=32, int8=True, jitter=True)
    lora = [synth.make_lora(1024, 1024, 64, seed=3)]
    qk = synth.make_qk(768, 128, seed=4, angles="axial")
    x0, _ = run_scratch(inp, 256, 256, 512, False, lora, 64, qk)
    x1, _ = run_scratch(inp, 256, 256, 512, True, lora, 64, qk)
    assert torch.equal(x0, x1)


def test_weight_scratch_full_size_block_T4096_D3072():
    inp = synth.make_inputs(4096, 3072, 24, 8192, seed=33, int8=True, jitter=True)
    x0, _ = run_scratch(inp, 2048, 2048, 0, False)
    x1, _ = run_scratch(inp, 2048, 2048, 0, True)
    assert torch.equal(x0, x1)


def test_headline_stack_chunk_sweep_is_bit_identical():
    """The 4-block int8 + final workload at full size (T = 32768) for query
    slabs and MLP chunks from 256 to 32768 tokens: every setting gives the
    same bits as the unchunked run."""
    name = "dit4_int8_final_T32768_D3072"
    inp = synth.make_workload(name, seed=1)
    T, D = inp.x.shape
    dev = runner.upload(inp)
    stream = torch.cuda.current_stream()
    ref = None
    settings = [(c, c) for c in (256, 512, 1024, 2048, 4096, 8192, 16384, 32768)]
    settings += [(256, 32768), (32768, 256), (1024, 8192), (0, 0)]
    for cm, ca in settings:
        st = runner.DitStack(T, D, 24, 8192, cm, ca, weight_scratch=(cm == ca))
        x = dev.x.clone()
        out = st.forward(x, dev, stream)
        st.check()
        if ref is None:
            ref = (x, out)
        else:
            assert torch.equal(x, ref[0]), (cm, ca)
            assert torch.equal(out, ref[1]), (cm, ca)
        del st


@pytest.mark.parametrize("final", [True, False])
def test_forward_host_pipeline_matches_per_batch_forwards(final):
    # three different token batches from pinned host memory through the
    # double-buffered host path, against one device forward per batch
    T, D, H, F = 1000, 256, 4, 704
    inp = synth.make_inputs(T, D, H, F, seed=21, blocks=2, int8=True, final=final,
                            jitter=True)
    dev = runner.upload(inp)
    g = torch.Generator().manual_seed(5)
    xs = [torch.randn(T, D, generator=g).pin_memory() for _ in range(3)]
    cols = 64 if final else D
    outs = [torch.full((T, cols), float("nan")).pin_memory() for _ in range(3)]
    stack = runner.DitStack(T, D, H, F, 256, 384, 256)
    for _ in range(2):  # the second call reuses the stack's buffers
        stack.forward_host(xs, dev, outs)
        torch.cuda.synchronize()
        stack.check()
        for xh, oh in zip(xs, outs):
            x = xh.cuda()
            ref = stack.forward(x, dev)
            stack.check()
            ref = (ref if final else x).cpu()
            assert torch.equal(oh.view(torch.int32), ref.view(torch.int32))
        for o in outs:
            o.fill_(float("nan"))


def test_final_layer_rows_with_large_offsets():
    # rows with a large common offset and rows of very different spread: the
    # head's statistics come from sums of the row shifted by its first
    # element, which must hold its accuracy when the offset dwarfs the spread
    T, D = 777, 1024
    g = torch.Generator().manual_seed(11)
    x = torch.randn(T, D, generator=g)
    x *= torch.exp(torch.randn(T, 1, generator=g))          # spread 0.1 .. 10
    x += torch.randn(T, 1, generator=g) * 100.0             # offsets ~ 100
    x[5] += 1.0e4
    wf = (torch.randn(64, D, generator=g) * 0.02).float()
    mod = (torch.randn(2, D, generator=g) * 0.1).float()
    plan = ds.block_plan(T, D, 8, 704, 0, 0)
    out = torch.full((T, 64), float("nan"), device="cuda")
    plan.final_forward(x.cuda(), wf.cuda(), None, mod.cuda(), out)
    torch.cuda.synchronize()
    ref = ob.final_layer(x.double().numpy(), wf.double().numpy(), mod.double().numpy())
    got = out.cpu().double().numpy()
    # the same fp32 bound as the plain rows (after LN every row's output is
    # of the same size, whatever its offset and spread)
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max()


@pytest.mark.parametrize("int8", [False, True])
def test_final_layer_several_tiles_per_cta(int8):
    # more 128-row tiles than multiprocessors (every CTA of the persistent
    # grid runs two or three tiles, the last one ragged), against the full
    # oracle: the tile loop's hand-over of the statistics and the
    # tensor-memory partial-sum buffers from one tile to the next
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T, D = 128 * (2 * sms + 5) + 77, 512
    inp = synth.make_inputs(T, D, 4, 704, seed=21, int8=int8, final=True, jitter=True,
                            blocks=0)
    dev = runner.upload(inp)
    plan = ds.block_plan(T, D, 4, 704, 0, 0)
    out = torch.full((T, 64), float("nan"), device="cuda")
    plan.final_forward(dev.x, dev.wf, dev.wf_scale, dev.mod_f, out)
    torch.cuda.synchronize()
    ref = ob.final_layer(inp.x.double().numpy(), final64(inp), inp.mod_f.double().numpy())
    got = out.cpu().double().numpy()
    assert np.isfinite(got).all()
    assert np.abs(got - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())
