"""Host-side driver of libditstream for PyTorch users.

PyTorch supplies device memory and streams only: this module uploads
weights, allocates the plan's workspace with ``torch.empty`` (so the caching
allocator accounts for it) and calls the C ABI.  Every step of the block runs
in the library's CUDA kernels; nothing here computes.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional

import torch

from . import ditstream
from .synth import DitInputs


@dataclass
class DeviceBlock:
    tensors: dict            # device tensors (kept alive)
    struct: ditstream.BlockWeights
    mod: torch.Tensor        # [6, D] fp32 on device


@dataclass
class DeviceInputs:
    x: torch.Tensor                        # [T, D] fp32 (pristine copy)
    blocks: List[DeviceBlock]
    mod_f: Optional[torch.Tensor] = None
    wf: Optional[torch.Tensor] = None
    wf_scale: Optional[torch.Tensor] = None


def upload(inp: DitInputs, device="cuda") -> DeviceInputs:
    """Copy seeded CPU inputs to the device (weights stay resident)."""
    blocks = []
    for bw, mod in zip(inp.blocks, inp.mods):
        t = {k: v.to(device).contiguous() for k, v in bw.named().items()}
        sc = None
        if bw.scales is not None:
            sc = {k: v.to(device).contiguous() for k, v in bw.scales.items()}
            t.update({k + "_scale": v for k, v in sc.items()})
        st = ditstream.block_weights(t["wqkv"], t["wo"], t["wgate"], t["wup"],
                                     t["wdown"], scales=sc)
        blocks.append(DeviceBlock(t, st, mod.to(device).contiguous()))
    out = DeviceInputs(x=inp.x.to(device).contiguous(), blocks=blocks)
    if inp.mod_f is not None:
        out.mod_f = inp.mod_f.to(device).contiguous()
        out.wf = inp.wf.to(device).contiguous()
        if inp.wf_scale is not None:
            out.wf_scale = inp.wf_scale.to(device).contiguous()
    return out


@dataclass
class DeviceQk:
    tensors: dict            # device tensors (kept alive)
    struct: ditstream.QkArgs


def upload_qk(qk: dict, device="cuda") -> DeviceQk:
    """Copy Q/K transform inputs (``synth.make_qk``) to the device."""
    t = {k: (v.to(device).contiguous() if isinstance(v, torch.Tensor) else None)
         for k, v in qk.items() if k != "eps"}
    st = ditstream.qk_args(t["q_norm"], t["k_norm"], t["cos"], t["sin"],
                           qk.get("eps", 1e-6))
    return DeviceQk(t, st)


@dataclass
class DeviceLora:
    tensors: dict            # device tensors (kept alive)
    struct: ditstream.BlockLora


_LORA_WEIGHT = dict(qkv="wqkv", o="wo", gate="wgate", up="wup", down="wdown")


def upload_lora(lora: dict, block: DeviceBlock, stream=None) -> DeviceLora:
    """Place adapters (``synth.make_lora``) on the device for one block:
    A as given, B prepared by ``dit_lora_prepare`` (alpha folded in and, for
    int8 weights, divided by the adapted weight's row scales)."""
    keep, packed = {}, {}
    for name, (A, B, alpha) in lora.items():
        a = A.to("cuda").contiguous()
        b = B.to("cuda").contiguous()
        rows, rank = b.shape
        bp = torch.empty_like(b)
        scale = block.tensors.get(_LORA_WEIGHT[name] + "_scale")
        ditstream.lora_prepare(b, rows, rank, rank, alpha, scale, bp, rank, stream)
        keep[name] = (a, b, bp)
        packed[name] = (a, bp, rank)
    return DeviceLora(keep, ditstream.block_lora(**packed))


class DitStack:
    """A stack of DiT blocks (one plan, one workspace) plus an optional
    final layer.  ``forward`` updates ``x`` in place and returns the final
    layer's output when there is one."""

    def __init__(self, T, D, heads, F, mlp_chunk, attn_chunk, ffn_slice=0,
                 device="cuda", lora_rank=0, weight_scratch=False, kv_offload=0):
        self.plan = ditstream.block_plan(T, D, heads, F, mlp_chunk, attn_chunk,
                                         ffn_slice)
        if lora_rank:
            self.plan.set_lora_rank(lora_rank)
        self.kv_host = None
        if kv_offload:  # K/V of all tokens in pinned host memory
            self.plan.set_kv_offload(kv_offload)
            self.kv_host = torch.empty(self.plan.kv_host_bytes(), dtype=torch.uint8,
                                       pin_memory=True)
            self.plan.bind_kv_host(self.kv_host)
        self.weight_scratch = None
        if weight_scratch:  # int8 weights expanded to bf16 ahead of the GEMMs
            self.weight_scratch = torch.empty(self.plan.weight_scratch_bytes(),
                                              dtype=torch.uint8, device=device)
            self.plan.bind_weight_scratch(self.weight_scratch)
        self.T, self.D = T, D
        self.workspace = torch.empty(self.plan.workspace_bytes(),
                                     dtype=torch.uint8, device=device)
        self.plan.bind_workspace(self.workspace)
        self.device = device

    def forward(self, x: torch.Tensor, dev: DeviceInputs, stream=None,
                out: Optional[torch.Tensor] = None,
                qk: Optional[DeviceQk] = None,
                lora: Optional[List[DeviceLora]] = None):
        """``lora``: one DeviceLora (or None) per block."""
        if stream is None:
            stream = torch.cuda.current_stream(x.device)
        for i, b in enumerate(dev.blocks):
            ad = None if lora is None else lora[i]
            self.plan.forward(x, b.struct, b.mod, stream,
                              qk=None if qk is None else qk.struct,
                              lora=None if ad is None else ad.struct)
        if dev.wf is not None:
            if out is None:
                out = torch.empty(self.T, 64, dtype=torch.float32,
                                  device=x.device)
            self.plan.final_forward(x, dev.wf, dev.wf_scale, dev.mod_f, out,
                                    stream)
            return out
        return None

    def forward_host(self, x_host: List[torch.Tensor], dev: DeviceInputs,
                     out_host: List[torch.Tensor], stream=None,
                     qk: Optional[DeviceQk] = None,
                     lora: Optional[List[DeviceLora]] = None):
        """Run the stack over a sequence of token batches held in pinned
        host memory, writing each batch's result (the final layer's output,
        or x without a final layer) into the matching pinned ``out_host``
        tensor.  Two device buffers alternate: while batch i computes on
        ``stream``, a copy stream brings batch i + 1 in and takes batch i - 1's
        result out, so the host link overlaps the kernels.  Asynchronous:
        ``stream`` has waited for every copy when this returns, so
        synchronising it makes the results valid."""
        if stream is None:
            stream = torch.cuda.current_stream()
        n = len(x_host)
        if len(out_host) != n:
            raise ValueError("one output buffer per input batch")
        if n == 0:
            return
        final = dev.wf is not None
        if getattr(self, "_io", None) is None:
            xs = [torch.empty(self.T, self.D, dtype=torch.float32, device=self.device)
                  for _ in range(2)]
            outs = ([torch.empty(self.T, 64, dtype=torch.float32, device=self.device)
                     for _ in range(2)] if final else [None, None])
            self._io = (torch.cuda.Stream(device=self.device), xs, outs)
        copy, xs, outs = self._io
        if final and outs[0] is None:
            raise ValueError("forward_host: the stack was first run without a final layer")
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        copy.wait_stream(stream)  # the buffers' previous users are done

        def bring_in(i):
            with torch.cuda.stream(copy):
                xs[i % 2].copy_(x_host[i], non_blocking=True)
                ev_in[i % 2].record(copy)

        bring_in(0)
        for i in range(n):
            b = i % 2
            if i + 1 < n:  # same stream as batch i - 1's copy-out: ordered after it
                bring_in(i + 1)
            stream.wait_event(ev_in[b])
            res = self.forward(xs[b], dev, stream, out=outs[b], qk=qk, lora=lora)
            ev_done[b].record(stream)
            copy.wait_event(ev_done[b])
            with torch.cuda.stream(copy):
                out_host[i].copy_(res if res is not None else xs[b], non_blocking=True)
        stream.wait_stream(copy)

    def check(self, stream=None):
        """Synchronise and raise if a kernel recorded a device-side error."""
        if stream is None:
            stream = torch.cuda.current_stream()
        s = self.plan.sync_status(stream)
        if s != ditstream.OK:
            raise ditstream.DitError(s, "dit_block_sync_status")
