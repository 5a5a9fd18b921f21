"""Seeded synthetic inputs for the DiT block (shared by tests, bench and oracle).

This module draws random numbers and nothing else: it holds none of the
block's arithmetic, imports neither the CUDA library nor the oracle, and is
the only code that both sides use.  Every tensor is drawn on the CPU from a
``torch.Generator`` seeded with ``seed`` in a fixed order, so the oracle and
the GPU path see identical bits on any machine.

Distributions (the video-DiT workloads of "LayerStream: H3 Chunking" and
"ComfyUI-StaticPipeline" have no public weights; these synthetic draws stand
in for them):

* residual stream ``x``       : N(0, 1) fp32, [T, D], token order frames x
  patches row-major (irrelevant without positional terms);
* linear weights             : N(0, 0.02) fp32 rounded to bf16 (RNE), or
  int8 uniform on [-127, 127] with one fp32 scale per output row
  (0.02/127, optionally times U(0.5, 1.5) so row/column mix-ups show);
* ``modulation`` [6, D] fp32 : shift/scale rows N(0, 0.1), gate rows U(0, 1);
* final layer                : ``mod_f`` [2, D] N(0, 0.1); ``W_f`` [64, D]
  N(0, 0.02) fp32 (or int8 like the block weights);
* optional Q/K transform      : RMSNorm weights [d] N(1, 0.1); rotary angle
  tables [T, d/2] fp32 (see ``make_qk``);
* optional LoRA adapters      : A [r, in], B [out, r] ~ N(0, 0.02) rounded to
  bf16, alpha given (see ``make_lora``).
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

# Named workloads: video DiT blocks of the sizes the method is run at.
WORKLOADS: Dict[str, dict] = {
    # 2 frames x 16x16 patches, small enough for the full float64 oracle.
    "dit_T512_D256": dict(T=512, D=256, heads=4, F=704, mlp_chunk=128,
                          attn_chunk=128, ffn_slice=0, int8=False, blocks=1,
                          final=False),
    # 4 frames x 32x32 patches.
    "dit_T4096_D1024": dict(T=4096, D=1024, heads=16, F=2816, mlp_chunk=512,
                            attn_chunk=512, ffn_slice=0, int8=False,
                            blocks=1, final=False),
    # 16 frames x 32x32 patches, 24 heads x 128.
    "dit_T16384_D3072": dict(T=16384, D=3072, heads=24, F=8192,
                             mlp_chunk=8192, attn_chunk=8192, ffn_slice=0,
                             int8=False, blocks=1, final=False),
    # 64 frames x 32x32 patches, FFN sliced 4 x 2048.
    "dit_T65536_D3072": dict(T=65536, D=3072, heads=24, F=8192,
                             mlp_chunk=4096, attn_chunk=4096, ffn_slice=2048,
                             int8=False, blocks=1, final=False),
    # 32 frames x 32x32 patches: 4 int8 blocks + fp32 final layer.
    "dit4_int8_final_T32768_D3072": dict(T=32768, D=3072, heads=24, F=8192,
                                         mlp_chunk=8192, attn_chunk=8192,
                                         ffn_slice=0, int8=True, blocks=4,
                                         final=True),
    # bf16 block at 32k tokens.
    "dit_T32768_D3072": dict(T=32768, D=3072, heads=24, F=8192,
                             mlp_chunk=8192, attn_chunk=8192, ffn_slice=0,
                             int8=False, blocks=1, final=False),
}

FINAL_OUT = 64  # output channels of the final layer


@dataclass
class BlockWeights:
    """One block's weights as CPU tensors, row-major [out, in].

    bf16 blocks fill ``wqkv .. wdown``; int8 blocks fill the same names with
    int8 tensors and ``*_scale`` with fp32 [out] scales."""

    wqkv: torch.Tensor
    wo: torch.Tensor
    wgate: torch.Tensor
    wup: torch.Tensor
    wdown: torch.Tensor
    scales: Optional[Dict[str, torch.Tensor]] = None

    @property
    def int8(self) -> bool:
        return self.wqkv.dtype == torch.int8

    def named(self):
        return dict(wqkv=self.wqkv, wo=self.wo, wgate=self.wgate,
                    wup=self.wup, wdown=self.wdown)


@dataclass
class DitInputs:
    x: torch.Tensor                       # [T, D] fp32
    blocks: List[BlockWeights]
    mods: List[torch.Tensor]              # each [6, D] fp32
    mod_f: Optional[torch.Tensor] = None  # [2, D] fp32
    wf: Optional[torch.Tensor] = None     # [64, D] fp32 or int8
    wf_scale: Optional[torch.Tensor] = None
    meta: dict = field(default_factory=dict)


def _normal(g, shape, std):
    return torch.randn(*shape, generator=g, dtype=torch.float32) * std


def _int8(g, shape):
    return torch.randint(-127, 128, shape, generator=g,
                         dtype=torch.int16).to(torch.int8)


def _scales(g, n, jitter):
    s = torch.full((n,), 0.02 / 127.0, dtype=torch.float32)
    if jitter:
        s = s * (0.5 + torch.rand(n, generator=g, dtype=torch.float32))
    return s


def make_block_weights(g, D, F, int8=False, jitter=False) -> BlockWeights:
    shapes = dict(wqkv=(3 * D, D), wo=(D, D), wgate=(F, D), wup=(F, D),
                  wdown=(D, F))
    if not int8:
        ws = {k: _normal(g, s, 0.02).to(torch.bfloat16)
              for k, s in shapes.items()}
        return BlockWeights(**ws)
    ws = {k: _int8(g, s) for k, s in shapes.items()}
    sc = {k: _scales(g, s[0], jitter) for k, s in shapes.items()}
    return BlockWeights(**ws, scales=sc)


def make_modulation(g, D) -> torch.Tensor:
    m = torch.empty(6, D, dtype=torch.float32)
    for r in (0, 1, 3, 4):                 # shift1, scale1, shift2, scale2
        m[r] = _normal(g, (D,), 0.1)
    for r in (2, 5):                       # gate1, gate2
        m[r] = torch.rand(D, generator=g, dtype=torch.float32)
    return m


def make_inputs(T, D, heads, F, seed=0, blocks=1, int8=False, final=False,
                jitter=False, x_std=1.0) -> DitInputs:
    """Draw x, ``blocks`` sets of weights + modulation and the final layer."""
    if D % heads:
        raise ValueError("D must be a multiple of heads")
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    x = _normal(g, (T, D), x_std)
    bw, mods = [], []
    for _ in range(blocks):
        bw.append(make_block_weights(g, D, F, int8=int8, jitter=jitter))
        mods.append(make_modulation(g, D))
    out = DitInputs(x=x, blocks=bw, mods=mods,
                    meta=dict(T=T, D=D, heads=heads, F=F, seed=seed,
                              int8=int8, jitter=jitter))
    if final:
        out.mod_f = _normal(g, (2, D), 0.1)
        if int8:
            out.wf = _int8(g, (FINAL_OUT, D))
            out.wf_scale = _scales(g, FINAL_OUT, jitter)
        else:
            out.wf = _normal(g, (FINAL_OUT, D), 0.02)
    return out


def make_workload(name: str, seed=0, T: Optional[int] = None,
                  jitter=False) -> DitInputs:
    c = dict(WORKLOADS[name])
    if T is not None:
        c["T"] = T
    return make_inputs(c["T"], c["D"], c["heads"], c["F"], seed=seed,
                       blocks=c["blocks"], int8=c["int8"], final=c["final"],
                       jitter=jitter)


def axial_angles(T, head_dim, grid_hw=(32, 32), base=10000.0) -> torch.Tensor:
    """Rotary angles [T, head_dim/2] of a video laid out frame by frame, each
    frame ``grid_hw`` patches row-major: the pairs are split between the
    frame, row and column index (the last two get (d/2)//3 pairs each, the
    frame the rest) and pair j of an axis with n pairs turns at
    base^(-j/n) radians per step.  An input table, like the weights: the
    block applies whatever angles it is given."""
    h, w = grid_hw
    t = torch.arange(T, dtype=torch.float64)
    pos = (torch.div(t, h * w, rounding_mode="floor"),
           torch.remainder(torch.div(t, w, rounding_mode="floor"), h),
           torch.remainder(t, w))
    half = head_dim // 2
    n_hw = half // 3
    cols = []
    for p_axis, n in zip(pos, (half - 2 * n_hw, n_hw, n_hw)):
        inv = base ** (-torch.arange(n, dtype=torch.float64) / n)
        cols.append(p_axis[:, None] * inv[None, :])
    return torch.cat(cols, dim=1)


def make_qk(T, head_dim, seed=0, angles="axial", norm=True) -> dict:
    """Q/K transform inputs: fp32 ``q_norm``/``k_norm`` [head_dim] (or None)
    and ``cos``/``sin`` [T, head_dim/2] (or None) of ``angles`` = "axial"
    (``axial_angles``), "random" (U(0, 2 pi) per entry) or None."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = dict(q_norm=None, k_norm=None, cos=None, sin=None, eps=1e-6)
    if norm:
        out["q_norm"] = 1.0 + _normal(g, (head_dim,), 0.1)
        out["k_norm"] = 1.0 + _normal(g, (head_dim,), 0.1)
    if angles is not None:
        if angles == "axial":
            th = axial_angles(T, head_dim)
        elif angles == "random":
            th = torch.rand(T, head_dim // 2, generator=g, dtype=torch.float64) * 6.283185307179586
        else:
            raise ValueError(angles)
        out["cos"] = torch.cos(th).float()
        out["sin"] = torch.sin(th).float()
    return out


LORA_SHAPES = ("qkv", "o", "gate", "up", "down")


def make_lora(D, F, rank, seed=0, names=LORA_SHAPES, std=0.02, alpha=1.0) -> dict:
    """Adapters name -> (A bf16 [rank, in], B bf16 [out, rank], alpha) for
    the linears ``names`` of a block (in/out: qkv D/3D, o D/D, gate and up
    D/F, down F/D)."""
    dims = dict(qkv=(D, 3 * D), o=(D, D), gate=(D, F), up=(D, F), down=(F, D))
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    out = {}
    for n in names:
        i, o = dims[n]
        out[n] = (_normal(g, (rank, i), std).to(torch.bfloat16),
                  _normal(g, (o, rank), std).to(torch.bfloat16), float(alpha))
    return out
