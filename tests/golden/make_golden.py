"""Write the oracle regression fixtures under tests/golden/.

Calls only ``oracle`` and the seeded input generator; no value here comes
from the CUDA path.  Run from the repository root:

    python tests/golden/make_golden.py
"""

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from memory_bounded_video_gb300 import synth  # noqa: E402
from oracle import block as ob  # noqa: E402


def weights64(bw):
    return ob.DitWeights(**{k: v.double().numpy() for k, v in bw.named().items()})


def tiny_block():
    T, D, H, F = 16, 8, 2, 16
    inp = synth.make_inputs(T, D, H, F, seed=7, x_std=1.0)
    # larger weights than the workloads so that every stage moves the output
    w = weights64(inp.blocks[0])
    for k in ("wqkv", "wo", "wgate", "wup", "wdown"):
        setattr(w, k, getattr(w, k) * 25.0)
    x = inp.x.double().numpy()
    mod = inp.mods[0].double().numpy()
    x2 = ob.dit_block(x, w, mod, H)
    return dict(
        what="one DiT block, float64 oracle, T=16 D=8 heads=2 F=16",
        source=("oracle.block.dit_block on synth.make_inputs(16, 8, 2, 16, "
                "seed=7) with every weight multiplied by 25"),
        weight_multiplier=25.0, T=T, D=D, heads=H, F=F, seed=7,
        x2=[[float(v) for v in r] for r in x2])


def main():
    with open(os.path.join(HERE, "block_tiny_seed7.json"), "w") as f:
        json.dump(tiny_block(), f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
