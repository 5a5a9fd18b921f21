"""Regression pin: the oracle still reproduces its committed tiny fixture.

The fixture was written by ``tests/golden/make_golden.py`` (oracle + seeded
generator only).  It guards against an accidental change of the oracle's
arithmetic; the independent pins are in ``test_oracle_pins.py``."""

import json
import os

import numpy as np

from memory_bounded_video_gb300 import synth
from oracle import block as ob

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_block_fixture():
    with open(os.path.join(HERE, "golden", "block_tiny_seed7.json")) as f:
        g = json.load(f)
    inp = synth.make_inputs(g["T"], g["D"], g["heads"], g["F"], seed=g["seed"])
    w = ob.DitWeights(**{k: v.double().numpy() * g["weight_multiplier"]
                         for k, v in inp.blocks[0].named().items()})
    x2 = ob.dit_block(inp.x.double().numpy(), w, inp.mods[0].double().numpy(),
                      g["heads"])
    np.testing.assert_allclose(x2, np.array(g["x2"]), rtol=1e-12, atol=1e-12)
