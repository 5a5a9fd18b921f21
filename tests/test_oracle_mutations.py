"""Plant plausible mistakes in the oracle (on the CPU) and check the pins see them.

Each mutant rewrites one step of ``oracle.block.dit_block`` the way a slip
would (a swapped modulation row, a transposed weight, a dropped ``1 +``, the
wrong softmax scale, the activation on the wrong projection, a missing gate)
and must disagree with the scalar-loop brute force of
``test_oracle_pins.brute_block``."""

import math

import numpy as np
import pytest

from oracle import block as ob
from test_oracle_pins import brute_block, rand_mod, rand_weights


def mutant_block(x, w, mod, heads, slip):
    D = w.D
    wq, wk, wv = w.q_k_v()
    m = mod.copy()
    if slip == "swap_shift_scale":
        m[[0, 1]] = m[[1, 0]]
    if slip == "gate_row_4":
        m[[4, 5]] = m[[5, 4]]

    def lnmod(v, sh, sc):
        n = ob.layernorm(v)
        if slip == "drop_one_plus":
            return n * sc + sh
        return n * (1 + sc) + sh

    a = lnmod(x, m[0], m[1])
    q, k, v = a @ wq.T, a @ wk.T, a @ wv.T
    if slip == "q_k_swapped_rows":
        q, k = k, q
    if slip == "scale_sqrt_D":
        q = q * math.sqrt(D // heads) / math.sqrt(D)
    o = ob.mha_attention(q, k, v, heads)
    wo = w.wo.T if slip == "transpose_wo" else w.wo
    g1 = 1.0 if slip == "no_gate1" else m[2]
    x1 = x + g1 * (o @ wo.T)
    b = lnmod(x1, m[3], m[4])
    g, u = b @ w.wgate.T, b @ w.wup.T
    if slip == "silu_on_up":
        g, u = u, g
    h = ob.silu(g) * u
    return x1 + m[5] * (h @ w.wdown.T)


SLIPS = ["swap_shift_scale", "gate_row_4", "drop_one_plus",
         "q_k_swapped_rows", "scale_sqrt_D", "transpose_wo", "no_gate1",
         "silu_on_up"]


@pytest.mark.parametrize("slip", SLIPS)
def test_brute_force_pin_catches(slip):
    rng = np.random.default_rng(99)
    T, D, H, F = 5, 4, 2, 6
    x = rng.normal(size=(T, D))
    w = rand_weights(D, F, std=0.6, rng=rng)
    mod = rand_mod(D, rng=rng)
    ref = brute_block(x, w, mod, H)
    # the unmutated path agrees, the mutant does not
    np.testing.assert_allclose(mutant_block(x, w, mod, H, None), ref,
                               rtol=1e-12, atol=1e-13)
    assert np.abs(mutant_block(x, w, mod, H, slip) - ref).max() > 1e-6
