"""Pins of the oracle's activation-space LoRA (CPU only).

"ComfyUI-StaticPipeline", section "Activation-space LoRA (bypass mode)":
y = W x + alpha B (A x), applied to the activations so the weights stay
packed; section "Four levels of chunking": the delta is added in place,
chunk by chunk."""

import math

import numpy as np
import pytest

from oracle import block as ob
from test_oracle_pins import brute_attention, rand_mod, rand_weights


def adapters(D, F, r, rng, names=("qkv", "o", "gate", "up", "down"), scale=0.3):
    shapes = dict(qkv=(3 * D, D), o=(D, D), gate=(F, D), up=(F, D), down=(D, F))
    out = {}
    for i, n in enumerate(names):
        o_, i_ = shapes[n]
        out[n] = (rng.normal(0, scale, (r, i_)), rng.normal(0, scale, (o_, r)),
                  0.5 + 0.25 * i)
    return out


def case(T=40, D=16, H=2, F=48, r=4, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.normal(size=(T, D))
    w = rand_weights(D, F, std=0.25)
    mod = rand_mod(D)
    return x, w, mod, H, adapters(D, F, r, rng)


def test_bypass_equals_merged_weights():
    x, w, mod, H, lora = case()
    got = ob.dit_block(x, w, mod, H, lora=lora)
    ref = ob.dit_block(x, ob.merge_lora(w, lora), mod, H)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    # and each adapter alone
    for name in lora:
        one = {name: lora[name]}
        np.testing.assert_allclose(ob.dit_block(x, w, mod, H, lora=one),
                                   ob.dit_block(x, ob.merge_lora(w, one), mod, H),
                                   rtol=1e-12, atol=1e-12)


def test_zero_up_projection_is_no_adapter():
    x, w, mod, H, lora = case(seed=1)
    zero = {k: (A, np.zeros_like(B), a) for k, (A, B, a) in lora.items()}
    np.testing.assert_array_equal(ob.dit_block(x, w, mod, H, lora=zero),
                                  ob.dit_block(x, w, mod, H))


def test_delta_is_rank_r():
    rng = np.random.default_rng(3)
    t = rng.normal(size=(30, 12))
    A, B = rng.normal(size=(3, 12)), rng.normal(size=(20, 3))
    d = ob.lora_delta(t, (A, B, 0.7))
    assert np.linalg.matrix_rank(d) == 3
    np.testing.assert_allclose(d, 0.7 * t @ (B @ A).T, rtol=1e-12)


@pytest.mark.parametrize("ca,cm,fs", [(8, 8, 0), (16, 24, 16), (40, 7, 8), (1, 40, 24)])
def test_chunked_with_lora_equals_unchunked(ca, cm, fs):
    x, w, mod, H, lora = case(seed=2)
    ref = ob.dit_block(x, w, mod, H, lora=lora)
    got = ob.dit_block_chunked(x, w, mod, H, ca, cm, fs, lora=lora)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    rows = np.array([0, 5, 39])
    got_r, _ = ob.dit_block_rows(x, w, mod, H, rows, lora=lora)
    np.testing.assert_allclose(got_r, ref[rows], rtol=1e-12, atol=1e-12)


def brute_block_lora(x, w, mod, H, lora):
    """Scalar loops: every adapted linear as sum_k W[o,k] t[k] +
    alpha sum_j B[o,j] sum_k A[j,k] t[k]."""
    T, D = x.shape
    F = w.wgate.shape[0]

    def lin(t, W, ad, row0=0):
        A, B, al = ad
        n_out = W.shape[0]
        out = []
        for row in t:
            ua = [sum(A[j][k] * row[k] for k in range(len(row))) for j in range(len(A))]
            out.append([sum(W[o][k] * row[k] for k in range(len(row))) +
                        al * sum(B[row0 + o][j] * ua[j] for j in range(len(A)))
                        for o in range(n_out)])
        return np.array(out)

    def lnmod(v, sh, sc):
        out = []
        for row in v:
            mu = sum(row) / D
            var = sum((e - mu) ** 2 for e in row) / D
            out.append([(row[c] - mu) / math.sqrt(var + 1e-6) * (1 + sc[c]) + sh[c]
                        for c in range(D)])
        return np.array(out)

    a = lnmod(x, mod[0], mod[1])
    q = lin(a, w.wqkv[:D], lora["qkv"], 0)
    k = lin(a, w.wqkv[D:2 * D], lora["qkv"], D)
    v = lin(a, w.wqkv[2 * D:], lora["qkv"], 2 * D)
    o = brute_attention(q.tolist(), k.tolist(), v.tolist(), H)
    x1 = x + mod[2] * lin(o, w.wo, lora["o"])
    b = lnmod(x1, mod[3], mod[4])
    g = lin(b, w.wgate, lora["gate"])
    u = lin(b, w.wup, lora["up"])
    h = g / (1 + np.exp(-g)) * u
    assert h.shape[1] == F
    return x1 + mod[5] * lin(h, w.wdown, lora["down"])


def small():
    return case(T=5, D=8, H=2, F=6, r=3, seed=4)


def test_block_with_lora_brute_force():
    x, w, mod, H, lora = small()
    np.testing.assert_allclose(ob.dit_block(x, w, mod, H, lora=lora),
                               brute_block_lora(x, w, mod, H, lora),
                               rtol=1e-11, atol=1e-12)


_DELTA = ob.lora_delta


def _k_rows_from_q(t, ad, rows=None):
    if isinstance(rows, slice) and rows.start and rows.start > 0:
        D = rows.stop - rows.start
        rows = slice(rows.start - D, rows.stop - D)   # K and V take the rows before theirs
    return _DELTA(t, ad, rows)


def _alpha_twice(t, ad, rows=None):
    return _DELTA(t, (ad[0], ad[1], ad[2] * ad[2]), rows) if ad is not None else 0.0


def _transposed_product(t, ad, rows=None):
    if ad is None:
        return 0.0
    A, B, al = ad
    Bs = B if rows is None else B[rows]
    # (t A^T) B^T computed as t (A^T B^T) with A, B each reversed along r
    return al * (t @ A[::-1].T) @ Bs.T


SLIPS = {"k_v_rows_from_the_wrong_range": _k_rows_from_q, "alpha_squared": _alpha_twice,
         "rank_order_mismatch": _transposed_product}


@pytest.mark.parametrize("slip", sorted(SLIPS))
def test_brute_force_catches_lora_slips(slip, monkeypatch):
    monkeypatch.setattr(ob, "lora_delta", SLIPS[slip])
    x, w, mod, H, lora = small()
    got = ob.dit_block(x, w, mod, H, lora=lora)
    assert not np.allclose(got, brute_block_lora(x, w, mod, H, lora), rtol=1e-8, atol=1e-9)


def test_brute_force_catches_gate_delta_after_activation():
    x, w, mod, H, lora = small()
    D = w.D
    ref = brute_block_lora(x, w, mod, H, lora)
    # the gate adapter added after silu instead of before
    no_gate = dict(lora)
    A, B, al = no_gate.pop("gate")
    _, taps = ob.dit_block(x, w, mod, H, taps=True, lora=no_gate)
    b = taps["b"]
    g = b @ w.wgate.T
    u = b @ w.wup.T + ob.lora_delta(b, lora["up"])
    h = (ob.silu(g) + ob.lora_delta(b, (A, B, al))) * u
    wrong = taps["x1"] + mod[5] * (h @ w.wdown.T + ob.lora_delta(h, lora["down"]))
    assert wrong.shape == (5, D)
    assert not np.allclose(wrong, ref, rtol=1e-8, atol=1e-9)
