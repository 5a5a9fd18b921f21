"""Pins of the oracle's optional Q/K transform (per-head RMSNorm, rotary
embedding of interleaved channel pairs by given angles) — CPU only.

"Proposal: Generic memory-aware streaming execution for transformer models"
(attention streaming plan): the model's Q normalisation and positional
transform are applied to each streamed Q region."""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fnn

from oracle import block as ob
from test_oracle_pins import brute_attention, rand_mod, rand_weights

RNG = np.random.default_rng(77)


def standard_angles(T, d, base=10000.0):
    pos = np.arange(T)[:, None]
    inv = base ** (-np.arange(0, d, 2) / d)[None, :]
    return pos * inv


def test_rms_norm_equals_library():
    x = RNG.normal(0, 3, (17, 64))
    g = RNG.normal(1, 0.2, 64)
    ref = Fnn.rms_norm(torch.from_numpy(x), (64,), torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(ob.rms_norm(x, g), ref, rtol=1e-13)


def test_rope_is_complex_multiplication():
    T, d = 9, 16
    x = RNG.normal(size=(T, d))
    th = RNG.uniform(0, 2 * np.pi, (T, d // 2))
    z = (x[:, 0::2] + 1j * x[:, 1::2]) * np.exp(1j * th)
    got = ob.rope_rotate(x, np.cos(th), np.sin(th))
    np.testing.assert_allclose(got[:, 0::2], z.real, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(got[:, 1::2], z.imag, rtol=1e-13, atol=1e-14)
    # each pair keeps its length; zero angles are the identity
    np.testing.assert_allclose(np.hypot(got[:, 0::2], got[:, 1::2]),
                               np.hypot(x[:, 0::2], x[:, 1::2]), rtol=1e-13)
    np.testing.assert_array_equal(ob.rope_rotate(x, np.ones((T, d // 2)),
                                                 np.zeros((T, d // 2))), x)


def test_rope_scores_depend_on_position_difference_only():
    d, T = 32, 40
    th = standard_angles(T, d)
    c, s = np.cos(th), np.sin(th)
    q = RNG.normal(size=(1, d))
    k = RNG.normal(size=(1, d))
    Q = ob.rope_rotate(np.repeat(q, T, 0), c, s)
    K = ob.rope_rotate(np.repeat(k, T, 0), c, s)
    for p, r, shift in [(5, 3, 7), (30, 2, 5), (10, 10, 20)]:
        np.testing.assert_allclose(Q[p] @ K[r], Q[p + shift] @ K[r + shift],
                                   rtol=1e-12, atol=1e-12)


def test_qk_transform_is_per_head():
    T, H, d = 6, 3, 8
    t = RNG.normal(size=(T, H * d))
    g = RNG.normal(1, 0.1, d)
    th = RNG.uniform(0, 6, (T, d // 2))
    out = ob.qk_transform(t, H, g, np.cos(th), np.sin(th))
    for h in range(H):
        u = t[:, h * d:(h + 1) * d]
        exp = ob.rope_rotate(ob.rms_norm(u, g), np.cos(th), np.sin(th))
        np.testing.assert_allclose(out[:, h * d:(h + 1) * d], exp, rtol=1e-13)
    np.testing.assert_array_equal(ob.qk_transform(t, H, None, None, None), t)


def qk_inputs(T, d):
    th = RNG.uniform(0, 2 * np.pi, (T, d // 2))
    return dict(q_norm=RNG.normal(1, 0.1, d), k_norm=RNG.normal(1, 0.1, d),
                cos=np.cos(th), sin=np.sin(th), eps=1e-6)


@pytest.mark.parametrize("ca,cm,fs", [(32, 32, 0), (24, 40, 16), (1, 96, 8)])
def test_chunked_with_qk_equals_unchunked(ca, cm, fs):
    T, D, H, F = 96, 16, 2, 64
    x = RNG.normal(size=(T, D))
    w = rand_weights(D, F, std=0.25)
    mod = rand_mod(D)
    qk = qk_inputs(T, D // H)
    ref = ob.dit_block(x, w, mod, H, qk=qk)
    got = ob.dit_block_chunked(x, w, mod, H, ca, cm, fs, qk=qk)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    rows = np.array([0, 7, 50, 95])
    got_r, _ = ob.dit_block_rows(x, w, mod, H, rows, qk=qk)
    np.testing.assert_allclose(got_r, ref[rows], rtol=1e-12, atol=1e-12)


def brute_x1(x, w, mod, H, qk):
    """Scalar loops: LN-mod, projections, per-head RMS norm, rotation as a
    complex product, attention, gated residual."""
    T, D = x.shape
    d = D // H
    a = []
    for t in range(T):
        mu = sum(x[t]) / D
        var = sum((v - mu) ** 2 for v in x[t]) / D
        a.append([(x[t][c] - mu) / math.sqrt(var + 1e-6) * (1 + mod[1][c]) + mod[0][c]
                  for c in range(D)])

    def proj(rows):
        return [[sum(a[t][i] * rows[o][i] for i in range(D)) for o in range(D)]
                for t in range(T)]

    def transform(m, gamma):
        out = [row[:] for row in m]
        for t in range(T):
            for h in range(H):
                u = m[t][h * d:(h + 1) * d]
                r = math.sqrt(sum(v * v for v in u) / d + 1e-6)
                u = [u[i] / r * gamma[i] for i in range(d)]
                for i in range(d // 2):
                    z = complex(u[2 * i], u[2 * i + 1]) * complex(qk["cos"][t][i],
                                                                  qk["sin"][t][i])
                    out[t][h * d + 2 * i] = z.real
                    out[t][h * d + 2 * i + 1] = z.imag
        return out

    q = transform(proj(w.wqkv[:D]), qk["q_norm"])
    k = transform(proj(w.wqkv[D:2 * D]), qk["k_norm"])
    v = proj(w.wqkv[2 * D:])
    o = brute_attention(q, k, v, H)
    return x + mod[2] * (o @ w.wo.T)


def small_case():
    rng = np.random.default_rng(5)
    T, D, H, F = 5, 8, 2, 6
    x = rng.normal(size=(T, D))
    w = rand_weights(D, F, std=0.5)
    mod = rand_mod(D)
    th = rng.uniform(0, 2 * np.pi, (T, D // H // 2))
    qk = dict(q_norm=rng.normal(1, 0.3, D // H), k_norm=rng.normal(1, 0.3, D // H),
              cos=np.cos(th), sin=np.sin(th), eps=1e-6)
    return x, w, mod, H, qk


def test_block_with_qk_brute_force():
    x, w, mod, H, qk = small_case()
    _, taps = ob.dit_block(x, w, mod, H, taps=True, qk=qk)
    np.testing.assert_allclose(taps["x1"], brute_x1(x, w, mod, H, qk),
                               rtol=1e-12, atol=1e-13)


_ROPE, _RMS = ob.rope_rotate, ob.rms_norm


def _rope_sign_slip(x, cos, sin):
    return _ROPE(x, cos, -np.asarray(sin))


def _rope_halves_slip(x, cos, sin):
    # pairs (i, i + d/2) instead of (2i, 2i + 1)
    x = np.asarray(x, np.float64)
    h = x.shape[1] // 2
    out = np.empty_like(x)
    out[:, :h] = x[:, :h] * cos - x[:, h:] * sin
    out[:, h:] = x[:, :h] * sin + x[:, h:] * cos
    return out


def _layernorm_slip(x, gamma, eps=1e-6):
    # centred (LayerNorm) instead of RMS
    return ob.layernorm(x, eps) * gamma


QK_SLIPS = {
    "rope_sign": ("rope_rotate", _rope_sign_slip),
    "rope_halves": ("rope_rotate", _rope_halves_slip),
    "layernorm_not_rms": ("rms_norm", _layernorm_slip),
    "norm_without_gamma": ("rms_norm", lambda x, g, eps=1e-6: _RMS(x, np.ones_like(g), eps)),
}


@pytest.mark.parametrize("slip", sorted(QK_SLIPS))
def test_brute_force_catches_qk_slips(slip, monkeypatch):
    name, fn = QK_SLIPS[slip]
    monkeypatch.setattr(ob, name, fn)
    x, w, mod, H, qk = small_case()
    _, taps = ob.dit_block(x, w, mod, H, taps=True, qk=qk)
    assert not np.allclose(taps["x1"], brute_x1(x, w, mod, H, qk), rtol=1e-9, atol=1e-10)


def test_brute_force_catches_q_k_norm_swap():
    x, w, mod, H, qk = small_case()
    swapped = dict(qk, q_norm=qk["k_norm"], k_norm=qk["q_norm"])
    _, taps = ob.dit_block(x, w, mod, H, taps=True, qk=swapped)
    assert not np.allclose(taps["x1"], brute_x1(x, w, mod, H, qk), rtol=1e-9, atol=1e-10)


def test_chunked_pin_catches_slab_local_positions(monkeypatch):
    # a Q/K slab rotated by the angles of positions 0.. instead of its own
    T, D, H, F = 64, 16, 2, 32
    rng = np.random.default_rng(8)
    x = rng.normal(size=(T, D))
    w = rand_weights(D, F, std=0.25)
    mod = rand_mod(D)
    qk = qk_inputs(T, D // H)
    ref = ob.dit_block(x, w, mod, H, qk=qk)
    orig = ob._qk_one
    monkeypatch.setattr(ob, "_qk_one", lambda t, heads, q, which, rows=None: orig(
        t, heads, q, which, None if rows is None else rows - rows[0]))
    got = ob.dit_block_chunked(x, w, mod, H, 16, 16, 0, qk=qk)
    assert not np.allclose(got, ref, rtol=1e-9, atol=1e-10)
