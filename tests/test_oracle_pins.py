"""Pins of the float64 oracle against things other than itself (CPU only).

Each test ties one oracle function to a library routine, a closed form, an
invariant or a brute-force loop on tiny inputs, chosen so that a plausible
slip (a dropped term, a wrong sign, a transposed weight, a swapped
modulation row) fails at least one of them.  The method is the one of
"LayerStream: H3 Chunking" ("How the slicing works") and "Proposal: Generic
memory-aware streaming execution for transformer models" ("MLP planning").
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as Fnn
from scipy.special import expit

from oracle import block as ob

RNG = np.random.default_rng(1234)


def rand_weights(D, F, std=0.3, rng=RNG):
    return ob.DitWeights(
        wqkv=rng.normal(0, std, (3 * D, D)), wo=rng.normal(0, std, (D, D)),
        wgate=rng.normal(0, std, (F, D)), wup=rng.normal(0, std, (F, D)),
        wdown=rng.normal(0, std, (D, F)))


def rand_mod(D, rng=RNG):
    m = rng.normal(0, 0.3, (6, D))
    m[2] = rng.uniform(0, 1, D)
    m[5] = rng.uniform(0, 1, D)
    return m


# ---------------------------------------------------------------- LayerNorm

def test_layernorm_equals_library_layer_norm():
    x = RNG.normal(0, 2, (37, 96)) + 3.0
    ref = Fnn.layer_norm(torch.from_numpy(x), (96,), eps=1e-6).numpy()
    np.testing.assert_allclose(ob.layernorm(x), ref, rtol=0, atol=1e-13)


def test_layernorm_row_moments():
    x = RNG.normal(0, 0.7, (20, 64)) - 1.5
    n = ob.layernorm(x)
    var_in = x.var(axis=1)
    np.testing.assert_allclose(n.mean(axis=1), 0, atol=1e-14)
    # biased variance of the output is var / (var + eps)
    np.testing.assert_allclose(n.var(axis=1), var_in / (var_in + 1e-6),
                               rtol=1e-13)


def test_layernorm_two_channel_closed_form():
    # D = 2: (u, v) -> (+-delta / sqrt(delta^2 + eps)), delta = (u - v) / 2.
    for u, v in [(1.0, -1.0), (3.0, 1.0), (0.25, 0.75), (-2.0, 5.0)]:
        delta = (u - v) / 2
        e = delta / math.sqrt(delta * delta + 1e-6)
        np.testing.assert_allclose(ob.layernorm([[u, v]])[0], [e, -e],
                                   rtol=1e-15)


def test_modulate_rows_roles():
    n = RNG.normal(size=(3, 5))
    sh = RNG.normal(size=5)
    sc = RNG.normal(size=5)
    np.testing.assert_array_equal(ob.modulate(n, 0 * sh, 0 * sc), n)
    np.testing.assert_allclose(ob.modulate(n, sh, 0 * sc), n + sh)
    np.testing.assert_allclose(ob.modulate(n, 0 * sh, sc), n + n * sc)
    # scale = -1 collapses the normalised row to the shift
    np.testing.assert_allclose(ob.modulate(n, sh, -np.ones(5)),
                               np.broadcast_to(sh, n.shape))


# ---------------------------------------------------------------- attention

def brute_attention(q, k, v, heads):
    """Scalar loops straight from softmax(q.k / sqrt(d)) v."""
    Tq, D = len(q), len(q[0])
    d = D // heads
    out = [[0.0] * D for _ in range(Tq)]
    for h in range(heads):
        for i in range(Tq):
            s = []
            for j in range(len(k)):
                acc = 0.0
                for c in range(h * d, (h + 1) * d):
                    acc += q[i][c] * k[j][c]
                s.append(acc / math.sqrt(d))
            e = [math.exp(t) for t in s]
            z = sum(e)
            for c in range(h * d, (h + 1) * d):
                out[i][c] = sum(e[j] * v[j][c] for j in range(len(k))) / z
    return np.array(out)


def test_attention_equals_brute_force_loops():
    q = RNG.normal(size=(5, 6))
    k = RNG.normal(size=(7, 6))
    v = RNG.normal(size=(7, 6))
    got = ob.mha_attention(q, k, v, heads=3)
    ref = brute_attention(q.tolist(), k.tolist(), v.tolist(), 3)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_attention_equals_library_sdpa():
    T, H, d = 40, 4, 16
    q = RNG.normal(0, 2, (T, H * d))
    k = RNG.normal(0, 2, (T + 9, H * d))
    v = RNG.normal(size=(T + 9, H * d))

    def heads(a):
        return torch.from_numpy(a).reshape(a.shape[0], H, d).transpose(0, 1)

    ref = Fnn.scaled_dot_product_attention(heads(q), heads(k), heads(v))
    ref = ref.transpose(0, 1).reshape(T, H * d).numpy()
    np.testing.assert_allclose(ob.mha_attention(q, k, v, H), ref,
                               rtol=1e-12, atol=1e-13)


def test_attention_identity_values_give_probability_rows():
    # With V = I (d = number of keys) the output row is the softmax row.
    T = 8
    q = RNG.normal(0, 3, (5, T))
    k = RNG.normal(0, 3, (T, T))
    p = ob.mha_attention(q, k, np.eye(T), heads=1)
    assert (p > 0).all()
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
    # the largest logit gets the largest weight
    np.testing.assert_array_equal(p.argmax(1), (q @ k.T).argmax(1))


def test_attention_equal_value_rows_return_that_row():
    v_row = RNG.normal(size=8)
    q = RNG.normal(0, 4, (6, 8))
    k = RNG.normal(0, 4, (11, 8))
    v = np.tile(v_row, (11, 1))
    np.testing.assert_allclose(ob.mha_attention(q, k, v, heads=2),
                               np.tile(v_row, (6, 1)), rtol=1e-13)


def test_attention_zero_keys_average_values():
    q = RNG.normal(size=(4, 8))
    v = RNG.normal(size=(9, 8))
    got = ob.mha_attention(q, np.zeros((9, 8)), v, heads=2)
    np.testing.assert_allclose(got, np.tile(v.mean(0), (4, 1)), rtol=1e-13)


def test_attention_heads_use_their_own_columns():
    # Scaling head 1's query columns sharpens only head 1's output.
    q = RNG.normal(size=(3, 8))
    k = RNG.normal(size=(6, 8))
    v = RNG.normal(size=(6, 8))
    base = ob.mha_attention(q, k, v, 2)
    q2 = q.copy()
    q2[:, 4:] *= 5
    got = ob.mha_attention(q2, k, v, 2)
    np.testing.assert_array_equal(got[:, :4], base[:, :4])
    assert np.abs(got[:, 4:] - base[:, 4:]).max() > 1e-3


def test_attention_scale_is_inverse_sqrt_head_dim():
    # Two keys, one query: weight ratio is exp((q.k1 - q.k2) / sqrt(d)).
    d = 16
    q = np.zeros((1, d))
    q[0, 0] = 2.0
    k = np.zeros((2, d))
    k[0, 0] = 1.5
    v = np.zeros((2, d))
    v[0, 1] = 1.0
    p0 = ob.mha_attention(q, k, v, 1)[0, 1]
    z = math.exp(3.0 / math.sqrt(d))
    np.testing.assert_allclose(p0, z / (z + 1.0), rtol=1e-14)


# ---------------------------------------------------------------- SwiGLU

def test_silu_matches_library_sigmoid():
    z = np.linspace(-30, 30, 601)
    np.testing.assert_allclose(ob.silu(z), z * expit(z), rtol=1e-14,
                               atol=1e-300)
    assert ob.silu(np.array([0.0]))[0] == 0.0
    assert ob.silu(np.array([-800.0]))[0] == 0.0  # no overflow to nan


def test_swiglu_brute_force_and_roles():
    D, F = 3, 4
    w = rand_weights(D, F)
    b = RNG.normal(size=(2, D))
    got = ob.swiglu_mlp(b, w)
    ref = np.zeros((2, D))
    for t in range(2):
        for o in range(D):
            acc = 0.0
            for f in range(F):
                g = sum(b[t, i] * w.wgate[f, i] for i in range(D))
                u = sum(b[t, i] * w.wup[f, i] for i in range(D))
                acc += (g / (1 + math.exp(-g))) * u * w.wdown[o, f]
            ref[t, o] = acc
    np.testing.assert_allclose(got, ref, rtol=1e-13)
    # the activation sits on the gate projection, not the up projection:
    # with W_up = W_gate the result is silu(g) g, which is not odd in g
    w2 = ob.DitWeights(w.wqkv, w.wo, w.wgate, w.wgate.copy(), np.eye(D, F))
    h_pos = ob.swiglu_mlp(b, w2)
    h_neg = ob.swiglu_mlp(-b, w2)
    assert np.abs(h_pos + h_neg).max() > 1e-3
    g = b @ w.wgate.T
    np.testing.assert_allclose(h_pos, (g * g * expit(g))[:, :D], rtol=1e-13)


# ---------------------------------------------------------------- block

def brute_block(x, w, mod, heads):
    """Whole block in scalar loops, weights indexed W[out][in]."""
    T, D = x.shape
    F = w.wgate.shape[0]

    def ln_mod(row, sh, sc):
        mu = sum(row) / D
        var = sum((r - mu) ** 2 for r in row) / D
        return [(row[c] - mu) / math.sqrt(var + 1e-6) * (1 + sc[c]) + sh[c]
                for c in range(D)]

    def lin(vec, W, n_out):
        return [sum(vec[i] * W[o][i] for i in range(len(vec)))
                for o in range(n_out)]

    a = [ln_mod(list(x[t]), mod[0], mod[1]) for t in range(T)]
    q = [lin(a[t], w.wqkv[0:D], D) for t in range(T)]
    k = [lin(a[t], w.wqkv[D:2 * D], D) for t in range(T)]
    v = [lin(a[t], w.wqkv[2 * D:], D) for t in range(T)]
    o = brute_attention(q, k, v, heads)
    x1 = [[x[t][c] + mod[2][c] * lin(list(o[t]), w.wo, D)[c]
           for c in range(D)] for t in range(T)]
    out = []
    for t in range(T):
        b = ln_mod(x1[t], mod[3], mod[4])
        g = lin(b, w.wgate, F)
        u = lin(b, w.wup, F)
        h = [g[f] / (1 + math.exp(-g[f])) * u[f] for f in range(F)]
        m = lin(h, w.wdown, D)
        out.append([x1[t][c] + mod[5][c] * m[c] for c in range(D)])
    return np.array(out)


def test_block_equals_brute_force_loops():
    T, D, H, F = 5, 4, 2, 6
    x = RNG.normal(size=(T, D))
    w = rand_weights(D, F, std=0.6)
    mod = rand_mod(D)
    np.testing.assert_allclose(ob.dit_block(x, w, mod, H),
                               brute_block(x, w, mod, H), rtol=1e-12,
                               atol=1e-13)


def test_block_two_token_hand_example():
    # Hand-worked: x rows (1,-1), (3,1) both normalise to c(1,-1),
    # c = 1/sqrt(1+1e-6); with zero shift/scale, Wv = I, Wo = diag(2,1),
    # gate1 = (0.5,1) the attention branch adds c(1,-1) to both rows;
    # x1 rows normalise to k(1,-1), k = (1+c)/sqrt((1+c)^2+1e-6); with
    # Wg = Wu = Wd = I and gate2 = 1 the MLP adds (k silu(k), k silu(-k)).
    x = np.array([[1.0, -1.0], [3.0, 1.0]])
    I2 = np.eye(2)
    w = ob.DitWeights(wqkv=np.vstack([RNG.normal(size=(2, 2)),
                                      RNG.normal(size=(2, 2)), I2]),
                      wo=np.diag([2.0, 1.0]), wgate=I2, wup=I2, wdown=I2)
    mod = np.zeros((6, 2))
    mod[2] = [0.5, 1.0]
    mod[5] = [1.0, 1.0]
    c = 1 / math.sqrt(1 + 1e-6)
    k = (1 + c) / math.sqrt((1 + c) ** 2 + 1e-6)

    def silu(z):
        return z / (1 + math.exp(-z))

    x1 = x + np.array([c, -c])
    exp = x1 + np.array([k * silu(k), -k * silu(-k)])
    np.testing.assert_allclose(ob.dit_block(x, w, mod, 1), exp, rtol=1e-14)


@pytest.mark.parametrize("ca,cm,fs", [(0, 0, 0), (32, 32, 0), (24, 40, 16),
                                      (96, 7, 48), (1, 96, 8), (50, 0, 64)])
def test_chunked_schedule_equals_unchunked(ca, cm, fs):
    T, D, H, F = 96, 16, 2, 64
    x = RNG.normal(size=(T, D))
    w = rand_weights(D, F, std=0.25)
    mod = rand_mod(D)
    ref = ob.dit_block(x, w, mod, H)
    got = ob.dit_block_chunked(x, w, mod, H, ca, cm, fs)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_block_is_token_permutation_equivariant():
    T, D, H, F = 33, 8, 2, 24
    x = RNG.normal(size=(T, D))
    w = rand_weights(D, F)
    mod = rand_mod(D)
    perm = RNG.permutation(T)
    np.testing.assert_allclose(ob.dit_block(x[perm], w, mod, H),
                               ob.dit_block(x, w, mod, H)[perm], rtol=1e-12,
                               atol=1e-13)


def test_zero_gates_leave_residual_unchanged():
    T, D, H, F = 12, 8, 2, 16
    x = RNG.normal(size=(T, D))
    w = rand_weights(D, F)
    mod = rand_mod(D)
    mod[2] = 0
    mod[5] = 0
    np.testing.assert_array_equal(ob.dit_block(x, w, mod, H), x)


def test_gate_rows_are_two_and_five():
    T, D, H, F = 10, 8, 2, 16
    x = RNG.normal(size=(T, D))
    w = rand_weights(D, F)
    mod = rand_mod(D)
    _, t = ob.dit_block(x, w, mod, H, taps=True)
    m2 = mod.copy()
    m2[5] = 0  # only the MLP gate closed -> output is x1
    np.testing.assert_allclose(ob.dit_block(x, w, m2, H), t["x1"],
                               rtol=0, atol=0)
    m3 = mod.copy()
    m3[2] = 0  # attention gate closed -> x1 = x
    _, t3 = ob.dit_block(x, w, m3, H, taps=True)
    np.testing.assert_array_equal(t3["x1"], x)


def test_uniform_attention_closed_form():
    # Wq = 0 makes every softmax row uniform: O = mean_t(V) for all queries,
    # so x1 = x + gate1 * (mean_t(a) Wv^T) Wo^T.
    T, D, H, F = 20, 8, 2, 16
    x = RNG.normal(size=(T, D))
    w = rand_weights(D, F)
    w.wqkv[:D] = 0
    mod = rand_mod(D)
    _, t = ob.dit_block(x, w, mod, H, taps=True)
    a_mean = ob.ln_modulate(x, mod[0], mod[1]).mean(axis=0)
    exp_x1 = x + mod[2] * ((w.wqkv[2 * D:] @ a_mean) @ w.wo.T)
    np.testing.assert_allclose(t["x1"], exp_x1, rtol=1e-12, atol=1e-13)


def test_row_sampled_block_equals_full_block():
    T, D, H, F = 64, 16, 4, 32
    x = RNG.normal(size=(T, D))
    w = rand_weights(D, F)
    mod = rand_mod(D)
    rows = np.array([0, 5, 17, 63])
    full = ob.dit_block(x, w, mod, H)
    got, _ = ob.dit_block_rows(x, w, mod, H, rows)
    np.testing.assert_allclose(got, full[rows], rtol=1e-13, atol=1e-14)


# ---------------------------------------------------------------- final layer / int8

def test_final_layer_equals_library_ops():
    x = RNG.normal(size=(9, 32))
    wf = RNG.normal(size=(64, 32))
    mod_f = RNG.normal(0, 0.3, (2, 32))
    n = Fnn.layer_norm(torch.from_numpy(x), (32,), eps=1e-6)
    ref = Fnn.linear(n * (1 + torch.from_numpy(mod_f[1]))
                     + torch.from_numpy(mod_f[0]), torch.from_numpy(wf))
    np.testing.assert_allclose(ob.final_layer(x, wf, mod_f), ref.numpy(),
                               rtol=1e-12, atol=1e-13)


def test_dequant_scales_rows_not_columns():
    q = np.ones((3, 5), dtype=np.int8)
    q[1] = -127
    s = np.array([0.5, 2.0, 4.0])
    w = ob.dequant_int8(q, s)
    np.testing.assert_array_equal(w[0], 0.5)
    np.testing.assert_array_equal(w[1], -254.0)
    np.testing.assert_array_equal(w[2], 4.0)
    with pytest.raises(ValueError):
        ob.dequant_int8(q, np.ones(5))


def test_block_flops_counts_the_contractions():
    # Count multiply-adds of the oracle's contractions by their shapes.
    T, D, F = 512, 256, 704
    macs = (T * D * 3 * D + T * D * D + 2 * T * D * F + T * F * D
            + 2 * T * T * D)
    assert ob.block_flops(T, D, F) == 2 * macs == 1090519040
