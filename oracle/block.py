"""Plain float64 definition of one bounded-activation DiT block (CPU, numpy).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): nothing in the product
path imports this module.

What the block computes
-----------------------
"LayerStream: H3 Chunking", section "The wall is activations, not weights",
lists what a block holds: projections (q, k, v), the MLP expansion, fp32
norm and head copies, and the residual stream.  Section "How the slicing
works" gives the order of operations: norm + modulation, the projections and
the MLP are token-wise and add into the residual stream in place; attention
needs every key and value, so K and V are kept for all tokens while queries
are recomputed per slice, attended, projected and added into the residual.
"Proposal: Generic memory-aware streaming execution for transformer models"
(section "MLP planning") describes the gated MLP as gate/up projection,
gated activation, down projection.

Because every streamed schedule on those pages computes the same function
("same math, smaller working set"; the proposal's "Safety and fallback
behavior" asks that decompositions keep the model's computation), the oracle
computes that function directly, unchunked, in float64:

    a   = LN(x) * (1 + scale1) + shift1
    Q   = a Wq^T,  K = a Wk^T,  V = a Wv^T      (Wqkv rows: Q, K, V)
    O_h = softmax(Q_h K_h^T / sqrt(d)) V_h       (per head, non-causal)
    x1  = x + gate1 * (O Wo^T)
    b   = LN(x1) * (1 + scale2) + shift2
    x2  = x1 + gate2 * ((silu(b Wg^T) * (b Wu^T)) Wd^T)

Readings where the pages are silent:

* LN is LayerNorm over the hidden axis, biased variance, eps 1e-6, no affine.
* ``modulation`` is [6, D] with rows shift1, scale1, gate1, shift2, scale2,
  gate2; modulation is ``n * (1 + scale) + shift``; the residual is gated
  per channel, ``x += gate * branch``.
* SwiGLU is ``silu(gate_proj) * up_proj`` with separate W_gate / W_up;
  ``silu(z) = z / (1 + exp(-z))``.
* No biases anywhere.  Q/K normalisation and rotary embedding are optional
  (``qk``); see ``qk_transform``.
* Activation-space LoRA is optional (``lora``): each adapted linear gives
  ``t W^T + alpha (t A^T) B^T`` ("ComfyUI-StaticPipeline", section
  "Activation-space LoRA (bypass mode)": y = W x + alpha B (A x), weights
  left packed).  The fused Q/K/V projection has one adapter whose B rows
  follow Wqkv's (Q, K, V); the down projection's A is [r, F].
* Weights are row-major [out, in] (the ``nn.Linear.weight`` convention);
  head h owns hidden columns h*d .. (h+1)*d-1 of Q, K, V and O.
* INT8 weights are ``W = s_row * q`` with one float scale per output row
  ("MiniMax-H3-Comfy-NPU" article, section 2.2).
* The final layer is ``(LN(x) * (1 + scale_f) + shift_f) W_f^T`` in fp32
  arithmetic on the pages ("LayerStream: H3 Chunking": the fp32 output head
  runs unsliced); here float64.

Parity: every function below is pinned by ``tests/test_oracle_*.py``.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

LN_EPS = 1e-6
F64 = np.float64


@dataclass
class DitWeights:
    """Float64 weights of one block, each row-major [out, in]."""

    wqkv: np.ndarray   # [3D, D]  rows 0..D-1 = Q, D..2D-1 = K, 2D..3D-1 = V
    wo: np.ndarray     # [D, D]
    wgate: np.ndarray  # [F, D]
    wup: np.ndarray    # [F, D]
    wdown: np.ndarray  # [D, F]

    @property
    def D(self) -> int:
        return self.wo.shape[0]

    @property
    def F(self) -> int:
        return self.wgate.shape[0]

    def q_k_v(self):
        D = self.D
        return self.wqkv[:D], self.wqkv[D:2 * D], self.wqkv[2 * D:3 * D]


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=F64)


def dequant_int8(q, scale) -> np.ndarray:
    """W = s_row * q for an int8 matrix q [N, K] and scales s [N].

    "MiniMax-H3-Comfy-NPU" section 2.2: one ``weight_scale`` per output row,
    which is sliced together with the rows."""
    q = np.asarray(q)
    if q.dtype != np.int8:
        raise TypeError("int8 weights expected")
    s = _f64(scale)
    if s.shape != (q.shape[0],):
        raise ValueError("one scale per output row expected")
    return s[:, None] * q.astype(F64)


def layernorm(x, eps: float = LN_EPS) -> np.ndarray:
    """Row-wise LayerNorm over the last axis, biased variance, no affine.

    The pages only say "norms" ("LayerStream: H3 Chunking", "How the
    slicing works"); LayerNorm with eps 1e-6 and no affine is the reading."""
    x = _f64(x)
    mu = x.mean(axis=-1, keepdims=True)
    xc = x - mu
    var = (xc * xc).mean(axis=-1, keepdims=True)
    return xc / np.sqrt(var + eps)


def modulate(n, shift, scale) -> np.ndarray:
    """adaLN modulation ``n * (1 + scale) + shift`` (per channel)."""
    return _f64(n) * (1.0 + _f64(scale)) + _f64(shift)


def ln_modulate(x, shift, scale, eps: float = LN_EPS) -> np.ndarray:
    """Norm + modulation, the first token-wise step of each branch."""
    return modulate(layernorm(x, eps), shift, scale)


def mha_attention(q, k, v, heads: int) -> np.ndarray:
    """Non-causal multi-head softmax attention, one query per row.

    "LayerStream: H3 Chunking", "How the slicing works": every query needs
    every key and value.  Per head h (hidden columns h*d .. (h+1)*d-1):
    ``O_h = softmax(Q_h K_h^T / sqrt(d)) V_h``.  The max subtraction is the
    usual overflow guard; it cancels exactly in real arithmetic."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    Tq, D = q.shape
    if k.shape != v.shape or k.shape[1] != D or D % heads:
        raise ValueError("bad attention shapes")
    d = D // heads
    out = np.empty((Tq, D), dtype=F64)
    for h in range(heads):
        cols = slice(h * d, (h + 1) * d)
        s = (q[:, cols] @ k[:, cols].T) / math.sqrt(d)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, cols] = p @ v[:, cols]
    return out


def silu(z) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z)) (the SwiGLU gate activation)."""
    z = _f64(z)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu_mlp(b, w: DitWeights) -> np.ndarray:
    """Gated MLP: ``(silu(b Wg^T) * (b Wu^T)) Wd^T``.

    "Proposal: Generic memory-aware streaming execution ...", "MLP planning":
    input projection, gated activation, output projection."""
    b = _f64(b)
    h = silu(b @ w.wgate.T) * (b @ w.wup.T)
    return h @ w.wdown.T


def rms_norm(x, gamma, eps: float = LN_EPS) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * gamma."""
    x = _f64(x)
    return x / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps) * _f64(gamma)


def rope_rotate(x, cos, sin) -> np.ndarray:
    """Rotate channel pairs (2i, 2i+1) of x [T, d] by the angles whose cosine
    and sine are cos, sin [T, d/2]: (x0, x1) -> (x0 c - x1 s, x0 s + x1 c)."""
    x = _f64(x)
    c, s = _f64(cos), _f64(sin)
    x0, x1 = x[:, 0::2], x[:, 1::2]
    out = np.empty_like(x)
    out[:, 0::2] = x0 * c - x1 * s
    out[:, 1::2] = x0 * s + x1 * c
    return out


def qk_transform(t, heads: int, gamma, cos, sin, eps: float = LN_EPS) -> np.ndarray:
    """Per-head RMSNorm (weights gamma [d], or none) then rotary embedding
    (tables cos/sin [T, d/2], or none) of a Q or K matrix [T, H*d].

    "Proposal: Generic memory-aware streaming execution for transformer
    models", attention streaming plan: the model's Q normalisation and
    positional transform are applied to each streamed Q region (and to K).
    The pages name the steps only; per-head RMSNorm with a learned weight and
    the rotation of interleaved pairs by caller-given angles are the
    readings taken."""
    t = _f64(t)
    T, D = t.shape
    d = D // heads
    out = np.empty_like(t)
    for h in range(heads):
        u = t[:, h * d:(h + 1) * d]
        if gamma is not None:
            u = rms_norm(u, gamma, eps)
        if cos is not None:
            u = rope_rotate(u, cos, sin)
        out[:, h * d:(h + 1) * d] = u
    return out


def _qk_one(t, heads, qk, which, rows=None):
    """The Q (which = "q") or K ("k") transform of ``qk`` applied to t, whose
    rows are the tokens ``rows`` (all tokens from 0 when None)."""
    if qk is None:
        return t
    cos, sin = qk.get("cos"), qk.get("sin")
    if cos is not None and rows is not None:
        cos, sin = _f64(cos)[rows], _f64(sin)[rows]
    return qk_transform(t, heads, qk.get(which + "_norm"), cos, sin,
                        qk.get("eps", LN_EPS))


def lora_delta(t, adapter, rows=None):
    """``alpha * (t A^T) B[rows]^T`` for an adapter (A [r, in], B [out, r],
    alpha), or 0 when there is none.

    "ComfyUI-StaticPipeline", section "Activation-space LoRA (bypass mode)":
    the adapter is applied to the activations, y = W x + alpha B (A x),
    instead of being merged into the (packed) weights."""
    if adapter is None:
        return 0.0
    A, B, alpha = adapter
    B = _f64(B)
    if rows is not None:
        B = B[rows]
    return alpha * ((_f64(t) @ _f64(A).T) @ B.T)


def merge_lora(w: DitWeights, lora) -> DitWeights:
    """The weights with every adapter merged in, W + alpha B A (the form the
    bypass avoids; used to pin ``lora_delta`` by linearity)."""
    out = DitWeights(*(getattr(w, k).copy() for k in
                       ("wqkv", "wo", "wgate", "wup", "wdown")))
    for name, attr in (("qkv", "wqkv"), ("o", "wo"), ("gate", "wgate"),
                       ("up", "wup"), ("down", "wdown")):
        ad = _ad(lora, name)
        if ad is not None:
            A, B, alpha = ad
            setattr(out, attr, getattr(out, attr) + alpha * (_f64(B) @ _f64(A)))
    return out


def _ad(lora, name):
    return None if lora is None else lora.get(name)


def dit_block(x, w: DitWeights, mod, heads: int, eps: float = LN_EPS,
              taps: bool = False, qk=None, lora=None):
    """Unchunked forward of one block; returns x2 (and the stage taps).

    ``mod`` is [6, D]: shift1, scale1, gate1, shift2, scale2, gate2.
    ``qk`` (optional): dict with q_norm, k_norm ([d] or None), cos, sin
    ([T, d/2] or None) and eps — the Q/K transform before attention.
    ``lora`` (optional): dict name -> (A, B, alpha) for the linears "qkv",
    "o", "gate", "up", "down" — see ``lora_delta``."""
    x = _f64(x)
    mod = _f64(mod)
    D = w.D
    wq, wk, wv = w.q_k_v()
    a = ln_modulate(x, mod[0], mod[1], eps)
    ad = _ad(lora, "qkv")
    q = a @ wq.T + lora_delta(a, ad, slice(0, D))
    k = a @ wk.T + lora_delta(a, ad, slice(D, 2 * D))
    v = a @ wv.T + lora_delta(a, ad, slice(2 * D, 3 * D))
    q, k = _qk_one(q, heads, qk, "q"), _qk_one(k, heads, qk, "k")
    o = mha_attention(q, k, v, heads)
    x1 = x + mod[2] * (o @ w.wo.T + lora_delta(o, _ad(lora, "o")))
    b = ln_modulate(x1, mod[3], mod[4], eps)
    g = b @ w.wgate.T + lora_delta(b, _ad(lora, "gate"))
    u = b @ w.wup.T + lora_delta(b, _ad(lora, "up"))
    h = silu(g) * u
    x2 = x1 + mod[5] * (h @ w.wdown.T + lora_delta(h, _ad(lora, "down")))
    if not taps:
        return x2
    return x2, dict(a=a, q=q, k=k, v=v, o=o, x1=x1, b=b, h=h, x2=x2)


def dit_block_chunked(x, w: DitWeights, mod, heads: int, attn_chunk: int,
                      mlp_chunk: int, ffn_slice: int, eps: float = LN_EPS, qk=None,
                      lora=None):
    """The pages' bounded schedule, written out on token slices (self-check).

    "LayerStream: H3 Chunking", "How the slicing works": pass one keeps
    K and V for all tokens; pass two recomputes Q per slice, attends it to
    the full K/V, projects and adds into the residual; the MLP runs on token
    slices.  "Proposal ...", "MLP planning": each FFN feature slice is
    projected, activated, passed through the matching down-projection slice
    and accumulated.  A chunk of 0 means unchunked.  Used only to check that
    the schedule equals ``dit_block`` (which it must, up to rounding)."""
    x = _f64(x).copy()
    mod = _f64(mod)
    T, D = x.shape
    F = w.F
    ca = attn_chunk or T
    cm = mlp_chunk or T
    fs = ffn_slice or F
    wq, wk, wv = w.q_k_v()
    K = np.empty((T, D))
    V = np.empty((T, D))
    aq = _ad(lora, "qkv")
    for s in range(0, T, ca):                       # pass one: K/V only
        a = ln_modulate(x[s:s + ca], mod[0], mod[1], eps)
        k = a @ wk.T + lora_delta(a, aq, slice(D, 2 * D))
        K[s:s + ca] = _qk_one(k, heads, qk, "k", np.arange(s, min(s + ca, T)))
        V[s:s + ca] = a @ wv.T + lora_delta(a, aq, slice(2 * D, 3 * D))
    for s in range(0, T, ca):                       # pass two: Q slab
        a = ln_modulate(x[s:s + ca], mod[0], mod[1], eps)
        q = a @ wq.T + lora_delta(a, aq, slice(0, D))
        q = _qk_one(q, heads, qk, "q", np.arange(s, min(s + ca, T)))
        o = mha_attention(q, K, V, heads)
        x[s:s + ca] += mod[2] * (o @ w.wo.T + lora_delta(o, _ad(lora, "o")))
    ag, au, adn = _ad(lora, "gate"), _ad(lora, "up"), _ad(lora, "down")
    for c in range(0, T, cm):                       # MLP token chunks
        b = ln_modulate(x[c:c + cm], mod[3], mod[4], eps)
        acc = np.zeros((b.shape[0], D))
        ud = 0.0                                    # down adapter: h A_d^T
        for f in range(0, F, fs):                   # FFN feature slices
            fr = slice(f, f + fs)
            g = b @ w.wgate[fr].T + lora_delta(b, ag, fr)
            u = b @ w.wup[fr].T + lora_delta(b, au, fr)
            hf = silu(g) * u
            acc += hf @ w.wdown[:, fr].T
            if adn is not None:
                ud = ud + hf @ _f64(adn[0])[:, fr].T
        if adn is not None:
            acc += adn[2] * (ud @ _f64(adn[1]).T)
        x[c:c + cm] += mod[5] * acc
    return x


def dit_block_rows(x, w: DitWeights, mod, heads: int, rows,
                   eps: float = LN_EPS, kv=None, qk=None, lora=None):
    """The block's output on selected token rows only.

    Every stage but attention is token-wise, so the output rows ``rows``
    need K and V of all tokens (computed here, or passed in as ``kv``) and
    every other stage only on those rows.  Returns (x2[rows], taps)."""
    x = _f64(x)
    mod = _f64(mod)
    rows = np.asarray(rows, dtype=np.int64)
    wq, wk, wv = w.q_k_v()
    D = w.D
    aq = _ad(lora, "qkv")
    if kv is None:
        a_all = ln_modulate(x, mod[0], mod[1], eps)
        k = a_all @ wk.T + lora_delta(a_all, aq, slice(D, 2 * D))
        kv = (_qk_one(k, heads, qk, "k"),
              a_all @ wv.T + lora_delta(a_all, aq, slice(2 * D, 3 * D)))
    K, V = kv
    xr = x[rows]
    a = ln_modulate(xr, mod[0], mod[1], eps)
    q = _qk_one(a @ wq.T + lora_delta(a, aq, slice(0, D)), heads, qk, "q", rows)
    o = mha_attention(q, K, V, heads)
    x1 = xr + mod[2] * (o @ w.wo.T + lora_delta(o, _ad(lora, "o")))
    b = ln_modulate(x1, mod[3], mod[4], eps)
    h = silu(b @ w.wgate.T + lora_delta(b, _ad(lora, "gate"))) * \
        (b @ w.wup.T + lora_delta(b, _ad(lora, "up")))
    x2 = x1 + mod[5] * (h @ w.wdown.T + lora_delta(h, _ad(lora, "down")))
    return x2, dict(q=q, o=o, x1=x1, b=b, h=h, k=K, v=V)


def final_layer(x, wf, mod_f, eps: float = LN_EPS) -> np.ndarray:
    """Output head: ``(LN(x) * (1 + scale_f) + shift_f) W_f^T``.

    ``mod_f`` is [2, D] (shift_f, scale_f), ``wf`` is [P, D].  "LayerStream:
    H3 Chunking", "How the slicing works": the fp32 output head runs stock
    (unsliced) for exactness."""
    mod_f = _f64(mod_f)
    return ln_modulate(x, mod_f[0], mod_f[1], eps) @ _f64(wf).T


def block_flops(T: int, D: int, F: int) -> int:
    """Algorithmic flops of one block: Q/K/V projections (6 D^2 per token,
    Q counted once), O projection (2 D^2), MLP (6 D F) and the two attention
    contractions (4 T D per query token).  Norms, softmax and elementwise
    work are not counted."""
    return T * (8 * D * D + 6 * D * F) + 4 * T * T * D
