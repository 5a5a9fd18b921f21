"""ctypes binding of libditstream (argument marshalling only).

Every function here forwards to the C ABI declared in ``include/ditstream.h``
with the same name (minus the ``dit_`` prefix); all compute runs in the CUDA
kernels of the library.  Device buffers may be given as integers (device
addresses) or as objects with ``data_ptr()`` (e.g. torch tensors); streams as
integers (``cudaStream_t``) or objects with ``cuda_stream``.  A non-OK status
raises :class:`DitError`.  There is no fallback: if the library is missing,
:func:`load` raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libditstream.so")

OK = 0
ERR_INVALID_ARG = -1
ERR_CHUNK_ALIGN = -2
ERR_ALIGN = -3
ERR_NO_WORKSPACE = -4
ERR_WORKSPACE_TOO_SMALL = -5
ERR_CUDA = -6
ERR_TIMEOUT = -7
ERR_UNSUPPORTED_ARCH = -8

W_BF16 = 0
W_INT8 = 1

EPI_STORE_BF16 = 0
EPI_STORE_F32 = 1
EPI_KV = 2
EPI_RESID = 3
EPI_SWIGLU = 4
EPI_DOWN = 5

GEMM_FLAG_INJECT_STALL = 1

# Exported symbols of the C ABI (checked by the CPU tests against the header).
SYMBOLS = (
    "dit_block_plan", "dit_block_plan_ex", "dit_block_plan_destroy",
    "dit_block_plan_info", "dit_block_workspace_bytes",
    "dit_block_bind_workspace", "dit_block_forward", "dit_block_sync_status",
    "dit_final_forward", "dit_status_string", "dit_last_cuda_error",
    "dit_abi_version", "dit_modln_cast", "dit_gemm", "dit_attention",
    "dit_block_profile_enable", "dit_block_profile_read",
    "dit_block_forward_static", "dit_block_plan_auto", "dit_block_forward_qk",
    "dit_block_forward_ex", "dit_block_plan_set_lora_rank", "dit_lora_prepare",
    "dit_block_weight_scratch_bytes", "dit_block_bind_weight_scratch", "dit_int8_to_bf16",
    "dit_block_plan_set_kv_offload", "dit_block_kv_host_bytes", "dit_block_bind_kv_host",
    "dit_attention_part", "dit_attention_split_bytes", "dit_attention_ex",
    "dit_attention_schedule", "dit_gemm_split_bytes", "dit_gemm_ex",
)

STATIC_SCRATCH_BYTES = 64 << 20

# Kernel kinds of the per-kernel timing record (DIT_K_*).
KINDS = ("modln", "gemm_kv", "gemm_q", "attention", "gemm_o", "gemm_swiglu",
         "gemm_down", "final", "lora_u", "expand")
# work unit of each kind: flops (tensor-core kinds) or bytes (memory-bound)
KIND_UNITS = ("bytes", "flops", "flops", "flops", "flops", "flops", "flops",
              "bytes", "flops", "bytes")


class DitError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.dit_status_string(status).decode() if _lib else str(status)
        if status == ERR_CUDA and _lib:
            msg += ": " + _lib.dit_last_cuda_error().decode()
        super().__init__(f"{where}: {msg} (status {status})")


class BlockWeights(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int),
                ("wqkv", ctypes.c_void_p), ("wo", ctypes.c_void_p),
                ("wgate", ctypes.c_void_p), ("wup", ctypes.c_void_p),
                ("wdown", ctypes.c_void_p),
                ("wqkv_scale", ctypes.c_void_p), ("wo_scale", ctypes.c_void_p),
                ("wgate_scale", ctypes.c_void_p), ("wup_scale", ctypes.c_void_p),
                ("wdown_scale", ctypes.c_void_p)]


class GemmArgs(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int), ("M", ctypes.c_int64),
                ("N", ctypes.c_int), ("K", ctypes.c_int),
                ("a", ctypes.c_void_p), ("lda", ctypes.c_int64),
                ("b0", ctypes.c_void_p), ("b1", ctypes.c_void_p),
                ("ldb", ctypes.c_int64), ("b_dtype", ctypes.c_int),
                ("b0_scale", ctypes.c_void_p), ("b1_scale", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("ldo", ctypes.c_int64),
                ("out2", ctypes.c_void_p), ("ldo2", ctypes.c_int64),
                ("row_offset", ctypes.c_int64), ("split_n", ctypes.c_int),
                ("x", ctypes.c_void_p), ("ldx", ctypes.c_int64),
                ("gate", ctypes.c_void_p),
                ("acc", ctypes.c_void_p), ("ldacc", ctypes.c_int64),
                ("acc_load", ctypes.c_int), ("acc_final", ctypes.c_int),
                ("flags", ctypes.c_int),
                ("qk_norm", ctypes.c_void_p), ("rope_cos", ctypes.c_void_p),
                ("rope_sin", ctypes.c_void_p), ("head_dim", ctypes.c_int),
                ("qk_eps", ctypes.c_float),
                ("lora_u0", ctypes.c_void_p), ("lora_ldu0", ctypes.c_int64),
                ("lora_l0", ctypes.c_void_p), ("lora_ldl0", ctypes.c_int64),
                ("lora_rank0", ctypes.c_int),
                ("lora_u1", ctypes.c_void_p), ("lora_ldu1", ctypes.c_int64),
                ("lora_l1", ctypes.c_void_p), ("lora_ldl1", ctypes.c_int64),
                ("lora_rank1", ctypes.c_int),
                ("rope_pos0", ctypes.c_int64)]


class LoraArgs(ctypes.Structure):
    """dit_lora_t: one adapter (A [rank, in], prepared B [out, rank])."""
    _fields_ = [("a", ctypes.c_void_p), ("b", ctypes.c_void_p), ("rank", ctypes.c_int)]


class BlockLora(ctypes.Structure):
    """dit_block_lora_t: the adapters of one block (absent ones zero)."""
    _fields_ = [("qkv", LoraArgs), ("o", LoraArgs), ("gate", LoraArgs),
                ("up", LoraArgs), ("down", LoraArgs)]


class QkArgs(ctypes.Structure):
    """dit_qk_t: per-head Q/K RMSNorm weights and rotary angle tables."""
    _fields_ = [("q_norm", ctypes.c_void_p), ("k_norm", ctypes.c_void_p),
                ("rope_cos", ctypes.c_void_p), ("rope_sin", ctypes.c_void_p),
                ("eps", ctypes.c_float)]


_lib: Optional[ctypes.CDLL] = None


def _declare(lib):
    c_int, c_int64, c_size, vp = (ctypes.c_int, ctypes.c_int64, ctypes.c_size_t,
                                  ctypes.c_void_p)
    pp = ctypes.POINTER(ctypes.c_void_p)
    sig = {
        "dit_block_plan": (c_int, [c_int64, c_int, c_int, c_int, c_int, c_int, pp]),
        "dit_block_plan_ex": (c_int, [c_int64, c_int, c_int, c_int, c_int, c_int,
                                      c_int, pp]),
        "dit_block_plan_destroy": (None, [vp]),
        "dit_block_plan_info": (c_int, [vp] + [vp] * 7),
        "dit_block_workspace_bytes": (c_size, [vp]),
        "dit_block_bind_workspace": (c_int, [vp, vp, c_size]),
        "dit_block_forward": (c_int, [vp, vp, ctypes.POINTER(BlockWeights), vp, vp]),
        "dit_block_sync_status": (c_int, [vp, vp]),
        "dit_final_forward": (c_int, [vp, vp, vp, vp, vp, vp, vp]),
        "dit_status_string": (ctypes.c_char_p, [c_int]),
        "dit_last_cuda_error": (ctypes.c_char_p, []),
        "dit_abi_version": (c_int, []),
        "dit_modln_cast": (c_int, [vp, c_int64, c_int, vp, vp, vp, vp]),
        "dit_gemm": (c_int, [ctypes.POINTER(GemmArgs), vp, vp]),
        "dit_attention": (c_int, [vp, c_int64, c_int64, vp, c_int64, vp, c_int64,
                                  c_int64, c_int, c_int, vp, c_int64, vp, vp]),
        "dit_block_profile_enable": (c_int, [vp, c_int]),
        "dit_block_profile_read": (c_int, [vp, vp, vp, vp]),
        "dit_block_forward_static": (c_int, [vp, vp, ctypes.POINTER(BlockWeights),
                                             vp, vp]),
        "dit_block_plan_auto": (c_int, [c_int64, c_int, c_int, c_int, c_size, pp]),
        "dit_block_forward_qk": (c_int, [vp, vp, ctypes.POINTER(BlockWeights), vp,
                                         ctypes.POINTER(QkArgs), vp]),
        "dit_block_forward_ex": (c_int, [vp, vp, ctypes.POINTER(BlockWeights), vp,
                                         ctypes.POINTER(QkArgs), ctypes.POINTER(BlockLora),
                                         vp]),
        "dit_block_plan_set_lora_rank": (c_int, [vp, c_int]),
        "dit_block_weight_scratch_bytes": (c_size, [vp]),
        "dit_block_bind_weight_scratch": (c_int, [vp, vp, c_size]),
        "dit_int8_to_bf16": (c_int, [vp, c_int64, vp, vp]),
        "dit_block_plan_set_kv_offload": (c_int, [vp, c_int]),
        "dit_block_kv_host_bytes": (c_size, [vp]),
        "dit_block_bind_kv_host": (c_int, [vp, vp, c_size]),
        "dit_attention_part": (c_int, [vp, c_int64, c_int64, vp, c_int64, vp, c_int64,
                                       c_int64, c_int, c_int, vp, c_int64, vp, vp, vp,
                                       c_int64, c_int, c_int, vp, vp]),
        "dit_lora_prepare": (c_int, [vp, c_int64, c_int, c_int64, ctypes.c_float, vp, vp,
                                     c_int64, vp]),
        "dit_attention_split_bytes": (c_size, [c_int, c_int]),
        "dit_gemm_split_bytes": (c_size, [c_int]),
        "dit_gemm_ex": (c_int, [ctypes.POINTER(GemmArgs), vp, c_size, c_int, vp, vp]),
        "dit_attention_ex": (c_int, [vp, c_int64, c_int64, vp, c_int64, vp, c_int64,
                                     c_int64, c_int, c_int, vp, c_int64, vp, c_size, c_int,
                                     vp, vp]),
        "dit_attention_schedule": (c_int, [c_int, c_int, c_int, c_int, vp, vp, vp,
                                           c_int64, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Open the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(
                f"libditstream not built ({path} missing): run "
                "`python -m memory_bounded_video_gb300.build`")
        lib = ctypes.CDLL(path)
        _declare(lib)
        _lib = lib
    return _lib


def ptr(t) -> Optional[int]:
    """Device address of a buffer given as int, None or tensor-like."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return int(t.data_ptr())


def stream_handle(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _check(status: int, where: str):
    if status != OK:
        raise DitError(status, where)


def status_string(s: int) -> str:
    return load().dit_status_string(s).decode()


def abi_version() -> int:
    return load().dit_abi_version()


class BlockPlan:
    """Owns a ``dit_plan_t``; see ``dit_block_plan_ex``.  With
    ``budget_bytes`` set the chunk sizes are chosen by
    ``dit_block_plan_auto`` instead."""

    def __init__(self, T, D, heads, ffn, mlp_chunk_tokens=0, attn_chunk_tokens=0,
                 ffn_slice=0, budget_bytes=None):
        lib = load()
        h = ctypes.c_void_p()
        if budget_bytes is not None:
            _check(lib.dit_block_plan_auto(T, D, heads, ffn, int(budget_bytes),
                                           ctypes.byref(h)), "dit_block_plan_auto")
        else:
            _check(lib.dit_block_plan_ex(T, D, heads, ffn, mlp_chunk_tokens,
                                         attn_chunk_tokens, ffn_slice,
                                         ctypes.byref(h)), "dit_block_plan_ex")
        self._h = h
        self._ws = None

    def __del__(self):
        if getattr(self, "_h", None) and _lib is not None:
            _lib.dit_block_plan_destroy(self._h)
            self._h = None

    @property
    def handle(self):
        return self._h

    def info(self) -> dict:
        T = ctypes.c_int64()
        ints = [ctypes.c_int() for _ in range(6)]
        _check(load().dit_block_plan_info(self._h, ctypes.byref(T),
                                          *[ctypes.byref(i) for i in ints]),
               "dit_block_plan_info")
        keys = ("D", "heads", "ffn", "mlp_chunk", "attn_chunk", "ffn_slice")
        return dict(T=T.value, **{k: v.value for k, v in zip(keys, ints)})

    def workspace_bytes(self) -> int:
        return int(load().dit_block_workspace_bytes(self._h))

    def bind_workspace(self, buf, nbytes: Optional[int] = None):
        if nbytes is None:
            nbytes = buf.numel() * buf.element_size()
        _check(load().dit_block_bind_workspace(self._h, ptr(buf), nbytes),
               "dit_block_bind_workspace")
        self._ws = buf  # keep the caller's buffer alive with the plan

    def forward(self, x, weights: BlockWeights, modulation, stream=None,
                qk: Optional["QkArgs"] = None, lora: Optional["BlockLora"] = None):
        if lora is not None:
            _check(load().dit_block_forward_ex(
                self._h, ptr(x), ctypes.byref(weights), ptr(modulation),
                None if qk is None else ctypes.byref(qk), ctypes.byref(lora),
                stream_handle(stream)), "dit_block_forward_ex")
        elif qk is None:
            _check(load().dit_block_forward(self._h, ptr(x), ctypes.byref(weights),
                                            ptr(modulation), stream_handle(stream)),
                   "dit_block_forward")
        else:
            _check(load().dit_block_forward_qk(self._h, ptr(x), ctypes.byref(weights),
                                               ptr(modulation), ctypes.byref(qk),
                                               stream_handle(stream)),
                   "dit_block_forward_qk")

    def weight_scratch_bytes(self) -> int:
        return int(load().dit_block_weight_scratch_bytes(self._h))

    def bind_weight_scratch(self, buf, nbytes: Optional[int] = None):
        """Bind (or, with None, unbind) the int8 weight-expansion scratch."""
        if buf is None:
            _check(load().dit_block_bind_weight_scratch(self._h, None, 0),
                   "dit_block_bind_weight_scratch")
        else:
            if nbytes is None:
                nbytes = buf.numel() * buf.element_size()
            _check(load().dit_block_bind_weight_scratch(self._h, ptr(buf), nbytes),
                   "dit_block_bind_weight_scratch")
        self._wscratch = buf

    def set_kv_offload(self, key_block_tokens: int):
        """K/V of all tokens in pinned host memory, streamed back in key
        blocks (before binding a workspace)."""
        _check(load().dit_block_plan_set_kv_offload(self._h, key_block_tokens),
               "dit_block_plan_set_kv_offload")

    def kv_host_bytes(self) -> int:
        return int(load().dit_block_kv_host_bytes(self._h))

    def bind_kv_host(self, buf, nbytes: Optional[int] = None):
        """Bind a pinned host buffer (e.g. ``torch.empty(..., pin_memory=True)``)."""
        if nbytes is None:
            nbytes = buf.numel() * buf.element_size()
        _check(load().dit_block_bind_kv_host(self._h, ptr(buf), nbytes),
               "dit_block_bind_kv_host")
        self._kv_host = buf

    def set_lora_rank(self, max_rank: int):
        """Reserve workspace for adapters of rank <= max_rank (before binding)."""
        _check(load().dit_block_plan_set_lora_rank(self._h, max_rank),
               "dit_block_plan_set_lora_rank")

    def forward_static(self, x, weights: BlockWeights, modulation, stream=None):
        """dit_block_forward_static: the same forward with the library's
        fixed device scratch instead of a bound workspace, for callers that
        cannot allocate device memory."""
        _check(load().dit_block_forward_static(self._h, ptr(x), ctypes.byref(weights),
                                               ptr(modulation),
                                               stream_handle(stream)),
               "dit_block_forward_static")

    def sync_status(self, stream=None) -> int:
        return load().dit_block_sync_status(self._h, stream_handle(stream))

    def profile_enable(self, on: bool = True):
        _check(load().dit_block_profile_enable(self._h, int(bool(on))),
               "dit_block_profile_enable")

    def profile_read(self) -> dict:
        """Per kernel kind: {"ms", "launches", "work"} since the last read."""
        n = len(KINDS)
        ms = (ctypes.c_double * n)()
        cnt = (ctypes.c_int64 * n)()
        work = (ctypes.c_double * n)()
        _check(load().dit_block_profile_read(self._h, ms, cnt, work),
               "dit_block_profile_read")
        return {k: dict(ms=ms[i], launches=cnt[i], work=work[i],
                        unit=KIND_UNITS[i]) for i, k in enumerate(KINDS)}

    def final_forward(self, x, wf, wf_scale, mod_f, out, stream=None):
        _check(load().dit_final_forward(self._h, ptr(x), ptr(wf), ptr(wf_scale),
                                        ptr(mod_f), ptr(out),
                                        stream_handle(stream)),
               "dit_final_forward")


def block_plan(T, D, heads, ffn, mlp_chunk_tokens, attn_chunk_tokens,
               ffn_slice=0) -> BlockPlan:
    return BlockPlan(T, D, heads, ffn, mlp_chunk_tokens, attn_chunk_tokens,
                     ffn_slice)


def block_plan_auto(T, D, heads, ffn, budget_bytes) -> BlockPlan:
    """The largest chunks whose workspace fits ``budget_bytes``."""
    return BlockPlan(T, D, heads, ffn, budget_bytes=budget_bytes)


def block_weights(wqkv, wo, wgate, wup, wdown, scales=None) -> BlockWeights:
    """Pack device weight buffers into the C struct (bf16, or int8 + scales)."""
    w = BlockWeights()
    w.dtype = W_INT8 if scales is not None else W_BF16
    w.wqkv, w.wo, w.wgate, w.wup, w.wdown = (ptr(wqkv), ptr(wo), ptr(wgate),
                                             ptr(wup), ptr(wdown))
    if scales is not None:
        w.wqkv_scale = ptr(scales["wqkv"])
        w.wo_scale = ptr(scales["wo"])
        w.wgate_scale = ptr(scales["wgate"])
        w.wup_scale = ptr(scales["wup"])
        w.wdown_scale = ptr(scales["wdown"])
    return w


def qk_args(q_norm=None, k_norm=None, rope_cos=None, rope_sin=None,
            eps=1e-6) -> QkArgs:
    """Pack device buffers of the Q/K transform into a ``dit_qk_t``."""
    a = QkArgs()
    a.q_norm, a.k_norm = ptr(q_norm), ptr(k_norm)
    a.rope_cos, a.rope_sin = ptr(rope_cos), ptr(rope_sin)
    a.eps = eps
    return a


def lora_prepare(b, rows, rank, ld_b, alpha, row_scale, b_out, ld_out, stream=None):
    """dit_lora_prepare: b_out = bf16(alpha * b / row_scale) (row_scale may be None)."""
    _check(load().dit_lora_prepare(ptr(b), rows, rank, ld_b, alpha, ptr(row_scale),
                                   ptr(b_out), ld_out, stream_handle(stream)),
           "dit_lora_prepare")


def block_lora(**adapters) -> BlockLora:
    """Pack adapters given as name=(a, b_prepared, rank) into a ``BlockLora``."""
    bl = BlockLora()
    for name, (a, b, rank) in adapters.items():
        setattr(bl, name, LoraArgs(ptr(a), ptr(b), rank))
    return bl


def attention_part(q, Tq, ldq, k, ldk, vt, ldvt, T_block, heads, head_dim, o, ldo,
                   o_state, m_state, l_state, ld_state, first, last, dev_status=None,
                   stream=None):
    _check(load().dit_attention_part(ptr(q), Tq, ldq, ptr(k), ldk, ptr(vt), ldvt, T_block,
                                     heads, head_dim, ptr(o), ldo, ptr(o_state),
                                     ptr(m_state), ptr(l_state), ld_state, int(first),
                                     int(last), ptr(dev_status), stream_handle(stream)),
           "dit_attention_part")


def int8_to_bf16(q, n, out, stream=None):
    _check(load().dit_int8_to_bf16(ptr(q), n, ptr(out), stream_handle(stream)),
           "dit_int8_to_bf16")


def modln_cast(x, rows, D, shift, scale, out, stream=None):
    _check(load().dit_modln_cast(ptr(x), rows, D, ptr(shift), ptr(scale),
                                 ptr(out), stream_handle(stream)),
           "dit_modln_cast")


def gemm(args: GemmArgs, dev_status=None, stream=None):
    _check(load().dit_gemm(ctypes.byref(args), ptr(dev_status),
                           stream_handle(stream)), "dit_gemm")


def attention(q, Tq, ldq, k, ldk, vt, ldvt, T, heads, head_dim, o, ldo,
              dev_status=None, stream=None):
    _check(load().dit_attention(ptr(q), Tq, ldq, ptr(k), ldk, ptr(vt), ldvt, T,
                                heads, head_dim, ptr(o), ldo, ptr(dev_status),
                                stream_handle(stream)), "dit_attention")


def attention_split_bytes(head_dim, slots):
    return int(load().dit_attention_split_bytes(head_dim, slots))


def attention_ex(q, Tq, ldq, k, ldk, vt, ldvt, T, heads, head_dim, o, ldo, split_ws=None,
                 split_bytes=0, max_ctas=0, dev_status=None, stream=None):
    _check(load().dit_attention_ex(ptr(q), Tq, ldq, ptr(k), ldk, ptr(vt), ldvt, T, heads,
                                   head_dim, ptr(o), ldo, ptr(split_ws), split_bytes,
                                   max_ctas, ptr(dev_status), stream_handle(stream)),
           "dit_attention_ex")


def attention_schedule(units, n_kv, max_ctas, slots):
    """(n_cta, n_split, items): the persistent attention's work list, each
    item (cta, index, unit, k0, k1, src_slot, dst_slot)."""
    lib = load()
    n_cta, n_split, n = ctypes.c_int(), ctypes.c_int(), ctypes.c_int64()
    _check(lib.dit_attention_schedule(units, n_kv, max_ctas, slots, ctypes.byref(n_cta),
                                      ctypes.byref(n_split), None, 0, ctypes.byref(n)),
           "dit_attention_schedule")
    buf = (ctypes.c_int * (7 * max(n.value, 1)))()
    _check(lib.dit_attention_schedule(units, n_kv, max_ctas, slots, ctypes.byref(n_cta),
                                      ctypes.byref(n_split), buf, n.value, ctypes.byref(n)),
           "dit_attention_schedule")
    items = [tuple(buf[7 * i:7 * i + 7]) for i in range(n.value)]
    return n_cta.value, n_split.value, items


def gemm_split_bytes(slots):
    return int(load().dit_gemm_split_bytes(slots))


def gemm_ex(args: GemmArgs, split_ws=None, split_bytes=0, max_ctas=0, dev_status=None,
            stream=None):
    _check(load().dit_gemm_ex(ctypes.byref(args), ptr(split_ws), split_bytes, max_ctas,
                              ptr(dev_status), stream_handle(stream)), "dit_gemm_ex")
