"""CPU checks of the C ABI: the library loads, exports what the header
declares, validates arguments and lays out its workspace as documented.
No kernel is launched (no GPU needed)."""

import ctypes
import os
import re

import pytest

from memory_bounded_video_gb300 import build as dbuild
from memory_bounded_video_gb300 import ditstream as ds

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ditstream.h")


@pytest.fixture(scope="module")
def lib():
    dbuild.build()
    return ds.load()


def header_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^DIT_API [^(]*?\b(dit_\w+)\(", src, re.M)))


def header_defines():
    src = open(HEADER).read()
    return {k: int(v) for k, v in
            re.findall(r"#define (DIT\w+) \(?(-?\d+)\)?", src)}


def test_every_declared_symbol_is_exported(lib):
    declared = header_functions()
    assert len(declared) >= 15
    assert sorted(ds.SYMBOLS) == declared
    for name in declared:
        assert hasattr(lib, name), name


def test_binding_constants_match_header():
    d = header_defines()
    pairs = dict(DIT_OK=ds.OK, DIT_ERR_INVALID_ARG=ds.ERR_INVALID_ARG,
                 DIT_ERR_CHUNK_ALIGN=ds.ERR_CHUNK_ALIGN, DIT_ERR_ALIGN=ds.ERR_ALIGN,
                 DIT_ERR_NO_WORKSPACE=ds.ERR_NO_WORKSPACE,
                 DIT_ERR_WORKSPACE_TOO_SMALL=ds.ERR_WORKSPACE_TOO_SMALL,
                 DIT_ERR_CUDA=ds.ERR_CUDA, DIT_ERR_TIMEOUT=ds.ERR_TIMEOUT,
                 DIT_ERR_UNSUPPORTED_ARCH=ds.ERR_UNSUPPORTED_ARCH,
                 DIT_W_BF16=ds.W_BF16, DIT_W_INT8=ds.W_INT8,
                 DIT_EPI_STORE_BF16=ds.EPI_STORE_BF16,
                 DIT_EPI_STORE_F32=ds.EPI_STORE_F32, DIT_EPI_KV=ds.EPI_KV,
                 DIT_EPI_RESID=ds.EPI_RESID, DIT_EPI_SWIGLU=ds.EPI_SWIGLU,
                 DIT_EPI_DOWN=ds.EPI_DOWN, DIT_NUM_KINDS=len(ds.KINDS),
                 DIT_K_MODLN=ds.KINDS.index("modln"),
                 DIT_K_ATTENTION=ds.KINDS.index("attention"),
                 DIT_K_FINAL=ds.KINDS.index("final"),
                 DIT_K_LORA_U=ds.KINDS.index("lora_u"),
                 DIT_K_EXPAND=ds.KINDS.index("expand"),
                 DIT_LORA_MAX_RANK=256,
                 DITSTREAM_ABI_VERSION=None)
    for k, v in pairs.items():
        if v is not None:
            assert d[k] == v, k


def test_struct_layouts_match_header():
    # field order and count of the two POD structs
    src = open(HEADER).read()
    body = re.search(r"typedef struct \{([^}]*)\} dit_gemm_args_t;", src).group(1)
    fields = re.findall(r"\b(\w+);", re.sub(r"/\*.*?\*/", "", body, flags=re.S))
    assert fields == [f for f, _ in ds.GemmArgs._fields_]
    body = re.search(r"typedef struct \{([^}]*)\} dit_block_weights_t;", src).group(1)
    fields = re.findall(r"\b(\w+);", body)
    assert fields == [f for f, _ in ds.BlockWeights._fields_]
    body = re.search(r"typedef struct \{([^}]*)\} dit_lora_t;", src).group(1)
    assert re.findall(r"\b(\w+);", body) == [f for f, _ in ds.LoraArgs._fields_]
    body = re.search(r"typedef struct \{([^}]*)\} dit_block_lora_t;", src).group(1)
    names = re.search(r"dit_lora_t ([\w, ]+);", body).group(1).replace(" ", "").split(",")
    assert names == [f for f, _ in ds.BlockLora._fields_]
    body = re.search(r"typedef struct \{([^}]*)\} dit_qk_t;", src).group(1)
    fields = re.findall(r"\b(\w+);", re.sub(r"/\*.*?\*/", "", body, flags=re.S))
    assert fields == [f for f, _ in ds.QkArgs._fields_]


def test_status_strings(lib):
    assert ds.abi_version() == header_defines()["DITSTREAM_ABI_VERSION"]
    for s in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        assert ds.status_string(s) and ds.status_string(s) != "unknown status"
    assert ds.status_string(-99) == "unknown status"


@pytest.mark.parametrize("args,status", [
    ((0, 256, 4, 704, 128, 128), ds.ERR_INVALID_ARG),       # T = 0
    ((512, 250, 4, 704, 128, 128), ds.ERR_INVALID_ARG),     # D % 128
    ((512, 320, 5, 704, 128, 128), ds.ERR_INVALID_ARG),     # D % 128 with d = 64
    ((512, 256, 3, 704, 128, 128), ds.ERR_INVALID_ARG),     # D % heads
    ((512, 256, 8, 704, 128, 128), ds.ERR_INVALID_ARG),     # d = 32
    ((512, 256, 4, 700, 128, 128), ds.ERR_INVALID_ARG),     # ffn % 64
    ((512, 256, 4, 704, 100, 128), ds.ERR_CHUNK_ALIGN),
    ((512, 256, 4, 704, 128, 64), ds.ERR_CHUNK_ALIGN),
    ((512, 256, 4, 704, -128, 128), ds.ERR_INVALID_ARG),
])
def test_plan_rejects_bad_arguments(lib, args, status):
    h = ctypes.c_void_p()
    assert lib.dit_block_plan(*args, ctypes.byref(h)) == status
    assert not h.value


def test_plan_ex_rejects_bad_ffn_slice(lib):
    h = ctypes.c_void_p()
    assert lib.dit_block_plan_ex(512, 256, 4, 704, 128, 128, 96,
                                 ctypes.byref(h)) == ds.ERR_INVALID_ARG
    assert lib.dit_block_plan_ex(512, 256, 4, 704, 128, 128, 768,
                                 ctypes.byref(h)) == ds.ERR_INVALID_ARG


def rup(v, a=1024):
    return (v + a - 1) // a * a


def split_region(ca, H, hd):
    """Bytes of the attention hand-off state: slots for the most CTAs that
    share a slab's partial last wave on a 128..160-multiprocessor device,
    256 rows x (head_dim + 2) fp32 values each (the rule is restated in
    test_attention_schedule.grid)."""
    from test_attention_schedule import grid
    units = -(-ca // 256) * H
    slots = max(grid(units, 1 << 20, sm, 160)[1] for sm in range(128, 161))
    return slots * 256 * (hd + 2) * 4


def gemm_region(T, D, F, cm, ca, fs):
    """Bytes of the GEMMs' hand-off state: 128 KiB slots for the most CTAs
    that any of the plan's GEMM launches (K/V, Q, O, gate/up, down at full
    and ragged chunk / slice sizes, in 128 x BN one-CTA tiles or 256 x BN
    pair tiles, two slots per cut pair tile) would cut its last wave over on
    a 128..160-SM device, at most 64."""
    from test_attention_schedule import grid

    def units(M, N, two_b, pair):
        bm = 256 if pair else 128
        bn = 128 if two_b else 256
        return -(-M // bm) * -(-N // bn)

    slots = 0
    def need(M, N, K, two_b):
        nonlocal slots
        if M <= 0 or N <= 0 or K <= 0:
            return
        u = units(M, N, two_b, False)
        slots = max([slots] + [grid(u, K // 64, sm, 64)[1] for sm in range(128, 161)])
        u = units(M, N, two_b, True)
        slots = max([slots] + [2 * grid(u, K // 64, w, 32)[1] for w in range(64, 81)])
    for M in (ca, T % ca):
        need(M, 2 * D, D, False)
        need(M, D, D, False)
    for M in (cm, T % cm):
        for fw in (fs, F % fs):
            need(M, fw, D, True)
            need(M, D, fw, False)
    return slots * 128 * 1024


def expected_workspace_offload(T, D, H, F, cm, ca, fs, kvb):
    """dit_block_workspace_bytes with K/V offload: the two ring slots and the
    carried attention state replace K and V^T."""
    cm = T if cm == 0 or cm >= T else cm
    ca = T if ca == 0 or ca >= T else ca
    fs = fs or F
    phase = 1024 + 2 * rup(4 * kvb * D)
    attn = rup(rup(phase + 2 * ca * D) + 2 * ca * D)
    attn = rup(rup(rup(attn + 4 * ca * D) + 4 * ca * H) + 4 * ca * H)
    attn = rup(attn + split_region(ca, H, D // H))
    mlp = rup(rup(phase + 2 * cm * D) + 2 * cm * fs)
    if fs < F:
        mlp = rup(mlp + 4 * cm * D)
    g = gemm_region(T, D, F, cm, ca, fs)
    return rup(max(attn, mlp) + g) if g else max(attn, mlp)


def expected_workspace(T, D, F, cm, ca, fs, R=0, H=24):
    """The layout documented for dit_block_workspace_bytes (and, with a
    LoRA rank R, dit_block_plan_set_lora_rank), restated."""
    cm = T if cm == 0 or cm >= T else cm
    ca = T if ca == 0 or ca >= T else ca
    fs = fs or F
    k = 1024
    vt = rup(k + 2 * T * D)
    phase = rup(vt + 2 * D * rup(T, 128))
    attn = rup(rup(phase + 2 * ca * D) + 2 * ca * D)
    mlp = rup(rup(phase + 2 * cm * D) + 2 * cm * fs)
    if fs < F:
        mlp = rup(mlp + 4 * cm * D)
    if R:
        attn = rup(rup(attn + 2 * ca * R) + 2 * ca * R)    # u of Q/K/V and O
        mlp = rup(rup(rup(mlp + 2 * cm * R) + 2 * cm * R) + 2 * cm * R)  # gate, up, down
        if fs < F:
            mlp = rup(mlp + 4 * cm * R)                     # down's fp32 carry
    attn = rup(attn + split_region(ca, H, D // H))          # attention hand-off state
    g = gemm_region(T, D, F, cm, ca, fs)                    # GEMM hand-off state
    return rup(max(attn, mlp) + g) if g else max(attn, mlp)


@pytest.mark.parametrize("cfg", [
    (512, 256, 4, 704, 128, 128, 0),
    (4096, 1024, 16, 2816, 0, 512, 0),
    (16384, 3072, 24, 8192, 8192, 0, 0),
    (65536, 3072, 24, 8192, 4096, 4096, 2048),
    (1000, 1024, 8, 2816, 256, 384, 1024),
])
def test_workspace_layout_and_info(lib, cfg):
    T, D, H, F, cm, ca, fs = cfg
    p = ds.block_plan(T, D, H, F, cm, ca, fs)
    assert p.workspace_bytes() == expected_workspace(T, D, F, cm, ca, fs, H=H)
    info = p.info()
    assert info["T"] == T and info["D"] == D and info["heads"] == H
    assert info["mlp_chunk"] == (T if cm == 0 or cm >= T else cm)
    assert info["attn_chunk"] == (T if ca == 0 or ca >= T else ca)
    assert info["ffn_slice"] == (fs or F)


@pytest.mark.parametrize("cfg", [
    (512, 256, 4, 704, 128, 128, 0, 32),
    (1000, 1024, 8, 2816, 256, 384, 1024, 64),
    (32768, 3072, 24, 8192, 8192, 8192, 0, 256),
])
def test_workspace_with_lora_rank(lib, cfg):
    T, D, H, F, cm, ca, fs, R = cfg
    p = ds.block_plan(T, D, H, F, cm, ca, fs)
    p.set_lora_rank(R)
    assert p.workspace_bytes() == expected_workspace(T, D, F, cm, ca, fs, R, H=H)
    p.set_lora_rank(0)
    assert p.workspace_bytes() == expected_workspace(T, D, F, cm, ca, fs, H=H)


def test_lora_rank_rules(lib):
    p = ds.block_plan(512, 256, 4, 704, 128, 128)
    for bad in (-32, 16, 48, 288):
        with pytest.raises(ds.DitError) as e:
            p.set_lora_rank(bad)
        assert e.value.status == ds.ERR_INVALID_ARG
    assert lib.dit_block_plan_set_lora_rank(None, 32) == ds.ERR_INVALID_ARG


def test_lora_arguments_validated_before_launch(lib):
    base = dict(mode=ds.EPI_STORE_F32, M=128, N=256, K=64, a=16, lda=64, b0=16,
                ldb=64, out=16, ldo=256)
    lo = dict(lora_u0=16, lora_ldu0=64, lora_l0=16, lora_ldl0=64, lora_rank0=64)
    cases = [
        (dict(lora_u0=16), ds.ERR_INVALID_ARG),                       # l missing
        (dict(lora_l0=16, lora_rank0=64, lora_ldl0=64), ds.ERR_INVALID_ARG),
        ({**lo, "lora_rank0": 12}, ds.ERR_INVALID_ARG),               # rank % 8
        ({**lo, "lora_rank0": 264, "lora_ldu0": 264, "lora_ldl0": 264}, ds.ERR_INVALID_ARG),
        ({**lo, "lora_ldu0": 32}, ds.ERR_INVALID_ARG),                 # ldu < rank
        ({**lo, "lora_ldl0": 68}, ds.ERR_INVALID_ARG),                 # stride % 16 B
        ({**lo, "lora_u0": 24}, ds.ERR_ALIGN),
        ({**lo, "lora_l1": 16, "lora_u1": 16, "lora_rank1": 64, "lora_ldu1": 64,
          "lora_ldl1": 64}, ds.ERR_INVALID_ARG),                      # half 1: SWIGLU only
        (dict(mode=ds.EPI_STORE_BF16, ldo=256, out=16, acc_load=1), ds.ERR_ALIGN),  # no acc
    ]
    for kw, want in cases:
        g = ds.GemmArgs(**{**base, **kw})
        assert lib.dit_gemm(ctypes.byref(g), None, None) == want, kw
    # dit_lora_prepare
    assert lib.dit_lora_prepare(16, 100, 0, 64, 1.0, None, 16, 64, None) == ds.ERR_INVALID_ARG
    assert lib.dit_lora_prepare(16, 100, 64, 60, 1.0, None, 16, 64, None) == ds.ERR_INVALID_ARG
    assert lib.dit_lora_prepare(24, 100, 64, 64, 1.0, None, 16, 64, None) == ds.ERR_ALIGN


def test_forward_ex_validates_adapters_before_launch(lib):
    # no workspace is bound, so even a valid call stops before any launch
    p = ds.block_plan(512, 256, 4, 704, 128, 128)
    p.set_lora_rank(64)
    w = ds.block_weights(16, 16, 16, 16, 16)
    for kw, want in [(dict(o=(16, 16, 48)), ds.ERR_INVALID_ARG),     # rank % 32
                     (dict(up=(16, 16, 128)), ds.ERR_INVALID_ARG),   # above the plan's
                     (dict(down=(8, 16, 32)), ds.ERR_ALIGN),
                     (dict(qkv=(16, 16, 64), gate=(16, 16, 32)), ds.ERR_NO_WORKSPACE),
                     (dict(qkv=(16, None, 64)), ds.ERR_NO_WORKSPACE)]:  # absent adapter
        with pytest.raises(ds.DitError) as e:
            p.forward(16, w, 16, lora=ds.block_lora(**kw))
        assert e.value.status == want, kw


@pytest.mark.parametrize("D,F", [(256, 704), (3072, 8192), (1024, 1024)])
def test_weight_scratch_size_and_binding(lib, D, F):
    p = ds.block_plan(512, D, D // 64, F, 128, 128)
    need = 2 * max(4 * D * D, 3 * D * F)
    assert p.weight_scratch_bytes() == need
    assert lib.dit_block_bind_weight_scratch(p.handle, 256 + 16, need) == ds.ERR_ALIGN
    assert lib.dit_block_bind_weight_scratch(p.handle, 256, need - 1) == \
        ds.ERR_WORKSPACE_TOO_SMALL
    assert lib.dit_block_bind_weight_scratch(p.handle, 256, need) == ds.OK
    assert lib.dit_block_bind_weight_scratch(p.handle, None, 0) == ds.OK  # unbind
    assert lib.dit_int8_to_bf16(16, 24, 16, None) == ds.ERR_INVALID_ARG   # n % 16
    assert lib.dit_int8_to_bf16(8, 32, 16, None) == ds.ERR_ALIGN


@pytest.mark.parametrize("cfg", [
    (65536, 3072, 24, 8192, 4096, 4096, 2048, 4096),
    (1000, 256, 4, 704, 128, 384, 0, 256),
    (32768, 3072, 24, 8192, 8192, 8192, 0, 8192),
])
def test_kv_offload_workspace_does_not_grow_with_T(lib, cfg):
    T, D, H, F, cm, ca, fs, kvb = cfg
    p = ds.block_plan(T, D, H, F, cm, ca, fs)
    p.set_kv_offload(kvb)
    assert p.workspace_bytes() == expected_workspace_offload(T, D, H, F, cm, ca, fs, kvb)
    assert p.kv_host_bytes() == 2 * T * D + 2 * D * kvb * ((T + kvb - 1) // kvb)
    q = ds.block_plan(2 * T, D, H, F, cm, ca, fs)
    q.set_kv_offload(kvb)
    assert q.workspace_bytes() == p.workspace_bytes()   # independent of T
    if T == 65536:  # below the resident K/V floor alone (4*T*D = 768 MiB)
        assert p.workspace_bytes() < 4 * T * D / 3


def test_kv_offload_rules(lib):
    p = ds.block_plan(1000, 256, 4, 704, 128, 128)
    with pytest.raises(ds.DitError) as e:
        p.set_kv_offload(100)
    assert e.value.status == ds.ERR_CHUNK_ALIGN
    p.set_kv_offload(256)
    assert lib.dit_block_bind_kv_host(p.handle, None, 1 << 20) == ds.ERR_INVALID_ARG
    assert lib.dit_block_bind_kv_host(p.handle, 8, 1 << 20) == ds.ERR_ALIGN
    assert lib.dit_block_bind_kv_host(p.handle, 16, 100) == ds.ERR_WORKSPACE_TOO_SMALL
    # an offloading plan without its host buffer fails closed
    w = ds.block_weights(16, 16, 16, 16, 16)
    with pytest.raises(ds.DitError) as e:
        p.forward(16, w, 16)
    assert e.value.status == ds.ERR_NO_WORKSPACE


def test_workspace_beyond_kv_floor_is_bounded_by_chunk():
    # 4*T*D (K and V) grows with T; the rest depends on the chunks only.
    D, F = 3072, 8192
    rest = []
    for T in (8192, 16384, 32768, 65536):
        total = expected_workspace(T, D, F, 4096, 4096, 2048)
        rest.append(total - 4 * T * D)
    assert max(rest) - min(rest) <= 4 * 1024
    assert ds.block_plan(65536, D, 24, F, 4096, 4096, 2048).workspace_bytes() \
        - 4 * 65536 * D == rest[-1]


def test_forward_without_workspace_fails_closed(lib):
    p = ds.block_plan(512, 256, 4, 704, 128, 128)
    w = ds.block_weights(16, 16, 16, 16, 16)
    with pytest.raises(ds.DitError) as e:
        p.forward(None, w, 16)
    assert e.value.status == ds.ERR_INVALID_ARG  # null x
    with pytest.raises(ds.DitError) as e:
        p.forward(16, w, 16)
    assert e.value.status == ds.ERR_NO_WORKSPACE


def test_stage_entry_points_validate_before_launch(lib):
    # misaligned or invalid arguments are rejected on the host
    assert lib.dit_modln_cast(8, 4, 256, 16, 16, 16, None) == ds.ERR_ALIGN
    assert lib.dit_modln_cast(16, 4, 200, 16, 16, 16, None) == ds.ERR_INVALID_ARG
    g = ds.GemmArgs(mode=ds.EPI_STORE_BF16, M=128, N=100, K=64, a=16, lda=64,
                    b0=16, ldb=64, out=16, ldo=128)
    assert lib.dit_gemm(ctypes.byref(g), None, None) == ds.ERR_INVALID_ARG
    g.N, g.mode = 128, 99
    assert lib.dit_gemm(ctypes.byref(g), None, None) == ds.ERR_INVALID_ARG
    assert lib.dit_attention(16, 128, 256, 16, 256, 16, 512, 512, 4, 32, 16,
                             256, None, None) == ds.ERR_INVALID_ARG
    assert lib.dit_attention(16, 128, 256, 16, 256, 16, 500, 512, 4, 64, 16,
                             256, None, None) == ds.ERR_INVALID_ARG


def test_qk_transform_arguments_validated_before_launch(lib):
    # every call below is rejected on the host: nothing is launched
    base = dict(mode=ds.EPI_STORE_BF16, M=128, N=256, K=64, a=16, lda=64, b0=16,
                ldb=64, out=16, ldo=256, head_dim=128, qk_eps=1e-6)
    cases = [
        (dict(mode=ds.EPI_RESID, x=16, ldx=256, gate=16, qk_norm=16), ds.ERR_INVALID_ARG),
        (dict(qk_norm=16, head_dim=96), ds.ERR_INVALID_ARG),
        (dict(qk_norm=16, N=192, ldo=192), ds.ERR_INVALID_ARG),  # N % d
        (dict(rope_cos=16), ds.ERR_INVALID_ARG),                  # sin missing
        (dict(rope_sin=16), ds.ERR_INVALID_ARG),
        (dict(qk_norm=16, qk_eps=0.0), ds.ERR_INVALID_ARG),
        (dict(qk_norm=16, rope_pos0=-1), ds.ERR_INVALID_ARG),
        (dict(qk_norm=8), ds.ERR_ALIGN),
        (dict(rope_cos=16, rope_sin=24), ds.ERR_ALIGN),
        (dict(mode=ds.EPI_KV, out2=16, ldo2=4096, split_n=192, N=384, ldo=192,
              rope_cos=16, rope_sin=16), ds.ERR_INVALID_ARG),      # split_n % d
    ]
    for kw, want in cases:
        g = ds.GemmArgs(**{**base, **kw})
        assert lib.dit_gemm(ctypes.byref(g), None, None) == want, kw


def test_forward_qk_validates_before_launch(lib):
    # no workspace is bound, so even a valid call stops before any launch
    p = ds.block_plan(512, 256, 4, 704, 128, 128)
    w = ds.block_weights(16, 16, 16, 16, 16)
    for qk, want in [(ds.qk_args(rope_cos=16), ds.ERR_INVALID_ARG),
                     (ds.qk_args(q_norm=16, eps=0.0), ds.ERR_INVALID_ARG),
                     (ds.qk_args(k_norm=8), ds.ERR_ALIGN),
                     (ds.qk_args(q_norm=16), ds.ERR_NO_WORKSPACE)]:
        with pytest.raises(ds.DitError) as e:
            p.forward(16, w, 16, qk=qk)
        assert e.value.status == want


def test_plan_auto_picks_largest_chunks_that_fit(lib):
    T, D, H, F = 65536, 3072, 24, 8192
    floor = 4 * T * D
    # unlimited budget: one slab of all tokens, unsliced FFN
    p = ds.block_plan_auto(T, D, H, F, 1 << 40)
    info = p.info()
    assert info["attn_chunk"] == T and info["mlp_chunk"] == T
    assert info["ffn_slice"] == F
    prev = None
    for extra_mib in (40, 88, 200, 500, 1500):
        budget = floor + 2 * 1024 * 1024 + extra_mib * 2**20
        p = ds.block_plan_auto(T, D, H, F, budget)
        info = p.info()
        assert p.workspace_bytes() <= budget
        # the chosen chunks are maximal: the next larger attention chunk
        # would not fit
        ca = info["attn_chunk"]
        if ca < T:
            bigger = ds.block_plan(T, D, H, F, 128, ca + 128)
            assert bigger.workspace_bytes() > budget
        if prev is not None:
            assert info["attn_chunk"] >= prev["attn_chunk"]
            assert info["mlp_chunk"] >= prev["mlp_chunk"]
        prev = info


def test_plan_auto_rejects_budgets_below_the_kv_floor(lib):
    T, D = 8192, 1024
    h = ctypes.c_void_p()
    st = lib.dit_block_plan_auto(T, D, 16, 2816, 4 * T * D, ctypes.byref(h))
    assert st == ds.ERR_WORKSPACE_TOO_SMALL and not h.value
    st = lib.dit_block_plan_auto(T, 1000, 16, 2816, 1 << 40, ctypes.byref(h))
    assert st == ds.ERR_INVALID_ARG


def test_plan_auto_slices_the_ffn_only_when_needed(lib):
    T, D, H, F = 16384, 3072, 24, 8192
    # enough for 4096-token attention slabs but not for a 4096-token MLP
    # chunk with the full FFN intermediate
    attn_4096 = ds.block_plan(T, D, H, F, 128, 4096).workspace_bytes()
    p = ds.block_plan_auto(T, D, H, F, attn_4096)
    info = p.info()
    assert p.workspace_bytes() <= attn_4096
    if info["ffn_slice"] < F:
        unsliced = ds.block_plan(T, D, H, F, info["mlp_chunk"], info["attn_chunk"])
        assert unsliced.workspace_bytes() > attn_4096


def test_final_forward_validates_before_launch(lib):
    # argument and alignment errors come back before any CUDA call (the
    # pointers below are never dereferenced)
    h = ctypes.c_void_p()
    assert lib.dit_block_plan(1000, 256, 4, 704, 0, 0, ctypes.byref(h)) == ds.OK
    try:
        ok_ptr = ctypes.c_void_p(0x10000)
        bad_ptr = ctypes.c_void_p(0x10004)  # not 16-byte aligned
        assert lib.dit_final_forward(None, ok_ptr, ok_ptr, None, ok_ptr, ok_ptr,
                                     None) == ds.ERR_INVALID_ARG
        for i in range(4):  # x, wf, mod_f, out missing in turn
            args = [ok_ptr, ok_ptr, None, ok_ptr, ok_ptr]
            args[[0, 1, 3, 4][i]] = None
            assert lib.dit_final_forward(h, *args, None) == ds.ERR_INVALID_ARG
        for i in range(4):  # x, wf, mod_f, out misaligned in turn
            args = [ok_ptr, ok_ptr, None, ok_ptr, ok_ptr]
            args[[0, 1, 3, 4][i]] = bad_ptr
            assert lib.dit_final_forward(h, *args, None) == ds.ERR_ALIGN
    finally:
        lib.dit_block_plan_destroy(h)
