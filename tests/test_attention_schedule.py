"""CPU checks of the persistent attention kernel's work list.

The kernel computes its items from the same host/device code that
dit_attention_schedule runs on the host, so these checks cover what the
device executes: every (unit, key tile) once, each cut unit a chain of key
ranges handing state from CTA to CTA through distinct slots, a processing
order in which no CTA waits for a hand-off, and the balance of key tiles
per CTA that removes the partial last wave."""

import random

import pytest

from memory_bounded_video_gb300 import build as dbuild
from memory_bounded_video_gb300 import ditstream as ds


@pytest.fixture(scope="module", autouse=True)
def lib():
    dbuild.build()
    return ds.load()


def grid(units, n_kv, max_cta, slots):
    """(CTAs, CTAs sharing the remainder, whole units each, remainder units,
    whole units each without the extension), restating the documented rule:
    F = U // G whole units per CTA and the R = U % G remaining units cut into
    n ranges, n the larger of min(G, R*F, R*n_kv) (any ranges of at least
    n_kv / F tiles) and R*q, q = min(F + 1, G // R, n_kv) (q aligned ranges
    per unit), or, when that exceeds the slots, min(the first, slots); used
    when the longest range, ceil(R * n_kv / n), is shorter than a unit.  The
    extended split (F >= 1, G <= slots) instead cuts the last R + G units
    into G ranges, leaving F - 1 whole units per CTA, when that makes the
    busiest CTA's load, (F - 1) * n_kv + ceil((R + G) * n_kv / G), shorter
    by more than n_kv // 16 key tiles."""
    G = max(1, min(units, max_cta))
    F, R = divmod(units, G)
    if R == 0:
        return G, 0, F, 0, F
    n1 = min(G, R * F, R * n_kv)
    q = min(F + 1, G // R, n_kv)
    n = max(n1, R * q)
    if n > slots:
        n = min(n1, slots)
    longest = -(-R * n_kv // n) if n > 0 else n_kv
    split = n > 0 and longest < n_kv
    cur = F * n_kv + longest if split else (F + 1) * n_kv
    ext_max = (F - 1) * n_kv + -(-(R + G) * n_kv // G)
    if F >= 1 and G <= slots and ext_max + n_kv // 16 < cur:
        return G, G, F - 1, R + G, F
    if split:
        return G, n, F, R, F
    return G, 0, F, R, F


CASES = [
    (768, 256, 148, 160),    # 32k keys, 8192-query slab, 24 heads (the bench)
    (384, 256, 148, 160),    # 4096-query slab
    (1536, 256, 148, 160),   # 16384-query slab
    (3072, 256, 148, 160),   # all 32768 queries
    (384, 512, 148, 160),    # 64k keys, 4096-query slab
    (200, 256, 148, 160),    # one whole unit per CTA plus a cut remainder
    (256, 32, 148, 160),     # 4096 tokens, 16 heads of 64
    (768, 256, 148, 0),      # no hand-off space: round robin
    (768, 256, 152, 160),
    (100, 256, 148, 160),    # fewer units than multiprocessors
    (50, 8, 7, 8), (23, 5, 7, 8), (40, 3, 7, 8), (1000, 1, 13, 13),
    (97, 64, 13, 13), (13, 4, 13, 13), (5, 9, 13, 13), (29, 2, 9, 9),
    (17, 17, 16, 16), (33, 6, 16, 3),
]
_rng = random.Random(11)
CASES += [(_rng.randint(1, 400), _rng.randint(1, 40), _rng.randint(1, 40), 40)
          for _ in range(60)]
# few units left over (where the extended split applies): U = F * G + R with
# R small against G
_rng2 = random.Random(12)
for _ in range(40):
    _g = _rng2.randint(2, 40)
    CASES.append((_rng2.randint(1, 6) * _g + _rng2.randint(1, max(1, _g // 4)),
                  _rng2.randint(1, 64), _g, 40))


def by_cta(items):
    out = {}
    for c, i, u, k0, k1, src, dst in items:
        out.setdefault(c, []).append((i, u, k0, k1, src, dst))
    for c in out:
        out[c].sort()
        assert [it[0] for it in out[c]] == list(range(len(out[c])))
    return out


@pytest.mark.parametrize("units,n_kv,max_cta,slots", CASES)
def test_schedule_covers_every_key_tile_once_as_chains(units, n_kv, max_cta, slots):
    n_cta, n_split, items = ds.attention_schedule(units, n_kv, max_cta, slots)
    G, n_pc, F, R, _ = grid(units, n_kv, max_cta, slots)
    assert (n_cta, n_split) == (G, n_pc)
    pieces = {}
    for c, i, u, k0, k1, src, dst in items:
        assert 0 <= c < n_cta and 0 <= u < units and 0 <= k0 < k1 <= n_kv
        pieces.setdefault(u, []).append((k0, k1, c, src, dst))
    assert sorted(pieces) == list(range(units))
    written, read = set(), set()
    for u, ps in pieces.items():
        ps.sort()
        assert ps[0][0] == 0 and ps[0][3] == -1          # starts fresh
        assert ps[-1][1] == n_kv and ps[-1][4] == -1     # ends with the output
        for a, b in zip(ps, ps[1:]):
            assert a[1] == b[0]                          # contiguous key ranges
            assert a[4] == b[3] != -1                    # handed through one slot
            assert b[2] == a[2] + 1 == a[4]              # to the next CTA, slot c
            assert 0 < a[4] < max(n_split, 1)
            written.add(a[4])
            read.add(b[3])
    assert len(written) == len(read) == sum(len(ps) - 1 for ps in pieces.values())
    if n_split == 0:  # round robin: units c, c + G, ... whole
        for c, its in by_cta(items).items():
            assert [it[1] for it in its] == list(range(c, units, n_cta))
            assert all(it[2:] == (0, n_kv, -1, -1) for it in its)


@pytest.mark.parametrize("units,n_kv,max_cta,slots", CASES)
def test_schedule_never_waits_and_balances_key_tiles(units, n_kv, max_cta, slots):
    """Every CTA runs its items back to back, an item taking its key tiles
    in time; an item that continues a unit must not start before the piece
    before it has ended on the CTA before."""
    n_cta, n_split, items = ds.attention_schedule(units, n_kv, max_cta, slots)
    G, n_pc, F, R, F0 = grid(units, n_kv, max_cta, slots)
    per = by_cta(items)
    start, end = {}, {}
    for c, its in per.items():
        t = 0
        for i, u, k0, k1, src, dst in its:
            start[(u, k0)] = t
            t += k1 - k0
            end[(u, k1)] = t
    for (u, k0), t in start.items():
        if k0 > 0:
            assert end[(u, k0)] <= t, (u, k0)
    loads = [sum(k1 - k0 for _, _, k0, k1, _, _ in its) for its in per.values()]
    assert sum(loads) == units * n_kv
    if n_pc:
        assert max(loads) == F * n_kv + -(-R * n_kv // n_pc)
        assert max(loads) < (F0 + 1) * n_kv  # shorter than with a last wave
    else:
        assert max(loads) == -(-units // n_cta) * n_kv


def test_schedule_of_the_32k_token_slab():
    # 8192-query slabs of 24 heads against 32768 keys on 148 SMs: 768 units,
    # 5.19 waves.  One CTA per unit needs 6 waves (1536 key tiles on the
    # busiest SM); the split needs 1332, the mean being 1328.4.
    n_cta, n_split, items = ds.attention_schedule(768, 256, 148, 160)
    assert (n_cta, n_split) == (148, 140)
    loads = {}
    for c, i, u, k0, k1, src, dst in items:
        loads[c] = loads.get(c, 0) + k1 - k0
    assert max(loads.values()) == 1332 and min(loads.values()) == 1280


def test_schedule_of_the_32k_token_slab_on_152_sms():
    # the same slab on 152 SMs: 768 units are 5.05 waves, and the 8 left over
    # could be cut into at most 48 ranges (1323 key tiles on the busiest SM
    # against a mean of 1293.5); the extended split cuts the last 160 units
    # into 152 ranges of 269-270 key tiles after 4 whole units per CTA
    n_cta, n_split, items = ds.attention_schedule(768, 256, 152, 160)
    assert (n_cta, n_split) == (152, 152)
    loads, count = {}, {}
    for c, i, u, k0, k1, src, dst in items:
        loads[c] = loads.get(c, 0) + k1 - k0
        count[c] = count.get(c, 0) + 1
    assert max(loads.values()) == 1294 and min(loads.values()) == 1293
    assert max(count.values()) <= 7
    # without the extension (as the GEMMs split): 48 ranges, 1323 tiles
    assert ds.attention_schedule(768, 256, 152, 151)[1] == 48


def test_plan_workspace_holds_the_hand_off_space():
    # a 8192-query slab of 24 heads needs hand-off slots
    big = ds.block_plan(32768, 3072, 24, 8192, 8192, 8192)
    small = ds.block_plan(4096, 1024, 16, 2816, 4096, 4096)
    slots = max(grid(768, 1 << 20, sm, 160)[1] for sm in range(128, 161))
    assert slots == 160
    base = 1024 + 2 * 32768 * 3072 + 2 * 3072 * 32768
    attn = base + 4 * 8192 * 3072 + slots * 256 * 130 * 4
    mlp = base + 2 * 8192 * 3072 + 2 * 8192 * 8192
    # plus the GEMMs' hand-off state: 8192-row chunks of 3072 outputs are 768
    # tiles (5.05 waves on 152 SMs: 8 left over, each cut into 6 K ranges);
    # the K/V projection's 1536 tiles (10.1 waves) would use 152 slots and
    # get the 64 there are
    from test_abi import gemm_region
    g = gemm_region(32768, 3072, 8192, 8192, 8192, 8192)
    assert g == 64 * 128 * 1024
    assert ds.attention_schedule(768, 48, 152, 64)[1] == 48
    assert ds.attention_schedule(1536, 48, 152, 64)[1] == 64
    assert big.workspace_bytes() == max(attn, mlp) + g
    # the 4096-token block: 256 units, one whole unit per CTA and a remainder,
    # split by the extended rule on every device size (160 slots of 64-wide
    # state); its attention phase stays below the MLP phase, which sets the
    # workspace
    small_slots = max(grid(256, 1 << 20, sm, 160)[1] for sm in range(128, 161))
    assert small_slots == 160
    small_attn = (1024 + 4 * 4096 * 1024 + 4 * 4096 * 1024 + small_slots * 256 * 66 * 4)
    small_mlp = 1024 + 4 * 4096 * 1024 + 2 * 4096 * 1024 + 2 * 4096 * 2816
    assert small_attn < small_mlp
    assert small.workspace_bytes() == (small_mlp
                                       + gemm_region(4096, 1024, 2816, 4096, 4096, 2816))


def test_split_bytes_and_arguments(lib):
    assert ds.attention_split_bytes(128, 160) == 1024 + 160 * 256 * 130 * 4
    assert ds.attention_split_bytes(64, 1) == 1024 + 256 * 66 * 4
    assert ds.attention_split_bytes(96, 4) == 0
    assert ds.attention_split_bytes(128, 161) == 0
    for bad in ((0, 4, 4, 4), (4, 0, 4, 4), (4, 4, 0, 4), (4, 4, 4, -1)):
        with pytest.raises(ds.DitError) as e:
            ds.attention_schedule(*bad)
        assert e.value.status == ds.ERR_INVALID_ARG
    # argument checks before any launch: head_dim, alignment, too small
    with pytest.raises(ds.DitError) as e:
        ds.attention_ex(16, 256, 1024, 16, 1024, 16, 256, 256, 8, 96, 16, 1024)
    assert e.value.status == ds.ERR_INVALID_ARG
    with pytest.raises(ds.DitError) as e:
        ds.attention_ex(16, 256, 1024, 16, 1024, 16, 256, 256, 8, 128, 16, 1024,
                        split_ws=8, split_bytes=4096)
    assert e.value.status == ds.ERR_ALIGN
    with pytest.raises(ds.DitError) as e:
        ds.attention_ex(16, 256, 1024, 16, 1024, 16, 256, 256, 8, 128, 16, 1024,
                        split_ws=16, split_bytes=512)
    assert e.value.status == ds.ERR_WORKSPACE_TOO_SMALL
