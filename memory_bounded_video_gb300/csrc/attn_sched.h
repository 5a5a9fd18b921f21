// Work schedule of the persistent attention kernel (host and device code).
//
// A unit is one head and one pair of 128-query tiles, attended against all
// n_kv key tiles in ascending order.  With U units on G CTAs (G = min(U,
// SMs)), CTA c takes the F = U / G whole units c, c + G, ..., c + (F-1) G,
// the order in which a one-unit-per-CTA grid would run them.  The R = U % G
// remaining units would otherwise run as a last, mostly idle wave; instead
// their R * n_kv key tiles, laid out unit by unit, are cut into n_pc equal
// contiguous ranges, one per CTA c < n_pc.  A range covers the end of one
// unit (piece A) and possibly the start of the next (piece B).
//
// A unit cut between CTAs is still computed as one pass over its keys: the
// CTA holding keys [k0, k1) takes over the running max, sum and unnormalised
// fp32 output at k0 from the CTA before it (slot c, flag c) and, if the unit
// goes on past k1, hands them to the CTA after it (slot c + 1), so every
// output element sees the same operations in the same order as in one CTA.
// A piece that starts a unit has no input and is run first; the piece that
// continues a unit at chain position p (p CTAs before it hold earlier keys of
// that unit) is run after p whole units, by which time the piece before it,
// run at position p - 1 on the CTA before, has long finished.  Positions are
// at most F when n_pc <= R * F, since a unit then spans at most F + 1
// ranges, or when every unit is cut into the same q <= F + 1 aligned ranges;
// a larger position is clamped to F (correct, only slower).
//
// When R is small against G (few CTAs could share it), the attention takes
// one whole unit per CTA into the shared part as well (extended split; with
// F = 1 that leaves no whole unit before the pieces): the
// R + G units after the first (F - 1) G are cut into G equal ranges, each
// longer than a unit and shorter than two, so a range is the end of one unit
// (piece A), at most one whole unit, and the start of another (piece B), and
// every CTA carries about the mean load.  A CTA runs its whole units first
// (all CTAs in step, so those sharing a head share its K/V tiles in L2),
// then piece B, the whole unit, and piece A last.  Each cut unit spans two
// ranges, its start piece B of CTA c and its end piece A of CTA c + 1; with
// W whole-unit tiles per CTA, B ends at W + |B| and A starts at W + L - |A|
// on the next CTA (L its range's length), so since |B| + |A| = n_kv <= L no
// CTA waits.  (Running B first instead let the CTAs' whole units drift apart
// by up to a unit and doubled the launch's DRAM reads.)
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define DS_HD __host__ __device__ __forceinline__
#else
#define DS_HD inline
#endif

namespace ds {

// Most CTAs that may share the remainder: one state slot and one flag each.
constexpr int kAttnSplitSlots = 160;


struct AttnItem {
    int u;       // unit: query pair u % n_qpairs, head u / n_qpairs
    int k0, k1;  // key tiles [k0, k1)
    int src;     // slot holding the state at k0 (k0 > 0), else -1
    int dst;     // slot to hand the state at k1 to (k1 < n_kv), else -1
};

struct AttnGrid {
    int units, n_kv, n_cta;
    int full;           // whole units per CTA (split mode); 0: round robin
    int n_pc;           // CTAs sharing the remainder (0: no split)
    int64_t rem_tiles;  // remainder key tiles R * n_kv ((R + G) * n_kv extended)
    int rem_u0;         // first remainder unit, full * n_cta
    int ext;            // extended split: ranges between one and two units long
};

// Grid and split for U units of n_kv key tiles on at most max_cta CTAs;
// slots: state slots available (0: no split; slot c is used by CTAs c - 1
// and c, for 0 < c < n_pc); extend: the extended split may be chosen.
DS_HD AttnGrid attn_grid(int units, int n_kv, int max_cta, int slots, bool extend = false) {
    AttnGrid g{};
    g.units = units;
    g.n_kv = n_kv;
    g.n_cta = units < max_cta ? units : max_cta;
    if (g.n_cta < 1) g.n_cta = 1;
    const int F = units / g.n_cta, R = units % g.n_cta;
    if (R > 0) {
        // Ranges of any length at least n_kv / F keep every unit within
        // F + 1 ranges; ranges of exactly n_kv / q (q of them per unit,
        // aligned to the units) allow q = F + 1.  The more CTAs share the
        // remainder, the shorter the longest range.
        int64_t n1 = g.n_cta;
        if (int64_t(R) * F < n1) n1 = int64_t(R) * F;
        if (int64_t(R) * n_kv < n1) n1 = int64_t(R) * n_kv;
        int64_t q = F + 1;
        if (g.n_cta / R < q) q = g.n_cta / R;
        if (n_kv < q) q = n_kv;
        int64_t n = n1 > R * q ? n1 : R * q;
        // with fewer slots than that, as many contiguous ranges as there are
        // slots (still at most R * F of them)
        if (n > slots) n = n1 < slots ? n1 : slots;
        // split only if the longest range is shorter than a unit (else every
        // remainder unit stays whole, round robin)
        const int64_t longest = n > 0 ? (int64_t(R) * n_kv + n - 1) / n : n_kv;
        if (longest < n_kv) {
            g.full = F;
            g.n_pc = int(n);
            g.rem_tiles = int64_t(R) * n_kv;
            g.rem_u0 = F * g.n_cta;
        }
        // extended split: at least one whole unit per CTA to move into the
        // shared part, a slot per CTA, and a busiest CTA shorter by more than
        // n_kv / 16 key tiles
        const int64_t cur = g.n_pc ? int64_t(F) * n_kv + longest : int64_t(F + 1) * n_kv;
        const int64_t G = g.n_cta;
        const int64_t ext_max = int64_t(F - 1) * n_kv + (int64_t(R + G) * n_kv + G - 1) / G;
        if (extend && F >= 1 && G <= slots && ext_max + n_kv / 16 < cur) {
            g.full = F - 1;
            g.n_pc = g.n_cta;
            g.rem_tiles = int64_t(R + G) * n_kv;
            g.rem_u0 = (F - 1) * g.n_cta;
            g.ext = 1;
        }
    }
    return g;
}

// Multiprocessor counts a plan sizes its hand-off space for (the plan is
// made without a device; a device outside the range may split less).
constexpr int kAttnMinSms = 128, kAttnMaxSms = 160;

// State slots that `units` units of n_kv key tiles may need on any device
// with kAttnMinSms..kAttnMaxSms multiprocessors when at most `cap` slots
// are available (0: none would split).
inline int attn_slots_needed(int units, int n_kv = 1 << 20, int cap = kAttnSplitSlots,
                             bool extend = false) {
    int need = 0;
    for (int sm = kAttnMinSms; sm <= kAttnMaxSms; ++sm) {
        const AttnGrid g = attn_grid(units, n_kv, sm, cap, extend);
        if (g.n_pc > need) need = g.n_pc;
    }
    return need;
}

// The tensor-core GEMM uses the same split with output tiles as units and
// K-steps of 64 as key tiles: a slot holds one CTA's raw fp32 accumulator
// (128 x 256 values), and a plan provides at most 64 slots.
constexpr int kGemmSplitSlots = 64;
constexpr size_t kGemmSlotBytes = size_t(128) * 256 * 4;

// GEMM tiles of an M x N output in either tile shape the GEMM uses: 128 x BN
// on one CTA, or 256 x BN on a cluster pair (BN = 256, or with two B operands
// 128 per operand).
inline int gemm_units(int64_t M, int N, bool two_b, bool pair) {
    const int bm = pair ? 256 : 128;
    const int bn = two_b ? 128 : 256;
    return int((M + bm - 1) / bm) * ((N + bn - 1) / bn);
}

// Hand-off slots a GEMM launch of `units` tiles and `k_steps` K-steps may use
// on a device of 128 to 160 SMs (pair tiles: 64 to 80 pairs, two slots per
// cut, one per CTA), at most kGemmSplitSlots.
inline int gemm_slots_needed(int units, int k_steps, bool pair) {
    if (!pair) return attn_slots_needed(units, k_steps, kGemmSplitSlots);
    int need = 0;
    for (int w = kAttnMinSms / 2; w <= kAttnMaxSms / 2; ++w) {
        const AttnGrid g = attn_grid(units, k_steps, w, kGemmSplitSlots / 2);
        if (2 * g.n_pc > need) need = 2 * g.n_pc;
    }
    return need;
}

// The pieces of CTA c and where piece A goes among its whole units.
struct AttnCta {
    int count;  // items
    int has_a, has_b, pos_a;
    int has_m, m_u;  // extended split: a whole unit between pieces A and B
    AttnItem a, b;
};

DS_HD AttnCta attn_cta(const AttnGrid &g, int c) {
    AttnCta s{};
    if (g.n_pc == 0) {  // round robin: units c, c + G, ... below U
        s.count = c < g.units ? (g.units - c + g.n_cta - 1) / g.n_cta : 0;
        return s;
    }
    s.count = g.full;
    if (c >= g.n_pc) return s;
    const int64_t nkv = g.n_kv;
    const int64_t lo = int64_t(c) * g.rem_tiles / g.n_pc;
    const int64_t hi = int64_t(c + 1) * g.rem_tiles / g.n_pc;
    const int64_t ja = lo / nkv;
    const int64_t end_a = hi < (ja + 1) * nkv ? hi : (ja + 1) * nkv;
    s.has_a = 1;
    s.a.u = int(g.rem_u0 + ja);
    s.a.k0 = int(lo - ja * nkv);
    s.a.k1 = int(end_a - ja * nkv);
    s.a.src = s.a.k0 > 0 ? c : -1;
    s.a.dst = s.a.k1 < nkv ? c + 1 : -1;
    if (hi > (ja + 1) * nkv) {  // the range goes on into the next unit
        int64_t jb = ja + 1;
        if (hi - jb * nkv > nkv) {  // extended: a whole unit, then the next
            s.has_m = 1;
            s.m_u = int(g.rem_u0 + jb);
            ++jb;
        }
        s.has_b = 1;
        s.b.u = int(g.rem_u0 + jb);
        s.b.k0 = 0;
        s.b.k1 = int(hi - jb * nkv);
        s.b.src = -1;
        s.b.dst = s.b.k1 < nkv ? c + 1 : -1;
    }
    if (g.ext) {
        s.pos_a = g.full + s.has_b + s.has_m;  // last
    } else if (s.a.k0 > 0) {
        // chain position: CTAs before c whose ranges hold keys of unit ja;
        // the first is the one whose range holds its key tile 0
        const int64_t first = ((ja * nkv + 1) * g.n_pc - 1) / g.rem_tiles;
        int64_t pos = c - first;
        if (pos > g.full) pos = g.full;
        s.pos_a = int(pos);
    }
    s.count += s.has_a + s.has_b + s.has_m;
    return s;
}

// Item idx (0 <= idx < count) of CTA c, in processing order.
DS_HD AttnItem attn_item(const AttnGrid &g, const AttnCta &s, int c, int idx) {
    int i = idx;
    AttnItem w;
    w.k0 = 0;
    w.k1 = g.n_kv;
    w.src = w.dst = -1;
    if (g.ext) {  // whole units, piece B, the range's whole unit, piece A
        if (i < g.full) {
            w.u = c + i * g.n_cta;
            return w;
        }
        i -= g.full;
        if (s.has_b) {
            if (i == 0) return s.b;
            --i;
        }
        if (s.has_m) {
            if (i == 0) {
                w.u = s.m_u;
                return w;
            }
            --i;
        }
        return s.a;
    }
    if (s.has_b) {
        if (i == 0) return s.b;
        --i;
    }
    if (s.has_a) {
        if (i == s.pos_a) return s.a;
        if (i > s.pos_a) --i;
    }
    w.u = c + i * g.n_cta;
    return w;
}

}  // namespace ds
