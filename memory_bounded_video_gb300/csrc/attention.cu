// Flash-style attention of one query slab against the full K/V on sm_103a.
//
// "LayerStream: H3 Chunking" ("How the slicing works"): every query needs
// every key and value, so pass two attends each query slice to the K and V
// kept for all tokens.  Per CTA: one head and two 128-query tiles (A, B);
// the key loop runs over all T keys in tiles of 128, always in ascending
// order, so a query's output does not depend on the slab it belongs to.
//
// Persistent: one CTA per SM works through a list of (unit, key range)
// items (attn_sched.h), where a unit is one head and one pair of query tiles;
// the last, partial wave of units (with one more whole unit per CTA when few
// are left over) is cut into key ranges shared by the CTAs, handing the
// softmax state from CTA to CTA, so that every SM gets about the same number
// of key tiles.
//
// Roles (384 threads):
//   warp 0        TMA: per item both Q tiles, then K_j and V_j^T tiles
//                 through one shared ring (K_0, V_0, K_1, V_1, ...)
//   warp 1        TMEM owner; one lane issues the tcgen05.mma:
//                   S_X  = Q_X K_j^T  (M=128, N=128, K=d)     -> TMEM S[X]
//                   O_X += P_X V_j    (M=128, N=d,   K=128)   -> TMEM O[X]
//                 (P_X from TMEM, aliasing S_X; V_j from shared memory)
//                 in the order S_A S_B | PV_A S_A' PV_B S_B' | ... so the
//                 tensor core works on one tile while the other's softmax runs
//   warps 4..7    softmax of tile A, one query row per thread
//   warps 8..11   softmax of tile B
// Softmax per key tile: the S row into registers (one tensor-memory load
// latency for the whole tile), P = exp2(S*log2e/sqrt(d) - m) against the
// running reference max m as bf16 written back into the first 64 columns of
// the same TMEM region (P is the A operand of the PV MMA, read straight from
// tensor memory, so P never touches shared memory), the running sum l.  The
// reference max m is only moved when the tile max exceeds it by more than 8
// (log2 units); then the row of O is rescaled in TMEM and the tile's P
// recomputed.  The tile max is taken only where it can matter: a row whose
// probabilities sum to at most 2^8 has no score above m + 8.  Otherwise P may
// reach 2^8, which bf16 and the fp32 accumulator represent without loss of
// range; O / l is unchanged in exact arithmetic.
//
// V arrives transposed (V^T [H*d, T], written so by the K/V projection's
// epilogue), which makes both MMAs K-major in both operands.
#include "attn_sched.h"
#include "internal.h"
#include "ptx.cuh"

namespace ds {

namespace {

constexpr int kBQ = 128;    // queries per tile
constexpr int kBKV = 128;   // keys per tile
constexpr int kThreads = 384;
constexpr float kRescaleLog2 = 8.0f;
// 2^kRescaleLog2: a row whose probabilities against its reference max sum to
// at most this has no score above that max + kRescaleLog2 (each probability
// is at most the fp32 sum of all of them, which are >= 0)
constexpr float kRescaleSum = 256.0f;
static_assert(kRescaleSum == 256.0f && kRescaleLog2 == 8.0f, "kRescaleSum = 2^kRescaleLog2");

template <int HD>
struct ACfg {
    static constexpr int RING = HD == 128 ? 5 : 8;       // K/V ring stages
    static constexpr int Q_BYTES = kBQ * HD * 2;          // one Q tile
    static constexpr int TILE_BYTES = kBKV * HD * 2;      // one K or V^T tile
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_RING = OFF_Q + 2 * Q_BYTES;
    static constexpr int OFF_BAR = OFF_RING + RING * TILE_BYTES;
    static constexpr int SMEM_BYTES = OFF_BAR + 512 + 1024;  // + barriers, schedule
    static constexpr int TMEM_COLS = 512;
    static constexpr int COL_O = 2 * kBKV;                // S_A S_B | O_A O_B
};

struct AttnParams {
    int64_t Tq, T;
    int n_kv;
    float scale_log2;  // log2(e) / sqrt(d)
    __nv_bfloat16 *o;
    int64_t ldo;
    int *status;
    // Keys in several launches (a block each, in ascending order): the
    // running max m, sum l and unnormalised fp32 O of every (query, head)
    // carried between them.  first: no state yet; last: normalise and store
    // O.  One launch over all keys is first = last = 1.
    float *o_state;           // [Tq, H*HD], row stride ld_state
    float *m_state, *l_state; // [Tq, H]
    int64_t ld_state;
    int heads;
    int first, last;
    // persistent schedule and the hand-off space of split units
    AttnGrid g;
    int n_qpairs;             // query-tile pairs per head
    int *split_flags;         // [slots]
    float *split_state;       // [slots][256 * (HD + 2)]: m, l, O
};

DEV float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// The whole S row of a tile (128 fp32 columns) into registers: four loads
// in flight, one wait (a wait covers every earlier load of the thread, so
// loads waited for one by one would each pay the full latency).
DEV void tile_load(uint32_t saddr, uint32_t (&s)[kBKV]) {
#pragma unroll
    for (int c0 = 0; c0 < kBKV; c0 += 32)
        tmem_ld32(saddr + c0, *reinterpret_cast<uint32_t(*)[32]>(s + c0));
#pragma unroll
    for (int c0 = 0; c0 < kBKV; c0 += 32) tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(s + c0));
}

// Row max of a tile held in registers; keys >= nvalid masked.
template <bool MASK>
DEV float row_max(const uint32_t (&s)[kBKV], int nvalid) {
    float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
    for (int c = 0; c < kBKV; c += 4) {
        float v0 = __uint_as_float(s[c]), v1 = __uint_as_float(s[c + 1]);
        float v2 = __uint_as_float(s[c + 2]), v3 = __uint_as_float(s[c + 3]);
        if (MASK) {
            if (c >= nvalid) v0 = -INFINITY;
            if (c + 1 >= nvalid) v1 = -INFINITY;
            if (c + 2 >= nvalid) v2 = -INFINITY;
            if (c + 3 >= nvalid) v3 = -INFINITY;
        }
        m0 = fmaxf(m0, v0);
        m1 = fmaxf(m1, v1);
        m2 = fmaxf(m2, v2);
        m3 = fmaxf(m3, v3);
    }
    return fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
}

// row_exp's arithmetic for the 32 keys c0.. of the row (the same
// instructions in the same order, so the same bits): P written over the
// tile's S columns, the fp32 probabilities added into the running sums
// (s0, s1) and (s2, s3).
template <bool MASK>
DEV void chunk_exp(const uint32_t (&s)[kBKV], int c0, uint32_t saddr, uint64_t sl2x2,
                   uint64_t negm2, int nvalid, uint64_t &s01, uint64_t &s23) {
    uint32_t pk[16];
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
        uint64_t x01 = (uint64_t(s[c0 + c + 1]) << 32) | s[c0 + c];
        uint64_t x23 = (uint64_t(s[c0 + c + 3]) << 32) | s[c0 + c + 2];
        asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x01) : "l"(sl2x2), "l"(negm2));
        asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x23) : "l"(sl2x2), "l"(negm2));
        float p0 = ex2(__uint_as_float(uint32_t(x01)));
        float p1 = ex2(__uint_as_float(uint32_t(x01 >> 32)));
        float p2 = ex2(__uint_as_float(uint32_t(x23)));
        float p3 = ex2(__uint_as_float(uint32_t(x23 >> 32)));
        if (MASK) {
            if (c0 + c >= nvalid) p0 = 0.f;
            if (c0 + c + 1 >= nvalid) p1 = 0.f;
            if (c0 + c + 2 >= nvalid) p2 = 0.f;
            if (c0 + c + 3 >= nvalid) p3 = 0.f;
        }
        const uint64_t p01 = (uint64_t(__float_as_uint(p1)) << 32) | __float_as_uint(p0);
        const uint64_t p23 = (uint64_t(__float_as_uint(p3)) << 32) | __float_as_uint(p2);
        asm("add.rn.f32x2 %0, %0, %1;" : "+l"(s01) : "l"(p01));
        asm("add.rn.f32x2 %0, %0, %1;" : "+l"(s23) : "l"(p23));
        pk[c >> 1] = pack_bf16x2(p0, p1);
        pk[(c >> 1) + 1] = pack_bf16x2(p2, p3);
    }
    tmem_st16(saddr + (c0 >> 1), pk);
}

DEV uint64_t pair_of(float v) {
    return (uint64_t(__float_as_uint(v)) << 32) | __float_as_uint(v);
}

DEV float sum_of(uint64_t s01, uint64_t s23) {
    const float s0 = __uint_as_float(uint32_t(s01)), s1 = __uint_as_float(uint32_t(s01 >> 32));
    const float s2 = __uint_as_float(uint32_t(s23)), s3 = __uint_as_float(uint32_t(s23 >> 32));
    return (s0 + s1) + (s2 + s3);
}

// P = exp2(S * sl2 - m) of a tile held in registers, as bf16 written over
// the tile's S columns in tensor memory (keys 2i, 2i+1 -> column i); returns
// the sum of the fp32 probabilities.  The scale-and-shift and the four
// running sums use packed two-lane fp32 instructions (each lane rounds as the
// scalar instruction would, in the same order), which cuts the instructions
// the softmax issues per score.
template <bool MASK>
DEV float row_exp(const uint32_t (&s)[kBKV], uint32_t saddr, float sl2, float m, int nvalid) {
    uint64_t s01 = 0, s23 = 0;  // (s0, s1), (s2, s3): four running sums
    const uint64_t sl2x2 = (uint64_t(__float_as_uint(sl2)) << 32) | __float_as_uint(sl2);
    const uint64_t negm2 = (uint64_t(__float_as_uint(-m)) << 32) | __float_as_uint(-m);
#pragma unroll
    for (int c0 = 0; c0 < kBKV; c0 += 32) {
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
            uint64_t x01 = (uint64_t(s[c0 + c + 1]) << 32) | s[c0 + c];
            uint64_t x23 = (uint64_t(s[c0 + c + 3]) << 32) | s[c0 + c + 2];
            asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x01) : "l"(sl2x2), "l"(negm2));
            asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x23) : "l"(sl2x2), "l"(negm2));
            float p0 = ex2(__uint_as_float(uint32_t(x01)));
            float p1 = ex2(__uint_as_float(uint32_t(x01 >> 32)));
            float p2 = ex2(__uint_as_float(uint32_t(x23)));
            float p3 = ex2(__uint_as_float(uint32_t(x23 >> 32)));
            if (MASK) {
                if (c0 + c >= nvalid) p0 = 0.f;
                if (c0 + c + 1 >= nvalid) p1 = 0.f;
                if (c0 + c + 2 >= nvalid) p2 = 0.f;
                if (c0 + c + 3 >= nvalid) p3 = 0.f;
            }
            const uint64_t p01 = (uint64_t(__float_as_uint(p1)) << 32) | __float_as_uint(p0);
            const uint64_t p23 = (uint64_t(__float_as_uint(p3)) << 32) | __float_as_uint(p2);
            asm("add.rn.f32x2 %0, %0, %1;" : "+l"(s01) : "l"(p01));
            asm("add.rn.f32x2 %0, %0, %1;" : "+l"(s23) : "l"(p23));
            pk[c >> 1] = pack_bf16x2(p0, p1);
            pk[(c >> 1) + 1] = pack_bf16x2(p2, p3);
        }
        tmem_st16(saddr + (c0 >> 1), pk);
    }
    const float s0 = __uint_as_float(uint32_t(s01)), s1 = __uint_as_float(uint32_t(s01 >> 32));
    const float s2 = __uint_as_float(uint32_t(s23)), s3 = __uint_as_float(uint32_t(s23 >> 32));
    return (s0 + s1) + (s2 + s3);
}

// The same while the row comes into registers: the load of each 32-column
// chunk is in flight during the previous chunk's exponentials (a wait covers
// every earlier load, so chunk c + 1 is issued after the wait for chunk c).
// P of chunk c overwrites columns 16c.., whose S values are already loaded.
// Returns the sum; the whole row is in registers afterwards.  Used at head
// dimension 64 (0.0986 -> 0.0946 ms for 4096 x 4096 x 16 heads, same bits);
// at 128 the same code spills at the 168-register allocation and the launch
// of 8192 x 32768 x 24 heads took 2.045 ms against 2.01-2.02 with the whole
// row loaded before the exponentials.
template <bool MASK>
DEV float row_load_exp(uint32_t (&s)[kBKV], uint32_t saddr, float sl2, float m, int nvalid) {
    uint64_t s01 = 0, s23 = 0;
    auto chunk = [&](int c0) -> uint32_t(&)[32] {
        return *reinterpret_cast<uint32_t(*)[32]>(s + c0);
    };
    tmem_ld32(saddr, chunk(0));
    tmem_ld_wait(chunk(0));
#pragma unroll
    for (int c0 = 0; c0 < kBKV; c0 += 32) {
        if (c0 + 32 < kBKV) tmem_ld32(saddr + c0 + 32, chunk(c0 + 32));
        chunk_exp<MASK>(s, c0, saddr, pair_of(sl2), pair_of(-m), nvalid, s01, s23);
        if (c0 + 32 < kBKV) tmem_ld_wait(chunk(c0 + 32));
    }
    return sum_of(s01, s23);
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    using C = ACfg<HD>;
    constexpr int kSlotFloats = 2 * kBQ * (HD + 2);  // m, l, O of 256 rows
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
    // bars: q_full, ring_full[RING], ring_empty[RING], s_full[2], p_full[2],
    //       o_full, drain, q_empty, handed (split state written)
    constexpr int B_Q = 0, B_RF = 1, B_RE = B_RF + C::RING, B_SF = B_RE + C::RING,
                  B_PF = B_SF + 2, B_O = B_PF + 2, B_DR = B_O + 1, B_QE = B_DR + 1,
                  B_HD = B_QE + 1, NBAR = B_HD + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBAR);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const uint32_t bar0 = smem_u32(bars);
    auto bar = [&](int i) { return bar0 + 8u * i; };

    const int warp = warp_id(), lane = lane_id();
    const int cta = blockIdx.x;
    const int n_kv = p.n_kv;
    // this CTA's pieces, in shared memory (kept out of the registers of the
    // softmax loop)
    AttnCta *cs_smem = reinterpret_cast<AttnCta *>(sm + C::OFF_BAR + 256);
    if (threadIdx.x == 0) *cs_smem = attn_cta(p.g, cta);
    const AttnCta &cs = *cs_smem;

    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q), 1);
        for (int s = 0; s < C::RING; ++s) {
            mbar_init(bar(B_RF + s), 1);
            mbar_init(bar(B_RE + s), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(B_SF + x), 1);
            mbar_init(bar(B_PF + x), 4);  // one arrival per softmax warp
        }
        mbar_init(bar(B_O), 1);
        mbar_init(bar(B_DR), 1);
        mbar_init(bar(B_QE), 1);
        mbar_init(bar(B_HD), 8);  // one arrival per softmax warp
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx wc{abort_flag, p.status};
    const uint32_t sQ = smem_u32(sm + C::OFF_Q);
    const uint32_t sRing = smem_u32(sm + C::OFF_RING);

    if (warp < 4) {
        // The TMA and MMA warps (and the two idle warps of their warpgroup)
        // hand registers to the softmax warpgroups: 4*32*152 + 8*32*176 =
        // 64,512 = the launch's 384 threads x 168, and per SM sub-partition
        // 152 + 176 + 176 <= 512 per lane.  Measured 1.7 % (d = 128) and
        // 5 % (d = 64) faster than 168 for every warp.
        asm volatile("setmaxnreg.dec.sync.aligned.u32 152;" ::: "memory");
    }
    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int rs = 0, nq = 0;             // ring stage; Q loads
            int nl = 0;                     // ring loads issued
            uint32_t rph = 0;               // ring pass parity
            bool ok = true;
            auto ring_load = [&](int head, int j, int kind) -> bool {
                if (!mbar_wait(bar(B_RE + rs), rph ^ 1u, wc)) return false;
                mbar_arrive_expect_tx(bar(B_RF + rs), C::TILE_BYTES);
                const uint32_t dst = sRing + rs * C::TILE_BYTES;
                if (kind == 0) {
#pragma unroll
                    for (int b = 0; b < HD / 64; ++b)
                        tma_load_2d(dst + b * (kBKV * 128), &tmK, bar(B_RF + rs),
                                    head * HD + 64 * b, j * kBKV);
                } else {
#pragma unroll
                    for (int b = 0; b < kBKV / 64; ++b)
                        tma_load_2d(dst + b * (HD * 128), &tmV, bar(B_RF + rs),
                                    j * kBKV + 64 * b, head * HD);
                }
                ++nl;
                if (++rs == C::RING) {
                    rs = 0;
                    rph ^= 1u;
                }
                return true;
            };
            for (int idx = 0; ok && idx < cs.count; ++idx) {
                const AttnItem it = attn_item(p.g, cs, cta, idx);
                const int qpair = it.u % p.n_qpairs, head = it.u / p.n_qpairs;
                // the item's first K/V tiles go ahead of its Q, which must
                // wait until the previous item's last S MMAs have read Q
                ok = ring_load(head, it.k0, 0) && ring_load(head, it.k0, 1);
                if (ok && idx > 0) ok = mbar_wait(bar(B_QE), uint32_t((idx - 1) & 1), wc);
                if (!ok) break;
                mbar_arrive_expect_tx(bar(B_Q), 2 * C::Q_BYTES);
#pragma unroll
                for (int x = 0; x < 2; ++x)
#pragma unroll
                    for (int b = 0; b < HD / 64; ++b)
                        tma_load_2d(sQ + x * C::Q_BYTES + b * (kBQ * 128), &tmQ, bar(B_Q),
                                    head * HD + 64 * b, (2 * qpair + x) * kBQ);
                ++nq;
                for (int j = it.k0 + 1; ok && j < it.k1; ++j)
                    ok = ring_load(head, j, 0) && ring_load(head, j, 1);
            }
            if (!ok) {  // let the copies in flight land before the CTA exits
                if (nq > 0) mbar_wait_quiet(bar(B_Q), uint32_t((nq - 1) & 1), kWaitLimitNs);
                for (int i = 0; i < C::RING && i < nl; ++i) {  // the last loads issued
                    if (--rs < 0) {
                        rs = C::RING - 1;
                        rph ^= 1u;
                    }
                    mbar_wait_quiet(bar(B_RF + rs), rph, kWaitLimitNs);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            // One thread issues 32 MMAs per key tile (~1,000 tensor cycles at
            // d = 128), so every instruction of this loop is on the critical
            // path: shared-memory descriptors are computed once and stepped by
            // constant offsets (16 bytes per unit of the address field, which
            // cannot overflow), and the last key tile of an item is peeled so
            // that the loop body has no branches but the waits.
            constexpr uint32_t ID_S = idesc_bf16_f32(kBQ, kBKV);
            constexpr uint32_t ID_PV = idesc_bf16_f32(kBQ, HD);
            const uint64_t dq0 = desc_sw128(sQ), dring = desc_sw128(sRing);
            auto issue_s = [&](int x, int stage) {
                const uint64_t dq = dq0 + uint64_t(x * (C::Q_BYTES >> 4));
                const uint64_t dk = dring + uint64_t(stage * (C::TILE_BYTES >> 4));
                const uint32_t d = tmem + uint32_t(x * kBKV);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint64_t off = uint64_t(((kk >> 2) * (kBQ * 128) + (kk & 3) * 32) >> 4);
                    mma_bf16_ss(d, dq + off, dk + off, ID_S, kk > 0);
                }
                mma_commit(bar(B_SF + x));
            };
            auto issue_pv = [&](int x, int stage, bool acc) {
                const uint64_t dv = dring + uint64_t(stage * (C::TILE_BYTES >> 4));
                const uint32_t pt = tmem + uint32_t(x * kBKV);  // P_X: lanes 0..127
                const uint32_t d = tmem + uint32_t(C::COL_O + x * HD);
#pragma unroll
                for (int kk = 0; kk < kBKV / 16; ++kk) {
                    const uint64_t offv = uint64_t(((kk >> 2) * (HD * 128) + (kk & 3) * 32) >> 4);
                    mma_bf16_ts(d, pt + uint32_t(8 * kk), dv + offv, ID_PV,
                                (acc || kk > 0) ? 1u : 0u);
                }
            };
            // ring entries are read in the order they were filled (K_0, V_0,
            // K_1, ...): the stage and its fill parity advance one by one
            int rs = 0;
            uint32_t rph = 0, tph = 0;  // ring pass parity; key tile parity
            auto advance = [&]() {
                if (++rs == C::RING) {
                    rs = 0;
                    rph ^= 1u;
                }
            };
            bool ok = true;
            for (int idx = 0; ok && idx < cs.count; ++idx) {
                const AttnItem it = attn_item(p.g, cs, cta, idx);
                const int nt = it.k1 - it.k0;
                // O starts from a carried state unless this is the start of
                // the unit's first launch
                const bool carried = it.k0 > 0 || !p.first;
                if (!mbar_wait(bar(B_Q), uint32_t(idx & 1), wc) ||
                    !mbar_wait(bar(B_RF + rs), rph, wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                issue_s(0, rs);
                issue_s(1, rs);
                mma_commit(bar(B_RE + rs));
                advance();
                for (int jj = 0; jj + 1 < nt; ++jj) {
                    const int sv = rs;  // V_j
                    if (!mbar_wait(bar(B_RF + sv), rph, wc) || !mbar_wait(bar(B_PF + 0), tph, wc)) {
                        ok = false;
                        break;
                    }
                    advance();
                    tc_fence_after();
                    issue_pv(0, sv, jj > 0 || carried);
                    const int sk = rs;  // K_{j+1}
                    if (!mbar_wait(bar(B_RF + sk), rph, wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_s(0, sk);
                    if (!mbar_wait(bar(B_PF + 1), tph, wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_pv(1, sv, jj > 0 || carried);
                    mma_commit(bar(B_RE + sv));
                    issue_s(1, sk);
                    mma_commit(bar(B_RE + sk));
                    advance();
                    tph ^= 1u;
                }
                if (!ok) break;
                // the item's last S MMAs are issued: Q may be reloaded once
                // they are complete
                mma_commit(bar(B_QE));
                {  // last key tile: PV only
                    const int sv = rs;
                    if (!mbar_wait(bar(B_RF + sv), rph, wc) || !mbar_wait(bar(B_PF + 0), tph, wc)) {
                        ok = false;
                        break;
                    }
                    advance();
                    tc_fence_after();
                    issue_pv(0, sv, nt > 1 || carried);
                    if (!mbar_wait(bar(B_PF + 1), tph, wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    issue_pv(1, sv, nt > 1 || carried);
                    mma_commit(bar(B_RE + sv));
                    tph ^= 1u;
                }
                mma_commit(bar(B_O));
            }
            if (!ok) {
                mma_commit(bar(B_DR));
                mbar_wait_quiet(bar(B_DR), 0, kWaitLimitNs);
            }
        }
    } else if (warp >= 4) {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 176;" ::: "memory");
        // ---------------------------------------------------- softmax
        const int x = (warp - 4) >> 2;          // tile A or B
        const int qd = warp & 3;                // TMEM lane quadrant
        const int row = qd * 32 + lane;         // query row within the tile
        const int urow = x * kBQ + row;         // row within the unit's 256
        const uint32_t lane_base = tmem + (uint32_t(qd * 32) << 16);
        const uint32_t saddr = lane_base + uint32_t(x * kBKV);
        const uint32_t oaddr = lane_base + uint32_t(C::COL_O + x * HD);
        const float sl2 = p.scale_log2;
        const int last_valid = int(p.T - int64_t(n_kv - 1) * kBKV);  // keys in last tile
        // O of this row (HD fp32 values, 4 columns per float4, consecutive
        // float4s `step` apart) into TMEM; rows beyond the queries read zeros
        auto o_to_tmem = [&](const float *src, size_t step, bool valid) {
            const float4 *s4 = reinterpret_cast<const float4 *>(src);
#pragma unroll
            for (int c0 = 0; c0 < HD; c0 += 32) {
                uint32_t r[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 v = valid ? s4[size_t((c0 >> 2) + i) * step]
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
                    r[4 * i] = __float_as_uint(v.x);
                    r[4 * i + 1] = __float_as_uint(v.y);
                    r[4 * i + 2] = __float_as_uint(v.z);
                    r[4 * i + 3] = __float_as_uint(v.w);
                }
                __syncwarp();
                tmem_st32_sync(oaddr + c0, r);
            }
        };
        // O of this row from TMEM to dst (fp32, the same layout), if valid
        auto o_from_tmem = [&](float *dst, size_t step, bool valid) {
            float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
            for (int c0 = 0; c0 < HD; c0 += 32) {
                uint32_t r[32];
                __syncwarp();
                tmem_ld32(oaddr + c0, r);
                tmem_ld_wait(r);
                if (valid) {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        d4[size_t((c0 >> 2) + i) * step] =
                            make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                        __uint_as_float(r[4 * i + 2]),
                                        __uint_as_float(r[4 * i + 3]));
                }
            }
        };
        // query row of this thread in item `it` (global index) and its head
        auto qrow_of = [&](const AttnItem &it) {
            return (2 * int64_t(it.u % p.n_qpairs) + x) * kBQ + row;
        };
        bool ok = true;
        int tc = 0;  // key tiles done
        for (int idx = 0; ok && idx < cs.count; ++idx) {
            float m = -INFINITY, l = 0.f;
            int k0, nt;
            {
                const AttnItem it = attn_item(p.g, cs, cta, idx);
                k0 = it.k0;
                nt = it.k1 - it.k0;
                // the state this item starts from: the CTA before's at k0
                // (the unit's earlier keys ran there), or the earlier
                // launches' (earlier key blocks); O goes into TMEM before
                // this item's first PV MMA, which accumulates onto it
                const float *src = nullptr;
                size_t step = 1;  // float4s between column groups
                bool valid = true;
                if (it.k0 > 0) {
                    const bool w = flag_wait(p.split_flags + it.src, wc);
                    if (!__all_sync(0xffffffffu, w)) {
                        ok = false;
                        break;
                    }
                    const float *slot = p.split_state + size_t(it.src) * kSlotFloats;
                    m = slot[urow];
                    l = slot[2 * kBQ + urow];
                    src = slot + 4 * kBQ + 4 * size_t(urow);  // column-group major
                    step = 2 * kBQ;
                } else if (!p.first) {
                    const int64_t qrow = qrow_of(it);
                    const int head = it.u / p.n_qpairs;
                    valid = qrow < p.Tq;
                    m = valid ? p.m_state[qrow * p.heads + head] : 0.f;
                    l = valid ? p.l_state[qrow * p.heads + head] : 0.f;
                    src = p.o_state + qrow * p.ld_state + int64_t(head) * HD;
                }
                if (src) o_to_tmem(src, step, valid);
            }
            const bool fresh = k0 == 0 && p.first;
            for (int jj = 0; jj < nt; ++jj) {
                const int j = k0 + jj;
                bool w = mbar_wait(bar(B_SF + x), uint32_t((tc + jj) & 1), wc);
                w = __all_sync(0xffffffffu, w);
                if (!w) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const bool masked = (j == n_kv - 1) && last_valid < kBKV;
                // the tile's S row in registers, for the exponentials and,
                // when needed, the max
                uint32_t sr[kBKV];
                float alpha = 1.0f;
                bool rescale = false;
                float sum;
                if (jj == 0 && fresh) {  // no reference max yet: the tile's own
                    tile_load(saddr, sr);
                    m = (masked ? row_max<true>(sr, last_valid) : row_max<false>(sr, kBKV)) * sl2;
                    sum = masked ? row_exp<true>(sr, saddr, sl2, m, last_valid)
                                 : row_exp<false>(sr, saddr, sl2, m, kBKV);
                } else {
                    // P against the reference max first.  A row can need its
                    // max moved (a score above m + kRescaleLog2) only if its
                    // probabilities sum to more than kRescaleSum, so the
                    // tile max is computed only for warps with such a row;
                    // the rows that move their max are exactly those the
                    // max-first order moves, and their P is redone.
                    if constexpr (HD == 64) {
                        sum = masked ? row_load_exp<true>(sr, saddr, sl2, m, last_valid)
                                     : row_load_exp<false>(sr, saddr, sl2, m, kBKV);
                    } else {
                        tile_load(saddr, sr);
                        sum = masked ? row_exp<true>(sr, saddr, sl2, m, last_valid)
                                     : row_exp<false>(sr, saddr, sl2, m, kBKV);
                    }
                    if (__any_sync(0xffffffffu, sum > kRescaleSum)) {
                        const float mx =
                            (masked ? row_max<true>(sr, last_valid) : row_max<false>(sr, kBKV)) *
                            sl2;
                        if (__any_sync(0xffffffffu, mx > m + kRescaleLog2)) {
                            // Move the reference max of the rows that need it:
                            // O_row *= 2^(m - m_new), l likewise.  The branch
                            // is warp-uniform (the TMEM accesses are
                            // warp-collective); the other rows keep m, their P
                            // and sum are recomputed unchanged and they are
                            // multiplied by exactly 1, so each row's result
                            // depends on that row alone.
                            const float m_new = (mx > m + kRescaleLog2) ? mx : m;
                            alpha = ex2(m - m_new);
                            m = m_new;
                            rescale = true;
                            tmem_st_wait();  // the first P is stored before it is overwritten
                            sum = masked ? row_exp<true>(sr, saddr, sl2, m, last_valid)
                                         : row_exp<false>(sr, saddr, sl2, m, kBKV);
                        }
                    }
                }
                if (rescale) {
                    // O is rescaled after P is written (the S row is out of
                    // the registers by then); the PV MMA that accumulates
                    // onto O waits for this thread's arrival below
#pragma unroll
                    for (int c0 = 0; c0 < HD; c0 += 32) {
                        uint32_t r[32];
                        tmem_ld32(oaddr + c0, r);
                        tmem_ld_wait(r);
#pragma unroll
                        for (int c = 0; c < 32; ++c)
                            r[c] = __float_as_uint(__uint_as_float(r[c]) * alpha);
                        tmem_st32_sync(oaddr + c0, r);
                    }
                    l *= alpha;
                }
                l += sum;
                tmem_st_wait();    // P is in tensor memory before the PV MMA reads it
                tc_fence_before(); // S/O/P accesses finish before the next MMAs
                mbar_arrive_warp(bar(B_PF + x));
            }
            if (!ok) break;
            // the item is looked up again rather than kept in registers
            // across the key loop
            const AttnItem it = attn_item(p.g, cs, cta, idx);
            const int64_t qrow = qrow_of(it);
            const int head = it.u / p.n_qpairs;
            const bool valid = qrow < p.Tq;
            {
                const bool w = mbar_wait(bar(B_O), uint32_t(idx & 1), wc);
                if (!__all_sync(0xffffffffu, w)) {
                    ok = false;
                    break;
                }
            }
            tc_fence_after();
            if (it.k1 < n_kv || !p.last) {
                // hand m, l and O at key tile k1 on: to the CTA that continues
                // the unit (all 256 rows write, then one thread sets the flag;
                // a CTA hands on at most once, since only its range's end can
                // fall inside a unit), or to the next key block's launch
                const bool split = it.k1 < n_kv;
                float *slot = p.split_state + size_t(split ? it.dst : 0) * kSlotFloats;
                float *mp = split ? slot + urow : p.m_state + qrow * p.heads + head;
                float *lp = split ? slot + 2 * kBQ + urow : p.l_state + qrow * p.heads + head;
                // the slot's O is column-group major (float4 j of row r at
                // j * 256 + r: a warp's rows move 512 contiguous bytes)
                float *dst = split ? slot + 4 * kBQ + 4 * size_t(urow)
                                   : p.o_state + qrow * p.ld_state + int64_t(head) * HD;
                const bool v = split || valid;
                if (v) {
                    *mp = m;
                    *lp = l;
                }
                o_from_tmem(dst, split ? size_t(2 * kBQ) : size_t(1), v);
                if (split) {
                    __threadfence();
                    mbar_arrive_warp(bar(B_HD));
                    if (x == 0 && row == 0) {
                        if (!mbar_wait(bar(B_HD), 0u, wc)) {
                            ok = false;
                        } else {
                            __threadfence();
                            flag_release(p.split_flags + it.dst);
                        }
                    }
                    ok = __all_sync(0xffffffffu, ok);
                }
            } else {
                const float inv = 1.0f / l;
                uint4 *dst = reinterpret_cast<uint4 *>(p.o + qrow * p.ldo + int64_t(head) * HD);
#pragma unroll
                for (int c0 = 0; c0 < HD; c0 += 32) {
                    uint32_t r[32];
                    __syncwarp();
                    tmem_ld32(oaddr + c0, r);
                    tmem_ld_wait(r);
                    if (valid) {
#pragma unroll
                        for (int c = 0; c < 32; c += 8) {
                            uint4 v;
                            v.x = pack_bf16x2(__uint_as_float(r[c]) * inv,
                                              __uint_as_float(r[c + 1]) * inv);
                            v.y = pack_bf16x2(__uint_as_float(r[c + 2]) * inv,
                                              __uint_as_float(r[c + 3]) * inv);
                            v.z = pack_bf16x2(__uint_as_float(r[c + 4]) * inv,
                                              __uint_as_float(r[c + 5]) * inv);
                            v.w = pack_bf16x2(__uint_as_float(r[c + 6]) * inv,
                                              __uint_as_float(r[c + 7]) * inv);
                            dst[(c0 + c) >> 3] = v;
                        }
                    }
                }
            }
            // this item's TMEM reads are done before the next item's MMAs
            // write O (the first PV waits for this thread's P arrival)
            tc_fence_before();
            tc += nt;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    // every thread of this CTA is past its wait on the flag it consumed:
    // leave it zero for the next launch
    if (threadIdx.x == 0 && cs.has_a && cs.a.src >= 0) p.split_flags[cs.a.src] = 0;
}

template <int HD>
dit_status_t run(const void *q, int64_t Tq, int64_t ldq, const void *k, int64_t ldk,
                 const void *vt, int64_t ldvt, int64_t T, int heads, void *o, int64_t ldo,
                 const AttnState *state, const AttnSplit *split, int *dev_status,
                 cudaStream_t s) {
    using C = ACfg<HD>;
    const uint64_t D = uint64_t(heads) * HD;
    const CUtensorMapDataType bf16 = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tQ, tK, tV;
    if (!make_tmap_2d(&tQ, bf16, q, D, uint64_t(Tq), uint64_t(ldq) * 2, 64, kBQ) ||
        !make_tmap_2d(&tK, bf16, k, D, uint64_t(T), uint64_t(ldk) * 2, 64, kBKV) ||
        !make_tmap_2d(&tV, bf16, vt, uint64_t(T), D, uint64_t(ldvt) * 2, 64, HD))
        return DIT_ERR_INVALID_ARG;
    AttnParams p{};
    p.Tq = Tq;
    p.T = T;
    p.n_kv = int((T + kBKV - 1) / kBKV);
    p.scale_log2 = 1.4426950408889634f / sqrtf(float(HD));
    p.o = reinterpret_cast<__nv_bfloat16 *>(o);
    p.ldo = ldo;
    p.status = dev_status;
    p.heads = heads;
    p.first = p.last = 1;
    if (state) {
        p.o_state = state->o;
        p.m_state = state->m;
        p.l_state = state->l;
        p.ld_state = state->ld;
        p.first = state->first;
        p.last = state->last;
    }
    const int64_t qtiles = (Tq + kBQ - 1) / kBQ;
    p.n_qpairs = int((qtiles + 1) / 2);
    int max_cta = sm_count();
    if (split && split->max_ctas > 0 && split->max_ctas < max_cta) max_cta = split->max_ctas;
    const int slots = (split && split->flags && split->state) ? split->slots : 0;
    p.g = attn_grid(p.n_qpairs * heads, p.n_kv, max_cta, slots, true);
    if (p.g.n_pc > 0) {
        p.split_flags = split->flags;
        p.split_state = split->state;
    }
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(
            attn_fwd_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return cuda_fail(e);
        attr_done = true;
    }
    // CTAs that hand state to one another must all be resident at once: a
    // cooperative launch guarantees it (one CTA per SM, at most one per SM)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.g.n_cta));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = p.g.n_pc > 0 ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, attn_fwd_kernel<HD>, tQ, tK, tV, p);
    if (e != cudaSuccess) return cuda_fail(e);
    return check_launch();
}

}  // namespace

dit_status_t launch_attention(const void *q, int64_t Tq, int64_t ldq, const void *k,
                              int64_t ldk, const void *vt, int64_t ldvt, int64_t T,
                              int heads, int head_dim, void *o, int64_t ldo, int *dev_status,
                              cudaStream_t s, const AttnState *state,
                              const AttnSplit *split) {
    if (Tq < 0 || T <= 0 || heads <= 0 || (head_dim != 64 && head_dim != 128))
        return DIT_ERR_INVALID_ARG;
    if (!q || !k || !vt || !o) return DIT_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o)) return DIT_ERR_ALIGN;
    const int64_t D = int64_t(heads) * head_dim;
    if (ldq < D || ldk < D || ldo < D || ldvt < T) return DIT_ERR_INVALID_ARG;
    if (ldq % 8 || ldk % 8 || ldo % 8 || ldvt % 8) return DIT_ERR_INVALID_ARG;
    if (Tq > (int64_t(1) << 31) - 2 * kBQ || T > (int64_t(1) << 31) - kBKV ||
        (Tq + 2 * kBQ - 1) / (2 * kBQ) * heads > (int64_t(1) << 30))
        return DIT_ERR_INVALID_ARG;
    if (split && split->slots > 0) {
        if (!split->flags || !split->state || split->slots > kAttnSplitSlots)
            return DIT_ERR_INVALID_ARG;
        if (!aligned16(split->state)) return DIT_ERR_ALIGN;
    }
    if (state) {
        if (!state->o || !state->m || !state->l) return DIT_ERR_INVALID_ARG;
        if (!aligned16(state->o) || state->ld < D || state->ld % 4) return DIT_ERR_ALIGN;
        if (T % kBKV && !state->last) return DIT_ERR_INVALID_ARG;  // only the last block ragged
    }
    if (Tq == 0) return DIT_OK;
    if (head_dim == 64)
        return run<64>(q, Tq, ldq, k, ldk, vt, ldvt, T, heads, o, ldo, state, split, dev_status,
                       s);
    return run<128>(q, Tq, ldq, k, ldk, vt, ldvt, T, heads, o, ldo, state, split, dev_status,
                    s);
}

}  // namespace ds
