// Tensor-core GEMM for sm_103a:  acc[M, N] = A[M, K] * B[N, K]^T
// (bf16 A, bf16 or int8 B, fp32 accumulation in tensor memory) with the
// block's fused epilogues: K/V store, Q store (both optionally with the
// per-head Q/K RMSNorm and rotary embedding), gated fp32 residual add,
// SwiGLU, and the down projection's accumulate-across-FFN-slices.
//
// Structure (one CTA per SM, persistent over 128 x BN output tiles):
//   warp 0      TMA producer: A and B k-blocks (64 wide) into a shared-memory
//               ring (bf16 tiles in the 128-byte swizzle the MMA reads)
//   warp 1      allocates TMEM; one lane issues tcgen05.mma (M=128, N=BN,
//               K=16) into one of two TMEM accumulators
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (one token row per
//               thread), the fused math, stores to global
//   warps 6-8,10 (int8 B only) dequantise: each int8 B tile staged by TMA is
//               converted to bf16 (exact: |q| <= 127) into the swizzled layout
//               of the MMA operand; the per-row scale multiplies the fp32
//               accumulator in the epilogue (W = s_row * q, "MiniMax-H3-Comfy-
//               NPU" section 2.2)
// The accumulator is double-buffered, so the epilogue of tile i overlaps the
// main loop of tile i+1.
//
// Work split (attn_sched.h, output tiles as units and K-steps as key tiles):
// each CTA runs its whole tiles in the order of a one-tile-per-CTA grid, and
// when the last, partial wave is worth cutting, its tiles' K-steps are cut
// into equal ranges shared by all CTAs.  A range that continues a tile starts
// from the raw fp32 accumulator the CTA before handed on (a state slot and a
// release/acquire flag; cooperative launch), so every output element is
// still one accumulation over K in the same order.
//
// Activation-space LoRA ("ComfyUI-StaticPipeline", "Activation-space LoRA
// (bypass mode)": y = W x + alpha B (A x)) continues the same accumulation:
// after W's K-steps, each 64-wide K-step of U L^T (U = x A^T, L = alpha B)
// takes two ring stages, one per half of the accumulator's columns (an M=128,
// N=128 MMA each: the two 128-row halves of the output tile, or for SwiGLU
// the gate and the up accumulator with their own U and L).  A LoRA stage
// holds a bf16 U tile where A's tile goes and a bf16 L tile at the start of
// the B area; with int8 weights the MMA reads it there directly and the
// converter warps skip the stage.
//
// Per-row exactness: every output element is the same fp32 accumulation over
// K in the same order (k-blocks of 64, MMAs of 16), whatever M, the tile
// schedule or the grid — so results do not depend on how tokens are chunked.
#include "attn_sched.h"
#include "internal.h"
#include "ptx.cuh"

namespace ds {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;

struct GemmParams {
    int64_t M;
    int N, K;
    int num_m, num_n, num_k;
    void *out;
    int64_t ldo;
    void *out2;
    int64_t ldo2;
    int64_t row_offset;
    int64_t pos0;  // rotary position of row 0 (Q/K transform)
    int split_n;
    float *x;
    int64_t ldx;
    const float *gate;
    float *acc;
    int64_t ldacc;
    int acc_load, acc_final;
    const float *s0, *s1;  // int8 per-row scales of B0 / B1
    int bscale;            // bf16 B holding int8 values: apply s0 / s1 too
    int inject_stall;      // DIT_GEMM_FLAG_INJECT_STALL test hook
    int *status;
    // Q/K transform (STORE_BF16, and K columns of KV); qk == 0: off
    int qk;
    const float *qk_norm;  // [head_dim] or null
    const float *rope_cos, *rope_sin;  // [positions, head_dim / 2] or null
    int head_dim;
    float qk_eps;
    int group_n;  // tile order: groups of group_n N-blocks, M-blocks within
    // work split: tiles as units, K-steps as key tiles (attn_sched.h); the
    // hand-off flags and slots of raw fp32 accumulators [MH*128][HALF_COLS]
    AttnGrid g;
    int *split_flags;
    float *split_state;
    // LoRA: K-steps of U L^T after the main ones (two half stages each)
    int num_lk;
    int lora_on0, lora_on1;
};

constexpr int kLoraRows = 128;                    // rows of a half's L tile
constexpr int kLoraStageBytes = (kBM + kLoraRows) * kBK * 2;

// MH: 128-row halves of the M tile of a one-CTA tile.  MH = 2 runs two
// M = 128 MMAs per K-step on one converted int8 B tile (half the conversion
// per multiply-add, with the N tile halved so that both halves'
// accumulators fit TMEM twice); no launch uses it now that launches without
// LoRA run on pair tiles, and LoRA launches use MH = 1.
//
// P (pair): a cluster of two CTAs computes a 256 x 256 output tile (SwiGLU:
// 256 rows x 128 features of gate and of up) with M = 256, N = 256 MMAs
// issued by the leading CTA (cta_group::2).  Each CTA stages its own 128 rows
// of A and half of the B rows (the N-block's first or second 128 rows; for
// SwiGLU the gate or the up tile) and keeps its 128 rows x 256 columns of the
// accumulator in its own tensor memory, so its epilogue is the MH = 1 one.
// Per K-step a CTA then stages half the B rows of the one-CTA 128 x 256
// tile for the same multiply-adds, and an int8 CTA converts half as many;
// the one-CTA tiles' main loops ran at 78-80 % tensor-pipe activity for bf16.
template <int MODE, bool I8, int MH = 1, bool P = false>
struct Cfg {
    static_assert(!P || MH == 1, "pair tiles hold one 128-row half per CTA");
    static constexpr int NB = (MODE == DIT_EPI_SWIGLU) ? 2 : 1;  // B operands
    static constexpr int BN = ((MODE == DIT_EPI_SWIGLU) ? 128 : 256) / MH;
    static constexpr int A_ROWS = kBM * MH;                 // rows of A per CTA
    static constexpr int BM = A_ROWS * (P ? 2 : 1);         // rows of A per tile
    static constexpr int B_ROWS = P ? 128 : NB * BN;        // B rows staged per CTA
    static constexpr int B_BOX = P ? 128 : BN;              // rows of one B TMA box
    static constexpr int MMA_M = P ? 256 : kBM;
    // Warps: 0 TMA producer, 1 MMA issuer (a pair's leader), 2 int8 B
    // producer (int8 pair), 3 forwarder (int8 pair, second CTA), 4..7
    // epilogue (TMEM lane quadrants 0..3), then the int8 -> bf16 converters.
    // One-CTA int8 tiles: warps 8, 10, 11, 12, 14, 15, two on each
    // sub-partition but the MMA issuer's (1), whose single thread bounds the
    // main loop (four converter warps took 640-700 cycles per 8 KB stage,
    // longer than a K-step of the MMAs).  Int8 pair tiles: warps 8..15 in
    // four groups of two, group g converting the CTA's K-steps j with
    // j % 4 == g, so four stages are converted at once and each group's
    // per-stage latency (wait, loads, stores, proxy fence, arrival) overlaps
    // the others' (one group of six: 0.64 ms for the SwiGLU launch of 8192 x
    // 8192 x 3072; two groups of three 0.59; three of two 0.53; four of two,
    // with two warps on the issuer's sub-partition, 0.52; with the int8 tile
    // staged in place and a 7-stage ring, 0.50).
    static constexpr bool QR = P && I8;
    static constexpr int CONV_WARPS = QR ? 8 : 6;           // int8 only
    static constexpr int CONV_GROUPS = QR ? 4 : 1;
    static constexpr int THREADS = I8 ? 512 : 256;
    static constexpr int A_BYTES = A_ROWS * kBK * 2;
    static constexpr int BQ_BYTES = B_ROWS * kBK;          // int8 B staging
    static constexpr int C_BYTES = B_ROWS * kBK * 2;       // one bf16 B tile
    // QR (int8 pair): one ring of A + converted-B stages, freed by one commit
    // per K-step.  The int8 B tile (8 KB) lands by TMA in the upper half of
    // its stage's converted-B slot (16 KB), and a converter group reads all
    // of it into registers before any of the group writes the bf16 tile over
    // the slot, so no separate int8 ring takes shared memory: the ring is 7
    // stages deep (6 with the fp32 epilogue tile) instead of 5 beside a
    // 7-stage int8 ring.  The conversion of a stage can start only when the
    // MMA of the stage's previous use is done, and the ring's depth is what
    // hides that chain (conversion, proxy fence, the peer's arrival, the MMA
    // and its commit).
    // TMA ring: bf16: A + B; int8 one-CTA: A + int8 B; QR: A + converted B
    // (the A tile completes on the converted-B barrier, so the MMA issuer
    // waits once per K-step).
    static constexpr bool EPI_T =
        MODE == DIT_EPI_RESID || MODE == DIT_EPI_DOWN || MODE == DIT_EPI_STORE_F32;
    static constexpr int STAGES = P ? (I8 ? (EPI_T ? 6 : 7) : 6) : 4;
    static constexpr int STAGE_BYTES = A_BYTES + (QR ? C_BYTES : I8 ? BQ_BYTES : C_BYTES);
    static constexpr int TMA_BYTES = QR ? A_BYTES : STAGE_BYTES;
    // fp32 epilogues (gated residual, down projection, fp32 store) move each
    // warp's 32 x 32 blocks through a padded shared-memory tile so that
    // every global access of a warp is one contiguous 128-byte row segment
    // (with one row per lane each access touched 32 lines, and the residual
    // epilogue took longer than the tile's main loop); the rings give up a
    // stage for it.
    static constexpr int T_BYTES = EPI_T ? 4 * 32 * 36 * 4 : 0;
    // int8 one-CTA: ring of converted bf16 B tiles read by the MMA (3 stages),
    // decoupled from the TMA ring so TMA latency and conversion overlap.
    static constexpr int CSTAGES = (I8 && !QR) ? (EPI_T ? 2 : 3) : 0;
    static constexpr int OFF_QIN = A_BYTES + BQ_BYTES;  // QR: int8 tile within a stage
    static constexpr int OFF_C = STAGES * STAGE_BYTES;
    static constexpr int OFF_T = OFF_C + CSTAGES * C_BYTES;
    static constexpr int HALF_COLS = NB * BN;      // fp32 TMEM columns per M half
    static constexpr int ACC_COLS = MH * HALF_COLS;  // per accumulator buffer
    static constexpr int TMEM_COLS = 2 * ACC_COLS;
    static constexpr int OUT_COLS = BN;       // output columns per tile
    static constexpr int SLOT_FLOATS = MH * kBM * HALF_COLS;  // one CTA's accumulator
    // barriers (up to byte 384), TMEM slot, abort flag; this CTA's work list
    // at byte 384
    static constexpr int BAR_BYTES = 512;
    static constexpr int SMEM_BYTES = OFF_T + T_BYTES + BAR_BYTES + 1024;
    static_assert(2 * STAGES + 32 <= 48 && CSTAGES <= 8,
                  "barriers overlap the work list");
    // A converter group's K-steps are CONV_GROUPS apart; its wait for a ring
    // slot's previous use to be freed is only unambiguous (mbarrier phase
    // parity) while that use is at most one ring cycle back, which needs
    // CONV_GROUPS <= the ring depth.
    static_assert(!QR || (CONV_GROUPS <= STAGES && CONV_GROUPS <= 8),
                  "converter groups outrun the ring");
    static_assert(!QR || 2 * BQ_BYTES == C_BYTES, "int8 tile fills half a converted slot");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Output tile of persistent work index t.  Tiles go in groups of group_n
// N-blocks; within a group M-block by M-block, N fastest.  The CTAs in flight
// then share the group's B tiles (kept to a size that stays in L2) and each
// A row block; a group of all N-blocks is plain M-major order.
DEV void tile_of(const GemmParams &p, int t, int &mb, int &nb) {
    const int per_group = p.group_n * p.num_m;
    const int g = t / per_group;
    const int r = t - g * per_group;
    const int n0 = g * p.group_n;
    const int gw = min(p.group_n, p.num_n - n0);
    mb = r / gw;
    nb = n0 + (r - (r / gw) * gw);
}

// LoRA half h of output tile nb: whether it has work, and the first row of
// its L tile (the tile's rows h*128.. for one B operand; SwiGLU: the tile's
// rows of the gate (h = 0) or up (h = 1) adapter).
template <int MODE, bool I8, int MH>
DEV bool lora_half_on(const GemmParams &p, int h, int nb) {
    using C = Cfg<MODE, I8, MH>;
    if (h == 0) return p.lora_on0 != 0;
    if (C::NB == 2) return p.lora_on1 != 0;
    return p.lora_on1 != 0 && nb * C::BN + kLoraRows < p.N;
}

template <int MODE, bool I8, int MH>
DEV int lora_row(int h, int nb) {
    using C = Cfg<MODE, I8, MH>;
    return C::NB == 2 ? nb * C::BN : nb * C::BN + h * kLoraRows;
}

DEV void store_bf16x32(__nv_bfloat16 *dst, const float (&f)[32]) {
    uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 v;
        v.x = pack_bf16x2(f[8 * i + 0], f[8 * i + 1]);
        v.y = pack_bf16x2(f[8 * i + 2], f[8 * i + 3]);
        v.z = pack_bf16x2(f[8 * i + 4], f[8 * i + 5]);
        v.w = pack_bf16x2(f[8 * i + 6], f[8 * i + 7]);
        d[i] = v;
    }
}

// x[0..31] += gate[0..31] * f[0..31], one fp32 rounding per element.
DEV void gated_residual32(float *x, const float *gate, const float (&f)[32]) {
    float4 *xv = reinterpret_cast<float4 *>(x);
    const float4 *gv = reinterpret_cast<const float4 *>(gate);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float4 a = xv[i];
        const float4 g = __ldg(gv + i);
        a.x = __fmaf_rn(g.x, f[4 * i + 0], a.x);
        a.y = __fmaf_rn(g.y, f[4 * i + 1], a.y);
        a.z = __fmaf_rn(g.z, f[4 * i + 2], a.z);
        a.w = __fmaf_rn(g.w, f[4 * i + 3], a.w);
        xv[i] = a;
    }
}

// f[0..31] *= s[0..31] (per-output-row int8 weight scales).
DEV void scale32(float (&f)[32], const float *s) {
    const float4 *sv = reinterpret_cast<const float4 *>(s);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float4 v = __ldg(sv + i);
        f[4 * i + 0] *= v.x;
        f[4 * i + 1] *= v.y;
        f[4 * i + 2] *= v.z;
        f[4 * i + 3] *= v.w;
    }
}

DEV float silu(float z) { return z / (1.0f + __expf(-z)); }

// Two floats (as raw bits) -> one bf16x2 word by taking their high halves.
// Exact for the values produced below: small integers whose low 16 mantissa
// bits are zero.
DEV uint32_t hi_halves(uint32_t f_lo, uint32_t f_hi) { return __byte_perm(f_lo, f_hi, 0x7632u); }

// Four int8 (one word, already XORed with 0x80808080 so each byte is
// u = q + 128) -> four bf16 (two bf16x2 words), exact.  u placed in the low
// mantissa bits of 2^23 is the float 2^23 + u; one packed subtraction of
// 2^23 + 128 leaves q, which has at most 8 significant bits, so its bf16
// value is the high half of its fp32 bits.
DEV uint2 int8x4_to_bf16x4(uint32_t u) {
    const uint64_t bias2 = 0xCB000080CB000080ull;  // (-(2^23 + 128)) x 2
    uint64_t a = (uint64_t(__byte_perm(u, 0x4B000000u, 0x7541u)) << 32) |
                 __byte_perm(u, 0x4B000000u, 0x7540u);
    uint64_t b = (uint64_t(__byte_perm(u, 0x4B000000u, 0x7543u)) << 32) |
                 __byte_perm(u, 0x4B000000u, 0x7542u);
    asm("add.rn.f32x2 %0, %0, %1;" : "+l"(a) : "l"(bias2));
    asm("add.rn.f32x2 %0, %0, %1;" : "+l"(b) : "l"(bias2));
    uint2 r;
    r.x = hi_halves(uint32_t(a), uint32_t(a >> 32));
    r.y = hi_halves(uint32_t(b), uint32_t(b >> 32));
    return r;
}

// Eight int8 (two words) -> eight bf16 (four bf16x2 words), exact.
DEV uint4 int8x8_to_bf16x8(uint2 w) {
    const uint2 lo = int8x4_to_bf16x4(w.x ^ 0x80808080u);
    const uint2 hi = int8x4_to_bf16x4(w.y ^ 0x80808080u);
    return make_uint4(lo.x, lo.y, hi.x, hi.y);
}

// One 32-column chunk of the accumulator row as fp32, with the int8 row
// scales applied.
template <bool I8>
DEV void load_chunk(const GemmParams &p, uint32_t taddr, int n, float (&f)[32]) {
    uint32_t r[32];
    tmem_ld32(taddr, r);
    tmem_ld_wait(r);
#pragma unroll
    for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(r[j]);
    if (I8 || p.bscale) scale32(f, p.s0 + n);
}

// Q/K epilogue with the per-head transform: for each head of d columns in
// the tile, the sum of squares over its accumulator columns (first pass over
// TMEM), then the RMSNorm scale and weight, the rotation of pairs (2i, 2i+1)
// by the angles of the row's position, and the bf16 store (second pass).
// "Proposal: Generic memory-aware streaming execution for transformer
// models", attention section (Q normalisation and positional transform on
// each bounded Q region).  V columns of KV pass through as in the plain
// epilogue.
template <int MODE, bool I8, int MH>
DEV void epilogue_qk_tile(const GemmParams &p, uint32_t taddr, int64_t m, int nb) {
    using C = Cfg<MODE, I8, MH>;
    const bool row_ok = m < p.M;
    const int d = p.head_dim;
    const int64_t pos = p.pos0 + m;           // rotary position
    const int64_t tok = p.row_offset + m;     // KV: destination row of K, column of V^T
    __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(p.out) +
                          (MODE == DIT_EPI_KV ? tok : m) * p.ldo;
#pragma unroll 1
    for (int h0 = 0; h0 < C::OUT_COLS; h0 += d) {
        const int nh = nb * C::BN + h0;  // first column of the head (warp-uniform)
        if (nh >= p.N) break;
        if (MODE == DIT_EPI_KV && nh >= p.split_n) {
#pragma unroll 1
            for (int c0 = 0; c0 < d; c0 += 32) {
                __syncwarp();
                float f[32];
                load_chunk<I8>(p, taddr + h0 + c0, nh + c0, f);
                if (!row_ok) continue;
                __nv_bfloat16 *vt = reinterpret_cast<__nv_bfloat16 *>(p.out2) +
                                    int64_t(nh + c0 - p.split_n) * p.ldo2 + tok;
#pragma unroll
                for (int j = 0; j < 32; ++j) vt[int64_t(j) * p.ldo2] = __float2bfloat16_rn(f[j]);
            }
            continue;
        }
        float inv_rms = 1.0f;
        if (p.qk_norm) {
            float ss = 0.0f;
#pragma unroll 1
            for (int c0 = 0; c0 < d; c0 += 32) {
                __syncwarp();
                float f[32];
                load_chunk<I8>(p, taddr + h0 + c0, nh + c0, f);
#pragma unroll
                for (int j = 0; j < 32; ++j) ss = __fmaf_rn(f[j], f[j], ss);
            }
            // d is a power of two: the mean is exact
            inv_rms = rsqrtf(ss * (1.0f / float(d)) + p.qk_eps);
        }
#pragma unroll 1
        for (int c0 = 0; c0 < d; c0 += 32) {
            __syncwarp();
            float f[32];
            load_chunk<I8>(p, taddr + h0 + c0, nh + c0, f);
            if (!row_ok) continue;
            if (p.qk_norm) {
                const float4 *g = reinterpret_cast<const float4 *>(p.qk_norm + c0);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 w = __ldg(g + i);
                    f[4 * i + 0] = f[4 * i + 0] * inv_rms * w.x;
                    f[4 * i + 1] = f[4 * i + 1] * inv_rms * w.y;
                    f[4 * i + 2] = f[4 * i + 2] * inv_rms * w.z;
                    f[4 * i + 3] = f[4 * i + 3] * inv_rms * w.w;
                }
            }
            if (p.rope_cos) {
                const int64_t off = pos * (d / 2) + c0 / 2;
                const float4 *cv = reinterpret_cast<const float4 *>(p.rope_cos + off);
                const float4 *sv = reinterpret_cast<const float4 *>(p.rope_sin + off);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 c4 = __ldg(cv + i), s4 = __ldg(sv + i);
                    const float cs[4] = {c4.x, c4.y, c4.z, c4.w};
                    const float sn[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float a = f[8 * i + 2 * k], b = f[8 * i + 2 * k + 1];
                        f[8 * i + 2 * k] = a * cs[k] - b * sn[k];
                        f[8 * i + 2 * k + 1] = a * sn[k] + b * cs[k];
                    }
                }
            }
            store_bf16x32(orow + nh + c0, f);
        }
    }
}

// fp32 epilogues (gated residual, down projection, fp32 store) of a warp's
// 32 rows m0.. through its shared-memory tile T (32 rows of 36 floats): per
// 32 columns each lane writes its accumulator row into T as float4s, then
// each group of 8 lanes reads one row back (lane & 7 picks the 16-byte
// piece), so one warp access moves four whole 128-byte row segments instead
// of touching 32 rows.  The row stride of 36 floats keeps both the writes
// and the reads free of bank conflicts.  The arithmetic per element is the
// row path's: scale, then one fused multiply-add onto x (or a plain store).
constexpr int kEpiLd = 36;  // floats per row of an epilogue tile
template <int MODE, bool I8, int MH>
DEV void epilogue_tile_f32(const GemmParams &p, uint32_t taddr, int64_t m0, int nb, float *T) {
    using C = Cfg<MODE, I8, MH>;
    const int lane = lane_id();
    const int64_t left = p.M - m0;
    const int rows = left < 32 ? int(left) : 32;  // <= 0: no row of this warp
    const bool scaled = (I8 || p.bscale) && !(MODE == DIT_EPI_DOWN && !p.acc_final);
    const bool resid = MODE == DIT_EPI_RESID || (MODE == DIT_EPI_DOWN && p.acc_final);
    const int sub = lane >> 3;       // row within a group of four
    const int c4 = (lane & 7) * 4;   // this lane's four columns
    float4 *tw = reinterpret_cast<float4 *>(T + lane * kEpiLd);
#pragma unroll 1
    for (int c0 = 0; c0 < C::OUT_COLS; c0 += 32) {
        __syncwarp();
        uint32_t r[32];
        tmem_ld32(taddr + c0, r);
        tmem_ld_wait(r);
        const int n = nb * C::BN + c0;  // warp-uniform; N is a multiple of 32
        if (rows <= 0 || n >= p.N) continue;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            tw[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
        __syncwarp();
        const float4 s = scaled ? __ldg(reinterpret_cast<const float4 *>(p.s0 + n + c4))
                                : make_float4(1.f, 1.f, 1.f, 1.f);
        const float4 g = resid ? __ldg(reinterpret_cast<const float4 *>(p.gate + n + c4))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        float *base;
        int64_t ld;
        if (resid) {
            base = p.x + m0 * p.ldx + n + c4;
            ld = p.ldx;
        } else if (MODE == DIT_EPI_DOWN) {
            base = p.acc + m0 * p.ldacc + n + c4;
            ld = p.ldacc;
        } else {
            base = reinterpret_cast<float *>(p.out) + m0 * p.ldo + n + c4;
            ld = p.ldo;
        }
        if (resid) {
            float4 xv[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int i = 4 * k + sub;
                if (i < rows) xv[k] = *reinterpret_cast<const float4 *>(base + int64_t(i) * ld);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int i = 4 * k + sub;
                if (i < rows) {
                    float4 v = *reinterpret_cast<const float4 *>(T + i * kEpiLd + c4);
                    if (scaled) {
                        v.x *= s.x;
                        v.y *= s.y;
                        v.z *= s.z;
                        v.w *= s.w;
                    }
                    float4 a = xv[k];
                    a.x = __fmaf_rn(g.x, v.x, a.x);
                    a.y = __fmaf_rn(g.y, v.y, a.y);
                    a.z = __fmaf_rn(g.z, v.z, a.z);
                    a.w = __fmaf_rn(g.w, v.w, a.w);
                    *reinterpret_cast<float4 *>(base + int64_t(i) * ld) = a;
                }
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int i = 4 * k + sub;
                if (i < rows) {
                    float4 v = *reinterpret_cast<const float4 *>(T + i * kEpiLd + c4);
                    if (scaled) {
                        v.x *= s.x;
                        v.y *= s.y;
                        v.z *= s.z;
                        v.w *= s.w;
                    }
                    *reinterpret_cast<float4 *>(base + int64_t(i) * ld) = v;
                }
            }
        }
    }
}

template <int MODE, bool I8, int MH>
DEV void epilogue_tile(const GemmParams &p, uint32_t taddr, int64_t m, int nb, float *T) {
    using C = Cfg<MODE, I8, MH>;
    if constexpr (C::EPI_T) {
        epilogue_tile_f32<MODE, I8, MH>(p, taddr, m - lane_id(), nb, T);
        return;
    }
    if constexpr (MODE == DIT_EPI_STORE_BF16 || MODE == DIT_EPI_KV) {
        if (p.qk) {
            epilogue_qk_tile<MODE, I8, MH>(p, taddr, m, nb);
            return;
        }
    }
    const bool row_ok = m < p.M;
#pragma unroll 1
    for (int c0 = 0; c0 < C::OUT_COLS; c0 += 32) {
        __syncwarp();
        uint32_t r[32];
        tmem_ld32(taddr + c0, r);
        uint32_t u[32];
        if constexpr (MODE == DIT_EPI_SWIGLU) {
            tmem_ld32(taddr + C::BN + c0, u);
            tmem_ld_wait(u);
        }
        tmem_ld_wait(r);
        const int n = nb * C::BN + c0;
        if (!row_ok || n >= p.N) continue;
        float f[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(r[j]);
        // The DOWN carry stays unscaled (the row scale is the same for every
        // FFN slice and is applied once, with the residual add).
        if ((I8 || p.bscale) && !(MODE == DIT_EPI_DOWN && !p.acc_final)) scale32(f, p.s0 + n);
        if constexpr (MODE == DIT_EPI_STORE_BF16) {
            store_bf16x32(reinterpret_cast<__nv_bfloat16 *>(p.out) + m * p.ldo + n, f);
        } else if constexpr (MODE == DIT_EPI_STORE_F32) {
            float4 *d = reinterpret_cast<float4 *>(reinterpret_cast<float *>(p.out) +
                                                   m * p.ldo + n);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                d[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
        } else if constexpr (MODE == DIT_EPI_KV) {
            const int64_t tok = p.row_offset + m;
            if (n < p.split_n) {
                store_bf16x32(reinterpret_cast<__nv_bfloat16 *>(p.out) + tok * p.ldo + n, f);
            } else {
                __nv_bfloat16 *vt = reinterpret_cast<__nv_bfloat16 *>(p.out2) +
                                    int64_t(n - p.split_n) * p.ldo2 + tok;
#pragma unroll
                for (int j = 0; j < 32; ++j) vt[int64_t(j) * p.ldo2] = __float2bfloat16_rn(f[j]);
            }
        } else if constexpr (MODE == DIT_EPI_RESID) {
            gated_residual32(p.x + m * p.ldx + n, p.gate + n, f);
        } else if constexpr (MODE == DIT_EPI_SWIGLU) {
            float g[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) g[j] = __uint_as_float(u[j]);
            if (I8 || p.bscale) scale32(g, p.s1 + n);
            float h[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) h[j] = silu(f[j]) * g[j];
            store_bf16x32(reinterpret_cast<__nv_bfloat16 *>(p.out) + m * p.ldo + n, h);
        } else if constexpr (MODE == DIT_EPI_DOWN) {
            if (p.acc_final) {
                gated_residual32(p.x + m * p.ldx + n, p.gate + n, f);
            } else {
                float4 *d = reinterpret_cast<float4 *>(p.acc + m * p.ldacc + n);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    d[i] = make_float4(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3]);
            }
        }
    }
}

// A thread's row of a raw fp32 accumulator between TMEM (COLS columns from
// taddr) and a hand-off slot of ROWS rows.  The slot is column-group major:
// the 4 columns 4j..4j+3 of row r are float4 number j * ROWS + r, so a warp's
// 32 rows move 512 contiguous bytes per access (row-major slots cost a cache
// line per thread and made each hand-off several times slower).
template <int COLS, int ROWS>
DEV void slot_to_tmem(const float *slot, int row, uint32_t taddr) {
    const float4 *s4 = reinterpret_cast<const float4 *>(slot) + row;
#pragma unroll 1
    for (int c0 = 0; c0 < COLS; c0 += 32) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 v = s4[size_t((c0 >> 2) + i) * ROWS];
            r[4 * i] = __float_as_uint(v.x);
            r[4 * i + 1] = __float_as_uint(v.y);
            r[4 * i + 2] = __float_as_uint(v.z);
            r[4 * i + 3] = __float_as_uint(v.w);
        }
        __syncwarp();
        tmem_st32_sync(taddr + c0, r);
    }
}
template <int COLS, int ROWS>
DEV void tmem_to_slot(uint32_t taddr, float *slot, int row) {
    float4 *d4 = reinterpret_cast<float4 *>(slot) + row;
#pragma unroll 1
    for (int c0 = 0; c0 < COLS; c0 += 32) {
        uint32_t r[32];
        __syncwarp();
        tmem_ld32(taddr + c0, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            d4[size_t((c0 >> 2) + i) * ROWS] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                            __uint_as_float(r[4 * i + 2]),
                                            __uint_as_float(r[4 * i + 3]));
    }
}

// DOWN with acc_load: write the carried fp32 accumulator of tile t into the
// TMEM buffer before the tile's MMAs start (they then accumulate onto it).
template <int MODE, bool I8, int MH>
DEV void preload_tile(const GemmParams &p, uint32_t taddr, int64_t m, int nb) {
    using C = Cfg<MODE, I8, MH>;
    const bool row_ok = m < p.M;
#pragma unroll 1
    for (int c0 = 0; c0 < C::OUT_COLS; c0 += 32) {
        const int n = nb * C::BN + c0;
        uint32_t r[32];
        if (row_ok && n < p.N) {
            const float4 *s = reinterpret_cast<const float4 *>(p.acc + m * p.ldacc + n);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 v = s[i];
                r[4 * i] = __float_as_uint(v.x);
                r[4 * i + 1] = __float_as_uint(v.y);
                r[4 * i + 2] = __float_as_uint(v.z);
                r[4 * i + 3] = __float_as_uint(v.w);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = 0u;
        }
        __syncwarp();
        tmem_st32_sync(taddr + c0, r);
    }
}

template <int MODE, bool I8, int MH, bool P>
__global__ void __launch_bounds__(Cfg<MODE, I8, MH, P>::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB0,
                   const __grid_constant__ CUtensorMap tmB1,
                   const __grid_constant__ CUtensorMap tmU0,
                   const __grid_constant__ CUtensorMap tmL0,
                   const __grid_constant__ CUtensorMap tmU1,
                   const __grid_constant__ CUtensorMap tmL1, const GemmParams p) {
    using C = Cfg<MODE, I8, MH, P>;
    constexpr int S = C::STAGES;
    constexpr int CS = C::CSTAGES;
    constexpr bool QR = C::QR;
    constexpr int G = P ? 2 : 1;  // cta_group of every tcgen05 instruction here
    extern __shared__ uint8_t smem_raw[];
    uint8_t *tiles = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(tiles + C::OFF_T + C::T_BYTES);
    // bars: full[S], empty[S], cfull[8], cempty[8] (QR: qfull), qempty[8]
    // (QR: the converter groups' load-before-store barriers),
    // tfull[2], tempty[2], drain, handed (split accumulator written); then the
    // TMEM slot and the abort flag; this CTA's work list at byte 384
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * S + 30);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    AttnCta *cs_smem = reinterpret_cast<AttnCta *>(reinterpret_cast<uint8_t *>(bars) + 384);
    // work unit owner: the CTA, or the cluster pair; rank 0 of a pair issues
    // the MMAs for both
    const int cta = P ? int(cluster_id_x()) : int(blockIdx.x);
    const int rank = P ? int(cluster_ctarank()) : 0;
    const bool leader = rank == 0;
    if (threadIdx.x == 0) *cs_smem = attn_cta(p.g, cta);
    const AttnCta &cs = *cs_smem;

    const int warp = warp_id();
    const int lane = lane_id();
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto cfull_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
    auto cempty_bar = [&](int s) { return bar0 + 8u * (2 * S + 8 + s); };
    auto qfull_bar = [&](int s) { return bar0 + 8u * (2 * S + 8 + s); };  // QR only
    auto gsync_bar = [&](int g) { return bar0 + 8u * (2 * S + 16 + g); };  // QR only
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * S + 24 + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * S + 26 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * S + 28);
    const uint32_t handed_bar = bar0 + 8u * (2 * S + 29);
    // the leader's copy of a barrier (pair: where the peer reports to)
    auto lead = [&](uint32_t bar) { return P ? mapa_shared(bar, 0) : bar; };
    constexpr uint32_t kConvThreads = 32 * C::CONV_WARPS;
    constexpr uint32_t kGroupThreads = kConvThreads / C::CONV_GROUPS;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
            // QR: stage s ready: the A producer's arrival with the A tile's
            // bytes, the converters' arrivals, and at the pair's leader the
            // peer's forwarded arrival
            if (QR) mbar_init(cfull_bar(s), kGroupThreads + 1 + (leader ? 1 : 0));
        }
        for (int s = 0; s < CS; ++s) {
            mbar_init(cfull_bar(s), kGroupThreads);
            mbar_init(cempty_bar(s), 1);
        }
        if (QR) {
            for (int s = 0; s < S; ++s) mbar_init(qfull_bar(s), 1);
            for (int g = 0; g < C::CONV_GROUPS; ++g) mbar_init(gsync_bar(g), kGroupThreads);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 128 + (P ? 4 : 0));  // pair: + the peer's 4 warps
        }
        mbar_init(drain_bar, 1);
        mbar_init(handed_bar, 4);  // one arrival per epilogue warp
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB0);
        if (C::NB == 2) tma_prefetch_desc(&tmB1);
        if (p.num_lk) {
            tma_prefetch_desc(&tmU0);
            tma_prefetch_desc(&tmL0);
            tma_prefetch_desc(&tmU1);
            tma_prefetch_desc(&tmL1);
        }
    }
    if (warp == 1) {
        tmem_alloc<G>(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish<G>();
    }
    tc_fence_before();
    __syncthreads();
    if constexpr (P) cluster_sync();  // both CTAs' barriers exist before any remote arrival
    tc_fence_after();
    // int8 (512 threads, launched with 128 registers each): the epilogue
    // warpgroup takes 168 from the producer / issuer warpgroup and the
    // converters (112 + 168 + 2 x 112 per thread: 64,512 of the 65,536; the
    // smallest split without spills)
    if constexpr (I8) {
        if (warp < 4)
            asm volatile("setmaxnreg.dec.sync.aligned.u32 112;" ::: "memory");
        else if (warp < 8)
            asm volatile("setmaxnreg.inc.sync.aligned.u32 168;" ::: "memory");
        else
            asm volatile("setmaxnreg.dec.sync.aligned.u32 112;" ::: "memory");
    }
    const uint32_t tmem = *tmem_slot;
    const WaitCtx wc{abort_flag, p.status};
    const bool preload = (MODE == DIT_EPI_DOWN || MODE == DIT_EPI_STORE_BF16) && p.acc_load;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------------------------------------- TMA producer
            // (QR: A only; the int8 B tiles come from warp 2)
            int stage = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            // this CTA's B operand and rows within the N-block (pair: its half)
            const CUtensorMap *tb = (P && C::NB == 2 && rank == 1) ? &tmB1 : &tmB0;
            const int b_row0 = (P && C::NB == 1) ? rank * C::B_BOX : 0;
            for (int idx = 0; idx < cs.count && ok; ++idx) {
                const AttnItem it = attn_item(p.g, cs, cta, idx);
                int mb, nb;
                tile_of(p, it.u, mb, nb);
                const int a_row = mb * C::BM + rank * C::A_ROWS;
                for (int kb = it.k0; kb < it.k1; ++kb) {
                    if (!mbar_wait(empty_bar(stage), ph ^ 1u, wc)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sA = smem_u32(tiles + stage * C::STAGE_BYTES);
                    const uint32_t sB = sA + C::A_BYTES;
                    // test hook: CTA 0 withholds its first copy (the stage's
                    // transaction count then never completes)
                    const bool withhold = p.inject_stall && blockIdx.x == 0 && issued == 0;
                    if (P && !I8) {
                        // bf16 pair: both CTAs' tiles complete on the leader's
                        // barrier, armed by the leader for both
                        if (leader) mbar_arrive_expect_tx(full_bar(stage), 2 * C::TMA_BYTES);
                        if (!withhold) {
                            const uint32_t fb = lead(full_bar(stage));
                            tma_load_2d_pair(sA, &tmA, fb, kb * kBK, a_row);
                            tma_load_2d_pair(sB, tb, fb, kb * kBK, nb * C::BN + b_row0);
                        }
                    } else {
                        const uint32_t fb = QR ? cfull_bar(stage) : full_bar(stage);
                        mbar_arrive_expect_tx(fb, C::TMA_BYTES);
                        if (!withhold) {
                            tma_load_2d(sA, &tmA, fb, kb * kBK, a_row);
                            if (!QR)
                                tma_load_2d(sB, tb, fb, kb * kBK, nb * C::BN + b_row0);
                            if (!P && C::NB == 2)
                                tma_load_2d(sB + C::B_BOX * kBK * (I8 ? 1 : 2), &tmB1, fb,
                                            kb * kBK, nb * C::BN);
                        }
                    }
                    ++issued;
                    if (++stage == S) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
                // LoRA K-steps (after the tile's last W K-step): U and L
                // tiles, one half stage per accumulator half (one-CTA tiles)
                const int num_lk = (!P && it.k1 == p.num_k) ? p.num_lk : 0;
                for (int lk = 0; lk < num_lk && ok; ++lk) {
                    for (int h = 0; h < 2; ++h) {
                        if (!mbar_wait(empty_bar(stage), ph ^ 1u, wc)) {
                            ok = false;
                            break;
                        }
                        const uint32_t sA = smem_u32(tiles + stage * C::STAGE_BYTES);
                        if (lora_half_on<MODE, I8, MH>(p, h, nb)) {
                            mbar_arrive_expect_tx(full_bar(stage), kLoraStageBytes);
                            tma_load_2d(sA, h ? &tmU1 : &tmU0, full_bar(stage), lk * kBK,
                                        mb * kBM);
                            tma_load_2d(sA + C::A_BYTES, h ? &tmL1 : &tmL0, full_bar(stage),
                                        lk * kBK, lora_row<MODE, I8, MH>(h, nb));
                        } else {
                            mbar_arrive(full_bar(stage));  // nothing to load
                        }
                        ++issued;
                        if (++stage == S) {
                            stage = 0;
                            ph ^= 1u;
                        }
                    }
                }
            }
            if (!ok) {  // let the copies already in flight land before exit
                if ((P && !I8 && !leader) || QR) {
                    // they complete on the leader's barriers, or on barriers
                    // that also wait for the converters: give them time
                    const uint64_t t0 = globaltimer();
                    while (globaltimer() - t0 < 200000ull) __nanosleep(1000);
                } else {
                    const int64_t first = issued > S ? issued - S : 0;
                    for (int64_t i = first; i < issued; ++i)
                        mbar_wait_quiet(full_bar(int(i % S)), uint32_t((i / S) & 1),
                                        kWaitLimitNs);
                }
            }
        }
    } else if (warp == 1 && (!P || leader)) {
        if (lane == 0) {
            // ---------------------------------------------- MMA issuer
            // The NB B tiles are contiguous in shared memory (rows of B1 follow
            // those of B0; pair: the peer's half follows this CTA's), so one
            // MMA with N = NB * BN covers both; its accumulator columns BN..
            // are the B1 results.
            constexpr uint32_t IDESC = idesc_bf16_f32(C::MMA_M, C::NB * C::BN);
            constexpr uint32_t IDESC_L = idesc_bf16_f32(kBM, kLoraRows);
            constexpr uint16_t kPairMask = 0x3;
            auto commit = [&](uint32_t bar) {
                if constexpr (P)
                    mma_commit_pair_mc(bar, kPairMask);  // the same barrier in both CTAs
                else
                    mma_commit(bar);
            };
            int stage = 0, cstage = 0;
            uint32_t ph = 0, cph = 0;
            // descriptors of the first TMA stage and the first converted-B stage
            const uint64_t da0 = desc_sw128(smem_u32(tiles));
            const uint64_t dc0 = desc_sw128(smem_u32(tiles + C::OFF_C));
            bool ok = true;
            for (int idx = 0; idx < cs.count && ok; ++idx) {
                const AttnItem it = attn_item(p.g, cs, cta, idx);
                // accumulator buffer idx % 2, ready (drained, and holding the
                // carry if the item starts from one) once per use
                const int buf = idx & 1;
                if (!mbar_wait(tempty_bar(buf), uint32_t((idx >> 1) & 1), wc)) {
                    ok = false;
                    break;
                }
                // the first K-step accumulates onto a carry: the CTA before's
                // partial sum at k0, or the caller's accumulator
                const bool carried = it.k0 > 0 || preload;
                tc_fence_after();
                const uint32_t d = tmem + uint32_t(buf * C::ACC_COLS);
                for (int kb = it.k0; kb < it.k1; ++kb) {
                    // the stage's tiles (bf16 pair: both CTAs'); int8
                    // one-CTA: and the converted B; int8 pair: one barrier
                    // for this CTA's A tile and converted B and the peer's
                    // signal that its stage is ready
                    if ((QR && !mbar_wait(cfull_bar(stage), ph, wc)) ||
                        (!QR && !mbar_wait(full_bar(stage), ph, wc)) ||
                        (I8 && !QR && !mbar_wait(cfull_bar(cstage), cph, wc))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // descriptors of the stage's tiles, stepped from the ring's
                    // first stage by whole stages and through K (16 elements =
                    // 32 bytes = 2 in the address field) and the M halves (128
                    // rows = 16 KB); the field cannot overflow
                    const uint64_t da = da0 + uint64_t(stage * (C::STAGE_BYTES >> 4));
                    const uint64_t db = (I8 && !QR)
                                            ? dc0 + uint64_t(cstage * (C::C_BYTES >> 4))
                                            : da + uint64_t(C::A_BYTES >> 4);
                    const uint32_t accum0 = kb != it.k0 || carried;
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        if constexpr (P) {
                            mma_bf16_ss_pair(d, da + uint64_t(2 * k), db + uint64_t(2 * k), IDESC,
                                             k == 0 ? accum0 : 1u);
                        } else {
#pragma unroll
                            for (int mh = 0; mh < MH; ++mh)
                                mma_bf16_ss(d + uint32_t(mh * C::HALF_COLS),
                                            da + uint64_t(mh * (kBM * 128 / 16) + 2 * k),
                                            db + uint64_t(2 * k), IDESC, k == 0 ? accum0 : 1u);
                        }
                    }
                    commit(empty_bar(stage));
                    if (++stage == S) {
                        stage = 0;
                        ph ^= 1u;
                    }
                    if (I8 && !QR) {
                        commit(cempty_bar(cstage));
                        if (++cstage == CS) {
                            cstage = 0;
                            cph ^= 1u;
                        }
                    }
                }
                if (!ok) break;
                if constexpr (!P) {
                    int mb, nb;
                    tile_of(p, it.u, mb, nb);
                    const int num_lk = it.k1 == p.num_k ? p.num_lk : 0;
                    for (int lk = 0; lk < num_lk && ok; ++lk) {
                        for (int h = 0; h < 2; ++h) {
                            if (!mbar_wait(full_bar(stage), ph, wc)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            if (lora_half_on<MODE, I8, MH>(p, h, nb)) {
                                const uint32_t sU = smem_u32(tiles + stage * C::STAGE_BYTES);
                                const uint32_t sL = sU + C::A_BYTES;
#pragma unroll
                                for (int k = 0; k < kBK / 16; ++k)
                                    mma_bf16_ss(d + uint32_t(h * kLoraRows),
                                                desc_sw128(sU + 32u * k),
                                                desc_sw128(sL + 32u * k), IDESC_L, 1u);
                            }
                            mma_commit(empty_bar(stage));
                            if (++stage == S) {
                                stage = 0;
                                ph ^= 1u;
                            }
                        }
                    }
                    if (!ok) break;
                }
                commit(tfull_bar(buf));
            }
            if (!ok) {  // every issued MMA must finish before TMEM is freed
                if constexpr (P)
                    mma_commit_pair_mc(drain_bar, 0x1);  // this CTA's barrier only
                else
                    mma_commit(drain_bar);
                mbar_wait_quiet(drain_bar, 0, kWaitLimitNs);
            }
        }
    } else if (warp == 2 && QR) {
        if (lane == 0) {
            // ---------------------------------------------- int8 B producer (QR)
            // into the upper half of the stage's converted-B slot, once the
            // MMAs of the stage's previous use are done
            const CUtensorMap *tb = (C::NB == 2 && rank == 1) ? &tmB1 : &tmB0;
            const int b_row0 = C::NB == 1 ? rank * C::B_BOX : 0;
            int stage = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int idx = 0; idx < cs.count && ok; ++idx) {
                const AttnItem it = attn_item(p.g, cs, cta, idx);
                int mb, nb;
                tile_of(p, it.u, mb, nb);
                for (int kb = it.k0; kb < it.k1; ++kb) {
                    if (!mbar_wait(empty_bar(stage), ph ^ 1u, wc)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(qfull_bar(stage), C::BQ_BYTES);
                    tma_load_2d(smem_u32(tiles + stage * C::STAGE_BYTES + C::OFF_QIN), tb,
                                qfull_bar(stage), kb * kBK, nb * C::BN + b_row0);
                    ++issued;
                    if (++stage == S) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (!ok) {
                const int64_t first = issued > S ? issued - S : 0;
                for (int64_t i = first; i < issued; ++i)
                    mbar_wait_quiet(qfull_bar(int(i % S)), uint32_t((i / S) & 1), kWaitLimitNs);
            }
        }
    } else if (QR && (warp == 1 || warp == 3)) {
        if (!leader && lane == 0) {
            // ---------------------------------------------- forwarders (QR)
            // the pair's second CTA: once its converters have filled the B
            // half of stage s and its A tile has landed there, arrive on the
            // leader's barrier of the stage.  A remote arrival holds its
            // thread for several hundred ns, so two otherwise idle warps (1,
            // the MMA issuer at the leader; 3) take the K-steps in turn.  (A
            // 16-byte bulk copy completing on the leader's barrier, which
            // does not hold the thread, took 1.5-2.3 us to land, queued
            // behind this CTA's tile loads; the down projection's launch of
            // 8192 x 3072 x 8192 ran 1 % slower with it.  A cluster-scope
            // release held each arriving thread so long that two forwarders
            // fell behind: the SwiGLU launch took 0.72 ms against 0.51.)
            const int mine = warp == 3 ? 0 : 1;
            int stage = 0, turn = 0;
            uint32_t ph = 0;
            bool ok = true;
            for (int idx = 0; idx < cs.count && ok; ++idx) {
                const AttnItem it = attn_item(p.g, cs, cta, idx);
                for (int kb = it.k0; kb < it.k1; ++kb) {
                    if (turn == mine) {
                        if (!mbar_wait(cfull_bar(stage), ph, wc)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_remote(lead(cfull_bar(stage)));
                    }
                    turn ^= 1;
                    if (++stage == S) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
            }
        }
    } else if (warp >= 4 && warp < 8) {
        // -------------------------------------------------- epilogue
        const int q = warp & 3;  // TMEM lane quadrant this warp may access
        const uint32_t lane_base = tmem + (uint32_t(q * 32) << 16);
        // hand-off flags and slots: one per CTA of a pair
        auto hslot = [&](int i) { return P ? 2 * i + rank : i; };
        // this warp's fp32 epilogue tile (32 rows of 36 floats)
        float *epi_t = reinterpret_cast<float *>(tiles + C::OFF_T) + q * (32 * 36);
        // Buffer j % 2 ready for item j: drained (this warp's epilogue of item
        // j - 2 is done, by program order) and, if the item starts from a
        // carry, holding it: the CTA before's raw accumulator at K-step k0
        // (waited for by its flag), or the caller's accumulator.
        auto prepare = [&](int j) -> bool {
            const AttnItem it = attn_item(p.g, cs, cta, j);
            const uint32_t base = lane_base + uint32_t((j & 1) * C::ACC_COLS);
            if (it.k0 > 0) {
                const bool w = flag_wait(p.split_flags + hslot(it.src), wc);
                if (!__all_sync(0xffffffffu, w)) return false;
                const float *slot = p.split_state + size_t(hslot(it.src)) * C::SLOT_FLOATS;
#pragma unroll 1
                for (int mh = 0; mh < MH; ++mh)
                    slot_to_tmem<C::HALF_COLS, MH * kBM>(slot, mh * kBM + q * 32 + lane,
                                                         base + uint32_t(mh * C::HALF_COLS));
            } else if (preload) {
                int mb, nb;
                tile_of(p, it.u, mb, nb);
#pragma unroll 1
                for (int mh = 0; mh < MH; ++mh)
                    preload_tile<MODE, I8, MH>(
                        p, base + uint32_t(mh * C::HALF_COLS),
                        int64_t(mb) * C::BM + rank * C::A_ROWS + mh * kBM + q * 32 + lane, nb);
            }
            tc_fence_before();
            if (P && !leader)
                mbar_arrive_remote_warp(lead(tempty_bar(j & 1)));
            else
                mbar_arrive(tempty_bar(j & 1));
            return true;
        };
        bool ok = true;
        for (int j = 0; ok && j < 2 && j < cs.count; ++j) ok = prepare(j);
        for (int idx = 0; ok && idx < cs.count; ++idx) {
            const int buf = idx & 1;
            {
                const bool w = mbar_wait(tfull_bar(buf), uint32_t((idx >> 1) & 1), wc);
                if (!__all_sync(0xffffffffu, w)) break;
            }
            tc_fence_after();
            const AttnItem it = attn_item(p.g, cs, cta, idx);
            const uint32_t base = lane_base + uint32_t(buf * C::ACC_COLS);
            if (it.k1 < p.num_k) {
                // hand the raw accumulator at K-step k1 to the CTA that
                // continues the tile: all rows write, then one thread sets the
                // flag (a CTA hands on at most once: only its range's end can
                // fall inside a tile)
                float *slot = p.split_state + size_t(hslot(it.dst)) * C::SLOT_FLOATS;
#pragma unroll 1
                for (int mh = 0; mh < MH; ++mh)
                    tmem_to_slot<C::HALF_COLS, MH * kBM>(base + uint32_t(mh * C::HALF_COLS), slot,
                                                         mh * kBM + q * 32 + lane);
                __threadfence();
                mbar_arrive_warp(handed_bar);
                if (warp == 4 && lane == 0) {
                    if (!mbar_wait(handed_bar, 0u, wc)) {
                        ok = false;
                    } else {
                        __threadfence();
                        flag_release(p.split_flags + hslot(it.dst));
                    }
                }
                ok = __all_sync(0xffffffffu, ok);
            } else {
                int mb, nb;
                tile_of(p, it.u, mb, nb);
#pragma unroll 1
                for (int mh = 0; mh < MH; ++mh)
                    epilogue_tile<MODE, I8, MH>(
                        p, base + uint32_t(mh * C::HALF_COLS),
                        int64_t(mb) * C::BM + rank * C::A_ROWS + mh * kBM + q * 32 + lane, nb,
                        epi_t);
            }
            if (ok && idx + 2 < cs.count) ok = prepare(idx + 2);
        }
    } else if (I8 && warp >= 8 && (QR || (warp & 3) != 1)) {
        // -------------------------------------------------- int8 -> bf16
        // Staged int8 rows (64 bytes each, B_ROWS rows) become 128-byte bf16
        // rows of a converted-B tile; 16-byte chunk c of row r lands at chunk
        // c ^ (r % 8) of the row (the 128-byte swizzle), rows in 8-row groups
        // of 1024 bytes.  One-CTA tiles: from the TMA stage into the
        // converted-B ring; QR: in place, from the upper half of the A + B
        // stage's B slot (where the int8 tile landed once the MMAs of the
        // stage's previous use were done) over the whole slot.  Group g of
        // CONV_GROUPS converts the CTA's K-steps j with j % CONV_GROUPS == g.
        const int tid_all =
            (QR ? warp - 8 : (warp - 8) - (warp > 9) - (warp > 13)) * 32 + lane;
        const int grp = tid_all / int(kGroupThreads);
        const int tid = tid_all % int(kGroupThreads);
        int stage = 0, cstage = 0, turn = 0;
        uint32_t ph = 0, cph = 0, gph = 0;
        bool ok = true;
        for (int idx = 0; ok && idx < cs.count; ++idx) {
            const AttnItem it = attn_item(p.g, cs, cta, idx);
            for (int kb = it.k0; kb < it.k1; ++kb) {
              const bool mine = turn == grp;
              if (++turn == C::CONV_GROUPS) turn = 0;
              if (mine) {
                bool w;
                if constexpr (QR)
                    w = mbar_wait(qfull_bar(stage), ph, wc);  // the slot was free for it
                else
                    w = mbar_wait(full_bar(stage), ph, wc) &&
                        mbar_wait(cempty_bar(cstage), cph ^ 1u, wc);
                w = __all_sync(0xffffffffu, w);
                if (!w) {
                    ok = false;
                    break;
                }
                const uint8_t *sq = tiles + stage * C::STAGE_BYTES + (QR ? C::OFF_QIN : C::A_BYTES);
                uint8_t *dst0 = QR ? tiles + stage * C::STAGE_BYTES + C::A_BYTES
                                   : tiles + C::OFF_C + cstage * C::C_BYTES;
                // Thread tid owns pieces of 8 int8: rows r = tid / 8 + kStep i
                // (kStep = the group's threads / 8; the last piece is ragged),
                // chunk c = tid % 8.  Loads go ahead of the conversions so
                // their latency overlaps (one-CTA: in batches; QR: all).
                constexpr int kStep = int(kGroupThreads) / 8;
                constexpr int kPieces = (C::B_ROWS + kStep - 1) / kStep;
                constexpr int kBatch = kPieces < 6 ? kPieces : 6;
                const int r0 = tid >> 3, c8 = tid & 7;
                const uint8_t *src = sq + r0 * kBK + c8 * 8;
                // row r's chunk c lands at chunk c ^ (r % 8): with kStep a
                // multiple of 8 that is the same chunk for every piece
                auto dst_of = [&](int i) -> uint8_t * {
                    const int r = r0 + i * kStep;
                    const int sw = (kStep % 8 == 0) ? (r0 & 7) : (r & 7);
                    return dst0 + r * 128 + ((c8 ^ sw) << 4);
                };
                if constexpr (QR) {
                    // the bf16 tile overwrites the int8 tile it comes from:
                    // the whole group's pieces go into registers first, and
                    // the group's barrier (bounded wait) orders every load
                    // before any store
                    uint2 w8[kPieces];
#pragma unroll
                    for (int i = 0; i < kPieces; ++i) {
                        const bool in = r0 + i * kStep < C::B_ROWS;
                        w8[i] = in ? *reinterpret_cast<const uint2 *>(src + i * kStep * kBK)
                                   : make_uint2(0u, 0u);
                    }
                    mbar_arrive(gsync_bar(grp));
                    bool gw = mbar_wait(gsync_bar(grp), gph, wc);
                    gph ^= 1u;
                    gw = __all_sync(0xffffffffu, gw);
                    if (!gw) {
                        ok = false;
                        break;
                    }
#pragma unroll
                    for (int i = 0; i < kPieces; ++i) {
                        const bool in = r0 + i * kStep < C::B_ROWS;
                        if (in) *reinterpret_cast<uint4 *>(dst_of(i)) = int8x8_to_bf16x8(w8[i]);
                    }
                } else {
#pragma unroll
                    for (int i0 = 0; i0 < kPieces; i0 += kBatch) {
                        uint2 w8[kBatch];
#pragma unroll
                        for (int i = 0; i < kBatch; ++i) {
                            const bool in =
                                i0 + i < kPieces && r0 + (i0 + i) * kStep < C::B_ROWS;
                            w8[i] = in ? *reinterpret_cast<const uint2 *>(src + (i0 + i) * kStep *
                                                                          kBK)
                                       : make_uint2(0u, 0u);
                        }
#pragma unroll
                        for (int i = 0; i < kBatch; ++i) {
                            const bool in =
                                i0 + i < kPieces && r0 + (i0 + i) * kStep < C::B_ROWS;
                            if (in)
                                *reinterpret_cast<uint4 *>(dst_of(i0 + i)) =
                                    int8x8_to_bf16x8(w8[i]);
                        }
                    }
                }
                fence_proxy_async_smem();  // the tensor core reads what we wrote
                // every converter thread arrives as soon as its own stores are
                // fenced (one arrival per warp after __syncwarp measured 3-5 %
                // slower)
                mbar_arrive(cfull_bar(QR ? stage : cstage));
              }
                if constexpr (!QR) {
                    if (++cstage == CS) {
                        cstage = 0;
                        cph ^= 1u;
                    }
                }
                if (++stage == S) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
            // the tile's LoRA stages hold bf16 tiles the MMA reads directly
            const int num_lk = (!P && it.k1 == p.num_k) ? p.num_lk : 0;
            for (int i = 0; ok && i < 2 * num_lk; ++i) {
                if (++stage == S) {
                    stage = 0;
                    ph ^= 1u;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    // pair: neither CTA frees its tensor memory or leaves (its barriers may
    // still take the other's arrivals) before both are done
    if constexpr (P) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc<G>(tmem, C::TMEM_COLS);
    }
    // every thread of this CTA is past its wait on the flag it consumed:
    // leave it zero for the next launch
    if (threadIdx.x == 0 && cs.has_a && cs.a.src >= 0)
        p.split_flags[P ? 2 * cs.a.src + rank : cs.a.src] = 0;
}

// Per (mode, B type, tile shape, device): 0 until the kernel's shared-memory
// attribute is set; then, for pair kernels, the most clusters of two that can
// be resident at once (queried once).
int &attr_flag(int mode, bool i8, int shape) {
    static int done[8][2][3][64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    return done[mode][i8 ? 1 : 0][shape][dev & 63];
}

template <int MODE, bool I8, int MH, bool P>
dit_status_t run(const dit_gemm_args_t &a, int *dev_status, cudaStream_t s,
                 const AttnSplit *split) {
    using C = Cfg<MODE, I8, MH, P>;
    static_assert(size_t(C::SLOT_FLOATS) * 4 == kGemmSlotBytes, "hand-off slot size");
    CUtensorMap tA, tB0, tB1;
    if (!make_tmap_2d(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.a, uint64_t(a.K), uint64_t(a.M),
                      uint64_t(a.lda) * 2, kBK, C::A_ROWS))
        return DIT_ERR_INVALID_ARG;
    const CUtensorMapDataType bdt =
        I8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const uint64_t bel = I8 ? 1 : 2;
    const CUtensorMapSwizzle bsw = I8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
    if (!make_tmap_2d(&tB0, bdt, a.b0, uint64_t(a.K), uint64_t(a.N), uint64_t(a.ldb) * bel, kBK,
                      C::B_BOX, bsw))
        return DIT_ERR_INVALID_ARG;
    tB1 = tB0;
    if (C::NB == 2 && !make_tmap_2d(&tB1, bdt, a.b1, uint64_t(a.K), uint64_t(a.N),
                                    uint64_t(a.ldb) * bel, kBK, C::B_BOX, bsw))
        return DIT_ERR_INVALID_ARG;

    // LoRA operand maps (unused ones alias A's map)
    CUtensorMap tU0 = tA, tL0 = tA, tU1 = tA, tL1 = tA;
    int rmax = 0;
    if (a.lora_l0) {
        if (!make_tmap_2d(&tU0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.lora_u0,
                          uint64_t(a.lora_rank0), uint64_t(a.M), uint64_t(a.lora_ldu0) * 2, kBK,
                          kBM) ||
            !make_tmap_2d(&tL0, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.lora_l0,
                          uint64_t(a.lora_rank0), uint64_t(a.N), uint64_t(a.lora_ldl0) * 2, kBK,
                          kLoraRows))
            return DIT_ERR_INVALID_ARG;
        rmax = a.lora_rank0;
    }
    if (C::NB == 2 && a.lora_l1) {
        if (!make_tmap_2d(&tU1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.lora_u1,
                          uint64_t(a.lora_rank1), uint64_t(a.M), uint64_t(a.lora_ldu1) * 2, kBK,
                          kBM) ||
            !make_tmap_2d(&tL1, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.lora_l1,
                          uint64_t(a.lora_rank1), uint64_t(a.N), uint64_t(a.lora_ldl1) * 2, kBK,
                          kLoraRows))
            return DIT_ERR_INVALID_ARG;
        if (a.lora_rank1 > rmax) rmax = a.lora_rank1;
    }
    if (C::NB == 1) {  // one adapter: its two halves cover the tile's rows
        tU1 = tU0;
        tL1 = tL0;
    }
    if (P && rmax) return DIT_ERR_INVALID_ARG;  // LoRA K-steps use one-CTA tiles

    GemmParams p{};
    p.M = a.M;
    p.N = a.N;
    p.K = a.K;
    p.num_m = int((a.M + C::BM - 1) / C::BM);
    p.num_n = (a.N + C::BN - 1) / C::BN;
    p.num_k = a.K / kBK;
    {  // N-blocks per tile group: the group's B tiles within ~48 MB of L2
        const int64_t b_block = int64_t(C::NB) * C::BN * a.K * (I8 ? 1 : 2);
        int64_t gn = (int64_t(48) << 20) / b_block;
        if (gn < 1) gn = 1;
        p.group_n = gn < p.num_n ? int(gn) : p.num_n;
    }
    p.out = a.out;
    p.ldo = a.ldo;
    p.out2 = a.out2;
    p.ldo2 = a.ldo2;
    p.row_offset = a.row_offset;
    p.pos0 = a.rope_pos0;
    p.split_n = a.split_n;
    p.x = a.x;
    p.ldx = a.ldx;
    p.gate = a.gate;
    p.acc = a.acc;
    p.ldacc = a.ldacc;
    p.acc_load = a.acc_load;
    p.acc_final = a.acc_final;
    p.s0 = a.b0_scale;
    p.s1 = a.b1_scale;
    p.bscale = (!I8 && a.b0_scale) ? 1 : 0;
    p.inject_stall = (a.flags & DIT_GEMM_FLAG_INJECT_STALL) != 0;
    p.status = dev_status;
    p.qk = (a.qk_norm || a.rope_cos) ? 1 : 0;
    p.qk_norm = a.qk_norm;
    p.rope_cos = a.rope_cos;
    p.rope_sin = a.rope_sin;
    p.head_dim = a.head_dim;
    p.qk_eps = a.qk_eps;
    p.num_lk = (rmax + kBK - 1) / kBK;
    p.lora_on0 = a.lora_l0 != nullptr;
    p.lora_on1 = C::NB == 2 ? a.lora_l1 != nullptr : a.lora_l0 != nullptr;

    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;

    const int shape = P ? 2 : MH - 1;
    int &done = attr_flag(MODE, I8, shape);
    if (!done) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<MODE, I8, MH, P>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             C::SMEM_BYTES);
        if (e != cudaSuccess) return cuda_fail(e);
        done = 1;
        if (P) {
            cfg.gridDim = dim3(2u * unsigned(sm_count() / 2));
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            e = cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<MODE, I8, MH, P>, &cfg);
            if (e != cudaSuccess) return cuda_fail(e);
            if (n < 1) return DIT_ERR_CUDA;
            done = n;
        }
    }
    // workers: CTAs, or resident pairs
    const int units = p.num_m * p.num_n;
    int max_w = P ? done : sm_count();
    if (split && split->max_ctas > 0) {
        const int cap = P ? (split->max_ctas >= 2 ? split->max_ctas / 2 : 1) : split->max_ctas;
        if (cap < max_w) max_w = cap;
    }
    // No split where the epilogue, not the main loop, bounds a tile: the bf16
    // gated-residual launch's fp32 read-modify-write (about 20 us per 128 x
    // 256 tile against 16 us of MMAs, measured) would only gain work.
    const bool split_pays = I8 || MODE != DIT_EPI_RESID;
    int slots = (split_pays && split && split->flags && split->state) ? split->slots : 0;
    if (P) slots /= 2;  // a cut pair tile hands on two slots, one per CTA
    p.g = attn_grid(units, p.num_k, max_w, slots);
    if (p.g.n_pc > 0) {
        p.split_flags = split->flags;
        p.split_state = split->state;
    }
    // CTAs that hand accumulators to one another must all be resident at
    // once: a cooperative launch guarantees it (at most one CTA per SM)
    auto launch = [&]() {
        cudaLaunchAttribute used[2];
        int na = 0;
        if (P) used[na++] = attr[0];
        if (p.g.n_pc > 0) used[na++] = attr[1];
        cfg.gridDim = dim3(unsigned(p.g.n_cta * (P ? 2 : 1)));
        cfg.attrs = used;
        cfg.numAttrs = na;
        return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<MODE, I8, MH, P>, tA, tB0, tB1, tU0, tL0,
                                  tU1, tL1, p);
    };
    cudaError_t e = launch();
    if (e != cudaSuccess && P && p.g.n_pc > 0) {
        // no cooperative launch of clusters here: run whole tiles only
        (void)cudaGetLastError();
        p.g = attn_grid(units, p.num_k, max_w, 0);
        p.split_flags = nullptr;
        p.split_state = nullptr;
        e = launch();
    }
    if (e != cudaSuccess) return cuda_fail(e);
    return check_launch();
}

template <int MODE>
dit_status_t run_b(const dit_gemm_args_t &a, int *dev_status, cudaStream_t s,
                   const AttnSplit *split) {
    // LoRA K-steps are laid out for one-CTA tiles of 128 rows; everything
    // else runs on pair tiles
    const bool lora = a.lora_l0 || a.lora_l1;
    if (a.b_dtype == DIT_W_BF16)
        return lora ? run<MODE, false, 1, false>(a, dev_status, s, split)
                    : run<MODE, false, 1, true>(a, dev_status, s, split);
    return lora ? run<MODE, true, 1, false>(a, dev_status, s, split)
                : run<MODE, true, 1, true>(a, dev_status, s, split);
}

bool ld_ok(int64_t ld, int64_t min_ld, int elem_bytes) {
    return ld >= min_ld && (ld * elem_bytes) % 16 == 0;
}

}  // namespace

dit_status_t launch_gemm(const dit_gemm_args_t &a, int *dev_status, cudaStream_t s,
                         const AttnSplit *split) {
    if (a.M < 0 || a.N <= 0 || a.K <= 0 || a.N % 32 || a.K % kBK) return DIT_ERR_INVALID_ARG;
    if (a.M > (int64_t(1) << 31) - kBM) return DIT_ERR_INVALID_ARG;
    if (a.b_dtype != DIT_W_BF16 && a.b_dtype != DIT_W_INT8)
        return DIT_ERR_INVALID_ARG;
    if (a.flags & ~DIT_GEMM_FLAG_INJECT_STALL) return DIT_ERR_INVALID_ARG;
    const bool i8 = a.b_dtype != DIT_W_BF16;
    if (!a.a || !a.b0) return DIT_ERR_INVALID_ARG;
    if (!aligned16(a.a) || !aligned16(a.b0)) return DIT_ERR_ALIGN;
    if (!ld_ok(a.lda, a.K, 2) || !ld_ok(a.ldb, a.K, i8 ? 1 : 2)) return DIT_ERR_INVALID_ARG;
    if (i8 || a.b0_scale) {  // bf16 B may carry row scales too (expanded int8)
        if (!a.b0_scale || !aligned16(a.b0_scale)) return DIT_ERR_ALIGN;
        if (a.mode == DIT_EPI_SWIGLU && (!a.b1_scale || !aligned16(a.b1_scale)))
            return DIT_ERR_ALIGN;
    }
    if (a.qk_norm || a.rope_cos || a.rope_sin) {
        if (a.mode != DIT_EPI_STORE_BF16 && a.mode != DIT_EPI_KV) return DIT_ERR_INVALID_ARG;
        if (a.head_dim != 64 && a.head_dim != 128) return DIT_ERR_INVALID_ARG;
        if (a.N % a.head_dim || (a.mode == DIT_EPI_KV && a.split_n % a.head_dim))
            return DIT_ERR_INVALID_ARG;
        if (!a.rope_cos != !a.rope_sin || a.rope_pos0 < 0) return DIT_ERR_INVALID_ARG;
        if (a.qk_norm && !(a.qk_eps > 0.0f)) return DIT_ERR_INVALID_ARG;
        if (!aligned16(a.qk_norm) || !aligned16(a.rope_cos) || !aligned16(a.rope_sin))
            return DIT_ERR_ALIGN;
    }
    if (a.lora_l0 || a.lora_l1 || a.lora_u0 || a.lora_u1) {
        if ((a.lora_l1 || a.lora_u1) && a.mode != DIT_EPI_SWIGLU) return DIT_ERR_INVALID_ARG;
        auto half_ok = [](const void *u, int64_t ldu, const void *l, int64_t ldl, int r) {
            if (!u && !l) return DIT_OK;
            if (!u || !l || r <= 0 || r > DIT_LORA_MAX_RANK || r % 8) return DIT_ERR_INVALID_ARG;
            if (!ld_ok(ldu, r, 2) || !ld_ok(ldl, r, 2)) return DIT_ERR_INVALID_ARG;
            if (!aligned16(u) || !aligned16(l)) return DIT_ERR_ALIGN;
            return DIT_OK;
        };
        dit_status_t e = half_ok(a.lora_u0, a.lora_ldu0, a.lora_l0, a.lora_ldl0, a.lora_rank0);
        if (e == DIT_OK)
            e = half_ok(a.lora_u1, a.lora_ldu1, a.lora_l1, a.lora_ldl1, a.lora_rank1);
        if (e != DIT_OK) return e;
    }
    if (split && split->slots > 0) {
        if (!split->flags || !split->state || split->slots > kGemmSplitSlots)
            return DIT_ERR_INVALID_ARG;
        if (!aligned16(split->state)) return DIT_ERR_ALIGN;
    }
    if (a.M == 0) return DIT_OK;
    switch (a.mode) {
        case DIT_EPI_STORE_BF16:
            if (!a.out || !aligned16(a.out)) return DIT_ERR_ALIGN;
            if (!ld_ok(a.ldo, a.N, 2)) return DIT_ERR_INVALID_ARG;
            if (a.acc_load) {
                if (!a.acc || !aligned16(a.acc)) return DIT_ERR_ALIGN;
                if (!ld_ok(a.ldacc, a.N, 4)) return DIT_ERR_INVALID_ARG;
            }
            return run_b<DIT_EPI_STORE_BF16>(a, dev_status, s, split);
        case DIT_EPI_STORE_F32:
            if (!a.out || !aligned16(a.out)) return DIT_ERR_ALIGN;
            if (!ld_ok(a.ldo, a.N, 4)) return DIT_ERR_INVALID_ARG;
            return run_b<DIT_EPI_STORE_F32>(a, dev_status, s, split);
        case DIT_EPI_KV:
            if (!a.out || !a.out2 || !aligned16(a.out)) return DIT_ERR_ALIGN;
            if (a.split_n < 0 || a.split_n % 32 || a.split_n > a.N || a.row_offset < 0)
                return DIT_ERR_INVALID_ARG;
            if (!ld_ok(a.ldo, a.split_n, 2) || a.ldo2 < a.row_offset + a.M)
                return DIT_ERR_INVALID_ARG;
            return run_b<DIT_EPI_KV>(a, dev_status, s, split);
        case DIT_EPI_RESID:
            if (!a.x || !a.gate || !aligned16(a.x) || !aligned16(a.gate)) return DIT_ERR_ALIGN;
            if (!ld_ok(a.ldx, a.N, 4)) return DIT_ERR_INVALID_ARG;
            return run_b<DIT_EPI_RESID>(a, dev_status, s, split);
        case DIT_EPI_SWIGLU:
            if (!a.b1 || !aligned16(a.b1) || !a.out || !aligned16(a.out)) return DIT_ERR_ALIGN;
            if (!ld_ok(a.ldo, a.N, 2)) return DIT_ERR_INVALID_ARG;
            return run_b<DIT_EPI_SWIGLU>(a, dev_status, s, split);
        case DIT_EPI_DOWN:
            if (a.acc_final) {
                if (!a.x || !a.gate || !aligned16(a.x) || !aligned16(a.gate))
                    return DIT_ERR_ALIGN;
                if (!ld_ok(a.ldx, a.N, 4)) return DIT_ERR_INVALID_ARG;
            }
            if (a.acc_load || !a.acc_final) {
                if (!a.acc || !aligned16(a.acc)) return DIT_ERR_ALIGN;
                if (!ld_ok(a.ldacc, a.N, 4)) return DIT_ERR_INVALID_ARG;
            }
            return run_b<DIT_EPI_DOWN>(a, dev_status, s, split);
        default:
            return DIT_ERR_INVALID_ARG;
    }
}

}  // namespace ds
