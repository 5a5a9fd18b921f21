// Output head in fp32: out[t, :] = (LN(x[t]) * (1 + scale_f) + shift_f) W_f^T,
// W_f [64, D] fp32, or int8 with one fp32 scale per output row.
// "LayerStream: H3 Chunking" ("How the slicing works"): the fp32 head runs
// unsliced; it is token-wise, so each tile of token rows is independent.
//
// One read of x.  With y_k = (x_k - mean) * rstd * (1 + scale_k) + shift_k,
//   out_j = sum_k y_k W_jk
//         = rstd * (sum_k z_k W'_jk - mean(z) * c_j) + e_j,
// where z_k = x_k - p is the row shifted by its first element p, W'_jk =
// (1 + scale_k) W_jk, c_j = sum_k W'_jk and e_j = sum_k shift_k W_jk: the
// same sum in exact arithmetic, rearranged so the contraction starts before
// the row's statistics are known.  The row's mean and variance come from the
// shifted sums sum z and sum z^2 gathered while the row is staged (the
// shifted-data form of the variance: the shift keeps mean(z) of the order of
// the row's spread, so the subtractions lose nothing even when the row has a
// large common offset).
//
// The contraction sum_k z_k W'_jk runs on the tensor cores at fp32-level
// precision: each operand is split into two tf32 parts (v = hi + lo, hi =
// v rounded to tf32, lo = v - hi rounded to tf32, so hi + lo carries about
// 22 significant bits) and three products are accumulated in fp32 in
// tensor memory by two tcgen05.mma.kind::tf32 per k step: hi_z [W'hi; W'lo]
// (N = 128: hi_z W'hi and hi_z W'lo side by side) and lo_z W'hi (N = 64,
// onto hi_z W'hi); the dropped lo_z W'lo term is below 2^-22 of each
// product.  The tensor-memory accumulator only ever holds a partial sum over
// 128 values of k: the partials are added in fp32 registers, round-to-
// nearest, so the long sum over D is not left to the accumulator
// (accumulating all of D there measured 25 times the error of an fp32 FMA
// loop against the float64 oracle).  Statistics, modulation, the final
// combination and the output are fp32 CUDA-core work.
//
// Persistent CTAs, one per SM, over 128-row tiles (the MMA's M = 128, N = 64
// outputs).  Warps 0..7 stage: per 32-wide k chunk they copy their pieces of
// x and W_f from global memory into a raw shared-memory ring (cp.async, two
// chunks ahead), read them back, shift, gather the row sums, modulate, split
// and store the four operand tiles of a shared-memory ring stage in the
// 128-byte-swizzle K-major layout.  Warps 8..11 (one accumulator row per
// thread) add each finished partial from tensor memory (two 128-column
// buffers, allocated by warp 8) into registers and, after a tile's last
// partial, combine and write out; warp 8's lane 0 also issues the MMAs.
// Twelve warps (three per SM sub-partition) leave each thread up to 168
// registers; a thirteenth warp for the MMAs would cap every thread at 128.
#include "internal.h"
#include "ptx.cuh"

namespace ds {

namespace {

constexpr int kOut = 64;                    // output channels (MMA N)
constexpr int kRows = 128;                  // token rows per tile (MMA M)
constexpr int kKC = 32;                     // k per chunk: one 128-byte fp32 row
constexpr int kStages = 3;                  // operand ring depth
constexpr int kStagers = 256;               // warps 0..7
constexpr int kThreads = 384;               // 8..11: partial sums; 8 also MMA issuer
constexpr int kDrain = 4;                   // chunks per tensor-memory partial sum
constexpr int kPartCols = 2 * kOut;         // a partial: hi*hi + lo*hi | hi*lo
constexpr int kTmemCols = 2 * kPartCols;    // two partial-sum buffers
constexpr int kATile = kRows * 128;         // one split part of the x chunk
constexpr int kBTile = kOut * 128;          // one split part of the W chunk
constexpr int kStageBytes = 2 * kATile + 2 * kBTile;
constexpr int kRaw = 3;                     // chunks of raw x and W in flight
constexpr int kPieces = 6;                  // per stager and chunk: 4 of x, 2 of W
constexpr int kRawBytes = kPieces * kStagers * 16;  // one chunk, [piece][stager] x 16 B
constexpr int kOffRaw = kStages * kStageBytes;
constexpr int kOffSt = kOffRaw + kRaw * kRawBytes;  // [128][2] mean(z), rstd
constexpr int kOffCe = kOffSt + kRows * 8;          // [64][2]  c_j, e_j
constexpr int kOffBar = kOffCe + kOut * 8;
// barriers: full[3], empty[3], tfull[2], tempty[2], drain, stats_ready,
// stats_free; then the TMEM slot and the abort flag
constexpr int kNumBars = 2 * kStages + 7;
constexpr int kSmemBytes = kOffBar + 8 * kNumBars + 16 + 1024;
static_assert(kStageBytes % 1024 == 0 && kATile % 1024 == 0 && kBTile % 1024 == 0,
              "operand tiles start on 1024-byte swizzle atoms");
static_assert(kSmemBytes <= 232448, "shared memory");

// Instruction descriptor, kind::tf32: D = f32, A = B = tf32, both K-major,
// dense; N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(N >> 3) << 17) |
           (uint32_t(M >> 4) << 24);
}

template <uint32_t IDESC>
DEV void mma_tf32_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(IDESC), "r"(accumulate)
        : "memory");
}

DEV float tf32_rna(float v) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return __uint_as_float(r);
}

// v -> (hi, lo) tf32 parts, written to the two tiles at byte offset `off`.
DEV void split_store(uint8_t *hi_tile, uint8_t *lo_tile, int off, float4 v) {
    float4 h, l;
    h.x = tf32_rna(v.x);
    h.y = tf32_rna(v.y);
    h.z = tf32_rna(v.z);
    h.w = tf32_rna(v.w);
    l.x = tf32_rna(v.x - h.x);
    l.y = tf32_rna(v.y - h.y);
    l.z = tf32_rna(v.z - h.z);
    l.w = tf32_rna(v.w - h.w);
    *reinterpret_cast<float4 *>(hi_tile + off) = h;
    *reinterpret_cast<float4 *>(lo_tile + off) = l;
}

// 16 consecutive 32-bit columns of this thread's TMEM lane, waited for.
DEV void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
          "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Asynchronous copies global -> shared (bypassing the registers): 16 bytes
// (zero-filled when src_bytes is 0) or 4 bytes.
DEV void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(src_bytes)
                 : "memory");
}
DEV void cp_async4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
DEV void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Byte offset of 16-byte chunk q of row r in a 128-byte-swizzle K-major tile.
DEV int sw128(int r, int q) { return (r >> 3) * 1024 + (r & 7) * 128 + ((q ^ (r & 7)) << 4); }

template <bool INT8>
__global__ void __launch_bounds__(kThreads, 1)
    final_layer_kernel(const float *__restrict__ x, int64_t T, int D,
                       const void *__restrict__ wf, const float *__restrict__ wscale,
                       const float *__restrict__ mod_f, float *__restrict__ out,
                       int64_t ntiles, int *status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kNumBars);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *st = reinterpret_cast<float *>(sm + kOffSt);
    float *ce = reinterpret_cast<float *>(sm + kOffCe);
    const uint32_t bar0 = smem_u32(bars);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kStages + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kStages + 4);
    const uint32_t ready_bar = bar0 + 8u * (2 * kStages + 5);  // statistics written
    const uint32_t free_bar = bar0 + 8u * (2 * kStages + 6);   // statistics read
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), kStagers);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 128);
        }
        mbar_init(drain_bar, 1);
        mbar_init(ready_bar, kStagers);
        mbar_init(free_bar, 128);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 8) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtx wc{abort_flag, status};
    const int nch = D / kKC;
    const int nparts = (nch + kDrain - 1) / kDrain;  // partial sums per tile

    if (warp < 8) {
        // ---------------------------------------------------- stagers
        // x chunk: float4 column q of rows srow + 32 s; W chunk: float4
        // column q of outputs (tid + 256 s) / 8
        const float *shift = mod_f;
        const float *scale = mod_f + D;
        const int q = tid & 7;
        const int srow = tid >> 3;
        int stage = 0;
        uint32_t ph = 0;
        bool ok = true;
        int ti = 0;
        for (int64_t tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++ti) {
            const int64_t row0 = tile * kRows;
            float p[4], s1[4], s2[4], cpart[2], epart[2];
#pragma unroll
            for (int s = 0; s < 4; ++s) {
                const int64_t t = row0 + srow + 32 * s;
                p[s] = t < T ? __ldg(x + t * D) : 0.f;
                s1[s] = 0.f;
                s2[s] = 0.f;
            }
            cpart[0] = cpart[1] = epart[0] = epart[1] = 0.f;

            // chunk c's raw x and W pieces of this thread into raw slot c % kRaw
            // (every thread reads back only what it copied itself)
            const uint32_t raw0 = smem_u32(sm + kOffRaw) + 16u * tid;
            auto fetch = [&](int c) {
                if (c < nch) {
                    const uint32_t slot = raw0 + uint32_t((c % kRaw) * kRawBytes);
                    const int k = c * kKC + 4 * q;
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        const int64_t t = row0 + srow + 32 * s;
                        cp_async16(slot + uint32_t(s * kStagers * 16),
                                   t < T ? x + t * D + k : x, t < T ? 16u : 0u);
                    }
#pragma unroll
                    for (int s = 0; s < 2; ++s) {
                        const int j = (tid + kStagers * s) >> 3;
                        const uint32_t dst = slot + uint32_t((4 + s) * kStagers * 16);
                        if (INT8)
                            cp_async4(dst, reinterpret_cast<const int8_t *>(wf) + int64_t(j) * D + k);
                        else
                            cp_async16(dst, reinterpret_cast<const float *>(wf) + int64_t(j) * D + k,
                                       16u);
                    }
                }
                cp_async_commit();  // an empty group past the end keeps the count
            };
            // chunk c from the raw slot into registers (its copies are done)
            auto take = [&](int c, float4 (&xr)[4], float4 (&wr)[2]) {
                const uint8_t *slot = sm + kOffRaw + (c % kRaw) * kRawBytes + 16 * tid;
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    xr[s] = *reinterpret_cast<const float4 *>(slot + s * kStagers * 16);
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    const uint8_t *src = slot + (4 + s) * kStagers * 16;
                    if (INT8) {
                        const char4 qv = *reinterpret_cast<const char4 *>(src);
                        const float sc = __ldg(wscale + ((tid + kStagers * s) >> 3));
                        wr[s] = make_float4(float(qv.x) * sc, float(qv.y) * sc,
                                            float(qv.z) * sc, float(qv.w) * sc);
                    } else {
                        wr[s] = *reinterpret_cast<const float4 *>(src);
                    }
                }
            };
            // one chunk from registers into ring stage `stage`
            auto put = [&](int c, const float4 (&xr)[4], const float4 (&wr)[2]) -> bool {
                bool w = mbar_wait(empty_bar(stage), ph ^ 1u, wc);  // its MMAs are done
                if (!__all_sync(0xffffffffu, w)) return false;
                uint8_t *s0 = sm + stage * kStageBytes;
#pragma unroll
                for (int s = 0; s < 4; ++s) {
                    float4 z = xr[s];
                    z.x -= p[s];
                    z.y -= p[s];
                    z.z -= p[s];
                    z.w -= p[s];
                    s1[s] += (z.x + z.y) + (z.z + z.w);
                    s2[s] = __fmaf_rn(z.x, z.x, s2[s]);
                    s2[s] = __fmaf_rn(z.y, z.y, s2[s]);
                    s2[s] = __fmaf_rn(z.z, z.z, s2[s]);
                    s2[s] = __fmaf_rn(z.w, z.w, s2[s]);
                    split_store(s0, s0 + kATile, sw128(srow + 32 * s, q), z);
                }
                const int k = c * kKC + 4 * q;
                const float4 sc = __ldg(reinterpret_cast<const float4 *>(scale + k));
                const float4 sh = __ldg(reinterpret_cast<const float4 *>(shift + k));
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    const int j = (tid + kStagers * s) >> 3;
                    const float4 wv = wr[s];
                    epart[s] = __fmaf_rn(sh.x, wv.x, epart[s]);
                    epart[s] = __fmaf_rn(sh.y, wv.y, epart[s]);
                    epart[s] = __fmaf_rn(sh.z, wv.z, epart[s]);
                    epart[s] = __fmaf_rn(sh.w, wv.w, epart[s]);
                    const float4 wm = make_float4(wv.x * (1.0f + sc.x), wv.y * (1.0f + sc.y),
                                                  wv.z * (1.0f + sc.z), wv.w * (1.0f + sc.w));
                    cpart[s] += (wm.x + wm.y) + (wm.z + wm.w);
                    split_store(s0 + 2 * kATile, s0 + 2 * kATile + kBTile, sw128(j, q), wm);
                }
                fence_proxy_async_smem();  // the tensor core reads what we wrote
                mbar_arrive(full_bar(stage));
                if (++stage == kStages) {
                    stage = 0;
                    ph ^= 1u;
                }
                return true;
            };

            // kRaw - 1 chunks in flight ahead of the one being stored
#pragma unroll
            for (int c = 0; c < kRaw - 1; ++c) fetch(c);
            for (int c = 0; ok && c < nch; ++c) {
                fetch(c + kRaw - 1);
                cp_async_wait<kRaw - 1>();  // chunk c's group is complete
                float4 xr[4], wr[2];
                take(c, xr, wr);
                ok = put(c, xr, wr);
            }
            if (!ok) {
                cp_async_wait<0>();  // no copy lands after the CTA has left
                break;
            }

            // the row statistics and c, e: sums over the 8 lanes of a staging
            // group (consecutive lanes, fixed order), written once the
            // previous tile's epilogue has read them
            if (ti > 0) {
                const bool w = mbar_wait(free_bar, uint32_t((ti - 1) & 1), wc);
                if (!__all_sync(0xffffffffu, w)) break;
            }
#pragma unroll
            for (int s = 0; s < 4; ++s) {
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    s1[s] += __shfl_xor_sync(0xffffffffu, s1[s], o);
                    s2[s] += __shfl_xor_sync(0xffffffffu, s2[s], o);
                }
                if (q == 0) {
                    const float mz = s1[s] / float(D);
                    const float var = fmaxf(s2[s] / float(D) - mz * mz, 0.f);
                    st[2 * (srow + 32 * s)] = mz;
                    st[2 * (srow + 32 * s) + 1] = rsqrtf(var + 1e-6f);
                }
            }
#pragma unroll
            for (int s = 0; s < 2; ++s) {
#pragma unroll
                for (int o = 1; o < 8; o <<= 1) {
                    cpart[s] += __shfl_xor_sync(0xffffffffu, cpart[s], o);
                    epart[s] += __shfl_xor_sync(0xffffffffu, epart[s], o);
                }
                if (q == 0) {
                    const int j = (tid + kStagers * s) >> 3;
                    ce[2 * j] = cpart[s];
                    ce[2 * j + 1] = epart[s];
                }
            }
            mbar_arrive(ready_bar);
        }
    } else {
        // ---------------------------------------------- partial sums, output
        // warps 8..11: thread = accumulator row 32 (warp % 4) + lane (the
        // warp's TMEM lane quadrant).  Warp 8's lane 0 also issues the MMAs;
        // warp 8 sums a partial once the next partial's first chunk is issued
        // (the tile's last one after its last chunk), so the tensor core has
        // work queued while it waits.
        const bool issuer = warp == 8;
        const int r = 32 * (warp & 3) + lane;
        const uint32_t lane_base = tmem + (uint32_t(32 * (warp & 3)) << 16);
        int stage = 0;         // issuer: ring position
        uint32_t ph = 0;
        int64_t pi_iss = 0;    // issuer: partials started
        int64_t pi = 0;        // partials summed by this warp
        bool ok = true;
        float acc[kOut];
        // add partial pi of this warp's quadrant to acc (warp-collective)
        auto sum_partial = [&]() -> bool {
            const int buf = int(pi & 1);
            const bool w = mbar_wait(tfull_bar(buf), uint32_t((pi >> 1) & 1), wc);
            if (!__all_sync(0xffffffffu, w)) return false;
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < kOut; c0 += 16) {
                uint32_t v[16], u[16];
                tmem_ld16(lane_base + uint32_t(buf * kPartCols + c0), v);
                tmem_ld16(lane_base + uint32_t(buf * kPartCols + kOut + c0), u);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    acc[c0 + j] += __uint_as_float(v[j]) + __uint_as_float(u[j]);
            }
            tc_fence_before();
            mbar_arrive(tempty_bar(buf));
            ++pi;
            return true;
        };
        // the MMAs of chunk c: a partial's first chunk starts its buffer
        // afresh once the buffer's previous partial has been summed by all
        // four warps; its last chunk signals the buffer full
        auto issue = [&](int c) -> bool {
            const int c_in = c % kDrain;
            const int buf = int(pi_iss & 1);
            if (c_in == 0 && pi_iss >= 2) {
                if (!mbar_wait(tempty_bar(buf), uint32_t(((pi_iss >> 1) - 1) & 1), wc))
                    return false;
                tc_fence_after();
            }
            if (!mbar_wait(full_bar(stage), ph, wc)) return false;
            tc_fence_after();
            const uint32_t s0 = smem_u32(sm + stage * kStageBytes);
            const uint32_t d = tmem + uint32_t(buf * kPartCols);
#pragma unroll
            for (int k = 0; k < kKC / 8; ++k) {  // K = 8 tf32 = 32 bytes per MMA
                const uint64_t ahi = desc_sw128(s0 + 32u * k);
                const uint64_t alo = desc_sw128(s0 + kATile + 32u * k);
                // W'hi rows then W'lo rows: one N = 128 operand
                const uint64_t bhl = desc_sw128(s0 + 2 * kATile + 32u * k);
                const uint32_t acc = (c_in > 0 || k > 0) ? 1u : 0u;
                mma_tf32_ss<idesc_tf32(kRows, 2 * kOut)>(d, ahi, bhl, acc);
                mma_tf32_ss<idesc_tf32(kRows, kOut)>(d, alo, bhl, 1u);
            }
            mma_commit(empty_bar(stage));
            if (++stage == kStages) {
                stage = 0;
                ph ^= 1u;
            }
            if (c_in == kDrain - 1 || c == nch - 1) {
                mma_commit(tfull_bar(buf));
                ++pi_iss;
            }
            return true;
        };
        int ti = 0;
        for (int64_t tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++ti) {
#pragma unroll
            for (int j = 0; j < kOut; ++j) acc[j] = 0.f;
            if (issuer) {
                for (int c = 0; ok && c < nch; ++c) {
                    bool w = true;
                    if (lane == 0) w = issue(c);
                    ok = __all_sync(0xffffffffu, w);
                    if (ok && c % kDrain == 0 && c > 0) ok = sum_partial();
                }
                if (ok) ok = sum_partial();  // the tile's last partial
            } else {
                for (int part = 0; ok && part < nparts; ++part) ok = sum_partial();
            }
            if (!ok) break;
            const bool w = mbar_wait(ready_bar, uint32_t(ti & 1), wc);
            if (!__all_sync(0xffffffffu, w)) {
                ok = false;
                break;
            }
            const int64_t t = tile * kRows + r;
            const float mz = st[2 * r], rs = st[2 * r + 1];
            if (t < T) {
                float4 *dst = reinterpret_cast<float4 *>(out + t * kOut);
#pragma unroll
                for (int i = 0; i < kOut / 4; ++i) {
                    float o[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int j = 4 * i + u;
                        o[u] = __fmaf_rn(__fmaf_rn(-mz, ce[2 * j], acc[j]), rs, ce[2 * j + 1]);
                    }
                    dst[i] = make_float4(o[0], o[1], o[2], o[3]);
                }
            }
            mbar_arrive(free_bar);
        }
        if (issuer && !ok && lane == 0) {  // every issued MMA finishes before the memory is freed
            mma_commit(drain_bar);
            mbar_wait_quiet(drain_bar, 0, kWaitLimitNs);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <bool INT8>
dit_status_t run(const float *x, int64_t T, int D, const void *wf, const float *wf_scale,
                 const float *mod_f, float *out, int *status, cudaStream_t s) {
    static int attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(final_layer_kernel<INT8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
        if (e != cudaSuccess) return cuda_fail(e);
        if (dev >= 0 && dev < 64) attr_set[dev] = 1;  // the same value from any thread
    }
    const int64_t ntiles = (T + kRows - 1) / kRows;
    const int64_t grid = ntiles < sm_count() ? ntiles : sm_count();
    final_layer_kernel<INT8><<<int(grid), kThreads, kSmemBytes, s>>>(x, T, D, wf, wf_scale,
                                                                       mod_f, out, ntiles, status);
    return check_launch();
}

}  // namespace

dit_status_t launch_final(const float *x, int64_t T, int D, const void *wf,
                          const float *wf_scale, const float *mod_f, float *out,
                          int *dev_status, cudaStream_t s) {
    if (T < 0 || D <= 0 || D % kKC || !x || !wf || !mod_f || !out) return DIT_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(mod_f) || !aligned16(out) || !aligned16(wf))
        return DIT_ERR_ALIGN;
    if (T == 0) return DIT_OK;
    if (T > (int64_t(1) << 40)) return DIT_ERR_INVALID_ARG;
    return wf_scale ? run<true>(x, T, D, wf, wf_scale, mod_f, out, dev_status, s)
                    : run<false>(x, T, D, wf, nullptr, mod_f, out, dev_status, s);
}

}  // namespace ds
