// Flash-style attention of one query slab against the full K/V on sm_103a.
//
// "LayerStream: H3 Chunking" ("How the slicing works"): every query needs
// every key and value, so pass two attends each query slice to the K and V
// kept for all tokens.  Per CTA: one head and 128 queries; the key loop runs
// over all T keys in tiles of 128, always in ascending order, so a query's
// output does not depend on the slab it belongs to.
//
// Roles (192 threads, one CTA per SM):
//   warp 0      TMA: the Q tile once, then K and V^T tiles into 2-stage rings
//   warp 1      TMEM owner; one lane issues the tcgen05.mma:
//                 S_j  = Q K_j^T  (M=128, N=128, K=d)   -> TMEM S[j%2]
//                 PV_j = P_j V_j  (M=128, N=d,   K=128) -> TMEM PV[j%2]
//   warps 2..5  softmax, one query row per thread: S_j from TMEM, running
//               max and sum in fp32, P_j = exp2(S*log2e/sqrt(d) - m) as bf16
//               into shared memory (128-byte-swizzled K-major, the A operand
//               of the PV MMA), and O = alpha*O + PV_{j-1} in registers.
// S and PV are double-buffered in TMEM so the tensor core computes S_{j+1}
// and PV_j while the softmax threads work on S_j.
//
// V arrives transposed (V^T [H*d, T], written so by the K/V projection's
// epilogue), which makes both MMAs K-major in both operands.
#include "internal.h"
#include "ptx.cuh"

namespace ds {

namespace {

constexpr int kBQ = 128;    // queries per CTA
constexpr int kBKV = 128;   // keys per tile
constexpr int kThreads = 192;

template <int HD>
struct ACfg {
    static constexpr int KS = 2;                         // K stages
    static constexpr int VS = 2;                         // V stages
    static constexpr int Q_BYTES = kBQ * HD * 2;
    static constexpr int K_BYTES = kBKV * HD * 2;
    static constexpr int V_BYTES = HD * kBKV * 2;
    static constexpr int P_BYTES = kBQ * kBKV * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + KS * K_BYTES;
    static constexpr int OFF_P = OFF_V + VS * V_BYTES;
    static constexpr int OFF_BAR = OFF_P + 2 * P_BYTES;
    static constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;
    static constexpr int TMEM_COLS = 512;                 // S0 S1 PV0 PV1
    static constexpr int COL_PV = 2 * kBKV;
};

struct AttnParams {
    int64_t Tq, T;
    int n_kv;
    float scale_log2;  // log2(e) / sqrt(d)
    __nv_bfloat16 *o;
    int64_t ldo;
    int *status;
};

DEV float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
    using C = ACfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
    // bars: q_full, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS],
    //       s_full[2], p_full[2], pv_full[2], drain
    constexpr int B_Q = 0, B_KF = 1, B_KE = B_KF + C::KS, B_VF = B_KE + C::KS,
                  B_VE = B_VF + C::VS, B_SF = B_VE + C::VS, B_PF = B_SF + 2, B_PV = B_PF + 2,
                  B_DR = B_PV + 2, NBAR = B_DR + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NBAR);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const uint32_t bar0 = smem_u32(bars);
    auto bar = [&](int i) { return bar0 + 8u * i; };

    const int warp = warp_id(), lane = lane_id();
    const int qt = blockIdx.x, head = blockIdx.y;
    const int n_kv = p.n_kv;

    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q), 1);
        for (int s = 0; s < C::KS; ++s) {
            mbar_init(bar(B_KF + s), 1);
            mbar_init(bar(B_KE + s), 1);
        }
        for (int s = 0; s < C::VS; ++s) {
            mbar_init(bar(B_VF + s), 1);
            mbar_init(bar(B_VE + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_SF + b), 1);
            mbar_init(bar(B_PF + b), 128);
            mbar_init(bar(B_PV + b), 1);
        }
        mbar_init(bar(B_DR), 1);
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
    const uint32_t sK = smem_u32(sm + C::OFF_K);
    const uint32_t sV = smem_u32(sm + C::OFF_V);
    const uint32_t sP = smem_u32(sm + C::OFF_P);

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            bool ok = true;
            int k_issued = 0, v_issued = 0;
            mbar_arrive_expect_tx(bar(B_Q), C::Q_BYTES);
#pragma unroll
            for (int b = 0; b < HD / 64; ++b)
                tma_load_2d(sQ + b * (kBQ * 128), &tmQ, bar(B_Q), head * HD + 64 * b, qt * kBQ);
            auto load_k = [&](int j) -> bool {
                const int s = j % C::KS;
                if (!mbar_wait(bar(B_KE + s), uint32_t((j / C::KS) & 1) ^ 1u, wc)) return false;
                mbar_arrive_expect_tx(bar(B_KF + s), C::K_BYTES);
                const uint32_t dst = sK + s * C::K_BYTES;
#pragma unroll
                for (int b = 0; b < HD / 64; ++b)
                    tma_load_2d(dst + b * (kBKV * 128), &tmK, bar(B_KF + s), head * HD + 64 * b,
                                j * kBKV);
                ++k_issued;
                return true;
            };
            auto load_v = [&](int j) -> bool {
                const int s = j % C::VS;
                if (!mbar_wait(bar(B_VE + s), uint32_t((j / C::VS) & 1) ^ 1u, wc)) return false;
                mbar_arrive_expect_tx(bar(B_VF + s), C::V_BYTES);
                const uint32_t dst = sV + s * C::V_BYTES;
#pragma unroll
                for (int b = 0; b < kBKV / 64; ++b)
                    tma_load_2d(dst + b * (HD * 128), &tmV, bar(B_VF + s), j * kBKV + 64 * b,
                                head * HD);
                ++v_issued;
                return true;
            };
            ok = load_k(0);
            if (ok && n_kv > 1) ok = load_k(1);
            for (int j = 0; ok && j < n_kv; ++j) {
                ok = load_v(j);
                if (ok && j + 2 < n_kv) ok = load_k(j + 2);
            }
            if (!ok) {  // let the copies in flight land before the CTA exits
                mbar_wait_quiet(bar(B_Q), 0, kWaitLimitNs);
                for (int j = k_issued > C::KS ? k_issued - C::KS : 0; j < k_issued; ++j)
                    mbar_wait_quiet(bar(B_KF + j % C::KS), uint32_t((j / C::KS) & 1),
                                    kWaitLimitNs);
                for (int j = v_issued > C::VS ? v_issued - C::VS : 0; j < v_issued; ++j)
                    mbar_wait_quiet(bar(B_VF + j % C::VS), uint32_t((j / C::VS) & 1),
                                    kWaitLimitNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            constexpr uint32_t ID_S = idesc_bf16_f32(kBQ, kBKV);
            constexpr uint32_t ID_PV = idesc_bf16_f32(kBQ, HD);
            bool ok = mbar_wait(bar(B_Q), 0, wc);
            auto issue_s = [&](int j) -> bool {
                const int s = j % C::KS;
                if (!mbar_wait(bar(B_KF + s), uint32_t((j / C::KS) & 1), wc)) return false;
                tc_fence_after();
                const uint32_t kbase = sK + s * C::K_BYTES;
                const uint32_t d = tmem + uint32_t((j & 1) * kBKV);
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * (kBQ * 128) + (kk & 3) * 32;
                    const uint32_t offk = (kk >> 2) * (kBKV * 128) + (kk & 3) * 32;
                    mma_bf16_ss(d, desc_sw128(sQ + off), desc_sw128(kbase + offk), ID_S,
                                kk > 0);
                }
                mma_commit(bar(B_KE + s));
                mma_commit(bar(B_SF + (j & 1)));
                return true;
            };
            if (ok) ok = issue_s(0);
            if (ok && n_kv > 1) ok = issue_s(1);
            for (int j = 0; ok && j < n_kv; ++j) {
                if (!mbar_wait(bar(B_PF + (j & 1)), uint32_t((j >> 1) & 1), wc)) {
                    ok = false;
                    break;
                }
                const int s = j % C::VS;
                if (!mbar_wait(bar(B_VF + s), uint32_t((j / C::VS) & 1), wc)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t pbase = sP + (j & 1) * C::P_BYTES;
                const uint32_t vbase = sV + s * C::V_BYTES;
                const uint32_t d = tmem + uint32_t(C::COL_PV + (j & 1) * HD);
#pragma unroll
                for (int kk = 0; kk < kBKV / 16; ++kk) {
                    const uint32_t offp = (kk >> 2) * (kBQ * 128) + (kk & 3) * 32;
                    const uint32_t offv = (kk >> 2) * (HD * 128) + (kk & 3) * 32;
                    mma_bf16_ss(d, desc_sw128(pbase + offp), desc_sw128(vbase + offv), ID_PV,
                                kk > 0);
                }
                mma_commit(bar(B_VE + s));
                mma_commit(bar(B_PV + (j & 1)));
                if (j + 2 < n_kv) ok = issue_s(j + 2);
            }
            if (!ok) {
                mma_commit(bar(B_DR));
                mbar_wait_quiet(bar(B_DR), 0, kWaitLimitNs);
            }
        }
    } else {
        // ---------------------------------------------------- softmax
        const int qd = warp & 3;
        const int row = qd * 32 + lane;  // query row within the tile
        const uint32_t lane_base = tmem + (uint32_t(qd * 32) << 16);
        const float sl2 = p.scale_log2;
        float o[HD];
#pragma unroll
        for (int c = 0; c < HD; ++c) o[c] = 0.f;
        float m = -INFINITY, l = 0.f, alpha_prev = 1.f;
        const int last_valid = int(p.T - int64_t(n_kv - 1) * kBKV);  // keys in last tile
        bool ok = true;
        auto consume_pv = [&](int jj, float alpha) -> bool {
            bool w = mbar_wait(bar(B_PV + (jj & 1)), uint32_t((jj >> 1) & 1), wc);
            w = __all_sync(0xffffffffu, w);
            if (!w) return false;
            tc_fence_after();
            const uint32_t pvaddr = lane_base + uint32_t(C::COL_PV + (jj & 1) * HD);
#pragma unroll
            for (int c0 = 0; c0 < HD; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(pvaddr + c0, r);
                tmem_ld_wait(r);
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    o[c0 + c] = __fmaf_rn(o[c0 + c], alpha, __uint_as_float(r[c]));
            }
            return true;
        };
        for (int j = 0; j < n_kv; ++j) {
            bool w = mbar_wait(bar(B_SF + (j & 1)), uint32_t((j >> 1) & 1), wc);
            w = __all_sync(0xffffffffu, w);
            if (!w) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t saddr = lane_base + uint32_t((j & 1) * kBKV);
            const int nvalid = (j == n_kv - 1) ? last_valid : kBKV;
            // pass 1: row max of this tile
            float mx = -INFINITY;
#pragma unroll
            for (int c0 = 0; c0 < kBKV; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(saddr + c0, r);
                tmem_ld_wait(r);
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if (c0 + c < nvalid) mx = fmaxf(mx, __uint_as_float(r[c]));
            }
            const float m_new = fmaxf(m, mx * sl2);
            const float alpha = ex2(m - m_new);  // 0 on the first tile
            // pass 2: probabilities, their sum, bf16 P row into shared memory
            float sum = 0.f;
            const uint32_t prow = sP + (j & 1) * C::P_BYTES + row * 128;
#pragma unroll
            for (int c0 = 0; c0 < kBKV; c0 += 32) {
                uint32_t r[32];
                tmem_ld32(saddr + c0, r);
                tmem_ld_wait(r);
                uint32_t pk[16];
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    float p0 = ex2(__fmaf_rn(__uint_as_float(r[c]), sl2, -m_new));
                    float p1 = ex2(__fmaf_rn(__uint_as_float(r[c + 1]), sl2, -m_new));
                    if (c0 + c >= nvalid) p0 = 0.f;
                    if (c0 + c + 1 >= nvalid) p1 = 0.f;
                    sum += p0 + p1;
                    pk[c >> 1] = pack_bf16x2(p0, p1);
                }
                // 32 keys = 64 bytes = four 16-byte chunks of one 128-byte row
                const uint32_t blk = prow + (c0 >> 6) * (kBQ * 128);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int chunk = ((c0 & 63) >> 3) + u;
                    const uint32_t addr = blk + uint32_t(((chunk ^ (row & 7)) << 4));
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                                 "r"(pk[4 * u]), "r"(pk[4 * u + 1]), "r"(pk[4 * u + 2]),
                                 "r"(pk[4 * u + 3])
                                 : "memory");
                }
            }
            l = __fmaf_rn(l, alpha, sum);
            m = m_new;
            fence_proxy_async_smem();  // P is read by the tensor core (async proxy)
            tc_fence_before();         // S_j reads finish before S_{j+2} overwrites
            mbar_arrive(bar(B_PF + (j & 1)));
            if (j > 0 && !consume_pv(j - 1, alpha_prev)) {
                ok = false;
                break;
            }
            alpha_prev = alpha;
        }
        if (ok && n_kv > 0) ok = consume_pv(n_kv - 1, alpha_prev);
        const int64_t qrow = int64_t(qt) * kBQ + row;
        if (ok && qrow < p.Tq) {
            const float inv = 1.0f / l;
            uint4 *dst = reinterpret_cast<uint4 *>(p.o + qrow * p.ldo + int64_t(head) * HD);
#pragma unroll
            for (int c = 0; c < HD; c += 8) {
                uint4 v;
                v.x = pack_bf16x2(o[c] * inv, o[c + 1] * inv);
                v.y = pack_bf16x2(o[c + 2] * inv, o[c + 3] * inv);
                v.z = pack_bf16x2(o[c + 4] * inv, o[c + 5] * inv);
                v.w = pack_bf16x2(o[c + 6] * inv, o[c + 7] * inv);
                dst[c >> 3] = v;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int HD>
dit_status_t run(const void *q, int64_t Tq, int64_t ldq, const void *k, int64_t ldk,
                 const void *vt, int64_t ldvt, int64_t T, int heads, void *o, int64_t ldo,
                 int *dev_status, cudaStream_t s) {
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
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(
            attn_fwd_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
        if (e != cudaSuccess) return cuda_fail(e);
        attr_done = true;
    }
    const dim3 grid(unsigned((Tq + kBQ - 1) / kBQ), unsigned(heads));
    attn_fwd_kernel<HD><<<grid, kThreads, C::SMEM_BYTES, s>>>(tQ, tK, tV, p);
    return check_launch();
}

}  // namespace

dit_status_t launch_attention(const void *q, int64_t Tq, int64_t ldq, const void *k,
                              int64_t ldk, const void *vt, int64_t ldvt, int64_t T,
                              int heads, int head_dim, void *o, int64_t ldo, int *dev_status,
                              cudaStream_t s) {
    if (Tq < 0 || T <= 0 || heads <= 0 || (head_dim != 64 && head_dim != 128))
        return DIT_ERR_INVALID_ARG;
    if (!q || !k || !vt || !o) return DIT_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o)) return DIT_ERR_ALIGN;
    const int64_t D = int64_t(heads) * head_dim;
    if (ldq < D || ldk < D || ldo < D || ldvt < T) return DIT_ERR_INVALID_ARG;
    if (ldq % 8 || ldk % 8 || ldo % 8 || ldvt % 8) return DIT_ERR_INVALID_ARG;
    if (Tq > (int64_t(1) << 31) - kBQ || T > (int64_t(1) << 31) - kBKV || heads > 65535)
        return DIT_ERR_INVALID_ARG;
    if (Tq == 0) return DIT_OK;
    if (head_dim == 64)
        return run<64>(q, Tq, ldq, k, ldk, vt, ldvt, T, heads, o, ldo, dev_status, s);
    return run<128>(q, Tq, ldq, k, ldk, vt, ldvt, T, heads, o, ldo, dev_status, s);
}

}  // namespace ds
