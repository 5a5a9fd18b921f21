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
// large common offset).  All arithmetic is fp32.
//
// Persistent CTAs of 256 threads, one per SM, over tiles of R = 32 * RI token
// rows (RI = 4: 128 rows).  The D axis goes in chunks of 32: the shifted x chunk [R, 32] and the
// modulated W chunk [64, 32] sit in shared memory (double-buffered; the next
// chunk's global loads are in flight in registers while the current one is
// multiplied), and every thread accumulates an RI-row x 8-output register
// tile: the 8 lanes of a row group read the same x float4 (a broadcast) and
// the 4 lanes of an output group the same W float4.
#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace ds {

namespace {

constexpr int kOut = 64;            // output channels
constexpr int kKC = 32;             // k per chunk
constexpr int kLd = kKC + 4;        // padded shared-memory row (floats)
constexpr int kThreads = 256;
constexpr int kWq = kOut * kKC / 4;  // float4s of one W chunk
constexpr int kWper = kWq / kThreads;
static_assert(kWq % kThreads == 0, "each thread stages whole float4s of W");

template <int RI>
struct FinalCfg {
    static constexpr int R = 32 * RI;  // token rows per tile (8 warps x 4 row lanes x RI)
    static constexpr size_t SMEM =
        sizeof(float) * (2 * size_t(R) * kLd + 2 * size_t(kOut) * kLd + 2 * R + 2 * kOut);
};

template <int RI, bool INT8>
__global__ void __launch_bounds__(kThreads, 1)
    final_layer_kernel(const float *__restrict__ x, int64_t T, int D,
                       const void *__restrict__ wf, const float *__restrict__ wscale,
                       const float *__restrict__ mod_f, float *__restrict__ out,
                       int64_t ntiles) {
    using C = FinalCfg<RI>;
    extern __shared__ __align__(16) float sm[];
    float *xs = sm;                     // [2][R][kLd]   shifted x chunk
    float *ws = xs + 2 * C::R * kLd;    // [2][64][kLd]  modulated W chunk
    float *st = ws + 2 * kOut * kLd;    // [R][2]        mean(z), rstd
    float *ce = st + 2 * C::R;          // [64][2]       c_j, e_j
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float *shift = mod_f;
    const float *scale = mod_f + D;
    const int nch = D / kKC;
    // staging roles: float4 column q of the chunk; x rows srow + 32 s; W
    // float4s f = tid + 256 s -> output f / 8, the same column q
    const int q = tid & 7;
    const int srow = tid >> 3;
    // multiply roles: rows 4 RI warp + rg + 4 i, outputs og + 8 jj
    const int rg = lane >> 3, og = lane & 7;
    const int crow = 4 * RI * warp + rg;

    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
        const int64_t row0 = tile * C::R;
        float p[RI], s1[RI], s2[RI];
#pragma unroll
        for (int s = 0; s < RI; ++s) {
            const int64_t t = row0 + srow + 32 * s;
            p[s] = t < T ? __ldg(x + t * D) : 0.f;
            s1[s] = 0.f;
            s2[s] = 0.f;
        }
        float cpart[kWper], epart[kWper];
#pragma unroll
        for (int s = 0; s < kWper; ++s) cpart[s] = epart[s] = 0.f;

        float4 xr[RI], wr[kWper];
        auto load = [&](int c) {
            const int k = c * kKC + 4 * q;
#pragma unroll
            for (int s = 0; s < RI; ++s) {
                const int64_t t = row0 + srow + 32 * s;
                xr[s] = t < T ? __ldcs(reinterpret_cast<const float4 *>(x + t * D + k))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int s = 0; s < kWper; ++s) {
                const int j = (tid + kThreads * s) >> 3;
                if (INT8) {
                    const char4 qv = __ldg(reinterpret_cast<const char4 *>(
                        reinterpret_cast<const int8_t *>(wf) + int64_t(j) * D + k));
                    const float sc = __ldg(wscale + j);
                    wr[s] = make_float4(float(qv.x) * sc, float(qv.y) * sc, float(qv.z) * sc,
                                        float(qv.w) * sc);
                } else {
                    wr[s] = __ldg(reinterpret_cast<const float4 *>(
                        reinterpret_cast<const float *>(wf) + int64_t(j) * D + k));
                }
            }
        };
        // shift x, gather the row sums, modulate W, gather c and e, store
        auto stage = [&](int c, int buf) {
            const int k = c * kKC + 4 * q;
            float *xb = xs + buf * C::R * kLd;
            float *wb = ws + buf * kOut * kLd;
#pragma unroll
            for (int s = 0; s < RI; ++s) {
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
                *reinterpret_cast<float4 *>(xb + (srow + 32 * s) * kLd + 4 * q) = z;
            }
            const float4 sc = __ldg(reinterpret_cast<const float4 *>(scale + k));
            const float4 sh = __ldg(reinterpret_cast<const float4 *>(shift + k));
#pragma unroll
            for (int s = 0; s < kWper; ++s) {
                const int j = (tid + kThreads * s) >> 3;
                const float4 w = wr[s];
                epart[s] = __fmaf_rn(sh.x, w.x, epart[s]);
                epart[s] = __fmaf_rn(sh.y, w.y, epart[s]);
                epart[s] = __fmaf_rn(sh.z, w.z, epart[s]);
                epart[s] = __fmaf_rn(sh.w, w.w, epart[s]);
                const float4 wm = make_float4(w.x * (1.0f + sc.x), w.y * (1.0f + sc.y),
                                              w.z * (1.0f + sc.z), w.w * (1.0f + sc.w));
                cpart[s] += (wm.x + wm.y) + (wm.z + wm.w);
                *reinterpret_cast<float4 *>(wb + j * kLd + 4 * q) = wm;
            }
        };

        float acc[RI][8];
#pragma unroll
        for (int i = 0; i < RI; ++i)
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) acc[i][jj] = 0.f;

        load(0);
        stage(0, 0);
        __syncthreads();
        for (int c = 0; c < nch; ++c) {
            if (c + 1 < nch) load(c + 1);
            const float *xb = xs + (c & 1) * C::R * kLd;
            const float *wb = ws + (c & 1) * kOut * kLd;
#pragma unroll
            for (int k4 = 0; k4 < kKC / 4; ++k4) {
                float4 a[RI], b[8];
#pragma unroll
                for (int i = 0; i < RI; ++i)
                    a[i] = *reinterpret_cast<const float4 *>(xb + (crow + 4 * i) * kLd +
                                                             4 * k4);
#pragma unroll
                for (int jj = 0; jj < 8; ++jj)
                    b[jj] = *reinterpret_cast<const float4 *>(wb + (og + 8 * jj) * kLd +
                                                              4 * k4);
#pragma unroll
                for (int i = 0; i < RI; ++i)
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        acc[i][jj] = __fmaf_rn(a[i].x, b[jj].x, acc[i][jj]);
                        acc[i][jj] = __fmaf_rn(a[i].y, b[jj].y, acc[i][jj]);
                        acc[i][jj] = __fmaf_rn(a[i].z, b[jj].z, acc[i][jj]);
                        acc[i][jj] = __fmaf_rn(a[i].w, b[jj].w, acc[i][jj]);
                    }
            }
            if (c + 1 < nch) stage(c + 1, (c + 1) & 1);
            __syncthreads();
        }

        // the row statistics and c, e: sums over the 8 lanes of a staging
        // group (consecutive lanes, fixed order)
#pragma unroll
        for (int s = 0; s < RI; ++s) {
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
        for (int s = 0; s < kWper; ++s) {
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                cpart[s] += __shfl_xor_sync(0xffffffffu, cpart[s], o);
                epart[s] += __shfl_xor_sync(0xffffffffu, epart[s], o);
            }
            if (q == 0) {
                const int j = (tid + kThreads * s) >> 3;
                ce[2 * j] = cpart[s];
                ce[2 * j + 1] = epart[s];
            }
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < RI; ++i) {
            const int r = crow + 4 * i;
            const int64_t t = row0 + r;
            const float mz = st[2 * r], rs = st[2 * r + 1];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = og + 8 * jj;
                const float v =
                    __fmaf_rn(__fmaf_rn(-mz, ce[2 * j], acc[i][jj]), rs, ce[2 * j + 1]);
                if (t < T) out[t * kOut + j] = v;
            }
        }
        // (the next tile rewrites the statistics only after the barriers of
        // its chunk loop, so these reads are done by then)
    }
}

template <int RI, bool INT8>
dit_status_t run(const float *x, int64_t T, int D, const void *wf, const float *wf_scale,
                 const float *mod_f, float *out, cudaStream_t s) {
    using C = FinalCfg<RI>;
    static std::atomic<unsigned long long> attr_set{0};  // one bit per device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (!bit || !(attr_set.load() & bit)) {
        e = cudaFuncSetAttribute(final_layer_kernel<RI, INT8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::SMEM));
        if (e != cudaSuccess) return cuda_fail(e);
        attr_set.fetch_or(bit);
    }
    const int64_t ntiles = (T + C::R - 1) / C::R;
    const int64_t grid = ntiles < sm_count() ? ntiles : sm_count();
    final_layer_kernel<RI, INT8><<<int(grid), kThreads, C::SMEM, s>>>(
        x, T, D, wf, wf_scale, mod_f, out, ntiles);
    return check_launch();
}

}  // namespace

dit_status_t launch_final(const float *x, int64_t T, int D, const void *wf,
                          const float *wf_scale, const float *mod_f, float *out,
                          cudaStream_t s) {
    if (T < 0 || D <= 0 || D % kKC || !x || !wf || !mod_f || !out) return DIT_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(mod_f) || !aligned16(out) || !aligned16(wf))
        return DIT_ERR_ALIGN;
    if (T == 0) return DIT_OK;
    if (T > (int64_t(1) << 40)) return DIT_ERR_INVALID_ARG;
    return wf_scale ? run<4, true>(x, T, D, wf, wf_scale, mod_f, out, s)
                    : run<4, false>(x, T, D, wf, nullptr, mod_f, out, s);
}

}  // namespace ds
