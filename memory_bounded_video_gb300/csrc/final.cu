// Output head in fp32: out[t, :] = (LN(x[t]) * (1 + scale_f) + shift_f) W_f^T,
// W_f [64, D] fp32, or int8 with one fp32 scale per output row.
// "LayerStream: H3 Chunking" ("How the slicing works"): the fp32 head runs
// unsliced; it is token-wise, so each CTA owns 64 token rows.
//
// Per CTA (256 threads): row statistics (one warp per row, two passes over
// the row), then the D axis in chunks of 64: the normalised-modulated chunk
// and the matching W_f chunk are staged transposed in shared memory and every
// thread accumulates a 4-row x 4-output register tile in ascending k.
#include "internal.h"
#include "ptx.cuh"

namespace ds {

namespace {

constexpr int kRows = 64;    // token rows per CTA
constexpr int kOut = 64;     // output channels
constexpr int kKC = 64;      // k chunk
constexpr int kPad = 68;     // padded row of the transposed tiles (floats)
constexpr int kThreads = 256;

template <bool INT8>
__global__ void __launch_bounds__(kThreads)
    final_layer_kernel(const float *__restrict__ x, int64_t T, int D,
                       const void *__restrict__ wf, const float *__restrict__ wscale,
                       const float *__restrict__ mod_f, float *__restrict__ out) {
    __shared__ __align__(16) float xs[kKC * kPad];  // [k][row]
    __shared__ __align__(16) float ws[kKC * kPad];  // [k][out]
    __shared__ float mean_s[kRows], rstd_s[kRows];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row0 = int64_t(blockIdx.x) * kRows;
    const float *shift = mod_f;
    const float *scale = mod_f + D;

    for (int r = warp; r < kRows; r += kThreads / 32) {
        const int64_t t = row0 + r;
        float mean = 0.f, rstd = 0.f;
        if (t < T) {
            const float4 *xr = reinterpret_cast<const float4 *>(x + t * D);
            float s = 0.f;
            for (int c = lane; c < D / 4; c += 32) {
                const float4 v = xr[c];
                s += (v.x + v.y) + (v.z + v.w);
            }
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            mean = s / float(D);
            float q = 0.f;
            for (int c = lane; c < D / 4; c += 32) {
                const float4 v = xr[c];
                const float a = v.x - mean, b = v.y - mean, cc = v.z - mean, d = v.w - mean;
                q += (a * a + b * b) + (cc * cc + d * d);
            }
            for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
            rstd = rsqrtf(q / float(D) + 1e-6f);
        }
        if (lane == 0) {
            mean_s[r] = mean;
            rstd_s[r] = rstd;
        }
    }
    __syncthreads();

    const int rg = tid >> 4;   // rows rg*4 .. rg*4+3
    const int og = tid & 15;   // outputs og*4 .. og*4+3
    float acc[4][4] = {};
    for (int k0 = 0; k0 < D; k0 += kKC) {
        // stage the modulated-normalised x chunk and the W chunk, transposed
        for (int i = tid; i < kRows * (kKC / 4); i += kThreads) {
            const int r = i / (kKC / 4), c4 = i % (kKC / 4);
            const int64_t t = row0 + r;
            const int k = k0 + 4 * c4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < T) {
                const float4 xv = *reinterpret_cast<const float4 *>(x + t * D + k);
                const float4 sc = __ldg(reinterpret_cast<const float4 *>(scale + k));
                const float4 sh = __ldg(reinterpret_cast<const float4 *>(shift + k));
                const float m = mean_s[r], rs = rstd_s[r];
                v.x = __fmaf_rn((xv.x - m) * rs, 1.0f + sc.x, sh.x);
                v.y = __fmaf_rn((xv.y - m) * rs, 1.0f + sc.y, sh.y);
                v.z = __fmaf_rn((xv.z - m) * rs, 1.0f + sc.z, sh.z);
                v.w = __fmaf_rn((xv.w - m) * rs, 1.0f + sc.w, sh.w);
            }
            xs[(4 * c4 + 0) * kPad + r] = v.x;
            xs[(4 * c4 + 1) * kPad + r] = v.y;
            xs[(4 * c4 + 2) * kPad + r] = v.z;
            xs[(4 * c4 + 3) * kPad + r] = v.w;
        }
        for (int i = tid; i < kOut * (kKC / 4); i += kThreads) {
            const int o = i / (kKC / 4), c4 = i % (kKC / 4);
            const int k = k0 + 4 * c4;
            float4 w;
            if (INT8) {
                const char4 qv = *reinterpret_cast<const char4 *>(
                    reinterpret_cast<const int8_t *>(wf) + int64_t(o) * D + k);
                const float s = __ldg(wscale + o);
                w = make_float4(float(qv.x) * s, float(qv.y) * s, float(qv.z) * s,
                                float(qv.w) * s);
            } else {
                w = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(wf) +
                                                      int64_t(o) * D + k);
            }
            ws[(4 * c4 + 0) * kPad + o] = w.x;
            ws[(4 * c4 + 1) * kPad + o] = w.y;
            ws[(4 * c4 + 2) * kPad + o] = w.z;
            ws[(4 * c4 + 3) * kPad + o] = w.w;
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < kKC; ++k) {
            const float4 a = *reinterpret_cast<const float4 *>(xs + k * kPad + 4 * rg);
            const float4 b = *reinterpret_cast<const float4 *>(ws + k * kPad + 4 * og);
            const float av[4] = {a.x, a.y, a.z, a.w};
            const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = __fmaf_rn(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t t = row0 + 4 * rg + i;
        if (t < T)
            *reinterpret_cast<float4 *>(out + t * kOut + 4 * og) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    }
}

}  // namespace

dit_status_t launch_final(const float *x, int64_t T, int D, const void *wf,
                          const float *wf_scale, const float *mod_f, float *out,
                          cudaStream_t s) {
    if (T < 0 || D <= 0 || D % kKC || !x || !wf || !mod_f || !out) return DIT_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(mod_f) || !aligned16(out) || !aligned16(wf))
        return DIT_ERR_ALIGN;
    if (T == 0) return DIT_OK;
    const int64_t grid = (T + kRows - 1) / kRows;
    if (grid > 0x7fffffff) return DIT_ERR_INVALID_ARG;
    if (wf_scale)
        final_layer_kernel<true><<<int(grid), kThreads, 0, s>>>(x, T, D, wf, wf_scale, mod_f,
                                                                out);
    else
        final_layer_kernel<false><<<int(grid), kThreads, 0, s>>>(x, T, D, wf, nullptr, mod_f,
                                                                 out);
    return check_launch();
}

}  // namespace ds
