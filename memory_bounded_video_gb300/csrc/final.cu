// Output head in fp32: out[t, :] = (LN(x[t]) * (1 + scale_f) + shift_f) W_f^T,
// W_f [64, D] fp32, or int8 with one fp32 scale per output row.
// "LayerStream: H3 Chunking" ("How the slicing works"): the fp32 head runs
// unsliced; it is token-wise, so each CTA owns 64 token rows.
//
// Per CTA (256 threads): row statistics (one warp per row, two passes over
// the row), then the D axis in chunks of 64: the normalised-modulated chunk
// and the matching W_f chunk are staged transposed in shared memory (each
// thread one 4 x 4 block of each) and every thread accumulates a 4-row x
// 4-output register tile in ascending k.
#include "internal.h"
#include "ptx.cuh"

namespace ds {

namespace {

constexpr int kRows = 64;    // token rows per CTA
constexpr int kOut = 64;     // output channels
constexpr int kKC = 64;      // k chunk
constexpr int kPad = 68;     // padded row of the transposed tiles (floats)
constexpr int kThreads = 256;
static_assert(kRows == 64 && kOut == 64 && kKC == 64 && kThreads == 256,
              "each thread stages one 4 x 4 block of the x and W chunks");

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
        // stage the modulated-normalised x chunk and the W chunk, transposed.
        // Thread tid owns a 4 x 4 block of each (rows or outputs 4 (tid % 16)
        // .., k 4 (tid / 16) ..): four 16-byte loads (the two half-warps
        // read the two halves of each 32-byte sector) and four 16-byte
        // shared stores, which hit distinct banks within each quarter-warp
        // (one scalar store per element, with consecutive threads 272 floats
        // apart, collided eight ways).
        {
            const int b4 = (tid & 15) * 4;  // first row / output of the block
            const int c4 = tid >> 4;        // k = k0 + 4 c4 .. + 3
            const int k = k0 + 4 * c4;
            float v[4][4];
            const float4 sc = __ldg(reinterpret_cast<const float4 *>(scale + k));
            const float4 sh = __ldg(reinterpret_cast<const float4 *>(shift + k));
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int r = b4 + i;
                const int64_t t = row0 + r;
                float4 xv = make_float4(0.f, 0.f, 0.f, 0.f);
                if (t < T) {
                    xv = *reinterpret_cast<const float4 *>(x + t * D + k);
                    const float m = mean_s[r], rs = rstd_s[r];
                    xv.x = __fmaf_rn((xv.x - m) * rs, 1.0f + sc.x, sh.x);
                    xv.y = __fmaf_rn((xv.y - m) * rs, 1.0f + sc.y, sh.y);
                    xv.z = __fmaf_rn((xv.z - m) * rs, 1.0f + sc.z, sh.z);
                    xv.w = __fmaf_rn((xv.w - m) * rs, 1.0f + sc.w, sh.w);
                }
                v[0][i] = xv.x;
                v[1][i] = xv.y;
                v[2][i] = xv.z;
                v[3][i] = xv.w;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<float4 *>(xs + (4 * c4 + j) * kPad + b4) =
                    make_float4(v[j][0], v[j][1], v[j][2], v[j][3]);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int o = b4 + i;
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
                v[0][i] = w.x;
                v[1][i] = w.y;
                v[2][i] = w.z;
                v[3][i] = w.w;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                *reinterpret_cast<float4 *>(ws + (4 * c4 + j) * kPad + b4) =
                    make_float4(v[j][0], v[j][1], v[j][2], v[j][3]);
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
