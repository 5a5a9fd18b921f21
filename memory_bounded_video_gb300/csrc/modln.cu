// Norm + modulation + cast of token rows.
//   y = (x - mean) * rsqrt(var + 1e-6) * (1 + scale) + shift  -> bf16 (RNE)
// Token-wise ("LayerStream: H3 Chunking", "How the slicing works"), HBM-bound:
// 4*D bytes read and 2*D bytes written per row.  The row lives in the
// registers of the warps that share it, mean and biased variance come from
// warp-shuffle reductions and a fixed-order combination of the warps'
// partial sums, so a row's result is the same whichever slab it is
// processed in.
#include "internal.h"
#include "ptx.cuh"

namespace ds {

namespace {

constexpr int kWarpsPerBlock = 8;

// W warps share a row (W divides NV): warp j of the row's group holds float4
// columns [j*NV/W*32, (j+1)*NV/W*32) in registers (NV/W per lane, 128-bit
// coalesced loads); the W partial sums of the mean and of the squared
// deviations are combined through shared memory in the same fixed order for
// every row.  Few registers per thread leave several blocks per SM, so many
// rows are in flight (a whole 3072-wide row per warp needed 185 registers
// and allowed one block per SM: 4.4 TB/s).
template <int NV, int W>
__global__ void __launch_bounds__(32 * kWarpsPerBlock)
    modln_cast_kernel(const float *__restrict__ x, int64_t rows, const float *__restrict__ shift,
                      const float *__restrict__ scale, __nv_bfloat16 *__restrict__ out) {
    constexpr int D = NV * 128;
    constexpr int RB = kWarpsPerBlock / W;  // rows per block and step
    constexpr int PV = NV / W;              // float4 per lane
    __shared__ float red[2][kWarpsPerBlock];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = warp / W, j = warp % W;
    const int c4_0 = j * PV * 32 + lane;
    for (int64_t base = int64_t(blockIdx.x) * RB; base < rows;
         base += int64_t(gridDim.x) * RB) {
        const int64_t r = base + g;
        const bool on = r < rows;
        const float4 *xr = reinterpret_cast<const float4 *>(x + r * D);
        float4 v[PV];
#pragma unroll
        for (int i = 0; i < PV; ++i)
            v[i] = on ? __ldcs(xr + c4_0 + 32 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < PV; ++i) s += (v[i].x + v[i].y) + (v[i].z + v[i].w);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) red[0][warp] = s;
        __syncthreads();
        float st = 0.f;
#pragma unroll
        for (int k = 0; k < W; ++k) st += red[0][g * W + k];
        const float mean = st * (1.0f / D);
        float q = 0.f;
#pragma unroll
        for (int i = 0; i < PV; ++i) {
            const float a = v[i].x - mean, b = v[i].y - mean, c = v[i].z - mean,
                        d = v[i].w - mean;
            q += (a * a + b * b) + (c * c + d * d);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
        if (lane == 0) red[1][warp] = q;
        __syncthreads();
        float qt = 0.f;
#pragma unroll
        for (int k = 0; k < W; ++k) qt += red[1][g * W + k];
        const float rstd = rsqrtf(qt * (1.0f / D) + 1e-6f);
        if (on) {
            uint2 *orow = reinterpret_cast<uint2 *>(out + r * D);
#pragma unroll
            for (int i = 0; i < PV; ++i) {
                const int c4 = c4_0 + 32 * i;
                const float4 sc = __ldg(reinterpret_cast<const float4 *>(scale) + c4);
                const float4 sh = __ldg(reinterpret_cast<const float4 *>(shift) + c4);
                const float y0 = __fmaf_rn((v[i].x - mean) * rstd, 1.0f + sc.x, sh.x);
                const float y1 = __fmaf_rn((v[i].y - mean) * rstd, 1.0f + sc.y, sh.y);
                const float y2 = __fmaf_rn((v[i].z - mean) * rstd, 1.0f + sc.z, sh.z);
                const float y3 = __fmaf_rn((v[i].w - mean) * rstd, 1.0f + sc.w, sh.w);
                uint2 pk;
                pk.x = pack_bf16x2(y0, y1);
                pk.y = pack_bf16x2(y2, y3);
                orow[c4] = pk;
            }
        }
        __syncthreads();  // red is reused by the next step
    }
}

// warps per row: 4 where it divides NV (wide rows), else 2, else 1
template <int NV>
constexpr int warps_per_row() {
    return NV % 4 == 0 ? 4 : (NV % 2 == 0 ? 2 : 1);
}

template <int NV>
dit_status_t run(const float *x, int64_t rows, const float *shift, const float *scale,
                 void *out, cudaStream_t s) {
    constexpr int W = warps_per_row<NV>();
    constexpr int RB = kWarpsPerBlock / W;
    const int64_t blocks_needed = (rows + RB - 1) / RB;
    // one wave of resident blocks, each looping over row groups: a second,
    // partial wave of block launches measured 4 % slower (24.8 against 23.7
    // us for 8192 x 3072)
    static int per_sm = 0;  // the same value from any thread
    if (!per_sm) {
        int n = 0;
        const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &n, modln_cast_kernel<NV, W>, 32 * kWarpsPerBlock, 0);
        if (e != cudaSuccess) return cuda_fail(e);
        per_sm = n > 0 ? n : 1;
    }
    const int64_t cap = int64_t(sm_count()) * per_sm;
    const int grid = int(blocks_needed < cap ? blocks_needed : cap);
    modln_cast_kernel<NV, W><<<grid, 32 * kWarpsPerBlock, 0, s>>>(
        x, rows, shift, scale, reinterpret_cast<__nv_bfloat16 *>(out));
    return check_launch();
}

}  // namespace

dit_status_t launch_modln(const float *x, int64_t rows, int D, const float *shift,
                          const float *scale, void *out, cudaStream_t s) {
    if (rows < 0 || D <= 0 || D % 128 || !x || !shift || !scale || !out)
        return DIT_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(shift) || !aligned16(scale) || !aligned16(out))
        return DIT_ERR_ALIGN;
    if (rows == 0) return DIT_OK;
    switch (D / 128) {
#define DS_CASE(nv) \
    case nv:        \
        return run<nv>(x, rows, shift, scale, out, s);
        DS_CASE(1)
        DS_CASE(2)
        DS_CASE(3)
        DS_CASE(4)
        DS_CASE(5)
        DS_CASE(6)
        DS_CASE(8)
        DS_CASE(10)
        DS_CASE(12)
        DS_CASE(16)
        DS_CASE(20)
        DS_CASE(24)
        DS_CASE(32)
#undef DS_CASE
        default:
            return DIT_ERR_INVALID_ARG;
    }
}

}  // namespace ds
