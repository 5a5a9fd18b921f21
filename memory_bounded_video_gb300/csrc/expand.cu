// int8 weights expanded to bf16 ahead of their GEMMs.
//
// An int8 weight value q (|q| <= 127) has at most 8 significant bits, so its
// bf16 value is exact.  With the expanded copy the GEMM runs its bf16 main
// loop and applies the same per-row scale to the fp32 accumulator ("MiniMax-
// H3-Comfy-NPU" section 2.2: W = s_row * q): the MMAs see the same operands
// in the same order as with the in-kernel conversion, so the result bits are
// the same, and the shared-memory conversion traffic that bounds the int8
// main loop is gone.  HBM-bound: n bytes read, 2n written.
#include <cuda_bf16.h>

#include "internal.h"

namespace ds {
namespace {

__device__ __forceinline__ uint32_t bf16x2_of(int lo, int hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(float(lo), float(hi));
    return *reinterpret_cast<uint32_t *>(&v);
}

// 16 int8 per thread and step (one 16-byte load, two 16-byte stores).
__global__ void expand_int8_kernel(const int8_t *__restrict__ q, int64_t n16,
                                   __nv_bfloat16 *__restrict__ out) {
    const int4 *src = reinterpret_cast<const int4 *>(q);
    uint4 *dst = reinterpret_cast<uint4 *>(out);
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n16;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int4 v = __ldcs(src + i);  // read once: do not keep in L2
        const uint32_t w[4] = {uint32_t(v.x), uint32_t(v.y), uint32_t(v.z), uint32_t(v.w)};
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int b0 = int(int8_t(w[k] & 0xffu)), b1 = int(int8_t((w[k] >> 8) & 0xffu));
            const int b2 = int(int8_t((w[k] >> 16) & 0xffu)), b3 = int(int8_t(w[k] >> 24));
            o[2 * k] = bf16x2_of(b0, b1);
            o[2 * k + 1] = bf16x2_of(b2, b3);
        }
        dst[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

}  // namespace

dit_status_t launch_expand_int8(const void *q, int64_t n, void *out, cudaStream_t s) {
    if (!q || !out || n < 0 || n % 16) return DIT_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(out)) return DIT_ERR_ALIGN;
    if (n == 0) return DIT_OK;
    const int64_t n16 = n / 16;
    int64_t blocks = (n16 + 255) / 256;
    const int64_t cap = int64_t(sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    expand_int8_kernel<<<int(blocks), 256, 0, s>>>(static_cast<const int8_t *>(q), n16,
                                                   static_cast<__nv_bfloat16 *>(out));
    return check_launch();
}

}  // namespace ds

extern "C" dit_status_t dit_int8_to_bf16(const void *q, int64_t n, void *out,
                                         dit_stream_t stream) {
    return ds::launch_expand_int8(q, n, out, static_cast<cudaStream_t>(stream));
}
