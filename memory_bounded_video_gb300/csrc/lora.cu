// Activation-space LoRA adapter preparation.
//
// "ComfyUI-StaticPipeline", section "Activation-space LoRA (bypass mode)":
// y = W x + alpha B (A x) with W left packed.  The GEMM adds the delta as
// extra K-steps of u B'^T into W's fp32 accumulator (u = x A^T), so B' must
// carry alpha and, for int8 W, the inverse of W's row scale (the epilogue
// multiplies the whole accumulator by that scale).  This runs once per
// adapter, when it is placed on the device.
#include <cuda_bf16.h>

#include "internal.h"

namespace ds {
namespace {

__global__ void lora_prepare_kernel(const __nv_bfloat16 *__restrict__ b, int64_t rows, int rank,
                                    int64_t ld_b, float alpha, const float *__restrict__ scale,
                                    __nv_bfloat16 *__restrict__ out, int64_t ld_out) {
    const int64_t n_el = rows * rank;
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n_el;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t n = i / rank;
        const int j = int(i - n * rank);
        float v = alpha * __bfloat162float(b[n * ld_b + j]);
        if (scale) v = __fdiv_rn(v, scale[n]);
        out[n * ld_out + j] = __float2bfloat16_rn(v);
    }
}

}  // namespace
}  // namespace ds

extern "C" dit_status_t dit_lora_prepare(const void *b, int64_t rows, int rank, int64_t ld_b,
                                         float alpha, const float *row_scale, void *b_out,
                                         int64_t ld_out, dit_stream_t stream) {
    if (!b || !b_out || rows <= 0 || rank <= 0 || rank > DIT_LORA_MAX_RANK)
        return DIT_ERR_INVALID_ARG;
    if (ld_b < rank || ld_out < rank || ld_b % 8 || ld_out % 8) return DIT_ERR_INVALID_ARG;
    if (!ds::aligned16(b) || !ds::aligned16(b_out)) return DIT_ERR_ALIGN;
    const int64_t n_el = rows * rank;
    int64_t blocks = (n_el + 255) / 256;
    const int64_t cap = int64_t(ds::sm_count()) * 8;
    if (blocks > cap) blocks = cap;
    ds::lora_prepare_kernel<<<int(blocks), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __nv_bfloat16 *>(b), rows, rank, ld_b, alpha, row_scale,
        static_cast<__nv_bfloat16 *>(b_out), ld_out);
    return ds::check_launch();
}
