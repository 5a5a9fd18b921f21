// Host-side internals shared by the translation units of libditstream.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "ditstream.h"

// A block plan: sizes, the workspace layout and the per-kernel timing record.
struct dit_plan {
    int64_t T;
    int D, heads, head_dim, F;
    int cm, ca, fs;  // effective mlp chunk, attention chunk, FFN slice
    int64_t t_pad;   // row stride of V^T
    int lora_r = 0;  // LoRA rank the workspace holds (0: none)
    // workspace layout (byte offsets)
    size_t off_k, off_vt, off_a, off_q, off_b, off_h, off_acc, total;
    size_t off_uq, off_uo;                   // LoRA u of Q/K/V and O (attention phase)
    size_t off_ug, off_uu, off_ud, off_udc;  // LoRA u of gate, up, down; down's carry
    uint8_t *ws;
    size_t ws_bytes;
    // optional bf16 scratch for int8 weights expanded ahead of their GEMMs
    uint8_t *wscratch = nullptr;
    size_t wscratch_bytes = 0;
    // K/V offload: key block size (0: K/V resident), the device ring and the
    // carried attention state in the workspace, the host K/V buffer and the
    // copy stream with its events (slot filled / slot used)
    int kvb = 0;
    size_t off_ring = 0, ring_slot = 0, off_ost = 0, off_mst = 0, off_lst = 0;
    // hand-off state of the persistent attention's split units (slots of
    // it; 0: none) in the attention phase; their flags sit in the header
    int split_slots = 0;
    size_t off_split = 0;
    // the GEMMs' hand-off state (slots of kGemmSlotBytes), outside the phases
    int gsplit_slots = 0;
    size_t off_gsplit = 0;
    uint8_t *kv_host = nullptr;      // device address of the pinned host buffer
    size_t kv_host_bytes = 0;
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t ev_filled[2] = {nullptr, nullptr};   // pass 2: slot holds a key block
    cudaEvent_t ev_used[2] = {nullptr, nullptr};     // pass 2: attention done with slot
    cudaEvent_t ev_written[2] = {nullptr, nullptr};  // pass 1: GEMM wrote slot
    cudaEvent_t ev_free[2] = {nullptr, nullptr};     // pass 1: slot copied out
    // per-kernel timing (dit_block_profile_*)
    struct Rec {
        int kind;
        cudaEvent_t a, b;
        double work;
    };
    bool prof = false;
    std::vector<cudaEvent_t> pool;
    size_t pool_used = 0;
    std::vector<Rec> recs;
};

namespace ds {

// Workspace header: the device status word at byte 0, the attention
// hand-off flags at kFlagsOffset; zeroed when the workspace is bound.
constexpr size_t kFlagsOffset = 256;
constexpr size_t kHeaderBytes = 1024;

// Record a CUDA error for dit_last_cuda_error() and return DIT_ERR_CUDA.
dit_status_t cuda_fail(cudaError_t e);
// Check for a launch error right after a launch.
dit_status_t check_launch();

// Multiprocessor count of the current device (cached per device).
int sm_count();

// 2-D tensor map (row-major matrix: `inner` elements per row, `outer` rows,
// `row_bytes` between rows) with a box of box_inner x box_outer elements and
// the given shared-memory swizzle (128-byte by default); out-of-range
// elements read as zero.
bool make_tmap_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base,
                  uint64_t inner, uint64_t outer, uint64_t row_bytes,
                  uint32_t box_inner, uint32_t box_outer,
                  CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

dit_status_t launch_modln(const float *x, int64_t rows, int D, const float *shift,
                          const float *scale, void *out, cudaStream_t s);

struct AttnSplit;
// split: the hand-off space of the work split (flags, kGemmSlotBytes slots);
// null or no slots: whole tiles only.
dit_status_t launch_gemm(const dit_gemm_args_t &a, int *dev_status, cudaStream_t s,
                         const AttnSplit *split = nullptr);

// Carried softmax state for attention over keys in several launches.
struct AttnState {
    float *o;        // unnormalised fp32 O [Tq, H*d], row stride ld
    float *m, *l;    // running max and sum [Tq, H]
    int64_t ld;
    int first, last; // this launch has the first / last key block
};

// Hand-off space of the persistent attention kernel's split units: a flag
// per slot (zero before a launch; a launch leaves the flags it used zero
// again) and per slot the running max and sum of 256 query rows and their
// unnormalised fp32 output [256, head_dim].  slots = 0: no split.
struct AttnSplit {
    int *flags;    // [slots]
    float *state;  // [slots][256 * (head_dim + 2)]
    int slots;
    int max_ctas;  // CTAs at most (0: one per multiprocessor)
};

// Bytes of the split state for `slots` slots (the flags not included).
inline size_t attn_split_state_bytes(int slots, int head_dim) {
    return size_t(slots) * 256 * size_t(head_dim + 2) * 4;
}

dit_status_t launch_attention(const void *q, int64_t Tq, int64_t ldq, const void *k,
                              int64_t ldk, const void *vt, int64_t ldvt, int64_t T,
                              int heads, int head_dim, void *o, int64_t ldo,
                              int *dev_status, cudaStream_t s,
                              const AttnState *state = nullptr,
                              const AttnSplit *split = nullptr);

// dev_status: where a bounded wait that ran out records DIT_ERR_TIMEOUT (may
// be null).
dit_status_t launch_final(const float *x, int64_t T, int D, const void *wf,
                          const float *wf_scale, const float *mod_f, float *out,
                          int *dev_status, cudaStream_t s);

// bf16 copy of n int8 values (exact); n % 16 == 0, both 16-byte aligned.
dit_status_t launch_expand_int8(const void *q, int64_t n, void *out, cudaStream_t s);

// The block forward over the scratch at `ws` (a bound workspace or the
// static scratch); per-kernel timing goes to the plan's record only when
// `prof` is set, and the plan is not otherwise modified.
dit_status_t block_forward(const dit_plan *p, uint8_t *ws, bool prof, float *x,
                           const dit_block_weights_t *w, const float *mod, const dit_qk_t *qk,
                           const dit_block_lora_t *lora, dit_stream_t stream);

// Device address of the static scratch's status word on the current device,
// or null when no static forward has set that device up yet.
int *static_status_word();

inline bool aligned16(const void *p) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace ds
