// libditstream C ABI: plans, workspace layout, the bounded block schedule
// and the stage entry points.  Host code only; kernels live in modln.cu,
// gemm.cu, attention.cu and final.cu.
//
// Block schedule ("LayerStream: H3 Chunking", "How the slicing works";
// "Proposal: Generic memory-aware streaming execution for transformer
// models", attention streaming plan and "MLP planning"), all on one stream:
//   pass 1, per attention slab s:  modln(x_s; shift1, scale1) -> a_s
//                                  [K | V^T] rows s  = a_s Wkv^T       (KV)
//   pass 2, per attention slab s:  modln(x_s; shift1, scale1) -> a_s
//                                  Q_s = a_s Wq^T                     (STORE)
//                                  O_s = attention(Q_s, K, V)
//                                  x_s += gate1 * O_s Wo^T            (RESID)
//   MLP, per token chunk c:        modln(x_c; shift2, scale2) -> b_c
//     per FFN slice f:             h_f = silu(b_c Wg_f^T) * b_c Wu_f^T (SWIGLU)
//                                  acc (+)= h_f Wd_f^T; on the last slice
//                                  x_c += gate2 * acc                  (DOWN)
// Pass 2 reads x_s before writing it, and K/V come from pass 1, so every
// query attends to the pre-attention keys and values of all tokens.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "attn_sched.h"
#include "internal.h"

namespace ds {

namespace {
thread_local char g_err[256] = "";

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Signature of the driver's cuTensorMapEncodeTiled (fetched at run time so
// the library needs no link-time dependency on libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

bool load_encode() {
    if (g_encode) return true;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return false;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    return true;
}

bool modln_supports(int D) {
    if (D <= 0 || D % 128) return false;
    switch (D / 128) {
        case 1: case 2: case 3: case 4: case 5: case 6: case 8: case 10: case 12:
        case 16: case 20: case 24: case 32:
            return true;
        default:
            return false;
    }
}

}  // namespace

dit_status_t cuda_fail(cudaError_t e) {
    snprintf(g_err, sizeof(g_err), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return DIT_ERR_CUDA;
}

dit_status_t check_launch() {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DIT_OK : cuda_fail(e);
}

int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cache[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 148;
    }
    return cache[dev];
}

bool make_tmap_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *base, uint64_t inner,
                  uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                  CUtensorMapSwizzle swizzle) {
    if (!load_encode()) return false;
    if (inner == 0 || outer == 0 || row_bytes % 16 || !aligned16(base)) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Whether the block's GEMMs may cut their last wave into K ranges (the work
// split, a cooperative launch).  DITSTREAM_GEMM_SPLIT=0 in the environment
// turns it off for the process: every GEMM then runs whole tiles, with the
// same result bits.  This is for tools that cannot launch a cooperative grid
// of thread-block clusters (Nsight Compute reports such a launch as failed).
bool gemm_split_on() {
    static const bool on = [] {
        const char *v = std::getenv("DITSTREAM_GEMM_SPLIT");
        return !(v && std::strcmp(v, "0") == 0);
    }();
    return on;
}

// Launch `fn` (returning a dit_status_t) bracketed by profiling events when
// a plan is given and has profiling enabled.
template <class Fn>
dit_status_t timed(dit_plan *p, cudaStream_t st, int kind, double work, Fn &&fn) {
    if (!p || !p->prof) return fn();
    cudaEvent_t ev[2];
    for (int i = 0; i < 2; ++i) {
        if (p->pool_used == p->pool.size()) {
            cudaEvent_t e;
            const cudaError_t err = cudaEventCreate(&e);
            if (err != cudaSuccess) return cuda_fail(err);
            p->pool.push_back(e);
        }
        ev[i] = p->pool[p->pool_used++];
    }
    cudaError_t err = cudaEventRecord(ev[0], st);
    if (err != cudaSuccess) return cuda_fail(err);
    const dit_status_t r = fn();
    if (r != DIT_OK) return r;
    err = cudaEventRecord(ev[1], st);
    if (err != cudaSuccess) return cuda_fail(err);
    p->recs.push_back({kind, ev[0], ev[1], work});
    return DIT_OK;
}

}  // namespace ds

using namespace ds;

extern "C" {

int dit_abi_version(void) { return DITSTREAM_ABI_VERSION; }

const char *dit_last_cuda_error(void) { return g_err; }

const char *dit_status_string(dit_status_t s) {
    switch (s) {
        case DIT_OK: return "ok";
        case DIT_ERR_INVALID_ARG: return "invalid argument";
        case DIT_ERR_CHUNK_ALIGN: return "chunk size must be 0 or a multiple of 128";
        case DIT_ERR_ALIGN: return "device pointer not 16-byte aligned";
        case DIT_ERR_NO_WORKSPACE: return "no workspace bound to the plan";
        case DIT_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than dit_block_workspace_bytes";
        case DIT_ERR_CUDA: return "CUDA error";
        case DIT_ERR_TIMEOUT: return "a bounded device wait timed out";
        case DIT_ERR_UNSUPPORTED_ARCH: return "device is not sm_103";
        default: return "unknown status";
    }
}

namespace {

// Workspace layout of a plan (byte offsets, 1 KiB-aligned regions).
void layout(dit_plan *p) {
    const size_t A = 1024;
    const size_t Dz = size_t(p->D);
    const size_t R = size_t(p->lora_r);
    size_t phase;
    if (p->kvb) {  // K/V in host memory: a two-slot ring of key blocks
        p->off_k = p->off_vt = 0;
        p->off_ring = A;  // [0, 1024): header (status word, attention flags)
        p->ring_slot = round_up(4 * size_t(p->kvb) * Dz, A);
        phase = p->off_ring + 2 * p->ring_slot;
    } else {
        p->off_k = A;  // [0, 1024): header (status word, attention flags)
        p->off_vt = round_up(p->off_k + 2 * size_t(p->T) * Dz, A);
        phase = round_up(p->off_vt + 2 * Dz * size_t(p->t_pad), A);
    }
    // attention phase: a_s / O_s share one region (a_s is dead once Q_s exists)
    p->off_a = phase;
    p->off_q = round_up(p->off_a + 2 * size_t(p->ca) * Dz, A);
    size_t attn_end = round_up(p->off_q + 2 * size_t(p->ca) * Dz, A);
    p->off_uq = attn_end;
    p->off_uo = round_up(p->off_uq + 2 * size_t(p->ca) * R, A);
    if (R) attn_end = round_up(p->off_uo + 2 * size_t(p->ca) * R, A);
    if (p->kvb) {  // carried attention state: O fp32 [C_a, D], m and l [C_a, H]
        p->off_ost = attn_end;
        p->off_mst = round_up(p->off_ost + 4 * size_t(p->ca) * Dz, A);
        p->off_lst = round_up(p->off_mst + 4 * size_t(p->ca) * size_t(p->heads), A);
        attn_end = round_up(p->off_lst + 4 * size_t(p->ca) * size_t(p->heads), A);
    }
    // hand-off state of the attention's split units, when a slab has enough
    // (query pair, head) units to leave a partial wave on some device
    const int64_t units = (int64_t(p->ca) + 255) / 256 * p->heads;
    p->split_slots =
        units < (int64_t(1) << 30) ? attn_slots_needed(int(units), 1 << 20, kAttnSplitSlots, true) : 0;
    p->off_split = 0;
    if (p->split_slots) {
        p->off_split = attn_end;
        attn_end = round_up(p->off_split + attn_split_state_bytes(p->split_slots, p->head_dim), A);
    }
    // MLP phase (aliases the attention phase: the two never overlap in time)
    p->off_b = phase;
    p->off_h = round_up(p->off_b + 2 * size_t(p->cm) * Dz, A);
    p->off_acc = round_up(p->off_h + 2 * size_t(p->cm) * size_t(p->fs), A);
    size_t mlp_end = p->off_acc;
    if (p->fs < p->F) mlp_end = round_up(p->off_acc + 4 * size_t(p->cm) * Dz, A);
    p->off_ug = mlp_end;
    p->off_uu = round_up(p->off_ug + 2 * size_t(p->cm) * R, A);
    p->off_ud = round_up(p->off_uu + 2 * size_t(p->cm) * R, A);
    p->off_udc = round_up(p->off_ud + 2 * size_t(p->cm) * R, A);
    if (R) {
        mlp_end = p->off_udc;
        if (p->fs < p->F) mlp_end = round_up(p->off_udc + 4 * size_t(p->cm) * R, A);
    }
    p->total = attn_end > mlp_end ? attn_end : mlp_end;
    // the GEMMs' hand-off state, used within single launches of every phase:
    // slots for the most CTAs that any of the plan's GEMM launches (either
    // tile shape, full and ragged chunks and FFN slices) may cut its last
    // wave over on a device of 128 to 160 SMs, at most kGemmSplitSlots
    int gs = 0;
    auto need = [&](int64_t M, int N, int K, bool two_b) {
        if (M <= 0 || N <= 0 || K <= 0) return;
        for (bool pair : {false, true}) {
            const int n = gemm_slots_needed(gemm_units(M, N, two_b, pair), K / 64, pair);
            if (n > gs) gs = n;
        }
    };
    const int D = p->D;
    for (int64_t M : {int64_t(p->ca), p->T % p->ca}) {
        need(M, 2 * D, D, false);  // K, V
        need(M, D, D, false);      // Q, O
    }
    for (int64_t M : {int64_t(p->cm), p->T % p->cm})
        for (int fw : {p->fs, p->F % p->fs}) {
            need(M, fw, D, true);   // gate / up
            need(M, D, fw, false);  // down
        }
    p->gsplit_slots = gs;
    p->off_gsplit = 0;
    if (gs) {
        p->off_gsplit = round_up(p->total, A);
        p->total = round_up(p->off_gsplit + size_t(gs) * kGemmSlotBytes, A);
    }
}

}  // namespace

size_t dit_block_weight_scratch_bytes(const dit_plan_t *p) {
    if (!p) return 0;
    const size_t D = size_t(p->D), F = size_t(p->F);
    const size_t attn = 4 * D * D, mlp = 3 * D * F;
    return 2 * (attn > mlp ? attn : mlp);
}

dit_status_t dit_block_bind_weight_scratch(dit_plan_t *p, void *dev_ptr, size_t bytes) {
    if (!p) return DIT_ERR_INVALID_ARG;
    if (!dev_ptr) {
        p->wscratch = nullptr;
        p->wscratch_bytes = 0;
        return DIT_OK;
    }
    if (reinterpret_cast<uintptr_t>(dev_ptr) % 256) return DIT_ERR_ALIGN;
    if (bytes < dit_block_weight_scratch_bytes(p)) return DIT_ERR_WORKSPACE_TOO_SMALL;
    p->wscratch = static_cast<uint8_t *>(dev_ptr);
    p->wscratch_bytes = bytes;
    return DIT_OK;
}

dit_status_t dit_block_plan_set_kv_offload(dit_plan_t *p, int key_block_tokens) {
    if (!p || p->ws) return DIT_ERR_INVALID_ARG;
    if (key_block_tokens < 0) return DIT_ERR_INVALID_ARG;
    if (key_block_tokens % 128) return DIT_ERR_CHUNK_ALIGN;
    p->kvb = key_block_tokens;
    layout(p);
    return DIT_OK;
}

size_t dit_block_kv_host_bytes(const dit_plan_t *p) {
    if (!p || !p->kvb) return 0;
    const size_t n_kb = (size_t(p->T) + p->kvb - 1) / p->kvb;
    return 2 * size_t(p->T) * size_t(p->D) + 2 * size_t(p->D) * size_t(p->kvb) * n_kb;
}

dit_status_t dit_block_bind_kv_host(dit_plan_t *p, void *host_ptr, size_t bytes) {
    if (!p || !host_ptr) return DIT_ERR_INVALID_ARG;
    if (!aligned16(host_ptr)) return DIT_ERR_ALIGN;
    if (bytes < dit_block_kv_host_bytes(p)) return DIT_ERR_WORKSPACE_TOO_SMALL;
    void *dev = nullptr;
    cudaError_t e = cudaHostGetDevicePointer(&dev, host_ptr, 0);
    if (e != cudaSuccess) return cuda_fail(e);
    if (!p->copy_stream) {
        e = cudaStreamCreateWithFlags(&p->copy_stream, cudaStreamNonBlocking);
        for (int i = 0; i < 2 && e == cudaSuccess; ++i)
            for (cudaEvent_t *ev : {&p->ev_filled[i], &p->ev_used[i], &p->ev_written[i],
                                    &p->ev_free[i]})
                if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    p->kv_host = static_cast<uint8_t *>(dev);
    p->kv_host_bytes = bytes;
    return DIT_OK;
}

dit_status_t dit_block_plan_set_lora_rank(dit_plan_t *p, int max_rank) {
    if (!p || p->ws) return DIT_ERR_INVALID_ARG;
    if (max_rank < 0 || max_rank > DIT_LORA_MAX_RANK || max_rank % 32) return DIT_ERR_INVALID_ARG;
    p->lora_r = max_rank;
    layout(p);
    return DIT_OK;
}

dit_status_t dit_block_plan_ex(int64_t T, int D, int heads, int ffn, int mlp_chunk_tokens,
                               int attn_chunk_tokens, int ffn_slice, dit_plan_t **out) {
    if (!out) return DIT_ERR_INVALID_ARG;
    *out = nullptr;
    if (T <= 0 || T > (int64_t(1) << 30) || heads <= 0 || D <= 0 || D % heads ||
        !modln_supports(D))
        return DIT_ERR_INVALID_ARG;
    const int hd = D / heads;
    if (hd != 64 && hd != 128) return DIT_ERR_INVALID_ARG;
    if (ffn < 64 || ffn % 64) return DIT_ERR_INVALID_ARG;
    if (mlp_chunk_tokens < 0 || attn_chunk_tokens < 0 || ffn_slice < 0)
        return DIT_ERR_INVALID_ARG;
    if (mlp_chunk_tokens % 128 || attn_chunk_tokens % 128) return DIT_ERR_CHUNK_ALIGN;
    if (ffn_slice % 64 || ffn_slice > ffn) return DIT_ERR_INVALID_ARG;

    dit_plan *p = new (std::nothrow) dit_plan();
    if (!p) return DIT_ERR_INVALID_ARG;
    p->T = T;
    p->D = D;
    p->heads = heads;
    p->head_dim = hd;
    p->F = ffn;
    auto clamp = [&](int c) -> int { return (c == 0 || c >= T) ? int(T) : c; };
    p->cm = clamp(mlp_chunk_tokens);
    p->ca = clamp(attn_chunk_tokens);
    p->fs = ffn_slice == 0 ? ffn : ffn_slice;
    p->t_pad = int64_t(round_up(size_t(T), 128));
    layout(p);
    p->ws = nullptr;
    p->ws_bytes = 0;
    *out = p;
    return DIT_OK;
}

dit_status_t dit_block_plan_auto(int64_t T, int D, int heads, int ffn, size_t budget_bytes,
                                 dit_plan_t **out) {
    // "LayerStream: H3 Chunking" ("The two numbers you set"): use the largest
    // chunk that fits; "Proposal: ... streaming execution" ("Automatic chunk
    // sizing"): choose the largest chunks that fit a memory envelope.  The
    // attention slab is the largest multiple of 128 (or all T tokens) whose
    // plan fits; the MLP takes the largest token chunk, with the FFN unsliced
    // if that fits and sliced (halving down to 1024 features) only when it is
    // needed to fit that chunk.  Every choice gives the same result bits.
    if (!out) return DIT_ERR_INVALID_ARG;
    *out = nullptr;
    dit_plan_t *probe = nullptr;
    dit_status_t r = dit_block_plan_ex(T, D, heads, ffn, 128, 128, 0, &probe);
    if (r != DIT_OK) return r;
    dit_block_plan_destroy(probe);
    auto total = [&](int cm, int ca, int fs) -> size_t {
        dit_plan_t *q = nullptr;
        if (dit_block_plan_ex(T, D, heads, ffn, cm, ca, fs, &q) != DIT_OK) return SIZE_MAX;
        const size_t b = q->total;
        dit_block_plan_destroy(q);
        return b;
    };
    // candidate chunk sizes, largest first: all T tokens, then multiples of 128
    const int64_t top = (T + 127) / 128 * 128;
    auto chunk_of = [&](int64_t c) -> int { return c >= T ? 0 : int(c); };
    int ca = -1;
    for (int64_t c = top; c >= 128 && ca < 0; c -= 128)
        if (total(128, chunk_of(c), 0) <= budget_bytes) ca = chunk_of(c);
    if (ca < 0) return DIT_ERR_WORKSPACE_TOO_SMALL;
    // For each FFN slice width (unsliced, then halvings down to 1024) the
    // largest MLP token chunk that fits; slicing is taken only when it buys a
    // token chunk at least 25% larger than a wider slice does (its fp32
    // carry adds 4*C_m*D bytes of workspace and HBM traffic per slice).
    int cm = -1, fs = 0;
    int64_t best_tokens = 0;
    for (int f = ffn; f >= 64; f = (f / 2) / 64 * 64) {
        if (f != ffn && f < 1024) break;
        const int fs_try = f == ffn ? 0 : f;
        int cm_f = -1;
        int64_t tokens = 0;
        for (int64_t c = top; c >= 128; c -= 128)
            if (total(chunk_of(c), ca, fs_try) <= budget_bytes) {
                cm_f = chunk_of(c);
                tokens = c < T ? c : T;
                break;
            }
        if (cm_f < 0) continue;
        if (cm < 0 || tokens * 4 >= best_tokens * 5) {
            cm = cm_f;
            fs = fs_try;
            best_tokens = tokens;
        }
    }
    if (cm < 0) return DIT_ERR_WORKSPACE_TOO_SMALL;
    return dit_block_plan_ex(T, D, heads, ffn, cm, ca, fs, out);
}

dit_status_t dit_block_plan(int64_t T, int D, int heads, int ffn, int mlp_chunk_tokens,
                            int attn_chunk_tokens, dit_plan_t **out) {
    return dit_block_plan_ex(T, D, heads, ffn, mlp_chunk_tokens, attn_chunk_tokens, 0, out);
}

void dit_block_plan_destroy(dit_plan_t *plan) {
    if (!plan) return;
    for (cudaEvent_t e : plan->pool) cudaEventDestroy(e);
    for (int i = 0; i < 2; ++i)
        for (cudaEvent_t e : {plan->ev_filled[i], plan->ev_used[i], plan->ev_written[i],
                              plan->ev_free[i]})
            if (e) cudaEventDestroy(e);
    if (plan->copy_stream) cudaStreamDestroy(plan->copy_stream);
    delete plan;
}

dit_status_t dit_block_profile_enable(dit_plan_t *p, int enable) {
    if (!p) return DIT_ERR_INVALID_ARG;
    p->prof = enable != 0;
    return DIT_OK;
}

dit_status_t dit_block_profile_read(dit_plan_t *p, double *ms, int64_t *launches, double *work) {
    if (!p) return DIT_ERR_INVALID_ARG;
    double t[DIT_NUM_KINDS] = {0}, w[DIT_NUM_KINDS] = {0};
    int64_t n[DIT_NUM_KINDS] = {0};
    dit_status_t r = DIT_OK;
    for (const auto &rec : p->recs) {
        float e = 0.f;
        cudaError_t err = cudaEventSynchronize(rec.b);
        if (err == cudaSuccess) err = cudaEventElapsedTime(&e, rec.a, rec.b);
        if (err != cudaSuccess) {
            r = cuda_fail(err);
            break;
        }
        t[rec.kind] += e;
        w[rec.kind] += rec.work;
        n[rec.kind] += 1;
    }
    p->recs.clear();
    p->pool_used = 0;
    for (int k = 0; k < DIT_NUM_KINDS; ++k) {
        if (ms) ms[k] = t[k];
        if (launches) launches[k] = n[k];
        if (work) work[k] = w[k];
    }
    return r;
}

dit_status_t dit_block_plan_info(const dit_plan_t *p, int64_t *T, int *D, int *heads, int *ffn,
                                 int *mlp_chunk, int *attn_chunk, int *ffn_slice) {
    if (!p) return DIT_ERR_INVALID_ARG;
    if (T) *T = p->T;
    if (D) *D = p->D;
    if (heads) *heads = p->heads;
    if (ffn) *ffn = p->F;
    if (mlp_chunk) *mlp_chunk = p->cm;
    if (attn_chunk) *attn_chunk = p->ca;
    if (ffn_slice) *ffn_slice = p->fs;
    return DIT_OK;
}

size_t dit_block_workspace_bytes(const dit_plan_t *p) { return p ? p->total : 0; }

dit_status_t dit_block_bind_workspace(dit_plan_t *p, void *dev_ptr, size_t bytes) {
    if (!p || !dev_ptr) return DIT_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(dev_ptr) & 255u) return DIT_ERR_ALIGN;
    if (bytes < p->total) return DIT_ERR_WORKSPACE_TOO_SMALL;
    int dev = 0, major = 0, minor = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (major != 10 || minor != 3) return DIT_ERR_UNSUPPORTED_ARCH;
    e = cudaMemset(dev_ptr, 0, kHeaderBytes);
    if (e != cudaSuccess) return cuda_fail(e);
    p->ws = static_cast<uint8_t *>(dev_ptr);
    p->ws_bytes = bytes;
    return DIT_OK;
}

dit_status_t dit_block_forward(const dit_plan_t *cp, float *x, const dit_block_weights_t *w,
                               const float *mod, dit_stream_t stream) {
    return dit_block_forward_qk(cp, x, w, mod, nullptr, stream);
}

dit_status_t dit_block_forward_qk(const dit_plan_t *cp, float *x, const dit_block_weights_t *w,
                                  const float *mod, const dit_qk_t *qk, dit_stream_t stream) {
    return dit_block_forward_ex(cp, x, w, mod, qk, nullptr, stream);
}

}  // extern "C"

namespace ds {

// The block schedule over the scratch at `ws` (the plan's bound workspace,
// or the library's static scratch), with per-kernel timing recorded in the
// plan only when `prof` is set; the plan itself is not modified otherwise.
dit_status_t block_forward(const dit_plan *cp, uint8_t *ws, bool prof, float *x,
                           const dit_block_weights_t *w, const float *mod, const dit_qk_t *qk,
                           const dit_block_lora_t *lora, dit_stream_t stream) {
    if (!cp || !x || !w || !mod) return DIT_ERR_INVALID_ARG;
    const dit_plan *p = cp;
    // the timing record is the one part of the plan a forward may change
    dit_plan *tp = prof ? const_cast<dit_plan *>(cp) : nullptr;
    if (qk) {
        if (!qk->rope_cos != !qk->rope_sin) return DIT_ERR_INVALID_ARG;
        if ((qk->q_norm || qk->k_norm) && !(qk->eps > 0.0f)) return DIT_ERR_INVALID_ARG;
        if (!aligned16(qk->q_norm) || !aligned16(qk->k_norm) || !aligned16(qk->rope_cos) ||
            !aligned16(qk->rope_sin))
            return DIT_ERR_ALIGN;
    }
    // an adapter is present when both of its matrices are given
    auto on = [&](const dit_lora_t &l) { return lora && l.a && l.b; };
    if (lora) {
        for (const dit_lora_t *l : {&lora->qkv, &lora->o, &lora->gate, &lora->up, &lora->down}) {
            if (!on(*l)) continue;
            if (l->rank <= 0 || l->rank % 32 || l->rank > p->lora_r) return DIT_ERR_INVALID_ARG;
            if (!aligned16(l->a) || !aligned16(l->b)) return DIT_ERR_ALIGN;
        }
    }
    if (!ws || (p->kvb && !p->kv_host)) return DIT_ERR_NO_WORKSPACE;
    if (!w->wqkv || !w->wo || !w->wgate || !w->wup || !w->wdown) return DIT_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(mod) || !aligned16(w->wqkv) || !aligned16(w->wo) ||
        !aligned16(w->wgate) || !aligned16(w->wup) || !aligned16(w->wdown))
        return DIT_ERR_ALIGN;
    if (w->dtype != DIT_W_BF16 && w->dtype != DIT_W_INT8) return DIT_ERR_INVALID_ARG;
    const bool i8 = w->dtype == DIT_W_INT8;
    if (i8) {
        if (!w->wqkv_scale || !w->wo_scale || !w->wgate_scale || !w->wup_scale ||
            !w->wdown_scale)
            return DIT_ERR_INVALID_ARG;
        if (!aligned16(w->wqkv_scale) || !aligned16(w->wo_scale) ||
            !aligned16(w->wgate_scale) || !aligned16(w->wup_scale) ||
            !aligned16(w->wdown_scale))
            return DIT_ERR_ALIGN;
    }
    // int8 weights expanded into the weight scratch run as bf16 with scales
    const bool expand = i8 && p->wscratch;
    const int bdt = expand ? DIT_W_BF16 : w->dtype;
    const int64_t el = (i8 && !expand) ? 1 : 2;  // bytes per weight element

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t T = p->T;
    const int D = p->D, F = p->F;
    const int64_t Dl = D;
    int *status = reinterpret_cast<int *>(ws);
    // the GEMMs' hand-off space for split tiles (flags shared with the
    // attention's: every launch leaves the flags it used zero)
    const AttnSplit gsplit{reinterpret_cast<int *>(ws + kFlagsOffset),
                           reinterpret_cast<float *>(ws + p->off_gsplit),
                           gemm_split_on() ? p->gsplit_slots : 0, 0};
    // K [T, D] and V^T [D, T_pad]: in the workspace, or (offload) in the
    // host buffer, written there by pass one through its device mapping
    void *K = p->kvb ? static_cast<void *>(p->kv_host) : static_cast<void *>(ws + p->off_k);
    void *Vt = p->kvb ? static_cast<void *>(p->kv_host + 2 * size_t(T) * size_t(D))
                      : static_cast<void *>(ws + p->off_vt);
    void *a = ws + p->off_a;
    void *Q = ws + p->off_q;
    void *b = ws + p->off_b;
    void *h = ws + p->off_h;
    float *acc = reinterpret_cast<float *>(ws + p->off_acc);
    void *u_q = ws + p->off_uq;
    void *u_o = ws + p->off_uo;
    void *u_g = ws + p->off_ug;
    void *u_u = ws + p->off_uu;
    void *u_d = ws + p->off_ud;
    float *u_dc = reinterpret_cast<float *>(ws + p->off_udc);
    const float *shift1 = mod, *scale1 = mod + Dl, *gate1 = mod + 2 * Dl;
    const float *shift2 = mod + 3 * Dl, *scale2 = mod + 4 * Dl, *gate2 = mod + 5 * Dl;
    const uint8_t *wqkv = static_cast<const uint8_t *>(w->wqkv);
    const void *wo_m = w->wo;
    dit_status_t r;
    auto expand_into = [&](const void *q, int64_t n, uint8_t *dst) -> dit_status_t {
        return timed(tp, st, DIT_K_EXPAND, 3.0 * n,
                     [&] { return launch_expand_int8(q, n, dst, st); });
    };
    if (expand) {  // attention-phase weights: Wqkv [3D, D], Wo [D, D]
        if ((r = expand_into(w->wqkv, 3 * Dl * Dl, p->wscratch)) != DIT_OK ||
            (r = expand_into(w->wo, Dl * Dl, p->wscratch + 6 * Dl * Dl)) != DIT_OK)
            return r;
        wqkv = p->wscratch;
        wo_m = p->wscratch + 6 * Dl * Dl;
    }

    // the GEMM's Q/K transform fields for Q (which = 0) or K (which = 1)
    auto set_qk = [&](dit_gemm_args_t &g, int which) {
        if (!qk) return;
        g.qk_norm = which ? qk->k_norm : qk->q_norm;
        g.rope_cos = qk->rope_cos;
        g.rope_sin = qk->rope_sin;
        g.head_dim = p->head_dim;
        g.qk_eps = qk->eps;
    };
    // LoRA: u = t A^T (bf16 [rows, rank]); A's columns col0.. of row stride lda_a
    auto lora_u = [&](const void *t, int64_t ldt, int64_t rows, int K_, const dit_lora_t &l,
                      int64_t col0, int64_t lda_a, void *u, float *carry, int load,
                      int final_) -> dit_status_t {
        dit_gemm_args_t g{};
        g.M = rows;
        g.N = l.rank;
        g.K = K_;
        g.a = t;
        g.lda = ldt;
        g.b0 = static_cast<const uint8_t *>(l.a) + col0 * 2;
        g.ldb = lda_a;
        g.b_dtype = DIT_W_BF16;
        if (final_) {  // bf16 u, from the fp32 carry when there is one
            g.mode = DIT_EPI_STORE_BF16;
            g.out = u;
            g.ldo = l.rank;
            g.acc_load = load;
            g.acc = carry;
            g.ldacc = l.rank;
        } else {  // fp32 carry of a K-sliced u (the down adapter over FFN slices)
            g.mode = DIT_EPI_DOWN;
            g.acc = carry;
            g.ldacc = l.rank;
            g.acc_load = load;
            g.acc_final = 0;
        }
        return timed(tp, st, DIT_K_LORA_U, 2.0 * rows * l.rank * K_,
                     [&] { return launch_gemm(g, status, st, &gsplit); });
    };
    // LoRA K-steps of a GEMM: u [rows, rank] and rows row0.. of the prepared B
    auto attach = [&](dit_gemm_args_t &g, int half, const void *u, const dit_lora_t &l,
                      int64_t row0) {
        const void *lb = static_cast<const uint8_t *>(l.b) + row0 * l.rank * 2;
        if (half == 0) {
            g.lora_u0 = u;
            g.lora_ldu0 = l.rank;
            g.lora_l0 = lb;
            g.lora_ldl0 = l.rank;
            g.lora_rank0 = l.rank;
        } else {
            g.lora_u1 = u;
            g.lora_ldu1 = l.rank;
            g.lora_l1 = lb;
            g.lora_ldl1 = l.rank;
            g.lora_rank1 = l.rank;
        }
    };
    const dit_lora_t none{};
    const dit_lora_t &l_qkv = lora ? lora->qkv : none;
    const dit_lora_t &l_o = lora ? lora->o : none;
    const dit_lora_t &l_g = lora ? lora->gate : none;
    const dit_lora_t &l_u = lora ? lora->up : none;
    const dit_lora_t &l_d = lora ? lora->down : none;
    auto lflops = [&](const dit_lora_t &l, int64_t rows, int n_out) {
        return on(l) ? 2.0 * rows * n_out * l.rank : 0.0;
    };

    // K/V offload: the two ring slots stage pass one's K/V on their way to
    // the host buffer and bring key blocks back in pass two; the copies run
    // on the plan's copy stream, ordered against the kernels by events.  The
    // host buffer holds K [T, D] and, per key block b, V^T_b [D, kvb]: every
    // copy is one contiguous range (a strided V^T copy ran at a third of the
    // contiguous copy's bandwidth).
    const int64_t kvb = p->kvb;
    const int64_t n_kb = kvb ? (T + kvb - 1) / kvb : 0;
    const int64_t n_total = kvb ? n_kb * ((T + p->ca - 1) / p->ca) : 0;
    cudaStream_t cs = p->copy_stream;
    auto slot_k = [&](int slot) { return ws + p->off_ring + size_t(slot) * p->ring_slot; };
    auto slot_vt = [&](int slot) { return slot_k(slot) + 2 * size_t(kvb) * size_t(D); };
    uint8_t *hK = static_cast<uint8_t *>(K);
    uint8_t *hVt = static_cast<uint8_t *>(Vt);  // offload: V^T blocks [n_kb][D][kvb]
    const size_t vt_block_bytes = 2 * size_t(kvb) * size_t(D);
    auto fetch = [&](int64_t c) -> dit_status_t {  // c-th block of pass two
        const int slot = int(c & 1);
        const int64_t b = c % n_kb, k0 = b * kvb;
        const int64_t kb = (T - k0 < kvb) ? T - k0 : kvb;
        cudaError_t e = cudaStreamWaitEvent(cs, p->ev_used[slot], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(slot_k(slot), hK + 2 * k0 * Dl, size_t(2 * kb * Dl),
                                cudaMemcpyDefault, cs);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(slot_vt(slot), hVt + size_t(b) * vt_block_bytes, vt_block_bytes,
                                cudaMemcpyDefault, cs);
        if (e == cudaSuccess) e = cudaEventRecord(p->ev_filled[slot], cs);
        return e == cudaSuccess ? DIT_OK : cuda_fail(e);
    };

    // pass 1: K and V of every token
    for (int64_t s = 0; s < T; s += p->ca) {
        const int64_t rows = (T - s < p->ca) ? T - s : p->ca;
        if ((r = timed(tp, st, DIT_K_MODLN, 6.0 * rows * D,
                       [&] { return launch_modln(x + s * Dl, rows, D, shift1, scale1, a, st); })) !=
            DIT_OK)
            return r;
        if (on(l_qkv) && (r = lora_u(a, D, rows, D, l_qkv, 0, D, u_q, nullptr, 0, 1)) != DIT_OK)
            return r;
        // resident: one GEMM into K / V^T; offload: one per part of a key
        // block in the slab, into the block's ring slot (slot b % 2, part at
        // the block's column t0 % kvb), copied out when the block is complete
        for (int64_t t0 = s; t0 < s + rows;) {
            const int64_t b = kvb ? t0 / kvb : 0;
            const int64_t c0 = kvb ? t0 - b * kvb : 0;
            const int64_t t1 = kvb ? ((s + rows < (b + 1) * kvb) ? s + rows : (b + 1) * kvb)
                                   : s + rows;
            const int64_t sr = t1 - t0;
            const int slot = int(b & 1);
            dit_gemm_args_t g{};
            g.mode = DIT_EPI_KV;
            g.M = sr;
            g.N = 2 * D;
            g.K = D;
            g.a = static_cast<const uint8_t *>(a) + 2 * (t0 - s) * Dl;
            g.lda = D;
            g.b0 = wqkv + Dl * Dl * el;  // rows D..3D-1: Wk then Wv
            g.ldb = D;
            g.b_dtype = bdt;
            g.b0_scale = i8 ? w->wqkv_scale + Dl : nullptr;
            g.ldo = D;
            g.split_n = D;
            g.rope_pos0 = t0;
            if (!kvb) {
                g.out = K;
                g.out2 = Vt;
                g.ldo2 = p->t_pad;
                g.row_offset = s;
            } else {
                if (c0 == 0) {  // the block's first part: its slot must be copied out
                    cudaError_t e = cudaStreamWaitEvent(st, p->ev_free[slot], 0);
                    if (e != cudaSuccess) return cuda_fail(e);
                }
                g.out = slot_k(slot);
                g.out2 = slot_vt(slot);
                g.ldo2 = kvb;
                g.row_offset = c0;
            }
            set_qk(g, 1);
            if (on(l_qkv))
                attach(g, 0, static_cast<const uint8_t *>(u_q) + 2 * (t0 - s) * l_qkv.rank,
                       l_qkv, Dl);
            if ((r = timed(tp, st, DIT_K_GEMM_KV, 2.0 * sr * 2 * D * D + lflops(l_qkv, sr, 2 * D),
                           [&] { return launch_gemm(g, status, st, &gsplit); })) != DIT_OK)
                return r;
            if (kvb && (t1 % kvb == 0 || t1 == T)) {  // block b complete
                const int64_t k0 = b * kvb;
                cudaError_t e = cudaEventRecord(p->ev_written[slot], st);
                if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, p->ev_written[slot], 0);
                if (e == cudaSuccess)
                    e = cudaMemcpyAsync(hK + 2 * k0 * Dl, slot_k(slot), size_t(2 * (t1 - k0) * Dl),
                                        cudaMemcpyDefault, cs);
                if (e == cudaSuccess)
                    e = cudaMemcpyAsync(hVt + size_t(b) * vt_block_bytes, slot_vt(slot),
                                        vt_block_bytes, cudaMemcpyDefault, cs);
                if (e == cudaSuccess) e = cudaEventRecord(p->ev_free[slot], cs);
                if (e != cudaSuccess) return cuda_fail(e);
            }
            t0 = t1;
        }
    }
    // the attention's hand-off space for split units
    const AttnSplit split{reinterpret_cast<int *>(ws + kFlagsOffset),
                          reinterpret_cast<float *>(ws + p->off_split), p->split_slots, 0};
    int64_t kv_c = 0;  // blocks of pass two consumed so far
    // pass two's first block; the copy stream is in order, so it follows
    // pass one's copies to the host
    if (kvb && (r = fetch(0)) != DIT_OK) return r;
    // pass 2: Q per slab, attention against all keys, O-projection into x
    for (int64_t s = 0; s < T; s += p->ca) {
        const int64_t rows = (T - s < p->ca) ? T - s : p->ca;
        if ((r = timed(tp, st, DIT_K_MODLN, 6.0 * rows * D,
                       [&] { return launch_modln(x + s * Dl, rows, D, shift1, scale1, a, st); })) !=
            DIT_OK)
            return r;
        if (on(l_qkv) && (r = lora_u(a, D, rows, D, l_qkv, 0, D, u_q, nullptr, 0, 1)) != DIT_OK)
            return r;
        dit_gemm_args_t g{};
        g.mode = DIT_EPI_STORE_BF16;
        g.M = rows;
        g.N = D;
        g.K = D;
        g.a = a;
        g.lda = D;
        g.b0 = wqkv;
        g.ldb = D;
        g.b_dtype = bdt;
        g.b0_scale = i8 ? w->wqkv_scale : nullptr;
        g.out = Q;
        g.ldo = D;
        g.rope_pos0 = s;  // rotary position of the slab's first token
        set_qk(g, 0);
        if (on(l_qkv)) attach(g, 0, u_q, l_qkv, 0);
        if ((r = timed(tp, st, DIT_K_GEMM_Q, 2.0 * rows * D * D + lflops(l_qkv, rows, D),
                       [&] { return launch_gemm(g, status, st, &gsplit); })) != DIT_OK)
            return r;
        // O_s overwrites a_s (dead once Q_s exists)
        if (!kvb) {
            if ((r = timed(tp, st, DIT_K_ATTENTION, 4.0 * rows * double(T) * D, [&] {
                     return launch_attention(Q, rows, D, K, D, Vt, p->t_pad, T, p->heads,
                                             p->head_dim, a, D, status, st, nullptr, &split);
                 })) != DIT_OK)
                return r;
        } else {
            for (int64_t b = 0; b < n_kb; ++b, ++kv_c) {
                if (kv_c + 1 < n_total && (r = fetch(kv_c + 1)) != DIT_OK) return r;
                const int slot = int(kv_c & 1);
                const int64_t kb = (T - b * kvb < kvb) ? T - b * kvb : kvb;
                cudaError_t e = cudaStreamWaitEvent(st, p->ev_filled[slot], 0);
                if (e != cudaSuccess) return cuda_fail(e);
                AttnState as{reinterpret_cast<float *>(ws + p->off_ost),
                             reinterpret_cast<float *>(ws + p->off_mst),
                             reinterpret_cast<float *>(ws + p->off_lst), Dl, b == 0,
                             b == n_kb - 1};
                if ((r = timed(tp, st, DIT_K_ATTENTION, 4.0 * rows * double(kb) * D, [&] {
                         return launch_attention(Q, rows, D, slot_k(slot), D, slot_vt(slot),
                                                 kvb, kb, p->heads, p->head_dim, a, D, status,
                                                 st, &as, &split);
                     })) != DIT_OK)
                    return r;
                e = cudaEventRecord(p->ev_used[slot], st);
                if (e != cudaSuccess) return cuda_fail(e);
            }
        }
        if (on(l_o) && (r = lora_u(a, D, rows, D, l_o, 0, D, u_o, nullptr, 0, 1)) != DIT_OK)
            return r;
        dit_gemm_args_t o{};
        o.mode = DIT_EPI_RESID;
        o.M = rows;
        o.N = D;
        o.K = D;
        o.a = a;
        o.lda = D;
        o.b0 = wo_m;
        o.ldb = D;
        o.b_dtype = bdt;
        o.b0_scale = i8 ? w->wo_scale : nullptr;
        o.x = x + s * Dl;
        o.ldx = D;
        o.gate = gate1;
        if (on(l_o)) attach(o, 0, u_o, l_o, 0);
        if ((r = timed(tp, st, DIT_K_GEMM_O, 2.0 * rows * D * D + lflops(l_o, rows, D),
                       [&] { return launch_gemm(o, status, st, &gsplit); })) != DIT_OK)
            return r;
    }
    // MLP: token chunks x FFN feature slices
    const uint8_t *wg = static_cast<const uint8_t *>(w->wgate);
    const uint8_t *wu = static_cast<const uint8_t *>(w->wup);
    const uint8_t *wd = static_cast<const uint8_t *>(w->wdown);
    if (expand) {  // MLP-phase weights over the attention ones (stream order)
        const int64_t nf = int64_t(F) * Dl;
        uint8_t *sg = p->wscratch, *su = sg + 2 * nf, *sd = su + 2 * nf;
        if ((r = expand_into(w->wgate, nf, sg)) != DIT_OK ||
            (r = expand_into(w->wup, nf, su)) != DIT_OK ||
            (r = expand_into(w->wdown, nf, sd)) != DIT_OK)
            return r;
        wg = sg;
        wu = su;
        wd = sd;
    }
    for (int64_t c = 0; c < T; c += p->cm) {
        const int64_t rows = (T - c < p->cm) ? T - c : p->cm;
        if ((r = timed(tp, st, DIT_K_MODLN, 6.0 * rows * D,
                       [&] { return launch_modln(x + c * Dl, rows, D, shift2, scale2, b, st); })) !=
            DIT_OK)
            return r;
        if (on(l_g) && (r = lora_u(b, D, rows, D, l_g, 0, D, u_g, nullptr, 0, 1)) != DIT_OK)
            return r;
        if (on(l_u) && (r = lora_u(b, D, rows, D, l_u, 0, D, u_u, nullptr, 0, 1)) != DIT_OK)
            return r;
        for (int f = 0; f < F; f += p->fs) {
            const int fw = (F - f < p->fs) ? F - f : p->fs;
            const bool last = f + fw >= F;
            dit_gemm_args_t g{};
            g.mode = DIT_EPI_SWIGLU;
            g.M = rows;
            g.N = fw;
            g.K = D;
            g.a = b;
            g.lda = D;
            g.b0 = wg + int64_t(f) * Dl * el;
            g.b1 = wu + int64_t(f) * Dl * el;
            g.ldb = D;
            g.b_dtype = bdt;
            g.b0_scale = i8 ? w->wgate_scale + f : nullptr;
            g.b1_scale = i8 ? w->wup_scale + f : nullptr;
            g.out = h;
            g.ldo = p->fs;
            if (on(l_g)) attach(g, 0, u_g, l_g, f);
            if (on(l_u)) attach(g, 1, u_u, l_u, f);
            if ((r = timed(tp, st, DIT_K_GEMM_SWIGLU,
                           4.0 * rows * fw * D + lflops(l_g, rows, fw) + lflops(l_u, rows, fw),
                           [&] { return launch_gemm(g, status, st, &gsplit); })) != DIT_OK)
                return r;
            // the down adapter's u = h A_d^T accumulates over the FFN slices
            // (fp32 carry; bf16 after the last), in the unsliced K order
            if (on(l_d) &&
                (r = lora_u(h, p->fs, rows, fw, l_d, f, F, u_d, u_dc, f > 0, last)) != DIT_OK)
                return r;
            dit_gemm_args_t d{};
            d.mode = DIT_EPI_DOWN;
            d.M = rows;
            d.N = D;
            d.K = fw;
            d.a = h;
            d.lda = p->fs;
            d.b0 = wd + int64_t(f) * el;  // columns f .. f+fw-1 of Wdown [D, F]
            d.ldb = F;
            d.b_dtype = bdt;
            d.b0_scale = i8 ? w->wdown_scale : nullptr;
            d.acc = acc;
            d.ldacc = D;
            d.acc_load = f > 0;
            d.acc_final = last;
            d.x = x + c * Dl;
            d.ldx = D;
            d.gate = gate2;
            if (last && on(l_d)) attach(d, 0, u_d, l_d, 0);
            if ((r = timed(tp, st, DIT_K_GEMM_DOWN,
                           2.0 * rows * D * fw + (last ? lflops(l_d, rows, D) : 0.0),
                           [&] { return launch_gemm(d, status, st, &gsplit); })) != DIT_OK)
                return r;
        }
    }
    return DIT_OK;
}

}  // namespace ds

extern "C" {

dit_status_t dit_block_forward_ex(const dit_plan_t *p, float *x, const dit_block_weights_t *w,
                                  const float *mod, const dit_qk_t *qk,
                                  const dit_block_lora_t *lora, dit_stream_t stream) {
    if (!p) return DIT_ERR_INVALID_ARG;
    return block_forward(p, p->ws, p->prof, x, w, mod, qk, lora, stream);
}

dit_status_t dit_block_sync_status(const dit_plan_t *p, dit_stream_t stream) {
    if (!p) return DIT_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    // the plan's workspace header, and the static scratch's when a static
    // forward has set up the current device (shared by every static call)
    int v = 0;
    for (uint8_t *hdr : {p->ws, reinterpret_cast<uint8_t *>(static_status_word())}) {
        if (!hdr) continue;
        int s = 0;
        e = cudaMemcpyAsync(&s, hdr, sizeof(int), cudaMemcpyDeviceToHost, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        // after a failure the hand-off flags may be left set: clear them with
        // the status word
        if (e == cudaSuccess && s != 0) e = cudaMemsetAsync(hdr, 0, kHeaderBytes, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(e);
        if (v == 0) v = s;
    }
    return v == 0 ? DIT_OK : (v == DIT_ERR_TIMEOUT ? DIT_ERR_TIMEOUT : DIT_ERR_CUDA);
}

dit_status_t dit_final_forward(const dit_plan_t *cp, const float *x, const void *wf,
                               const float *wf_scale, const float *mod_f, float *out,
                               dit_stream_t stream) {
    dit_plan *p = const_cast<dit_plan *>(cp);
    if (!p) return DIT_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const double bytes = 4.0 * double(p->T) * p->D + 4.0 * 64 * p->D + 4.0 * 64 * double(p->T);
    return timed(p, st, DIT_K_FINAL, bytes, [&] {
        return launch_final(x, p->T, p->D, wf, wf_scale, mod_f, out,
                            p->ws ? reinterpret_cast<int *>(p->ws) : nullptr, st);
    });
}

dit_status_t dit_modln_cast(const float *x, int64_t rows, int D, const float *shift,
                            const float *scale, void *out_bf16, dit_stream_t stream) {
    return launch_modln(x, rows, D, shift, scale, out_bf16, static_cast<cudaStream_t>(stream));
}

dit_status_t dit_gemm(const dit_gemm_args_t *args, int *dev_status, dit_stream_t stream) {
    if (!args) return DIT_ERR_INVALID_ARG;
    return launch_gemm(*args, dev_status, static_cast<cudaStream_t>(stream));
}

size_t dit_gemm_split_bytes(int slots) {
    if (slots < 0 || slots > kGemmSplitSlots) return 0;
    return kHeaderBytes + size_t(slots) * kGemmSlotBytes;
}

dit_status_t dit_gemm_ex(const dit_gemm_args_t *args, void *split_ws, size_t split_bytes,
                         int max_ctas, int *dev_status, dit_stream_t stream) {
    if (!args || max_ctas < 0) return DIT_ERR_INVALID_ARG;
    AttnSplit split{nullptr, nullptr, 0, max_ctas};
    if (split_ws) {
        if (!aligned16(split_ws)) return DIT_ERR_ALIGN;
        if (split_bytes < kHeaderBytes) return DIT_ERR_WORKSPACE_TOO_SMALL;
        size_t n = (split_bytes - kHeaderBytes) / kGemmSlotBytes;
        if (n > size_t(kGemmSplitSlots)) n = kGemmSplitSlots;
        split.flags = static_cast<int *>(split_ws);
        split.state = reinterpret_cast<float *>(static_cast<uint8_t *>(split_ws) + kHeaderBytes);
        split.slots = int(n);
    }
    return launch_gemm(*args, dev_status, static_cast<cudaStream_t>(stream), &split);
}

dit_status_t dit_attention_part(const void *q, int64_t Tq, int64_t ldq, const void *k,
                                int64_t ldk, const void *vt, int64_t ldvt, int64_t T_block,
                                int heads, int head_dim, void *o, int64_t ldo, float *o_state,
                                float *m_state, float *l_state, int64_t ld_state, int first,
                                int last, int *dev_status, dit_stream_t stream) {
    AttnState as{o_state, m_state, l_state, ld_state, first != 0, last != 0};
    return launch_attention(q, Tq, ldq, k, ldk, vt, ldvt, T_block, heads, head_dim, o, ldo,
                            dev_status, static_cast<cudaStream_t>(stream), &as);
}

size_t dit_attention_split_bytes(int head_dim, int slots) {
    if ((head_dim != 64 && head_dim != 128) || slots < 0 || slots > kAttnSplitSlots) return 0;
    return kHeaderBytes + attn_split_state_bytes(slots, head_dim);
}

dit_status_t dit_attention_ex(const void *q, int64_t Tq, int64_t ldq, const void *k,
                              int64_t ldk, const void *vt, int64_t ldvt, int64_t T, int heads,
                              int head_dim, void *o, int64_t ldo, void *split_ws,
                              size_t split_bytes, int max_ctas, int *dev_status,
                              dit_stream_t stream) {
    if (max_ctas < 0 || (head_dim != 64 && head_dim != 128)) return DIT_ERR_INVALID_ARG;
    AttnSplit split{nullptr, nullptr, 0, max_ctas};
    if (split_ws) {
        if (!aligned16(split_ws)) return DIT_ERR_ALIGN;
        if (split_bytes < kHeaderBytes) return DIT_ERR_WORKSPACE_TOO_SMALL;
        const size_t per = attn_split_state_bytes(1, head_dim);
        size_t n = (split_bytes - kHeaderBytes) / per;
        if (n > size_t(kAttnSplitSlots)) n = kAttnSplitSlots;
        split.flags = static_cast<int *>(split_ws);
        split.state = reinterpret_cast<float *>(static_cast<uint8_t *>(split_ws) + kHeaderBytes);
        split.slots = int(n);
    }
    return launch_attention(q, Tq, ldq, k, ldk, vt, ldvt, T, heads, head_dim, o, ldo, dev_status,
                            static_cast<cudaStream_t>(stream), nullptr, &split);
}

dit_status_t dit_attention_schedule(int units, int n_kv, int max_ctas, int slots, int *n_cta,
                                    int *n_split, int *items, int64_t cap, int64_t *n_items) {
    if (units <= 0 || n_kv <= 0 || max_ctas <= 0 || slots < 0 || cap < 0)
        return DIT_ERR_INVALID_ARG;
    const AttnGrid g = attn_grid(units, n_kv, max_ctas, slots, true);
    if (n_cta) *n_cta = g.n_cta;
    if (n_split) *n_split = g.n_pc;
    int64_t n = 0;
    for (int c = 0; c < g.n_cta; ++c) {
        const AttnCta cs = attn_cta(g, c);
        for (int i = 0; i < cs.count; ++i, ++n) {
            if (!items || n >= cap) continue;
            const AttnItem it = attn_item(g, cs, c, i);
            int *row = items + 7 * n;
            row[0] = c;
            row[1] = i;
            row[2] = it.u;
            row[3] = it.k0;
            row[4] = it.k1;
            row[5] = it.src;
            row[6] = it.dst;
        }
    }
    if (n_items) *n_items = n;
    return DIT_OK;
}

dit_status_t dit_attention(const void *q, int64_t Tq, int64_t ldq, const void *k, int64_t ldk,
                           const void *vt, int64_t ldvt, int64_t T, int heads, int head_dim,
                           void *o, int64_t ldo, int *dev_status, dit_stream_t stream) {
    return launch_attention(q, Tq, ldq, k, ldk, vt, ldvt, T, heads, head_dim, o, ldo, dev_status,
                            static_cast<cudaStream_t>(stream));
}

}  // extern "C"
