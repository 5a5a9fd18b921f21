/*
 * libditstream — bounded-activation forward pass of one video-DiT block on
 * NVIDIA GB300 (sm_103a).  Plain C ABI: device pointers, sizes and a CUDA
 * stream handle; no C++ or framework types cross this boundary.
 *
 * The method.  "LayerStream: H3 Chunking" (section "How the slicing works"):
 * norm, modulation, the projections and the MLP are token-wise and run on
 * token slices that add into the residual stream in place; attention runs in
 * two passes — pass one keeps only K and V for all tokens, pass two
 * recomputes the queries of one slice, attends them to the full K/V,
 * projects and adds into the residual.  "Proposal: Generic memory-aware
 * streaming execution for transformer models" (section "MLP planning"): a
 * gated MLP may also be cut along its FFN feature axis, each slice passing
 * through the matching slice of the down projection and accumulating into
 * the output.  Section "The two numbers you set" of the first page defines
 * the two knobs: mlp_chunk_tokens and attn_chunk_tokens (0 = unchunked
 * attention).
 *
 * What one block computes (all matrices row-major, weights [out, in]):
 *   a  = LN(x) * (1 + scale1) + shift1                     -> bf16
 *   K, V = a Wk^T, a Wv^T   (all tokens, kept)             -> bf16
 *   Q_s  = a_s Wq^T         (per attention slab s)         -> bf16
 *   O_s  = softmax(Q_s K^T / sqrt(d)) V   per head         -> bf16
 *   x_s += gate1 * (O_s Wo^T)                              (fp32, in place)
 *   b  = LN(x) * (1 + scale2) + shift2  (per MLP chunk)    -> bf16
 *   h_f = silu(b Wg_f^T) * (b Wu_f^T)   (per FFN slice f)  -> bf16
 *   x_c += gate2 * sum_f h_f Wd[:, f]^T                    (fp32, in place)
 * LN is LayerNorm over D, biased variance, eps 1e-6, no affine.
 * modulation is float [6, D] with rows shift1, scale1, gate1, shift2,
 * scale2, gate2.  Accumulation is fp32 throughout.
 *
 * Exactness.  Every kernel computes a token's row with the same operations
 * in the same order whatever the chunk sizes, so the output is bit-identical
 * for every (mlp_chunk_tokens, attn_chunk_tokens) and every ffn_slice.
 *
 * Errors.  No function aborts, traps or prints.  Host-side checks return a
 * negative dit_status_t without launching anything.  Device waits are
 * bounded: a wait that runs out records DIT_ERR_TIMEOUT in the plan's device
 * status word and the kernel returns; dit_block_sync_status() reports it.
 *
 * Threading.  A plan is not re-entrant: one forward at a time per plan (it
 * owns one workspace).  Different plans may run concurrently on different
 * streams.
 */
#ifndef DITSTREAM_H
#define DITSTREAM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DITSTREAM_ABI_VERSION 7

#if defined(__GNUC__)
#define DIT_API __attribute__((visibility("default")))
#else
#define DIT_API
#endif

typedef int dit_status_t;

#define DIT_OK 0
#define DIT_ERR_INVALID_ARG (-1)        /* bad size, NULL pointer, bad mode */
#define DIT_ERR_CHUNK_ALIGN (-2)        /* chunk not 0 and not a multiple of 128 */
#define DIT_ERR_ALIGN (-3)              /* device pointer not 16-byte aligned */
#define DIT_ERR_NO_WORKSPACE (-4)       /* forward before bind_workspace */
#define DIT_ERR_WORKSPACE_TOO_SMALL (-5)
#define DIT_ERR_CUDA (-6)               /* launch / runtime error: see dit_last_cuda_error() */
#define DIT_ERR_TIMEOUT (-7)            /* a bounded device wait ran out */
#define DIT_ERR_UNSUPPORTED_ARCH (-8)   /* current device is not sm_103 */

/* CUDA stream handle (a cudaStream_t); NULL = the legacy default stream. */
typedef void *dit_stream_t;

/* Weight element types. */
#define DIT_W_BF16 0
#define DIT_W_INT8 1

/* One block's weights: borrowed, read-only device pointers, row-major
 * [out, in] (the nn.Linear.weight layout), 16-byte aligned.
 *   wqkv  [3D, D]  rows 0..D-1 = Wq, D..2D-1 = Wk, 2D..3D-1 = Wv;
 *                  head h owns rows h*d .. h*d+d-1 of each third
 *   wo    [D, D]
 *   wgate [F, D]   (SwiGLU gate projection: silu is applied to it)
 *   wup   [F, D]
 *   wdown [D, F]
 * dtype DIT_W_BF16: bf16 elements.  dtype DIT_W_INT8: int8 elements q and
 * one fp32 scale per output row in the matching *_scale pointer; the weight
 * is W[r, :] = scale[r] * q[r, :] ("MiniMax-H3-Comfy-NPU", section 2.2: one
 * weight_scale per output row, sliced with the rows).  Scales are ignored
 * for bf16. */
typedef struct {
    int dtype;
    const void *wqkv;
    const void *wo;
    const void *wgate;
    const void *wup;
    const void *wdown;
    const float *wqkv_scale;
    const float *wo_scale;
    const float *wgate_scale;
    const float *wup_scale;
    const float *wdown_scale;
} dit_block_weights_t;

typedef struct dit_plan dit_plan_t;

/* Plan one block: T tokens, hidden D, `heads` heads of d = D/heads, SwiGLU
 * width ffn.  Pure host work; allocates no device memory.
 *   T >= 1; D % 128 == 0; d in {64, 128}; ffn % 64 == 0 and ffn >= 64.
 *   mlp_chunk_tokens, attn_chunk_tokens: 0 (one slab of all T tokens) or a
 *   multiple of 128; values >= T are clamped to T ("The two numbers you set":
 *   attn_chunk_tokens = 0 turns the two-pass slicing off; the MLP half is
 *   still chunked by mlp_chunk_tokens).
 * The FFN is not feature-sliced (slice width = ffn); see dit_block_plan_ex.
 * No CUDA call is made here (the device is checked when a workspace is
 * bound).  On success *out receives a plan owned by the caller
 * (dit_block_plan_destroy).  Errors: DIT_ERR_INVALID_ARG,
 * DIT_ERR_CHUNK_ALIGN. */
DIT_API dit_status_t dit_block_plan(int64_t T, int D, int heads, int ffn,
                            int mlp_chunk_tokens, int attn_chunk_tokens,
                            dit_plan_t **out);

/* As dit_block_plan, plus ffn_slice: 0 (= ffn) or a multiple of 64 that is
 * <= ffn — the FFN feature-slice width ("MLP planning").  With a slice width
 * below ffn the down projection's fp32 accumulator is carried across slices
 * in the workspace, so the result stays bit-identical to ffn_slice = ffn. */
DIT_API dit_status_t dit_block_plan_ex(int64_t T, int D, int heads, int ffn,
                               int mlp_chunk_tokens, int attn_chunk_tokens,
                               int ffn_slice, dit_plan_t **out);

/* Plan with automatic chunk sizes: the largest chunks whose workspace fits
 * budget_bytes ("LayerStream: H3 Chunking", "The two numbers you set": use
 * the largest chunk that fits; "Proposal: Generic memory-aware streaming
 * execution ...", "Automatic chunk sizing").  The attention slab is chosen
 * first (largest multiple of 128 tokens, or all T, that fits); then the MLP
 * token chunk, largest first, with the FFN unsliced unless a slice width of
 * ffn/2, ffn/4, ... (at least 1024 features) lets a token chunk at least 25%
 * larger fit (a slice's fp32 carry costs 4*C_m*D bytes).
 * Any choice gives bit-identical results.  Errors: as dit_block_plan, and
 * DIT_ERR_WORKSPACE_TOO_SMALL when even 128-token chunks do not fit (K and V
 * of all T tokens alone take 4*T*D bytes). */
DIT_API dit_status_t dit_block_plan_auto(int64_t T, int D, int heads, int ffn,
                                         size_t budget_bytes, dit_plan_t **out);

DIT_API void dit_block_plan_destroy(dit_plan_t *plan);

/* Effective sizes of a plan after clamping: fills any non-NULL pointer. */
DIT_API dit_status_t dit_block_plan_info(const dit_plan_t *plan, int64_t *T, int *D,
                                 int *heads, int *ffn, int *mlp_chunk,
                                 int *attn_chunk, int *ffn_slice);

/* Exact device workspace bytes the plan needs:
 *   1024 (header: status word, attention hand-off flags)
 *   + K [T, D] bf16 + V^T [D, roundup(T, 128)] bf16
 *   + max(attention phase 4 * C_a * D + hand-off state,
 *         MLP phase 2 * C_m * D + 2 * C_m * F_s + (F_s < F ? 4 * C_m * D : 0))
 *   + the GEMMs' hand-off state
 * each region rounded up to 1 KiB, plus the LoRA regions when the plan has a
 * LoRA rank (dit_block_plan_set_lora_rank).  The attention's hand-off state
 * is that of dit_attention_ex: slots x 1024 * (head_dim + 2) bytes, slots the
 * most CTAs that would share the split part (the partial last wave, or with
 * the extended split one range per CTA) of ceil(C_a / 256) * heads units on
 * a device of 128 to 160 multiprocessors (0 when no such device would split;
 * at most 160).  The GEMMs' is that of dit_gemm_ex: 128 KiB per
 * slot, slots the most that any of the plan's GEMM launches (K/V, Q, O,
 * gate/up, down, at full and ragged chunk and slice sizes, in either tile
 * shape) would use on such a device, at most 64.  K/V for all tokens is the floor that grows with T ("Where
 * people get burned": K and V of the whole sequence stay resident);
 * everything else is bounded by the chunk sizes. */
DIT_API size_t dit_block_workspace_bytes(const dit_plan_t *plan);

/* Bind caller-owned device memory (>= dit_block_workspace_bytes, 256-byte
 * aligned) as the plan's workspace and clear its header (status word and
 * hand-off flags).  The current
 * device must be of compute capability 10.3.  The library never allocates
 * device memory itself.  Errors: DIT_ERR_INVALID_ARG, DIT_ERR_ALIGN,
 * DIT_ERR_WORKSPACE_TOO_SMALL, DIT_ERR_UNSUPPORTED_ARCH, DIT_ERR_CUDA. */
DIT_API dit_status_t dit_block_bind_workspace(dit_plan_t *plan, void *dev_ptr,
                                      size_t bytes);

/* K/V offload below the K/V floor.  "LayerStream: H3 Chunking" ("Where
 * people get burned"): K and V of the whole sequence stay resident, a floor
 * that chunking cannot go under; only K/V offload can.  With
 * key_block_tokens > 0 (a multiple of 128) K [T, D] and V^T [D, T_pad] of
 * all tokens live in caller-owned pinned host memory instead of the device
 * workspace:
 *   - pass one's K/V projection writes each key block into a device ring
 *     slot, copied out to the host buffer on the plan's copy stream;
 *   - pass two streams them back, per query slab, in blocks of
 *     key_block_tokens keys through a two-slot device ring (copies on the
 *     plan's own copy stream, one block ahead of the attention), and the
 *     attention carries its running max, sum and fp32 output from block to
 *     block in the workspace.
 * Key tiles are visited in the same order with the same arithmetic, so the
 * output bits equal the resident schedule's.  The workspace then holds the
 * ring (2 x 4 * key_block_tokens * D bytes) and the carried state
 * (4 * C_a * D + 8 * C_a * heads bytes) instead of 4 * T * D, so it no longer
 * grows with T.
 * dit_block_plan_set_kv_offload: before a workspace is bound (else
 * DIT_ERR_INVALID_ARG); 0 turns it off (the default).
 * dit_block_kv_host_bytes: bytes of the host buffer, 2 T D + 2 D kvb n_kb
 * (K [T, D], then V^T per key block [n_kb][D][kvb], n_kb = ceil(T / kvb),
 * so that every copy is one contiguous range); 0 when offload is off.
 * dit_block_bind_kv_host: bind the host buffer (allocated with
 * cudaHostAlloc or registered with cudaHostRegister, so that the device can
 * address it; 16-byte aligned, >= dit_block_kv_host_bytes) and create the
 * plan's copy stream and events on the current device (released by
 * dit_block_plan_destroy).  Errors: DIT_ERR_INVALID_ARG,
 * DIT_ERR_ALIGN, DIT_ERR_WORKSPACE_TOO_SMALL, DIT_ERR_CUDA (the buffer is not
 * mapped for the device).  A forward of an offloading plan without a bound
 * host buffer returns DIT_ERR_NO_WORKSPACE. */
DIT_API dit_status_t dit_block_plan_set_kv_offload(dit_plan_t *plan, int key_block_tokens);
DIT_API size_t dit_block_kv_host_bytes(const dit_plan_t *plan);
DIT_API dit_status_t dit_block_bind_kv_host(dit_plan_t *plan, void *host_ptr, size_t bytes);

/* Optional weight scratch for int8 blocks.  An int8 weight value q
 * (|q| <= 127) is exact in bf16, so with a scratch bound the forward expands
 * each phase's int8 weights into it (Wqkv and Wo before pass one; Wgate,
 * Wup and Wdown after pass two) and runs the bf16 tensor-core main loop,
 * applying the same per-row scale to the fp32 accumulator as the int8 path
 * ("MiniMax-H3-Comfy-NPU" section 2.2: W = s_row * q).  The MMAs see the
 * same operands in the same order, so the output bits are the same as
 * without the scratch; the GEMMs skip the in-kernel shared-memory conversion,
 * for 2 * max(4 D^2, 3 D F) bytes of weight scratch (independent of T and of
 * the chunks; the resident weights stay int8).  bf16 weights ignore it.
 * dit_block_weight_scratch_bytes: the size needed.
 * dit_block_bind_weight_scratch: bind caller-owned device memory (>= that
 * size, 256-byte aligned); dev_ptr = NULL unbinds.  Errors:
 * DIT_ERR_INVALID_ARG, DIT_ERR_ALIGN, DIT_ERR_WORKSPACE_TOO_SMALL. */
DIT_API size_t dit_block_weight_scratch_bytes(const dit_plan_t *plan);
DIT_API dit_status_t dit_block_bind_weight_scratch(dit_plan_t *plan, void *dev_ptr,
                                                   size_t bytes);

/* One block forward, in place on x [T, D] fp32 (device, caller-owned,
 * 16-byte aligned).  modulation: device float [6, D].  Asynchronous on
 * `stream`; returns the launch-time status.  Device-side errors are read by
 * dit_block_sync_status().  Errors: DIT_ERR_INVALID_ARG, DIT_ERR_ALIGN,
 * DIT_ERR_NO_WORKSPACE, DIT_ERR_CUDA.
 * The GEMMs cut their last wave of output tiles into K ranges in a
 * cooperative launch; with the environment variable DITSTREAM_GEMM_SPLIT=0
 * (read once per process) they run whole tiles only, with the same output
 * bits, for tools that cannot launch cooperative cluster grids. */
DIT_API dit_status_t dit_block_forward(const dit_plan_t *plan, float *x,
                               const dit_block_weights_t *w,
                               const float *modulation, dit_stream_t stream);

/* Optional per-head transform of Q and K, applied in the fp32 epilogues of
 * the Q and K projections before their bf16 store.  For one token at
 * sequence position p and one head h, with u its head_dim values of Q (or K):
 *   u <- u / sqrt(mean(u^2) + eps) * norm          when norm != NULL
 *   (u[2i], u[2i+1]) <- (u[2i] c - u[2i+1] s, u[2i] s + u[2i+1] c),
 *       c = rope_cos[p, i], s = rope_sin[p, i]     when rope_cos != NULL
 * norm is q_norm for Q and k_norm for K: device fp32 [head_dim], the same for
 * every head.  rope_cos, rope_sin: device fp32 [T, head_dim / 2] row-major,
 * 16-byte aligned, both NULL or both set; one row of angles per token, shared
 * by all heads and by Q and K (a 3-D video rotary embedding is one such
 * table, laid out by the caller).  eps > 0.
 * "Proposal: Generic memory-aware streaming execution for transformer
 * models", attention section: the model's Q normalisation and positional
 * transform are applied to each bounded Q region before its attention; the
 * block description lists optional Q/K normalisation and a RoPE step.  The
 * page names the steps only: the RMSNorm with a learned weight and the
 * rotation of interleaved pairs are this library's reading. */
typedef struct {
    const float *q_norm;    /* [head_dim] or NULL */
    const float *k_norm;    /* [head_dim] or NULL */
    const float *rope_cos;  /* [T, head_dim / 2] or NULL */
    const float *rope_sin;  /* [T, head_dim / 2] or NULL */
    float eps;
} dit_qk_t;

/* dit_block_forward with the Q/K transform `qk` (NULL: none, identical to
 * dit_block_forward).  The transform is row-local and uses each token's
 * position in the whole sequence, so the output stays bit-identical across
 * chunk settings.  Errors: as dit_block_forward; DIT_ERR_INVALID_ARG when
 * only one of rope_cos / rope_sin is set or eps <= 0, DIT_ERR_ALIGN for a
 * table or weight not 16-byte aligned. */
DIT_API dit_status_t dit_block_forward_qk(const dit_plan_t *plan, float *x,
                                          const dit_block_weights_t *w,
                                          const float *modulation,
                                          const dit_qk_t *qk, dit_stream_t stream);

/* Activation-space LoRA ("ComfyUI-StaticPipeline", section "Activation-space
 * LoRA (bypass mode)"): an adapted linear computes y = W x + alpha B (A x)
 * with W left as it is (bf16 or packed int8).  Here the delta joins W's
 * product inside the same tensor-core accumulation: u = x A^T (bf16, one
 * small GEMM per token chunk), then ceil(rank / 64) extra K-steps of
 * u B'^T after W's, so every fused epilogue (SwiGLU, gated residual, the
 * down projection's carry) sees W x + delta before its nonlinearity.
 * B' = alpha * B (divided by W's int8 row scale, which the epilogue applies)
 * is made once per adapter by dit_lora_prepare.
 *   a: device bf16 [rank, in] row-major (in = D, or ffn for "down");
 *   b: device bf16 [out, rank] row-major, the output of dit_lora_prepare;
 *   rank: multiple of 32, at most the plan's LoRA rank; a == NULL or
 *   b == NULL: no adapter on that linear.
 * The fused Q/K/V projection has one adapter whose B rows follow Wqkv's
 * (out = 3D: rows of Q, then K, then V). */
typedef struct {
    const void *a;
    const void *b;
    int rank;
} dit_lora_t;

typedef struct {
    dit_lora_t qkv, o, gate, up, down;
} dit_block_lora_t;

#define DIT_LORA_MAX_RANK 256

/* b_out[n, j] = bf16_rne(alpha * b[n, j] / row_scale[n]) for n < rows,
 * j < rank (row_scale == NULL: no division).  b, b_out: device bf16, row
 * strides ld_b, ld_out elements (>= rank, multiples of 8); row_scale: the
 * int8 scales of the adapted weight's rows (the same rows as b's), or NULL
 * for bf16 weights.  Asynchronous on `stream`.
 * Errors: DIT_ERR_INVALID_ARG, DIT_ERR_ALIGN, DIT_ERR_CUDA. */
DIT_API dit_status_t dit_lora_prepare(const void *b, int64_t rows, int rank, int64_t ld_b,
                                      float alpha, const float *row_scale, void *b_out,
                                      int64_t ld_out, dit_stream_t stream);

/* Reserve workspace for adapters of rank <= max_rank (a multiple of 32, at
 * most DIT_LORA_MAX_RANK; 0 = none, the default).  Must be called before a
 * workspace is bound (else DIT_ERR_INVALID_ARG).  The workspace grows by
 * 4*C_a*R (u of the Q/K/V and O adapters) plus 6*C_m*R, and 4*C_m*R more when
 * the FFN is sliced (u of gate, up, down and the down adapter's fp32 carry). */
DIT_API dit_status_t dit_block_plan_set_lora_rank(dit_plan_t *plan, int max_rank);

/* dit_block_forward with the optional Q/K transform (`qk`, see dit_qk_t)
 * and activation-space LoRA adapters (`lora`); either may be NULL.  The
 * output stays bit-identical across chunk settings and FFN slice widths.
 * Errors: as dit_block_forward_qk; DIT_ERR_INVALID_ARG when an adapter's
 * rank is not a multiple of 32 or exceeds the plan's LoRA rank,
 * DIT_ERR_ALIGN for an adapter matrix not 16-byte aligned. */
DIT_API dit_status_t dit_block_forward_ex(const dit_plan_t *plan, float *x,
                                          const dit_block_weights_t *w,
                                          const float *modulation, const dit_qk_t *qk,
                                          const dit_block_lora_t *lora,
                                          dit_stream_t stream);

/* Block forward that allocates nothing.  The method's pages have no
 * counterpart to this entry point: it exists for callers that cannot
 * allocate device memory (code that runs under an allocator owning every
 * device byte, or where allocation is not allowed), so it needs no
 * workspace bound to the plan.  Same computation, kernels and result bits as
 * dit_block_forward; the scratch is a file-scope device array of 64 MiB
 * (DIT_STATIC_SCRATCH_BYTES) that every device loading the library holds
 * until the process exits.
 *   - Plans whose dit_block_workspace_bytes exceeds that size are rejected
 *     with DIT_ERR_WORKSPACE_TOO_SMALL before anything is launched.
 *   - The first call on a device sets up the scratch address for that
 *     device (with that device current) and clears the scratch's header;
 *     make that first call before any stream capture.  Under lazy module
 *     loading (the CUDA default) the driver reserves the 64 MiB array on
 *     that first call, so the device's free memory drops by that much then;
 *     later calls reserve nothing.
 *   - All calls share one scratch, which keeps the last call's contents:
 *     calls whose work overlaps on the GPU (concurrent streams, several
 *     host threads) race and give wrong results.  Serialise them.  The plan
 *     is only read: ordinary calls on the same plan (with its own bound
 *     workspace) do not interfere with static ones.
 *   - Each call clears the scratch's hand-off flags; its status word is
 *     kept.  A bounded device wait that runs out in a static call is
 *     recorded there and reported (and cleared) by the next
 *     dit_block_sync_status on that device, for any plan.
 *   - No per-kernel timing is recorded, whatever the plan's profiling flag.
 *   - Calls no cudaMalloc/cudaFree or any other allocating routine.
 * Errors: as dit_block_forward, plus DIT_ERR_WORKSPACE_TOO_SMALL and
 * DIT_ERR_UNSUPPORTED_ARCH. */
#define DIT_STATIC_SCRATCH_BYTES (64u << 20)
DIT_API dit_status_t dit_block_forward_static(const dit_plan_t *plan, float *x,
                                              const dit_block_weights_t *w,
                                              const float *modulation,
                                              dit_stream_t stream);

/* Synchronise `stream`, read and clear the plan's device status word (after
 * a failure also the attention hand-off flags, which a launch that gave up
 * may have left set).  Once a dit_block_forward_static call has set up the
 * current device, the static scratch's status word is read and cleared the
 * same way, so a wait that ran out in any static call on this device is
 * reported here.  Returns DIT_OK, DIT_ERR_TIMEOUT or DIT_ERR_CUDA. */
DIT_API dit_status_t dit_block_sync_status(const dit_plan_t *plan, dit_stream_t stream);

/* Final layer (output head), fp32 arithmetic, unsliced:
 *   out[t, :] = (LN(x[t]) * (1 + scale_f) + shift_f) W_f^T
 * x [T, D] fp32; mod_f [2, D] fp32 (shift_f, scale_f); W_f [64, D] fp32 when
 * wf_scale == NULL, else int8 with fp32 scales [64]; out [T, 64] fp32.
 * "LayerStream: H3 Chunking" ("How the slicing works"): the fp32 output head
 * runs stock.  Uses the plan's T and D only; needs no workspace (when one is
 * bound, a bounded device wait that runs out is recorded in its status word
 * and reported by dit_block_sync_status).  Arithmetic is fp32-level: the
 * statistics and the output in fp32, the D-long contraction on the tensor
 * cores as three products of operands split into two tf32 parts each, with
 * fp32 partial sums over 128 values of k.  Asynchronous on `stream`.
 * Errors: DIT_ERR_INVALID_ARG (null pointer, D not a multiple of 32),
 * DIT_ERR_ALIGN (a pointer not 16-byte aligned), DIT_ERR_CUDA. */
DIT_API dit_status_t dit_final_forward(const dit_plan_t *plan, const float *x,
                               const void *wf, const float *wf_scale,
                               const float *mod_f, float *out,
                               dit_stream_t stream);

/* ----------------------------------------------------------------------
 * Per-kernel timing.  When enabled, every kernel that dit_block_forward and
 * dit_final_forward launch is bracketed by two CUDA events recorded on the
 * launching stream.  dit_block_profile_read() waits for those events, adds
 * up, per kernel kind, the elapsed milliseconds, the launch count and the
 * algorithmic work (flops for the tensor-core kinds: 2*M*N*K per GEMM,
 * 4*rows*T*D per attention launch; bytes for the memory-bound kinds:
 * 6*rows*D per modln launch, 4*T*D + 4*64*D + 4*64*T per final-layer launch),
 * writes them to the caller's arrays of DIT_NUM_KINDS entries (any may be
 * NULL) and clears the record.  Events are created by the library and kept
 * with the plan.
 * ---------------------------------------------------------------------- */
#define DIT_K_MODLN 0
#define DIT_K_GEMM_KV 1
#define DIT_K_GEMM_Q 2
#define DIT_K_ATTENTION 3
#define DIT_K_GEMM_O 4
#define DIT_K_GEMM_SWIGLU 5
#define DIT_K_GEMM_DOWN 6
#define DIT_K_FINAL 7
#define DIT_K_LORA_U 8      /* LoRA u = x A^T GEMMs (dit_block_forward_ex) */
#define DIT_K_EXPAND 9      /* int8 -> bf16 weight expansion (weight scratch) */
#define DIT_NUM_KINDS 10

DIT_API dit_status_t dit_block_profile_enable(dit_plan_t *plan, int enable);
DIT_API dit_status_t dit_block_profile_read(dit_plan_t *plan, double *ms,
                                            int64_t *launches, double *work);

DIT_API const char *dit_status_string(dit_status_t s);
/* Text of the last CUDA error seen by this thread's calls ("" if none). */
DIT_API const char *dit_last_cuda_error(void);
DIT_API int dit_abi_version(void);

/* ----------------------------------------------------------------------
 * Stage entry points: the individual kernels of the block, for per-stage
 * checks.  Same conventions as above.  `dev_status` is an optional device
 * int (NULL allowed) that receives DIT_ERR_TIMEOUT if a bounded wait ran
 * out.  bf16 data is passed as raw 16-bit patterns (void *).
 * ---------------------------------------------------------------------- */

/* Norm + modulation + cast ("How the slicing works": norms and modulation
 * are token-wise).  out[r, c] = bf16_rne((x[r,c] - mu_r) * rsqrt(var_r +
 * 1e-6) * (1 + scale[c]) + shift[c]) for r < rows; x fp32 [rows, D] row-major;
 * out bf16 [rows, D].  D % 128 == 0. */
DIT_API dit_status_t dit_modln_cast(const float *x, int64_t rows, int D,
                            const float *shift, const float *scale,
                            void *out_bf16, dit_stream_t stream);

/* Epilogues of the tensor-core GEMM  acc[M, N] = A[M, K] B[N, K]^T
 * (A bf16, B bf16 or int8 with per-row fp32 scale applied to acc). */
#define DIT_EPI_STORE_BF16 0  /* out bf16 [M, N], row stride ldo; if acc_load
                                 the fp32 accumulator starts from acc[m, n]  */
#define DIT_EPI_STORE_F32 1   /* out fp32 [M, N], row stride ldo             */
#define DIT_EPI_KV 2          /* n < split_n: out (K) bf16 [row_offset+m, n],
                                 stride ldo; n >= split_n: out2 (V^T) bf16
                                 [n - split_n, row_offset + m], stride ldo2 */
#define DIT_EPI_RESID 3       /* x[m, n] += gate[n] * acc  (fp32, stride ldx) */
#define DIT_EPI_SWIGLU 4      /* two B operands b0 (gate) and b1 (up), each
                                 [N, K]: out bf16 [m, n] = silu(acc0) * acc1 */
#define DIT_EPI_DOWN 5        /* accumulate over FFN slices: if acc_load the
                                 fp32 accumulator starts from acc[m, n], else
                                 from 0; if acc_final x[m, n] += gate[n]*acc,
                                 else acc[m, n] = acc (fp32, stride ldacc)    */

typedef struct {
    int mode;               /* DIT_EPI_* */
    int64_t M;              /* rows of A (tokens) */
    int N;                  /* output columns, N % 32 == 0 */
    int K;                  /* contraction, K % 64 == 0 */
    const void *a;          /* bf16 [M, K], row stride lda elements */
    int64_t lda;
    const void *b0;         /* [N, K], row stride ldb elements */
    const void *b1;         /* second B (SWIGLU only) */
    int64_t ldb;
    int b_dtype;            /* DIT_W_BF16 or DIT_W_INT8 */
    const float *b0_scale;  /* per-row scales [N]: int8 B, or bf16 B holding
                               int8 values (dit_int8_to_bf16); else NULL */
    const float *b1_scale;
    void *out;              /* STORE_*, KV (K), SWIGLU */
    int64_t ldo;
    void *out2;             /* KV: V^T */
    int64_t ldo2;
    int64_t row_offset;     /* KV: row of K (column of V^T) that A's row 0 lands in */
    int split_n;            /* KV: first V column */
    float *x;               /* RESID, DOWN */
    int64_t ldx;
    const float *gate;      /* RESID, DOWN: [N] */
    float *acc;             /* DOWN: fp32 carry [M, N] */
    int64_t ldacc;
    int acc_load;
    int acc_final;
    int flags;              /* 0, or DIT_GEMM_FLAG_* test hooks */
    /* Q/K transform (see dit_qk_t) on STORE_BF16 output and on the K columns
     * (n < split_n) of KV output; off when qk_norm and rope_cos are NULL.
     * Heads are head_dim (64 or 128) consecutive columns; the rotary position
     * of row m is rope_pos0 + m. */
    const float *qk_norm;   /* [head_dim] or NULL */
    const float *rope_cos;  /* [positions, head_dim / 2] or NULL */
    const float *rope_sin;
    int head_dim;
    float qk_eps;
    /* LoRA K-steps (see dit_lora_t): after the K-steps of A B^T the
     * accumulator takes ceil(rank / 64) more of U L^T, U = lora_u bf16
     * [M, rank] (row stride lora_ldu), L = lora_l bf16 [N, rank] (row stride
     * lora_ldl), rank % 8 == 0, <= DIT_LORA_MAX_RANK.  Half 0 (lora_*0)
     * feeds every output column (SWIGLU: the gate's), half 1 only the up
     * accumulator of SWIGLU.  lora_l0 == NULL and lora_l1 == NULL: off. */
    const void *lora_u0;
    int64_t lora_ldu0;
    const void *lora_l0;
    int64_t lora_ldl0;
    int lora_rank0;
    const void *lora_u1;
    int64_t lora_ldu1;
    const void *lora_l1;
    int64_t lora_ldl1;
    int lora_rank1;
    int64_t rope_pos0;      /* rotary position of A's row 0 (Q/K transform) */
} dit_gemm_args_t;

/* Test hook for failure detection: CTA 0's producer arms its first
 * shared-memory stage but withholds the copy, so the MMA's bounded wait runs
 * out.  The kernel then records DIT_ERR_TIMEOUT in *dev_status, lets its
 * in-flight copies and MMAs land, frees its tensor memory and returns
 * (after about two wait limits, ~4 s); the CUDA context stays usable. */
#define DIT_GEMM_FLAG_INJECT_STALL 1

DIT_API dit_status_t dit_gemm(const dit_gemm_args_t *args, int *dev_status,
                      dit_stream_t stream);

/* dit_gemm with the work split of its persistent grid: the output tiles of
 * a launch go to at most max_ctas CTAs (0: one per multiprocessor); when the
 * tiles that would form a last, partial wave are worth cutting, their K-steps
 * (64 wide) are cut into ranges shared by all CTAs, each continuing the raw
 * fp32 accumulator of the range before it, so every output element is still
 * one accumulation over K in the same order: the result equals dit_gemm bit
 * for bit.  split_ws: device memory of dit_gemm_split_bytes(slots) bytes,
 * 16-byte aligned, zero before its first use (a successful launch leaves it
 * so); bytes [0, 1024) hold one flag per slot, the rest `slots` accumulator
 * slots of 128 KiB (slots = (split_bytes - 1024) / 131072, at most 64).  A
 * launch splits only if it needs no more slots than that; split_ws = NULL
 * never splits.  Launches sharing one split_ws must not overlap on the
 * device.  Errors: as dit_gemm. */
DIT_API size_t dit_gemm_split_bytes(int slots);
DIT_API dit_status_t dit_gemm_ex(const dit_gemm_args_t *args, void *split_ws,
                                 size_t split_bytes, int max_ctas, int *dev_status,
                                 dit_stream_t stream);

/* dit_attention over one block of a longer key sequence (keys k0 .. k0 +
 * T_block - 1 of it, k and vt pointing at that block), carrying the softmax
 * state between the blocks, which must be passed in ascending key order:
 * o_state fp32 [Tq, H*d] (row stride ld_state, a multiple of 4), m_state and
 * l_state fp32 [Tq, H] hold the running max, sum and unnormalised output.
 * first != 0: the state is started here; last != 0: the output is
 * normalised into o (bf16), else the state is written back.  Every block but
 * the last holds a multiple of 128 keys.  The result equals one dit_attention
 * call over all the keys bit for bit. */
DIT_API dit_status_t dit_attention_part(const void *q, int64_t Tq, int64_t ldq,
                                        const void *k, int64_t ldk, const void *vt,
                                        int64_t ldvt, int64_t T_block, int heads,
                                        int head_dim, void *o, int64_t ldo, float *o_state,
                                        float *m_state, float *l_state, int64_t ld_state,
                                        int first, int last, int *dev_status,
                                        dit_stream_t stream);

/* out[i] = bf16(q[i]) for n int8 values q (exact: |q| <= 127 needs 8 bits).
 * n % 16 == 0; q, out 16-byte aligned.  The weight scratch's expansion. */
DIT_API dit_status_t dit_int8_to_bf16(const void *q, int64_t n, void *out,
                                      dit_stream_t stream);

/* Non-causal multi-head attention of Tq queries against T keys:
 *   o[i, h*d:(h+1)*d] = softmax(q_h[i] . k_h^T / sqrt(d)) v_h
 * q bf16 [Tq, H*d] (stride ldq), k bf16 [T, H*d] (stride ldk), V given
 * transposed: vt bf16 [H*d, ldvt] with vt[c, j] = V[j, c] (ldvt >= T,
 * ldvt % 8 == 0), o bf16 [Tq, H*d] (stride ldo).  head_dim in {64, 128}.
 * The key loop visits key tiles in one fixed order, so a query row's result
 * does not depend on Tq or on the other queries. */
DIT_API dit_status_t dit_attention(const void *q, int64_t Tq, int64_t ldq,
                           const void *k, int64_t ldk, const void *vt,
                           int64_t ldvt, int64_t T, int heads, int head_dim,
                           void *o, int64_t ldo, int *dev_status,
                           dit_stream_t stream);

/* dit_attention with the persistent kernel's work split.  The (query pair,
 * head) units of a launch are spread over at most max_ctas CTAs (0: one per
 * multiprocessor); the units that would form a last, partial wave (and,
 * when few are left over, one more whole unit per CTA) are cut into key
 * ranges shared by the CTAs, each range continuing the running max, sum and
 * fp32 output of the range before it, so that every CTA gets about the same
 * number of key tiles.  Key tiles are still visited in ascending order
 * with the same arithmetic: the result equals dit_attention bit for bit.
 * split_ws: device memory of dit_attention_split_bytes(head_dim, slots)
 * bytes, 16-byte aligned, zero before its first use (the call leaves it so
 * after a successful launch); bytes [0, 1024) hold one flag per slot, the
 * rest the hand-off state of `slots` slots (slots = (split_bytes - 1024) /
 * (1024 * (head_dim + 2)), at most 160).  A launch splits only if it needs no
 * more slots than that; split_ws = NULL never splits.  Launches sharing one
 * split_ws must not overlap on the device.  Errors: as dit_attention. */
DIT_API size_t dit_attention_split_bytes(int head_dim, int slots);
DIT_API dit_status_t dit_attention_ex(const void *q, int64_t Tq, int64_t ldq,
                                      const void *k, int64_t ldk, const void *vt,
                                      int64_t ldvt, int64_t T, int heads, int head_dim,
                                      void *o, int64_t ldo, void *split_ws,
                                      size_t split_bytes, int max_ctas, int *dev_status,
                                      dit_stream_t stream);

/* The persistent attention's work list, computed on the host exactly as the
 * kernel computes it: `units` (query pair, head) units of n_kv key tiles on
 * at most max_ctas CTAs with `slots` hand-off slots.  Writes the CTA count
 * and the number of CTAs that share the remainder (0: none), and, while
 * they fit in `cap` rows, one row of 7 ints per work item in each CTA's
 * processing order: (cta, index, unit, first key tile, end key tile, slot
 * read at the start or -1, slot written at the end or -1); *n_items is the
 * total.  Host only; for checking the schedule. */
DIT_API dit_status_t dit_attention_schedule(int units, int n_kv, int max_ctas, int slots,
                                            int *n_cta, int *n_split, int *items,
                                            int64_t cap, int64_t *n_items);

#ifdef __cplusplus
}
#endif

#endif /* DITSTREAM_H */
