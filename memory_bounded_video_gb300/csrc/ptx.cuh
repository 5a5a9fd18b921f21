// Inline-PTX helpers for sm_103a: mbarriers, TMA tile loads, tcgen05 (TMEM
// allocation, MMA, commit, TMEM load/store) and the shared-memory matrix
// descriptors of the 5th-generation tensor cores.  Written from the public
// PTX ISA description of these instructions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#define DEV __device__ __forceinline__

namespace ds {

// Device status codes (mirror of include/ditstream.h).
constexpr int kErrTimeout = -7;

// A bounded wait gives up after this many nanoseconds (~2 s): long enough
// for a time-sliced shared GPU, short enough that a lost arrival is reported
// instead of hanging the device.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

DEV uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

DEV uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------ mbarrier
DEV void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
                 : "memory");
}
DEV void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
DEV void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
DEV void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar)
                 : "memory");
}
// One arrival for the whole warp (the barrier counts warps, not threads):
// after __syncwarp, lane 0 arrives with release semantics, so every lane's
// earlier writes and fences are ordered before the arrival.  One atomic on
// the barrier word instead of 32.  All lanes of the warp must call it.
DEV void mbar_arrive_warp(uint32_t bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}
DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
        "r"(bytes)
        : "memory");
}
DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Per-CTA failure state for bounded waits.  `abort` lives in shared memory;
// once any wait of the CTA runs out every later wait returns false at once.
struct WaitCtx {
    volatile int *abort;  // shared
    int *status;          // global, may be null
};

DEV void record_timeout(const WaitCtx &w) {
    *w.abort = 1;
    if (w.status) atomicCAS(w.status, 0, kErrTimeout);
}

// Wait for the phase of parity `parity` of barrier `bar` to complete.
// Returns false (after recording DIT_ERR_TIMEOUT) if it did not within the
// limit, or if another wait of this CTA already gave up.
DEV bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtx &w) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    uint32_t n = 0;
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((++n & 255u) == 0) {
            if (*w.abort) return false;
            if (globaltimer() - t0 > kWaitLimitNs) {
                record_timeout(w);
                return false;
            }
        }
    }
}

// Short wait used during teardown after a failure: never records anything.
DEV void mbar_wait_quiet(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > limit_ns) return;
    }
}

// ------------------------------------------------------------ clusters
DEV uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
DEV uint32_t cluster_id_x() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
// All threads of every CTA of the cluster: arrive (release) and wait
// (acquire).  Only reached on paths every thread takes; every other wait in
// the kernels that use it is bounded, so it cannot wait forever.
DEV void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Shared-memory address of the same variable in CTA `rank` of the cluster.
DEV uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// Arrive on a barrier of another CTA of the cluster (address from
// mapa_shared), with release semantics at CTA scope, the form used for
// cross-CTA pipeline barriers in tensor-core GEMMs; at cluster scope the
// arrival cost the issuing thread about 400 ns more (measured: the pair
// GEMM's K-step went from 365 to 742 ns with one such arrival per K-step).
// The issuing thread still waits several hundred ns for it, so pipelines
// keep it off their per-K-step critical threads.
DEV void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}
// One such arrival for the whole warp; all lanes call it.
DEV void mbar_arrive_remote_warp(uint32_t cluster_addr) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive_remote(cluster_addr);
}

// ------------------------------------------------------------ hand-off flags
// A CTA that continues another CTA's partial result waits for that CTA's
// flag (global int, 0 or 1): release / acquire at device scope.
DEV void flag_release(int *f) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(f), "r"(1) : "memory");
}
DEV int flag_acquire(const int *f) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v;
}

// Bounded wait for a hand-off flag; false (with the timeout recorded) if it
// was not set within the limit or another wait of this CTA gave up.
DEV bool flag_wait(const int *f, const WaitCtx &w) {
    if (flag_acquire(f)) return true;
    const uint64_t t0 = globaltimer();
    while (true) {
        __nanosleep(128);
        if (flag_acquire(f)) return true;
        if (*w.abort) return false;
        if (globaltimer() - t0 > kWaitLimitNs) {
            record_timeout(w);
            return false;
        }
    }
}

// ------------------------------------------------------------ TMA
DEV void tma_prefetch_desc(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m))
                 : "memory");
}
// 2-D tiled load of box (x = inner coordinate, y = outer) into shared memory,
// completing `bytes` of transaction on barrier `bar`.
DEV void tma_load_2d(uint32_t dst, const CUtensorMap *m, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

// Pair form: a CTA of a cluster pair loads into its own shared memory and
// completes the bytes on barrier `cluster_bar` of either CTA of the pair
// (mapa_shared address), so the pair's leader can wait for both CTAs' tiles
// on one barrier armed with both CTAs' bytes.
DEV void tma_load_2d_pair(uint32_t dst, const CUtensorMap *m, uint32_t cluster_bar, int x,
                          int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes."
        "cta_group::2 [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(cluster_bar), "r"(x), "r"(y)
        : "memory");
}

// ------------------------------------------------------------ tcgen05
// G = 1: this CTA's tensor memory.  G = 2: the same columns in both CTAs of
// a cluster pair, for MMAs issued with cta_group::2; one warp of each CTA of
// the pair executes the allocation (and later the deallocation) together.
// A kernel uses one value of G for all of its tcgen05 instructions.
template <int G = 1>
DEV void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    if constexpr (G == 1)
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         dst_smem),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         dst_smem),
                     "r"(ncols)
                     : "memory");
}
template <int G = 1>
DEV void tmem_relinquish() {
    if constexpr (G == 1)
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    else
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
template <int G = 1>
DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    if constexpr (G == 1)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                     "r"(ncols)
                     : "memory");
    else
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr),
                     "r"(ncols)
                     : "memory");
}
DEV void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
DEV void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, both K-major, kind::f16 (bf16 inputs,
// fp32 accumulate).  Issued by one thread.
DEV void mma_bf16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                     uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (bf16 inputs, fp32
// accumulate).  A (M = 128 rows) lives in tensor memory: row i in lane i,
// two consecutive K elements per 32-bit column (the lower K index in the low
// half), so one K=16 step spans 8 columns starting at a_tmem.
DEV void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                     uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when all previously issued tcgen05.mma of this thread
// have completed.
DEV void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            bar)
        : "memory");
}

// Pair form (cta_group::2), issued by one thread of the pair's leading CTA:
// D (M = 256: rows 0..127 in the leader's tensor memory, 128..255 in the
// peer's, same columns) (+)= A * B^T, where each CTA holds its 128 rows of A
// and its half of B's N rows (the leader rows 0..N/2-1) at the same
// shared-memory offsets the descriptors give.
DEV void mma_bf16_ss_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on barrier `bar` (same offset) in every CTA of `cta_mask` when
// all pair MMAs issued so far by this thread have completed.
DEV void mma_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster."
        "b64 [%0], %1;" ::"r"(bar),
        "h"(cta_mask)
        : "memory");
}

// Instruction descriptor, kind::f16: D = f32, A = B = bf16, both K-major,
// dense, no negation; N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) |
           (uint32_t(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a K-major operand stored in the
// 128-byte-swizzle layout that a TMA tile load with SWIZZLE_128B writes:
// rows of 128 bytes (64 bf16 along K), 8-row core groups 1024 bytes apart
// (stride byte offset), tile base 1024-byte aligned.  Advancing along K
// inside the 128-byte row is done by adding the byte offset to `saddr`.
DEV uint64_t desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= uint64_t((saddr & 0x3FFFFu) >> 4);      // start address
    d |= uint64_t(1) << 16;                      // leading byte offset (unused)
    d |= uint64_t(1024 >> 4) << 32;              // stride byte offset
    d |= uint64_t(1) << 46;                      // descriptor version
    d |= uint64_t(2) << 61;                      // SWIZZLE_128B
    return d;
}

#define DS_R32(r)                                                                           \
    "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),     \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),         \
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),      \
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),      \
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),      \
        "=r"(r[31])
#define DS_W32(r)                                                                           \
    "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), \
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),  \
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]),            \
        "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),            \
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])

#define DS_RW32(r)                                                                          \
    "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),     \
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),         \
        "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),      \
        "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),      \
        "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),      \
        "+r"(r[31])

// Thread i of the warp reads TMEM lane (lane field of taddr) + i, 32
// consecutive 32-bit columns starting at the column field of taddr.  The
// registers are valid only after tmem_ld_wait(r), which names them so that
// no use can be scheduled before the wait.  Warp-collective: the whole warp
// must be converged.
DEV void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : DS_R32(r)
        : "r"(taddr)
        : "memory");
}
DEV void tmem_ld_wait(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;" : DS_RW32(r)::"memory");
}

// Write 32 consecutive 32-bit columns of this thread's TMEM lane, then wait
// for the store to complete (the source registers stay live until then).
DEV void tmem_st32_sync(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        DS_W32(r)
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" : DS_RW32(r)::"memory");
}

// Write 16 consecutive 32-bit columns of this thread's TMEM lane (no wait).
DEV void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
        "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
        "r"(r[14]), "r"(r[15])
        : "memory");
}
DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

DEV uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

DEV int warp_id() { return threadIdx.x >> 5; }
DEV int lane_id() { return threadIdx.x & 31; }

DEV bool elect_one_lane() { return lane_id() == 0; }

}  // namespace ds
