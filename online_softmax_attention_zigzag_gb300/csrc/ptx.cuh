// ptx.cuh -- inline-PTX wrappers for sm_103a: mbarrier, TMA bulk-tensor loads,
// tcgen05 (TMEM allocation, MMA, commit, TMEM load/store, fences) and bounded waits.
// Every wait here gives up after a time limit, records an error and lets the caller
// unwind; nothing traps.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace ra {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Abort state shared by the CTA: a flag in shared memory plus the library's device
// error word.  A wait that runs out raises both; every other wait polls the flag and
// unwinds too.
struct WaitCtl {
    volatile int* abort_flag;  // shared memory
    int* err;                  // device error record (may be null): status, set, barrier, where
    uint64_t timeout_ns;
};

constexpr int kErrTimeout = -5;  // RA_ERR_TIMEOUT

// Record the abort; the first wait to run out also records which barrier (its
// shared-memory address) and which thread of which CTA gave up.
__device__ __forceinline__ void raise_abort(const WaitCtl& w, uint64_t* bar) {
    *w.abort_flag = 1;
    if (w.err) {
        atomicExch(w.err, kErrTimeout);
        if (atomicCAS(w.err + 1, 0, 1) == 0) {
            w.err[2] = static_cast<int>(smem_u32(bar));
            w.err[3] = static_cast<int>((blockIdx.x << 10) | threadIdx.x);
        }
    }
}

// Wait until `bar` completes the phase with parity `parity`; false on abort/timeout.
// The abort flag and the clock are checked every 64 polls only, to keep the loop short;
// sleep_ns > 0 backs off between polls (for waiters that are not latency-critical).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtl& w,
                                          uint32_t sleep_ns = 0) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (sleep_ns) __nanosleep(sleep_ns);
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0u) {
            if (*w.abort_flag) return false;
            if (globaltimer_ns() - t0 > w.timeout_ns) {
                raise_abort(w, bar);
                return false;
            }
        }
    }
}

// As mbar_wait, but gives up only when its own time limit runs out, not when another role
// has raised the abort flag (it still raises the flag itself).  For the roles that feed a
// named barrier: they keep arriving for every tile whose gating MMA was issued, so that a
// waiter on that barrier is never left without its arrival.  The host never sets a limit
// below 1 s, far above the time a queued MMA takes to complete.
__device__ __forceinline__ bool mbar_wait_noabort(uint64_t* bar, uint32_t parity, const WaitCtl& w) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0u && globaltimer_ns() - t0 > w.timeout_ns) {
            raise_abort(w, bar);
            return false;
        }
    }
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for two barrier phases at once: both are polled with non-blocking reads issued back
// to back, so that when both have already completed the check costs one shared-memory round
// trip instead of two; false on abort/timeout.  Every lane of the warp takes part.
__device__ __forceinline__ bool mbar_wait2_w(uint64_t* a, uint32_t pa, uint64_t* b, uint32_t pb, const WaitCtl& w) {
    bool da = false, db = false;
    uint64_t t0 = 0;
    for (uint32_t i = 0;; ++i) {
        const bool ra = da || mbar_test_wait(a, pa);
        const bool rb = db || mbar_test_wait(b, pb);
        da = ra;
        db = rb;
        if (__all_sync(0xffffffffu, ra && rb)) return true;
        if (i == 0) t0 = globaltimer_ns();
        if ((i & 63u) == 63u) {
            if (*w.abort_flag) return false;
            if (globaltimer_ns() - t0 > w.timeout_ns) {
                raise_abort(w, da ? b : a);
                return false;
            }
        }
    }
}

// Bounded wait that ignores the abort flag (used to drain in-flight work on abort).
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > timeout_ns) return;
    }
}

// Named barrier `id` over `nthreads` threads (a multiple of 32); returns the AND of every
// participating thread's `ok`, so that a failed wait reaches the whole group.
__device__ __forceinline__ bool named_bar_and(int id, int nthreads, bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.and.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(ok ? 1u : 0u), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// Hardware named barrier `id` over `nthreads` threads: arrive without waiting / arrive and
// wait for the rest.
__device__ __forceinline__ void named_bar_arrive(int id, int nthreads) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Wait on an mbarrier phase with every lane of the warp; the verdict is the warp's.
__device__ __forceinline__ bool mbar_wait_w(uint64_t* bar, uint32_t parity, const WaitCtl& wc) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, wc));
}

// Dynamic work items of the persistent kernels.  A launch owns two counters in global
// memory (zero at launch): the next item index and the number of CTAs done.  In each CTA
// one loader thread draws indices and hands them to the other roles through a ring of
// kItemRing slots in shared memory, guarded by `full` (count 1) and `empty` (count = the
// number of takers) mbarriers.
constexpr int kItemRing = 4;

// Loader: draw entry k of the CTA's item sequence and publish it (-1 past the last item);
// -2 on abort.
__device__ __forceinline__ int publish_item(unsigned int* counter, int n_items, uint64_t* full, uint64_t* empty,
                                            volatile int* ring, uint32_t k, const WaitCtl& wc) {
    const uint32_t slot = k % kItemRing;
    if (!mbar_wait(&empty[slot], ((k / kItemRing) & 1u) ^ 1u, wc, 32)) return -2;
    int item = static_cast<int>(atomicAdd(counter, 1u));
    if (item >= n_items) item = -1;
    ring[slot] = item;
    mbar_arrive(&full[slot]);
    return item;
}

// Taker: entry k as the loader published it (an item index, -1 at the end), -2 on abort.
// Every taker takes every entry, in order; one arrival per taker (`leader`: one lane of
// a warp, or a lone issuing thread) frees the slot.
__device__ __forceinline__ int take_item(uint64_t* full, uint64_t* empty, const volatile int* ring, uint32_t k,
                                         bool leader, const WaitCtl& wc, bool honour_abort = true) {
    const uint32_t slot = k % kItemRing;
    const uint32_t par = (k / kItemRing) & 1u;
    if (!(honour_abort ? mbar_wait(&full[slot], par, wc) : mbar_wait_noabort(&full[slot], par, wc))) return -2;
    const int item = ring[slot];
    __syncwarp(__activemask());
    if (leader) mbar_arrive(&empty[slot]);
    return item;
}

// End of a launch: the last CTA to finish zeroes the counters for the next launch that
// uses them.  Called by one thread per CTA after every role is done.
__device__ __forceinline__ void finish_items(unsigned int* counter) {
    __threadfence();
    if (atomicAdd(counter + 1, 1u) == gridDim.x - 1) {
        counter[0] = 0u;
        counter[1] = 0u;
        __threadfence();
    }
}

// ------------------------------------------------------------------ TMA
// 2-D tiled TMA load of box (x, y) that completes its bytes on `bar`, with an L2 cache
// policy (from make_policy_*) attached to the loaded lines.
__device__ __forceinline__ void tma_load_2d_hint(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int x,
                                                 int y, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
// L2 policies: keep lines that many CTAs re-read (K, V); let streamed lines (Q, out) go first.
__device__ __forceinline__ uint64_t make_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t make_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void st_stream_f4(float4* dst, float4 v, uint64_t policy) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(dst),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "l"(policy)
                 : "memory");
}
// 32-byte streaming store (dst 32-byte aligned)
__device__ __forceinline__ void st_stream_f8(float* dst, const float (&v)[8], uint64_t policy) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(
                     dst),
                 "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]), "l"(policy)
                 : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// tcgen05 issue for issuers that run as a whole warp (descriptors and counters stay
// warp-uniform): one elected lane issues the instruction; every lane must take part.  The
// elected lane is the same for every call with the full mask, so a commit tracks the MMAs
// issued before it.
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void mma_ss_e(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc], A read from tensor memory.
__device__ __forceinline__ void mma_ts_e(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when every tcgen05 operation the elected lane issued so far is done.
__device__ __forceinline__ void mma_commit_e(uint64_t* bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A K-major,
// B K-major (b_mn_major = 0) or MN-major (1), shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int b_mn_major) {
    return (1u << 4)                                  // D format: f32
           | (1u << 7)                                // A format: bf16
           | (1u << 10)                               // B format: bf16
           | (static_cast<uint32_t>(b_mn_major) << 16)  // B major-ness
           | (static_cast<uint32_t>(N >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);   // M / 16
}

// desc + off computed where it is used: an opaque add keeps the compiler from hoisting
// every (descriptor, K-slice) pair out of the loops into registers.
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t off16) {
    uint64_t r;
    asm volatile("add.s64 %0, %1, %2;" : "=l"(r) : "l"(desc), "l"(static_cast<uint64_t>(off16)));
    return r;
}

// Shared-memory matrix descriptor with 128-byte swizzle.
// lbo/sbo are byte offsets: for K-major operands sbo is the distance between
// consecutive 8-row groups (1024 B for 128-byte rows) and lbo is unused; for
// MN-major operands lbo is the distance between 64-element column blocks and sbo
// the distance between 8-row groups along K.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((smem_addr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
    d |= static_cast<uint64_t>(2) << 61;  // swizzle: 128 B
    return d;
}

// 32 lanes x 32 columns of 32-bit TMEM words: thread t of the warp gets lane
// (base lane + t), columns [col, col+32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
// As tmem_ld32, and `mx` receives the largest of the 32 fp32 values this thread loads
// (tcgen05.ld.red, sm_103a).
__device__ __forceinline__ void tmem_ld32_max(uint32_t taddr, uint32_t (&r)[32], float& mx) {
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
          "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31]), "=f"(mx)
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
// 32 lanes x 16 columns: thread t writes lane (base lane + t), columns [col, col+16).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------ math
// 2^x with the hardware approximation (MUFU.EX2), flush-to-zero; 2^-inf = +0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pair arithmetic of sm_100+ (one instruction for two lanes of work).
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0,
                                      float c1) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\tfma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void fmul2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
    asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// acc += lo + hi of a packed bf16 pair, each half added exactly into fp32
__device__ __forceinline__ void add_bf16x2_f32(float& acc0, float& acc1, uint32_t pk) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\tadd.rn.f32.bf16 %0, lo, %0;\n\t"
        "add.rn.f32.bf16 %1, hi, %1;\n\t}"
        : "+f"(acc0), "+f"(acc1)
        : "r"(pk));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace ra
