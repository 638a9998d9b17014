// attn_bwd.cu -- backward pass of the fused ring attention on tcgen05 tensor cores.
//
// The pages give the forward only (the training FLOP count of "Interrogating
// parallelism, part 5" covers a backward pass but does not describe it); this is the
// exact gradient of that forward.  With P_ij = exp(q_i . k_j - lse_i) over visible keys,
// D_i = dout_i . out_i and dS_ij = P_ij (dout_i . v_j - D_i):
//     dV_j = sum_i P_ij dout_i,   dK_j = sum_i dS_ij q_i,   dQ_i = sum_j dS_ij k_j,
// a KV head summing over the query heads that use it.  In the dq kernel a query tile meets
// the KV blocks hop by hop in ring order, as in the forward.  In the dk/dv kernel a key
// tile meets the query tiles from the end of the sequence down, every query head of its
// group at each position, which keeps the Q and dO tiles the CTAs read at one time in L2
// (see for_each_query_tile).  Only the order of the fp32 sums depends on either order.
//
// Three kernels, all on the caller's stream:
//   * bwd_delta_kernel   D_i = dout_i . out_i, one warp per row (HBM-bound);
//   * bwd_kernel<D, true>   (dq) one 128-row query tile per work item: per key tile
//                        S = Q K^T and dP = dO V^T into TMEM, then dS (bf16) into TMEM,
//                        then dQ += dS K with dS read from TMEM;
//   * bwd_kernel<D, false>  (dk/dv) one 128-row key tile per work item: per query tile
//                        S^T = K Q^T and dP^T = V dO^T, then P^T and dS^T (bf16) into
//                        TMEM, then dV += P^T dO and dK += dS^T Q.
// Splitting dq from dk/dv recomputes S and dP once more (7 tile products instead of 5)
// but needs no atomics and gives a deterministic result.
//
// Each CTA is persistent and draws its work items (query tiles for dq, key tiles for
// dk/dv, listed by KV head and decreasing work) from a counter in global memory as it
// finishes the previous one; its loader hands the index to the other roles through a ring
// in shared memory.  (Dealing the 2048 key tiles of the 32k GQA dk/dv launch out
// statically in snake order left the CTAs ~20% apart.)  Warps 0-7 compute (warpgroup h
// handles columns [64h, 64h+64) of the 128 x 128 tile product, thread = TMEM lane = row),
// warp 8 issues the MMAs (the whole warp runs the issuer so that its descriptors stay
// warp-uniform; one elected lane issues each instruction), warp 9 the TMA loads (one
// thread).  In the dq kernel
// warp 8 issues S and dP only and warp 10 issues dQ += dS K, so that neither issuer's waits
// hold up the other's products; a K ring slot is then released by both, and a dS buffer is
// handed back by warp 10 once its dQ product is done.  The compute warps copy S (S^T) and dP
// (dP^T) from TMEM into registers and release those columns at once, so the next tile's
// products run on the tensor cores while this tile's exponentials are computed; the
// streamed operands move through separate shared-memory rings (three slots for the one
// the next tile's first product needs, two for the other).  Every operand form used here
// (both operands K-major from shared memory; A from TMEM with an MN-major B) is one the
// forward kernel uses too.
//   dq TMEM:    S [0,128), dP [128,256), dQ [256, 256+D), dS in [384 + 64b, +64), b = j%2.
//   dk/dv TMEM: S^T [0,128), dP^T [128,256), dV [256,384), dK [384,512); warpgroup h puts
//               P^T in [128+64h, +32) and dS^T in [128+64h+32, +32) over its own dP^T.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ra {
namespace {

constexpr int kTile = 128;
constexpr int kThreads = 352;
// warp 8: MMA issuer (dQ kernel: S and dP products); warp 9: TMA loads; warp 10: the dQ
// kernel's second issuer (dQ += dS K)
constexpr int kMmaWarp = 8, kLoadWarp = 9, kMma2Warp = 10;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 256;
constexpr uint32_t kItemTakers = 10;  // work-item takers: 2 MMA issuer warps + 8 compute warps

// Shared memory of both kernels: two resident tiles (Q, dO or K, V), then ring A (three
// slots: K for dq, Q for dk/dv) and ring B (two slots: V for dq, dO for dk/dv).
template <int D>
struct BwdCfg {
    static constexpr int kTileBytes = kTile * D * 2;  // one 128 x D bf16 tile
    static constexpr int kBoxBytes = kTile * 64 * 2;  // one 128-row, 64-column block
    static constexpr int kSlotsA = 3, kSlotsB = 2;
    static constexpr int kAOff = 2 * kTileBytes;
    static constexpr int kBOff = kAOff + kSlotsA * kTileBytes;
    static constexpr int kBarOff = kBOff + kSlotsB * kTileBytes;
    static constexpr int kNumBars = 40;
    static constexpr int kRingOff = kBarOff + kNumBars * 8 + 16;  // item ids, loader -> other roles
    static constexpr int kSmem = kRingOff + 16 + 1024;  // + slack to align the base
};

// Rank-major (or natural) row of natural position pos of head `head`.
__device__ __forceinline__ int row_of(const AttnBwdParams& p, int head, int pos) {
    const Ring& R = p.ring;
    if (p.natural) return head * R.S + pos;
    const int k = pos / R.m;
    const bool second = R.layout == 1 && k >= R.c;
    const int s = second ? 2 * R.c - 1 - k : k;
    return head * R.S + s * R.n_r + (second ? R.m : 0) + (pos - k * R.m);
}

// A 128-row tile of a [heads * S, d] tensor starting at `row` (check build: a row outside the
// tensor is recorded and replaced by row 0).
__device__ __forceinline__ int checked_tile_row(int row, int heads, const Ring& R, int* err, int site) {
    if (!RA_CHECKED(row >= 0 && static_cast<long long>(row) + kTile <= static_cast<long long>(heads) * R.S, err, site))
        return 0;
    return row;
}

__device__ __forceinline__ int rank_of(const Ring& R, int pos) {
    const int k = pos / R.m;
    return (R.layout == 1 && k >= R.c) ? 2 * R.c - 1 - k : k;
}

// dq work item: query head hq, natural position qp of the tile.  Items are KV-head-major
// and, within a KV head, by decreasing causal work (last tiles first).
__device__ __forceinline__ void dq_item(const AttnBwdParams& p, int item, int& hq, int& qp) {
    const Ring& R = p.ring;
    const int per_kv = R.g * p.n_tiles;
    const int hk = item / per_kv;
    const int rem = item - hk * per_kv;
    const int ti = rem / R.g;
    hq = hk * R.g + (rem - ti * R.g);
    qp = (R.causal ? p.n_tiles - 1 - ti : ti) * kTile;
}

// dk/dv work item: KV head hk, natural position kp of the key tile (first tiles carry
// the most causal work, so ascending position is decreasing work).
__device__ __forceinline__ void kv_item(const AttnBwdParams& p, int item, int& hk, int& kp) {
    hk = item / p.n_tiles;
    kp = (item - hk * p.n_tiles) * kTile;
}

// Key tiles a query tile at qp meets, in ring order: hop h brings rank (r - h) mod c's
// block; under the causal mask tiles wholly after the query tile are skipped.
template <class F>
__device__ __forceinline__ void for_each_key_tile(const Ring& R, int qp, F&& f) {
    const int r = rank_of(R, qp);
    for (int hop = 0; hop < R.c; ++hop) {
        const int s = (r - hop + R.c) % R.c;
        for (int slot = 0; slot < R.nslot; ++slot) {
            const int base = (slot ? 2 * R.c - 1 - s : s) * R.m;
            for (int t0 = base; t0 < base + R.m; t0 += kTile) {
                if (R.causal && t0 > qp) break;
                if (!f(t0)) return;
            }
        }
    }
}

__device__ __forceinline__ int count_key_tiles(const Ring& R, int qp) {
    int n = 0;
    for_each_key_tile(R, qp, [&](int) { ++n; return true; });
    return n;
}

// Query tiles the key tile at kp meets, every query head of the KV group for each tile
// position, positions in descending natural order (down to kp under the causal mask).
// Every CTA of a launch starts its item at the end of the sequence and moves down at the
// same rate (a position costs the same for every key tile), so the CTAs read the same Q
// and dO tiles at about the same time and each tile comes from DRAM about once; the
// ring's order (hop h meets rank (s + h) mod c, each CTA starting at its own rank) had
// every CTA in a different part of the 8 heads' Q and dO and read them ~9 times over.
// Only the order of the fp32 sums into dK, dV depends on it.
template <class F>
__device__ __forceinline__ void for_each_query_tile(const Ring& R, int hk, int kp, F&& f) {
    const int lo = R.causal ? kp : 0;
    for (int t0 = R.S - kTile; t0 >= lo; t0 -= kTile)
        for (int x = 0; x < R.g; ++x)
            if (!f(hk * R.g + x, t0)) return;
}

// The query tile for_each_query_tile visits after (hq, t0) for the key tile at kp;
// false when (hq, t0) is the last.
__device__ __forceinline__ bool next_query_tile(const Ring& R, int hk, int kp, int hq, int t0, int& nhq, int& nt0) {
    nhq = hq + 1;
    nt0 = t0;
    if (nhq == (hk + 1) * R.g) {
        nhq = hk * R.g;
        nt0 = t0 - kTile;
    }
    return nt0 >= (R.causal ? kp : 0);
}

__device__ __forceinline__ int count_query_tiles(const Ring& R, int hk, int kp) {
    (void)hk;
    return ((R.S - (R.causal ? kp : 0)) / kTile) * R.g;
}

// Named barrier over one compute warpgroup (128 threads); returns the AND of `ok`.
__device__ __forceinline__ bool group_bar_and(int h, bool ok) { return named_bar_and(1 + h, 128, ok); }
// dK/dV kernel: P^T and dS^T handed to the MMA warp on named barriers 3 and 4 (the eight
// compute warps arrive, the MMA warp syncs)
constexpr int kPtBar = 3, kDsBar = 4, kHandThreads = 8 * 32 + 32;

// D[tmem] = A B^T with A (128 x D) and B (128 x D) both K-major in shared memory (128-byte
// swizzle, 64-column boxes): the 128 x 128 tile products S, dP, S^T, dP^T.
template <int D>
__device__ __forceinline__ void issue_kk(uint32_t d_tmem, uint32_t a_base, uint32_t b_base) {
    using C = BwdCfg<D>;
    constexpr uint32_t idesc = idesc_bf16(kTile, kTile, 0);
    const uint64_t ad = sdesc_sw128(a_base, 16, 1024);
    const uint64_t bd = sdesc_sw128(b_base, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk / 4) * C::kBoxBytes + (kk % 4) * 32) >> 4;
        mma_ss_e(d_tmem, desc_add(ad, off), desc_add(bd, off), idesc, kk > 0 ? 1u : 0u);
    }
}

// D[tmem] (+)= A B: A (128 x 128, bf16 packed in TMEM: columns [64h, 64h+64) of the
// product in TMEM columns a_tmem + h * a_half + [0, 32)), B (128 x D) from shared memory
// as an MN-major operand (the tile's rows are the contraction index).
template <int D>
__device__ __forceinline__ void issue_tm(uint32_t d_tmem, uint32_t a_tmem, uint32_t a_half, uint32_t b_base,
                                         bool accumulate) {
    using C = BwdCfg<D>;
    constexpr uint32_t idesc = idesc_bf16(kTile, D, 1);
    const uint64_t bd = sdesc_sw128(b_base, C::kBoxBytes, 1024);
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk) {
        const uint32_t acol = (kk / 4) * a_half + (kk % 4) * 8;
        mma_ts_e(d_tmem, a_tmem + acol, desc_add(bd, (kk * 16 * 128) >> 4), idesc,
                 (accumulate || kk > 0) ? 1u : 0u);
    }
}

// Load a 128 x D bf16 tile (rows row..row+127) as 64 x 64 boxes: 64-column block cb,
// 64-row block rb at byte cb * 16384 + rb * 8192, the layout of one 128-byte-swizzled
// K-major operand of 128 rows.
template <int D>
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int row,
                                          uint64_t policy) {
#pragma unroll
    for (int cb = 0; cb < D / 64; ++cb)
#pragma unroll
        for (int rb = 0; rb < 2; ++rb)
            tma_load_2d_hint(dst + cb * 16384 + rb * 8192, map, bar, cb * 64, row + rb * 64, policy);
}

// 64 fp32 TMEM columns of this thread's lane, in two 32-column loads.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
    uint32_t r0[32], r1[32];
    tmem_ld32(taddr, r0);
    tmem_ld32(taddr + 32, r1);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        v[i] = __uint_as_float(r0[i]);
        v[32 + i] = __uint_as_float(r1[i]);
    }
}

// Write `cols` fp32 accumulator columns of this lane to global memory (row-contiguous).
template <int COLS>
__device__ __forceinline__ void store_acc(uint32_t taddr, float* dst) {
#pragma unroll
    for (int cc = 0; cc < COLS; cc += 32) {
        uint32_t r[32];
        tmem_ld32(taddr + cc, r);
        tmem_wait_ld();
        float4* d4 = reinterpret_cast<float4*>(dst + cc);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            d4[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
    }
}

// Barriers shared by both kernels' layouts (slot rings A: 3, B: 2).
struct Bars {
    uint64_t *res_full, *res_empty;  // resident tiles landed / item's MMAs done with them
    uint64_t *s_full, *dp_full;      // S (S^T) / dP (dP^T) in TMEM
    uint64_t *s_free, *dp_free;      // 256 compute threads copied S / dP out of TMEM
    uint64_t *ds_full;               // [2] dq: dS buffer written (the dk/dv kernel hands dS^T
                                     //     and P^T over on named barriers kDsBar and kPtBar)
    uint64_t *pt_full;               // the same barrier as ds_full[1]; unused by the dk/dv kernel
    uint64_t *acc_done, *acc_free, *drain, *drain2;
    uint64_t *ds_free;  // [2] dQ kernel: the dQ product that read dS buffer b is done
    uint64_t *a_full, *a_empty, *b_full, *b_empty;
    uint64_t *item_full, *item_empty;  // [kItemRing] each: item ids handed from the loader
    __device__ explicit Bars(uint64_t* b)
        : res_full(b), res_empty(b + 1), s_full(b + 2), dp_full(b + 3), s_free(b + 4), dp_free(b + 5),
          ds_full(b + 6), pt_full(b + 7), acc_done(b + 8), acc_free(b + 9), drain(b + 10), drain2(b + 11), ds_free(b + 12), a_full(b + 16), a_empty(b + 19),
          b_full(b + 22), b_empty(b + 24), item_full(b + 26), item_empty(b + 30) {}
};

__device__ __forceinline__ void init_bars(const Bars& b, uint32_t a_releases) {
    mbar_init(b.res_full, 1);
    mbar_init(b.res_empty, 1);
    mbar_init(b.s_full, 1);
    mbar_init(b.dp_full, 1);
    mbar_init(b.s_free, 256);
    mbar_init(b.dp_free, 256);
    mbar_init(&b.ds_full[0], 256);
    mbar_init(&b.ds_full[1], 256);
    mbar_init(b.acc_done, 1);
    mbar_init(b.acc_free, 256);
    mbar_init(b.drain, 1);
    mbar_init(b.drain2, 1);
    mbar_init(&b.ds_free[0], 1);
    mbar_init(&b.ds_free[1], 1);
    for (int s = 0; s < 3; ++s) {
        mbar_init(&b.a_full[s], 1);
        mbar_init(&b.a_empty[s], a_releases);
    }
    for (int s = 0; s < 2; ++s) {
        mbar_init(&b.b_full[s], 1);
        mbar_init(&b.b_empty[s], 1);
    }
    for (int s = 0; s < kItemRing; ++s) {
        mbar_init(&b.item_full[s], 1);
        mbar_init(&b.item_empty[s], kItemTakers);
    }
}

// Wait (one poller warp per warpgroup, the rest in the group's named barrier).
__device__ __forceinline__ bool group_wait(uint64_t* bar, uint32_t parity, int h, int wq, const WaitCtl& wc,
                                           bool honour_abort = true) {
    bool ok = true;
    if (wq == 0)
        ok = __all_sync(0xffffffffu, honour_abort ? mbar_wait(bar, parity, wc) : mbar_wait_noabort(bar, parity, wc));
    return group_bar_and(h, ok);
}

// Wait with every lane of the warp polling (no named barrier).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& wc) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, wc));
}

// Copy 64 fp32 TMEM columns of this lane into registers, then release them.
__device__ __forceinline__ void tmem_take64(uint32_t taddr, float (&v)[64], uint64_t* free_bar) {
    tmem_ld64(taddr, v);
    tc_fence_before();
    mbar_arrive(free_bar);
}

// Loader helper: wait for slot `i % n` of a ring to be empty and load one tile into it.
template <int D>
__device__ __forceinline__ bool ring_load(uint8_t* ring, uint64_t* full, uint64_t* empty, uint32_t i, int n,
                                          const CUtensorMap* map, int row, uint64_t policy, const WaitCtl& wc) {
    using C = BwdCfg<D>;
    const uint32_t s = i % n;
    if (!mbar_wait(&empty[s], ((i / n) & 1u) ^ 1u, wc, 32)) return false;
    mbar_arrive_expect_tx(&full[s], C::kTileBytes);
    load_tile<D>(ring + s * C::kTileBytes, map, &full[s], row, policy);
    return true;
}

__device__ __forceinline__ bool ring_wait_w(uint64_t* full, uint32_t i, int n, const WaitCtl& wc) {
    return mbar_wait_w(&full[i % n], (i / n) & 1u, wc);
}

// Let every copy issued into a ring land before the CTA's shared memory goes away.
__device__ __forceinline__ void ring_drain(uint64_t* full, uint32_t issued, int n, uint64_t timeout_ns) {
    for (uint32_t s = 0; s < (uint32_t)n && s < issued; ++s) {
        const uint32_t last = issued - 1 - ((issued - 1 - s) % n);
        drain_wait(&full[s], (last / n) & 1u, timeout_ns);
    }
}

// ------------------------------------------------------------------ dq kernel
template <int D>
__device__ void dq_load(const AttnBwdParams& p, const CUtensorMap* tq, const CUtensorMap* tdo,
                        const CUtensorMap* tk, const CUtensorMap* tv, uint8_t* smem, const Bars& b,
                        volatile int* ring, const WaitCtl& wc) {
    using C = BwdCfg<D>;
    const Ring& R = p.ring;
    const uint64_t keep = make_policy_evict_last(), stream = make_policy_evict_first();
    uint32_t ka = 0, vb = 0, qit = 0;
    bool ok = true;
    for (uint32_t n_it = 0; ok; ++n_it) {
        const int item = publish_item(p.sched, p.n_items, b.item_full, b.item_empty, ring, n_it, wc);
        if (item == -2) { ok = false; break; }
        if (item < 0) break;
        int hq, qp;
        dq_item(p, item, hq, qp);
        if (!mbar_wait(b.res_empty, (qit & 1u) ^ 1u, wc, 32)) { ok = false; break; }
        ++qit;
        mbar_arrive_expect_tx(b.res_full, 2 * C::kTileBytes);
        const int qrow = checked_tile_row(row_of(p, hq, qp), R.Hq, R, p.err, kSiteBwdQRow);
        load_tile<D>(smem, tq, b.res_full, qrow, stream);
        load_tile<D>(smem + C::kTileBytes, tdo, b.res_full, qrow, stream);
        const int hk = hq / R.g;
        for_each_key_tile(R, qp, [&](int t0) -> bool {
            const int krow = checked_tile_row(row_of(p, hk, t0), R.Hkv, R, p.err, kSiteBwdKvRow);
            if (!ring_load<D>(smem + C::kAOff, b.a_full, b.a_empty, ka, C::kSlotsA, tk, krow, keep, wc) ||
                !ring_load<D>(smem + C::kBOff, b.b_full, b.b_empty, vb, C::kSlotsB, tv, krow, keep, wc)) {
                ok = false;
                return false;
            }
            ++ka;
            ++vb;
            return true;
        });
    }
    if (!ok) {
        ring_drain(b.a_full, ka, C::kSlotsA, wc.timeout_ns);
        ring_drain(b.b_full, vb, C::kSlotsB, wc.timeout_ns);
        if (qit > 0) drain_wait(b.res_full, (qit - 1) & 1u, wc.timeout_ns);
    }
}

// dQ kernel, first issuer: S = Q K^T and dP = dO V^T, each as soon as the compute warps
// have copied the previous tile's out of TMEM.
template <int D>
__device__ void dq_mma(const AttnBwdParams& p, uint8_t* smem, const Bars& b, uint32_t tmem, volatile int* ring, const WaitCtl& wc) {
    using C = BwdCfg<D>;
    const Ring& R = p.ring;
    const uint32_t sQ = smem_u32(smem), sdO = sQ + C::kTileBytes;
    const uint32_t sA = sQ + C::kAOff, sB = sQ + C::kBOff;
    uint32_t idx = 0, qit = 0, sf = 0, dpf = 0;
    bool ok = true;
    for (uint32_t n_it = 0; ok; ++n_it) {
        const int item = take_item(b.item_full, b.item_empty, ring, n_it, (threadIdx.x & 31) == 0, wc);
        if (item == -2) { ok = false; break; }
        if (item < 0) break;
        int hq, qp;
        dq_item(p, item, hq, qp);
        const int nj = count_key_tiles(R, qp);
        const uint32_t i0 = idx;
        if (!mbar_wait_w(b.res_full, qit & 1u, wc)) { ok = false; break; }
        // S(0), dP(0)
        if (!ring_wait_w(b.a_full, i0, C::kSlotsA, wc)) { ok = false; break; }
        tc_fence_after();
        issue_kk<D>(tmem, sQ, sA + (i0 % C::kSlotsA) * C::kTileBytes);
        mma_commit_e(b.s_full);
        mma_commit_e(&b.a_empty[i0 % C::kSlotsA]);  // this issuer is done with K(0)
        if (!ring_wait_w(b.b_full, i0, C::kSlotsB, wc)) { ok = false; break; }
        tc_fence_after();
        issue_kk<D>(tmem + kTile, sdO, sB + (i0 % C::kSlotsB) * C::kTileBytes);
        mma_commit_e(b.dp_full);
        mma_commit_e(&b.b_empty[i0 % C::kSlotsB]);  // V(0) is done once dP(0) is
        for (int j = 0; j + 1 < nj && ok; ++j) {
            const uint32_t i = i0 + j;
            // the next S as soon as this tile's S is out of TMEM and K(j+1) has landed,
            // likewise dP with V(j+1); each pair is checked at once (both are usually complete
            // already, and each check is a shared-memory read behind the tensor core's)
            const uint32_t na = i + 1;
            if (!mbar_wait2_w(b.s_free, sf & 1u, &b.a_full[na % C::kSlotsA], (na / C::kSlotsA) & 1u, wc)) {
                ok = false;
                break;
            }
            ++sf;
            tc_fence_after();
            issue_kk<D>(tmem, sQ, sA + ((i + 1) % C::kSlotsA) * C::kTileBytes);
            mma_commit_e(b.s_full);
            mma_commit_e(&b.a_empty[(i + 1) % C::kSlotsA]);
            if (!mbar_wait2_w(b.dp_free, dpf & 1u, &b.b_full[na % C::kSlotsB], (na / C::kSlotsB) & 1u, wc)) {
                ok = false;
                break;
            }
            ++dpf;
            tc_fence_after();
            issue_kk<D>(tmem + kTile, sdO, sB + ((i + 1) % C::kSlotsB) * C::kTileBytes);
            mma_commit_e(b.dp_full);
            mma_commit_e(&b.b_empty[(i + 1) % C::kSlotsB]);
        }
        if (!ok) break;
        // the last tile's S and dP still have to be copied out before the next item's
        if (!mbar_wait_w(b.s_free, sf & 1u, wc) || !mbar_wait_w(b.dp_free, dpf & 1u, wc)) { ok = false; break; }
        ++sf;
        ++dpf;
        idx = i0 + nj;
        mma_commit_e(b.res_empty);  // Q and dO of this item are done with
        ++qit;
    }
    if (!ok) {
        // every MMA issued so far must finish before TMEM is released
        mma_commit_e(b.drain);
        drain_wait(b.drain, 0, wc.timeout_ns);
    }
}

// dQ kernel, second issuer: dQ += dS K for every key tile, as the compute warps hand dS over.
template <int D>
__device__ void dq_mma2(const AttnBwdParams& p, uint8_t* smem, const Bars& b, uint32_t tmem, volatile int* ring,
                        const WaitCtl& wc) {
    using C = BwdCfg<D>;
    const Ring& R = p.ring;
    const uint32_t sA = smem_u32(smem) + C::kAOff;
    uint32_t idx = 0, it = 0, dsit[2] = {0, 0};
    bool ok = true;
    for (uint32_t n_it = 0; ok; ++n_it) {
        const int item = take_item(b.item_full, b.item_empty, ring, n_it, (threadIdx.x & 31) == 0, wc);
        if (item == -2) { ok = false; break; }
        if (item < 0) break;
        int hq, qp;
        dq_item(p, item, hq, qp);
        const int nj = count_key_tiles(R, qp);
        for (int j = 0; j < nj && ok; ++j) {
            const uint32_t i = idx + j;
            const int bb = j & 1;
            if (!mbar_wait_w(&b.ds_full[bb], dsit[bb] & 1u, wc)) { ok = false; break; }
            ++dsit[bb];
            if (j == 0 && !mbar_wait_w(b.acc_free, (it & 1u) ^ 1u, wc)) { ok = false; break; }
            // K(j) landed before the S(j) that led to this dS; its slot cannot have been
            // refilled, since this issuer has not released it yet
            if (!ring_wait_w(b.a_full, i, C::kSlotsA, wc)) { ok = false; break; }
            tc_fence_after();
            // dQ += dS K, dS from TMEM buffer j % 2, K from its ring slot as an MN-major B
            issue_tm<D>(tmem + kAccCol, tmem + 384 + 64 * bb, 32, sA + (i % C::kSlotsA) * C::kTileBytes, j > 0);
            mma_commit_e(&b.a_empty[i % C::kSlotsA]);
            mma_commit_e(&b.ds_free[bb]);
        }
        if (!ok) break;
        idx += nj;
        mma_commit_e(b.acc_done);
        ++it;
    }
    if (!ok) {
        mma_commit_e(b.drain2);
        drain_wait(b.drain2, 0, wc.timeout_ns);
    }
}

template <int D>
__device__ void dq_compute(const AttnBwdParams& p, const Bars& b, uint32_t tmem, volatile int* ring, const WaitCtl& wc) {
    const Ring& R = p.ring;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int h = warp / 4, wq = warp % 4;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_tm = tmem + lane_off + h * 64;           // my 64 key columns of S
    const uint32_t dp_tm = tmem + lane_off + kTile + h * 64;  // and of dP
    const uint32_t acc_tm = tmem + lane_off + kAccCol + h * (D / 2);
    uint32_t sf = 0, dpf = 0, it = 0, dsf[2] = {0, 0};
    bool ok = true;
    for (uint32_t n_it = 0; ok; ++n_it) {
        const int item = take_item(b.item_full, b.item_empty, ring, n_it, lane == 0, wc);
        if (item == -2) { ok = false; break; }
        if (item < 0) break;
        int hq, qp;
        dq_item(p, item, hq, qp);
        const int grow = row_of(p, hq, qp) + row;
        const bool row_ok = RA_CHECKED(grow >= 0 && grow < R.Hq * R.S, p.err, kSiteBwdLseRow);
        const float nl = row_ok ? -__ldg(p.lse + grow) * kLog2e : 0.f;
        const float dl = row_ok ? __ldg(p.delta + grow) : 0.f;
        const int qpos = qp + row;
        uint32_t jj = 0;  // tile within the item
        for_each_key_tile(R, qp, [&](int t0) -> bool {
            if (!warp_wait(b.s_full, sf & 1u, wc)) { ok = false; return false; }
            ++sf;
            tc_fence_after();
            float x[64];
            tmem_take64(s_tm, x, b.s_free);
            const int lim = qpos - (t0 + h * 64);  // my keys [0, lim] are visible
            // only tiles on the diagonal mask; branch on the warp, not per element
            if (__any_sync(0xffffffffu, R.causal && lim < 63)) {
                const int lm = R.causal ? lim : 63;
#pragma unroll
                for (int i = 0; i < 64; i += 2) {
                    float p0, p1;
                    ffma2(p0, p1, x[i], x[i + 1], kLog2e, kLog2e, nl, nl);
                    x[i] = (i > lm) ? 0.f : ex2(p0);
                    x[i + 1] = (i + 1 > lm) ? 0.f : ex2(p1);
                }
            } else {
#pragma unroll
                for (int i = 0; i < 64; i += 2) {
                    float p0, p1;
                    ffma2(p0, p1, x[i], x[i + 1], kLog2e, kLog2e, nl, nl);
                    x[i] = ex2(p0);
                    x[i + 1] = ex2(p1);
                }
            }
            if (!warp_wait(b.dp_full, dpf & 1u, wc)) { ok = false; return false; }
            ++dpf;
            tc_fence_after();
            float dp[64];
            tmem_take64(dp_tm, dp, b.dp_free);
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                float a0, a1;
                fadd2(a0, a1, dp[2 * i], dp[2 * i + 1], -dl, -dl);  // dP - D
                fmul2(a0, a1, a0, a1, x[2 * i], x[2 * i + 1]);     // P (dP - D)
                pk[i] = pack_bf16x2(a0, a1);
            }
            const int bb = jj & 1;  // dS buffer, as the MMA issuer counts it
            // the dQ product of two tiles ago, issued by the other issuer, has read it
            if (!warp_wait(&b.ds_free[bb], (dsf[bb] & 1u) ^ 1u, wc)) { ok = false; return false; }
            ++dsf[bb];
            tmem_st32(tmem + lane_off + 384 + 64 * bb + 32 * h, pk);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&b.ds_full[bb]);
            ++jj;
            return true;
        });
        if (!ok) break;
        if (!warp_wait(b.acc_done, it & 1u, wc)) { ok = false; break; }
        ++it;
        tc_fence_after();
        if (RA_CHECKED(row_ok, p.err, kSiteBwdGradRow))
            store_acc<D / 2>(acc_tm, p.dq + static_cast<size_t>(grow) * D + h * (D / 2));
        tc_fence_before();
        mbar_arrive(b.acc_free);
    }
}

// ------------------------------------------------------------------ dk/dv kernel
template <int D>
__device__ void kv_load(const AttnBwdParams& p, const CUtensorMap* tq, const CUtensorMap* tdo,
                        const CUtensorMap* tk, const CUtensorMap* tv, uint8_t* smem, const Bars& b,
                        volatile int* ring, const WaitCtl& wc) {
    using C = BwdCfg<D>;
    const Ring& R = p.ring;
    // Q, dO are re-read by every key tile of their KV group: keep them in L2
    const uint64_t keep = make_policy_evict_last(), stream = make_policy_evict_first();
    uint32_t qa = 0, ob = 0, kit = 0;
    bool ok = true;
    for (uint32_t n_it = 0; ok; ++n_it) {
        const int item = publish_item(p.sched, p.n_items, b.item_full, b.item_empty, ring, n_it, wc);
        if (item == -2) { ok = false; break; }
        if (item < 0) break;
        int hk, kp;
        kv_item(p, item, hk, kp);
        if (!mbar_wait(b.res_empty, (kit & 1u) ^ 1u, wc, 32)) { ok = false; break; }
        ++kit;
        mbar_arrive_expect_tx(b.res_full, 2 * C::kTileBytes);
        const int krow = checked_tile_row(row_of(p, hk, kp), R.Hkv, R, p.err, kSiteBwdKvRow);
        load_tile<D>(smem, tk, b.res_full, krow, stream);
        load_tile<D>(smem + C::kTileBytes, tv, b.res_full, krow, stream);
        for_each_query_tile(R, hk, kp, [&](int hq, int t0) -> bool {
            const int qrow = checked_tile_row(row_of(p, hq, t0), R.Hq, R, p.err, kSiteBwdQRow);
            if (!ring_load<D>(smem + C::kAOff, b.a_full, b.a_empty, qa, C::kSlotsA, tq, qrow, keep, wc) ||
                !ring_load<D>(smem + C::kBOff, b.b_full, b.b_empty, ob, C::kSlotsB, tdo, qrow, keep, wc)) {
                ok = false;
                return false;
            }
            ++qa;
            ++ob;
            return true;
        });
    }
    if (!ok) {
        ring_drain(b.a_full, qa, C::kSlotsA, wc.timeout_ns);
        ring_drain(b.b_full, ob, C::kSlotsB, wc.timeout_ns);
        if (kit > 0) drain_wait(b.res_full, (kit - 1) & 1u, wc.timeout_ns);
    }
}

template <int D>
__device__ void kv_mma(const AttnBwdParams& p, uint8_t* smem, const Bars& b, uint32_t tmem, volatile int* ring, const WaitCtl& wc) {
    using C = BwdCfg<D>;
    const Ring& R = p.ring;
    const uint32_t sK = smem_u32(smem), sV = sK + C::kTileBytes;
    const uint32_t sA = sK + C::kAOff, sB = sK + C::kBOff;
    uint32_t idx = 0, kit = 0, pf = 0, dsf = 0;
    bool ok = true;
    for (uint32_t n_it = 0; ok; ++n_it) {
        const int item = take_item(b.item_full, b.item_empty, ring, n_it, (threadIdx.x & 31) == 0, wc);
        if (item == -2) { ok = false; break; }
        if (item < 0) break;
        int hk, kp;
        kv_item(p, item, hk, kp);
        const int n = count_query_tiles(R, hk, kp);
        const uint32_t i0 = idx;
        if (!mbar_wait_w(b.res_full, kit & 1u, wc)) { ok = false; break; }
        // S^T(0) = K Q(0)^T, dP^T(0) = V dO(0)^T
        if (!ring_wait_w(b.a_full, i0, C::kSlotsA, wc)) { ok = false; break; }
        tc_fence_after();
        issue_kk<D>(tmem, sK, sA + (i0 % C::kSlotsA) * C::kTileBytes);
        mma_commit_e(b.s_full);
        if (!ring_wait_w(b.b_full, i0, C::kSlotsB, wc)) { ok = false; break; }
        tc_fence_after();
        issue_kk<D>(tmem + kTile, sV, sB + (i0 % C::kSlotsB) * C::kTileBytes);
        mma_commit_e(b.dp_full);
        // Per query tile t the tensor pipe takes dV(t), S^T(t+1), dK(t), dP^T(t+1) in that
        // order.  P^T(t) sits over S^T(t)'s columns and dS^T(t) over dP^T(t)'s, so each
        // product that overwrites them comes after the one that reads them (the pipe runs
        // a CTA's MMAs in issue order), and only dK(t) and dP^T(t+1) lie between one dS^T
        // and the next.
        for (int t = 0; t < n && ok; ++t) {
            const uint32_t i = i0 + t;
            const bool more = t + 1 < n;
            if (__any_sync(0xffffffffu, *wc.abort_flag != 0)) { ok = false; break; }
            named_bar_sync(kPtBar, kHandThreads);
            ++pf;
            if (t == 0 && !mbar_wait_w(b.acc_free, (kit & 1u) ^ 1u, wc)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sq = sA + (i % C::kSlotsA) * C::kTileBytes;
            const uint32_t sdo = sB + (i % C::kSlotsB) * C::kTileBytes;
            issue_tm<D>(tmem + kAccCol, tmem, 64, sdo, t > 0);  // dV += P^T dO
            mma_commit_e(&b.b_empty[i % C::kSlotsB]);
            if (more) {  // S^T(t+1) over P^T(t), which dV(t) has read
                if (!ring_wait_w(b.a_full, i + 1, C::kSlotsA, wc)) { ok = false; break; }
                tc_fence_after();
                issue_kk<D>(tmem, sK, sA + ((i + 1) % C::kSlotsA) * C::kTileBytes);
                mma_commit_e(b.s_full);
            }
            if (__any_sync(0xffffffffu, *wc.abort_flag != 0)) { ok = false; break; }
            named_bar_sync(kDsBar, kHandThreads);
            ++dsf;
            tc_fence_after();
            issue_tm<D>(tmem + kAccCol + D, tmem + kTile, 64, sq, t > 0);  // dK += dS^T Q
            mma_commit_e(&b.a_empty[i % C::kSlotsA]);
            if (more) {  // dP^T(t+1) over dS^T(t), which dK(t) has read
                if (!ring_wait_w(b.b_full, i + 1, C::kSlotsB, wc)) { ok = false; break; }
                tc_fence_after();
                issue_kk<D>(tmem + kTile, sV, sB + ((i + 1) % C::kSlotsB) * C::kTileBytes);
                mma_commit_e(b.dp_full);
            }
        }
        if (!ok) break;
        idx = i0 + n;
        mma_commit_e(b.res_empty);
        mma_commit_e(b.acc_done);
        ++kit;
    }
    if (!ok) {
        mma_commit_e(b.drain);
        drain_wait(b.drain, 0, wc.timeout_ns);
    }
}

template <int D>
__device__ void kv_compute(const AttnBwdParams& p, const Bars& b, uint32_t tmem, volatile int* ring, const WaitCtl& wc) {
    const Ring& R = p.ring;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int h = warp / 4, wq = warp % 4;
    const int row = wq * 32 + lane;  // key row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_tm = tmem + lane_off + h * 64;           // my 64 query columns of S^T
    const uint32_t dp_tm = tmem + lane_off + kTile + h * 64;  // and of dP^T (P^T, dS^T go here)
    const uint32_t dv_tm = tmem + lane_off + kAccCol + h * (D / 2);
    const uint32_t dk_tm = tmem + lane_off + kAccCol + D + h * (D / 2);
    uint32_t sf = 0, dpf = 0, it = 0;
    bool ok = true;
    // The MMA warp waits for P^T and dS^T on named barriers, which cannot time out.  These
    // warps arrive for every tile whose S^T (for P^T) and dP^T (for dS^T) the MMA warp queued
    // (those complete), and it queues S^T(t+1) only after taking P^T(t) and dP^T(t+1) only
    // after taking dS^T(t), so no phase gets a second arrival; their waits ignore the abort
    // flag and give up only on their own time limit, which products the MMA warp queued
    // cannot reach, so it is never left without an arrival.
    for (uint32_t n_it = 0; ok; ++n_it) {
        const int item = take_item(b.item_full, b.item_empty, ring, n_it, lane == 0, wc, false);
        if (item == -2) { ok = false; break; }
        if (item < 0) break;
        int hk, kp;
        kv_item(p, item, hk, kp);
        const int kpos = kp + row;
        // Lane l of every warp holds -lse log2(e) and -D of query columns 2l and 2l+1 of its
        // warpgroup's 64, fetched one step ahead (the loads' L2 latency hides behind a
        // step); the loops take a column's value from its lane with a shuffle.  (Staged in
        // shared memory instead, the values were read while the tensor core's operand
        // reads held shared memory busy, which doubled the exponential loop.)
        // (raw values travel a step; they are scaled where they are used, so that no
        // instruction waits for the loads until then).  The chunk map of a position is
        // worked out once for the g heads that share it.
        int map_t0 = -1, map_row = 0;
        auto fetch = [&](int hq, int t0, float2& a, float2& dd) {
            if (t0 != map_t0) {
                map_t0 = t0;
                map_row = row_of(p, 0, t0);
            }
            const int r0 = hq * R.S + map_row;  // first row of the query tile
            if (!RA_CHECKED(r0 >= 0 && static_cast<long long>(r0) + kTile <= static_cast<long long>(R.Hq) * R.S, p.err,
                            kSiteBwdLseRow)) {
                a = dd = make_float2(0.f, 0.f);
                return;
            }
            const int c = r0 + h * 64 + 2 * lane;
            a = __ldg(reinterpret_cast<const float2*>(p.lse + c));
            dd = __ldg(reinterpret_cast<const float2*>(p.delta + c));
        };
        float2 lse_next, d_next;
        fetch(hk * R.g, R.S - kTile, lse_next, d_next);
        for_each_query_tile(R, hk, kp, [&](int hq, int t0) -> bool {
            const float2 lse_cur = lse_next, d_cur = d_next;
            int nhq, nt0;
            if (next_query_tile(R, hk, kp, hq, t0, nhq, nt0)) fetch(nhq, nt0, lse_next, d_next);
            if (!group_wait(b.s_full, sf & 1u, h, wq, wc, false)) { ok = false; return false; }
            ++sf;
            const float4 vals = make_float4(-lse_cur.x * kLog2e, -lse_cur.y * kLog2e, -d_cur.x, -d_cur.y);
            tc_fence_after();
            float x[64];
            tmem_ld64(s_tm, x);
            const int lo = kpos - (t0 + h * 64);  // my query columns [lo, 64) see my key
            // only tiles on the diagonal mask; branch on the warp, not per element
            if (__any_sync(0xffffffffu, R.causal && lo > 0)) {
                const int lm = R.causal ? lo : 0;
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    float p0, p1;
                    ffma2(p0, p1, x[2 * k], x[2 * k + 1], kLog2e, kLog2e, __shfl_sync(0xffffffffu, vals.x, k),
                          __shfl_sync(0xffffffffu, vals.y, k));
                    x[2 * k] = (2 * k < lm) ? 0.f : ex2(p0);
                    x[2 * k + 1] = (2 * k + 1 < lm) ? 0.f : ex2(p1);
                }
            } else {
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    float p0, p1;
                    ffma2(p0, p1, x[2 * k], x[2 * k + 1], kLog2e, kLog2e, __shfl_sync(0xffffffffu, vals.x, k),
                          __shfl_sync(0xffffffffu, vals.y, k));
                    x[2 * k] = ex2(p0);
                    x[2 * k + 1] = ex2(p1);
                }
            }
            {
                // P^T (bf16) over the first 32 of my own S^T columns, whose values are in
                // registers: dV(t) can start while dS^T is still being formed
                uint32_t pp[32];
#pragma unroll
                for (int k = 0; k < 32; ++k) pp[k] = pack_bf16x2(x[2 * k], x[2 * k + 1]);
                tmem_st32(s_tm, pp);
                tmem_wait_st();
                tc_fence_before();
                named_bar_arrive(kPtBar, kHandThreads);
            }
            if (!group_wait(b.dp_full, dpf & 1u, h, wq, wc, false)) { ok = false; return false; }
            ++dpf;
            tc_fence_after();
            uint32_t pd[32];
            // dP^T in two 32-column chunks, each packed as soon as it is used, so that P, dP^T
            // and the packed words are never all live at once
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t r[32];
                tmem_ld32(dp_tm + 32 * c, r);
                tmem_wait_ld();
#pragma unroll
                for (int k2 = 0; k2 < 16; ++k2) {
                    const int k = 16 * c + k2;  // query columns 2k, 2k+1: -D from lane k
                    float a0, a1;
                    fadd2(a0, a1, __uint_as_float(r[2 * k2]), __uint_as_float(r[2 * k2 + 1]),
                          __shfl_sync(0xffffffffu, vals.z, k), __shfl_sync(0xffffffffu, vals.w, k));
                    fmul2(a0, a1, a0, a1, x[2 * k], x[2 * k + 1]);
                    pd[k] = pack_bf16x2(a0, a1);
                }
            }
            tmem_st32(dp_tm, pd);  // dS^T over the first 32 of my own dP^T columns
            tmem_wait_st();
            tc_fence_before();
            named_bar_arrive(kDsBar, kHandThreads);
            return true;
        });
        if (!ok) break;
        if (!group_wait(b.acc_done, it & 1u, h, wq, wc, false)) { ok = false; break; }
        ++it;
        tc_fence_after();
        const size_t grow = static_cast<size_t>(row_of(p, hk, kp) + row);
        if (RA_CHECKED(grow < static_cast<size_t>(R.Hkv) * R.S, p.err, kSiteBwdGradRow)) {
            store_acc<D / 2>(dv_tm, p.dv + grow * D + h * (D / 2));
            store_acc<D / 2>(dk_tm, p.dk + grow * D + h * (D / 2));
        }
        tc_fence_before();
        mbar_arrive(b.acc_free);
    }
}

// ------------------------------------------------------------------ kernels
template <int D, bool DQ>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ AttnBwdParams p, const __grid_constant__ CUtensorMap tq,
               const __grid_constant__ CUtensorMap tdo, const __grid_constant__ CUtensorMap tk,
               const __grid_constant__ CUtensorMap tv) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    const Bars b(bars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kBarOff + C::kNumBars * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kBarOff + C::kNumBars * 8 + 4);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        init_bars(b, DQ ? 2u : 1u);  // dQ kernel: a K slot is released by both issuers
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kLoadWarp && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tdo);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl wc{abort_flag, p.err, p.timeout_ns};
    volatile int* ring = reinterpret_cast<volatile int*>(smem + C::kRingOff);
    if (warp < 8) {
        if constexpr (DQ) dq_compute<D>(p, b, tmem, ring, wc);
        else kv_compute<D>(p, b, tmem, ring, wc);
    } else if (warp == kMmaWarp) {  // the whole warp: see mma_ss_e
        if constexpr (DQ) dq_mma<D>(p, smem, b, tmem, ring, wc);
        else kv_mma<D>(p, smem, b, tmem, ring, wc);
    } else if (warp == kLoadWarp) {
        if (lane == 0) {
            if constexpr (DQ) dq_load<D>(p, &tq, &tdo, &tk, &tv, smem, b, ring, wc);
            else kv_load<D>(p, &tq, &tdo, &tk, &tv, smem, b, ring, wc);
        }
    } else if (warp == kMma2Warp) {
        if (lane == 0 || DQ) {
            if constexpr (DQ) {
                dq_mma2<D>(p, smem, b, tmem, ring, wc);
            } else {  // no second issuer in the dk/dv kernel: take the items only
                for (uint32_t n_it = 0; take_item(b.item_full, b.item_empty, ring, n_it, true, wc) >= 0; ++n_it) {
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
    if (threadIdx.x == 0) finish_items(p.sched);
}

// ------------------------------------------------------------------ D = dout . out
// Lane l holds elements [l*E, l*E + E) of a row (E = D / 32); a warp takes R consecutive rows
// per iteration and issues all their loads before reducing, so 2R independent loads per lane
// are in flight (one row at a time leaves an HBM-bound kernel latency-bound).
template <int D, int R>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const uint16_t* __restrict__ dout,
                                                        const float* __restrict__ out, float* __restrict__ delta,
                                                        long long rows) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const long long warp = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
    for (long long r0 = warp * R; r0 < rows; r0 += warps * R) {
        float acc[R];
        if constexpr (E == 4) {
            float4 o[R];
            uint2 g[R];
#pragma unroll
            for (int k = 0; k < R; ++k) {
                if (r0 + k < rows) {
                    const size_t base = static_cast<size_t>(r0 + k) * D + lane * E;
                    o[k] = *reinterpret_cast<const float4*>(out + base);
                    g[k] = *reinterpret_cast<const uint2*>(dout + base);
                }
            }
#pragma unroll
            for (int k = 0; k < R; ++k)
                acc[k] = (r0 + k < rows)
                             ? o[k].x * __uint_as_float(g[k].x << 16) + o[k].y * __uint_as_float(g[k].x & 0xffff0000u) +
                                   o[k].z * __uint_as_float(g[k].y << 16) + o[k].w * __uint_as_float(g[k].y & 0xffff0000u)
                             : 0.f;
        } else {
            float2 o[R];
            uint32_t g[R];
#pragma unroll
            for (int k = 0; k < R; ++k) {
                if (r0 + k < rows) {
                    const size_t base = static_cast<size_t>(r0 + k) * D + lane * E;
                    o[k] = *reinterpret_cast<const float2*>(out + base);
                    g[k] = *reinterpret_cast<const uint32_t*>(dout + base);
                }
            }
#pragma unroll
            for (int k = 0; k < R; ++k)
                acc[k] = (r0 + k < rows) ? o[k].x * __uint_as_float(g[k] << 16) + o[k].y * __uint_as_float(g[k] & 0xffff0000u)
                                         : 0.f;
        }
#pragma unroll
        for (int k = 0; k < R; ++k)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], off);
        if (lane < R && r0 + lane < rows) {
            float v = acc[0];
#pragma unroll
            for (int k = 1; k < R; ++k) v = (lane == k) ? acc[k] : v;
            delta[r0 + lane] = v;
        }
    }
}

template <int D>
int launch_bwd_d(const AttnBwdParams& p0, const float* out, const void* dout, const CUtensorMap& tq,
                 const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo, int sms, cudaStream_t stream) {
    using C = BwdCfg<D>;
    const Ring& R = p0.ring;
    const long long rows = static_cast<long long>(R.Hq) * R.S;
    constexpr int kRows = 4;
    long long blocks = (rows + 8 * kRows - 1) / (8 * kRows);
    if (blocks > static_cast<long long>(sms) * 8) blocks = static_cast<long long>(sms) * 8;
    bwd_delta_kernel<D, kRows><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint16_t*>(dout), out, const_cast<float*>(p0.delta), rows);
    if (cudaGetLastError() != cudaSuccess) return -4;

    AttnBwdParams p = p0;
    p.n_items = R.Hq * p.n_tiles;
    auto kq = bwd_kernel<D, true>;
    if (cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess) return -4;
    kq<<<p.n_items < sms ? p.n_items : sms, kThreads, C::kSmem, stream>>>(p, tq, tdo, tk, tv);
    if (cudaGetLastError() != cudaSuccess) return -4;

    p.n_items = R.Hkv * p.n_tiles;
    p.sched = p0.sched + 2;  // the dk/dv launch's own counter pair
    auto kkv = bwd_kernel<D, false>;
    if (cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem) != cudaSuccess) return -4;
    kkv<<<p.n_items < sms ? p.n_items : sms, kThreads, C::kSmem, stream>>>(p, tq, tdo, tk, tv);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace

int launch_attn_bwd(const AttnBwdParams& p, const float* out, const void* dout, const CUtensorMap& tq,
                    const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo, int sms,
                    cudaStream_t stream) {
    if (p.ring.d == 128) return launch_bwd_d<128>(p, out, dout, tq, tk, tv, tdo, sms, stream);
    if (p.ring.d == 64) return launch_bwd_d<64>(p, out, dout, tq, tk, tv, tdo, sms, stream);
    return -2;
}

}  // namespace ra
