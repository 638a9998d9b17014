// attn_bwd.cu -- backward pass of the fused ring attention on tcgen05 tensor cores.
//
// The pages give the forward only (the training FLOP count of "Interrogating
// parallelism, part 5" covers a backward pass but does not describe it); this is the
// exact gradient of that forward.  With P_ij = exp(q_i . k_j - lse_i) over visible keys,
// D_i = dout_i . out_i and dS_ij = P_ij (dout_i . v_j - D_i):
//     dV_j = sum_i P_ij dout_i,   dK_j = sum_i dS_ij q_i,   dQ_i = sum_j dS_ij k_j,
// a KV head summing over the query heads that use it.  The ring order is kept: a query
// tile meets the KV blocks hop by hop as in the forward (the dq kernel), and a KV block
// travels round the ring with its dK, dV accumulators, meeting rank (s + h) mod c's
// queries at hop h (the dk/dv kernel).  Only the order of the fp32 sums depends on it.
//
// Three kernels, all on the caller's stream:
//   * bwd_delta_kernel   D_i = dout_i . out_i, one warp per row (HBM-bound);
//   * bwd_dq_kernel      one 128-row query tile per work item: per key tile
//                        S = Q K^T and dP = dO V^T into TMEM, then dS (bf16) into TMEM,
//                        then dQ += dS K with dS read from TMEM;
//   * bwd_dkdv_kernel    one 128-row key tile per work item: per query tile
//                        S^T = K Q^T and dP^T = V dO^T, then P^T and dS^T (bf16) into
//                        TMEM, then dV += P^T dO and dK += dS^T Q.
// Splitting dq from dk/dv recomputes S and dP once more (7 tile products instead of 5)
// but needs no atomics and gives a deterministic result.
//
// Each CTA is persistent: warps 0-7 compute (warpgroup h handles key or query columns
// [64h, 64h+64) of the 128 x 128 tile, thread = TMEM lane = row), warp 8 issues the
// MMAs (one thread), warp 9 the TMA loads (one thread).  Every operand form used here
// (both operands K-major from shared memory; A from TMEM with an MN-major B) is one the
// forward kernel uses too.  TMEM: S [0,128), dP [128,256), accumulators from 256.  The
// packed bf16 P / dS of column half h overwrite the first 32 columns of that half's own
// S / dP columns, so the halves never touch each other's columns.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ra {
namespace {

constexpr int kTile = 128;
constexpr int kThreads = 320;
constexpr int kMmaWarp = 8, kLoadWarp = 9;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kAccCol = 256;

template <int D>
struct BwdCfg {
    static constexpr int kTileBytes = kTile * D * 2;  // one 128 x D bf16 tile
    static constexpr int kBoxBytes = kTile * 64 * 2;  // one 128 x 64 TMA box
    static constexpr int kBoxes = D / 64;
    static constexpr int kStages = (D == 128) ? 2 : 4;
    // dq kernel: Q, dO resident; stages of (K, V)
    static constexpr int kDqStageBytes = 2 * kTileBytes;
    static constexpr int kDqKVOff = 2 * kTileBytes;
    static constexpr int kDqBarOff = kDqKVOff + kStages * kDqStageBytes;
    // dk/dv kernel: K, V resident; stages of (Q, dO, lse[128], delta[128])
    static constexpr int kKvStageBytes = 2 * kTileBytes + 1024;
    static constexpr int kKvQOff = 2 * kTileBytes;
    static constexpr int kKvBarOff = kKvQOff + kStages * kKvStageBytes;
    static constexpr int kNumBars = 16 + 2 * kStages;
    static constexpr int kDqSmem = kDqBarOff + kNumBars * 8 + 16 + 1024;  // + slack to align the base
    static constexpr int kKvSmem = kKvBarOff + kNumBars * 8 + 16 + 1024;
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

// Query tiles the key tile at kp meets as its block travels: hop h visits rank
// (s + h) mod c; each query tile is met once per query head of the KV group.
template <class F>
__device__ __forceinline__ void for_each_query_tile(const Ring& R, int hk, int kp, F&& f) {
    const int s = rank_of(R, kp);
    for (int hop = 0; hop < R.c; ++hop) {
        const int r = (s + hop) % R.c;
        for (int slot = 0; slot < R.nslot; ++slot) {
            const int base = (slot ? 2 * R.c - 1 - r : r) * R.m;
            const int first = (R.causal && kp > base) ? kp : base;
            for (int t0 = first; t0 < base + R.m; t0 += kTile)
                for (int x = 0; x < R.g; ++x)
                    if (!f(hk * R.g + x, t0)) return;
        }
    }
}

__device__ __forceinline__ int count_query_tiles(const Ring& R, int hk, int kp) {
    int n = 0;
    for_each_query_tile(R, hk, kp, [&](int, int) { ++n; return true; });
    return n;
}

__device__ __forceinline__ int item_of_round(int round) {
    const int b = (round & 1) ? (gridDim.x - 1 - blockIdx.x) : blockIdx.x;
    return round * gridDim.x + b;
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > timeout_ns) return;
    }
}

// Named barrier over one compute warpgroup (128 threads); returns the AND of `ok`.
__device__ __forceinline__ bool group_bar_and(int h, bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.and.pred po, %2, 128, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(ok ? 1u : 0u), "r"(1 + h)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t off16) {
    uint64_t r;
    asm volatile("add.s64 %0, %1, %2;" : "=l"(r) : "l"(desc), "l"(static_cast<uint64_t>(off16)));
    return r;
}

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
        mma_ss(d_tmem, desc_add(ad, off), desc_add(bd, off), idesc, kk > 0 ? 1u : 0u);
    }
}

// D[tmem] (+)= A B: A (128 x 128, bf16 packed in TMEM by column halves: keys or queries
// [64h, 64h+64) in columns a_col + 64h + [0, 32)), B (128 x D) from shared memory as an
// MN-major operand (the tile's rows are the contraction index).
template <int D>
__device__ __forceinline__ void issue_tm(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_base, bool accumulate) {
    using C = BwdCfg<D>;
    constexpr uint32_t idesc = idesc_bf16(kTile, D, 1);
    const uint64_t bd = sdesc_sw128(b_base, C::kBoxBytes, 1024);
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk) {
        const uint32_t acol = (kk / 4) * 64 + (kk % 4) * 8;
        mma_ts(d_tmem, a_tmem + acol, desc_add(bd, (kk * 16 * 128) >> 4), idesc,
               (accumulate || kk > 0) ? 1u : 0u);
    }
}

// Load a 128 x D bf16 tile (rows row..row+127) as D/64 boxes.
template <int D>
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int row,
                                          uint64_t policy) {
    using C = BwdCfg<D>;
#pragma unroll
    for (int bx = 0; bx < C::kBoxes; ++bx) tma_load_2d_hint(dst + bx * C::kBoxBytes, map, bar, bx * 64, row, policy);
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

// ------------------------------------------------------------------ dq kernel
// Barriers: 0 q_full (Q, dO landed), 1 q_empty (item's MMAs done with Q, dO), 2 s_full
// (S, dP in TMEM), 3 ds_full (256 compute threads wrote dS), 4 acc_done (item's dQ
// complete), 5 acc_free (256 threads read dQ out), 6 drain (abort only), then kv_full
// and kv_empty per stage (K and V of one key tile).
struct DqBars {
    uint64_t *q_full, *q_empty, *s_full, *ds_full, *acc_done, *acc_free, *drain, *kv_full, *kv_empty;
    __device__ DqBars(uint64_t* b, int stages)
        : q_full(b), q_empty(b + 1), s_full(b + 2), ds_full(b + 3), acc_done(b + 4), acc_free(b + 5),
          drain(b + 6), kv_full(b + 16), kv_empty(b + 16 + stages) {}
};

template <int D>
__device__ void dq_load(const AttnBwdParams& p, const CUtensorMap* tq, const CUtensorMap* tdo,
                        const CUtensorMap* tk, const CUtensorMap* tv, uint8_t* smem, const DqBars& b,
                        const WaitCtl& wc) {
    using C = BwdCfg<D>;
    const Ring& R = p.ring;
    const uint64_t keep = make_policy_evict_last(), stream = make_policy_evict_first();
    uint32_t kv_idx = 0, qit = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
        if (round * (int)gridDim.x >= p.n_items) break;
        const int item = item_of_round(round);
        if (item >= p.n_items) continue;
        int hq, qp;
        dq_item(p, item, hq, qp);
        if (!mbar_wait(b.q_empty, (qit & 1u) ^ 1u, wc, 32)) { ok = false; break; }
        ++qit;
        mbar_arrive_expect_tx(b.q_full, 2 * C::kTileBytes);
        const int qrow = row_of(p, hq, qp);
        load_tile<D>(smem, tq, b.q_full, qrow, stream);
        load_tile<D>(smem + C::kTileBytes, tdo, b.q_full, qrow, stream);
        const int hk = hq / R.g;
        for_each_key_tile(R, qp, [&](int t0) -> bool {
            const uint32_t s = kv_idx % C::kStages;
            if (!mbar_wait(&b.kv_empty[s], ((kv_idx / C::kStages) & 1u) ^ 1u, wc, 32)) { ok = false; return false; }
            mbar_arrive_expect_tx(&b.kv_full[s], 2 * C::kTileBytes);
            uint8_t* st = smem + C::kDqKVOff + s * C::kDqStageBytes;
            const int krow = row_of(p, hk, t0);
            load_tile<D>(st, tk, &b.kv_full[s], krow, keep);
            load_tile<D>(st + C::kTileBytes, tv, &b.kv_full[s], krow, keep);
            ++kv_idx;
            return true;
        });
    }
    if (!ok) {
        // let every copy already issued land before the CTA's shared memory goes away
        for (uint32_t s = 0; s < (uint32_t)C::kStages && s < kv_idx; ++s) {
            const uint32_t last = kv_idx - 1 - ((kv_idx - 1 - s) % C::kStages);
            drain_wait(&b.kv_full[s], (last / C::kStages) & 1u, wc.timeout_ns);
        }
        if (qit > 0) drain_wait(b.q_full, (qit - 1) & 1u, wc.timeout_ns);
    }
}

template <int D>
__device__ void dq_mma(const AttnBwdParams& p, uint8_t* smem, const DqBars& b, uint32_t tmem, const WaitCtl& wc) {
    using C = BwdCfg<D>;
    const Ring& R = p.ring;
    const uint32_t sQ = smem_u32(smem), sdO = sQ + C::kTileBytes, sKV = sQ + C::kDqKVOff;
    uint32_t kv_idx = 0, qit = 0, dsit = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
        if (round * (int)gridDim.x >= p.n_items) break;
        const int item = item_of_round(round);
        if (item >= p.n_items) continue;
        int hq, qp;
        dq_item(p, item, hq, qp);
        const int nj = count_key_tiles(R, qp);
        if (!mbar_wait(b.q_full, qit & 1u, wc)) { ok = false; break; }
        uint32_t st = kv_idx % C::kStages;
        if (!mbar_wait(&b.kv_full[st], (kv_idx / C::kStages) & 1u, wc)) { ok = false; break; }
        tc_fence_after();
        issue_kk<D>(tmem, sQ, sKV + st * C::kDqStageBytes);                            // S = Q K^T
        issue_kk<D>(tmem + kTile, sdO, sKV + st * C::kDqStageBytes + C::kTileBytes);  // dP = dO V^T
        mma_commit(b.s_full);
        for (int j = 0; j < nj && ok; ++j) {
            if (!mbar_wait(b.ds_full, dsit & 1u, wc)) { ok = false; break; }
            ++dsit;
            if (j == 0 && !mbar_wait(b.acc_free, (qit & 1u) ^ 1u, wc)) { ok = false; break; }
            tc_fence_after();
            issue_tm<D>(tmem + kAccCol, tmem, sKV + st * C::kDqStageBytes, j > 0);  // dQ += dS K
            mma_commit(&b.kv_empty[st]);
            ++kv_idx;
            if (j + 1 < nj) {
                st = kv_idx % C::kStages;
                if (!mbar_wait(&b.kv_full[st], (kv_idx / C::kStages) & 1u, wc)) { ok = false; break; }
                tc_fence_after();
                issue_kk<D>(tmem, sQ, sKV + st * C::kDqStageBytes);
                issue_kk<D>(tmem + kTile, sdO, sKV + st * C::kDqStageBytes + C::kTileBytes);
                mma_commit(b.s_full);
            }
        }
        if (!ok) break;
        mma_commit(b.q_empty);
        mma_commit(b.acc_done);
        ++qit;
    }
    if (!ok) {
        // every MMA issued so far must finish before TMEM is released
        mma_commit(b.drain);
        drain_wait(b.drain, 0, wc.timeout_ns);
    }
}

template <int D>
__device__ void dq_compute(const AttnBwdParams& p, const DqBars& b, uint32_t tmem, const WaitCtl& wc) {
    const Ring& R = p.ring;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int h = warp / 4, wq = warp % 4;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_tm = tmem + lane_off + h * 64;           // my 64 key columns of S
    const uint32_t dp_tm = tmem + lane_off + kTile + h * 64;  // and of dP
    const uint32_t acc_tm = tmem + lane_off + kAccCol + h * (D / 2);
    uint32_t sit = 0, it = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
        if (round * (int)gridDim.x >= p.n_items) break;
        const int item = item_of_round(round);
        if (item >= p.n_items) continue;
        int hq, qp;
        dq_item(p, item, hq, qp);
        const int grow = row_of(p, hq, qp) + row;
        const float nl = -__ldg(p.lse + grow) * kLog2e;
        const float dl = __ldg(p.delta + grow);
        const int qpos = qp + row;
        for_each_key_tile(R, qp, [&](int t0) -> bool {
            bool w_ok = true;
            if (wq == 0) w_ok = __all_sync(0xffffffffu, mbar_wait(b.s_full, sit & 1u, wc));
            w_ok = group_bar_and(h, w_ok);
            ++sit;
            if (!w_ok) { ok = false; return false; }
            tc_fence_after();
            float s[64], dp[64];
            tmem_ld64(s_tm, s);
            tmem_ld64(dp_tm, dp);
            const int lim = qpos - (t0 + h * 64);  // my keys [0, lim] are visible
            const bool mask = R.causal && lim < 63;
            uint32_t pk[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                float p0, p1;
                ffma2(p0, p1, s[2 * i], s[2 * i + 1], kLog2e, kLog2e, nl, nl);
                p0 = ex2(p0);
                p1 = ex2(p1);
                if (mask) {
                    p0 = (2 * i > lim) ? 0.f : p0;
                    p1 = (2 * i + 1 > lim) ? 0.f : p1;
                }
                pk[i] = pack_bf16x2(p0 * (dp[2 * i] - dl), p1 * (dp[2 * i + 1] - dl));
            }
            tmem_st32(s_tm, pk);  // dS over the first 32 of my own S columns
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(b.ds_full);
            return true;
        });
        if (!ok) break;
        bool d_ok = true;
        if (wq == 0) d_ok = __all_sync(0xffffffffu, mbar_wait(b.acc_done, it & 1u, wc));
        if (!group_bar_and(h, d_ok)) { ok = false; break; }
        ++it;
        tc_fence_after();
        store_acc<D / 2>(acc_tm, p.dq + static_cast<size_t>(grow) * D + h * (D / 2));
        tc_fence_before();
        mbar_arrive(b.acc_free);
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ AttnBwdParams p, const __grid_constant__ CUtensorMap tq,
                  const __grid_constant__ CUtensorMap tdo, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kDqBarOff);
    const DqBars b(bars, C::kStages);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kDqBarOff + C::kNumBars * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kDqBarOff + C::kNumBars * 8 + 4);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        mbar_init(b.q_full, 1);
        mbar_init(b.q_empty, 1);
        mbar_init(b.s_full, 1);
        mbar_init(b.ds_full, 256);
        mbar_init(b.acc_done, 1);
        mbar_init(b.acc_free, 256);
        mbar_init(b.drain, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&b.kv_full[s], 1);
            mbar_init(&b.kv_empty[s], 1);
        }
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
    if (warp < 8) {
        dq_compute<D>(p, b, tmem, wc);
    } else if (warp == kMmaWarp) {
        if (lane == 0) dq_mma<D>(p, smem, b, tmem, wc);
    } else if (warp == kLoadWarp) {
        if (lane == 0) dq_load<D>(p, &tq, &tdo, &tk, &tv, smem, b, wc);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ dk/dv kernel
// Barriers: 0 kv_full (K, V landed), 1 kv_empty (item's MMAs done with K, V), 2 s_full
// (S^T, dP^T in TMEM), 3 p_full (256 compute threads wrote P^T, dS^T), 4 acc_done,
// 5 acc_free (256), 6 drain, then qd_full and qd_empty per stage (Q, dO, lse, D of one
// query tile).
struct KvBars {
    uint64_t *kv_full, *kv_empty, *s_full, *p_full, *acc_done, *acc_free, *drain, *qd_full, *qd_empty;
    __device__ KvBars(uint64_t* b, int stages)
        : kv_full(b), kv_empty(b + 1), s_full(b + 2), p_full(b + 3), acc_done(b + 4), acc_free(b + 5),
          drain(b + 6), qd_full(b + 16), qd_empty(b + 16 + stages) {}
};

template <int D>
__device__ void kv_load(const AttnBwdParams& p, const CUtensorMap* tq, const CUtensorMap* tdo,
                        const CUtensorMap* tk, const CUtensorMap* tv, uint8_t* smem, const KvBars& b,
                        const WaitCtl& wc) {
    using C = BwdCfg<D>;
    const Ring& R = p.ring;
    // Q, dO tiles are re-read by every key tile of their KV group: keep them in L2
    const uint64_t keep = make_policy_evict_last(), stream = make_policy_evict_first();
    uint32_t idx = 0, kit = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
        if (round * (int)gridDim.x >= p.n_items) break;
        const int item = item_of_round(round);
        if (item >= p.n_items) continue;
        int hk, kp;
        kv_item(p, item, hk, kp);
        if (!mbar_wait(b.kv_empty, (kit & 1u) ^ 1u, wc, 32)) { ok = false; break; }
        ++kit;
        mbar_arrive_expect_tx(b.kv_full, 2 * C::kTileBytes);
        const int krow = row_of(p, hk, kp);
        load_tile<D>(smem, tk, b.kv_full, krow, stream);
        load_tile<D>(smem + C::kTileBytes, tv, b.kv_full, krow, stream);
        for_each_query_tile(R, hk, kp, [&](int hq, int t0) -> bool {
            const uint32_t s = idx % C::kStages;
            if (!mbar_wait(&b.qd_empty[s], ((idx / C::kStages) & 1u) ^ 1u, wc, 32)) { ok = false; return false; }
            mbar_arrive_expect_tx(&b.qd_full[s], 2 * C::kTileBytes + 2 * kTile * 4);
            uint8_t* st = smem + C::kKvQOff + s * C::kKvStageBytes;
            const int qrow = row_of(p, hq, t0);
            load_tile<D>(st, tq, &b.qd_full[s], qrow, keep);
            load_tile<D>(st + C::kTileBytes, tdo, &b.qd_full[s], qrow, keep);
            bulk_load_1d(st + 2 * C::kTileBytes, p.lse + qrow, kTile * 4, &b.qd_full[s]);
            bulk_load_1d(st + 2 * C::kTileBytes + kTile * 4, p.delta + qrow, kTile * 4, &b.qd_full[s]);
            ++idx;
            return true;
        });
    }
    if (!ok) {
        for (uint32_t s = 0; s < (uint32_t)C::kStages && s < idx; ++s) {
            const uint32_t last = idx - 1 - ((idx - 1 - s) % C::kStages);
            drain_wait(&b.qd_full[s], (last / C::kStages) & 1u, wc.timeout_ns);
        }
        if (kit > 0) drain_wait(b.kv_full, (kit - 1) & 1u, wc.timeout_ns);
    }
}

template <int D>
__device__ void kv_mma(const AttnBwdParams& p, uint8_t* smem, const KvBars& b, uint32_t tmem, const WaitCtl& wc) {
    using C = BwdCfg<D>;
    const Ring& R = p.ring;
    const uint32_t sK = smem_u32(smem), sV = sK + C::kTileBytes, sQD = sK + C::kKvQOff;
    uint32_t idx = 0, kit = 0, pit = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
        if (round * (int)gridDim.x >= p.n_items) break;
        const int item = item_of_round(round);
        if (item >= p.n_items) continue;
        int hk, kp;
        kv_item(p, item, hk, kp);
        const int n = count_query_tiles(R, hk, kp);
        if (!mbar_wait(b.kv_full, kit & 1u, wc)) { ok = false; break; }
        uint32_t st = idx % C::kStages;
        if (!mbar_wait(&b.qd_full[st], (idx / C::kStages) & 1u, wc)) { ok = false; break; }
        tc_fence_after();
        issue_kk<D>(tmem, sK, sQD + st * C::kKvStageBytes);                           // S^T = K Q^T
        issue_kk<D>(tmem + kTile, sV, sQD + st * C::kKvStageBytes + C::kTileBytes);  // dP^T = V dO^T
        mma_commit(b.s_full);
        for (int i = 0; i < n && ok; ++i) {
            if (!mbar_wait(b.p_full, pit & 1u, wc)) { ok = false; break; }
            ++pit;
            if (i == 0 && !mbar_wait(b.acc_free, (kit & 1u) ^ 1u, wc)) { ok = false; break; }
            tc_fence_after();
            const uint32_t sq = sQD + st * C::kKvStageBytes;
            issue_tm<D>(tmem + kAccCol, tmem, sq + C::kTileBytes, i > 0);          // dV += P^T dO
            issue_tm<D>(tmem + kAccCol + D, tmem + kTile, sq, i > 0);              // dK += dS^T Q
            mma_commit(&b.qd_empty[st]);
            ++idx;
            if (i + 1 < n) {
                st = idx % C::kStages;
                if (!mbar_wait(&b.qd_full[st], (idx / C::kStages) & 1u, wc)) { ok = false; break; }
                tc_fence_after();
                issue_kk<D>(tmem, sK, sQD + st * C::kKvStageBytes);
                issue_kk<D>(tmem + kTile, sV, sQD + st * C::kKvStageBytes + C::kTileBytes);
                mma_commit(b.s_full);
            }
        }
        if (!ok) break;
        mma_commit(b.kv_empty);
        mma_commit(b.acc_done);
        ++kit;
    }
    if (!ok) {
        mma_commit(b.drain);
        drain_wait(b.drain, 0, wc.timeout_ns);
    }
}

template <int D>
__device__ void kv_compute(const AttnBwdParams& p, uint8_t* smem, const KvBars& b, uint32_t tmem,
                           const WaitCtl& wc) {
    using C = BwdCfg<D>;
    const Ring& R = p.ring;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int h = warp / 4, wq = warp % 4;
    const int row = wq * 32 + lane;  // key row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_tm = tmem + lane_off + h * 64;           // my 64 query columns of S^T
    const uint32_t dp_tm = tmem + lane_off + kTile + h * 64;  // and of dP^T
    const uint32_t dv_tm = tmem + lane_off + kAccCol + h * (D / 2);
    const uint32_t dk_tm = tmem + lane_off + kAccCol + D + h * (D / 2);
    uint32_t idx = 0, sit = 0, it = 0;
    bool ok = true;
    for (int round = 0; ok; ++round) {
        if (round * (int)gridDim.x >= p.n_items) break;
        const int item = item_of_round(round);
        if (item >= p.n_items) continue;
        int hk, kp;
        kv_item(p, item, hk, kp);
        const int kpos = kp + row;
        for_each_query_tile(R, hk, kp, [&](int, int t0) -> bool {
            const uint32_t st = idx % C::kStages;
            bool w_ok = true;
            if (wq == 0)
                w_ok = __all_sync(0xffffffffu, mbar_wait(b.s_full, sit & 1u, wc) &&
                                                   mbar_wait(&b.qd_full[st], (idx / C::kStages) & 1u, wc));
            w_ok = group_bar_and(h, w_ok);
            ++sit;
            ++idx;
            if (!w_ok) { ok = false; return false; }
            tc_fence_after();
            float s[64], dp[64];
            tmem_ld64(s_tm, s);
            tmem_ld64(dp_tm, dp);
            const float* sl = reinterpret_cast<const float*>(smem + C::kKvQOff + st * C::kKvStageBytes +
                                                             2 * C::kTileBytes) + h * 64;
            const float* sd = sl + kTile;
            const int lo = kpos - (t0 + h * 64);  // my query columns [lo, 64) see my key
            const bool mask = R.causal && lo > 0;
            uint32_t pp[32], pd[32];
#pragma unroll
            for (int i4 = 0; i4 < 16; ++i4) {
                const float4 l4 = reinterpret_cast<const float4*>(sl)[i4];
                const float4 d4 = reinterpret_cast<const float4*>(sd)[i4];
                const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
                const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
                for (int e = 0; e < 4; e += 2) {
                    const int i = i4 * 4 + e;
                    float p0, p1;
                    ffma2(p0, p1, s[i], s[i + 1], kLog2e, kLog2e, -lv[e] * kLog2e, -lv[e + 1] * kLog2e);
                    p0 = ex2(p0);
                    p1 = ex2(p1);
                    if (mask) {
                        p0 = (i < lo) ? 0.f : p0;
                        p1 = (i + 1 < lo) ? 0.f : p1;
                    }
                    pp[i / 2] = pack_bf16x2(p0, p1);
                    pd[i / 2] = pack_bf16x2(p0 * (dp[i] - dv[e]), p1 * (dp[i + 1] - dv[e + 1]));
                }
            }
            tmem_st32(s_tm, pp);   // P^T over the first 32 of my own S^T columns
            tmem_st32(dp_tm, pd);  // dS^T over the first 32 of my own dP^T columns
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(b.p_full);
            return true;
        });
        if (!ok) break;
        bool d_ok = true;
        if (wq == 0) d_ok = __all_sync(0xffffffffu, mbar_wait(b.acc_done, it & 1u, wc));
        if (!group_bar_and(h, d_ok)) { ok = false; break; }
        ++it;
        tc_fence_after();
        const size_t grow = static_cast<size_t>(row_of(p, hk, kp) + row);
        store_acc<D / 2>(dv_tm, p.dv + grow * D + h * (D / 2));
        store_acc<D / 2>(dk_tm, p.dk + grow * D + h * (D / 2));
        tc_fence_before();
        mbar_arrive(b.acc_free);
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ AttnBwdParams p, const __grid_constant__ CUtensorMap tq,
                    const __grid_constant__ CUtensorMap tdo, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv) {
    using C = BwdCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kKvBarOff);
    const KvBars b(bars, C::kStages);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kKvBarOff + C::kNumBars * 8);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kKvBarOff + C::kNumBars * 8 + 4);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        mbar_init(b.kv_full, 1);
        mbar_init(b.kv_empty, 1);
        mbar_init(b.s_full, 1);
        mbar_init(b.p_full, 256);
        mbar_init(b.acc_done, 1);
        mbar_init(b.acc_free, 256);
        mbar_init(b.drain, 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&b.qd_full[s], 1);
            mbar_init(&b.qd_empty[s], 1);
        }
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
    if (warp < 8) {
        kv_compute<D>(p, smem, b, tmem, wc);
    } else if (warp == kMmaWarp) {
        if (lane == 0) kv_mma<D>(p, smem, b, tmem, wc);
    } else if (warp == kLoadWarp) {
        if (lane == 0) kv_load<D>(p, &tq, &tdo, &tk, &tv, smem, b, wc);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ D = dout . out
// One warp per row; lane l holds elements [l*E, l*E + E) of the row (E = D / 32).
template <int D>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const uint16_t* __restrict__ dout,
                                                        const float* __restrict__ out, float* __restrict__ delta,
                                                        long long rows) {
    constexpr int E = D / 32;
    const int lane = threadIdx.x & 31;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
    for (long long r = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; r < rows;
         r += warps) {
        const size_t base = static_cast<size_t>(r) * D + lane * E;
        float acc = 0.f;
        if constexpr (E == 4) {
            const float4 o = *reinterpret_cast<const float4*>(out + base);
            const uint2 g = *reinterpret_cast<const uint2*>(dout + base);
            acc = o.x * __uint_as_float(g.x << 16) + o.y * __uint_as_float(g.x & 0xffff0000u) +
                  o.z * __uint_as_float(g.y << 16) + o.w * __uint_as_float(g.y & 0xffff0000u);
        } else {
            const float2 o = *reinterpret_cast<const float2*>(out + base);
            const uint32_t g = *reinterpret_cast<const uint32_t*>(dout + base);
            acc = o.x * __uint_as_float(g << 16) + o.y * __uint_as_float(g & 0xffff0000u);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) delta[r] = acc;
    }
}

template <int D>
int launch_bwd_d(const AttnBwdParams& p0, const float* out, const void* dout, const CUtensorMap& tq,
                 const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo, int sms, cudaStream_t stream) {
    using C = BwdCfg<D>;
    const Ring& R = p0.ring;
    const long long rows = static_cast<long long>(R.Hq) * R.S;
    long long blocks = (rows + 7) / 8;
    if (blocks > static_cast<long long>(sms) * 16) blocks = static_cast<long long>(sms) * 16;
    bwd_delta_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint16_t*>(dout), out, const_cast<float*>(p0.delta), rows);
    if (cudaGetLastError() != cudaSuccess) return -4;

    AttnBwdParams p = p0;
    p.n_items = R.Hq * p.n_tiles;
    auto kq = bwd_dq_kernel<D>;
    if (cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDqSmem) != cudaSuccess) return -4;
    kq<<<p.n_items < sms ? p.n_items : sms, kThreads, C::kDqSmem, stream>>>(p, tq, tdo, tk, tv);
    if (cudaGetLastError() != cudaSuccess) return -4;

    p.n_items = R.Hkv * p.n_tiles;
    auto kkv = bwd_dkdv_kernel<D>;
    if (cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kKvSmem) != cudaSuccess)
        return -4;
    kkv<<<p.n_items < sms ? p.n_items : sms, kThreads, C::kKvSmem, stream>>>(p, tq, tdo, tk, tv);
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
