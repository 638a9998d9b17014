// attn_bf16.cu -- fused ring attention on the tcgen05 tensor cores of sm_103a.
//
// What it computes ("Ring Attention and Ulysses shard a sequence two different
// ways...", section "Ring Attention: point-to-point rotation, and an online softmax
// that never sees the whole row at once"): every virtual rank keeps its query rows
// fixed and visits the KV blocks in ring order -- hop h brings the block rank
// (r - h) mod c started with ("Interrogating parallelism, part 5", "How does
// attention survive being split?") -- folding each block into a running max, a
// running sum and a rescaled output.  Chunks are contiguous or zigzag (rank i holds
// chunks i and 2c-1-i, "What breaks the load balance?").  Under the causal mask,
// key tiles that lie wholly after a query tile are never visited.
//
// A second mode ("Interrogating parallelism, part 5", "Why did Llama 3 not use a
// ring?") takes the K/V of every rank as all-gathered and applies a document mask:
// keys are visited in natural order from the start of the earliest document the item
// touches, and a key is visible to a row when it lies between the start of the row's
// document and the row itself.
//
// Design (one CTA per SM, persistent, 352 threads):
//   * a work item is two 128-row query tiles (units) that share every K/V tile: two
//     query heads of one KV group at the same positions, or two adjacent tiles of one
//     head; items are listed by groups of KV heads, then by decreasing causal work, and
//     each CTA's loader draws the next one from a global counter when it needs it;
//   * warp 10 (one thread) streams Q tiles and, in visiting order, K and V tiles into
//     shared memory with TMA (128-byte swizzle), through a ring of stages guarded by
//     mbarriers; a stage pairs the V tile of one key tile with the K tile of the next,
//     which is what the MMA issuers consume together (one wait, one release per tile);
//   * warps 8 and 9 issue tcgen05.mma for units 0 and 1 (the whole warp runs the issuer,
//     keeping descriptors and counters warp-uniform; one elected lane issues each
//     instruction): S_x = Q_x K^T
//     into TMEM, and after softmax O_x += P_x V with P_x read from TMEM.  They take
//     turns batch by batch through a counter in shared memory, so the tensor pipe sees
//     each unit's batch whole while one issuer's waits and commits overlap the other's
//     batch;
//   * warps 0-7 are two softmax warpgroups, one per unit; thread t owns row t of its
//     unit and all 128 key columns of every score tile.  They read S from TMEM (with
//     loads that also return each thread's largest score, the row max of a tile no mask
//     touches), mask, update the running max and sums with exp2, write P (bf16) back to
//     TMEM (and hand it to the issuer: on a named barrier on the ring), rescale O
//     in TMEM when the running max rose by more than 2^8, and at the end write
//     out = O / (sum of the bf16 P) and lse = m + ln(sum of the exact p).
//   One unit's softmax overlaps the other unit's MMAs.
//
// TMEM (512 columns x 128 lanes, fp32): S_0 [0,128), S_1 [128,256) -- P_x is stored
// as packed bf16 pairs in the upper half of S_x's columns -- O_0 [256, 256+D),
// O_1 [256+D, 256+2D).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace ra {
namespace {

constexpr int kTile = 128;
constexpr int kThreads = 352;
constexpr int kPBar = 1;              // named barriers kPBar + x: unit x's P hand-off on the ring
constexpr int kPBarThreads = 4 * 32 + 32;  // its softmax warpgroup and its issuer warp
constexpr int kMmaWarp = 8, kLoadWarp = 10;  // warp 8 + x issues the MMAs of unit x
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kItemTakers = 10;  // work-item takers: 2 MMA issuers + 8 softmax warps
constexpr float kLn2 = 0.69314718055994531f;
// The running max used for P is only moved when the true max exceeds it by more
// than this (log2 units): P then stays below 2^8 and O needs no rescale otherwise.
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct Cfg {
    static constexpr int kTileBytes = kTile * D * 2;   // one 128 x D bf16 tile
    static constexpr int kBoxBytes = kTile * 64 * 2;   // one 128 x 64 TMA box (16 KB)
    static constexpr int kBoxes = D / 64;
    // A stage holds the V tile of one key tile and the K tile of the next (128 KB in all).
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kStages = (D == 128) ? 2 : 4;
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = 2 * kTileBytes;
    static constexpr int kBarOff = kKVOff + kStages * kStageBytes;
    static constexpr int kNumBars = 16 + 2 * kStages + 2 * kItemRing;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kRingOff = kMiscOff + 16;  // item ids handed from the loader to the other roles
    static constexpr int kSmemBytes = kRingOff + 4 * kItemRing + 1024;  // + slack to align the base
    static constexpr uint32_t kTmemCols = 512;
    static constexpr uint32_t kOCol = 256;
};

struct Bars {
    uint64_t* q_full;    // [2] loader -> mma (TMA bytes)
    uint64_t* q_empty;   // [2] mma -> loader (last S MMA of an item done)
    uint64_t* s_full;    // [2] mma -> softmax
    uint64_t* p_full;    // [2] softmax (128 threads) -> mma: all of P written (document mask; the
                         //     ring hands P over on named barrier kPBar + x instead)
    uint64_t* p_half;    // [2] softmax (128 threads) -> mma: P of keys [0, 64) written (and O rescaled)
    uint64_t* o_done;    // [2] mma -> softmax (last PV of an item done)
    uint64_t* o_free;    // [2] softmax (128 threads) -> mma (O read out)
    uint64_t* drain;     // [1] mma, on abort only
    uint64_t* kv_full;   // [stages]
    uint64_t* kv_empty;  // [stages]
    uint64_t* item_full;   // [kItemRing] loader -> issuers, softmax warps (item id written)
    uint64_t* item_empty;  // [kItemRing] issuers, softmax warps (one arrival each) -> loader
};

// A work item: up to two query tiles (units) of one rank that share a KV head.
struct Item {
    int hq[2];    // query head of each unit; hq[1] < 0 when the item has one unit
    int hk;       // KV head
    int pos[2];   // natural position of each unit's first row
    int r;        // virtual rank holding the units
    int qrow[2];  // row of each unit's first query in q / out / lse
    int pmax;     // last natural query position in the item
    int klo;      // document mask: first natural key position visited (a multiple of 128)
};

// Natural tile index of local tile t of rank r (local rows: chunk r, then for zigzag
// chunk 2c-1-r; "What breaks the load balance?").
__device__ __forceinline__ int rank_tile(const Ring& R, int r, int t) {
    const int x = t * kTile;
    const int slot = x / R.m;
    const int k = (slot == 0) ? r : 2 * R.c - 1 - r;
    return (k * R.m + (x - slot * R.m)) / kTile;
}

// Items are ordered KV-head-major (all of one KV head's items, then the next), and
// within a KV head by decreasing causal work (last query tiles first): the K/V tiles in
// use at any time are then one head's, which stay in L2, and the snake assignment of
// items to CTAs still deals out decreasing work.
template <bool DOC>
__device__ __forceinline__ void decode_item(const AttnBf16Params& p, int item, Item& it) {
    const Ring& R = p.ring;
    int t0, t1;
    // Items are grouped by KV heads (p.kv_group heads per group, chosen by the host so
    // that a group's K and V stay in L2); within a group, by decreasing causal work
    // (last query tiles first), then by head.  upk: items per (KV head, tile position).
    const int upk = (p.pair_mode == kPairHeads) ? R.g / 2 : (p.pair_mode == kPairPositions ? 1 : R.g);
    const int n_pi = (p.pair_mode == kPairPositions) ? p.n_tiles / 2 : p.n_tiles;
    const int per_pi = upk * p.kv_group;
    const int grp = item / (n_pi * per_pi), rem = item - grp * (n_pi * per_pi);
    const int pi = rem / per_pi, r2 = rem - pi * per_pi;
    it.hk = grp * p.kv_group + r2 / upk;
    const int u = r2 - (r2 / upk) * upk;
    if (p.pair_mode == kPairHeads) {
        t0 = t1 = p.n_tiles - 1 - pi;
        it.hq[0] = it.hk * R.g + 2 * u;
        it.hq[1] = it.hq[0] + 1;
    } else if (p.pair_mode == kPairPositions) {
        t1 = p.n_tiles - 1 - 2 * pi;
        t0 = t1 - 1;
        it.hq[0] = it.hq[1] = it.hk;  // one query head per KV head
    } else {
        t0 = t1 = p.n_tiles - 1 - pi;
        it.hq[0] = it.hk * R.g + u;
        it.hq[1] = -1;
    }
    if (p.rank_sel >= 0) {  // tile indices count one rank's local tiles: map them to natural tiles
        t0 = rank_tile(R, p.rank_sel, t0);
        t1 = rank_tile(R, p.rank_sel, t1);
    }
    it.pos[0] = t0 * kTile;
    it.pos[1] = t1 * kTile;
    // rank and local row of a natural position (both units share chunk and rank)
    int local0;
    if (R.layout == 1) {
        const int k = it.pos[0] / R.m;
        it.r = (k < R.c) ? k : 2 * R.c - 1 - k;
        local0 = ((k < R.c) ? 0 : R.m) + (it.pos[0] - k * R.m);
    } else {
        it.r = it.pos[0] / R.n_r;
        local0 = it.pos[0] - it.r * R.n_r;
    }
    const int local1 = local0 + (it.pos[1] - it.pos[0]);
    const int rbase = it.r * R.n_r;
    it.qrow[0] = it.hq[0] * R.S + (p.natural ? it.pos[0] : rbase + local0);
    it.qrow[1] = (it.hq[1] < 0) ? -1 : it.hq[1] * R.S + (p.natural ? it.pos[1] : rbase + local1);
    it.pmax = max(it.pos[0], it.pos[1]) + kTile - 1;
    // document mask: no key before the start of the document of the item's first row is
    // visible to any of its rows (starts do not decrease along the sequence)
    const int p0 = min(it.pos[0], it.pos[1]);
    it.klo = (DOC && RA_CHECKED(p0 >= 0 && p0 < R.S, p.err, kSiteFwdDocStart))
                 ? (__ldg(p.doc_start + p0) / kTile) * kTile
                 : 0;
}

// Row of natural key position pos of KV head hk in k / v (rank-major unless p.natural).
__device__ __forceinline__ int kv_row_of(const AttnBf16Params& p, int hk, int pos) {
    const Ring& R = p.ring;
    if (p.natural) return hk * R.S + pos;
    const int k = pos / R.m;                            // natural chunk
    const bool second = R.layout == 1 && k >= R.c;      // zigzag: the rank's second chunk
    const int s = second ? 2 * R.c - 1 - k : k;         // rank holding it
    return hk * R.S + s * R.n_r + (second ? R.m : 0) + (pos - k * R.m);
}

// Visit the item's key tiles in ring order: f(kv_row, key_pos).  kv_row is the row of
// the tile's first key in k / v; key_pos its natural position.
template <class F>
__device__ __forceinline__ void for_each_ring_tile(const AttnBf16Params& p, const Item& it, F&& f) {
    const Ring& R = p.ring;
    for (int hop = R.hop_lo; hop < R.hop_hi; ++hop) {
        int s = it.r - hop;
        if (s < 0) s += R.c;
        for (int slot = 0; slot < R.nslot; ++slot) {
            const int k = (slot == 0) ? s : 2 * R.c - 1 - s;  // natural chunk
            const int base = slot * R.m;                      // its first local row in the block
            const int lo = max(R.kv_lo, base);
            int hi = min(R.kv_hi, base + R.m);
            if (R.causal) hi = min(hi, base + max(0, it.pmax - k * R.m + 1));
            for (int x = lo; x < hi; x += kTile) {
                const int pos = k * R.m + (x - base);
                const int row = it.hk * R.S + (p.natural ? pos : s * R.n_r + x);
                if (!f(row, pos)) return;
            }
        }
    }
}

__device__ __forceinline__ int count_ring_tiles(const AttnBf16Params& p, const Item& it) {
    const Ring& R = p.ring;
    int n = 0;
    for (int hop = R.hop_lo; hop < R.hop_hi; ++hop) {
        int s = it.r - hop;
        if (s < 0) s += R.c;
        for (int slot = 0; slot < R.nslot; ++slot) {
            const int k = (slot == 0) ? s : 2 * R.c - 1 - s;
            const int base = slot * R.m;
            const int lo = max(R.kv_lo, base);
            int hi = min(R.kv_hi, base + R.m);
            if (R.causal) hi = min(hi, base + max(0, it.pmax - k * R.m + 1));
            if (hi > lo) n += (hi - lo + kTile - 1) / kTile;
        }
    }
    return n;
}

// With the document mask the K/V of every rank have been gathered: the keys are visited
// in natural order, from the item's first document start to its last row.
template <bool DOC, class F>
__device__ __forceinline__ void for_each_kv_tile(const AttnBf16Params& p, const Item& it, F&& f) {
    if constexpr (DOC) {
        for (int pos = it.klo; pos <= it.pmax; pos += kTile)
            if (!f(kv_row_of(p, it.hk, pos), pos)) return;
    } else {
        for_each_ring_tile(p, it, f);
    }
}

template <bool DOC>
__device__ __forceinline__ int count_kv_tiles(const AttnBf16Params& p, const Item& it) {
    if constexpr (DOC) {
        return (it.pmax + 1 - it.klo) / kTile;
    } else {
        return count_ring_tiles(p, it);
    }
}

// ------------------------------------------------------------------ TMA producer
// Stage sequence of an item with n key tiles: K(0); then V(j-1) with K(j) for j = 1..n-1;
// then V(n-1).  V sits at the stage base, K one tile above it.
template <int D, bool DOC>
__device__ void load_role(const AttnBf16Params& p, const CUtensorMap* tq, const CUtensorMap* tk,
                          const CUtensorMap* tv, uint8_t* sQ, uint8_t* sKV, const Bars& b, volatile int* ring,
                          const WaitCtl& wc) {
    using C = Cfg<D>;
    uint32_t st_idx = 0, qit[2] = {0, 0};
    bool ok = true;
    // K/V tiles are re-read by every query tile of their head group: keep them in L2;
    // Q tiles are read once: let them go first
    const uint64_t keep = make_policy_evict_last(), stream = make_policy_evict_first();
    // wait for the next stage to be empty and announce the bytes it will receive
    auto claim = [&](uint32_t bytes, uint32_t& s) -> bool {
        s = st_idx % C::kStages;
        if (!mbar_wait(&b.kv_empty[s], ((st_idx / C::kStages) & 1u) ^ 1u, wc, 32)) return false;
        mbar_arrive_expect_tx(&b.kv_full[s], bytes);
        ++st_idx;
        return true;
    };
    auto load_tile = [&](uint32_t s, int off, const CUtensorMap* map, int row) {
        if (!RA_CHECKED(row >= 0 && static_cast<long long>(row) + kTile <= static_cast<long long>(p.ring.Hkv) * p.ring.S,
                        p.err, kSiteFwdKvRow))
            row = 0;
        for (int bx = 0; bx < C::kBoxes; ++bx)
            tma_load_2d_hint(sKV + s * C::kStageBytes + off + bx * C::kBoxBytes, map, &b.kv_full[s], bx * 64, row,
                             keep);
    };
    for (uint32_t k = 0; ok; ++k) {
        // draw the next item and publish it (or the end of the sequence)
        const int item = publish_item(p.sched, p.n_items, b.item_full, b.item_empty, ring, k, wc);
        if (item == -2) { ok = false; break; }
        if (item < 0) break;
        Item it;
        decode_item<DOC>(p, item, it);
        if (count_kv_tiles<DOC>(p, it) == 0) continue;
        const int nx = (it.hq[1] >= 0) ? 2 : 1;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            if (x >= nx || !ok) break;
            if (!mbar_wait(&b.q_empty[x], (qit[x] & 1u) ^ 1u, wc, 32)) { ok = false; break; }
            ++qit[x];
            mbar_arrive_expect_tx(&b.q_full[x], C::kTileBytes);
            int qrow = x ? it.qrow[1] : it.qrow[0];
            if (!RA_CHECKED(qrow >= 0 && static_cast<long long>(qrow) + kTile <= static_cast<long long>(p.ring.Hq) * p.ring.S,
                            p.err, kSiteFwdQRow))
                qrow = 0;
#pragma unroll
            for (int bx = 0; bx < C::kBoxes; ++bx)
                tma_load_2d_hint(sQ + x * C::kTileBytes + bx * C::kBoxBytes, tq, &b.q_full[x], bx * 64, qrow, stream);
        }
        if (!ok) break;
        int prev = -1;  // row of the previous tile, whose V goes with this tile's K
        for_each_kv_tile<DOC>(p, it, [&](int row, int) -> bool {
            uint32_t s;
            if (!claim(prev < 0 ? C::kTileBytes : C::kStageBytes, s)) { ok = false; return false; }
            if (prev >= 0) load_tile(s, 0, tv, prev);
            load_tile(s, C::kTileBytes, tk, row);
            prev = row;
            return true;
        });
        if (!ok) break;
        uint32_t s;
        if (!claim(C::kTileBytes, s)) { ok = false; break; }
        load_tile(s, 0, tv, prev);
    }
    if (!ok) {
        // let every copy already issued land before the CTA's shared memory goes away
        for (uint32_t s = 0; s < (uint32_t)C::kStages && s < st_idx; ++s) {
            const uint32_t last = st_idx - 1 - ((st_idx - 1 - s) % C::kStages);
            drain_wait(&b.kv_full[s], (last / C::kStages) & 1u, wc.timeout_ns);
        }
        for (int x = 0; x < 2; ++x)
            if (qit[x] > 0) drain_wait(&b.q_full[x], (qit[x] - 1) & 1u, wc.timeout_ns);
    }
}

// ------------------------------------------------------------------ MMA issuer
// The two halves of a 128-byte-swizzle descriptor: the low word carries (address >> 4)
// and the leading byte offset, the high word the stride, version and swizzle, which are
// the same for every operand here.
__device__ __forceinline__ uint32_t sdesc_lo(uint32_t smem_addr, uint32_t lbo) {
    return ((smem_addr >> 4) & 0x3FFFu) | (((lbo >> 4) & 0x3FFFu) << 16);
}
constexpr uint32_t kSdescHi = (1024u >> 4) | (1u << 14) | (2u << 29);  // sbo 1024 B, version 1, 128 B swizzle

// Eight MMAs along K into one accumulator, descriptors stepped in their low words.
__device__ __forceinline__ void mma_ss8(uint32_t d_tmem, uint32_t alo, uint32_t blo, uint32_t idesc, uint32_t acc,
                                        uint32_t step_lo4, uint32_t step_box) {
    // K slice kk sits at byte offset (kk / 4) * box + (kk % 4) * 32
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk / 4) * step_box + (kk % 4) * step_lo4;
        asm volatile(
            "{\n\t.reg .b64 da, db;\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "mov.b64 da, {%1, %5};\n\tmov.b64 db, {%2, %5};\n\telect.sync _|e, 0xffffffff;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n\t}" ::"r"(d_tmem),
            "r"(alo + off), "r"(blo + off), "r"(idesc), "r"(kk > 0 ? 1u : acc), "r"(kSdescHi)
            : "memory");
    }
}

template <int D>
__device__ __forceinline__ void issue_s(uint32_t tmem, int x, uint32_t q_base, uint32_t k_base) {
    using C = Cfg<D>;
    static_assert(D == 128 || D == 64, "head dimension");
    constexpr uint32_t idesc = idesc_bf16(kTile, kTile, 0);
    const uint32_t d_tmem = tmem + x * kTile;
    const uint32_t qlo = sdesc_lo(q_base, 16), klo = sdesc_lo(k_base, 16);
    if constexpr (D == 128) {
        mma_ss8(d_tmem, qlo, klo, idesc, 0u, 32 >> 4, C::kBoxBytes >> 4);
    } else {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint32_t off = (kk * 32) >> 4;
            const uint64_t qa = (static_cast<uint64_t>(kSdescHi) << 32) | (qlo + off);
            const uint64_t kb = (static_cast<uint64_t>(kSdescHi) << 32) | (klo + off);
            asm volatile(
                "{\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
                "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                "l"(qa), "l"(kb), "r"(idesc), "r"(kk > 0 ? 1u : 0u)
                : "memory");
        }
    }
}

template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tmem, int x, uint32_t v_base, bool accumulate) {
    using C = Cfg<D>;
    constexpr uint32_t idesc = idesc_bf16(kTile, D, 1);
    const uint32_t d_tmem = tmem + C::kOCol + x * D;
    const uint32_t a_tmem = tmem + x * kTile + 64;
    const uint32_t vlo = sdesc_lo(v_base, C::kBoxBytes);
    const uint32_t acc = accumulate ? 1u : 0u;
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk) {
        asm volatile(
            "{\n\t.reg .b64 db;\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "mov.b64 db, {%2, %5};\n\telect.sync _|e, 0xffffffff;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %3, p;\n\t}" ::"r"(d_tmem),
            "r"(a_tmem + kk * 8), "r"(vlo + ((kk * 16 * 128) >> 4)), "r"(idesc), "r"(kk > 0 ? 1u : acc),
            "r"(kSdescHi)
            : "memory");
    }
}

template <int D, int K0, int K1>
__device__ __forceinline__ void issue_pv_part(uint32_t tmem, int x, uint32_t v_base, bool accumulate) {
    using C = Cfg<D>;
    constexpr uint32_t idesc = idesc_bf16(kTile, D, 1);
    const uint32_t d_tmem = tmem + C::kOCol + x * D;
    const uint32_t a_tmem = tmem + x * kTile + 64;
    const uint32_t vlo = sdesc_lo(v_base, C::kBoxBytes);
    const uint32_t acc = accumulate ? 1u : 0u;
#pragma unroll
    for (int kk = K0; kk < K1; ++kk) {
        asm volatile(
            "{\n\t.reg .b64 db;\n\t.reg .pred p, e;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "mov.b64 db, {%2, %5};\n\telect.sync _|e, 0xffffffff;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %3, p;\n\t}" ::"r"(d_tmem),
            "r"(a_tmem + kk * 8), "r"(vlo + ((kk * 16 * 128) >> 4)), "r"(idesc), "r"(kk > 0 ? 1u : acc),
            "r"(kSdescHi)
            : "memory");
    }
}

// Wait until `turn` reaches `mine` (bounded: gives up on abort or after the timeout).
__device__ __forceinline__ bool wait_turn(volatile uint32_t* turn, uint32_t mine, const WaitCtl& wc) {
    if (*turn == mine) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 1;; ++i) {
        if (*turn == mine) return true;
        if ((i & 255u) == 0u) {
            if (*wc.abort_flag) return false;
            if (globaltimer_ns() - t0 > wc.timeout_ns) {
                raise_abort(wc, reinterpret_cast<uint64_t*>(const_cast<uint32_t*>(turn)));
                return false;
            }
        }
    }
}

// One issuer warp per unit x (run by the whole warp; tcgen05 instructions from one elected
// lane, which tcgen05.commit tracks).  The two issuers take turns batch by batch (a batch is
// the MMAs one unit issues between two softmax hand-offs), so the tensor pipe sees the
// units' batches whole and in the order of the single-issuer schedule, while each
// issuer's waits and commits overlap the other's batch.  `turn` counts the batches
// issued so far; both issuers derive every batch's number from the item sequence.
// Each K/V stage is released once per issuer (the barrier counts two): by a commit after
// the unit's last MMA on it, or, in an item without a unit 1, by issuer 1's plain
// arrival once the stage is loaded, which keeps both within one phase of every stage.
template <int D, bool DOC>
__device__ void mma_role(const AttnBf16Params& p, int x, uint8_t* sQ, uint8_t* sKV, const Bars& b, uint32_t tmem,
                         volatile uint32_t* turn, const volatile int* ring, const WaitCtl& wc) {
    using C = Cfg<D>;
    const uint32_t sQa = smem_u32(sQ) + x * C::kTileBytes, sKVa = smem_u32(sKV);
    uint32_t st_idx = 0, qit = 0, pit = 0, seq = 0;
    bool ok = true;
    auto wait_stage = [&](uint32_t& s, uint32_t& base) -> bool {
        s = st_idx % C::kStages;
        base = sKVa + s * C::kStageBytes;
        const bool r = mbar_wait_w(&b.kv_full[s], (st_idx / C::kStages) & 1u, wc);
        ++st_idx;
        return r;
    };
    for (uint32_t k = 0; ok; ++k) {
        const int item = take_item(b.item_full, b.item_empty, ring, k, (threadIdx.x & 31) == 0, wc);
        if (item == -2) { ok = false; break; }
        if (item < 0) break;
        Item it;
        decode_item<DOC>(p, item, it);
        const int nj = count_kv_tiles<DOC>(p, it);
        if (nj == 0) continue;
        const int nx = (it.hq[1] >= 0) ? 2 : 1;
        if (x >= nx) {  // no unit 1: pass every stage of the item
            for (int i = 0; i <= nj && ok; ++i) {
                uint32_t s, base;
                if (!wait_stage(s, base)) { ok = false; break; }
                if ((threadIdx.x & 31) == 0) mbar_arrive(&b.kv_empty[s]);
            }
            seq += 1 + nj;
            continue;
        }
        // batch numbers: S(0) of unit x is seq + x, tile j of unit x is seq + nx (j + 1) + x
        if (!mbar_wait_w(&b.q_full[x], qit & 1u, wc)) { ok = false; break; }
        uint32_t s, base;
        if (!wait_stage(s, base)) { ok = false; break; }
        if (!__all_sync(0xffffffffu, wait_turn(turn, seq + x, wc))) { ok = false; break; }
        tc_fence_after();
        issue_s<D>(tmem, x, sQa, base + C::kTileBytes);
        mma_commit_e(&b.s_full[x]);
        *turn = seq + x + 1;
        mma_commit_e(&b.kv_empty[s]);
        if (nj == 1) mma_commit_e(&b.q_empty[x]);
        for (int j = 0; j < nj && ok; ++j) {
            // this stage holds V(j) and, unless j is the last tile, K(j+1)
            if (!wait_stage(s, base)) { ok = false; break; }
            // Under the document mask items are short, and P of the tile's first 64 keys
            // goes into O while the softmax finishes the rest; in the ring, all of P at once.
            // Each check reads shared memory, which the tensor core's operand reads keep busy
            // (~130 cycles even when already satisfied), so the one expected to be satisfied
            // comes first and the last arrival leads straight to the issue: on the ring the
            // other unit's batch is usually queued before this unit's P is written; under the
            // document mask (short items) it is usually the other way round.
            const uint32_t mine = seq + nx * (j + 1) + x;
            if constexpr (DOC) {
                if (!mbar_wait_w(&b.p_half[x], pit & 1u, wc)) { ok = false; break; }
                if (j == 0 && !mbar_wait_w(&b.o_free[x], (qit & 1u) ^ 1u, wc)) { ok = false; break; }
                if (!__all_sync(0xffffffffu, wait_turn(turn, mine, wc))) { ok = false; break; }
            } else {
                if (!__all_sync(0xffffffffu, wait_turn(turn, mine, wc))) { ok = false; break; }
                if (j == 0 && !mbar_wait_w(&b.o_free[x], (qit & 1u) ^ 1u, wc)) { ok = false; break; }
                // P on the unit's named barrier: the hardware releases the issuer as the last
                // softmax warp arrives, sooner than an mbarrier's wake (1-3% on the ring).  It
                // cannot time out: it is entered only while no role has given up, after S(j) was
                // queued, and the softmax arrives for every tile whose S it sees (see there).
                if (__any_sync(0xffffffffu, *wc.abort_flag != 0)) { ok = false; break; }
                named_bar_sync(kPBar + x, kPBarThreads);
            }
            tc_fence_after();
            if constexpr (DOC) {
                issue_pv_part<D, 0, kTile / 32>(tmem, x, base, j > 0);
                if (!mbar_wait_w(&b.p_full[x], pit & 1u, wc)) { ok = false; break; }
                tc_fence_after();
                issue_pv_part<D, kTile / 32, kTile / 16>(tmem, x, base, true);
            } else {
                issue_pv<D>(tmem, x, base, j > 0);
            }
            ++pit;
            if (j + 1 < nj) {
                issue_s<D>(tmem, x, sQa, base + C::kTileBytes);
                mma_commit_e(&b.s_full[x]);
            } else {
                mma_commit_e(&b.o_done[x]);
            }
            *turn = mine + 1;
            mma_commit_e(&b.kv_empty[s]);
            if (j + 2 == nj) mma_commit_e(&b.q_empty[x]);
        }
        seq += nx * (nj + 1);
        ++qit;
    }
    if (!ok) {
        // every MMA this warp issued must finish before TMEM is released
        mma_commit_e(&b.drain[x]);
        drain_wait(&b.drain[x], 0, wc.timeout_ns);
    }
}

// ------------------------------------------------------------------ softmax warpgroups
// Warpgroup x owns query tile x; thread t owns row t (TMEM lane t) and all 128 key
// columns of every score tile, so a row's max and sums never leave its thread.  Each
// warp waits on the tile's barriers by itself: the warps of a warpgroup share nothing
// but the arrival that hands P to the MMA issuer.
template <int D, bool DOC>
__device__ void softmax_role(const AttnBf16Params& p, int x, const Bars& b, uint32_t tmem, const volatile int* ring,
                             const WaitCtl& wc) {
    using C = Cfg<D>;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_tmem = tmem + lane_off + x * kTile;       // 128 score columns
    const uint32_t p_tmem = s_tmem + 64;                        // 64 packed P columns over S's upper half
    const uint32_t o_tmem = tmem + lane_off + C::kOCol + x * D;
    const bool causal = p.ring.causal != 0;
    uint32_t sit = 0, iit = 0;
    bool ok = true;
    // On the ring the issuer waits for P on a hardware named barrier, which cannot time out.
    // These warps arrive on it for every tile whose S the issuer queued (that S completes),
    // and the issuer queues S(j+1) only after taking P(j), so no phase gets a second
    // arrival; their waits ignore the abort flag and give up only on their own time limit,
    // which S the issuer queued cannot reach, so the issuer is never left without P.
    constexpr bool kFlagAware = DOC;
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        return __all_sync(0xffffffffu, kFlagAware ? mbar_wait(bar, parity, wc) : mbar_wait_noabort(bar, parity, wc));
    };
    for (uint32_t k = 0; ok; ++k) {
        const int item = take_item(b.item_full, b.item_empty, ring, k, lane == 0, wc, kFlagAware);
        if (__any_sync(0xffffffffu, item == -2)) {
            ok = false;
            break;
        }
        if (item < 0) break;
        Item it;
        decode_item<DOC>(p, item, it);
        const int my_hq = x ? it.hq[1] : it.hq[0];
        if (my_hq < 0) continue;
        const int nj = count_kv_tiles<DOC>(p, it);
        const size_t grow = static_cast<size_t>((x ? it.qrow[1] : it.qrow[0]) + row);
        float* orow = p.out + grow * D;
        const bool row_ok =
            RA_CHECKED(grow < static_cast<size_t>(p.ring.Hq) * p.ring.S, p.err, kSiteFwdOutRow);
        if (nj == 0) {  // a message with no visible key for this tile
            if (row_ok) {
                float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int i = 0; i < D / 4; ++i) reinterpret_cast<float4*>(orow)[i] = z;
                p.lse[grow] = -INFINITY;
            }
            continue;
        }
        const int tpos = x ? it.pos[1] : it.pos[0];
        const int qpos = tpos + row;
        // first key of my document
        const int doc_lo =
            (DOC && RA_CHECKED(qpos >= 0 && qpos < p.ring.S, p.err, kSiteFwdDocStart)) ? __ldg(p.doc_start + qpos) : 0;
        // l: sum of the exact p (for lse); lr: sum of p as rounded to bf16 for the P V
        // product, so that out = O / lr weighs every key consistently (a key that
        // dominates the row then comes out exactly, whatever its rounding)
        float m = -INFINITY, l = 0.f, lr = 0.f;
        int j = 0;
        for_each_kv_tile<DOC>(p, it, [&](int, int kpos) -> bool {
            if (!wait(&b.s_full[x], sit & 1u)) {
                ok = false;
                return false;
            }
            ++sit;
            tc_fence_after();
            float s[kTile];
            float pm0, pm1, pm2, pm3;  // the largest score of each 32-column load
            {
                uint32_t r0[32], r1[32], r2[32], r3[32];
                tmem_ld32_max(s_tmem + 0, r0, pm0);
                tmem_ld32_max(s_tmem + 32, r1, pm1);
                tmem_ld32_max(s_tmem + 64, r2, pm2);
                tmem_ld32_max(s_tmem + 96, r3, pm3);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    s[i] = __uint_as_float(r0[i]);
                    s[32 + i] = __uint_as_float(r1[i]);
                    s[64 + i] = __uint_as_float(r2[i]);
                    s[96 + i] = __uint_as_float(r3[i]);
                }
            }
            bool masked = false;
            if constexpr (DOC) {
                // my keys [lo, hi] are visible: my document's start up to my own position
                const int hi = qpos - kpos, lo = doc_lo - kpos;
                if (lo > 0 || hi < kTile - 1) {
                    masked = true;
#pragma unroll
                    for (int i = 0; i < kTile; ++i) s[i] = (i > hi || i < lo) ? -INFINITY : s[i];
                }
            } else if (causal && kpos + kTile - 1 > tpos) {  // the tile may cross the diagonal
                masked = true;
                const int lim = qpos - kpos;                  // my keys [0, lim] are visible
#pragma unroll
                for (int i = 0; i < kTile; ++i) s[i] = (i > lim) ? -INFINITY : s[i];
            }
            // row max: from the loads themselves unless some score of the warp was masked
            float mx = fmaxf(fmaxf(pm0, pm1), fmaxf(pm2, pm3));
            if (__any_sync(0xffffffffu, masked)) {
                float c[8];
#pragma unroll
                for (int a = 0; a < 8; ++a) c[a] = fmaxf(s[2 * a], s[2 * a + 1]);
#pragma unroll
                for (int i = 16; i < kTile; i += 16)
#pragma unroll
                    for (int a = 0; a < 8; ++a) c[a] = fmax3(c[a], s[i + 2 * a], s[i + 2 * a + 1]);
                mx = fmaxf(fmax3(c[0], c[1], c[2]), fmax3(c[3], c[4], fmax3(c[5], c[6], c[7])));
            }
            const float m_new = fmaxf(m, mx * kLog2e);
            float f = 1.f;
            bool need = false;
            if (j == 0) {
                m = m_new;
            } else if (m_new > m + kRescaleLog2) {
                need = true;
                f = ex2(m - m_new);
                l *= f;
                lr *= f;
                m = m_new;
            }
            const float nmu = (m == -INFINITY) ? 0.f : -m;
            // per-tile partial sums of p: two packed pairs under the document mask, one on the
            // ring, whose softmax then needs no spill slot (measured: each is the faster there)
            constexpr int kAcc = DOC ? 4 : 2;
            float se[kAcc] = {}, sr[kAcc] = {};
            // P goes to TMEM in four stores of 16 columns (32 keys each): a 16-word packing
            // buffer keeps the softmax within its registers, where two 32-word ones spilled
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float t0, t1;
                    ffma2(t0, t1, s[qq * 32 + 2 * i], s[qq * 32 + 2 * i + 1], kLog2e, kLog2e, nmu, nmu);
                    const float a = ex2(t0), c2 = ex2(t1);
                    const int q2 = DOC ? 2 * (i & 1) : 0;
                    fadd2(se[q2], se[q2 + 1], se[q2], se[q2 + 1], a, c2);
                    pk[i] = pack_bf16x2(a, c2);
                    add_bf16x2_f32(sr[q2], sr[q2 + 1], pk[i]);
                }
                // every score is in registers: P may overwrite S's upper half
                tmem_st16(p_tmem + qq * 16, pk);
                if (DOC && qq == 1) {  // hand the first 64 keys' P (and a rescaled O) over at once
                    // O is stable here: the commit that signalled this S also covered the
                    // previous P V, and this tile's P V waits for this arrival.
                    if (__any_sync(0xffffffffu, need)) {
#pragma unroll
                        for (int cc = 0; cc < D; cc += 32) {
                            uint32_t o0[32];
                            tmem_ld32(o_tmem + cc, o0);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) o0[i] = __float_as_uint(__uint_as_float(o0[i]) * f);
                            tmem_st32(o_tmem + cc, o0);
                        }
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&b.p_half[x]);
                }
            }
            if constexpr (!DOC) {
                // O is stable here: the commit that signalled this S also covered the
                // previous P V, and the next P V waits for this tile's arrivals.
                if (__any_sync(0xffffffffu, need)) {
#pragma unroll
                    for (int cc = 0; cc < D; cc += 32) {
                        uint32_t o0[32];
                        tmem_ld32(o_tmem + cc, o0);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o0[i] = __float_as_uint(__uint_as_float(o0[i]) * f);
                        tmem_st32(o_tmem + cc, o0);
                    }
                }
            }
            if constexpr (DOC) {
                l += (se[0] + se[1]) + (se[2] + se[3]);
                lr += (sr[0] + sr[1]) + (sr[2] + sr[3]);
            } else {
                l += se[0] + se[1];
                lr += sr[0] + sr[1];
            }
            tmem_wait_st();
            tc_fence_before();
            if constexpr (DOC) {
                mbar_arrive(&b.p_full[x]);
            } else {
                named_bar_arrive(kPBar + x, kPBarThreads);
            }
            ++j;
            return true;
        });
        if (!ok) break;
        // epilogue: out = O / lr, lse = m + log2(l), both in natural-log units
        if (!wait(&b.o_done[x], iit & 1u)) {
            ok = false;
            break;
        }
        ++iit;
        tc_fence_after();
        const float inv = (lr > 0.f) ? 1.f / lr : 0.f;
        const uint64_t out_policy = make_policy_evict_first();  // written once, read by the host
        // read all of O, hand its columns back, then store: 32-byte stores when `out` allows
        float o[D];
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
            uint32_t r[32];
            tmem_ld32(o_tmem + cc, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[cc + i] = __uint_as_float(r[i]);
        }
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&b.o_free[x]);
#pragma unroll
        for (int i = 0; i < D; ++i) o[i] *= inv;
        if (!row_ok) continue;
        if ((reinterpret_cast<uintptr_t>(p.out) & 31u) == 0u) {
#pragma unroll
            for (int i = 0; i < D; i += 8) {
                float w8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) w8[e] = o[i + e];
                st_stream_f8(orow + i, w8, out_policy);
            }
        } else {
            float4* dst = reinterpret_cast<float4*>(orow);
#pragma unroll
            for (int i = 0; i < D / 4; ++i)
                st_stream_f4(dst + i, make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]), out_policy);
        }
        p.lse[grow] = (l > 0.f) ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
}

template <int D, bool DOC>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bf16_kernel(const __grid_constant__ AttnBf16Params p, const __grid_constant__ CUtensorMap tq,
                     const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sQ = smem + C::kQOff;
    uint8_t* sKV = smem + C::kKVOff;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    Bars b;
    b.q_full = bars + 0;
    b.q_empty = bars + 2;
    b.s_full = bars + 4;
    b.p_full = bars + 6;
    b.o_done = bars + 8;
    b.o_free = bars + 10;
    b.drain = bars + 12;
    b.kv_full = bars + 14;
    b.kv_empty = bars + 14 + C::kStages;
    b.item_full = bars + 14 + 2 * C::kStages;
    b.item_empty = bars + 14 + 2 * C::kStages + kItemRing;
    b.p_half = bars + 14 + 2 * C::kStages + 2 * kItemRing;
    volatile int* ring = reinterpret_cast<volatile int*>(smem + C::kRingOff);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);
    volatile uint32_t* turn = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff + 8);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int x = 0; x < 2; ++x) {
            mbar_init(&b.q_full[x], 1);
            mbar_init(&b.q_empty[x], 1);
            mbar_init(&b.s_full[x], 1);
            mbar_init(&b.p_full[x], 128);
            mbar_init(&b.p_half[x], 128);
            mbar_init(&b.o_done[x], 1);
            mbar_init(&b.o_free[x], 128);
        }
        mbar_init(&b.drain[0], 1);
        mbar_init(&b.drain[1], 1);
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&b.kv_full[s], 1);
            mbar_init(&b.kv_empty[s], 2);  // released once by each unit's issuer
        }
        for (int s = 0; s < kItemRing; ++s) {
            mbar_init(&b.item_full[s], 1);
            mbar_init(&b.item_empty[s], kItemTakers);
        }
        *abort_flag = 0;
        *turn = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == kLoadWarp && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl wc{abort_flag, p.err, p.timeout_ns};

    // warps 0-7: two softmax warpgroups, warpgroup x = warp / 4 owns unit x (full rows);
    // warps 8 and 9 issue the MMAs of units 0 and 1; warp 10 loads
    if (warp < 8) {
        softmax_role<D, DOC>(p, warp / 4, b, tmem, ring, wc);
    } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
        mma_role<D, DOC>(p, warp - kMmaWarp, sQ, sKV, b, tmem, turn, ring, wc);
    } else if (warp == kLoadWarp) {
        if (lane == 0) load_role<D, DOC>(p, &tq, &tk, &tv, sQ, sKV, b, ring, wc);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, C::kTmemCols);
    if (threadIdx.x == 0) finish_items(p.sched);
}

template <int D, bool DOC>
int launch_d(const AttnBf16Params& p, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
             int grid, cudaStream_t stream) {
    using C = Cfg<D>;
    auto kern = attn_bf16_kernel<D, DOC>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
        return -4;
    kern<<<grid, kThreads, C::kSmemBytes, stream>>>(p, tq, tk, tv);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace

size_t attn_bf16_smem_bytes(int d) {
    return d == 128 ? Cfg<128>::kSmemBytes : Cfg<64>::kSmemBytes;
}

int launch_attn_bf16(const AttnBf16Params& p, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, int grid, cudaStream_t stream) {
    const bool doc = p.doc_start != nullptr;
    if (p.ring.d == 128) return doc ? launch_d<128, true>(p, tq, tk, tv, grid, stream)
                                    : launch_d<128, false>(p, tq, tk, tv, grid, stream);
    if (p.ring.d == 64) return doc ? launch_d<64, true>(p, tq, tk, tv, grid, stream)
                                   : launch_d<64, false>(p, tq, tk, tv, grid, stream);
    return -2;
}

}  // namespace ra
