// internal.h -- parameter blocks and launchers shared by the translation units of
// libringattn.so.  Not part of the public ABI (that is include/ringattn.h).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ra {

// ------------------------------------------------------------------ check build
// Index checks of the check build (compiled with -DRA_CHECK, libringattn_check.so): at every
// site where a kernel derives a memory index from the ring's chunk and work-item arithmetic
// (TMA row coordinates, output rows, document starts, source slabs), the index is checked
// against the tensor it addresses.  A failed check records RA_ERR_BOUNDS and the site
// number in the device error word (read with ringattn_sync_status / ringattn_last_timeout)
// and the access is skipped (a store), read as zero (a load) or moved to row 0 (a TMA load,
// so the pipeline's byte counts still complete); nothing traps.  In the normal build
// RA_CHECKED(cond, err, site) is `true` and the condition is not evaluated.
constexpr int kErrBounds = -6;  // RA_ERR_BOUNDS
enum CheckSite : int {
    kSiteFwdQRow = 1, kSiteFwdKvRow = 2, kSiteFwdOutRow = 3, kSiteFwdDocStart = 4,
    kSiteBwdQRow = 11, kSiteBwdKvRow = 12, kSiteBwdLseRow = 13, kSiteBwdGradRow = 14,
    kSitePermuteSlab = 21, kSiteRelayoutSrc = 31, kSiteF32Row = 41
};
#if defined(__CUDACC__) && defined(RA_CHECK)
__device__ __forceinline__ bool ra_check(bool ok, int* err, int site) {
    if (!ok && err) {
        atomicCAS(err, 0, kErrBounds);
        if (atomicCAS(err + 1, 0, 1) == 0) {
            err[2] = site;
            err[3] = static_cast<int>((blockIdx.x << 10) | threadIdx.x);
        }
    }
    return ok;
}
#define RA_CHECKED(cond, err, site) ::ra::ra_check((cond), (err), (site))
#else
#define RA_CHECKED(cond, err, site) true
#endif

// Ring geometry, fixed per call.
//   n_r  rows per rank (S / c);  m  rows per chunk (n_r, or n_r / 2 for zigzag);
//   nslot chunks per rank (1 or 2).  A rank's local row x lies in chunk slot x / m;
//   slot 0 holds natural chunk r, slot 1 (zigzag) natural chunk 2c-1-r.
struct Ring {
    int S, Hq, Hkv, g, d, c, causal, layout;
    int n_r, m, nslot;
    // messages visited: hops [hop_lo, hop_hi) and, inside each held block, local
    // key rows [kv_lo, kv_hi) (the whole block for the fused path)
    int hop_lo, hop_hi, kv_lo, kv_hi;
};

// How query tiles are grouped two by two onto the two softmax warpgroups of a CTA.
enum PairMode : int {
    kPairHeads = 0,      // two query heads of one KV group at the same position
    kPairPositions = 1,  // two adjacent 128-row tiles of one head, same chunk
    kSingles = 2         // one tile per work item
};

struct AttnBf16Params {
    Ring ring;
    int natural;    // 1: tensors in natural order (chunk map folded into addressing)
    int pair_mode;
    int rank_sel;   // -1: every rank's query rows; r >= 0: only virtual rank r's rows
    int n_tiles;    // 128-row query tiles per head (S / 128, or S / (128 c) for one rank)
    int n_items;
    int kv_group;   // KV heads per ordering group of work items (divides Hkv)
    // [2] item counter and finished-CTA counter in global memory: zero at launch; the
    // last CTA of the launch zeroes them again
    unsigned int* sched;
    float* out;
    float* lse;
    // document mask over all-gathered K/V: first natural position of the document of
    // every natural position (null: the ring, with or without the causal mask)
    const int* doc_start;
    int* err;
    unsigned long long timeout_ns;
};

// Backward pass (attn_bwd.cu): gradients of the fused forward, in the forward's layout.
struct AttnBwdParams {
    Ring ring;
    int natural;       // 1: tensors in natural order
    int n_tiles;       // 128-row tiles per head (S / 128)
    int n_items;       // dq kernel: Hq * n_tiles; dk/dv kernel: Hkv * n_tiles
    const float* lse;  // [Hq, S] natural log, from the forward
    const float* delta;  // [Hq, S] dout . out per row (bwd_delta_kernel)
    // [4] item counter and finished-CTA counter of the dq launch, then of the dk/dv launch
    // (global memory, zero at launch; the last CTA of each launch zeroes its pair again)
    unsigned int* sched;
    float* dq;
    float* dk;
    float* dv;
    int* err;
    unsigned long long timeout_ns;
};

struct AttnF32Params {
    Ring ring;
    int kv_block;
    int* err;  // device error word (check build)
    const float* q;
    const float* k;
    const float* v;
    float* out;
    float* lse;
};

int launch_attn_bf16(const AttnBf16Params& p, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, int grid, cudaStream_t stream);
int launch_attn_f32(const AttnF32Params& p, cudaStream_t stream);
int launch_permute(const void* src, void* dst, int S, int H, int row_bytes, int c, int layout, int inverse,
                   int* err, cudaStream_t stream);
int launch_merge(float* o_run, float* lse_run, const float* o_part, const float* lse_part, long long rows,
                 int d, cudaStream_t stream);
int launch_selftest_timeout(int* err, unsigned long long timeout_ns, cudaStream_t stream);
int launch_doc_start(const int* doc_id, int* doc_start, int S, cudaStream_t stream);
// Ulysses relayout between sequence-sharded [S, H, row] (rank-major tokens) and
// head-sharded [H, S, row] (natural tokens); relayout_fits checks the index ranges.
bool relayout_fits(long long S, int H, int row_bytes, int c, int layout);
int launch_relayout(const void* src, void* dst, int S, int H, int row_bytes, int c, int layout, int to_heads,
                    int* err, cudaStream_t stream);

int launch_attn_bwd(const AttnBwdParams& p, const float* out, const void* dout, const CUtensorMap& tq,
                    const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo, int sms,
                    cudaStream_t stream);

// Shared-memory footprint of the bf16 kernel for head dimension d.
size_t attn_bf16_smem_bytes(int d);

}  // namespace ra
