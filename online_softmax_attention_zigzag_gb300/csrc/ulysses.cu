// ulysses.cu -- the data movement of Ulysses' two all-to-alls, all c virtual ranks on
// one GPU ("Ring Attention and Ulysses shard a sequence two different ways...", section
// "Ulysses: an all-to-all relayout instead of a rotation": an all-to-all turns the
// sequence-sharded layout -- each rank its own tokens, every head -- into a head-sharded
// one -- each rank a subset of the heads over the whole sequence -- and a second one
// turns the attention's result back).
//
// With every rank on one GPU the ranks' shards sit side by side, so each all-to-all is
// one relayout of the whole tensor:
//   sequence-sharded  [S, H, row]  tokens in rank-major order (rank 0's tokens first; a
//                     zigzag rank holds natural chunk r, then chunk 2c-1-r), heads inner;
//   head-sharded      [H, S, row]  heads outer, tokens in natural order; rank r's share
//                     is the H/c consecutive heads [r H/c, (r+1) H/c).
// A row is one (token, head) vector of `row` bytes (d bf16 values, d fp32 values, or one
// fp32 lse).  The kernel walks the destination one chunk-sized slab at a time, so each
// source row address comes from one chunk-base lookup and a division by a constant.
#include "fastdiv.h"
#include "internal.h"

namespace ra {
namespace {

struct RelayoutArgs {
    long long S;          // tokens
    int H;                // heads
    int rowv;             // vectors per row
    int m;                // tokens per chunk
    int n_r;              // tokens per rank (m, or 2m for zigzag)
    int c, layout, to_heads;
    int nslab;            // destination slabs: H * chunks (to heads) or chunks (to sequence)
    unsigned slab_vecs;   // vectors per destination slab
    FastDiv div_rowv;     // by rowv
    FastDiv div_hrow;     // by H * rowv
    long long total_vecs; // vectors in the source tensor (check build)
    int* err;             // device error word (check build)
};

// Rank-major token index of the first token of natural chunk k.
__device__ __forceinline__ long long chunk_token_base(const RelayoutArgs& a, int k) {
    if (a.layout == 0) return static_cast<long long>(k) * a.m;
    return k < a.c ? static_cast<long long>(k) * a.n_r : static_cast<long long>(2 * a.c - 1 - k) * a.n_r + a.m;
}

// Grid: x = blocks sharing one slab, y = slab.  Four independent vectors per thread per
// iteration keep enough loads in flight to approach the copy bandwidth.
template <typename V>
__global__ void __launch_bounds__(256) relayout_kernel(const V* __restrict__ src, V* __restrict__ dst,
                                                       const RelayoutArgs a) {
    constexpr int kUnroll = 4;
    const int slab = blockIdx.y;
    long long dst_base, src_tok;  // dst vector offset of the slab; rank-major / natural token base
    int h = 0;
    if (a.to_heads) {
        // slab = (head h, natural chunk k): m rows of head h, contiguous in dst
        const int nch = a.nslab / a.H;
        h = slab / nch;
        const int k = slab - h * nch;
        dst_base = (static_cast<long long>(h) * a.S + static_cast<long long>(k) * a.m) * a.rowv;
        src_tok = chunk_token_base(a, k);
    } else {
        // slab = rank-major chunk j = (rank r, slot): m tokens x every head, contiguous in dst
        const int j = slab;
        const int r = a.layout == 1 ? j >> 1 : j;
        const int k = (a.layout == 1 && (j & 1)) ? 2 * a.c - 1 - r : r;
        dst_base = static_cast<long long>(j) * a.m * a.H * a.rowv;
        src_tok = static_cast<long long>(k) * a.m;  // natural position of the slab's first token
    }
    const unsigned stride = gridDim.x * blockDim.x;
    for (unsigned base = blockIdx.x * blockDim.x + threadIdx.x; base < a.slab_vecs; base += stride * kUnroll) {
        V vals[kUnroll];
        long long dsto[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const unsigned i = base + u * stride;
            dsto[u] = -1;
            if (i < a.slab_vecs) {
                long long s;
                if (a.to_heads) {
                    const unsigned row = fdiv(i, a.div_rowv);  // token within the chunk
                    const unsigned v = i - row * a.rowv;
                    s = ((src_tok + row) * a.H + h) * a.rowv + v;
                } else {
                    const unsigned row = fdiv(i, a.div_hrow);  // token within the chunk
                    const unsigned rem = i - row * a.H * a.rowv;
                    const unsigned hh = fdiv(rem, a.div_rowv);
                    const unsigned v = rem - hh * a.rowv;
                    s = (static_cast<long long>(hh) * a.S + src_tok + row) * a.rowv + v;
                }
                if (RA_CHECKED(s >= 0 && s < a.total_vecs, a.err, kSiteRelayoutSrc)) {
                    vals[u] = src[s];
                    dsto[u] = dst_base + i;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (dsto[u] >= 0) dst[dsto[u]] = vals[u];
    }
}

template <typename V>
int launch_relayout_v(const void* src, void* dst, RelayoutArgs a, cudaStream_t stream) {
    int dev = 0, sms = 152;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // about 8 CTAs of 256 threads per SM in total, but no more than the slab needs
    const long long per_block = 256LL * 4;
    long long bx = (static_cast<long long>(sms) * 8 + a.nslab - 1) / a.nslab;
    const long long need = (a.slab_vecs + per_block - 1) / per_block;
    if (bx > need) bx = need;
    if (bx < 1) bx = 1;
    dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(a.nslab));
    relayout_kernel<V><<<grid, 256, 0, stream>>>(static_cast<const V*>(src), static_cast<V*>(dst), a);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace

bool relayout_fits(long long S, int H, int row_bytes, int c, int layout) {
    if (S < 1 || H < 1 || c < 1 || row_bytes < 4 || row_bytes % 4 != 0) return false;
    const int nch = c * (layout == 1 ? 2 : 1);
    if (S % nch != 0) return false;
    const long long m = S / nch;
    // per-slab indices and the divisors are 31-bit even with 4-byte vectors (the kernel
    // falls back to them for unaligned buffers); slab counts fit a grid's y extent
    return m * H * (row_bytes / 4) < (1LL << 31) && static_cast<long long>(H) * nch < 65536;
}

int launch_relayout(const void* src, void* dst, int S, int H, int row_bytes, int c, int layout, int to_heads,
                    int* err, cudaStream_t stream) {
    const bool vec16 = row_bytes % 16 == 0 && (reinterpret_cast<uintptr_t>(src) & 15u) == 0 &&
                       (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
    RelayoutArgs a;
    const int nch = c * (layout == 1 ? 2 : 1);
    a.S = S;
    a.H = H;
    a.rowv = vec16 ? row_bytes / 16 : row_bytes / 4;
    a.m = S / nch;
    a.n_r = S / c;
    a.c = c;
    a.layout = layout;
    a.to_heads = to_heads;
    a.nslab = to_heads ? H * nch : nch;
    a.slab_vecs = static_cast<unsigned>(to_heads ? static_cast<long long>(a.m) * a.rowv
                                                 : static_cast<long long>(a.m) * H * a.rowv);
    a.div_rowv = make_fastdiv(static_cast<unsigned>(a.rowv));
    a.div_hrow = make_fastdiv(static_cast<unsigned>(H * a.rowv));
    a.total_vecs = static_cast<long long>(S) * H * a.rowv;
    a.err = err;
    if (a.slab_vecs == 0) return 0;
    return vec16 ? launch_relayout_v<uint4>(src, dst, a, stream) : launch_relayout_v<uint32_t>(src, dst, a, stream);
}

}  // namespace ra
