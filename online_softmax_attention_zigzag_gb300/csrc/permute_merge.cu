// permute_merge.cu -- the HBM-bound kernels of the path:
//   * chunk permutation between natural and rank-major order (contiguous: identity
//     map of c chunks; zigzag: natural chunk k of 2c goes to rank k if k < c, else to
//     rank 2c-1-k as its second chunk -- "Interrogating parallelism, part 5", "What
//     breaks the load balance?");
//   * the exact (O, LSE) merge of a ring message's partial into a running result
//     (same page, "How does attention survive being split?");
//   * a self-test kernel whose only wait is never satisfied and runs out.
#include "internal.h"
#include "ptx.cuh"

namespace ra {
namespace {

// ------------------------------------------------------------------ permutation
// The tensor is H * nchunks slabs of `slab` bytes; a chunk moves whole, so the copy is one
// contiguous slab-to-slab copy per destination slab.  Grid: y (and z) = destination slab,
// x = blocks sharing it; four independent vectors per thread per iteration keep enough
// loads in flight to approach the copy bandwidth.
template <typename V>
__global__ void __launch_bounds__(256) permute_kernel(const V* __restrict__ src, V* __restrict__ dst,
                                                      long long slab_vecs, int nchunks, int c, int layout,
                                                      int inverse, long long nslabs, int* err) {
    constexpr int kUnroll = 4;
    const long long slab = static_cast<long long>(blockIdx.z) * gridDim.y + blockIdx.y;
    if (slab >= nslabs) return;
    const long long h = slab / nchunks;
    const int dslab = static_cast<int>(slab - h * nchunks);
    // natural chunk <-> rank-major chunk
    int sslab;
    if (layout == 1) {
        if (!inverse) {  // dst is rank-major: rank-major chunk j = 2r + slot
            const int r = dslab >> 1, slot = dslab & 1;
            sslab = slot ? 2 * c - 1 - r : r;
        } else {         // dst is natural chunk k
            const int k = dslab;
            sslab = (k < c) ? 2 * k : 2 * (2 * c - 1 - k) + 1;
        }
    } else {
        sslab = dslab;
    }
    if (!RA_CHECKED(sslab >= 0 && sslab < nchunks, err, kSitePermuteSlab)) return;
    const V* sp = src + (h * nchunks + sslab) * slab_vecs;
    V* dp = dst + slab * slab_vecs;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long base = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; base < slab_vecs;
         base += stride * kUnroll) {
        V vals[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const long long i = base + u * stride;
            if (i < slab_vecs) vals[u] = sp[i];
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const long long i = base + u * stride;
            if (i < slab_vecs) dp[i] = vals[u];
        }
    }
}

template <typename V>
int launch_permute_v(const void* src, void* dst, long long slab_bytes, int H, int nchunks, int c, int layout,
                     int inverse, int* err, cudaStream_t stream) {
    const long long slab_vecs = slab_bytes / static_cast<long long>(sizeof(V));
    const long long nslabs = static_cast<long long>(H) * nchunks;
    if (slab_vecs == 0 || nslabs == 0) return 0;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // about 8 CTAs of 256 threads per SM in total, but no more than a slab needs
    const long long per_block = 256LL * 4;
    long long bx = (static_cast<long long>(sms) * 8 + nslabs - 1) / nslabs;
    const long long need = (slab_vecs + per_block - 1) / per_block;
    if (bx > need) bx = need;
    if (bx < 1) bx = 1;
    const long long gy = nslabs < 65535 ? nslabs : 65535;
    const long long gz = (nslabs + gy - 1) / gy;
    if (gz > 65535) return -2;
    dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(gy), static_cast<unsigned>(gz));
    permute_kernel<V><<<grid, 256, 0, stream>>>(static_cast<const V*>(src), static_cast<V*>(dst), slab_vecs, nchunks,
                                               c, layout, inverse, nslabs, err);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// ------------------------------------------------------------------ merge
__device__ __forceinline__ float mix(float x, float wa, bool use_a, float y, float wb, bool use_b) {
    return (use_a ? x * wa : 0.f) + (use_b ? y * wb : 0.f);
}

// One warp per row at a time; the lanes stride over the row.  Every lane reads
// lse_run before the warp synchronises and lane 0 overwrites it, so the in-place
// update never races.
template <bool kVec4>
__global__ void __launch_bounds__(256) merge_kernel(float* __restrict__ o_run, float* __restrict__ lse_run,
                                                    const float* __restrict__ o_part,
                                                    const float* __restrict__ lse_part, long long rows, int d) {
    const int lane = threadIdx.x & 31;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
    for (long long row = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32; row < rows;
         row += warps) {
        const float a = lse_run[row];
        const float b = lse_part[row];
        const float M = fmaxf(a, b);
        float wa, wb, lse;
        if (M == -INFINITY) {  // neither partial saw a key
            wa = 0.f;
            wb = 0.f;
            lse = -INFINITY;
        } else {
            const float ea = expf(a - M), eb = expf(b - M);  // exp(-inf) = 0: weight 0
            const float tot = ea + eb;
            wa = ea / tot;
            wb = eb / tot;
            lse = M + logf(tot);
        }
        // a side with no key contributes exactly nothing, whatever its o holds
        const bool use_a = a != -INFINITY, use_b = b != -INFINITY;
        const size_t base = static_cast<size_t>(row) * d;
        if (kVec4) {
            float4* orun = reinterpret_cast<float4*>(o_run + base);
            const float4* opart = reinterpret_cast<const float4*>(o_part + base);
            for (int i = lane; i < d / 4; i += 32) {
                const float4 x = orun[i], y = opart[i];
                orun[i] = make_float4(mix(x.x, wa, use_a, y.x, wb, use_b), mix(x.y, wa, use_a, y.y, wb, use_b),
                                      mix(x.z, wa, use_a, y.z, wb, use_b), mix(x.w, wa, use_a, y.w, wb, use_b));
            }
        } else {
            for (int i = lane; i < d; i += 32)
                o_run[base + i] = mix(o_run[base + i], wa, use_a, o_part[base + i], wb, use_b);
        }
        __syncwarp();
        if (lane == 0) lse_run[row] = lse;
    }
}

// d = 128 (one float4 of each row per lane): a warp takes R consecutive rows per iteration
// and issues every load of them before any arithmetic, so 2R independent 16-byte loads per
// lane are in flight (one row at a time left the merge latency-bound at ~71% of HBM).
template <int R>
__global__ void __launch_bounds__(256) merge_kernel_d128(float4* __restrict__ o_run, float* __restrict__ lse_run,
                                                         const float4* __restrict__ o_part,
                                                         const float* __restrict__ lse_part, long long rows) {
    const int lane = threadIdx.x & 31;
    const long long warp = static_cast<long long>(blockIdx.x) * (blockDim.x / 32) + threadIdx.x / 32;
    const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x / 32);
    for (long long r0 = warp * R; r0 < rows; r0 += warps * R) {
        float4 x[R], y[R];
        float a[R], b[R];
#pragma unroll
        for (int k = 0; k < R; ++k) {
            const long long row = r0 + k;
            if (row < rows) {
                a[k] = lse_run[row];
                b[k] = lse_part[row];
                x[k] = o_run[row * 32 + lane];
                y[k] = o_part[row * 32 + lane];
            }
        }
        float lse_new = 0.f;  // lane k keeps row r0 + k's result
#pragma unroll
        for (int k = 0; k < R; ++k) {
            const long long row = r0 + k;
            if (row >= rows) break;
            const float M = fmaxf(a[k], b[k]);
            float wa = 0.f, wb = 0.f, lse = -INFINITY;
            if (M != -INFINITY) {  // else neither partial saw a key
                const float ea = expf(a[k] - M), eb = expf(b[k] - M);  // exp(-inf) = 0: weight 0
                const float tot = ea + eb;
                wa = ea / tot;
                wb = eb / tot;
                lse = M + logf(tot);
            }
            // a side with no key contributes exactly nothing, whatever its o holds
            const bool ua = a[k] != -INFINITY, ub = b[k] != -INFINITY;
            o_run[row * 32 + lane] = make_float4(mix(x[k].x, wa, ua, y[k].x, wb, ub), mix(x[k].y, wa, ua, y[k].y, wb, ub),
                                                 mix(x[k].z, wa, ua, y[k].z, wb, ub), mix(x[k].w, wa, ua, y[k].w, wb, ub));
            if (lane == k) lse_new = lse;
        }
        // every lane has read the R lse values above before any lane writes one back
        __syncwarp();
        if (lane < R && r0 + lane < rows) lse_run[r0 + lane] = lse_new;
    }
}

// ------------------------------------------------------------------ bounded-wait self test
__global__ void selftest_timeout_kernel(int* err, unsigned long long timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtl wc{&abort_flag, err, timeout_ns};
        // nothing ever arrives on `bar`: the wait must give up and record the error
        (void)mbar_wait(&bar, 0, wc);
    }
}

}  // namespace

int launch_permute(const void* src, void* dst, int S, int H, int row_bytes, int c, int layout, int inverse,
                   int* err, cudaStream_t stream) {
    const int nchunks = c * (layout == 1 ? 2 : 1);
    const long long slab = static_cast<long long>(S / nchunks) * row_bytes;
    const uintptr_t align = reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) |
                            static_cast<uintptr_t>(slab);
    if ((align & 15) == 0) return launch_permute_v<uint4>(src, dst, slab, H, nchunks, c, layout, inverse, err, stream);
    if ((align & 7) == 0) return launch_permute_v<uint2>(src, dst, slab, H, nchunks, c, layout, inverse, err, stream);
    if ((align & 3) == 0) return launch_permute_v<uint32_t>(src, dst, slab, H, nchunks, c, layout, inverse, err, stream);
    if ((align & 1) == 0) return launch_permute_v<uint16_t>(src, dst, slab, H, nchunks, c, layout, inverse, err, stream);
    return launch_permute_v<uint8_t>(src, dst, slab, H, nchunks, c, layout, inverse, err, stream);
}

int launch_merge(float* o_run, float* lse_run, const float* o_part, const float* lse_part, long long rows, int d,
                 cudaStream_t stream) {
    if (rows == 0) return 0;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long warps_needed = rows;
    long long blocks = (warps_needed + 7) / 8;
    const long long cap = static_cast<long long>(sms) * 8;
    if (blocks > cap) blocks = cap;
    const bool vec = (d % 4 == 0) && ((reinterpret_cast<uintptr_t>(o_run) | reinterpret_cast<uintptr_t>(o_part)) & 15) == 0;
    if (vec && d == 128) {
        constexpr int kRows = 4;
        long long b4 = (rows + 8 * kRows - 1) / (8 * kRows);
        if (b4 > cap) b4 = cap;
        merge_kernel_d128<kRows><<<static_cast<unsigned>(b4), 256, 0, stream>>>(
            reinterpret_cast<float4*>(o_run), lse_run, reinterpret_cast<const float4*>(o_part), lse_part, rows);
    } else if (vec)
        merge_kernel<true><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(o_run, lse_run, o_part, lse_part, rows, d);
    else
        merge_kernel<false><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(o_run, lse_run, o_part, lse_part, rows, d);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// ------------------------------------------------------------------ document starts
// For a packed sequence whose document ids do not decrease, the first position of the
// document of token i is the first position whose id is not below doc_id[i]: a binary
// search over [0, i] (thread per token).  Whatever the ids, the result lies in [0, i].
__global__ void doc_start_kernel(const int* __restrict__ doc_id, int* __restrict__ doc_start, int S) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= S) return;
    const int id = doc_id[i];
    int lo = 0, hi = i;
    while (lo < hi) {
        const int mid = lo + (hi - lo) / 2;
        if (doc_id[mid] < id) lo = mid + 1;
        else hi = mid;
    }
    doc_start[i] = lo;
}

int launch_doc_start(const int* doc_id, int* doc_start, int S, cudaStream_t stream) {
    doc_start_kernel<<<(S + 255) / 256, 256, 0, stream>>>(doc_id, doc_start, S);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int launch_selftest_timeout(int* err, unsigned long long timeout_ns, cudaStream_t stream) {
    selftest_timeout_kernel<<<1, 32, 0, stream>>>(err, timeout_ns);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace ra
