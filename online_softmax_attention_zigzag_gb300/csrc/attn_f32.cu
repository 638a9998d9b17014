// attn_f32.cu -- ring attention in fp32 on the CUDA cores (FFMA), one online update
// per ring message of kv_block keys, in the order of the update rule of "Ring
// Attention and Ulysses shard a sequence two different ways..." (section "Ring
// Attention: point-to-point rotation, and an online softmax that never sees the
// whole row at once"):
//     block_max = max of the message's scores; new_max = max(running_max, block_max);
//     correction = exp(running_max - new_max); p = exp(score - new_max);
//     running_sum = running_sum * correction + sum p;  out = out * correction + p V.
// Hop h visits the block of rank (r - h) mod c ("Interrogating parallelism, part 5",
// "How does attention survive being split?").  A message whose keys are all masked
// for a row leaves that row unchanged.
//
// One thread owns one query row; a CTA owns 128 consecutive local rows of one
// (head, rank), so every thread of a CTA walks the same messages and the K/V rows
// are staged once per CTA in shared memory, 32 keys at a time.
#include <cfloat>

#include "internal.h"

namespace ra {
namespace {

constexpr int kRows = 128;
constexpr int kKeys = 32;

// Two sweeps per message with CTA-uniform control flow: pass 1 finds the message
// max, pass 2 applies correction and accumulates; masked rows skip arithmetic only.
template <int DP>
__global__ void __launch_bounds__(kRows) attn_f32_kernel(const AttnF32Params p) {
    const Ring& R = p.ring;
    const int h = blockIdx.z, r = blockIdx.y;
    const int local = blockIdx.x * kRows + threadIdx.x;
    const bool active = local < R.n_r;
    const int hk = h / R.g;
    const int d = R.d;
    int qpos;
    {
        const int lr = active ? local : 0;
        const int slot = lr / R.m;
        const int chunk = (slot == 0) ? r : 2 * R.c - 1 - r;
        qpos = chunk * R.m + (lr - slot * R.m);
    }
    const size_t qrow = static_cast<size_t>(h) * R.S + static_cast<size_t>(r) * R.n_r + (active ? local : 0);

    const bool row_ok = !active || RA_CHECKED(qrow < static_cast<size_t>(R.Hq) * R.S, p.err, kSiteF32Row);
    float q[DP], o[DP];
#pragma unroll
    for (int t = 0; t < DP; ++t) {
        q[t] = (active && row_ok && t < d) ? p.q[qrow * d + t] : 0.f;
        o[t] = 0.f;
    }
    float run_max = -INFINITY, run_sum = 0.f;

    __shared__ float sk[kKeys][DP];
    __shared__ float sv[kKeys][DP];

    for (int hop = R.hop_lo; hop < R.hop_hi; ++hop) {
        int s = r - hop;
        if (s < 0) s += R.c;
        const size_t kv_base = static_cast<size_t>(hk) * R.S + static_cast<size_t>(s) * R.n_r;
        for (int m0 = R.kv_lo; m0 < R.kv_hi; m0 += p.kv_block) {
            const int m1 = min(m0 + p.kv_block, R.kv_hi);
            // ---- pass 1: block max
            float bmax = -INFINITY;
            for (int k0 = m0; k0 < m1; k0 += kKeys) {
                const int nk = min(kKeys, m1 - k0);
                __syncthreads();
                for (int e = threadIdx.x; e < nk * DP; e += kRows) {
                    const int kr = e / DP, t = e % DP;
                    const size_t kvr = kv_base + k0 + kr;
                    const bool ok = RA_CHECKED(kvr < static_cast<size_t>(R.Hkv) * R.S, p.err, kSiteF32Row);
                    sk[kr][t] = (t < d && ok) ? p.k[kvr * d + t] : 0.f;
                }
                __syncthreads();
                for (int kr = 0; kr < nk; ++kr) {
                    const int lk = k0 + kr;
                    const int slot = lk / R.m;
                    const int kpos = ((slot == 0) ? s : 2 * R.c - 1 - s) * R.m + (lk - slot * R.m);
                    if (R.causal && kpos > qpos) continue;
                    float acc = 0.f;
#pragma unroll
                    for (int t = 0; t < DP; ++t) acc = fmaf(q[t], sk[kr][t], acc);
                    bmax = fmaxf(bmax, acc);
                }
            }
            const bool visible = bmax != -INFINITY;
            const float new_max = visible ? fmaxf(run_max, bmax) : run_max;
            if (visible) {
                const float corr = expf(run_max - new_max);
                run_sum *= corr;
#pragma unroll
                for (int t = 0; t < DP; ++t) o[t] *= corr;
            }
            // ---- pass 2: p = exp(score - new_max), accumulate sum and p V
            for (int k0 = m0; k0 < m1; k0 += kKeys) {
                const int nk = min(kKeys, m1 - k0);
                __syncthreads();
                for (int e = threadIdx.x; e < nk * DP; e += kRows) {
                    const int kr = e / DP, t = e % DP;
                    const size_t kvr = kv_base + k0 + kr;
                    const bool ok = RA_CHECKED(kvr < static_cast<size_t>(R.Hkv) * R.S, p.err, kSiteF32Row);
                    const size_t off = kvr * d + t;
                    sk[kr][t] = (t < d && ok) ? p.k[off] : 0.f;
                    sv[kr][t] = (t < d && ok) ? p.v[off] : 0.f;
                }
                __syncthreads();
                if (!visible) continue;
                for (int kr = 0; kr < nk; ++kr) {
                    const int lk = k0 + kr;
                    const int slot = lk / R.m;
                    const int kpos = ((slot == 0) ? s : 2 * R.c - 1 - s) * R.m + (lk - slot * R.m);
                    if (R.causal && kpos > qpos) continue;
                    float acc = 0.f;
#pragma unroll
                    for (int t = 0; t < DP; ++t) acc = fmaf(q[t], sk[kr][t], acc);
                    const float pe = expf(acc - new_max);
                    run_sum += pe;
#pragma unroll
                    for (int t = 0; t < DP; ++t) o[t] = fmaf(pe, sv[kr][t], o[t]);
                }
            }
            run_max = new_max;
        }
    }
    if (!active || !row_ok) return;
    const bool seen = run_sum > 0.f;
    const float inv = seen ? 1.f / run_sum : 0.f;
    for (int t = 0; t < d; ++t) p.out[qrow * d + t] = o[t] * inv;
    p.lse[qrow] = seen ? run_max + logf(run_sum) : -INFINITY;
}

template <int DP>
int launch_dp(const AttnF32Params& p, cudaStream_t stream) {
    const Ring& R = p.ring;
    dim3 grid((R.n_r + kRows - 1) / kRows, R.c, R.Hq);
    attn_f32_kernel<DP><<<grid, kRows, 0, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace

int launch_attn_f32(const AttnF32Params& p, cudaStream_t stream) {
    const int d = p.ring.d;
    if (d <= 8) return launch_dp<8>(p, stream);
    if (d <= 16) return launch_dp<16>(p, stream);
    if (d <= 32) return launch_dp<32>(p, stream);
    if (d <= 64) return launch_dp<64>(p, stream);
    if (d <= 128) return launch_dp<128>(p, stream);
    return -2;
}

}  // namespace ra
