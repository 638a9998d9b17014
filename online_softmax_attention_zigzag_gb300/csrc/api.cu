// api.cu -- the C ABI of libringattn.so (declared in include/ringattn.h): argument
// validation, device checks, TMA descriptors, work geometry and kernel launches.
// Host code only; the compute is in attn_bf16.cu, attn_f32.cu and permute_merge.cu.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <nvtx3/nvToolsExt.h>

#include <climits>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "ringattn.h"
#include "internal.h"

namespace {

// NVTX range over one entry point's host work (argument checks and the launches it
// enqueues), so that a timeline tool shows permute, attention, merge and the other
// calls by name.  Without a tool attached a push/pop costs a few nanoseconds.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// Device error word: bounded waits that run out write RA_ERR_TIMEOUT here.  It is a
// static device variable, so the library allocates nothing; host code reaches it
// through the address cudaGetSymbolAddress returns for the current device.
__device__ int g_err_word[4];  // status, record set, barrier address, (block << 10 | thread)
// Work-item counters of the fused kernel, one pair per launch slot.  A launch takes the
// next slot in turn; its last CTA zeroes the pair again, so a slot is clean for the launch
// that takes it kSchedSlots launches later.  (Two launches in flight at once that held the
// same slot would share counters: that needs kSchedSlots launches in flight together.)
constexpr int kSchedSlots = 256;
__device__ unsigned int g_sched[2 * kSchedSlots];
// Scratch of ringattn_fwd_docmask_noalloc: the document start of every position, for
// callers that cannot allocate it.  A file-scope device array, so it exists on every
// device that loads the library and is never allocated or freed by a call.  In host
// code the name is only a stand-in for the symbol: the device address comes from
// cudaGetSymbolAddress, looked up in device_info() with the device current.
__device__ __align__(256) int g_doc_start_scratch[RINGATTN_DOCMASK_NOALLOC_MAX_S];

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    int status = RA_OK;  // RA_ERR_ARCH when the device is not sm_103
    int sms = 0;
    int* err = nullptr;
    unsigned int* sched = nullptr;  // g_sched on this device
    int* doc_scratch = nullptr;     // g_doc_start_scratch on this device
    unsigned int next_slot = 0;     // guarded by g_mu
};

std::mutex g_mu;
int g_last_timeout[3] = {0, 0, 0};  // barrier address, CTA, thread of the last recorded timeout
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Current device's info; performs the one-time set-up for that device.
int device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return RA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return RA_ERR_CUDA;
        if (major != 10 || minor != 3) {
            d.status = RA_ERR_ARCH;
        } else {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return RA_ERR_CUDA;
            d.err = static_cast<int*>(p);
            if (cudaGetSymbolAddress(&p, g_sched) != cudaSuccess) return RA_ERR_CUDA;
            d.sched = static_cast<unsigned int*>(p);
            if (cudaGetSymbolAddress(&p, g_doc_start_scratch) != cudaSuccess || !p) return RA_ERR_CUDA;
            d.doc_scratch = static_cast<int*>(p);
            d.status = RA_OK;
        }
        d.ready = true;
    }
    if (d.status != RA_OK) return d.status;
    *out = &d;
    return RA_OK;
}

// n consecutive counter slots (pairs of words) of the device's ring, taken in turn.
unsigned int* sched_slots(DeviceInfo* dev, int n) {
    std::lock_guard<std::mutex> lock(g_mu);
    unsigned int i = dev->next_slot % kSchedSlots;
    if (i + n > static_cast<unsigned int>(kSchedSlots)) {  // keep the n slots contiguous
        dev->next_slot += kSchedSlots - i;
        i = 0;
    }
    dev->next_slot += n;
    return dev->sched + 2 * i;
}

int get_encoder() {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_encode) return RA_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return RA_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return RA_OK;
}

// [rows, d] bf16 tensor, boxes of box_rows rows x 64 columns, 128-byte swizzle.
int encode_bf16_map(CUtensorMap* map, const void* base, long long rows, int d, int box_rows = 128) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * 2};
    cuuint32_t box[2] = {64, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? RA_OK : RA_ERR_CUDA;
}

// The attention kernels' wait limit.  Never below 1 s: the warps that feed a hardware
// named barrier (whose waiter cannot give up) stop arriving only when their own limit runs
// out, so that limit must stay far above the time a queued MMA takes to complete.
unsigned long long wait_timeout_ns() {
    static unsigned long long ns = [] {
        const char* e = std::getenv("RINGATTN_WAIT_TIMEOUT_MS");
        long long ms = e ? std::atoll(e) : 2000;
        if (ms < 1000) ms = 1000;
        if (ms > 600000) ms = 600000;
        return static_cast<unsigned long long>(ms) * 1000000ull;
    }();
    return ns;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Geometry checks shared by every attention entry point.
int make_ring(int S, int Hq, int Hkv, int d, int c, int causal, int layout, int kv_block, ra::Ring* R) {
    if (S < 1 || Hq < 1 || Hkv < 1 || d < 1 || c < 1 || kv_block < 1) return RA_ERR_INVALID_ARG;
    if ((causal != 0 && causal != 1) || (layout != 0 && layout != 1)) return RA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return RA_ERR_INVALID_ARG;
    const int nch = c * (layout == 1 ? 2 : 1);
    if (S % nch != 0) return RA_ERR_INVALID_ARG;
    const int m = S / nch;
    if (m % kv_block != 0) return RA_ERR_INVALID_ARG;
    if (static_cast<long long>(Hq) * S > INT_MAX || static_cast<long long>(Hq) * S * d > (1LL << 40))
        return RA_ERR_UNSUPPORTED;
    R->S = S;
    R->Hq = Hq;
    R->Hkv = Hkv;
    R->g = Hq / Hkv;
    R->d = d;
    R->c = c;
    R->causal = causal;
    R->layout = layout;
    R->n_r = S / c;
    R->m = m;
    R->nslot = layout == 1 ? 2 : 1;
    R->hop_lo = 0;
    R->hop_hi = c;
    R->kv_lo = 0;
    R->kv_hi = S / c;
    return RA_OK;
}

int select_hop(ra::Ring* R, int kv_block, int hop, int sub) {
    if (hop < 0 || hop >= R->c) return RA_ERR_INVALID_ARG;
    if (sub < 0 || sub >= R->n_r / kv_block) return RA_ERR_INVALID_ARG;
    R->hop_lo = hop;
    R->hop_hi = hop + 1;
    R->kv_lo = sub * kv_block;
    R->kv_hi = (sub + 1) * kv_block;
    return RA_OK;
}

int fwd_bf16(const void* q, const void* k, const void* v, float* out, float* lse, int S, int Hq, int Hkv, int d,
             int c, int causal, int layout, int kv_block, int natural, int hop, int sub, int rank,
             cudaStream_t stream, const int* doc_id = nullptr, int* doc_start = nullptr) {
    if (!q || !k || !v || !out || !lse) return RA_ERR_INVALID_ARG;
    if (rank < -1 || rank >= c) return RA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse))
        return RA_ERR_INVALID_ARG;
    ra::Ring R;
    int st = make_ring(S, Hq, Hkv, d, c, causal, layout, kv_block, &R);
    if (st != RA_OK) return st;
    if (d != 64 && d != 128) return RA_ERR_UNSUPPORTED;
    if (R.m % 128 != 0 || kv_block % 128 != 0) return RA_ERR_UNSUPPORTED;
    if (hop >= 0 && (st = select_hop(&R, kv_block, hop, sub)) != RA_OK) return st;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != RA_OK) return st;
    if ((st = get_encoder()) != RA_OK) return st;

    ra::AttnBf16Params p;
    p.ring = R;
    p.natural = natural;
    p.rank_sel = rank;
    p.n_tiles = (rank >= 0 ? R.n_r : S) / 128;
    const int tiles_per_chunk = R.m / 128;
    if (R.g % 2 == 0) {
        p.pair_mode = ra::kPairHeads;
        p.n_items = p.n_tiles * (Hq / 2);
    } else if (R.g == 1 && tiles_per_chunk % 2 == 0) {
        p.pair_mode = ra::kPairPositions;
        p.n_items = (p.n_tiles / 2) * Hq;
    } else {
        p.pair_mode = ra::kSingles;
        p.n_items = p.n_tiles * Hq;
    }
    // Order work items by groups of KV heads whose K and V take a third of L2 at most:
    // within a group the items go by decreasing work across the group's heads; across
    // groups, one group's K/V is live at a time, so K and V come from DRAM once.  The
    // CTAs draw items from this list as they finish (a counter in global memory), which
    // evens out their work whatever the list's shape.
    {
        constexpr double kBudget = 40e6;
        const double kv_head_bytes = static_cast<double>(S) * d * 4.0;  // K and V of one head, bf16
        p.kv_group = 1;
        for (int gsz = Hkv; gsz >= 1; --gsz)
            if (Hkv % gsz == 0 && gsz * kv_head_bytes <= kBudget) {
                p.kv_group = gsz;
                break;
            }
    }
    p.sched = sched_slots(dev, 1);
    p.out = out;
    p.lse = lse;
    p.doc_start = doc_start;
    p.err = dev->err;
    p.timeout_ns = wait_timeout_ns();

    CUtensorMap tq, tk, tv;
    if (encode_bf16_map(&tq, q, static_cast<long long>(Hq) * S, d) != RA_OK ||
        encode_bf16_map(&tk, k, static_cast<long long>(Hkv) * S, d) != RA_OK ||
        encode_bf16_map(&tv, v, static_cast<long long>(Hkv) * S, d) != RA_OK)
        return RA_ERR_CUDA;
    const int grid = p.n_items < dev->sms ? p.n_items : dev->sms;
    if (doc_id && ra::launch_doc_start(doc_id, doc_start, S, stream) != 0) return RA_ERR_CUDA;
    return ra::launch_attn_bf16(p, tq, tk, tv, grid, stream);
}

int fwd_f32(const float* q, const float* k, const float* v, float* out, float* lse, int S, int Hq, int Hkv, int d,
            int c, int causal, int layout, int kv_block, int hop, int sub, cudaStream_t stream) {
    if (!q || !k || !v || !out || !lse) return RA_ERR_INVALID_ARG;
    ra::Ring R;
    int st = make_ring(S, Hq, Hkv, d, c, causal, layout, kv_block, &R);
    if (st != RA_OK) return st;
    if (d > 128) return RA_ERR_UNSUPPORTED;
    if (R.c > 65535 || Hq > 65535) return RA_ERR_UNSUPPORTED;
    if (hop >= 0 && (st = select_hop(&R, kv_block, hop, sub)) != RA_OK) return st;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != RA_OK) return st;
    ra::AttnF32Params p;
    p.ring = R;
    p.kv_block = kv_block;
    p.err = dev->err;
    p.q = q;
    p.k = k;
    p.v = v;
    p.out = out;
    p.lse = lse;
    return ra::launch_attn_f32(p, stream);
}

// ------------------------------------------------------------------ host-buffer path
// ringattn_fwd_host runs the natural-order kernel once per group of KV heads, so that the
// copies of one group overlap the attention of another: H2D of group g+1 and D2H of group
// g-1 run on two internal streams (one per copy direction) while group g computes.  The
// launches alternate between the caller's stream and a third internal stream, so that a
// launch's CTAs take the SMs its predecessor's last CTAs leave (each launch ends with a
// tail of long work items; the launches are independent: different heads, their own
// work-item counters).  Streams and events are created once per device and kept until exit.
constexpr int kMaxGroups = 16;
constexpr int kMaxLaunches = kMaxGroups + 4;  // the first and last group may run as three launches

struct HostPipe {
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr, comp = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t in[kMaxLaunches] = {}, out[kMaxLaunches] = {};
    std::mutex mu;  // one call enqueues at a time per device
};

HostPipe g_pipe[kMaxDevices];

int host_pipe(HostPipe** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return RA_ERR_UNSUPPORTED;
    HostPipe& hp = g_pipe[dev];
    std::lock_guard<std::mutex> lock(g_mu);
    if (!hp.ready) {
        const unsigned ef = cudaEventDisableTiming;
        if (cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&hp.comp, cudaStreamNonBlocking) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp.start, ef) != cudaSuccess ||
            cudaEventCreateWithFlags(&hp.done, ef) != cudaSuccess)
            return RA_ERR_CUDA;
        for (int i = 0; i < kMaxLaunches; ++i)
            if (cudaEventCreateWithFlags(&hp.in[i], ef) != cudaSuccess ||
                cudaEventCreateWithFlags(&hp.out[i], ef) != cudaSuccess)
                return RA_ERR_CUDA;
        hp.ready = true;
    }
    *out = &hp;
    return RA_OK;
}

// Byte offsets of the device copies inside the host path's workspace, each 256-byte aligned:
// q, k, v (bf16), out, lse (fp32), all [H, S, ...] in natural order; off[5] = total.
void host_workspace_layout(int S, int Hq, int Hkv, int d, long long off[6]) {
    const long long sz[5] = {2LL * Hq * S * d, 2LL * Hkv * S * d, 2LL * Hkv * S * d, 4LL * Hq * S * d,
                             4LL * Hq * S};
    long long o = 0;
    for (int i = 0; i < 5; ++i) {
        off[i] = o;
        o += (sz[i] + 255) / 256 * 256;
    }
    off[5] = o;
}

// Number of KV-head groups: as many as divide Hkv (at most kMaxGroups) while every group
// still holds at least four waves of work items, so that no launch is mostly tail.
int host_groups(int S, int Hq, int Hkv, int sms) {
    const long long items = static_cast<long long>(S / 128) * Hq / 2;  // about two tiles per item
    int best = 1;
    for (int gcount = 1; gcount <= Hkv && gcount <= kMaxGroups; ++gcount)
        if (Hkv % gcount == 0 && items / gcount >= 4LL * sms) best = gcount;
    return best;
}

int fwd_host(const void* q_h, const void* k_h, const void* v_h, float* out_h, float* lse_h, int S, int Hq,
             int Hkv, int d, int c, int causal, int layout, int kv_block, void* ws, size_t ws_bytes,
             cudaStream_t stream) {
    if (!q_h || !k_h || !v_h || !out_h || !lse_h || !ws) return RA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return RA_ERR_INVALID_ARG;
    ra::Ring R;
    int st = make_ring(S, Hq, Hkv, d, c, causal, layout, kv_block, &R);
    if (st != RA_OK) return st;
    if (d != 64 && d != 128) return RA_ERR_UNSUPPORTED;
    if (R.m % 128 != 0 || kv_block % 128 != 0) return RA_ERR_UNSUPPORTED;
    long long off[6];
    host_workspace_layout(S, Hq, Hkv, d, off);
    if (static_cast<long long>(ws_bytes) < off[5]) return RA_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != RA_OK) return st;
    HostPipe* hp = nullptr;
    if ((st = host_pipe(&hp)) != RA_OK) return st;

    char* base = static_cast<char*>(ws);
    const int G = host_groups(S, Hq, Hkv, dev->sms);
    const int hq_g = Hq / G, hkv_g = Hkv / G;
    // Launches: one per group, except that the first and the last group run as two halves
    // of their query heads when a group has one KV head: the first launch then starts after
    // less input has crossed, and the last results start back sooner.  Each half is the
    // same per-head computation, so the result does not depend on the split.
    struct Launch { int g, h0, hn; };  // group g, its query heads [h0, h0 + hn)
    Launch L[kMaxLaunches];
    int nl = 0;
    const bool halves = G >= 2 && hkv_g == 1 && hq_g % 2 == 0;
    const bool quarters = halves && hq_g % 4 == 0;
    for (int gi = 0; gi < G; ++gi) {
        if (quarters && gi == 0) {  // quarter, quarter, half
            L[nl++] = {gi, 0, hq_g / 4};
            L[nl++] = {gi, hq_g / 4, hq_g / 4};
            L[nl++] = {gi, hq_g / 2, hq_g / 2};
        } else if (quarters && gi == G - 1) {  // half, quarter, quarter
            L[nl++] = {gi, 0, hq_g / 2};
            L[nl++] = {gi, hq_g / 2, hq_g / 4};
            L[nl++] = {gi, 3 * hq_g / 4, hq_g / 4};
        } else if (halves && (gi == 0 || gi == G - 1)) {
            L[nl++] = {gi, 0, hq_g / 2};
            L[nl++] = {gi, hq_g / 2, hq_g / 2};
        } else {
            L[nl++] = {gi, 0, hq_g};
        }
    }
    const size_t qh_b = 2ull * S * d, oh_b = 4ull * S * d, lh_b = 4ull * S;  // one query head's rows
    const size_t kv_b = 2ull * hkv_g * S * d;
    std::lock_guard<std::mutex> lock(hp->mu);
    // the copies and the second compute stream start only after the work already queued on
    // `stream`
    if (cudaEventRecord(hp->start, stream) != cudaSuccess || cudaStreamWaitEvent(hp->h2d, hp->start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(hp->comp, hp->start, 0) != cudaSuccess)
        return RA_ERR_CUDA;
    for (int li = 0; li < nl; ++li) {
        const int gi = L[li].g;
        const size_t h0 = static_cast<size_t>(gi) * hq_g + L[li].h0;  // first query head of the launch
        if (L[li].h0 == 0 &&  // K and V once per group, ahead of its first launch
            (cudaMemcpyAsync(base + off[1] + gi * kv_b, static_cast<const char*>(k_h) + gi * kv_b, kv_b,
                             cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess ||
             cudaMemcpyAsync(base + off[2] + gi * kv_b, static_cast<const char*>(v_h) + gi * kv_b, kv_b,
                             cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess))
            return RA_ERR_CUDA;
        if (cudaMemcpyAsync(base + off[0] + h0 * qh_b, static_cast<const char*>(q_h) + h0 * qh_b, L[li].hn * qh_b,
                            cudaMemcpyHostToDevice, hp->h2d) != cudaSuccess ||
            cudaEventRecord(hp->in[li], hp->h2d) != cudaSuccess)
            return RA_ERR_CUDA;
    }
    for (int li = 0; li < nl; ++li) {
        const int gi = L[li].g;
        const size_t h0 = static_cast<size_t>(gi) * hq_g + L[li].h0;
        float* od = reinterpret_cast<float*>(base + off[3] + h0 * oh_b);
        float* ld = reinterpret_cast<float*>(base + off[4] + h0 * lh_b);
        cudaStream_t ks = (li % 2 == 0) ? stream : hp->comp;  // launches alternate between two streams
        if (cudaStreamWaitEvent(ks, hp->in[li], 0) != cudaSuccess) return RA_ERR_CUDA;
        st = fwd_bf16(base + off[0] + h0 * qh_b, base + off[1] + gi * kv_b, base + off[2] + gi * kv_b, od, ld, S,
                      L[li].hn, hkv_g, d, c, causal, layout, kv_block, 1, -1, 0, -1, ks);
        if (st != RA_OK) return st;
        if (cudaEventRecord(hp->out[li], ks) != cudaSuccess || cudaStreamWaitEvent(hp->d2h, hp->out[li], 0) != cudaSuccess ||
            cudaMemcpyAsync(reinterpret_cast<char*>(out_h) + h0 * oh_b, od, L[li].hn * oh_b, cudaMemcpyDeviceToHost,
                            hp->d2h) != cudaSuccess ||
            cudaMemcpyAsync(reinterpret_cast<char*>(lse_h) + h0 * lh_b, ld, L[li].hn * lh_b, cudaMemcpyDeviceToHost,
                            hp->d2h) != cudaSuccess)
            return RA_ERR_CUDA;
    }
    // `stream` completes only once the last result has reached the host
    if (cudaEventRecord(hp->done, hp->d2h) != cudaSuccess || cudaStreamWaitEvent(stream, hp->done, 0) != cudaSuccess)
        return RA_ERR_CUDA;
    return RA_OK;
}

}  // namespace

extern "C" {

int ringattn_fwd(const void* q, const void* k, const void* v, float* out, float* lse, int S, int Hq, int Hkv, int d,
                 int c, int causal, int layout, int kv_block, ra_stream_t stream) {
    NvtxRange nvtx("ringattn_fwd");
    return fwd_bf16(q, k, v, out, lse, S, Hq, Hkv, d, c, causal, layout, kv_block, 0, -1, 0, -1,
                    reinterpret_cast<cudaStream_t>(stream));
}

int ringattn_fwd_rank(const void* q, const void* k, const void* v, float* out, float* lse, int S, int Hq, int Hkv,
                      int d, int c, int causal, int layout, int kv_block, int rank, ra_stream_t stream) {
    NvtxRange nvtx("ringattn_fwd_rank");
    if (rank < 0) return RA_ERR_INVALID_ARG;
    return fwd_bf16(q, k, v, out, lse, S, Hq, Hkv, d, c, causal, layout, kv_block, 0, -1, 0, rank,
                    reinterpret_cast<cudaStream_t>(stream));
}

int ringattn_fwd_docmask(const void* q, const void* k, const void* v, float* out, float* lse, const int* doc_id,
                         int* doc_start, int S, int Hq, int Hkv, int d, int c, int layout, ra_stream_t stream) {
    NvtxRange nvtx("ringattn_fwd_docmask");
    if (!doc_id || !doc_start || static_cast<const void*>(doc_id) == static_cast<const void*>(doc_start))
        return RA_ERR_INVALID_ARG;
    if (((reinterpret_cast<uintptr_t>(doc_id) | reinterpret_cast<uintptr_t>(doc_start)) & 3u) != 0)
        return RA_ERR_INVALID_ARG;
    if (c < 1 || (layout != 0 && layout != 1)) return RA_ERR_INVALID_ARG;
    const int nch = c * (layout == 1 ? 2 : 1);
    if (S < 1 || S % nch != 0) return RA_ERR_INVALID_ARG;
    // kv_block plays no part here (no ring messages): pass the chunk, always valid
    return fwd_bf16(q, k, v, out, lse, S, Hq, Hkv, d, c, 1, layout, S / nch, 0, -1, 0, -1,
                    reinterpret_cast<cudaStream_t>(stream), doc_id, doc_start);
}

int ringattn_fwd_docmask_noalloc(const void* q, const void* k, const void* v, float* out, float* lse,
                                 const int* doc_id, int S, int Hq, int Hkv, int d, int c, int layout,
                                 ra_stream_t stream) {
    NvtxRange nvtx("ringattn_fwd_docmask_noalloc");
    if (!doc_id || (reinterpret_cast<uintptr_t>(doc_id) & 3u) != 0) return RA_ERR_INVALID_ARG;
    if (S > RINGATTN_DOCMASK_NOALLOC_MAX_S) return RA_ERR_UNSUPPORTED;  // beyond the static scratch
    if (c < 1 || (layout != 0 && layout != 1)) return RA_ERR_INVALID_ARG;
    const int nch = c * (layout == 1 ? 2 : 1);
    if (S < 1 || S % nch != 0) return RA_ERR_INVALID_ARG;
    // the scratch address comes from the device's one-time set-up (device_info)
    DeviceInfo* dev = nullptr;
    int st = device_info(&dev);
    if (st != RA_OK) return st;
    // doc_start_kernel rewrites scratch[0, S) on `stream` before the attention kernel
    // reads it, so nothing left by an earlier call is ever read
    return fwd_bf16(q, k, v, out, lse, S, Hq, Hkv, d, c, 1, layout, S / nch, 0, -1, 0, -1,
                    reinterpret_cast<cudaStream_t>(stream), doc_id, dev->doc_scratch);
}

int ringattn_host_workspace_bytes(int S, int Hq, int Hkv, int d, long long* bytes) {
    if (!bytes || S < 1 || Hq < 1 || Hkv < 1 || d < 1) return RA_ERR_INVALID_ARG;
    long long off[6];
    host_workspace_layout(S, Hq, Hkv, d, off);
    *bytes = off[5];
    return RA_OK;
}

int ringattn_fwd_host(const void* q_h, const void* k_h, const void* v_h, float* out_h, float* lse_h, int S, int Hq,
                      int Hkv, int d, int c, int causal, int layout, int kv_block, void* workspace,
                      long long workspace_bytes, ra_stream_t stream) {
    NvtxRange nvtx("ringattn_fwd_host");
    if (workspace_bytes < 0) return RA_ERR_INVALID_ARG;
    return fwd_host(q_h, k_h, v_h, out_h, lse_h, S, Hq, Hkv, d, c, causal, layout, kv_block, workspace,
                    static_cast<size_t>(workspace_bytes), reinterpret_cast<cudaStream_t>(stream));
}

int ringattn_relayout(const void* src, void* dst, int S, int H, int row_bytes, int c, int layout, int to_heads,
                      ra_stream_t stream) {
    NvtxRange nvtx("ringattn_relayout");
    if (!src || !dst || src == dst) return RA_ERR_INVALID_ARG;
    if (S < 1 || H < 1 || row_bytes < 1 || c < 1) return RA_ERR_INVALID_ARG;
    if ((layout != 0 && layout != 1) || (to_heads != 0 && to_heads != 1)) return RA_ERR_INVALID_ARG;
    if (S % (c * (layout == 1 ? 2 : 1)) != 0) return RA_ERR_INVALID_ARG;
    if (((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 3u) != 0) return RA_ERR_INVALID_ARG;
    if (!ra::relayout_fits(S, H, row_bytes, c, layout)) return RA_ERR_UNSUPPORTED;
    const long long bytes = static_cast<long long>(H) * S * row_bytes;
    const char* a = static_cast<const char*>(src);
    const char* b = static_cast<const char*>(dst);
    if (a < b + bytes && b < a + bytes) return RA_ERR_INVALID_ARG;  // overlapping buffers
    DeviceInfo* dev = nullptr;
    int st = device_info(&dev);
    if (st != RA_OK) return st;
    return ra::launch_relayout(src, dst, S, H, row_bytes, c, layout, to_heads, dev->err,
                               reinterpret_cast<cudaStream_t>(stream));
}

int ringattn_ulysses_fwd(const void* q_seq, const void* k_seq, const void* v_seq, float* out_seq, float* lse_seq,
                         int S, int Hq, int Hkv, int d, int c, int causal, int layout, void* workspace,
                         long long workspace_bytes, ra_stream_t stream) {
    NvtxRange nvtx("ringattn_ulysses_fwd");
    if (!q_seq || !k_seq || !v_seq || !out_seq || !lse_seq || !workspace) return RA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || workspace_bytes < 0) return RA_ERR_INVALID_ARG;
    if (!aligned16(q_seq) || !aligned16(k_seq) || !aligned16(v_seq) || !aligned16(out_seq) ||
        (reinterpret_cast<uintptr_t>(lse_seq) & 3u) != 0)
        return RA_ERR_INVALID_ARG;
    if (c < 1 || Hq < 1 || Hq % c != 0) return RA_ERR_INVALID_ARG;  // each rank gets Hq/c query heads
    // the sequence shards: the ring's chunking for (c, layout) (no messages: kv_block 1)
    ra::Ring R;
    int st = make_ring(S, Hq, Hkv, d, c, causal, layout, 1, &R);
    if (st != RA_OK) return st;
    // the attention: every rank's heads over the whole sequence (c = 1 in the kernel)
    if ((st = make_ring(S, Hq, Hkv, d, 1, causal, 0, S, &R)) != RA_OK) return st;
    if (d != 64 && d != 128) return RA_ERR_UNSUPPORTED;
    if (S % 128 != 0) return RA_ERR_UNSUPPORTED;
    if (!ra::relayout_fits(S, Hq, 4 * d, c, layout) || !ra::relayout_fits(S, Hkv, 2 * d, c, layout))
        return RA_ERR_UNSUPPORTED;
    long long off[6];
    host_workspace_layout(S, Hq, Hkv, d, off);
    if (workspace_bytes < off[5]) return RA_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != RA_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    void *qh = ws + off[0], *kh = ws + off[1], *vh = ws + off[2];
    float* oh = reinterpret_cast<float*>(ws + off[3]);
    float* lh = reinterpret_cast<float*>(ws + off[4]);
    // all-to-all: sequence shards -> head shards
    if (ra::launch_relayout(q_seq, qh, S, Hq, 2 * d, c, layout, 1, dev->err, s) != 0 ||
        ra::launch_relayout(k_seq, kh, S, Hkv, 2 * d, c, layout, 1, dev->err, s) != 0 ||
        ra::launch_relayout(v_seq, vh, S, Hkv, 2 * d, c, layout, 1, dev->err, s) != 0)
        return RA_ERR_CUDA;
    // local attention of every rank's heads over the whole sequence, one launch for all ranks
    if ((st = fwd_bf16(qh, kh, vh, oh, lh, S, Hq, Hkv, d, 1, causal, 0, S, 1, -1, 0, -1, s)) != RA_OK) return st;
    // all-to-all back: head shards -> sequence shards
    if (ra::launch_relayout(oh, out_seq, S, Hq, 4 * d, c, layout, 0, dev->err, s) != 0 ||
        ra::launch_relayout(lh, lse_seq, S, Hq, 4, c, layout, 0, dev->err, s) != 0)
        return RA_ERR_CUDA;
    return RA_OK;
}

}  // extern "C"

namespace {

int bwd_bf16(const void* q, const void* k, const void* v, const float* out, const float* lse, const void* dout,
             float* dq, float* dk, float* dv, float* delta, int S, int Hq, int Hkv, int d, int c, int causal,
             int layout, int kv_block, int natural, cudaStream_t stream) {
    if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv || !delta) return RA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(lse) || !aligned16(dout) ||
        !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(delta))
        return RA_ERR_INVALID_ARG;
    ra::Ring R;
    int st = make_ring(S, Hq, Hkv, d, c, causal, layout, kv_block, &R);
    if (st != RA_OK) return st;
    if (d != 64 && d != 128) return RA_ERR_UNSUPPORTED;
    if (R.m % 128 != 0 || kv_block % 128 != 0) return RA_ERR_UNSUPPORTED;
    DeviceInfo* dev = nullptr;
    if ((st = device_info(&dev)) != RA_OK) return st;
    if ((st = get_encoder()) != RA_OK) return st;
    ra::AttnBwdParams p;
    p.ring = R;
    p.natural = natural;
    p.n_tiles = S / 128;
    p.n_items = 0;
    p.lse = lse;
    p.delta = delta;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.err = dev->err;
    p.timeout_ns = wait_timeout_ns();
    p.sched = sched_slots(dev, 2);
    CUtensorMap tq, tk, tv, tdo;
    // the backward kernels move 64-row boxes (half tiles are their streaming unit)
    if (encode_bf16_map(&tq, q, static_cast<long long>(Hq) * S, d, 64) != RA_OK ||
        encode_bf16_map(&tk, k, static_cast<long long>(Hkv) * S, d, 64) != RA_OK ||
        encode_bf16_map(&tv, v, static_cast<long long>(Hkv) * S, d, 64) != RA_OK ||
        encode_bf16_map(&tdo, dout, static_cast<long long>(Hq) * S, d, 64) != RA_OK)
        return RA_ERR_CUDA;
    return ra::launch_attn_bwd(p, out, dout, tq, tk, tv, tdo, dev->sms, stream) == 0 ? RA_OK : RA_ERR_CUDA;
}

}  // namespace

extern "C" {

int ringattn_bwd(const void* q, const void* k, const void* v, const float* out, const float* lse, const void* dout,
                 float* dq, float* dk, float* dv, float* delta, int S, int Hq, int Hkv, int d, int c, int causal,
                 int layout, int kv_block, ra_stream_t stream) {
    NvtxRange nvtx("ringattn_bwd");
    return bwd_bf16(q, k, v, out, lse, dout, dq, dk, dv, delta, S, Hq, Hkv, d, c, causal, layout, kv_block, 0,
                    reinterpret_cast<cudaStream_t>(stream));
}

int ringattn_bwd_natural(const void* q, const void* k, const void* v, const float* out, const float* lse,
                         const void* dout, float* dq, float* dk, float* dv, float* delta, int S, int Hq, int Hkv,
                         int d, int c, int causal, int layout, int kv_block, ra_stream_t stream) {
    NvtxRange nvtx("ringattn_bwd_natural");
    return bwd_bf16(q, k, v, out, lse, dout, dq, dk, dv, delta, S, Hq, Hkv, d, c, causal, layout, kv_block, 1,
                    reinterpret_cast<cudaStream_t>(stream));
}

int ringattn_fwd_natural(const void* q, const void* k, const void* v, float* out, float* lse, int S, int Hq,
                         int Hkv, int d, int c, int causal, int layout, int kv_block, ra_stream_t stream) {
    NvtxRange nvtx("ringattn_fwd_natural");
    return fwd_bf16(q, k, v, out, lse, S, Hq, Hkv, d, c, causal, layout, kv_block, 1, -1, 0, -1,
                    reinterpret_cast<cudaStream_t>(stream));
}

int ringattn_fwd_hop(const void* q, const void* k, const void* v, float* o_part, float* lse_part, int S, int Hq,
                     int Hkv, int d, int c, int causal, int layout, int kv_block, int hop, int sub,
                     ra_stream_t stream) {
    NvtxRange nvtx("ringattn_fwd_hop");
    if (hop < 0) return RA_ERR_INVALID_ARG;
    return fwd_bf16(q, k, v, o_part, lse_part, S, Hq, Hkv, d, c, causal, layout, kv_block, 0, hop, sub, -1,
                    reinterpret_cast<cudaStream_t>(stream));
}

int ringattn_fwd_f32(const float* q, const float* k, const float* v, float* out, float* lse, int S, int Hq,
                     int Hkv, int d, int c, int causal, int layout, int kv_block, ra_stream_t stream) {
    NvtxRange nvtx("ringattn_fwd_f32");
    return fwd_f32(q, k, v, out, lse, S, Hq, Hkv, d, c, causal, layout, kv_block, -1, 0,
                   reinterpret_cast<cudaStream_t>(stream));
}

int ringattn_fwd_hop_f32(const float* q, const float* k, const float* v, float* o_part, float* lse_part, int S,
                         int Hq, int Hkv, int d, int c, int causal, int layout, int kv_block, int hop, int sub,
                         ra_stream_t stream) {
    NvtxRange nvtx("ringattn_fwd_hop_f32");
    if (hop < 0) return RA_ERR_INVALID_ARG;
    return fwd_f32(q, k, v, o_part, lse_part, S, Hq, Hkv, d, c, causal, layout, kv_block, hop, sub,
                   reinterpret_cast<cudaStream_t>(stream));
}

int ringattn_merge(float* o_run, float* lse_run, const float* o_part, const float* lse_part, long long rows, int d,
                   ra_stream_t stream) {
    NvtxRange nvtx("ringattn_merge");
    if (rows < 0 || d < 1 || d > 4096) return RA_ERR_INVALID_ARG;
    if (rows > 0 && (!o_run || !lse_run || !o_part || !lse_part)) return RA_ERR_INVALID_ARG;
    if (rows == 0) return RA_OK;
    DeviceInfo* dev = nullptr;
    int st = device_info(&dev);
    if (st != RA_OK) return st;
    return ra::launch_merge(o_run, lse_run, o_part, lse_part, rows, d, reinterpret_cast<cudaStream_t>(stream));
}

int ringattn_permute(const void* src, void* dst, int S, int H, int row_bytes, int c, int layout, int inverse,
                     ra_stream_t stream) {
    NvtxRange nvtx("ringattn_permute");
    if (!src || !dst || src == dst) return RA_ERR_INVALID_ARG;
    if (S < 1 || H < 1 || row_bytes < 1 || c < 1) return RA_ERR_INVALID_ARG;
    if ((layout != 0 && layout != 1) || (inverse != 0 && inverse != 1)) return RA_ERR_INVALID_ARG;
    if (S % (c * (layout == 1 ? 2 : 1)) != 0) return RA_ERR_INVALID_ARG;
    const long long bytes = static_cast<long long>(H) * S * row_bytes;
    const char* a = static_cast<const char*>(src);
    const char* b = static_cast<const char*>(dst);
    if (a < b + bytes && b < a + bytes) return RA_ERR_INVALID_ARG;  // overlapping buffers
    DeviceInfo* dev = nullptr;
    int st = device_info(&dev);
    if (st != RA_OK) return st;
    return ra::launch_permute(src, dst, S, H, row_bytes, c, layout, inverse, dev->err,
                              reinterpret_cast<cudaStream_t>(stream));
}

int ringattn_rank_work(int S, int c, int causal, int layout, int tile, long long* units, long long* pairs,
                       long long* tiles) {
    if (S < 1 || c < 1 || tile < 1 || (causal != 0 && causal != 1) || (layout != 0 && layout != 1))
        return RA_ERR_INVALID_ARG;
    const int nch = c * (layout == 1 ? 2 : 1);
    if (S % nch != 0) return RA_ERR_INVALID_ARG;
    const long long m = S / nch, n_r = S / c;
    const long long kv_tiles_per_chunk = (m + tile - 1) / tile;
    for (int r = 0; r < c; ++r) {
        const int nslot = layout == 1 ? 2 : 1;
        long long u = 0, pr = 0, t = 0;
        for (int slot = 0; slot < nslot; ++slot) {
            const long long qc = slot == 0 ? r : 2LL * c - 1 - r;  // natural chunk
            const long long a = qc * m;                            // its first position
            u += causal ? qc + 1 : nch;
            pr += causal ? m * a + m * (m + 1) / 2 : m * S;
        }
        // query tiles over the rank's local rows; positions grow with the local row
        for (long long t0 = 0; t0 < n_r; t0 += tile) {
            const long long last = (t0 + tile < n_r ? t0 + tile : n_r) - 1;
            const long long slot = last / m;
            const long long qc = slot == 0 ? r : 2LL * c - 1 - r;
            const long long qmax = qc * m + (last - slot * m);
            for (long long kc = 0; kc < nch; ++kc) {
                if (!causal) {
                    t += kv_tiles_per_chunk;
                } else if (qmax >= kc * m) {
                    const long long n = (qmax - kc * m) / tile + 1;
                    t += n < kv_tiles_per_chunk ? n : kv_tiles_per_chunk;
                }
            }
        }
        if (units) units[r] = u;
        if (pairs) pairs[r] = pr;
        if (tiles) tiles[r] = t;
    }
    return RA_OK;
}

int ringattn_sync_status(ra_stream_t stream) {
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return RA_ERR_CUDA;
    DeviceInfo* dev = nullptr;
    int st = device_info(&dev);
    if (st != RA_OK) return st;
    int rec[4] = {0, 0, 0, 0};
    if (cudaMemcpy(rec, dev->err, sizeof(rec), cudaMemcpyDeviceToHost) != cudaSuccess) return RA_ERR_CUDA;
    if (rec[0] != 0) {
        {
            std::lock_guard<std::mutex> lock(g_mu);
            g_last_timeout[0] = rec[2];
            g_last_timeout[1] = rec[3] >> 10;
            g_last_timeout[2] = rec[3] & 1023;
        }
        const int zero[4] = {0, 0, 0, 0};
        if (cudaMemcpy(dev->err, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return RA_ERR_CUDA;
        // a bounded wait that ran out, or (check build) an index check that failed
        return rec[0] == RA_ERR_BOUNDS ? RA_ERR_BOUNDS : RA_ERR_TIMEOUT;
    }
    return RA_OK;
}

int ringattn_selftest_timeout(long long timeout_ns, ra_stream_t stream) {
    if (timeout_ns < 1000 || timeout_ns > 10000000000LL) return RA_ERR_INVALID_ARG;
    DeviceInfo* dev = nullptr;
    int st = device_info(&dev);
    if (st != RA_OK) return st;
    return ra::launch_selftest_timeout(dev->err, static_cast<unsigned long long>(timeout_ns),
                                       reinterpret_cast<cudaStream_t>(stream));
}

int ringattn_last_timeout(int* info) {
    if (!info) return RA_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    info[0] = g_last_timeout[0];
    info[1] = g_last_timeout[1];
    info[2] = g_last_timeout[2];
    return RA_OK;
}

const char* ringattn_strerror(int status) {
    switch (status) {
        case RA_OK: return "ok";
        case RA_ERR_INVALID_ARG: return "invalid argument";
        case RA_ERR_UNSUPPORTED: return "unsupported shape or size";
        case RA_ERR_ARCH: return "current device is not compute capability 10.3 (sm_103)";
        case RA_ERR_CUDA: return "CUDA runtime error";
        case RA_ERR_TIMEOUT: return "a bounded device wait ran out";
        case RA_ERR_BOUNDS: return "a device index check failed (check build)";
        default: return "unknown status";
    }
}

}  // extern "C"
