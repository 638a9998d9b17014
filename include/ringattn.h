/*
 * ringattn.h -- C ABI of libringattn.so: the per-rank hot path of ring attention
 * (context parallelism) with contiguous or zigzag chunking, all c virtual ranks on
 * one GB300 (sm_103a) GPU.
 *
 * The operation (sources are the pages' titles and sections):
 *  - "Ring Attention and Ulysses shard a sequence two different ways...", section
 *    "Ring Attention: point-to-point rotation, and an online softmax that never sees
 *    the whole row at once": each rank keeps its queries fixed and attends to KV
 *    blocks one hop at a time, merging with a running max, a running sum and a
 *    correction factor exp(old max - new max).
 *  - "Interrogating parallelism, part 5", section "How does attention survive being
 *    split?": rank i sends its KV block to rank i+1, so at hop h rank r holds the
 *    block of rank (r - h) mod c; the merged result is exact.
 *  - same page, section "What breaks the load balance?": contiguous chunking gives
 *    rank i chunk i of c; zigzag chunking gives rank i chunks i and 2c-1-i of 2c.
 *  - "Context & Expert Parallelism", section "Context parallelism: splitting the
 *    sequence": under the causal mask token i attends to every token j <= i.
 *
 * Per (query head h, query position i) every entry point computes, up to rounding,
 *     out[h,i,:] = sum_j softmax_j(q_i . k_j) v_j,   lse[h,i] = ln sum_j exp(q_i . k_j)
 * over the visible keys j (all keys, or j <= i when causal), with kv head h / (Hq/Hkv).
 * No 1/sqrt(d) scale is applied (the pages' rule uses q @ k.T as is); callers that
 * want one scale q before the call.
 *
 * Conventions shared by every entry point:
 *  - Pointers are DEVICE pointers unless stated otherwise; the caller allocates and
 *    owns every buffer.  Inputs are read-only; outputs are fully overwritten.
 *  - Tensors are head-major, [H, S, row] with H = batch * heads (batch folds into
 *    heads: kv head of query head b*Hq+h is b*Hkv + h/g).
 *  - "Rank-major" order stores rank 0's local rows, then rank 1's, ...; a zigzag rank
 *    holds chunk r then chunk 2c-1-r.  ringattn_permute converts from/to natural order.
 *  - layout: 0 = contiguous (c chunks), 1 = zigzag (2c chunks).  causal: 0 or 1.
 *  - kv_block: rows of one simulated ring message; it must divide a chunk
 *    (S/c contiguous, S/(2c) zigzag).  A rank's KV block is split into messages of
 *    kv_block rows, visited in ring order.
 *  - stream: a cudaStream_t (0 = legacy default stream).  Calls are asynchronous:
 *    they validate, enqueue kernels on `stream` and return.
 *  - Errors: every argument is validated on the host before any launch; on a bad
 *    argument the call returns a negative ra_status and touches no device memory.
 *    RA_ERR_ARCH: the current device is not compute capability 10.3.  RA_ERR_CUDA: a
 *    CUDA runtime call or launch failed.  Device-side waits are bounded; one that
 *    runs out records RA_ERR_TIMEOUT, read with ringattn_sync_status.  The limit is
 *    the environment variable RINGATTN_WAIT_TIMEOUT_MS, read once per process (default
 *    2000, clamped to 1000 .. 600000).  It is never below 1 s because the warps that
 *    feed a hardware named barrier (forward P hand-off, backward P^T and dS^T hand-offs)
 *    stop arriving only when it runs out, and the waiting side of such a barrier cannot
 *    give up.  No exception crosses the ABI and there is no CPU fallback.
 *  - Check build: the same sources compiled with -DRA_CHECK give libringattn_check.so,
 *    the same ABI with an index check at every place a kernel derives a memory index
 *    from the chunk and work-item arithmetic (TMA row coordinates, output rows, document
 *    starts, source slabs and rows).  A failed check records RA_ERR_BOUNDS (read with
 *    ringattn_sync_status) and the access is skipped, read as zero, or moved to row 0;
 *    nothing traps.  The normal library never records RA_ERR_BOUNDS.
 *  - The library allocates no device memory per call; scratch it needs is passed in,
 *    except for ringattn_fwd_docmask_noalloc, which uses a static device array.
 *  - The first call of any entry point on a device performs the library's one-time
 *    set-up for that device (its attributes and the device addresses of the library's
 *    static arrays), with that device current; make that first call before any stream
 *    capture begins.
 *  - The fused bf16 kernels (ringattn_fwd*, ringattn_bwd*) hand out their work items
 *    from counters in a static device array of 256 slots: a launch takes the next slot
 *    in turn (the backward takes two) and its last block zeroes it again.  Launches in
 *    flight at the same time on any streams use different slots unless 256 or more of
 *    them are in flight together.  A call captured into a CUDA graph keeps the slot it
 *    took at capture: two executable graphs instantiated from one capture must not run
 *    at the same time.
 */
#ifndef RINGATTN_H
#define RINGATTN_H

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* ra_stream_t; /* same type as cudaStream_t */

typedef enum {
    RA_OK = 0,
    RA_ERR_INVALID_ARG = -1,
    RA_ERR_UNSUPPORTED = -2,
    RA_ERR_ARCH = -3,
    RA_ERR_CUDA = -4,
    RA_ERR_TIMEOUT = -5,
    RA_ERR_BOUNDS = -6
} ra_status;

/*
 * ringattn_fwd -- fused ring attention, bf16 in, fp32 out (tcgen05 tensor cores).
 * q:   [Hq,  S, d] bf16, rank-major.      k, v: [Hkv, S, d] bf16, rank-major.
 * out: [Hq,  S, d] fp32, rank-major.      lse:  [Hq, S] fp32 natural log, rank-major.
 * Every rank's query tiles visit the KV blocks in ring order (hop 0 = own block);
 * each 128-row key tile is one exact online-softmax update (finer than kv_block,
 * which only has to be valid here), and key tiles that the causal mask hides
 * entirely are skipped.
 * Requires d in {64, 128}; S/(c*(layout?2:1)) and kv_block multiples of 128;
 * Hq % Hkv == 0; 16-byte aligned pointers.
 */
int ringattn_fwd(const void* q, const void* k, const void* v, float* out, float* lse,
                 int S, int Hq, int Hkv, int d, int c, int causal, int layout, int kv_block,
                 ra_stream_t stream);

/*
 * ringattn_fwd_rank -- as ringattn_fwd, restricted to the query rows that virtual rank
 * `rank` (0 <= rank < c) holds: its local rows of out and lse are written, every other
 * row is left untouched.  This is one rank's share of the ring ("Interrogating
 * parallelism, part 5", "What breaks the load balance?": under the causal mask rank i
 * of a contiguous split does i+1 units of work, every zigzag rank 2c+1), so timing one
 * call per rank measures the load balance of the two layouts.  Same requirements and
 * rank-major layout as ringattn_fwd; the rows it writes are bitwise those of
 * ringattn_fwd.
 */
int ringattn_fwd_rank(const void* q, const void* k, const void* v, float* out, float* lse,
                      int S, int Hq, int Hkv, int d, int c, int causal, int layout, int kv_block,
                      int rank, ra_stream_t stream);

/*
 * ringattn_fwd_docmask -- all-gathered K/V under a document mask, bf16 in, fp32 out
 * ("Interrogating parallelism, part 5", section "Why did Llama 3 not use a ring?": the
 * keys and values are all-gathered first, then each rank computes attention for its
 * local query chunks; this carries the document mask that keeps attention inside each
 * document of a packed sequence).  For every rank's query rows:
 *     out[h,i,:] = sum_j softmax_j(q_i . k_j) v_j   over j <= i with doc_id[j] == doc_id[i]
 * (causal inside a document), lse as for ringattn_fwd.  Keys are visited in natural
 * order from the first key of the earliest document a query tile touches; key tiles
 * outside every row's document are skipped.
 * q, k, v, out, lse: as ringattn_fwd (rank-major for c and layout; one message per
 * chunk, no kv_block).
 * doc_id:    [S] int32 device, NATURAL order, the document of every position; ids must
 *            not decrease along the sequence (documents packed one after another).  One
 *            packing is shared by every head; batch entries with different packings
 *            are separate calls.  Ids that decrease give an unspecified result (never
 *            an out-of-bounds access).
 * doc_start: [S] int32 device scratch owned by the caller, distinct from doc_id; the
 *            call overwrites it with the first position of every position's document
 *            (computed from doc_id on `stream` before the attention kernel runs).
 * Requirements as ringattn_fwd otherwise: d in {64, 128}, S/(c*(layout?2:1)) a
 * multiple of 128, Hq % Hkv == 0, 16-byte aligned q, k, v, out, lse; 4-byte aligned
 * doc_id and doc_start.
 */
int ringattn_fwd_docmask(const void* q, const void* k, const void* v, float* out, float* lse,
                         const int* doc_id, int* doc_start, int S, int Hq, int Hkv, int d, int c,
                         int layout, ra_stream_t stream);

/*
 * ringattn_fwd_docmask_noalloc -- ringattn_fwd_docmask for callers that cannot allocate
 * device memory.  The pages have no counterpart: this is a convenience of the library.
 *
 * Who needs it: code that must not call cudaMalloc at the point where it runs attention
 * -- for example a host that runs under a fixed memory budget handed out up front, a
 * plug-in whose host process owns every allocation, or code that must not make the
 * implicit device synchronisation cudaMalloc/cudaFree can cause.  Such a caller is
 * handed q, k, v, out, lse and doc_id by whoever owns its memory, but has no way to get
 * the extra [S] int32 scratch that ringattn_fwd_docmask asks for.
 *
 * What it does: exactly ringattn_fwd_docmask, same arguments minus doc_start, same
 * result, with the document starts kept in a static device array inside the library
 * (RINGATTN_DOCMASK_NOALLOC_MAX_S int32 entries, 1 MiB, held by every GPU that loads the
 * library until the process exits).  The call allocates nothing and frees nothing.
 *
 * Limits and sharing:
 *  - S > RINGATTN_DOCMASK_NOALLOC_MAX_S is rejected with RA_ERR_UNSUPPORTED before any
 *    device work; use ringattn_fwd_docmask with caller-owned scratch for longer sequences.
 *  - Every call on a device shares the one array, and the array keeps what the last call
 *    wrote.  Each call rewrites entries [0, S) on `stream` before reading them, so stale
 *    contents never matter to a call on its own; but two calls whose work overlaps on the
 *    GPU (different streams, no ordering between them) race on the array and give wrong
 *    results.  Order such calls on one stream or with events.
 *  - The array's device address is looked up in the library's one-time set-up of each
 *    device, which the first call of any entry point on that device performs (with that
 *    device current); as for every entry point, make that first call before any stream
 *    capture begins.
 * Requirements and errors otherwise as ringattn_fwd_docmask.
 */
#define RINGATTN_DOCMASK_NOALLOC_MAX_S 262144
int ringattn_fwd_docmask_noalloc(const void* q, const void* k, const void* v, float* out, float* lse,
                                 const int* doc_id, int S, int Hq, int Hkv, int d, int c, int layout,
                                 ra_stream_t stream);

/*
 * ringattn_fwd_host -- ringattn_fwd_natural on HOST buffers: copies q, k, v to the device,
 * computes, and copies out and lse back, with the copies overlapped with the attention.
 * The computation is that of ringattn_fwd_natural (same sources, same result); the KV
 * heads are split into G groups (G divides Hkv, at most 16, each group at least four
 * waves of work items), and while group g computes, the inputs of later groups travel
 * host->device and the results of earlier groups device->host.  The launches alternate
 * between `stream` and a compute stream of the library's, so that one group's CTAs start
 * on the SMs the previous group's last CTAs leave; the library creates its streams (one
 * per copy direction and that compute stream) once per device and keeps them until exit.
 * q_h, k_h, v_h: HOST [Hq|Hkv, S, d] bf16, natural order.  out_h: HOST [Hq, S, d] fp32,
 *     lse_h: HOST [Hq, S] fp32, natural order.  Page-locked memory (cudaHostAlloc or
 *     cudaHostRegister) is needed for the copies to run asynchronously and overlap;
 *     pageable memory gives the same result with copies that block the calling thread.
 *     The host buffers must stay valid, and out_h/lse_h unread, until `stream` has
 *     completed the call (e.g. cudaStreamSynchronize(stream)).
 * workspace: DEVICE buffer of at least ringattn_host_workspace_bytes(S, Hq, Hkv, d)
 *     bytes, 256-byte aligned, owned by the caller; it receives the device copies.  Calls
 *     sharing one workspace must be ordered (same stream, or events).
 * stream: the work starts after everything queued on `stream` before the call, and
 *     `stream` completes only after the last result has reached the host.
 * Requirements as ringattn_fwd otherwise.  Arguments are validated before anything is
 * enqueued; RA_ERR_CUDA can leave part of the work enqueued.
 */
int ringattn_fwd_host(const void* q_h, const void* k_h, const void* v_h, float* out_h, float* lse_h,
                      int S, int Hq, int Hkv, int d, int c, int causal, int layout, int kv_block,
                      void* workspace, long long workspace_bytes, ra_stream_t stream);

/*
 * ringattn_host_workspace_bytes -- host only.  Device workspace that ringattn_fwd_host
 * needs for this geometry: q, k, v (bf16) and out, lse (fp32), each rounded up to 256
 * bytes.  Writes the count to *bytes.
 */
int ringattn_host_workspace_bytes(int S, int Hq, int Hkv, int d, long long* bytes);

/*
 * ringattn_relayout -- the data movement of one Ulysses all-to-all, every virtual rank
 * on this GPU ("Ring Attention and Ulysses shard a sequence two different ways...",
 * section "Ulysses: an all-to-all relayout instead of a rotation": an all-to-all swaps
 * the sequence-sharded layout for a head-sharded one, and back after attention).
 *   sequence-sharded: [S, H, row] -- tokens in rank-major order (rank r's tokens are its
 *       chunk for `layout`: contiguous chunk r, or zigzag chunks r then 2c-1-r), heads
 *       inner: each rank's shard is its tokens with every head, as an activation is held;
 *   head-sharded:     [H, S, row] -- heads outer, tokens in natural order: rank r's share
 *       is heads [r*H/c, (r+1)*H/c) over the whole sequence.
 * to_heads = 1 moves src (sequence-sharded) to dst (head-sharded); 0 the reverse.  A row
 * is one (token, head) vector of row_bytes bytes.  Bit-exact copy; every dst byte is
 * written.  src and dst must not overlap.
 * Requires row_bytes a multiple of 4 and 4-byte aligned src, dst (16-byte rows on
 * 16-byte aligned buffers move as 16-byte vectors), S a multiple of the chunk count,
 * (S/chunks) * H * row_bytes/4 < 2^31 and H * chunks < 65536 (else RA_ERR_UNSUPPORTED).
 */
int ringattn_relayout(const void* src, void* dst, int S, int H, int row_bytes, int c, int layout,
                      int to_heads, ra_stream_t stream);

/*
 * ringattn_ulysses_fwd -- attention by Ulysses' scheme, every virtual rank on this GPU
 * (same page and section as ringattn_relayout): relayout q, k, v from sequence shards to
 * head shards, attend every rank's heads over the whole sequence (one launch of the fused
 * kernel for all ranks, natural order, no ring), relayout out and lse back.  The result
 * is the same attention as ringattn_fwd's, in the sequence-sharded layout.
 * q_seq: [S, Hq, d] bf16, k_seq, v_seq: [S, Hkv, d] bf16, out_seq: [S, Hq, d] fp32,
 *     lse_seq: [S, Hq] fp32 -- all sequence-sharded (rank-major tokens, heads inner).
 * Rank r takes query heads [r*Hq/c, (r+1)*Hq/c), so Hq % c == 0; it uses the KV heads of
 * those query heads (h / (Hq/Hkv)), which puts one KV head on c/Hkv ranks when c > Hkv
 * (on one GPU each KV head is stored once).
 * workspace: DEVICE, at least ringattn_host_workspace_bytes(S, Hq, Hkv, d) bytes,
 *     256-byte aligned, caller-owned: it holds the head-sharded q, k, v, out, lse.
 * Requires d in {64, 128}, S a multiple of 128 and of the chunk count, 16-byte aligned
 * q_seq, k_seq, v_seq, out_seq and 4-byte aligned lse_seq.
 */
int ringattn_ulysses_fwd(const void* q_seq, const void* k_seq, const void* v_seq, float* out_seq,
                         float* lse_seq, int S, int Hq, int Hkv, int d, int c, int causal, int layout,
                         void* workspace, long long workspace_bytes, ra_stream_t stream);

/*
 * ringattn_bwd -- gradients of ringattn_fwd with respect to q, k and v (bf16 in, fp32 out).
 * The pages give no backward pass (the training FLOP count of "Interrogating parallelism,
 * part 5" implies one); this computes the exact gradient of the forward's attention:
 * with P_ij = exp(q_i . k_j - lse_i) over visible keys, D_i = dout_i . out_i and
 * dS_ij = P_ij (dout_i . v_j - D_i):
 *     dq_i = sum_j dS_ij k_j,   dk_j = sum_i dS_ij q_i,   dv_j = sum_i P_ij dout_i,
 * a KV head summing over the query heads that use it.  The ring order is kept: each query
 * tile meets the KV blocks hop by hop, and each KV block travels the ring with its dk, dv
 * accumulators (only the order of fp32 sums depends on it).  P and dS are rounded to bf16
 * for the tensor-core products; all sums are fp32.
 * q, k, v, dout: bf16, rank-major as in ringattn_fwd (dout: [Hq, S, d]).
 * out, lse: ringattn_fwd's outputs for these q, k, v (fp32, rank-major).
 * dq: [Hq, S, d], dk, dv: [Hkv, S, d] fp32, rank-major, fully overwritten.
 * delta: [Hq, S] fp32 DEVICE scratch owned by the caller; overwritten with D.
 * Requirements as ringattn_fwd (d in {64, 128}, chunks and kv_block multiples of 128,
 * Hq % Hkv == 0), every pointer 16-byte aligned.
 */
int ringattn_bwd(const void* q, const void* k, const void* v, const float* out, const float* lse,
                 const void* dout, float* dq, float* dk, float* dv, float* delta, int S, int Hq,
                 int Hkv, int d, int c, int causal, int layout, int kv_block, ra_stream_t stream);

/*
 * ringattn_bwd_natural -- as ringattn_bwd with every tensor (q, k, v, out, lse, dout, dq, dk,
 * dv, delta) in NATURAL sequence order: the chunk map is applied in the kernels' tile
 * addressing, as in ringattn_fwd_natural.  Same result, same requirements.
 */
int ringattn_bwd_natural(const void* q, const void* k, const void* v, const float* out,
                         const float* lse, const void* dout, float* dq, float* dk, float* dv,
                         float* delta, int S, int Hq, int Hkv, int d, int c, int causal, int layout,
                         int kv_block, ra_stream_t stream);

/*
 * ringattn_fwd_natural -- as ringattn_fwd, but q, k, v, out and lse are in NATURAL
 * sequence order: the zigzag/contiguous chunk map is applied in the kernel's tile
 * addressing, so no permutation pass is needed.  Same result, same requirements.
 */
int ringattn_fwd_natural(const void* q, const void* k, const void* v, float* out, float* lse,
                         int S, int Hq, int Hkv, int d, int c, int causal, int layout,
                         int kv_block, ra_stream_t stream);

/*
 * ringattn_fwd_f32 -- the same computation in fp32 with FFMA (no tensor cores), one
 * online update per kv_block message exactly as the pages' rule.  Any 1 <= d <= 128;
 * S divisible by the chunk count; kv_block divides a chunk.  Rank-major layout.
 */
int ringattn_fwd_f32(const float* q, const float* k, const float* v, float* out, float* lse,
                     int S, int Hq, int Hkv, int d, int c, int causal, int layout, int kv_block,
                     ra_stream_t stream);

/*
 * ringattn_fwd_hop / ringattn_fwd_hop_f32 -- one ring message: every rank attends
 * to message `sub` (0 <= sub < (S/c)/kv_block) of the KV block it holds at hop `hop`
 * (0 <= hop < c) and writes the normalised partial o_part [Hq,S,d] fp32 and its
 * log-sum-exp lse_part [Hq,S] fp32 (rank-major).  Rows that see no key in that
 * message get o_part = 0 and lse_part = -inf.  Folding every message's partial
 * into a running (out, lse) with ringattn_merge, in ring order, gives ringattn_fwd's
 * result.  Requirements as ringattn_fwd (bf16) or ringattn_fwd_f32.
 */
int ringattn_fwd_hop(const void* q, const void* k, const void* v, float* o_part, float* lse_part,
                     int S, int Hq, int Hkv, int d, int c, int causal, int layout, int kv_block,
                     int hop, int sub, ra_stream_t stream);
int ringattn_fwd_hop_f32(const float* q, const float* k, const float* v, float* o_part,
                         float* lse_part, int S, int Hq, int Hkv, int d, int c, int causal,
                         int layout, int kv_block, int hop, int sub, ra_stream_t stream);

/*
 * ringattn_merge -- exact merge of a partial into a running result, in place:
 *   lse' = ln(exp(lse_run) + exp(lse_part))
 *   o'   = o_run * exp(lse_run - lse') + o_part * exp(lse_part - lse')
 * ("Interrogating parallelism, part 5", "How does attention survive being split?":
 * partials over disjoint key sets combine exactly).  A partial with lse = -inf has
 * weight 0; two -inf partials give o = 0, lse = -inf.  rows >= 0 rows of d fp32
 * (any 1 <= d <= 4096); o_run/lse_run are read and overwritten.  To start a ring,
 * fill o_run with 0 and lse_run with -inf (or copy the first partial).
 */
int ringattn_merge(float* o_run, float* lse_run, const float* o_part, const float* lse_part,
                   long long rows, int d, ra_stream_t stream);

/*
 * ringattn_permute -- move rows between natural and rank-major order.
 * src, dst: [H, S, row_bytes] bytes, distinct buffers.  inverse = 0: natural ->
 * rank-major; 1: rank-major -> natural.  row_bytes >= 1 (2*d for bf16 Q/K/V, 4*d
 * for fp32 out, 4 for lse).  Bit-exact copy ("What breaks the load balance?": the
 * zigzag assignment is index bookkeeping only).
 */
int ringattn_permute(const void* src, void* dst, int S, int H, int row_bytes, int c, int layout,
                     int inverse, ra_stream_t stream);

/*
 * ringattn_rank_work -- host only, no device use.  Per rank r < c (each output array
 * has c entries; any may be NULL), for one head:
 *   units[r] -- (query chunk, key chunk) pairs with a visible key, the pages' count
 *               (contiguous causal: r+1; zigzag causal: 2c+1);
 *   pairs[r] -- visible (query, key) pairs;
 *   tiles[r] -- (query tile, key tile) pairs of `tile` rows with a visible pair, the
 *               tiles the fused kernel computes when tile = 128.
 */
int ringattn_rank_work(int S, int c, int causal, int layout, int tile, long long* units,
                       long long* pairs, long long* tiles);

/*
 * ringattn_sync_status -- synchronise `stream`, then return RA_ERR_TIMEOUT if a
 * bounded device wait of any earlier call on the current device ran out, or (check
 * build only) RA_ERR_BOUNDS if an index check failed; the record is cleared.  Returns
 * RA_ERR_CUDA if the synchronisation failed, else RA_OK.
 */
int ringattn_sync_status(ra_stream_t stream);

/*
 * ringattn_selftest_timeout -- launch one tiny kernel whose single wait is on a
 * barrier that nothing signals, bounded by timeout_ns (1e3 .. 1e10).  The kernel gives
 * up, records RA_ERR_TIMEOUT and exits, leaving the context usable; the caller reads
 * the record with ringattn_sync_status.  Exists to test the failure path.
 */
int ringattn_selftest_timeout(long long timeout_ns, ra_stream_t stream);

/*
 * ringattn_last_timeout -- host only.  Where the last device error that
 * ringattn_sync_status reported happened: info[0] = shared-memory address of the barrier
 * whose wait ran out (RA_ERR_TIMEOUT) or the number of the index check that failed
 * (RA_ERR_BOUNDS), info[1] = CTA index, info[2] = thread index within the CTA (all 0 if
 * none yet).
 * info must hold 3 ints.  A diagnostic for reports; the values are not stable across
 * library versions.
 */
int ringattn_last_timeout(int* info);

/* ringattn_strerror -- static description of a status code. */
const char* ringattn_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* RINGATTN_H */
