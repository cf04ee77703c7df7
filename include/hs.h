/*
 * hs.h -- C ABI of the HiSparse swap-in path on one GB300 GPU.
 *
 * The operation (HiSparse blog, section "Efficient swap-in kernel"; the
 * papercache summary of it, section 2 "Method", steps 1-3): for every request
 * at every decode step, take the indexer's top-k token indices and
 *   (1) find which of them miss in the request's hot device buffer,
 *   (2) choose eviction victims by LRU among the slots not hit this step,
 *   (3) update the token->slot page table, the slot->token table and the
 *       per-slot last-use stamps, and fetch each missing KV row from the
 *       pinned host pool into its victim slot.
 * The result is a [B, K] list of buffer slots that a sparse-attention kernel
 * reads.  With a resident tail (vLLM "Hybrid HiSparse" post, section "Mixed
 * Residency"), tokens in the last T positions of the context live on the
 * device and resolve in place; a request starts with an empty buffer (same
 * post, "No Residency").
 *
 * Exact semantics (the library reproduces them bit for bit):
 *   - one token per page; stamps hold the step of last use (steps count from
 *     1, stamp 0 = never used); a hit refreshes its slot's stamp;
 *   - victims are the m slots not hit this step with the smallest
 *     (stamp, slot index) pairs -- ties go to the lowest slot index; the i-th
 *     miss in top-k row order is paired with the i-th victim in ascending slot
 *     order;
 *   - a tail token t (C - T <= t < len) resolves to slot S + (t mod T) and
 *     touches no table; it counts as neither hit nor miss;
 *   - index -1 is padding (out = -1).  An index < -1 or >= the request's
 *     current length, or a repeat of an earlier index in the same row, is a
 *     device-side input error: out = -1 for that entry, the state is left as
 *     if the entry were absent, and an error bit is latched (hs_stats).
 *
 * Layouts (row-major, all int32 unless stated):
 *   topk_idx, out_slot         [B][K]
 *   token->slot table          [B][C]        (-1 = not in the buffer)
 *   slot->token table, stamps  [B][S]
 *   device buffer (uint8)      [B][S + T][R] (slots [0,S) hot, [S,S+T) tail)
 *   host pool (uint8, pinned and mapped)  [B][H][R], H = host_ratio * S,
 *                              row t of request b holds token t (t < C - T)
 *
 * Ownership: the library allocates and frees everything in a handle (device
 * tables, buffer, scratch, pinned host pool).  Pointers passed in by the
 * caller stay the caller's and must remain valid until the stream reaches the
 * work that uses them.  A handle is bound to the device that was current at
 * hs_create; calls switch to that device and restore the caller's.
 *
 * Errors: host-side checks return a negative HS_ERR_* synchronously and
 * enqueue nothing.  Device-side input errors never trap; they are latched in
 * the handle's error word (HS_E_* bits, read by hs_stats).
 *
 * Streams: hs_stream_t is cudaStream_t (NULL = the legacy default stream).
 * hs_resolve, hs_resolve_multi, hs_resolve_layers, hs_append and
 * hs_reset_requests only enqueue work (no host synchronisation, no
 * allocation), so a sequence of them can be captured in a CUDA graph.
 * Calls that read or set state from the host (hs_stats, hs_export_*,
 * hs_import_state, hs_set_lengths, hs_set_tail_rows, hs_reset) synchronise
 * the device first.
 */
#ifndef HS_H
#define HS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct hs_handle hs_handle;
typedef struct CUstream_st* hs_stream_t;

/* Return codes. */
#define HS_OK                 0
#define HS_ERR_ARG           -1  /* bad size, null pointer, or bad handle */
#define HS_ERR_TOPK_GT_SLOTS -2  /* K > buffer_slots: the LRU step needs K <= S */
#define HS_ERR_CAPACITY      -3  /* host pool too small: host_ratio * S < ctx_len - resident_tail */
#define HS_ERR_ALLOC         -4  /* device or pinned host allocation failed */
#define HS_ERR_CUDA          -5  /* a CUDA runtime call or launch failed */
#define HS_ERR_LIMIT         -6  /* a size beyond the kernels' limits below */

/* Device-side error bits (hs_stats_t.err_bits). */
#define HS_E_RANGE   1  /* an index < -1 or >= the request's current length */
#define HS_E_DUP     2  /* an index repeated within one top-k row */
#define HS_E_APPEND  4  /* hs_append with no room in the resident tail */
#define HS_E_STATE   8  /* inconsistent state met and repaired for this step
                           (caller-owned tables of hs_resolve_noalloc, or a step
                           counter run past HS_MAX_STEP): a step counter outside
                           [0, HS_MAX_STEP) or a stamp outside [0, step - 1] was
                           clamped, a token->slot entry outside [-1, S) was taken
                           as a miss, or a slot->token entry outside [-1, C) was
                           not written through.  Results stay in range; LRU
                           order among the repaired entries is unspecified. */

/* Kernel limits.  The step counter runs up to HS_MAX_STEP (stamps and the
 * in-kernel claim of a slot, step + K, stay below 2^31). */
#define HS_MAX_STEP       0x7fffefff
#define HS_MAX_TOPK       4096
#define HS_MAX_SLOTS      16384
#define HS_MAX_BATCH      4096
#define HS_MAX_ROW_BYTES  65536
#define HS_MAX_LAYERS     16      /* handles per hs_resolve_layers call */

typedef struct {
    int64_t steps;         /* resolves issued on the handle (its step counter) */
    int64_t hits;          /* cumulative buffer hits */
    int64_t misses;        /* cumulative misses (= rows fetched from host) */
    int64_t inplace;       /* cumulative resident-tail resolves */
    int64_t bytes_copied;  /* misses * row_bytes */
    int32_t err_bits;      /* HS_E_* latched since create / reset */
    int32_t reserved;
} hs_stats_t;

/*
 * Create the swap-in state for `batch` requests of one layer.
 *   ctx_len        C, capacity in tokens (valid positions [0, C))
 *   row_bytes      R, bytes per KV row; a multiple of 16
 *   buffer_slots   S, hot-buffer slots per request (SGLang's device_buffer_size)
 *   host_ratio     H = host_ratio * S host rows per request (SGLang's
 *                  host_to_device_ratio); must cover C - resident_tail
 *   resident_tail  T >= 0, device-resident tail tokens (0 = no mixed residency)
 * All tables start empty, stamps 0, step 0, every request's length = C
 * (use hs_set_lengths for a growing context).  The host pool is allocated
 * but not filled: write the cold rows through hs_host_pool before resolving
 * (its placement follows hs_set_host_pool_pages).
 * Returns HS_OK and *out, or an HS_ERR_* code (then *out = NULL).
 * Source: HiSparse blog, "ベンチマークテスト" (the deployment's top_k,
 * device_buffer_size and host_to_device_ratio); vLLM Hybrid HiSparse post,
 * "Mixed Residency" (the device-resident tail) and "メモリ管理と統合" (a hot
 * buffer of 2x top-K rows per request by default).
 */
int hs_create(int batch, int ctx_len, int row_bytes, int buffer_slots, int host_ratio,
              int resident_tail, hs_handle** out);

/* Free everything the handle owns.  Synchronises the device first.  NULL is a no-op.
 * Source: no passage (the handle's lifetime; the pages define no API). */
void hs_destroy(hs_handle* h);

/*
 * One decode step for all B requests: resolve topk_idx (device, [B][K]) into
 * out_slot (device, [B][K]) and fetch every missing row from the host pool
 * into the device buffer, on `stream`.  1 <= K <= min(S, HS_MAX_TOPK).
 * Asynchronous; graph-capturable.  Calls on one handle must be ordered (one
 * stream, or streams joined by events): each step reads the state the
 * previous step wrote.
 * Source: HiSparse blog, "効率的なSwap-inカーネル", steps (1)-(3); papercache
 * summary, section 2 "方法细节"; vLLM Hybrid HiSparse post, "Mixed Residency"
 * (tail tokens in place, a hit refreshes its LRU entry, a miss copies one row
 * from pinned host memory into the LRU slot, no wait on the CPU) and "No
 * Residency" (a request starts with an empty buffer).
 */
int hs_resolve(hs_handle* h, const int32_t* topk_idx, int K, int32_t* out_slot,
               hs_stream_t stream);

/*
 * Several draft positions in one step (speculative decoding; vLLM Hybrid
 * HiSparse post, "Speculative Decoding": a per-step resolver plan over the
 * request's shared hot state).  topk_idx (device, [B][P][K]) holds P top-k
 * rows per request; they are resolved as one row of P*K entries, and a
 * repeated token -- across positions or within one -- is not an error: it
 * gets the slot of its first occurrence and is fetched and counted once.
 * out_slot is [B][P][K].  1 <= P*K <= min(S, HS_MAX_TOPK).  A retried step
 * is simply another call.  Asynchronous; graph-capturable.
 * Source: vLLM Hybrid HiSparse post, "vLLM エコシステムとの統合", item
 * "Speculative Decoding".
 */
int hs_resolve_multi(hs_handle* h, const int32_t* topk_idx, int P, int K, int32_t* out_slot,
                     hs_stream_t stream);

/*
 * The step of L independent layers in one launch.  The pages name better
 * overlap of the miss I/O with other work as the way to cut its overhead
 * (HiSparse blog, section "今後の展望" (outlook)): here the CTAs of all
 * layers share the GPU, so while some resolve their tables others fetch
 * rows, and a layer's idle start is hidden behind the others' copies.
 * handles, topk_idx and out_slot are HOST arrays of L entries: handle l
 * resolves topk_idx[l] (device, [B][K]) into out_slot[l] (device, [B][K])
 * with exactly the result of hs_resolve on that handle.  The handles must be
 * distinct, made on one device, and share B, S and row_bytes; their
 * context length, tail, policy and tail mode may differ.  One fused launch of
 * L * B CTAs whatever the handles' copy mode.  1 <= L <= HS_MAX_LAYERS,
 * 1 <= K <= min(S, HS_MAX_TOPK).  Prefer it, or hs_resolve per layer on one
 * stream, to hs_resolve per layer on concurrent streams: several cluster
 * launches reading large pools at once ran slower than the same launches in
 * sequence (measured: 64 requests x 4 layers of 9.5 GB pools, 1.0 ms per step
 * on a stream per layer against 0.57 ms on one stream and 0.54 ms here).
 * Asynchronous; graph-capturable.  Errors:
 * HS_ERR_ARG (a NULL array, entry or handle, a handle given twice, shapes
 * that differ, another device), HS_ERR_TOPK_GT_SLOTS, HS_ERR_LIMIT.
 * Source: HiSparse blog, "今後の展望", and papercache summary, section 4
 * "结论与未来工作" (better overlap as the way to cut the miss I/O overhead);
 * the per-layer step is hs_resolve's.
 */
int hs_resolve_layers(hs_handle* const* handles, int L, const int32_t* const* topk_idx, int K,
                      int32_t* const* out_slot, hs_stream_t stream);

/*
 * hs_resolve_layers from host memory: topk_idx[l] and out_slot[l] are host
 * buffers ([B][K] each), with the same rules as hs_resolve_host (mapped
 * pinned buffers are read and written by the kernel directly, others are
 * staged); synchronises the stream before returning.  Not graph-capturable.
 * Every check of hs_resolve_layers is made before anything is staged or
 * enqueued.
 * Source: as hs_resolve_layers; the host buffers are this library's end-to-end
 * entry, with no passage of their own.
 */
int hs_resolve_layers_host(hs_handle* const* handles, int L, const int32_t* const* topk_idx, int K,
                           int32_t* const* out_slot, hs_stream_t stream);

/*
 * The same step from host memory: topk_idx (host, [B][K]) in, out_slot (host,
 * [B][K]) out; synchronises the stream before returning.  When both buffers
 * are page-locked and mapped into the device address space (cudaHostAlloc,
 * cudaMallocHost, or cudaHostRegister with mapping), the kernels read and
 * write them across the host link directly (every CTA of a request's cluster
 * reads its top-k row, so with the default cluster size this call launches
 * clusters of at most 4 CTAs above HS_CLUSTER_WIDE_BATCH requests); otherwise
 * they are staged
 * through device buffers with two cudaMemcpyAsync.  The choice follows
 * cudaHostGetDevicePointer: on a system whose GPU addresses pageable host
 * memory (a Grace host), it can accept ordinary malloc'd buffers too, and
 * those are then read and written in place as well.  Not graph-capturable
 * (it synchronises).
 * Source: as hs_resolve; the host buffers are this library's end-to-end
 * entry, with no passage of their own.
 */
int hs_resolve_host(hs_handle* h, const int32_t* topk_idx, int K, int32_t* out_slot,
                    hs_stream_t stream);

/*
 * Copy-engine variant of hs_resolve, kept for comparison with the zero-copy
 * row fetch.  The resolve kernel writes the miss lists; the host reads the
 * miss tokens back (one stream synchronisation per call), gathers the
 * missing rows from the pinned pool into a pinned staging area with host
 * threads, moves the whole area with one cudaMemcpyAsync, and a kernel
 * writes every row into its victim slot.  Results are identical to
 * hs_resolve.  Not graph-capturable.  The first call allocates the staging
 * areas (B * min(S, HS_MAX_TOPK) rows on the host and on the device) and
 * starts the host threads.
 * Source: HiSparse blog, "効率的なSwap-inカーネル", step (3) (fetch the
 * needed entries from host into device memory), done here by the copy engine
 * instead of the kernel, for comparison.
 */
int hs_resolve_ce(hs_handle* h, const int32_t* topk_idx, int K, int32_t* out_slot,
                  hs_stream_t stream);

/*
 * Read the counters and, if last_miss is not NULL, the last step's miss count
 * of every request (host, [B]).  Synchronises the device first.
 * Source: HiSparse blog, "効率的なSwap-inカーネル" (the figure of miss counts
 * against hot-buffer size and eviction strategy: misses are the path's own
 * measure).
 */
int hs_stats(hs_handle* h, hs_stats_t* out, int32_t* last_miss);

/* Host pointer of the pinned, device-mapped host pool [B][H][R]; its size in bytes.
 * Source: HiSparse blog, "HiSparseの設計" (inactive KV entries are offloaded to
 * host memory); vLLM Hybrid HiSparse post, "Mixed Residency" (pinned host memory). */
uint8_t* hs_host_pool(hs_handle* h);
size_t hs_host_pool_bytes(hs_handle* h);

/*
 * Where hs_create places host pools, for the whole process (later handles
 * only; a handle keeps the pool it was created with):
 *   HS_POOL_PAGES_AUTO  (default) a pool of at least HS_POOL_HUGE_MIN_BYTES
 *                       and one transparent huge page (hs_huge_page_bytes)
 *                       goes into anonymous memory aligned to that size and
 *                       advised for huge pages, then is page-locked and mapped
 *                       with cudaHostRegister; smaller pools come from
 *                       cudaHostAlloc(..., cudaHostAllocMapped)
 *   HS_POOL_PAGES_BASE  always cudaHostAlloc
 *   HS_POOL_PAGES_HUGE  the huge-page placement for any non-empty pool, when
 *                       the host has huge pages
 * A huge-page pool prefers the host NUMA node nearest the GPU
 * (cudaDevAttrHostNumaId, when the device names one) and is not inherited by
 * forked children (MADV_DONTFORK; a cudaHostAlloc pool is not either).  The
 * huge-page placement falls back to cudaHostAlloc when mmap or the
 * registration fails; whether the kernel backs the range with huge pages
 * depends on its free memory.  Why it matters: with base pages, a pool of tens
 * of GB whose rows are read by several SMs per request (cluster and split
 * launches) spends much of a step on address translation; huge pages let the
 * GPU map it with large pages.  The first seconds of steps on a huge-page pool
 * are slow and uneven (measured; the cause is not known), hence the size
 * floor.  Either placement is pinned, mapped and read the same way, with
 * bit-identical results.  Returns HS_OK or HS_ERR_ARG
 * (unknown mode).  hs_host_pool_pages reports a handle's placement
 * (HS_POOL_PAGES_HUGE or HS_POOL_PAGES_BASE); hs_huge_page_bytes is the host's
 * transparent huge page size (0: none).
 * Source: no passage (host memory placement; the pages keep cold KV in
 * pinned host memory without saying how it is mapped).
 */
#define HS_POOL_HUGE_MIN_BYTES (1ull << 34) /* 16 GiB */
#define HS_POOL_PAGES_AUTO 0
#define HS_POOL_PAGES_BASE 1
#define HS_POOL_PAGES_HUGE 2
int hs_set_host_pool_pages(int mode);
int hs_host_pool_pages(hs_handle* h);
size_t hs_huge_page_bytes(void);

/* Device pointer of the buffer [B][S+T][R] that out_slot indexes; its size in bytes.
 * Source: HiSparse blog, "HiSparseの設計" (the hot device buffer in HBM);
 * vLLM Hybrid HiSparse post, "Mixed Residency" (the tail stays on the GPU). */
uint8_t* hs_device_buffer(hs_handle* h);
size_t hs_device_buffer_bytes(hs_handle* h);

/*
 * Set the current length of every request (host, [B]; each in [0, C]).
 * Setup only: synchronises the device first.
 * Source: vLLM Hybrid HiSparse post, "エージェント的ワークロードにおける KV
 * キャッシュ圧迫の解決" (contexts that grow over time) and "Mixed Residency".
 */
int hs_set_lengths(hs_handle* h, const int32_t* len_host);

/*
 * Mixed residency, growing context: for every request b write row b of
 * rows_dev (device, [B][R]) as token len[b] into tail slot S + (len[b] mod T)
 * and advance len[b].  With a fixed tail, a request whose next token is
 * outside [C - T, C) is left unchanged and HS_E_APPEND is latched; with a
 * sliding tail (hs_set_tail_mode) only len[b] = C is refused, and the token
 * leaving the tail is first written back to the host pool.  Asynchronous;
 * graph-capturable.  Requires T > 0.
 * Source: vLLM Hybrid HiSparse post, "Mixed Residency" (the request's tail
 * stays on the GPU) and "Full Residency" (pages copied to host memory ahead
 * of eviction, the sliding tail's write-back).
 */
int hs_append(hs_handle* h, const uint8_t* rows_dev, hs_stream_t stream);

/*
 * Setup only: write tokens [first_token, first_token + n) of request b from
 * rows_host (host, [n][R]) into their tail slots S + (t mod T).  All tokens
 * must lie in [C - T, C).  Synchronous.
 * Source: vLLM Hybrid HiSparse post, "Mixed Residency" (the tail rows live
 * on the device).
 */
int hs_set_tail_rows(hs_handle* h, int b, int first_token, int n, const uint8_t* rows_host);

/*
 * Copy the state to host memory (any pointer may be NULL to skip it):
 * tok_slot [B][C], slot_tok [B][S], stamp [B][S], step (one int32).
 * Synchronises the device first.
 * Source: no passage (a test, checkpoint and resume aid).
 */
int hs_export_state(hs_handle* h, int32_t* tok_slot, int32_t* slot_tok, int32_t* stamp,
                    int32_t* step);

/*
 * Resume from a saved state: load tok_slot [B][C], slot_tok [B][S], stamp
 * [B][S] (host arrays, the layout hs_export_state writes) and the step
 * counter.  The state is checked on the host first and refused with
 * HS_ERR_ARG unless it is one the path can reach: slot -> token entries in
 * [-1, C - T), token -> slot entries in [-1, S) and -1 for tail tokens, the
 * two maps inverse to each other, every stamp in [0, step], 0 <= step <= HS_MAX_STEP.
 * Buffer bytes are not part of the state (write them, or let misses refill
 * them).  Counters and error bits are cleared.  Synchronous.
 * Source: no passage (a test, checkpoint and resume aid).
 */
int hs_import_state(hs_handle* h, const int32_t* tok_slot, const int32_t* slot_tok,
                    const int32_t* stamp, int32_t step);

/* Copy request b's buffer rows [S+T][R] to host memory.  Synchronous.
 * Source: no passage (a test, checkpoint and resume aid). */
int hs_export_buffer(hs_handle* h, int b, uint8_t* dst_host);

/* Back to the start state: empty tables, stamps 0, step 0, counters and error bits 0,
 * lengths = C.  The host pool and buffer bytes are kept.  Synchronous.
 * Source: vLLM Hybrid HiSparse post, "No Residency" (the start state: placeholders
 * only, rows loaded when the indexer selects them). */
int hs_reset(hs_handle* h);

/*
 * Give batch slots to new requests (continuous batching).  A request starts
 * with an empty hot buffer and loads rows only when the indexer selects them
 * (vLLM Hybrid HiSparse post, "No Residency").  For each of the n entries of
 * req_ids (device, int32 [n]), request b = req_ids[i] gets token->slot all -1,
 * slot->token all -1, stamps 0 and length lengths[i] (device, int32 [n]; NULL
 * means C).  Its host-pool rows and resident-tail rows are the caller's to
 * write (hs_host_pool; hs_set_tail_rows or hs_append); its buffer bytes are
 * left as they are and are never read before a miss refills them.  Other
 * requests, the step counter and the counters are untouched.  An id outside
 * [0, B) or a length outside [0, C] is skipped and latches HS_E_RANGE; a
 * repeated id is reset once more.  0 <= n <= HS_MAX_BATCH.  Asynchronous and
 * graph-capturable, ordered with the handle's other calls by the stream.
 * Source: vLLM Hybrid HiSparse post, "No Residency".
 */
int hs_reset_requests(hs_handle* h, const int32_t* req_ids, int n, const int32_t* lengths,
                      hs_stream_t stream);

/*
 * Measurement helper: stream `bytes` (a multiple of 16) from pinned host
 * memory `src_host` (allocated with cudaHostAlloc(..., cudaHostAllocMapped)
 * or returned by hs_host_pool) into device memory `dst_dev` with 128-bit
 * zero-copy loads -- the access pattern of the row fetch, but sequential.
 * `blocks` = 0 picks the default grid.  Asynchronous.
 * Source: HiSparse blog, "今後の展望" (the CPU-GPU bandwidth of Grace
 * Blackwell systems bounds the miss I/O); this probe measures it.
 */
int hs_h2d_read(const void* src_host, void* dst_dev, size_t bytes, int blocks,
                hs_stream_t stream);

/*
 * How the step is launched (all give identical results):
 *   HS_COPY_FUSED    one kernel; each request's CTA resolves its row and then
 *                    fetches its own missing rows from the host pool;
 *   HS_COPY_SPLIT    a resolve kernel, then a grid-wide copy kernel over the
 *                    misses of all requests;
 *   HS_COPY_CLUSTER  one kernel with a thread-block cluster of several CTAs
 *                    per request: the first CTA resolves the row, the others
 *                    read its miss list from distributed shared memory, load
 *                    their first rows while it chooses the victims, and the
 *                    cluster copies the rows together (more SMs per request
 *                    than FUSED, one launch unlike SPLIT);
 *   HS_COPY_AUTO     (default) cluster when B <= HS_CLUSTER_MAX_BATCH and the
 *                    device runs a cluster size of 2 or more for the handle
 *                    (hs_cluster_size); beyond HS_CLUSTER_MAX_BATCH requests
 *                    fused.  Without such a cluster size: fused when
 *                    B >= HS_FUSED_MIN_BATCH, or when one
 *                    request's hot buffer (S * row_bytes) is at most
 *                    HS_FUSED_MAX_REQUEST_BYTES, so that no step gives one CTA
 *                    much to copy; split otherwise.  A function of the handle
 *                    alone, so hs_resolve_launches answers per handle.
 * Source: HiSparse blog, "効率的なSwap-inカーネル" (one dedicated kernel does
 * steps (1)-(3)); the split and cluster forms are this library's, with no
 * passage.
 */
#define HS_COPY_AUTO     0
#define HS_COPY_FUSED    1
#define HS_COPY_SPLIT    2
#define HS_COPY_CLUSTER  3
#define HS_FUSED_MIN_BATCH 16
#define HS_FUSED_MAX_REQUEST_BYTES (1 << 20)
#define HS_MAX_CLUSTER   16
#define HS_CLUSTER_WIDE_BATCH 4
#define HS_CLUSTER_MAX_BATCH 128
int hs_set_copy_mode(hs_handle* h, int mode);

/*
 * CTAs of the split mode's grid-wide copy kernel (HS_COPY_SPLIT, and the
 * copy-engine variant's scatter): n = 0 (default) launches one per SM times
 * the kernel's occupancy; 1 <= n <= HS_MAX_COPY_CTAS launches n.  Every n
 * gives the same results.  A small grid leaves the other SMs to kernels on
 * other streams while the rows cross the host link, which a few dozen CTAs
 * keep busy: the overlap of the miss I/O with other work.  When the step runs
 * beside compute on other streams, HS_COPY_SPLIT with about 48 copy CTAs (or
 * HS_COPY_FUSED for a small batch) overlaps far better than the default
 * cluster launch, which takes every SM while it runs.  Returns HS_OK or
 * HS_ERR_ARG.
 * Source: HiSparse blog, "今後の展望", and papercache summary, section 4
 * "结论与未来工作" (overlapping the miss I/O with other work as the way to cut
 * its overhead).
 */
#define HS_MAX_COPY_CTAS 65535
int hs_set_copy_ctas(hs_handle* h, int n);

/*
 * Eviction policy (HiSparse blog, "Efficient swap-in kernel": the miss count
 * depends on the buffer size and the eviction strategy):
 *   HS_POLICY_LRU   victims are the least recently used slots; a hit
 *                   refreshes its slot's stamp (default);
 *   HS_POLICY_FIFO  victims are the slots filled longest ago; a hit keeps its
 *                   slot's fill stamp (the slot is still not evicted in the
 *                   step that hits it);
 *   HS_POLICY_RANDOM  victims are a uniform random choice among the slots not
 *                   hit this step, empty slots first: each slot gets a key, 0
 *                   when empty, else 1 + the top 30 bits of one SplitMix64
 *                   output (Steele, Lea and Flood, OOPSLA 2014) of the state
 *                   seed XOR (step << 32 | request << 14 | slot), and the
 *                   victims are the smallest (key, slot) pairs; stamps keep
 *                   the step of last use, as under LRU.  The seed is set with
 *                   hs_set_eviction_seed (default 0).
 * Ties go to the lowest slot index under all three.  Takes effect at the next
 * hs_resolve; switching mid-run keeps the stamps as they are.  The
 * allocation-free entry point runs LRU only.
 * Source: HiSparse blog, "効率的なSwap-inカーネル"; papercache summary,
 * section 2 "方法细节" (the eviction strategy is one axis of the miss count).
 */
#define HS_POLICY_LRU   0
#define HS_POLICY_FIFO  1
#define HS_POLICY_RANDOM 2
int hs_set_policy(hs_handle* h, int policy);
int hs_set_eviction_seed(hs_handle* h, uint64_t seed);

/*
 * Which tokens the resident tail holds (vLLM Hybrid HiSparse post, "Mixed
 * Residency": the tail stays on the GPU, older pages move to host memory):
 *   HS_TAIL_FIXED    the last T positions of the capacity, [C - T, C)
 *                    (default; hs_append fills it until len reaches C);
 *   HS_TAIL_SLIDING  the last T tokens written, [len - T, len) per request.
 *                    hs_append first writes the row of the token leaving the
 *                    tail (position len - T) back to its host-pool row, so it
 *                    is from then on an ordinary host-backed token (the post's
 *                    "Full Residency" pre-copy).  hs_set_tail_rows then takes
 *                    any token below C: write the current last T tokens.
 * Setup only (before the first hs_resolve); sliding needs resident_tail > 0.
 * Source: vLLM Hybrid HiSparse post, "Mixed Residency" and "Full Residency".
 */
#define HS_TAIL_FIXED    0
#define HS_TAIL_SLIDING  1
int hs_set_tail_mode(hs_handle* h, int mode);

/*
 * CTAs per request in HS_COPY_CLUSTER mode.  n = 0 (the default) picks 16
 * for up to HS_CLUSTER_WIDE_BATCH requests when all of their clusters run at
 * once (else 8 under the same condition), and 5 otherwise (4, then 2, then
 * 1, when the device cannot run it); otherwise 2 <= n <= HS_MAX_CLUSTER, refused
 * (HS_ERR_LIMIT) when the device cannot run clusters of n such CTAs.
 * hs_cluster_size returns the size in use (1 when no cluster size fits: the
 * cluster mode then launches the fused kernel); hs_resolve_host reading
 * mapped top-k rows takes at most 4 of the default (see there).
 * Source: no passage (a launch-shape knob of this library).
 */
int hs_set_cluster_size(hs_handle* h, int n);
int hs_cluster_size(hs_handle* h);

/* The launch the next hs_resolve on this handle makes: HS_COPY_FUSED,
 * HS_COPY_SPLIT or HS_COPY_CLUSTER (never HS_COPY_AUTO), or HS_ERR_ARG.
 * Source: no passage (a measurement aid). */
int hs_launch_mode(hs_handle* h);

/* Kernel launches one hs_resolve makes on this handle (1 fused or cluster, 2 split), or HS_ERR_ARG.
 * Source: no passage (a measurement aid). */
int hs_resolve_launches(hs_handle* h);

/*
 * Measurement aid: when `before_copy` and `after_copy` (cudaEvent_t) are not
 * NULL, every later hs_resolve on this handle records them on its stream
 * around the row-copy kernel (split mode) or around the single fused kernel
 * (fused mode), so that kernel's duration can be read with
 * cudaEventElapsedTime.  In split mode the copy then no longer overlaps the
 * tail of the resolve kernel.  Pass NULL, NULL to switch it off.
 * Source: no passage (a measurement aid).
 */
int hs_profile_events(hs_handle* h, void* before_copy, void* after_copy);

/*
 * ---- Allocation-free variant -------------------------------------------
 * Source: no passage -- the pages have no counterpart: this entry point exists
 * for callers of the library, not because the method needs it.
 *
 * For callers that must not have a library allocate device memory -- an
 * engine that has reserved nearly all HBM for its own KV pool, or a decode
 * loop in which an allocation would synchronise the device.  The caller owns
 * all state and passes it in.  The step is hs_resolve's with a handle's
 * defaults, and only those: LRU eviction, the fixed resident tail [C - T, C),
 * one top-k row per request, and two launches (the resolve kernel, then the
 * grid-wide row-copy kernel; HS_COPY_SPLIT).
 *
 *   tok_slot [B][C], slot_tok [B][S] (start at -1), stamp [B][S] (start at 0),
 *   lengths [B], device_buffer [B][S+T][R]: device memory.
 *   host_pool [B][host_rows][R]: pinned host memory mapped into the device
 *   address space (cudaHostAlloc with cudaHostAllocMapped, cudaHostRegister
 *   with cudaHostRegisterMapped, or a handle's hs_host_pool), host pointer;
 *   all B * host_rows * R bytes must lie in the allocation or registration
 *   that holds its first byte, as the driver reports it.
 *   control: device memory, one hs_control_t, zeroed by the caller before
 *   the first step; the step counter and counters advance in it.
 * Alignment: host_pool and device_buffer 16 bytes, control 8 bytes, the
 * int32 arrays 4 bytes.  A pointer that breaks it, a pool whose extent the
 * driver does not know or that is shorter than B * host_rows * R bytes, is
 * refused with HS_ERR_ARG before anything is enqueued.  The tables are not
 * checked on the host; the kernels check every entry they would use as an
 * index and repair and flag what is out of range (HS_E_STATE).
 *
 * The per-step miss lists live in a fixed device array inside the library
 * (HS_NOALLOC_SCRATCH_BYTES, held on every device that loads the library
 * until the process exits), so B * K may not exceed HS_NOALLOC_MAX_ENTRIES
 * (HS_ERR_LIMIT otherwise).  The first call on a device looks up that
 * array's address and sets kernel attributes; make that first call before
 * any stream capture (while `stream` is being captured, a call that would do
 * it returns HS_ERR_ARG and enqueues nothing).  A set-up that failed is not
 * kept: the next call tries it again.  All calls on a device share the
 * array: calls whose work overlaps on the GPU race, so order them on one
 * stream.  Returns HS_OK or an HS_ERR_* code, synchronously, like hs_resolve.
 */
#define HS_NOALLOC_MAX_ENTRIES    524288   /* B * K */
#define HS_NOALLOC_SCRATCH_BYTES  (2 * 4 * HS_NOALLOC_MAX_ENTRIES + 4 * HS_MAX_BATCH)

typedef struct {
    int32_t step;       /* resolves done; this call's step is step + 1 */
    int32_t err_bits;   /* HS_E_* bits, OR-ed in */
    uint64_t hits;      /* cumulative counters, added to */
    uint64_t misses;
    uint64_t inplace;
} hs_control_t;

int hs_resolve_noalloc(int batch, int ctx_len, int row_bytes, int buffer_slots, int host_rows,
                       int resident_tail, const int32_t* topk_idx, int K, int32_t* out_slot,
                       int32_t* tok_slot, int32_t* slot_tok, int32_t* stamp,
                       const int32_t* lengths, const uint8_t* host_pool, uint8_t* device_buffer,
                       hs_control_t* control, hs_stream_t stream);

/* Static text for a return code.  Source: no passage. */
const char* hs_error_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* HS_H */
