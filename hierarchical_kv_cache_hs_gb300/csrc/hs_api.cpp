// Host side of the C ABI declared in include/hs.h: handle lifetime,
// argument checks, launches and state export.  The host never reads device
// data on the resolve path; everything it enqueues is graph-capturable.
#include <cuda_runtime.h>
#include <sys/mman.h>
#include <sys/syscall.h>
#include <unistd.h>

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <new>
#include <thread>

#include "hs_gather_pool.h"
#include "hs_internal.h"

struct hs_handle {
    int B, C, R, S, T, H, cold;
    int device;
    int32_t* d_tok_slot;   // [B][C]
    int32_t* d_slot_tok;   // [B][S]
    int32_t* d_stamp;      // [B][S]
    int32_t* d_len;        // [B]
    uint8_t* d_buf;        // [B][S+T][R]
    uint8_t* h_pool;       // pinned, mapped [B][H][R]
    uint8_t* d_pool;       // device address of h_pool
    size_t pool_map_len;   // > 0: h_pool is an mmap of this length, registered
                           // with CUDA; 0: from cudaHostAlloc
    int32_t* d_miss_tok;   // [B][S] scratch: this step's miss tokens
    int32_t* d_miss_slot;  // [B][S] scratch: their victim slots
    int32_t* d_miss_cnt;   // [B]
    HsDevState* d_st;
    unsigned* d_done;      // CTAs finished in the current fused launch
    int32_t* d_stage_in;   // [B][min(S, HS_MAX_TOPK)] for hs_resolve_host
    int32_t* d_stage_out;
    cudaEvent_t prof_before, prof_after;  // optional, around the copy kernel
    int copy_mode;         // HS_COPY_*
    int cluster_n;         // CTAs per request in cluster mode (1: no cluster fits)
    int cluster_host_n;    // the same when the kernel reads the top-k rows from
                           // host memory (hs_resolve_host): every CTA of a
                           // cluster reads its request's row across the link
    int policy;            // HS_POLICY_*
    unsigned long long evict_seed;  // HS_POLICY_RANDOM's seed
    int tail_mode;         // HS_TAIL_*
    int copy_grid;         // the copy kernel's default grid: SMs x its occupancy
    int copy_ctas;         // hs_set_copy_ctas: the grid in use when > 0
    int copy_unroll;
    int copy_rows_per_group;
    size_t pool_bytes, buf_bytes;
    // Copy-engine variant (allocated on its first call).
    uint8_t* ce_h_stage;   // pinned host staging [B * min(S, HS_MAX_TOPK)][R]
    uint8_t* ce_d_stage;   // device staging, same size
    int32_t* ce_h_cnt;     // pinned [B]
    int32_t* ce_h_tok;     // pinned [B][S]
    GatherPool* ce_pool;
};

namespace {

// Switch to the handle's device for the duration of a call.
struct DeviceGuard {
    int prev = -1;
    bool switched = false;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) == cudaSuccess && prev != dev) {
            switched = cudaSetDevice(dev) == cudaSuccess;
        }
    }
    ~DeviceGuard()
    {
        if (switched) cudaSetDevice(prev);
    }
};

template <class T>
cudaError_t dalloc(T** p, size_t n)
{
    *p = nullptr;
    if (n == 0) n = 1;
    return cudaMalloc(reinterpret_cast<void**>(p), n * sizeof(T));
}

// How host pools are placed (hs_set_host_pool_pages), process-wide.
std::atomic<int> g_pool_pages{HS_POOL_PAGES_AUTO};

// Size of a transparent huge page on this host (the kernel's PMD mapping
// size), or 0 when the kernel offers none.
size_t huge_page_bytes()
{
    static const size_t bytes = [] {
        size_t v = 0;
        if (FILE* f = std::fopen("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size", "r")) {
            unsigned long long x = 0;
            if (std::fscanf(f, "%llu", &x) == 1) v = (size_t)x;
            std::fclose(f);
        }
        return v;
    }();
    return bytes;
}

// Ask for the pages of [p, p + len) on the host NUMA node nearest the GPU,
// before their first touch, as a preference (MPOL_PREFERRED).  Nothing
// happens when the device reports no node or the call fails.
void prefer_gpu_node(void* p, size_t len, int device)
{
    int node = -1;
    if (cudaDeviceGetAttribute(&node, cudaDevAttrHostNumaId, device) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    if (node < 0 || node >= 1024) return;
    unsigned long mask[1024 / (8 * sizeof(unsigned long))] = {};
    mask[node / (8 * sizeof(unsigned long))] = 1ul << (node % (8 * sizeof(unsigned long)));
    const int kPreferred = 1;  // MPOL_PREFERRED
    syscall(SYS_mbind, p, len, kPreferred, mask, (unsigned long)(node + 2), 0u);
}

// The host pool, n bytes.  A pool of at least HS_POOL_HUGE_MIN_BYTES and one
// huge page (or any size under HS_POOL_PAGES_HUGE) is placed in anonymous
// memory aligned to the huge-page size and advised for huge pages before its
// first touch, then page-locked and mapped with cudaHostRegister, so the GPU
// can map it with large pages: with the base pages of cudaHostAlloc, a pool of
// tens of GB read from several SMs per request spends much of the step on
// address translation.  Smaller pools stay in cudaHostAlloc memory, whose
// first steps after set-up run at full speed (the huge-page placement's
// first seconds of steps are slow and uneven).  Whether the kernel backs the
// range with huge pages is up to it (memory fragmentation); any failure here
// falls back to cudaHostAlloc.
bool alloc_pool(hs_handle* h, size_t n)
{
    const int mode = g_pool_pages.load();
    const size_t hp = huge_page_bytes();
    const long pg = sysconf(_SC_PAGESIZE);
    const bool big = n >= hp && n >= (size_t)HS_POOL_HUGE_MIN_BYTES;
    if (mode != HS_POOL_PAGES_BASE && hp > 0 && pg > 0 &&
        (big || (mode == HS_POOL_PAGES_HUGE && n > 0))) {
        const size_t len = (n + (size_t)pg - 1) / (size_t)pg * (size_t)pg;
        void* m = mmap(nullptr, len + hp, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
        if (m != MAP_FAILED) {
            const uintptr_t lo = (uintptr_t)m, hi = lo + len + hp;
            const uintptr_t a = (lo + hp - 1) / hp * hp;  // a multiple of the page size too
            if (a > lo) munmap(m, a - lo);
            if (hi > a + len) munmap(reinterpret_cast<void*>(a + len), hi - (a + len));
            void* p = reinterpret_cast<void*>(a);
            madvise(p, len, MADV_HUGEPAGE);
            // A forked child does not inherit the pool (it would otherwise copy
            // every pinned page at the fork).
            madvise(p, len, MADV_DONTFORK);
            prefer_gpu_node(p, len, h->device);
            if (cudaHostRegister(p, n, cudaHostRegisterMapped) == cudaSuccess) {
                h->h_pool = static_cast<uint8_t*>(p);
                h->pool_map_len = len;
                return true;
            }
            cudaGetLastError();
            munmap(p, len);
        }
    }
    void* p = nullptr;
    if (cudaHostAlloc(&p, n ? n : 1, cudaHostAllocMapped) != cudaSuccess) return false;
    h->h_pool = static_cast<uint8_t*>(p);
    h->pool_map_len = 0;
    return true;
}

void free_pool(hs_handle* h)
{
    if (!h->h_pool) return;
    if (h->pool_map_len > 0) {
        cudaHostUnregister(h->h_pool);
        munmap(h->h_pool, h->pool_map_len);
    } else {
        cudaFreeHost(h->h_pool);
    }
    h->h_pool = nullptr;
}

void free_all(hs_handle* h)
{
    if (!h) return;
    cudaFree(h->d_tok_slot);
    cudaFree(h->d_slot_tok);
    cudaFree(h->d_stamp);
    cudaFree(h->d_len);
    cudaFree(h->d_buf);
    cudaFree(h->d_miss_tok);
    cudaFree(h->d_miss_slot);
    cudaFree(h->d_miss_cnt);
    cudaFree(h->d_st);
    cudaFree(h->d_done);
    cudaFree(h->d_stage_in);
    cudaFree(h->d_stage_out);
    free_pool(h);
    if (h->ce_h_stage) cudaFreeHost(h->ce_h_stage);
    cudaFree(h->ce_d_stage);
    if (h->ce_h_cnt) cudaFreeHost(h->ce_h_cnt);
    if (h->ce_h_tok) cudaFreeHost(h->ce_h_tok);
    delete h->ce_pool;
}

int fill_start_state(hs_handle* h)
{
    const size_t B = (size_t)h->B;
    if (cudaMemset(h->d_tok_slot, 0xff, B * h->C * sizeof(int32_t)) != cudaSuccess) return HS_ERR_CUDA;
    if (cudaMemset(h->d_slot_tok, 0xff, B * h->S * sizeof(int32_t)) != cudaSuccess) return HS_ERR_CUDA;
    if (cudaMemset(h->d_stamp, 0, B * h->S * sizeof(int32_t)) != cudaSuccess) return HS_ERR_CUDA;
    if (cudaMemset(h->d_miss_cnt, 0, B * sizeof(int32_t)) != cudaSuccess) return HS_ERR_CUDA;
    if (cudaMemset(h->d_st, 0, sizeof(HsDevState)) != cudaSuccess) return HS_ERR_CUDA;
    if (cudaMemset(h->d_done, 0, sizeof(unsigned)) != cudaSuccess) return HS_ERR_CUDA;
    std::vector<int32_t> len(B, h->C);
    if (cudaMemcpy(h->d_len, len.data(), B * sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess)
        return HS_ERR_CUDA;
    return cudaDeviceSynchronize() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

// State reads and setup calls wait for all work on the device, so a stream
// the caller has since destroyed is never touched.
int sync_last(hs_handle*)
{
    return cudaDeviceSynchronize() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

bool valid(const hs_handle* h)
{
    return h != nullptr && h->B > 0;
}

// The launch of a step: HS_COPY_FUSED, HS_COPY_SPLIT or HS_COPY_CLUSTER.  A
// cluster mode whose cluster size is 1 runs the fused kernel.  HS_COPY_AUTO:
// a cluster per request up to HS_CLUSTER_MAX_BATCH requests when a cluster
// size of 2 or more runs on the device (beyond it, one CTA per request
// already fills several waves of the SMs, whose later waves resolve while the
// earlier ones copy); otherwise fused, or split below HS_FUSED_MIN_BATCH
// requests when one request's hot buffer (which bounds what a step gives one
// CTA to copy) is over HS_FUSED_MAX_REQUEST_BYTES.
int launch_kind(const hs_handle* h)
{
    if (h->copy_mode == HS_COPY_CLUSTER)
        return h->cluster_n >= 2 ? HS_COPY_CLUSTER : HS_COPY_FUSED;
    if (h->copy_mode != HS_COPY_AUTO) return h->copy_mode;
    if (h->B <= HS_CLUSTER_MAX_BATCH && h->cluster_n >= 2) return HS_COPY_CLUSTER;
    return (h->B >= HS_FUSED_MIN_BATCH ||
            (long long)h->S * h->R <= (long long)HS_FUSED_MAX_REQUEST_BYTES)
               ? HS_COPY_FUSED
               : HS_COPY_SPLIT;
}

// CTAs per request in cluster mode (measured on GB300, 1-256 requests of
// 2048-of-4096 slots): 16 up to HS_CLUSTER_WIDE_BATCH requests, when all of
// their clusters run at once (8 when 16 do not fit), else 5; each size falls
// back to the next smaller one the device cannot run.  Above 4 requests,
// clusters of 5 were the fastest of 2, 3, 4, 5, 6, 8 and 16 at every batch
// size measured (up to 3 % ahead of 4), also past one wave of the SMs:
// later clusters resolve while earlier ones copy.
int auto_cluster_size(const hs_handle* h)
{
    const int kmax = h->S < HS_MAX_TOPK ? h->S : HS_MAX_TOPK;
    if (h->B <= HS_CLUSTER_WIDE_BATCH)
        for (int n = HS_MAX_CLUSTER; n > 4; n >>= 1)
            if (hs_cluster_max_active(kmax, h->S, n, h->copy_unroll) >= h->B) return n;
    // Otherwise 5 CTAs per request (measured faster than 4 at every batch
    // from 8 to 128 requests), or the largest of 4 and 2 that the device runs.
    for (int n : {5, 4, 2})
        if (hs_cluster_max_active(kmax, h->S, n, h->copy_unroll) >= 1) return n;
    return 1;
}

// The default sizes: auto_cluster_size for the device-resident top-k rows,
// and at most 4 above HS_CLUSTER_WIDE_BATCH requests when the rows are read
// from host memory.  Each CTA of a cluster reads its request's row across
// the host link, so a fifth CTA adds B * K * 4 bytes of link traffic per
// step; measured through hs_resolve_host, clusters of 4 were 1-2.5 % faster
// than 5 at 32 and 64 requests, where 5 were faster with the rows on the device.
void set_auto_cluster_size(hs_handle* h)
{
    h->cluster_n = auto_cluster_size(h);
    h->cluster_host_n = (h->B > HS_CLUSTER_WIDE_BATCH && h->cluster_n > 4) ? 4 : h->cluster_n;
}

}  // namespace

extern "C" {

const char* hs_error_string(int code)
{
    switch (code) {
    case HS_OK: return "ok";
    case HS_ERR_ARG: return "invalid argument";
    case HS_ERR_TOPK_GT_SLOTS: return "top-k larger than the buffer slots";
    case HS_ERR_CAPACITY: return "host pool smaller than the host-backed context";
    case HS_ERR_ALLOC: return "allocation failed";
    case HS_ERR_CUDA: return "CUDA runtime error";
    case HS_ERR_LIMIT: return "size beyond the kernel limits";
    default: return "unknown error";
    }
}

int hs_create(int batch, int ctx_len, int row_bytes, int buffer_slots, int host_ratio,
              int resident_tail, hs_handle** out)
{
    if (!out) return HS_ERR_ARG;
    *out = nullptr;
    if (batch <= 0 || ctx_len <= 0 || row_bytes <= 0 || buffer_slots <= 0 || host_ratio <= 0 ||
        resident_tail < 0 || resident_tail > ctx_len || (row_bytes % 16) != 0)
        return HS_ERR_ARG;
    if (batch > HS_MAX_BATCH || buffer_slots > HS_MAX_SLOTS || row_bytes > HS_MAX_ROW_BYTES)
        return HS_ERR_LIMIT;
    const long long H = (long long)host_ratio * buffer_slots;
    if (H < (long long)ctx_len - resident_tail) return HS_ERR_CAPACITY;
    if (H > 0x7fffffffLL) return HS_ERR_LIMIT;

    hs_handle* h = new (std::nothrow) hs_handle();
    if (!h) return HS_ERR_ALLOC;
    h->B = batch;
    h->C = ctx_len;
    h->R = row_bytes;
    h->S = buffer_slots;
    h->T = resident_tail;
    h->H = (int)H;
    h->cold = ctx_len - resident_tail;
    if (cudaGetDevice(&h->device) != cudaSuccess) {
        delete h;
        return HS_ERR_CUDA;
    }

    const size_t B = (size_t)batch;
    const int kmax = buffer_slots < HS_MAX_TOPK ? buffer_slots : HS_MAX_TOPK;
    h->pool_bytes = B * (size_t)h->H * (size_t)row_bytes;
    h->buf_bytes = B * (size_t)(buffer_slots + resident_tail) * (size_t)row_bytes;
    bool ok = dalloc(&h->d_tok_slot, B * ctx_len) == cudaSuccess &&
              dalloc(&h->d_slot_tok, B * buffer_slots) == cudaSuccess &&
              dalloc(&h->d_stamp, B * buffer_slots) == cudaSuccess &&
              dalloc(&h->d_len, B) == cudaSuccess &&
              dalloc(&h->d_buf, h->buf_bytes) == cudaSuccess &&
              dalloc(&h->d_miss_tok, B * buffer_slots) == cudaSuccess &&
              dalloc(&h->d_miss_slot, B * buffer_slots) == cudaSuccess &&
              dalloc(&h->d_miss_cnt, B) == cudaSuccess &&
              dalloc(&h->d_st, 1) == cudaSuccess &&
              dalloc(&h->d_done, 1) == cudaSuccess &&
              dalloc(&h->d_stage_in, B * kmax) == cudaSuccess &&
              dalloc(&h->d_stage_out, B * kmax) == cudaSuccess;
    if (ok) {
        ok = alloc_pool(h, h->pool_bytes);
        if (ok) {
            void* dp = nullptr;
            ok = cudaHostGetDevicePointer(&dp, h->h_pool, 0) == cudaSuccess;
            h->d_pool = static_cast<uint8_t*>(dp);
        }
    }
    if (!ok) {
        cudaGetLastError();
        free_all(h);
        delete h;
        return HS_ERR_ALLOC;
    }
    if (hs_prepare_resolve() != cudaSuccess) {
        free_all(h);
        delete h;
        return HS_ERR_CUDA;
    }
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, h->device);
    if (sms <= 0) sms = 1;
    h->copy_unroll = hs_copy_unroll_for(row_bytes);
    h->copy_grid = sms * hs_copy_blocks_per_sm(h->copy_unroll, batch);
    h->copy_rows_per_group = hs_copy_rows_per_group(row_bytes, h->copy_unroll);
    h->copy_mode = HS_COPY_AUTO;
    set_auto_cluster_size(h);
    h->policy = HS_POLICY_LRU;
    h->tail_mode = HS_TAIL_FIXED;
    const int rc = fill_start_state(h);
    if (rc != HS_OK) {
        free_all(h);
        delete h;
        return rc;
    }
    *out = h;
    return HS_OK;
}

void hs_destroy(hs_handle* h)
{
    if (!h) return;
    DeviceGuard g(h->device);
    cudaDeviceSynchronize();
    free_all(h);
    h->B = 0;
    delete h;
}

static int resolve_impl(hs_handle* h, const int32_t* topk_idx, int K, int32_t* out_slot,
                        hs_stream_t stream, int alias, bool host_topk = false);

int hs_resolve(hs_handle* h, const int32_t* topk_idx, int K, int32_t* out_slot,
               hs_stream_t stream)
{
    return resolve_impl(h, topk_idx, K, out_slot, stream, 0);
}

int hs_resolve_multi(hs_handle* h, const int32_t* topk_idx, int P, int K, int32_t* out_slot,
                     hs_stream_t stream)
{
    if (!valid(h) || P <= 0 || K <= 0) return HS_ERR_ARG;
    const long long PK = (long long)P * K;
    if (PK > h->S) return HS_ERR_TOPK_GT_SLOTS;
    if (PK > HS_MAX_TOPK) return HS_ERR_LIMIT;
    return resolve_impl(h, topk_idx, (int)PK, out_slot, stream, 1);
}

// The resolve kernel's arguments for one handle's step.
static ResolveArgs resolve_args(const hs_handle* h, const int32_t* topk_idx, int K,
                                int32_t* out_slot, int alias)
{
    ResolveArgs ra;
    ra.topk = topk_idx;
    ra.out = out_slot;
    ra.tok_slot = h->d_tok_slot;
    ra.slot_tok = h->d_slot_tok;
    ra.stamp = h->d_stamp;
    ra.len = h->d_len;
    ra.miss_tok = h->d_miss_tok;
    ra.miss_slot = h->d_miss_slot;
    ra.miss_cnt = h->d_miss_cnt;
    ra.st = h->d_st;
    ra.K = K;
    ra.C = h->C;
    ra.S = h->S;
    ra.T = h->T;
    ra.cold = h->cold;
    ra.list_stride = h->S;
    ra.hash_bits = hs_hash_bits(K);
    ra.pool = h->d_pool;
    ra.buf = h->d_buf;
    ra.H = h->H;
    ra.R = h->R;
    ra.rows_per_group = h->copy_rows_per_group;
    ra.done = h->d_done;
    ra.fifo = h->policy == HS_POLICY_FIFO ? 1 : 0;
    ra.random = h->policy == HS_POLICY_RANDOM ? 1 : 0;
    ra.seed = h->evict_seed;
    ra.sliding = h->tail_mode == HS_TAIL_SLIDING ? 1 : 0;
    ra.alias = alias;
    return ra;
}

static int resolve_impl(hs_handle* h, const int32_t* topk_idx, int K, int32_t* out_slot,
                        hs_stream_t stream, int alias, bool host_topk)
{
    if (!valid(h) || !topk_idx || !out_slot || K <= 0) return HS_ERR_ARG;
    if (K > h->S) return HS_ERR_TOPK_GT_SLOTS;
    if (K > HS_MAX_TOPK) return HS_ERR_LIMIT;
    DeviceGuard g(h->device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const ResolveArgs ra = resolve_args(h, topk_idx, K, out_slot, alias);

    const bool prof = h->prof_before && h->prof_after;
    const int kind = launch_kind(h);
    if (kind != HS_COPY_SPLIT) {
        // One launch: each request's CTA (or cluster of CTAs) fetches its own
        // rows.  The profiling events then bracket the whole step.
        if (prof && cudaEventRecord(h->prof_before, s) != cudaSuccess) return HS_ERR_CUDA;
        const cudaError_t e = kind == HS_COPY_CLUSTER
            ? hs_launch_swapin_cluster(ra, h->B, host_topk ? h->cluster_host_n : h->cluster_n,
                                       h->copy_unroll, s)
            : hs_launch_swapin(ra, h->B, h->copy_unroll, s);
        if (e != cudaSuccess) return HS_ERR_CUDA;
        if (prof && cudaEventRecord(h->prof_after, s) != cudaSuccess) return HS_ERR_CUDA;
        return HS_OK;
    }
    if (hs_launch_resolve(ra, h->B, s) != cudaSuccess) return HS_ERR_CUDA;

    CopyArgs ca;
    ca.miss_cnt = h->d_miss_cnt;
    ca.miss_tok = h->d_miss_tok;
    ca.miss_slot = h->d_miss_slot;
    ca.pool = h->d_pool;
    ca.buf = h->d_buf;
    ca.st = h->d_st;
    ca.B = h->B;
    ca.S = h->S;
    ca.T = h->T;
    ca.R = h->R;
    ca.list_stride = h->S;
    ca.H = h->H;
    ca.rows_per_group = h->copy_rows_per_group;
    ca.advance_step = 1;
    ca.flat_src = 0;
    if (prof && cudaEventRecord(h->prof_before, s) != cudaSuccess) return HS_ERR_CUDA;
    if (hs_launch_copy(ca, h->copy_ctas > 0 ? h->copy_ctas : h->copy_grid, h->copy_unroll, s, !prof) != cudaSuccess) return HS_ERR_CUDA;
    if (prof && cudaEventRecord(h->prof_after, s) != cudaSuccess) return HS_ERR_CUDA;
    return HS_OK;
}

// Every host-side check of a several-layer step, shared by the device- and
// host-buffer entry points so that neither enqueues anything (a staging copy
// included) for arguments the launch would refuse.
static int check_layers(hs_handle* const* handles, int L, const void* const* topk_idx, int K,
                        const void* const* out_slot)
{
    if (!handles || !topk_idx || !out_slot || L <= 0 || K <= 0) return HS_ERR_ARG;
    if (L > HS_MAX_LAYERS) return HS_ERR_LIMIT;
    const hs_handle* h0 = handles[0];
    if (!valid(h0)) return HS_ERR_ARG;
    for (int l = 0; l < L; ++l) {
        const hs_handle* h = handles[l];
        if (!valid(h) || !topk_idx[l] || !out_slot[l]) return HS_ERR_ARG;
        if (h->B != h0->B || h->S != h0->S || h->R != h0->R || h->device != h0->device)
            return HS_ERR_ARG;
        for (int k = 0; k < l; ++k)
            if (handles[k] == h) return HS_ERR_ARG;
    }
    if (K > h0->S) return HS_ERR_TOPK_GT_SLOTS;
    if (K > HS_MAX_TOPK) return HS_ERR_LIMIT;
    return HS_OK;
}

int hs_resolve_layers(hs_handle* const* handles, int L, const int32_t* const* topk_idx, int K,
                      int32_t* const* out_slot, hs_stream_t stream)
{
    const int rc = check_layers(handles, L, reinterpret_cast<const void* const*>(topk_idx), K,
                                reinterpret_cast<const void* const*>(out_slot));
    if (rc != HS_OK) return rc;
    const hs_handle* h0 = handles[0];
    DeviceGuard g(h0->device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    LayerArgs p;
    p.B = h0->B;
    for (int l = 0; l < L; ++l) p.l[l] = resolve_args(handles[l], topk_idx[l], K, out_slot[l], 0);
    // Profiling events of any handle bracket the one launch.
    for (int l = 0; l < L; ++l) {
        const hs_handle* h = handles[l];
        if (h->prof_before && h->prof_after && cudaEventRecord(h->prof_before, s) != cudaSuccess)
            return HS_ERR_CUDA;
    }
    if (hs_launch_swapin_layers(p, L, h0->copy_unroll, s) != cudaSuccess) return HS_ERR_CUDA;
    for (int l = 0; l < L; ++l) {
        const hs_handle* h = handles[l];
        if (h->prof_before && h->prof_after && cudaEventRecord(h->prof_after, s) != cudaSuccess)
            return HS_ERR_CUDA;
    }
    return HS_OK;
}

int hs_resolve_layers_host(hs_handle* const* handles, int L, const int32_t* const* topk_idx, int K,
                           int32_t* const* out_slot, hs_stream_t stream)
{
    // All checks first: the staging buffers below hold B * min(S, HS_MAX_TOPK)
    // entries of each handle, which only a checked K and shape respect.
    const int rc0 = check_layers(handles, L, reinterpret_cast<const void* const*>(topk_idx), K,
                                 reinterpret_cast<const void* const*>(out_slot));
    if (rc0 != HS_OK) return rc0;
    const hs_handle* h0 = handles[0];
    DeviceGuard g(h0->device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Device addresses of mapped buffers; the others go through each handle's
    // staging buffers.
    const int32_t* d_in[HS_MAX_LAYERS];
    int32_t* d_out[HS_MAX_LAYERS];
    bool staged_out[HS_MAX_LAYERS];
    for (int l = 0; l < L; ++l) {
        hs_handle* h = handles[l];
        const size_t bytes = (size_t)h->B * (size_t)K * sizeof(int32_t);
        void* p = nullptr;
        if (cudaHostGetDevicePointer(&p, const_cast<int32_t*>(topk_idx[l]), 0) == cudaSuccess) {
            d_in[l] = static_cast<const int32_t*>(p);
        } else {
            cudaGetLastError();
            if (cudaMemcpyAsync(h->d_stage_in, topk_idx[l], bytes, cudaMemcpyHostToDevice, s) !=
                cudaSuccess)
                return HS_ERR_CUDA;
            d_in[l] = h->d_stage_in;
        }
        p = nullptr;
        staged_out[l] = cudaHostGetDevicePointer(&p, out_slot[l], 0) != cudaSuccess;
        if (staged_out[l]) cudaGetLastError();
        d_out[l] = staged_out[l] ? h->d_stage_out : static_cast<int32_t*>(p);
    }
    const int rc = hs_resolve_layers(handles, L, d_in, K, d_out, stream);
    if (rc != HS_OK) return rc;
    for (int l = 0; l < L; ++l) {
        if (!staged_out[l]) continue;
        const size_t bytes = (size_t)handles[l]->B * (size_t)K * sizeof(int32_t);
        if (cudaMemcpyAsync(out_slot[l], handles[l]->d_stage_out, bytes, cudaMemcpyDeviceToHost, s) !=
            cudaSuccess)
            return HS_ERR_CUDA;
    }
    return cudaStreamSynchronize(s) == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

int hs_resolve_ce(hs_handle* h, const int32_t* topk_idx, int K, int32_t* out_slot,
                  hs_stream_t stream)
{
    if (!valid(h) || !topk_idx || !out_slot || K <= 0) return HS_ERR_ARG;
    if (K > h->S) return HS_ERR_TOPK_GT_SLOTS;
    if (K > HS_MAX_TOPK) return HS_ERR_LIMIT;
    DeviceGuard g(h->device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t B = (size_t)h->B, S = (size_t)h->S, R = (size_t)h->R;
    if (!h->ce_pool) {
        const size_t rows = B * (size_t)(h->S < HS_MAX_TOPK ? h->S : HS_MAX_TOPK);
        // Each pointer is stored only once its allocation has succeeded, so the
        // error path below frees exactly what exists.
        void* p = nullptr;
        bool ok = cudaHostAlloc(&p, rows * R, cudaHostAllocDefault) == cudaSuccess;
        if (ok) h->ce_h_stage = static_cast<uint8_t*>(p);
        ok = ok && cudaMalloc(&p, rows * R) == cudaSuccess;
        if (ok) h->ce_d_stage = static_cast<uint8_t*>(p);
        ok = ok && cudaHostAlloc(&p, B * sizeof(int32_t), cudaHostAllocDefault) == cudaSuccess;
        if (ok) h->ce_h_cnt = static_cast<int32_t*>(p);
        ok = ok && cudaHostAlloc(&p, B * S * sizeof(int32_t), cudaHostAllocDefault) == cudaSuccess;
        if (ok) h->ce_h_tok = static_cast<int32_t*>(p);
        unsigned n = std::thread::hardware_concurrency();
        if (ok) h->ce_pool = new (std::nothrow) GatherPool(n ? (int)n : 4);
        if (!ok || !h->ce_pool) {
            // Release what was allocated so that a later call starts afresh.
            cudaGetLastError();
            if (h->ce_h_stage) cudaFreeHost(h->ce_h_stage);
            if (h->ce_d_stage) cudaFree(h->ce_d_stage);
            if (h->ce_h_cnt) cudaFreeHost(h->ce_h_cnt);
            if (h->ce_h_tok) cudaFreeHost(h->ce_h_tok);
            h->ce_h_stage = nullptr;
            h->ce_d_stage = nullptr;
            h->ce_h_cnt = nullptr;
            h->ce_h_tok = nullptr;
            return HS_ERR_ALLOC;
        }
    }

    // (1)-(3) on the device: the resolve kernel writes the miss lists.
    ResolveArgs ra = {};
    ra.topk = topk_idx;
    ra.out = out_slot;
    ra.tok_slot = h->d_tok_slot;
    ra.slot_tok = h->d_slot_tok;
    ra.stamp = h->d_stamp;
    ra.len = h->d_len;
    ra.miss_tok = h->d_miss_tok;
    ra.miss_slot = h->d_miss_slot;
    ra.miss_cnt = h->d_miss_cnt;
    ra.st = h->d_st;
    ra.K = K;
    ra.C = h->C;
    ra.S = h->S;
    ra.T = h->T;
    ra.cold = h->cold;
    ra.list_stride = h->S;
    ra.hash_bits = hs_hash_bits(K);
    ra.R = h->R;
    ra.H = h->H;
    ra.rows_per_group = 1;
    ra.fifo = h->policy == HS_POLICY_FIFO ? 1 : 0;
    ra.random = h->policy == HS_POLICY_RANDOM ? 1 : 0;
    ra.seed = h->evict_seed;
    ra.sliding = h->tail_mode == HS_TAIL_SLIDING ? 1 : 0;
    ra.alias = 0;
    if (hs_launch_resolve(ra, h->B, s) != cudaSuccess) return HS_ERR_CUDA;

    // The host needs the miss tokens: one read-back and one synchronisation.
    if (cudaMemcpyAsync(h->ce_h_cnt, h->d_miss_cnt, B * sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
            cudaSuccess ||
        cudaMemcpyAsync(h->ce_h_tok, h->d_miss_tok, B * S * sizeof(int32_t), cudaMemcpyDeviceToHost,
                        s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return HS_ERR_CUDA;
    std::vector<long long> off(B + 1, 0);
    // A request's misses never exceed K, which the staging area is sized for;
    // the clamp keeps the host gather inside it whatever the device wrote.
    for (size_t b = 0; b < B; ++b) {
        const int32_t c = h->ce_h_cnt[b];
        off[b + 1] = off[b] + (c < 0 ? 0 : c > K ? K : c);
    }
    const long long M = off[B];

    // Host threads gather the rows into the staging area in flattened
    // (request, miss) order -- the order the scatter kernel expects.
    const long long chunk = 256;
    const int ntasks = (int)((M + chunk - 1) / chunk);
    const uint8_t* pool = h->h_pool;
    uint8_t* stage = h->ce_h_stage;
    const int32_t* toks = h->ce_h_tok;
    const long long H = h->H;
    std::function<void(int)> gather = [&](int task) {
        const long long r0 = (long long)task * chunk;
        const long long r1 = r0 + chunk < M ? r0 + chunk : M;
        size_t b = 0;
        while (b + 1 < B && off[b + 1] <= r0) ++b;
        for (long long r = r0; r < r1; ++r) {
            while (off[b + 1] <= r) ++b;
            const long long i = r - off[b];
            const int32_t t = toks[b * S + (size_t)i];
            if (t < 0 || t >= H) continue;  // never written by the resolve kernel
            std::memcpy(stage + (size_t)r * R, pool + ((long long)b * H + t) * (long long)R, R);
        }
    };
    h->ce_pool->run(ntasks, gather);

    // One large copy-engine transfer, then the rows go to their slots.
    if (M > 0 && cudaMemcpyAsync(h->ce_d_stage, h->ce_h_stage, (size_t)M * R,
                                 cudaMemcpyHostToDevice, s) != cudaSuccess)
        return HS_ERR_CUDA;
    CopyArgs ca;
    ca.miss_cnt = h->d_miss_cnt;
    ca.miss_tok = h->d_miss_tok;
    ca.miss_slot = h->d_miss_slot;
    ca.pool = h->ce_d_stage;
    ca.buf = h->d_buf;
    ca.st = h->d_st;
    ca.B = h->B;
    ca.S = h->S;
    ca.T = h->T;
    ca.R = h->R;
    ca.list_stride = h->S;
    ca.H = h->H;
    ca.rows_per_group = h->copy_rows_per_group;
    ca.advance_step = 1;
    ca.flat_src = 1;
    if (hs_launch_copy(ca, h->copy_ctas > 0 ? h->copy_ctas : h->copy_grid, h->copy_unroll, s, false) != cudaSuccess) return HS_ERR_CUDA;
    return HS_OK;
}

int hs_resolve_launches(hs_handle* h)
{
    if (!valid(h)) return HS_ERR_ARG;
    return launch_kind(h) == HS_COPY_SPLIT ? 2 : 1;
}

int hs_launch_mode(hs_handle* h)
{
    return valid(h) ? launch_kind(h) : HS_ERR_ARG;
}

int hs_set_cluster_size(hs_handle* h, int n)
{
    if (!valid(h) || n < 0 || n == 1) return HS_ERR_ARG;
    if (n > HS_MAX_CLUSTER) return HS_ERR_LIMIT;
    DeviceGuard g(h->device);
    if (n == 0) {
        set_auto_cluster_size(h);
        return HS_OK;
    }
    const int kmax = h->S < HS_MAX_TOPK ? h->S : HS_MAX_TOPK;
    if (hs_cluster_max_active(kmax, h->S, n, h->copy_unroll) < 1) return HS_ERR_LIMIT;
    h->cluster_n = n;
    h->cluster_host_n = n;
    return HS_OK;
}

int hs_cluster_size(hs_handle* h)
{
    return valid(h) ? h->cluster_n : HS_ERR_ARG;
}

int hs_set_tail_mode(hs_handle* h, int mode)
{
    if (!valid(h) || (mode != HS_TAIL_FIXED && mode != HS_TAIL_SLIDING)) return HS_ERR_ARG;
    if (mode == HS_TAIL_SLIDING && h->T <= 0) return HS_ERR_ARG;
    h->tail_mode = mode;
    return HS_OK;
}

int hs_set_policy(hs_handle* h, int policy)
{
    if (!valid(h) || (policy != HS_POLICY_LRU && policy != HS_POLICY_FIFO && policy != HS_POLICY_RANDOM))
        return HS_ERR_ARG;
    h->policy = policy;
    return HS_OK;
}

int hs_set_eviction_seed(hs_handle* h, uint64_t seed)
{
    if (!valid(h)) return HS_ERR_ARG;
    h->evict_seed = seed;
    return HS_OK;
}

int hs_set_copy_mode(hs_handle* h, int mode)
{
    if (!valid(h) || mode < HS_COPY_AUTO || mode > HS_COPY_CLUSTER) return HS_ERR_ARG;
    h->copy_mode = mode;
    return HS_OK;
}

int hs_set_copy_ctas(hs_handle* h, int n)
{
    if (!valid(h) || n < 0 || n > HS_MAX_COPY_CTAS) return HS_ERR_ARG;
    h->copy_ctas = n;
    return HS_OK;
}

int hs_resolve_host(hs_handle* h, const int32_t* topk_idx, int K, int32_t* out_slot,
                    hs_stream_t stream)
{
    if (!valid(h) || !topk_idx || !out_slot || K <= 0) return HS_ERR_ARG;
    if (K > h->S) return HS_ERR_TOPK_GT_SLOTS;
    if (K > HS_MAX_TOPK) return HS_ERR_LIMIT;
    DeviceGuard g(h->device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Pinned, mapped host buffers: the kernels read the top-k rows and write
    // out_slot across the host link themselves -- no staging copies.
    void* d_in = nullptr;
    void* d_out = nullptr;
    if (cudaHostGetDevicePointer(&d_in, const_cast<int32_t*>(topk_idx), 0) == cudaSuccess &&
        cudaHostGetDevicePointer(&d_out, out_slot, 0) == cudaSuccess) {
        const int rc = resolve_impl(h, static_cast<const int32_t*>(d_in), K,
                                    static_cast<int32_t*>(d_out), stream, 0, true);
        if (rc != HS_OK) return rc;
        return cudaStreamSynchronize(s) == cudaSuccess ? HS_OK : HS_ERR_CUDA;
    }
    cudaGetLastError();  // not mapped: clear the lookup's error and stage through the device
    const size_t bytes = (size_t)h->B * (size_t)K * sizeof(int32_t);
    if (cudaMemcpyAsync(h->d_stage_in, topk_idx, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return HS_ERR_CUDA;
    const int rc = hs_resolve(h, h->d_stage_in, K, h->d_stage_out, stream);
    if (rc != HS_OK) return rc;
    if (cudaMemcpyAsync(out_slot, h->d_stage_out, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return HS_ERR_CUDA;
    return cudaStreamSynchronize(s) == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

int hs_stats(hs_handle* h, hs_stats_t* out, int32_t* last_miss)
{
    if (!valid(h) || !out) return HS_ERR_ARG;
    DeviceGuard g(h->device);
    if (sync_last(h) != HS_OK) return HS_ERR_CUDA;
    HsDevState st;
    if (cudaMemcpy(&st, h->d_st, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) return HS_ERR_CUDA;
    out->steps = st.step;
    out->hits = (int64_t)st.hits;
    out->misses = (int64_t)st.misses;
    out->inplace = (int64_t)st.inplace;
    out->bytes_copied = (int64_t)st.misses * h->R;
    out->err_bits = st.err;
    out->reserved = 0;
    if (last_miss &&
        cudaMemcpy(last_miss, h->d_miss_cnt, (size_t)h->B * sizeof(int32_t), cudaMemcpyDeviceToHost) !=
            cudaSuccess)
        return HS_ERR_CUDA;
    return HS_OK;
}

uint8_t* hs_host_pool(hs_handle* h) { return valid(h) ? h->h_pool : nullptr; }
size_t hs_host_pool_bytes(hs_handle* h) { return valid(h) ? h->pool_bytes : 0; }

int hs_set_host_pool_pages(int mode)
{
    if (mode != HS_POOL_PAGES_AUTO && mode != HS_POOL_PAGES_BASE && mode != HS_POOL_PAGES_HUGE)
        return HS_ERR_ARG;
    g_pool_pages.store(mode);
    return HS_OK;
}

int hs_host_pool_pages(hs_handle* h)
{
    if (!valid(h)) return HS_ERR_ARG;
    return h->pool_map_len > 0 ? HS_POOL_PAGES_HUGE : HS_POOL_PAGES_BASE;
}

size_t hs_huge_page_bytes(void) { return huge_page_bytes(); }
uint8_t* hs_device_buffer(hs_handle* h) { return valid(h) ? h->d_buf : nullptr; }
size_t hs_device_buffer_bytes(hs_handle* h) { return valid(h) ? h->buf_bytes : 0; }

int hs_set_lengths(hs_handle* h, const int32_t* len_host)
{
    if (!valid(h) || !len_host) return HS_ERR_ARG;
    for (int b = 0; b < h->B; ++b)
        if (len_host[b] < 0 || len_host[b] > h->C) return HS_ERR_ARG;
    DeviceGuard g(h->device);
    if (sync_last(h) != HS_OK) return HS_ERR_CUDA;
    if (cudaMemcpy(h->d_len, len_host, (size_t)h->B * sizeof(int32_t), cudaMemcpyHostToDevice) !=
        cudaSuccess)
        return HS_ERR_CUDA;
    return HS_OK;
}

int hs_append(hs_handle* h, const uint8_t* rows_dev, hs_stream_t stream)
{
    if (!valid(h) || !rows_dev || h->T <= 0) return HS_ERR_ARG;
    DeviceGuard g(h->device);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    AppendArgs a;
    a.rows = rows_dev;
    a.buf = h->d_buf;
    a.len = h->d_len;
    a.st = h->d_st;
    a.S = h->S;
    a.T = h->T;
    a.R = h->R;
    a.C = h->C;
    a.cold = h->cold;
    a.pool = h->d_pool;
    a.H = h->H;
    a.sliding = h->tail_mode == HS_TAIL_SLIDING ? 1 : 0;
    if (hs_launch_append(a, h->B, s) != cudaSuccess) return HS_ERR_CUDA;
    return HS_OK;
}

int hs_reset_requests(hs_handle* h, const int32_t* req_ids, int n, const int32_t* lengths,
                      hs_stream_t stream)
{
    if (!valid(h) || n < 0 || (n > 0 && !req_ids)) return HS_ERR_ARG;
    if (n > HS_MAX_BATCH) return HS_ERR_LIMIT;
    if (n == 0) return HS_OK;
    DeviceGuard g(h->device);
    ResetArgs a;
    a.ids = req_ids;
    a.lengths = lengths;
    a.tok_slot = h->d_tok_slot;
    a.slot_tok = h->d_slot_tok;
    a.stamp = h->d_stamp;
    a.len = h->d_len;
    a.st = h->d_st;
    a.B = h->B;
    a.C = h->C;
    a.S = h->S;
    if (hs_launch_reset_requests(a, n, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return HS_ERR_CUDA;
    return HS_OK;
}

int hs_set_tail_rows(hs_handle* h, int b, int first_token, int n, const uint8_t* rows_host)
{
    if (!valid(h) || !rows_host || b < 0 || b >= h->B || n < 0 || h->T <= 0) return HS_ERR_ARG;
    const int lowest = h->tail_mode == HS_TAIL_SLIDING ? 0 : h->cold;
    if (first_token < lowest || (long long)first_token + n > h->C) return HS_ERR_ARG;
    DeviceGuard g(h->device);
    if (sync_last(h) != HS_OK) return HS_ERR_CUDA;
    const size_t R = (size_t)h->R;
    uint8_t* base = h->d_buf + (size_t)b * (size_t)(h->S + h->T) * R;
    // Consecutive tokens occupy consecutive tail slots until t mod T wraps.
    for (int i = 0; i < n;) {
        const int t = first_token + i;
        const int slot = t % h->T;
        int run = h->T - slot;
        if (run > n - i) run = n - i;
        if (cudaMemcpy(base + (size_t)(h->S + slot) * R, rows_host + (size_t)i * R, (size_t)run * R,
                       cudaMemcpyHostToDevice) != cudaSuccess)
            return HS_ERR_CUDA;
        i += run;
    }
    return HS_OK;
}

int hs_export_state(hs_handle* h, int32_t* tok_slot, int32_t* slot_tok, int32_t* stamp,
                    int32_t* step)
{
    if (!valid(h)) return HS_ERR_ARG;
    DeviceGuard g(h->device);
    if (sync_last(h) != HS_OK) return HS_ERR_CUDA;
    const size_t B = (size_t)h->B;
    if (tok_slot && cudaMemcpy(tok_slot, h->d_tok_slot, B * h->C * sizeof(int32_t),
                               cudaMemcpyDeviceToHost) != cudaSuccess)
        return HS_ERR_CUDA;
    if (slot_tok && cudaMemcpy(slot_tok, h->d_slot_tok, B * h->S * sizeof(int32_t),
                               cudaMemcpyDeviceToHost) != cudaSuccess)
        return HS_ERR_CUDA;
    if (stamp && cudaMemcpy(stamp, h->d_stamp, B * h->S * sizeof(int32_t),
                            cudaMemcpyDeviceToHost) != cudaSuccess)
        return HS_ERR_CUDA;
    if (step) {
        HsDevState st;
        if (cudaMemcpy(&st, h->d_st, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess)
            return HS_ERR_CUDA;
        *step = st.step;
    }
    return HS_OK;
}

int hs_import_state(hs_handle* h, const int32_t* tok_slot, const int32_t* slot_tok,
                    const int32_t* stamp, int32_t step)
{
    if (!valid(h) || !tok_slot || !slot_tok || !stamp || step < 0 || step > HS_MAX_STEP)
        return HS_ERR_ARG;
    const size_t C = (size_t)h->C, S = (size_t)h->S;
    for (int b = 0; b < h->B; ++b) {
        const int32_t* ts = tok_slot + (size_t)b * C;
        const int32_t* st = slot_tok + (size_t)b * S;
        const int32_t* sp = stamp + (size_t)b * S;
        size_t occupied = 0;
        for (size_t v = 0; v < S; ++v) {
            const int32_t t = st[v];
            if (sp[v] < 0 || sp[v] > step) return HS_ERR_ARG;
            if (t == -1) continue;
            if (t < 0 || t >= h->cold || ts[t] != (int32_t)v) return HS_ERR_ARG;
            ++occupied;
        }
        size_t mapped = 0;
        for (size_t t = 0; t < C; ++t) {
            const int32_t v = ts[t];
            if (v == -1) continue;
            if (v < 0 || (size_t)v >= S || (int)t >= h->cold || st[v] != (int32_t)t) return HS_ERR_ARG;
            ++mapped;
        }
        if (mapped != occupied) return HS_ERR_ARG;
    }
    DeviceGuard g(h->device);
    if (sync_last(h) != HS_OK) return HS_ERR_CUDA;
    const size_t B = (size_t)h->B;
    if (cudaMemcpy(h->d_tok_slot, tok_slot, B * C * sizeof(int32_t), cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        cudaMemcpy(h->d_slot_tok, slot_tok, B * S * sizeof(int32_t), cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        cudaMemcpy(h->d_stamp, stamp, B * S * sizeof(int32_t), cudaMemcpyHostToDevice) != cudaSuccess)
        return HS_ERR_CUDA;
    HsDevState st = {};
    st.step = step;
    if (cudaMemcpy(h->d_st, &st, sizeof(st), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(h->d_done, 0, sizeof(unsigned)) != cudaSuccess)
        return HS_ERR_CUDA;
    return HS_OK;
}

int hs_export_buffer(hs_handle* h, int b, uint8_t* dst_host)
{
    if (!valid(h) || !dst_host || b < 0 || b >= h->B) return HS_ERR_ARG;
    DeviceGuard g(h->device);
    if (sync_last(h) != HS_OK) return HS_ERR_CUDA;
    const size_t row = (size_t)(h->S + h->T) * (size_t)h->R;
    if (cudaMemcpy(dst_host, h->d_buf + (size_t)b * row, row, cudaMemcpyDeviceToHost) != cudaSuccess)
        return HS_ERR_CUDA;
    return HS_OK;
}

int hs_reset(hs_handle* h)
{
    if (!valid(h)) return HS_ERR_ARG;
    DeviceGuard g(h->device);
    if (sync_last(h) != HS_OK) return HS_ERR_CUDA;
    return fill_start_state(h);
}

int hs_profile_events(hs_handle* h, void* before_copy, void* after_copy)
{
    if (!valid(h) || (before_copy == nullptr) != (after_copy == nullptr)) return HS_ERR_ARG;
    h->prof_before = static_cast<cudaEvent_t>(before_copy);
    h->prof_after = static_cast<cudaEvent_t>(after_copy);
    return HS_OK;
}

int hs_h2d_read(const void* src_host, void* dst_dev, size_t bytes, int blocks, hs_stream_t stream)
{
    if (!src_host || !dst_dev || bytes == 0 || (bytes % 16) != 0 || blocks < 0) return HS_ERR_ARG;
    void* dsrc = nullptr;
    if (cudaHostGetDevicePointer(&dsrc, const_cast<void*>(src_host), 0) != cudaSuccess) {
        cudaGetLastError();
        return HS_ERR_ARG;
    }
    int grid = blocks;
    if (grid == 0) {
        int dev = 0, sms = 1;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        grid = sms * 4;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (hs_launch_h2d_read(static_cast<const uint8_t*>(dsrc), static_cast<uint8_t*>(dst_dev), bytes,
                           grid, s) != cudaSuccess)
        return HS_ERR_CUDA;
    return HS_OK;
}

}  // extern "C"
