// hs_resolve_noalloc: the swap-in step for callers that must not allocate.
//
// Some callers cannot let a library allocate device memory: serving engines
// that reserve almost all of HBM for their own KV pool at start-up (a
// cudaMalloc from a library then fails or fragments that reservation), and
// decode loops where an allocation would synchronise the device and stall
// the step.  Such a caller owns the swap-in state itself (tables, stamps,
// lengths, buffer, pinned host pool and a small control block) and passes
// pointers to it.  The only memory this path needs beyond that -- the
// per-step miss lists that the resolve kernel hands to the copy kernel --
// lives in the fixed-size device array below, so the call allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU on which the
// library's module is loaded holds it until the process exits.  From host
// code its name is only a stand-in, so the device address is looked up once
// per device with cudaGetSymbolAddress (on the first call made with that
// device current) and passed to the kernels.  All calls share the array and
// it keeps the last call's contents; nothing in it has to start at zero (the
// resolve kernel writes every list entry and count the copy kernel reads).
// Calls on one device whose work overlaps on the GPU (for example on two
// streams) race on that device's array; order them on one stream.  Each
// device has its own copy of the array.
#include <cstddef>
#include <mutex>

#include "hs_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kListEntries = (size_t)HS_NOALLOC_MAX_ENTRIES;     // B * K
constexpr size_t kScratchBytes = 2 * kListEntries * sizeof(int32_t)  // miss tokens, victim slots
                                 + (size_t)HS_MAX_BATCH * sizeof(int32_t);  // miss counts

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct DeviceScratch {
    std::once_flag once;
    cudaError_t status = cudaErrorNotReady;
    unsigned char* ptr = nullptr;
};

DeviceScratch g_dev[kMaxDevices];

static_assert(sizeof(hs_control_t) == sizeof(HsDevState), "control block layout");
static_assert(offsetof(hs_control_t, step) == offsetof(HsDevState, step), "control step");
static_assert(offsetof(hs_control_t, err_bits) == offsetof(HsDevState, err), "control err");
static_assert(offsetof(hs_control_t, hits) == offsetof(HsDevState, hits), "control hits");
static_assert(offsetof(hs_control_t, misses) == offsetof(HsDevState, misses), "control misses");
static_assert(offsetof(hs_control_t, inplace) == offsetof(HsDevState, inplace), "control inplace");

// Per-device set-up, run once with that device current: the scratch address
// and the resolve kernel's shared-memory limit.  Neither allocates.
DeviceScratch* scratch_for(int dev)
{
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    DeviceScratch* d = &g_dev[dev];
    std::call_once(d->once, [d]() {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e == cudaSuccess) e = hs_prepare_resolve();
        d->ptr = static_cast<unsigned char*>(p);
        d->status = e;
    });
    return d->status == cudaSuccess ? d : nullptr;
}

}  // namespace

extern "C" int hs_resolve_noalloc(int batch, int ctx_len, int row_bytes, int buffer_slots,
                                  int host_rows, int resident_tail, const int32_t* topk_idx, int K,
                                  int32_t* out_slot, int32_t* tok_slot, int32_t* slot_tok,
                                  int32_t* stamp, const int32_t* lengths, const uint8_t* host_pool,
                                  uint8_t* device_buffer, hs_control_t* control,
                                  hs_stream_t stream)
{
    if (!topk_idx || !out_slot || !tok_slot || !slot_tok || !stamp || !lengths || !host_pool ||
        !device_buffer || !control)
        return HS_ERR_ARG;
    if (batch <= 0 || ctx_len <= 0 || row_bytes <= 0 || (row_bytes % 16) != 0 ||
        buffer_slots <= 0 || host_rows < 0 || resident_tail < 0 || resident_tail > ctx_len ||
        K <= 0)
        return HS_ERR_ARG;
    if (K > buffer_slots) return HS_ERR_TOPK_GT_SLOTS;
    if (host_rows < ctx_len - resident_tail) return HS_ERR_CAPACITY;
    // Sizes the fixed scratch array (and the kernels) cannot take.
    if (batch > HS_MAX_BATCH || buffer_slots > HS_MAX_SLOTS || K > HS_MAX_TOPK ||
        row_bytes > HS_MAX_ROW_BYTES || (long long)batch * K > HS_NOALLOC_MAX_ENTRIES)
        return HS_ERR_LIMIT;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HS_ERR_CUDA;
    DeviceScratch* d = scratch_for(dev);
    if (!d) return HS_ERR_CUDA;

    // The pool must be pinned and mapped; this looks up its device address.
    void* pool_dev = nullptr;
    if (cudaHostGetDevicePointer(&pool_dev, const_cast<uint8_t*>(host_pool), 0) != cudaSuccess) {
        cudaGetLastError();
        return HS_ERR_ARG;
    }

    int32_t* miss_tok = reinterpret_cast<int32_t*>(d->ptr);
    int32_t* miss_slot = miss_tok + (size_t)batch * K;
    int32_t* miss_cnt = miss_tok + 2 * kListEntries;
    HsDevState* st = reinterpret_cast<HsDevState*>(control);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    ResolveArgs ra;
    ra.topk = topk_idx;
    ra.out = out_slot;
    ra.tok_slot = tok_slot;
    ra.slot_tok = slot_tok;
    ra.stamp = stamp;
    ra.len = lengths;
    ra.miss_tok = miss_tok;
    ra.miss_slot = miss_slot;
    ra.miss_cnt = miss_cnt;
    ra.st = st;
    ra.K = K;
    ra.C = ctx_len;
    ra.S = buffer_slots;
    ra.T = resident_tail;
    ra.cold = ctx_len - resident_tail;
    ra.list_stride = K;
    ra.hash_bits = hs_hash_bits(K);
    ra.pool = nullptr;
    ra.buf = nullptr;
    ra.H = host_rows;
    ra.R = row_bytes;
    ra.rows_per_group = 1;
    ra.done = nullptr;
    ra.fifo = 0;
    ra.sliding = 0;
    ra.alias = 0;
    if (hs_launch_resolve(ra, batch, s) != cudaSuccess) return HS_ERR_CUDA;

    int sms = 1;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    CopyArgs ca;
    ca.miss_cnt = miss_cnt;
    ca.miss_tok = miss_tok;
    ca.miss_slot = miss_slot;
    ca.pool = static_cast<const uint8_t*>(pool_dev);
    ca.buf = device_buffer;
    ca.st = st;
    ca.B = batch;
    ca.S = buffer_slots;
    ca.T = resident_tail;
    ca.R = row_bytes;
    ca.list_stride = K;
    ca.H = host_rows;
    const int unroll = hs_copy_unroll_for(row_bytes);
    ca.rows_per_group = hs_copy_rows_per_group(row_bytes, unroll);
    ca.advance_step = 1;
    ca.flat_src = 0;
    const int grid = (sms > 0 ? sms : 1) * hs_copy_blocks_per_sm(unroll, batch);
    if (hs_launch_copy(ca, grid, unroll, s, true) != cudaSuccess) return HS_ERR_CUDA;
    return HS_OK;
}
