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
// code its name is only a stand-in, so the device address is looked up per
// device with cudaGetSymbolAddress (on the first call made with that device
// current) and passed to the kernels.  That set-up is kept only once it has
// succeeded: a call that finds it failed tries it again.  It is refused while
// the call's stream is being captured into a CUDA graph, so the first call on
// a device must come before any capture.  All calls share the array and it
// keeps the last call's contents; nothing in it has to start at zero (the
// resolve kernel writes every list entry and count the copy kernel reads).
// Calls on one device whose work overlaps on the GPU (for example on two
// streams) race on that device's array; order them on one stream.  Each
// device has its own copy of the array.
//
// The step itself is the one hs_resolve takes with its defaults -- LRU
// eviction, the fixed resident tail [C - T, C) -- in two launches: the
// resolve kernel, then the grid-wide row-copy kernel.
#include <cuda.h>

#include <atomic>
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
    std::mutex mu;
    std::atomic<bool> ready{false};
    unsigned char* ptr = nullptr;
};

DeviceScratch g_dev[kMaxDevices];

// cuPointerGetAttribute and cuMemGetAddressRange, found through the runtime
// so that the library does not link the driver library itself.
using PointerGetAttributeFn = CUresult (*)(void*, CUpointer_attribute, CUdeviceptr);
using GetAddressRangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);
std::atomic<PointerGetAttributeFn> g_get_attr{nullptr};
std::atomic<GetAddressRangeFn> g_get_range{nullptr};

cudaError_t driver_fn(const char* name, void** fn)
{
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    *fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion(name, fn, CUDA_VERSION, cudaEnableDefault, &q);
    if (e == cudaSuccess && (q != cudaDriverEntryPointSuccess || !*fn)) e = cudaErrorSymbolNotFound;
    return e;
}

static_assert(sizeof(hs_control_t) == sizeof(HsDevState), "control block layout");
static_assert(offsetof(hs_control_t, step) == offsetof(HsDevState, step), "control step");
static_assert(offsetof(hs_control_t, err_bits) == offsetof(HsDevState, err), "control err");
static_assert(offsetof(hs_control_t, hits) == offsetof(HsDevState, hits), "control hits");
static_assert(offsetof(hs_control_t, misses) == offsetof(HsDevState, misses), "control misses");
static_assert(offsetof(hs_control_t, inplace) == offsetof(HsDevState, inplace), "control inplace");

// Per-device set-up with that device current: the scratch address, the
// resolve kernel's shared-memory limit and the pointer-attribute query.  None
// of it allocates.  Returns HS_OK and the scratch address; HS_ERR_ARG when
// the set-up is still to do and `s` is being captured; HS_ERR_CUDA when a
// call failed (nothing is kept, so the next call tries again).
int scratch_for(int dev, cudaStream_t s, unsigned char** out)
{
    if (dev < 0 || dev >= kMaxDevices) return HS_ERR_CUDA;
    DeviceScratch* d = &g_dev[dev];
    if (!d->ready.load(std::memory_order_acquire)) {
        std::lock_guard<std::mutex> lock(d->mu);
        if (!d->ready.load(std::memory_order_relaxed)) {
            cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
            if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
                cudaGetLastError();
                return HS_ERR_CUDA;
            }
            if (cs != cudaStreamCaptureStatusNone) return HS_ERR_ARG;
            void* p = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e == cudaSuccess) e = hs_prepare_resolve();
            void* fa = nullptr;
            void* fr = nullptr;
            if (e == cudaSuccess) e = driver_fn("cuPointerGetAttribute", &fa);
            if (e == cudaSuccess) e = driver_fn("cuMemGetAddressRange", &fr);
            if (e == cudaSuccess) {
                g_get_attr.store(reinterpret_cast<PointerGetAttributeFn>(fa));
                g_get_range.store(reinterpret_cast<GetAddressRangeFn>(fr));
            }
            if (e != cudaSuccess) {
                cudaGetLastError();
                return HS_ERR_CUDA;
            }
            d->ptr = static_cast<unsigned char*>(p);
            d->ready.store(true, std::memory_order_release);
        }
    }
    *out = d->ptr;
    return HS_OK;
}

// The copy kernel reads B * host_rows * R bytes from the pool: they must lie
// inside the one pinned allocation that holds its first byte.  The driver
// reports that allocation's extent (as an address range of the pointer, else
// as the range of the allocation); memory whose extent it does not know is
// refused.
bool pool_inside_allocation(const void* pool_dev, size_t bytes)
{
    const CUdeviceptr p = (CUdeviceptr)(uintptr_t)pool_dev;
    CUdeviceptr start = 0;
    size_t size = 0;
    bool known = false;
    if (PointerGetAttributeFn get = g_get_attr.load())
        known = get(&start, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, p) == CUDA_SUCCESS &&
                get(&size, CU_POINTER_ATTRIBUTE_RANGE_SIZE, p) == CUDA_SUCCESS && size > 0;
    if (!known) {
        GetAddressRangeFn range = g_get_range.load();
        known = range && range(&start, &size, p) == CUDA_SUCCESS && size > 0;
    }
    if (!known || p < start || p - start >= size) return false;
    return bytes <= size - (size_t)(p - start);
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

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

    // Alignment the kernels' accesses need: 16-byte row loads and stores,
    // 64-bit counter atomics in the control block, 32-bit table entries.
    if (!aligned(host_pool, 16) || !aligned(device_buffer, 16) || !aligned(control, 8) ||
        !aligned(topk_idx, 4) || !aligned(out_slot, 4) || !aligned(tok_slot, 4) ||
        !aligned(slot_tok, 4) || !aligned(stamp, 4) || !aligned(lengths, 4))
        return HS_ERR_ARG;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HS_ERR_CUDA;
    unsigned char* scratch = nullptr;
    const int rc = scratch_for(dev, s, &scratch);
    if (rc != HS_OK) return rc;

    // The pool must be pinned and mapped; this looks up its device address.
    void* pool_dev = nullptr;
    if (cudaHostGetDevicePointer(&pool_dev, const_cast<uint8_t*>(host_pool), 0) != cudaSuccess) {
        cudaGetLastError();
        return HS_ERR_ARG;
    }
    if (!pool_inside_allocation(pool_dev, (size_t)batch * (size_t)host_rows * (size_t)row_bytes))
        return HS_ERR_ARG;

    int32_t* miss_tok = reinterpret_cast<int32_t*>(scratch);
    int32_t* miss_slot = miss_tok + (size_t)batch * K;
    int32_t* miss_cnt = miss_tok + 2 * kListEntries;
    HsDevState* st = reinterpret_cast<HsDevState*>(control);

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
    ra.random = 0;
    ra.seed = 0;
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
