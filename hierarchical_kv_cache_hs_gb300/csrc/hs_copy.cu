// Row fetch of the HiSparse swap-in path: the "fetch the needed entries from
// host into device memory" half of step (3) of the HiSparse blog's swap-in
// kernel, one row from pinned host memory into each victim slot (vLLM Hybrid
// HiSparse post, "Mixed Residency").
//
// The rows of all requests are flattened into one list (prefix sum of the
// per-request miss counts, computed by every CTA in shared memory) so that no
// SM idles on a request with few misses; each warp takes an equal contiguous
// run of it.  A warp copies `rows_per_group`
// rows at a time: its first lanes look up one row each (request, token,
// victim slot), then every lane streams 16-byte chunks of those rows with
// zero-copy loads from the mapped host pool -- U independent loads in flight
// per lane before the matching stores to HBM.
//
// Also here: the resident-tail append, the reset of single requests (a batch
// slot taken by a new request) and a sequential host-read probe used to
// measure the host->device link.
#include "hs_internal.h"

namespace {

constexpr int CT = HS_COPY_THREADS;
constexpr int CW = CT / 32;
constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ uint4 ld_host_v4(const uint8_t* p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st_v4(uint8_t* p, const uint4& v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

template <int U>
__global__ void __launch_bounds__(CT) hs_copy_kernel(CopyArgs a)
{
    extern __shared__ int s_pref[];  // [B + 1]
    __shared__ int s_w[CW];

    // Wait until the resolve grid has finished and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // Advance the step counter (wrapping: the next resolve clamps a counter
    // outside its range and reports it).
    if (a.advance_step && blockIdx.x == 0 && tid == 0) a.st->step = (int)((unsigned)a.st->step + 1u);

    // Exclusive prefix of the miss counts over requests.
    int carry = 0;
    for (int base = 0; base < a.B; base += CT) {
        const int v = (base + tid < a.B) ? a.miss_cnt[base + tid] : 0;
        int incl = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int n = __shfl_up_sync(FULL, incl, d);
            if (lane >= d) incl += n;
        }
        if (lane == 31) s_w[warp] = incl;
        __syncthreads();
        int off = 0, tot = 0;
        for (int w = 0; w < CW; ++w) {
            const int x = s_w[w];
            if (w < warp) off += x;
            tot += x;
        }
        if (base + tid < a.B) s_pref[base + tid] = carry + off + incl - v;
        carry += tot;
        __syncthreads();
    }
    if (tid == 0) s_pref[a.B] = carry;
    __syncthreads();

    const int total = s_pref[a.B];
    const int cpr = a.R >> 4;  // 16-byte chunks per row
    const int G = a.rows_per_group;
    const long long slots = (long long)(a.S + a.T);
    const int gw = (int)((blockIdx.x * (unsigned)CT + tid) >> 5);
    const int nw = (int)((gridDim.x * (unsigned)CT) >> 5);

    // Each warp copies one contiguous run of the flattened list, so it reads
    // the rows of one or two requests: a narrow window of the host pool per
    // SM.  (Striding the groups over the whole grid scattered every SM's reads
    // over the whole pool, and cost a third of the rate on 38 GB of pools.)
    const long long per = ((total + nw - 1) / nw + G - 1) / G * G;
    const long long beg = (long long)gw * per;
    const long long end = beg + per < total ? beg + per : total;
    for (long long r0 = beg; r0 < end; r0 += G) {
        long long src = 0, dst = 0;
        const long long r = r0 + lane;
        if (lane < G && r < end) {
            int lo = 0, hi = a.B - 1;  // request b with s_pref[b] <= r < s_pref[b + 1]
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_pref[mid] <= r) lo = mid; else hi = mid - 1;
            }
            const int i = (int)(r - s_pref[lo]);
            const size_t li = (size_t)lo * a.list_stride + i;
            // Flat source: row r of a staging area (the copy-engine variant);
            // otherwise token t of request lo in the host pool.
            src = a.flat_src ? r * a.R : ((long long)lo * a.H + a.miss_tok[li]) * a.R;
            dst = ((long long)lo * slots + a.miss_slot[li]) * a.R;
        }
        const int nrows = (int)((end - r0) < G ? (end - r0) : G);
        const int nch = nrows * cpr;
        for (int c0 = 0; c0 < nch; c0 += 32 * U) {
            uint4 v[U];
            long long d[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * 32 + lane;
                const int rr = c < nch ? c / cpr : 0;
                const long long s = __shfl_sync(FULL, src, rr);
                d[u] = __shfl_sync(FULL, dst, rr);
                const int off = (c - rr * cpr) << 4;
                d[u] += off;
                if (c < nch) v[u] = ld_host_v4(a.pool + s + off);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * 32 + lane;
                if (c < nch) st_v4(a.buf + d[u], v[u]);
            }
        }
    }
}

__global__ void hs_append_kernel(AppendArgs a)
{
    const int b = blockIdx.x;
    const int len = a.len[b];
    const bool ok = a.T > 0 && len < a.C && (a.sliding || len >= a.cold);
    if (ok) {
        const uint4* src = reinterpret_cast<const uint4*>(a.rows + (size_t)b * a.R);
        uint4* dst = reinterpret_cast<uint4*>(
            a.buf + ((size_t)b * (a.S + a.T) + a.S + len % a.T) * a.R);
        // Sliding tail: the slot still holds token len - T, which leaves the
        // tail now; its row goes back to its host row first (zero-copy
        // stores into the mapped pool), chunk by chunk before the overwrite.
        uint4* back = (a.sliding && len >= a.T)
            ? reinterpret_cast<uint4*>(a.pool + ((size_t)b * a.H + (size_t)(len - a.T)) * a.R)
            : nullptr;
        for (int c = threadIdx.x; c < (a.R >> 4); c += blockDim.x) {
            if (back) back[c] = dst[c];
            dst[c] = src[c];
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        if (ok) a.len[b] = len + 1;
        else atomicOr(&a.st->err, HS_E_APPEND);
    }
}

// One CTA per listed request: empty tables, stamps 0 ("never used", so the
// request's slots are the first victims, lowest index first), new length.
__global__ void hs_reset_requests_kernel(ResetArgs a)
{
    const int b = a.ids[blockIdx.x];
    const int len = a.lengths ? a.lengths[blockIdx.x] : a.C;
    if (b < 0 || b >= a.B || len < 0 || len > a.C) {
        if (threadIdx.x == 0) atomicOr(&a.st->err, HS_E_RANGE);
        return;
    }
    int32_t* ts = a.tok_slot + (size_t)b * a.C;
    int32_t* sl = a.slot_tok + (size_t)b * a.S;
    int32_t* sp = a.stamp + (size_t)b * a.S;
    for (int t = threadIdx.x; t < a.C; t += blockDim.x) ts[t] = -1;
    for (int v = threadIdx.x; v < a.S; v += blockDim.x) {
        sl[v] = -1;
        sp[v] = 0;
    }
    if (threadIdx.x == 0) a.len[b] = len;
}

constexpr int PROBE_U = 8;

__global__ void __launch_bounds__(CT) hs_h2d_read_kernel(const uint8_t* src, uint8_t* dst,
                                                         size_t nchunks)
{
    const size_t stride = (size_t)gridDim.x * CT;
    size_t i = (size_t)blockIdx.x * CT + threadIdx.x;
    for (; i + (PROBE_U - 1) * stride < nchunks; i += PROBE_U * stride) {
        uint4 v[PROBE_U];
#pragma unroll
        for (int u = 0; u < PROBE_U; ++u) v[u] = ld_host_v4(src + ((i + u * stride) << 4));
#pragma unroll
        for (int u = 0; u < PROBE_U; ++u) st_v4(dst + ((i + u * stride) << 4), v[u]);
    }
    for (; i < nchunks; i += stride) st_v4(dst + (i << 4), ld_host_v4(src + (i << 4)));
}

}  // namespace

int hs_copy_unroll_for(int row_bytes)
{
    const int cpr = row_bytes >> 4;
    // Prefer the unroll whose warp group (32 * U chunks) holds whole rows.
    if (cpr <= 32 * 9 && (32 * 9) % cpr == 0) return 9;
    return 8;
}

int hs_copy_rows_per_group(int row_bytes, int unroll)
{
    const int cpr = row_bytes >> 4;
    int g = (32 * unroll) / cpr;
    if (g < 1) g = 1;
    if (g > 32) g = 32;
    return g;
}

cudaError_t hs_launch_copy(const CopyArgs& a, int grid, int unroll, cudaStream_t s, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(CT);
    cfg.dynamicSmemBytes = sizeof(int) * ((size_t)a.B + 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    if (pdl) {
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    if (unroll == 9) return cudaLaunchKernelEx(&cfg, hs_copy_kernel<9>, a);
    return cudaLaunchKernelEx(&cfg, hs_copy_kernel<8>, a);
}

int hs_copy_blocks_per_sm(int unroll, int B)
{
    int n = 0;
    const size_t smem = sizeof(int) * ((size_t)B + 1);
    cudaError_t e = unroll == 9
        ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, hs_copy_kernel<9>, CT, smem)
        : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, hs_copy_kernel<8>, CT, smem);
    return (e == cudaSuccess && n > 0) ? n : 1;
}

cudaError_t hs_launch_append(const AppendArgs& a, int B, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)B);
    cfg.blockDim = dim3(128);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, hs_append_kernel, a);
}

cudaError_t hs_launch_reset_requests(const ResetArgs& a, int n, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)n);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, hs_reset_requests_kernel, a);
}

cudaError_t hs_launch_h2d_read(const uint8_t* src, uint8_t* dst, size_t bytes, int grid,
                               cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(CT);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, hs_h2d_read_kernel, src, dst, bytes >> 4);
}
