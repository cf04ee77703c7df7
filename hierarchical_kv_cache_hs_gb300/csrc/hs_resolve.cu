// Resolve kernel of the HiSparse swap-in path: steps (1)-(3) of the swap-in
// kernel of the HiSparse blog ("Efficient swap-in kernel"): miss
// identification, LRU victim selection and the page-table update.  The host
// row fetch of step (3) runs in the copy kernel that follows (hs_copy.cu).
//
// One CTA of 1024 threads per request.  Everything the request's step needs
// stays in shared memory:
//   - a 2K-entry open-addressing hash of the row's indices, which finds
//     repeated indices (the first occurrence wins);
//   - the request's S stamps (read once, written back once, coalesced);
//   - the miss list in top-k row order (block scan of per-thread counts);
//   - the victim list in ascending slot order.
// Victims are the m smallest (stamp, slot) pairs.  A block-wide radix select
// over the stamps (8-bit digits, most significant first, only the digits
// that the current step counter can populate) finds the m-th smallest stamp
// tau; every slot below tau is a victim, and so are the lowest-index slots
// equal to tau until m are taken.  Slots hit in this step carry the current
// step -- larger than every other stamp -- so they are never chosen.
#include <climits>

#include "hs_internal.h"

namespace {

constexpr int NT = HS_RESOLVE_THREADS;
constexpr int NW = NT / 32;
constexpr int EMAX = HS_MAX_TOPK / NT;  // top-k entries per thread
constexpr unsigned FULL = 0xffffffffu;

static_assert(NW == 32, "block scans assume 32 warps");
static_assert(EMAX * NT == HS_MAX_TOPK, "entries per thread");

enum : int { C_NONE = 0, C_BAD = 1, C_TAIL = 2, C_HIT = 3, C_MISS = 4 };

__device__ __forceinline__ int warp_incl_scan(int v, int lane)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int n = __shfl_up_sync(FULL, v, d);
        if (lane >= d) v += n;
    }
    return v;
}

// Block-wide exclusive scan (all NT threads call it); *total = block sum.
__device__ __forceinline__ int block_excl_scan(int v, int* s_w, int* total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int incl = warp_incl_scan(v, lane);
    if (lane == 31) s_w[warp] = incl;
    __syncthreads();
    if (warp == 0) s_w[lane] = warp_incl_scan(s_w[lane], lane);
    __syncthreads();
    const int off = warp ? s_w[warp - 1] : 0;
    *total = s_w[NW - 1];
    __syncthreads();
    return off + incl - v;
}

__device__ __forceinline__ int hs_region_a_ints(int hash_bits)
{
    const int hc2 = 2 << hash_bits;
    return hc2 > NW * 256 ? hc2 : NW * 256;
}

__global__ void __launch_bounds__(NT, 1) hs_resolve_kernel(ResolveArgs a)
{
    extern __shared__ __align__(16) int smem[];
    __shared__ int s_w[32];
    __shared__ int s_cnt[3];  // hits, in-place, error bits
    __shared__ int s_sel[2];  // selected digit, count below it

    // The copy grid may be scheduled as soon as every resolve CTA is running;
    // it waits for this grid's completion before reading anything.
    asm volatile("griddepcontrol.launch_dependents;");

    const int hc = 1 << a.hash_bits;
    int* s_hkey = smem;                                  // [hc]  (phase 1)
    int* s_hj = smem + hc;                               // [hc]  (phase 1)
    int* s_hist = smem;                                  // [NW][256] (phase 2, reuses the hash)
    int* s_stamp = smem + hs_region_a_ints(a.hash_bits); // [S]
    int* s_mtok = s_stamp + a.S;                         // [K]
    int* s_mj = s_mtok + a.K;                            // [K]
    int* s_vic = s_mj + a.K;                             // [K]

    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = a.K, S = a.S;
    const int step = a.st->step + 1;
    const int len = a.len[b];
    const int32_t* g_topk = a.topk + (size_t)b * K;
    int32_t* g_out = a.out + (size_t)b * K;
    int32_t* g_stamp = a.stamp + (size_t)b * S;
    const int32_t* g_tok_slot = a.tok_slot + (size_t)b * a.C;

    for (int i = tid; i < hc; i += NT) {
        s_hkey[i] = -1;
        s_hj[i] = INT_MAX;
    }
    for (int i = tid; i < S; i += NT) s_stamp[i] = g_stamp[i];
    if (tid < 3) s_cnt[tid] = 0;
    __syncthreads();

    // ---- (1) classify, drop repeats, gather the page table -------------
    // Thread tid owns the contiguous entries [tid*E, tid*E + E) so that a
    // block scan of per-thread miss counts yields row order.
    const int E = (K + NT - 1) / NT;
    const int j0 = tid * E;
    int tk[EMAX], cl[EMAX], hs[EMAX], sl[EMAX];
    int err = 0;
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        tk[e] = -1;
        cl[e] = C_NONE;
        hs[e] = 0;
        sl[e] = -1;
        const int j = j0 + e;
        if (e < E && j < K) {
            const int t = g_topk[j];
            tk[e] = t;
            if (t == -1) {
                cl[e] = C_NONE;
            } else if (t < -1 || t >= len || t >= a.C) {
                cl[e] = C_BAD;
                err |= HS_E_RANGE;
            } else {
                unsigned h = ((unsigned)t * 0x9E3779B1u) >> (32 - a.hash_bits);
                for (;;) {
                    const int k = atomicCAS(&s_hkey[h], -1, t);
                    if (k == -1 || k == t) break;
                    h = (h + 1) & (unsigned)(hc - 1);
                }
                atomicMin(&s_hj[h], j);
                hs[e] = (int)h;
                cl[e] = C_MISS;  // valid; refined below
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        if (cl[e] == C_MISS) {
            if (s_hj[hs[e]] != j0 + e) {
                cl[e] = C_BAD;
                err |= HS_E_DUP;
            } else if (tk[e] >= a.cold) {
                cl[e] = C_TAIL;
                sl[e] = S + tk[e] % a.T;
            } else {
                sl[e] = g_tok_slot[tk[e]];
            }
        }
    }
    int nh = 0, ni = 0, nm = 0;
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        const int j = j0 + e;
        if (cl[e] == C_MISS) {
            if (sl[e] >= 0) {
                cl[e] = C_HIT;
                s_stamp[sl[e]] = step;  // a hit refreshes its LRU entry
                g_out[j] = sl[e];
                ++nh;
            } else {
                ++nm;
            }
        } else if (cl[e] == C_TAIL) {
            g_out[j] = sl[e];
            ++ni;
        } else if (e < E && j < K) {
            g_out[j] = -1;
        }
    }
    nh = __reduce_add_sync(FULL, nh);
    ni = __reduce_add_sync(FULL, ni);
    err = __reduce_or_sync(FULL, err);
    if (lane == 0) {
        if (nh) atomicAdd(&s_cnt[0], nh);
        if (ni) atomicAdd(&s_cnt[1], ni);
        if (err) atomicOr(&s_cnt[2], err);
    }

    int m = 0;
    int pos = block_excl_scan(nm, s_w, &m);
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        if (cl[e] == C_MISS) {
            s_mtok[pos] = tk[e];
            s_mj[pos] = j0 + e;
            ++pos;
        }
    }

    if (m > 0) {
        // ---- (2) LRU victims: radix select of the m-th smallest stamp ----
        const int nbits = 32 - __clz(step);
        unsigned prefix = 0, pmask = 0;
        int remaining = m;
        const int s_pad = (S + NT - 1) / NT * NT;
        for (int d = (nbits - 1) >> 3; d >= 0; --d) {
            const int shift = 8 * d;
            for (int i = tid; i < NW * 256; i += NT) s_hist[i] = 0;
            __syncthreads();
            for (int i = tid; i < s_pad; i += NT) {
                int dig = 256;
                if (i < S) {
                    const unsigned k = (unsigned)s_stamp[i];
                    if ((k & pmask) == prefix) dig = (int)((k >> shift) & 255u);
                }
                const unsigned peers = __match_any_sync(FULL, dig);
                if (dig < 256 && lane == __ffs(peers) - 1)
                    atomicAdd(&s_hist[warp * 256 + dig], __popc(peers));
            }
            __syncthreads();
            int c = 0, incl = 0;
            if (tid < 256) {
#pragma unroll 8
                for (int w = 0; w < NW; ++w) c += s_hist[w * 256 + tid];
                incl = warp_incl_scan(c, lane);
                if (lane == 31) s_w[warp] = incl;
            }
            __syncthreads();
            if (tid < 256) {
                int off = 0;
                for (int w = 0; w < warp; ++w) off += s_w[w];
                const int excl = off + incl - c;
                if (c > 0 && excl < remaining && remaining <= excl + c) {
                    s_sel[0] = tid;
                    s_sel[1] = excl;
                }
            }
            __syncthreads();
            prefix |= (unsigned)s_sel[0] << shift;
            pmask |= 255u << shift;
            remaining -= s_sel[1];
        }
        const int tau = (int)prefix;
        const int need_eq = remaining;  // slots equal to tau taken, lowest index first

        // Victims in ascending slot order: thread tid owns slots [tid*Q, tid*Q + Q).
        const int Q = (S + NT - 1) / NT;
        const int q0 = tid * Q;
        int nl = 0, ne = 0;
        for (int q = 0; q < Q; ++q) {
            const int s = q0 + q;
            if (s < S) {
                const int k = s_stamp[s];
                nl += k < tau;
                ne += k == tau;
            }
        }
        int tot;
        const int packed = block_excl_scan((nl << 16) | ne, s_w, &tot);
        int lb = packed >> 16, eb = packed & 0xffff;
        for (int q = 0; q < Q; ++q) {
            const int s = q0 + q;
            if (s < S) {
                const int k = s_stamp[s];
                // Exactly m slots qualify; the bound only keeps a corrupted
                // stamp from writing past the list.
                if (k < tau) {
                    const int p = lb + (eb < need_eq ? eb : need_eq);
                    if (p < m) s_vic[p] = s;
                    ++lb;
                } else if (k == tau) {
                    if (eb < need_eq && lb + eb < m) s_vic[lb + eb] = s;
                    ++eb;
                }
            }
        }
        __syncthreads();

        // ---- (3) pair the i-th miss (row order) with the i-th victim ------
        int32_t* g_slot_tok = a.slot_tok + (size_t)b * S;
        int32_t* g_tok_slot_w = a.tok_slot + (size_t)b * a.C;
        int32_t* g_mtok = a.miss_tok + (size_t)b * a.list_stride;
        int32_t* g_mslot = a.miss_slot + (size_t)b * a.list_stride;
        for (int i = tid; i < m; i += NT) {
            const int t = s_mtok[i];
            const int v = s_vic[i];
            const int old = g_slot_tok[v];
            if (old >= 0) g_tok_slot_w[old] = -1;  // the evicted token leaves the table
            g_slot_tok[v] = t;
            g_tok_slot_w[t] = v;
            s_stamp[v] = step;
            g_out[s_mj[i]] = v;
            g_mtok[i] = t;
            g_mslot[i] = v;
        }
    }
    __syncthreads();
    for (int i = tid; i < S; i += NT) g_stamp[i] = s_stamp[i];
    if (tid == 0) {
        a.miss_cnt[b] = m;
        if (s_cnt[0]) atomicAdd(&a.st->hits, (unsigned long long)s_cnt[0]);
        if (s_cnt[1]) atomicAdd(&a.st->inplace, (unsigned long long)s_cnt[1]);
        if (m) atomicAdd(&a.st->misses, (unsigned long long)m);
        if (s_cnt[2]) atomicOr(&a.st->err, s_cnt[2]);
    }
}

}  // namespace

int hs_hash_bits(int K)
{
    int bits = 6;
    while ((1 << bits) < 2 * K) ++bits;
    return bits;
}

size_t hs_resolve_smem_bytes(int K, int S)
{
    const int hb = hs_hash_bits(K);
    const int hc2 = 2 << hb;
    const int region_a = hc2 > NW * 256 ? hc2 : NW * 256;
    return sizeof(int) * ((size_t)region_a + (size_t)S + 3u * (size_t)K);
}

cudaError_t hs_prepare_resolve()
{
    const size_t most = hs_resolve_smem_bytes(HS_MAX_TOPK, HS_MAX_SLOTS);
    return cudaFuncSetAttribute(hs_resolve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)most);
}

cudaError_t hs_launch_resolve(const ResolveArgs& a, int B, cudaStream_t s)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)B);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = hs_resolve_smem_bytes(a.K, a.S);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, hs_resolve_kernel, a);
}
