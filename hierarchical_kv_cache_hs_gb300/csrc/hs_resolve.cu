// Swap-in kernel of the HiSparse path: steps (1)-(3) of the HiSparse blog's
// swap-in kernel ("Efficient swap-in kernel"): miss identification, LRU
// victim selection, and the page-table update with the host -> device row
// fetch.
//
// One CTA of 512 threads resolves each request.  Everything the request's
// step needs stays in its shared memory:
//   - the request's S stamps and S slot -> token entries, loaded once,
//     together with the top-k row, at the start;
//   - a 2K-entry open-addressing hash of the row's indices that finds
//     repeated indices (the first occurrence wins), built while the
//     page-table gathers are in flight;
//   - the miss list in top-k row order (block scan of per-thread counts);
//   - the victim list in ascending slot order;
//   - the out_slot row, kept until the victims are known and then written
//     once, each thread's contiguous entries as 16-byte stores (out_slot may
//     be mapped host memory, where scattered 4-byte writes slowed the step
//     by 6 %).
//
// Victims are the m slots with the smallest (stamp, slot) pairs.  One
// 1024-bin histogram of stamp ages (step - stamp, ages >= 1023 share the
// oldest bin) locates the m-th oldest stamp tau: when it falls in an exact
// bin, tau is that bin's stamp; when it falls in the shared oldest bin, a
// radix select over the stamps of that bin (8-bit digits, most significant
// first) finds it.  Every slot older than tau is a victim, and so are the
// lowest-index slots with stamp tau until m are taken; one packed block scan
// gives each victim its position in ascending slot order.  Slots hit in this
// step carry the current step -- younger than every other slot -- so they
// are never chosen.
//
// Three variants:
//   CLUSTER (hs_swapin_cluster_kernel) a thread-block cluster of 2-16 CTAs
//           per request.  Rank 0 runs the resolve below; the other ranks
//           (cluster_helper) gather the page table themselves and load their
//           share of the candidate misses before rank 0's miss list exists,
//           then copy rows from rank 0's lists through distributed shared
//           memory.  Rank 0 ranks the candidates the same way, so every miss
//           is fetched ahead once or put on its copy list.  The CTAs hand off
//           through three phases of the hardware cluster barrier.  One
//           launch; more SMs per request than FUSED.
//   FUSED   the CTA then updates the tables and copies its own missing rows
//           from the mapped host pool into the buffer (zero-copy 128-bit
//           loads, U in flight per lane); the last CTA to finish advances the
//           step counter.  One launch per step.  Half of the warps load
//           their first row group into registers as soon as the miss list
//           exists, so the host link is busy while the victims are chosen
//           (unless one round of the copy loop takes every row).
//           (Staging rows in shared memory instead -- cp.async, or bulk
//           copies on mbarriers issued by a separate fetch warp -- was
//           measured no faster.)
//   !FUSED  the CTA writes the miss / victim lists to global memory for the
//           grid-wide copy kernel (hs_copy.cu), which advances the counter.
//
// hs_resolve_kernel runs one handle's B CTAs (B clusters for
// hs_swapin_cluster_kernel); hs_resolve_layers_kernel runs the FUSED per-CTA
// body for several independent handles (layers) in one grid, CTA x serving
// request x mod B of layer x / B.
#include <climits>

#include "hs_internal.h"

namespace {

constexpr int NT = HS_RESOLVE_THREADS;
constexpr int NW = NT / 32;
constexpr int EMAX = HS_MAX_TOPK / NT;   // top-k entries per thread
constexpr int NB = HS_AGE_BINS;          // age bins
constexpr int NSUB = HS_AGE_SUBHIST;     // age sub-histograms (NW / NSUB warps share one)
constexpr int BPT = NB / NT;             // bins per thread in the bin scan
constexpr unsigned FULL = 0xffffffffu;

static_assert(NW <= 32, "one warp scans the warp totals");
static_assert(EMAX * NT == HS_MAX_TOPK, "entries per thread");
static_assert(BPT * NT == NB, "bins per thread");

enum : int { C_NONE = 0, C_BAD = 1, C_TAIL = 2, C_HIT = 3, C_MISS = 4 };

// One SplitMix64 output for the state x (Steele, Lea and Flood, "Fast
// Splittable Pseudorandom Number Generators", OOPSLA 2014): the state
// advanced by the golden-ratio increment, two xor-shift-multiply rounds and a
// final xor-shift.
__device__ __forceinline__ unsigned long long splitmix64(unsigned long long x)
{
    unsigned long long z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// The key that orders slot s for eviction (smallest first).  LRU and FIFO:
// its stamp.  Random eviction: a slot hit this step (stamp == step) never
// goes (INT_MAX), an empty slot goes first (0), and any other slot gets 1 +
// the top 30 bits of SplitMix64 of seed ^ (step << 32 | request << 14 | s).
__device__ __forceinline__ int evict_key(const ResolveArgs& a, int s, int stamp, int slot_tok,
                                         int step, int b)
{
    if (!a.random) return stamp;
    if (stamp == step) return INT_MAX;
    if (slot_tok < 0) return 0;
    const unsigned long long x = ((unsigned long long)(unsigned)step << 32) |
                                 ((unsigned long long)(unsigned)b << 14) | (unsigned)s;
    return 1 + (int)(splitmix64(a.seed ^ x) >> 34);
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int n = __shfl_up_sync(FULL, v, d);
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
    if (warp == 0) {
        const int x = lane < NW ? s_w[lane] : 0;
        const int y = warp_incl_scan(x, lane);
        if (lane < NW) s_w[lane] = y;
    }
    __syncthreads();
    const int off = warp ? s_w[warp - 1] : 0;
    *total = s_w[NW - 1];
    __syncthreads();
    return off + incl - v;
}

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

// 16-byte asynchronous copy global -> shared (bypasses L1), and its fences.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc)
{
    const unsigned d = (unsigned)__cvta_generic_to_shared(smem_dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// One warp copies `nrows` rows: lane r < nrows holds row r's source and
// destination byte offsets.  Every lane streams 16-byte chunks, U loads in
// flight before the matching stores.
template <int U>
__device__ __forceinline__ void copy_row_group(const uint8_t* pool_b, uint8_t* buf_b, long long src,
                                               long long dst, int nrows, int cpr, int lane)
{
    const int nch = nrows * cpr;
    for (int c0 = 0; c0 < nch; c0 += 32 * U) {
        uint4 v[U];
        long long d[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int cc = c0 + u * 32 + lane;
            const int rr = cc < nch ? cc / cpr : 0;
            const long long s = __shfl_sync(FULL, src, rr);
            const int off = (cc - rr * cpr) << 4;
            d[u] = __shfl_sync(FULL, dst, rr) + off;
            if (cc < nch) v[u] = ld_host_v4(pool_b + s + off);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int cc = c0 + u * 32 + lane;
            if (cc < nch) st_v4(buf_b + d[u], v[u]);
        }
    }
}

// ---- thread-block clusters: one request's CTAs on several SMs -------------
// The copy-list length of the cluster's resolving CTA, read by the others
// through distributed shared memory (a file-scope variable has the same
// offset in every CTA of the kernel).
__shared__ int s_cluster_mc;  // misses on the copy list (not fetched ahead)

__device__ __forceinline__ unsigned cluster_rank()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_size()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ unsigned cluster_index()
{
    unsigned r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
// Hardware cluster barrier, split into its two halves.  Every thread of every
// CTA of the cluster arrives once per phase and waits before it arrives
// again; .release publishes the thread's earlier shared-memory writes to the
// CTAs that wait (.acquire) on the phase.  (The forms without .aligned: they
// do not need the warp to be converged where they are called.)
__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
// The shared-memory address of `p` in CTA `rank` of this cluster.
__device__ __forceinline__ unsigned cluster_map(const void* p, unsigned rank)
{
    const unsigned a = (unsigned)__cvta_generic_to_shared(p);
    unsigned r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
__device__ __forceinline__ int ld_cluster_s32(unsigned addr)
{
    int v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ int ld_cluster_u16(unsigned addr)
{
    unsigned short v;
    asm volatile("ld.shared::cluster.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
    return (int)v;
}

// A stamp clamped into [0, step - 1], the range the victim search assumes.
__device__ __forceinline__ int clamp_stamp(int k, int step)
{
    return k < 0 ? 0 : (k >= step ? step - 1 : k);
}

// One thread's top-k entries [j0, j0 + E) (entries at or past K read as -1),
// as 16-byte (else 8-byte) loads where the run is whole and aligned: the row
// may be mapped host memory, where each 4-byte load of a warp would move its
// own sectors across the host link.
__device__ __forceinline__ void load_row(int (&tk)[EMAX], const int32_t* g_row, int j0, int E,
                                         int K)
{
    const int32_t* src = g_row + j0;
    if (j0 + E <= K && (E & 3) == 0 && ((uintptr_t)src & 15u) == 0) {
#pragma unroll
        for (int e = 0; e < EMAX; e += 4) {
            int4 v = make_int4(-1, -1, -1, -1);
            if (e < E) v = *reinterpret_cast<const int4*>(src + e);
            tk[e] = v.x;
            tk[e + 1] = v.y;
            tk[e + 2] = v.z;
            tk[e + 3] = v.w;
        }
    } else if (j0 + E <= K && (E & 1) == 0 && ((uintptr_t)src & 7u) == 0) {
#pragma unroll
        for (int e = 0; e < EMAX; e += 2) {
            int2 v = make_int2(-1, -1);
            if (e < E) v = *reinterpret_cast<const int2*>(src + e);
            tk[e] = v.x;
            tk[e + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int e = 0; e < EMAX; ++e) tk[e] = (e < E && j0 + e < K) ? src[e] : -1;
    }
}

// One thread's out_slot entries [j0, j0 + E) that lie below K, written with
// 16-byte (else 8-byte) stores where the run is whole and aligned.  A warp's
// stores then cover whole lines: out_slot may be mapped host memory, where
// scattered 4-byte writes each take a transaction on the host link.
__device__ __forceinline__ void write_out(int32_t* g_out, const int (&o)[EMAX], int j0, int E,
                                          int K)
{
    int32_t* dst = g_out + j0;
    const int n = j0 + E <= K ? E : (K > j0 ? K - j0 : 0);
    if (n == E && (E & 3) == 0 && ((uintptr_t)dst & 15u) == 0) {
#pragma unroll
        for (int e = 0; e < EMAX; e += 4)
            if (e < E) *reinterpret_cast<int4*>(dst + e) = make_int4(o[e], o[e + 1], o[e + 2], o[e + 3]);
    } else if (n == E && (E & 1) == 0 && ((uintptr_t)dst & 7u) == 0) {
#pragma unroll
        for (int e = 0; e < EMAX; e += 2)
            if (e < E) *reinterpret_cast<int2*>(dst + e) = make_int2(o[e], o[e + 1]);
    } else {
#pragma unroll
        for (int e = 0; e < EMAX; ++e)
            if (e < n) dst[e] = o[e];
    }
}

// One request's step: CTA `b` of the `nblocks` that serve one handle.
// CLUSTER: this CTA is rank 0 of a cluster of `ncl` CTAs serving request b;
// the others (cluster_helper) fetch rows from its miss and victim lists.
template <bool FUSED, int U, bool CLUSTER = false>
__device__ __forceinline__ void resolve_cta(const ResolveArgs& a, const int b,
                                            const unsigned nblocks, const int ncl = 1)
{
    extern __shared__ __align__(16) int smem[];
    __shared__ int s_w[32];
    __shared__ int s_cnt[3];  // hits, in-place, error bits
    __shared__ int s_sel[3];  // selected bin / digit, count below it, flag

    if (!FUSED) {
        // The copy grid may be scheduled as soon as every resolve CTA is
        // running; it waits for this grid's completion before reading.
        asm volatile("griddepcontrol.launch_dependents;");
    }

    const int K = a.K, S = a.S;
    const int hc = 1 << a.hash_bits;
    const int region_a = hs_resolve_region_a_ints(a.hash_bits, K);
    int* s_hkey = smem;                       // [hc]   phase 1
    int* s_hj = smem + hc;                    // [hc]   phase 1
    int* s_hist = smem;                       // [NSUB][NB], phase 2 (reuses the hash)
    int* s_out = smem + NSUB * NB;            // [E][NT] after the miss list (reuses the hash)
    int* s_stamp = smem + region_a;           // [S]
    int* s_slot_tok = s_stamp + S;            // [S]
    int* s_mtok = s_slot_tok + S;             // [K]
    uint16_t* s_mj = reinterpret_cast<uint16_t*>(s_mtok + K);  // [K]
    uint16_t* s_vic = s_mj + K;                                 // [K]
    // The two uint16 arrays hold 2K entries (4K bytes), so the word array after
    // them is 4-byte aligned for every K.
    unsigned* s_hitbits = reinterpret_cast<unsigned*>(s_vic + K);  // [ceil(S/32)]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // State the caller owns (the allocation-free entry point) may be
    // inconsistent; each repair below latches HS_E_STATE.  The step counter
    // must leave room for the claims step + K - j to stay below 2^31.
    int bad_state = 0;
    int step0 = a.st->step;
    if (step0 < 0 || step0 >= HS_MAX_STEP) {
        step0 = step0 < 0 ? 0 : HS_MAX_STEP - 1;
        bad_state = HS_E_STATE;
    }
    const int step = step0 + 1;
    const int len = a.len[b];
    // First tail position: fixed at C - T, or sliding with the request's length.
    const int cold = a.sliding ? (len - a.T > 0 ? len - a.T : 0) : a.cold;
    const int32_t* g_topk = a.topk + (size_t)b * K;
    int32_t* g_out = a.out + (size_t)b * K;
    int32_t* g_stamp = a.stamp + (size_t)b * S;
    int32_t* g_slot_tok = a.slot_tok + (size_t)b * S;
    int32_t* g_tok_slot = a.tok_slot + (size_t)b * a.C;

    // ---- loads: top-k row (registers), stamps and slot -> token (shared) --
    // Thread tid owns the contiguous entries [tid*E, tid*E + E) so that a
    // block scan of per-thread miss counts yields row order.
    const int E = (K + NT - 1) / NT;
    const int j0 = tid * E;
    int tk[EMAX];
    load_row(tk, g_topk, j0, E, K);
    // The two S-entry rows go to shared memory with asynchronous 16-byte
    // copies when they are 16-byte aligned, so all of them are in flight at
    // once; otherwise with plain loads.
    const bool vec_rows = (S & 3) == 0 &&
        (((uintptr_t)g_stamp | (uintptr_t)g_slot_tok | (uintptr_t)s_stamp) & 15u) == 0;
    if (vec_rows) {
        for (int i = tid; i < (S >> 2); i += NT) {
            cp_async16(s_stamp + 4 * i, g_stamp + 4 * i);
            cp_async16(s_slot_tok + 4 * i, g_slot_tok + 4 * i);
        }
        cp_async_commit();
    } else {
        for (int i = tid; i < S; i += NT) {
            s_stamp[i] = g_stamp[i];
            s_slot_tok[i] = g_slot_tok[i];
        }
    }
    for (int i = tid; i < hc; i += NT) {
        s_hkey[i] = -1;
        s_hj[i] = INT_MAX;
    }
    if (a.fifo)
        for (int i = tid; i < ((S + 31) >> 5); i += NT) s_hitbits[i] = 0u;
    // ---- (1) classify, gather the page table, find repeats ----------------
    // The page-table gathers are issued before waiting for the stamp rows, so
    // their DRAM latency overlaps the wait.
    int cl[EMAX], hs[EMAX], sl[EMAX];
    // out_slot values of the thread's entries, written to memory once per
    // step (write_out below).  A miss holds -(2 + its miss index) until its
    // victim is known; under aliasing a repeated miss holds
    // -(2 + K + row of its first occurrence).
    int ov[EMAX];
    int err = 0;
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        const int t = tk[e];
        cl[e] = C_NONE;
        sl[e] = -1;
        hs[e] = 0;
        if (e < E && j0 + e < K && t != -1) {
            if (t < -1 || t >= len || t >= a.C) {
                cl[e] = C_BAD;
                err |= HS_E_RANGE;
            } else {
                cl[e] = C_MISS;  // valid; refined below
                if (t < cold) sl[e] = g_tok_slot[t];
            }
        }
    }
    if (vec_rows) cp_async_wait_all();
    // Every stamp must lie in [0, step - 1] for the victim search to place
    // exactly m victims: each thread clamps the stamps it loaded itself (as
    // 16-byte words when it copied them so, which keeps the reads free of
    // bank conflicts).
    if (vec_rows) {
        int4* s4 = reinterpret_cast<int4*>(s_stamp);
        for (int i = tid; i < (S >> 2); i += NT) {
            const int4 k = s4[i];
            if ((unsigned)k.x >= (unsigned)step || (unsigned)k.y >= (unsigned)step ||
                (unsigned)k.z >= (unsigned)step || (unsigned)k.w >= (unsigned)step) {
                s4[i] = make_int4(clamp_stamp(k.x, step), clamp_stamp(k.y, step),
                                  clamp_stamp(k.z, step), clamp_stamp(k.w, step));
                bad_state = HS_E_STATE;
            }
        }
    } else {
        for (int i = tid; i < S; i += NT) {
            const int k = s_stamp[i];
            if ((unsigned)k >= (unsigned)step) {
                s_stamp[i] = clamp_stamp(k, step);
                bad_state = HS_E_STATE;
            }
        }
    }
    err |= bad_state;
    if (tid < 3) s_cnt[tid] = 0;
    __syncthreads();

    // Cluster: the other CTAs fetch rows ahead of the miss list.  They rank the
    // candidate misses of each warp's entries -- valid cold tokens outside the
    // buffer, repeats included -- in row order, and the first (ncl - 1) * G of
    // each warp are theirs.  This CTA ranks them the same way, so each miss
    // either was fetched ahead or goes on the copy list, never both.
    unsigned pfmask = 0;
    if (CLUSTER) {
        const int PF = (a.rows_per_group * (a.R >> 4) <= 32 * U) ? (ncl - 1) * a.rows_per_group : 0;
        unsigned cmask = 0;
        int c = 0;
#pragma unroll
        for (int e = 0; e < EMAX; ++e)
            if (cl[e] == C_MISS && tk[e] < cold && (sl[e] < 0 || sl[e] >= S)) {
                cmask |= 1u << e;
                ++c;
            }
        int q = warp_incl_scan(c, lane) - c;
#pragma unroll
        for (int e = 0; e < EMAX; ++e)
            if ((cmask >> e) & 1u) {
                if (q < PF) pfmask |= 1u << e;
                ++q;
            }
    }

    // Repeated indices: the first occurrence in row order wins.  A resident
    // token claims its slot by raising the slot's stamp word to
    // step + K - j (the largest value belongs to the smallest j); every other
    // valid token (a miss or a tail token) goes through the hash.
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        // A page-table entry outside [-1, S) is corrupt state: resolve as a miss.
        if (sl[e] < -1 || sl[e] >= S) {
            sl[e] = -1;
            err |= HS_E_STATE;
        }
        if (cl[e] == C_MISS && sl[e] >= 0) atomicMax(&s_stamp[sl[e]], step + (K - (j0 + e)));
    }
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        if (cl[e] == C_MISS && sl[e] < 0) {
            const int t = tk[e];
            unsigned h = ((unsigned)t * 0x9E3779B1u) >> (32 - a.hash_bits);
            for (;;) {
                const int k = atomicCAS(&s_hkey[h], -1, t);
                if (k == -1 || k == t) break;
                h = (h + 1) & (unsigned)(hc - 1);
            }
            atomicMin(&s_hj[h], j0 + e);
            hs[e] = (int)h;
        }
    }
    __syncthreads();
    int nh = 0, ni = 0, nm = 0, nmc = 0;
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        const int j = j0 + e;
        if (cl[e] == C_MISS) {
            if (sl[e] >= 0) {
                // A repeat reads either the winner's claim or the normalised
                // stamp; both differ from its own claim step + K - j.
                if (s_stamp[sl[e]] != step + (K - j)) {
                    cl[e] = C_BAD;
                    if (a.alias) {
                        ov[e] = sl[e];  // the same resident slot as its first occurrence
                    } else {
                        err |= HS_E_DUP;
                        ov[e] = -1;
                    }
                } else {
                    cl[e] = C_HIT;
                    // LRU: a hit refreshes its entry.  FIFO: the slot only
                    // looks new while victims are chosen; its fill stamp is
                    // kept at write-back.
                    s_stamp[sl[e]] = step;
                    if (a.fifo) atomicOr(&s_hitbits[sl[e] >> 5], 1u << (sl[e] & 31));
                    ov[e] = sl[e];
                    ++nh;
                }
            } else if (s_hj[hs[e]] != j) {
                cl[e] = C_BAD;
                if (!a.alias) {
                    err |= HS_E_DUP;
                    ov[e] = -1;
                } else if (tk[e] >= cold) {
                    ov[e] = S + tk[e] % a.T;
                } else {
                    // A repeated miss takes its first occurrence's slot.
                    ov[e] = -(2 + K + s_hj[hs[e]]);
                }
            } else if (tk[e] >= cold) {
                cl[e] = C_TAIL;
                ov[e] = S + tk[e] % a.T;
                ++ni;
            } else {
                ++nm;
                if (!((pfmask >> e) & 1u)) ++nmc;
            }
        } else {
            ov[e] = -1;
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

    int m = 0, mc = 0, pos, pos2 = 0;
    if (CLUSTER) {
        // Both scans at once: misses, and misses not fetched ahead (counts
        // below 2^16).
        int tot;
        const int packed = block_excl_scan((nm << 16) | nmc, s_w, &tot);
        pos = packed >> 16;
        pos2 = packed & 0xffff;
        m = tot >> 16;
        mc = tot & 0xffff;
    } else {
        pos = block_excl_scan(nm, s_w, &m);
    }
    // The copy list (cluster only): the indices of the misses not fetched
    // ahead, in the hash's region, which the scan's barriers have retired.
    uint16_t* s_clist = reinterpret_cast<uint16_t*>(s_out + E * NT);
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        if (cl[e] == C_MISS) {
            s_mtok[pos] = tk[e];
            s_mj[pos] = (uint16_t)(j0 + e);
            ov[e] = -(2 + pos);
            if (CLUSTER && !((pfmask >> e) & 1u)) s_clist[pos2++] = (uint16_t)pos;
            ++pos;
        }
    }
    if (CLUSTER) {
        // Phase 1 of the cluster barrier: the miss list and the copy list are
        // complete.
        if (tid == 0) s_cluster_mc = mc;
        cluster_arrive_release();
    }

    if (m == 0) {
        write_out(g_out, ov, j0, E, K);
    } else {
        // The hash is no longer read (the scan above passed a barrier), so
        // its region keeps the thread's out values through phase 2, entry e
        // at e * NT + tid: a warp's accesses hit 32 different banks.
#pragma unroll
        for (int e = 0; e < EMAX; ++e)
            if (e < E) s_out[e * NT + tid] = ov[e];

        // ---- (2) LRU victims ----------------------------------------------
        // Age histogram: bin NB-1-min(age, NB-1), so older slots sit in lower
        // bins and the shared bin 0 holds every age >= NB-1.
        for (int i = tid; i < NSUB * NB; i += NT) s_hist[i] = 0;
        __syncthreads();
        // Fused: the miss list is complete, the victims are not chosen yet.
        // Half of the warps already load their first group of rows into
        // registers, so the host link is busy during the victim search; each
        // group is stored once its slots are known.  A warp issuing host loads
        // waits while the SM's memory path is full, so the other half runs the
        // victim search unhindered (measured: all 16 warps 1.8 % faster per
        // step than none; 8 warps a further 1.8 % faster at 32 requests and no
        // slower at 64 or 256).  When one round of the copy loop takes every
        // row (m <= NW * G0) the early loads only delay the victim search.
        uint4 pre[U];
        const int G0 = a.rows_per_group;
        const int cpr0 = a.R >> 4;
        const bool prefetch = FUSED && !CLUSTER && G0 * cpr0 <= 32 * U && warp < NW / 2 &&
                              m > NW * G0;
        if (prefetch && warp * G0 < m) {
            const uint8_t* pool_b0 = a.pool + (size_t)b * (size_t)a.H * a.R;
            const int r0 = warp * G0;
            long long src = 0;
            if (lane < G0 && r0 + lane < m) src = (long long)s_mtok[r0 + lane] * a.R;
            const int nch = ((m - r0) < G0 ? (m - r0) : G0) * cpr0;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int cc = u * 32 + lane;
                const int rr = cc < nch ? cc / cpr0 : 0;
                const long long sg = __shfl_sync(FULL, src, rr);
                if (cc < nch) pre[u] = ld_host_v4(pool_b0 + sg + ((cc - rr * cpr0) << 4));
            }
        }
        const int s_pad = (S + NT - 1) / NT * NT;
        int* my_hist = s_hist + (warp % NSUB) * NB;
        // Random eviction has no age order: every slot counts as "oldest"
        // (bin 0), so the radix select below runs over the keys.
        for (int i = tid; i < s_pad; i += NT) {
            int bin = NB;
            if (i < S) {
                const int age = step - s_stamp[i];
                bin = a.random ? 0 : NB - 1 - (age < NB - 1 ? age : NB - 1);
            }
            const unsigned peers = __match_any_sync(FULL, bin);
            if (bin < NB && lane == __ffs(peers) - 1) atomicAdd(&my_hist[bin], __popc(peers));
        }
        __syncthreads();
        int c[BPT];
        int csum = 0;
#pragma unroll
        for (int q = 0; q < BPT; ++q) {
            const int bin = tid * BPT + q;
            int x = 0;
#pragma unroll
            for (int h = 0; h < NSUB; ++h) x += s_hist[h * NB + bin];
            c[q] = x;
            csum += x;
        }
        int tot_bins;
        int below = block_excl_scan(csum, s_w, &tot_bins);
#pragma unroll
        for (int q = 0; q < BPT; ++q) {
            if (c[q] > 0 && below < m && m <= below + c[q]) {
                s_sel[0] = tid * BPT + q;
                s_sel[1] = below;
            }
            below += c[q];
        }
        __syncthreads();
        const int bsel = s_sel[0];
        int tau, need_eq;
        if (bsel > 0) {
            tau = step - (NB - 1 - bsel);  // one exact stamp per bin
            need_eq = m - s_sel[1];
        } else {
            // The m-th oldest slot is among the ages >= NB-1: radix select
            // over the stamps <= lim, most significant digit first.
            // (random eviction: every key below INT_MAX, which marks a hit)
            const int lim = a.random ? INT_MAX - 1 : step - (NB - 1);
            const int nbits = 32 - __clz(lim > 0 ? lim : 1);
            unsigned prefix = 0, pmask = 0;
            int remaining = m;
            for (int d = (nbits - 1) >> 3; d >= 0; --d) {
                const int shift = 8 * d;
                for (int i = tid; i < NSUB * NB; i += NT) s_hist[i] = 0;
                __syncthreads();
                for (int i = tid; i < s_pad; i += NT) {
                    int dig = 256;
                    if (i < S) {
                        const int k = evict_key(a, i, s_stamp[i], s_slot_tok[i], step, b);
                        if (k <= lim && ((unsigned)k & pmask) == prefix)
                            dig = (int)(((unsigned)k >> shift) & 255u);
                    }
                    const unsigned peers = __match_any_sync(FULL, dig);
                    if (dig < 256 && lane == __ffs(peers) - 1)
                        atomicAdd(&my_hist[dig], __popc(peers));
                }
                __syncthreads();
                int cd = 0, incl = 0;
                if (tid < 256) {
#pragma unroll
                    for (int h = 0; h < NSUB; ++h) cd += s_hist[h * NB + tid];
                    incl = warp_incl_scan(cd, lane);
                    if (lane == 31) s_w[warp] = incl;
                }
                __syncthreads();
                if (tid < 256) {
                    int off = 0;
                    for (int w = 0; w < warp; ++w) off += s_w[w];
                    const int excl = off + incl - cd;
                    if (cd > 0 && excl < remaining && remaining <= excl + cd) {
                        s_sel[0] = tid;
                        s_sel[1] = excl;
                    }
                }
                __syncthreads();
                prefix |= (unsigned)s_sel[0] << shift;
                pmask |= 255u << shift;
                remaining -= s_sel[1];
                __syncthreads();
            }
            tau = (int)prefix;
            need_eq = remaining;
        }

        // Victims in ascending slot order: thread tid owns slots [tid*Q, tid*Q + Q).
        const int Q = (S + NT - 1) / NT;
        const int q0 = tid * Q;
        int nl = 0, ne = 0;
        const bool vec_q = !a.random && (Q & 3) == 0 && q0 + Q <= S &&  // 16-byte aligned, all in range
                           ((uintptr_t)s_stamp & 15u) == 0;
        if (vec_q) {
            for (int q = 0; q < Q; q += 4) {
                const int4 k4 = *reinterpret_cast<const int4*>(s_stamp + q0 + q);
                nl += (k4.x < tau) + (k4.y < tau) + (k4.z < tau) + (k4.w < tau);
                ne += (k4.x == tau) + (k4.y == tau) + (k4.z == tau) + (k4.w == tau);
            }
        } else {
            for (int q = 0; q < Q; ++q) {
                const int s = q0 + q;
                if (s < S) {
                    const int k = evict_key(a, s, s_stamp[s], s_slot_tok[s], step, b);
                    nl += k < tau;
                    ne += k == tau;
                }
            }
        }
        int tot;
        const int packed = block_excl_scan((nl << 16) | ne, s_w, &tot);
        int lb = packed >> 16, eb = packed & 0xffff;
        // Exactly m slots qualify; the bounds only keep a corrupted stamp from
        // writing past the list.
        auto place = [&](int s, int k) {
            if (k < tau) {
                const int p = lb + (eb < need_eq ? eb : need_eq);
                if (p < m) s_vic[p] = (uint16_t)s;
                ++lb;
            } else if (k == tau) {
                if (eb < need_eq && lb + eb < m) s_vic[lb + eb] = (uint16_t)s;
                ++eb;
            }
        };
        if (nl | ne) {
            if (vec_q) {
                for (int q = 0; q < Q; q += 4) {
                    const int4 k4 = *reinterpret_cast<const int4*>(s_stamp + q0 + q);
                    place(q0 + q, k4.x);
                    place(q0 + q + 1, k4.y);
                    place(q0 + q + 2, k4.z);
                    place(q0 + q + 3, k4.w);
                }
            } else {
                for (int q = 0; q < Q; ++q) {
                    const int s = q0 + q;
                    if (s < S) place(s, evict_key(a, s, s_stamp[s], s_slot_tok[s], step, b));
                }
            }
        }
        __syncthreads();

        // The i-th miss (row order) is paired with the i-th victim, so every
        // out value is known now: one write of the thread's entries.
        {
            int fo[EMAX];
#pragma unroll
            for (int e = 0; e < EMAX; ++e) {
                int o = e < E ? s_out[e * NT + tid] : -1;
                if (o <= -2) {
                    int i = -o - 2;
                    if (i >= K) {
                        // first occurrence at row i - K: find its miss index
                        // (the miss rows are ascending)
                        const int jf = i - K;
                        int lo = 0, hi = m;
                        while (lo < hi) {
                            const int mid = (lo + hi) >> 1;
                            if ((int)s_mj[mid] < jf) lo = mid + 1;
                            else hi = mid;
                        }
                        i = lo;
                    }
                    o = i < m ? (int)s_vic[i] : -1;
                }
                fo[e] = o;
                // Cluster: the final slots replace the miss indices, for the
                // CTAs whose rows were fetched ahead (each thread rewrites only
                // its own entries).
                if (CLUSTER && e < E) s_out[e * NT + tid] = o;
            }
            write_out(g_out, fo, j0, E, K);
        }

        if (!FUSED) {
            // ---- (3) pair the i-th miss (row order) with the i-th victim ----
            int32_t* g_mtok = a.miss_tok + (size_t)b * a.list_stride;
            int32_t* g_mslot = a.miss_slot + (size_t)b * a.list_stride;
            for (int i = tid; i < m; i += NT) {
                const int t = s_mtok[i];
                const int v = s_vic[i];
                const int old = s_slot_tok[v];
                // the evicted token leaves the table (an entry outside
                // [-1, C) is corrupt state and is not written through)
                if (old >= 0 && old < a.C) g_tok_slot[old] = -1;
                else if (old != -1) atomicOr(&s_cnt[2], HS_E_STATE);
                g_slot_tok[v] = t;
                g_tok_slot[t] = v;
                s_stamp[v] = step;
                g_mtok[i] = t;
                g_mslot[i] = v;
            }
        } else if (!CLUSTER) {
            // ---- (3) table update + host fetch, G rows per warp at a time ----
            const int G = a.rows_per_group;
            const int cpr = a.R >> 4;  // 16-byte chunks per row
            const uint8_t* pool_b = a.pool + (size_t)b * (size_t)a.H * a.R;
            uint8_t* buf_b = a.buf + (size_t)b * (size_t)(S + a.T) * a.R;
            for (int r0 = warp * G; r0 < m; r0 += NW * G) {
                long long src = 0, dst = 0;
                const int i = r0 + lane;
                if (lane < G && i < m) {
                    const int t = s_mtok[i];
                    const int v = s_vic[i];
                    const int old = s_slot_tok[v];
                    if (old >= 0 && old < a.C) g_tok_slot[old] = -1;
                    else if (old != -1) atomicOr(&s_cnt[2], HS_E_STATE);
                    g_slot_tok[v] = t;
                    g_tok_slot[t] = v;
                    s_stamp[v] = step;
                    src = (long long)t * a.R;
                    dst = (long long)v * a.R;
                }
                const int nrows = (m - r0) < G ? (m - r0) : G;
                if (prefetch && r0 == warp * G) {
                    // the group loaded before the victim search
                    const int nch = nrows * cpr;
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int cc = u * 32 + lane;
                        const int rr = cc < nch ? cc / cpr : 0;
                        const long long dg = __shfl_sync(FULL, dst, rr) + ((cc - rr * cpr) << 4);
                        if (cc < nch) st_v4(buf_b + dg, pre[u]);
                    }
                } else {
                    copy_row_group<U>(pool_b, buf_b, src, dst, nrows, cpr, lane);
                }
            }
        }
    }
    if (CLUSTER) {
        cluster_wait();            // phase 1 done: the other CTAs have read the page table
        cluster_arrive_release();  // phase 2: the victims are placed
        if (m > 0) {
            // ---- (3) table update for every miss, then this CTA's rows ----
            for (int i = tid; i < m; i += NT) {
                const int t = s_mtok[i];
                const int v = s_vic[i];
                const int old = s_slot_tok[v];
                if (old >= 0 && old < a.C) g_tok_slot[old] = -1;
                else if (old != -1) atomicOr(&s_cnt[2], HS_E_STATE);
                g_slot_tok[v] = t;
                g_tok_slot[t] = v;
                s_stamp[v] = step;
            }
            // Row group g of the copy list (entries [g*G, g*G + G)) belongs
            // to cluster warp g mod (ncl * NW); this CTA's warps come after
            // the other CTAs'.
            const int G = a.rows_per_group;
            const int cpr = a.R >> 4;
            const uint8_t* pool_b = a.pool + (size_t)b * (size_t)a.H * a.R;
            uint8_t* buf_b = a.buf + (size_t)b * (size_t)(S + a.T) * a.R;
            const int ncw = ncl * NW;
            for (int g = (ncl - 1) * NW + warp; g * G < mc; g += ncw) {
                const int r0 = g * G;
                long long src = 0, dst = 0;
                if (lane < G && r0 + lane < mc) {
                    const int i = s_clist[r0 + lane];
                    src = (long long)s_mtok[i] * a.R;
                    dst = (long long)s_vic[i] * a.R;
                }
                copy_row_group<U>(pool_b, buf_b, src, dst, (mc - r0) < G ? (mc - r0) : G, cpr, lane);
            }
        }
        cluster_wait();            // phase 2 done
    }
    __syncthreads();
    if (a.fifo) {
        for (int i = tid; i < S; i += NT)
            if (!((s_hitbits[i >> 5] >> (i & 31)) & 1u)) g_stamp[i] = s_stamp[i];
    } else {
        for (int i = tid; i < S; i += NT) g_stamp[i] = s_stamp[i];
    }
    if (tid == 0) {
        a.miss_cnt[b] = m;
        if (s_cnt[0]) atomicAdd(&a.st->hits, (unsigned long long)s_cnt[0]);
        if (s_cnt[1]) atomicAdd(&a.st->inplace, (unsigned long long)s_cnt[1]);
        if (m) atomicAdd(&a.st->misses, (unsigned long long)m);
        if (s_cnt[2]) atomicOr(&a.st->err, s_cnt[2]);
        if (FUSED) {
            // Every CTA read the step counter before this point; the last one
            // to arrive advances it for the next call and re-arms the count.
            __threadfence();
            const unsigned prev = atomicAdd(a.done, 1u);
            if (prev == nblocks - 1) {
                *a.done = 0u;
                a.st->step = step;
            }
        }
    }
    if (CLUSTER) {
        // Phase 3: this CTA's lists stay in shared memory until the other
        // CTAs of the cluster have read them.
        cluster_arrive_release();
        cluster_wait();
    }
}

// A CTA of rank >= 1 in a request's cluster.  Before rank 0 has its miss
// list, it loads the top-k row and gathers the page table itself, ranks each
// warp's candidate misses as rank 0 does (valid cold tokens outside the
// buffer, in row order), and its warp w loads candidates
// [(rank - 1) * G, rank * G) of warp w's entries into registers.  Once rank
// 0 has placed the victims, each of those rows that is a miss goes to its
// victim slot (rank 0's out values in shared memory give its miss index), and
// the CTA copies its share of the rows on rank 0's copy list (group g to
// cluster warp g mod (ncl * NW), ranks 1.. first).  It writes no table.  The
// barrier phases match resolve_cta<CLUSTER>: 1 page table read / miss lists
// built, 2 victims placed, 3 lists read.
template <int U>
__device__ __forceinline__ void cluster_helper(const ResolveArgs& a, const int b, const int rank,
                                               const int ncl)
{
    extern __shared__ __align__(16) int smem[];
    const int K = a.K, S = a.S;
    const int E = (K + NT - 1) / NT;
    // rank 0's layout (the same dynamic shared memory size in every CTA)
    int* s_out = smem + NSUB * NB;
    uint16_t* s_clist = reinterpret_cast<uint16_t*>(s_out + E * NT);
    int* s_mtok = smem + hs_resolve_region_a_ints(a.hash_bits, K) + 2 * S;
    uint16_t* s_vic = reinterpret_cast<uint16_t*>(s_mtok + K) + K;
    const unsigned r_out = cluster_map(s_out, 0);
    const unsigned r_clist = cluster_map(s_clist, 0);
    const unsigned r_mtok = cluster_map(s_mtok, 0);
    const unsigned r_vic = cluster_map(s_vic, 0);
    const unsigned r_mc = cluster_map(&s_cluster_mc, 0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = a.rows_per_group;
    const int cpr = a.R >> 4;
    const int ncw = ncl * NW;
    const uint8_t* pool_b = a.pool + (size_t)b * (size_t)a.H * a.R;
    uint8_t* buf_b = a.buf + (size_t)b * (size_t)(S + a.T) * a.R;
    // This CTA's own shared memory: the rows its warps fetch ahead, [NW][G]
    // tokens and [NW][G] row positions.
    int* s_pf_tok = smem;
    int* s_pf_j = smem + NW * G;

    // ---- fetch ahead: this CTA's candidates, ranked as rank 0 ranks them ----
    const int len = a.len[b];
    const int cold = a.sliding ? (len - a.T > 0 ? len - a.T : 0) : a.cold;
    const int32_t* g_topk = a.topk + (size_t)b * K;
    const int32_t* g_tok_slot = a.tok_slot + (size_t)b * a.C;
    const int j0 = tid * E;
    int tk[EMAX], sl[EMAX];
    load_row(tk, g_topk, j0, E, K);
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        const int t = tk[e];
        sl[e] = -1;
        if (t >= 0 && t < len && t < a.C && t < cold) sl[e] = g_tok_slot[t];
    }
    const bool fits = G * cpr <= 32 * U;  // a row group fits the registers
    const int lo = (rank - 1) * G;
    unsigned cmask = 0;
    int c = 0;
#pragma unroll
    for (int e = 0; e < EMAX; ++e) {
        const int t = tk[e];
        if (t >= 0 && t < len && t < a.C && t < cold && (sl[e] < 0 || sl[e] >= S)) {
            cmask |= 1u << e;
            ++c;
        }
    }
    const int incl = warp_incl_scan(c, lane);
    int q = incl - c;
#pragma unroll
    for (int e = 0; e < EMAX; ++e)
        if ((cmask >> e) & 1u) {
            if (fits && q >= lo && q < lo + G) {
                s_pf_tok[warp * G + (q - lo)] = tk[e];
                s_pf_j[warp * G + (q - lo)] = j0 + e;
            }
            ++q;
        }
    const int wtot = __shfl_sync(FULL, incl, 31);
    const int np = fits ? (wtot - lo < 0 ? 0 : (wtot - lo > G ? G : wtot - lo)) : 0;
    // Phase 1: this CTA's page-table reads are done (their values are in
    // use), so rank 0 may update the tables; the loads below may then wait
    // for room in this SM's memory path without holding rank 0 up.
    cluster_arrive_release();
    __syncwarp();
    uint4 pre[U];
    int jr = 0;
    const int nch = np * cpr;
    if (np > 0) {
        long long src = 0;
        if (lane < np) {
            src = (long long)s_pf_tok[warp * G + lane] * a.R;
            jr = s_pf_j[warp * G + lane];
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int cc = u * 32 + lane;
            const int rr = cc < nch ? cc / cpr : 0;
            const long long sg = __shfl_sync(FULL, src, rr);
            if (cc < nch) pre[u] = ld_host_v4(pool_b + sg + ((cc - rr * cpr) << 4));
        }
    }
    cluster_wait();            // rank 0's miss and copy lists are complete
    cluster_arrive_relaxed();  // phase 2
    cluster_wait();            // rank 0's victims are placed, its final slots in shared memory
    const int mc = ld_cluster_s32(r_mc);
    if (np > 0) {
        // Each row fetched ahead goes to its entry's final slot: a victim for
        // a miss, its first occurrence's slot for a repeat that aliases it;
        // -1 (a repeat refused as an error) drops it.
        long long dst = -1;
        if (lane < np) {
            const int o = ld_cluster_s32(r_out + 4u * (unsigned)((jr % E) * NT + jr / E));
            if (o >= 0 && o < S) dst = (long long)o * a.R;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int cc = u * 32 + lane;
            const int rr = cc < nch ? cc / cpr : 0;
            const long long dg = __shfl_sync(FULL, dst, rr);
            if (cc < nch && dg >= 0) st_v4(buf_b + dg + ((cc - rr * cpr) << 4), pre[u]);
        }
    }
    // This CTA's share of the copy list.  The next group's entries are read
    // from rank 0 while the current group's rows are copied.
    int g = (rank - 1) * NW + warp;
    int inext = (lane < G && g * G + lane < mc) ? ld_cluster_u16(r_clist + 2u * (unsigned)(g * G + lane)) : -1;
    for (; g * G < mc; g += ncw) {
        const int r0 = g * G;
        long long src = 0, dst = 0;
        if (inext >= 0) {
            src = (long long)ld_cluster_s32(r_mtok + 4u * (unsigned)inext) * a.R;
            dst = (long long)ld_cluster_u16(r_vic + 2u * (unsigned)inext) * a.R;
        }
        const int gn = g + ncw;
        inext = (lane < G && gn * G + lane < mc) ? ld_cluster_u16(r_clist + 2u * (unsigned)(gn * G + lane)) : -1;
        copy_row_group<U>(pool_b, buf_b, src, dst, (mc - r0) < G ? (mc - r0) : G, cpr, lane);
    }
    cluster_arrive_release();  // phase 3: done with rank 0's lists
    cluster_wait();
}

template <bool FUSED, int U>
__global__ void __launch_bounds__(NT, 1) hs_resolve_kernel(ResolveArgs a)
{
    resolve_cta<FUSED, U>(a, blockIdx.x, gridDim.x);
}

// One cluster of ncl CTAs per request (cluster x serves request x): rank 0
// resolves and copies a share of the rows, the others fetch the rest.
template <int U>
__global__ void __launch_bounds__(NT, 1) hs_swapin_cluster_kernel(ResolveArgs a)
{
    const int rank = (int)cluster_rank();
    const int ncl = (int)cluster_size();
    const int b = (int)cluster_index();
    if (rank == 0) resolve_cta<true, U, true>(a, b, gridDim.x / (unsigned)ncl, ncl);
    else cluster_helper<U>(a, b, rank, ncl);
}

// Independent layers in one grid: CTA x serves request x mod B of layer
// x / B.  The layers' CTAs then share the SMs, so while some resolve
// others fetch rows, and one launch covers the whole step.
template <int U>
__global__ void __launch_bounds__(NT, 1) hs_resolve_layers_kernel(const __grid_constant__ LayerArgs p)
{
    const int layer = blockIdx.x / p.B;
    resolve_cta<true, U>(p.l[layer], blockIdx.x - layer * p.B, (unsigned)p.B);
}

}  // namespace

size_t hs_resolve_smem_bytes(int K, int S)
{
    return hs_resolve_base_bytes(K, S, hs_hash_bits(K));
}

cudaError_t hs_prepare_resolve()
{
    const int most = (int)hs_resolve_smem_bytes(HS_MAX_TOPK, HS_MAX_SLOTS);
    cudaError_t e = cudaFuncSetAttribute(hs_resolve_kernel<false, 9>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(hs_resolve_kernel<true, 9>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(hs_resolve_kernel<true, 8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(hs_resolve_layers_kernel<9>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(hs_resolve_layers_kernel<8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(hs_swapin_cluster_kernel<9>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(hs_swapin_cluster_kernel<8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(hs_swapin_cluster_kernel<9>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(hs_swapin_cluster_kernel<8>,
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    return e;
}

// The kernel places its stamp row right after region A and copies into it
// with 16-byte asynchronous copies: refuse a layout that would misalign it.
static bool layout_ok(const ResolveArgs& a)
{
    return a.hash_bits == hs_hash_bits(a.K) && (hs_resolve_region_a_ints(a.hash_bits, a.K) & 3) == 0;
}

cudaError_t hs_launch_resolve(const ResolveArgs& a, int B, cudaStream_t s)
{
    if (!layout_ok(a)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)B);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = hs_resolve_smem_bytes(a.K, a.S);
    cfg.stream = s;
    return cudaLaunchKernelEx(&cfg, hs_resolve_kernel<false, 9>, a);
}

cudaError_t hs_launch_swapin(const ResolveArgs& a, int B, int unroll, cudaStream_t s)
{
    if (!layout_ok(a)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)B);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = hs_resolve_smem_bytes(a.K, a.S);
    cfg.stream = s;
    if (unroll == 9) return cudaLaunchKernelEx(&cfg, hs_resolve_kernel<true, 9>, a);
    return cudaLaunchKernelEx(&cfg, hs_resolve_kernel<true, 8>, a);
}

cudaError_t hs_launch_swapin_layers(const LayerArgs& p, int L, int unroll, cudaStream_t s)
{
    for (int l = 0; l < L; ++l)
        if (!layout_ok(p.l[l])) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(L * p.B));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = hs_resolve_smem_bytes(p.l[0].K, p.l[0].S);
    cfg.stream = s;
    if (unroll == 9) return cudaLaunchKernelEx(&cfg, hs_resolve_layers_kernel<9>, p);
    return cudaLaunchKernelEx(&cfg, hs_resolve_layers_kernel<8>, p);
}

static cudaLaunchConfig_t cluster_config(const ResolveArgs& a, int B, int ncl, cudaStream_t s,
                                         cudaLaunchAttribute* attr)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(B * ncl));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = hs_resolve_smem_bytes(a.K, a.S);
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ncl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

cudaError_t hs_launch_swapin_cluster(const ResolveArgs& a, int B, int ncl, int unroll,
                                     cudaStream_t s)
{
    if (!layout_ok(a) || ncl < 2 || ncl > HS_MAX_CLUSTER) return cudaErrorInvalidValue;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = cluster_config(a, B, ncl, s, attr);
    if (unroll == 9) return cudaLaunchKernelEx(&cfg, hs_swapin_cluster_kernel<9>, a);
    return cudaLaunchKernelEx(&cfg, hs_swapin_cluster_kernel<8>, a);
}

int hs_cluster_max_active(int K, int S, int ncl, int unroll)
{
    ResolveArgs a = {};
    a.K = K;
    a.S = S;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = cluster_config(a, 1, ncl, nullptr, attr);
    int n = 0;
    const cudaError_t e = unroll == 9
        ? cudaOccupancyMaxActiveClusters(&n, hs_swapin_cluster_kernel<9>, &cfg)
        : cudaOccupancyMaxActiveClusters(&n, hs_swapin_cluster_kernel<8>, &cfg);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}
