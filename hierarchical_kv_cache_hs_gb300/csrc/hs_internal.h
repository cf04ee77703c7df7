// Private declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "hs.h"

// Device-resident per-handle control word: the step counter, latched error
// bits and cumulative counters.  The resolve kernel reads `step` (this call's
// step is step + 1), the copy kernel that follows it advances `step`.
struct HsDevState {
    int32_t step;
    int32_t err;
    unsigned long long hits;
    unsigned long long misses;
    unsigned long long inplace;
};

struct ResolveArgs {
    const int32_t* topk;   // [B][K]
    int32_t* out;          // [B][K]
    int32_t* tok_slot;     // [B][C]
    int32_t* slot_tok;     // [B][S]
    int32_t* stamp;        // [B][S]
    const int32_t* len;    // [B]
    int32_t* miss_tok;     // [B][list_stride]  miss tokens, top-k row order
    int32_t* miss_slot;    // [B][list_stride]  their victim slots
    int32_t* miss_cnt;     // [B]
    HsDevState* st;
    int K, C, S, T, cold;
    int list_stride;
    int hash_bits;         // dedup hash capacity = 1 << hash_bits >= 2K
    // Fused variant only: the row fetch and the step advance.
    const uint8_t* pool;   // device-usable address of the mapped pinned pool [B][H][R]
    uint8_t* buf;          // [B][S+T][R]
    long long H;
    int R;
    int rows_per_group;
    unsigned* done;        // CTAs finished this call (returns to 0 after each call)
    int fifo;              // 1: FIFO eviction (hits keep their fill stamp), 0: LRU
    int random;            // 1: random eviction (keys from seed, step, request, slot)
    unsigned long long seed;  // random eviction's seed
    int sliding;           // 1: the tail is [len - T, len) per request; 0: [C - T, C)
    int alias;             // 1: a repeated token takes its first occurrence's slot (several
                           //    draft positions in one row); 0: a repeat is an error
};

// Several handles' steps in one launch (hs_resolve_layers): the first L
// entries are used, all with the same K and S; each handle has B CTAs.
struct LayerArgs {
    ResolveArgs l[HS_MAX_LAYERS];
    int B;
};

struct CopyArgs {
    const int32_t* miss_cnt;
    const int32_t* miss_tok;
    const int32_t* miss_slot;
    const uint8_t* pool;   // device-usable address of the mapped pinned pool [B][H][R]
    uint8_t* buf;          // [B][S+T][R]
    HsDevState* st;
    int B, S, T, R, list_stride;
    long long H;
    int rows_per_group;    // rows a warp copies together (its lanes < rows_per_group own one row each)
    int advance_step;      // 1: block 0 advances st->step after the primary grid finished
    int flat_src;          // 1: `pool` is a staging area holding the rows in flattened order
};

struct AppendArgs {
    const uint8_t* rows;   // [B][R]
    uint8_t* buf;
    int32_t* len;
    HsDevState* st;
    int S, T, R, C, cold;
    uint8_t* pool;         // sliding tail: device-usable address of the mapped host pool
    long long H;
    int sliding;
};

struct ResetArgs {
    const int32_t* ids;      // [n] requests to reset
    const int32_t* lengths;  // [n] or NULL (= C)
    int32_t* tok_slot;
    int32_t* slot_tok;
    int32_t* stamp;
    int32_t* len;
    HsDevState* st;
    int B, C, S;
};

// Launch geometry and shared-memory layout of the resolve kernel.
constexpr int HS_RESOLVE_THREADS = 512;
constexpr int HS_COPY_THREADS = 256;
constexpr int HS_AGE_BINS = 1024;
constexpr int HS_AGE_SUBHIST = 4;

// Bits of the dedup hash: at least 2K entries, so it is at most half full.
__host__ __device__ inline int hs_hash_bits(int K)
{
    int bits = 6;
    while ((1 << bits) < 2 * K) ++bits;
    return bits;
}

// Ints of the region shared by the dedup hash (2 << hash_bits) in phase 1 and,
// once the miss list exists, the age histograms (HS_AGE_SUBHIST * HS_AGE_BINS)
// followed by the out_slot values, entry e of thread tid at e * threads + tid
// (ceil(K / threads) * threads ints), and the cluster kernel's copy list
// (uint16 [K]).  From K = 1025 on the hash alone is larger than all of them.
// A multiple of 4 ints, so that the stamp row after it starts on the 16-byte
// boundary its asynchronous copies and int4 reads need.
__host__ __device__ inline int hs_resolve_region_a_ints(int hash_bits, int K)
{
    const int hc2 = 2 << hash_bits;
    const int per_thread = (K + HS_RESOLVE_THREADS - 1) / HS_RESOLVE_THREADS;
    const int later =
        (HS_AGE_SUBHIST * HS_AGE_BINS + per_thread * HS_RESOLVE_THREADS + (K + 1) / 2 + 3) & ~3;
    return hc2 > later ? hc2 : later;
}

// Shared memory of the resolve kernel: region A (hash; then histograms and
// the out_slot row), stamps [S], slot -> token
// [S], miss tokens [K] (ints); miss row positions [K], victims [K] (uint16);
// the hit bitmap [ceil(S/32)] (words).
__host__ __device__ inline size_t hs_resolve_base_bytes(int K, int S, int hash_bits)
{
    const size_t ints = (size_t)hs_resolve_region_a_ints(hash_bits, K) + 2u * (size_t)S + (size_t)K;
    size_t bytes = 4u * ints + 2u * 2u * (size_t)K;
    bytes += 4u * (size_t)((S + 31) >> 5);
    return bytes;
}

size_t hs_resolve_smem_bytes(int K, int S);
cudaError_t hs_prepare_resolve();
// Resolve only: writes the miss lists for hs_launch_copy.
cudaError_t hs_launch_resolve(const ResolveArgs& a, int B, cudaStream_t s);
// Resolve + row fetch in one launch; advances the step counter itself.
cudaError_t hs_launch_swapin(const ResolveArgs& a, int B, int unroll, cudaStream_t s);
// The same for L handles at once (L * B CTAs).
cudaError_t hs_launch_swapin_layers(const LayerArgs& p, int L, int unroll, cudaStream_t s);
// Resolve + row fetch with a cluster of ncl CTAs per request (B * ncl CTAs).
cudaError_t hs_launch_swapin_cluster(const ResolveArgs& a, int B, int ncl, int unroll,
                                     cudaStream_t s);
// Clusters of ncl swap-in CTAs that fit on the device at once (0 if none).
int hs_cluster_max_active(int K, int S, int ncl, int unroll);

// Copy kernel: `pdl` lets it launch while the resolve grid drains (it waits
// on the resolve grid's completion before reading the miss lists).
cudaError_t hs_launch_copy(const CopyArgs& a, int grid, int unroll, cudaStream_t s, bool pdl);
int hs_copy_unroll_for(int row_bytes);
int hs_copy_rows_per_group(int row_bytes, int unroll);
int hs_copy_blocks_per_sm(int unroll, int B);

cudaError_t hs_launch_append(const AppendArgs& a, int B, cudaStream_t s);
cudaError_t hs_launch_reset_requests(const ResetArgs& a, int n, cudaStream_t s);
cudaError_t hs_launch_h2d_read(const uint8_t* src, uint8_t* dst, size_t bytes, int grid,
                               cudaStream_t s);
