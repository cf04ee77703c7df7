/*
 * CPU ORACLE for the HiSparse swap-in path -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the package smoke check and the benchmark's CPU-baseline
 * leg may load this.  The product path never calls it and shares no code
 * with it (no headers, helpers or tables).
 *
 * What it computes, one request at a time, in plain sequential C:
 *
 *   The swap-in kernel of the HiSparse blog ("Efficient swap-in kernel"
 *   section; the papercache summary, section 2 "Method", steps 1-3) does
 *   three things per decode step:
 *     (1) find which top-k indices miss in the device buffer,
 *     (2) choose eviction candidates by LRU,
 *     (3) update the page table and fetch the missing entries from host
 *         memory into device memory.
 *   The vLLM "Hybrid HiSparse" post ("Mixed Residency") adds: tokens in the
 *   resident tail are read in place; tokens in the hot buffer are read with
 *   their LRU entry refreshed; a miss copies a single row from pinned host
 *   memory into the LRU slot.  Its "No Residency" state is the start state
 *   here: an empty buffer, rows load only when the indexer selects them.
 *
 * Eviction policy: the pages compare eviction strategies by their miss
 * counts (HiSparse blog, "Efficient swap-in kernel": a larger buffer with
 * LRU misses far less).  Besides LRU the oracle offers FIFO, the plainest
 * alternative: a slot's stamp is the step it was filled, hits do not refresh
 * it, and a slot hit in this step is still never evicted in that step.
 * The third point on that axis is random eviction: the victims are a uniform
 * random choice among the slots not hit this step, empty slots first.  Each
 * such slot gets a key, 0 when it is empty and otherwise 1 plus the top 30
 * bits of one SplitMix64 output (Steele, Lea and Flood, "Fast Splittable
 * Pseudorandom Number Generators", OOPSLA 2014, with the output function as
 * Vigna publishes it) of the state seed XOR (step << 32 | request << 14 |
 * slot); the victims are the slots with the smallest (key, slot) pairs.
 * Stamps keep the step of last use, as under LRU.
 *
 * Resident tail, two readings of which tokens it holds:
 *   fixed    the last T positions of the capacity, [C - T, C) (a growing
 *            context appends into it until it is full);
 *   sliding  the last T tokens written, [len - T, len): a token that leaves
 *            the tail on an append is written back to its host row and from
 *            then on is an ordinary host-backed token (vLLM Hybrid HiSparse
 *            post, "Full Residency" and "Mixed Residency": the tail stays on
 *            the GPU while older pages move to host memory, copied there so
 *            that eviction needs no further copy).
 *
 * Several draft positions (speculative decoding; vLLM Hybrid HiSparse post,
 * "Speculative Decoding": a per-step resolver plan over the request's shared
 * hot state): the P top-k rows of one step are resolved as one concatenated
 * row.  In this "alias" mode a repeated token is not an error: it gets the
 * slot of its first occurrence, and only first occurrences are counted,
 * fetched and paired with victims.
 *
 * Readings where the pages are silent (each is a plain choice):
 *   - one token per page: the table maps token -> slot;
 *   - a stamp is the step counter at last use (hit or fill); steps start
 *     at 1, stamp 0 = never used, so empty slots go first;
 *   - victims are the slots not hit this step with the smallest
 *     (stamp, slot) pairs: ties go to the lowest slot index;
 *   - the i-th miss in top-k row order is paired with the i-th victim in
 *     ascending slot order;
 *   - a tail token t (t >= C - T) resolves to slot S + (t mod T), touches no
 *     table and counts neither as hit nor miss;
 *   - -1 is padding; an index < -1 or >= the current length, or a repeat of
 *     an earlier index of the same row, is an error: out = -1, an error bit
 *     is set, the state is untouched for that entry.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_E_RANGE 1
#define OR_E_DUP 2
#define OR_E_NOROOM 8

#define OR_POLICY_LRU 0
#define OR_POLICY_FIFO 1
#define OR_POLICY_RANDOM 2

typedef struct {
    int32_t stamp;
    int32_t slot;
} or_pair;

static int or_cmp_pair(const void* a, const void* b)
{
    const or_pair* x = (const or_pair*)a;
    const or_pair* y = (const or_pair*)b;
    if (x->stamp != y->stamp) return x->stamp < y->stamp ? -1 : 1;
    if (x->slot != y->slot) return x->slot < y->slot ? -1 : 1;
    return 0;
}

/* One SplitMix64 output for the state x: advance by the golden-ratio
 * increment, then the two xor-shift-multiply rounds and a final xor-shift. */
static uint64_t or_splitmix64(uint64_t x)
{
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* Random-eviction key of slot s of request req at step `step`; see the header. */
static int32_t or_random_key(uint64_t seed, int32_t step, int32_t req, int32_t s, int32_t empty)
{
    if (empty) return 0;
    const uint64_t x = ((uint64_t)(uint32_t)step << 32) | ((uint64_t)(uint32_t)req << 14) | (uint64_t)(uint32_t)s;
    return 1 + (int32_t)(or_splitmix64(seed ^ x) >> 34);
}

/* The generator alone, for its known-answer test. */
uint64_t or_splitmix64_at(uint64_t x) { return or_splitmix64(x); }

static int or_cmp_int(const void* a, const void* b)
{
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/*
 * Empty state of one request: tok_slot[C] = -1, slot_tok[S] = -1, stamp[S] = 0.
 */
void or_init(int32_t C, int32_t S, int32_t* tok_slot, int32_t* slot_tok, int32_t* stamp)
{
    for (int32_t t = 0; t < C; ++t) tok_slot[t] = -1;
    for (int32_t s = 0; s < S; ++s) { slot_tok[s] = -1; stamp[s] = 0; }
}

/*
 * One resolve of one request at step `step` (>= 1, the handle's counter after
 * it was advanced for this call).
 *
 *   C, S, T, R   capacity, buffer slots, resident tail, row bytes
 *   len          current length: valid indices are [0, len)
 *   tok_slot[C], slot_tok[S], stamp[S]   the request's state (updated)
 *   buf[(S+T)*R]                          the request's device-buffer model
 *   host[(C-T)*R]                         host rows of the request, by token
 *   topk[K]                               this step's top-k row
 *   out[K]                                resolved slots
 *   counts[3]                             hits, misses, in-place
 *
 * Returns the error bits (OR_E_*).
 */
static int32_t or_resolve_core(int32_t C, int32_t S, int32_t T, int32_t R, int32_t len,
                               int32_t* tok_slot, int32_t* slot_tok, int32_t* stamp, uint8_t* buf,
                               const uint8_t* host, const int32_t* topk, int32_t K, int32_t step,
                               int32_t* out, int32_t* counts, int32_t policy, int32_t sliding,
                               int32_t alias, int32_t req, uint64_t seed)
{
    int32_t err = 0;
    int32_t hits = 0, nmiss = 0, inplace = 0;
    /* First position of the resident tail. */
    const int32_t cold = sliding ? (len - T > 0 ? len - T : 0) : C - T;

    unsigned char* seen = (unsigned char*)calloc((size_t)(C > 0 ? C : 1), 1);
    int32_t* first = (int32_t*)malloc(sizeof(int32_t) * (size_t)(C > 0 ? C : 1));
    int32_t* alias_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)(K > 0 ? K : 1));
    unsigned char* hit = (unsigned char*)calloc((size_t)(S > 0 ? S : 1), 1);
    int32_t* miss_tok = (int32_t*)malloc(sizeof(int32_t) * (size_t)(K > 0 ? K : 1));
    int32_t* miss_pos = (int32_t*)malloc(sizeof(int32_t) * (size_t)(K > 0 ? K : 1));
    or_pair* cand = (or_pair*)malloc(sizeof(or_pair) * (size_t)(S > 0 ? S : 1));
    int32_t* victims = (int32_t*)malloc(sizeof(int32_t) * (size_t)(K > 0 ? K : 1));

    /* Step 1: classify every entry in row order; hits and misses. */
    for (int32_t j = 0; j < K; ++j) {
        int32_t t = topk[j];
        out[j] = -1;
        if (t == -1) continue;                       /* padding */
        if (t < -1 || t >= len || t >= C) { err |= OR_E_RANGE; continue; }
        if (seen[t]) {                               /* repeat of an earlier entry */
            if (alias) alias_of[j] = first[t];
            else err |= OR_E_DUP;
            continue;
        }
        seen[t] = 1;
        first[t] = j;
        alias_of[j] = -1;
        if (t >= cold) {                             /* resident tail: in place */
            out[j] = S + t % T;
            inplace += 1;
            continue;
        }
        if (tok_slot[t] >= 0) {                      /* hit */
            out[j] = tok_slot[t];
            hit[tok_slot[t]] = 1;
            hits += 1;
        } else {                                     /* miss, kept in row order */
            miss_tok[nmiss] = t;
            miss_pos[nmiss] = j;
            nmiss += 1;
        }
    }

    /* Under LRU (and random) a hit refreshes the slot's entry; under FIFO it
     * does not. */
    if (policy != OR_POLICY_FIFO)
        for (int32_t s = 0; s < S; ++s)
            if (hit[s]) stamp[s] = step;

    /* Step 2: victims among the slots not hit this step: the smallest
     * (stamp, slot) pairs, or (key, slot) pairs under random eviction. */
    int32_t ncand = 0;
    for (int32_t s = 0; s < S; ++s) {
        if (hit[s]) continue;
        cand[ncand].stamp = policy == OR_POLICY_RANDOM
                                ? or_random_key(seed, step, req, s, slot_tok[s] < 0)
                                : stamp[s];
        cand[ncand].slot = s;
        ncand += 1;
    }
    if (nmiss > ncand) {
        /* Cannot happen when K <= S; reported rather than assumed. */
        err |= OR_E_NOROOM;
        nmiss = ncand;
    }
    qsort(cand, (size_t)ncand, sizeof(or_pair), or_cmp_pair);
    for (int32_t i = 0; i < nmiss; ++i) victims[i] = cand[i].slot;
    qsort(victims, (size_t)nmiss, sizeof(int32_t), or_cmp_int);

    /* Step 3: page-table update and host -> device fetch, one row per miss. */
    for (int32_t i = 0; i < nmiss; ++i) {
        int32_t t = miss_tok[i];
        int32_t v = victims[i];
        int32_t old = slot_tok[v];
        if (old >= 0) tok_slot[old] = -1;
        slot_tok[v] = t;
        tok_slot[t] = v;
        stamp[v] = step;
        out[miss_pos[i]] = v;
        memcpy(buf + (size_t)v * (size_t)R, host + (size_t)t * (size_t)R, (size_t)R);
    }

    /* Repeats (alias mode) take their first occurrence's slot. */
    if (alias)
        for (int32_t j = 0; j < K; ++j) {
            int32_t t = topk[j];
            if (t >= 0 && t < len && t < C && seen[t] && first[t] != j) out[j] = out[alias_of[j]];
        }

    counts[0] = hits;
    counts[1] = nmiss;
    counts[2] = inplace;

    free(seen); free(first); free(alias_of); free(hit); free(miss_tok); free(miss_pos); free(cand); free(victims);
    return err;
}

int32_t or_resolve_full(int32_t C, int32_t S, int32_t T, int32_t R, int32_t len,
                        int32_t* tok_slot, int32_t* slot_tok, int32_t* stamp, uint8_t* buf,
                        const uint8_t* host, const int32_t* topk, int32_t K, int32_t step,
                        int32_t* out, int32_t* counts, int32_t policy, int32_t sliding,
                        int32_t alias)
{
    return or_resolve_core(C, S, T, R, len, tok_slot, slot_tok, stamp, buf, host, topk, K, step,
                           out, counts, policy, sliding, alias, 0, 0);
}

/* Any policy, with the request's index and the seed that random eviction keys on. */
int32_t or_resolve_keyed(int32_t C, int32_t S, int32_t T, int32_t R, int32_t len,
                         int32_t* tok_slot, int32_t* slot_tok, int32_t* stamp, uint8_t* buf,
                         const uint8_t* host, const int32_t* topk, int32_t K, int32_t step,
                         int32_t* out, int32_t* counts, int32_t policy, int32_t sliding,
                         int32_t alias, int32_t req, uint64_t seed)
{
    return or_resolve_core(C, S, T, R, len, tok_slot, slot_tok, stamp, buf, host, topk, K, step,
                           out, counts, policy, sliding, alias, req, seed);
}

int32_t or_resolve_ex(int32_t C, int32_t S, int32_t T, int32_t R, int32_t len,
                      int32_t* tok_slot, int32_t* slot_tok, int32_t* stamp, uint8_t* buf,
                      const uint8_t* host, const int32_t* topk, int32_t K, int32_t step,
                      int32_t* out, int32_t* counts, int32_t policy, int32_t sliding)
{
    return or_resolve_full(C, S, T, R, len, tok_slot, slot_tok, stamp, buf, host, topk, K, step,
                           out, counts, policy, sliding, 0);
}

/* Fixed tail, chosen eviction policy. */
int32_t or_resolve_policy(int32_t C, int32_t S, int32_t T, int32_t R, int32_t len,
                          int32_t* tok_slot, int32_t* slot_tok, int32_t* stamp, uint8_t* buf,
                          const uint8_t* host, const int32_t* topk, int32_t K, int32_t step,
                          int32_t* out, int32_t* counts, int32_t policy)
{
    return or_resolve_ex(C, S, T, R, len, tok_slot, slot_tok, stamp, buf, host, topk, K, step,
                         out, counts, policy, 0);
}

/* The LRU step (the swap-in kernel's policy). */
int32_t or_resolve(int32_t C, int32_t S, int32_t T, int32_t R, int32_t len,
                   int32_t* tok_slot, int32_t* slot_tok, int32_t* stamp, uint8_t* buf,
                   const uint8_t* host, const int32_t* topk, int32_t K, int32_t step,
                   int32_t* out, int32_t* counts)
{
    return or_resolve_policy(C, S, T, R, len, tok_slot, slot_tok, stamp, buf, host, topk, K,
                             step, out, counts, OR_POLICY_LRU);
}

/*
 * Mixed residency: write the next token (position *len) into the resident
 * tail, slot S + (*len mod T), and advance the length.  Only a token that
 * belongs to the tail ([C - T, C)) can be appended; otherwise nothing is
 * written and OR_E_RANGE is returned.
 */
int32_t or_append(int32_t C, int32_t S, int32_t T, int32_t R, int32_t* len,
                  uint8_t* buf, const uint8_t* row)
{
    int32_t t = *len;
    if (T <= 0 || t < C - T || t >= C) return OR_E_RANGE;
    memcpy(buf + (size_t)(S + t % T) * (size_t)R, row, (size_t)R);
    *len = t + 1;
    return 0;
}

/*
 * Sliding tail: append token *len.  When the tail already holds T tokens, the
 * oldest one (position *len - T, in the same tail slot) is first written back
 * to its host row.  Only a token below the capacity C can be appended;
 * otherwise nothing changes and OR_E_RANGE is returned.
 */
int32_t or_append_sliding(int32_t C, int32_t S, int32_t T, int32_t R, int32_t* len,
                          uint8_t* buf, uint8_t* host, const uint8_t* row)
{
    int32_t t = *len;
    if (T <= 0 || t >= C) return OR_E_RANGE;
    uint8_t* slot = buf + (size_t)(S + t % T) * (size_t)R;
    if (t >= T) memcpy(host + (size_t)(t - T) * (size_t)R, slot, (size_t)R);
    memcpy(slot, row, (size_t)R);
    *len = t + 1;
    return 0;
}
