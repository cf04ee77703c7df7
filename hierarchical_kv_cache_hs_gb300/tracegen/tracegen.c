/*
 * Seeded synthetic inputs for the HiSparse swap-in path.
 *
 * This module produces the two kinds of input the swap-in path consumes:
 *   - per-step top-k token index rows, standing in for the DSA indexer's
 *     output (HiSparse blog, "Efficient swap-in kernel": the kernel receives
 *     the indexer's top-k selection every decode step; top_k = 2048 in the
 *     launch configurations of the "Benchmarks" section);
 *   - KV row bytes (a 576-element bf16 MLA row = 1152 bytes, filled with
 *     uniform random bits), keyed by (layer, request, token) so that the
 *     same token has the same bytes wherever it lives.
 *
 * It holds none of the method's arithmetic: no page table, no LRU, no copy
 * logic.  Both the CUDA path and the CPU oracle consume what it produces.
 *
 * Random numbers: a counter-based splitmix64.  Every step of every
 * (layer, request) has its own key, so rows can be generated for requests in
 * parallel and a step's draws do not depend on how many draws earlier steps
 * made (only on the previous step's row, which the carry-over reuses).
 *
 * Row composition for step s of one (layer, request), with n = current
 * length (positions [0, n) are selectable):
 *   carry  = floor(carry_pct * K / 100) indices drawn uniformly without
 *            replacement from the previous step's row (step 0: this quota is
 *            moved to the Zipf component);
 *   zipf   = floor(zipf_pct * K / 100) draws from Zipf(a) over positions,
 *            P(p) proportional to (p + 1)^-a for p in [0, n);
 *   rest   = K - carry - zipf draws from the third component: Zipf again,
 *            uniform over [0, n), or uniform over the recent window
 *            [n - W, n).
 * A draw that repeats an index already in the row is redrawn.  After
 * TG_MAX_DRAWS_PER_INDEX repeats for one index (a row that takes nearly every
 * position) the next free position after the last draw is taken instead,
 * cyclically within the component's range.  The finished row is shuffled with
 * Fisher-Yates so that its order carries no structure.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define TG_GOLDEN 0x9E3779B97F4A7C15ULL

/* splitmix64 finaliser applied to (x + golden). */
static inline uint64_t tg_mix(uint64_t x)
{
    uint64_t z = x + TG_GOLDEN;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

typedef struct {
    uint64_t key;
    uint64_t ctr;
} tg_stream;

static inline uint64_t tg_next(tg_stream* s)
{
    uint64_t v = tg_mix(s->key + s->ctr * TG_GOLDEN);
    s->ctr += 1;
    return v;
}

/* Uniform integer in [0, n), n >= 1 (multiply-high mapping). */
static inline int64_t tg_below(tg_stream* s, int64_t n)
{
    unsigned __int128 p = (unsigned __int128)tg_next(s) * (unsigned __int128)(uint64_t)n;
    return (int64_t)(p >> 64);
}

/* Uniform double in [0, 1) with 53 random bits. */
static inline double tg_unit(tg_stream* s)
{
    return (double)(tg_next(s) >> 11) * (1.0 / 9007199254740992.0);
}

static uint64_t tg_row_key_of(uint64_t seed, int32_t wl, int32_t layer, int32_t b, int32_t step)
{
    uint64_t k = tg_mix(seed);
    k = tg_mix(k ^ (uint64_t)(uint32_t)wl);
    k = tg_mix(k ^ (uint64_t)(uint32_t)layer);
    k = tg_mix(k ^ (uint64_t)(uint32_t)b);
    k = tg_mix(k ^ (uint64_t)(uint32_t)step);
    return k;
}

static uint64_t tg_bytes_key_of(uint64_t seed, int32_t wl, int32_t layer, int32_t b, int32_t tok)
{
    uint64_t k = tg_mix(seed ^ 0x4B56524F57ULL); /* distinct domain from the rows */
    k = tg_mix(k ^ (uint64_t)(uint32_t)wl);
    k = tg_mix(k ^ (uint64_t)(uint32_t)layer);
    k = tg_mix(k ^ (uint64_t)(uint32_t)b);
    k = tg_mix(k ^ (uint64_t)(uint32_t)tok);
    return k;
}

enum { TG_THIRD_ZIPF = 0, TG_THIRD_UNIFORM = 1, TG_THIRD_RECENT = 2 };

typedef struct {
    uint64_t seed;
    int32_t workload;   /* workload id, part of every key */
    int32_t K;          /* indices per row */
    int32_t len0;       /* length before the first step */
    int32_t grow;       /* tokens appended per step before drawing */
    int32_t carry_pct;
    int32_t zipf_pct;
    int32_t third;      /* TG_THIRD_* */
    int32_t recent;     /* window W for TG_THIRD_RECENT */
    double zipf_a;      /* Zipf exponent */
} tg_params;

/* Cumulative Zipf weights: cdf[i] = sum_{p <= i} (p + 1)^-a, i < n. */
int tg_zipf_cdf(double a, int32_t n, double* cdf)
{
    if (n <= 0 || !cdf) return -1;
    double acc = 0.0;
    for (int32_t i = 0; i < n; ++i) {
        acc += pow((double)i + 1.0, -a);
        cdf[i] = acc;
    }
    return 0;
}

/* Smallest p in [0, n) with cdf[p] > x (x < cdf[n-1]). */
static int32_t tg_zipf_pick(const double* cdf, int32_t n, double x)
{
    int32_t lo = 0, hi = n - 1;
    while (lo < hi) {
        int32_t mid = lo + (hi - lo) / 2;
        if (cdf[mid] > x) hi = mid; else lo = mid + 1;
    }
    return lo;
}

/* Length n at step s (0-based). */
int32_t tg_len_at(const tg_params* p, int32_t s)
{
    return p->len0 + p->grow * (s + 1);
}

#define TG_MAX_DRAWS_PER_INDEX 100000

/*
 * The first position in [lo, hi) not taken at this epoch, searching cyclically
 * from `from`; -1 when every one is taken.  Used only once a component's
 * random draws have hit TG_MAX_DRAWS_PER_INDEX (a row that takes nearly every
 * position), so rows that the draws alone can fill are unchanged.
 */
static int32_t tg_next_free(const uint32_t* mark, uint32_t epoch, int32_t lo, int32_t hi,
                            int32_t from)
{
    int32_t q = (from >= lo && from < hi) ? from : lo;
    for (int32_t k = lo; k < hi; ++k) {
        if (mark[q] != epoch) return q;
        q = (q + 1 == hi) ? lo : q + 1;
    }
    return -1;
}

/*
 * Rows of steps [0, nsteps) of one (layer, request).  out + s * step_stride
 * receives step s's K indices.  cdf must cover max length over the steps.
 * Returns 0, or -1 on bad arguments / a component that cannot be filled.
 */
int tg_trace_request(const tg_params* p, const double* cdf, int32_t cdf_n,
                     int32_t layer, int32_t b, int32_t nsteps,
                     int32_t* out, int64_t step_stride)
{
    const int32_t K = p->K;
    if (K <= 0 || nsteps <= 0 || !out || !cdf) return -1;
    int32_t nmax = tg_len_at(p, nsteps - 1);
    if (nmax > cdf_n || p->len0 + p->grow < K) return -1;
    if (p->carry_pct < 0 || p->zipf_pct < 0 || p->carry_pct + p->zipf_pct > 100) return -1;
    if (p->third == TG_THIRD_RECENT && p->recent < K) return -1;

    uint32_t* mark = (uint32_t*)calloc((size_t)nmax, sizeof(uint32_t));
    int32_t* tmp = (int32_t*)malloc((size_t)K * sizeof(int32_t));
    if (!mark || !tmp) { free(mark); free(tmp); return -1; }

    const int32_t carry_q = (int32_t)(((int64_t)p->carry_pct * K) / 100);
    const int32_t zipf_q = (int32_t)(((int64_t)p->zipf_pct * K) / 100);
    const int32_t rest_q = K - carry_q - zipf_q;
    int rc = 0;

    for (int32_t s = 0; s < nsteps && rc == 0; ++s) {
        const int32_t n = tg_len_at(p, s);
        const uint32_t epoch = (uint32_t)s + 1u;
        tg_stream st = { tg_row_key_of(p->seed, p->workload, layer, b, s), 0 };
        int32_t* row = out + (int64_t)s * step_stride;
        int32_t cnt = 0;

        int32_t zq = zipf_q;
        if (s == 0) {
            zq += carry_q;
        } else {
            const int32_t* prev = out + (int64_t)(s - 1) * step_stride;
            memcpy(tmp, prev, (size_t)K * sizeof(int32_t));
            for (int32_t i = 0; i < carry_q; ++i) {
                int32_t j = i + (int32_t)tg_below(&st, K - i);
                int32_t x = tmp[i]; tmp[i] = tmp[j]; tmp[j] = x;
                row[cnt++] = tmp[i];
                mark[tmp[i]] = epoch;
            }
        }

        /* Zipf component. */
        const double total = cdf[n - 1];
        for (int32_t got = 0; got < zq && rc == 0; ) {
            int64_t tries = 0;
            for (;;) {
                int32_t pos = tg_zipf_pick(cdf, n, tg_unit(&st) * total);
                if (mark[pos] != epoch) { mark[pos] = epoch; row[cnt++] = pos; ++got; break; }
                if (++tries > TG_MAX_DRAWS_PER_INDEX) {
                    pos = tg_next_free(mark, epoch, 0, n, pos);
                    if (pos < 0) { rc = -1; break; }
                    mark[pos] = epoch; row[cnt++] = pos; ++got; break;
                }
            }
        }
        /* Third component. */
        for (int32_t got = 0; got < rest_q && rc == 0; ) {
            int64_t tries = 0;
            for (;;) {
                int32_t pos, lo = 0;
                if (p->third == TG_THIRD_ZIPF) {
                    pos = tg_zipf_pick(cdf, n, tg_unit(&st) * total);
                } else if (p->third == TG_THIRD_UNIFORM) {
                    pos = (int32_t)tg_below(&st, n);
                } else {
                    int32_t w = p->recent < n ? p->recent : n;
                    lo = n - w;
                    pos = lo + (int32_t)tg_below(&st, w);
                }
                if (mark[pos] != epoch) { mark[pos] = epoch; row[cnt++] = pos; ++got; break; }
                if (++tries > TG_MAX_DRAWS_PER_INDEX) {
                    pos = tg_next_free(mark, epoch, lo, n, pos);
                    if (pos < 0) { rc = -1; break; }
                    mark[pos] = epoch; row[cnt++] = pos; ++got; break;
                }
            }
        }
        /* Fisher-Yates shuffle of the finished row. */
        for (int32_t i = K - 1; i > 0 && rc == 0; --i) {
            int32_t j = (int32_t)tg_below(&st, (int64_t)i + 1);
            int32_t x = row[i]; row[i] = row[j]; row[j] = x;
        }
    }
    free(mark);
    free(tmp);
    return rc;
}

/*
 * Bytes of tokens [t0, t0 + n) of (layer, request) into dst, row t0 + i at
 * dst + i * dst_stride.  Word w of a row is mix(key + w * golden), stored
 * little-endian; a tail shorter than 8 bytes takes the low bytes.
 */
int tg_fill_rows(uint64_t seed, int32_t workload, int32_t layer, int32_t b,
                 int32_t t0, int32_t n, int32_t row_bytes,
                 uint8_t* dst, int64_t dst_stride)
{
    if (n < 0 || row_bytes <= 0 || (!dst && n > 0)) return -1;
    for (int32_t i = 0; i < n; ++i) {
        tg_stream st = { tg_bytes_key_of(seed, workload, layer, b, t0 + i), 0 };
        uint8_t* d = dst + (int64_t)i * dst_stride;
        int32_t w = 0;
        for (; w + 8 <= row_bytes; w += 8) {
            uint64_t v = tg_next(&st);
            for (int k = 0; k < 8; ++k) d[w + k] = (uint8_t)(v >> (8 * k));
        }
        if (w < row_bytes) {
            uint64_t v = tg_next(&st);
            for (int k = 0; w + k < row_bytes; ++k) d[w + k] = (uint8_t)(v >> (8 * k));
        }
    }
    return 0;
}

/* Raw stream values, for testing the generator against its definition. */
uint64_t tg_stream_value(uint64_t key, uint64_t ctr)
{
    tg_stream st = { key, ctr };
    return tg_next(&st);
}

uint64_t tg_splitmix64(uint64_t x)
{
    return tg_mix(x);
}
