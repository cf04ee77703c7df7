/*
 * A plain C program driving the swap-in library through its C ABI alone
 * (include/hs.h): create a handle, fill the pinned host pool, resolve a few
 * decode steps from host buffers, and check the counters against what the
 * rows must give.  No CUDA header or call is needed on the caller's side.
 *
 * Build (from the repository root, after libhs.so is built):
 *   cc -O2 -I include hierarchical_kv_cache_hs_gb300/examples/resolve_from_c.c \
 *      -L hierarchical_kv_cache_hs_gb300 -lhs -Wl,-rpath,$PWD/hierarchical_kv_cache_hs_gb300 \
 *      -o resolve_from_c
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "hs.h"

#define B 4        /* requests */
#define C 8192     /* context tokens */
#define R 1152     /* bytes per KV row */
#define S 512      /* hot-buffer slots per request */
#define K 256      /* top-k per step */
#define STEPS 6

static int fail(const char* what, int rc)
{
    fprintf(stderr, "%s: %s (%d)\n", what, hs_error_string(rc), rc);
    return 1;
}

int main(void)
{
    hs_handle* h = NULL;
    int rc = hs_create(B, C, R, S, C / S, 0, &h);
    if (rc != HS_OK) return fail("hs_create", rc);

    /* Host pool [B][H][R]: row t of request b holds (b + t) mod 251 everywhere. */
    uint8_t* pool = hs_host_pool(h);
    const size_t H = (size_t)(C / S) * S;
    for (size_t b = 0; b < B; ++b)
        for (size_t t = 0; t < C; ++t) memset(pool + (b * H + t) * R, (int)((b + t) % 251), R);

    int32_t* topk = malloc(sizeof(int32_t) * B * K);
    int32_t* out = malloc(sizeof(int32_t) * B * K);
    if (!topk || !out) return 1;
    /* Step s selects tokens s*K/2 .. s*K/2 + K - 1: half of each row is new. */
    int64_t expect_misses = 0;
    for (int s = 0; s < STEPS; ++s) {
        for (int b = 0; b < B; ++b)
            for (int j = 0; j < K; ++j) topk[b * K + j] = s * (K / 2) + j;
        rc = hs_resolve_host(h, topk, K, out, NULL);
        if (rc != HS_OK) return fail("hs_resolve_host", rc);
        expect_misses += (int64_t)B * (s == 0 ? K : K / 2);
        for (int i = 0; i < B * K; ++i)
            if (out[i] < 0 || out[i] >= S) {
                fprintf(stderr, "step %d: slot %d out of range\n", s, out[i]);
                return 1;
            }
    }
    hs_stats_t st;
    rc = hs_stats(h, &st, NULL);
    if (rc != HS_OK) return fail("hs_stats", rc);
    /* Every slot the last step returned holds its token's row. */
    uint8_t* row = malloc((size_t)(S) * R);
    int bad = 0;
    for (int b = 0; b < B && row; ++b) {
        if (hs_export_buffer(h, b, row) != HS_OK) return 1;
        for (int j = 0; j < K; ++j) {
            const int t = (STEPS - 1) * (K / 2) + j;
            if (row[(size_t)out[b * K + j] * R] != (uint8_t)((b + t) % 251)) ++bad;
        }
    }
    printf("steps %lld hits %lld misses %lld (expected %lld) errors 0x%x bad rows %d\n",
           (long long)st.steps, (long long)st.hits, (long long)st.misses, (long long)expect_misses,
           st.err_bits, bad);
    hs_destroy(h);
    free(topk);
    free(out);
    free(row);
    return (st.misses == expect_misses && st.err_bits == 0 && bad == 0) ? 0 : 1;
}
