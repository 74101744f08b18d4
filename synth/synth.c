/*
 * Seeded synthetic input generator.
 *
 * Serves both the oracle tests and the CUDA path with identical bytes. It holds
 * none of the MoE layer's arithmetic: it only draws random numbers and maps them
 * through lookup tables that the Python side builds (value distributions, code
 * distributions). Nothing here decodes a weight format.
 *
 * Random stream: counter-based SplitMix64 (Steele, Lea, Flood, "Fast Splittable
 * Pseudorandom Number Generators", OOPSLA 2014). Word i of the stream with key K
 * is mix64(K + (i + 1) * GOLDEN), so any range of a stream can be produced
 * independently and in parallel, and the result does not depend on the number
 * of threads.
 */
#include <stdint.h>
#include <stddef.h>
#include <pthread.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_word(uint64_t key, uint64_t i) {
    return mix64(key + (i + 1) * GOLDEN);
}

/* Key for a (seed, a, b, c) tuple, e.g. (seed, layer, expert, tensor tag). */
uint64_t synth_key(uint64_t seed, uint64_t a, uint64_t b, uint64_t c) {
    uint64_t k = mix64(seed + GOLDEN);
    k = mix64(k ^ (a + 0x1000193ULL));
    k = mix64(k ^ (b + 0x2000387ULL));
    k = mix64(k ^ (c + 0x30005A1ULL));
    return k;
}

uint64_t synth_word(uint64_t key, uint64_t i) { return stream_word(key, i); }

/* ---- threaded range driver ------------------------------------------------ */

typedef void (*range_fn)(void* ctx, size_t lo, size_t hi);

typedef struct { range_fn fn; void* ctx; size_t lo, hi; } job_t;

static void* job_run(void* p) {
    job_t* j = (job_t*)p;
    j->fn(j->ctx, j->lo, j->hi);
    return NULL;
}

/* Splits [0, n) into chunks aligned to `align` items and runs them on up to
 * `nthreads` threads. The output never depends on the thread count. */
static void run_parallel(range_fn fn, void* ctx, size_t n, size_t align, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    size_t min_chunk = (size_t)1 << 20;
    if (n < min_chunk * 2 || nthreads == 1) { fn(ctx, 0, n); return; }
    size_t per = (n + nthreads - 1) / nthreads;
    per = (per + align - 1) / align * align;
    pthread_t th[256];
    job_t jobs[256];
    int live[256];
    int nj = 0;
    for (int t = 0; t < nthreads; ++t) {
        size_t lo = (size_t)t * per, hi = lo + per;
        if (lo >= n) break;
        if (hi > n) hi = n;
        jobs[t].fn = fn; jobs[t].ctx = ctx; jobs[t].lo = lo; jobs[t].hi = hi;
        live[t] = pthread_create(&th[t], NULL, job_run, &jobs[t]) == 0;
        if (!live[t]) fn(ctx, lo, hi);
        nj = t + 1;
    }
    for (int t = 0; t < nj; ++t)
        if (live[t]) pthread_join(th[t], NULL);
}

/* ---- 16-bit table fills: out[i] = tab[u16_i] ------------------------------
 * u16_i is 16-bit lane (i % 4) of stream word (i / 4). */

typedef struct { void* out; uint64_t key; const void* tab; } tab16_ctx;

static void fill_tab16_u16_range(void* c, size_t lo, size_t hi) {
    tab16_ctx* x = (tab16_ctx*)c;
    uint16_t* out = (uint16_t*)x->out;
    const uint16_t* tab = (const uint16_t*)x->tab;
    size_t i = lo;
    while (i < hi) {
        uint64_t w = stream_word(x->key, i >> 2);
        for (unsigned l = (unsigned)(i & 3); l < 4 && i < hi; ++l, ++i)
            out[i] = tab[(w >> (16 * l)) & 0xFFFF];
    }
}

static void fill_tab16_f32_range(void* c, size_t lo, size_t hi) {
    tab16_ctx* x = (tab16_ctx*)c;
    float* out = (float*)x->out;
    const float* tab = (const float*)x->tab;
    size_t i = lo;
    while (i < hi) {
        uint64_t w = stream_word(x->key, i >> 2);
        for (unsigned l = (unsigned)(i & 3); l < 4 && i < hi; ++l, ++i)
            out[i] = tab[(w >> (16 * l)) & 0xFFFF];
    }
}

void synth_fill_tab16_u16(uint16_t* out, size_t n, uint64_t key, const uint16_t* tab, int nthreads) {
    tab16_ctx c = { out, key, tab };
    run_parallel(fill_tab16_u16_range, &c, n, 4, nthreads);
}

void synth_fill_tab16_f32(float* out, size_t n, uint64_t key, const float* tab, int nthreads) {
    tab16_ctx c = { out, key, tab };
    run_parallel(fill_tab16_f32_range, &c, n, 4, nthreads);
}

/* ---- nibble-pair fills: out[i] = tab[b0] | tab[b1] << 4 -------------------
 * b0, b1 are bytes 2*(i%4) and 2*(i%4)+1 of stream word (i / 4); tab maps a
 * random byte to a 4-bit code (its entries are < 16). */

typedef struct { uint8_t* out; uint64_t key; const uint8_t* tab; } nib_ctx;

static void fill_nibbles_range(void* c, size_t lo, size_t hi) {
    nib_ctx* x = (nib_ctx*)c;
    size_t i = lo;
    while (i < hi) {
        uint64_t w = stream_word(x->key, i >> 2);
        for (unsigned l = (unsigned)(i & 3); l < 4 && i < hi; ++l, ++i) {
            unsigned b0 = (unsigned)(w >> (16 * l)) & 0xFF;
            unsigned b1 = (unsigned)(w >> (16 * l + 8)) & 0xFF;
            x->out[i] = (uint8_t)((x->tab[b0] & 0xF) | ((x->tab[b1] & 0xF) << 4));
        }
    }
}

void synth_fill_nibbles(uint8_t* out, size_t n, uint64_t key, const uint8_t* tab256, int nthreads) {
    nib_ctx c = { out, key, tab256 };
    run_parallel(fill_nibbles_range, &c, n, 4, nthreads);
}

/* ---- byte fills: out[i] = lo + (byte_i % (hi - lo + 1)) ------------------- */

typedef struct { uint8_t* out; uint64_t key; unsigned lo, span; } byte_ctx;

static void fill_bytes_range(void* c, size_t lo, size_t hi) {
    byte_ctx* x = (byte_ctx*)c;
    size_t i = lo;
    while (i < hi) {
        uint64_t w = stream_word(x->key, i >> 3);
        for (unsigned l = (unsigned)(i & 7); l < 8 && i < hi; ++l, ++i)
            x->out[i] = (uint8_t)(x->lo + ((unsigned)(w >> (8 * l)) & 0xFF) % x->span);
    }
}

void synth_fill_bytes(uint8_t* out, size_t n, uint64_t key, unsigned lo, unsigned hi, int nthreads) {
    byte_ctx c = { out, key, lo, hi - lo + 1 };
    run_parallel(fill_bytes_range, &c, n, 8, nthreads);
}

/* ---- byte-table fills: out[i] = tab256[byte_i] ----------------------------- */

typedef struct { uint8_t* out; uint64_t key; const uint8_t* tab; } tab8_ctx;

static void fill_tab8_range(void* c, size_t lo, size_t hi) {
    tab8_ctx* x = (tab8_ctx*)c;
    size_t i = lo;
    while (i < hi) {
        uint64_t w = stream_word(x->key, i >> 3);
        for (unsigned l = (unsigned)(i & 7); l < 8 && i < hi; ++l, ++i)
            x->out[i] = x->tab[(w >> (8 * l)) & 0xFF];
    }
}

void synth_fill_tab8(uint8_t* out, size_t n, uint64_t key, const uint8_t* tab256, int nthreads) {
    tab8_ctx c = { out, key, tab256 };
    run_parallel(fill_tab8_range, &c, n, 8, nthreads);
}

/* Uniform doubles in [0, 1) from the top 53 bits of each stream word. */
void synth_fill_uniform(double* out, size_t n, uint64_t key) {
    for (size_t i = 0; i < n; ++i)
        out[i] = (double)(stream_word(key, i) >> 11) * (1.0 / 9007199254740992.0);
}
