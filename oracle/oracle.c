/*
 * ORACLE — test infrastructure, not the product.
 *
 * A plain, slow, single-threaded fp32 CPU implementation of the routed
 * Mixture-of-Experts layer with a device-side LRU expert cache, used only to
 * check the CUDA path. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load it. It shares no code, header, table or constant with
 * the CUDA library, and must be built with -ffp-contract=off so that every
 * multiply and add below rounds exactly as written.
 *
 * What it follows:
 *  - "FreeToken量子化：MoE推論のセットアップガイド" (freetoken.wiki, architecture
 *    page), paragraphs on the two-tier expert memory (host holds every routed
 *    expert, VRAM is one expert cache shared by all MoE layers), on prefill
 *    whole-layer double buffering (the next layer's experts stream over PCIe
 *    while the current layer computes, when the cache has room) and on decode
 *    (an LRU over recently selected experts; a hit runs on the GPU, a miss is
 *    copied into the cache over PCIe).
 *  - The blog post on reading FreeToken's numbers (bhrtaym-blog.com), section on
 *    the four MoE backends (the `offload` backend: experts in host RAM, LRU slots
 *    on the GPU, misses streamed over PCIe) and section on the supported weight
 *    formats (MXFP4, NVFP4, FP8, BF16).
 *  - The weight formats themselves follow the OCP Microscaling Formats (MX) v1.0
 *    specification (E2M1 elements, E8M0 block scale over 32 elements) and the
 *    NVFP4 definition (E2M1 elements, an E4M3 scale per 16 elements and one fp32
 *    scale per tensor).
 *
 * Readings where the pages are silent (each one is also listed in the design
 * notes):
 *  - router logits are summed in one fixed order (orc_router_logits) so that
 *    the top-k decision is reproducible bit for bit;
 *  - top-k is taken on the logits (softmax is strictly increasing), ordered by
 *    logit descending, ties to the lower expert index;
 *  - gates are the full softmax renormalised over the k selected experts;
 *  - the LRU batch rule and the prefill prefetch rule (orc_lru_batch).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Codecs (format definitions)                                               */
/* ------------------------------------------------------------------------- */

/* E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa. Exponent 0 is
 * subnormal: value = mantissa * 2^(1-1) * 1/2. Otherwise
 * value = 2^(e-1) * (1 + m/2). Magnitudes: 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
float orc_e2m1(unsigned code) {
    unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    float v;
    if (e == 0) v = 0.5f * (float)m;
    else v = ldexpf(1.0f + 0.5f * (float)m, (int)e - 1);
    return s ? -v : v;
}

/* E4M3 (the "FN" variant): bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0
 * mantissa. No infinities; exponent 15 with mantissa 7 is NaN. Exponent 0 is
 * subnormal: value = m/8 * 2^-6. Largest finite value 448. */
float orc_e4m3fn(unsigned b) {
    unsigned s = (b >> 7) & 1u, e = (b >> 3) & 15u, m = b & 7u;
    float v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexpf((float)m / 8.0f, -6);
    else v = ldexpf(1.0f + (float)m / 8.0f, (int)e - 7);
    return s ? -v : v;
}

/* E8M0: an unsigned biased exponent, value 2^(b-127); 0xFF is NaN. */
float orc_e8m0(unsigned b) {
    if (b == 255u) return NAN;
    return ldexpf(1.0f, (int)b - 127);
}

/* bf16 is the upper half of an IEEE binary32. */
float orc_bf16(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* binary32 -> bf16, round to nearest, ties to even (NaN kept quiet). */
uint16_t orc_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void orc_bf16_to_f32(const uint16_t* in, size_t n, float* out) {
    for (size_t i = 0; i < n; ++i) out[i] = orc_bf16(in[i]);
}

void orc_f32_to_bf16(const float* in, size_t n, uint16_t* out) {
    for (size_t i = 0; i < n; ++i) out[i] = orc_bf16_rne(in[i]);
}

enum { ORC_FP32 = 0, ORC_BF16 = 1, ORC_NVFP4 = 2, ORC_MXFP4 = 3, ORC_FP8 = 4 };

/* Dequantise one [N, K] weight tensor stored row-major along K.
 *  FP32:  data = float[N*K]
 *  BF16:  data = uint16[N*K]
 *  NVFP4: data = packed codes uint8[N*K/2] (element 2i in the low nibble of
 *         byte i), scales = E4M3 bytes [N*K/16]; w = code * scale * gscale
 *  MXFP4: data = packed codes as above, scales = E8M0 bytes [N*K/32];
 *         w = code * scale
 *  FP8:   data = E4M3 (FN) bytes uint8[N*K], one per element; no block
 *         scales; w = code * gscale (one fp32 scale per tensor, as NVFP4's) */
void orc_dequant(int fmt, const void* data, const uint8_t* scales, float gscale,
                 int N, int K, float* out) {
    for (int n = 0; n < N; ++n) {
        for (int kk = 0; kk < K; ++kk) {
            size_t i = (size_t)n * K + kk;
            float w;
            if (fmt == ORC_FP32) {
                w = ((const float*)data)[i];
            } else if (fmt == ORC_BF16) {
                w = orc_bf16(((const uint16_t*)data)[i]);
            } else if (fmt == ORC_FP8) {
                w = orc_e4m3fn(((const uint8_t*)data)[i]) * gscale;
            } else {
                uint8_t byte = ((const uint8_t*)data)[i / 2];
                unsigned code = (i & 1) ? (byte >> 4) : (byte & 0xF);
                float c = orc_e2m1(code);
                if (fmt == ORC_NVFP4) {
                    float s = orc_e4m3fn(scales[(size_t)n * (K / 16) + kk / 16]);
                    w = (c * s) * gscale;
                } else {
                    float s = orc_e8m0(scales[(size_t)n * (K / 32) + kk / 32]);
                    w = c * s;
                }
            }
            out[i] = w;
        }
    }
}

/* ------------------------------------------------------------------------- */
/* Router                                                                    */
/* ------------------------------------------------------------------------- */

/* logits[t, e] = sum_h x[t, h] * w[e, h], summed in one fixed order:
 * H is cut into chunks of 8 consecutive elements; chunk c belongs to partial
 * sum c mod 32; each partial sum starts at 0 and takes its chunks in increasing
 * h with a fused multiply-add; the 32 partial sums are then combined by
 * pairwise halving: for o = 16, 8, 4, 2, 1, p[i] <- p[i] + p[i xor o] for every
 * i, and the result is p[0]. Requires H % 8 == 0. */
void orc_router_logits(const float* x, const float* w, int T, int E, int H, float* logits) {
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            float p[32];
            for (int i = 0; i < 32; ++i) p[i] = 0.0f;
            for (int c = 0; c < H / 8; ++c) {
                for (int h = 8 * c; h < 8 * c + 8; ++h)
                    p[c % 32] = fmaf(x[(size_t)t * H + h], w[(size_t)e * H + h], p[c % 32]);
            }
            for (int o = 16; o >= 1; o /= 2) {
                float q[32];
                for (int i = 0; i < 32; ++i) q[i] = p[i] + p[i ^ o];
                for (int i = 0; i < 32; ++i) p[i] = q[i];
            }
            logits[(size_t)t * E + e] = p[0];
        }
    }
}

/* For each token: softmax over all E logits, the k experts with the largest
 * logits (ties to the lower index; NaN counts as -inf), ordered by logit
 * descending then index ascending, and the gates = softmax probabilities of
 * the selected experts renormalised to sum to 1. probs may be NULL. */
void orc_router_topk(const float* logits, int T, int E, int k,
                     int32_t* idx, float* gates, float* probs) {
    float* p = (float*)malloc(sizeof(float) * (size_t)E);
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (size_t)t * E;
        float mx = -INFINITY;
        for (int e = 0; e < E; ++e) if (!isnan(l[e]) && l[e] > mx) mx = l[e];
        float den = 0.0f;
        for (int e = 0; e < E; ++e) {
            p[e] = isnan(l[e]) ? 0.0f : expf(l[e] - mx);
            den += p[e];
        }
        for (int e = 0; e < E; ++e) p[e] = p[e] / den;
        if (probs) memcpy(probs + (size_t)t * E, p, sizeof(float) * (size_t)E);
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            float bv = 0.0f;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                float v = isnan(l[e]) ? -INFINITY : l[e];
                if (best < 0 || v > bv) { best = e; bv = v; }
            }
            taken[best] = 1;
            idx[(size_t)t * k + j] = best;
        }
        float s = 0.0f;
        for (int j = 0; j < k; ++j) s += p[idx[(size_t)t * k + j]];
        for (int j = 0; j < k; ++j) gates[(size_t)t * k + j] = p[idx[(size_t)t * k + j]] / s;
    }
    free(p);
    free(taken);
}

/* Group the T*k assignments a = t*k + j by expert with a stable counting sort:
 * counts[e], offsets[e] (exclusive prefix sums, offsets[E] = T*k),
 * perm[row] = a (rows expert-major, then ascending a), inv_perm[a] = row, and
 * the ascending list of experts with at least one assignment (returns its
 * length). */
int orc_permute(const int32_t* idx, int T, int E, int k, int32_t* counts, int32_t* offsets,
                int32_t* perm, int32_t* inv_perm, int32_t* uniq) {
    int n = T * k;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int a = 0; a < n; ++a) counts[idx[a]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* fill = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    for (int a = 0; a < n; ++a) {
        int e = idx[a];
        int row = offsets[e] + fill[e]++;
        perm[row] = a;
        inv_perm[a] = row;
    }
    free(fill);
    int nu = 0;
    for (int e = 0; e < E; ++e) if (counts[e] > 0) uniq[nu++] = e;
    return nu;
}

/* ------------------------------------------------------------------------- */
/* LRU expert cache                                                          */
/* ------------------------------------------------------------------------- */

/* One global pool of S slots shared by all L layers. table[l*E + e] is the slot
 * holding expert e of layer l, or -1; owner[s] is the key held by slot s, or -1;
 * stamp[s] orders slots by recency (0 = never filled, older first).
 *
 * A batch touches the sorted, distinct experts members[0..n) of one layer at
 * clock c = ++*clock: member p gets stamp c*65536 + p. Hits only restamp. The
 * misses take, in ascending member order, the slots with the smallest
 * (stamp, slot index) among slots that hold neither a member of this batch nor
 * one of the keys in protect[0..n_protect). This is a textbook LRU serving the
 * batch with its members pinned: misses in ascending order take free slots
 * lowest index first, then the least recently used unpinned entry, and all
 * members are then refreshed in ascending order (so free, never-filled slots,
 * stamp 0, go before any filled one). Events are written in member order: expert, hit flag,
 * slot, evicted key (-1 if the slot was empty).
 * Returns the number of misses, or -1 if there are not enough slots. */
int orc_lru_batch(int L, int E, int S, int32_t* table, int32_t* owner, uint64_t* stamp,
                  uint64_t* clock, int layer, const int32_t* members, int n,
                  const int32_t* protect, int n_protect,
                  int32_t* ev_expert, int32_t* ev_hit, int32_t* ev_slot, int32_t* ev_evicted) {
    (void)L;
    unsigned char* blocked = (unsigned char*)calloc((size_t)S, 1);
    for (int p = 0; p < n; ++p) {
        int s = table[(size_t)layer * E + members[p]];
        if (s >= 0) blocked[s] = 1;
    }
    for (int q = 0; q < n_protect; ++q) {
        int s = table[protect[q]];
        if (s >= 0) blocked[s] = 1;
    }
    int misses = 0, free_slots = 0;
    for (int p = 0; p < n; ++p) if (table[(size_t)layer * E + members[p]] < 0) misses++;
    for (int s = 0; s < S; ++s) if (!blocked[s]) free_slots++;
    if (misses > free_slots) { free(blocked); return -1; }
    uint64_t c = ++*clock;
    for (int p = 0; p < n; ++p) {
        int32_t key = layer * E + members[p];
        int s = table[key];
        ev_expert[p] = members[p];
        if (s >= 0) {
            stamp[s] = c * 65536u + (uint64_t)p;
            ev_hit[p] = 1; ev_slot[p] = s; ev_evicted[p] = -1;
            continue;
        }
        int best = -1;
        for (int v = 0; v < S; ++v) {
            if (blocked[v]) continue;
            if (best < 0 || stamp[v] < stamp[best]) best = v;
        }
        blocked[best] = 1;
        int32_t old = owner[best];
        if (old >= 0) table[old] = -1;
        owner[best] = key;
        table[key] = best;
        stamp[best] = c * 65536u + (uint64_t)p;
        ev_hit[p] = 0; ev_slot[p] = best; ev_evicted[p] = old;
    }
    free(blocked);
    return misses;
}

/* ------------------------------------------------------------------------- */
/* Experts and the layer                                                     */
/* ------------------------------------------------------------------------- */

static float dot(const float* a, const float* b, int n) {
    float s = 0.0f;
    for (int i = 0; i < n; ++i) s = s + a[i] * b[i];
    return s;
}

/* SwiGLU expert: y = W_down (act(W_gate x) * (W_up x)), act(z) = z / (1 + e^-z)
 * (SiLU), or act(z) = z when mode == 1 (the linear stand-in used by the
 * closed-form tests). Wg, Wu: [I, H]; Wd: [H, I]. h receives the I values of
 * the intermediate (may be NULL). */
void orc_expert_ffn(const float* x, const float* Wg, const float* Wu, const float* Wd,
                    int H, int I, int mode, float* y, float* h_out) {
    float* h = (float*)malloc(sizeof(float) * (size_t)I);
    for (int i = 0; i < I; ++i) {
        float g = dot(Wg + (size_t)i * H, x, H);
        float u = dot(Wu + (size_t)i * H, x, H);
        float a = mode == 1 ? g : g / (1.0f + expf(-g));
        h[i] = a * u;
    }
    for (int r = 0; r < H; ++r) y[r] = dot(Wd + (size_t)r * I, h, I);
    if (h_out) memcpy(h_out, h, sizeof(float) * (size_t)I);
    free(h);
}

/* Output of the layer for the tokens in toks[0..nt): for token t,
 * out = sum over j = 0..k-1 (in that order) of gates[t,j] * expert_{idx[t,j]}(x_t),
 * plus, unweighted, each always-on shared expert. Wg/Wu/Wd[e] are the
 * dequantised weights of expert e (e < E routed, E.. shared); a routed entry
 * may be NULL when no selected token uses it. out row i belongs to toks[i]. */
void orc_layer_tokens(const float* x, int H, int I, int E, int n_shared, int k, int mode,
                      const int32_t* idx, const float* gates,
                      const float* const* Wg, const float* const* Wu, const float* const* Wd,
                      const int32_t* toks, int nt, float* out) {
    float* y = (float*)malloc(sizeof(float) * (size_t)H);
    for (int i = 0; i < nt; ++i) {
        int t = toks[i];
        const float* xt = x + (size_t)t * H;
        float* o = out + (size_t)i * H;
        for (int r = 0; r < H; ++r) o[r] = 0.0f;
        for (int j = 0; j < k; ++j) {
            int e = idx[(size_t)t * k + j];
            float g = gates[(size_t)t * k + j];
            orc_expert_ffn(xt, Wg[e], Wu[e], Wd[e], H, I, mode, y, NULL);
            for (int r = 0; r < H; ++r) o[r] = o[r] + g * y[r];
        }
        for (int s = 0; s < n_shared; ++s) {
            orc_expert_ffn(xt, Wg[E + s], Wu[E + s], Wd[E + s], H, I, mode, y, NULL);
            for (int r = 0; r < H; ++r) o[r] = o[r] + y[r];
        }
    }
    free(y);
}

/* The combine step of orc_layer_tokens on its own, for callers that computed
 * the expert outputs separately (one expert at a time over many tokens):
 * out = sum over j = 0..k-1 (in that order) of gates[j] * y[j], then plus,
 * unweighted, y[k + s] for each shared expert s. y holds k + n_shared rows of
 * H floats. Same operations, in the same order, as orc_layer_tokens. */
void orc_combine(int H, int k, int n_shared, const float* gates, const float* const* y, float* out) {
    for (int r = 0; r < H; ++r) out[r] = 0.0f;
    for (int j = 0; j < k; ++j)
        for (int r = 0; r < H; ++r) out[r] = out[r] + gates[j] * y[j][r];
    for (int s = 0; s < n_shared; ++s)
        for (int r = 0; r < H; ++r) out[r] = out[r] + y[k + s][r];
}

/* ------------------------------------------------------------------------- */
/* Activation quantisers (for the tolerance study of block-scaled MMA)       */
/* ------------------------------------------------------------------------- */
/* A block-scaled tensor-core MMA (OCP MX formats, NVFP4) multiplies two
 * narrow operands, so the activations would have to be quantised on the fly.
 * These functions define that quantisation; orc_expert_ffn_q evaluates an
 * expert with it, so that its distance from orc_expert_ffn can be measured.
 * Nothing in the layer as specified uses them. */

/* nearest E4M3 (FN) value, ties to the even code, saturating at +-448 */
float orc_e4m3_rne(float v) {
    float a = fabsf(v);
    if (a >= 448.0f) a = 448.0f;
    else {
        int e;
        frexpf(a, &e);                   /* a = f * 2^e, f in [0.5, 1) */
        int ue = e - 1;                  /* a in [2^ue, 2^(ue+1)) */
        if (ue < -6) ue = -6;            /* subnormals share the spacing of 2^-6 */
        float q = ldexpf(1.0f, ue - 3);  /* 3 mantissa bits */
        a = rintf(a / q) * q;            /* rintf: ties to even under the default mode */
        if (a > 448.0f) a = 448.0f;
    }
    return v < 0 ? -a : a;
}

/* nearest E2M1 value, ties to the even code, saturating at +-6:
 * grid 0, 0.5, 1, 1.5, 2, 3, 4, 6 (codes 0..7; even codes 0, 1, 2, 4) */
float orc_e2m1_rne(float v) {
    static const float grid[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    float a = fabsf(v), best = 0.0f;
    int bc = 0;
    for (int c = 0; c < 8; ++c) {
        float d = fabsf(a - grid[c]), db = fabsf(a - best);
        if (d < db || (d == db && (c & 1) == 0 && (bc & 1) == 1)) {
            best = grid[c];
            bc = c;
        }
    }
    return v < 0 ? -best : best;
}

/* kind 1, MXFP8 (OCP MX v1.0, E4M3 elements): blocks of 32 consecutive
 * elements share X = 2^(floor(log2 amax) - 8), 8 being E4M3's largest
 * exponent; each element becomes X * e4m3_rne(x / X) (values above 448 X
 * saturate, as the specification allows). An all-zero block stays zero.
 * kind 2, NVFP4: g = amax(x) / (448 * 6) over the vector; blocks of 16 share
 * s = e4m3_rne(amax_blk / (6 g)); each element becomes
 * e2m1_rne(x / (s g)) * s * g. n is a multiple of the block size. */
void orc_quant_act(int kind, const float* x, int n, float* out) {
    if (kind == 1) {
        for (int b = 0; b < n; b += 32) {
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[b + i]));
            if (amax == 0.0f) {
                for (int i = 0; i < 32; ++i) out[b + i] = 0.0f;
                continue;
            }
            int e;
            frexpf(amax, &e);
            float X = ldexpf(1.0f, (e - 1) - 8);
            for (int i = 0; i < 32; ++i) out[b + i] = orc_e4m3_rne(x[b + i] / X) * X;
        }
    } else {
        float amax = 0.0f;
        for (int i = 0; i < n; ++i) amax = fmaxf(amax, fabsf(x[i]));
        if (amax == 0.0f) {
            for (int i = 0; i < n; ++i) out[i] = 0.0f;
            return;
        }
        float g = amax / (448.0f * 6.0f);
        for (int b = 0; b < n; b += 16) {
            float ab = 0.0f;
            for (int i = 0; i < 16; ++i) ab = fmaxf(ab, fabsf(x[b + i]));
            float sc = orc_e4m3_rne(ab / (6.0f * g));
            float d = sc * g;
            for (int i = 0; i < 16; ++i) out[b + i] = d == 0.0f ? 0.0f : orc_e2m1_rne(x[b + i] / d) * d;
        }
    }
}

/* orc_expert_ffn with the activations quantised by orc_quant_act(kind): x
 * before gate/up, h before down (the two operands a block-scaled MMA would
 * take in a narrow format) */
void orc_expert_ffn_q(const float* x, const float* Wg, const float* Wu, const float* Wd,
                      int H, int I, int mode, int kind, float* y) {
    float* xq = (float*)malloc(sizeof(float) * (size_t)H);
    float* h = (float*)malloc(sizeof(float) * (size_t)I);
    float* hq = (float*)malloc(sizeof(float) * (size_t)I);
    orc_quant_act(kind, x, H, xq);
    for (int i = 0; i < I; ++i) {
        float g = dot(Wg + (size_t)i * H, xq, H);
        float u = dot(Wu + (size_t)i * H, xq, H);
        float a = mode == 1 ? g : g / (1.0f + expf(-g));
        h[i] = a * u;
    }
    orc_quant_act(kind, h, I, hq);
    for (int r = 0; r < H; ++r) y[r] = dot(Wd + (size_t)r * I, hq, I);
    free(xq);
    free(h);
    free(hq);
}

/* ------------------------------------------------------------------------- */
/* Resizing the pool at a safe point                                         */
/* ------------------------------------------------------------------------- */

typedef struct {
    uint64_t stamp;
    int32_t slot;
} orc_slot_age;

static int orc_by_recency(const void* a, const void* b) {
    const orc_slot_age* x = (const orc_slot_age*)a;
    const orc_slot_age* y = (const orc_slot_age*)b;
    if (x->stamp != y->stamp) return x->stamp > y->stamp ? -1 : 1; /* most recent first */
    return x->slot < y->slot ? -1 : (x->slot > y->slot);
}

/* Resize the pool from S_old to S_new slots at a safe point, keeping the most
 * recently used experts (the cache is "resized and rebuilt at the scheduler's
 * safe points" on the freetoken.wiki architecture page; the pages do not say
 * which experts survive, so the reading here keeps the LRU order):
 *  - the min(S_new, resident) cached experts with the largest stamps stay;
 *  - a kept expert whose slot is below S_new keeps that slot; the other kept
 *    experts move, in ascending order of their old slot, to the lowest slots
 *    below S_new that hold no kept expert;
 *  - every other expert leaves the cache (its table entry becomes -1);
 *  - stamps move with their experts, free slots get stamp 0 and owner -1, and
 *    the clock is unchanged.
 * new_owner / new_stamp receive the S_new-slot state, table is updated in
 * place, and moved[s] (s < S_old) receives the new slot of old slot s's
 * expert, or -1 if it was dropped or empty. Returns the number kept. */
int orc_lru_resize(int L, int E, int S_old, int32_t* table, const int32_t* owner, const uint64_t* stamp,
                   int S_new, int32_t* new_owner, uint64_t* new_stamp, int32_t* moved) {
    (void)L;
    (void)E;
    orc_slot_age* res = (orc_slot_age*)malloc(sizeof(orc_slot_age) * (size_t)(S_old > 0 ? S_old : 1));
    int n = 0;
    for (int s = 0; s < S_old; ++s) {
        moved[s] = -1;
        if (owner[s] >= 0) {
            res[n].stamp = stamp[s];
            res[n].slot = s;
            n++;
        }
    }
    qsort(res, (size_t)n, sizeof(orc_slot_age), orc_by_recency);
    int keep = n < S_new ? n : S_new;
    unsigned char* kept = (unsigned char*)calloc((size_t)(S_old > 0 ? S_old : 1), 1);
    for (int i = 0; i < keep; ++i) kept[res[i].slot] = 1;
    for (int s = 0; s < S_new; ++s) {
        new_owner[s] = -1;
        new_stamp[s] = 0;
    }
    /* kept experts already below S_new stay where they are */
    for (int s = 0; s < S_old && s < S_new; ++s)
        if (kept[s]) moved[s] = s;
    /* the others fill the free slots below S_new, in ascending old-slot order */
    int hole = 0;
    for (int s = S_new; s < S_old; ++s) {
        if (!kept[s]) continue;
        while (hole < S_new && hole < S_old && kept[hole]) hole++;
        moved[s] = hole;
        hole++;
    }
    for (int s = 0; s < S_old; ++s) {
        if (owner[s] < 0) continue;
        if (moved[s] >= 0) {
            new_owner[moved[s]] = owner[s];
            new_stamp[moved[s]] = stamp[s];
            table[owner[s]] = moved[s];
        } else {
            table[owner[s]] = -1;
        }
    }
    free(res);
    free(kept);
    return keep;
}
