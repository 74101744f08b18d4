// Router (logits, softmax + top-k + renormalisation), permutation by expert and
// the device-side LRU expert cache of the routed MoE layer, fused into one
// launch per call.
//
// Follows "FreeToken量子化：MoE推論のセットアップガイド" (freetoken.wiki,
// architecture page): decode keeps a shared LRU over recently selected
// experts; a hit runs on the GPU, a miss is copied into the cache over PCIe;
// prefill streams the next layer's experts while the current layer computes
// when the cache has room. Summation order, tie-break and the batch LRU rule
// are fixed readings, stated at each step.
//
// k_route runs in two phases:
//  A (every CTA)  router logits in the fixed fp32 order. Decode (T <= 8, BF16
//                 or FP32 weights; FP4 / FP8 decode runs in the fused decode kernel):
//                 one warp per expert for all tokens, the activations are also
//                 reordered for the expert kernels. Prefill: one CTA per 8
//                 tokens over all experts, followed by that CTA's softmax/top-k.
//  B (the CTA that finishes last, found with a completion counter; nothing
//                 waits) decode top-k, per-expert counts and offsets, the stable
//                 permutation, the active-expert list, the LRU batch (and the
//                 prefill prefetch batch) and the call record the host reads.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "moe_internal.h"
#include "route_common.cuh"

namespace moe {

constexpr int kRouteThreads = 512;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kPrefillTokTile = 8;  // tokens per phase-A CTA (prefill)
constexpr int kPrefillEpw = 4;      // experts per warp per pass (prefill)

// --------------------------------------------------------------------------
// activation loads
// --------------------------------------------------------------------------

template <int ACT>
__device__ __forceinline__ float ld_act(const void* p, size_t i) {
    if constexpr (ACT == ACT_BF16) {
        uint16_t b = reinterpret_cast<const uint16_t*>(p)[i];
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    } else {
        return reinterpret_cast<const float*>(p)[i];
    }
}

// 8 consecutive activations starting at element i (i % 8 == 0)
template <int ACT>
__device__ __forceinline__ void ld_act8(const void* p, size_t i, float (&v)[8]) {
    if constexpr (ACT == ACT_BF16) {
        uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p) + i);
        uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[2 * j] = __uint_as_float(w[j] << 16);
            v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    } else {
        const float4* f = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + i);
        float4 a = f[0], b = f[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

// --------------------------------------------------------------------------
// activations -> bf16 in the device K-order (decode with BF16 weights), from
// the token rows already staged in shared memory: xs holds rows [t0, t0 + nt);
// work split over `nthr` threads starting at `tid`
// --------------------------------------------------------------------------

template <int ACT>
__device__ void xprep_rows(const unsigned char* xs, void* __restrict__ xh, int fmt, int H, int t0, int nt,
                           size_t tid, size_t nthr) {
    if (fmt != FMT_BF16) return;
    const int h4 = H / 4;
    const size_t n4 = static_cast<size_t>(nt) * h4;
    for (size_t idx = tid; idx < n4; idx += nthr) {
        const int t = static_cast<int>(idx / h4);
        const int p = 4 * static_cast<int>(idx % h4);   // device position
        const int j = p >> 7, w = p & 127, q = w >> 5, s = (w & 31) >> 2;
        const size_t src = static_cast<size_t>(t) * H + 128 * j + 16 * s + 4 * q;
        const float v0 = ld_act<ACT>(xs, src), v1 = ld_act<ACT>(xs, src + 1);
        const float v2 = ld_act<ACT>(xs, src + 2), v3 = ld_act<ACT>(xs, src + 3);
        __nv_bfloat162 a = __floats2bfloat162_rn(v0, v1), b = __floats2bfloat162_rn(v2, v3);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t*>(&a);
        o.y = *reinterpret_cast<uint32_t*>(&b);
        *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(xh) + static_cast<size_t>(t0 + t) * H + p) = o;
    }
}

// global -> shared copy of n 16-byte vectors; each thread issues up to 8 loads
// before its first store, so the copy costs one memory round trip per 8 vectors
__device__ __forceinline__ void copy_g2s(unsigned char* dst, const unsigned char* src, size_t n) {
    constexpr int kB = 8;
    const size_t nthr = blockDim.x;
    for (size_t i0 = threadIdx.x; i0 < n; i0 += nthr * kB) {
        uint4 v[kB];
#pragma unroll
        for (int i = 0; i < kB; ++i) {
            const size_t k = i0 + i * nthr;
            if (k < n) v[i] = __ldg(reinterpret_cast<const uint4*>(src) + k);
        }
#pragma unroll
        for (int i = 0; i < kB; ++i) {
            const size_t k = i0 + i * nthr;
            if (k < n) reinterpret_cast<uint4*>(dst)[k] = v[i];
        }
    }
}

// --------------------------------------------------------------------------
// router logits of one warp in the fixed summation order
//   H is cut into 8-element chunks; chunk c belongs to lane c mod 32, which
//   accumulates its chunks in increasing h with fused multiply-adds from 0;
//   the 32 lane sums then combine by xor-butterfly (o = 16, 8, 4, 2, 1).
// EPW experts (rows e0.. of router_w, e >= E contributes nothing) x nt tokens
// whose rows sit in shared memory; every lane returns the finished sums. Each
// lane first loads NB of its chunks (all independent), then runs its FMA
// chain over them in order, so a batch costs one memory round trip.
// --------------------------------------------------------------------------

__device__ __forceinline__ uint64_t route_gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

template <int ACT>
struct RawChunk {
    uint4 v[ACT == ACT_BF16 ? 1 : 2];
};

template <int ACT>
__device__ __forceinline__ void ld_chunk(const void* p, size_t i, RawChunk<ACT>& r) {
    const uint4* q = reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned char*>(p) +
                                                    i * (ACT == ACT_BF16 ? 2 : 4));
    r.v[0] = __ldg(q);
    if constexpr (ACT != ACT_BF16) r.v[1] = __ldg(q + 1);
}

template <int ACT>
__device__ __forceinline__ void cvt_chunk(const RawChunk<ACT>& r, float (&v)[8]) {
    if constexpr (ACT == ACT_BF16) {
        const uint32_t w[4] = {r.v[0].x, r.v[0].y, r.v[0].z, r.v[0].w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[2 * j] = __uint_as_float(w[j] << 16);
            v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    } else {
        const uint32_t w[8] = {r.v[0].x, r.v[0].y, r.v[0].z, r.v[0].w, r.v[1].x, r.v[1].y, r.v[1].z, r.v[1].w};
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(w[j]);
    }
}

// the first batch of a warp's router chunks (lane's chunks lane, lane+32, ...)
template <int ACT, int EPW, int NB>
__device__ __forceinline__ void router_batch(const void* __restrict__ router_w, int H, int E, int e0, int cb,
                                             RawChunk<ACT> (&raw)[NB][EPW]) {
    const int nchunk = H / 8;
#pragma unroll
    for (int i = 0; i < NB; ++i) {
        const int c = cb + 32 * i;
#pragma unroll
        for (int e = 0; e < EPW; ++e)
            if (c < nchunk && e0 + e < E) ld_chunk<ACT>(router_w, static_cast<size_t>(e0 + e) * H + 8 * c, raw[i][e]);
    }
}

// pre: this lane's first batch, already loaded with router_batch (or null);
// XT: element type of the token rows in shared memory
template <int ACT, int EPW, int NB, int XT = ACT>
__device__ __forceinline__ void warp_logits(const void* __restrict__ router_w, const unsigned char* xs, int H,
                                            int E, int e0, int nt, int lane, float (&acc)[EPW][8],
                                            const RawChunk<ACT> (*pre)[EPW] = nullptr) {
#pragma unroll
    for (int e = 0; e < EPW; ++e)
#pragma unroll
        for (int t = 0; t < 8; ++t) acc[e][t] = 0.0f;
    const int nchunk = H / 8;
    for (int cb = lane; cb < nchunk; cb += 32 * NB) {
        RawChunk<ACT> raw[NB][EPW];
        if (pre && cb == lane) {
#pragma unroll
            for (int i = 0; i < NB; ++i)
#pragma unroll
                for (int e = 0; e < EPW; ++e) raw[i][e] = pre[i][e];
        } else {
            router_batch<ACT, EPW, NB>(router_w, H, E, e0, cb, raw);
        }
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            const int c = cb + 32 * i;
            if (c >= nchunk) break;
            float wv[EPW][8];
#pragma unroll
            for (int e = 0; e < EPW; ++e) {
                if (e0 + e < E) {
                    cvt_chunk<ACT>(raw[i][e], wv[e]);
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) wv[e][j] = 0.0f;
                }
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                if (t < nt) {
                    float xv[8];
                    ld_act8<XT>(xs, static_cast<size_t>(t) * H + 8 * c, xv);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
#pragma unroll
                        for (int e = 0; e < EPW; ++e) acc[e][t] = __fmaf_rn(xv[j], wv[e][j], acc[e][t]);
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < EPW; ++e)
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            float v = acc[e][t];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
            acc[e][t] = v;
        }
}

// Fixed-order logits of two (token, expert) pairs at once (b optional), the
// same operations in the same order as warp_logits<ACT, 1, 8> with one token:
// lane l accumulates chunks l, l + 32, ... in increasing order, then the
// partials are combined by xor-halving. Both rows' loads are issued together.
template <int ACT>
__device__ __forceinline__ void pair_logits(const void* __restrict__ router_w, const unsigned char* xs, int H, int ea,
                                            int ta, int eb, int tb, bool has_b, int lane, float& la, float& lb) {
    constexpr int NB = 8;
    float sa = 0.0f, sb = 0.0f;
    const int nchunk = H / 8;
    for (int cb = lane; cb < nchunk; cb += 32 * NB) {
        RawChunk<ACT> ra[NB], rb[NB];
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            const int c = cb + 32 * i;
            if (c < nchunk) {
                ld_chunk<ACT>(router_w, static_cast<size_t>(ea) * H + 8 * c, ra[i]);
                if (has_b) ld_chunk<ACT>(router_w, static_cast<size_t>(eb) * H + 8 * c, rb[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            const int c = cb + 32 * i;
            if (c >= nchunk) break;
            float wv[8], xv[8];
            cvt_chunk<ACT>(ra[i], wv);
            ld_act8<ACT>(xs, static_cast<size_t>(ta) * H + 8 * c, xv);
#pragma unroll
            for (int j = 0; j < 8; ++j) sa = __fmaf_rn(xv[j], wv[j], sa);
            if (has_b) {
                cvt_chunk<ACT>(rb[i], wv);
                ld_act8<ACT>(xs, static_cast<size_t>(tb) * H + 8 * c, xv);
#pragma unroll
                for (int j = 0; j < 8; ++j) sb = __fmaf_rn(xv[j], wv[j], sb);
            }
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        sa = __fadd_rn(sa, __shfl_xor_sync(0xffffffffu, sa, o));
        sb = __fadd_rn(sb, __shfl_xor_sync(0xffffffffu, sb, o));
    }
    la = sa;
    lb = sb;
}

// phase-B shared memory; the work area follows it
struct RouteShared {
    int32_t cnt[kMaxExperts];
    int32_t off[kMaxExperts];
    int32_t members[kMaxExperts];
    int32_t e2u[kMaxExperts];
    int32_t trow[2][kMaxExperts];  // LRU table rows of this layer and of layer+1
    int32_t topk[kDecodeMaxT * kMaxTopK];
    float gates[kDecodeMaxT * kMaxTopK];
    int32_t scan_a[kRouteWarps], scan_b[kRouteWarps];
    int32_t nu;
    unsigned long long tks[kDecodeMaxT][32];  // top-k scratch of token t's warp
    LruShared lru;
};

constexpr size_t kRouteSharedBytes = (sizeof(RouteShared) + 15) / 16 * 16;
// pools up to this many slots keep their stamps and owners in shared memory during phase B
constexpr int kLruCachedSlots = 4096;

// block-wide exclusive scan of two ints per thread (sum over threads in tid order);
// returns the exclusive prefixes and the totals
__device__ __forceinline__ void block_scan2(int va, int vb, int& ea, int& eb, int& ta, int& tb, int32_t* sa,
                                            int32_t* sb) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    int ia = va, ib = vb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int ya = __shfl_up_sync(0xffffffffu, ia, o);
        const int yb = __shfl_up_sync(0xffffffffu, ib, o);
        if (lane >= o) { ia += ya; ib += yb; }
    }
    if (lane == 31) { sa[warp] = ia; sb[warp] = ib; }
    __syncthreads();
    int wa = 0, wb = 0;
    ta = 0; tb = 0;
    for (int w = 0; w < nwarps; ++w) {
        if (w < warp) { wa += sa[w]; wb += sb[w]; }
        ta += sa[w];
        tb += sb[w];
    }
    ea = wa + ia - va;
    eb = wb + ib - vb;
    __syncthreads();
}

// layout of the work area behind RouteShared: [keys | per-warp counts] (a union:
// the permutation is done before the cache lookup), then the stamp and owner
// copies of a small pool
__host__ __device__ inline size_t route_area_union(int S, int E) {
    size_t P = 1;
    while (P < static_cast<size_t>(S)) P <<= 1;
    const size_t keys = P * 8, wc = static_cast<size_t>(kRouteWarps) * E * 4;
    return (keys > wc ? keys : wc);
}

__host__ __device__ inline size_t route_area_bytes(int S, int E) {
    return route_area_union(S, E) + (S <= kLruCachedSlots ? static_cast<size_t>(S) * 12 : 0);
}

// --------------------------------------------------------------------------
// phase B: everything after the logits (and, for prefill, the top-k)
// --------------------------------------------------------------------------

// bmark (trace only, prefill): times of the steps below, written by thread 0
__device__ void route_phase_b(const CallArgs& a, RouteShared& rs, unsigned char* area, bool decode,
                              unsigned long long* bmark) {
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
    auto bm = [&](int i) {
        if (bmark && tid == 0) bmark[i] = route_gtimer();
    };
    const int T = a.T, E = a.E, k = a.k, n = T * k, S = a.S;
    CallInfo* info = a.info;
    LruShared& sm = rs.lru;
    // start every independent load of the cache state now: one round trip
    const bool pf_possible = a.prefetch && T > kDecodeMaxT && a.layer + 1 < a.L;
    const bool cached = S <= kLruCachedSlots;
    LruView lv;
    lv.bind(a);
    lv.trow0 = rs.trow[0];
    lv.trow1 = pf_possible ? rs.trow[1] : nullptr;
    unsigned long long* st_s = reinterpret_cast<unsigned long long*>(area + route_area_union(S, E));
    int32_t* own_s = reinterpret_cast<int32_t*>(st_s + S);
    lv.st_s = cached ? st_s : nullptr;
    lv.own_s = cached ? own_s : nullptr;
    {
        // every thread issues all its loads before its first store
        constexpr int kB = 8;
        const unsigned long long clock = tid == 0 ? *a.clock : 0ull;
        for (int e0 = tid; e0 < E; e0 += nthr * 2) {
            int32_t v[2][2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int e = e0 + i * nthr;
                if (e < E) {
                    v[i][0] = a.table[a.layer * E + e];
                    v[i][1] = pf_possible ? a.table[(a.layer + 1) * E + e] : -1;
                }
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int e = e0 + i * nthr;
                if (e < E) {
                    rs.trow[0][e] = v[i][0];
                    rs.trow[1][e] = v[i][1];
                }
            }
        }
        if (cached)
            for (int s0 = tid; s0 < S; s0 += nthr * kB) {
                unsigned long long sv[kB];
                int32_t ov[kB];
#pragma unroll
                for (int i = 0; i < kB; ++i) {
                    const int s = s0 + i * nthr;
                    if (s < S) {
                        sv[i] = a.stamp[s];
                        ov[i] = a.owner[s];
                    }
                }
#pragma unroll
                for (int i = 0; i < kB; ++i) {
                    const int s = s0 + i * nthr;
                    if (s < S) {
                        st_s[s] = sv[i];
                        own_s[s] = ov[i];
                    }
                }
            }
        if (tid == 0) sm.clock = clock;
    }
    // decode: top-k of every token (one warp each)
    if (decode) {
        if (warp < T) {
            int sel;
            float g;
            warp_topk<true>(a.logits + static_cast<size_t>(warp) * E, E, k, lane, sel, g, rs.tks[warp]);
            if (lane < k) {
                rs.topk[warp * k + lane] = sel;
                rs.gates[warp * k + lane] = g;
                a.topk[warp * k + lane] = sel;
                a.gates[warp * k + lane] = g;
            }
        }
        for (int i = tid; i < (E + a.n_shared) * kDecodeMaxT; i += nthr) a.tok_row[i] = -1;
    }
    bm(0);
    if (decode) {
        for (int e = tid; e < E; e += nthr) rs.cnt[e] = 0;
    } else {
        // the routing CTAs added their counts; reset the accumulator for the next call
        for (int e = tid; e < E; e += nthr) {
            rs.cnt[e] = __ldcg(a.cacc + e);
            a.cacc[e] = 0;
        }
    }
    __syncthreads();
    auto topk_at = [&](int i) -> int { return rs.topk[i]; };
    auto gate_at = [&](int i) -> float { return rs.gates[i]; };
    if (decode) {
        for (int i = tid; i < n; i += nthr) atomicAdd(&rs.cnt[topk_at(i)], 1);
        __syncthreads();
    }
    // offsets (exclusive) and the active list: each thread owns `per` consecutive experts
    const int per = (E + nthr - 1) / nthr;
    {
        int sc = 0, sz = 0;
        for (int i = 0; i < per; ++i) {
            const int e = tid * per + i;
            if (e < E) { sc += rs.cnt[e]; sz += rs.cnt[e] > 0; }
        }
        int ec, ez, tc, tz;
        block_scan2(sc, sz, ec, ez, tc, tz, rs.scan_a, rs.scan_b);
        for (int i = 0; i < per; ++i) {
            const int e = tid * per + i;
            if (e < E) {
                const int c = rs.cnt[e];
                rs.off[e] = ec;
                rs.e2u[e] = c > 0 ? ez : -1;
                a.offsets[e] = ec;
                a.counts[e] = c;
                a.e2u[e] = c > 0 ? ez : -1;
                if (c > 0) {
                    rs.members[ez] = e;
                    a.act_expert[ez] = e;
                    a.act_row0[ez] = ec;
                    a.act_cnt[ez] = c;
                    if (decode) {
                        DecExpert* d = reinterpret_cast<DecExpert*>(a.dplan + kDecPlanHeader) + ez;
                        d->row0 = ec;
                        d->cnt = c;
                    }
                }
                ec += c;
                ez += c > 0;
            }
        }
        if (tid == 0) {
            a.offsets[E] = tc;
            rs.nu = tz;
            *a.n_uniq = tz;
        }
    }
    __syncthreads();
    bm(1);
    // prefill: the rows of expert e before routing CTA b (the sum of e's count
    // column over earlier CTAs) are summed by k_perm_rows, one CTA per column
    // decode: stable permutation, warp w owns the contiguous assignment range [w*chunk, (w+1)*chunk)
    if (decode) {
        int32_t* wc = reinterpret_cast<int32_t*>(area);  // [kRouteWarps][E]
        const int nwarps = nthr >> 5;
        const int chunk = (n + nwarps - 1) / nwarps;
        const int a0 = min(n, warp * chunk), a1 = min(n, a0 + chunk);
        for (int i = tid; i < nwarps * E; i += nthr) wc[i] = 0;
        if (decode) {
            // plan token tables of the routed experts: empty until the permutation fills them
            DecExpert* dp = reinterpret_cast<DecExpert*>(a.dplan + kDecPlanHeader);
            for (int i = tid; i < rs.nu * kDecodeMaxT; i += nthr) {
                DecExpert& d = dp[i / kDecodeMaxT];
                d.tok[i % kDecodeMaxT] = -1;
                d.hrow[i % kDecodeMaxT] = -1;
                d.gate[i % kDecodeMaxT] = 0.0f;
            }
        }
        __syncthreads();
        for (int i = a0 + lane; i < a1; i += 32) atomicAdd(&wc[warp * E + topk_at(i)], 1);
        __syncthreads();
        for (int e = tid; e < E; e += nthr) {
            int run = rs.off[e];
            for (int w = 0; w < nwarps; ++w) {
                const int c = wc[w * E + e];
                wc[w * E + e] = run;
                run += c;
            }
        }
        __syncthreads();
        const uint32_t lt = (1u << lane) - 1u;
        for (int base = a0; base < a1; base += 32) {
            const int i = base + lane;
            const bool valid = i < a1;
            const int e = valid ? topk_at(i) : -1 - lane;
            const uint32_t peers = __match_any_sync(0xffffffffu, e);
            int row = 0;
            if (valid) row = wc[warp * E + e] + __popc(peers & lt);
            __syncwarp();
            if (valid && lane == 31 - __clz(peers)) wc[warp * E + e] += __popc(peers);
            __syncwarp();
            if (valid) {
                const int t = i / k;
                a.perm[row] = i;
                a.inv_perm[i] = row;
                a.row_tok[row] = t;
                a.row_gate[row] = gate_at(i);
                if (decode) {
                    const int u = rs.e2u[e];
                    a.tok_row[u * kDecodeMaxT + t] = row;
                    DecExpert& d = reinterpret_cast<DecExpert*>(a.dplan + kDecPlanHeader)[u];
                    d.tok[row - rs.off[e]] = t;
                    d.gate[row - rs.off[e]] = gate_at(i);
                    d.hrow[t] = row;
                }
            }
        }
    }
    __syncthreads();
    bm(2);
    // LRU: demand batch of this layer's experts
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(area);
    const int nu = rs.nu;
    const int m = lru_batch(lv, sm, keys, a.layer, rs.members, nu, nullptr, 0, 0);
    bm(3);
    if (m < 0) {
        if (tid == 0) {
            info->n_uniq = nu;
            info->n_hit = info->n_miss = info->n_pf = info->n_pf_hit = info->n_pf_miss = 0;
            info->n_events = 0;
            info->dev_err = *reinterpret_cast<volatile int32_t*>(a.dev_err);
            info->device_copied = 0;
            info->copy_ns = 0;
            info->status = -4;  // MOE_ERR_CAPACITY
            *a.n_active = 0;
            if (decode) *reinterpret_cast<int32_t*>(a.dplan) = 0;
            if (a.self_release) *a.ready = a.seq;
            __threadfence_system();
            info->done = a.seq;
        }
        return;
    }
    for (int p = tid; p < nu; p += nthr) {
        const int s = sm.member_slot[p];
        a.act_ptr[p] = a.pool + static_cast<size_t>(s) * a.lay.bytes;
        a.act_slot[p] = s;
        if (decode) reinterpret_cast<DecExpert*>(a.dplan + kDecPlanHeader)[p].ptr = a.act_ptr[p];
    }
    for (int p = tid; p < nu; p += nthr) {
        info->ev_layer[p] = a.layer;
        info->ev_expert[p] = rs.members[p];
        info->ev_hit[p] = 1;
        info->ev_slot[p] = sm.member_slot[p];
        info->ev_evicted[p] = sm.member_old[p];
        info->ev_prefetch[p] = 0;
    }
    __syncthreads();
    for (int r = tid; r < m; r += nthr) {
        const int p = sm.miss_p[r];
        info->ev_hit[p] = 0;
        info->miss_layer[r] = a.layer;
        info->miss_expert[r] = rs.members[p];
        info->miss_slot[r] = sm.member_slot[p];
    }
    __syncthreads();
    bm(4);
    int n_pf = 0, m_pf = 0;
    const bool do_pf = pf_possible && a.S >= nu + E;
    if (do_pf) {
        m_pf = lru_batch(lv, sm, keys, a.layer + 1, nullptr, E, rs.members, nu, a.layer);
        n_pf = E;
        if (m_pf < 0) { m_pf = 0; n_pf = 0; }  // cannot happen when S >= nu + E
        for (int p = tid; p < n_pf; p += nthr) {
            info->ev_layer[nu + p] = a.layer + 1;
            info->ev_expert[nu + p] = p;
            info->ev_hit[nu + p] = 1;
            info->ev_slot[nu + p] = sm.member_slot[p];
            info->ev_evicted[nu + p] = sm.member_old[p];
            info->ev_prefetch[nu + p] = 1;
        }
        __syncthreads();
        for (int r = tid; r < m_pf; r += nthr) {
            const int p = sm.miss_p[r];
            info->ev_hit[nu + p] = 0;
            info->miss_layer[m + r] = a.layer + 1;
            info->miss_expert[m + r] = p;
            info->miss_slot[m + r] = sm.member_slot[p];
        }
    }
    // shared experts: resident, after the routed ones in the active list
    for (int s = 0; s < a.n_shared; ++s) {
        const int u = nu + s;
        if (tid == 0) {
            a.act_expert[u] = E + s;
            a.act_row0[u] = T * k + s * T;
            a.act_cnt[u] = T;
            a.act_ptr[u] = a.shared_base + static_cast<size_t>(s) * a.lay.bytes;
            a.act_slot[u] = -(1 + a.layer * a.n_shared + s);
        }
        for (int t = tid; t < T; t += nthr) {
            a.row_tok[T * k + s * T + t] = t;
            a.row_gate[T * k + s * T + t] = 1.0f;
            if (decode) a.tok_row[u * kDecodeMaxT + t] = T * k + s * T + t;
        }
        if (decode && tid < kDecodeMaxT) {
            DecExpert& d = reinterpret_cast<DecExpert*>(a.dplan + kDecPlanHeader)[u];
            const int t = tid;
            d.tok[t] = t < T ? t : -1;
            d.hrow[t] = t < T ? T * k + s * T + t : -1;
            d.gate[t] = t < T ? 1.0f : 0.0f;
            if (t == 0) {
                d.ptr = a.shared_base + static_cast<size_t>(s) * a.lay.bytes;
                d.row0 = T * k + s * T;
                d.cnt = T;
            }
        }
    }
    if (decode && tid == 0) *reinterpret_cast<int32_t*>(a.dplan) = nu + a.n_shared;
    __syncthreads();
    bm(5);
    if (tid == 0) {
        *a.n_active = nu + a.n_shared;
        info->n_uniq = nu;
        info->n_hit = nu - m;
        info->n_miss = m;
        info->n_pf = n_pf;
        info->n_pf_hit = n_pf - m_pf;
        info->n_pf_miss = m_pf;
        info->n_events = nu + n_pf;
        info->dev_err = *reinterpret_cast<volatile int32_t*>(a.dev_err);
        info->device_copied = 0;  // this call's misses are the host's to copy
        info->copy_ns = 0;
        info->status = 0;
        if (a.self_release && m == 0) *a.ready = a.seq;
        __threadfence_system();
        info->done = a.seq;
    }
    bm(6);
}

// --------------------------------------------------------------------------
// the fused routing kernel
// --------------------------------------------------------------------------

template <int ACT, bool DECODE>
__global__ void __launch_bounds__(kRouteThreads) k_route(CallArgs a) {
    extern __shared__ __align__(16) unsigned char route_smem[];
    __shared__ int s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // trace only (prefill): first CTA entry, last phase-A finish, phase-B end in
    // the last slot of the per-call ring
    unsigned long long* rtr = (!DECODE && a.trace) ? a.trace + static_cast<size_t>(a.trace_ctas) * kTracePoints +
                                                        (kTraceCalls - 1) * 4
                                                  : nullptr;
    if (rtr && threadIdx.x == 0) atomicMin(rtr, static_cast<unsigned long long>(route_gtimer()));
    // trace only: the last CTA's phase-A steps in the two slots before it (it
    // runs in the last wave, after its SM has run routing CTAs already)
    unsigned long long* rsub = (rtr && blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) ? rtr - 8 : nullptr;
    if (rsub) rsub[0] = route_gtimer();
    const int T = a.T, E = a.E, H = a.H;
    const size_t esz = ACT == ACT_BF16 ? 2 : 4;
    // ---------------- phase A
    if constexpr (DECODE) {
        // warp w: expert blockIdx.x * 16 + w. Its first router chunks are loaded
        // before the x rows [T][H] are staged, so both share one round trip.
        constexpr int NB = ACT == ACT_BF16 ? 8 : 4;  // chunks per lane per round trip
        const int e0 = blockIdx.x * kRouteWarps + warp;
        RawChunk<ACT> pre[NB][1];
        router_batch<ACT, 1, NB>(a.router_w, H, E, e0, lane, pre);
        copy_g2s(route_smem, reinterpret_cast<const unsigned char*>(a.hidden), static_cast<size_t>(T) * H * esz / 16);
        __syncthreads();
        if (e0 < E) {
            float acc[1][8];
            warp_logits<ACT, 1, NB>(a.router_w, route_smem, H, E, e0, T, lane, acc, pre);
            if (lane < T) {
                float v = acc[0][0];
#pragma unroll
                for (int t = 1; t < 8; ++t) v = lane == t ? acc[0][t] : v;
                a.logits[static_cast<size_t>(lane) * E + e0] = v;
            }
        }
        xprep_rows<ACT>(route_smem, a.xh, a.fmt, H, 0, T, static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x,
                        static_cast<size_t>(gridDim.x) * blockDim.x);
    } else {
        // 8 tokens per CTA, all experts; logits [8][E] in shared memory, then
        // top-k, then this CTA's share of the permutation (ranks, counts)
        const int t0 = blockIdx.x * kPrefillTokTile;
        const int nt = min(kPrefillTokTile, T - t0);
        const int k = a.k;
        float* lg = reinterpret_cast<float*>(route_smem + static_cast<size_t>(kPrefillTokTile) * H * esz);
        int32_t* s_tk = reinterpret_cast<int32_t*>(lg + static_cast<size_t>(kPrefillTokTile) * E);
        int32_t* s_cnt = s_tk + kPrefillTokTile * kMaxTopK;
        unsigned long long* s_scr = reinterpret_cast<unsigned long long*>(
            route_smem + (reinterpret_cast<unsigned char*>(s_cnt + E) - route_smem + 7) / 8 * 8);
        float* lsel = reinterpret_cast<float*>(s_scr + kPrefillTokTile * 32);  // [8][E] logits the top-k reads
        float* wn = lsel + static_cast<size_t>(kPrefillTokTile) * E;          // [E] router row norms
        int32_t* cand = reinterpret_cast<int32_t*>(wn + E);                   // [8 E] (token << 16 | expert)
        copy_g2s(route_smem, reinterpret_cast<const unsigned char*>(a.hidden) + static_cast<size_t>(t0) * H * esz,
                 static_cast<size_t>(nt) * H * esz / 16);
        for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
        const bool tc = ACT == ACT_BF16 && a.tc_router;
        if (tc) {
            // The tensor cores' logits L~ differ from the fixed-order ones L by at
            // most B_te = H 2^-21 ||x_t|| ||w_e|| (each sum's rounding is below
            // H 2^-23 sum |x_h w_h| <= H 2^-23 ||x_t|| ||w_e||, with a factor 2 to
            // spare). The k-th largest of L~ - B is a lower bound of the k-th
            // largest L, so only experts with L~ + B reaching it can be selected:
            // those get their exact logits, the others -inf, and the top-k below
            // is the top-k of the exact logits.
            // E is a multiple of 32: the CTA's logit rows are whole 16-byte vectors
            const float4* src4 = reinterpret_cast<const float4*>(a.logits + static_cast<size_t>(t0) * E);
            for (int i0 = threadIdx.x; i0 < nt * E / 4; i0 += 4 * blockDim.x) {
                float4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (i0 + j * blockDim.x < nt * E / 4) v[j] = __ldcg(src4 + i0 + j * blockDim.x);
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (i0 + j * blockDim.x < nt * E / 4) reinterpret_cast<float4*>(lg)[i0 + j * blockDim.x] = v[j];
            }
            for (int e = threadIdx.x; e < E; e += blockDim.x) wn[e] = __ldcg(a.wnorm + e);
            if (threadIdx.x == 0) s_last = 0;  // candidate count (s_last is free until the hand-off)
        }
        __syncthreads();
        if (rsub) rsub[1] = route_gtimer();
        if (tc) {
            // trace only: warp 0's sub-steps (norm, bounds, top-k of the bounds, candidates)
            unsigned long long* csub = (rsub && lane == 0 && warp == 0) ? rsub - 8 : nullptr;
            if (warp < nt) {
                const int t = warp;
                const unsigned char* xr = route_smem + static_cast<size_t>(t) * H * esz;
                float ss = 0.0f;
                for (int c = lane; c < H / 8; c += 32) {
                    float xv[8];
                    ld_act8<ACT>(xr, 8 * c, xv);
#pragma unroll
                    for (int j = 0; j < 8; ++j) ss = __fmaf_rn(xv[j], xv[j], ss);
                }
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
                const float cb = ldexpf(static_cast<float>(H), -21) * sqrtf(ss) * (1.0f + 1.0f / 1024.0f);
                if (csub) csub[0] = route_gtimer();
                const float* lrow = lg + static_cast<size_t>(t) * E;
                float* orow = lsel + static_cast<size_t>(t) * E;
                for (int e = lane; e < E; e += 32) orow[e] = lrow[e] - cb * wn[e];
                __syncwarp();
                if (csub) csub[1] = route_gtimer();
                int sel;
                float gd;
                warp_topk<false>(orow, E, k, lane, sel, gd, s_scr + warp * 32);
                const float tau = orow[__shfl_sync(0xffffffffu, sel, k - 1)];
                __syncwarp();
                if (csub) csub[2] = route_gtimer();
                for (int e = lane; e < E; e += 32) {
                    if (lrow[e] + cb * wn[e] >= tau) cand[atomicAdd(&s_last, 1)] = (t << 16) | e;
                    orow[e] = -INFINITY;
                }
                if (csub) csub[3] = route_gtimer();
            }
            __syncthreads();
            if (rsub) rsub[2] = route_gtimer();
            const int ncand = s_last;
            if (rsub) rsub[7] = static_cast<unsigned long long>(ncand);
            // two candidates per warp and pass, their router rows in flight together
            for (int p = warp; p < ncand; p += 2 * kRouteWarps) {
                const int q = p + kRouteWarps;
                const bool has_b = q < ncand;
                const int ta = cand[p] >> 16, ea = cand[p] & 0xFFFF;
                const int tb = has_b ? cand[q] >> 16 : ta, eb = has_b ? cand[q] & 0xFFFF : ea;
                float la, lb;
                pair_logits<ACT>(a.router_w, route_smem, H, ea, ta, eb, tb, has_b, lane, la, lb);
                if (lane == 0) {
                    lsel[static_cast<size_t>(ta) * E + ea] = la;
                    if (has_b) lsel[static_cast<size_t>(tb) * E + eb] = lb;
                }
            }
            __syncthreads();
            if (rsub) rsub[3] = route_gtimer();
        }
        constexpr int kPass = kRouteWarps * kPrefillEpw;
        for (int eb = 0; eb < E && !tc; eb += kPass) {
            const int e0 = eb + warp * kPrefillEpw;
            if (e0 < E) {
                float acc[kPrefillEpw][8];
                warp_logits<ACT, kPrefillEpw, 1>(a.router_w, route_smem, H, E, e0, nt, lane, acc);
                if (lane == 0) {
#pragma unroll
                    for (int e = 0; e < kPrefillEpw; ++e)
#pragma unroll
                        for (int t = 0; t < 8; ++t)
                            if (t < nt && e0 + e < E) lg[t * E + e0 + e] = acc[e][t];
                }
            }
        }
        __syncthreads();
        if (warp < nt) {
            int sel;
            float g;
            warp_topk<false>((tc ? lsel : lg) + warp * E, E, k, lane, sel, g, s_scr + warp * 32);
            if (rsub) rsub[4] = route_gtimer();
            if (lane < k) {
                const size_t o = static_cast<size_t>(t0 + warp) * k + lane;
                a.topk[o] = sel;
                a.gates[o] = g;
                s_tk[warp * k + lane] = sel;
            }
        }
        __syncthreads();
        // ranks among this CTA's assignments to the same expert (ascending
        // assignment order), per-expert counts: the stable permutation then
        // puts assignment a at offsets[e] + (rows of e in earlier CTAs) + rank
        if (warp == 0) {
            const int na = nt * k;
            const uint32_t lt = (1u << lane) - 1u;
            for (int base = 0; base < na; base += 32) {
                const int i = base + lane;
                const bool valid = i < na;
                const int e = valid ? s_tk[i] : -1 - lane;
                const uint32_t peers = __match_any_sync(0xffffffffu, e);
                int r = 0;
                if (valid) r = s_cnt[e] + __popc(peers & lt);
                __syncwarp();
                if (valid && lane == 31 - __clz(peers)) s_cnt[e] += __popc(peers);
                __syncwarp();
                if (valid) a.lrank[static_cast<size_t>(t0) * k + i] = static_cast<int16_t>(r);
            }
        }
        __syncthreads();
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            const int c = s_cnt[e];
            a.cntT[static_cast<size_t>(e) * a.nb_max + blockIdx.x] = static_cast<int16_t>(c);
            if (c) atomicAdd(&a.cacc[e], c);
        }
    }
    // ---------------- hand-off: the last CTA to finish runs phase B
    __syncthreads();
    if (rsub) rsub[5] = route_gtimer();
    if (rtr && threadIdx.x == 0) atomicMax(rtr + 1, static_cast<unsigned long long>(route_gtimer()));
    if (threadIdx.x == 0) {
        __threadfence();
        const int prev = atomicAdd(a.route_done, 1);
        s_last = prev == static_cast<int>(gridDim.x) - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    RouteShared& rs = *reinterpret_cast<RouteShared*>(route_smem);
    // trace only: phase B's steps two ring slots before the phase-A marks
    route_phase_b(a, rs, route_smem + kRouteSharedBytes, DECODE, rtr ? rtr - 24 : nullptr);
    if (threadIdx.x == 0) *a.route_done = 0;
    if (rtr && threadIdx.x == 0) rtr[2] = route_gtimer();
}

// prefill: places every assignment of routing CTA b (8 tokens) at
// offsets[e] + rows of e in earlier CTAs + its rank among CTA b's assignments
// to e. The rows of e in earlier CTAs are the sum of e's count column over
// b' < b: a warp per assignment, 8 assignments per warp in flight at once.
__global__ void __launch_bounds__(256) k_perm_rows(CallArgs a) {
    constexpr int kPerWarp = 8;
    __shared__ int s_base[kPrefillTokTile * kMaxTopK];
    const int b = blockIdx.x, k = a.k;
    const int t0 = b * kPrefillTokTile, nt = min(kPrefillTokTile, a.T - t0);
    const int n = nt * k;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
    for (int i0 = warp * kPerWarp; i0 < n; i0 += nwarps * kPerWarp) {
        uint4 v[kPerWarp][2];
#pragma unroll
        for (int j = 0; j < kPerWarp; ++j) {
            const int i = i0 + j;
            const int16_t* col = i < n ? a.cntT + static_cast<size_t>(a.topk[t0 * k + i]) * a.nb_max : nullptr;
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // columns 256 h + 8 lane .. + 7 (nb <= 512 per pass)
                const int c0 = 256 * h + 8 * lane;
                v[j][h] = col && c0 < b ? __ldcg(reinterpret_cast<const uint4*>(col + c0)) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int j = 0; j < kPerWarp; ++j) {
            const int i = i0 + j;
            int sum = 0;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int c0 = 256 * h + 8 * lane;
                const uint32_t w[4] = {v[j][h].x, v[j][h].y, v[j][h].z, v[j][h].w};
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int x = static_cast<int>((q & 1) ? (w[q >> 1] >> 16) : (w[q >> 1] & 0xFFFFu));
                    sum += c0 + q < b ? x : 0;
                }
            }
            // columns past 512 (T > 4096): the rest of the row, one vector per lane per step
            const int16_t* col = i < n ? a.cntT + static_cast<size_t>(a.topk[t0 * k + i]) * a.nb_max : nullptr;
            for (int c0 = 512 + 8 * lane; col && c0 < b; c0 += 256) {
                const uint4 u = __ldcg(reinterpret_cast<const uint4*>(col + c0));
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int x = static_cast<int>((q & 1) ? (w[q >> 1] >> 16) : (w[q >> 1] & 0xFFFFu));
                    sum += c0 + q < b ? x : 0;
                }
            }
            sum = __reduce_add_sync(0xffffffffu, sum);
            if (lane == 0 && i < n) s_base[i] = sum;
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int asg = t0 * k + i;
        const int e = a.topk[asg];
        const int row = a.offsets[e] + s_base[i] + a.lrank[asg];
        a.perm[row] = asg;
        a.inv_perm[asg] = row;
        a.row_tok[row] = asg / k;
        a.row_gate[row] = a.gates[asg];
    }
}

// dynamic shared memory of one k_route launch
static size_t route_smem_bytes(const CallArgs& a, bool decode) {
    const size_t esz = a.act == ACT_BF16 ? 2 : 4;
    const size_t phase_a = decode ? static_cast<size_t>(a.T) * a.H * esz
                                  : static_cast<size_t>(kPrefillTokTile) * a.H * esz +
                                        static_cast<size_t>(kPrefillTokTile) * a.E * 4 +
                                        static_cast<size_t>(kPrefillTokTile) * kMaxTopK * 4 + static_cast<size_t>(a.E) * 4 +
                                        8 + static_cast<size_t>(kPrefillTokTile) * 32 * 8 +
                                        static_cast<size_t>(kPrefillTokTile) * a.E * 4 * 2 + static_cast<size_t>(a.E) * 4;
    return std::max(phase_a, kRouteSharedBytes + route_area_bytes(a.S, a.E));
}

// the opt-in per-block limit is 227 KB including static shared memory
size_t route_smem_limit() { return 226 * 1024; }

cudaError_t launch_route(const CallArgs& a, cudaStream_t s) {
    const bool decode = a.T <= kDecodeMaxT;
    const size_t smem = route_smem_bytes(a, decode);
    if (smem > route_smem_limit()) return cudaErrorInvalidValue;
    if (decode) {
        const int grid = (a.E + kRouteWarps - 1) / kRouteWarps;
        if (a.act == ACT_BF16) k_route<ACT_BF16, true><<<grid, kRouteThreads, smem, s>>>(a);
        else k_route<ACT_FP32, true><<<grid, kRouteThreads, smem, s>>>(a);
    } else {
        const int grid = (a.T + kPrefillTokTile - 1) / kPrefillTokTile;
        CallArgs b = a;
        b.tc_router = 0;
        if (router_tc_eligible(a)) {
            const cudaError_t e = launch_router_tc(a, s);
            if (e != cudaSuccess) return e;
            b.tc_router = 1;
        }
        if (b.act == ACT_BF16) k_route<ACT_BF16, false><<<grid, kRouteThreads, smem, s>>>(b);
        else k_route<ACT_FP32, false><<<grid, kRouteThreads, smem, s>>>(b);
        k_perm_rows<<<grid, 256, 0, s>>>(b);
    }
    return cudaGetLastError();
}

// dynamic shared memory limits are raised once per process
cudaError_t routing_set_attributes() {
    cudaError_t e;
    cudaFuncAttributes fa;  // loads the kernel now (see experts_preload)
    if ((e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(&k_perm_rows)))) return e;
    const int big = static_cast<int>(route_smem_limit());
    if ((e = cudaFuncSetAttribute(k_route<ACT_BF16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, big))) return e;
    if ((e = cudaFuncSetAttribute(k_route<ACT_BF16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, big))) return e;
    if ((e = cudaFuncSetAttribute(k_route<ACT_FP32, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, big))) return e;
    if ((e = cudaFuncSetAttribute(k_route<ACT_FP32, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, big))) return e;
    return cudaSuccess;
}

}  // namespace moe
