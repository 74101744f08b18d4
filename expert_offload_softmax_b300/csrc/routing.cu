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
//  A (every CTA)  router logits in the fixed fp32 order. Decode (T <= 8): one
//                 warp per expert for all tokens, the activations are also
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

namespace moe {

constexpr int kRouteThreads = 512;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kPrefillTokTile = 8;  // tokens per phase-A CTA (prefill)
constexpr int kPrefillEpw = 2;      // experts per warp per pass (prefill)

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
// activations -> device K-order (f16 for FP4 weights, bf16 for BF16 weights)
// for rows [t0, t1); work split over `nthr` threads starting at `tid`
// --------------------------------------------------------------------------

template <int ACT>
__device__ void xprep_rows(const void* __restrict__ hidden, void* __restrict__ xh, int fmt, int H, int t0,
                           int t1, size_t tid, size_t nthr) {
    if (fmt == FMT_FP32) return;
    const bool f16 = fmt != FMT_BF16;
    const int h4 = H / 4;
    const size_t n4 = static_cast<size_t>(t1 - t0) * h4;
    for (size_t idx = tid; idx < n4; idx += nthr) {
        const int t = t0 + static_cast<int>(idx / h4);
        const int p = 4 * static_cast<int>(idx % h4);   // device position
        const int j = p >> 7, w = p & 127, q = w >> 5, s = (w & 31) >> 2;
        const size_t src = static_cast<size_t>(t) * H + 128 * j + 16 * s + 4 * q;
        const float v0 = ld_act<ACT>(hidden, src), v1 = ld_act<ACT>(hidden, src + 1);
        const float v2 = ld_act<ACT>(hidden, src + 2), v3 = ld_act<ACT>(hidden, src + 3);
        uint2 o;
        if (f16) {
            __half2 a = __floats2half2_rn(v0, v1), b = __floats2half2_rn(v2, v3);
            o.x = *reinterpret_cast<uint32_t*>(&a);
            o.y = *reinterpret_cast<uint32_t*>(&b);
        } else {
            __nv_bfloat162 a = __floats2bfloat162_rn(v0, v1), b = __floats2bfloat162_rn(v2, v3);
            o.x = *reinterpret_cast<uint32_t*>(&a);
            o.y = *reinterpret_cast<uint32_t*>(&b);
        }
        *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(xh) + static_cast<size_t>(t) * H + p) = o;
    }
}

// --------------------------------------------------------------------------
// router logits of one warp in the fixed summation order
//   H is cut into 8-element chunks; chunk c belongs to lane c mod 32, which
//   accumulates its chunks in increasing h with fused multiply-adds from 0;
//   the 32 lane sums then combine by xor-butterfly (o = 16, 8, 4, 2, 1).
// EPW experts (rows e0.. of router_w, e >= E contributes nothing) x nt tokens
// whose rows sit in shared memory; every lane returns the finished sums.
// --------------------------------------------------------------------------

template <int ACT, int EPW>
__device__ __forceinline__ void warp_logits(const void* __restrict__ router_w, const unsigned char* xs, int H,
                                            int E, int e0, int nt, int lane, float (&acc)[EPW][8]) {
#pragma unroll
    for (int e = 0; e < EPW; ++e)
#pragma unroll
        for (int t = 0; t < 8; ++t) acc[e][t] = 0.0f;
    const int nchunk = H / 8;
#pragma unroll 2
    for (int c = lane; c < nchunk; c += 32) {
        float wv[EPW][8];
#pragma unroll
        for (int e = 0; e < EPW; ++e) {
            if (e0 + e < E) {
                ld_act8<ACT>(router_w, static_cast<size_t>(e0 + e) * H + 8 * c, wv[e]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) wv[e][i] = 0.0f;
            }
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            if (t < nt) {
                float xv[8];
                ld_act8<ACT>(xs, static_cast<size_t>(t) * H + 8 * c, xv);
#pragma unroll
                for (int e = 0; e < EPW; ++e)
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[e][t] = __fmaf_rn(xv[i], wv[e][i], acc[e][t]);
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

// --------------------------------------------------------------------------
// softmax + top-k + renormalisation of one token, one warp
//   selection on the logits: larger first, ties to the lower expert index,
//   NaN treated as -inf; gates = softmax probabilities of the selected experts
//   divided by their sum. Lane j < k returns selection j.
// --------------------------------------------------------------------------

template <bool GLOBAL>
__device__ __forceinline__ void warp_topk(const float* lrow, int E, int k, int lane, int& sel, float& gate) {
    constexpr int kPer = kMaxExperts / 32;
    const int per = (E + 31) / 32;
    float v[kPer];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        v[i] = -INFINITY;
        const int e = lane + 32 * i;
        if (i < per && e < E) {
            float x = GLOBAL ? __ldcg(lrow + e) : lrow[e];
            if (x != x) x = -INFINITY;
            v[i] = x;
            mx = fmaxf(mx, x);
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float den = 0.0f;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
        if (i < per && v[i] != -INFINITY) den += expf(v[i] - mx);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    uint32_t taken = 0;
    float psum = 0.0f, pj = 0.0f;
    int ej = 0;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kPer; ++i) {
            const int e = lane + 32 * i;
            if (i < per && e < E && !((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < be))) {
                bv = v[i];
                be = e;
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        const float p = bv == -INFINITY ? 0.0f : expf(bv - mx) / den;
        psum += p;
        if (lane == j) { pj = p; ej = be; }
    }
    sel = ej;
    gate = pj / psum;
}

// --------------------------------------------------------------------------
// device LRU cache (phase B, one CTA)
//   One pool of S slots shared by all layers; table[l*E+e] -> slot, owner[s]
//   -> key, stamp[s] recency (0 = never filled). A batch serves the ascending,
//   distinct experts of one layer at clock c = ++clock; member p gets stamp
//   c*65536 + p. Hits only restamp. Misses, in member order, take the slots
//   with the smallest (stamp, slot index) among slots holding neither a member
//   nor a protected key. A prefill call with prefetch enabled, layer+1 < L and
//   S >= n_uniq + E then runs a second batch over all E experts of layer+1,
//   protecting this layer's experts.
// --------------------------------------------------------------------------

struct LruShared {
    uint32_t blocked[kMaxSlots / 32];
    int32_t member_slot[kMaxExperts];
    int32_t member_old[kMaxExperts];
    int32_t miss_p[kMaxExperts];
    int32_t victim[kMaxExperts];
    int32_t scan[kRouteWarps];
    unsigned long long red[2][kRouteWarps];
    int32_t n_free;
    unsigned long long clock;
};

// phase-B shared memory; the keys / per-warp count area follows it
struct RouteShared {
    int32_t cnt[kMaxExperts];
    int32_t off[kMaxExperts];
    int32_t members[kMaxExperts];
    int32_t topk[kDecodeMaxT * kMaxTopK];
    float gates[kDecodeMaxT * kMaxTopK];
    int32_t scan_a[kRouteWarps], scan_b[kRouteWarps];
    int32_t nu;
    LruShared lru;
};

constexpr size_t kRouteSharedBytes = (sizeof(RouteShared) + 15) / 16 * 16;

__device__ __forceinline__ unsigned long long slot_key(unsigned long long stamp, int s) {
    return (stamp << 14) | static_cast<unsigned long long>(s);
}

// members: the batch's experts (ascending), or nullptr for 0..n-1.
// Returns the number of misses, or -1 (not enough slots; nothing changed).
__device__ int lru_batch(const CallArgs& a, LruShared& sm, unsigned long long* keys, int layer,
                         const int32_t* members, int n, const int32_t* protect, int n_protect, int protect_layer) {
    const int tid = threadIdx.x, nthr = blockDim.x, S = a.S, E = a.E;
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
    for (int i = tid; i < (S + 31) / 32; i += nthr) sm.blocked[i] = 0u;
    if (tid == 0) sm.n_free = 0;
    __syncthreads();
    for (int p = tid; p < n; p += nthr) {
        const int e = members ? members[p] : p;
        const int s = a.table[layer * E + e];
        sm.member_slot[p] = s;
        sm.member_old[p] = -1;
        if (s >= 0) atomicOr(&sm.blocked[s >> 5], 1u << (s & 31));
    }
    for (int q = tid; q < n_protect; q += nthr) {
        const int s = a.table[protect_layer * E + protect[q]];
        if (s >= 0) atomicOr(&sm.blocked[s >> 5], 1u << (s & 31));
    }
    __syncthreads();
    // misses in member order
    int running = 0;
    for (int base = 0; base < n; base += nthr) {
        const int p = base + tid;
        const int m = (p < n && sm.member_slot[p] < 0) ? 1 : 0;
        const unsigned bal = __ballot_sync(0xffffffffu, m);
        if (lane == 0) sm.scan[warp] = __popc(bal);
        __syncthreads();
        int wb = 0, tot = 0;
        for (int w = 0; w < nwarps; ++w) {
            if (w < warp) wb += sm.scan[w];
            tot += sm.scan[w];
        }
        if (m) sm.miss_p[running + wb + __popc(bal & ((1u << lane) - 1u))] = p;
        running += tot;
        __syncthreads();
    }
    int nfree = 0;
    for (int i = tid; i < (S + 31) / 32; i += nthr) {
        const int bits = min(32, S - 32 * i);
        const uint32_t valid = bits == 32 ? 0xffffffffu : ((1u << bits) - 1u);
        nfree += __popc(~sm.blocked[i] & valid);
    }
    atomicAdd(&sm.n_free, nfree);
    __syncthreads();
    const int m = running;
    if (m > sm.n_free) return -1;
    if (tid == 0) {
        sm.clock = *a.clock + 1;
        *a.clock = sm.clock;
    }
    __syncthreads();
    const unsigned long long c = sm.clock;
    // hits restamp
    for (int p = tid; p < n; p += nthr)
        if (sm.member_slot[p] >= 0) a.stamp[sm.member_slot[p]] = (c << 16) | static_cast<unsigned long long>(p);
    if (m > 0) {
        // keys of the candidate slots; blocked slots never win
        int P = 1;
        while (P < S) P <<= 1;
        const int span = m <= 32 ? S : P;
        for (int s = tid; s < span; s += nthr)
            keys[s] = (s < S && !((sm.blocked[s >> 5] >> (s & 31)) & 1u)) ? slot_key(a.stamp[s], s) : ~0ull;
        __syncthreads();
        if (m <= 32) {
            // m rounds of a block-wide minimum; slot s is only ever read by thread s mod nthr
            for (int r = 0; r < m; ++r) {
                unsigned long long best = ~0ull;
                for (int s = tid; s < S; s += nthr) best = keys[s] < best ? keys[s] : best;
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) {
                    const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
                    best = y < best ? y : best;
                }
                if (lane == 0) sm.red[r & 1][warp] = best;
                __syncthreads();
                unsigned long long b = ~0ull;
                for (int w = 0; w < nwarps; ++w) b = sm.red[r & 1][w] < b ? sm.red[r & 1][w] : b;
                const int v = static_cast<int>(b & 0x3FFFull);
                if (tid == 0) sm.victim[r] = v;
                if (v % nthr == tid) keys[v] = ~0ull;
            }
        } else {
            // bitonic sort of the P keys, ascending
            for (int kk = 2; kk <= P; kk <<= 1) {
                for (int j = kk >> 1; j > 0; j >>= 1) {
                    for (int i = tid; i < P / 2; i += nthr) {
                        const int lo = (i / j) * 2 * j + (i % j), hi = lo + j;
                        const bool up = (lo & kk) == 0;
                        const unsigned long long x = keys[lo], y = keys[hi];
                        if ((x > y) == up) { keys[lo] = y; keys[hi] = x; }
                    }
                    __syncthreads();
                }
            }
            for (int r = tid; r < m; r += nthr) sm.victim[r] = static_cast<int>(keys[r] & 0x3FFFull);
        }
        __syncthreads();
    }
    // fill the victims
    for (int r = tid; r < m; r += nthr) {
        const int p = sm.miss_p[r];
        const int v = sm.victim[r];
        const int e = members ? members[p] : p;
        const int32_t key = layer * E + e;
        const int32_t old = a.owner[v];
        if (old >= 0) a.table[old] = -1;
        a.owner[v] = key;
        a.table[key] = v;
        a.stamp[v] = (c << 16) | static_cast<unsigned long long>(p);
        sm.member_slot[p] = v;
        sm.member_old[p] = old;
    }
    __syncthreads();
    return m;
}

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

// --------------------------------------------------------------------------
// phase B: everything after the logits (and, for prefill, the top-k)
// --------------------------------------------------------------------------

__device__ void route_phase_b(const CallArgs& a, RouteShared& rs, unsigned char* area, bool decode) {
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31, warp = tid >> 5;
    const int T = a.T, E = a.E, k = a.k, n = T * k;
    CallInfo* info = a.info;
    // decode: top-k of every token (one warp each)
    if (decode) {
        if (warp < T) {
            int sel;
            float g;
            warp_topk<true>(a.logits + static_cast<size_t>(warp) * E, E, k, lane, sel, g);
            if (lane < k) {
                rs.topk[warp * k + lane] = sel;
                rs.gates[warp * k + lane] = g;
                a.topk[warp * k + lane] = sel;
                a.gates[warp * k + lane] = g;
            }
        }
        for (int i = tid; i < (E + a.n_shared) * kDecodeMaxT; i += nthr) a.tok_row[i] = -1;
    }
    for (int e = tid; e < E; e += nthr) rs.cnt[e] = 0;
    __syncthreads();
    auto topk_at = [&](int i) -> int { return decode ? rs.topk[i] : __ldcg(a.topk + i); };
    auto gate_at = [&](int i) -> float { return decode ? rs.gates[i] : __ldcg(a.gates + i); };
    for (int i = tid; i < n; i += nthr) atomicAdd(&rs.cnt[topk_at(i)], 1);
    __syncthreads();
    // offsets (exclusive) and the active list: each thread owns experts 2*tid, 2*tid+1, ...
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
                a.offsets[e] = ec;
                a.counts[e] = c;
                a.e2u[e] = c > 0 ? ez : -1;
                if (c > 0) {
                    rs.members[ez] = e;
                    a.act_expert[ez] = e;
                    a.act_row0[ez] = ec;
                    a.act_cnt[ez] = c;
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
    // stable permutation: warp w owns the contiguous assignment range [w*chunk, (w+1)*chunk)
    {
        int32_t* wc = reinterpret_cast<int32_t*>(area);  // [kRouteWarps][E]
        const int nwarps = nthr >> 5;
        const int chunk = (n + nwarps - 1) / nwarps;
        const int a0 = min(n, warp * chunk), a1 = min(n, a0 + chunk);
        for (int i = tid; i < nwarps * E; i += nthr) wc[i] = 0;
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
                if (decode) a.tok_row[a.e2u[e] * kDecodeMaxT + t] = row;
            }
        }
    }
    __syncthreads();
    // LRU: demand batch of this layer's experts
    unsigned long long* keys = reinterpret_cast<unsigned long long*>(area);
    LruShared& sm = rs.lru;
    const int nu = rs.nu;
    const int m = lru_batch(a, sm, keys, a.layer, rs.members, nu, nullptr, 0, 0);
    if (m < 0) {
        if (tid == 0) {
            info->n_uniq = nu;
            info->n_hit = info->n_miss = info->n_pf = info->n_pf_hit = info->n_pf_miss = 0;
            info->n_events = 0;
            info->dev_err = *reinterpret_cast<volatile int32_t*>(a.dev_err);
            *a.n_active = 0;
            __threadfence_system();
            info->status = -4;  // MOE_ERR_CAPACITY
        }
        return;
    }
    for (int p = tid; p < nu; p += nthr) {
        const int s = sm.member_slot[p];
        a.act_ptr[p] = a.pool + static_cast<size_t>(s) * a.lay.bytes;
        a.act_slot[p] = s;
        info->ev_layer[p] = a.layer;
        info->ev_expert[p] = rs.members[p];
        info->ev_hit[p] = 1;
        info->ev_slot[p] = s;
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
    int n_pf = 0, m_pf = 0;
    const bool do_pf = a.prefetch && T > kDecodeMaxT && a.layer + 1 < a.L && a.S >= nu + E;
    if (do_pf) {
        m_pf = lru_batch(a, sm, keys, a.layer + 1, nullptr, E, rs.members, nu, a.layer);
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
    }
    __syncthreads();
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
        __threadfence_system();
        info->status = 0;
    }
}

// --------------------------------------------------------------------------
// the fused routing kernel
// --------------------------------------------------------------------------

template <int ACT, bool DECODE>
__global__ void __launch_bounds__(kRouteThreads) k_route(CallArgs a) {
    extern __shared__ __align__(16) unsigned char route_smem[];
    __shared__ int s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = a.T, E = a.E, H = a.H;
    const size_t esz = ACT == ACT_BF16 ? 2 : 4;
    // ---------------- phase A
    if constexpr (DECODE) {
        // x rows [T][H] in shared memory; warp w: expert blockIdx.x * 16 + w
        {
            const size_t bytes = static_cast<size_t>(T) * H * esz;
            const uint4* src = reinterpret_cast<const uint4*>(a.hidden);
            uint4* dst = reinterpret_cast<uint4*>(route_smem);
            for (size_t i = threadIdx.x; i < bytes / 16; i += blockDim.x) dst[i] = src[i];
        }
        xprep_rows<ACT>(a.hidden, a.xh, a.fmt, H, 0, T, static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x,
                        static_cast<size_t>(gridDim.x) * blockDim.x);
        __syncthreads();
        const int e0 = blockIdx.x * kRouteWarps + warp;
        if (e0 < E) {
            float acc[1][8];
            warp_logits<ACT, 1>(a.router_w, route_smem, H, E, e0, T, lane, acc);
            if (lane < T) {
                float v = acc[0][0];
#pragma unroll
                for (int t = 1; t < 8; ++t) v = lane == t ? acc[0][t] : v;
                a.logits[static_cast<size_t>(lane) * E + e0] = v;
            }
        }
    } else {
        // 8 tokens per CTA, all experts; logits [8][E] in shared memory, then top-k
        const int t0 = blockIdx.x * kPrefillTokTile;
        const int nt = min(kPrefillTokTile, T - t0);
        float* lg = reinterpret_cast<float*>(route_smem + static_cast<size_t>(kPrefillTokTile) * H * esz);
        {
            const size_t bytes = static_cast<size_t>(nt) * H * esz;
            const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned char*>(a.hidden) +
                                                              static_cast<size_t>(t0) * H * esz);
            uint4* dst = reinterpret_cast<uint4*>(route_smem);
            for (size_t i = threadIdx.x; i < bytes / 16; i += blockDim.x) dst[i] = src[i];
        }
        if (a.fmt != FMT_BF16) xprep_rows<ACT>(a.hidden, a.xh, a.fmt, H, t0, t0 + nt, threadIdx.x, blockDim.x);
        __syncthreads();
        constexpr int kPass = kRouteWarps * kPrefillEpw;
        for (int eb = 0; eb < E; eb += kPass) {
            const int e0 = eb + warp * kPrefillEpw;
            if (e0 < E) {
                float acc[kPrefillEpw][8];
                warp_logits<ACT, kPrefillEpw>(a.router_w, route_smem, H, E, e0, nt, lane, acc);
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
            warp_topk<false>(lg + warp * E, E, a.k, lane, sel, g);
            if (lane < a.k) {
                const size_t o = static_cast<size_t>(t0 + warp) * a.k + lane;
                a.topk[o] = sel;
                a.gates[o] = g;
            }
        }
    }
    // ---------------- hand-off: the last CTA to finish runs phase B
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const int prev = atomicAdd(a.route_done, 1);
        s_last = prev == static_cast<int>(gridDim.x) - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    RouteShared& rs = *reinterpret_cast<RouteShared*>(route_smem);
    route_phase_b(a, rs, route_smem + kRouteSharedBytes, DECODE);
    if (threadIdx.x == 0) *a.route_done = 0;
}

// dynamic shared memory of one k_route launch
static size_t route_smem_bytes(const CallArgs& a, bool decode) {
    const size_t esz = a.act == ACT_BF16 ? 2 : 4;
    const size_t phase_a = decode ? static_cast<size_t>(a.T) * a.H * esz
                                  : static_cast<size_t>(kPrefillTokTile) * a.H * esz +
                                        static_cast<size_t>(kPrefillTokTile) * a.E * 4;
    size_t P = 1;
    while (P < static_cast<size_t>(a.S)) P <<= 1;
    const size_t area = std::max(P * 8, static_cast<size_t>(kRouteWarps) * a.E * 4);
    return std::max(phase_a, kRouteSharedBytes + area);
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
        if (a.act == ACT_BF16) k_route<ACT_BF16, false><<<grid, kRouteThreads, smem, s>>>(a);
        else k_route<ACT_FP32, false><<<grid, kRouteThreads, smem, s>>>(a);
    }
    return cudaGetLastError();
}

// dynamic shared memory limits are raised once per process
cudaError_t routing_set_attributes() {
    cudaError_t e;
    const int big = static_cast<int>(route_smem_limit());
    if ((e = cudaFuncSetAttribute(k_route<ACT_BF16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, big))) return e;
    if ((e = cudaFuncSetAttribute(k_route<ACT_BF16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, big))) return e;
    if ((e = cudaFuncSetAttribute(k_route<ACT_FP32, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, big))) return e;
    if ((e = cudaFuncSetAttribute(k_route<ACT_FP32, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, big))) return e;
    return cudaSuccess;
}

}  // namespace moe
