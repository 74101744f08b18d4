// Device routines shared by the routing kernels: the softmax / top-k /
// renormalisation of one token on one warp, and the device LRU batch of the
// expert cache (one CTA). Follows "FreeToken量子化：MoE推論のセットアップガイド"
// (freetoken.wiki, architecture page): decode keeps an LRU over recently
// selected experts in one cache shared by all MoE layers. The tie-break and
// the batch LRU rule are fixed readings, stated below.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_internal.h"

namespace moe {

constexpr int kLruMaxWarps = 32;  // blocks of up to 1024 threads

// --------------------------------------------------------------------------
// softmax + top-k + renormalisation of one token, one warp
//   selection on the logits: larger first, ties to the lower expert index,
//   NaN treated as -inf; gates = softmax probabilities of the selected experts
//   divided by their sum. Lane j < k returns selection j.
// --------------------------------------------------------------------------

// float -> unsigned with the same order (NaN never reaches it; callers turn
// -0.0 into +0.0 first, since the two compare equal)
__device__ __forceinline__ uint32_t ord_key(float v) {
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// KPER: logits per lane the code is unrolled for (E <= 32 * KPER). Each round
// takes the lane-local best untaken logit, then the warp maximum and the
// lowest expert index holding it with two warp-wide reductions.
template <bool GLOBAL, int KPER>
__device__ __forceinline__ void warp_topk_n(const float* lrow, int E, int k, int lane, int& sel, float& gate) {
    float v[KPER];
    uint32_t key[KPER];
#pragma unroll
    for (int i = 0; i < KPER; ++i) {
        const int e = lane + 32 * i;
        float x = -INFINITY;
        if (e < E) x = GLOBAL ? __ldcg(lrow + e) : lrow[e];
        if (x != x) x = -INFINITY;
        x = __fadd_rn(x, 0.0f);  // -0.0 -> +0.0: the two zeros are one logit value (equal, lower index wins)
        v[i] = x;
        key[i] = ord_key(x);
    }
    uint32_t kmax = 0u;
#pragma unroll
    for (int i = 0; i < KPER; ++i) kmax = key[i] > kmax ? key[i] : kmax;
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    const uint32_t mu = (kmax & 0x80000000u) ? (kmax & 0x7FFFFFFFu) : ~kmax;
    const float mx = __uint_as_float(mu);
    float den = 0.0f;
#pragma unroll
    for (int i = 0; i < KPER; ++i)
        if (v[i] != -INFINITY) den += expf(v[i] - mx);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    uint32_t taken = 0;
    int ej = 0;
    float bvj = -INFINITY;
    for (int j = 0; j < k; ++j) {
        uint32_t bk = 0u;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < KPER; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && key[i] > bk) { bk = key[i]; be = e; }
        }
        // lanes whose local best is below the warp best offer no index
        const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
        const int we = static_cast<int>(__reduce_min_sync(0xffffffffu, static_cast<uint32_t>(bk == wk ? be : 0x7fffffff)));
        if ((we & 31) == lane) taken |= 1u << (we >> 5);
        if (lane == j) {
            ej = we;
            const uint32_t u = (wk & 0x80000000u) ? (wk & 0x7FFFFFFFu) : ~wk;
            bvj = __uint_as_float(u);
        }
    }
    // lane j < k holds selection j; gates = its probability / sum over the k
    const float pj = (lane < k && bvj != -INFINITY) ? expf(bvj - mx) / den : 0.0f;
    float psum = lane < k ? pj : 0.0f;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
    sel = ej;
    gate = pj / psum;
}

template <bool GLOBAL>
__device__ __forceinline__ void warp_topk(const float* lrow, int E, int k, int lane, int& sel, float& gate) {
    if (E <= 256) warp_topk_n<GLOBAL, 8>(lrow, E, k, lane, sel, gate);
    else warp_topk_n<GLOBAL, kMaxExperts / 32>(lrow, E, k, lane, sel, gate);
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
    int32_t scan[kLruMaxWarps];
    unsigned long long red[2][kLruMaxWarps];
    int32_t n_free;
    unsigned long long clock;
};

// The LRU state phase B works on: global arrays, with shared-memory copies
// (loaded once at the start of phase B) of the stamps and owners of a small
// pool and of the table rows of this layer and the next. Every write goes to
// both.
struct LruView {
    const CallArgs* a;
    int32_t* trow0;               // table row of a.layer
    int32_t* trow1;               // table row of a.layer + 1 (prefill prefetch)
    unsigned long long* st_s;     // [S] stamps, or null
    int32_t* own_s;               // [S] owners, or null
    __device__ int table(int layer, int e) const {
        if (layer == a->layer) return trow0[e];
        if (trow1 && layer == a->layer + 1) return trow1[e];
        return a->table[layer * a->E + e];
    }
    __device__ void set_table(int key, int v) const {
        a->table[key] = v;
        const int l = key / a->E, e = key % a->E;
        if (l == a->layer) trow0[e] = v;
        else if (trow1 && l == a->layer + 1) trow1[e] = v;
    }
    __device__ unsigned long long stamp(int s) const { return st_s ? st_s[s] : a->stamp[s]; }
    __device__ void set_stamp(int s, unsigned long long v) const {
        a->stamp[s] = v;
        if (st_s) st_s[s] = v;
    }
    __device__ int owner(int s) const { return own_s ? own_s[s] : a->owner[s]; }
    __device__ void set_owner(int s, int v) const {
        a->owner[s] = v;
        if (own_s) own_s[s] = v;
    }
};

__device__ __forceinline__ unsigned long long slot_key(unsigned long long stamp, int s) {
    return (stamp << 14) | static_cast<unsigned long long>(s);
}

// members: the batch's experts (ascending), or nullptr for 0..n-1.
// Returns the number of misses, or -1 (not enough slots; nothing changed).
__device__ inline int lru_batch(const CallArgs& a, const LruView& lv, LruShared& sm, unsigned long long* keys, int layer,
                         const int32_t* members, int n, const int32_t* protect, int n_protect, int protect_layer) {
    const int tid = threadIdx.x, nthr = blockDim.x, S = a.S;
    const int lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
    for (int i = tid; i < (S + 31) / 32; i += nthr) sm.blocked[i] = 0u;
    if (tid == 0) sm.n_free = 0;
    __syncthreads();
    for (int p = tid; p < n; p += nthr) {
        const int e = members ? members[p] : p;
        const int s = lv.table(layer, e);
        sm.member_slot[p] = s;
        sm.member_old[p] = -1;
        if (s >= 0) atomicOr(&sm.blocked[s >> 5], 1u << (s & 31));
    }
    for (int q = tid; q < n_protect; q += nthr) {
        const int s = lv.table(protect_layer, protect[q]);
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
    const unsigned long long c = sm.clock + 1;
    // hits restamp
    for (int p = tid; p < n; p += nthr)
        if (sm.member_slot[p] >= 0) lv.set_stamp(sm.member_slot[p], (c << 16) | static_cast<unsigned long long>(p));
    if (m > 0) {
        // keys of the candidate slots; blocked slots never win
        int P = 1;
        while (P < S) P <<= 1;
        const int span = m <= 32 ? S : P;
        for (int s = tid; s < span; s += nthr)
            keys[s] = (s < S && !((sm.blocked[s >> 5] >> (s & 31)) & 1u)) ? slot_key(lv.stamp(s), s) : ~0ull;
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
    // fill the victims (distinct slots; the evicted keys are not members)
    for (int r = tid; r < m; r += nthr) {
        const int p = sm.miss_p[r];
        const int v = sm.victim[r];
        const int e = members ? members[p] : p;
        const int32_t key = layer * a.E + e;
        const int32_t old = lv.owner(v);
        if (old >= 0) lv.set_table(old, -1);
        lv.set_owner(v, key);
        lv.set_table(key, v);
        lv.set_stamp(v, (c << 16) | static_cast<unsigned long long>(p));
        sm.member_slot[p] = v;
        sm.member_old[p] = old;
    }
    __syncthreads();
    if (tid == 0) {
        sm.clock = c;
        *a.clock = c;
    }
    __syncthreads();
    return m;
}

}  // namespace moe
