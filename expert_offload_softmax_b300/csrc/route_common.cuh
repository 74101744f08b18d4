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

// The same selection with one pass instead of k rounds, using 32 words of
// warp-private scratch. Every logit becomes one 64-bit key, (ordered logit,
// inverted index), so that a larger key means a larger logit or, on equal
// logits, a lower index: the selection order above. The k-th largest of the
// 32 lane maxima is a lower bound tau of the k-th largest key, since k lanes
// hold a key >= tau; only keys >= tau can be selected (at least k, at most
// k * KPER of them, usually a few more than k). When they fit in 32 they are
// compacted into the scratch and each is ranked by counting the larger ones;
// otherwise the function returns false and selects nothing.
template <bool GLOBAL, int KPER>
__device__ __forceinline__ bool warp_topk_pass(const float* lrow, int E, int k, int lane, unsigned long long* scr,
                                               int& sel, float& gate) {
    unsigned long long key[KPER];
    unsigned long long lm = 0ull;
#pragma unroll
    for (int i = 0; i < KPER; ++i) {
        const int e = lane + 32 * i;
        key[i] = 0ull;
        if (e < E) {
            float x = GLOBAL ? __ldcg(lrow + e) : lrow[e];
            if (x != x) x = -INFINITY;
            x = __fadd_rn(x, 0.0f);  // -0.0 -> +0.0
            key[i] = (static_cast<unsigned long long>(ord_key(x)) << 32) | (0xFFFFFFFFu - static_cast<uint32_t>(e));
        }
        lm = key[i] > lm ? key[i] : lm;
    }
    // rank of this lane's maximum among the 32 (keys of valid logits are distinct;
    // lanes without one hold 0, below all of them, and k <= min(32, E))
    int r = 0;
#pragma unroll
    for (int j = 0; j < 32; ++j) r += __shfl_sync(0xffffffffu, lm, j) > lm;
    const unsigned int bal = __ballot_sync(0xffffffffu, r == k - 1);
    const unsigned long long tau = __shfl_sync(0xffffffffu, lm, __ffs(bal) - 1);
    int cnt = 0;
#pragma unroll
    for (int i = 0; i < KPER; ++i) cnt += key[i] >= tau;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (total > 32) return false;
    int pos = incl - cnt;
#pragma unroll
    for (int i = 0; i < KPER; ++i)
        if (key[i] >= tau) scr[pos++] = key[i];
    __syncwarp();
    const unsigned long long mine = lane < total ? scr[lane] : 0ull;
    int rank = 0;
    for (int j = 0; j < total; ++j) rank += scr[j] > mine;
    __syncwarp();
    if (lane < total && rank < k) scr[rank] = mine;
    __syncwarp();
    const unsigned long long kj = scr[lane < k ? lane : 0];
    const unsigned long long k0 = scr[0];
    __syncwarp();  // the scratch may be reused after this
    const uint32_t uj = static_cast<uint32_t>(kj >> 32), u0 = static_cast<uint32_t>(k0 >> 32);
    const float vj = __uint_as_float((uj & 0x80000000u) ? (uj & 0x7FFFFFFFu) : ~uj);
    const float mx = __uint_as_float((u0 & 0x80000000u) ? (u0 & 0x7FFFFFFFu) : ~u0);
    // gates: softmax restricted to the k selected (the full softmax's
    // denominator cancels in the renormalisation)
    const float pj = (lane < k && vj != -INFINITY) ? expf(vj - mx) : 0.0f;
    float psum = pj;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
    sel = lane < k ? static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(kj)) : 0;
    gate = pj / psum;
    return true;
}

// top-k of one row of E logits by one warp; lane j < k gets selection j.
// scr: 32 words of scratch private to the warp, or null (round-based only)
// (not inlined: one copy of this code serves every call site of a kernel, which
// keeps the kernel's instructions within the SM's instruction cache)
template <bool GLOBAL>
__device__ __noinline__ void warp_topk(const float* lrow, int E, int k, int lane, int& sel, float& gate,
                                       unsigned long long* scr = nullptr) {
    if (E <= 256) {
        if (scr && warp_topk_pass<GLOBAL, 8>(lrow, E, k, lane, scr, sel, gate)) return;
        warp_topk_n<GLOBAL, 8>(lrow, E, k, lane, sel, gate);
    } else {
        if (scr && warp_topk_pass<GLOBAL, kMaxExperts / 32>(lrow, E, k, lane, scr, sel, gate)) return;
        warp_topk_n<GLOBAL, kMaxExperts / 32>(lrow, E, k, lane, sel, gate);
    }
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
    // the LRU arrays and sizes, copied out of the call's arguments (a load
    // through a pointer to a kernel argument is a memory round trip)
    int32_t* gtable;              // [L*E] -> slot
    unsigned long long* gstamp;   // [S]
    int32_t* gowner;              // [S]
    unsigned long long* gclock;
    int E, S, layer;
    int32_t* trow0;               // table row of `layer`
    int32_t* trow1;               // table row of layer + 1 (prefill prefetch)
    unsigned long long* st_s;     // [S] stamps, or null
    int32_t* own_s;               // [S] owners, or null
    __device__ __forceinline__ void bind(const CallArgs& a) {
        gtable = a.table;
        gstamp = a.stamp;
        gowner = a.owner;
        gclock = a.clock;
        E = a.E;
        S = a.S;
        layer = a.layer;
    }
    __device__ int table(int l, int e) const {
        if (l == layer) return trow0[e];
        if (trow1 && l == layer + 1) return trow1[e];
        return gtable[l * E + e];
    }
    __device__ void set_table(int key, int v) const {
        gtable[key] = v;
        const int l = key / E, e = key - l * E;
        if (l == layer) trow0[e] = v;
        else if (trow1 && l == layer + 1) trow1[e] = v;
    }
    __device__ unsigned long long stamp(int s) const { return st_s ? st_s[s] : gstamp[s]; }
    __device__ void set_stamp(int s, unsigned long long v) const {
        gstamp[s] = v;
        if (st_s) st_s[s] = v;
    }
    __device__ int owner(int s) const { return own_s ? own_s[s] : gowner[s]; }
    __device__ void set_owner(int s, int v) const {
        gowner[s] = v;
        if (own_s) own_s[s] = v;
    }
};

__device__ __forceinline__ unsigned long long slot_key(unsigned long long stamp, int s) {
    return (stamp << 14) | static_cast<unsigned long long>(s);
}

// members: the batch's experts (ascending), or nullptr for 0..n-1.
// Returns the number of misses, or -1 (not enough slots; nothing changed).
static __device__ __noinline__ int lru_batch(const LruView& lv, LruShared& sm, unsigned long long* keys, int layer,
                         const int32_t* members, int n, const int32_t* protect, int n_protect, int protect_layer) {
    const int tid = threadIdx.x, nthr = blockDim.x, S = lv.S;
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
        const int32_t key = layer * lv.E + e;
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
        *lv.gclock = c;
    }
    __syncthreads();
    return m;
}

}  // namespace moe
