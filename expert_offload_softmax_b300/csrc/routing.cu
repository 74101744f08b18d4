// Router (logits, softmax + top-k + renormalisation), permutation by expert and
// the device-side LRU expert cache of the routed MoE layer.
//
// Follows "FreeToken量子化：MoE推論のセットアップガイド" (freetoken.wiki,
// architecture page): decode keeps a shared LRU over recently selected
// experts; a hit runs on the GPU, a miss is copied into the cache over PCIe;
// prefill streams the next layer's experts while the current layer computes
// when the cache has room. Summation order, tie-break and the batch LRU rule
// are fixed readings, stated at each kernel.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "moe_internal.h"

namespace moe {

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
// --------------------------------------------------------------------------

template <int ACT, bool F16>
__global__ void k_xprep(const void* __restrict__ hidden, void* __restrict__ xh, int T, int H) {
    const size_t n4 = static_cast<size_t>(T) * H / 4;
    const int h4 = H / 4;
    for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < n4;
         idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(idx / h4);
        const int p = 4 * static_cast<int>(idx % h4);   // device position
        const int j = p >> 7, w = p & 127, q = w >> 5, s = (w & 31) >> 2;
        const size_t src = static_cast<size_t>(t) * H + 128 * j + 16 * s + 4 * q;
        float v0 = ld_act<ACT>(hidden, src), v1 = ld_act<ACT>(hidden, src + 1);
        float v2 = ld_act<ACT>(hidden, src + 2), v3 = ld_act<ACT>(hidden, src + 3);
        uint2 o;
        if constexpr (F16) {
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
// router logits in the fixed summation order
//   H is cut into 8-element chunks; chunk c belongs to lane c mod 32, which
//   accumulates its chunks in increasing h with fused multiply-adds from 0;
//   the 32 lane sums then combine by xor-butterfly (o = 16, 8, 4, 2, 1).
// Block: 8 warps x EPW experts per warp, 8 tokens; x tile staged in shared memory.
// --------------------------------------------------------------------------

template <int ACT, int EPW>
__global__ void __launch_bounds__(256) k_logits(CallArgs a) {
    extern __shared__ __align__(16) unsigned char smem_x[];
    const int T = a.T, E = a.E, H = a.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (blockIdx.x == 0 && blockIdx.y == 0) {
        for (int i = threadIdx.x; i < E; i += blockDim.x) a.counts[i] = 0;
        if (T <= kDecodeMaxT)
            for (int i = threadIdx.x; i < (E + a.n_shared) * kDecodeMaxT; i += blockDim.x) a.tok_row[i] = -1;
    }
    const int t0 = blockIdx.y * 8;
    const int nt = min(8, T - t0);
    const size_t esz = ACT == ACT_BF16 ? 2 : 4;
    // stage x rows [nt][H]
    {
        const size_t bytes = static_cast<size_t>(nt) * H * esz;
        const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned char*>(a.hidden) +
                                                          static_cast<size_t>(t0) * H * esz);
        uint4* dst = reinterpret_cast<uint4*>(smem_x);
        for (size_t i = threadIdx.x; i < bytes / 16; i += blockDim.x) dst[i] = src[i];
    }
    __syncthreads();
    const int e0 = (blockIdx.x * 8 + warp) * EPW;
    float acc[EPW][8];
#pragma unroll
    for (int e = 0; e < EPW; ++e)
#pragma unroll
        for (int t = 0; t < 8; ++t) acc[e][t] = 0.0f;
    const int nchunk = H / 8;
    for (int c = lane; c < nchunk; c += 32) {
        float wv[EPW][8];
#pragma unroll
        for (int e = 0; e < EPW; ++e) {
            if (e0 + e < E) ld_act8<ACT>(a.router_w, static_cast<size_t>(e0 + e) * H + 8 * c, wv[e]);
            else
#pragma unroll
                for (int i = 0; i < 8; ++i) wv[e][i] = 0.0f;
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            if (t < nt) {
                float xv[8];
                ld_act8<ACT>(smem_x, static_cast<size_t>(t) * H + 8 * c, xv);
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
    if (lane == 0) {
#pragma unroll
        for (int e = 0; e < EPW; ++e)
#pragma unroll
            for (int t = 0; t < 8; ++t)
                if (t < nt && e0 + e < E) a.logits[static_cast<size_t>(t0 + t) * E + e0 + e] = acc[e][t];
    }
}

// --------------------------------------------------------------------------
// softmax + top-k + renormalisation, one warp per token
//   selection on the logits: larger first, ties to the lower expert index,
//   NaN treated as -inf; gates = softmax probabilities of the selected experts
//   divided by their sum.
// --------------------------------------------------------------------------

__global__ void __launch_bounds__(256) k_topk(CallArgs a) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= a.T) return;
    const int E = a.E, k = a.k;
    const int per = (E + 31) / 32;
    float v[kMaxExperts / 32];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i) {
        if (i < per) {
            const int e = lane + 32 * i;
            float x = e < E ? a.logits[static_cast<size_t>(t) * E + e] : -INFINITY;
            if (x != x) x = -INFINITY;
            v[i] = x;
            mx = fmaxf(mx, x);
        } else {
            v[i] = -INFINITY;
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float den = 0.0f;
#pragma unroll
    for (int i = 0; i < kMaxExperts / 32; ++i)
        if (i < per && lane + 32 * i < E && v[i] != -INFINITY) den += expf(v[i] - mx);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    uint32_t taken = 0;
    float psel[kMaxTopK];
    int isel[kMaxTopK];
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int be = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < kMaxExperts / 32; ++i) {
            const int e = lane + 32 * i;
            if (i < per && e < E && !((taken >> i) & 1u)) {
                if (v[i] > bv || (v[i] == bv && e < be)) { bv = v[i]; be = e; }
            }
        }
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oe = __shfl_xor_sync(0xffffffffu, be, o);
            if (ov > bv || (ov == bv && oe < be)) { bv = ov; be = oe; }
        }
        if ((be & 31) == lane) taken |= 1u << (be >> 5);
        isel[j] = be;
        psel[j] = bv == -INFINITY ? 0.0f : expf(bv - mx) / den;
    }
    if (lane == 0) {
        float s = 0.0f;
        for (int j = 0; j < k; ++j) s += psel[j];
        for (int j = 0; j < k; ++j) {
            a.topk[static_cast<size_t>(t) * k + j] = isel[j];
            a.gates[static_cast<size_t>(t) * k + j] = psel[j] / s;
            atomicAdd(&a.counts[isel[j]], 1);
        }
    }
}

// --------------------------------------------------------------------------
// stable counting sort of the assignments a = t*k + j by expert, one block per
// expert: offsets, perm / inv_perm, per-row token and gate, active-expert list
// --------------------------------------------------------------------------

constexpr int kPermThreads = 256;
constexpr int kPermPer = 16;  // consecutive assignments per thread per pass

__device__ __forceinline__ int block_sum_int(int v, int* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    int s = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) s += red[w];
    return s;
}

__global__ void __launch_bounds__(kPermThreads) k_perm(CallArgs a) {
    __shared__ int red[kPermThreads / 32];
    __shared__ int wex[kPermThreads / 32];
    const int e = blockIdx.x, E = a.E, k = a.k, T = a.T;
    const int n = T * k;
    int off = 0, nz = 0;
    for (int i = threadIdx.x; i < e; i += blockDim.x) {
        const int c = a.counts[i];
        off += c;
        nz += c > 0;
    }
    off = block_sum_int(off, red);
    nz = block_sum_int(nz, red);
    const int cnt = a.counts[e];
    if (e == 0) {
        int tot = 0;
        for (int i = threadIdx.x; i < E; i += blockDim.x) tot += a.counts[i] > 0;
        tot = block_sum_int(tot, red);
        if (threadIdx.x == 0) *a.n_uniq = tot;
    }
    if (threadIdx.x == 0) {
        a.offsets[e] = off;
        if (e == E - 1) a.offsets[E] = off + cnt;
        a.e2u[e] = cnt > 0 ? nz : -1;
        if (cnt > 0) {
            a.act_expert[nz] = e;
            a.act_row0[nz] = off;
            a.act_cnt[nz] = cnt;
        }
    }
    if (cnt == 0) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int running = 0;
    for (int base = 0; base < n; base += kPermThreads * kPermPer) {
        const int a0 = base + threadIdx.x * kPermPer;
        uint32_t mask = 0;
#pragma unroll
        for (int i = 0; i < kPermPer; ++i) {
            const int ai = a0 + i;
            if (ai < n && a.topk[ai] == e) mask |= 1u << i;
        }
        const int mine = __popc(mask);
        int incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) wex[warp] = incl;
        __syncthreads();
        int wbase = 0, total = 0;
        for (int w = 0; w < kPermThreads / 32; ++w) {
            if (w < warp) wbase += wex[w];
            total += wex[w];
        }
        int row = off + running + wbase + incl - mine;
        while (mask) {
            const int i = __ffs(mask) - 1;
            mask &= mask - 1;
            const int ai = a0 + i;
            a.perm[row] = ai;
            a.inv_perm[ai] = row;
            a.row_tok[row] = ai / k;
            a.row_gate[row] = a.gates[ai];
            if (T <= kDecodeMaxT) a.tok_row[nz * kDecodeMaxT + ai / k] = row;
            ++row;
        }
        running += total;
        __syncthreads();
    }
}

// --------------------------------------------------------------------------
// device LRU cache (one block)
//   One pool of S slots shared by all layers; table[l*E+e] -> slot, owner[s]
//   -> key, stamp[s] recency (0 = never filled). A batch serves the ascending,
//   distinct experts of one layer at clock c = ++clock; member p gets stamp
//   c*65536 + p. Hits only restamp. Misses, in member order, take the slots
//   with the smallest (stamp, slot index) among slots holding neither a member
//   nor a protected key. A prefill call with prefetch enabled, layer+1 < L and
//   S >= n_uniq + E then runs a second batch over all E experts of layer+1,
//   protecting this layer's experts.
// --------------------------------------------------------------------------

constexpr int kLruThreads = 1024;

struct LruSmem {
    uint32_t blocked[kMaxSlots / 32];
    int32_t member_slot[kMaxExperts];
    int32_t member_old[kMaxExperts];
    int32_t miss_p[kMaxExperts];
    int32_t victim[kMaxExperts];
    int32_t scan[kLruThreads / 32];
    unsigned long long red_key[kLruThreads / 32];
    int32_t n_miss, n_free, status;
    unsigned long long clock;
};

__device__ __forceinline__ unsigned long long slot_key(const unsigned long long* stamp, int s) {
    return (stamp[s] << 14) | static_cast<unsigned long long>(s);
}

// returns number of misses, or -1 (not enough slots; nothing changed)
__device__ int lru_batch(const CallArgs& a, LruSmem& sm, unsigned long long* skeys, int layer,
                         const int32_t* members, int n, const int32_t* protect, int n_protect,
                         int32_t protect_layer, bool is_prefetch) {
    const int tid = threadIdx.x, S = a.S, E = a.E;
    for (int i = tid; i < (S + 31) / 32; i += blockDim.x) sm.blocked[i] = 0u;
    if (tid == 0) { sm.n_miss = 0; sm.n_free = 0; }
    __syncthreads();
    for (int p = tid; p < n; p += blockDim.x) {
        const int s = a.table[layer * E + members[p]];
        sm.member_slot[p] = s;
        sm.member_old[p] = -1;
        if (s >= 0) atomicOr(&sm.blocked[s >> 5], 1u << (s & 31));
    }
    for (int q = tid; q < n_protect; q += blockDim.x) {
        const int s = a.table[protect_layer * E + protect[q]];
        if (s >= 0) atomicOr(&sm.blocked[s >> 5], 1u << (s & 31));
    }
    __syncthreads();
    // misses in member order (prefix over chunks of blockDim)
    int running = 0;
    for (int base = 0; base < n; base += blockDim.x) {
        const int p = base + tid;
        const int m = (p < n && sm.member_slot[p] < 0) ? 1 : 0;
        const unsigned bal = __ballot_sync(0xffffffffu, m);
        const int lane = tid & 31, warp = tid >> 5;
        if (lane == 0) sm.scan[warp] = __popc(bal);
        __syncthreads();
        int wb = 0, tot = 0;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
            if (w < warp) wb += sm.scan[w];
            tot += sm.scan[w];
        }
        if (m) sm.miss_p[running + wb + __popc(bal & ((1u << lane) - 1u))] = p;
        running += tot;
        __syncthreads();
    }
    int nfree = 0;
    for (int s = tid; s < S; s += blockDim.x) nfree += !((sm.blocked[s >> 5] >> (s & 31)) & 1u);
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
    for (int p = tid; p < n; p += blockDim.x)
        if (sm.member_slot[p] >= 0) a.stamp[sm.member_slot[p]] = (c << 16) | static_cast<unsigned long long>(p);
    // victims: the m smallest (stamp, slot) keys among unblocked slots
    if (m > 0 && m <= 32) {
        for (int r = 0; r < m; ++r) {
            unsigned long long best = ~0ull;
            for (int s = tid; s < S; s += blockDim.x)
                if (!((sm.blocked[s >> 5] >> (s & 31)) & 1u)) {
                    const unsigned long long kk = slot_key(a.stamp, s);
                    best = kk < best ? kk : best;
                }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) {
                const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
                best = y < best ? y : best;
            }
            if ((tid & 31) == 0) sm.red_key[tid >> 5] = best;
            __syncthreads();
            if (tid == 0) {
                unsigned long long b = ~0ull;
                for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) b = sm.red_key[w] < b ? sm.red_key[w] : b;
                const int v = static_cast<int>(b & 0x3FFFull);
                sm.victim[r] = v;
                sm.blocked[v >> 5] |= 1u << (v & 31);
            }
            __syncthreads();
        }
    } else if (m > 32) {
        int P = 1;
        while (P < S) P <<= 1;
        for (int s = tid; s < P; s += blockDim.x)
            skeys[s] = (s < S && !((sm.blocked[s >> 5] >> (s & 31)) & 1u)) ? slot_key(a.stamp, s) : ~0ull;
        __syncthreads();
        for (int kk = 2; kk <= P; kk <<= 1) {
            for (int j = kk >> 1; j > 0; j >>= 1) {
                for (int i = tid; i < P; i += blockDim.x) {
                    const int ixj = i ^ j;
                    if (ixj > i) {
                        const bool up = (i & kk) == 0;
                        const unsigned long long x = skeys[i], y = skeys[ixj];
                        if ((x > y) == up) { skeys[i] = y; skeys[ixj] = x; }
                    }
                }
                __syncthreads();
            }
        }
        for (int r = tid; r < m; r += blockDim.x) sm.victim[r] = static_cast<int>(skeys[r] & 0x3FFFull);
        __syncthreads();
    }
    // fill the victims
    for (int r = tid; r < m; r += blockDim.x) {
        const int p = sm.miss_p[r];
        const int v = sm.victim[r];
        const int32_t key = layer * E + members[p];
        const int32_t old = a.owner[v];
        if (old >= 0) a.table[old] = -1;
        a.owner[v] = key;
        a.table[key] = v;
        a.stamp[v] = (c << 16) | static_cast<unsigned long long>(p);
        sm.member_slot[p] = v;
        sm.member_old[p] = old;
    }
    __syncthreads();
    (void)is_prefetch;
    return m;
}

__global__ void __launch_bounds__(kLruThreads) k_lru(CallArgs a) {
    extern __shared__ __align__(16) unsigned char lru_dyn[];
    __shared__ LruSmem sm;
    __shared__ int32_t s_members[kMaxExperts];
    unsigned long long* skeys = reinterpret_cast<unsigned long long*>(lru_dyn);
    CallInfo* info = a.info;
    const int tid = threadIdx.x, E = a.E;
    const int nu = *a.n_uniq;
    for (int i = tid; i < nu; i += blockDim.x) s_members[i] = a.act_expert[i];
    __syncthreads();
    const int m = lru_batch(a, sm, skeys, a.layer, s_members, nu, nullptr, 0, 0, false);
    if (m < 0) {
        if (tid == 0) {
            info->status = -4;  // MOE_ERR_CAPACITY
            info->n_uniq = nu;
            info->n_hit = info->n_miss = info->n_pf = info->n_pf_hit = info->n_pf_miss = 0;
            info->n_events = 0;
            info->dev_err = *reinterpret_cast<volatile int32_t*>(a.dev_err);
            *a.n_active = 0;
        }
        return;
    }
    // demand results
    for (int p = tid; p < nu; p += blockDim.x) {
        const int s = sm.member_slot[p];
        a.act_ptr[p] = a.pool + static_cast<size_t>(s) * a.lay.bytes;
        a.act_slot[p] = s;
        info->ev_layer[p] = a.layer;
        info->ev_expert[p] = s_members[p];
        info->ev_hit[p] = sm.member_old[p] == -1 && 0;  // set below
        info->ev_slot[p] = s;
        info->ev_evicted[p] = sm.member_old[p];
        info->ev_prefetch[p] = 0;
    }
    // hit flags: a member is a miss iff it appears in miss_p[0..m)
    __syncthreads();
    for (int p = tid; p < nu; p += blockDim.x) info->ev_hit[p] = 1;
    __syncthreads();
    for (int r = tid; r < m; r += blockDim.x) {
        const int p = sm.miss_p[r];
        info->ev_hit[p] = 0;
        info->miss_layer[r] = a.layer;
        info->miss_expert[r] = s_members[p];
        info->miss_slot[r] = sm.member_slot[p];
    }
    __syncthreads();
    int n_pf = 0, m_pf = 0;
    const bool do_pf = a.prefetch && a.T > kDecodeMaxT && a.layer + 1 < a.L && a.S >= nu + E;
    if (do_pf) {
        // protect this layer's experts (still listed in s_members), members = all E of layer+1
        __shared__ int32_t s_all[kMaxExperts];
        for (int i = tid; i < E; i += blockDim.x) s_all[i] = i;
        __syncthreads();
        m_pf = lru_batch(a, sm, skeys, a.layer + 1, s_all, E, s_members, nu, a.layer, true);
        n_pf = E;
        if (m_pf < 0) { m_pf = 0; n_pf = 0; }  // cannot happen when S >= nu + E
        for (int p = tid; p < n_pf; p += blockDim.x) {
            info->ev_layer[nu + p] = a.layer + 1;
            info->ev_expert[nu + p] = p;
            info->ev_hit[nu + p] = 1;
            info->ev_slot[nu + p] = sm.member_slot[p];
            info->ev_evicted[nu + p] = sm.member_old[p];
            info->ev_prefetch[nu + p] = 1;
        }
        __syncthreads();
        for (int r = tid; r < m_pf; r += blockDim.x) {
            const int p = sm.miss_p[r];
            info->ev_hit[nu + p] = 0;
            info->miss_layer[m + r] = a.layer + 1;
            info->miss_expert[m + r] = p;
            info->miss_slot[m + r] = sm.member_slot[p];
        }
    }
    // shared experts: resident, after the routed ones in the active list
    const int T = a.T, k = a.k;
    for (int s = 0; s < a.n_shared; ++s) {
        const int u = nu + s;
        if (tid == 0) {
            a.act_expert[u] = E + s;
            a.act_row0[u] = T * k + s * T;
            a.act_cnt[u] = T;
            a.act_ptr[u] = a.shared_base + static_cast<size_t>(s) * a.lay.bytes;
            a.act_slot[u] = -(1 + a.layer * a.n_shared + s);
        }
        for (int t = tid; t < T; t += blockDim.x) {
            a.row_tok[T * k + s * T + t] = t;
            a.row_gate[T * k + s * T + t] = 1.0f;
            if (T <= kDecodeMaxT) a.tok_row[u * kDecodeMaxT + t] = T * k + s * T + t;
        }
    }
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

cudaError_t launch_router(const CallArgs& a, cudaStream_t s) {
    if (a.fmt != FMT_FP32) {
        const size_t n4 = static_cast<size_t>(a.T) * a.H / 4;
        const int blocks = static_cast<int>(std::min<size_t>((n4 + 255) / 256, 148 * 8));
        const bool f16 = a.fmt != FMT_BF16;
        if (a.act == ACT_BF16) {
            if (f16) k_xprep<ACT_BF16, true><<<blocks, 256, 0, s>>>(a.hidden, a.xh, a.T, a.H);
            else k_xprep<ACT_BF16, false><<<blocks, 256, 0, s>>>(a.hidden, a.xh, a.T, a.H);
        } else {
            if (f16) k_xprep<ACT_FP32, true><<<blocks, 256, 0, s>>>(a.hidden, a.xh, a.T, a.H);
            else k_xprep<ACT_FP32, false><<<blocks, 256, 0, s>>>(a.hidden, a.xh, a.T, a.H);
        }
    }
    const size_t smem = static_cast<size_t>(8) * a.H * (a.act == ACT_BF16 ? 2 : 4);
    const int ty = (a.T + 7) / 8;
    if (a.T <= kDecodeMaxT) {
        dim3 grid((a.E + 7) / 8, ty);
        if (a.act == ACT_BF16) k_logits<ACT_BF16, 1><<<grid, 256, smem, s>>>(a);
        else k_logits<ACT_FP32, 1><<<grid, 256, smem, s>>>(a);
    } else {
        dim3 grid((a.E + 15) / 16, ty);
        if (a.act == ACT_BF16) k_logits<ACT_BF16, 2><<<grid, 256, smem, s>>>(a);
        else k_logits<ACT_FP32, 2><<<grid, 256, smem, s>>>(a);
    }
    k_topk<<<(a.T + 7) / 8, 256, 0, s>>>(a);
    k_perm<<<a.E, kPermThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_cache(const CallArgs& a, cudaStream_t s) {
    int P = 1;
    while (P < a.S) P <<= 1;
    const size_t dyn = static_cast<size_t>(P) * sizeof(unsigned long long);
    k_lru<<<1, kLruThreads, dyn, s>>>(a);
    return cudaGetLastError();
}

// dynamic shared memory limits are raised once per process
cudaError_t routing_set_attributes() {
    cudaError_t e;
    const int big = 200 * 1024;
    if ((e = cudaFuncSetAttribute(k_logits<ACT_BF16, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, big))) return e;
    if ((e = cudaFuncSetAttribute(k_logits<ACT_BF16, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, big))) return e;
    if ((e = cudaFuncSetAttribute(k_logits<ACT_FP32, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, big))) return e;
    if ((e = cudaFuncSetAttribute(k_logits<ACT_FP32, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, big))) return e;
    const int lru = static_cast<int>(kSortMax * sizeof(unsigned long long));
    if ((e = cudaFuncSetAttribute(k_lru, cudaFuncAttributeMaxDynamicSharedMemorySize, lru))) return e;
    return cudaSuccess;
}

}  // namespace moe
