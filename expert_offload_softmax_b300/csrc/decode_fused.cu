// Decode call of the routed MoE layer (T <= 8 tokens, FP4 or FP8 expert weights) in
// one cooperative launch: router logits, softmax / top-k / renormalisation,
// the permutation by expert, the device LRU lookup of the expert cache, the
// copy of missed experts from the pinned host banks into their pool slots,
// gate/up + SwiGLU, and down + gate-weighted combine.
//
// Follows "FreeToken量子化：MoE推論のセットアップガイド" (freetoken.wiki,
// architecture page, decode paragraph): an LRU over recently selected experts;
// a hit runs on the GPU, a miss is copied into the cache over PCIe. Here the
// copy is made by the kernel itself, reading the pinned host bank through its
// mapped device view, so a call with misses needs no host round trip (with the
// cache flag MOE_CACHE_HOST_MISSES the host's copy engines do it instead, and
// the kernel waits for the release the host posts after them).
//
// At T <= 8 the layer is bound by streaming the active experts' packed
// weights from HBM once; the arithmetic is tiny. Phases:
//  P1  every CTA stages the token rows in shared memory; warps compute router
//      logits (one warp per expert, in the fixed summation order) into global
//      scratch; grid barrier.
//  P2  every CTA computes the same top-k, permutation and expert plan from the
//      logits and looks the experts up in the LRU table; CTA 0 alone updates
//      the LRU (stamps, victims), publishes the slots of the misses and writes
//      the call record the host reads for its statistics. With misses, all
//      CTAs copy the missed blobs (host -> pool slot) in parallel; barrier.
//  P3  warp 0 of each CTA streams 16-row weight tiles with cp.async.bulk into
//      a ring of shared-memory stages (mbarriers); warps 1-16 consume them with
//      mma.sync m16n8k16 (swap-AB: 16 weight rows x 8 token columns). Phase 1:
//      h = gate * silu(W_gate x) * (W_up x); barrier (the producer keeps
//      streaming phase-2 tiles across it); phase 2: out[t] = sum over experts
//      of W_down h. Each tile's K range is split over the 16 consumer warps; the
//      warp that finishes a tile last sums the 16 partials in warp order and
//      writes the result, so the reduction order is fixed.
//
// Exact arithmetic of the operands. NVFP4: code (E2M1) and block scale (E4M3)
// are both widened to f16 and multiplied there: the product has at most 6
// significant bits and lies in [2^-10, 2688], so it is exact in f16; the fp32
// per-tensor scale is applied after the dot product. MXFP4: the E8M0 scale is
// applied in fp32 to each 32-element partial sum. FP8: E4M3 codes are exact in
// f16 (|code| in [2^-9, 448]); the per-tensor scale comes after the dot
// product, as for NVFP4. Activations: each token row
// is scaled by a power of two so that its largest |x| lies in [2^14, 2^15)
// before rounding to f16 (exact for every element the f16 normal range holds),
// and h rows likewise by their token's largest |h|; the power of two is undone
// in fp32 after the dot product. So neither the bf16 range of the layer's
// inputs nor that of h is narrowed to f16's.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "mma_common.cuh"
#include "moe_internal.h"
#include "route_common.cuh"

namespace moe {
namespace {

constexpr int kConsumers = 16;
constexpr int kWarps = kConsumers + 1;
constexpr int kThreads = 32 * kWarps;
static_assert(kDecodeMaxT * kMaxTopK < 32 * kWarps, "one assignment per thread in the routing counts");
constexpr int kStageGroups = 2 * kChunkGroups;  // K groups (16 rows x 128) per pipeline stage
constexpr int kMaxStages = 12;
constexpr int kMaxAssign = kDecodeMaxT * kMaxTopK;
constexpr int kSlotsPerWarp = kStageGroups / kConsumers;  // K groups of a stage per consumer warp
static_assert(kStageGroups % kConsumers == 0, "a stage's groups split evenly over the consumer warps");
constexpr int kRedSlotBytes = kConsumers * 32 * 4 * 4;  // one tile's partial accumulators, one per consumer warp
constexpr int kRedSlots = 4;                            // tiles whose reduction can be in flight
constexpr int kSmemLimit = 220 * 1024;                  // dynamic bytes; a few KB static sit beside it
constexpr int kLruCached = 4096;                        // pools up to this size cache stamps/owners in smem

template <int FMT>
struct Fp4Cfg {
    static constexpr int kSbpg = tiled_scale_bytes(FMT);
    static constexpr int kRowBytes = tiled_row_bytes(FMT);  // one tile row of one K group
    static constexpr int kChunkBytes = kTileRows * kChunkGroups * kRowBytes;
    static constexpr int kStageBytes = 2 * kChunkBytes;
};

// per-CTA routing state (front of dynamic shared memory)
struct DecRoute {
    int32_t tk[kMaxAssign];       // expert of assignment a = t*k + j
    float g[kMaxAssign];          // its gate
    int32_t rank[kMaxAssign];     // its row: stable order by expert
    int32_t uidx[kMaxAssign];     // active index of its expert
    int32_t first[kMaxAssign];    // 1: the lowest assignment of its expert
    int32_t members[kMaxAssign];  // ascending distinct experts
    int32_t mslot[kMaxAssign];    // their pool slots (-1: miss, until the cache update assigns one)
    int32_t hit[kMaxAssign];      // 1: the member was in the cache
    int32_t missr[kMaxAssign];    // member index of the r-th miss
    int32_t rowtok[kMaxAssign + kDecodeMaxT];  // token of h row r
    int32_t trow[kMaxExperts];    // this layer's LRU table row as it was before the call
    float xsc[kDecodeMaxT], xun[kDecodeMaxT];  // activation power-of-two scale and its inverse
    float hsc[kDecodeMaxT], hun[kDecodeMaxT];
    unsigned int xmax[kDecodeMaxT], hmax[kDecodeMaxT];
    int32_t red_cnt[kRedSlots];   // arrivals at each reduction slot
    int32_t red_gen[kRedSlots];   // uses of each slot finished
    int32_t nu, n_miss, status, ok;
    unsigned long long t_copy0;
    unsigned long long seqbuf[24];  // T = 1: this CTA's stage sequence, set up while P1 waits for its rows
    unsigned long long tks[kDecodeMaxT][32];  // top-k scratch of token t's warp
};

// dynamic shared memory carve-up, computed on the host
struct DecGeom {
    int nst;          // pipeline stages
    int max_active;   // plan records
    int act_bytes;    // token rows (phase 1) / h rows (phase 2) in smem; 0: read from global
    int plan_off, ring_off, red_off, act_off, total;
    int stage_x;      // 1: P1 stages the raw token rows and this CTA's router rows at ring_off
    int lru_trow_off, lru_keys_off, lru_cache_off;  // CTA 0's cache-lookup scratch (aliases the ring)
};

__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
// suspends for up to ~20 us waiting for the phase of parity `parity`
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 20000;\n"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// bounded by wait_ns; false on abort or timeout
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                          unsigned long long wait_ns) {
    if (mbar_test(b, parity)) return true;
    const uint64_t t0 = gtimer();
    for (;;) {
        if (mbar_test(b, parity)) return true;
        if (*abort_flag) return false;
        if (gtimer() - t0 > wait_ns) return false;
    }
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(su32(dst)),
        "l"(src), "r"(bytes), "r"(su32(bar))
        : "memory");
}
// The same copy with an L2 eviction priority: expert weights stream through L2
// once per call (evict first), so that they do not push out what every call
// reuses (router rows, LRU state, the kernel's own code), which is kept with
// evict last.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            su32(dst)),
        "l"(src), "r"(bytes), "r"(su32(bar)), "l"(policy)
        : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_gpu64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_gpu64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumers) : "memory"); }
__device__ __forceinline__ uint4 lds128(const unsigned char* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ unsigned long long ld_relaxed_gpu64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
// Row `src` of the tagged decode logits into dst (E floats), waiting (bounded)
// for every entry to carry this call's sequence number: each entry is one
// 64-bit store, so the value is read together with the tag that validates it
// and no separate barrier is needed. False on timeout (this lane).
__device__ __forceinline__ bool poll_logits(const unsigned long long* src, int E, uint32_t seq, float* dst, int lane,
                                            unsigned long long wait_ns);

__device__ __forceinline__ void red_release_add64(unsigned long long* p, unsigned long long v) {
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ bool poll_logits(const unsigned long long* src, int E, uint32_t seq, float* dst, int lane,
                                            unsigned long long wait_ns) {
    const uint64_t t0 = gtimer();
    for (int base = 0; base < E; base += 256) {
        unsigned long long v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = base + lane + 32 * i;
            v[i] = e < E ? ld_relaxed_gpu64(src + e) : static_cast<unsigned long long>(seq) << 32;
        }
        for (;;) {
            bool done = true;
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (static_cast<uint32_t>(v[i] >> 32) != seq) {
                    done = false;
                    v[i] = ld_relaxed_gpu64(src + base + lane + 32 * i);
                }
            if (done) break;
            if (gtimer() - t0 > wait_ns) return false;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int e = base + lane + 32 * i;
            if (e < E) dst[e] = __uint_as_float(static_cast<uint32_t>(v[i]));
        }
    }
    return true;
}

// Grid-wide barriers on monotone arrival counters (never reset between calls):
// barrier k of a call has P participants, and every decode call adds exactly P
// to counter k (a call that skips the barrier adds the missing arrivals in one
// step), so the call's target is (calls before it + 1) * P, which the host
// passes. Arriving is a release add (it publishes the CTA's writes); waiting
// is one thread polling with relaxed loads, then an acquire fence.
__device__ __forceinline__ void bar_arrive(unsigned long long* cnt, unsigned long long n) { red_release_add64(cnt, n); }

__device__ __forceinline__ bool bar_wait(const CallArgs& a, const unsigned long long* cnt, unsigned long long target, int err_code) {
    if (ld_relaxed_gpu64(cnt) < target) {
        const uint64_t t0 = gtimer();
        while (ld_relaxed_gpu64(cnt) < target) {
            if (gtimer() - t0 > a.wait_ns) {
                atomicExch(a.dev_err, err_code);
                return false;
            }
        }
    }
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    return true;
}

// f16 of v * sc, two at a time (round to nearest)
__device__ __forceinline__ uint32_t f16x2_scaled(float lo, float hi, float sc) {
    __half2 h = __floats2half2_rn(lo * sc, hi * sc);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t hmul2u(uint32_t a, uint32_t b) {
    __half2 r = __hmul2(*reinterpret_cast<__half2*>(&a), *reinterpret_cast<__half2*>(&b));
    return *reinterpret_cast<uint32_t*>(&r);
}

// One 128-element K group of a staged 16-row chunk (ng groups) against one
// 8-column B run: acc0 + acc1 (rows g / g+8, columns 2q / 2q+1) += the group's
// dot products. NVFP4 (scale folded into the f16 operand): accumulates in the
// MMA, even steps into acc0 and odd steps into acc1 (two independent chains,
// so consecutive MMAs of a warp do not wait for each other). MXFP4: each
// 32-element block (two MMA steps from zero) times its E8M0 scale, in fp32,
// into acc0.
template <int FMT>
__device__ __forceinline__ void mma_group(const unsigned char* chunk, int ng, int w, int g, int q,
                                          const uint32_t (&b)[16], float (&acc0)[4], float (&acc1)[4]) {
    constexpr int kSbpg = Fp4Cfg<FMT>::kSbpg;
    if constexpr (FMT == FMT_FP8) {
        // E4M3 codes widen to f16 exactly; the per-tensor scale comes after
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const uint4 ra = lds128(chunk + fp8_code_off(ng, g, w, q, hf));
            const uint4 rb = lds128(chunk + fp8_code_off(ng, g + 8, w, q, hf));
            uint32_t oa[8], ob[8];
            e4m3x8_to_f16x2(make_uint2(ra.x, ra.y), *reinterpret_cast<uint32_t(*)[4]>(oa));
            e4m3x8_to_f16x2(make_uint2(ra.z, ra.w), *reinterpret_cast<uint32_t(*)[4]>(oa + 4));
            e4m3x8_to_f16x2(make_uint2(rb.x, rb.y), *reinterpret_cast<uint32_t(*)[4]>(ob));
            e4m3x8_to_f16x2(make_uint2(rb.z, rb.w), *reinterpret_cast<uint32_t(*)[4]>(ob + 4));
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const int s = 4 * hf + x;  // MMA step: word x of the half, elements i = 0, 1 | 2, 3
                const uint32_t A[4] = {oa[2 * x], ob[2 * x], oa[2 * x + 1], ob[2 * x + 1]};
                if (s & 1) mma_f16(acc1, A, b[2 * s], b[2 * s + 1], acc1);
                else mma_f16(acc0, A, b[2 * s], b[2 * s + 1], acc0);
            }
        }
        return;
    }
    const uint4 ra = lds128(chunk + fp4_code_off(ng, g, w, q));
    const uint4 rb = lds128(chunk + fp4_code_off(ng, g + 8, w, q));
    const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
    if constexpr (FMT == FMT_NVFP4) {
        uint32_t fa[4], fb[4];
        e4m3x8_to_f16x2(*reinterpret_cast<const uint2*>(chunk + fp4_scale_off(ng, kSbpg, g, w)), fa);
        e4m3x8_to_f16x2(*reinterpret_cast<const uint2*>(chunk + fp4_scale_off(ng, kSbpg, g + 8, w)), fb);
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            uint32_t oa[4], ob[4];
            fp4x8_to_f16x2(wa[x], oa);
            fp4x8_to_f16x2(wb[x], ob);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int s = 2 * x + h;  // MMA step; its 16 elements share one scale per row
                const uint32_t sel = (s & 1) ? 0x3232u : 0x1010u;
                const uint32_t sa = __byte_perm(fa[s >> 1], 0u, sel), sb = __byte_perm(fb[s >> 1], 0u, sel);
                const uint32_t A[4] = {hmul2u(oa[2 * h], sa), hmul2u(ob[2 * h], sb), hmul2u(oa[2 * h + 1], sa),
                                       hmul2u(ob[2 * h + 1], sb)};
                if (h == 0) mma_f16(acc0, A, b[2 * s], b[2 * s + 1], acc0);
                else mma_f16(acc1, A, b[2 * s], b[2 * s + 1], acc1);
            }
        }
    } else {
        const uint32_t va = *reinterpret_cast<const uint32_t*>(chunk + fp4_scale_off(ng, kSbpg, g, w));
        const uint32_t vb = *reinterpret_cast<const uint32_t*>(chunk + fp4_scale_off(ng, kSbpg, g + 8, w));
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            uint32_t oa[4], ob[4];
            fp4x8_to_f16x2(wa[x], oa);
            fp4x8_to_f16x2(wb[x], ob);
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int s = 2 * x + h;
                const uint32_t A[4] = {oa[2 * h], ob[2 * h], oa[2 * h + 1], ob[2 * h + 1]};
                mma_f16(d, A, b[2 * s], b[2 * s + 1], d);
            }
            const float sa = e8m0_to_f32((va >> (8 * x)) & 0xFFu), sb = e8m0_to_f32((vb >> (8 * x)) & 0xFFu);
            acc0[0] = __fmaf_rn(sa, d[0], acc0[0]);
            acc0[1] = __fmaf_rn(sa, d[1], acc0[1]);
            acc0[2] = __fmaf_rn(sb, d[2], acc0[2]);
            acc0[3] = __fmaf_rn(sb, d[3], acc0[3]);
        }
    }
}

// B run of one column for K group j: 32 f16 at device positions
// [128 j + 32 q, +32). From the staged rows (pitch bytes apart), or, when the
// rows did not fit in shared memory, converted here from global memory: token
// rows (x, canonical element order) or h rows (bf16, device order).
__device__ __forceinline__ void load_b_smem(const unsigned char* rows, int pitch, int r, int j, int q,
                                            uint32_t (&bq)[16]) {
    if (r < 0) {
#pragma unroll
        for (int i = 0; i < 16; ++i) bq[i] = 0u;
        return;
    }
    const unsigned char* p = rows + r * pitch + j * 256 + 64 * q;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const uint4 x = lds128(p + 16 * v);
        bq[4 * v] = x.x; bq[4 * v + 1] = x.y; bq[4 * v + 2] = x.z; bq[4 * v + 3] = x.w;
    }
}

template <int ACT>
__device__ __forceinline__ void load_b_xglobal(const void* hidden, int H, int t, int j, int q, float sc,
                                               uint32_t (&bq)[16]) {
    if (t < 0) {
#pragma unroll
        for (int i = 0; i < 16; ++i) bq[i] = 0u;
        return;
    }
    // device position 32q + 4s + i of group j holds element 16s + 4q + i
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        const size_t e0 = static_cast<size_t>(t) * H + 128 * j + 16 * s + 4 * q;
        float v[4];
        if constexpr (ACT == ACT_BF16) {
            const uint2 u = __ldg(reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(hidden) + e0));
            v[0] = __uint_as_float(u.x << 16); v[1] = __uint_as_float(u.x & 0xFFFF0000u);
            v[2] = __uint_as_float(u.y << 16); v[3] = __uint_as_float(u.y & 0xFFFF0000u);
        } else {
            const float4 f = __ldg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(hidden) + e0));
            v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
        }
        bq[2 * s] = f16x2_scaled(v[0], v[1], sc);
        bq[2 * s + 1] = f16x2_scaled(v[2], v[3], sc);
    }
}

__device__ __forceinline__ void load_b_hglobal(const uint16_t* hbuf, int I, int r, int j, int q, float sc,
                                               uint32_t (&bq)[16]) {
    if (r < 0) {
#pragma unroll
        for (int i = 0; i < 16; ++i) bq[i] = 0u;
        return;
    }
    const uint4* p = reinterpret_cast<const uint4*>(hbuf + static_cast<size_t>(r) * I + j * 128 + 32 * q);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const uint4 x = __ldcg(p + v);
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            bq[4 * v + i] = f16x2_scaled(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u), sc);
    }
}

// A pipeline stage: up to 16 K groups of 16 weight rows, made of one or more
// contiguous pieces of the blobs (one cp.async.bulk each).
// The stage sequence of one CTA, identical for its producer and consumers.
// CTA 0 runs the cache update and takes no tiles; CTA b >= 1 is worker b1 = b-1
// of G1 = G-1.
//  phase 1: gate/up tiles i = b1, b1 + G1, ... (active expert u = i / (I/8),
//           unit tile i mod (I/8)); a stage = up to two 8-group chunks.
//  phase 2: down row tiles rt = b1, b1 + G1, ...; for each, every active expert's
//           16-row tile: up to two chunks of one expert per stage when I >= 1024,
//           else the whole tiles of several experts (16 groups at most).
template <int FMT>
struct StageSeq {
    // blob offsets of the gate/up and down tiles and their strides, copied from
    // the kernel's arguments: a load through a pointer to a kernel argument is
    // a memory round trip, a register is not
    size_t gu, gu_tile, d, d_tile;
    const DecExpert* plan;
    int na, b1, G1;
    int UT, G1k, nch1, ns1, n1, my1, G1q, G1r;  // phase 1
    int G2k, nch2, nsu, epp, ns2, n2, my2;      // phase 2
    // Cursor: the stage this copy of the sequence stands at. The producer and
    // each consumer walk the stages in order, so the position advances by
    // additions; integer division (a long dependent chain on the GPU) only
    // runs once, here.
    int f, nf1;
    int u, ut, cs;        // phase 1: active expert, its unit tile, chunk step
    int rt, k2, u0, csu;  // phase 2: row tile, stage within it, first expert, chunk step

    __device__ void init(const CallArgs& ca, const DecExpert* pl, int na_, int blk, int grid) {
        gu = ca.lay.gu;
        gu_tile = ca.lay.gu_tile;
        d = ca.lay.d;
        d_tile = ca.lay.d_tile;
        plan = pl;
        na = na_;
        G1 = grid > 1 ? grid - 1 : 1;
        b1 = grid > 1 ? blk - 1 : blk;
        UT = ca.I / 8;
        G1k = ca.H / kGroupK;
        nch1 = (G1k + kChunkGroups - 1) / kChunkGroups;
        ns1 = (nch1 + 1) / 2;
        n1 = na * UT;
        my1 = (b1 >= 0 && b1 < n1) ? (n1 - 1 - b1) / G1 + 1 : 0;
        G1q = G1 / UT;
        G1r = G1 - G1q * UT;
        u = b1 >= 0 ? b1 / UT : 0;
        ut = b1 >= 0 ? b1 - u * UT : 0;
        cs = 0;
        G2k = ca.I / kGroupK;
        nch2 = (G2k + kChunkGroups - 1) / kChunkGroups;
        if (G2k >= kChunkGroups) {
            nsu = (nch2 + 1) / 2;
            epp = 1;
            ns2 = na * nsu;
        } else {
            nsu = 1;
            epp = kStageGroups / G2k;
            ns2 = (na + epp - 1) / epp;
        }
        n2 = ca.H / kTileRows;
        my2 = (b1 >= 0 && b1 < n2) ? (n2 - 1 - b1) / G1 + 1 : 0;
        rt = b1;
        k2 = u0 = csu = 0;
        f = 0;
        nf1 = my1 * ns1;
    }
    __device__ int count1() const { return my1 * ns1; }
    __device__ int count2() const { return my2 * ns2; }

    // phase 1, the current stage: chunks [c0, c0 + nc) of tile (u, ut); the
    // tile's last stage when cs == ns1 - 1
    __device__ int c0_1() const { return 2 * cs; }
    __device__ int nc_1() const { return min(2, nch1 - 2 * cs); }
    __device__ bool end1() const { return cs == ns1 - 1; }
    // phase 2, the current stage: row tile rt; experts [u0, u0 + nu); chunks
    // [c0, c0 + nc) of one expert, or the whole tiles of several
    __device__ void where2(int& rt_, int& u0_, int& nu_, int& c0, int& nc) const {
        rt_ = rt;
        u0_ = u0;
        if (epp == 1) {
            nu_ = 1;
            c0 = 2 * csu;
            nc = min(2, nch2 - c0);
        } else {
            nu_ = min(epp, na - u0);
            c0 = 0;
            nc = 1;
        }
    }
    __device__ bool end2() const { return k2 == ns2 - 1; }
    __device__ void advance() {
        if (f < nf1) {
            if (++cs == ns1) {  // next tile: i += G1
                cs = 0;
                u += G1q;
                ut += G1r;
                if (ut >= UT) {
                    ut -= UT;
                    ++u;
                }
            }
        } else {
            if (epp == 1) {
                if (++csu == nsu) {
                    csu = 0;
                    ++u0;
                }
            } else {
                u0 += epp;
            }
            if (++k2 == ns2) {  // next row tile
                k2 = u0 = csu = 0;
                rt += G1;
            }
        }
        ++f;
    }

    // Copy number `lane` of the current stage (all in registers: the producer
    // issues one copy per lane): its source, size and offset in the stage;
    // returns the number of copies of the stage (lanes at or above it have
    // none) and sets the stage's total bytes.
    __device__ int piece(int lane, const uint8_t*& src, uint32_t& bytes, uint32_t& off, uint32_t& total) const {
        constexpr uint32_t row = Fp4Cfg<FMT>::kRowBytes;  // bytes of one row of one K group
        if (f < nf1) {
            const int c0 = c0_1(), nc = nc_1();
            uint32_t g = 0;
            for (int c = c0; c < c0 + nc; ++c) g += fp4_chunk_groups(G1k, c);
            total = static_cast<uint32_t>(kTileRows) * g * row;
            src = plan[u].ptr + gu + static_cast<size_t>(ut) * gu_tile + tile_chunk_off(c0, Fp4Cfg<FMT>::kRowBytes);
            bytes = total;
            off = 0;
            return 1;
        }
        int rt_, u0_, nu_, c0, nc;
        where2(rt_, u0_, nu_, c0, nc);
        const size_t toff = d + static_cast<size_t>(rt_) * d_tile;
        if (epp == 1) {
            uint32_t g = 0;
            for (int c = c0; c < c0 + nc; ++c) g += fp4_chunk_groups(G2k, c);
            total = static_cast<uint32_t>(kTileRows) * g * row;
            src = plan[u0_].ptr + toff + tile_chunk_off(c0, Fp4Cfg<FMT>::kRowBytes);
            bytes = total;
            off = 0;
            return 1;
        }
        const uint32_t pb = static_cast<uint32_t>(kTileRows) * G2k * row;
        total = static_cast<uint32_t>(nu_) * pb;
        const int p = lane < nu_ ? lane : 0;
        src = plan[u0_ + p].ptr + toff;
        bytes = pb;
        off = static_cast<uint32_t>(p) * pb;
        return nu_;
    }
};

// TT: the call's token count when it is fixed at compile time (1: single-token
// decode, whose loops over tokens then fold away), else 0 (T from the call)
template <int FMT, int ACT, int TT>
__global__ void __launch_bounds__(kThreads, 1) k_decode(const __grid_constant__ CallArgs a, const __grid_constant__ DecGeom geo) {
    using C = Fp4Cfg<FMT>;
    extern __shared__ __align__(128) unsigned char dsm[];
    __shared__ __align__(8) uint64_t full[kMaxStages], empty[kMaxStages], p1bar;
    __shared__ int s_abort;

    DecRoute& R = *reinterpret_cast<DecRoute*>(dsm);
    DecExpert* plan = reinterpret_cast<DecExpert*>(dsm + geo.plan_off);
    unsigned char* ring = dsm + geo.ring_off;
    float* red = reinterpret_cast<float*>(dsm + geo.red_off);
    unsigned char* act = dsm + geo.act_off;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, b = blockIdx.x;
    const int T = TT ? TT : a.T, E = a.E, k = a.k, H = a.H, I = a.I, ns = a.n_shared;
    const int n = T * k;
    const int nst = geo.nst;
    const size_t esz = ACT == ACT_BF16 ? 2 : 4;
    const size_t B = a.lay.bytes;
    volatile int* abort_flag = &s_abort;
    // the call's grid barriers: logits written (all CTAs; only when E < G),
    // misses copied (all CTAs), h written (workers 1..G-1)
    const unsigned long long tgt0 = (a.dcall + 1) * static_cast<unsigned long long>(G);
    // decode logits carry the call's sequence number (the entries of earlier
    // calls and of the reset buffer, 0, never match it)
    const unsigned long long tgt2 = (a.dcall + 1) * static_cast<unsigned long long>(G - 1);
    const uint32_t lseq = static_cast<uint32_t>(a.dcall + 1);
    const unsigned long long tag = static_cast<unsigned long long>(lseq) << 32;
    // Every CTA computes logits when E >= G: then a CTA's logits, stored with
    // release semantics after it read its LRU table row, tell the cache-update
    // CTA that the row was read, and no barrier is needed; else barrier 1.
    const bool logits_barrier = E < G;

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumers);
        }
        mbar_init(&p1bar, 1);
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (tid < kRedSlots) {
        R.red_cnt[tid] = 0;
        R.red_gen[tid] = 0;
    }
    if (tid < kDecodeMaxT) {
        R.xmax[tid] = 0u;
        R.hmax[tid] = 0u;
    }
    // programmatic dependent launch: everything the previous call wrote is
    // visible after this; the next call's CTAs may be scheduled as ours exit
    const uint64_t t_entry = a.trace ? gtimer() : 0;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // per-token max |h| of the calls: two arrays by call parity; this call uses
    // its own (zeroed by the previous call, or at moe_cache_config) and zeroes
    // the next call's, which the previous call used and no one reads any more
    if (b == 0 && tid < kDecodeMaxT) a.hmax[((a.dcall + 1) & 1) * kDecodeMaxT + tid] = 0u;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // trace only: per call, the first CTA's entry, CTA 0's return from the
    // dependency wait, the last CTA's exit
    unsigned long long* tcall =
        a.trace ? a.trace + static_cast<size_t>(G) * kTracePoints + (a.dcall % kTraceCalls) * 4 : nullptr;
    if (tcall && tid == 0) {
        atomicMin(tcall, static_cast<unsigned long long>(t_entry));
        if (b == 0) {
            tcall[1] = gtimer();
            // the next call's slot: its CTAs start after every CTA of this one has exited
            unsigned long long* nxt = a.trace + static_cast<size_t>(G) * kTracePoints + ((a.dcall + 1) % kTraceCalls) * 4;
            nxt[0] = ~0ull;
            nxt[2] = 0ull;
        }
    }
    __syncthreads();
    // optional phase timeline (MOE_TRACE): per CTA, %globaltimer at fixed points
    auto mark = [&](int point) {
        if (a.trace) a.trace[static_cast<size_t>(b) * kTracePoints + point] = gtimer();
    };
    if (tid == 0) mark(0);

    // ---------------------------------------------------------------- P1: logits
    // This CTA's experts are e = b, b + G, ...; with the token rows they are
    // staged in shared memory by bulk copies (one round trip), then warp j
    // computes the logits of expert b + j*G for every token.
    const unsigned char* xsrc = reinterpret_cast<const unsigned char*>(a.hidden);
    {
        const uint32_t xbytes = static_cast<uint32_t>(T) * H * static_cast<uint32_t>(esz);
        const uint32_t rbytes = static_cast<uint32_t>(H) * static_cast<uint32_t>(esz);
        const int nexp = b < E ? (E - 1 - b) / G + 1 : 0;
        const bool staged = geo.stage_x != 0;  // token rows and this CTA's router rows fit (host-checked)
        if (staged && tid == 0) {
            mbar_expect_tx(&p1bar, xbytes + static_cast<uint32_t>(nexp) * rbytes);
            bulk_g2s(ring, a.hidden, xbytes, &p1bar);
            const uint64_t keep = l2_evict_last();
            for (int j = 0; j < nexp; ++j)
                bulk_g2s_hint(ring + xbytes + static_cast<size_t>(j) * rbytes,
                              reinterpret_cast<const unsigned char*>(a.router_w) + static_cast<size_t>(b + j * G) * rbytes,
                              rbytes, &p1bar, keep);
        }
        // this layer's table row before anything of this call changes it: CTA 0
        // rewrites entries of missed experts after the barrier below
        for (int e = tid; e < E; e += kThreads) R.trow[e] = __ldcg(a.table + static_cast<size_t>(a.layer) * E + e);
        if (TT == 1 && tid == 32) {
            // at T = 1 the call has k + n_shared active experts whatever the routing:
            // the stage sequence's divisions run here, off the path to P3
            StageSeq<FMT> tmp;
            tmp.init(a, plan, k + ns, b, G);
            *reinterpret_cast<StageSeq<FMT>*>(R.seqbuf) = tmp;
        }
        if (staged) {
            if (!mbar_wait(&p1bar, 0, abort_flag, a.wait_ns)) atomicExch(a.dev_err, MOE_DEVERR_TIMEOUT_PRODUCER);
            xsrc = ring;
        }
        __syncthreads();
        if (tid == 0) mark(10);
        // row maxima of the token rows (every CTA, from its own copy): warp t, token t
        if (kWarps - 1 - warp < T) {  // the last warps, beside the logit warps
            const int t = kWarps - 1 - warp;
            float m = 0.f;
            for (int i = 8 * lane; i < H; i += 8 * 32) {
                float v[8];
                const size_t o = static_cast<size_t>(t) * H + i;
                if constexpr (ACT == ACT_BF16) {
                    const uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(xsrc) + o);
                    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        v[2 * jj] = __uint_as_float(wd[jj] << 16);
                        v[2 * jj + 1] = __uint_as_float(wd[jj] & 0xFFFF0000u);
                    }
                } else {
                    const float4* f = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(xsrc) + o);
                    const float4 p0 = f[0], p1 = f[1];
                    v[0] = p0.x; v[1] = p0.y; v[2] = p0.z; v[3] = p0.w;
                    v[4] = p1.x; v[5] = p1.y; v[6] = p1.z; v[7] = p1.w;
                }
#pragma unroll
                for (int jj = 0; jj < 8; ++jj) m = fmaxf(m, fabsf(v[jj]));
            }
            const unsigned int mb = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
            if (lane == 0) R.xmax[t] = mb;
        }
        // router logits in the fixed order: lane l accumulates chunks l, l+32, ...
        // of 8 elements with fused multiply-adds, then the xor butterfly
        const int nchunk = H / 8;
        // release: this CTA's LRU table read (above, complete at the barrier)
        // precedes the tagged logits below, whose stores are then relaxed
        if (warp < nexp && lane == 0) asm volatile("fence.acq_rel.gpu;" ::: "memory");
        for (int j = warp; j < nexp; j += kWarps) {
            const int e = b + j * G;
            const unsigned char* wrow = staged ? ring + xbytes + static_cast<size_t>(j) * rbytes
                                               : reinterpret_cast<const unsigned char*>(a.router_w) + static_cast<size_t>(e) * rbytes;
            float acc[kDecodeMaxT];
#pragma unroll
            for (int t = 0; t < kDecodeMaxT; ++t) acc[t] = 0.f;
            for (int c = lane; c < nchunk; c += 32) {
                float wv[8];
                if constexpr (ACT == ACT_BF16) {
                    const uint4 u = staged ? *reinterpret_cast<const uint4*>(wrow + 16 * c)
                                           : __ldg(reinterpret_cast<const uint4*>(wrow + 16 * c));
                    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        wv[2 * jj] = __uint_as_float(wd[jj] << 16);
                        wv[2 * jj + 1] = __uint_as_float(wd[jj] & 0xFFFF0000u);
                    }
                } else {
                    const float4* f = reinterpret_cast<const float4*>(wrow + 32 * c);
                    const float4 p0 = staged ? f[0] : __ldg(f), p1 = staged ? f[1] : __ldg(f + 1);
                    wv[0] = p0.x; wv[1] = p0.y; wv[2] = p0.z; wv[3] = p0.w;
                    wv[4] = p1.x; wv[5] = p1.y; wv[6] = p1.z; wv[7] = p1.w;
                }
#pragma unroll
                for (int t = 0; t < kDecodeMaxT; ++t) {
                    if (t < T) {
                        const size_t o = static_cast<size_t>(t) * H + 8 * c;
                        float xv[8];
                        if constexpr (ACT == ACT_BF16) {
                            const uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(xsrc) + o);
                            const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj) {
                                xv[2 * jj] = __uint_as_float(wd[jj] << 16);
                                xv[2 * jj + 1] = __uint_as_float(wd[jj] & 0xFFFF0000u);
                            }
                        } else {
                            const float4* f = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(xsrc) + o);
                            const float4 p0 = f[0], p1 = f[1];
                            xv[0] = p0.x; xv[1] = p0.y; xv[2] = p0.z; xv[3] = p0.w;
                            xv[4] = p1.x; xv[5] = p1.y; xv[6] = p1.z; xv[7] = p1.w;
                        }
#pragma unroll
                        for (int jj = 0; jj < 8; ++jj) acc[t] = __fmaf_rn(xv[jj], wv[jj], acc[t]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < kDecodeMaxT; ++t) {
                if (t < T) {
                    float v = acc[t];
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
                    if (lane == 0) st_relaxed_gpu64(a.dlog + static_cast<size_t>(t) * E + e, tag | __float_as_uint(v));
                }
            }
        }
        __syncthreads();
        // activation scales; token rows -> f16 device order in smem (CTAs with phase-1 work)
        if (tid == 0) mark(11);
        if (tid < kDecodeMaxT) pow2_scale(R.xmax[tid], R.xsc[tid], R.xun[tid]);
        __syncthreads();
        if (geo.act_bytes && b != 0) {
            const int xp = H * 2 + 16;
            const int h4 = H / 4;
            for (int t = 0; t < T; ++t) {
                for (int i4 = tid; i4 < h4; i4 += kThreads) {
                    const int p = 4 * i4;  // device position
                    const int j = p >> 7, w = p & 127, q = w >> 5, s = (w & 31) >> 2;
                    const size_t src = static_cast<size_t>(t) * H + 128 * j + 16 * s + 4 * q;
                    float v[4];
    #pragma unroll
                    for (int i = 0; i < 4; ++i)
                        v[i] = ACT == ACT_BF16
                                   ? __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(xsrc)[src + i]) << 16)
                                   : reinterpret_cast<const float*>(xsrc)[src + i];
                    uint2 o;
                    o.x = f16x2_scaled(v[0], v[1], R.xsc[t]);
                    o.y = f16x2_scaled(v[2], v[3], R.xsc[t]);
                    *reinterpret_cast<uint2*>(act + t * xp + 2 * p) = o;
                }
            }
        }
        __syncthreads();
        if (tid == 0) {
            mark(1);
            R.ok = 1;
            if (logits_barrier) {
                bar_arrive(a.bar_cnt, 1);
                R.ok = bar_wait(a, a.bar_cnt, tgt0, MOE_DEVERR_TIMEOUT_EPILOGUE) ? 1 : 0;
            }
            mark(2);
        }
        __syncthreads();
    }
    if (!R.ok) return;  // every CTA gives up the same way; nothing is in flight

    // ---------------------------------------------------------------- P2: routing (every CTA)
    if (T == 1) {
        // One token: its k experts are distinct, so the expert-major order is
        // the ascending order of the selected experts and every expert has one
        // row. Warp 0 builds the same records as the general path below from
        // registers: lane j < k holds selection j and its rank r.
        if (warp == 0) {
            int sel;
            float gv;
            float* lrow = reinterpret_cast<float*>(ring);  // the staged rows are no longer needed
            const bool got = __all_sync(0xffffffffu, poll_logits(a.dlog, E, lseq, lrow, lane, a.wait_ns));
            if (!got && lane == 0) {
                atomicExch(a.dev_err, MOE_DEVERR_TIMEOUT_EPILOGUE);
                R.ok = 0;
            }
            __syncwarp();
            warp_topk<false>(lrow, E, k, lane, sel, gv, R.tks[0]);
            if (lane == 0) mark(12);
            const bool live = lane < k;
            int r = 0;
            for (int i = 0; i < k; ++i) r += __shfl_sync(0xffffffffu, sel, i) < sel;
            int slot = 0;
            if (live) {
                R.tk[lane] = sel;
                R.g[lane] = gv;
                R.rank[lane] = r;
                R.first[lane] = 1;
                R.uidx[lane] = r;
                R.rowtok[r] = 0;
                R.members[r] = sel;
                slot = R.trow[sel];
                R.mslot[r] = slot;
                R.hit[r] = slot >= 0 ? 1 : 0;
                DecExpert& d = plan[r];
                d.ptr = slot >= 0 ? a.pool + static_cast<size_t>(slot) * B : nullptr;
                d.row0 = r;
                d.cnt = 1;
                // a resident expert's per-tensor scales, now rather than at P3
                d.pad = slot >= 0 ? 1 : 0;
                if (slot >= 0) {
                    if constexpr (FMT == FMT_NVFP4 || FMT == FMT_FP8) {
                        const float4 v = __ldcg(reinterpret_cast<const float4*>(d.ptr + a.lay.gsc));
                        d.gs[0] = v.x;
                        d.gs[1] = v.y;
                        d.gs[2] = v.z;
                    } else {
                        d.gs[0] = d.gs[1] = d.gs[2] = 1.0f;
                    }
                }
#pragma unroll
                for (int t = 0; t < kDecodeMaxT; ++t) {
                    d.tok[t] = t == 0 ? 0 : -1;
                    d.hrow[t] = t == 0 ? r : -1;
                    d.gate[t] = t == 0 ? gv : 0.f;
                }
            }
            // misses in member (rank) order
            const bool miss = live && slot < 0;
            const unsigned int mm = __reduce_or_sync(0xffffffffu, miss ? 1u << r : 0u);
            if (miss) R.missr[__popc(mm & ((1u << r) - 1u))] = r;
            for (int sidx = lane; sidx < ns; sidx += 32) {
                DecExpert& d = plan[k + sidx];
                d.ptr = a.shared_base + static_cast<size_t>(sidx) * B;
                d.row0 = k + sidx;
                d.cnt = 1;
                d.pad = 1;
                if constexpr (FMT == FMT_NVFP4 || FMT == FMT_FP8) {
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(d.ptr + a.lay.gsc));
                    d.gs[0] = v.x;
                    d.gs[1] = v.y;
                    d.gs[2] = v.z;
                } else {
                    d.gs[0] = d.gs[1] = d.gs[2] = 1.0f;
                }
#pragma unroll
                for (int t = 0; t < kDecodeMaxT; ++t) {
                    d.tok[t] = t == 0 ? 0 : -1;
                    d.hrow[t] = t == 0 ? k + sidx : -1;
                    d.gate[t] = t == 0 ? 1.0f : 0.f;
                }
                R.rowtok[k + sidx] = 0;
            }
            if (lane == 0) {
                R.nu = k;
                R.status = k > a.S ? -4 : 0;  // MOE_ERR_CAPACITY
                R.n_miss = __popc(mm);
            }
        }
    } else {
        if (warp < T) {
            int sel;
            float gv;
            float* lrow = reinterpret_cast<float*>(ring) + static_cast<size_t>(warp) * E;
            const bool got =
                __all_sync(0xffffffffu, poll_logits(a.dlog + static_cast<size_t>(warp) * E, E, lseq, lrow, lane, a.wait_ns));
            if (!got && lane == 0) {
                atomicExch(a.dev_err, MOE_DEVERR_TIMEOUT_EPILOGUE);
                R.ok = 0;
            }
            __syncwarp();
            warp_topk<false>(lrow, E, k, lane, sel, gv, R.tks[warp]);
            if (lane < k) {
                R.tk[warp * k + lane] = sel;
                R.g[warp * k + lane] = gv;
            }
        }
        __syncthreads();
        if (tid == 0) mark(12);
        // stable order by expert: row of assignment i = #{j : e_j < e_i or (e_j == e_i and j < i)}
        int my_first = 0;
        for (int i = tid; i < n; i += kThreads) {
            const int e = R.tk[i];
            int rk = 0, first = 1;
    #pragma unroll 16
            for (int j2 = 0; j2 < n; ++j2) {
                const int f = R.tk[j2];
                rk += (f < e) || (f == e && j2 < i);
                first &= !(f == e && j2 < i);
            }
            R.rank[i] = rk;
            R.first[i] = first;
            R.rowtok[rk] = i / k;
            my_first += first;
        }
        const int nu = __syncthreads_count(my_first);  // n <= 256 < threads: one assignment per thread
        for (int i = tid; i < n; i += kThreads) {
            const int e = R.tk[i];
            int u = 0;
    #pragma unroll 16
            for (int j2 = 0; j2 < n; ++j2) u += R.first[j2] && R.tk[j2] < e;
            R.uidx[i] = u;
            if (R.first[i]) R.members[u] = e;
        }
        if (tid == 0) {
            R.nu = nu;
            R.status = nu > a.S ? -4 : 0;  // MOE_ERR_CAPACITY: the call leaves the cache as it was
        }
        __syncthreads();
        const int na = nu + ns;
        for (int u = tid; u < na; u += kThreads) {
            DecExpert& d = plan[u];
            for (int t = 0; t < kDecodeMaxT; ++t) {
                d.tok[t] = -1;
                d.hrow[t] = -1;
                d.gate[t] = 0.f;
            }
            d.cnt = 0;
            d.pad = 0;  // per-tensor scales not loaded yet
            if (u < nu) {
                const int s = R.trow[R.members[u]];
                R.mslot[u] = s;
                R.hit[u] = s >= 0 ? 1 : 0;
                d.ptr = s >= 0 ? a.pool + static_cast<size_t>(s) * B : nullptr;
            } else {
                const int sidx = u - nu;
                d.ptr = a.shared_base + static_cast<size_t>(sidx) * B;
                d.row0 = n + sidx * T;
                d.cnt = T;
                for (int t = 0; t < T; ++t) {
                    d.tok[t] = t;
                    d.hrow[t] = n + sidx * T + t;
                    d.gate[t] = 1.0f;
                }
            }
        }
        for (int i = tid; i < ns * T; i += kThreads) R.rowtok[n + i] = i % T;
        __syncthreads();
        for (int i = tid; i < n; i += kThreads)
            if (R.first[i]) plan[R.uidx[i]].row0 = R.rank[i];
        // the r-th missed member, in member order
        for (int p = tid; p < nu; p += kThreads)
            if (!R.hit[p]) {
                int r = 0;
    #pragma unroll 16
                for (int p2 = 0; p2 < p; ++p2) r += !R.hit[p2];
                R.missr[r] = p;
            }
        const int n_miss_all = __syncthreads_count(tid < nu && !R.hit[tid]);
        if (tid == 0) R.n_miss = n_miss_all;
        for (int i = tid; i < n; i += kThreads) {
            DecExpert& d = plan[R.uidx[i]];
            const int t = i / k, nn = R.rank[i] - d.row0;
            d.tok[nn] = t;
            d.gate[nn] = R.g[i];
            d.hrow[t] = R.rank[i];
            atomicAdd(&d.cnt, 1);
        }
    }
    __syncthreads();
    if (!R.ok) return;  // a logits wait gave up (the device error is set)
    // CTA 0 rewrites LRU table entries below: every CTA's read of its table row
    // happened before its release of the logits this CTA has now read
    if (b == 0) asm volatile("fence.acq_rel.gpu;" ::: "memory");
    const int nu = R.nu, na = nu + ns;
    const int n_miss = R.n_miss;
    const bool capacity_err = R.status != 0;
    if (tid == 0) mark(3);

    // ---------------------------------------------------------------- P2b: CTA 0 updates the cache
    CallInfo* info = a.info;
    auto write_record = [&](int m, unsigned long long copy_ns) {
        // the call record the host reads (statistics, event log); written last: done
        for (int p = tid; p < nu; p += kThreads) {
            info->ev_layer[p] = a.layer;
            info->ev_expert[p] = R.members[p];
            info->ev_hit[p] = R.hit[p];
        }
        __syncthreads();
        if (tid == 0) {
            info->n_uniq = nu;
            info->n_hit = capacity_err ? 0 : nu - m;
            info->n_miss = capacity_err ? 0 : m;
            info->n_pf = info->n_pf_hit = info->n_pf_miss = 0;
            info->n_events = capacity_err ? 0 : nu;
            info->dev_err = *reinterpret_cast<volatile int32_t*>(a.dev_err);
            info->status = capacity_err ? -4 : 0;
            info->device_copied = a.device_misses;
            info->copy_ns = copy_ns;
            __threadfence_system();
            info->done = a.seq;
        }
    };
    if (b == 0 && tid == 0) {
        // barriers this call will not hold still count their participants
        const bool holds_copy_barrier = !capacity_err && n_miss > 0 && a.device_misses;
        if (!holds_copy_barrier) bar_arrive(a.bar_cnt + 1, static_cast<unsigned long long>(G));
        if (capacity_err) bar_arrive(a.bar_cnt + 2, static_cast<unsigned long long>(G - 1));
    }
    if (b == 0) {
        // routing results for moe_debug_routing
        for (int i = tid; i < n; i += kThreads) {
            a.topk[i] = R.tk[i];
            a.gates[i] = R.g[i];
            a.perm[R.rank[i]] = i;
            a.inv_perm[i] = R.rank[i];
        }
        for (int e = tid; e < E; e += kThreads) a.counts[e] = 0;
        __syncthreads();
        for (int u = tid; u < nu; u += kThreads) {
            a.counts[R.members[u]] = plan[u].cnt;
            a.act_expert[u] = R.members[u];
        }
        if (tid == 0) *a.n_uniq = nu;
        if (!capacity_err) {
            // the LRU batch (scratch over the ring: no stage is in use yet)
            LruShared& sm = *reinterpret_cast<LruShared*>(ring);
            int32_t* trow = reinterpret_cast<int32_t*>(dsm + geo.lru_trow_off);
            unsigned long long* keys = reinterpret_cast<unsigned long long*>(dsm + geo.lru_keys_off);
            const bool cached = geo.lru_cache_off > 0;
            unsigned long long* st_s = cached ? reinterpret_cast<unsigned long long*>(dsm + geo.lru_cache_off) : nullptr;
            int32_t* own_s = cached ? reinterpret_cast<int32_t*>(st_s + a.S) : nullptr;
            for (int e = tid; e < E; e += kThreads) trow[e] = __ldcg(a.table + static_cast<size_t>(a.layer) * E + e);
            if (cached)
                for (int s = tid; s < a.S; s += kThreads) {
                    st_s[s] = __ldcg(a.stamp + s);
                    own_s[s] = __ldcg(a.owner + s);
                }
            if (tid == 0) sm.clock = __ldcg(a.clock);
            __syncthreads();
            LruView lv;
            lv.bind(a);
            lv.trow0 = trow;
            lv.trow1 = nullptr;
            lv.st_s = st_s;
            lv.own_s = own_s;
            const int m = lru_batch(lv, sm, keys, a.layer, R.members, nu, nullptr, 0, 0);
            // m == n_miss: the members that missed are those whose table entry was -1
            for (int r = tid; r < m; r += kThreads) {
                const int p = sm.miss_p[r];
                a.pub->slot[r] = sm.member_slot[p];
                info->miss_layer[r] = a.layer;
                info->miss_expert[r] = R.members[p];
                info->miss_slot[r] = sm.member_slot[p];
            }
            for (int p = tid; p < nu; p += kThreads) {
                info->ev_slot[p] = sm.member_slot[p];
                info->ev_evicted[p] = sm.member_old[p];
                info->ev_prefetch[p] = 0;
            }
            __syncthreads();
            if (tid == 0 && m > 0) {
                __threadfence();
                st_release_gpu64(&a.pub->seq, a.seq);
            }
            if (!(m > 0 && a.device_misses)) write_record(m, 0ull);
        } else {
            write_record(0, 0ull);
        }
        __syncthreads();
        if (tid == 0) mark(4);
    }
    if (capacity_err) return;

    // ---------------------------------------------------------------- P2c: misses
    if (n_miss > 0) {
        if (tid == 0) {
            bool ok = true;
            if (!a.device_misses) ok = wait_ready(a);  // the host's copies have landed
            if (ok) {
                const uint64_t t0 = gtimer();
                while (ld_acquire_gpu64(&a.pub->seq) < a.seq) {
                    if (gtimer() - t0 > a.wait_ns) {
                        atomicExch(a.dev_err, MOE_DEVERR_TIMEOUT_READY);
                        ok = false;
                        break;
                    }
                }
            }
            R.ok = ok ? 1 : 0;
            R.t_copy0 = gtimer();
        }
        __syncthreads();
        if (!R.ok) return;
        for (int r = tid; r < n_miss; r += kThreads) {
            const int p = R.missr[r];
            const int s = __ldcg(&a.pub->slot[r]);
            R.mslot[p] = s;
            plan[p].ptr = a.pool + static_cast<size_t>(s) * B;
        }
        __syncthreads();
        if (a.device_misses) {
            // copy the missed blobs: CTA b takes a contiguous share of the 16-byte vectors
            const size_t per_blob = B / 16;
            const size_t total = per_blob * n_miss;
            const size_t share = (total + G - 1) / G;
            const size_t v0 = share * b, v1 = min(total, v0 + share);
            const uint8_t* bank = a.banks[a.layer];
            constexpr int kU = 4;
            for (size_t v = v0 + tid; v < v1; v += static_cast<size_t>(kThreads) * kU) {
                uint4 x[kU];
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const size_t vv = v + static_cast<size_t>(u) * kThreads;
                    if (vv < v1) {
                        const size_t r = vv / per_blob, off = vv % per_blob;
                        const int e = R.members[R.missr[r]];
                        x[u] = __ldcs(reinterpret_cast<const uint4*>(bank + static_cast<size_t>(e) * B) + off);
                    }
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const size_t vv = v + static_cast<size_t>(u) * kThreads;
                    if (vv < v1) {
                        const size_t r = vv / per_blob, off = vv % per_blob;
                        reinterpret_cast<uint4*>(const_cast<uint8_t*>(a.pool) + static_cast<size_t>(R.mslot[R.missr[r]]) * B)[off] = x[u];
                    }
                }
            }
            // the bulk copies (async proxy) of every CTA read these bytes next
            asm volatile("fence.proxy.async.global;" ::: "memory");
            __syncthreads();
            if (tid == 0) {
                bar_arrive(a.bar_cnt + 1, 1);
                R.ok = bar_wait(a, a.bar_cnt + 1, tgt0, MOE_DEVERR_TIMEOUT_PRODUCER) ? 1 : 0;
            }
            __syncthreads();
            if (!R.ok) return;
            if (b == 0) {
                const unsigned long long dt = gtimer() - R.t_copy0;
                write_record(n_miss, dt);
            }
        }
        __syncthreads();
    }

    if (tid == 0) mark(5);
    // ---------------------------------------------------------------- P3: experts
    static_assert(sizeof(StageSeq<FMT>) <= sizeof(DecRoute::seqbuf), "stage sequence buffer");
    StageSeq<FMT> seq;
    if (TT == 1) seq = *reinterpret_cast<const StageSeq<FMT>*>(R.seqbuf);
    else seq.init(a, plan, na, b, G);
    const int nf1 = seq.count1(), nf2 = seq.count2();
    const int xp = H * 2 + 16, hp = I * 2 + 16;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        int stage = 0;
        uint32_t phase = 0;
        const uint64_t stream = l2_evict_first();
        bool ok = true;
        const int nf = nf1 + nf2;
        if (lane == 0) mark(20);
        int f = 0;
        for (; f < nf && ok; ++f) {
            const uint8_t* src;
            uint32_t bytes, off, total;
            const int np = seq.piece(lane, src, bytes, off, total);
            int got = 1;
            if (lane == 0) {
                // a slot's first use needs no wait: the ring starts empty
                got = (f < nst || mbar_wait(&empty[stage], phase ^ 1u, abort_flag, a.wait_ns)) && !*abort_flag;
                if (got) mbar_expect_tx(&full[stage], total);
            }
            got = __shfl_sync(0xffffffffu, got, 0);
            if (!got) {
                ok = false;
                break;
            }
            if (lane < np) bulk_g2s_hint(ring + stage * C::kStageBytes + off, src, bytes, &full[stage], stream);
            if (lane == 0 && (f == 0 || f == nf1 - 1)) mark(f == 0 ? 16 : 17);
            seq.advance();
            if (++stage == nst) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok && lane == 0 && !*abort_flag) {
            atomicExch(a.dev_err, MOE_DEVERR_TIMEOUT_PRODUCER);
            *abort_flag = 1;
        }
        if (a.trace && lane == 0) {
            // trace only: when the producer had issued everything, when phase 1's last stage landed
            mark(18);
            if (nf1 > 0 && nf1 <= f && f - nf1 < nst) {  // its slot has not been reused since
                const uint64_t t0 = gtimer();
                while (!mbar_test(&full[(nf1 - 1) % nst], static_cast<uint32_t>(((nf1 - 1) / nst) & 1)) &&
                       gtimer() - t0 < a.wait_ns) {
                }
                mark(19);
            }
        }
        // every copy this warp issued (stages 0 .. f-1) must land before the
        // CTA may exit: the last use of each slot, with its phase parity
        if (lane == 0)
            for (int g2 = f > nst ? f - nst : 0; g2 < f; ++g2) {
                const uint64_t t0 = gtimer();
                while (!mbar_test(&full[g2 % nst], static_cast<uint32_t>((g2 / nst) & 1)) && gtimer() - t0 < a.wait_ns) {
                }
            }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- consumers
        const int w = warp - 1, ct = tid - 32;
        const int g = lane >> 2, q = lane & 3;
        // NVFP4 / FP8 per-tensor scales live in the blobs
        for (int u = ct; u < na; u += 32 * kConsumers) {
            if (plan[u].pad) continue;  // loaded with the plan
            if constexpr (FMT == FMT_NVFP4 || FMT == FMT_FP8) {
                const float4 v = __ldcg(reinterpret_cast<const float4*>(plan[u].ptr + a.lay.gsc));  // may be this call's copy
                plan[u].gs[0] = v.x; plan[u].gs[1] = v.y; plan[u].gs[2] = v.z;
            } else {
                plan[u].gs[0] = plan[u].gs[1] = plan[u].gs[2] = 1.0f;
            }
        }
        consumer_sync();
        const uint16_t* hb = reinterpret_cast<const uint16_t*>(a.hbuf);
        int stage = 0;
        uint32_t phase = 0;
        bool dead = false;
        auto wait_full = [&]() -> const unsigned char* {
            if (!dead && !mbar_wait(&full[stage], phase, abort_flag, a.wait_ns)) {
                dead = true;
                atomicExch(a.dev_err, MOE_DEVERR_TIMEOUT_MMA);
                *abort_flag = 1;
            }
            return ring + stage * C::kStageBytes;
        };
        auto release = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == nst) {
                stage = 0;
                phase ^= 1u;
            }
        };
        // this warp's partial of finished tile number ti (counted over both
        // phases) into reduction slot ti mod kRedSlots, once that slot's previous
        // tile has been summed (bounded wait); true for the warp that arrives
        // last, which then holds the tile's sum in v, in warp order. The caller
        // has already released the tile's stages, so the weight stream goes on.
        int ti = 0;
        auto tile_reduce = [&](const float (&acc)[4], float (&v)[4]) -> bool {
            const int slot = ti % kRedSlots, use = ti / kRedSlots;
            ++ti;
            float* sl = red + slot * (kConsumers * 32 * 4);
            volatile int32_t* gen = &R.red_gen[slot];
            if (*gen != use) {
                const uint64_t t0 = gtimer();
                while (*gen != use) {
                    if (gtimer() - t0 > a.wait_ns) {
                        dead = true;
                        atomicExch(a.dev_err, MOE_DEVERR_TIMEOUT_EPILOGUE);
                        *abort_flag = 1;
                        break;
                    }
                }
            }
            *reinterpret_cast<float4*>(sl + (w * 32 + lane) * 4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
            __threadfence_block();
            __syncwarp();
            int last = 0;
            if (lane == 0) last = atomicAdd(&R.red_cnt[slot], 1) == kConsumers - 1;
            last = __shfl_sync(0xffffffffu, last, 0);
            if (!last) return false;
            __threadfence_block();
            v[0] = v[1] = v[2] = v[3] = 0.f;
#pragma unroll
            for (int y = 0; y < kConsumers; ++y) {
                const float4 p = *reinterpret_cast<const float4*>(sl + (y * 32 + lane) * 4);
                v[0] += p.x; v[1] += p.y; v[2] += p.z; v[3] += p.w;
            }
            __syncwarp();
            if (lane == 0) {
                R.red_cnt[slot] = 0;
                __threadfence_block();
                *gen = use + 1;  // the slot is free for tile ti + kRedSlots
            }
            return true;
        };
        // ---------------- phase 1: gate/up + SwiGLU
        {
            float acc[2 * kSlotsPerWarp][4] = {};  // independent chains: (group slot, even/odd step)
            for (int f = 0; f < nf1; ++f) {
                const int u = seq.u, ut = seq.ut, c0 = seq.c0_1(), nc = seq.nc_1();
                const bool tile_end = seq.end1();
                seq.advance();
                const DecExpert& m = plan[u];
                const int tok = m.tok[g];
                const unsigned char* st = wait_full();
                if (ct == 0 && (f == 0 || f == nf1 - 1)) mark(f == 0 ? 13 : 14);
#pragma unroll
                for (int h = 0; h < kSlotsPerWarp; ++h) {
                    const int gs = w + kConsumers * h;  // group slot of this stage: chunk gs / 8, group gs % 8
                    const int half = gs / kChunkGroups, ww = gs % kChunkGroups;
                    const int c = c0 + half;
                    if (half < nc) {
                        const int ng = fp4_chunk_groups(seq.G1k, c);
                        if (ww < ng && !dead) {
                            const int j = c * kChunkGroups + ww;
                            uint32_t bq[16];
                            if (geo.act_bytes) load_b_smem(act, xp, tok, j, q, bq);
                            else load_b_xglobal<ACT>(a.hidden, H, tok, j, q, tok >= 0 ? R.xsc[tok] : 1.f, bq);
                            mma_group<FMT>(st + half * C::kChunkBytes, ng, ww, g, q, bq, acc[2 * h], acc[2 * h + 1]);
                        }
                    }
                }
                release();
                if (tile_end) {
                    float v[4], part[4];
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        part[x] = acc[0][x];
#pragma unroll
                        for (int y = 1; y < 2 * kSlotsPerWarp; ++y) part[x] += acc[y][x];
                    }
                    if (tile_reduce(part, v)) {
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const int nn = 2 * q + h2;
                            float hv = 0.f;
                            if (nn < m.cnt) {
                                const int t = m.tok[nn];
                                const int r = m.row0 + nn;
                                const float gate = v[h2] * m.gs[0] * R.xun[t], up = v[2 + h2] * m.gs[1] * R.xun[t];
                                const float av = a.mode == 1 ? gate : silu(gate);
                                hv = av * up * m.gate[nn];
                                const __nv_bfloat16 hb16 = __float2bfloat16_rn(hv);
                                reinterpret_cast<__nv_bfloat16*>(a.hbuf)[static_cast<size_t>(r) * I + dpos(ut * 8 + g)] = hb16;
                                // this CTA's max |h| of token t, as the bits of an fp32
                                const uint32_t hbits = (static_cast<uint32_t>(__bfloat16_as_ushort(hb16)) << 16) & 0x7FFFFFFFu;
                                atomicMax(&R.hmax[t], hbits);
                            }
                        }
                    }
#pragma unroll
                    for (int y = 0; y < 2 * kSlotsPerWarp; ++y) acc[y][0] = acc[y][1] = acc[y][2] = acc[y][3] = 0.f;
                }
            }
        }
        // ---------------- barrier: every h row of the call is written (workers only)
        consumer_sync();
        if (ct == 0) mark(6);
        if (b != 0) {
            if (ct == 0) {
                // this CTA's per-token max |h| into the call's maxima, before its arrival publishes them
                for (int t = 0; t < T; ++t)
                    if (R.hmax[t]) atomicMax(a.hmax + (a.dcall & 1) * kDecodeMaxT + t, R.hmax[t]);
                bar_arrive(a.bar_cnt + 2, 1);
                R.ok = (bar_wait(a, a.bar_cnt + 2, tgt2, MOE_DEVERR_TIMEOUT_EPILOGUE) && !*abort_flag) ? 1 : 0;
            }
            consumer_sync();
            if (!R.ok) *abort_flag = 1;
        }
        // ---------------- phase 2: down projection + combine
        if (nf2 > 0) {
            const int hrows = n + ns * T;
            // Every h row of the call (bf16, read once) into shared memory as f16,
            // scaled by a power of two per token from the call's maxima (published
            // by every worker before barrier 2), when the rows fit; otherwise the
            // MMA operands are read from global memory with the same scales.
            {
                const int per_row = I / 8;
                const float inv_pr = 1.0f / static_cast<float>(per_row);
                if (ct < T) {
                    const unsigned int mb = __ldcg(a.hmax + (a.dcall & 1) * kDecodeMaxT + ct);
                    R.hmax[ct] = mb;
                    pow2_scale(mb, R.hsc[ct], R.hun[ct]);
                }
                consumer_sync();
                if (geo.act_bytes) {
                    const int nvec = hrows * per_row;  // row r holds vectors [r * per_row, (r + 1) * per_row): h is contiguous
                    const uint4* hv = reinterpret_cast<const uint4*>(hb);
                    for (int i0 = ct; i0 < nvec; i0 += 4 * 32 * kConsumers) {
                        uint4 x[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {  // four loads in flight
                            const int i = i0 + j * 32 * kConsumers;
                            x[j] = i < nvec ? __ldcg(hv + i) : make_uint4(0u, 0u, 0u, 0u);
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int i = i0 + j * 32 * kConsumers;
                            if (i < nvec) {
                                int r = __float2int_rz(static_cast<float>(i) * inv_pr);
                                r += (r + 1) * per_row <= i;
                                r -= r * per_row > i;
                                const float sc = R.hsc[R.rowtok[r]];
                                uint4 o;
                                o.x = f16x2_scaled(__uint_as_float(x[j].x << 16), __uint_as_float(x[j].x & 0xFFFF0000u), sc);
                                o.y = f16x2_scaled(__uint_as_float(x[j].y << 16), __uint_as_float(x[j].y & 0xFFFF0000u), sc);
                                o.z = f16x2_scaled(__uint_as_float(x[j].z << 16), __uint_as_float(x[j].z & 0xFFFF0000u), sc);
                                o.w = f16x2_scaled(__uint_as_float(x[j].w << 16), __uint_as_float(x[j].w & 0xFFFF0000u), sc);
                                *reinterpret_cast<uint4*>(act + r * hp + 16 * (i - r * per_row)) = o;
                            }
                        }
                    }
                    consumer_sync();
                }
                if (ct == 0) mark(7);
            }
            // with several experts per stage: this warp's expert and K group in each of its slots
            int p2[kSlotsPerWarp], w2[kSlotsPerWarp];
#pragma unroll
            for (int h = 0; h < kSlotsPerWarp; ++h) {
                const int gs = w + kConsumers * h;  // group slot of this stage
                p2[h] = seq.epp == 1 ? 0 : gs / seq.G2k;
                w2[h] = gs - p2[h] * seq.G2k;
            }
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int f = 0; f < nf2; ++f) {
                int rt, u0, nu_, c0, nc;
                seq.where2(rt, u0, nu_, c0, nc);
                const bool tile_end = seq.end2();
                seq.advance();
                const unsigned char* st = wait_full();
                if (ct == 0 && f == nf2 - 1) mark(15);
#pragma unroll
                for (int h = 0; h < kSlotsPerWarp; ++h) {
                    int u, c, ww, ng, off;
                    if (seq.epp == 1) {
                        const int gs = w + kConsumers * h, half = gs / kChunkGroups;  // chunk c0 + half, group gs % 8
                        u = u0;
                        c = c0 + half;
                        ww = gs % kChunkGroups;
                        ng = c < c0 + nc ? fp4_chunk_groups(seq.G2k, c) : 0;
                        off = half * C::kChunkBytes;
                    } else {
                        const int p = p2[h];
                        u = u0 + p;
                        c = 0;
                        ww = w2[h];
                        ng = p < nu_ ? seq.G2k : 0;
                        off = p * kTileRows * seq.G2k * C::kRowBytes;
                    }
                    if (ww < ng && !dead) {
                        const int hr = plan[u].hrow[g];
                        const int j = c * kChunkGroups + ww;
                        uint32_t bq[16];
                        if (geo.act_bytes) load_b_smem(act, hp, hr, j, q, bq);
                        else load_b_hglobal(hb, I, hr, j, q, R.hsc[g < T ? g : 0], bq);
                        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
                        mma_group<FMT>(st + off, ng, ww, g, q, bq, d0, d1);
                        const float gsd = plan[u].gs[2];
#pragma unroll
                        for (int x = 0; x < 4; ++x) acc[x] = __fmaf_rn(gsd, d0[x] + d1[x], acc[x]);
                    }
                }
                release();
                if (tile_end) {
                    float v[4];
                    if (tile_reduce(acc, v)) {
                        const int r0 = rt * kTileRows;
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const int t = 2 * q + h2;
                            if (t < T) {
#pragma unroll
                                for (int rr = 0; rr < 2; ++rr) {
                                    const size_t o = static_cast<size_t>(t) * H + r0 + g + 8 * rr;
                                    const float x = v[2 * rr + h2] * R.hun[t];
                                    if constexpr (ACT == ACT_BF16)
                                        reinterpret_cast<__nv_bfloat16*>(a.out)[o] = __float2bfloat16_rn(x);
                                    else
                                        reinterpret_cast<float*>(a.out)[o] = x;
                                }
                            }
                        }
                    }
                    acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
                }
            }
        }
        consumer_sync();
        if (ct == 0) mark(8);
    }
    __syncthreads();
    if (tid == 0) mark(9);
    if (tcall && tid == 0) atomicMax(tcall + 2, static_cast<unsigned long long>(gtimer()));
}

template <int FMT>
size_t lru_need(const CallArgs& a, int* trow_off, int* keys_off, int* cache_off, int base) {
    size_t o = base + (sizeof(LruShared) + 127) / 128 * 128;
    *trow_off = static_cast<int>(o);
    o += (static_cast<size_t>(a.E) * 4 + 127) / 128 * 128;
    *keys_off = static_cast<int>(o);
    size_t P = 1;
    while (P < static_cast<size_t>(a.S)) P <<= 1;
    o += P * 8;
    if (a.S <= kLruCached) {
        *cache_off = static_cast<int>(o);
        o += static_cast<size_t>(a.S) * 12;
    } else {
        *cache_off = 0;
    }
    return o;
}

template <int FMT>
bool geometry(const CallArgs& a, int grid, DecGeom& g) {
    const int T = a.T, H = a.H, I = a.I, k = a.k, ns = a.n_shared;
    const size_t esz = a.act == ACT_BF16 ? 2 : 4;
    g.max_active = std::min(a.E, T * k) + ns;
    size_t o = (sizeof(DecRoute) + 127) / 128 * 128;
    g.plan_off = static_cast<int>(o);
    o += static_cast<size_t>(g.max_active) * sizeof(DecExpert);
    o = (o + 127) / 128 * 128;
    g.ring_off = static_cast<int>(o);
    const size_t fixed = o;
    const size_t stage = Fp4Cfg<FMT>::kStageBytes;
    const size_t red = static_cast<size_t>(kRedSlots) * kRedSlotBytes;
    const size_t act_need = std::max(static_cast<size_t>(T) * (H * 2 + 16),
                                     static_cast<size_t>(T) * (k + ns) * (I * 2 + 16));
    // P1 stages the token rows and this CTA's router rows at ring_off
    const size_t rows_per_cta = (static_cast<size_t>(a.E) + grid - 1) / grid;
    const size_t p1_stage = static_cast<size_t>(T) * H * esz + rows_per_cta * H * esz;
    int to, ko, co;
    const size_t lru_end = lru_need<FMT>(a, &to, &ko, &co, static_cast<int>(fixed));
    if (lru_end > static_cast<size_t>(kSmemLimit)) return false;
    for (int with_act = 1; with_act >= 0; --with_act) {
        const size_t actb = with_act ? (act_need + 127) / 128 * 128 : 0;
        if (fixed + red + actb + 2 * stage > static_cast<size_t>(kSmemLimit)) continue;
        int nst = static_cast<int>((kSmemLimit - fixed - red - actb) / stage);
        nst = std::min(nst, kMaxStages);
        g.nst = nst;
        g.act_bytes = static_cast<int>(actb);
        g.red_off = static_cast<int>(fixed + static_cast<size_t>(nst) * stage);
        g.act_off = static_cast<int>(g.red_off + red);
        const size_t ring_end = g.act_off + actb;
        g.total = static_cast<int>(std::max(ring_end, lru_end));
        g.stage_x = fixed + p1_stage <= static_cast<size_t>(g.total) && p1_stage < (1u << 20) ? 1 : 0;
        g.lru_trow_off = to;
        g.lru_keys_off = ko;
        g.lru_cache_off = co;
        return g.total <= kSmemLimit;
    }
    return false;
}

template <int FMT, int ACT>
cudaError_t launch_one(const CallArgs& a, int grid, cudaStream_t s, bool pdl) {
    DecGeom geo{};
    if (grid < 2) return cudaErrorInvalidValue;  // CTA 0 runs the cache update beside the others' work
    if (!geometry<FMT>(a, grid, geo)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(geo.total);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return a.T == 1 ? cudaLaunchKernelEx(&cfg, k_decode<FMT, ACT, 1>, a, geo)
                    : cudaLaunchKernelEx(&cfg, k_decode<FMT, ACT, 0>, a, geo);
}

}  // namespace

template <int FMT, int ACT>
cudaError_t set_attr() {
    cudaError_t e;
    const int lim = kSmemLimit;
    if ((e = cudaFuncSetAttribute(k_decode<FMT, ACT, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim))) return e;
    return cudaFuncSetAttribute(k_decode<FMT, ACT, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
}

cudaError_t decode_set_attributes() {
    cudaError_t e;
    if ((e = set_attr<FMT_NVFP4, ACT_BF16>())) return e;
    if ((e = set_attr<FMT_NVFP4, ACT_FP32>())) return e;
    if ((e = set_attr<FMT_MXFP4, ACT_BF16>())) return e;
    if ((e = set_attr<FMT_MXFP4, ACT_FP32>())) return e;
    if ((e = set_attr<FMT_FP8, ACT_BF16>())) return e;
    return set_attr<FMT_FP8, ACT_FP32>();
}

cudaError_t launch_decode(const CallArgs& a, int num_sms, cudaStream_t s, bool pdl) {
    const bool bf = a.act == ACT_BF16;
    if (a.fmt == FMT_NVFP4)
        return bf ? launch_one<FMT_NVFP4, ACT_BF16>(a, num_sms, s, pdl) : launch_one<FMT_NVFP4, ACT_FP32>(a, num_sms, s, pdl);
    if (a.fmt == FMT_FP8)
        return bf ? launch_one<FMT_FP8, ACT_BF16>(a, num_sms, s, pdl) : launch_one<FMT_FP8, ACT_FP32>(a, num_sms, s, pdl);
    return bf ? launch_one<FMT_MXFP4, ACT_BF16>(a, num_sms, s, pdl) : launch_one<FMT_MXFP4, ACT_FP32>(a, num_sms, s, pdl);
}

}  // namespace moe
