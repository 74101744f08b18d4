// Decode expert FFNs (T <= 8 tokens) over FP4 expert weights (NVFP4, MXFP4):
// gate/up projection + SwiGLU, then down projection + gate-weighted combine,
// in one persistent cooperative kernel.
//
// Hits of the expert cache "run on the GPU" (freetoken.wiki architecture page,
// decode paragraph). At decode the layer is bound by streaming the active
// experts' packed weights from HBM once, so the kernel is built around that
// stream rather than around the (tiny) arithmetic:
//
//  * warp 0 is a producer: its 32 lanes issue cp.async.bulk copies in parallel
//    (one 16-row weight tile = 16 code runs + 16 scale runs per pipeline stage)
//    into a ring of shared-memory stages, completing on an mbarrier;
//  * warps 1-8 consume the stages with mma.sync m16n8k16 in swap-AB form
//    (16 weight rows x 8 token columns); FP4 codes and E4M3/E8M0 scales are
//    widened exactly in registers; each warp owns one 128-element K group of a
//    stage, and a fixed-order shared-memory reduction finishes every tile;
//  * phase 1 computes h = gate * silu(W_gate x) * (W_up x) for every active
//    expert; a grid barrier (consumers only, bounded wait) separates it from
//    phase 2, out[t] = sum over experts of W_down h. The producer does not stop
//    at the barrier: phase-2 weights stream into the ring while phase 1
//    finishes, so HBM stays busy across the dependency.
//
// Staged rows are 576 bytes apart (512 code bytes + 64) so that the 8 rows a
// quarter-warp reads fall into disjoint shared-memory banks.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "mma_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kConsumers = 8;                       // consumer warps
constexpr int kDecThreads = 32 * (kConsumers + 1);  // + the producer warp
constexpr int kRows = 16;                           // weight rows per stage (one m16 tile)
constexpr int kGroupsPerStage = 8;                  // 128-element K groups per stage (one per consumer)
constexpr int kCodeRun = kGroupsPerStage * 64;      // FP4 code bytes of one row per stage
constexpr int kCodePitch = kCodeRun + 64;           // staged row pitch (bank shift of 16 words)
constexpr int kStages = 10;
constexpr unsigned long long kDecWaitNs = 2000000000ull;  // 2 s per wait

template <int FMT>
struct DecCfg {
    static constexpr int kBlk = FMT == FMT_NVFP4 ? 16 : 32;
    static constexpr int kScaleRun = kGroupsPerStage * 128 / kBlk;  // scale bytes of one row per stage
    static constexpr int kScalePitch = FMT == FMT_NVFP4 ? 80 : 48;   // conflict-free 8-row reads
    static constexpr int kStageBytes = kRows * kCodePitch + kRows * kScalePitch;
    static constexpr int kStageStride = (kStageBytes + 127) / 128 * 128;
};

// per active expert, staged once per CTA by the consumers
struct ExpertMeta {
    int32_t row0, cnt;
    int32_t tok[kDecodeMaxT];   // token of the expert's row n (n < cnt), else -1
    int32_t hrow[kDecodeMaxT];  // h row of token t, else -1
    float gate[kDecodeMaxT];    // routing gate of the expert's row n
    float gs[3];                // per-tensor scales (gate, up, down); 1 for MXFP4
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

__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// bounded wait for the phase of parity `parity`; false on abort or timeout
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag) {
    if (mbar_test(b, parity)) return true;
    const uint64_t t0 = gtimer();
    for (;;) {
        if (mbar_test(b, parity)) return true;
        if (*abort_flag) return false;
        if (gtimer() - t0 > kDecWaitNs) return false;
    }
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(su32(dst)),
        "l"(src), "r"(bytes), "r"(su32(bar))
        : "memory");
}

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumers) : "memory"); }

__device__ __forceinline__ uint4 lds128(const unsigned char* p) { return *reinterpret_cast<const uint4*>(p); }

// 64-byte B run of one token column for one group (16 words); zeros for a null pointer
template <bool CG>
__device__ __forceinline__ void load_bcol(const uint16_t* p, uint32_t (&b)[16]) {
    if (p) {
        const uint4* v4 = reinterpret_cast<const uint4*>(p);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint4 x = CG ? __ldcg(v4 + v) : __ldg(v4 + v);
            b[4 * v] = x.x; b[4 * v + 1] = x.y; b[4 * v + 2] = x.z; b[4 * v + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) b[i] = 0u;
    }
}

// scales of one staged row for consumer group w, times mul
template <int FMT>
__device__ __forceinline__ void stage_scales(const unsigned char* srow, int w, float mul, float (&s)[8]) {
    if constexpr (FMT == FMT_NVFP4) {
        const uint2 v = *reinterpret_cast<const uint2*>(srow + 8 * w);
        e4m3x8_to_f32(v, s);
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i] *= mul;
    } else {
        const uint32_t v = *reinterpret_cast<const uint32_t*>(srow + 4 * w);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const float f = e8m0_to_f32((v >> (8 * b)) & 0xFFu) * mul;
            s[2 * b] = f;
            s[2 * b + 1] = f;
        }
    }
}

// one 128-element group of a staged 16-row tile against one 8-column B run:
// acc (rows g / g+8, columns 2q / 2q+1) += sum over the 8 MMA steps of scale * MMA
template <int FMT>
__device__ __forceinline__ void stage_group(const unsigned char* st, int w, int g, int q, float mul,
                                            const uint32_t (&b)[16], float (&acc)[4]) {
    using C = DecCfg<FMT>;
    const uint4 ra = lds128(st + g * kCodePitch + w * 64 + 16 * q);
    const uint4 rb = lds128(st + (g + 8) * kCodePitch + w * 64 + 16 * q);
    float sa[8], sb[8];
    stage_scales<FMT>(st + kRows * kCodePitch + g * C::kScalePitch, w, mul, sa);
    stage_scales<FMT>(st + kRows * kCodePitch + (g + 8) * C::kScalePitch, w, mul, sb);
    const uint32_t wa[4] = {ra.x, ra.y, ra.z, ra.w}, wb[4] = {rb.x, rb.y, rb.z, rb.w};
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        uint32_t oa[4], ob[4];
        fp4x8_to_f16x2(wa[x], oa);
        fp4x8_to_f16x2(wb[x], ob);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int s = 2 * x + h;
            const uint32_t A[4] = {oa[2 * h], ob[2 * h], oa[2 * h + 1], ob[2 * h + 1]};
            float d[4];
            const float z[4] = {0.f, 0.f, 0.f, 0.f};
            mma_f16(d, A, b[2 * s], b[2 * s + 1], z);
            acc[0] = __fmaf_rn(sa[s], d[0], acc[0]);
            acc[1] = __fmaf_rn(sa[s], d[1], acc[1]);
            acc[2] = __fmaf_rn(sb[s], d[2], acc[2]);
            acc[3] = __fmaf_rn(sb[s], d[3], acc[3]);
        }
    }
}

template <int FMT, int ACT>
__global__ void __launch_bounds__(kDecThreads, 1) k_dec_fp4(CallArgs a) {
    using C = DecCfg<FMT>;
    extern __shared__ unsigned char dec_raw[];
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
    __shared__ float red[2][kConsumers][32][4];
    __shared__ int s_abort, s_gb_ok;

    unsigned char* ring = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dec_raw) + 127) & ~uintptr_t(127));
    ExpertMeta* meta = reinterpret_cast<ExpertMeta*>(ring + kStages * C::kStageStride);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, I = a.I, T = a.T;
    const int na = *a.n_active;
    const int UT = I / 8;                  // gate/up unit tiles (8 units = 16 rows) per expert
    const int G1 = H / kGroupK, G2 = I / kGroupK;
    const int nch1 = (G1 + kGroupsPerStage - 1) / kGroupsPerStage;
    const int nch2 = (G2 + kGroupsPerStage - 1) / kGroupsPerStage;
    const int n1 = na * UT;                // phase-1 tasks
    const int n2 = H / kRows;              // phase-2 row tiles
    const int G = gridDim.x, b = blockIdx.x;
    const int my1 = b < n1 ? (n1 - 1 - b) / G + 1 : 0;
    const int rt_first = G - 1 - b;        // phase-2 tiles go to the CTAs with the least phase-1 work first
    const int my2 = rt_first < n2 ? (n2 - 1 - rt_first) / G + 1 : 0;
    volatile int* abort_flag = &s_abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumers);
        }
        s_abort = 0;
        s_gb_ok = 1;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        int stage = 0;
        uint32_t phase = 0;
        int issued[kStages];
#pragma unroll
        for (int s = 0; s < kStages; ++s) issued[s] = -1;
        bool ok = true;
        // phase 1: gate rows rg..rg+7 and up rows rg+64..rg+71 of unit tile ut
        const size_t rb1 = static_cast<size_t>(H) / 2;
        for (int i = 0; i < my1 && ok; ++i) {
            const int task = b + i * G;
            const int u = task / UT, ut = task % UT;
            const unsigned char* blob = a.act_ptr[u];
            const int i0 = ut * 8;
            const int rg = (i0 / 64) * 128 + (i0 % 64);
            const int li = lane & 15;
            const int drow = rg + (li < 8 ? li : 64 + li - 8);
            for (int c = 0; c < nch1 && ok; ++c) {
                const int ng = min(kGroupsPerStage, G1 - c * kGroupsPerStage);
                // per-lane row addresses: codes and scales of staged row li
                const unsigned char* crow = blob + a.lay.gu + static_cast<size_t>(drow) * rb1;
                const unsigned char* srow = blob + a.lay.gus + static_cast<size_t>(drow) * a.lay.gus_pitch;
                bool got = true;
                if (lane == 0) got = mbar_wait(&empty[stage], phase ^ 1u, abort_flag) && !*abort_flag;
                got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
                if (!got) { ok = false; break; }
                unsigned char* st = ring + stage * C::kStageStride;
                const uint32_t cb = static_cast<uint32_t>(ng) * 64;
                const uint32_t sbytes = (static_cast<uint32_t>(ng) * (128 / C::kBlk) + 15u) & ~15u;
                if (lane == 0) mbar_expect_tx(&full[stage], kRows * (cb + sbytes));
                __syncwarp();
                if (lane < 16) bulk_g2s(st + li * kCodePitch, crow + static_cast<size_t>(c) * kCodeRun, cb, &full[stage]);
                else bulk_g2s(st + kRows * kCodePitch + li * C::kScalePitch, srow + static_cast<size_t>(c) * C::kScaleRun,
                              sbytes, &full[stage]);
                issued[stage] = static_cast<int>(phase);
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
            }
        }
        // phase 2: rows r0..r0+15 of the down projection of every active expert
        const size_t rb2 = static_cast<size_t>(I) / 2;
        for (int i = 0; i < my2 && ok; ++i) {
            const int r0 = (rt_first + i * G) * kRows;
            const int li = lane & 15;
            for (int u = 0; u < na && ok; ++u) {
                const unsigned char* blob = a.act_ptr[u];
                const unsigned char* crow = blob + a.lay.d + static_cast<size_t>(r0 + li) * rb2;
                const unsigned char* srow = blob + a.lay.ds + static_cast<size_t>(r0 + li) * a.lay.ds_pitch;
                for (int c = 0; c < nch2 && ok; ++c) {
                    const int ng = min(kGroupsPerStage, G2 - c * kGroupsPerStage);
                    bool got = true;
                    if (lane == 0) got = mbar_wait(&empty[stage], phase ^ 1u, abort_flag) && !*abort_flag;
                    got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
                    if (!got) { ok = false; break; }
                    unsigned char* st = ring + stage * C::kStageStride;
                    const uint32_t cb = static_cast<uint32_t>(ng) * 64;
                    const uint32_t sbytes = (static_cast<uint32_t>(ng) * (128 / C::kBlk) + 15u) & ~15u;
                    if (lane == 0) mbar_expect_tx(&full[stage], kRows * (cb + sbytes));
                    __syncwarp();
                    if (lane < 16) bulk_g2s(st + li * kCodePitch, crow + static_cast<size_t>(c) * kCodeRun, cb, &full[stage]);
                    else bulk_g2s(st + kRows * kCodePitch + li * C::kScalePitch, srow + static_cast<size_t>(c) * C::kScaleRun,
                                  sbytes, &full[stage]);
                    issued[stage] = static_cast<int>(phase);
                    if (++stage == kStages) { stage = 0; phase ^= 1u; }
                }
            }
        }
        if (!ok && lane == 0 && !*abort_flag) {
            atomicExch(a.dev_err, MOE_DEVERR_TIMEOUT_PRODUCER);
            *abort_flag = 1;
        }
        // every copy this warp issued must land before the CTA may exit
        if (lane == 0) {
            for (int s = 0; s < kStages; ++s)
                if (issued[s] >= 0) {
                    const uint64_t t0 = gtimer();
                    while (!mbar_test(&full[s], static_cast<uint32_t>(issued[s])) && gtimer() - t0 < kDecWaitNs) {
                    }
                }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------------- consumers
        const int w = warp - 1, ct = threadIdx.x - 32;
        const int g = lane >> 2, q = lane & 3;
        // per-expert metadata into shared memory
        for (int u = ct; u < na; u += 32 * kConsumers) {
            ExpertMeta& m = meta[u];
            const int row0 = a.act_row0[u], cnt = a.act_cnt[u];
            m.row0 = row0;
            m.cnt = cnt;
#pragma unroll
            for (int n = 0; n < kDecodeMaxT; ++n) {
                m.tok[n] = n < cnt ? a.row_tok[row0 + n] : -1;
                m.gate[n] = n < cnt ? a.row_gate[row0 + n] : 0.0f;
                m.hrow[n] = n < T ? a.tok_row[u * kDecodeMaxT + n] : -1;
            }
            if constexpr (FMT == FMT_NVFP4) {
                const float* gsc = reinterpret_cast<const float*>(a.act_ptr[u] + a.lay.gsc);
                m.gs[0] = gsc[0]; m.gs[1] = gsc[1]; m.gs[2] = gsc[2];
            } else {
                m.gs[0] = m.gs[1] = m.gs[2] = 1.0f;
            }
        }
        consumer_sync();
        const uint16_t* xh = reinterpret_cast<const uint16_t*>(a.xh);
        const uint16_t* hb = reinterpret_cast<const uint16_t*>(a.hbuf);
        int stage = 0;
        uint32_t phase = 0;
        bool dead = false;
        int rbuf = 0;
        auto wait_full = [&]() -> const unsigned char* {
            if (!dead && !mbar_wait(&full[stage], phase, abort_flag)) {
                dead = true;
                atomicExch(a.dev_err, MOE_DEVERR_TIMEOUT_MMA);
                *abort_flag = 1;
            }
            return ring + stage * C::kStageStride;
        };
        auto release = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
        };
        // ---------------- phase 1: gate/up + SwiGLU
        {
            const int nf = my1 * nch1;
            // B run (activations) of flat stage f for this lane: token column g of the task's expert
            auto bsrc = [&](int f) -> const uint16_t* {
                const int i = f / nch1, c = f % nch1;
                const int task = b + i * G, u = task / UT;
                const int j = c * kGroupsPerStage + w;
                const int tok = meta[u].tok[g];
                return (j < G1 && tok >= 0) ? xh + static_cast<size_t>(tok) * H + j * kGroupK + 32 * q : nullptr;
            };
            uint32_t bn[16], bq[16];
            if (nf > 0) load_bcol<false>(bsrc(0), bn);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int f = 0; f < nf; ++f) {
                const int i = f / nch1, c = f % nch1;
                const int task = b + i * G, u = task / UT, ut = task % UT;
#pragma unroll
                for (int x = 0; x < 16; ++x) bq[x] = bn[x];
                if (f + 1 < nf) load_bcol<false>(bsrc(f + 1), bn);
                if (c == 0) acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
                const unsigned char* st = wait_full();
                const int ng = min(kGroupsPerStage, G1 - c * kGroupsPerStage);
                if (!dead && w < ng) stage_group<FMT>(st, w, g, q, 1.0f, bq, acc);
                release();
                if (c == nch1 - 1) {
#pragma unroll
                    for (int x = 0; x < 4; ++x) red[rbuf][w][lane][x] = acc[x];
                    consumer_sync();
                    if (w == 0) {
                        float v[4];
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            float s = 0.f;
#pragma unroll
                            for (int y = 0; y < kConsumers; ++y) s += red[rbuf][y][lane][x];
                            v[x] = s;
                        }
                        const ExpertMeta& m = meta[u];
                        const int unit = ut * 8 + g;
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const int n = 2 * q + h2;
                            if (n < m.cnt) {
                                const int r = m.row0 + n;
                                const float gate = v[h2] * m.gs[0], up = v[2 + h2] * m.gs[1];
                                const float act = a.mode == 1 ? gate : silu(gate);
                                reinterpret_cast<__half*>(a.hbuf)[static_cast<size_t>(r) * I + dpos(unit)] =
                                    __float2half_rn(act * up * m.gate[n]);
                            }
                        }
                    }
                    rbuf ^= 1;
                }
            }
        }
        // ---------------- grid barrier (consumers of every CTA)
        consumer_sync();
        if (ct == 0) {
            int okb = *abort_flag ? 0 : 1;
            if (okb) {
                unsigned int* cnt = a.grid_bar;
                volatile unsigned int* gen = a.grid_bar + 1;
                const unsigned int my_gen = *gen;
                __threadfence();
                const unsigned int prev = atomicAdd(cnt, 1u);
                if (prev == static_cast<unsigned int>(G) - 1u) {
                    *cnt = 0u;
                    __threadfence();
                    atomicAdd(a.grid_bar + 1, 1u);
                } else {
                    const uint64_t t0 = gtimer();
                    while (*gen == my_gen) {
                        if (gtimer() - t0 > kDecWaitNs) {
                            okb = 0;
                            atomicExch(a.dev_err, MOE_DEVERR_TIMEOUT_EPILOGUE);
                            *abort_flag = 1;
                            break;
                        }
                    }
                }
                __threadfence();
            }
            s_gb_ok = okb;
        }
        consumer_sync();
        // ---------------- phase 2: down projection + combine
        if (s_gb_ok) {
            const int per_tile = na * nch2;
            const int nf = my2 * per_tile;
            auto bsrc = [&](int f) -> const uint16_t* {
                const int r = f % per_tile, u = r / nch2, c = r % nch2;
                const int j = c * kGroupsPerStage + w;
                const int hr = meta[u].hrow[g];
                return (j < G2 && hr >= 0) ? hb + static_cast<size_t>(hr) * I + j * kGroupK + 32 * q : nullptr;
            };
            uint32_t bn[16], bq[16];
            if (nf > 0) load_bcol<true>(bsrc(0), bn);
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int f = 0; f < nf; ++f) {
                const int i = f / per_tile, r = f % per_tile, u = r / nch2, c = r % nch2;
#pragma unroll
                for (int x = 0; x < 16; ++x) bq[x] = bn[x];
                if (f + 1 < nf) load_bcol<true>(bsrc(f + 1), bn);
                if (r == 0) acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
                const unsigned char* st = wait_full();
                const int ng = min(kGroupsPerStage, G2 - c * kGroupsPerStage);
                if (!dead && w < ng) stage_group<FMT>(st, w, g, q, meta[u].gs[2], bq, acc);
                release();
                if (r == per_tile - 1) {
#pragma unroll
                    for (int x = 0; x < 4; ++x) red[rbuf][w][lane][x] = acc[x];
                    consumer_sync();
                    if (w == 0) {
                        float v[4];
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            float s = 0.f;
#pragma unroll
                            for (int y = 0; y < kConsumers; ++y) s += red[rbuf][y][lane][x];
                            v[x] = s;
                        }
                        const int r0 = (rt_first + i * G) * kRows;
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const int t = 2 * q + h2;
                            if (t < T) {
#pragma unroll
                                for (int rr = 0; rr < 2; ++rr) {
                                    const size_t o = static_cast<size_t>(t) * H + r0 + g + 8 * rr;
                                    const float x = v[2 * rr + h2];
                                    if constexpr (ACT == ACT_BF16)
                                        reinterpret_cast<__nv_bfloat16*>(a.out)[o] = __float2bfloat16_rn(x);
                                    else
                                        reinterpret_cast<float*>(a.out)[o] = x;
                                }
                            }
                        }
                    }
                    rbuf ^= 1;
                }
            }
        }
    }
    __syncthreads();
}

template <int FMT>
size_t dec_smem(int max_active) {
    return static_cast<size_t>(kStages) * DecCfg<FMT>::kStageStride + 128 +
           static_cast<size_t>(max_active) * sizeof(ExpertMeta);
}

template <int FMT, int ACT>
cudaError_t launch_one(const CallArgs& a, int grid, size_t smem, cudaStream_t s) {
    void* args[] = {const_cast<CallArgs*>(&a)};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(&k_dec_fp4<FMT, ACT>), dim3(grid),
                                       dim3(kDecThreads), args, smem, s);
}

constexpr int kDecMaxActive = kDecodeMaxT * kMaxTopK + 1;  // T*k routed + one shared expert

}  // namespace

bool decode_fp4_supported(int fmt, int T) { return (fmt == FMT_NVFP4 || fmt == FMT_MXFP4) && T <= kDecodeMaxT; }

cudaError_t decode_fp4_set_attributes() {
    cudaError_t e;
    const int nv = static_cast<int>(dec_smem<FMT_NVFP4>(kDecMaxActive));
    const int mx = static_cast<int>(dec_smem<FMT_MXFP4>(kDecMaxActive));
    if ((e = cudaFuncSetAttribute(k_dec_fp4<FMT_NVFP4, ACT_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, nv))) return e;
    if ((e = cudaFuncSetAttribute(k_dec_fp4<FMT_NVFP4, ACT_FP32>, cudaFuncAttributeMaxDynamicSharedMemorySize, nv))) return e;
    if ((e = cudaFuncSetAttribute(k_dec_fp4<FMT_MXFP4, ACT_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx))) return e;
    if ((e = cudaFuncSetAttribute(k_dec_fp4<FMT_MXFP4, ACT_FP32>, cudaFuncAttributeMaxDynamicSharedMemorySize, mx))) return e;
    return cudaSuccess;
}

cudaError_t launch_decode_fp4(const CallArgs& a, int num_sms, cudaStream_t s) {
    const int max_active = std::min(a.E, a.T * a.k) + a.n_shared;
    const bool bf = a.act == ACT_BF16;
    if (a.fmt == FMT_NVFP4) {
        const size_t smem = dec_smem<FMT_NVFP4>(max_active);
        return bf ? launch_one<FMT_NVFP4, ACT_BF16>(a, num_sms, smem, s) : launch_one<FMT_NVFP4, ACT_FP32>(a, num_sms, smem, s);
    }
    const size_t smem = dec_smem<FMT_MXFP4>(max_active);
    return bf ? launch_one<FMT_MXFP4, ACT_BF16>(a, num_sms, smem, s) : launch_one<FMT_MXFP4, ACT_FP32>(a, num_sms, smem, s);
}

}  // namespace moe
