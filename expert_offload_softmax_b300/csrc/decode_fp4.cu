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
constexpr int kRows = kTileRows;                    // weight rows per stage (one m16 tile)
constexpr int kGroupsPerStage = kChunkGroups;       // 128-element K groups per chunk (one per consumer)
constexpr int kChunksPerStage = 2;                  // a bulk copy costs about the same up to ~9 KB: copy >= 17 KB
constexpr int kStages = 7;
constexpr unsigned long long kDecWaitNs = 2000000000ull;  // 2 s per wait

template <int FMT>
struct DecCfg {
    static constexpr int kSbpg = FMT == FMT_NVFP4 ? 8 : 4;                     // scale bytes per group
    static constexpr int kChunkBytes = kRows * kGroupsPerStage * (64 + kSbpg);  // one full chunk of a tile
    static constexpr int kStageStride = (kChunksPerStage * kChunkBytes + 127) / 128 * 128;
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

// waits for the phase of parity `parity` for up to ~20 us (the thread is
// suspended, not spinning, and resumes as soon as the phase completes)
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

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned int atom_add_acqrel_gpu(unsigned int* p, unsigned int v) {
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void st_relaxed_gpu(unsigned int* p, unsigned int v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_add_release_gpu(unsigned int* p, unsigned int v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
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

// scales of staged row r for consumer group w of a chunk with ng groups, times mul
template <int FMT>
__device__ __forceinline__ void stage_scales(const unsigned char* st, int ng, int r, int w, float mul, float (&s)[8]) {
    const unsigned char* p = st + fp4_scale_off(ng, DecCfg<FMT>::kSbpg, r, w);
    if constexpr (FMT == FMT_NVFP4) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        e4m3x8_to_f32(v, s);
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i] *= mul;
    } else {
        const uint32_t v = *reinterpret_cast<const uint32_t*>(p);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const float f = e8m0_to_f32((v >> (8 * b)) & 0xFFu) * mul;
            s[2 * b] = f;
            s[2 * b + 1] = f;
        }
    }
}

// one 128-element group of a staged 16-row chunk (ng groups) against one
// 8-column B run: acc (rows g / g+8, columns 2q / 2q+1) += sum over the 8 MMA
// steps of scale * MMA
template <int FMT>
__device__ __forceinline__ void stage_group(const unsigned char* st, int ng, int w, int g, int q, float mul,
                                            const uint32_t (&b)[16], float (&acc)[4]) {
    const uint4 ra = lds128(st + fp4_code_off(ng, g, w, q));
    const uint4 rb = lds128(st + fp4_code_off(ng, g + 8, w, q));
    float sa[8], sb[8];
    stage_scales<FMT>(st, ng, g, w, mul, sa);
    stage_scales<FMT>(st, ng, g + 8, w, mul, sb);
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

// shared-memory activation rows are padded by 16 bytes (a 4-bank shift per row)
__host__ __device__ inline int act_pitch(int K) { return K * 2 + 16; }

// bytes of the activation area: the T token rows of x for phase 1, then the
// h rows of phase 2 in the same place; 0 when they do not fit (global loads)
__host__ __device__ inline int dec_act_bytes(int T, int H, int I, int rows, int budget) {
    const int x = T * act_pitch(H), h = rows * act_pitch(I);
    const int need = x > h ? x : h;
    return need <= budget ? need : 0;
}

template <int FMT, int ACT>
__global__ void __launch_bounds__(kDecThreads, 1) k_dec_fp4(CallArgs a, int max_active, int act_bytes) {
    using C = DecCfg<FMT>;
    extern __shared__ unsigned char dec_raw[];
    __shared__ __align__(8) uint64_t full[kStages], empty[kStages], init_bar;
    __shared__ float red[2][kConsumers][32][4];
    __shared__ int s_abort, s_gb_ok, s_ready;

    unsigned char* ring = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dec_raw) + 127) & ~uintptr_t(127));
    unsigned char* plan = ring + kStages * C::kStageStride;  // header + max_active records
    DecExpert* meta = reinterpret_cast<DecExpert*>(plan + kDecPlanHeader);
    unsigned char* act = plan + kDecPlanHeader + static_cast<size_t>(max_active) * sizeof(DecExpert);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int H = a.H, I = a.I, T = a.T;
    const int UT = I / 8;                  // gate/up unit tiles (8 units = 16 rows) per expert
    const int G1 = H / kGroupK, G2 = I / kGroupK;
    const int nch1 = (G1 + kGroupsPerStage - 1) / kGroupsPerStage;
    const int nch2 = (G2 + kGroupsPerStage - 1) / kGroupsPerStage;
    const int n2 = H / kRows;              // phase-2 row tiles
    const int G = gridDim.x, b = blockIdx.x;
    const int rt_first = G - 1 - b;        // phase-2 tiles go to the CTAs with the least phase-1 work first
    const int my2 = rt_first < n2 ? (n2 - 1 - rt_first) / G + 1 : 0;
    const int xp = act_pitch(H), hp = act_pitch(I);
    volatile int* abort_flag = &s_abort;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumers);
        }
        mbar_init(&init_bar, 1);
        s_abort = 0;
        s_gb_ok = 1;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // the plan and the token rows of x: one round trip
        const uint32_t pbytes = kDecPlanHeader + static_cast<uint32_t>(max_active) * sizeof(DecExpert);
        const uint32_t xrow = static_cast<uint32_t>(H) * 2;
        mbar_expect_tx(&init_bar, pbytes + (act_bytes ? static_cast<uint32_t>(T) * xrow : 0u));
        bulk_g2s(plan, a.dplan, pbytes, &init_bar);
        if (act_bytes)
            for (int t = 0; t < T; ++t)
                bulk_g2s(act + t * xp, reinterpret_cast<const unsigned char*>(a.xh) + static_cast<size_t>(t) * xrow,
                         xrow, &init_bar);
        // the call's expert weights must have landed in the pool
        s_ready = wait_ready(a) ? 1 : 0;
        if (!mbar_wait(&init_bar, 0, abort_flag)) {
            atomicExch(a.dev_err, MOE_DEVERR_TIMEOUT_PRODUCER);
            s_ready = 0;
        }
        if (!s_ready) s_abort = 1;
    }
    __syncthreads();
    const int na = s_ready ? *reinterpret_cast<const int32_t*>(plan) : 0;
    const int n1 = na * UT;                // phase-1 tasks
    const int my1 = b < n1 ? (n1 - 1 - b) / G + 1 : 0;

    if (warp == 0) {
        // ---------------------------------------------------------------- producer
        int stage = 0;
        uint32_t phase = 0;
        int issued[kStages];
#pragma unroll
        for (int s = 0; s < kStages; ++s) issued[s] = -1;
        bool ok = s_ready != 0;
        // one stage = up to kChunksPerStage consecutive chunks of a tile,
        // contiguous in the blob: one bulk copy
        auto issue = [&](const unsigned char* tile, int G, int c0, int nc) -> bool {
            bool got = true;
            if (lane == 0) {
                got = mbar_wait(&empty[stage], phase ^ 1u, abort_flag) && !*abort_flag;
                if (got) {
                    uint32_t bytes = 0;
                    for (int c = c0; c < c0 + nc; ++c) bytes += static_cast<uint32_t>(kRows) * fp4_chunk_groups(G, c) * (64 + C::kSbpg);
                    mbar_expect_tx(&full[stage], bytes);
                    bulk_g2s(ring + stage * C::kStageStride, tile + fp4_chunk_off(c0, C::kSbpg), bytes, &full[stage]);
                }
            }
            got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
            if (!got) return false;
            issued[stage] = static_cast<int>(phase);
            if (++stage == kStages) { stage = 0; phase ^= 1u; }
            return true;
        };
        // phase 1: the gate/up tile of unit tile ut
        for (int i = 0; i < my1 && ok; ++i) {
            const int task = b + i * G;
            const int u = task / UT, ut = task % UT;
            const unsigned char* tile = meta[u].ptr + a.lay.gu + static_cast<size_t>(ut) * a.lay.gu_tile;
            for (int c = 0; c < nch1 && ok; c += kChunksPerStage) ok = issue(tile, G1, c, min(kChunksPerStage, nch1 - c));
        }
        // phase 2: down tile rt of every active expert
        for (int i = 0; i < my2 && ok; ++i) {
            const int rt = rt_first + i * G;
            for (int u = 0; u < na && ok; ++u) {
                const unsigned char* tile = meta[u].ptr + a.lay.d + static_cast<size_t>(rt) * a.lay.d_tile;
                for (int c = 0; c < nch2 && ok; c += kChunksPerStage) ok = issue(tile, G2, c, min(kChunksPerStage, nch2 - c));
            }
        }
        if (!ok && lane == 0 && s_ready && !*abort_flag) {
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
        // NVFP4 per-tensor scales live in the blobs (readable once the call is released)
        for (int u = ct; u < na; u += 32 * kConsumers) {
            if constexpr (FMT == FMT_NVFP4) {
                const float4 v = *reinterpret_cast<const float4*>(meta[u].ptr + a.lay.gsc);
                meta[u].gs[0] = v.x; meta[u].gs[1] = v.y; meta[u].gs[2] = v.z;
            } else {
                meta[u].gs[0] = meta[u].gs[1] = meta[u].gs[2] = 1.0f;
            }
        }
        consumer_sync();
        const uint16_t* xh = reinterpret_cast<const uint16_t*>(a.xh);
        const uint16_t* hb = reinterpret_cast<const uint16_t*>(a.hbuf);
        int stage = 0;
        uint32_t phase = 0;
        bool dead = !s_ready;
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
        // B run (32 activations of token column g for group j) from the staged rows
        // in shared memory, or from global memory when they did not fit
        auto load_b = [&](const unsigned char* rows, int pitch, const uint16_t* grow, int K, int r, int j,
                          uint32_t (&bq)[16], bool cg) {
            if (r < 0) {
#pragma unroll
                for (int x = 0; x < 16; ++x) bq[x] = 0u;
            } else if (act_bytes) {
                const unsigned char* p = rows + r * pitch + j * 256 + 64 * q;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const uint4 x = lds128(p + 16 * v);
                    bq[4 * v] = x.x; bq[4 * v + 1] = x.y; bq[4 * v + 2] = x.z; bq[4 * v + 3] = x.w;
                }
            } else if (cg) {
                load_bcol<true>(grow + static_cast<size_t>(r) * K + j * kGroupK + 32 * q, bq);
            } else {
                load_bcol<false>(grow + static_cast<size_t>(r) * K + j * kGroupK + 32 * q, bq);
            }
        };
        const int ns1 = (nch1 + kChunksPerStage - 1) / kChunksPerStage;  // stages per gate/up tile
        const int ns2 = (nch2 + kChunksPerStage - 1) / kChunksPerStage;  // stages per down tile
        // ---------------- phase 1: gate/up + SwiGLU
        {
            const int nf = my1 * ns1;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int f = 0; f < nf; ++f) {
                const int i = f / ns1, sidx = f % ns1;
                const int task = b + i * G, u = task / UT, ut = task % UT;
                const int tok = meta[u].tok[g];
                if (sidx == 0) acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
                const unsigned char* st = wait_full();
#pragma unroll
                for (int cc = 0; cc < kChunksPerStage; ++cc) {
                    const int c = sidx * kChunksPerStage + cc;
                    if (c < nch1) {
                        const int ng = fp4_chunk_groups(G1, c);
                        if (w < ng) {
                            uint32_t bq[16];
                            load_b(act, xp, xh, H, tok, c * kGroupsPerStage + w, bq, false);
                            if (!dead) stage_group<FMT>(st + cc * C::kChunkBytes, ng, w, g, q, 1.0f, bq, acc);
                        }
                    }
                }
                release();
                if (sidx == ns1 - 1) {
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
                        const DecExpert& m = meta[u];
                        const int unit = ut * 8 + g;
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const int n = 2 * q + h2;
                            if (n < m.cnt) {
                                const int r = m.row0 + n;
                                const float gate = v[h2] * m.gs[0], up = v[2 + h2] * m.gs[1];
                                const float actv = a.mode == 1 ? gate : silu(gate);
                                reinterpret_cast<__half*>(a.hbuf)[static_cast<size_t>(r) * I + dpos(unit)] =
                                    __float2half_rn(actv * up * m.gate[n]);
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
            // arrivals counted with an acquire-release add (it publishes this CTA's
            // h rows); the last arrival resets the count and bumps the generation
            // with a release; everyone else polls it with acquire loads (bounded)
            int okb = *abort_flag ? 0 : 1;
            if (okb) {
                unsigned int* cnt = a.grid_bar;
                unsigned int* gen = a.grid_bar + 1;
                const unsigned int my_gen = ld_acquire_gpu(gen);
                const unsigned int prev = atom_add_acqrel_gpu(cnt, 1u);
                if (prev == static_cast<unsigned int>(G) - 1u) {
                    st_relaxed_gpu(cnt, 0u);
                    red_add_release_gpu(gen, 1u);
                } else {
                    const uint64_t t0 = gtimer();
                    while (ld_acquire_gpu(gen) == my_gen) {
                        if (gtimer() - t0 > kDecWaitNs) {
                            okb = 0;
                            atomicExch(a.dev_err, MOE_DEVERR_TIMEOUT_EPILOGUE);
                            *abort_flag = 1;
                            break;
                        }
                    }
                }
            }
            s_gb_ok = okb;
        }
        consumer_sync();
        // ---------------- phase 2: down projection + combine
        if (s_gb_ok && my2 > 0) {
            // every h row of the call into shared memory: one round trip
            const int hrows = T * (a.k + a.n_shared);
            if (act_bytes) {
                // each thread issues all its loads before its first store
                constexpr int kB = 8;
                constexpr int kNt = 32 * kConsumers;
                const int per_row = I / 8;  // uint4 per row
                const int n = hrows * per_row;
                for (int i0 = ct; i0 < n; i0 += kNt * kB) {
                    uint4 v[kB];
#pragma unroll
                    for (int x = 0; x < kB; ++x) {
                        const int i = i0 + x * kNt;
                        if (i < n) v[x] = __ldcg(reinterpret_cast<const uint4*>(hb + static_cast<size_t>(i / per_row) * I) + i % per_row);
                    }
#pragma unroll
                    for (int x = 0; x < kB; ++x) {
                        const int i = i0 + x * kNt;
                        if (i < n) *reinterpret_cast<uint4*>(act + (i / per_row) * hp + 16 * (i % per_row)) = v[x];
                    }
                }
                consumer_sync();
            }
            const int per_tile = na * ns2;
            const int nf = my2 * per_tile;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int f = 0; f < nf; ++f) {
                const int i = f / per_tile, r = f % per_tile, u = r / ns2, sidx = r % ns2;
                const int hr = meta[u].hrow[g];
                if (r == 0) acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
                const unsigned char* st = wait_full();
#pragma unroll
                for (int cc = 0; cc < kChunksPerStage; ++cc) {
                    const int c = sidx * kChunksPerStage + cc;
                    if (c < nch2) {
                        const int ng = fp4_chunk_groups(G2, c);
                        if (w < ng) {
                            uint32_t bq[16];
                            load_b(act, hp, hb, I, hr, c * kGroupsPerStage + w, bq, true);
                            if (!dead) stage_group<FMT>(st + cc * C::kChunkBytes, ng, w, g, q, meta[u].gs[2], bq, acc);
                        }
                    }
                }
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

constexpr int kDecSmemLimit = 216 * 1024;  // dynamic bytes; the static part (~8 KB) sits beside it

template <int FMT>
size_t dec_fixed_smem(int max_active) {
    return static_cast<size_t>(kStages) * DecCfg<FMT>::kStageStride + 128 + kDecPlanHeader +
           static_cast<size_t>(max_active) * sizeof(DecExpert);
}

template <int FMT, int ACT>
cudaError_t launch_one(const CallArgs& a, int grid, cudaStream_t s) {
    int max_active = std::min(a.E, a.T * a.k) + a.n_shared;
    const size_t fixed = dec_fixed_smem<FMT>(max_active);
    const int budget = static_cast<int>(kDecSmemLimit - fixed);
    int act_bytes = dec_act_bytes(a.T, a.H, a.I, a.T * (a.k + a.n_shared), budget);
    const size_t smem = fixed + act_bytes;
    void* args[] = {const_cast<CallArgs*>(&a), &max_active, &act_bytes};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(&k_dec_fp4<FMT, ACT>), dim3(grid),
                                       dim3(kDecThreads), args, smem, s);
}

}  // namespace

bool decode_fp4_supported(int fmt, int T) { return (fmt == FMT_NVFP4 || fmt == FMT_MXFP4) && T <= kDecodeMaxT; }

cudaError_t decode_fp4_set_attributes() {
    cudaError_t e;
    const int lim = kDecSmemLimit;
    if ((e = cudaFuncSetAttribute(k_dec_fp4<FMT_NVFP4, ACT_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim))) return e;
    if ((e = cudaFuncSetAttribute(k_dec_fp4<FMT_NVFP4, ACT_FP32>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim))) return e;
    if ((e = cudaFuncSetAttribute(k_dec_fp4<FMT_MXFP4, ACT_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim))) return e;
    if ((e = cudaFuncSetAttribute(k_dec_fp4<FMT_MXFP4, ACT_FP32>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim))) return e;
    return cudaSuccess;
}

cudaError_t launch_decode_fp4(const CallArgs& a, int num_sms, cudaStream_t s) {
    const bool bf = a.act == ACT_BF16;
    if (a.fmt == FMT_NVFP4)
        return bf ? launch_one<FMT_NVFP4, ACT_BF16>(a, num_sms, s) : launch_one<FMT_NVFP4, ACT_FP32>(a, num_sms, s);
    return bf ? launch_one<FMT_MXFP4, ACT_BF16>(a, num_sms, s) : launch_one<FMT_MXFP4, ACT_FP32>(a, num_sms, s);
}

}  // namespace moe
