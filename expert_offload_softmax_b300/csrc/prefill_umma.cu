// Prefill expert GEMMs of the routed MoE layer on the 5th-generation tensor
// cores: tcgen05.mma (kind::f16, BF16 operands, fp32 accumulators in tensor
// memory), operand tiles staged by TMA into 128-byte-swizzled shared memory,
// one persistent CTA per SM with warp-specialised roles.
//
// Prefill is where the layer is a real dense contraction: with T tokens and
// top-k routing every active expert sees about T*k/E tokens (128 at T=4096,
// E=256, k=8), so each expert's weights are streamed once and reused across
// its tokens. The pages' prefill paragraph (freetoken.wiki architecture page:
// whole-layer double buffering, the next layer's experts streaming over PCIe
// while the current layer computes) is served by the host runtime; these
// kernels are the "current layer computes" part.
//
// Swap-AB: the weight rows are the MMA's M = 128 operand (A), the tokens routed
// to one expert are N (B), K is the projection's input dimension. Both operands
// are K-major; the K permutation the library stores weights in (see
// moe_internal.h) is applied to the activations too, so every dot product is
// over the same pairs.
//
//  gate/up: per tile, 128 intermediate units x up to 128 tokens; two
//           accumulators (gate rows, up rows of the same units); the epilogue
//           applies SwiGLU and the routing gate and writes h (bf16).
//  down:    per tile, 128 output rows x up to 128 tokens; the epilogue writes
//           the expert's output rows Y (bf16), combined later per token.
//
// Roles (192 threads): warp 0 = TMA producer, warp 1 = MMA issuer and TMEM
// owner, warps 2-5 = epilogue (TMEM lane quarter = warp % 4). Every wait is
// bounded by %globaltimer; on timeout the kernel records an error, lets its
// copies and MMAs in flight finish (bounded again), frees its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>

#include "mma_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int BM = 128;  // weight rows per accumulator (MMA M)
constexpr int BN = 128;  // tokens per tile (MMA N at most)
constexpr int BK = 64;   // K per pipeline stage: 64 bf16 = one 128-byte swizzle row
constexpr int kThreads = 192;                   // BF16 weights: producer, MMA, 4 epilogue warps
constexpr int kXformWarps = 16;                 // FP4 / FP8 weights: + warps that widen the A tiles (4 per stage)
constexpr int kThreadsFp4 = kThreads + 32 * kXformWarps;
constexpr int kTileBytes = BM * BK * 2;  // 16 KB: one 128 x 64 bf16 operand tile

enum { MODE_GU = 0, MODE_DOWN = 1 };

template <int MODE, bool FP4 = false>
struct Cfg {
    static constexpr int kATiles = MODE == MODE_GU ? 2 : 1;           // gate + up, or down
    static constexpr int kStageBytes = (kATiles + 1) * kTileBytes;   // A tiles + B tile
    // FP4 / FP8: 4 stages, each written by four transform warps (see XPart)
    static constexpr int kStages = (MODE == MODE_GU || FP4) ? 4 : 6;
    static constexpr int kAccCols = kATiles * BN;                    // TMEM columns per accumulator set
    static constexpr int kTmemCols = 2 * kAccCols;                   // double-buffered: 512 / 256
    static constexpr int kSmem = kStages * kStageBytes + 1024;       // + alignment slack
};

// ------------------------------------------------------------------ PTX helpers

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

// Waits for the phase of parity `parity` to complete. Gives up (false) when
// another role of this CTA has aborted or after wait_ns (the handle's bound on
// every device wait, MOE_WAIT_MS).
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

__device__ __forceinline__ void tma_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];"
        ::"r"(su32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(su32(bar)), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
        ::"r"(su32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(su32(bar)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes, 8-row atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
    d |= static_cast<uint64_t>(1) << 16;                  // leading byte offset (unused when swizzled)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride byte offset: next 8-row atom
    d |= static_cast<uint64_t>(1) << 46;                  // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                  // 128-byte swizzle
    return d;
}

// Instruction descriptor: BF16 x BF16 -> F32, both operands K-major, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// the same for f16 A and B (A/B type fields 0)
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// gate/up with NVFP4 or FP8 weights runs on f16 operands: the codes (times
// NVFP4's E4M3 block scale) widen to f16 exactly in one conversion, and each
// token row of X is scaled by a power of two into f16's range (exact for every
// element of the row within 2^29 of its largest); everything else is bf16
template <int FMT, int MODE>
__host__ __device__ constexpr bool f16_operands() {
    return MODE == MODE_GU && (FMT == FMT_NVFP4 || FMT == FMT_FP8);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
                 : "memory");
}

// this thread's TMEM lane, 16 consecutive fp32 columns starting at taddr
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// this thread's TMEM lane, 32 consecutive fp32 columns starting at taddr
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// position of intermediate unit i in the library's K order
__device__ __forceinline__ int kpos(int i) {
    const int w = i & 127, s = w >> 4, q = (w >> 2) & 3, e = w & 3;
    return (i & ~127) + 32 * q + 4 * s + e;
}

// ------------------------------------------------------------------ kernel

struct TileSched {
    int32_t start[kMaxExperts + 2];  // first tile of active expert u; start[n_active] = total
};

__device__ __forceinline__ int find_expert(const TileSched& ts, int na, int t) {
    int lo = 0, hi = na - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (ts.start[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// FP4 and FP8 weights (NVFP4 / MXFP4 / FP8): the A tile of a pipeline stage
// (one 64-element K block of 128 weight rows, or 2 x 128 for gate/up) is
// written by four transform warps, each owning a quarter of its rows. Warp w serves
// stage w mod 4 and only that stage, so it is never more than one use ahead of
// the MMA (an mbarrier parity wait cannot tell use n from use n-2). A warp
// loads its rows' codes and block scales from the tiled blob (FP4: one
// position ahead, into a second register buffer; FP8, whose codes take twice
// the registers: one buffer, the next position's lines prefetched into L2),
// widens them to BF16 (exact: an E2M1 value times an E4M3 or E8M0 scale has at
// most 6 significant bits, an E4M3 value 4) and stores them in the layout a
// TMA load with 128-byte swizzling would have produced (row r at r*128 bytes,
// its 16-byte chunk c at position c ^ (r mod 8)). FP8's per-tensor scale, like
// NVFP4's, is applied in the epilogue.
// the rows of a stage's A tiles that transform warp `part` (0..3) writes: GU
// tile part % 2 (gate, up), rows 64 (part / 2) .. + 63; DOWN rows 32 part .. + 31
template <int MODE>
struct XPart {
    static constexpr int kParts = kXformWarps / 4;
    static constexpr int kRows = (MODE == MODE_GU ? 2 * BM : BM) / kParts;
    __device__ static int tile(int part) { return MODE == MODE_GU ? part & 1 : 0; }
    __device__ static int row0(int part) { return MODE == MODE_GU ? (part >> 1) * kRows : part * kRows; }
};

template <int FMT, int MODE>
struct XRows {
    static constexpr int kRows = XPart<MODE>::kRows / 32;  // rows per lane
    static constexpr int kUnits = FMT == FMT_FP8 ? 4 : 2;  // 16-byte code units per row and K block
    uint4 codes[kRows][kUnits];  // FP8: piece 4i + j = codes[i][j], see xload
    uint2 sc[kRows];
};

// tile row `trow` and tile base of row `rl` of part `part` of M tile mt
template <int MODE>
__device__ __forceinline__ const uint8_t* xrow(const CallArgs& a, const uint8_t* blob, int mt, int part, int rl, int& trow) {
    if constexpr (MODE == MODE_GU) {
        const int unit = mt * BM + XPart<MODE>::row0(part) + rl;
        trow = 8 * XPart<MODE>::tile(part) + unit % 8;  // gate rows 0-7, up rows 8-15 of the unit tile
        return blob + a.lay.gu + static_cast<size_t>(unit / 8) * a.lay.gu_tile;
    } else {
        const int row = mt * BM + XPart<MODE>::row0(part) + rl;
        trow = row % kTileRows;
        return blob + a.lay.d + static_cast<size_t>(row / kTileRows) * a.lay.d_tile;
    }
}

// loads, for K block kb of M tile mt of the expert at blob, the rows of part
// `part` (see XPart) that this lane owns
template <int FMT, int MODE>
__device__ __forceinline__ void xload(const CallArgs& a, const uint8_t* blob, int mt, int kb, int part, int lane,
                                      XRows<FMT, MODE>& x) {
    constexpr int kSbpg = tiled_scale_bytes(FMT);
    const int G = (MODE == MODE_GU ? a.H : a.I) / kGroupK;
    const int j = kb >> 1, h = kb & 1;  // K group, half of it
    const int c = j / kChunkGroups, w = j % kChunkGroups, ng = fp4_chunk_groups(G, c);
    if constexpr (FMT == FMT_FP8) {
        // FP8: step i of lane l takes 16-byte unit l & 3 of the K block (quad 2h + (l & 3) / 2, half
        // (l & 3) % 2) of row 8i + l / 4, so each load instruction covers 8 whole 64-byte row segments
        const int u = lane & 3;
#pragma unroll
        for (int i = 0; i < XRows<FMT, MODE>::kRows * 4; ++i) {
            int trow;
            const uint8_t* chunk = xrow<MODE>(a, blob, mt, part, 8 * i + (lane >> 2), trow) + tile_chunk_off(c, tiled_row_bytes(FMT));
            x.codes[i >> 2][i & 3] = __ldg(reinterpret_cast<const uint4*>(chunk + fp8_code_off(ng, trow, w, 2 * h + (u >> 1), u & 1)));
        }
    } else {
#pragma unroll
        for (int i = 0; i < XRows<FMT, MODE>::kRows; ++i) {
            int trow;
            const uint8_t* chunk = xrow<MODE>(a, blob, mt, part, lane + 32 * i, trow) + tile_chunk_off(c, tiled_row_bytes(FMT));
            x.codes[i][0] = __ldg(reinterpret_cast<const uint4*>(chunk + fp4_code_off(ng, trow, w, 2 * h)));
            x.codes[i][1] = __ldg(reinterpret_cast<const uint4*>(chunk + fp4_code_off(ng, trow, w, 2 * h + 1)));
            if constexpr (FMT == FMT_NVFP4)
                x.sc[i] = __ldg(reinterpret_cast<const uint2*>(chunk + fp4_scale_off(ng, kSbpg, trow, w)));
            else
                x.sc[i] = make_uint2(__ldg(reinterpret_cast<const uint32_t*>(chunk + fp4_scale_off(ng, kSbpg, trow, w))), 0u);
        }
    }
}

// FP8: asks L2 for the 128-byte lines that xload will read for this position
template <int MODE>
__device__ __forceinline__ void xprefetch_fp8(const CallArgs& a, const uint8_t* blob, int mt, int kb, int part, int lane) {
    const int G = (MODE == MODE_GU ? a.H : a.I) / kGroupK;
    const int j = kb >> 1;
    const int c = j / kChunkGroups, w = j % kChunkGroups, ng = fp4_chunk_groups(G, c);
    if ((lane & 3) != 0) return;
#pragma unroll
    for (int i = 0; i < XRows<FMT_FP8, MODE>::kRows * 4; ++i) {
        int trow;
        const uint8_t* chunk = xrow<MODE>(a, blob, mt, part, 8 * i + (lane >> 2), trow) + tile_chunk_off(c, tiled_row_bytes(FMT_FP8));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(chunk + (trow * ng + w) * 128) : "memory");
    }
}

// widens the loaded rows into the stage's A tile
template <int FMT, int MODE>
__device__ __forceinline__ void xstore(const XRows<FMT, MODE>& x, unsigned char* st, int part, int lane) {
#pragma unroll
    for (int i = 0; i < XRows<FMT, MODE>::kRows; ++i) {
        const int r = XPart<MODE>::row0(part) + lane + 32 * i;  // row of the 128-row A tile
        unsigned char* rowp = st + XPart<MODE>::tile(part) * kTileBytes + r * 128;
        if constexpr (FMT == FMT_FP8) {
            // pieces as xload took them: 16 codes = K positions 16u .. 16u+15 of row 8i' + lane / 4 -> chunks 2u, 2u+1
            const int u = lane & 3;
#pragma unroll
            for (int i2 = 0; i2 < 4; ++i2) {
                const int ip = 4 * i + i2;
                const int rr = XPart<MODE>::row0(part) + 8 * ip + (lane >> 2);
                unsigned char* rp = st + XPart<MODE>::tile(part) * kTileBytes + rr * 128;
                uint32_t f[8];
                e4m3x8_to_f16x2(make_uint2(x.codes[i][i2].x, x.codes[i][i2].y), *reinterpret_cast<uint32_t(*)[4]>(f));
                e4m3x8_to_f16x2(make_uint2(x.codes[i][i2].z, x.codes[i][i2].w), *reinterpret_cast<uint32_t(*)[4]>(f + 4));
                if constexpr (!f16_operands<FMT, MODE>()) {
#pragma unroll
                    for (int y = 0; y < 8; ++y) {
                        const __half2 hv = *reinterpret_cast<const __half2*>(&f[y]);
                        __nv_bfloat162 bv = __floats2bfloat162_rn(__low2float(hv), __high2float(hv));
                        f[y] = *reinterpret_cast<uint32_t*>(&bv);
                    }
                }
                *reinterpret_cast<uint4*>(rp + (((2 * u) ^ (rr & 7)) << 4)) = make_uint4(f[0], f[1], f[2], f[3]);
                *reinterpret_cast<uint4*>(rp + (((2 * u + 1) ^ (rr & 7)) << 4)) = make_uint4(f[4], f[5], f[6], f[7]);
            }
            continue;
        } else if constexpr (FMT == FMT_NVFP4 && f16_operands<FMT, MODE>()) {
            // code x block scale in f16: at most 6 significant bits, within [2^-10, 2688]
            uint32_t sh[4];
            e4m3x8_to_f16x2(x.sc[i], sh);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const uint32_t wv[4] = {x.codes[i][u].x, x.codes[i][u].y, x.codes[i][u].z, x.codes[i][u].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {  // 4 code bytes -> 8 elements -> one 16-byte chunk
                    uint32_t f[4];
                    fp4x8_to_f16x2(wv[q], f);
#pragma unroll
                    for (int y = 0; y < 4; ++y) {
                        const int st = (4 * q + y) >> 1;  // K step of this pair: its block scale
                        const uint32_t sc2 = __byte_perm(sh[st >> 1], 0u, (st & 1) ? 0x3232u : 0x1010u);
                        __half2 v = __hmul2(*reinterpret_cast<const __half2*>(&f[y]), *reinterpret_cast<const __half2*>(&sc2));
                        f[y] = *reinterpret_cast<uint32_t*>(&v);
                    }
                    const int c16 = 4 * u + q;
                    *reinterpret_cast<uint4*>(rowp + ((c16 ^ (r & 7)) << 4)) = make_uint4(f[0], f[1], f[2], f[3]);
                }
            }
            continue;
        }
        float s8[8];
        if constexpr (FMT == FMT_NVFP4) {
            e4m3x8_to_f32(x.sc[i], s8);
        } else {
#pragma unroll
            for (int b = 0; b < 4; ++b) s8[2 * b] = s8[2 * b + 1] = e8m0_to_f32((x.sc[i].x >> (8 * b)) & 0xFFu);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const uint32_t wv[4] = {x.codes[i][u].x, x.codes[i][u].y, x.codes[i][u].z, x.codes[i][u].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // 4 code bytes -> 8 elements -> one 16-byte chunk
                uint32_t f[4];
                fp4x8_to_f16x2(wv[q], f);
                uint32_t o[4];
#pragma unroll
                for (int y = 0; y < 4; ++y) {
                    const float sv = s8[(4 * q + y) >> 1];  // byte b of a unit holds K steps b/2
                    const __half2 hv = *reinterpret_cast<const __half2*>(&f[y]);
                    __nv_bfloat162 bv = __floats2bfloat162_rn(__low2float(hv) * sv, __high2float(hv) * sv);
                    o[y] = *reinterpret_cast<uint32_t*>(&bv);
                }
                const int c16 = 4 * u + q;
                *reinterpret_cast<uint4*>(rowp + ((c16 ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
}

template <int MODE, int FMT>
__global__ void __launch_bounds__(FMT == FMT_BF16 ? kThreads : kThreadsFp4, 1)
    k_umma_grouped(const __grid_constant__ CUtensorMap map_pool, const __grid_constant__ CUtensorMap map_shared,
                   const __grid_constant__ CUtensorMap map_b, CallArgs a) {
    constexpr bool kFp4 = FMT != FMT_BF16;
    using C = Cfg<MODE, kFp4>;
    extern __shared__ unsigned char dyn_raw[];
    __shared__ TileSched ts;
    __shared__ const uint8_t* s_ptr[kFp4 ? kMaxExperts + 1 : 1];  // blob of each active expert (FP4 / FP8)
    __shared__ int s_nnt[kFp4 ? kMaxExperts + 1 : 1];             // its token tiles (FP4 / FP8)
    __shared__ __align__(8) uint64_t bar_full[C::kStages], bar_empty[C::kStages], bar_afull[C::kStages];
    __shared__ __align__(8) uint64_t bar_tfull[2], bar_tempty[2], bar_drain;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~uintptr_t(1023));
    const int na = *a.n_active;
    const int n_mt = MODE == MODE_GU ? a.I / BM : a.H / BM;
    const int n_kb = MODE == MODE_GU ? a.H / BK : a.I / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(&bar_full[s], 1);
            mbar_init(&bar_empty[s], 1);
            mbar_init(&bar_afull[s], kXformWarps / C::kStages);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar_tfull[s], 1);
            mbar_init(&bar_tempty[s], 128);
        }
        mbar_init(&bar_drain, 1);
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&s_tmem)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // tile schedule: active expert u owns n_mt * ceil(cnt_u / BN) tiles, token tiles fastest
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base < na; base += 32) {
            const int u = base + lane;
            const int v = u < na ? n_mt * ((a.act_cnt[u] + BN - 1) / BN) : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            if (u < na) ts.start[u] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) ts.start[na] = carry;
    }
    if constexpr (kFp4)
        for (int u = threadIdx.x; u < na; u += blockDim.x) {
            s_ptr[u] = a.act_ptr[u];
            s_nnt[u] = (a.act_cnt[u] + BN - 1) / BN;
        }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    const int total = ts.start[na];
    volatile int* abort_flag = &s_abort;

    auto fail = [&](int code) {
        *abort_flag = 1;
        atomicExch(a.dev_err, code);
    };

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- producer
            int stage = 0;
            uint32_t phase = 0;
            int issued_phase[C::kStages];
#pragma unroll
            for (int s = 0; s < C::kStages; ++s) issued_phase[s] = -1;
            // the call's expert weights must have landed in the pool
            bool ok = MODE == MODE_DOWN || wait_ready(a);
            if (!ok) *abort_flag = 1;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
                const int u = find_expert(ts, na, t);
                const int local = t - ts.start[u];
                const int n_nt = (a.act_cnt[u] + BN - 1) / BN;
                const int mt = local / n_nt, nt = local % n_nt;
                const int sl = a.act_slot[u];
                const CUtensorMap* mA = sl >= 0 ? &map_pool : &map_shared;
                const int z = sl >= 0 ? sl : -sl - 1;
                const int brow = a.act_row0[u] + nt * BN;
                for (int kb = 0; kb < n_kb; ++kb) {
                    if (!mbar_wait(&bar_empty[stage], phase ^ 1u, abort_flag, a.wait_ns)) {
                        fail(MOE_DEVERR_TIMEOUT_PRODUCER);
                        ok = false;
                        break;
                    }
                    unsigned char* st = smem + stage * C::kStageBytes;
                    mbar_expect_tx(&bar_full[stage], kFp4 ? kTileBytes : C::kStageBytes);
                    if constexpr (kFp4) {
                        // A tiles come from the transform warps
                    } else if constexpr (MODE == MODE_GU) {
                        // gate rows of units [128 mt, 128 mt + 128) sit in two 64-row blocks
                        // 128 rows apart; the up rows follow each block
                        const int r0 = (mt * BM / 64) * 128;
                        tma_3d(st, mA, &bar_full[stage], kb * BK, r0, z);
                        tma_3d(st + kTileBytes / 2, mA, &bar_full[stage], kb * BK, r0 + 128, z);
                        tma_3d(st + kTileBytes, mA, &bar_full[stage], kb * BK, r0 + 64, z);
                        tma_3d(st + kTileBytes + kTileBytes / 2, mA, &bar_full[stage], kb * BK, r0 + 192, z);
                    } else {
                        tma_3d(st, mA, &bar_full[stage], kb * BK, mt * BM, z);
                    }
                    tma_2d(st + C::kATiles * kTileBytes, &map_b, &bar_full[stage], kb * BK, brow);
                    issued_phase[stage] = static_cast<int>(phase);
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // let the copies already issued land before the CTA can exit
                for (int s = 0; s < C::kStages; ++s)
                    if (issued_phase[s] >= 0) {
                        const uint64_t t0 = gtimer();
                        while (!mbar_test(&bar_full[s], static_cast<uint32_t>(issued_phase[s])) &&
                               gtimer() - t0 < a.wait_ns) {
                        }
                    }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
                const int u = find_expert(ts, na, t);
                const int local = t - ts.start[u];
                const int n_nt = (a.act_cnt[u] + BN - 1) / BN;
                const int nt = local % n_nt;
                const int rows = min(BN, a.act_cnt[u] - nt * BN);
                const uint32_t idesc = f16_operands<FMT, MODE>() ? idesc_f16(BM, (rows + 15) & ~15)
                                                                 : idesc_bf16(BM, (rows + 15) & ~15);
                const int acc = it & 1;
                const uint32_t aph = (it >> 1) & 1;
                if (!mbar_wait(&bar_tempty[acc], aph ^ 1u, abort_flag, a.wait_ns)) {
                    fail(MOE_DEVERR_TIMEOUT_MMA);
                    break;
                }
                tc_fence_after();
                const uint32_t d0 = tmem + acc * C::kAccCols;
                for (int kb = 0; kb < n_kb; ++kb) {
                    if (!mbar_wait(&bar_full[stage], phase, abort_flag, a.wait_ns) ||
                        (kFp4 && !mbar_wait(&bar_afull[stage], phase, abort_flag, a.wait_ns))) {
                        fail(MOE_DEVERR_TIMEOUT_MMA);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = su32(smem + stage * C::kStageBytes);
                    const uint32_t sb = sa + C::kATiles * kTileBytes;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t db = sdesc(sb + 32 * kk);
                        const uint32_t accum = (kb | kk) != 0;
                        umma_bf16(d0, sdesc(sa + 32 * kk), db, idesc, accum);
                        if constexpr (MODE == MODE_GU) umma_bf16(d0 + BN, sdesc(sa + kTileBytes + 32 * kk), db, idesc, accum);
                    }
                    umma_commit(&bar_empty[stage]);
                    if (++stage == C::kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (ok) umma_commit(&bar_tfull[acc]);
            }
            // every MMA issued by this thread has completed once bar_drain flips
            umma_commit(&bar_drain);
            const uint64_t t0 = gtimer();
            while (!mbar_test(&bar_drain, 0) && gtimer() - t0 < a.wait_ns) {
            }
        }
    } else if (warp >= 6) {
        // ---------------- A-tile transform (FP4 / FP8 weights, warps 6-21)
        if constexpr (kFp4) {
            const int xw = warp - 6;
            const int sidx = xw % C::kStages, part = xw / C::kStages;
            bool ok = true;
            if (lane == 0 && !wait_ready(a)) *abort_flag = 1;
            __syncwarp();
            if (*abort_flag) ok = false;
            // this warp's positions: sidx, sidx + 4, ... over this CTA's tiles (n_kb each)
            const int my_tiles = blockIdx.x < total ? (total - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
            const long long npos = static_cast<long long>(my_tiles) * n_kb;
            // everything from shared memory: a position costs no memory round trip
            auto where = [&](long long P, const uint8_t*& blob, int& mt, int& kb) {
                const int i = static_cast<int>(P) / n_kb;
                kb = static_cast<int>(P) - i * n_kb;
                const int t = blockIdx.x + i * gridDim.x;
                const int u = find_expert(ts, na, t);
                mt = (t - ts.start[u]) / s_nnt[u];
                blob = s_ptr[u];
            };
            auto process = [&](long long P, const XRows<FMT, MODE>& x) -> bool {
                const uint32_t ph = static_cast<uint32_t>((P / C::kStages) & 1);
                int got = 1;
                if (lane == 0) got = mbar_wait(&bar_empty[sidx], ph ^ 1u, abort_flag, a.wait_ns) ? 1 : 0;
                got = __shfl_sync(0xffffffffu, got, 0);
                if (!got) {
                    if (lane == 0) fail(MOE_DEVERR_TIMEOUT_PRODUCER);
                    return false;
                }
                xstore<FMT, MODE>(x, smem + sidx * C::kStageBytes, part, lane);
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar_afull[sidx]);
                return true;
            };
            const uint8_t* blob;
            int mt, kb;
            long long P = sidx;
            if constexpr (FMT == FMT_FP8) {
                XRows<FMT, MODE> xa;
                if (ok && P < npos) {
                    where(P, blob, mt, kb);
                    xload<FMT, MODE>(a, blob, mt, kb, part, lane, xa);
                }
                while (ok && P < npos) {
                    const long long P1 = P + C::kStages;
                    if (P1 < npos) {
                        where(P1, blob, mt, kb);
                        xprefetch_fp8<MODE>(a, blob, mt, kb, part, lane);
                    }
                    ok = process(P, xa);
                    if (!ok || P1 >= npos) break;
                    xload<FMT, MODE>(a, blob, mt, kb, part, lane, xa);
                    P = P1;
                }
            } else {
            XRows<FMT, MODE> xa, xb;
            if (ok && P < npos) {
                where(P, blob, mt, kb);
                xload<FMT, MODE>(a, blob, mt, kb, part, lane, xa);
            }
            while (ok && P < npos) {
                const long long P1 = P + C::kStages;
                if (P1 < npos) {
                    where(P1, blob, mt, kb);
                    xload<FMT, MODE>(a, blob, mt, kb, part, lane, xb);
                }
                ok = process(P, xa);
                if (!ok || P1 >= npos) break;
                const long long P2 = P1 + C::kStages;
                if (P2 < npos) {
                    where(P2, blob, mt, kb);
                    xload<FMT, MODE>(a, blob, mt, kb, part, lane, xa);
                }
                ok = process(P1, xb);
                P = P2;
            }
            }
        }
    } else {
        // ---------------- epilogue (warps 2-5)
        const int quarter = warp & 3;
        const int row_in_tile = quarter * 32 + lane;
        int it = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
            const int u = find_expert(ts, na, t);
            const int local = t - ts.start[u];
            const int cnt = a.act_cnt[u];
            const int n_nt = (cnt + BN - 1) / BN;
            const int mt = local / n_nt, nt = local % n_nt;
            const int rows = min(BN, cnt - nt * BN);
            const int r0 = a.act_row0[u] + nt * BN;
            const int acc = it & 1;
            const uint32_t aph = (it >> 1) & 1;
            if (!mbar_wait(&bar_tfull[acc], aph, abort_flag, a.wait_ns)) {
                fail(MOE_DEVERR_TIMEOUT_EPILOGUE);
                break;
            }
            tc_fence_after();
            const uint32_t tbase = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + acc * C::kAccCols;
            float gsc0 = 1.0f, gsc1 = 1.0f;
            if (a.fmt == FMT_NVFP4 || a.fmt == FMT_FP8) {
                const float* g = reinterpret_cast<const float*>(a.act_ptr[u] + a.lay.gsc);
                gsc0 = MODE == MODE_GU ? g[0] : g[2];
                gsc1 = g[1];
            }
            if constexpr (MODE == MODE_GU) {
                const int unit = mt * BM + row_in_tile;
                __nv_bfloat16* hrow = reinterpret_cast<__nv_bfloat16*>(a.hbuf) + kpos(unit);
                // 16 columns at a time: the FP4 / FP8 kernels run 22 warps on 80 registers
                for (int c0 = 0; c0 < rows; c0 += 16) {
                    float g[16], up[16];
                    tmem_ld16(tbase + c0, g);
                    tmem_ld16(tbase + BN + c0, up);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c0 + j < rows) {
                            const int r = r0 + c0 + j;
                            // f16 operands: undo the row's power of two first (exact)
                            const float un = f16_operands<FMT, MODE>() ? a.xunr[r] : 1.0f;
                            const float gv = (g[j] * un) * gsc0;
                            const float act = a.mode == 1 ? gv : gv / (1.0f + expf(-gv));
                            hrow[static_cast<size_t>(r) * a.I] =
                                __float2bfloat16_rn(act * ((up[j] * un) * gsc1) * a.row_gate[r]);
                        }
                    }
                }
            } else {
                const int hr = mt * BM + row_in_tile;
                __nv_bfloat16* ycol = reinterpret_cast<__nv_bfloat16*>(a.ybuf) + hr;
                for (int c0 = 0; c0 < rows; c0 += 16) {
                    float y[16];
                    tmem_ld16(tbase + c0, y);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (c0 + j < rows) ycol[static_cast<size_t>(r0 + c0 + j) * a.H] = __float2bfloat16_rn(y[j] * gsc0);
                }
            }
            tc_fence_before();
            mbar_arrive(&bar_tempty[acc]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols) : "memory");
    }
}

// ------------------------------------------------------------------ router logits on the tensor cores
// Approximate router logits of a prefill call, L~[t][e] = sum_h x[t][h] w[e][h]
// with BF16 operands and fp32 accumulation in TMEM: one CTA per 128 tokens, all
// E (<= 256, a multiple of 32) experts as the MMA's N, K = H in 64-element TMA
// stages. The sums are not in the fixed order of the router's definition; the
// routing kernel turns them into the exact top-k (it recomputes, in the fixed
// order, every logit that their error bound leaves in contention).
constexpr int kRouterStages = 4;
constexpr int kRouterBTile = 256 * BK * 2;  // router rows of one stage (E <= 256)
constexpr int kRouterStageBytes = kTileBytes + kRouterBTile;
constexpr int kRouterSmem = kRouterStages * kRouterStageBytes + 1024;

__global__ void __launch_bounds__(kThreads, 1)
    k_router_tc(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w, CallArgs a) {
    extern __shared__ unsigned char dyn_raw[];
    __shared__ __align__(8) uint64_t bar_full[kRouterStages], bar_empty[kRouterStages], bar_tfull, bar_drain;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(dyn_raw) + 1023) & ~uintptr_t(1023));
    const int E = a.E, H = a.H, T = a.T;
    const int n_kb = H / BK;
    const int t0 = blockIdx.x * BM;
    if (threadIdx.x == 0) {
        for (int st = 0; st < kRouterStages; ++st) {
            mbar_init(&bar_full[st], 1);
            mbar_init(&bar_empty[st], 1);
        }
        mbar_init(&bar_tfull, 1);
        mbar_init(&bar_drain, 1);
        s_abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(&s_tmem)), "r"(256)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;
    volatile int* abort_flag = &s_abort;
    auto fail = [&](int code) {
        *abort_flag = 1;
        atomicExch(a.dev_err, code);
    };
    if (warp == 0) {
        if (lane == 0) {
            // ---------------- producer: token tile and router rows of each K stage
            int stage = 0;
            uint32_t phase = 0;
            int issued_phase[kRouterStages];
#pragma unroll
            for (int st = 0; st < kRouterStages; ++st) issued_phase[st] = -1;
            bool ok = true;
            for (int kb = 0; kb < n_kb; ++kb) {
                if (!mbar_wait(&bar_empty[stage], phase ^ 1u, abort_flag, a.wait_ns)) {
                    fail(MOE_DEVERR_TIMEOUT_PRODUCER);
                    ok = false;
                    break;
                }
                unsigned char* st = smem + stage * kRouterStageBytes;
                mbar_expect_tx(&bar_full[stage], static_cast<uint32_t>(kTileBytes + E * BK * 2));
                tma_2d(st, &map_x, &bar_full[stage], kb * BK, t0);
                tma_2d(st + kTileBytes, &map_w, &bar_full[stage], kb * BK, 0);
                issued_phase[stage] = static_cast<int>(phase);
                if (++stage == kRouterStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok)
                for (int st = 0; st < kRouterStages; ++st)
                    if (issued_phase[st] >= 0) {
                        const uint64_t w0 = gtimer();
                        while (!mbar_test(&bar_full[st], static_cast<uint32_t>(issued_phase[st])) && gtimer() - w0 < a.wait_ns) {
                        }
                    }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer: D[128 tokens][E] += X_tile * W_tile^T
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            const uint32_t idesc = idesc_bf16(BM, E);
            for (int kb = 0; kb < n_kb; ++kb) {
                if (!mbar_wait(&bar_full[stage], phase, abort_flag, a.wait_ns)) {
                    fail(MOE_DEVERR_TIMEOUT_MMA);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = su32(smem + stage * kRouterStageBytes);
                const uint32_t sb = sa + kTileBytes;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    umma_bf16(tmem, sdesc(sa + 32 * kk), sdesc(sb + 32 * kk), idesc, (kb | kk) != 0);
                umma_commit(&bar_empty[stage]);
                if (++stage == kRouterStages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (ok) umma_commit(&bar_tfull);
            umma_commit(&bar_drain);
            const uint64_t w0 = gtimer();
            while (!mbar_test(&bar_drain, 0) && gtimer() - w0 < a.wait_ns) {
            }
        }
    } else {
        // ---------------- epilogue (warps 2-5): TMEM lane = token of the tile
        const int quarter = warp & 3;
        const int t = t0 + quarter * 32 + lane;
        if (mbar_wait(&bar_tfull, 0, abort_flag, a.wait_ns)) {
            tc_fence_after();
            const uint32_t tbase = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
            for (int c0 = 0; c0 < E; c0 += 32) {
                float v[32];
                tmem_ld32(tbase + c0, v);
                if (t < T) {
                    float4* dst = reinterpret_cast<float4*>(a.logits + static_cast<size_t>(t) * E + c0);
#pragma unroll
                    for (int j = 0; j < 8; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                }
            }
        } else {
            fail(MOE_DEVERR_TIMEOUT_EPILOGUE);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(256) : "memory");
    }
}

// Euclidean norm of every router row (BF16), rounded up: the fp32 sum of the
// exact squares of H terms is within H * 2^-24 of the true sum, and the factor
// 1 + 2^-10 covers that and the square root's rounding.
__global__ void __launch_bounds__(256) k_router_norms(const __nv_bfloat16* __restrict__ w, int E, int H, float* out) {
    const int e = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (e >= E) return;
    const uint4* row = reinterpret_cast<const uint4*>(w + static_cast<size_t>(e) * H);
    float ss = 0.0f;
    for (int c = lane; c < H / 8; c += 32) {
        const uint4 u = __ldg(row + c);
        const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float lo = __uint_as_float(q[j] << 16), hi = __uint_as_float(q[j] & 0xFFFF0000u);
            ss = __fmaf_rn(lo, lo, ss);
            ss = __fmaf_rn(hi, hi, ss);
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) out[e] = sqrtf(ss) * (1.0f + 1.0f / 1024.0f);
}

// per token row t: the power of two xsc[t] with max_h |x[t,h]| * xsc[t] in
// [2^14, 2^15) (1 for an all-zero row); one warp per token
template <int ACT>
__global__ void __launch_bounds__(256) k_xscale(CallArgs a) {
    const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (t >= a.T) return;
    unsigned int m = 0u;
    if constexpr (ACT == ACT_BF16) {
        const uint4* x = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(a.hidden) + static_cast<size_t>(t) * a.H);
        for (int i = lane; i < a.H / 8; i += 32) {
            const uint4 v = x[i];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) m = max(m, max((w[j] << 16) & 0x7FFFFFFFu, w[j] & 0x7FFF0000u));
        }
    } else {
        const float4* x = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.hidden) + static_cast<size_t>(t) * a.H);
        for (int i = lane; i < a.H / 4; i += 32) {
            const float4 v = x[i];
            m = max(m, max(max(__float_as_uint(v.x) & 0x7FFFFFFFu, __float_as_uint(v.y) & 0x7FFFFFFFu),
                           max(__float_as_uint(v.z) & 0x7FFFFFFFu, __float_as_uint(v.w) & 0x7FFFFFFFu)));
        }
    }
    m = __reduce_max_sync(0xffffffffu, m);
    if (lane == 0) {
        float sc, un;
        pow2_scale(m, sc, un);
        a.xsc[t] = sc;
    }
}

// X_perm[r] = hidden[row_tok[r]] in the weights' K order: bf16, or (F16) f16
// of the row times its token's power of two, whose inverse goes to xunr[r]
template <int ACT, bool F16>
__global__ void __launch_bounds__(256) k_gather_x(CallArgs a, int rows) {
    const int H = a.H;
    const size_t n8 = static_cast<size_t>(rows) * H / 8;
    for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < n8;
         idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int r = static_cast<int>(idx / (H / 8));
        const int p = 8 * static_cast<int>(idx % (H / 8));  // destination position
        const int j = p >> 7, w = p & 127, q = w >> 5, s = (w & 31) >> 2;
        const int tok = a.row_tok[r];
        const size_t src = static_cast<size_t>(tok) * H + 128 * j + 16 * s + 4 * q;
        float v[8];
        uint32_t o[4];
        if constexpr (ACT == ACT_BF16) {
            const uint16_t* x = reinterpret_cast<const uint16_t*>(a.hidden);
            const uint2 lo = *reinterpret_cast<const uint2*>(x + src);
            const uint2 hi = *reinterpret_cast<const uint2*>(x + src + 16);
            o[0] = lo.x; o[1] = lo.y; o[2] = hi.x; o[3] = hi.y;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[2 * i] = __uint_as_float(o[i] << 16);
                v[2 * i + 1] = __uint_as_float(o[i] & 0xFFFF0000u);
            }
        } else {
            const float* x = reinterpret_cast<const float*>(a.hidden);
            const float4 lo = *reinterpret_cast<const float4*>(x + src);
            const float4 hi = *reinterpret_cast<const float4*>(x + src + 16);
            v[0] = lo.x; v[1] = lo.y; v[2] = lo.z; v[3] = lo.w;
            v[4] = hi.x; v[5] = hi.y; v[6] = hi.z; v[7] = hi.w;
            if constexpr (!F16) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                    o[i] = *reinterpret_cast<uint32_t*>(&b);
                }
            }
        }
        if constexpr (F16) {
            const float sc = a.xsc[tok];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                __half2 hv = __floats2half2_rn(v[2 * i] * sc, v[2 * i + 1] * sc);
                o[i] = *reinterpret_cast<uint32_t*>(&hv);
            }
            if (p == 0) a.xunr[r] = 1.0f / sc;  // a power of two: exact
        }
        *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(a.xperm) + static_cast<size_t>(r) * H + p) =
            make_uint4(o[0], o[1], o[2], o[3]);
    }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

}  // namespace

// bf16 [rows][cols] row-major, box = box_rows x 64 columns, 128-byte swizzle
bool umma_map_2d(UmmaMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn || !base || rows == 0) return false;
    CUtensorMap* t = reinterpret_cast<CUtensorMap*>(m->bytes);
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    const cuuint32_t es[2] = {1, 1};
    return fn(t, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 [slots][rows][cols], slot stride in bytes; box = box_rows x 64 columns x 1 slot
bool umma_map_3d(UmmaMap* m, const void* base, uint64_t slots, uint64_t slot_bytes, uint64_t rows, uint64_t cols,
                 uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn || !base || slots == 0) return false;
    CUtensorMap* t = reinterpret_cast<CUtensorMap*>(m->bytes);
    const cuuint64_t dims[3] = {cols, rows, slots};
    const cuuint64_t strides[2] = {cols * 2, slot_bytes};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), box_rows, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(t, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// also loads the gather kernel (see experts_preload for why every kernel is loaded up front)
cudaError_t umma_set_attributes() {
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(k_router_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, kRouterSmem))) return e;
    {
        cudaFuncAttributes fa;
        if ((e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(&k_router_norms)))) return e;
    }
    cudaFuncAttributes fa;
    if ((e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(&k_gather_x<ACT_BF16, false>)))) return e;
    if ((e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(&k_gather_x<ACT_FP32, false>)))) return e;
    if ((e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(&k_gather_x<ACT_BF16, true>)))) return e;
    if ((e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(&k_gather_x<ACT_FP32, true>)))) return e;
    if ((e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(&k_xscale<ACT_BF16>)))) return e;
    if ((e = cudaFuncGetAttributes(&fa, reinterpret_cast<const void*>(&k_xscale<ACT_FP32>)))) return e;
#define MOE_UMMA_ATTR(MODE, FMT)                                                                         \
    if ((e = cudaFuncSetAttribute(k_umma_grouped<MODE, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                  Cfg<MODE, FMT != FMT_BF16>::kSmem)))                                   \
        return e;
    MOE_UMMA_ATTR(MODE_GU, FMT_BF16)
    MOE_UMMA_ATTR(MODE_DOWN, FMT_BF16)
    MOE_UMMA_ATTR(MODE_GU, FMT_NVFP4)
    MOE_UMMA_ATTR(MODE_DOWN, FMT_NVFP4)
    MOE_UMMA_ATTR(MODE_GU, FMT_MXFP4)
    MOE_UMMA_ATTR(MODE_DOWN, FMT_MXFP4)
    MOE_UMMA_ATTR(MODE_GU, FMT_FP8)
    MOE_UMMA_ATTR(MODE_DOWN, FMT_FP8)
#undef MOE_UMMA_ATTR
    return cudaSuccess;
}

static CUtensorMap as_map(const UmmaMap& m) {
    CUtensorMap t;
    std::memcpy(&t, m.bytes, sizeof(t));
    return t;
}

template <int FMT>
static void launch_gemms(const CallArgs& a, const UmmaMaps& maps, int num_sms, cudaStream_t s, cudaEvent_t ev_gu) {
    constexpr int threads = FMT == FMT_BF16 ? kThreads : kThreadsFp4;
    // FP4 / FP8 weights do not use the pool / shared tensor maps (their A tiles are built in shared memory)
    const CUtensorMap pg = as_map(FMT == FMT_BF16 ? maps.pool_gu : maps.x);
    const CUtensorMap sg = as_map(FMT == FMT_BF16 ? maps.shared_gu : maps.x);
    const CUtensorMap pd = as_map(FMT == FMT_BF16 ? maps.pool_d : maps.x);
    const CUtensorMap sd = as_map(FMT == FMT_BF16 ? maps.shared_d : maps.x);
    k_umma_grouped<MODE_GU, FMT><<<num_sms, threads, Cfg<MODE_GU, FMT != FMT_BF16>::kSmem, s>>>(pg, sg, as_map(maps.x), a);
    if (ev_gu) cudaEventRecord(ev_gu, s);
    k_umma_grouped<MODE_DOWN, FMT><<<num_sms, threads, Cfg<MODE_DOWN, FMT != FMT_BF16>::kSmem, s>>>(pd, sd, as_map(maps.h), a);
}

bool router_tc_eligible(const CallArgs& a) {
    return a.act == ACT_BF16 && a.T > kDecodeMaxT && a.E % 32 == 0 && a.E <= 256 && a.H % BK == 0;
}

// norms of the router rows, then the approximate logits of every token
cudaError_t launch_router_tc(const CallArgs& a, cudaStream_t s) {
    UmmaMap mx, mw;
    if (!umma_map_2d(&mx, a.hidden, static_cast<uint64_t>(a.T), static_cast<uint64_t>(a.H), BM) ||
        !umma_map_2d(&mw, a.router_w, static_cast<uint64_t>(a.E), static_cast<uint64_t>(a.H), static_cast<uint32_t>(a.E)))
        return cudaErrorInvalidValue;
    k_router_norms<<<(a.E + 7) / 8, 256, 0, s>>>(reinterpret_cast<const __nv_bfloat16*>(a.router_w), a.E, a.H, a.wnorm);
    k_router_tc<<<(a.T + BM - 1) / BM, kThreads, kRouterSmem, s>>>(as_map(mx), as_map(mw), a);
    return cudaGetLastError();
}

// gather, gate/up + SwiGLU, down; the combine is launched by the caller
cudaError_t launch_prefill_umma(const CallArgs& a, const UmmaMaps& maps, int num_sms, cudaStream_t s,
                                cudaEvent_t ev_gu, int* launches) {
    const int rows = a.T * (a.k + a.n_shared);
    const size_t n8 = static_cast<size_t>(rows) * a.H / 8;
    const int gb = static_cast<int>(std::min<size_t>((n8 + 255) / 256, static_cast<size_t>(num_sms) * 16));
    const bool f16 = a.fmt == FMT_NVFP4 || a.fmt == FMT_FP8;  // gate/up on f16 operands
    int n = 3;
    if (f16) {
        if (a.act == ACT_BF16) k_xscale<ACT_BF16><<<(a.T + 7) / 8, 256, 0, s>>>(a);
        else k_xscale<ACT_FP32><<<(a.T + 7) / 8, 256, 0, s>>>(a);
        ++n;
    }
    if (a.act == ACT_BF16) {
        if (f16) k_gather_x<ACT_BF16, true><<<gb, 256, 0, s>>>(a, rows);
        else k_gather_x<ACT_BF16, false><<<gb, 256, 0, s>>>(a, rows);
    } else {
        if (f16) k_gather_x<ACT_FP32, true><<<gb, 256, 0, s>>>(a, rows);
        else k_gather_x<ACT_FP32, false><<<gb, 256, 0, s>>>(a, rows);
    }
    switch (a.fmt) {
        case FMT_BF16: launch_gemms<FMT_BF16>(a, maps, num_sms, s, ev_gu); break;
        case FMT_NVFP4: launch_gemms<FMT_NVFP4>(a, maps, num_sms, s, ev_gu); break;
        case FMT_MXFP4: launch_gemms<FMT_MXFP4>(a, maps, num_sms, s, ev_gu); break;
        case FMT_FP8: launch_gemms<FMT_FP8>(a, maps, num_sms, s, ev_gu); break;
        default: return cudaErrorInvalidValue;
    }
    if (launches) *launches = n;
    return cudaGetLastError();
}

}  // namespace moe
