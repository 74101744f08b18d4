// Expert FFNs of the routed MoE layer: SwiGLU gate/up projection, down
// projection and the gate-weighted combine, over the active experts that the
// router and cache kernels listed (routed experts in ascending id, then the
// always-on shared experts).
//
// Hits of the cache "run on the GPU" (freetoken.wiki architecture page, decode
// paragraph); the expert weights come in the formats the FreeToken pages list
// (bhrtaym-blog post, section on supported models and quantisation formats:
// MXFP4, NVFP4, BF16).
//
// MMA kernels use mma.sync m16n8k16 in swap-AB form: the weight rows are the
// M = 16 operand, the tokens routed to the expert are the N = 8 columns. FP4
// codes are widened to f16 in registers (exact) and multiplied by their block
// scale after each 16-element MMA step, in fp32; activations are fed as f16
// (FP4 weights) or bf16 (BF16 weights). The per-tensor NVFP4 scale multiplies
// the finished dot product.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "mma_common.cuh"
#include "moe_internal.h"

namespace moe {

// per-step block scales of one row for one 128-element group
template <int FMT>
__device__ __forceinline__ void load_step_scales(const uint8_t* sc_row, int j, float mul, float (&s)[8]) {
    if constexpr (FMT == FMT_NVFP4) {
        const uint2 v = *reinterpret_cast<const uint2*>(sc_row + 8 * j);
        e4m3x8_to_f32(v, s);
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i] *= mul;
    } else if constexpr (FMT == FMT_MXFP4) {
        const uint32_t v = *reinterpret_cast<const uint32_t*>(sc_row + 4 * j);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const float f = e8m0_to_f32((v >> (8 * b)) & 0xFFu) * mul;
            s[2 * b] = f;
            s[2 * b + 1] = f;
        }
    }
}

// A operand words of one row for one group: FP4 -> 4 words (16 B); BF16 -> 16 words (64 B)
template <int FMT>
struct RowWords {
    static constexpr int N = FMT == FMT_BF16 ? 16 : 4;
    uint32_t w[N];
};

template <int FMT>
__device__ __forceinline__ void load_row(const uint8_t* row, int j, int q, RowWords<FMT>& r) {
    if constexpr (FMT == FMT_BF16) {
        const uint4* p = reinterpret_cast<const uint4*>(row + (static_cast<size_t>(j) * 128 + 32 * q) * 2);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint4 x = __ldg(p + v);
            r.w[4 * v] = x.x; r.w[4 * v + 1] = x.y; r.w[4 * v + 2] = x.z; r.w[4 * v + 3] = x.w;
        }
    } else {
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(row + static_cast<size_t>(j) * 64 + 16 * q));
        r.w[0] = x.x; r.w[1] = x.y; r.w[2] = x.z; r.w[3] = x.w;
    }
}

// A operand words of one row for all 8 MMA steps of a group: A[s][lo] holds
// elements +0,+1 and A[s][hi] elements +2,+3 of the row's share of step s
template <int FMT>
__device__ __forceinline__ void row_to_a(const RowWords<FMT>& r, uint32_t (&A)[8][4], int lo, int hi) {
    if constexpr (FMT == FMT_BF16) {
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            A[s][lo] = r.w[2 * s];
            A[s][hi] = r.w[2 * s + 1];
        }
    } else {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            uint32_t o[4];
            fp4x8_to_f16x2(r.w[w], o);
            A[2 * w][lo] = o[0];
            A[2 * w][hi] = o[1];
            A[2 * w + 1][lo] = o[2];
            A[2 * w + 1][hi] = o[3];
        }
    }
}

// FP4 tiled blobs: the 16 code bytes of lane quad q and the step scales of row
// r (0-15) of a tile, for K-group j of G
template <int FMT>
__device__ __forceinline__ void load_tile_row(const uint8_t* tile, int G, int sbpg, int r, int j, int q, float mul,
                                              RowWords<FMT>& x, float (&s)[8]) {
    const int c = j / kChunkGroups, w = j % kChunkGroups;
    const int ng = fp4_chunk_groups(G, c);
    const uint8_t* chunk = tile + fp4_chunk_off(c, sbpg);
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(chunk + fp4_code_off(ng, r, w, q)));
    x.w[0] = v.x; x.w[1] = v.y; x.w[2] = v.z; x.w[3] = v.w;
    // the group's scale bytes sit where a row-major scale row would hold group 0
    load_step_scales<FMT>(chunk + fp4_scale_off(ng, sbpg, r, w), 0, mul, s);
}

// both rows (M rows 0-7 and 8-15) of one lane for group j: BF16 from row
// pointers ra/rb, FP4 from rows ta/tb of `tile`
template <int FMT>
__device__ __forceinline__ void load_pair(const uint8_t* ra, const uint8_t* rb, const uint8_t* tile, int ta, int tb,
                                          int G, int sbpg, int j, int q, float mul, RowWords<FMT>& x, RowWords<FMT>& y,
                                          float (&sa)[8], float (&sb)[8]) {
    if constexpr (FMT == FMT_BF16) {
        load_row<FMT>(ra, j, q, x);
        load_row<FMT>(rb, j, q, y);
    } else {
        load_tile_row<FMT>(tile, G, sbpg, ta, j, q, mul, x, sa);
        load_tile_row<FMT>(tile, G, sbpg, tb, j, q, mul, y, sb);
    }
}

// 64-byte B run (32 activations of one column for one group) -> 16 words; zeros if p is null
__device__ __forceinline__ void load_b(const uint16_t* p, uint32_t (&b)[16]) {
    if (p) {
        const uint4* v4 = reinterpret_cast<const uint4*>(p);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint4 x = v4[v];
            b[4 * v] = x.x; b[4 * v + 1] = x.y; b[4 * v + 2] = x.z; b[4 * v + 3] = x.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) b[i] = 0u;
    }
}

// one group (8 MMA steps) of a 16-row x (8 * NC)-column tile; rows ra (M rows
// 0-7) and rb (M rows 8-15); bptr[c] = this lane's B run of column tile c
template <int FMT, int NC>
__device__ __forceinline__ void mma_group(const RowWords<FMT>& ra, const RowWords<FMT>& rb, const float (&sa)[8],
                                          const float (&sb)[8], const uint16_t* const (&bptr)[NC], int ncols,
                                          float (&acc)[NC][4]) {
    uint32_t A[8][4];
    row_to_a<FMT>(ra, A, 0, 2);
    row_to_a<FMT>(rb, A, 1, 3);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        if (c < ncols) {
            uint32_t bw[16];
            load_b(bptr[c], bw);
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                if constexpr (FMT == FMT_BF16) {
                    mma_bf16(acc[c], A[s], bw[2 * s], bw[2 * s + 1], acc[c]);
                } else {
                    float d[4];
                    const float z[4] = {0.f, 0.f, 0.f, 0.f};
                    mma_f16(d, A[s], bw[2 * s], bw[2 * s + 1], z);
                    acc[c][0] = __fmaf_rn(sa[s], d[0], acc[c][0]);
                    acc[c][1] = __fmaf_rn(sa[s], d[1], acc[c][1]);
                    acc[c][2] = __fmaf_rn(sb[s], d[2], acc[c][2]);
                    acc[c][3] = __fmaf_rn(sb[s], d[3], acc[c][3]);
                }
            }
        }
    }
}

// --------------------------------------------------------------------------
// gate/up + SwiGLU: h[r, i] = gate_r * act(W_gate x_t)_i * (W_up x_t)_i
// grid (I/8 unit tiles, max active experts), 4 warps split K = H by group
// --------------------------------------------------------------------------

// thread 0 of every CTA waits for the call's weights; false if the wait gave up
__device__ __forceinline__ bool cta_wait_ready(const CallArgs& a) {
    __shared__ int s_ok;
    if (threadIdx.x == 0) s_ok = wait_ready(a) ? 1 : 0;
    __syncthreads();
    return s_ok != 0;
}

template <int FMT, int NC>
__global__ void __launch_bounds__(128) k_gu(CallArgs a) {
    if (!cta_wait_ready(a)) return;
    const int u = blockIdx.y;
    if (u >= *a.n_active) return;
    __shared__ float red[4][NC][32][4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const int H = a.H, I = a.I, G = H / kGroupK;
    const uint8_t* blob = a.act_ptr[u];
    const int row0 = a.act_row0[u], cnt = a.act_cnt[u];
    const int i0 = blockIdx.x * 8;
    const int rg = (i0 / 64) * 128 + (i0 % 64) + g;  // device gu row of gate unit i0+g
    const int ru = rg + 64;                           // and of its up unit
    const size_t rowbytes = static_cast<size_t>(H) * 2;
    const uint8_t* row_g = blob + a.lay.gu + rg * rowbytes;  // BF16
    const uint8_t* row_u = blob + a.lay.gu + ru * rowbytes;
    const uint8_t* tile = blob + a.lay.gu + static_cast<size_t>(blockIdx.x) * a.lay.gu_tile;  // FP4
    float gs_gate = 1.0f, gs_up = 1.0f;
    if constexpr (FMT == FMT_NVFP4) {
        const float* gsc = reinterpret_cast<const float*>(blob + a.lay.gsc);
        gs_gate = gsc[0];
        gs_up = gsc[1];
    }
    const uint16_t* xh = reinterpret_cast<const uint16_t*>(a.xh);
    for (int cb = 0; cb < cnt; cb += 8 * NC) {
        const int ncols = min(NC, (cnt - cb + 7) / 8);
        float acc[NC][4];
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.0f;
        int tok[NC];
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const int n = cb + 8 * c + g;
            tok[c] = n < cnt ? a.row_tok[row0 + n] : -1;
        }
        for (int j = warp; j < G; j += 4) {
            RowWords<FMT> ra, rb;
            float sa[8], sb[8];
            load_pair<FMT>(row_g, row_u, tile, g, 8 + g, G, a.lay.sbpg, j, q, 1.0f, ra, rb, sa, sb);
            const uint16_t* bp[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c)
                bp[c] = tok[c] >= 0 ? xh + static_cast<size_t>(tok[c]) * H + j * 128 + 32 * q : nullptr;
            mma_group<FMT, NC>(ra, rb, sa, sb, bp, ncols, acc);
        }
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int i = 0; i < 4; ++i) red[warp][c][lane][i] = acc[c][i];
        __syncthreads();
        // epilogue: warp w finishes column tiles c = w, w+4, ...
        for (int c = warp; c < ncols; c += 4) {
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                v[i] = ((red[0][c][lane][i] + red[1][c][lane][i]) + red[2][c][lane][i]) + red[3][c][lane][i];
            const int unit = i0 + g;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int n = cb + 8 * c + 2 * q + h;
                if (n < cnt) {
                    const int r = row0 + n;
                    const float gate = v[h] * gs_gate, up = v[2 + h] * gs_up;
                    const float act = a.mode == 1 ? gate : silu(gate);
                    const float hv = act * up * a.row_gate[r];
                    const size_t o = static_cast<size_t>(r) * I + dpos(unit);
                    if constexpr (FMT == FMT_BF16) reinterpret_cast<__nv_bfloat16*>(a.hbuf)[o] = __float2bfloat16_rn(hv);
                    else reinterpret_cast<__half*>(a.hbuf)[o] = __float2half_rn(hv);
                }
            }
        }
        __syncthreads();
    }
}

// --------------------------------------------------------------------------
// decode down projection + combine: out[t, r] = sum over active experts u of
// (W_down,u h_{u,t})[r]; the gate is already folded into h. The token index is
// the MMA column, so all experts accumulate into one tile.
// grid (H/16 row tiles), 4 warps split K = I by group
// --------------------------------------------------------------------------

template <int FMT, int ACT>
__global__ void __launch_bounds__(128) k_down_dec(CallArgs a) {
    __shared__ float red[4][32][4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const int H = a.H, I = a.I, T = a.T, GI = I / kGroupK;
    const int r0 = blockIdx.x * 16 + g;
    const int na = *a.n_active;
    const size_t rowbytes = static_cast<size_t>(I) * 2;
        const uint16_t* hb = reinterpret_cast<const uint16_t*>(a.hbuf);
    float acc[1][4] = {{0.f, 0.f, 0.f, 0.f}};
    for (int u = 0; u < na; ++u) {
        const uint8_t* blob = a.act_ptr[u];
        const int hr = g < T ? a.tok_row[u * kDecodeMaxT + g] : -1;
        float gsd = 1.0f;
        if constexpr (FMT == FMT_NVFP4) gsd = reinterpret_cast<const float*>(blob + a.lay.gsc)[2];
        const uint8_t* rowa = blob + a.lay.d + r0 * rowbytes;  // BF16
        const uint8_t* rowb = blob + a.lay.d + (r0 + 8) * rowbytes;
        const uint8_t* tile = blob + a.lay.d + static_cast<size_t>(blockIdx.x) * a.lay.d_tile;  // FP4
        for (int j = warp; j < GI; j += 4) {
            RowWords<FMT> ra, rb;
            float sa[8], sb[8];
            load_pair<FMT>(rowa, rowb, tile, g, 8 + g, GI, a.lay.sbpg, j, q, gsd, ra, rb, sa, sb);
            const uint16_t* bp[1] = {hr >= 0 ? hb + static_cast<size_t>(hr) * I + j * 128 + 32 * q : nullptr};
            mma_group<FMT, 1>(ra, rb, sa, sb, bp, 1, acc);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) red[warp][lane][i] = acc[0][i];
    __syncthreads();
    if (warp == 0) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = ((red[0][lane][i] + red[1][lane][i]) + red[2][lane][i]) + red[3][lane][i];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int t = 2 * q + h;
            if (t < T) {
#pragma unroll
                for (int rr = 0; rr < 2; ++rr) {
                    const size_t o = static_cast<size_t>(t) * H + r0 + 8 * rr;
                    const float x = v[2 * rr + h];
                    if constexpr (ACT == ACT_BF16) reinterpret_cast<__nv_bfloat16*>(a.out)[o] = __float2bfloat16_rn(x);
                    else reinterpret_cast<float*>(a.out)[o] = x;
                }
            }
        }
    }
}

// --------------------------------------------------------------------------
// prefill down projection: Y[r, :] = W_down,u h_r for every row r of expert u
// grid (H/16 row tiles, max active experts)
// --------------------------------------------------------------------------

template <int FMT, int NC>
__global__ void __launch_bounds__(128) k_down_rows(CallArgs a) {
    const int u = blockIdx.y;
    if (u >= *a.n_active) return;
    __shared__ float red[4][NC][32][4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const int H = a.H, I = a.I, GI = I / kGroupK;
    const uint8_t* blob = a.act_ptr[u];
    const int row0 = a.act_row0[u], cnt = a.act_cnt[u];
    const int r0 = blockIdx.x * 16 + g;
    const size_t rowbytes = static_cast<size_t>(I) * 2;
        float gsd = 1.0f;
    if constexpr (FMT == FMT_NVFP4) gsd = reinterpret_cast<const float*>(blob + a.lay.gsc)[2];
    const uint8_t* rowa = blob + a.lay.d + r0 * rowbytes;  // BF16
    const uint8_t* rowb = blob + a.lay.d + (r0 + 8) * rowbytes;
    const uint8_t* tile = blob + a.lay.d + static_cast<size_t>(blockIdx.x) * a.lay.d_tile;  // FP4
    const uint16_t* hb = reinterpret_cast<const uint16_t*>(a.hbuf);
    __nv_bfloat16* Y = reinterpret_cast<__nv_bfloat16*>(a.ybuf);
    for (int cb = 0; cb < cnt; cb += 8 * NC) {
        const int ncols = min(NC, (cnt - cb + 7) / 8);
        float acc[NC][4];
#pragma unroll
        for (int c = 0; c < NC; ++c) acc[c][0] = acc[c][1] = acc[c][2] = acc[c][3] = 0.0f;
        for (int j = warp; j < GI; j += 4) {
            RowWords<FMT> ra, rb;
            float sa[8], sb[8];
            load_pair<FMT>(rowa, rowb, tile, g, 8 + g, GI, a.lay.sbpg, j, q, gsd, ra, rb, sa, sb);
            const uint16_t* bp[NC];
#pragma unroll
            for (int c = 0; c < NC; ++c) {
                const int n = cb + 8 * c + g;
                bp[c] = n < cnt ? hb + static_cast<size_t>(row0 + n) * I + j * 128 + 32 * q : nullptr;
            }
            mma_group<FMT, NC>(ra, rb, sa, sb, bp, ncols, acc);
        }
#pragma unroll
        for (int c = 0; c < NC; ++c)
#pragma unroll
            for (int i = 0; i < 4; ++i) red[warp][c][lane][i] = acc[c][i];
        __syncthreads();
        for (int c = warp; c < ncols; c += 4) {
            float v[4];
#pragma unroll
            for (int i = 0; i < 4; ++i)
                v[i] = ((red[0][c][lane][i] + red[1][c][lane][i]) + red[2][c][lane][i]) + red[3][c][lane][i];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int n = cb + 8 * c + 2 * q + h;
                if (n < cnt) {
                    const size_t o = static_cast<size_t>(row0 + n) * H;
                    Y[o + r0] = __float2bfloat16_rn(v[h]);
                    Y[o + r0 + 8] = __float2bfloat16_rn(v[2 + h]);
                }
            }
        }
        __syncthreads();
    }
}

// out[t, :] = sum_j Y[inv_perm[t*k + j], :] (j ascending) + sum_s Y[shared row of t]
template <int ACT>
__global__ void __launch_bounds__(256) k_combine(CallArgs a) {
    const int H = a.H, T = a.T, k = a.k;
    const size_t n8 = static_cast<size_t>(T) * H / 8;
    const __nv_bfloat16* Y = reinterpret_cast<const __nv_bfloat16*>(a.ybuf);
    for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < n8;
         idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const int t = static_cast<int>(idx / (H / 8));
        const int c = 8 * static_cast<int>(idx % (H / 8));
        float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const int nrows = k + a.n_shared;
        for (int j = 0; j < nrows; ++j) {
            const int r = j < k ? a.inv_perm[t * k + j] : T * k + (j - k) * T + t;
            const uint4 v = *reinterpret_cast<const uint4*>(Y + static_cast<size_t>(r) * H + c);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                s[2 * i] += __uint_as_float(w[i] << 16);
                s[2 * i + 1] += __uint_as_float(w[i] & 0xFFFF0000u);
            }
        }
        if constexpr (ACT == ACT_BF16) {
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                __nv_bfloat162 b = __floats2bfloat162_rn(s[2 * i], s[2 * i + 1]);
                o[i] = *reinterpret_cast<uint32_t*>(&b);
            }
            *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.out) + static_cast<size_t>(t) * H + c) =
                make_uint4(o[0], o[1], o[2], o[3]);
        } else {
            float* o = reinterpret_cast<float*>(a.out) + static_cast<size_t>(t) * H + c;
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = s[i];
        }
    }
}

// --------------------------------------------------------------------------
// FP32 weights: plain SIMT kernels (small shapes)
// --------------------------------------------------------------------------

template <int ACT>
__device__ __forceinline__ float ldx(const void* p, size_t i) {
    if constexpr (ACT == ACT_BF16)
        return __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(p)[i]) << 16);
    else
        return reinterpret_cast<const float*>(p)[i];
}

template <int ACT>
__global__ void __launch_bounds__(256) k_gu_f32(CallArgs a) {
    if (!cta_wait_ready(a)) return;
    const int u = blockIdx.y;
    if (u >= *a.n_active) return;
    const int H = a.H, I = a.I;
    const float* Wg = reinterpret_cast<const float*>(a.act_ptr[u] + a.lay.gu);
    const float* Wu = Wg + static_cast<size_t>(I) * H;
    const int row0 = a.act_row0[u], cnt = a.act_cnt[u];
    float* hb = reinterpret_cast<float*>(a.hbuf);
    for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < cnt * I; idx += gridDim.x * blockDim.x) {
        const int n = idx / I, i = idx % I, r = row0 + n, t = a.row_tok[r];
        float gs = 0.f, us = 0.f;
        for (int h = 0; h < H; ++h) {
            const float x = ldx<ACT>(a.hidden, static_cast<size_t>(t) * H + h);
            gs = __fadd_rn(gs, __fmul_rn(Wg[static_cast<size_t>(i) * H + h], x));
            us = __fadd_rn(us, __fmul_rn(Wu[static_cast<size_t>(i) * H + h], x));
        }
        const float act = a.mode == 1 ? gs : gs / (1.0f + expf(-gs));
        hb[static_cast<size_t>(r) * I + i] = act * us * a.row_gate[r];
    }
}

template <int ACT>
__global__ void __launch_bounds__(256) k_down_f32(CallArgs a) {
    const int H = a.H, I = a.I, T = a.T, k = a.k;
    const float* hb = reinterpret_cast<const float*>(a.hbuf);
    const int nu = *a.n_uniq;
    for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < T * H; idx += gridDim.x * blockDim.x) {
        const int t = idx / H, c = idx % H;
        float acc = 0.f;
        for (int j = 0; j < k + a.n_shared; ++j) {
            int r, u;
            if (j < k) {
                r = a.inv_perm[t * k + j];
                u = a.e2u[a.topk[t * k + j]];
            } else {
                r = T * k + (j - k) * T + t;
                u = nu + (j - k);
            }
            const float* Wd = reinterpret_cast<const float*>(a.act_ptr[u] + a.lay.d);
            float y = 0.f;
            for (int i = 0; i < I; ++i)
                y = __fadd_rn(y, __fmul_rn(Wd[static_cast<size_t>(c) * I + i], hb[static_cast<size_t>(r) * I + i]));
            acc = __fadd_rn(acc, y);
        }
        if constexpr (ACT == ACT_BF16) reinterpret_cast<__nv_bfloat16*>(a.out)[idx] = __float2bfloat16_rn(acc);
        else reinterpret_cast<float*>(a.out)[idx] = acc;
    }
}

// --------------------------------------------------------------------------

template <int FMT, int ACT>
static int launch_mma_path(const CallArgs& a, cudaStream_t s, cudaEvent_t ev_gu, cudaEvent_t ev_down, int num_sms) {
    const int max_active = min(a.E, a.T * a.k) + a.n_shared;
    if (a.T <= kDecodeMaxT && decode_fp4_supported(FMT, a.T)) {
        if (launch_decode_fp4(a, num_sms, s) != cudaSuccess) return -1;
        if (ev_gu) cudaEventRecord(ev_gu, s);
        if (ev_down) cudaEventRecord(ev_down, s);
        return 1;
    }
    if (a.T <= kDecodeMaxT) {
        k_gu<FMT, 1><<<dim3(a.I / 8, max_active), 128, 0, s>>>(a);
        if (ev_gu) cudaEventRecord(ev_gu, s);
        k_down_dec<FMT, ACT><<<a.H / 16, 128, 0, s>>>(a);
        if (ev_down) cudaEventRecord(ev_down, s);
        return 2;
    }
    k_gu<FMT, 8><<<dim3(a.I / 8, max_active), 128, 0, s>>>(a);
    if (ev_gu) cudaEventRecord(ev_gu, s);
    k_down_rows<FMT, 8><<<dim3(a.H / 16, max_active), 128, 0, s>>>(a);
    if (ev_down) cudaEventRecord(ev_down, s);
    const size_t n8 = static_cast<size_t>(a.T) * a.H / 8;
    const int blocks = static_cast<int>(std::min<size_t>((n8 + 255) / 256, 148 * 16));
    k_combine<ACT><<<blocks, 256, 0, s>>>(a);
    return 3;
}

cudaError_t launch_experts(const CallArgs& a, cudaStream_t s, cudaEvent_t ev_gu, cudaEvent_t ev_down,
                           const UmmaMaps* maps, int num_sms, int* launches) {
    int n = 0;
    if (prefill_uses_umma(a.fmt, a.T)) {
        if (!maps || !maps->have_pool || !maps->have_io) return cudaErrorInvalidValue;
        cudaError_t e = launch_prefill_umma(a, *maps, num_sms, s, ev_gu, &n);
        if (e != cudaSuccess) return e;
        if (ev_down) cudaEventRecord(ev_down, s);
        const size_t n8 = static_cast<size_t>(a.T) * a.H / 8;
        const int blocks = static_cast<int>(std::min<size_t>((n8 + 255) / 256, static_cast<size_t>(num_sms) * 16));
        if (a.act == ACT_BF16) k_combine<ACT_BF16><<<blocks, 256, 0, s>>>(a);
        else k_combine<ACT_FP32><<<blocks, 256, 0, s>>>(a);
        if (launches) *launches = n + 1;
        return cudaGetLastError();
    }
    if (a.fmt == FMT_FP32) {
        const int max_active = min(a.E, a.T * a.k) + a.n_shared;
        const int gx = min((a.T * a.I + 255) / 256, 64);
        const int gd = min((a.T * a.H + 255) / 256, 148 * 8);
        if (a.act == ACT_BF16) k_gu_f32<ACT_BF16><<<dim3(gx, max_active), 256, 0, s>>>(a);
        else k_gu_f32<ACT_FP32><<<dim3(gx, max_active), 256, 0, s>>>(a);
        if (ev_gu) cudaEventRecord(ev_gu, s);
        if (a.act == ACT_BF16) k_down_f32<ACT_BF16><<<gd, 256, 0, s>>>(a);
        else k_down_f32<ACT_FP32><<<gd, 256, 0, s>>>(a);
        if (ev_down) cudaEventRecord(ev_down, s);
        n = 2;
    } else {
        const bool bf = a.act == ACT_BF16;
        switch (a.fmt) {
            case FMT_BF16:
                n = bf ? launch_mma_path<FMT_BF16, ACT_BF16>(a, s, ev_gu, ev_down, num_sms)
                       : launch_mma_path<FMT_BF16, ACT_FP32>(a, s, ev_gu, ev_down, num_sms);
                break;
            case FMT_NVFP4:
                n = bf ? launch_mma_path<FMT_NVFP4, ACT_BF16>(a, s, ev_gu, ev_down, num_sms)
                       : launch_mma_path<FMT_NVFP4, ACT_FP32>(a, s, ev_gu, ev_down, num_sms);
                break;
            case FMT_MXFP4:
                n = bf ? launch_mma_path<FMT_MXFP4, ACT_BF16>(a, s, ev_gu, ev_down, num_sms)
                       : launch_mma_path<FMT_MXFP4, ACT_FP32>(a, s, ev_gu, ev_down, num_sms);
                break;
            default:
                return cudaErrorInvalidValue;
        }
        if (n < 0) return cudaErrorLaunchFailure;
    }
    if (launches) *launches = n;
    return cudaGetLastError();
}

// Loads every expert kernel of this file now. The expert kernels of a call
// wait on the device for the call's copies, which the service thread issues;
// with lazy module loading, the first launch of a kernel behind a waiting one
// would load its module while the wait runs and hold up those copies until the
// wait gives up. Querying a kernel's attributes loads it.
cudaError_t experts_preload() {
    cudaFuncAttributes fa;
    const void* fns[] = {
        reinterpret_cast<const void*>(&k_gu<FMT_BF16, 1>), reinterpret_cast<const void*>(&k_gu<FMT_BF16, 8>),
        reinterpret_cast<const void*>(&k_gu<FMT_NVFP4, 1>), reinterpret_cast<const void*>(&k_gu<FMT_NVFP4, 8>),
        reinterpret_cast<const void*>(&k_gu<FMT_MXFP4, 1>), reinterpret_cast<const void*>(&k_gu<FMT_MXFP4, 8>),
        reinterpret_cast<const void*>(&k_down_dec<FMT_BF16, ACT_BF16>),
        reinterpret_cast<const void*>(&k_down_dec<FMT_BF16, ACT_FP32>),
        reinterpret_cast<const void*>(&k_down_dec<FMT_NVFP4, ACT_BF16>),
        reinterpret_cast<const void*>(&k_down_dec<FMT_NVFP4, ACT_FP32>),
        reinterpret_cast<const void*>(&k_down_dec<FMT_MXFP4, ACT_BF16>),
        reinterpret_cast<const void*>(&k_down_dec<FMT_MXFP4, ACT_FP32>),
        reinterpret_cast<const void*>(&k_down_rows<FMT_BF16, 8>), reinterpret_cast<const void*>(&k_down_rows<FMT_NVFP4, 8>),
        reinterpret_cast<const void*>(&k_down_rows<FMT_MXFP4, 8>),
        reinterpret_cast<const void*>(&k_combine<ACT_BF16>), reinterpret_cast<const void*>(&k_combine<ACT_FP32>),
        reinterpret_cast<const void*>(&k_gu_f32<ACT_BF16>), reinterpret_cast<const void*>(&k_gu_f32<ACT_FP32>),
        reinterpret_cast<const void*>(&k_down_f32<ACT_BF16>), reinterpret_cast<const void*>(&k_down_f32<ACT_FP32>),
    };
    for (const void* f : fns) {
        const cudaError_t e = cudaFuncGetAttributes(&fa, f);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace moe
