// Expert FFNs of the routed MoE layer: SwiGLU gate/up projection, down
// projection and the gate-weighted combine, over the active experts that the
// router and cache kernels listed (routed experts in ascending id, then the
// always-on shared experts).
//
// Hits of the cache "run on the GPU" (freetoken.wiki architecture page, decode
// paragraph); the expert weights come in the formats the FreeToken pages list
// (bhrtaym-blog post, section on supported models and quantisation formats:
// MXFP4, NVFP4, FP8, BF16).
//
// Here: decode with BF16 weights (mma.sync m16n8k16 in swap-AB form: the weight
// rows are the M = 16 operand, the tokens routed to the expert the N = 8
// columns; bf16 operands, fp32 accumulation), the prefill combine, and plain
// SIMT kernels for FP32 weights. Decode with FP4 or FP8 weights runs in the fused
// decode kernel, prefill in the tensor-core grouped GEMMs.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "mma_common.cuh"
#include "moe_internal.h"

namespace moe {

// A operand words of one BF16 weight row for one 128-element group (64 bytes)
struct RowWords {
    uint32_t w[16];
};

__device__ __forceinline__ void load_row(const uint8_t* row, int j, int q, RowWords& r) {
    const uint4* p = reinterpret_cast<const uint4*>(row + (static_cast<size_t>(j) * 128 + 32 * q) * 2);
#pragma unroll
    for (int v = 0; v < 4; ++v) {
        const uint4 x = __ldg(p + v);
        r.w[4 * v] = x.x; r.w[4 * v + 1] = x.y; r.w[4 * v + 2] = x.z; r.w[4 * v + 3] = x.w;
    }
}

// A operand words of one row for all 8 MMA steps of a group: A[s][lo] holds
// elements +0,+1 and A[s][hi] elements +2,+3 of the row's share of step s
__device__ __forceinline__ void row_to_a(const RowWords& r, uint32_t (&A)[8][4], int lo, int hi) {
#pragma unroll
    for (int s = 0; s < 8; ++s) {
        A[s][lo] = r.w[2 * s];
        A[s][hi] = r.w[2 * s + 1];
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
template <int NC>
__device__ __forceinline__ void mma_group(const RowWords& ra, const RowWords& rb, const uint16_t* const (&bptr)[NC],
                                          int ncols, float (&acc)[NC][4]) {
    uint32_t A[8][4];
    row_to_a(ra, A, 0, 2);
    row_to_a(rb, A, 1, 3);
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        if (c < ncols) {
            uint32_t bw[16];
            load_b(bptr[c], bw);
#pragma unroll
            for (int s = 0; s < 8; ++s) mma_bf16(acc[c], A[s], bw[2 * s], bw[2 * s + 1], acc[c]);
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

__global__ void __launch_bounds__(128) k_gu(CallArgs a) {
    if (!cta_wait_ready(a)) return;
    const int u = blockIdx.y;
    if (u >= *a.n_active) return;
    __shared__ float red[4][32][4];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
    const int H = a.H, I = a.I, G = H / kGroupK;
    const uint8_t* blob = a.act_ptr[u];
    const int row0 = a.act_row0[u], cnt = a.act_cnt[u];
    const int i0 = blockIdx.x * 8;
    const int rg = (i0 / 64) * 128 + (i0 % 64) + g;  // device gu row of gate unit i0+g
    const int ru = rg + 64;                           // and of its up unit
    const size_t rowbytes = static_cast<size_t>(H) * 2;
    const uint8_t* row_g = blob + a.lay.gu + rg * rowbytes;
    const uint8_t* row_u = blob + a.lay.gu + ru * rowbytes;
    const uint16_t* xh = reinterpret_cast<const uint16_t*>(a.xh);
    float acc[1][4] = {{0.f, 0.f, 0.f, 0.f}};
    const int tok = g < cnt ? a.row_tok[row0 + g] : -1;
    for (int j = warp; j < G; j += 4) {
        RowWords ra, rb;
        load_row(row_g, j, q, ra);
        load_row(row_u, j, q, rb);
        const uint16_t* bp[1] = {tok >= 0 ? xh + static_cast<size_t>(tok) * H + j * 128 + 32 * q : nullptr};
        mma_group<1>(ra, rb, bp, 1, acc);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) red[warp][lane][i] = acc[0][i];
    __syncthreads();
    if (warp == 0) {
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = ((red[0][lane][i] + red[1][lane][i]) + red[2][lane][i]) + red[3][lane][i];
        const int unit = i0 + g;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = 2 * q + h;
            if (n < cnt) {
                const int r = row0 + n;
                const float gate = v[h], up = v[2 + h];
                const float act = a.mode == 1 ? gate : silu(gate);
                reinterpret_cast<__nv_bfloat16*>(a.hbuf)[static_cast<size_t>(r) * I + dpos(unit)] =
                    __float2bfloat16_rn(act * up * a.row_gate[r]);
            }
        }
    }
}

// --------------------------------------------------------------------------
// decode down projection + combine: out[t, r] = sum over active experts u of
// (W_down,u h_{u,t})[r]; the gate is already folded into h. The token index is
// the MMA column, so all experts accumulate into one tile.
// grid (H/16 row tiles), 4 warps split K = I by group
// --------------------------------------------------------------------------

template <int ACT>
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
        const uint8_t* rowa = blob + a.lay.d + r0 * rowbytes;
        const uint8_t* rowb = blob + a.lay.d + (r0 + 8) * rowbytes;
        for (int j = warp; j < GI; j += 4) {
            RowWords ra, rb;
            load_row(rowa, j, q, ra);
            load_row(rowb, j, q, rb);
            const uint16_t* bp[1] = {hr >= 0 ? hb + static_cast<size_t>(hr) * I + j * 128 + 32 * q : nullptr};
            mma_group<1>(ra, rb, bp, 1, acc);
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

// decode with BF16 weights: gate/up + SwiGLU, then down + combine
template <int ACT>
static int launch_bf16_decode(const CallArgs& a, cudaStream_t s, cudaEvent_t ev_gu, cudaEvent_t ev_down) {
    const int max_active = min(a.E, a.T * a.k) + a.n_shared;
    k_gu<<<dim3(a.I / 8, max_active), 128, 0, s>>>(a);
    if (ev_gu) cudaEventRecord(ev_gu, s);
    k_down_dec<ACT><<<a.H / 16, 128, 0, s>>>(a);
    if (ev_down) cudaEventRecord(ev_down, s);
    return 2;
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
    } else if (a.fmt == FMT_BF16 && a.T <= kDecodeMaxT) {
        n = a.act == ACT_BF16 ? launch_bf16_decode<ACT_BF16>(a, s, ev_gu, ev_down)
                              : launch_bf16_decode<ACT_FP32>(a, s, ev_gu, ev_down);
    } else {
        return cudaErrorInvalidValue;  // FP4 / FP8 decode runs in the fused decode kernel
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
        reinterpret_cast<const void*>(&k_gu),
        reinterpret_cast<const void*>(&k_down_dec<ACT_BF16>), reinterpret_cast<const void*>(&k_down_dec<ACT_FP32>),
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
