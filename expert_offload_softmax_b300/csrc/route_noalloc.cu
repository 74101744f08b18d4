// Router top-k entry point that allocates nothing.
//
// moe_layer_forward needs a handle, and moe_init allocates that handle's device
// scratch with cudaMalloc. Some callers cannot do that: a plugin inside a host
// framework whose memory pool owns all device memory (a raw cudaMalloc there
// bypasses the framework's accounting and implicitly synchronises the device),
// or a latency-critical path that must not allocate at all. For them,
// moe_route_topk_noalloc computes the router part of the layer (logits in the
// fixed summation order, softmax, top-k with lowest-index ties, renormalised
// gates) into caller-provided outputs, with its logits scratch in a fixed-size
// file-scope device array instead of allocated memory.
//
// The array is a property of the loaded library: every GPU that uses it holds
// ROUTE_NOALLOC_MAX_LOGITS floats (4 MiB) until the process exits. All calls
// share it and it keeps the last call's contents; two calls whose work overlaps
// on the GPU (different streams, or different host threads) race on it.
// The first call on each device, with that device current, looks the array's
// device address up (cudaGetSymbolAddress) and raises the kernel's dynamic
// shared-memory limit; make that first call before any stream capture.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"
#include "moe_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxGridY = 65535;  // CUDA's limit on a grid's y extent

// logits scratch [T][E]
__device__ __align__(256) float g_route_scratch[MOE_ROUTE_NOALLOC_MAX_LOGITS];

std::mutex g_setup_mu;
float* g_scratch_ptr[kMaxDevices] = {};

template <int ACT>
__device__ __forceinline__ void na_ld8(const void* p, size_t i, float (&v)[8]) {
    if constexpr (ACT == moe::ACT_BF16) {
        const uint4 u = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p) + i);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[2 * j] = __uint_as_float(w[j] << 16);
            v[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    } else {
        const float4* f = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p) + i);
        const float4 a = f[0], b = f[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
}

// logits[t, e] in the fixed order: 8-element chunks, chunk c on lane c mod 32,
// fused multiply-adds in increasing h, then an xor butterfly over the lanes.
// One warp per expert, 8 tokens per block; the token rows sit in shared memory.
template <int ACT>
__global__ void __launch_bounds__(256) k_na_logits(const void* __restrict__ hidden, const void* __restrict__ w,
                                                   int T, int E, int H, float* __restrict__ logits) {
    extern __shared__ __align__(16) unsigned char na_x[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.y * 8, nt = min(8, T - t0);
    const size_t esz = ACT == moe::ACT_BF16 ? 2 : 4;
    const size_t bytes = static_cast<size_t>(nt) * H * esz;
    const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned char*>(hidden) +
                                                      static_cast<size_t>(t0) * H * esz);
    for (size_t i = threadIdx.x; i < bytes / 16; i += blockDim.x) reinterpret_cast<uint4*>(na_x)[i] = src[i];
    __syncthreads();
    const int e = blockIdx.x * 8 + warp;
    if (e >= E) return;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int c = lane; c < H / 8; c += 32) {
        float wv[8];
        na_ld8<ACT>(w, static_cast<size_t>(e) * H + 8 * c, wv);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            if (t < nt) {
                float xv[8];
                na_ld8<ACT>(na_x, static_cast<size_t>(t) * H + 8 * c, xv);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[t] = __fmaf_rn(xv[i], wv[i], acc[t]);
            }
        }
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        float v = acc[t];
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0 && t < nt) logits[static_cast<size_t>(t0 + t) * E + e] = v;
    }
}

// softmax over E, top-k on the logits (larger first, ties to the lower index,
// NaN as -inf), gates = selected probabilities / their sum; one warp per token
__global__ void __launch_bounds__(256) k_na_topk(const float* __restrict__ logits, int T, int E, int k,
                                                 int32_t* __restrict__ topk_idx, float* __restrict__ gates) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    constexpr int kPer = moe::kMaxExperts / 32;
    const int per = (E + 31) / 32;
    float v[kPer];
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        v[i] = -INFINITY;
        const int e = lane + 32 * i;
        if (i < per && e < E) {
            float x = logits[static_cast<size_t>(t) * E + e];
            if (x != x) x = -INFINITY;
            v[i] = x;
            mx = fmaxf(mx, x);
        }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float den = 0.f;
#pragma unroll
    for (int i = 0; i < kPer; ++i)
        if (i < per && lane + 32 * i < E && v[i] != -INFINITY) den += expf(v[i] - mx);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    uint32_t taken = 0;
    float psum = 0.f, pj = 0.f;
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
        const float p = bv == -INFINITY ? 0.f : expf(bv - mx) / den;
        psum += p;
        if (lane == j) { pj = p; ej = be; }  // lane j keeps selection j
    }
    if (lane < k) {
        topk_idx[static_cast<size_t>(t) * k + lane] = ej;
        gates[static_cast<size_t>(t) * k + lane] = pj / psum;
    }
}

// once per device: the scratch array's device address and the kernels' shared-memory limit
int setup_device(int dev, float** out) {
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_INVALID;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        const int big = 200 * 1024;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess ||
            cudaFuncSetAttribute(k_na_logits<moe::ACT_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, big) !=
                cudaSuccess ||
            cudaFuncSetAttribute(k_na_logits<moe::ACT_FP32>, cudaFuncAttributeMaxDynamicSharedMemorySize, big) !=
                cudaSuccess) {
            cudaGetLastError();  // this call's own failure
            return MOE_ERR_CUDA;
        }
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" int moe_route_topk_noalloc(const void* hidden, const void* router_w, int T, int E, int H, int k,
                                      int act_dtype, int32_t* topk_idx, float* gates, void* stream) {
    if (T < 0 || E < 1 || E > moe::kMaxExperts || k < 1 || k > moe::kMaxTopK || k > E) return MOE_ERR_INVALID;
    if (H < 8 || H % 8 != 0) return MOE_ERR_INVALID;
    if (act_dtype != MOE_ACT_FP32 && act_dtype != MOE_ACT_BF16) return MOE_ERR_INVALID;
    const size_t esz = act_dtype == MOE_ACT_BF16 ? 2 : 4;
    if (static_cast<size_t>(8) * H * esz > 200 * 1024) return MOE_ERR_INVALID;
    if (static_cast<size_t>(T) * E > static_cast<size_t>(MOE_ROUTE_NOALLOC_MAX_LOGITS)) return MOE_ERR_INVALID;
    if ((T + 7) / 8 > kMaxGridY) return MOE_ERR_INVALID;  // token blocks are the logits grid's y extent
    if (T == 0) return MOE_OK;
    if (!hidden || !router_w || !topk_idx || !gates) return MOE_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(router_w)) & 15u) return MOE_ERR_INVALID;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    float* scratch = nullptr;
    const int rc = setup_device(dev, &scratch);
    if (rc != MOE_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const dim3 grid((E + 7) / 8, (T + 7) / 8);
    size_t smem = static_cast<size_t>(8) * H * esz;
    // each launch's own status: an error another call left pending is neither
    // reported nor cleared here, and a failed launch of this call clears its own
    {
        void* args[] = {const_cast<void**>(&hidden), const_cast<void**>(&router_w), &T, &E, &H, &scratch};
        const void* fn = act_dtype == MOE_ACT_BF16 ? reinterpret_cast<const void*>(&k_na_logits<moe::ACT_BF16>)
                                                   : reinterpret_cast<const void*>(&k_na_logits<moe::ACT_FP32>);
        if (cudaLaunchKernel(fn, grid, dim3(256), args, smem, s) != cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
    }
    {
        void* args[] = {&scratch, &T, &E, &k, &topk_idx, &gates};
        smem = 0;
        if (cudaLaunchKernel(reinterpret_cast<const void*>(&k_na_topk), dim3((T + 7) / 8), dim3(256), args, smem, s) !=
            cudaSuccess) {
            cudaGetLastError();
            return MOE_ERR_CUDA;
        }
    }
    return MOE_OK;
}
