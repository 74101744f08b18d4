// Register-level helpers shared by the expert kernels: warp-level MMA, exact
// FP4 / E4M3 / E8M0 widening, the device K order of intermediate units, SiLU.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                        const float (&c)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                         const float (&c)[4]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}

// four bytes of packed E2M1 pairs -> four f16x2 (low nibble -> low half); exact
__device__ __forceinline__ void fp4x8_to_f16x2(uint32_t w, uint32_t (&o)[4]) {
    asm("{\n.reg .b8 b0, b1, b2, b3;\n"
        "mov.b32 {b0, b1, b2, b3}, %4;\n"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w));
}

// power of two p with max|v| * p in [2^14, 2^15) (1 for 0 or non-finite), and 1/p
__device__ __forceinline__ void pow2_scale(unsigned int maxbits, float& sc, float& un) {
    const int be = static_cast<int>((maxbits >> 23) & 0xFFu);
    if (maxbits == 0u || be == 0xFF) {
        sc = 1.0f;
        un = 1.0f;
        return;
    }
    int s = 141 - be;  // |v| < 2^(be - 126): |v| * 2^s < 2^15
    s = s > 127 ? 127 : s;
    sc = __uint_as_float(static_cast<unsigned int>(127 + s) << 23);
    const int u = -s;  // >= -127
    un = u >= -126 ? __uint_as_float(static_cast<unsigned int>(127 + u) << 23) : __uint_as_float(0x00400000u);
}

// eight E4M3 bytes -> four f16x2 (bytes 2i, 2i+1 -> word i); exact
__device__ __forceinline__ void e4m3x8_to_f16x2(uint2 v, uint32_t (&o)[4]) {
    asm("{\n.reg .b16 l0, h0, l1, h1;\n"
        "mov.b32 {l0, h0}, %4;\n"
        "mov.b32 {l1, h1}, %5;\n"
        "cvt.rn.f16x2.e4m3x2 %0, l0;\n"
        "cvt.rn.f16x2.e4m3x2 %1, h0;\n"
        "cvt.rn.f16x2.e4m3x2 %2, l1;\n"
        "cvt.rn.f16x2.e4m3x2 %3, h1;\n}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(v.x), "r"(v.y));
}

// eight E4M3 bytes -> eight floats (byte i -> o[i]); exact
__device__ __forceinline__ void e4m3x8_to_f32(uint2 v, float (&o)[8]) {
    uint32_t h[4];
    asm("{\n.reg .b16 l0, h0, l1, h1;\n"
        "mov.b32 {l0, h0}, %4;\n"
        "mov.b32 {l1, h1}, %5;\n"
        "cvt.rn.f16x2.e4m3x2 %0, l0;\n"
        "cvt.rn.f16x2.e4m3x2 %1, h0;\n"
        "cvt.rn.f16x2.e4m3x2 %2, l1;\n"
        "cvt.rn.f16x2.e4m3x2 %3, h1;\n}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(v.x), "r"(v.y));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 x = *reinterpret_cast<__half2*>(&h[i]);
        o[2 * i] = __low2float(x);
        o[2 * i + 1] = __high2float(x);
    }
}

// E8M0 byte -> 2^(b-127) as a float (b = 0 gives 2^-127)
__device__ __forceinline__ float e8m0_to_f32(uint32_t b) {
    return __uint_as_float(b == 0 ? 0x00400000u : (b << 23));
}

// position of intermediate unit i in the device K order (the order in which
// the down projection's weight rows store their K elements)
__device__ __forceinline__ int dpos(int i) {
    const int w = i & 127, s = w >> 4, q = (w >> 2) & 3, e = w & 3;
    return (i & ~127) + 32 * q + 4 * s + e;
}

__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }

__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

}  // namespace moe
