// Device helpers shared by the kernels of libdn: shared-memory addresses,
// the global timer, mbarriers and 1-D bulk copies (the asynchronous copy
// engine), exact int8 -> fp32 conversion and a fixed-order 16-term dot
// product, a warp sum.  One definition each, so the kernels cannot drift
// apart.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace dn {
namespace dev {

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// global -> shared bulk copy completed on an mbarrier (transaction bytes)
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Exact int8 -> fp32 for the four bytes of a 32-bit word: byte b taken as
// u = b ^ 0x80 (= b + 128) is placed in the mantissa of 2^23 (bit pattern
// 0x4B000000 | u, the float 8388608 + u); subtracting 8388608 + 128 is exact
// and leaves b (binary32 holds every integer below 2^24 exactly).
__device__ __forceinline__ void i8x4_to_f32(uint32_t w, float *f) {
    const uint32_t u = w ^ 0x80808080u;
    f[0] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)) - 8388736.0f;
    f[1] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651)) - 8388736.0f;
    f[2] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)) - 8388736.0f;
    f[3] = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653)) - 8388736.0f;
}

// Exact int4 -> fp32 for the eight nibbles of a 32-bit word (byte i: k = 2i
// in the low, k = 2i + 1 in the high nibble, two's complement): each nibble
// n taken as n ^ 8 (= n + 8) goes into the mantissa of 2^23, as in
// i8x4_to_f32, and 2^23 + 8 comes off.
__device__ __forceinline__ void i4x8_to_f32(uint32_t w, float *f) {
    const uint32_t u = w ^ 0x88888888u;
    const uint32_t lo = u & 0x0F0F0F0Fu, hi = (u >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7650 + i)) - 8388616.0f;
        f[2 * i + 1] = __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7650 + i)) - 8388616.0f;
    }
}

// 16-term dot product of w with 16 consecutive floats at xp (16-byte
// aligned) in four interleaved chains of four, combined in a fixed order
__device__ __forceinline__ float dot16(const float w[16], const float *xp) {
    const float4 a = *reinterpret_cast<const float4 *>(xp);
    const float4 b = *reinterpret_cast<const float4 *>(xp + 4);
    const float4 c = *reinterpret_cast<const float4 *>(xp + 8);
    const float4 d = *reinterpret_cast<const float4 *>(xp + 12);
    float t0 = w[0] * a.x, t1 = w[1] * a.y, t2 = w[2] * a.z, t3 = w[3] * a.w;
    t0 = fmaf(w[4], b.x, t0);
    t1 = fmaf(w[5], b.y, t1);
    t2 = fmaf(w[6], b.z, t2);
    t3 = fmaf(w[7], b.w, t3);
    t0 = fmaf(w[8], c.x, t0);
    t1 = fmaf(w[9], c.y, t1);
    t2 = fmaf(w[10], c.z, t2);
    t3 = fmaf(w[11], c.w, t3);
    t0 = fmaf(w[12], d.x, t0);
    t1 = fmaf(w[13], d.y, t1);
    t2 = fmaf(w[14], d.z, t2);
    t3 = fmaf(w[15], d.w, t3);
    return (t0 + t1) + (t2 + t3);
}

// butterfly sum over the 32 lanes (every lane gets the same, fixed-order result)
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace dev
}  // namespace dn
