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

// Packed pairs of fp32 (low word first) and the sm_100-family pair
// instructions: each element of a pair is rounded as its own scalar
// operation would be, so pair and scalar code give the same bits.
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
// i8x4_to_f32 as two pairs (k 0, 1) and (k 2, 3): the same exact values
__device__ __forceinline__ void i8x4_to_f32x2(uint32_t w, uint64_t &p01, uint64_t &p23) {
    const uint32_t u = w ^ 0x80808080u;
    const uint64_t m = f2_pack(0x4B000080u, 0x4B000080u);  // 8388736.0f twice
    p01 = f2_sub(f2_pack(__byte_perm(u, 0x4B000000u, 0x7650), __byte_perm(u, 0x4B000000u, 0x7651)), m);
    p23 = f2_sub(f2_pack(__byte_perm(u, 0x4B000000u, 0x7652), __byte_perm(u, 0x4B000000u, 0x7653)), m);
}
// i4x8_to_f32 as four pairs (k 2i, 2i + 1): the same exact values
__device__ __forceinline__ void i4x8_to_f32x2(uint32_t w, uint64_t p[4]) {
    const uint32_t u = w ^ 0x88888888u;
    const uint32_t lo = u & 0x0F0F0F0Fu, hi = (u >> 4) & 0x0F0F0F0Fu;
    const uint64_t m = f2_pack(0x4B000008u, 0x4B000008u);  // 8388616.0f twice
#pragma unroll
    for (int i = 0; i < 4; ++i)
        p[i] = f2_sub(f2_pack(__byte_perm(lo, 0x4B000000u, 0x7650 + i), __byte_perm(hi, 0x4B000000u, 0x7650 + i)), m);
}
// dot16 with the weights as pairs (w[2i], w[2i + 1]) in p[i]: the four
// chains of dot16 run as two pair chains, element for element the same
// operations, and combine in dot16's order (the same bits)
__device__ __forceinline__ float dot16x2(const uint64_t p[8], const float *xp) {
    const float4 a = *reinterpret_cast<const float4 *>(xp);
    const float4 b = *reinterpret_cast<const float4 *>(xp + 4);
    const float4 c = *reinterpret_cast<const float4 *>(xp + 8);
    const float4 d = *reinterpret_cast<const float4 *>(xp + 12);
    uint64_t t01 = f2_mul(p[0], f2_pack(__float_as_uint(a.x), __float_as_uint(a.y)));
    uint64_t t23 = f2_mul(p[1], f2_pack(__float_as_uint(a.z), __float_as_uint(a.w)));
    t01 = f2_fma(p[2], f2_pack(__float_as_uint(b.x), __float_as_uint(b.y)), t01);
    t23 = f2_fma(p[3], f2_pack(__float_as_uint(b.z), __float_as_uint(b.w)), t23);
    t01 = f2_fma(p[4], f2_pack(__float_as_uint(c.x), __float_as_uint(c.y)), t01);
    t23 = f2_fma(p[5], f2_pack(__float_as_uint(c.z), __float_as_uint(c.w)), t23);
    t01 = f2_fma(p[6], f2_pack(__float_as_uint(d.x), __float_as_uint(d.y)), t01);
    t23 = f2_fma(p[7], f2_pack(__float_as_uint(d.z), __float_as_uint(d.w)), t23);
    float t0, t1, t2, t3;
    f2_unpack(t01, t0, t1);
    f2_unpack(t23, t2, t3);
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
