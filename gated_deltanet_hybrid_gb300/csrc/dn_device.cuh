// Device helpers shared by the kernels of libdn: shared-memory addresses,
// the global timer, mbarriers and 1-D bulk copies (the asynchronous copy
// engine), exact int8 -> fp32 conversion and a fixed-order 16-term dot
// product, a warp sum, and the tcgen05 tensor-core primitives (matrix
// descriptors, MMAs with the A operand in tensor memory, tensor-memory loads
// and stores).  One definition each, so the kernels cannot drift
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

// ---- 5th-generation tensor cores (tcgen05) ----------------------------------

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor for the 128-byte swizzled K-major layout
// (bits 46..48 hold the descriptor format's fixed value 0b001): rows of 64 bf16
// (128 bytes) stored contiguously, 8-row groups 1024 bytes apart, and within
// each 1024-byte group the 16-byte chunk c of row r stored at chunk position
// c ^ (r & 7).  The leading offset is unused in this mode; a K step of 16
// elements inside the 128-byte row is a 32-byte advance of the start address
// (the hardware applies the XOR to the computed addresses), so groups must be
// 1024-byte aligned.  Layout-type field (bits 61..63) = 2.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// kind::f16 instruction descriptor: D fp32, A and B bf16, both K-major,
// N >> 3 at bits 17..22, M >> 4 at bits 24..28.
__device__ __forceinline__ uint32_t instr_desc(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

// Four K steps of 16: D (tensor memory) (+)= A (tensor memory, lane = row,
// 32-bit column = two consecutive k; 8 columns per step) x B (shared-memory
// descriptor, 32 bytes further per step)^T.  The first step overwrites D
// when `accumulate` is 0.  One asm block with precomputed operands: for
// 128 x 128 x 16 steps the issuing thread's own instruction count, not the
// tensor core, otherwise sets the pace.
__device__ __forceinline__ void mma_bf16_ts_x4(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 q, %4, %4;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %3, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%7], %8, %3, q;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%9], %10, %3, q;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(a_tmem + 8u), "l"(bdesc + 2u),
        "r"(a_tmem + 16u), "l"(bdesc + 4u), "r"(a_tmem + 24u), "l"(bdesc + 6u)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float v[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive 32-bit columns of this thread's tensor-memory lane, then
// wait until the stores are done
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t v[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
        "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
        "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Two K steps of 16 (K = 32), otherwise as mma_bf16_ts_x4
__device__ __forceinline__ void mma_bf16_ts_x2(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.eq.b32 q, %4, %4;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%5], %6, %3, q;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(a_tmem + 8u), "l"(bdesc + 2u)
        : "memory");
}

// 32 consecutive 32-bit columns of this thread's tensor-memory lane (wait
// included)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t r[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16 consecutive 32-bit columns of this thread's tensor-memory lane, then
// wait until the stores are done
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t v[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace dev
}  // namespace dn
