// int8 row-scaled GEMV on CUDA cores: y[b][o] = s[o] * sum_k W[o][k] * x[b][k].
//
// The projections of the gated-DeltaNet step are int8 matrices with one fp32
// scale per output row (page "feat(qwen36): the dense trunk places itself",
// section "What this adds", item 1; the fused in_proj is "qkv ++ z, one GEMV
// instead of two").  At small batch the step is a pure weight stream, so the
// kernel is built around the HBM read of W: one warp per output row, 16-byte
// loads of 16 int8 weights per lane (a warp covers 512 consecutive bytes of a
// row per iteration), all of a lane's loads for a row issued before any use,
// and a fixed xor-shuffle reduction order (bitwise-reproducible results).
// Each weight is converted once and used for every batch column of the
// chunk, so W is read from memory once per chunk of NB sequences.
#include "dn_internal.cuh"

namespace dn {
namespace {

constexpr int kWarps = 8;

// Exact int8 -> fp32 for the four bytes of a 32-bit word.  Byte b of the
// word, taken as unsigned u = b ^ 0x80 (= b + 128), is placed in the low
// mantissa bits of 2^23 (bit pattern 0x4B000000 | u, the float 8388608 + u);
// subtracting 8388608 + 128 is exact and leaves b.  (IEEE-754 binary32: any
// integer below 2^24 is exact, and at exponent 2^23 one mantissa unit is 1.)
__device__ __forceinline__ void i8x4_to_f32(uint32_t w, float &f0, float &f1, float &f2,
                                            float &f3) {
    const uint32_t u = w ^ 0x80808080u;
    f0 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)) - 8388736.0f;
    f1 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651)) - 8388736.0f;
    f2 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)) - 8388736.0f;
    f3 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653)) - 8388736.0f;
}

__device__ __forceinline__ void unpack16(const int4 v, float f[16]) {
    i8x4_to_f32((uint32_t)v.x, f[0], f[1], f[2], f[3]);
    i8x4_to_f32((uint32_t)v.y, f[4], f[5], f[6], f[7]);
    i8x4_to_f32((uint32_t)v.z, f[8], f[9], f[10], f[11]);
    i8x4_to_f32((uint32_t)v.w, f[12], f[13], f[14], f[15]);
}

__device__ __forceinline__ float dot16(const float w[16], const float *xp) {
    const float4 a = *reinterpret_cast<const float4 *>(xp);
    const float4 b = *reinterpret_cast<const float4 *>(xp + 4);
    const float4 c = *reinterpret_cast<const float4 *>(xp + 8);
    const float4 d = *reinterpret_cast<const float4 *>(xp + 12);
    float t = w[0] * a.x;
    t = fmaf(w[1], a.y, t);
    t = fmaf(w[2], a.z, t);
    t = fmaf(w[3], a.w, t);
    t = fmaf(w[4], b.x, t);
    t = fmaf(w[5], b.y, t);
    t = fmaf(w[6], b.z, t);
    t = fmaf(w[7], b.w, t);
    t = fmaf(w[8], c.x, t);
    t = fmaf(w[9], c.y, t);
    t = fmaf(w[10], c.z, t);
    t = fmaf(w[11], c.w, t);
    t = fmaf(w[12], d.x, t);
    t = fmaf(w[13], d.y, t);
    t = fmaf(w[14], d.z, t);
    t = fmaf(w[15], d.w, t);
    return t;
}

// One warp per output row.  Weights of the row are streamed UNROLL 16-byte
// chunks per lane at a time (loads first, then math).  NB batch columns share
// each converted weight.
template <int NB, int UNROLL>
__global__ void __launch_bounds__(kWarps * 32)
gemv_i8_kernel(const int8_t *__restrict__ W, const float *__restrict__ s,
               const float *__restrict__ x, float *__restrict__ y, int M, int K, int B,
               int32_t *__restrict__ rpos, int conv_k) {
    if (rpos != nullptr && blockIdx.x == 0) {
        // ring positions advance once per step, after the core kernel read them
        for (int b = threadIdx.x; b < B; b += blockDim.x) {
            int2 p = reinterpret_cast<int2 *>(rpos)[b];
            p.x = (p.x + 1) % conv_k;
            p.y = (p.y + 1) % (conv_k - 1);
            reinterpret_cast<int2 *>(rpos)[b] = p;
        }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int stride_rows = gridDim.x * kWarps;
    for (int row = blockIdx.x * kWarps + warp; row < M; row += stride_rows) {
        const int8_t *wr = W + (size_t)row * K;
        const float sc = s[row];
        for (int b0 = 0; b0 < B; b0 += NB) {
            float acc[NB];
#pragma unroll
            for (int j = 0; j < NB; ++j) acc[j] = 0.f;
            for (int kb = 0; kb < K; kb += 512 * UNROLL) {
                int4 wv[UNROLL];
#pragma unroll
                for (int u = 0; u < UNROLL; ++u) {
                    const int k0 = kb + u * 512 + lane * 16;
                    wv[u] = (k0 < K) ? __ldcs(reinterpret_cast<const int4 *>(wr + k0))
                                     : make_int4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < UNROLL; ++u) {
                    const int k0 = kb + u * 512 + lane * 16;
                    if (k0 < K) {
                        float wf[16];
                        unpack16(wv[u], wf);
#pragma unroll
                        for (int j = 0; j < NB; ++j)
                            if (b0 + j < B) acc[j] += dot16(wf, x + (size_t)(b0 + j) * K + k0);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < NB; ++j) {
                float v = acc[j];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                acc[j] = v;
            }
            if (lane == 0) {
#pragma unroll
                for (int j = 0; j < NB; ++j)
                    if (b0 + j < B) y[(size_t)(b0 + j) * M + row] = sc * acc[j];
            }
        }
    }
}

template <int NB, int UNROLL>
cudaError_t launch_nb(const int8_t *W, const float *s, const float *x, float *y, int M, int K,
                      int B, int32_t *rpos, int conv_k, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((M + kWarps - 1) / kWarps));
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, gemv_i8_kernel<NB, UNROLL>, W, s, x, y, M, K, B, rpos,
                              conv_k);
}

}  // namespace

cudaError_t launch_gemv_i8(const int8_t *W, const float *s, const float *x, float *y, int M,
                           int K, int B, int32_t *rpos_advance, int conv_k, cudaStream_t st) {
    // unroll so that one lane's loads of a row are in flight together
    if (B == 1) {
        if (K >= 2048) return launch_nb<1, 4>(W, s, x, y, M, K, B, rpos_advance, conv_k, st);
        return launch_nb<1, 1>(W, s, x, y, M, K, B, rpos_advance, conv_k, st);
    }
    if (B == 2) return launch_nb<2, 2>(W, s, x, y, M, K, B, rpos_advance, conv_k, st);
    if (B <= 4) return launch_nb<4, 2>(W, s, x, y, M, K, B, rpos_advance, conv_k, st);
    return launch_nb<8, 1>(W, s, x, y, M, K, B, rpos_advance, conv_k, st);
}

}  // namespace dn
