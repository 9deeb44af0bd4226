// int8 row-scaled projection on the 5th-generation tensor cores (tcgen05),
// for batches large enough that the GEMV becomes a dense contraction:
//   y[b][m] = s[m] * sum_k W[m][k] * x[b][k]
// (the fused in_proj "qkv ++ z" and the out_proj of the gated-DeltaNet step;
// int8 rows with one fp32 scale each, page "feat(qwen36): the dense trunk
// places itself", section "What this adds", item 1).
//
// Precision.  int8 weights are exact in bf16.  The fp32 activations are split
// into x = hi + lo with hi = bf16(x) and lo = bf16(x - hi), so that W*hi +
// W*lo reproduces W*x to about 2^-17 relative per term, with fp32 tensor-core
// accumulation.  hi and lo of sequence b are rows 2b and 2b+1 of the MMA's B
// operand (N = 2 * padded batch), so one MMA covers both halves and the
// epilogue adds columns 2b and 2b+1.
//
// Work split.  One CTA per (128-row tile of W, K split, batch chunk of <= 64).
// Warps 0-3 stream their 128 int8 rows from HBM with 16-byte loads (one tile
// ahead in registers), convert to bf16 and store them in the MMA's canonical
// K-major layout (8x16-byte core matrices); warps 4-5 convert the batch's x to
// hi/lo bf16 the same way; warp 6 issues tcgen05.mma (M=128, N=2*B, K=16)
// from one thread into a TMEM accumulator, STAGES shared-memory stages deep,
// with mbarriers between the roles.  The epilogue (warps 0-3) reads TMEM with
// tcgen05.ld.  With several K splits every CTA writes a partial tile; the
// last CTA of a tile to finish (atomic counter) sums the partials in split
// order, so results do not depend on scheduling.
//
// Every wait is bounded (about one second of the global timer); on timeout
// the kernel records an error in `err`, lets in-flight MMAs drain, frees its
// TMEM and returns.
#include <cuda_bf16.h>

#include "dn_internal.cuh"

namespace dn {
namespace {

constexpr int BM = 128;         // weight rows per tile (MMA M)
constexpr int BK = 64;          // K per pipeline stage
constexpr int STAGES = 3;
constexpr int NB_CHUNK = 64;    // sequences per CTA (MMA N = 2 * padded count <= 128)
constexpr int kThreads = 224;   // 7 warps
constexpr int kProducers = 192; // warps 0-5
constexpr uint32_t kCoreBytes = 128;             // one 8 x 16-byte core matrix
constexpr uint32_t kGroupBytes = (BK / 8) * 128; // 8 rows x BK bf16 = 1024 bytes
constexpr uint64_t kWaitLimitNs = 1000000000ull;

struct __align__(1024) GemmSmem {
    uint8_t a[STAGES][BM * BK * 2];            // 16 KB per stage
    uint8_t b[STAGES][2 * NB_CHUNK * BK * 2];  // 16 KB per stage
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t done;
    uint32_t tmem_base;
    int abort_flag;
    int last;
};

struct GemmParams {
    const int8_t *W;
    const float *s;
    const float *x;
    float *y;
    float *part;      // [ks][B][M] partials (ks > 1)
    int *counters;    // [chunks][M / BM], zero between launches
    int32_t *rpos;    // optional: ring positions to advance (out_proj)
    int *err;
    int M, K, B, ks, k_split, conv_k;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

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

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `bar` with the given parity.  Gives up (returns
// false) after about one second or when another role has aborted.
__device__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > kWaitLimitNs) return false;
        }
    }
}

__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, K-major, no swizzle: core matrices of
// 8 rows x 16 bytes; `lbo` = byte distance between core matrices along K,
// `sbo` = byte distance between 8-row groups.  Bits 46..48 hold the fixed
// value 0b001 of the tcgen05 descriptor format.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Instruction descriptor of kind::f16: D fp32, A and B bf16, both K-major,
// N >> 3 at bits 17..22, M >> 4 at bits 24..28.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
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

// byte offset of (row, 8-element K chunk) in a K-major no-swizzle tile
__device__ __forceinline__ uint32_t core_off(int row, int kc) {
    return (uint32_t)(row >> 3) * kGroupBytes + (uint32_t)kc * kCoreBytes + (uint32_t)(row & 7) * 16u;
}

// 4 int8 -> 4 bf16 (exact): byte ^ 0x80 placed in the mantissa of 2^23 gives
// 2^23 + b + 128; subtracting 2^23 + 128 is exact; the result is an integer
// of magnitude <= 128, exactly representable in bf16.
__device__ __forceinline__ uint2 i8x4_to_bf16x4(uint32_t w) {
    const uint32_t u = w ^ 0x80808080u;
    const float f0 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)) - 8388736.0f;
    const float f1 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651)) - 8388736.0f;
    const float f2 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)) - 8388736.0f;
    const float f3 = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653)) - 8388736.0f;
    __nv_bfloat162 p0 = __floats2bfloat162_rn(f0, f1);
    __nv_bfloat162 p1 = __floats2bfloat162_rn(f2, f3);
    return make_uint2(*reinterpret_cast<uint32_t *>(&p0), *reinterpret_cast<uint32_t *>(&p1));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__global__ void __launch_bounds__(kThreads, 2) gemm_i8_tc_kernel(const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    GemmSmem &sm = *reinterpret_cast<GemmSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int mt = blockIdx.x, ksi = blockIdx.y, chunk = blockIdx.z;
    const int m0 = mt * BM;
    const int b0 = chunk * NB_CHUNK;
    const int Bc = min(NB_CHUNK, p.B - b0);
    const int Bpad = (Bc + 7) & ~7;
    const int N = 2 * Bpad;  // multiple of 16, <= 128
    const int k_begin = ksi * p.k_split;
    const int T = p.k_split / BK;

    if (p.rpos != nullptr && mt == 0 && ksi == 0) {  // ring positions advance once per step
        for (int b = tid; b < Bc; b += kThreads) {
            int2 q = reinterpret_cast<int2 *>(p.rpos)[b0 + b];
            q.x = (q.x + 1) % p.conv_k;
            q.y = (q.y + 1) % (p.conv_k - 1);
            reinterpret_cast<int2 *>(p.rpos)[b0 + b] = q;
        }
    }

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sm.full[s], kProducers);
            mbar_init(&sm.empty[s], 1);
        }
        mbar_init(&sm.done, 1);
        sm.abort_flag = 0;
        sm.last = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {  // TMEM accumulator: 128 lanes x 128 fp32 columns
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&sm.tmem_base)),
                     "r"(128)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = sm.tmem_base;
    volatile int *abort_flag = &sm.abort_flag;

    if (warp < 4) {
        // ---- A producers: one weight row each, BK int8 per stage ----------
        const int r = tid;
        const int8_t *gw = p.W + (size_t)(m0 + r) * p.K + k_begin;
        int4 cur[BK / 16], nxt[BK / 16];
#pragma unroll
        for (int i = 0; i < BK / 16; ++i) cur[i] = __ldcs(reinterpret_cast<const int4 *>(gw) + i);
        for (int t = 0; t < T; ++t) {
            const int st = t % STAGES;
            if (t + 1 < T) {
#pragma unroll
                for (int i = 0; i < BK / 16; ++i)
                    nxt[i] = __ldcs(reinterpret_cast<const int4 *>(gw + (size_t)(t + 1) * BK) + i);
            }
            if (t >= STAGES && !mbar_wait(&sm.empty[st], ((t / STAGES) - 1) & 1, abort_flag)) {
                *abort_flag = 1;
                break;
            }
            const uint32_t base = smem_u32(sm.a[st]);
#pragma unroll
            for (int i = 0; i < BK / 16; ++i) {  // 16 int8 (k = 16i..16i+15) -> two core rows
                const uint2 q0 = i8x4_to_bf16x4((uint32_t)cur[i].x);  // k + 0..3
                const uint2 q1 = i8x4_to_bf16x4((uint32_t)cur[i].y);  // k + 4..7
                const uint2 q2 = i8x4_to_bf16x4((uint32_t)cur[i].z);  // k + 8..11
                const uint2 q3 = i8x4_to_bf16x4((uint32_t)cur[i].w);  // k + 12..15
                st_shared_v4(base + core_off(r, 2 * i), make_uint4(q0.x, q0.y, q1.x, q1.y));
                st_shared_v4(base + core_off(r, 2 * i + 1), make_uint4(q2.x, q2.y, q3.x, q3.y));
            }
            fence_async_smem();
            mbar_arrive(&sm.full[st]);
#pragma unroll
            for (int i = 0; i < BK / 16; ++i) cur[i] = nxt[i];
        }
    } else if (warp < 6) {
        // ---- B producers: x row b -> bf16 hi (row 2b) and lo (row 2b+1) ----
        const int b = tid - 128;  // 0..63
        const bool valid = b < Bc;
        const bool active = b < Bpad;
        const float *gx = p.x + (size_t)(b0 + (valid ? b : 0)) * p.K + k_begin;
        for (int t = 0; t < T; ++t) {
            const int st = t % STAGES;
            float4 v[BK / 4];
            if (valid) {
#pragma unroll
                for (int i = 0; i < BK / 4; ++i)
                    v[i] = __ldcg(reinterpret_cast<const float4 *>(gx + (size_t)t * BK) + i);
            } else {
#pragma unroll
                for (int i = 0; i < BK / 4; ++i) v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (t >= STAGES && !mbar_wait(&sm.empty[st], ((t / STAGES) - 1) & 1, abort_flag)) {
                *abort_flag = 1;
                break;
            }
            if (active) {
                const uint32_t base = smem_u32(sm.b[st]);
#pragma unroll
                for (int kc = 0; kc < BK / 8; ++kc) {
                    const float xs[8] = {v[2 * kc].x, v[2 * kc].y, v[2 * kc].z, v[2 * kc].w,
                                         v[2 * kc + 1].x, v[2 * kc + 1].y, v[2 * kc + 1].z,
                                         v[2 * kc + 1].w};
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        __nv_bfloat162 h = __floats2bfloat162_rn(xs[2 * j], xs[2 * j + 1]);
                        const float2 hf = __bfloat1622float2(h);
                        __nv_bfloat162 l = __floats2bfloat162_rn(xs[2 * j] - hf.x, xs[2 * j + 1] - hf.y);
                        hi[j] = *reinterpret_cast<uint32_t *>(&h);
                        lo[j] = *reinterpret_cast<uint32_t *>(&l);
                    }
                    st_shared_v4(base + core_off(2 * b, kc), make_uint4(hi[0], hi[1], hi[2], hi[3]));
                    st_shared_v4(base + core_off(2 * b + 1, kc), make_uint4(lo[0], lo[1], lo[2], lo[3]));
                }
            }
            fence_async_smem();
            mbar_arrive(&sm.full[st]);
        }
    } else if (lane == 0) {
        // ---- MMA issuer ---------------------------------------------------------
        const uint32_t idesc = instr_desc(BM, N);
        for (int t = 0; t < T; ++t) {
            const int st = t % STAGES;
            if (!mbar_wait(&sm.full[st], (t / STAGES) & 1, abort_flag)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const uint32_t a0 = smem_u32(sm.a[st]), bb0 = smem_u32(sm.b[st]);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
                const uint64_t ad = smem_desc(a0 + kk * 2 * kCoreBytes, kCoreBytes, kGroupBytes);
                const uint64_t bd = smem_desc(bb0 + kk * 2 * kCoreBytes, kCoreBytes, kGroupBytes);
                mma_bf16(tmem_d, ad, bd, idesc, (t > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&sm.empty[st]);  // frees the stage once these MMAs have read it
        }
        mma_commit(&sm.done);  // arrives when every MMA issued above has completed
    }

    // ---- epilogue: warps 0-3 read their 32 TMEM lanes (= weight rows) --------
    if (warp < 4) {
        bool ok = mbar_wait(&sm.done, 0, abort_flag) && !*abort_flag;
        ok = __all_sync(0xffffffffu, ok);  // tcgen05.ld is warp-collective
        tc_fence_after();
        const int r = warp * 32 + lane;
        const int m = m0 + r;
        const float sc = p.s[m];
        const uint32_t trow = tmem_d + ((uint32_t)(warp * 32) << 16);
        if (ok) {
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                if (c * 16 < N) {  // warp-uniform
                    float v[16];
                    tmem_ld16(trow + c * 16, v);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int b = c * 8 + j;
                        if (b < Bc) {
                            const float acc = v[2 * j] + v[2 * j + 1];
                            if (p.ks == 1)
                                p.y[(size_t)(b0 + b) * p.M + m] = sc * acc;
                            else
                                p.part[((size_t)ksi * p.B + b0 + b) * p.M + m] = acc;
                        }
                    }
                }
            }
        } else {
            atomicOr(p.err, 1);
        }
        if (p.ks > 1) {
            __threadfence();
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (tid == 0) {
                const int old = atomicAdd(&p.counters[chunk * gridDim.x + mt], 1);
                sm.last = (old == p.ks - 1);
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (sm.last) {
                __threadfence();
                for (int b = 0; b < Bc; ++b) {
                    float acc = 0.f;
                    for (int k = 0; k < p.ks; ++k)
                        acc += __ldcg(&p.part[((size_t)k * p.B + b0 + b) * p.M + m]);
                    p.y[(size_t)(b0 + b) * p.M + m] = sc * acc;
                }
                if (tid == 0) p.counters[chunk * gridDim.x + mt] = 0;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_d), "r"(128)
                     : "memory");
    }
}

}  // namespace

bool tc_gemm_supported(int M, int K) { return M % BM == 0 && K % BK == 0 && K >= BK; }

int tc_gemm_splits(int M, int K, int B) {
    const int tiles = (M / BM) * ((B + NB_CHUNK - 1) / NB_CHUNK);
    const int target = 2 * num_sms();
    int ks = 1;
    while (ks < 8 && tiles * ks * 2 <= target && K % (BK * ks * 2) == 0 && K / (ks * 2) >= 2 * BK)
        ks *= 2;
    return ks;
}

size_t tc_gemm_smem_bytes() { return sizeof(GemmSmem) + 1024; }

cudaError_t launch_gemm_i8_tc(const int8_t *W, const float *s, const float *x, float *y,
                              float *part, int *counters, int *err, int M, int K, int B, int ks,
                              int32_t *rpos_advance, int conv_k, cudaStream_t st) {
    static bool attr_set = false;
    const size_t smem = tc_gemm_smem_bytes();
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(gemm_i8_tc_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    GemmParams p;
    p.W = W;
    p.s = s;
    p.x = x;
    p.y = y;
    p.part = part;
    p.counters = counters;
    p.rpos = rpos_advance;
    p.err = err;
    p.M = M;
    p.K = K;
    p.B = B;
    p.ks = ks;
    p.k_split = K / ks;
    p.conv_k = conv_k;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(M / BM), (unsigned)ks, (unsigned)((B + NB_CHUNK - 1) / NB_CHUNK));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, gemm_i8_tc_kernel, p);
}

}  // namespace dn
