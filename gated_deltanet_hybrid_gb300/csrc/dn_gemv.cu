// int8 row-scaled GEMV on the CUDA cores for small batches:
//   y[b][o] = s[o] * sum_k W[o][k] * x[b][k]
//
// The projections of the gated-DeltaNet step are int8 matrices with one fp32
// scale per output row (page "feat(qwen36): the dense trunk places itself",
// section "What this adds", item 1; the fused in_proj is "qkv ++ z, one GEMV
// instead of two").  At small batch the step is a weight stream: the kernel
// is built so that every SM keeps about 128 KB of weights in flight.
//
// W is stored as contiguous 8 KB tiles of 128 rows x 64 int8 in four 16-k
// parts (dn_internal.cuh; shared with the tensor-core kernel) and the work is split exactly like the tensor-core
// projection (stream-K, dn_sched.cuh): one CTA per SM takes a contiguous
// range of units, each 4 consecutive k tiles of one row tile (32 KB; bulk
// copies this size keep the per-stage hand-off cost small against the HBM
// time).  Warp 0 streams the CTA's units with 1-D bulk copies
// (cp.async.bulk) into a 6-deep shared-memory ring; sixteen compute warps
// read each tile from shared memory (16 contiguous bytes per lane: 16
// weights of one row; a warp takes 8 rows x 4 k parts), convert int8 exactly
// to fp32 and multiply with the fp32 activations (read through L1) in four
// independent FMA chains, one accumulator per (row, sequence).  At the end
// of each segment the four lanes of a row (8 apart) are combined in a fixed
// shuffle order and the unscaled partial goes to its slot, to be summed and
// scaled by the consumer in slot order (bitwise-reproducible results).
//
// Every wait is bounded (about one second of the global timer); on timeout
// the kernel records an error in `err`, lets its copies land and returns.
#include <algorithm>

#include "dn_internal.cuh"
#include "dn_sched.cuh"

namespace dn {
namespace {

constexpr int KU = 4;                    // 64-wide k tiles per unit: one 32 KB bulk copy
constexpr int NSTAGE = 6;
constexpr int kCompute = 512;            // compute threads (warps 1..16), one 16-byte chunk each
constexpr int kThreads = 32 + kCompute;  // + producer warp
constexpr uint32_t kTile = kTileM * kTileK;  // 8 KB
constexpr uint32_t kUnit = KU * kTile;       // 32 KB
constexpr uint64_t kWaitLimitNs = 1000000000ull;

struct __align__(128) GemvSmem {
    uint8_t tile[NSTAGE][kUnit];
    uint64_t full[NSTAGE];
    uint64_t empty[NSTAGE];
    int abort_flag;
};

struct GemvParams {
    const uint8_t *Wt;
    const float *x;   // [B][K]
    float *part;      // [tiles][max_seg][64][128]
    int *nseg;        // [tiles]
    int *err;
    SchedView sv;   // units per row tile in sv.KT
    int K, B, KTt;  // KTt: 64-wide k tiles per row
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
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
__device__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                          bool ignore_abort = false) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (!ignore_abort && *abort_flag) return false;
            if (global_ns() - t0 > kWaitLimitNs) return false;
        }
    }
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

// 16-term dot product in four interleaved chains of four (fixed order)
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

template <int NB>
__global__ void __launch_bounds__(kThreads, 1) gemv_i8_stream_kernel(const GemvParams p) {
    extern __shared__ uint8_t smem_raw[];
    GemvSmem &sm = *reinterpret_cast<GemvSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int tid = threadIdx.x, warp = tid >> 5;
    const int c = blockIdx.x;
    const int u0 = sched_unit_start(c, p.sv), u1 = sched_unit_start(c + 1, p.sv);
    const int KT = p.sv.KT;
    if (tid == 0) {
        for (int s = 0; s < NSTAGE; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&sm.full[s])));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&sm.empty[s])),
                         "r"(kCompute));
        }
        sm.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    volatile int *abort_flag = &sm.abort_flag;

    if (warp == 0) {
        if (tid == 0) {  // ---- producer: bulk copies of the weight tiles ----
            int issued = 0;
            for (int u = u0; u < u1; ++u) {
                const int it = u - u0, st = it % NSTAGE;
                if (it >= NSTAGE && !mbar_wait(&sm.empty[st], ((it / NSTAGE) - 1) & 1, abort_flag)) {
                    *abort_flag = 1;
                    break;
                }
                const int tile = u / KT, j = u % KT;
                const int mt = tile % p.sv.MT;
                const int kt0 = j * KU, nk = min(KU, p.KTt - kt0);
                const uint32_t bytes = (uint32_t)nk * kTile;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                                 smem_u32(&sm.full[st])),
                             "r"(bytes)
                             : "memory");
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                        smem_u32(sm.tile[st])),
                    "l"(p.Wt + ((size_t)mt * p.KTt + kt0) * kTile), "r"(bytes), "r"(smem_u32(&sm.full[st]))
                    : "memory");
                issued = it + 1;
            }
            if (*abort_flag) {
                for (int it = issued > NSTAGE ? issued - NSTAGE : 0; it < issued; ++it)
                    mbar_wait(&sm.full[it % NSTAGE], (it / NSTAGE) & 1, abort_flag, true);
            }
        }
    } else {
        // ---- compute: lane l of compute warp w takes k part l/8 (16 of the
        //      tile's 64 k) of row 8w + l%8 of each 8 KB tile of the unit ---------
        pdl_wait();  // x and the partial buffers: after the previous kernel
        if (tid == 32) pdl_trigger();
        const int t = tid - 32;
        const int kp = (t >> 3) & 3;
        const int r = (t >> 5) * 8 + (t & 7);
        float acc[NB];
        int tile_cur = -1;
        for (int u = u0; u <= u1; ++u) {
            const int tile = u < u1 ? u / KT : -2;
            if (tile != tile_cur && tile_cur >= 0) {
                // end of a segment: combine the 4 lanes of each row, write the partial
#pragma unroll
                for (int j = 0; j < NB; ++j) {
                    float v = acc[j];
                    v += __shfl_xor_sync(0xffffffffu, v, 8);
                    v += __shfl_xor_sync(0xffffffffu, v, 16);
                    acc[j] = v;
                }
                const int slot = c - sched_cta_of_unit(tile_cur * KT, p.sv);
                if (t == 0 && u1 >= (tile_cur + 1) * KT) p.nseg[tile_cur] = slot + 1;
                if (kp == 0) {
                    float *ps = p.part + ((size_t)tile_cur * p.sv.max_seg + slot) * (64 * 128);
#pragma unroll
                    for (int j = 0; j < NB; ++j)
                        if (j < p.B) ps[j * 128 + r] = acc[j];
                }
            }
            if (u == u1) break;
            if (tile != tile_cur) {
#pragma unroll
                for (int j = 0; j < NB; ++j) acc[j] = 0.f;
                tile_cur = tile;
            }
            const int it = u - u0, st = it % NSTAGE;
            bool ok = mbar_wait(&sm.full[st], (it / NSTAGE) & 1, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                *abort_flag = 1;
                break;
            }
            const int kt0 = (u % KT) * KU, nk = min(KU, p.KTt - kt0);
            uint4 wv[KU];
#pragma unroll
            for (int i = 0; i < KU; ++i)
                if (i < nk) wv[i] = *reinterpret_cast<const uint4 *>(sm.tile[st] + i * kTile + kp * 2048 + r * 16);
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&sm.empty[st]))
                         : "memory");
#pragma unroll
            for (int i = 0; i < KU; ++i) {
                const int k0 = (kt0 + i) * kTileK + kp * 16;
                if (i < nk && k0 < p.K) {
                    float fa[16];
                    i8x4_to_f32(wv[i].x, fa);
                    i8x4_to_f32(wv[i].y, fa + 4);
                    i8x4_to_f32(wv[i].z, fa + 8);
                    i8x4_to_f32(wv[i].w, fa + 12);
#pragma unroll
                    for (int jb = 0; jb < NB; ++jb)
                        if (jb < p.B) acc[jb] += dot16(fa, p.x + (size_t)jb * p.K + k0);
                }
            }
        }
    }
    __syncthreads();
    if (tid == 0 && sm.abort_flag) atomicOr(p.err, 1);
}

template <int NB>
cudaError_t launch_nb(const uint8_t *Wt, const float *x, float *part, int *nseg, int *err, int M,
                      int K, int B, cudaStream_t st) {
    static int attr_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t smem = sizeof(GemvSmem) + 128;
    if (attr_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(gemv_i8_stream_kernel<NB>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr_dev = dev;
    }
    const GemmPlan g = plan_tc_gemm(M, K, B);
    GemvParams p;
    p.Wt = Wt;
    p.x = x;
    p.part = part;
    p.nseg = nseg;
    p.err = err;
    p.sv = SchedView{g.U, g.G, g.UT, g.MT, g.max_seg};
    p.K = K;
    p.B = B;
    p.KTt = g.KT;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)g.G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    PdlAttr pdl;
    pdl.apply(cfg);
    return cudaLaunchKernelEx(&cfg, gemv_i8_stream_kernel<NB>, p);
}

}  // namespace

cudaError_t launch_gemv_i8(const uint8_t *Wt, const float *x, float *part, int *nseg, int *err,
                           int M, int K, int B, cudaStream_t st) {
    if (B == 1) return launch_nb<1>(Wt, x, part, nseg, err, M, K, B, st);
    if (B == 2) return launch_nb<2>(Wt, x, part, nseg, err, M, K, B, st);
    if (B <= 4) return launch_nb<4>(Wt, x, part, nseg, err, M, K, B, st);
    return launch_nb<8>(Wt, x, part, nseg, err, M, K, B, st);
}

}  // namespace dn
