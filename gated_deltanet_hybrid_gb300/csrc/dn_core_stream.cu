// Persistent, bulk-copy-pipelined state kernel for large batches (one
// 128 x 128 state tile per (sequence, value head)).
//
// It runs the recurrence of the page's step ("qwen36: run the DeltaNet layer
// end to end on the card (Q36_DN_GPU=1)", section "What the PR does": the
// decay, the delta against the decayed state, the write-back, out = q^T S
// over the updated state) and the gated RMSNorm with silu(z), on the
// per-(sequence, head) records that dn_prep_kernel wrote (normalised q and k,
// v, silu(z), exp(g), beta).  Organised for HBM streaming:
//
//  * one CTA per SM walks a contiguous range of (sequence, head) items;
//  * each item's 64 KB state tile and its 2 KB record arrive by two
//    cp.async.bulk copies on one mbarrier into a 3-deep shared-memory ring;
//    the tile is updated in place by 16 warps (each thread keeps its 32
//    values in registers between the decay/delta pass and the write-back /
//    readout pass) and leaves by one bulk store; the loads of item i+2 are
//    issued as soon as the store of item i-1 has been read out of shared
//    memory.
//  * the first two state tiles are fetched before the kernel waits for
//    dn_prep_kernel (programmatic dependent launch), the records after.
//
// Every wait is bounded (about one second); on timeout the kernel records an
// error in `err`, waits (bounded) for its own bulk copies and returns.
#include <cuda_bf16.h>

#include <algorithm>

#include "dn_internal.cuh"

namespace dn {
namespace {

constexpr int D = 128;               // dk = dv
constexpr int NT = 512;              // threads
constexpr int STAGES = 3;
constexpr uint32_t kTileBytes = D * D * 4;
constexpr int REC = 4 * D + 4;       // record floats: q^ | k^ | v | silu(z) | exp(g), beta, 0, 0
constexpr uint32_t kRecBytes = REC * 4;
constexpr int LPR = D / 4;           // 32 lanes across a row (float4 each)
constexpr int RPP = NT / LPR;        // 16 rows per pass
constexpr int NP = D / RPP;          // 8 float4 per thread
constexpr uint64_t kWaitLimitNs = 1000000000ull;

struct StreamParams {
    const float *rec;      // [B][n_v][REC]
    const float *w_norm;   // [dv]
    float *S;              // [max_batch][n_v][128][128]
    float *nrm;            // fp32 output rows, or
    uint8_t *xb_out;       // packed bf16 hi/lo B-operand tiles
    int *err;
    int n_v, v_dim, kt_out, items;
    float norm_eps;
};

struct __align__(128) StreamSmem {
    float tile[STAGES][D * D];  // 3 x 64 KB
    float rec[STAGES][REC];     // 3 x 2064 B
    float red[RPP][D];          // 8 KB
    float delta[D];
    float ssq_o[4];
    float wn[D];                // gated-RMSNorm weight
    uint64_t full[STAGES];
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
__device__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0 && global_ns() - t0 > kWaitLimitNs) return false;
    }
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// the item's state tile and record, on the stage's barrier
__device__ __forceinline__ void load_tile(StreamSmem &sm, int st, const StreamParams &p, int item) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&sm.full[st])),
                 "r"(kTileBytes + kRecBytes)
                 : "memory");
    bulk_g2s(sm.tile[st], p.S + (size_t)item * (D * D), kTileBytes, &sm.full[st]);
}
__device__ __forceinline__ void load_rec(StreamSmem &sm, int st, const StreamParams &p, int item) {
    bulk_g2s(sm.rec[st], p.rec + (size_t)item * REC, kRecBytes, &sm.full[st]);
}
__device__ __forceinline__ void store_tile(float *dst, const float *src) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_u32(src)), "r"(kTileBytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void __launch_bounds__(NT, 1) dn_core_stream_kernel(const StreamParams p) {
    extern __shared__ uint8_t smem_raw[];
    StreamSmem &sm = *reinterpret_cast<StreamSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int i0 = (int)(((unsigned)blockIdx.x * (unsigned)p.items) / gridDim.x);
    const int i1 = (int)(((unsigned)(blockIdx.x + 1) * (unsigned)p.items) / gridDim.x);
    const int n_items = i1 - i0;

    if (t == 0) {
        for (int s = 0; s < STAGES; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&sm.full[s])));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (t < D) sm.wn[t] = p.w_norm[t];
    __syncthreads();
    int issued = 0;  // (thread 0) item loads issued so far
    if (t == 0) {
        // the state tiles do not depend on the previous kernel (dn_prep_kernel):
        // fetch them before waiting for it, the records after
        for (int j = 0; j < 2 && j < n_items; ++j, ++issued) load_tile(sm, j, p, i0 + j);
        pdl_wait();
        pdl_trigger();
        for (int j = 0; j < issued; ++j) load_rec(sm, j, p, i0 + j);
    } else {
        pdl_wait();
    }

    const int c4 = t % LPR, r0 = t / LPR;
    bool failed = false;
    for (int j = 0; j < n_items; ++j) {
        const int item = i0 + j;
        const int b = item / p.n_v, h = item % p.n_v;
        const int st = j % STAGES;
        const bool landed = mbar_wait(&sm.full[st], (j / STAGES) & 1);
        if (!__syncthreads_and(landed)) {
            failed = true;
            break;
        }
        const float *rq = sm.rec[st], *rk = rq + D, *rv = rq + 2 * D, *rz = rq + 3 * D;
        const float eg = rq[4 * D], bt = rq[4 * D + 1];
        float *tile = sm.tile[st];

        // decay, then what the decayed state predicts for k
        float4 s[NP];
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const int r = r0 + i * RPP;
            s[i] = *reinterpret_cast<const float4 *>(tile + r * D + c4 * 4);
            const float kr = rk[r];
            s[i].x *= eg;
            s[i].y *= eg;
            s[i].z *= eg;
            s[i].w *= eg;
            acc.x = fmaf(s[i].x, kr, acc.x);
            acc.y = fmaf(s[i].y, kr, acc.y);
            acc.z = fmaf(s[i].z, kr, acc.z);
            acc.w = fmaf(s[i].w, kr, acc.w);
        }
        *reinterpret_cast<float4 *>(&sm.red[r0][c4 * 4]) = acc;
        __syncthreads();
        // delta against the decayed state
        if (t < D) {
            float kv = 0.f;
#pragma unroll
            for (int r = 0; r < RPP; ++r) kv += sm.red[r][t];
            sm.delta[t] = bt * (rv[t] - kv);
        }
        __syncthreads();
        // write-back S += k delta^T, and the readout partials over the updated state
        const float4 d4 = *reinterpret_cast<const float4 *>(&sm.delta[c4 * 4]);
        acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const int r = r0 + i * RPP;
            const float kr = rk[r], qr = rq[r];
            s[i].x = fmaf(kr, d4.x, s[i].x);
            s[i].y = fmaf(kr, d4.y, s[i].y);
            s[i].z = fmaf(kr, d4.z, s[i].z);
            s[i].w = fmaf(kr, d4.w, s[i].w);
            *reinterpret_cast<float4 *>(tile + r * D + c4 * 4) = s[i];
            acc.x = fmaf(s[i].x, qr, acc.x);
            acc.y = fmaf(s[i].y, qr, acc.y);
            acc.z = fmaf(s[i].z, qr, acc.z);
            acc.w = fmaf(s[i].w, qr, acc.w);
        }
        *reinterpret_cast<float4 *>(&sm.red[r0][c4 * 4]) = acc;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // tile writes -> bulk store
        __syncthreads();
        if (t == 0) {
            store_tile(p.S + (size_t)item * (D * D), tile);
            // the stage of item j-1 is free once its store has read shared memory
            asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
            if (j + 2 < n_items) {
                load_tile(sm, (j + 2) % STAGES, p, item + 2);
                load_rec(sm, (j + 2) % STAGES, p, item + 2);
                issued = j + 3;
            }
        }
        // readout o = S^T q and gated RMSNorm over the head
        float o = 0.f;
        if (t < D) {
#pragma unroll
            for (int r = 0; r < RPP; ++r) o += sm.red[r][t];
            const float sq = warp_sum(o * o);
            if (lane == 0) sm.ssq_o[warp] = sq;
        }
        __syncthreads();
        if (t < D) {
            const float total = (sm.ssq_o[0] + sm.ssq_o[1]) + (sm.ssq_o[2] + sm.ssq_o[3]);
            const float rinv = 1.0f / sqrtf(total / (float)D + p.norm_eps);
            const float n = o * rinv * sm.wn[t] * rz[t];
            const int k = h * D + t;
            if (p.xb_out == nullptr) {
                p.nrm[(size_t)b * p.v_dim + k] = n;
            } else {
                const __nv_bfloat16 hi = __float2bfloat16_rn(n);
                const __nv_bfloat16 lo = __float2bfloat16_rn(n - __bfloat162float(hi));
                uint8_t *ot = p.xb_out + ((size_t)(b >> 6) * p.kt_out + (k >> 6)) * kOpTile;
                const int kc = (k & 63) >> 3, e = k & 7;
                const int rh = 2 * (b & 63), rl = rh + 1;
                *reinterpret_cast<__nv_bfloat16 *>(ot + op_chunk_offset(rh, kc) + e * 2) = hi;
                *reinterpret_cast<__nv_bfloat16 *>(ot + op_chunk_offset(rl, kc) + e * 2) = lo;
            }
        }
        // (red, delta and ssq_o are next written after the next item's first barrier)
    }
    if (t == 0) {
        if (failed) atomicOr(p.err, 1);
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        // let any load still in flight land before the CTA exits
        for (int j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j)
            (void)mbar_wait(&sm.full[j % STAGES], (j / STAGES) & 1);
    }
    __syncthreads();
}

}  // namespace

bool dn_core_stream_ok(const Dims &d, int B) {
    return d.dk == D && d.dv == D && (long)B * d.n_v >= 2L * num_sms();
}

size_t dn_core_stream_smem() { return sizeof(StreamSmem) + 128; }

cudaError_t launch_dn_core_stream(const Dims &d, const LayerDev &L, int B, const float *g,
                                  const float *beta, bool tc, cudaStream_t st) {
    static int attr_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (attr_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(dn_core_stream_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)dn_core_stream_smem());
        if (e != cudaSuccess) return e;
        attr_dev = dev;
    }
    // conv, ring, norms and gates of every (sequence, head) first
    cudaError_t e = launch_dn_prep(d, L, B, g, beta, st);
    if (e != cudaSuccess) return e;
    StreamParams p;
    p.rec = L.prep_rec;
    p.w_norm = L.w_norm;
    p.S = L.S;
    p.nrm = L.nrm;
    p.xb_out = tc ? L.xb_out : nullptr;
    p.err = L.err;
    p.n_v = d.n_v;
    p.v_dim = d.v_dim;
    p.kt_out = (d.v_dim + kTileK - 1) / kTileK;
    p.items = B * d.n_v;
    p.norm_eps = d.norm_eps;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min(num_sms(), p.items));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = dn_core_stream_smem();
    cfg.stream = st;
    PdlAttr pdl;
    pdl.apply(cfg);
    return cudaLaunchKernelEx(&cfg, dn_core_stream_kernel, p);
}

}  // namespace dn
