// Persistent, bulk-copy-pipelined kernel for large batches of 128 x 128
// heads: the whole part of the page's step ("qwen36: run the DeltaNet layer
// end to end on the card (Q36_DN_GPU=1)", section "What the PR does")
// between the in_proj and the out_proj - causal conv + SiLU with the ring
// advancing, the L2 norms of q and k, the decay, the delta against the
// decayed state, the write-back, out = q^T S over the updated state, and
// the gated RMSNorm with silu(z) - for one (sequence, value head) item at a
// time.  Organised for HBM streaming:
//
//  * one CTA per SM walks a contiguous range of items (b-major);
//  * each item's 64 KB state tile arrives by one cp.async.bulk copy on an
//    mbarrier into a 3-deep shared-memory ring, is updated in place by 16
//    warps (each thread keeps its 32 values in registers between the
//    decay/delta pass and the write-back/readout pass) and leaves by one bulk
//    store; the load of item j+2 is issued as soon as the store of item j-1
//    has been read out of shared memory;
//  * the item's inputs - its q and k rows (of its q/k head), its v and z rows,
//    one per thread (512 = 4 x 128 rows) - are built on the fly: the in_proj
//    output of a row is the sum of its segment partials in slot order
//    (dn_sched.cuh) times the row scale; q, k, v go through the conv over the
//    ring (K-1 history slots read, the newest written) and SiLU, z through
//    SiLU; q and k are L2-normalised with fp32 warp sums combined in a fixed
//    order.  The CTA's ring positions are read once into shared memory, so
//    an item's loads (segment count, partials, ring history, row scale and
//    conv weights) depend on nothing else and are issued one item ahead (as
//    volatile loads, so that the compiler keeps them there): their latency
//    hides behind the previous item's tile;
//  * the first two state tiles, and the first item's loads that do not come
//    from the in_proj kernel, are issued before the kernel waits for it
//    (programmatic dependent launch): the state, ring, gates and weights are
//    not written by it, the partials and segment counts are.
//
// Every wait is bounded (about one second); on timeout the kernel records an
// error in `err`, waits (bounded) for its own bulk copies and returns.
#include <cuda_bf16.h>

#include <algorithm>

#include "dn_internal.cuh"
#include "dn_sched.cuh"

namespace dn {
namespace {

constexpr int D = 128;               // dk = dv
constexpr int NT = 512;              // threads: one input row of the item each
constexpr int STAGES = 3;
constexpr uint32_t kTileBytes = D * D * 4;
constexpr int LPR = D / 4;           // 32 lanes across a row (float4 each)
constexpr int RPP = NT / LPR;        // 16 rows per pass
constexpr int NP = D / RPP;          // 8 float4 per thread
constexpr int PV = 6;                // partial slots fetched ahead (more are read on the spot)
constexpr int kMaxSeqCta = 64;       // sequences one CTA's item range may touch
constexpr uint64_t kWaitLimitNs = 1000000000ull;

struct StreamParams {
    const float *part_in;  // in_proj segment partials
    const int *nseg_in;
    const float *s_in;
    float *ring;           // [max_batch][conv_k][conv_ch]
    const int32_t *rpos;   // [max_batch][2]
    const float *wconv_t;  // [conv_k][conv_ch]
    const float *g, *beta; // [B][n_v]
    const float *w_norm;   // [dv]
    float *S;              // [max_batch][n_v][128][128]
    float *nrm;            // fp32 output rows, or
    uint8_t *xb_out;       // packed bf16 hi/lo B-operand tiles
    int *err;
    int MT, max_seg;       // in_proj row tiles and segment slots per tile
    int n_v, group, conv_ch, qk_dim, v_dim, kt_out, items;
    float l2_eps, q_scale, norm_eps;
};

struct __align__(128) StreamSmem {
    float tile[STAGES][D * D];  // 3 x 64 KB
    float rec[2][4 * D];        // the item's q^ | k^ | v | silu(z), double-buffered
    float gate[2][2];           // exp(g), beta
    float red[RPP][D];          // 8 KB
    float delta[D];
    float ssq_o[4];
    float ssq_qk[2][8];         // warp sums of squares (warps 0-3 q, 4-7 k), double-buffered
    float wn[D];                // gated-RMSNorm weight
    int dpos[kMaxSeqCta];       // ring positions of the CTA's sequences
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
// the item's state tile, on the stage's barrier
__device__ __forceinline__ void load_tile(StreamSmem &sm, int st, const StreamParams &p, int item) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(&sm.full[st])),
                 "r"(kTileBytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(sm.tile[st])),
        "l"(p.S + (size_t)item * (D * D)), "r"(kTileBytes), "r"(smem_u32(&sm.full[st]))
        : "memory");
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
// silu(a) = a / (1 + e^-a) with the hardware exponential and divide
// (__expf, __fdividef: a few ulp, far inside the step's tolerance; for
// a -> -inf the divisor overflows and the quotient is 0, silu's limit)
__device__ __forceinline__ float silu_f(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

// This thread's input row of item (b, h): region 0 q, 1 k, 2 v, 3 z (thread
// t serves row t % 128 of region t / 128).
struct RowRef {
    int b, c;          // sequence, in_proj row
    bool conv, ring_w; // goes through the conv; this item writes its ring slot
};
__device__ __forceinline__ RowRef row_of(const StreamParams &p, int b, int h, int hq, int t) {
    RowRef r;
    r.b = b;
    const int region = t >> 7, o = t & (D - 1);
    r.c = region == 0 ? hq * D + o
        : region == 1 ? p.qk_dim + hq * D + o
        : region == 2 ? 2 * p.qk_dim + h * D + o
                      : p.conv_ch + h * D + o;
    r.conv = region < 3;
    // q and k rows are shared by the value heads of a q/k head: the first writes
    r.ring_w = region == 2 || (region < 2 && h == hq * p.group);
    return r;
}

__device__ __forceinline__ float ld_cg(const float *ptr) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(ptr));
    return v;
}
__device__ __forceinline__ float ld_nc(const float *ptr) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(ptr));
    return v;
}

// One item ahead: the row's first PV segment partials, its ring history,
// scale and conv weights, and the item's gates.  Every load is
// unconditional, from an address that is valid whatever the row (slots past
// the segment count and the conv inputs of z rows are masked where they are
// used), because a select on a value still in flight would wait for it here.
template <int KC>
struct Ahead {
    float pv[PV], hist[KC - 1], sc, wc[KC], gv, bv;
    int ns;  // segment count of the row's tile
};

__device__ __forceinline__ int ld_cg_s32(const int *ptr) {
    int v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(ptr));
    return v;
}

// The loads that the in_proj kernel does not feed: ring history, row scale,
// conv weights, gates (for the first item they go out before the kernel
// waits for the in_proj kernel).
template <int KC>
__device__ __forceinline__ void load_ahead_fixed(const StreamParams &p, const StreamSmem &sm, int b0, int b,
                                                 int h, int hq, int t, Ahead<KC> &a) {
    const RowRef r = row_of(p, b, h, hq, t);
    const int item = b * p.n_v + h;
    const int cr = r.conv ? r.c : 0;  // z rows read channel 0's ring and weights
    const float *rb = p.ring + (size_t)r.b * KC * p.conv_ch + cr;
    int slot = sm.dpos[r.b - b0];
#pragma unroll
    for (int m = 0; m < KC - 1; ++m) {  // oldest input first
        a.hist[m] = ld_cg(rb + (size_t)slot * p.conv_ch);
        if (++slot == KC) slot = 0;
    }
    a.sc = ld_nc(p.s_in + r.c);
#pragma unroll
    for (int m = 0; m < KC; ++m) a.wc[m] = ld_nc(p.wconv_t + (size_t)m * p.conv_ch + cr);
    a.gv = ld_cg(p.g + item);  // [B][n_v] = item order
    a.bv = ld_cg(p.beta + item);
}
// The in_proj kernel's output for the row: segment count and partials.
template <int KC>
__device__ __forceinline__ void load_ahead_part(const StreamParams &p, int b, int h, int hq, int t,
                                                Ahead<KC> &a) {
    const RowRef r = row_of(p, b, h, hq, t);
    const int ptile = (r.b >> 6) * p.MT + (r.c >> 7);
    a.ns = ld_cg_s32(p.nseg_in + ptile);
    const float *pp = p.part_in + (size_t)ptile * p.max_seg * (64 * D) + (r.b & 63) * D + (r.c & (D - 1));
#pragma unroll
    for (int k = 0; k < PV; ++k)  // slots past max_seg fall back to slot 0
        a.pv[k] = ld_cg(pp + (size_t)(k < p.max_seg ? k : 0) * (64 * D));
}
template <int KC>
__device__ __forceinline__ void load_ahead(const StreamParams &p, const StreamSmem &sm, int b0, int b, int h,
                                           int hq, int t, Ahead<KC> &a) {
    load_ahead_part(p, b, h, hq, t, a);
    load_ahead_fixed(p, sm, b0, b, h, hq, t, a);
}

// The row's in_proj output, conv + SiLU (z: SiLU only); the ring slot of the
// new input is written by the item that owns the row.
template <int KC>
__device__ __forceinline__ float build_input(const StreamParams &p, const StreamSmem &sm, int b0, int b, int h,
                                             int hq, int t, const Ahead<KC> &a) {
    const RowRef r = row_of(p, b, h, hq, t);
    const int ns = a.ns;
    float acc = 0.f;
#pragma unroll
    for (int k = 0; k < PV; ++k)
        if (k < ns) acc += a.pv[k];  // slot order
    if (ns > PV) {
        const int ptile = (r.b >> 6) * p.MT + (r.c >> 7);
        const float *pp = p.part_in + (size_t)ptile * p.max_seg * (64 * D) + (r.b & 63) * D + (r.c & (D - 1));
        for (int k = PV; k < ns; ++k) acc += __ldcg(pp + (size_t)k * (64 * D));
    }
    const float xv = a.sc * acc;
    if (!r.conv) return silu_f(xv);
    float cv = 0.f;
#pragma unroll
    for (int m = 0; m < KC - 1; ++m) cv = fmaf(a.wc[m], a.hist[m], cv);
    cv = fmaf(a.wc[KC - 1], xv, cv);
    if (r.ring_w) {
        int ws = sm.dpos[r.b - b0] + KC - 1;  // the oldest slot, not read by this step
        if (ws >= KC) ws -= KC;
        p.ring[((size_t)r.b * KC + ws) * p.conv_ch + r.c] = xv;
    }
    return silu_f(cv);
}

// Gated RMSNorm of one item's readout (thread t < 128 holds o[t]; the warp
// sums of o^2 are in ssq_o) and the store of the result: fp32 rows for the
// CUDA-core out_proj, or bf16 hi/lo operand rows for the tensor-core one.
__device__ __forceinline__ void store_norm(const StreamParams &p, const StreamSmem &sm, float o, int b, int h,
                                           const float *rz, int t) {
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

template <int KC>
__global__ void __launch_bounds__(NT, 1) dn_core_stream_kernel(const StreamParams p) {
    extern __shared__ uint8_t smem_raw[];
    StreamSmem &sm = *reinterpret_cast<StreamSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int i0 = (int)(((unsigned)blockIdx.x * (unsigned)p.items) / gridDim.x);
    const int i1 = (int)(((unsigned)(blockIdx.x + 1) * (unsigned)p.items) / gridDim.x);
    const int n_items = i1 - i0;

    int issued = 0;  // (thread 0) tile loads issued so far
    if (t == 0) {
        for (int s = 0; s < STAGES; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&sm.full[s])));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        for (int j = 0; j < 2 && j < n_items; ++j, ++issued) load_tile(sm, j, p, i0 + j);
    }
    // the norm weights and the sequences' ring positions (advanced by the
    // previous step) in one round trip; the state is not written by the
    // in_proj kernel, its partials and segment counts are
    if (t < D) sm.wn[t] = p.w_norm[t];
    const int b0 = i0 / p.n_v;
    const int nseq = n_items > 0 ? (i1 - 1) / p.n_v - b0 + 1 : 0;
    for (int i = t; i < nseq; i += NT) sm.dpos[i] = p.rpos[2 * (b0 + i)];
    __syncthreads();
    // the item (b, h) and its q/k head hq, stepped without divisions
    int b = b0, h = i0 - b0 * p.n_v, hq = h / p.group;
    Ahead<KC> ac;  // item j
    if (n_items > 0) load_ahead_fixed(p, sm, b0, b, h, hq, t, ac);
    pdl_wait();
    if (t == 0) pdl_trigger();
    if (n_items > 0) load_ahead_part(p, b, h, hq, t, ac);

    const int c4 = t % LPR, r0 = t / LPR;
    bool failed = false;
    float o_prev = 0.f;      // (t < D) the previous item's readout, normalised after the next barrier
    int b_prev = 0, h_prev = 0;
    for (int j = 0; j < n_items; ++j) {
        const int item = i0 + j;
        const int st = j % STAGES, rbuf = j & 1;
        const int hn = h + 1 == p.n_v ? 0 : h + 1, bn = hn == 0 ? b + 1 : b;
        const int hqn = hn == 0 ? 0 : (hn == (hq + 1) * p.group ? hq + 1 : hq);

        // ---- the item's q^, k^, v, silu(z), gates; loads for the next item ----
        const float u = build_input(p, sm, b0, b, h, hq, t, ac);
        const float gv = ac.gv, bv = ac.bv;
        if (j + 1 < n_items) load_ahead(p, sm, b0, bn, hn, hqn, t, ac);
        if (warp < 8) {  // q (warps 0-3) and k (warps 4-7): sums of squares
            const float sq = warp_sum(u * u);
            if (lane == 0) sm.ssq_qk[rbuf][warp] = sq;
        }
        __syncthreads();
        if (j > 0 && t < D) store_norm(p, sm, o_prev, b_prev, h_prev, sm.rec[rbuf ^ 1] + 3 * D, t);
        float val = u;
        if (t < 2 * D) {
            const float *ssq = sm.ssq_qk[rbuf] + (t >> 7) * 4;
            val = u * (1.0f / sqrtf(((ssq[0] + ssq[1]) + (ssq[2] + ssq[3])) + p.l2_eps)) *
                  (t < D ? p.q_scale : 1.0f);
        }
        sm.rec[rbuf][t] = val;
        if (t == 0) {
            sm.gate[rbuf][0] = expf(gv);
            sm.gate[rbuf][1] = bv;
        }

        // ---- the state tile --------------------------------------------------
        const bool landed = mbar_wait(&sm.full[st], (j / STAGES) & 1);
        if (!__syncthreads_and(landed)) {
            failed = true;
            break;
        }
        const float *rq = sm.rec[rbuf], *rk = rq + D, *rv = rq + 2 * D;
        const float eg = sm.gate[rbuf][0], bt = sm.gate[rbuf][1];

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
                issued = j + 3;
            }
        }
        // readout o = S^T q; its gated RMSNorm over the head is finished after
        // the next barrier (the next item's first, or the one after the loop)
        if (t < D) {
            float o = 0.f;
#pragma unroll
            for (int r = 0; r < RPP; ++r) o += sm.red[r][t];
            const float sq = warp_sum(o * o);
            if (lane == 0) sm.ssq_o[warp] = sq;
            o_prev = o;
        }
        b_prev = b;
        h_prev = h;
        b = bn;
        h = hn;
        hq = hqn;
        // (red, delta, ssq_* and the other record buffer are next written after
        // a barrier of the next item)
    }
    __syncthreads();
    if (!failed && n_items > 0 && t < D) store_norm(p, sm, o_prev, b_prev, h_prev, sm.rec[(n_items - 1) & 1] + 3 * D, t);
    if (t == 0) {
        if (failed) atomicOr(p.err, 1);
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        // let any load still in flight land before the CTA exits
        for (int j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j)
            (void)mbar_wait(&sm.full[j % STAGES], (j / STAGES) & 1);
    }
    __syncthreads();
}

template <int KC>
cudaError_t launch_kc(const StreamParams &p, cudaStream_t st) {
    static std::atomic<uint64_t> attr_done{0};
    const size_t smem = sizeof(StreamSmem) + 128;
    const cudaError_t e = once_per_device(attr_done, [&](int) {
        return cudaFuncSetAttribute(dn_core_stream_kernel<KC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem);
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min(num_sms(), p.items));
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    PdlAttr pdl;
    pdl.apply(cfg);
    return cudaLaunchKernelEx(&cfg, dn_core_stream_kernel<KC>, p);
}

}  // namespace

bool dn_core_stream_ok(const Dims &d, int B) {
    const long items = (long)B * d.n_v, per_cta = (items + num_sms() - 1) / num_sms();
    return d.dk == D && d.dv == D && d.conv_k <= 4 && items >= 1 && per_cta / d.n_v + 2 <= kMaxSeqCta;
}

cudaError_t launch_dn_core_stream(const Dims &d, const LayerDev &L, int B, const float *g,
                                  const float *beta, bool tc, cudaStream_t st) {
    StreamParams p;
    p.part_in = L.part_in;
    p.nseg_in = L.nseg_in;
    p.s_in = L.s_in;
    p.ring = L.ring;
    p.rpos = L.rpos;
    p.wconv_t = L.wconv_t;
    p.g = g;
    p.beta = beta;
    p.w_norm = L.w_norm;
    p.S = L.S;
    p.nrm = L.nrm;
    p.xb_out = tc ? L.xb_out : nullptr;
    p.err = L.err;
    const GemmPlan gp = plan_tc_gemm(d.in_rows, d.hidden, B);
    p.MT = gp.MT;
    p.max_seg = gp.max_seg;
    p.n_v = d.n_v;
    p.group = d.n_v / d.n_qk;
    p.conv_ch = d.conv_ch;
    p.qk_dim = d.qk_dim;
    p.v_dim = d.v_dim;
    p.kt_out = (d.v_dim + kTileK - 1) / kTileK;
    p.items = B * d.n_v;
    p.l2_eps = d.l2_eps;
    p.q_scale = d.q_scale;
    p.norm_eps = d.norm_eps;
    switch (d.conv_k) {
        case 2: return launch_kc<2>(p, st);
        case 3: return launch_kc<3>(p, st);
        case 4: return launch_kc<4>(p, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dn
