// Persistent, bulk-copy-pipelined version of the fused gated-DeltaNet kernel
// for large batches (one 128 x 128 state tile per (sequence, value head)).
//
// Same arithmetic and order as dn_core.cu (page "qwen36: run the DeltaNet
// layer end to end on the card (Q36_DN_GPU=1)", section "What the PR does":
// conv + SiLU with the ring advancing, L2 norms of q and k, decay,
// delta against the decayed state, write-back, out = q^T S over the updated
// state, gated RMSNorm with silu(z)), organised for HBM streaming.  (The
// L2 norms are tree sums in fp32 here, a relative error near 1e-7; the norm
// factors are applied to the dot products instead of to q and k first.)
//
//  * one CTA per SM walks a contiguous range of (sequence, head) items;
//  * each item's 64 KB state tile arrives by one cp.async.bulk into a
//    3-deep shared-memory ring (an mbarrier per stage), is updated in place
//    by 16 "state" warps (each thread keeps its 32 values in registers
//    between the decay/delta pass and the write-back/readout pass), and
//    leaves by one bulk store; the load of item i+2 is issued as soon as the
//    store of item i-1 has been read out of shared memory;
//  * 4 "prep" warps compute item i+1's conv + SiLU (reading the in_proj
//    partials, ring slots and conv taps), update the ring, and sum the
//    squares of q and k while the state warps work on item i; the two roles
//    hand over double-buffered item vectors through mbarriers.
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
constexpr int NT = 512;              // threads
constexpr int STAGES = 3;
constexpr uint32_t kTileBytes = D * D * 4;
constexpr int LPR = D / 4;           // 32 lanes across a row (float4 each)
constexpr int RPP = NT / LPR;        // 16 rows per pass
constexpr int NP = D / RPP;          // 8 float4 per thread
constexpr uint64_t kWaitLimitNs = 1000000000ull;
constexpr int kMaxConvK = 4;       // taps handled here (longer convs use dn_core.cu)
constexpr int kMaxSegLoad = 4;       // partial slots per channel loaded ahead

struct StreamParams {
    const float *part_in;  // in_proj segment partials
    const int *nseg_in;    // segments per tile
    const float *s_in;
    SchedView sv;
    float *ring;           // [max_batch][conv_k][conv_ch]
    const int32_t *rpos;   // [max_batch][2]
    const float *wconv_t;  // [conv_k][conv_ch]
    const float *w_norm;   // [dv]
    float *S;              // [max_batch][n_v][128][128]
    float *nrm;            // fp32 output rows, or
    uint8_t *xb_out;       // packed bf16 hi/lo B-operand tiles
    const float *g, *beta; // [B][n_v]
    int *err;
    int n_qk, n_v, conv_k, conv_ch, qk_dim, in_rows, v_dim, kt_out, items, B, n_tiles_in;
    float l2_eps, norm_eps, q_scale;
};

constexpr int kMaxSmemTiles = 2048;  // in_proj tiles whose segment counts are cached in smem
constexpr int kMaxSeqs = 64;         // ring positions cached per CTA
constexpr int NS = 512;              // state threads (warps 0..15)
constexpr int NPREP = 128;           // prep threads (warps 16..19)
constexpr int NTH = NS + NPREP;
constexpr int kChan = 4;             // channels per prep thread (4 x 128 = q, k, v, z rows)

struct __align__(128) StreamSmem {
    float tile[STAGES][D * D];  // 3 x 64 KB
    float red[RPP][D];          // 8 KB
    float delta[D];
    // per-item vectors, double-buffered by item parity (written by the prep
    // warps for item j+1 while the state warps use item j): silu(conv) of the
    // raw q and k rows, v, silu(z), per-prep-warp sums of squares of q and k,
    // exp(g) and beta
    float q[2][D], k[2][D], v[2][D], zg[2][D];
    float ssq[2][NPREP / 32][2];
    float gate[2][2];
    float ssq_o[4];
    float wn[D];  // gated-RMSNorm weight
    int nseg[kMaxSmemTiles];
    int dpos[kMaxSeqs];
    uint64_t full[STAGES];     // state tile landed
    uint64_t prep_done[2];     // item vectors of a buffer ready
    uint64_t state_done[2];    // state warps finished with a buffer
    int abort_flag;
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
// Waits for the phase of `bar` with the given parity; false after about one
// second or once another role has aborted (unless ignore_abort).
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
__device__ __forceinline__ void state_sync() {  // the 512 state threads only
    asm volatile("bar.sync 1, 512;" ::: "memory");
}
__device__ __forceinline__ void load_tile(float *dst, const float *src, uint64_t *bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(kTileBytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(kTileBytes), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void store_tile(float *dst, const float *src) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_u32(src)), "r"(kTileBytes)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

__device__ __forceinline__ float silu_f(float a) { return a / (1.0f + expf(-a)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// in_proj row of channel slot ch (0..511) of value head h: q | k | v | z
__device__ __forceinline__ int item_channel(const StreamParams &p, int h, int ch) {
    const int hq = h / (p.n_v / p.n_qk);
    if (ch < D) return hq * D + ch;
    if (ch < 2 * D) return p.qk_dim + hq * D + (ch - D);
    if (ch < 3 * D) return 2 * p.qk_dim + h * D + (ch - 2 * D);
    return p.conv_ch + h * D + (ch - 3 * D);
}

__device__ __forceinline__ int nseg_of(const StreamParams &p, const StreamSmem &sm, int tile) {
    return tile < kMaxSmemTiles ? sm.nseg[tile] : p.nseg_in[tile];
}

// Prep warps: conv + SiLU of item `item`'s q, k, v rows (and silu(z)), the
// ring update, the q/k sums of squares and the gates, into buffer pb.  Prep
// thread pt owns channel slots pt, pt+128, pt+256, pt+384 (one q, k, v and z
// row).  All loads are issued before any is used.
__device__ __forceinline__ void prep_item(const StreamParams &p, StreamSmem &sm, int seq_lo, int item,
                                          int pb, int pt) {
    const int b = item / p.n_v, h = item % p.n_v;
    const int group = p.n_v / p.n_qk;
    const int K = p.conv_k;
    const int dpos = sm.dpos[b - seq_lo];
    int ws = dpos + K - 1;
    if (ws >= K) ws -= K;
    float xs[kChan][kMaxSegLoad], sc[kChan], past[kChan][kMaxConvK - 1], w[kChan][kMaxConvK];
    int ns[kChan], cc[kChan];
#pragma unroll
    for (int i = 0; i < kChan; ++i) {
        const int c = item_channel(p, h, pt + 128 * i);
        cc[i] = c;
        const int tile = (b >> 6) * p.sv.MT + (c >> 7);
        ns[i] = nseg_of(p, sm, tile);
        const float *pp = p.part_in + (size_t)tile * p.sv.max_seg * (64 * 128) + (b & 63) * 128 + (c & 127);
#pragma unroll
        for (int k = 0; k < kMaxSegLoad; ++k)
            xs[i][k] = (k < ns[i]) ? __ldcg(pp + (size_t)k * (64 * 128)) : 0.f;
        sc[i] = p.s_in[c];
        if (i < 3) {
            const float *rb = p.ring + (size_t)b * K * p.conv_ch + c;
            int slot = dpos;
#pragma unroll
            for (int m = 0; m < kMaxConvK; ++m) {
                w[i][m] = (m < K) ? p.wconv_t[(size_t)m * p.conv_ch + c] : 0.f;
                if (m < K - 1) {
                    past[i][m] = rb[(size_t)slot * p.conv_ch];
                    if (++slot == K) slot = 0;
                }
            }
        }
    }
    float u[kChan];
#pragma unroll
    for (int i = 0; i < kChan; ++i) {
        // the in_proj output of the channel: segment partials in slot order, scaled
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxSegLoad; ++k)
            if (k < ns[i]) acc += xs[i][k];
        if (ns[i] > kMaxSegLoad) {  // (longer than the shipped schedules produce)
            const int tile = (b >> 6) * p.sv.MT + (cc[i] >> 7);
            const float *pp = p.part_in + (size_t)tile * p.sv.max_seg * (64 * 128) + (b & 63) * 128 + (cc[i] & 127);
            for (int k = kMaxSegLoad; k < ns[i]; ++k) acc += __ldcg(pp + (size_t)k * (64 * 128));
        }
        const float xv = sc[i] * acc;
        if (i < 3) {
            float cv = 0.f;
#pragma unroll
            for (int m = 0; m < kMaxConvK; ++m) {  // oldest input first, newest last
                if (m < K - 1) cv = fmaf(w[i][m], past[i][m], cv);
                if (m == K - 1) cv = fmaf(w[i][m], xv, cv);
            }
            // q/k rows are shared by the group's value heads: the first head writes
            if (i == 2 || h % group == 0) p.ring[((size_t)b * K + ws) * p.conv_ch + cc[i]] = xv;
            u[i] = silu_f(cv);
        } else {
            u[i] = silu_f(xv);
        }
    }
    sm.q[pb][pt] = u[0];
    sm.k[pb][pt] = u[1];
    sm.v[pb][pt] = u[2];
    sm.zg[pb][pt] = u[3];
    const float sq = warp_sum(u[0] * u[0]);
    const float sk = warp_sum(u[1] * u[1]);
    if ((pt & 31) == 0) {
        sm.ssq[pb][pt >> 5][0] = sq;
        sm.ssq[pb][pt >> 5][1] = sk;
    }
    if (pt == 0) {
        sm.gate[pb][0] = expf(p.g[item]);
        sm.gate[pb][1] = p.beta[item];
    }
}

// true iff pred holds in all 512 state threads (a barrier among them)
__device__ __forceinline__ bool state_all(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 512, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

__global__ void __launch_bounds__(NTH, 1) dn_core_stream_kernel(const StreamParams p) {
    extern __shared__ uint8_t smem_raw[];
    StreamSmem &sm = *reinterpret_cast<StreamSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int i0 = (int)(((unsigned)blockIdx.x * (unsigned)p.items) / gridDim.x);
    const int i1 = (int)(((unsigned)(blockIdx.x + 1) * (unsigned)p.items) / gridDim.x);
    const int n_items = i1 - i0;
    const int seq_lo = i0 / p.n_v;

    if (t == 0) {
        for (int s = 0; s < STAGES; ++s) mbar_init(&sm.full[s], 1);
        for (int a = 0; a < 2; ++a) {
            mbar_init(&sm.prep_done[a], NPREP);
            mbar_init(&sm.state_done[a], NS);
        }
        sm.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // scalars every item needs: segment counts of the in_proj tiles, ring
    // positions of this CTA's sequences, the norm weight
    for (int i = t; i < min(p.n_tiles_in, kMaxSmemTiles); i += NTH) sm.nseg[i] = p.nseg_in[i];
    for (int i = t; i < kMaxSeqs && seq_lo + i < p.B; i += NTH) sm.dpos[i] = p.rpos[2 * (seq_lo + i)];
    if (t < D) sm.wn[t] = p.w_norm[t];
    __syncthreads();
    volatile int *abort_flag = &sm.abort_flag;
    int issued = 0;  // (thread 0) tile loads issued so far
    if (t == 0) {
        for (int j = 0; j < 2 && j < n_items; ++j, ++issued)
            load_tile(sm.tile[j], p.S + (size_t)(i0 + j) * (D * D), &sm.full[j]);
    }

    if (t >= NS) {
        // ---- prep warps: item vectors, up to two items ahead of the state warps
        const int pt = t - NS;
        for (int j = 0; j < n_items; ++j) {
            const int pb = j & 1;
            if (j >= 2 && !mbar_wait(&sm.state_done[pb], ((j >> 1) - 1) & 1, abort_flag)) {
                *abort_flag = 1;
                break;
            }
            prep_item(p, sm, seq_lo, i0 + j, pb, pt);
            mbar_arrive(&sm.prep_done[pb]);
        }
    } else {
        // ---- state warps --------------------------------------------------------------
        const int c4 = t % LPR, r0 = t / LPR;
        for (int j = 0; j < n_items; ++j) {
            const int item = i0 + j;
            const int b = item / p.n_v, h = item % p.n_v;
            const int st = j % STAGES, pb = j & 1;
            const bool ok = mbar_wait(&sm.prep_done[pb], (j >> 1) & 1, abort_flag) &&
                            mbar_wait(&sm.full[st], (j / STAGES) & 1, abort_flag);
            if (!ok) *abort_flag = 1;
            if (!state_all(ok)) break;

            // decay, then what the decayed state predicts for the raw k
            const float ssq_q = (sm.ssq[pb][0][0] + sm.ssq[pb][1][0]) + (sm.ssq[pb][2][0] + sm.ssq[pb][3][0]);
            const float ssq_k = (sm.ssq[pb][0][1] + sm.ssq[pb][1][1]) + (sm.ssq[pb][2][1] + sm.ssq[pb][3][1]);
            const float inv_q = 1.0f / sqrtf(ssq_q + p.l2_eps);
            const float inv_k = 1.0f / sqrtf(ssq_k + p.l2_eps);
            const float eg = sm.gate[pb][0], bt = sm.gate[pb][1];
            float *tile = sm.tile[st];
            float4 s[NP];
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < NP; ++i) {
                const int r = r0 + i * RPP;
                s[i] = *reinterpret_cast<const float4 *>(tile + r * D + c4 * 4);
                const float kr = sm.k[pb][r];
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
            state_sync();
            // delta against the decayed state (k normalised by inv_k); the
            // write-back uses the raw k: S += (inv_k k) delta^T = k (inv_k delta)^T
            if (t < D) {
                float kv = 0.f;
#pragma unroll
                for (int r = 0; r < RPP; ++r) kv += sm.red[r][t];
                sm.delta[t] = bt * (sm.v[pb][t] - kv * inv_k) * inv_k;
            }
            state_sync();
            // write-back and readout partials
            const float4 d4 = *reinterpret_cast<const float4 *>(&sm.delta[c4 * 4]);
            acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < NP; ++i) {
                const int r = r0 + i * RPP;
                const float kr = sm.k[pb][r], qr = sm.q[pb][r];
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
            state_sync();
            if (t == 0) {
                store_tile(p.S + (size_t)item * (D * D), tile);
                // the stage of item j-1 is free once its store has read shared memory
                asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
                if (j + 2 < n_items) {
                    const int sn = (j + 2) % STAGES;
                    load_tile(sm.tile[sn], p.S + (size_t)(item + 2) * (D * D), &sm.full[sn]);
                    issued = j + 3;
                }
            }
            // readout (q normalised by inv_q, times q_scale) and gated RMSNorm
            float o = 0.f;
            if (t < D) {
#pragma unroll
                for (int r = 0; r < RPP; ++r) o += sm.red[r][t];
                o *= inv_q * p.q_scale;
                const float sq = warp_sum(o * o);
                if (lane == 0) sm.ssq_o[warp] = sq;
            }
            state_sync();
            if (t < D) {
                const float total = (sm.ssq_o[0] + sm.ssq_o[1]) + (sm.ssq_o[2] + sm.ssq_o[3]);
                const float rinv = 1.0f / sqrtf(total / (float)D + p.norm_eps);
                const float n = o * rinv * sm.wn[t] * sm.zg[pb][t];
                const int k = h * D + t;
                if (p.xb_out == nullptr) {
                    p.nrm[(size_t)b * p.v_dim + k] = n;
                } else {
                    const __nv_bfloat16 hi = __float2bfloat16_rn(n);
                    const __nv_bfloat16 lo = __float2bfloat16_rn(n - __bfloat162float(hi));
                    uint8_t *ot = p.xb_out + ((size_t)(b >> 6) * p.kt_out + (k >> 6)) * kOpTile;
                    const int kc = (k & 63) >> 3, e = k & 7;
                    const int rh = 2 * (b & 63), rl = rh + 1;
                    *reinterpret_cast<__nv_bfloat16 *>(ot + (rh >> 3) * 1024 + kc * 128 + (rh & 7) * 16 + e * 2) = hi;
                    *reinterpret_cast<__nv_bfloat16 *>(ot + (rl >> 3) * 1024 + kc * 128 + (rl & 7) * 16 + e * 2) = lo;
                }
            }
            mbar_arrive(&sm.state_done[pb]);  // (after every read of buffer pb)
        }
    }
    __syncthreads();
    if (t == 0) {
        if (sm.abort_flag) atomicOr(p.err, 1);
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        // let any tile load still in flight land before the CTA exits
        for (int j = issued > STAGES ? issued - STAGES : 0; j < issued; ++j)
            (void)mbar_wait(&sm.full[j % STAGES], (j / STAGES) & 1, abort_flag, true);
    }
    __syncthreads();
}

}  // namespace

bool dn_core_stream_ok(const Dims &d, int B) {
    return d.dk == D && d.dv == D && d.conv_k <= kMaxConvK && (long)B * d.n_v >= 2L * num_sms();
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
    StreamParams p;
    p.part_in = L.part_in;
    p.nseg_in = L.nseg_in;
    p.s_in = L.s_in;
    {
        const GemmPlan gp = plan_tc_gemm(d.in_rows, d.hidden, B);
        p.sv = SchedView{gp.U, gp.G, gp.UT, gp.MT, gp.max_seg};
    }
    p.ring = L.ring;
    p.rpos = L.rpos;
    p.wconv_t = L.wconv_t;
    p.w_norm = L.w_norm;
    p.S = L.S;
    p.nrm = L.nrm;
    p.xb_out = tc ? L.xb_out : nullptr;
    p.g = g;
    p.beta = beta;
    p.err = L.err;
    p.n_qk = d.n_qk;
    p.n_v = d.n_v;
    p.conv_k = d.conv_k;
    p.conv_ch = d.conv_ch;
    p.qk_dim = d.qk_dim;
    p.in_rows = d.in_rows;
    p.v_dim = d.v_dim;
    p.kt_out = (d.v_dim + kTileK - 1) / kTileK;
    p.items = B * d.n_v;
    p.B = B;
    p.n_tiles_in = plan_tc_gemm(d.in_rows, d.hidden, B).tiles;
    p.l2_eps = d.l2_eps;
    p.norm_eps = d.norm_eps;
    p.q_scale = d.q_scale;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)std::min(num_sms(), p.items));
    cfg.blockDim = dim3(NTH);
    cfg.dynamicSmemBytes = dn_core_stream_smem();
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, dn_core_stream_kernel, p);
}

}  // namespace dn
