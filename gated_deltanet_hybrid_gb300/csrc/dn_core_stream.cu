// Persistent, bulk-copy-pipelined kernel for 128 x 128 heads: the whole part
// of the page's step ("qwen36: run the DeltaNet layer end to end on the card
// (Q36_DN_GPU=1)", section "What the PR does") between the in_proj and the
// out_proj - causal conv + SiLU with the ring advancing, the L2 norms of q
// and k, the decay, the delta against the decayed state, the write-back,
// out = q^T S over the updated state, and the gated RMSNorm with silu(z) -
// one (sequence, value head) item at a time.  Organised for HBM streaming:
//
//  * one CTA per SM walks a contiguous range of items (b-major, so the two
//    value heads of a q/k head follow each other); at large batches the
//    ranges are shorter than an even split and the rest of the items form a
//    pool handed out one at a time (an atomic counter, asked one item before
//    the answer is needed), so CTAs whose state streams run slower take
//    fewer items and all of them finish together.  The thread that issues
//    the tile copies publishes each position's item in a four-slot queue in
//    shared memory (one mbarrier per slot) for the producer warps; the step's
//    last kernel puts the counter back to zero;
//  * each item's 64 KB state tile arrives by one cp.async.bulk copy on an
//    mbarrier into a 3-deep shared-memory ring;
//  * 16 consumer warps (512 threads) read the tile into registers (32 values
//    per thread), decay it,
//    reduce it against k^ (delta), write it back and reduce it against q^
//    (readout) in registers, write it back into its stage and send it out
//    with one bulk store (global stores from registers would hold up the
//    load/store unit that the producers' loads need);
//  * 4 producer warps build the next item's inputs meanwhile, in a
//    double-buffered record, one warp per conv row kind and one for the z
//    rows and the gates (16-byte loads of four
//    channels per lane): for each of the item's q, k, v and z rows the
//    in_proj output (its segment partials summed in slot order, dn_sched.cuh,
//    times the row scale), then the conv over the ring (K-1 history slots
//    read, the newest written by the row's owner) and SiLU for q, k, v, SiLU
//    for z, the q/k L2 norms (one warp's fp32 shuffle sum, fixed order), the
//    query scale, the write strength and the decay of each key row (one
//    gate per head, or one per key channel).  The second value head of a q/k head reuses
//    the first one's q^ and k^.  Producers and consumers meet on two
//    mbarriers per record buffer (full, empty).  The loads of item j+1 are
//    issued as soon as item j's rows are computed;
//  * a stage takes the item three ahead once the bulk store of its item has
//    read it; the readout's gated RMSNorm is finished during the next item
//    by warps 4-7, which are otherwise idle while warps 0-3 form the delta;
//  * the first three state tiles, the ring positions and the norm weights
//    are requested before the kernel waits for the in_proj kernel
//    (programmatic dependent launch): the in_proj writes only the partials
//    and segment counts.  In pool mode the CTAs that start beside the
//    tensor-core in_proj (on the SMs it leaves free) also pull the first two
//    tiles of every other CTA into L2 while they wait (warm_l2).
//
// Every mbarrier wait is bounded (about one second of the global timer); on
// timeout the kernel records an error in `err`, leaves its loop (the
// consumers on a vote that all of them take, so no named barrier is left
// waiting; a producer warp on its own: it meets the others on mbarriers only),
// waits (bounded) for its own bulk copies and returns.
#include <cuda_bf16.h>

#include <algorithm>

#include "dn_device.cuh"
#include "dn_internal.cuh"
#include "dn_sched.cuh"

namespace dn {
namespace {

using dev::global_ns;
using dev::mbar_arrive;
using dev::smem_u32;
using dev::warp_sum;

constexpr int D = 128;               // dk = dv
constexpr int NC = 512;              // consumer threads (16 warps)
constexpr int NPW = 4;               // producer warps (q, k, v; z and the gates)
constexpr int NT = NC + 32 * NPW;    // 640
constexpr int STAGES = 3;
constexpr uint32_t kTileBytes = D * D * 4;
constexpr int LPR = D / 4;           // 32 lanes across a row (float4 each)
constexpr int RPP = NC / LPR;        // 16 rows per pass
constexpr int NP = D / RPP;          // 8 float4 per consumer thread
constexpr int PV = 4;                // partial slots loaded unconditionally (more are read on the spot)
constexpr int kMaxSeqCta = 64;       // sequences one CTA's item range may touch
// pool items per CTA: with at least kPoolPerCta + 4 items per CTA, each CTA's
// own range is that many items shorter than an even share
constexpr int kPoolPerCta = 3;
// the first tiles of each CTA that starts after the in_proj, which the CTAs
// that start beside it pull into L2 (pool mode)
constexpr int kWarmTiles = 2;
constexpr uint64_t kWaitLimitNs = 1000000000ull;
// named barriers (0 is __syncthreads)
constexpr int kBarCons = 1;          // the 512 consumer threads
// the consumer thread that issues the tile copies and stores (warp 15 has
// nothing else to do after the readout's barrier)
constexpr int kTma = NC - 32;

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
    int gw;                // log-decay values per head: 1, or 128 (per-key-channel gate)
    int dev_gates, in_rows; // g, beta from the a/b gate rows that follow the in_rows in_proj rows
    const float *gate_A;   // [n_v] (device gates)
    float l2_eps, q_scale, norm_eps;
    // item pool (nullptr: every CTA takes an even share of the items):
    // CTA c takes items [c * n_static, (c + 1) * n_static), then pool items
    // pool_base + k for the k the counter hands it, while k < pool_n
    int *pool;
    int n_static, pool_base, pool_n;
    int pf_ctas;  // CTAs 0 .. pf_ctas-1 start beside the in_proj and warm L2 (0: none)
};

struct __align__(128) StreamSmem {
    float tile[STAGES][D * D];  // 3 x 64 KB
    // (arrays read or written with 16-byte accesses are 16-byte aligned)
    alignas(16) float rec[2][5 * D];   // the item's q^ | k^ | v | silu(z) | exp(g) per key row, double-buffered
    alignas(16) float red[2][RPP][D];  // 2 x 8 KB: per-pass partial sums (kv, then readout)
    alignas(16) float delta[D];
    float beta[2];
    float ssq_o[4];             // readout warp sums of squares
    float o_prev[D];            // the last item's readout, normalised during the next item
    float zw_prev[D];           // its w_norm * silu(z)
    float wn[D];                // gated-RMSNorm weight
    int dpos[kMaxSeqCta];       // ring positions of the sequences of the CTA's own range
    int qitem[4];               // the item at position j >= 3 (-1: none), slot (j - 3) % 4
    uint64_t qfull[4];          // qitem slot written (one arrival by the copy thread)
    uint64_t full[STAGES];      // tile landed
    uint64_t rec_full[2];       // record built (one arrival per producer warp)
    uint64_t rec_empty[2];      // record read (one arrival per consumer warp)
    int failed;                 // a role gave up on a wait
};

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
// named barrier over `n` threads
__device__ __forceinline__ void bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// named barrier over `n` threads that also returns the AND of `ok`
__device__ __forceinline__ bool bar_and(int id, int n, bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok), "r"(id), "r"(n)
        : "memory");
    return r != 0;
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
// silu(a) = a / (1 + e^-a) with the hardware exponential and divide
// (__expf, __fdividef: a few ulp, far inside the step's tolerance; for
// a -> -inf the divisor overflows and the quotient is 0, silu's limit)
__device__ __forceinline__ float silu_f(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

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
__device__ __forceinline__ int ld_cg_s32(const int *ptr) {
    int v;
    asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(ptr));
    return v;
}
// The ring position of sequence b: from shared memory for the sequences of
// the CTA's own range, else (pool items) from global memory (written by the
// previous step's last kernel, which has completed)
__device__ __forceinline__ int ring_pos(const StreamParams &p, const StreamSmem &sm, int b0, int nseq, int b) {
    const unsigned i = (unsigned)(b - b0);
    return i < (unsigned)nseq ? sm.dpos[i] : ld_cg_s32(p.rpos + 2 * b);
}

// The item at position j of a CTA's walk, for the producer warps (-1: the
// walk has ended): the CTA's own range, then the queue slot the copy thread
// fills one to two items ahead of the consumers (waited for, bounded; false
// on timeout).
__device__ __forceinline__ bool item_at(StreamSmem &sm, int i0, int n_s, int j, int &item) {
    if (j < n_s) {
        item = i0 + j;
        return true;
    }
    if (j < 3) {
        item = -1;
        return true;
    }
    const int q = j - 3;
    if (!mbar_wait(&sm.qfull[q & 3], (q >> 2) & 1)) return false;
    item = sm.qitem[q & 3];
    return true;
}

// The loads of four channels c .. c+3 of one row kind (q, k, v or z) of an
// item, 16 bytes each: the in_proj segment partials (the first PV slots
// unconditionally, from clamped addresses, so no load waits for the segment
// count), the segment count, the row scales and, for q, k and v, the conv
// history and weights.
template <int KC>
struct RowLoads {
    float4 pv[PV], sc, hist[KC - 1], wc[KC];
    int ns;
};

__device__ __forceinline__ float4 ld_cg4(const float *ptr) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(ptr));
    return v;
}
__device__ __forceinline__ float4 ld_nc4(const float *ptr) {
    float4 v;
    asm volatile("ld.global.nc.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(ptr));
    return v;
}

// (dp: the sequence's ring position)
template <int KC>
__device__ __forceinline__ void load_row_fixed(const StreamParams &p, int dp, int b, int c, bool conv,
                                               RowLoads<KC> &r) {
    r.sc = ld_nc4(p.s_in + c);
    if (!conv) return;  // z rows (uniform across the warp)
    const float *rb = p.ring + (size_t)b * KC * p.conv_ch + c;
    int slot = dp;
#pragma unroll
    for (int m = 0; m < KC - 1; ++m) {  // oldest input first
        r.hist[m] = ld_cg4(rb + (size_t)slot * p.conv_ch);
        if (++slot == KC) slot = 0;
    }
#pragma unroll
    for (int m = 0; m < KC; ++m) r.wc[m] = ld_nc4(p.wconv_t + (size_t)m * p.conv_ch + c);
}

__device__ __forceinline__ const float *row_partials(const StreamParams &p, int b, int c) {
    const int ptile = (b >> 6) * p.MT + (c >> 7);
    return p.part_in + (size_t)ptile * p.max_seg * (64 * D) + (b & 63) * D + (c & (D - 1));
}

template <int KC>
__device__ __forceinline__ void load_row_part(const StreamParams &p, int b, int c, RowLoads<KC> &r) {
    r.ns = ld_cg_s32(p.nseg_in + (b >> 6) * p.MT + (c >> 7));
    const float *pp = row_partials(p, b, c);
#pragma unroll
    for (int k = 0; k < PV; ++k)  // slots past max_seg fall back to slot 0
        r.pv[k] = ld_cg4(pp + (size_t)(k < p.max_seg ? k : 0) * (64 * D));
}

__device__ __forceinline__ void add4(float4 &a, const float4 &b) {
    a.x += b.x;
    a.y += b.y;
    a.z += b.z;
    a.w += b.w;
}

// The four channels' in_proj output (partials in slot order, times the row scale)
template <int KC>
__device__ __forceinline__ float4 row_value(const StreamParams &p, int b, int c, const RowLoads<KC> &r) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int k = 0; k < PV; ++k)
        if (k < r.ns) add4(acc, r.pv[k]);
    if (r.ns > PV) {
        const float *pp = row_partials(p, b, c);
        for (int k = PV; k < r.ns; ++k) add4(acc, ld_cg4(pp + (size_t)k * (64 * D)));
    }
    return make_float4(r.sc.x * acc.x, r.sc.y * acc.y, r.sc.z * acc.z, r.sc.w * acc.w);
}

// conv over the history and the new input xv, then SiLU; the row's owner
// writes xv into the ring slot that this step does not read
template <int KC>
__device__ __forceinline__ float4 conv_silu(const StreamParams &p, int dp, int b, int c, float4 xv, bool owner,
                                            const RowLoads<KC> &r) {
    float4 cv = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < KC - 1; ++m) {
        cv.x = fmaf(r.wc[m].x, r.hist[m].x, cv.x);
        cv.y = fmaf(r.wc[m].y, r.hist[m].y, cv.y);
        cv.z = fmaf(r.wc[m].z, r.hist[m].z, cv.z);
        cv.w = fmaf(r.wc[m].w, r.hist[m].w, cv.w);
    }
    cv.x = fmaf(r.wc[KC - 1].x, xv.x, cv.x);
    cv.y = fmaf(r.wc[KC - 1].y, xv.y, cv.y);
    cv.z = fmaf(r.wc[KC - 1].z, xv.z, cv.z);
    cv.w = fmaf(r.wc[KC - 1].w, xv.w, cv.w);
    if (owner) {
        int ws = dp + KC - 1;  // the oldest slot, not read by this step
        if (ws >= KC) ws -= KC;
        *reinterpret_cast<float4 *>(p.ring + ((size_t)b * KC + ws) * p.conv_ch + c) = xv;
    }
    return make_float4(silu_f(cv.x), silu_f(cv.y), silu_f(cv.z), silu_f(cv.w));
}

// Gated RMSNorm of one item's readout o[i] (i = 0..127; the warp sums of
// o^2 are in ssq_o, zw = w_norm[i] * silu(z[i])) and the store of the
// result: fp32 rows for the CUDA-core out_proj, or bf16 hi/lo operand rows
// for the tensor-core one.
__device__ __forceinline__ void store_norm(const StreamParams &p, const StreamSmem &sm, float o, float zw, int b,
                                           int h, int i) {
    const float total = (sm.ssq_o[0] + sm.ssq_o[1]) + (sm.ssq_o[2] + sm.ssq_o[3]);
    const float rinv = 1.0f / sqrtf(total / (float)D + p.norm_eps);
    const float n = o * rinv * zw;
    const int k = h * D + i;
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

// softplus(a) = log(1 + e^a) as max(a, 0) + log1p(e^-|a|); sigmoid(b) = 1 / (1 + e^-b)
__device__ __forceinline__ float softplus_f(float a) { return fmaxf(a, 0.f) + log1pf(expf(-fabsf(a))); }
__device__ __forceinline__ float sigmoid_f(float b) { return 1.0f / (1.0f + expf(-b)); }

// An item's gates as seen by lane l of producer warp 3: the log-decays of key
// rows cl .. cl+3 (cl = 4l; one gate per head is repeated) and the write
// strength.  From the caller (g, beta), or - device gates - from the layer's
// a/b rows: the loads of a (four rows, or the head's one row) and b, which
// are summed and transformed when the record is built.
struct GateLoads {
    float4 g4;      // caller's log-decays
    float bv;       // caller's beta
    float4 pa[PV];  // a partials
    float4 sa;      // a row scales
    float pb[PV], sb, A;
    int nsa, nsb;
};

__device__ __forceinline__ int gate_a_row(const StreamParams &p, int h, int cl) {
    return p.in_rows + h * p.gw + (p.gw == 1 ? 0 : cl);
}
__device__ __forceinline__ int gate_b_row(const StreamParams &p, int h) { return p.in_rows + p.n_v * p.gw + h; }
__device__ __forceinline__ float4 splat(float v) { return make_float4(v, v, v, v); }

// the loads the in_proj does not feed
__device__ __forceinline__ void load_gates_fixed(const StreamParams &p, int h, int item, int cl, GateLoads &G) {
    if (!p.dev_gates) {
        G.g4 = p.gw == 1 ? splat(ld_cg(p.g + item)) : ld_cg4(p.g + (size_t)item * D + cl);
        G.bv = ld_cg(p.beta + item);
        return;
    }
    const int ca = gate_a_row(p, h, cl);
    G.sa = p.gw == 1 ? splat(ld_nc(p.s_in + ca)) : ld_nc4(p.s_in + ca);
    G.sb = ld_nc(p.s_in + gate_b_row(p, h));
    G.A = ld_nc(p.gate_A + h);
}
// the in_proj's partials of the gate rows
__device__ __forceinline__ void load_gates_part(const StreamParams &p, int b, int h, int cl, GateLoads &G) {
    if (!p.dev_gates) return;
    const int ca = gate_a_row(p, h, cl), cb = gate_b_row(p, h);
    G.nsa = ld_cg_s32(p.nseg_in + (b >> 6) * p.MT + (ca >> 7));
    G.nsb = ld_cg_s32(p.nseg_in + (b >> 6) * p.MT + (cb >> 7));
    const float *pa = row_partials(p, b, ca), *pb = row_partials(p, b, cb);
#pragma unroll
    for (int k = 0; k < PV; ++k) {  // slots past max_seg fall back to slot 0
        const size_t o = (size_t)(k < p.max_seg ? k : 0) * (64 * D);
        G.pa[k] = p.gw == 1 ? splat(ld_cg(pa + o)) : ld_cg4(pa + o);
        G.pb[k] = ld_cg(pb + o);
    }
}
// the item's log-decays (four key rows) and beta
__device__ __forceinline__ float4 gate_values(const StreamParams &p, int b, int h, int cl, const GateLoads &G,
                                              float &beta) {
    if (!p.dev_gates) {
        beta = G.bv;
        return G.g4;
    }
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    float bs = 0.f;
#pragma unroll
    for (int k = 0; k < PV; ++k) {
        if (k < G.nsa) add4(a, G.pa[k]);
        if (k < G.nsb) bs += G.pb[k];
    }
    if (G.nsa > PV || G.nsb > PV) {
        const float *pa = row_partials(p, b, gate_a_row(p, h, cl)), *pb = row_partials(p, b, gate_b_row(p, h));
        for (int k = PV; k < G.nsa; ++k) add4(a, p.gw == 1 ? splat(__ldcg(pa + (size_t)k * (64 * D))) : ld_cg4(pa + (size_t)k * (64 * D)));
        for (int k = PV; k < G.nsb; ++k) bs += __ldcg(pb + (size_t)k * (64 * D));
    }
    beta = sigmoid_f(G.sb * bs);
    return make_float4(-G.A * softplus_f(G.sa.x * a.x), -G.A * softplus_f(G.sa.y * a.y),
                       -G.A * softplus_f(G.sa.z * a.z), -G.A * softplus_f(G.sa.w * a.w));
}

// Producer warps 0-2: build the conv rows of the record (q^, k^, v) of
// every item of the CTA's walk, one item ahead of the consumers.  Warp `kind` builds
// one row kind (0 q, 1 k, 2 v), lane l channels 4l .. 4l+3 of the head,
// so a q or k norm is one warp's sum.  The loads of item j+1 are issued as
// soon as item j's values are computed (the registers are free again), so
// their latency hides behind the rest of item j.  (A failed wait ends the
// warp's loop on all of its lanes together.)
template <int KC>
__device__ void produce(const StreamParams &p, StreamSmem &sm, int i0, int n_s, int b0, int nseq, int kind,
                        int lane) {
    const int cl = 4 * lane;
    constexpr bool conv = true;
    const bool qk = kind < 2;
    const int base = kind == 0 ? 0 : kind == 1 ? p.qk_dim : 2 * p.qk_dim;
    int b = i0 / p.n_v, h = i0 - b * p.n_v, hq = h / p.group;
    int dp = ring_pos(p, sm, b0, nseq, b);
    RowLoads<KC> r;
    // the first item's loads that the in_proj does not feed go out before the wait
    int c = base + (qk ? hq : h) * D + cl;
    load_row_fixed(p, dp, b, c, conv, r);
    pdl_wait();
    load_row_part(p, b, c, r);
    bool reuse = false;  // item j has the q/k head of item j-1
    for (int j = 0;; ++j) {
        const int rb = j & 1;
        c = base + (qk ? hq : h) * D + cl;
        float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
        if (!(qk && reuse)) {
            // v rows belong to one item; q/k rows are written by the q/k head's first value head
            u = conv_silu(p, dp, b, c, row_value(p, b, c, r), kind == 2 || h == hq * p.group, r);
        }

        // item j+1 and its loads
        int nxt;
        if (!__all_sync(0xffffffffu, item_at(sm, i0, n_s, j + 1, nxt))) {
            sm.failed = 1;
            break;
        }
        const int bn = nxt / p.n_v, hn = nxt - bn * p.n_v, hqn = hn / p.group;
        const bool reuse_n = nxt >= 0 && bn == b && hqn == hq;
        int dpn = dp;
        if (nxt >= 0 && !(qk && reuse_n)) {
            const int cn = base + (qk ? hqn : hn) * D + cl;
            dpn = ring_pos(p, sm, b0, nseq, bn);
            load_row_fixed(p, dpn, bn, cn, conv, r);
            load_row_part(p, bn, cn, r);
        }
        float4 outv = u;
        if (qk) {
            if (!reuse) {
                const float ss = warp_sum((u.x * u.x + u.y * u.y) + (u.z * u.z + u.w * u.w));
                const float sc = (1.0f / sqrtf(ss + p.l2_eps)) * (kind == 0 ? p.q_scale : 1.0f);
                outv = make_float4(u.x * sc, u.y * sc, u.z * sc, u.w * sc);
            } else {
                outv = *reinterpret_cast<const float4 *>(&sm.rec[rb ^ 1][kind * D + cl]);
            }
        }
        // record buffer rb is free once the consumers are done with item j-2
        if (!__all_sync(0xffffffffu, j < 2 || mbar_wait(&sm.rec_empty[rb], ((j >> 1) - 1) & 1))) {
            sm.failed = 1;
            break;
        }
        *reinterpret_cast<float4 *>(&sm.rec[rb][kind * D + cl]) = outv;

        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.rec_full[rb]);  // release: the record's writes come first
        if (nxt < 0) break;
        b = bn;
        h = hn;
        hq = hqn;
        dp = dpn;
        reuse = reuse_n;
    }
}

// Producer warp 3: the z rows (silu(z)) and the gates (the decay of each
// key row, the write strength) of every item, one item ahead of the
// consumers, with their loads one item ahead of their use.  Its own loop, so
// that its registers do not add to those of the conv-row warps.
template <int KC>
__device__ void produce_z_gates(const StreamParams &p, StreamSmem &sm, int i0, int n_s, int lane) {
    const int cl = 4 * lane;
    int b = i0 / p.n_v, h = i0 - b * p.n_v;
    RowLoads<KC> r;  // (conv fields unused)
    GateLoads G;
    load_row_fixed(p, 0, b, p.conv_ch + h * D + cl, false, r);
    load_gates_fixed(p, h, i0, cl, G);
    pdl_wait();
    load_row_part(p, b, p.conv_ch + h * D + cl, r);
    load_gates_part(p, b, h, cl, G);
    for (int j = 0;; ++j) {
        const int rb = j & 1;
        const float4 xz = row_value(p, b, p.conv_ch + h * D + cl, r);
        const float4 uz = make_float4(silu_f(xz.x), silu_f(xz.y), silu_f(xz.z), silu_f(xz.w));
        float bj;
        const float4 gj = gate_values(p, b, h, cl, G, bj);
        int nxt;
        if (!__all_sync(0xffffffffu, item_at(sm, i0, n_s, j + 1, nxt))) {
            sm.failed = 1;
            break;
        }
        const int bn = nxt / p.n_v, hn = nxt - bn * p.n_v;
        if (nxt >= 0) {
            load_row_fixed(p, 0, bn, p.conv_ch + hn * D + cl, false, r);
            load_row_part(p, bn, p.conv_ch + hn * D + cl, r);
            load_gates_fixed(p, hn, nxt, cl, G);
            load_gates_part(p, bn, hn, cl, G);
        }
        if (!__all_sync(0xffffffffu, j < 2 || mbar_wait(&sm.rec_empty[rb], ((j >> 1) - 1) & 1))) {
            sm.failed = 1;
            break;
        }
        *reinterpret_cast<float4 *>(&sm.rec[rb][3 * D + cl]) = uz;
        *reinterpret_cast<float4 *>(&sm.rec[rb][4 * D + cl]) = make_float4(expf(gj.x), expf(gj.y), expf(gj.z), expf(gj.w));
        if (lane == 0) sm.beta[rb] = bj;
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.rec_full[rb]);
        if (nxt < 0) break;
        b = bn;
        h = hn;
    }
}

// Consumer warps (t = 0..511): the state update of every item.  Thread t
// holds rows r0 + 16 i (i < 8), columns 4 c4 .. 4 c4 + 3 of the tile.  The
// updated tile goes back into its stage and leaves by one bulk store; the
// stage takes the item STAGES ahead once that store has read it (checked
// during the next item).  The readout's gated RMSNorm is finished by warps
// 4-7 during the next item.  Thread kTma also decides the item of each
// position from 3 on (the CTA's own range, then the pool) two items ahead,
// when it requests that item's tile, and publishes it in the queue.
// Returns the number of tile copies issued.
__device__ int consume(const StreamParams &p, StreamSmem &sm, int i0, int n_s, int t) {
    const int warp = t >> 5, lane = t & 31;
    const int c4 = t % LPR, r0 = t / LPR;
    int issued = n_s < STAGES ? n_s : STAGES;
    int b_prev = 0, h_prev = 0;
    int grab = -1;  // (thread kTma) the pool's answer for the next position to decide
    bool clean = true;
    for (int j = 0;; ++j) {
        // (the queue slot was written two items ago, before a consumer barrier)
        const int item = j < n_s ? i0 + j : j < 3 ? -1 : sm.qitem[(j - 3) & 3];
        if (item < 0) break;
        const int b = item / p.n_v, h = item - b * p.n_v;
        const int st = j % STAGES, rb = j & 1;
        bool ok = mbar_wait(&sm.full[st], (j / STAGES) & 1);
        float *tile = sm.tile[st];
        float4 s[NP];
#pragma unroll
        for (int i = 0; i < NP; ++i) s[i] = *reinterpret_cast<const float4 *>(tile + (r0 + i * RPP) * D + c4 * 4);
        ok = ok && mbar_wait(&sm.rec_full[rb], (j >> 1) & 1);
        const float *rq = sm.rec[rb], *rk = rq + D, *rv = rq + 2 * D;
        const float bt = sm.beta[rb];
        const float *reg = rq + 4 * D;  // exp(g) of each key row
        float *red = &sm.red[rb][0][0];

        // decay, then what the decayed state predicts for k
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const float kr = rk[r0 + i * RPP], eg = reg[r0 + i * RPP];
            s[i].x *= eg;
            s[i].y *= eg;
            s[i].z *= eg;
            s[i].w *= eg;
            acc.x = fmaf(s[i].x, kr, acc.x);
            acc.y = fmaf(s[i].y, kr, acc.y);
            acc.z = fmaf(s[i].z, kr, acc.z);
            acc.w = fmaf(s[i].w, kr, acc.w);
        }
        *reinterpret_cast<float4 *>(red + r0 * D + c4 * 4) = acc;
        if (!bar_and(kBarCons, NC, ok)) {  // no consumer gives up on a wait alone
            sm.failed = 1;
            clean = false;
            break;
        }
        if (t == kTma && j >= 1) {
            // position j+2: its item, published for the producers, and its
            // tile into the stage of item j-1 (free once its bulk store has
            // read it)
            const int pos = j - 1 + STAGES;
            int nxt = -1;
            if (pos < n_s)
                nxt = i0 + pos;
            else if (grab >= 0 && grab < p.pool_n)
                nxt = p.pool_base + grab;
            sm.qitem[(pos - 3) & 3] = nxt;
            mbar_arrive(&sm.qfull[(pos - 3) & 3]);
            if (nxt >= 0) {
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                load_tile(sm, (j - 1) % STAGES, p, nxt);
                issued = pos + 1;
            }
            // ask the pool for position pos+1 now; the answer is read an item later
            grab = (p.pool != nullptr && nxt >= 0 && pos + 1 >= n_s) ? atomicAdd(p.pool, 1) : -1;
        }
        if (t < D) {
            // delta against the decayed state
            float kv = 0.f;
#pragma unroll
            for (int r = 0; r < RPP; ++r) kv += red[r * D + t];
            sm.delta[t] = bt * (rv[t] - kv);
        } else if (t < 2 * D && j >= 1) {
            store_norm(p, sm, sm.o_prev[t - D], sm.zw_prev[t - D], b_prev, h_prev, t - D);
        }
        bar_sync(kBarCons, NC);
        // write-back S += k delta^T into the stage, and the readout partials
        // over the updated state
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
        *reinterpret_cast<float4 *>(red + r0 * D + c4 * 4) = acc;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // tile writes -> bulk store
        bar_sync(kBarCons, NC);
        if (t == kTma) {
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                             p.S + (size_t)item * (D * D)),
                         "r"(smem_u32(tile)), "r"(kTileBytes)
                         : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        }
        if (t < D) {
            // readout o = S^T q over the updated state; its norm waits for the next item
            float o = 0.f;
#pragma unroll
            for (int r = 0; r < RPP; ++r) o += red[r * D + t];
            const float sq = warp_sum(o * o);
            if (lane == 0) sm.ssq_o[warp] = sq;
            sm.o_prev[t] = o;
            sm.zw_prev[t] = sm.wn[t] * rq[3 * D + t];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.rec_empty[rb]);
        b_prev = b;
        h_prev = h;
    }
    if (clean) {  // (uniform) the last item's norm
        bar_sync(kBarCons, NC);
        if (t >= D && t < 2 * D) store_norm(p, sm, sm.o_prev[t - D], sm.zw_prev[t - D], b_prev, h_prev, t - D);
    }
    return issued;
}

// Warm-up of L2 by the first pf_ctas CTAs.  The tensor-core in_proj leaves
// those SMs free, so these CTAs start while it runs, with nothing to do until
// it completes; the other CTAs start only as the in_proj's CTAs leave, a few
// microseconds before its end, and their first tile copies would come from
// HBM late.  So these CTAs pull the first kWarmTiles tiles of every other
// CTA into L2 (one prefetch per 128-byte line; the tiles of position 0 of all
// CTAs first).
__device__ void warm_l2(const StreamParams &p, int t) {
    const int G = gridDim.x, E = p.pf_ctas, late = G - E;
    for (int L = blockIdx.x; L < late * kWarmTiles; L += E) {
        const int pos = L / late, c = E + L % late;
        if (pos >= p.n_static) continue;
        const char *tile = reinterpret_cast<const char *>(p.S + (size_t)(c * p.n_static + pos) * (D * D));
        for (int off = t * 128; off < (int)kTileBytes; off += NT * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(tile + off));
    }
}

template <int KC>
__global__ void __launch_bounds__(NT, 1) dn_core_stream_kernel(const StreamParams p) {
    extern __shared__ uint8_t smem_raw[];
    StreamSmem &sm = *reinterpret_cast<StreamSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    // the CTA's own range [i0, i0 + n_s): n_s >= 1 (the grid has at most one
    // CTA per item; with a pool, n_s >= 4)
    int i0, n_s;
    if (p.pool != nullptr) {
        i0 = (int)blockIdx.x * p.n_static;
        n_s = p.n_static;
    } else {
        i0 = (int)(((unsigned)blockIdx.x * (unsigned)p.items) / gridDim.x);
        n_s = (int)(((unsigned)(blockIdx.x + 1) * (unsigned)p.items) / gridDim.x) - i0;
    }
    const int b0 = i0 / p.n_v;
    const int nseq = (i0 + n_s - 1) / p.n_v - b0 + 1;

    if (t == 0) {
        for (int s = 0; s < STAGES; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&sm.full[s])));
        for (int r = 0; r < 2; ++r) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&sm.rec_full[r])), "r"(NPW));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&sm.rec_empty[r])),
                         "r"(NC / 32));
        }
        for (int q = 0; q < 4; ++q)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&sm.qfull[q])));
        sm.failed = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // the state is not written by the in_proj kernel
        for (int j = 0; j < STAGES && j < n_s; ++j) load_tile(sm, j, p, i0 + j);
    }
    // the norm weights and the sequences' ring positions (advanced by the
    // previous step's last kernel, which has completed)
    if (t < D) sm.wn[t] = p.w_norm[t];
    for (int i = t; i < nseq; i += NT) sm.dpos[i] = p.rpos[2 * (b0 + i)];
    __syncthreads();

    if ((int)blockIdx.x < p.pf_ctas) warm_l2(p, t);
    int issued = 0;
    if (warp < NC / 32) {
        // (consumers read nothing the in_proj writes; the wait keeps
        // completion transitive, and the pool counter, zeroed by the previous
        // step's last kernel, is only asked after it)
        pdl_wait();
        if (t == 0) pdl_trigger();
        issued = consume(p, sm, i0, n_s, t);
    } else if (warp < NC / 32 + 3) {
        produce<KC>(p, sm, i0, n_s, b0, nseq, warp - NC / 32, lane);
    } else {
        produce_z_gates<KC>(p, sm, i0, n_s, lane);
    }
    __syncthreads();
    if (t == kTma) {
        asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        if (sm.failed) atomicOr(p.err, 1);
        // let any tile copy still in flight land before the CTA exits
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
        cudaError_t r = cudaFuncSetAttribute(dn_core_stream_kernel<KC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        // 640 threads at up to 96 registers and ~216 KB: one CTA must fit an SM
        int fit = 0;
        if (r == cudaSuccess) r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, dn_core_stream_kernel<KC>, NT, smem);
        if (r == cudaSuccess && fit < 1) r = cudaErrorLaunchOutOfResources;
        return r;
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
    const GemmPlan gp = plan_tc_gemm(d.proj_rows, plan_k(d, d.hidden, B), B);
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
    p.gw = d.gw;
    p.dev_gates = d.dev_gates;
    p.in_rows = d.in_rows;
    p.gate_A = L.gate_A;
    const int grid = std::min(num_sms(), p.items);
    p.pool = nullptr;
    p.n_static = p.pool_base = p.pool_n = p.pf_ctas = 0;
    if (L.pool != nullptr && p.items / grid >= kPoolPerCta + 4) {
        p.pool = L.pool;
        p.n_static = p.items / grid - kPoolPerCta;
        p.pool_base = grid * p.n_static;
        p.pool_n = p.items - p.pool_base;
        // the SMs the tensor-core in_proj leaves free host the first CTAs
        if (tc && grid == num_sms() && gp.G < grid) p.pf_ctas = grid - gp.G;
    }
    switch (d.conv_k) {
        case 2: return launch_kc<2>(p, st);
        case 3: return launch_kc<3>(p, st);
        case 4: return launch_kc<4>(p, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dn
