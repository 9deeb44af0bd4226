// Prompt processing: S > 1 tokens of each sequence through one layer, with
// the result of S decode steps (the page "qwen36: run the DeltaNet layer end
// to end on the card (Q36_DN_GPU=1)", section "What the PR does", keeps a
// prompt on its batched CPU path; here it runs on the card).
//
// The prompt goes through in blocks of up to kPrefillCols token columns (nb
// sequences x T tokens).  Per block:
//   1. the block's x rows are gathered, and the in_proj runs once over all
//      of its columns: a real GEMM, on the tensor cores (the decode kernels
//      with the columns as the batch; the CUDA-core GEMV for one column);
//   2. one kernel scales and sums the in_proj partials into xin;
//   3. one kernel per (column, head) runs the causal conv over the tokens
//      (the first K-1 reach back into the ring), SiLU, the q/k L2 norms and
//      the query scale, silu(z) and the gates (the caller's, or from the
//      layer's a/b rows), written head-major and token-contiguous;
//   4. one kernel moves the ring to the block's last K-1 inputs
//      (for 128-wide heads and blocks of several sequences 2-4 are one
//      kernel per (row tile, sequence), which reads each partial once and
//      keeps the conv window in registers);
//   5. the recurrence kernel: one block per (column slice, value head,
//      sequence) holds its dk x DJ slice of the state in registers for all T
//      tokens (read once and written once per block instead of once per
//      token) and walks them in order: decay, delta against the decayed
//      state, write-back, readout over the updated state; the next token's
//      inputs are loaded while the current one is computed (for 128-wide
//      keys with one decay per head: the chunked form of the same
//      recurrence, 5' below; for 128 x 128 heads, when the block holds a
//      (head, sequence) pair per SM, on the tensor cores, 5'' below);
//   6. the gated RMSNorm of every readout, written as the out_proj's input;
//   7. the out_proj over all columns, its reduction writing each token's row
//      of the caller's output and advancing the ring positions by T.
// Every reduction runs in a fixed order, so results do not depend on
// scheduling.
#include <cuda_bf16.h>

#include <algorithm>
#include <atomic>

#include "dn_device.cuh"
#include "dn_internal.cuh"
#include "dn_sched.cuh"

namespace dn {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float silu_f(float a) { return a / (1.0f + expf(-a)); }
__device__ __forceinline__ float softplus_f(float a) { return fmaxf(a, 0.f) + log1pf(expf(-fabsf(a))); }
__device__ __forceinline__ float sigmoid_f(float b) { return 1.0f / (1.0f + expf(-b)); }

struct Geo {
    int b0, nb, t0, T, S, cols;
};

constexpr int kChunk = 32;  // tokens per step of the chunked kernels

// 1. xg[j] = x[(b0 + j / T) * S + t0 + j % T]
__global__ void gather_rows_kernel(const float *__restrict__ x, float *__restrict__ xg, int hidden, Geo g) {
    const int j = blockIdx.y;
    const float4 *src = reinterpret_cast<const float4 *>(
        x + ((size_t)(g.b0 + j / g.T) * g.S + g.t0 + j % g.T) * hidden);
    float4 *dst = reinterpret_cast<float4 *>(xg + (size_t)j * hidden);
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < hidden / 4; i += gridDim.x * blockDim.x) dst[i] = src[i];
}

// 2. xin[j][c] = s[c] * (column j's segment partials of row c, in slot order)
__global__ void sum_rows_kernel(const float *__restrict__ part, const int *__restrict__ nseg,
                                const float *__restrict__ s, float *__restrict__ xin, int rows, int MT,
                                int max_seg) {
    pdl_wait();  // the projection before it
    const int j = blockIdx.y;
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= rows) return;
    const int tile = (j >> 6) * MT + (c >> 7);
    const int ns = nseg[tile];
    const float *pp = part + (size_t)tile * max_seg * (64 * 128) + (j & 63) * 128 + (c & 127);
    float acc = 0.f;
    for (int k = 0; k < ns; ++k) acc += __ldcg(pp + (size_t)k * (64 * 128));
    xin[(size_t)j * rows + c] = s[c] * acc;
}

struct PrepParams {
    const float *xin;      // [cols][proj_rows]
    const float *ring;     // [max_batch][K][conv_ch]
    const int32_t *rpos;   // [max_batch][2]
    const float *wconv_t;  // [K][conv_ch]
    const float *g, *beta; // caller's [batch][S][n_v][gw], [batch][S][n_v] (host gates)
    const float *gate_A;   // [n_v] (device gates)
    float *qn, *kn, *vv, *zs, *gg, *bb;
    Geo geo;
    int K, conv_ch, qk_dim, in_rows, proj_rows, n_qk, n_v, dk, dv, gw, dev_gates;
    float l2_eps, q_scale;
};

// the conv input of channel c at block token tau of local sequence b: a block
// column (tau >= 0) or the ring's history (tau < 0; history index tau + K - 1)
__device__ __forceinline__ float conv_in(const PrepParams &p, int b, int tau, int c, int dpos) {
    if (tau >= 0) return p.xin[(size_t)(b * p.geo.T + tau) * p.proj_rows + c];
    int slot = dpos + tau + p.K - 1;
    if (slot >= p.K) slot -= p.K;
    return p.ring[((size_t)(p.geo.b0 + b) * p.K + slot) * p.conv_ch + c];
}

__device__ __forceinline__ float conv_silu_at(const PrepParams &p, int b, int t, int c, int dpos) {
    float acc = 0.f;
    for (int m = 0; m < p.K; ++m)  // tap m meets token t - (K - 1) + m; tap K-1 the current one
        acc = fmaf(p.wconv_t[(size_t)m * p.conv_ch + c], conv_in(p, b, t - (p.K - 1) + m, c, dpos), acc);
    return silu_f(acc);
}

__device__ __forceinline__ float block_sum(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) t += red[i];  // fixed order
    __syncthreads();
    return t;
}

// 3. grid (n_qk + n_v, cols): block x < n_qk is q/k head x of column j;
// the others value head x - n_qk (v, silu(z), gates).  dk, dv <= 256 = threads.
__global__ void __launch_bounds__(kThreads) prep_kernel(const PrepParams p) {
    __shared__ float red[kThreads / 32];
    const int j = blockIdx.y, b = j / p.geo.T, t = j % p.geo.T;
    const int dpos = p.rpos[2 * (p.geo.b0 + b)];
    const int i = threadIdx.x;
    const int T = p.geo.T;
    if ((int)blockIdx.x < p.n_qk) {
        const int hq = blockIdx.x;
        float uq = 0.f, uk = 0.f;
        if (i < p.dk) {
            uq = conv_silu_at(p, b, t, hq * p.dk + i, dpos);
            uk = conv_silu_at(p, b, t, p.qk_dim + hq * p.dk + i, dpos);
        }
        const float sq = block_sum(uq * uq, red), sk = block_sum(uk * uk, red);
        if (i < p.dk) {
            const size_t o = (((size_t)b * p.n_qk + hq) * T + t) * p.dk + i;
            p.qn[o] = uq * (1.0f / sqrtf(sq + p.l2_eps)) * p.q_scale;
            p.kn[o] = uk * (1.0f / sqrtf(sk + p.l2_eps));
        }
        return;
    }
    const int h = blockIdx.x - p.n_qk;
    const size_t hv = ((size_t)b * p.n_v + h) * T + t;
    if (i < p.dv) {
        p.vv[hv * p.dv + i] = conv_silu_at(p, b, t, 2 * p.qk_dim + h * p.dv + i, dpos);
        p.zs[hv * p.dv + i] = silu_f(p.xin[(size_t)j * p.proj_rows + p.conv_ch + h * p.dv + i]);
    }
    const size_t tok = (size_t)(p.geo.b0 + b) * p.geo.S + p.geo.t0 + t;  // the caller's row
    for (int k = i; k < p.gw; k += kThreads) {
        p.gg[hv * p.gw + k] =
            p.dev_gates ? -p.gate_A[h] * softplus_f(p.xin[(size_t)j * p.proj_rows + p.in_rows + h * p.gw + k])
                        : p.g[(tok * p.n_v + h) * p.gw + k];
    }
    if (i == 0)
        p.bb[hv] = p.dev_gates ? sigmoid_f(p.xin[(size_t)j * p.proj_rows + p.in_rows + p.n_v * p.gw + h])
                               : p.beta[tok * p.n_v + h];
}

// 4. the ring after the block: the last K-1 of (history ++ the block's
// inputs), at the slots the advanced ring position (dpos + T) names.  One
// thread per (sequence, channel) reads everything before it writes.
__global__ void ring_block_kernel(const float *__restrict__ xin, float *__restrict__ ring,
                                  const int32_t *__restrict__ rpos, Geo g, int K, int conv_ch, int proj_rows) {
    const int b = blockIdx.y;
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= conv_ch) return;
    const int dpos = rpos[2 * (g.b0 + b)];
    float *rb = ring + (size_t)(g.b0 + b) * K * conv_ch + c;
    float hist[7], nw[7];  // K <= 8
    for (int m = 0; m < K - 1; ++m) {
        int slot = dpos + m;
        if (slot >= K) slot -= K;
        hist[m] = rb[(size_t)slot * conv_ch];
    }
    for (int m = 0; m < K - 1; ++m) {  // combined index T + m of history (K-1) ++ block (T)
        const int ci = g.T + m;
        nw[m] = ci < K - 1 ? hist[ci] : xin[(size_t)(b * g.T + ci - (K - 1)) * proj_rows + c];
    }
    const int dn = (dpos + g.T) % K;
    for (int m = 0; m < K - 1; ++m) {
        int slot = dn + m;
        if (slot >= K) slot -= K;
        rb[(size_t)slot * conv_ch] = nw[m];
    }
}

// 2-4 fused, for 128-wide heads (one in_proj row tile = one head).  One CTA
// of 128 threads per (row tile, sequence of the block); thread c takes row
// 128 mt + c through the block's T tokens, 32 at a time: the in_proj output
// (segment partials in slot order, times the row scale) and then, by the
// row's kind,
//   q, k rows:  conv over the ring's history and the block's inputs (the
//               window in registers), SiLU, the L2 norm over the tile (a
//               fixed-order sum through shared memory), the query scale;
//   v rows:     conv, SiLU (and the v head's CTA copies the caller's gates);
//   z rows:     SiLU;
//   gate rows:  (device gates) -A softplus(a), sigmoid(b);
// and at the end the conv rows' last K-1 inputs go into the ring, whose
// position moves with the reduction at the block's end.  Each partial and
// ring value is read once, and no scaled-row buffer goes through memory.
struct TileParams {
    const float *part;     // in_proj segment partials, their counts, the row scales
    const int *nseg;
    const float *s_in;
    float *ring;
    const int32_t *rpos;
    const float *wconv_t;
    const float *g, *beta;  // caller's gates (host gates)
    const float *gate_A;    // [n_v] (device gates)
    float *qn, *kn, *vv, *zs, *gg, *bb;
    Geo geo;
    int MT, max_seg, conv_ch, qk_dim, in_rows, proj_rows, n_qk, n_v, gw, dev_gates;
    float l2_eps, q_scale;
};

constexpr int kTileSlots = 4;  // partial slots loaded ahead (2 to 5 segments per tile on the 35B shape)

template <int K>
__global__ void __launch_bounds__(128) prep_tile_kernel(const TileParams p) {
    constexpr int D = 128;
    __shared__ float red[D][kChunk + 1];
    __shared__ float inv[kChunk];
    const int mt = blockIdx.x, b = blockIdx.y, c = threadIdx.x;
    const int row = mt * D + c, T = p.geo.T, sb = p.geo.b0 + b;
    const bool active = row < p.proj_rows;
    const bool conv = row < p.conv_ch;  // (q, k, v: uniform over the tile)
    const bool isq = row < p.qk_dim, isk = !isq && row < 2 * p.qk_dim;
    const float sc = active ? p.s_in[row] : 0.f;
    float w[K], prev[K - 1];  // taps; the last K-1 inputs before the current 32 tokens
    int dpos = 0;
#pragma unroll
    for (int m = 0; m < K; ++m) w[m] = 0.f;
#pragma unroll
    for (int m = 0; m < K - 1; ++m) prev[m] = 0.f;
    if (conv) {
        dpos = p.rpos[2 * sb];
#pragma unroll
        for (int m = 0; m < K; ++m) w[m] = p.wconv_t[(size_t)m * p.conv_ch + row];
#pragma unroll
        for (int m = 0; m < K - 1; ++m) {  // oldest first
            int slot = dpos + m;
            if (slot >= K) slot -= K;
            prev[m] = p.ring[((size_t)sb * K + slot) * p.conv_ch + row];
        }
    }
    for (int s0 = 0; s0 < T; s0 += kChunk) {
        const int nt = min(kChunk, T - s0);
        float x[kChunk], u[kChunk];
        // the partials of 16 tokens at a time: the first kTileSlots slots of
        // every token requested before any is summed (from clamped, always
        // valid addresses: tokens past nt take the last column, slots past
        // max_seg slot 0), the rest read on the spot
#pragma unroll
        for (int g0 = 0; g0 < kChunk; g0 += 16) {
            float pv[16][kTileSlots];
            int nsv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int j = b * T + s0 + min(g0 + i, nt - 1);  // block column
                const int tile = (j >> 6) * p.MT + mt;
                nsv[i] = p.nseg[tile];
                const float *pp = p.part + ((size_t)tile * p.max_seg * 64 + (j & 63)) * D + c;
#pragma unroll
                for (int k = 0; k < kTileSlots; ++k) pv[i][k] = __ldcg(pp + (size_t)(k < p.max_seg ? k : 0) * (64 * D));
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int tt = g0 + i;
                float acc = 0.f;
#pragma unroll
                for (int k = 0; k < kTileSlots; ++k)
                    if (k < nsv[i]) acc += pv[i][k];
                if (nsv[i] > kTileSlots) {
                    const int j = b * T + s0 + min(tt, nt - 1);
                    const int tile = (j >> 6) * p.MT + mt;
                    const float *pp = p.part + ((size_t)tile * p.max_seg * 64 + (j & 63)) * D + c;
                    for (int k = kTileSlots; k < nsv[i]; ++k) acc += __ldcg(pp + (size_t)k * (64 * D));
                }
                x[tt] = (active && tt < nt) ? sc * acc : 0.f;
            }
        }
        if (conv) {
#pragma unroll
            for (int tt = 0; tt < kChunk; ++tt) {
                float a = 0.f;
#pragma unroll
                for (int m = 0; m < K; ++m) {  // tap m meets input tt - (K - 1) + m; tap K-1 the current one
                    const int ti = tt - (K - 1) + m;
                    a = fmaf(w[m], ti >= 0 ? x[ti] : prev[ti + K - 1], a);
                }
                u[tt] = silu_f(a);
            }
            // the window for the next tokens: the last K-1 of (prev ++ x[0, nt)),
            // slid one input at a time (fixed register indices)
#pragma unroll
            for (int tt = 0; tt < kChunk; ++tt) {
                if (tt < nt) {
#pragma unroll
                    for (int m = 0; m < K - 2; ++m) prev[m] = prev[m + 1];
                    prev[K - 2] = x[tt];
                }
            }
        }
        if (isq || isk) {  // the head's L2 norm per token
#pragma unroll
            for (int tt = 0; tt < kChunk; ++tt) red[c][tt] = u[tt] * u[tt];
            __syncthreads();
            if (c < kChunk) {
                float ss = 0.f;
                for (int r = 0; r < D; ++r) ss += red[r][c];
                inv[c] = (1.0f / sqrtf(ss + p.l2_eps)) * (isq ? p.q_scale : 1.0f);
            }
            __syncthreads();
            const int hq = isq ? mt : mt - p.n_qk;
            float *dst = (isq ? p.qn : p.kn) + (((size_t)b * p.n_qk + hq) * T + s0) * D + c;
#pragma unroll
            for (int tt = 0; tt < kChunk; ++tt)
                if (tt < nt) dst[(size_t)tt * D] = u[tt] * inv[tt];
            __syncthreads();  // red and inv are taken again for the next tokens
        } else if (conv) {  // v
            const int h = mt - 2 * p.n_qk;
            float *dst = p.vv + (((size_t)b * p.n_v + h) * T + s0) * D + c;
#pragma unroll
            for (int tt = 0; tt < kChunk; ++tt)
                if (tt < nt) dst[(size_t)tt * D] = u[tt];
            if (!p.dev_gates) {  // the caller's gates of this head: (token, key channel) per thread
                for (int idx = c; idx < nt * p.gw; idx += D) {
                    const int tt = idx / p.gw, k = idx - tt * p.gw;
                    const size_t tok = (size_t)sb * p.geo.S + p.geo.t0 + s0 + tt;  // the caller's row
                    const size_t hv = ((size_t)b * p.n_v + h) * T + s0 + tt;
                    p.gg[hv * p.gw + k] = p.g[(tok * p.n_v + h) * p.gw + k];
                    if (k == 0) p.bb[hv] = p.beta[tok * p.n_v + h];
                }
            }
        } else if (row < p.in_rows) {  // z
            const int h = (row - p.conv_ch) / D;
            float *dst = p.zs + (((size_t)b * p.n_v + h) * T + s0) * D + c;
#pragma unroll
            for (int tt = 0; tt < kChunk; ++tt)
                if (tt < nt) dst[(size_t)tt * D] = silu_f(x[tt]);
        } else if (active) {  // the a/b gate rows (device gates)
            const int r = row - p.in_rows;
            const bool is_a = r < p.n_v * p.gw;
            const int h = is_a ? r / p.gw : r - p.n_v * p.gw, k = is_a ? r % p.gw : 0;
#pragma unroll
            for (int tt = 0; tt < kChunk; ++tt) {
                if (tt < nt) {
                    const size_t hv = ((size_t)b * p.n_v + h) * T + s0 + tt;
                    if (is_a)
                        p.gg[hv * p.gw + k] = -p.gate_A[h] * softplus_f(x[tt]);
                    else
                        p.bb[hv] = sigmoid_f(x[tt]);
                }
            }
        }
    }
    if (conv) {  // the ring after the block: its last K-1 inputs, at the advanced slots
        int slot = (dpos + T) % K;
#pragma unroll
        for (int m = 0; m < K - 1; ++m) {
            p.ring[((size_t)sb * K + slot) * p.conv_ch + row] = prev[m];
            if (++slot == K) slot = 0;
        }
    }
}

// 5. the recurrence over the block's T tokens for one column slice of one
// value head of one sequence: the dk x 32 slice of the state lives in
// registers (thread: rows r0 + 32 i, columns 4 c4 .. 4 c4 + 3).
constexpr int DJ = 32;

struct RecParams {
    float *S;  // layer state [max_batch][n_v][dk][dv]
    const float *qn, *kn, *vv, *gg, *bb;
    float *o;
    Geo geo;
    int n_v, n_qk, group, dv, gw;
    int *err;  // set when a bounded wait gives up
};

template <int DK>
__global__ void __launch_bounds__(kThreads, 2) recur_kernel(const RecParams p) {
    constexpr int LPR = DJ / 4;          // 8 lanes across a row of the slice
    constexpr int RPP = kThreads / LPR;  // 32 rows per pass
    constexpr int NP = DK / RPP;         // float4 of the state per thread
    static_assert(NP >= 1 && DK % RPP == 0, "tile");
    __shared__ __align__(16) float red[2][RPP][DJ];
    __shared__ __align__(16) float delta_s[DJ];

    const int tid = threadIdx.x;
    const int jc = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int hq = h / p.group, col0 = jc * DJ, T = p.geo.T;
    const int c4 = tid % LPR, r0 = tid / LPR;
    float *Sh = p.S + ((size_t)(p.geo.b0 + b) * p.n_v + h) * DK * p.dv + col0 + c4 * 4;
    float4 s[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i) s[i] = *reinterpret_cast<const float4 *>(Sh + (size_t)(r0 + i * RPP) * p.dv);

    const float *qb = p.qn + ((size_t)b * p.n_qk + hq) * T * DK;
    const float *kb = p.kn + ((size_t)b * p.n_qk + hq) * T * DK;
    const size_t hv = ((size_t)b * p.n_v + h) * T;
    // token t's inputs for this thread: its rows of k^, q^ and the decay,
    // and (threads < 32) its column of v and the write strength
    float kr[NP], qr[NP], eg[NP], vj = 0.f, bt = 0.f;
    float nkr[NP], nqr[NP], neg[NP], nvj = 0.f, nbt = 0.f;
    auto load = [&](int t, float *k_, float *q_, float *e_, float &v_, float &b_) {
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const int r = r0 + i * RPP;
            k_[i] = kb[(size_t)t * DK + r];
            q_[i] = qb[(size_t)t * DK + r];
            e_[i] = p.gg[(hv + t) * p.gw + (p.gw == 1 ? 0 : r)];
        }
        if (tid < DJ) {
            v_ = p.vv[(hv + t) * p.dv + col0 + tid];
            b_ = p.bb[hv + t];
        }
    };
    load(0, nkr, nqr, neg, nvj, nbt);
    for (int t = 0; t < T; ++t) {
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            kr[i] = nkr[i];
            qr[i] = nqr[i];
            eg[i] = expf(neg[i]);
        }
        vj = nvj;
        bt = nbt;
        if (t + 1 < T) load(t + 1, nkr, nqr, neg, nvj, nbt);
        // decay, then what the decayed state predicts for k
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            s[i].x *= eg[i];
            s[i].y *= eg[i];
            s[i].z *= eg[i];
            s[i].w *= eg[i];
            acc.x = fmaf(s[i].x, kr[i], acc.x);
            acc.y = fmaf(s[i].y, kr[i], acc.y);
            acc.z = fmaf(s[i].z, kr[i], acc.z);
            acc.w = fmaf(s[i].w, kr[i], acc.w);
        }
        *reinterpret_cast<float4 *>(&red[0][r0][c4 * 4]) = acc;
        __syncthreads();
        if (tid < DJ) {  // delta against the decayed state
            float kv = 0.f;
#pragma unroll 8
            for (int r = 0; r < RPP; ++r) kv += red[0][r][tid];
            delta_s[tid] = bt * (vj - kv);
        }
        __syncthreads();
        // write-back and the readout partials over the updated state
        const float4 d4 = *reinterpret_cast<const float4 *>(&delta_s[c4 * 4]);
        acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            s[i].x = fmaf(kr[i], d4.x, s[i].x);
            s[i].y = fmaf(kr[i], d4.y, s[i].y);
            s[i].z = fmaf(kr[i], d4.z, s[i].z);
            s[i].w = fmaf(kr[i], d4.w, s[i].w);
            acc.x = fmaf(s[i].x, qr[i], acc.x);
            acc.y = fmaf(s[i].y, qr[i], acc.y);
            acc.z = fmaf(s[i].z, qr[i], acc.z);
            acc.w = fmaf(s[i].w, qr[i], acc.w);
        }
        *reinterpret_cast<float4 *>(&red[1][r0][c4 * 4]) = acc;
        __syncthreads();
        if (tid < DJ) {
            float o = 0.f;
#pragma unroll 8
            for (int r = 0; r < RPP; ++r) o += red[1][r][tid];
            p.o[(hv + t) * p.dv + col0 + tid] = o;
        }
    }
#pragma unroll
    for (int i = 0; i < NP; ++i) *reinterpret_cast<float4 *>(Sh + (size_t)(r0 + i * RPP) * p.dv) = s[i];
}

// 5'. The same recurrence in chunks of kChunk tokens (dk = 128, one decay per
// head): per chunk, with S0 the slice's state at the chunk's start, the
// cumulative log-decay G_t of its tokens and gamma_t = exp(G_t), the delta
// rule unrolls to
//   u_t = beta_t (v_t - gamma_t S0^T k_t - sum_{s<t} exp(G_t - G_s) (k_t.k_s) u_s)
//   o_t = gamma_t S0^T q_t + sum_{s<=t} exp(G_t - G_s) (q_t.k_s) u_s
//   S   = gamma_n S0 + sum_t exp(G_n - G_t) k_t u_t^T
// (u_t is the token's delta, beta_t (v_t - k_t^T S'_t) of the decayed state
// S'_t; substitute S_{t-1} unrolled from S0 and collect terms).  The k.k and
// q.k products, S0^T k and S0^T q are dense products over the chunk, the
// lower-triangular solve for u runs in one warp (lane = column), and the
// state takes the chunk's outer products in registers: the state is read
// from shared memory a few times per chunk
// instead of reduced across the CTA at every token.  Exact algebra of the
// token recurrence; the rounding differs from it (fp32 throughout).
constexpr int kKP = 128 + 4;  // padded k / q rows: four rows a warp reads fall in distinct banks

struct ChunkSmem {
    float K[kChunk][kKP];
    float Q[kChunk][kKP];
    float S0[128][DJ];
    float V[kChunk][DJ];
    float P[kChunk][DJ];      // S0^T k_t (the slice's columns)
    float U[kChunk][DJ];
    float L[kChunk][kChunk];  // exp(G_t - G_s) k_t.k_s, s < t
    float M[kChunk][kChunk];  // exp(G_t - G_s) q_t.k_s, s <= t
    float G[kChunk], gam[kChunk], wn[kChunk], beta[kChunk];
};

__device__ __forceinline__ float dot4(const float4 a, const float4 b) {
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}
__device__ __forceinline__ void fma4(float4 &acc, float a, const float4 b) {
    acc.x = fmaf(a, b.x, acc.x);
    acc.y = fmaf(a, b.y, acc.y);
    acc.z = fmaf(a, b.z, acc.z);
    acc.w = fmaf(a, b.w, acc.w);
}

// grid (dv / DJ, n_v, nb); thread (r0, c4) = (tid / 8, tid % 8) holds rows
// r0 + 32 i (i < 4), columns 4 c4 .. 4 c4 + 3 of the slice's state; thread
// (tt, cq) (the same numbers) forms token tt's products for columns 4 cq ..
__global__ void __launch_bounds__(kThreads, 2) recur_chunk_kernel(const RecParams p) {
    constexpr int DK = 128;
    extern __shared__ __align__(16) uint8_t chunk_smem[];
    ChunkSmem &cs = *reinterpret_cast<ChunkSmem *>(chunk_smem);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int jc = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int hq = h / p.group, col0 = jc * DJ, T = p.geo.T;
    const int c4 = tid & 7, r0 = tid >> 3;
    const int tt = r0, cq = c4;
    float *Sh = p.S + ((size_t)(p.geo.b0 + b) * p.n_v + h) * DK * p.dv + col0 + c4 * 4;
    float4 s[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) s[i] = *reinterpret_cast<const float4 *>(Sh + (size_t)(r0 + 32 * i) * p.dv);
    const float *qb = p.qn + ((size_t)b * p.n_qk + hq) * T * DK;
    const float *kb = p.kn + ((size_t)b * p.n_qk + hq) * T * DK;
    const size_t hv = ((size_t)b * p.n_v + h) * T;
    const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);

    for (int c0 = 0; c0 < T; c0 += kChunk) {
        const int n = min(kChunk, T - c0);
        __syncthreads();  // the last chunk's reads of shared memory are done
        // 1. the chunk's k^, q^ rows, the slice's v, the gates (tokens past n
        //    are zero: no write, no decay), the state
        for (int idx = tid; idx < kChunk * DK / 4; idx += kThreads) {
            const int t = idx >> 5, r4 = idx & 31;
            float4 kv = zero4, qv = zero4;
            if (t < n) {
                kv = *reinterpret_cast<const float4 *>(kb + (size_t)(c0 + t) * DK + r4 * 4);
                qv = *reinterpret_cast<const float4 *>(qb + (size_t)(c0 + t) * DK + r4 * 4);
            }
            *reinterpret_cast<float4 *>(&cs.K[t][r4 * 4]) = kv;
            *reinterpret_cast<float4 *>(&cs.Q[t][r4 * 4]) = qv;
        }
        {
            float4 v4 = zero4;
            if (tt < n) v4 = *reinterpret_cast<const float4 *>(p.vv + (hv + c0 + tt) * p.dv + col0 + cq * 4);
            *reinterpret_cast<float4 *>(&cs.V[tt][cq * 4]) = v4;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) *reinterpret_cast<float4 *>(&cs.S0[r0 + 32 * i][c4 * 4]) = s[i];
        if (warp == 0) {
            float gv = lane < n ? p.gg[hv + c0 + lane] : 0.f;
            const float bv = lane < n ? p.bb[hv + c0 + lane] : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {  // inclusive prefix sum: G_t
                const float y = __shfl_up_sync(0xffffffffu, gv, o);
                if (lane >= o) gv += y;
            }
            const float gl = __shfl_sync(0xffffffffu, gv, n - 1);  // G of the chunk's last token
            cs.G[lane] = gv;
            cs.gam[lane] = expf(gv);
            cs.wn[lane] = expf(gl - gv);
            cs.beta[lane] = bv;
        }
        __syncthreads();
        // 2. L, M (token tt against tokens cq + 8 j, j < 4: consecutive padded
        //    rows across a quarter-warp, no bank conflicts), P = S0^T k_tt and
        //    S0^T q_tt (one read of S0 for both)
        float4 oi = zero4;
        {
            float a[4] = {0.f, 0.f, 0.f, 0.f}, m[4] = {0.f, 0.f, 0.f, 0.f};
            float4 pacc = zero4;
#pragma unroll 4
            for (int r = 0; r < DK; r += 4) {
                const float4 kt = *reinterpret_cast<const float4 *>(&cs.K[tt][r]);
                const float4 qt = *reinterpret_cast<const float4 *>(&cs.Q[tt][r]);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float4 ks = *reinterpret_cast<const float4 *>(&cs.K[cq + 8 * j][r]);
                    a[j] += dot4(kt, ks);
                    m[j] += dot4(qt, ks);
                }
                const float4 s0 = *reinterpret_cast<const float4 *>(&cs.S0[r][cq * 4]);
                const float4 s1 = *reinterpret_cast<const float4 *>(&cs.S0[r + 1][cq * 4]);
                const float4 s2 = *reinterpret_cast<const float4 *>(&cs.S0[r + 2][cq * 4]);
                const float4 s3 = *reinterpret_cast<const float4 *>(&cs.S0[r + 3][cq * 4]);
                fma4(pacc, kt.x, s0);
                fma4(pacc, kt.y, s1);
                fma4(pacc, kt.z, s2);
                fma4(pacc, kt.w, s3);
                fma4(oi, qt.x, s0);
                fma4(oi, qt.y, s1);
                fma4(oi, qt.z, s2);
                fma4(oi, qt.w, s3);
            }
            const float gt = cs.G[tt];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int si = cq + 8 * j;
                const float e = expf(gt - cs.G[si]);
                cs.L[tt][si] = si < tt ? e * a[j] : 0.f;
                cs.M[tt][si] = si <= tt ? e * m[j] : 0.f;
            }
            *reinterpret_cast<float4 *>(&cs.P[tt][cq * 4]) = pacc;
        }
        __syncthreads();
        // 3. warp 0: the triangular solve for u (lane = column)
        if (warp == 0) {
            float u[kChunk];
#pragma unroll
            for (int t = 0; t < kChunk; ++t) {
                float acc = fmaf(-cs.gam[t], cs.P[t][lane], cs.V[t][lane]);
#pragma unroll
                for (int s2 = 0; s2 < t; ++s2) acc = fmaf(-cs.L[t][s2], u[s2], acc);
                u[t] = cs.beta[t] * acc;
                cs.U[t][lane] = u[t];
            }
        }
        __syncthreads();
        // 4. the readouts o_tt, and the state after the chunk
        {
            const float gt = cs.gam[tt];
            float4 o4 = make_float4(gt * oi.x, gt * oi.y, gt * oi.z, gt * oi.w);
#pragma unroll 8
            for (int s2 = 0; s2 < kChunk; ++s2)
                fma4(o4, cs.M[tt][s2], *reinterpret_cast<const float4 *>(&cs.U[s2][cq * 4]));
            if (tt < n) *reinterpret_cast<float4 *>(p.o + (hv + c0 + tt) * p.dv + col0 + cq * 4) = o4;
        }
        {
            const float gn = cs.gam[n - 1];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                s[i].x *= gn;
                s[i].y *= gn;
                s[i].z *= gn;
                s[i].w *= gn;
            }
            for (int t = 0; t < n; ++t) {
                const float4 u4 = *reinterpret_cast<const float4 *>(&cs.U[t][c4 * 4]);
                const float w = cs.wn[t];
#pragma unroll
                for (int i = 0; i < 4; ++i) fma4(s[i], cs.K[t][r0 + 32 * i] * w, u4);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) *reinterpret_cast<float4 *>(Sh + (size_t)(r0 + 32 * i) * p.dv) = s[i];
}

// 5''. The chunked recurrence on the tensor cores (dk = dv = 128, one decay
// per head): the algebra of 5', with the three dense products of a chunk
// as tcgen05 MMAs (kind::f16, fp32 accumulation in tensor memory), each
// operand split into bf16 hi + lo and every product taken as
// hi*hi + hi*lo + lo*hi (about 2^-16 relative per term, far inside the
// decode step's tolerance).  One CTA of 128 threads per (value head,
// sequence); thread j owns value column j, which is tensor-memory lane j.
// The state lives in tensor memory for the whole block, transposed (lane j,
// column i holds S[i][j]), as the accumulator of the update.  Per chunk:
//   1. the gates; the chunk's k^, q^ rows as B operand tiles (64 rows: k^
//      tokens, then q^ tokens) and as the A operand [k^; q^] (lane = token
//      row); S0^T as an A operand; the accumulator scaled to gamma_n S0;
//   2. MMA: D1 = [k^; q^] k^^T (k.k and q.k), D2 = S0^T [k^; q^]^T
//      (S0^T k_t and S0^T q_t in lane j);
//   3. L, M from D1 with the decays; every thread solves the chunk's
//      lower-triangular system for its column of u (tokens in order) and
//      forms its column of the readouts;
//   4. MMA: S^T += U^T (w k^)^T with w_t = exp(G_n - G_t): A = U^T (lane j),
//      B = the chunk's weighted k^ as 128 rows of 32 tokens.
// Tensor memory (512 columns, one CTA per SM):
constexpr int kTcThreads = 128;
constexpr uint32_t kTcCols = 512;
constexpr uint32_t kColS = 0;       // S^T, fp32
constexpr uint32_t kColAsHi = 128;  // S0^T as bf16 pairs (k = i), hi and lo
constexpr uint32_t kColAsLo = 192;
constexpr uint32_t kColAkqHi = 256; // [k^; q^] as bf16 pairs, lanes 0-63 (64-127 zero)
constexpr uint32_t kColAkqLo = 320;
constexpr uint32_t kColD2 = 384;    // 64 columns: S0^T k_t (t < 32), S0^T q_t (32 + t)
constexpr uint32_t kColD1 = 448;    // 32 columns: k_r.k_s (lane r < 32), q_r.k_s (lane 32 + r)
constexpr uint32_t kColAuHi = 480;  // U^T as bf16 pairs (k = token), hi and lo
constexpr uint32_t kColAuLo = 496;

struct __align__(1024) TcChunkSmem {
    union {
        struct {
            // B operand tiles in the 128-byte swizzled K-major layout (op_chunk_offset)
            uint8_t bkq[2][2][8192];  // [hi, lo][k half]: 64 rows (k^ tokens, q^ tokens) x 64 k
            uint8_t bw[2][16384];     // [hi, lo]: 128 rows (key channel) x 32 tokens (the first 64 bytes)
        };
        float st[128 * 128];  // the state on its way in and out (bulk copies), [i][j]
    };
    float kf[kChunk][128];    // the chunk's k^ rows
    float L[kChunk][kChunk + 1];
    float M[kChunk][kChunk + 1];
    float G[kChunk], gam[kChunk], wn[kChunk], beta[kChunk];
    uint64_t mma_done, s_full;
    uint32_t tmem_base;
};

// x0, x1 -> bf16 pairs hi = bf16(x), lo = bf16(x - hi) (x0 in the low halves)
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

// mbarrier phase wait, bounded (about one second of the global timer)
__device__ bool tc_wait(uint64_t *bar, uint32_t parity) {
    const uint64_t t0 = dev::global_ns();
    for (uint32_t it = 0;; ++it) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred q;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(done)
            : "r"(dev::smem_u32(bar)), "r"(parity)
            : "memory");
        if (done) return true;
        if ((it & 63u) == 63u && dev::global_ns() - t0 > 1000000000ull) return false;
    }
}

// the MMAs of a 3-pass product: D (+)= A x B^T over K = 128 (two 64-k
// halves), A hi/lo in tensor memory, B hi/lo tiles 8 KB apart per k half
__device__ __forceinline__ void mma3_k128(uint32_t d, uint32_t a_hi, uint32_t a_lo, const uint8_t *b_hi,
                                          const uint8_t *b_lo, uint32_t idesc, bool accumulate) {
    for (int pass = 0; pass < 3; ++pass) {
        const uint32_t a = pass == 2 ? a_lo : a_hi;
        const uint8_t *bt = pass == 1 ? b_lo : b_hi;
        for (int kh = 0; kh < 2; ++kh)
            dev::mma_bf16_ts_x4(d, a + 32u * kh, dev::smem_desc_sw128(dev::smem_u32(bt + 8192 * kh)), idesc,
                                (accumulate || pass > 0 || kh > 0) ? 1u : 0u);
    }
}

__global__ void __launch_bounds__(kTcThreads, 1) recur_tc_kernel(const RecParams p) {
    constexpr int DK = 128;
    extern __shared__ uint8_t tc_smem_raw[];
    TcChunkSmem &cs = *reinterpret_cast<TcChunkSmem *>(
        (reinterpret_cast<uintptr_t>(tc_smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x, b = blockIdx.y;
    const int hq = h / p.group, T = p.geo.T;
    float *Sh = p.S + ((size_t)(p.geo.b0 + b) * p.n_v + h) * DK * DK;
    const float *qb = p.qn + ((size_t)b * p.n_qk + hq) * T * DK;
    const float *kb = p.kn + ((size_t)b * p.n_qk + hq) * T * DK;
    const size_t hv = ((size_t)b * p.n_v + h) * T;

    if (tid == 0) {
        dev::mbar_init(&cs.mma_done, 1);
        dev::mbar_init(&cs.s_full, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        // the head's state (64 KB) by one bulk copy
        dev::mbar_arrive_expect_tx(&cs.s_full, DK * DK * 4);
        dev::bulk_g2s(dev::smem_u32(cs.st), Sh, DK * DK * 4, &cs.s_full);
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         dev::smem_u32(&cs.tmem_base)),
                     "r"(kTcCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    dev::tc_fence_before();
    __syncthreads();
    dev::tc_fence_after();
    const uint32_t tbase = cs.tmem_base;
    const uint32_t tm = tbase + ((uint32_t)(warp * 32) << 16);  // this warp's lane quarter

    // the state into tensor memory, transposed (thread j takes column j)
    bool ok = tc_wait(&cs.s_full, 0);
    for (int i0 = 0; i0 < DK; i0 += 32) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(cs.st[(i0 + i) * DK + tid]);
        dev::tmem_st32(tm + kColS + i0, r);
    }
    if (warp >= 2) {  // rows 64-127 of [k^; q^]: zero for good
        uint32_t z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = 0u;
        for (uint32_t c = 0; c < 128; c += 32) dev::tmem_st32(tm + kColAkqHi + c, z);
    }

    uint32_t phase = 0;
    ok = __syncthreads_and(ok) != 0;  // (and the staging area is free again)
    for (int c0 = 0; c0 < T && ok; c0 += kChunk) {
        const int n = min(kChunk, T - c0);
        // 1. gates (tokens past n: no decay, no write)
        if (warp == 0) {
            float gv = lane < n ? p.gg[hv + c0 + lane] : 0.f;
            const float bv = lane < n ? p.bb[hv + c0 + lane] : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {  // inclusive prefix sum: G_t
                const float y = __shfl_up_sync(0xffffffffu, gv, o);
                if (lane >= o) gv += y;
            }
            const float gl = __shfl_sync(0xffffffffu, gv, n - 1);
            cs.G[lane] = gv;
            cs.gam[lane] = expf(gv);
            cs.wn[lane] = expf(gl - gv);
            cs.beta[lane] = bv;
        }
        float v[kChunk];  // column j of the chunk's v
#pragma unroll
        for (int t = 0; t < kChunk; ++t) v[t] = t < n ? p.vv[(hv + c0 + t) * p.dv + tid] : 0.f;
        // k^, q^ rows: B tiles and fp32 k^ (64 rows x 16 eight-wide k chunks;
        // every load issued before the first is used)
        float4 xs[2 * 64 * 16 / kTcThreads];
#pragma unroll
        for (int m = 0; m < 64 * 16 / kTcThreads; ++m) {
            const int it = tid + m * kTcThreads, row = it >> 4, kc = it & 15, t = row & 31;
            xs[2 * m] = xs[2 * m + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < n) {
                const float *src = (row < 32 ? kb : qb) + (size_t)(c0 + t) * DK + kc * 8;
                xs[2 * m] = *reinterpret_cast<const float4 *>(src);
                xs[2 * m + 1] = *reinterpret_cast<const float4 *>(src + 4);
            }
        }
#pragma unroll
        for (int m = 0; m < 64 * 16 / kTcThreads; ++m) {
            const int it = tid + m * kTcThreads, row = it >> 4, kc = it & 15, t = row & 31;
            const float4 x0 = xs[2 * m], x1 = xs[2 * m + 1];
            if (row < 32) {
                *reinterpret_cast<float4 *>(&cs.kf[t][kc * 8]) = x0;
                *reinterpret_cast<float4 *>(&cs.kf[t][kc * 8 + 4]) = x1;
            }
            uint4 hi, lo;
            split_bf16x2(x0.x, x0.y, hi.x, lo.x);
            split_bf16x2(x0.z, x0.w, hi.y, lo.y);
            split_bf16x2(x1.x, x1.y, hi.z, lo.z);
            split_bf16x2(x1.z, x1.w, hi.w, lo.w);
            const uint32_t off = op_chunk_offset(row, kc & 7);
            *reinterpret_cast<uint4 *>(cs.bkq[0][kc >> 3] + off) = hi;
            *reinterpret_cast<uint4 *>(cs.bkq[1][kc >> 3] + off) = lo;
        }
        // the A operand [k^; q^]: warp 0 the k^ tokens, warp 1 the q^ tokens
        if (warp < 2) {
            const float *src = (warp == 0 ? kb : qb) + (size_t)(c0 + lane) * DK;
            for (int half = 0; half < 2; ++half) {
                uint32_t hi[32], lo[32];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (lane < n) x = *reinterpret_cast<const float4 *>(src + half * 64 + 2 * e);
                    split_bf16x2(x.x, x.y, hi[e], lo[e]);
                    split_bf16x2(x.z, x.w, hi[e + 1], lo[e + 1]);
                }
                dev::tmem_st32(tm + kColAkqHi + 32u * half, hi);
                dev::tmem_st32(tm + kColAkqLo + 32u * half, lo);
            }
        }
        __syncthreads();
        // S0^T as the A operand, and the accumulator scaled to gamma_n S0
        {
            const float gn = cs.gam[n - 1];
            for (int i0 = 0; i0 < DK; i0 += 32) {
                uint32_t r[32], hi[16], lo[16];
                dev::tmem_ld32(tm + kColS + i0, r);
#pragma unroll
                for (int e = 0; e < 16; ++e)
                    split_bf16x2(__uint_as_float(r[2 * e]), __uint_as_float(r[2 * e + 1]), hi[e], lo[e]);
                dev::tmem_st16(tm + kColAsHi + i0 / 2, hi);
                dev::tmem_st16(tm + kColAsLo + i0 / 2, lo);
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(gn * __uint_as_float(r[e]));
                dev::tmem_st32(tm + kColS + i0, r);
            }
        }
        // 2. D1 and D2
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // B tiles -> the tensor core
        dev::tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            dev::tc_fence_after();
            mma3_k128(tbase + kColD1, tbase + kColAkqHi, tbase + kColAkqLo, cs.bkq[0][0], cs.bkq[1][0],
                      dev::instr_desc(128, 32), false);
            mma3_k128(tbase + kColD2, tbase + kColAsHi, tbase + kColAsLo, cs.bkq[0][0], cs.bkq[1][0],
                      dev::instr_desc(128, 64), false);
            dev::mma_commit(&cs.mma_done);
        }
        ok = tc_wait(&cs.mma_done, phase);
        phase ^= 1u;
        dev::tc_fence_after();
        // 3. L, M (warps 0 and 1: lane = token), S0^T k_t and S0^T q_t (lane j)
        if (warp < 2) {
            uint32_t r[32];
            dev::tmem_ld32(tm + kColD1, r);
            const float gt = cs.G[lane];
#pragma unroll
            for (int s2 = 0; s2 < kChunk; ++s2) {
                const float e = expf(gt - cs.G[s2]) * __uint_as_float(r[s2]);
                if (warp == 0)
                    cs.L[lane][s2] = s2 < lane ? e : 0.f;
                else
                    cs.M[lane][s2] = s2 <= lane ? e : 0.f;
            }
        }
        uint32_t pk[32], pq[32];
        dev::tmem_ld32(tm + kColD2, pk);
        dev::tmem_ld32(tm + kColD2 + 32, pq);
        __syncthreads();
        float u[kChunk];
#pragma unroll
        for (int t = 0; t < kChunk; ++t) {
            float acc = fmaf(-cs.gam[t], __uint_as_float(pk[t]), v[t]);
#pragma unroll
            for (int s2 = 0; s2 < t; ++s2) acc = fmaf(-cs.L[t][s2], u[s2], acc);
            u[t] = cs.beta[t] * acc;
        }
#pragma unroll
        for (int t = 0; t < kChunk; ++t) {
            if (t < n) {
                float o = cs.gam[t] * __uint_as_float(pq[t]);
#pragma unroll
                for (int s2 = 0; s2 <= t; ++s2) o = fmaf(cs.M[t][s2], u[s2], o);
                p.o[(hv + c0 + t) * p.dv + tid] = o;
            }
        }
        // 4. A = U^T (lane j), B = the weighted k^ (row i = this thread)
        {
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) split_bf16x2(u[2 * e], u[2 * e + 1], hi[e], lo[e]);
            dev::tmem_st16(tm + kColAuHi, hi);
            dev::tmem_st16(tm + kColAuLo, lo);
#pragma unroll
            for (int kc = 0; kc < 4; ++kc) {
                uint32_t wh[4], wl[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int t0 = 8 * kc + 2 * e;
                    split_bf16x2(cs.wn[t0] * cs.kf[t0][tid], cs.wn[t0 + 1] * cs.kf[t0 + 1][tid], wh[e], wl[e]);
                }
                const uint32_t off = op_chunk_offset(tid, kc);
                *reinterpret_cast<uint4 *>(cs.bw[0] + off) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                *reinterpret_cast<uint4 *>(cs.bw[1] + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
            }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        dev::tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            dev::tc_fence_after();
            const uint32_t idesc = dev::instr_desc(128, 128);
            for (int pass = 0; pass < 3; ++pass)
                dev::mma_bf16_ts_x2(tbase + kColS, tbase + (pass == 2 ? kColAuLo : kColAuHi),
                                    dev::smem_desc_sw128(dev::smem_u32(cs.bw[pass == 1 ? 1 : 0])), idesc, 1u);
            dev::mma_commit(&cs.mma_done);
        }
        ok = tc_wait(&cs.mma_done, phase) && ok;
        phase ^= 1u;
        dev::tc_fence_after();
        ok = __syncthreads_and(ok) != 0;
    }
    if (ok) {  // the state back, through the staging area and one bulk store
        for (int i0 = 0; i0 < DK; i0 += 32) {
            uint32_t r[32];
            dev::tmem_ld32(tm + kColS + i0, r);
#pragma unroll
            for (int i = 0; i < 32; ++i) cs.st[(i0 + i) * DK + tid] = __uint_as_float(r[i]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (tid == 0) {
            asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(Sh),
                         "r"(dev::smem_u32(cs.st)), "r"(DK * DK * 4)
                         : "memory");
            asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
        }
    }
    dev::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        dev::tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kTcCols)
                     : "memory");
    }
    if (tid == 0 && !ok) atomicOr(p.err, 1);
}

// 6. gated RMSNorm of every readout of the block: fp32 rows for the CUDA-core
// out_proj, or bf16 hi/lo B-operand tiles (column j = operand rows 2j, 2j+1
// of its 64-column chunk) for the tensor-core one.  grid (n_v, cols).
__global__ void __launch_bounds__(kThreads) norm_block_kernel(const float *__restrict__ o, const float *__restrict__ zs,
                                                              const float *__restrict__ w_norm, float *__restrict__ nrm,
                                                              uint8_t *__restrict__ xb_out, Geo g, int n_v, int dv,
                                                              int v_dim, int kt_out, float norm_eps) {
    __shared__ float red[kThreads / 32];
    const int h = blockIdx.x, j = blockIdx.y, b = j / g.T, t = j % g.T;
    const size_t row = (((size_t)b * n_v + h) * g.T + t) * dv;
    const int i = threadIdx.x;
    const float ov = i < dv ? o[row + i] : 0.f;
    const float ss = block_sum(ov * ov, red);
    if (i >= dv) return;
    const float n = ov * (1.0f / sqrtf(ss / (float)dv + norm_eps)) * w_norm[i] * zs[row + i];
    const int k = h * dv + i;
    if (xb_out == nullptr) {
        nrm[(size_t)j * v_dim + k] = n;
    } else {
        const __nv_bfloat16 hi = __float2bfloat16_rn(n);
        const __nv_bfloat16 lo = __float2bfloat16_rn(n - __bfloat162float(hi));
        uint8_t *ot = xb_out + ((size_t)(j >> 6) * kt_out + (k >> 6)) * kOpTile;
        const int kc = (k & 63) >> 3, e = k & 7;
        const int rh = 2 * (j & 63), rl = rh + 1;
        *reinterpret_cast<__nv_bfloat16 *>(ot + op_chunk_offset(rh, kc) + e * 2) = hi;
        *reinterpret_cast<__nv_bfloat16 *>(ot + op_chunk_offset(rl, kc) + e * 2) = lo;
    }
}

cudaError_t launch_recur_chunk(const RecParams &rp, int dv, int n_v, int nb, cudaStream_t st) {
    static std::atomic<uint64_t> attr_done{0};
    const cudaError_t e = once_per_device(attr_done, [&](int) {
        return cudaFuncSetAttribute(recur_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)sizeof(ChunkSmem));
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(dv / DJ), (unsigned)n_v, (unsigned)nb);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = sizeof(ChunkSmem);
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, recur_chunk_kernel, rp);
}

cudaError_t launch_recur_tc(const RecParams &rp, int n_v, int nb, cudaStream_t st) {
    // over half of an SM's shared memory: one CTA per SM, which then holds
    // all of its tensor memory
    const size_t smem = std::max<size_t>(sizeof(TcChunkSmem) + 1024, 116 * 1024);
    static std::atomic<uint64_t> attr_done{0};
    const cudaError_t e = once_per_device(attr_done, [&](int) {
        return cudaFuncSetAttribute(recur_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)n_v, (unsigned)nb);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, recur_tc_kernel, rp);
}

template <int DK>
cudaError_t launch_recur(const RecParams &rp, int dv, int n_v, int nb, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(dv / DJ), (unsigned)n_v, (unsigned)nb);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, recur_kernel<DK>, rp);
}

}  // namespace

cudaError_t launch_prefill_block(const Dims &d, const LayerDev &L, const PrefillDev &P, const PrefillBlock &blk,
                                 cudaStream_t st) {
    const Geo g{blk.b0, blk.nb, blk.t0, blk.T, blk.S, blk.nb * blk.T};
    const int cols = g.cols;
    const bool tc = cols >= kTcMinBatch;
    cudaError_t e;
    // 1. the block's x rows, the in_proj over all columns
    {
        cudaLaunchConfig_t c = {};
        c.gridDim = dim3((unsigned)((d.hidden / 4 + 255) / 256), (unsigned)cols);
        c.blockDim = dim3(256);
        c.stream = st;
        if ((e = cudaLaunchKernelEx(&c, gather_rows_kernel, blk.x, P.xg, d.hidden, g)) != cudaSuccess) return e;
    }
    if (tc) {
        if ((e = launch_pack_b(P.xg, P.xb_in, cols, d.hidden, st)) != cudaSuccess) return e;
        e = launch_gemm_i8_tc(L.w_in, P.xb_in, P.part_in, P.nseg_in, L.err, d.proj_rows, d.hidden, cols, st);
    } else {
        e = launch_gemv_i8(d.i4 ? L.w_in4 : L.w_in, P.xg, P.part_in, P.nseg_in, L.err, d.proj_rows, d.hidden, cols,
                           st, d.i4 != 0);
    }
    if (e != cudaSuccess) return e;
    const GemmPlan gpi = plan_tc_gemm(d.proj_rows, plan_k(d, d.hidden, cols), cols);
    if (d.dk == 128 && d.dv == 128 && d.conv_k <= 8 && gpi.MT * blk.nb >= num_sms()) {
        // 2-4 in one kernel, when its (row tile, sequence) CTAs cover the SMs
        // (one sequence's prompt has more parallelism in the three kernels)
        const GemmPlan &gp = gpi;
        TileParams tp;
        tp.part = P.part_in;
        tp.nseg = P.nseg_in;
        tp.s_in = L.s_in;
        tp.ring = L.ring;
        tp.rpos = L.rpos;
        tp.wconv_t = L.wconv_t;
        tp.g = blk.g;
        tp.beta = blk.beta;
        tp.gate_A = L.gate_A;
        tp.qn = P.qn;
        tp.kn = P.kn;
        tp.vv = P.vv;
        tp.zs = P.zs;
        tp.gg = P.gg;
        tp.bb = P.bb;
        tp.geo = g;
        tp.MT = gp.MT;
        tp.max_seg = gp.max_seg;
        tp.conv_ch = d.conv_ch;
        tp.qk_dim = d.qk_dim;
        tp.in_rows = d.in_rows;
        tp.proj_rows = d.proj_rows;
        tp.n_qk = d.n_qk;
        tp.n_v = d.n_v;
        tp.gw = d.gw;
        tp.dev_gates = d.dev_gates;
        tp.l2_eps = d.l2_eps;
        tp.q_scale = d.q_scale;
        cudaLaunchConfig_t c = {};
        c.gridDim = dim3((unsigned)gp.MT, (unsigned)blk.nb);
        c.blockDim = dim3(128);
        c.stream = st;
        switch (d.conv_k) {
            case 2: e = cudaLaunchKernelEx(&c, prep_tile_kernel<2>, tp); break;
            case 3: e = cudaLaunchKernelEx(&c, prep_tile_kernel<3>, tp); break;
            case 4: e = cudaLaunchKernelEx(&c, prep_tile_kernel<4>, tp); break;
            case 5: e = cudaLaunchKernelEx(&c, prep_tile_kernel<5>, tp); break;
            case 6: e = cudaLaunchKernelEx(&c, prep_tile_kernel<6>, tp); break;
            case 7: e = cudaLaunchKernelEx(&c, prep_tile_kernel<7>, tp); break;
            default: e = cudaLaunchKernelEx(&c, prep_tile_kernel<8>, tp); break;
        }
        if (e != cudaSuccess) return e;
    } else {
    // 2. scaled rows
    {
        const GemmPlan gp = plan_tc_gemm(d.proj_rows, plan_k(d, d.hidden, cols), cols);
        cudaLaunchConfig_t c = {};
        c.gridDim = dim3((unsigned)((d.proj_rows + 255) / 256), (unsigned)cols);
        c.blockDim = dim3(256);
        c.stream = st;
        if ((e = cudaLaunchKernelEx(&c, sum_rows_kernel, (const float *)P.part_in, (const int *)P.nseg_in,
                                    (const float *)L.s_in, P.xin, d.proj_rows, gp.MT, gp.max_seg)) != cudaSuccess)
            return e;
    }
    // 3. conv, SiLU, norms, gates
    {
        PrepParams pp;
        pp.xin = P.xin;
        pp.ring = L.ring;
        pp.rpos = L.rpos;
        pp.wconv_t = L.wconv_t;
        pp.g = blk.g;
        pp.beta = blk.beta;
        pp.gate_A = L.gate_A;
        pp.qn = P.qn;
        pp.kn = P.kn;
        pp.vv = P.vv;
        pp.zs = P.zs;
        pp.gg = P.gg;
        pp.bb = P.bb;
        pp.geo = g;
        pp.K = d.conv_k;
        pp.conv_ch = d.conv_ch;
        pp.qk_dim = d.qk_dim;
        pp.in_rows = d.in_rows;
        pp.proj_rows = d.proj_rows;
        pp.n_qk = d.n_qk;
        pp.n_v = d.n_v;
        pp.dk = d.dk;
        pp.dv = d.dv;
        pp.gw = d.gw;
        pp.dev_gates = d.dev_gates;
        pp.l2_eps = d.l2_eps;
        pp.q_scale = d.q_scale;
        cudaLaunchConfig_t c = {};
        c.gridDim = dim3((unsigned)(d.n_qk + d.n_v), (unsigned)cols);
        c.blockDim = dim3(kThreads);
        c.stream = st;
        if ((e = cudaLaunchKernelEx(&c, prep_kernel, pp)) != cudaSuccess) return e;
    }
    // 4. the ring moves on by T inputs (its positions move with the reduction in 7.)
    {
        cudaLaunchConfig_t c = {};
        c.gridDim = dim3((unsigned)((d.conv_ch + 255) / 256), (unsigned)blk.nb);
        c.blockDim = dim3(256);
        c.stream = st;
        if ((e = cudaLaunchKernelEx(&c, ring_block_kernel, (const float *)P.xin, L.ring, (const int32_t *)L.rpos, g,
                                    d.conv_k, d.conv_ch, d.proj_rows)) != cudaSuccess)
            return e;
    }
    }
    // 5. the recurrence
    {
        RecParams rp;
        rp.S = L.S;
        rp.qn = P.qn;
        rp.kn = P.kn;
        rp.vv = P.vv;
        rp.gg = P.gg;
        rp.bb = P.bb;
        rp.o = P.o;
        rp.geo = g;
        rp.n_v = d.n_v;
        rp.n_qk = d.n_qk;
        rp.group = d.n_v / d.n_qk;
        rp.dv = d.dv;
        rp.gw = d.gw;
        rp.err = L.err;
        // one decay per head: the chunked form; for 128 x 128 heads on the
        // tensor cores (one CTA per head and sequence) when that gives every
        // SM a CTA, else on the CUDA cores in 32-column slices
        if (d.dk == 128 && d.dv == 128 && d.gw == 1 && d.n_v * blk.nb >= num_sms())
            e = launch_recur_tc(rp, d.n_v, blk.nb, st);
        else if (d.dk == 128 && d.gw == 1)
            e = launch_recur_chunk(rp, d.dv, d.n_v, blk.nb, st);
        else switch (d.dk) {
            case 32: e = launch_recur<32>(rp, d.dv, d.n_v, blk.nb, st); break;
            case 64: e = launch_recur<64>(rp, d.dv, d.n_v, blk.nb, st); break;
            case 128: e = launch_recur<128>(rp, d.dv, d.n_v, blk.nb, st); break;
            case 256: e = launch_recur<256>(rp, d.dv, d.n_v, blk.nb, st); break;
            default: e = cudaErrorInvalidValue;
        }
        if (e != cudaSuccess) return e;
    }
    // 6. gated RMSNorm -> the out_proj's input
    const int kt_out = (d.v_dim + kTileK - 1) / kTileK;
    {
        cudaLaunchConfig_t c = {};
        c.gridDim = dim3((unsigned)d.n_v, (unsigned)cols);
        c.blockDim = dim3(kThreads);
        c.stream = st;
        if ((e = cudaLaunchKernelEx(&c, norm_block_kernel, (const float *)P.o, (const float *)P.zs,
                                    (const float *)L.w_norm, P.nrm, tc ? P.xb_out : (uint8_t *)nullptr, g, d.n_v,
                                    d.dv, d.v_dim, kt_out, d.norm_eps)) != cudaSuccess)
            return e;
    }
    // 7. the out_proj, each token's row of the output, ring positions + T
    if (tc)
        e = launch_gemm_i8_tc(L.w_out, P.xb_out, P.part_out, P.nseg_out, L.err, d.hidden, d.v_dim, cols, st);
    else
        e = launch_gemv_i8(d.i4 ? L.w_out4 : L.w_out, P.nrm, P.part_out, P.nseg_out, L.err, d.hidden, d.v_dim, cols,
                           st, d.i4 != 0);
    if (e != cudaSuccess) return e;
    return launch_splitk_reduce(P.part_out, P.nseg_out, L.s_out, blk.out + (size_t)blk.b0 * blk.S * d.hidden,
                                d.hidden, plan_k(d, d.v_dim, cols), cols, L.rpos + 2 * blk.b0, d.conv_k, st, blk.T, blk.S, blk.t0,
                                blk.T);
}

}  // namespace dn
