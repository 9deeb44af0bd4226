// The fused per-head part of the gated-DeltaNet decode step.
//
// Page "qwen36: run the DeltaNet layer end to end on the card
// (Q36_DN_GPU=1)", section "What the PR does": after the in_proj GEMV, the
// step runs the causal conv + SiLU with the ring advancing, then per value
// head the L2 norms of q and k (eps inside the square root), the
// decay, the delta against the decayed state, the write-back, out = q^T S
// over the updated state, and the gated RMSNorm with silu(z).  This kernel
// does all of that in one pass over the state.
//
// Work split: one thread block per (column slice jc, value head h, sequence
// b).  A head's dv columns are cut into JS slices of DJ columns; the JS
// blocks of a head form one thread-block cluster and meet only once, to sum
// the head's squared outputs for the RMSNorm through distributed shared
// memory.  Every column of the update (delta[j], S[:, j], o[j]) depends on
// its own column only, so no other exchange is needed.
//
// State traffic: the block's dk x DJ fp32 tile of S is loaded into registers
// with coalesced 16-byte loads before anything else happens (so the HBM
// reads overlap the conv and the norms), decayed, reduced against k, updated
// and stored back from registers: one read and one write of S per step.
// Reductions run in a fixed order, so results are bitwise reproducible.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "dn_internal.cuh"
#include "dn_sched.cuh"

namespace cg = cooperative_groups;

namespace dn {
namespace {

constexpr int kThreads = 256;

struct CoreParams {
    const float *part_in;  // in_proj segment partials (GEMV or tensor-core kernel),
    const float *s_in;     // summed in slot order and scaled here by s_in
    const int *nseg_in;    // segments per tile
    SchedView sv;          // their schedule
    float *ring;           // [max_batch][conv_k][conv_ch]
    const int32_t *rpos;   // [max_batch][2]
    const float *wconv_t;  // [conv_k][conv_ch]
    const float *w_norm;   // [dv]
    float *S;              // [max_batch][n_v][dk][dv]
    float *nrm;            // [B][v_dim] fp32 output, or
    uint8_t *xb_out;       // packed bf16 hi/lo B-operand tiles for the tensor-core out_proj
    const float *g;        // [B][n_v]
    const float *beta;     // [B][n_v]
    int n_qk, n_v, dv, conv_k, conv_ch, qk_dim, in_rows, v_dim, kt_out;
    int gw;                // log-decay values per head: 1, or dk (per-key-channel gate)
    int dev_gates;         // g, beta from the a/b gate rows after the in_proj rows
    const float *gate_A;   // [n_v] (device gates)
    float l2_eps, norm_eps, q_scale;
};

__device__ __forceinline__ float silu_f(float a) { return a / (1.0f + expf(-a)); }
// softplus(a) = log(1 + e^a) as max(a, 0) + log1p(e^-|a|); sigmoid(b) = 1 / (1 + e^-b)
__device__ __forceinline__ float softplus_f(float a) { return fmaxf(a, 0.f) + log1pf(expf(-fabsf(a))); }
__device__ __forceinline__ float sigmoid_f(float b) { return 1.0f / (1.0f + expf(-b)); }

// in_proj output row c of sequence b: read directly, or summed from the
// tensor-core kernel's segment partials in slot order, then scaled
__device__ __forceinline__ float in_proj_out(const CoreParams &p, int b, int c) {
    const int tile = (b >> 6) * p.sv.MT + (c >> 7);
    const int nseg = p.nseg_in[tile];
    const float *pt = p.part_in + (size_t)tile * p.sv.max_seg * (64 * 128) + (b & 63) * 128 + (c & 127);
    float acc = 0.f;
#pragma unroll 4
    for (int k = 0; k < nseg; ++k) acc += __ldcg(pt + (size_t)k * (64 * 128));
    return p.s_in[c] * acc;
}

template <int DK, int DJ, bool CLUSTER>
__global__ void __launch_bounds__(kThreads, 2) dn_core_kernel(const CoreParams p) {
    constexpr int LPR = DJ / 4;          // lanes across one row of the tile (float4 each)
    constexpr int RPP = kThreads / LPR;  // rows covered per pass
    constexpr int NP = DK / RPP;         // passes: float4 registers of S per thread
    static_assert(DJ % 4 == 0 && kThreads % LPR == 0 && DK % RPP == 0 && NP >= 1, "tile");

    __shared__ __align__(16) float q_s[DK];
    __shared__ __align__(16) float k_s[DK];
    __shared__ __align__(16) float v_s[DJ];
    __shared__ __align__(16) float delta_s[DJ];
    __shared__ __align__(16) float red[RPP][DJ];
    __shared__ __align__(16) float eg_s[DK];  // exp(log-decay) of each key row
    __shared__ float inv_s[2];
    __shared__ float bt_s;
    __shared__ float ssq_s;

    const int tid = threadIdx.x;
    const int jc = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int group = p.n_v / p.n_qk;
    const int hq = h / group;
    const int col0 = jc * DJ;  // first column of this slice within the head

    // ---- 1. issue the state loads first ------------------------------------
    const int c4 = tid % LPR, r0 = tid / LPR;
    float *Sh = p.S + ((size_t)(b * p.n_v + h) * DK) * p.dv + col0 + c4 * 4;
    float4 s[NP];
#pragma unroll
    for (int i = 0; i < NP; ++i)
        s[i] = __ldcs(reinterpret_cast<const float4 *>(Sh + (size_t)(r0 + i * RPP) * p.dv));

    // ---- 2. causal conv + SiLU for the q/k channels of q/k head hq and the
    //         DJ v channels of this slice; the ring takes the new inputs ----
    const int dpos = p.rpos[2 * b];
    const int K = p.conv_k;
    pdl_wait();  // the in_proj partials come from the previous kernel
    pdl_trigger();
    int wslot = dpos + K - 1;
    if (wslot >= K) wslot -= K;
    float *rb = p.ring + (size_t)b * K * p.conv_ch;
    // q/k channels are shared by the `group` value heads of a q/k head and by
    // all column slices: exactly one block (first head of the group, slice 0)
    // writes them into the ring
    const bool owner_qk = (h % group == 0) && (jc == 0);
    for (int j = tid; j < 2 * DK + DJ; j += kThreads) {
        int c;
        if (j < DK)
            c = hq * DK + j;
        else if (j < 2 * DK)
            c = p.qk_dim + hq * DK + (j - DK);
        else
            c = 2 * p.qk_dim + h * p.dv + col0 + (j - 2 * DK);
        const float xv = in_proj_out(p, b, c);
        float acc = 0.f;
        int slot = dpos;
        for (int m = 0; m < K - 1; ++m) {  // oldest input first
            acc = fmaf(p.wconv_t[(size_t)m * p.conv_ch + c], rb[(size_t)slot * p.conv_ch + c], acc);
            if (++slot == K) slot = 0;
        }
        acc = fmaf(p.wconv_t[(size_t)(K - 1) * p.conv_ch + c], xv, acc);
        if (j >= 2 * DK || owner_qk) rb[(size_t)wslot * p.conv_ch + c] = xv;
        const float u = silu_f(acc);
        if (j < DK)
            q_s[j] = u;
        else if (j < 2 * DK)
            k_s[j - DK] = u;
        else
            v_s[j - 2 * DK] = u;
    }
    __syncthreads();

    // ---- 3. L2 norms of q and k: fp32 tree sums (fixed order), a relative error
    //         near 1e-7 where the pages' CPU accumulates in double -------------
    const int warp = tid >> 5, lane = tid & 31;
    if (warp < 2) {
        const float *vec = warp == 0 ? q_s : k_s;
        float ss = 0.f;
        for (int i = lane; i < DK; i += 32) ss = fmaf(vec[i], vec[i], ss);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0) inv_s[warp] = 1.0f / sqrtf(ss + p.l2_eps);
    }
    __syncthreads();
    for (int i = tid; i < 2 * DK; i += kThreads) {
        if (i < DK)
            q_s[i] = q_s[i] * inv_s[0] * p.q_scale;
        else
            k_s[i - DK] = k_s[i - DK] * inv_s[1];
    }
    // the decay of each key row (one gate per head, or one per key channel)
    // and the write strength: from the caller, or from the layer's a/b rows
    for (int i = tid; i < DK; i += kThreads) {
        const int gi = p.gw == 1 ? 0 : i;
        const float gl = p.dev_gates ? -p.gate_A[h] * softplus_f(in_proj_out(p, b, p.in_rows + h * p.gw + gi))
                                     : p.g[((size_t)b * p.n_v + h) * p.gw + gi];
        eg_s[i] = expf(gl);
    }
    if (tid == 0)
        bt_s = p.dev_gates ? sigmoid_f(in_proj_out(p, b, p.in_rows + p.n_v * p.gw + h)) : p.beta[b * p.n_v + h];
    __syncthreads();

    // ---- 4. decay, then what the decayed state predicts for k ----------------
    const float bt = bt_s;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        const float kr = k_s[r0 + i * RPP], eg = eg_s[r0 + i * RPP];
        s[i].x *= eg;
        s[i].y *= eg;
        s[i].z *= eg;
        s[i].w *= eg;
        acc.x = fmaf(s[i].x, kr, acc.x);
        acc.y = fmaf(s[i].y, kr, acc.y);
        acc.z = fmaf(s[i].z, kr, acc.z);
        acc.w = fmaf(s[i].w, kr, acc.w);
    }
    *reinterpret_cast<float4 *>(&red[r0][c4 * 4]) = acc;
    __syncthreads();
    if (tid < DJ) {
        float kv = 0.f;
#pragma unroll 8
        for (int r = 0; r < RPP; ++r) kv += red[r][tid];
        delta_s[tid] = bt * (v_s[tid] - kv);
    }
    __syncthreads();

    // ---- 5. write-back S += k delta^T, store, and read out o = S^T q ---------
    const float4 d4 = *reinterpret_cast<const float4 *>(&delta_s[c4 * 4]);
    acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        const int r = r0 + i * RPP;
        const float kr = k_s[r], qr = q_s[r];
        s[i].x = fmaf(kr, d4.x, s[i].x);
        s[i].y = fmaf(kr, d4.y, s[i].y);
        s[i].z = fmaf(kr, d4.z, s[i].z);
        s[i].w = fmaf(kr, d4.w, s[i].w);
        __stcs(reinterpret_cast<float4 *>(Sh + (size_t)r * p.dv), s[i]);
        acc.x = fmaf(s[i].x, qr, acc.x);
        acc.y = fmaf(s[i].y, qr, acc.y);
        acc.z = fmaf(s[i].z, qr, acc.z);
        acc.w = fmaf(s[i].w, qr, acc.w);
    }
    *reinterpret_cast<float4 *>(&red[r0][c4 * 4]) = acc;
    __syncthreads();
    float o = 0.f;
    if (tid < DJ) {
#pragma unroll 8
        for (int r = 0; r < RPP; ++r) o += red[r][tid];
    }

    // ---- 6. gated RMSNorm over the head's dv outputs --------------------------
    if (warp == 0) {
        float ss = 0.f;
        for (int j = lane; j < DJ; j += 32) {
            float t = 0.f;
#pragma unroll 8
            for (int r = 0; r < RPP; ++r) t += red[r][j];
            ss = fmaf(t, t, ss);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (lane == 0) ssq_s = ss;
    }
    float total;
    if constexpr (CLUSTER) {
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        total = 0.f;
        const int nblk = (int)cluster.num_blocks();
        for (int r = 0; r < nblk; ++r) total += *cluster.map_shared_rank(&ssq_s, r);
        cluster.sync();  // peers keep their shared memory until everyone has read it
    } else {
        __syncthreads();
        total = ssq_s;
    }
    if (tid < DJ) {
        const float rinv = 1.0f / sqrtf(total / (float)p.dv + p.norm_eps);
        const float z = in_proj_out(p, b, p.conv_ch + h * p.dv + col0 + tid);
        const float n = o * rinv * p.w_norm[col0 + tid] * silu_f(z);
        const int k = h * p.dv + col0 + tid;
        if (p.xb_out == nullptr) {
            p.nrm[(size_t)b * p.v_dim + k] = n;
        } else {
            // row 2*(b%64) holds bf16(n), row 2*(b%64)+1 holds bf16(n - hi), in the
            // 8-row x 16-byte core-matrix layout of the out_proj's B operand
            const __nv_bfloat16 hi = __float2bfloat16_rn(n);
            const __nv_bfloat16 lo = __float2bfloat16_rn(n - __bfloat162float(hi));
            uint8_t *tile = p.xb_out + ((size_t)(b >> 6) * p.kt_out + (k >> 6)) * kOpTile;
            const int kc = (k & 63) >> 3, e = k & 7;
            const int rh = 2 * (b & 63), rl = rh + 1;
            *reinterpret_cast<__nv_bfloat16 *>(tile + op_chunk_offset(rh, kc) + e * 2) = hi;
            *reinterpret_cast<__nv_bfloat16 *>(tile + op_chunk_offset(rl, kc) + e * 2) = lo;
        }
    }
}

template <int DK, int DJ>
cudaError_t launch_core(const CoreParams &cp, int js, int n_v, int B, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)js, (unsigned)n_v, (unsigned)B);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (js > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = (unsigned)js;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, dn_core_kernel<DK, DJ, true>, cp);
    }
    return cudaLaunchKernelEx(&cfg, dn_core_kernel<DK, DJ, false>, cp);
}

// Widest slice a dk allows: a block's tile (dk x DJ floats over 256 threads)
// stays at 64 registers per thread.
constexpr int max_dj_of(int dk) { return dk >= 256 ? 64 : 128; }

template <int DK>
cudaError_t dispatch_dj(const CoreParams &cp, int dj, int js, int n_v, int B, cudaStream_t st) {
    switch (dj) {
        case 16:
            if constexpr (1024 / 16 <= DK) return launch_core<DK, 16>(cp, js, n_v, B, st);
            break;
        case 32:
            if constexpr (1024 / 32 <= DK) return launch_core<DK, 32>(cp, js, n_v, B, st);
            break;
        case 64: return launch_core<DK, 64>(cp, js, n_v, B, st);
        case 128:
            if constexpr (max_dj_of(DK) >= 128) return launch_core<DK, 128>(cp, js, n_v, B, st);
            break;
        default: break;
    }
    return cudaErrorInvalidValue;
}

// Smallest legal slice width for a dk: the tile's rows per pass (1024 / DJ)
// may not exceed dk.
int min_dj(int dk) {
    int dj = 16;
    while (1024 / dj > dk) dj *= 2;
    return dj;
}

}  // namespace

// Column slices per head: enough blocks to cover every SM at least once when
// the batch is small, at most 8 (a portable cluster), at least 16 columns and
// at most max_dj_of(dk) columns each.
int choose_js(const Dims &d, int B) {
    const int sms = num_sms();
    int js = 1;
    while (d.dv / js > max_dj_of(d.dk)) js *= 2;
    const int max_js = d.dv / min_dj(d.dk);
    while (js < 8 && js * 2 <= max_js && (long)B * d.n_v * js < sms) js *= 2;
    return js;
}

cudaError_t launch_dn_core(const Dims &d, const LayerDev &L, int B, const float *g,
                           const float *beta, bool tc, cudaStream_t st) {
    CoreParams cp;
    cp.ring = L.ring;
    cp.rpos = L.rpos;
    cp.wconv_t = L.wconv_t;
    cp.w_norm = L.w_norm;
    cp.S = L.S;
    cp.nrm = L.nrm;
    cp.xb_out = tc ? L.xb_out : nullptr;
    cp.part_in = L.part_in;
    cp.nseg_in = L.nseg_in;
    cp.s_in = L.s_in;
    {
        const GemmPlan gp = plan_tc_gemm(d.proj_rows, plan_k(d, d.hidden, B), B);
        cp.sv = SchedView{gp.U, gp.G, gp.UT, gp.MT, gp.max_seg};
    }
    cp.kt_out = (d.v_dim + kTileK - 1) / kTileK;
    cp.g = g;
    cp.beta = beta;
    cp.n_qk = d.n_qk;
    cp.n_v = d.n_v;
    cp.dv = d.dv;
    cp.conv_k = d.conv_k;
    cp.conv_ch = d.conv_ch;
    cp.qk_dim = d.qk_dim;
    cp.in_rows = d.in_rows;
    cp.v_dim = d.v_dim;
    cp.l2_eps = d.l2_eps;
    cp.norm_eps = d.norm_eps;
    cp.q_scale = d.q_scale;
    cp.gw = d.gw;
    cp.dev_gates = d.dev_gates;
    cp.gate_A = L.gate_A;
    const int js = choose_js(d, B);
    const int dj = d.dv / js;
    switch (d.dk) {
        case 32: return dispatch_dj<32>(cp, dj, js, d.n_v, B, st);
        case 64: return dispatch_dj<64>(cp, dj, js, d.n_v, B, st);
        case 128: return dispatch_dj<128>(cp, dj, js, d.n_v, B, st);
        case 256: return dispatch_dj<256>(cp, dj, js, d.n_v, B, st);
        default: return cudaErrorInvalidValue;
    }
}

// ---- ring conversion between the ABI layout and the device layout ----------
namespace {

// ABI: stage[b][(rp + m) % (K-1)][c] is the m-th oldest input (m = 0..K-2).
// Device: ring[seq][(dpos + m) % K][c], with dpos reset to 0 on import.
__global__ void ring_import_kernel(float *ring, int32_t *rpos, const float *stage,
                                   const int32_t *rp_stage, int seq0, int K, int C) {
    const int b = blockIdx.z, m = blockIdx.y;
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    const int rp = rp_stage[b];
    float *dst = ring + ((size_t)(seq0 + b) * K + m) * C;
    if (c < C) {
        if (m < K - 1) {
            int src = rp + m;
            if (src >= K - 1) src -= K - 1;
            dst[c] = stage[((size_t)b * (K - 1) + src) * C + c];
        } else {
            dst[c] = 0.f;
        }
    }
    if (m == 0 && blockIdx.x == 0 && threadIdx.x == 0) {
        rpos[2 * (seq0 + b)] = 0;
        rpos[2 * (seq0 + b) + 1] = rp;
    }
}

__global__ void ring_export_kernel(const float *ring, const int32_t *rpos, float *stage,
                                   int32_t *rp_stage, int seq0, int K, int C) {
    const int b = blockIdx.z, m = blockIdx.y;  // m = 0..K-2
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    const int dpos = rpos[2 * (seq0 + b)], rp = rpos[2 * (seq0 + b) + 1];
    int src = dpos + m;
    if (src >= K) src -= K;
    int dst = rp + m;
    if (dst >= K - 1) dst -= K - 1;
    if (c < C) stage[((size_t)b * (K - 1) + dst) * C + c] = ring[((size_t)(seq0 + b) * K + src) * C + c];
    if (m == 0 && blockIdx.x == 0 && threadIdx.x == 0) rp_stage[b] = rp;
}

}  // namespace

cudaError_t launch_ring_import(const Dims &d, const LayerDev &L, int seq0, int n,
                               cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((d.conv_ch + 255) / 256), (unsigned)d.conv_k, (unsigned)n);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, ring_import_kernel, L.ring, L.rpos, (const float *)L.ring_stage,
                              (const int32_t *)L.rp_stage, seq0, d.conv_k, d.conv_ch);
}

cudaError_t launch_ring_export(const Dims &d, const LayerDev &L, int seq0, int n,
                               cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((d.conv_ch + 255) / 256), (unsigned)(d.conv_k - 1), (unsigned)n);
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    return cudaLaunchKernelEx(&cfg, ring_export_kernel, (const float *)L.ring,
                              (const int32_t *)L.rpos, L.ring_stage, L.rp_stage, seq0, d.conv_k,
                              d.conv_ch);
}

}  // namespace dn
