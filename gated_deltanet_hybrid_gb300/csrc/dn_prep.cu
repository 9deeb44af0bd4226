// Per-sequence preparation of the state update for the persistent state
// kernel (large batches): the part of the page's step ("qwen36: run the
// DeltaNet layer end to end on the card (Q36_DN_GPU=1)", section "What the
// PR does") between the in_proj GEMV and the recurrence - causal conv + SiLU
// with the ring advancing, the L2 norms of q and k - plus silu(z) and the
// gates, written as one compact record per (sequence, value head):
//   rec[(b * n_v + h) * rec_len] = [ q^ (dk) | k^ (dk) | v_h (dv) | silu(z_h) (dv) |
//                                   exp(g) | beta | 0 | 0 ]
// with q^ = q / sqrt(sum q^2 + l2_eps) * q_scale and k^ = k / sqrt(sum k^2 + l2_eps)
// (fp32 tree sums in a fixed order).
//
// One block of 128 threads per (128-row tile of the in_proj output, group of
// kPrepSeqs sequences), one output row per thread for each sequence of the
// group, so the whole step is about one wave of short independent blocks
// with every load of a thread in flight at once: a thread sums its row's
// segment partials in slot order (dn_sched.cuh) and scales them, runs the
// conv over the ring (read K-1 slots, write the newest) and SiLU, and stores
// its element into the record(s).  Heads never straddle a warp (dk, dv are
// multiples of 32 and so are the region starts), so the sums of squares of a
// q or k head are warp sums combined in a fixed order over the dk/32 warps
// of the head.
#include "dn_internal.cuh"
#include "dn_sched.cuh"

namespace dn {
namespace {

constexpr int kPrepThreads = kTileM;  // one in_proj row each
constexpr int kPrepSeqs = 4;          // sequences per block (a group never straddles a 64-chunk)

struct PrepParams {
    const float *part_in;  // in_proj segment partials
    const int *nseg_in;
    const float *s_in;
    SchedView sv;
    float *ring;           // [max_batch][conv_k][conv_ch]
    const int32_t *rpos;   // [max_batch][2]
    const float *wconv_t;  // [conv_k][conv_ch]
    const float *g, *beta; // [B][n_v]
    float *rec;            // [B][n_v][rec_len]
    int B, n_qk, n_v, dk, dv, conv_ch, qk_dim, in_rows, rec_len;
    float l2_eps, q_scale;
};

__device__ __forceinline__ float silu_f(float a) { return a / (1.0f + expf(-a)); }

template <int KC>
__global__ void __launch_bounds__(kPrepThreads, 8) dn_prep_kernel(const PrepParams p) {
    constexpr int NS = kPrepSeqs;
    __shared__ float wsum[NS][kPrepThreads / 32];
    const int tile = blockIdx.x, b0 = blockIdx.y * NS;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int c = tile * kTileM + t;
    const bool active = c < p.in_rows;
    const int cc = active ? c : 0;
    const bool conv = c < p.conv_ch;
    bool live[NS];
#pragma unroll
    for (int j = 0; j < NS; ++j) live[j] = active && b0 + j < p.B;

    // loads of data that no kernel of this step writes first (the ring was
    // last written by the previous step, rpos advanced at its end)
    float wc[KC];
#pragma unroll
    for (int m = 0; m < KC; ++m) wc[m] = (active && conv) ? __ldg(p.wconv_t + (size_t)m * p.conv_ch + cc) : 0.f;
    const float sc = active ? __ldg(p.s_in + cc) : 0.f;
    float hist[NS][KC - 1];
    int ws[NS];
#pragma unroll
    for (int j = 0; j < NS; ++j) {
        const int b = min(b0 + j, p.B - 1);
        const float *rb = p.ring + (size_t)b * KC * p.conv_ch + cc;
        int slot = p.rpos[2 * b];
#pragma unroll
        for (int m = 0; m < KC - 1; ++m) {  // oldest input first
            hist[j][m] = (live[j] && conv) ? rb[(size_t)slot * p.conv_ch] : 0.f;
            if (++slot == KC) slot = 0;
        }
        ws[j] = slot;  // the slot after the newest history slot is the oldest: overwrite it
    }
    pdl_wait();  // the in_proj partials come from the previous kernel
    pdl_trigger();

    // in_proj output: segment partials in slot order, scaled (the group lies
    // in one 64-sequence chunk, so one segment count)
    const int ptile = (b0 >> 6) * p.sv.MT + tile;
    const int ns = p.nseg_in[ptile];
    const float *pp = p.part_in + (size_t)ptile * p.sv.max_seg * (64 * kTileM) + (b0 & 63) * kTileM + t;
    float pv[NS][4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int j = 0; j < NS; ++j)
            pv[j][k] = (k < ns && live[j]) ? __ldcg(pp + (size_t)k * (64 * kTileM) + j * kTileM) : 0.f;
    float u[NS];
    const bool qk = c < 2 * p.qk_dim;
#pragma unroll
    for (int j = 0; j < NS; ++j) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) acc += pv[j][k];
        for (int k = 4; k < ns; ++k)
            if (live[j]) acc += __ldcg(pp + (size_t)k * (64 * kTileM) + j * kTileM);
        const float xv = sc * acc;
        if (conv) {
            float cv = 0.f;
#pragma unroll
            for (int m = 0; m < KC - 1; ++m) cv = fmaf(wc[m], hist[j][m], cv);
            cv = fmaf(wc[KC - 1], xv, cv);
            if (live[j]) p.ring[((size_t)(b0 + j) * KC + ws[j]) * p.conv_ch + c] = xv;
            u[j] = silu_f(cv);
        } else {
            u[j] = silu_f(xv);  // z
        }
        // sums of squares of the q and k heads
        float sq = qk ? u[j] * u[j] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        if (lane == 0) wsum[j][warp] = sq;
    }
    __syncthreads();
    if (!active) return;

    const int L = p.rec_len;
    const int group = p.n_v / p.n_qk;
#pragma unroll
    for (int j = 0; j < NS; ++j) {
        if (!live[j]) continue;
        const int b = b0 + j;
        float *rec_b = p.rec + (size_t)b * p.n_v * L;
        if (qk) {
            const int is_k = c >= p.qk_dim;
            const int cq = c - is_k * p.qk_dim;
            const int hq = cq / p.dk, o = cq - hq * p.dk;
            const int w0 = warp - (o >> 5);  // first warp of the head in this block
            float ss = 0.f;
            for (int w = 0; w < (p.dk >> 5); ++w) ss += wsum[j][w0 + w];
            const float scale = 1.0f / sqrtf(ss + p.l2_eps) * (is_k ? 1.0f : p.q_scale);
            const float val = u[j] * scale;
            for (int gh = 0; gh < group; ++gh)
                rec_b[(size_t)(hq * group + gh) * L + is_k * p.dk + o] = val;
        } else if (conv) {
            const int cv = c - 2 * p.qk_dim;
            const int h = cv / p.dv, o = cv - h * p.dv;
            rec_b[(size_t)h * L + 2 * p.dk + o] = u[j];
        } else {
            const int cz = c - p.conv_ch;
            const int h = cz / p.dv, o = cz - h * p.dv;
            float *r = rec_b + (size_t)h * L + 2 * p.dk;
            r[p.dv + o] = u[j];
            if (o < 4) {
                const float gv = o == 0 ? expf(p.g[b * p.n_v + h]) : (o == 1 ? p.beta[b * p.n_v + h] : 0.f);
                r[2 * p.dv + o] = gv;
            }
        }
    }
}

}  // namespace

int prep_record_len(const Dims &d) { return 2 * d.dk + 2 * d.dv + 4; }

cudaError_t launch_dn_prep(const Dims &d, const LayerDev &L, int B, const float *g,
                           const float *beta, cudaStream_t st) {
    PrepParams p;
    p.part_in = L.part_in;
    p.nseg_in = L.nseg_in;
    p.s_in = L.s_in;
    const GemmPlan gp = plan_tc_gemm(d.in_rows, d.hidden, B);
    p.sv = SchedView{gp.U, gp.G, gp.UT, gp.MT, gp.max_seg};
    p.ring = L.ring;
    p.rpos = L.rpos;
    p.wconv_t = L.wconv_t;
    p.g = g;
    p.beta = beta;
    p.rec = L.prep_rec;
    p.B = B;
    p.n_qk = d.n_qk;
    p.n_v = d.n_v;
    p.dk = d.dk;
    p.dv = d.dv;
    p.conv_ch = d.conv_ch;
    p.qk_dim = d.qk_dim;
    p.in_rows = d.in_rows;
    p.rec_len = prep_record_len(d);
    p.l2_eps = d.l2_eps;
    p.q_scale = d.q_scale;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((d.in_rows + kTileM - 1) / kTileM), (unsigned)((B + kPrepSeqs - 1) / kPrepSeqs));
    cfg.blockDim = dim3(kPrepThreads);
    cfg.stream = st;
    PdlAttr pdl;
    pdl.apply(cfg);
    switch (d.conv_k) {
        case 2: return cudaLaunchKernelEx(&cfg, dn_prep_kernel<2>, p);
        case 3: return cudaLaunchKernelEx(&cfg, dn_prep_kernel<3>, p);
        case 4: return cudaLaunchKernelEx(&cfg, dn_prep_kernel<4>, p);
        case 5: return cudaLaunchKernelEx(&cfg, dn_prep_kernel<5>, p);
        case 6: return cudaLaunchKernelEx(&cfg, dn_prep_kernel<6>, p);
        case 7: return cudaLaunchKernelEx(&cfg, dn_prep_kernel<7>, p);
        case 8: return cudaLaunchKernelEx(&cfg, dn_prep_kernel<8>, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dn
