// int8 (or int4) row-scaled GEMV on the CUDA cores for small batches:
//   y[b][o] = s[o] * sum_k W[o][k] * x[b][k]
// (int4 layers: the same 8 KB tiles hold 128 k, 32 weights per 16-byte
// chunk, decoded exactly to fp32 in registers; the bytes to stream halve)
//
// The projections of the gated-DeltaNet step are int8 matrices with one fp32
// scale per output row (page "feat(qwen36): the dense trunk places itself",
// section "What this adds", item 1; the in_proj holds the q, k, v rows and
// the z rows in one matrix, so one GEMV serves both).  At small batch the step is a weight stream: the kernel
// is built so that every SM keeps about 128 KB of weights in flight.
//
// W is stored as contiguous 8 KB tiles of 128 rows x 64 int8 in four 16-k
// parts (dn_internal.cuh; shared with the tensor-core kernel) and the work is
// split exactly like the tensor-core projection (stream-K, dn_sched.cuh): up
// to one CTA per SM (two at batch 1), as few as keep every CTA at the same
// unit count, each takes a contiguous range of units, each unit 4
// consecutive k tiles of one row tile (32 KB).  The weights stream straight into registers: lane l
// of warp w loads 16 bytes (16 weights of row 8w + l%8, k part l/8) of each
// tile with a 16-byte load, so a warp reads 4 x 128 contiguous bytes, and the
// loads of the next D units are always in flight (a software pipeline over
// register slots; the loads are volatile so the compiler keeps them where
// they are issued); at batch 1 two CTAs per SM keep 8 warps per scheduler to
// hide the latency of the conversion and FMA chains.  Bulk copies into shared memory were tried first: at
// batch 1 the copies of one SM complete one after another and the weights
// stream at about half the HBM bandwidth.  Each lane converts int8 exactly
// to fp32 and multiplies with the fp32 activations (read through L1) in
// four independent FMA chains, one accumulator per (row, sequence).  At the
// end of each segment the four lanes of a row (8 apart) are combined in a
// fixed shuffle order and the unscaled partial goes to its slot, to be summed
// and scaled by the consumer in slot order (bitwise-reproducible results).
#include <algorithm>

#include "dn_device.cuh"
#include "dn_internal.cuh"
#include "dn_sched.cuh"

namespace dn {
namespace {

using dev::dot16x2;
using dev::i4x8_to_f32x2;
using dev::i8x4_to_f32x2;

constexpr int KU = 4;                    // 64-wide k tiles per unit (32 KB of weights)
// units in flight per thread, and CTAs per SM: one sequence leaves registers
// for two CTAs per SM (8 warps per scheduler), more sequences need them for
// their accumulators
template <int NB> struct Pipe { static constexpr int D = 4, CTAS = 1; };
template <> struct Pipe<1> { static constexpr int D = 2, CTAS = 2; };
constexpr int kThreads = 512;            // one 16-byte chunk of each 8 KB tile each
constexpr uint32_t kTile = kTileM * kTileK;  // 8 KB

struct GemvParams {
    const uint8_t *Wt;
    const float *x;   // [B][K]
    float *part;      // [tiles][max_seg][64][128]
    int *nseg;        // [tiles]
    SchedView sv;     // units per row tile in sv.KT
    int K, B, KTt;    // KTt: 64-wide k tiles per row
};

__device__ __forceinline__ uint4 ld_stream(const uint8_t *ptr) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr));
    return v;
}

// this thread's 16-byte chunk of each k tile of unit u.  The loads are
// unconditional (a k tile past the row's last one re-reads the last, and the
// compute skips it): a select on a value still in flight would wait for it.
__device__ __forceinline__ void load_unit(const GemvParams &p, int u, int kp, int r, uint4 w[KU]) {
    const int KT = p.sv.KT;
    const int mt = (u / KT) % p.sv.MT, kt0 = (u % KT) * KU;
    const uint8_t *row = p.Wt + (size_t)mt * p.KTt * kTile + kp * 2048 + r * 16;
#pragma unroll
    for (int i = 0; i < KU; ++i) w[i] = ld_stream(row + (size_t)min(kt0 + i, p.KTt - 1) * kTile);
}

template <int NB, bool I4>
__global__ void __launch_bounds__(kThreads, Pipe<NB>::CTAS) gemv_i8_stream_kernel(const GemvParams p) {
    constexpr int TK = I4 ? 128 : kTileK;  // k per tile
    constexpr int PK = TK / 4;             // k per 16-byte part
    constexpr int D = Pipe<NB>::D;
    const int t = threadIdx.x;
    const int c = blockIdx.x;
    const int u0 = sched_unit_start(c, p.sv), u1 = sched_unit_start(c + 1, p.sv);
    const int KT = p.sv.KT;
    // lane l of warp w: k part l/8 (16 of the tile's 64 k) of row 8w + l%8
    const int kp = (t >> 3) & 3;
    const int r = (t >> 5) * 8 + (t & 7);

    // the weights do not depend on the previous kernel: the first D units
    // are requested before waiting for it
    uint4 w[D][KU];
#pragma unroll
    for (int d = 0; d < D; ++d)
        if (u0 + d < u1) load_unit(p, u0 + d, kp, r, w[d]);
    pdl_wait();  // x and the partial buffers: after the previous kernel
    if (t == 0) pdl_trigger();

    float acc[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j) acc[j] = 0.f;
    int tile_cur = u0 < u1 ? u0 / KT : -1;
    for (int ub = u0; ub < u1; ub += D) {
#pragma unroll
        for (int d = 0; d < D; ++d) {
            const int u = ub + d;
            if (u >= u1) break;
            const int tile = u / KT;
            if (tile != tile_cur) {
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
#pragma unroll
                for (int j = 0; j < NB; ++j) acc[j] = 0.f;
                tile_cur = tile;
            }
            const int kt0 = (u % KT) * KU;
#pragma unroll
            for (int i = 0; i < KU; ++i) {
                const int k0 = (kt0 + i) * TK + kp * PK;
                if (kt0 + i < p.KTt && k0 < p.K) {
                    // weights as fp32 pairs and pair FMAs (dev::dot16x2: the bits
                    // of the scalar chains in half the instructions)
                    if constexpr (!I4) {
                        uint64_t wp[8];
                        i8x4_to_f32x2(w[d][i].x, wp[0], wp[1]);
                        i8x4_to_f32x2(w[d][i].y, wp[2], wp[3]);
                        i8x4_to_f32x2(w[d][i].z, wp[4], wp[5]);
                        i8x4_to_f32x2(w[d][i].w, wp[6], wp[7]);
#pragma unroll
                        for (int jb = 0; jb < NB; ++jb)
                            if (jb < p.B) acc[jb] += dot16x2(wp, p.x + (size_t)jb * p.K + k0);
                    } else {
                        // 32 weights: k0 .. k0+15 (K is a multiple of 16), then k0+16 ..
                        uint64_t wp[8];
                        i4x8_to_f32x2(w[d][i].x, wp);
                        i4x8_to_f32x2(w[d][i].y, wp + 4);
#pragma unroll
                        for (int jb = 0; jb < NB; ++jb)
                            if (jb < p.B) acc[jb] += dot16x2(wp, p.x + (size_t)jb * p.K + k0);
                        if (k0 + 16 < p.K) {
                            i4x8_to_f32x2(w[d][i].z, wp);
                            i4x8_to_f32x2(w[d][i].w, wp + 4);
#pragma unroll
                            for (int jb = 0; jb < NB; ++jb)
                                if (jb < p.B) acc[jb] += dot16x2(wp, p.x + (size_t)jb * p.K + k0 + 16);
                        }
                    }
                }
            }
            // refill the slot with the unit D ahead
            if (u + D < u1) load_unit(p, u + D, kp, r, w[d]);
        }
    }
    if (tile_cur >= 0) {  // the last segment
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
}

template <int NB, bool I4>
cudaError_t launch_nb(const uint8_t *Wt, const float *x, float *part, int *nseg, int M, int K, int B,
                      cudaStream_t st) {
    const GemmPlan g = plan_tc_gemm(M, I4 ? K / 2 : K, B);  // int4: 128 k per tile
    GemvParams p;
    p.Wt = Wt;
    p.x = x;
    p.part = part;
    p.nseg = nseg;
    p.sv = SchedView{g.U, g.G, g.UT, g.MT, g.max_seg};
    p.K = K;
    p.B = B;
    p.KTt = g.KT;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)g.G);
    cfg.blockDim = dim3(kThreads);
    cfg.stream = st;
    PdlAttr pdl;
    pdl.apply(cfg);
    return cudaLaunchKernelEx(&cfg, gemv_i8_stream_kernel<NB, I4>, p);
}

template <bool I4>
cudaError_t launch_gemv_b(const uint8_t *Wt, const float *x, float *part, int *nseg, int M, int K, int B,
                          cudaStream_t st) {
    if (B == 1) return launch_nb<1, I4>(Wt, x, part, nseg, M, K, B, st);
    if (B == 2) return launch_nb<2, I4>(Wt, x, part, nseg, M, K, B, st);
    if (B <= 4) return launch_nb<4, I4>(Wt, x, part, nseg, M, K, B, st);
    return launch_nb<8, I4>(Wt, x, part, nseg, M, K, B, st);
}

}  // namespace

cudaError_t launch_gemv_i8(const uint8_t *Wt, const float *x, float *part, int *nseg, int *err,
                           int M, int K, int B, cudaStream_t st, bool i4) {
    (void)err;  // no waits: nothing to report
    return i4 ? launch_gemv_b<true>(Wt, x, part, nseg, M, K, B, st)
              : launch_gemv_b<false>(Wt, x, part, nseg, M, K, B, st);
}

}  // namespace dn
