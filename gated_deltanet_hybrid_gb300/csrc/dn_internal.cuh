// Internal declarations shared by the translation units of libdn.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/dn.h"

namespace dn {

// Device-side layout of one layer.  All buffers are owned by the layer.
//   w_in    int8 [proj_rows][hidden]         (the in_proj rows, then the a/b gate rows)
//   s_in    f32  [proj_rows]
//   wconv_t f32  [conv_k][conv_ch]           (transposed: one tap is a contiguous row)
//   w_norm  f32  [dv]
//   w_out   int8 [hidden][v_dim]
//   s_out   f32  [hidden]
//   S       f32  [max_batch][n_v_heads][dk][dv]
//   ring    f32  [max_batch][conv_k][conv_ch] conv_k slots: the conv_k-1 inputs the
//                                             next step reads plus one slot that the
//                                             step writes, so no step ever writes a
//                                             slot that another block of the same
//                                             step reads
//   rpos    i32  [max_batch][2]              {slot of the oldest input in `ring`,
//                                             ring_pos as seen through the ABI}
//   nrm     f32  [max_batch][v_dim]          gated-RMSNorm output (scratch)
struct Dims {
    int hidden, n_qk, n_v, dk, dv, conv_k, max_batch;
    int qk_dim, v_dim, conv_ch, in_rows;
    int gw;  // log-decay values per head and step: dk with the per-key gate, else 1
    int dev_gates;  // the a/b gate rows follow the in_proj rows (DN_FLAG_DEVICE_GATES)
    int proj_rows;  // rows of the in_proj GEMM: in_rows, plus n_v * (gw + 1) gate rows
    int i4;         // int4 weights (DN_FLAG_INT4_WEIGHTS)
    float l2_eps, norm_eps, q_scale;
};

struct LayerDev {
    uint8_t *w_in;  // tiled int8 (see kTileM / kTileK)
    uint8_t *w_in4, *w_out4;  // int4 layers: the packed int4 tiles the CUDA-core GEMV streams
    float *s_in, *wconv_t, *w_norm;
    float *gate_A;  // [n_v] (device gates only)
    uint8_t *w_out;  // tiled int8
    float *s_out;
    float *S, *ring;
    int32_t *rpos;
    float *nrm;
    // staging used by dn_step with host pointers and by the state copies
    float *x_stage, *g_stage, *beta_stage, *out_stage;
    float *ring_stage;     // [max_batch][conv_k-1][conv_ch]
    int32_t *rp_stage;     // [max_batch]
    // tensor-core projections: split-K partials, per-tile arrival counters
    float *part_in, *part_out;
    int *nseg_in, *nseg_out;  // segments per tile of the last projection launch
    uint8_t *xb_in;        // packed B-operand tiles of x   [chunks][KT_in][16 KB]
    uint8_t *xb_out;       // packed B-operand tiles of the gated-norm output [chunks][KT_out][16 KB]
    int *err;              // device-side error word (bounded waits that gave up)
    int *pool;             // the state kernel's item-pool counter (zero between steps)
};

// Prompt processing (dn_prefill) works on blocks of up to kPrefillCols token
// columns: nb sequences x T tokens each, column j = sequence j / T, token
// j % T of the block.  Its scratch is allocated on the first dn_prefill call.
// (512 columns against 256: each head's state moves in and out of the
// recurrence once per 64 tokens of an 8-sequence prompt instead of 32, and
// half as many launches; 8 x 2048 tokens 1.94 -> 2.37 M tokens/s.)
constexpr int kPrefillCols = 512;
struct PrefillDev {
    float *xg;                 // [cols][hidden] the block's x rows
    uint8_t *xb_in;            // packed bf16 hi/lo tiles of xg (tensor-core in_proj)
    float *part_in;            // in_proj segment partials, and their counts
    int *nseg_in;
    float *xin;                // [cols][proj_rows] in_proj output, scaled
    float *qn, *kn;            // [nb][n_qk][T][dk] normalised q (times q_scale) and k
    float *vv, *zs;            // [nb][n_v][T][dv] v after conv + SiLU, silu(z)
    float *gg, *bb;            // [nb][n_v][T][gw] log-decays, [nb][n_v][T] write strengths
    float *o;                  // [nb][n_v][T][dv] readouts
    float *nrm;                // [cols][v_dim] gated-norm output (CUDA-core out_proj)
    uint8_t *xb_out;           // its packed tiles (tensor-core out_proj)
    float *part_out;
    int *nseg_out;
};

// One block of a prompt: sequences [b0, b0 + nb) of the layer, tokens
// [t0, t0 + T) of S; x, g, beta, out are the caller's [batch][S][...] arrays
// (g, beta NULL with device gates).
struct PrefillBlock {
    int b0, nb, t0, T, S;
    const float *x, *g, *beta;
    float *out;
};
cudaError_t launch_prefill_block(const Dims &d, const LayerDev &L, const PrefillDev &P, const PrefillBlock &blk,
                                 cudaStream_t st);

// Weight tiles used by every projection kernel: W [M][K] int8 is stored as
// [ceil(M/128)][ceil(K/64)][4 k parts][128 rows][16 int8], zero-padded, one
// 8 KB contiguous block per (m tile, k tile); k part p holds k 16p..16p+15 of
// the tile.  A warp reading 16 bytes per lane for 32 consecutive rows of one
// k part (or 8 rows x 4 parts, 8 lanes per part) touches 512 contiguous
// bytes per part, so shared-memory reads of a tile are free of bank conflicts.
constexpr int kTileM = 128;
constexpr int kTileK = 64;

// Both projection kernels leave unscaled per-segment partial sums of their
// stream-K schedule (dn_sched.cuh) in `part`; the consumer sums a tile's
// slots in slot order and applies the row scale: the core kernel for the
// in_proj, launch_splitk_reduce for the out_proj.
//
// CUDA-core version for batches < kTcMinBatch (fp32 activations x [B][K]).
// i4: Wt holds int4 tiles ([ceil(M/128)][ceil(K/128)][4 parts][128 rows][16 B],
// each 16-byte chunk 32 weights of one row, low nibble first).
cudaError_t launch_gemv_i8(const uint8_t *Wt, const float *x, float *part, int *nseg, int *err,
                           int M, int K, int B, cudaStream_t st, bool i4 = false);

// Batches from kTcMinBatch sequences (or prompt columns) take the tensor-core
// projections; below, the CUDA-core GEMV.  Measured on the 35B-shape layer:
// at batch 1 the GEMV step takes 20.5 us against 29.6 on the tensor cores,
// from batch 2 the tensor cores win (23.5 against 29.9 us at batch 2, 27.6
// against 83.0 at batch 7: the GEMV's conversion and FMA work grows with the
// batch, the tensor-core pipeline's does not).
constexpr int kTcMinBatch = 2;

// Tensor-core (tcgen05) version for batches >= kTcMinBatch: x arrives packed
// as bf16 hi/lo B-operand tiles (launch_pack_b, or written so by the core
// kernel).
// A schedule unit is KU consecutive 64-wide k tiles of one 128-row tile (the
// CUDA-core kernel, KU = 4) or of a pair of row tiles that share the
// activation operand (the tensor-core kernel, KU = 2, when there are enough
// units).  MP = row-tile groups of TP tiles, UT = units per group; partial
// sums are kept per row tile (MT tiles, up to max_seg segment slots each).
struct GemmPlan {
    int MT, TP, MP, KT, KU, UT, nchunks, U, G, max_seg, tiles;
};
GemmPlan plan_tc_gemm(int M, int K, int B);
// The k extent a projection of `B` columns is planned with: the CUDA-core
// GEMV of an int4 layer streams int4 tiles, 8 KB of which hold 128 k (the
// schedule of K/2 int8 columns); every other projection plans K.
inline int plan_k(const Dims &d, int K, int B) { return (d.i4 && B < kTcMinBatch) ? K / 2 : K; }
cudaError_t launch_pack_b(const float *x, uint8_t *xb, int B, int K, cudaStream_t st);
cudaError_t launch_gemm_i8_tc(const uint8_t *Wt, const uint8_t *xb, float *part, int *nseg, int *err,
                              int M, int K, int B, cudaStream_t st);
// y = s * (sum of partials); also advances ring positions (rpos_advance !=
// NULL).  Column j of the projection goes to row (j / T) * Sr + t0 + j % T of
// y and the B / T sequences' ring positions advance by `adv` (decode: the
// defaults, row j, one step).
cudaError_t launch_splitk_reduce(const float *part, const int *nseg, const float *s, float *y, int M,
                                 int K, int B, int32_t *rpos_advance, int conv_k, cudaStream_t st, int T = 1,
                                 int Sr = 1, int t0 = 0, int adv = 1, int *pool_reset = nullptr);
constexpr size_t kOpTile = 16384;  // bytes of one packed B-operand tile (64 seqs x 64 k, hi+lo)
// Byte offset, inside a packed B-operand tile (128 operand rows x 64 bf16;
// row 2b = hi, row 2b+1 = lo of sequence b), of the 16-byte chunk holding
// k 8*kc .. 8*kc+7 of operand row `row`.  The tile uses the 128-byte swizzled
// K-major layout: each row's 128 bytes contiguous, 8-row groups 1024 bytes
// apart, chunk kc of row r at chunk position kc ^ (r & 7).
__host__ __device__ __forceinline__ uint32_t op_chunk_offset(int row, int kc) {
    return (uint32_t)(row >> 3) * 1024u + (uint32_t)(row & 7) * 128u + ((uint32_t)(kc ^ (row & 7)) << 4);
}

// The fused conv / L2 / gated-delta / readout / gated-RMSNorm step.
// The in_proj result is read as the sum of its segment partials (part_in,
// scaled by s_in).  tc: the gated-norm output is written as packed B-operand
// tiles (xb_out) for the tensor-core out_proj instead of fp32 rows (nrm).
cudaError_t launch_dn_core(const Dims &d, const LayerDev &L, int B, const float *g,
                           const float *beta, bool tc, cudaStream_t st);

// Persistent bulk-copy-pipelined variant of the same step for large batches
// of 128 x 128 heads (conv_k <= 4).
bool dn_core_stream_ok(const Dims &d, int B);
cudaError_t launch_dn_core_stream(const Dims &d, const LayerDev &L, int B, const float *g,
                                  const float *beta, bool tc, cudaStream_t st);

// ring conversion between the ABI's conv_k-1 slots and the device's conv_k slots
cudaError_t launch_ring_import(const Dims &d, const LayerDev &L, int seq0, int n,
                               cudaStream_t st);
cudaError_t launch_ring_export(const Dims &d, const LayerDev &L, int seq0, int n,
                               cudaStream_t st);

int num_sms();

// dn_debug_expire_wait: one bounded wait that runs out after limit_us and
// sets the device error word (dn_debug.cu)
cudaError_t launch_expire_wait(int *err, int limit_us, cudaStream_t st);

// h += add (add may be NULL); xn = h / sqrt(mean(h^2) + eps), per sequence
cudaError_t launch_residual_prenorm(float *h, const float *add, float *xn, int B, int hidden, float eps,
                                    cudaStream_t st);

// Programmatic dependent launch.  Every kernel of a step is launched with
// the programmatic-serialization attribute (with_pdl), so it may start while
// the kernel before it is still running.  A kernel may only read read-only
// data (weights, the recurrent state when the previous kernel does not touch
// it) before pdl_wait(), which returns once the previous kernel has
// completed and its writes are visible.  Every kernel calls pdl_wait() before
// it completes, so "completed" is transitive down the chain: once a kernel's
// wait returns, every earlier kernel of the stream has completed too.  That
// lets the small kernels ahead of a projection (packing the activations, the
// out_proj reduction) signal pdl_trigger() first thing, so that the
// projection's CTAs are launched, and stream their weights, while those
// kernels still wait or run; the others signal it after their own wait.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Runs `set(device)` the first time a function is launched on each device
// (ordinals below 64; beyond that, every time): for per-function attributes
// such as a large dynamic shared-memory size.  Safe when several host
// threads launch on several devices.
template <typename Set>
cudaError_t once_per_device(std::atomic<uint64_t> &done, Set set) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t{1} << dev) : 0;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    e = set(dev);
    if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
    return e;
}

struct PdlAttr {
    cudaLaunchAttribute a[1];
    void apply(cudaLaunchConfig_t &cfg) {
        a[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        a[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = a;
        cfg.numAttrs = 1;
    }
};

}  // namespace dn
