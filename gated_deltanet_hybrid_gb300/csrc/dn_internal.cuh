// Internal declarations shared by the translation units of libdn.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dn.h"

namespace dn {

// Device-side layout of one layer.  All buffers are owned by the layer.
//   w_in    int8 [in_rows][hidden]           (as given)
//   s_in    f32  [in_rows]
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
//   qkvz    f32  [max_batch][in_rows]        in_proj output (scratch)
//   nrm     f32  [max_batch][v_dim]          gated-RMSNorm output (scratch)
struct Dims {
    int hidden, n_qk, n_v, dk, dv, conv_k, max_batch;
    int qk_dim, v_dim, conv_ch, in_rows;
    float l2_eps, norm_eps, q_scale;
};

struct LayerDev {
    int8_t *w_in;
    float *s_in, *wconv_t, *w_norm;
    int8_t *w_out;
    float *s_out;
    float *S, *ring;
    int32_t *rpos;
    float *qkvz, *nrm;
    // staging used by dn_step with host pointers and by the state copies
    float *x_stage, *g_stage, *beta_stage, *out_stage;
    float *ring_stage;     // [max_batch][conv_k-1][conv_ch]
    int32_t *rp_stage;     // [max_batch]
    // tensor-core projections: split-K partials, per-tile arrival counters
    float *part_in, *part_out;
    int *cnt_in, *cnt_out;
    int *err;              // device-side error word (bounded waits that gave up)
};

// y[b][o] = s[o] * sum_k W[o][k] * x[b][k] for b < B.  Optionally advances
// the per-sequence ring positions of `rpos` for b < B (done by block 0).
cudaError_t launch_gemv_i8(const int8_t *W, const float *s, const float *x, float *y, int M,
                           int K, int B, int32_t *rpos_advance, int conv_k, cudaStream_t st);

// Tensor-core (tcgen05) version of the same projection for batches >= 8.
bool tc_gemm_supported(int M, int K);
int tc_gemm_splits(int M, int K, int B);
cudaError_t launch_gemm_i8_tc(const int8_t *W, const float *s, const float *x, float *y,
                              float *part, int *counters, int *err, int M, int K, int B, int ks,
                              int32_t *rpos_advance, int conv_k, cudaStream_t st);
constexpr int kTcMinBatch = 8;

// The fused conv / L2 / gated-delta / readout / gated-RMSNorm step.
cudaError_t launch_dn_core(const Dims &d, const LayerDev &L, int B, const float *g,
                           const float *beta, cudaStream_t st);

// ring conversion between the ABI's conv_k-1 slots and the device's conv_k slots
cudaError_t launch_ring_import(const Dims &d, const LayerDev &L, int seq0, int n,
                               cudaStream_t st);
cudaError_t launch_ring_export(const Dims &d, const LayerDev &L, int seq0, int n,
                               cudaStream_t st);

int num_sms();

}  // namespace dn
