// A stack of gated-DeltaNet layers stepped one token at a time, with an
// unweighted RMS pre-norm before each layer and a residual add after it:
//   h <- h + layer_l(h / sqrt(mean(h^2) + eps))      for l = 0 .. n-1
// (the pages' 30 DeltaNet layers of the model, page "qwen36: run the
// DeltaNet layer end to end on the card (Q36_DN_GPU=1)", section "Measured";
// the stack between the layers is the residual stream of a decoder).
//
// The layers run through their own dn_step; between two layers one kernel
// adds the layer's output into the residual stream h and writes the next
// layer's normalised input in the same pass (one block per sequence, fp32
// sums of squares in a fixed tree order).
#include <cuda_runtime.h>

#include "dn_internal.cuh"

namespace dn {
namespace {

constexpr int kNormThreads = 256;

// h += add (if add != NULL); xn = h / sqrt(mean(h^2) + eps)
__global__ void __launch_bounds__(kNormThreads) residual_prenorm_kernel(float *__restrict__ h,
                                                                        const float *__restrict__ add,
                                                                        float *__restrict__ xn, int hidden,
                                                                        float eps) {
    __shared__ float wsum[kNormThreads / 32];
    pdl_trigger();  // the next layer's first kernels may be launched already
    pdl_wait();     // h and add come from the previous kernels
    float *hb = h + (size_t)blockIdx.x * hidden;
    const float *ab = add == nullptr ? nullptr : add + (size_t)blockIdx.x * hidden;
    float ss = 0.f;
    for (int i = threadIdx.x; i < hidden; i += kNormThreads) {
        float v = hb[i];
        if (ab != nullptr) {
            v += ab[i];
            hb[i] = v;
        }
        ss = fmaf(v, v, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) tot += wsum[w];
    const float inv = 1.0f / sqrtf(tot / (float)hidden + eps);
    float *xb = xn + (size_t)blockIdx.x * hidden;
    for (int i = threadIdx.x; i < hidden; i += kNormThreads) xb[i] = hb[i] * inv;
}

}  // namespace

cudaError_t launch_residual_prenorm(float *h, const float *add, float *xn, int B, int hidden, float eps,
                                    cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)B);
    cfg.blockDim = dim3(kNormThreads);
    cfg.stream = st;
    PdlAttr pdl;
    pdl.apply(cfg);
    return cudaLaunchKernelEx(&cfg, residual_prenorm_kernel, h, add, xn, hidden, eps);
}

}  // namespace dn
