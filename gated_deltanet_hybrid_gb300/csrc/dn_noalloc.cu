// dn_proj_i8_noalloc: the int8 row-scaled projection y = s * (W x) for callers
// that cannot allocate device memory.
//
// Who needs it: code that runs where it does not own the device allocator -
// for example a plug-in called from inside another runtime's memory pool or
// a tight inference loop whose memory budget was fixed up front - and so can
// call neither cudaMalloc nor anything that allocates behind its back
// (dn_create, torch).  The regular projection kernels keep their split-K
// partial sums in buffers that dn_create allocates; this variant keeps them
// in one file-scope static device array instead, so a call needs only the
// caller's inputs and outputs.
//
// It is the same work split as the CUDA-core projection (stream-K over units
// of 4 consecutive 64-wide k tiles of a 128-row tile, dn_sched.cuh; partial
// sums per segment, summed in slot order by a second kernel), but it reads W
// in the caller's row-major layout with ordinary 16-byte loads, since the
// caller cannot hand over the library's tiled copy.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "dn_device.cuh"
#include "dn_internal.cuh"
#include "dn_sched.cuh"

namespace dn {
namespace {

using dev::dot16;
using dev::i8x4_to_f32;

constexpr int kNaKU = 4;            // k tiles per unit
constexpr int kNaThreads = 512;     // one 16-byte chunk of a 128 x 64 tile each
constexpr int kNaMaxB = 8;          // sequences per call
constexpr int kNaMaxDim = 16384;    // M and K
// partial sums: [tiles][max_seg][kNaMaxB][128] floats; 1 Mi floats = 4 MiB
constexpr size_t kNaPartFloats = size_t(1) << 20;
constexpr int kNaMaxTiles = kNaMaxDim / kTileM;

// Scratch shared by every call on a device: segment partials, then the
// per-tile segment counts.  Host code must not pass this name to a kernel:
// on the host it only stands for the symbol (see scratch_ptr below).
static __device__ __align__(256) float g_na_scratch[kNaPartFloats + kNaMaxTiles];

struct NaParams {
    const int8_t *W;   // [M][K] row-major
    const float *x;    // [B][K]
    float *part;       // scratch partials
    int *nseg;         // scratch segment counts
    SchedView sv;      // units per row tile in sv.KT
    int M, K, KT, B;   // KT: 64-wide k tiles
};

// Stream-K partial sums: CTA c takes units [c*U/G, (c+1)*U/G); thread t
// covers row t/4 and 16 of the 64 k of each k tile of a unit.
__global__ void __launch_bounds__(kNaThreads) na_partials_kernel(const NaParams p) {
    const int t = threadIdx.x;
    const int c = blockIdx.x;
    const int u0 = sched_unit_start(c, p.sv), u1 = sched_unit_start(c + 1, p.sv);
    const int UT = p.sv.KT;
    const int kp = t & 3, r = t >> 2;
    float acc[kNaMaxB];
    int tile_cur = -1;
    for (int u = u0; u <= u1; ++u) {
        const int tile = u < u1 ? u / UT : -2;
        if (tile != tile_cur && tile_cur >= 0) {
            // end of a segment: combine the 4 lanes of each row, write the partial
#pragma unroll
            for (int j = 0; j < kNaMaxB; ++j) {
                float v = acc[j];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                acc[j] = v;
            }
            const int slot = c - sched_cta_of_unit(tile_cur * UT, p.sv);
            if (t == 0 && u1 >= (tile_cur + 1) * UT) p.nseg[tile_cur] = slot + 1;
            if (kp == 0) {
                float *ps = p.part + ((size_t)tile_cur * p.sv.max_seg + slot) * (kNaMaxB * kTileM);
#pragma unroll
                for (int j = 0; j < kNaMaxB; ++j)
                    if (j < p.B) ps[j * kTileM + r] = acc[j];
            }
        }
        if (u == u1) break;
        if (tile != tile_cur) {
#pragma unroll
            for (int j = 0; j < kNaMaxB; ++j) acc[j] = 0.f;
            tile_cur = tile;
        }
        const int row = tile * kTileM + r;
        const int kt0 = (u % UT) * kNaKU;
        int4 wv[kNaKU];
#pragma unroll
        for (int i = 0; i < kNaKU; ++i) {
            const int k0 = (kt0 + i) * kTileK + kp * 16;
            wv[i] = (row < p.M && kt0 + i < p.KT && k0 < p.K)
                        ? __ldcs(reinterpret_cast<const int4 *>(p.W + (size_t)row * p.K + k0))
                        : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < kNaKU; ++i) {
            const int k0 = (kt0 + i) * kTileK + kp * 16;
            if (row < p.M && kt0 + i < p.KT && k0 < p.K) {
                float fa[16];
                i8x4_to_f32((uint32_t)wv[i].x, fa);
                i8x4_to_f32((uint32_t)wv[i].y, fa + 4);
                i8x4_to_f32((uint32_t)wv[i].z, fa + 8);
                i8x4_to_f32((uint32_t)wv[i].w, fa + 12);
#pragma unroll
                for (int j = 0; j < kNaMaxB; ++j)
                    if (j < p.B) acc[j] += dot16(fa, p.x + (size_t)j * p.K + k0);
            }
        }
    }
}

// y[b][m] = s[m] * (the row tile's segment partials summed in slot order)
__global__ void na_reduce_kernel(const float *__restrict__ part, const int *__restrict__ nseg,
                                 const float *__restrict__ s, float *__restrict__ y, int M,
                                 int max_seg) {
    const int tile = blockIdx.x, b = blockIdx.y, r = threadIdx.x;
    const int m = tile * kTileM + r;
    if (m >= M) return;
    const int ns = nseg[tile];
    const float *pt = part + (size_t)tile * max_seg * (kNaMaxB * kTileM) + b * kTileM + r;
    float acc = 0.f;
#pragma unroll 4
    for (int k = 0; k < ns; ++k) acc += pt[(size_t)k * (kNaMaxB * kTileM)];
    y[(size_t)b * M + m] = s[m] * acc;
}

// Device address of g_na_scratch, looked up once per device (with that device
// current) and cached.
constexpr int kNaMaxDevices = 64;
float *g_na_ptr[kNaMaxDevices] = {};
std::mutex g_na_mu;

cudaError_t scratch_ptr(float **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kNaMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_na_mu);
    if (g_na_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_na_scratch);
        if (e != cudaSuccess) return e;
        g_na_ptr[dev] = static_cast<float *>(ptr);
    }
    *out = g_na_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace dn

extern "C" __attribute__((visibility("default"))) int dn_proj_i8_noalloc(
    const int8_t *W, const float *s, const float *x, float *y, int M, int K, int B, void *stream) {
    using namespace dn;
    if (W == nullptr || s == nullptr || x == nullptr || y == nullptr) return DN_EINVAL;
    if (M < 1 || M > kNaMaxDim || K < 16 || K > kNaMaxDim || K % 16 != 0) return DN_EINVAL;
    if (B < 1 || B > kNaMaxB) return DN_EINVAL;
    if (((uintptr_t)W | (uintptr_t)x) & 15u) return DN_EINVAL;  // 16-byte loads
    const int MT = (M + kTileM - 1) / kTileM;
    const int KT = (K + kTileK - 1) / kTileK;
    const int UT = (KT + kNaKU - 1) / kNaKU;
    const int U = MT * UT;
    const int G = std::min(num_sms(), U);
    const int max_seg = (UT + U / G - 1) / (U / G) + 1;
    if ((size_t)MT * max_seg * kNaMaxB * kTileM > kNaPartFloats) return DN_EINVAL;  // scratch too small
    float *scratch = nullptr;
    if (scratch_ptr(&scratch) != cudaSuccess) return DN_ECUDA;
    NaParams p;
    p.W = W;
    p.x = x;
    p.part = scratch;
    p.nseg = reinterpret_cast<int *>(scratch + kNaPartFloats);
    p.sv = SchedView{U, G, UT, MT, max_seg};
    p.M = M;
    p.K = K;
    p.KT = KT;
    p.B = B;
    const cudaStream_t st = (cudaStream_t)stream;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(kNaThreads);
    cfg.stream = st;
    if (cudaLaunchKernelEx(&cfg, na_partials_kernel, p) != cudaSuccess) return DN_ECUDA;
    cudaLaunchConfig_t rc = {};
    rc.gridDim = dim3((unsigned)MT, (unsigned)B);
    rc.blockDim = dim3(kTileM);
    rc.stream = st;
    if (cudaLaunchKernelEx(&rc, na_reduce_kernel, (const float *)p.part, (const int *)p.nseg, s, y, M,
                           max_seg) != cudaSuccess)
        return DN_ECUDA;
    return DN_OK;
}
