// int8 row-scaled projection on the 5th-generation tensor cores (tcgen05),
// for batches large enough that the GEMV becomes a dense contraction:
//   y[b][m] = s[m] * sum_k W[m][k] * x[b][k]
// (the fused in_proj of q, k, v and z rows and the out_proj of the step;
// int8 rows with one fp32 scale each, page "feat(qwen36): the dense trunk
// places itself", section "What this adds", item 1).
//
// Precision.  int8 weights are exact in bf16.  The fp32 activations arrive
// split into x = hi + lo with hi = bf16(x), lo = bf16(x - hi) (pack_b below),
// so W*hi + W*lo reproduces W*x to about 2^-17 relative per term, with fp32
// accumulation in tensor memory.  hi and lo of sequence b are rows 2b and
// 2b+1 of the MMA's B operand (N = 2 * padded batch), so one MMA covers both
// and the epilogue adds accumulator columns 2b and 2b+1.
//
// Layouts.  The layer stores W as contiguous 8 KB tiles [m tile][k tile]
// (128 rows x 64 int8 in four 16-k parts, dn_internal.cuh) and the
// activations as 16 KB tiles [batch chunk][k tile] holding 128 B-operand
// rows of 64 bf16 in the 128-byte swizzled K-major layout (op_chunk_offset).
// So every pipeline stage is two 1-D bulk copies (cp.async.bulk, completed
// on an mbarrier), and the k tiles of a row tile stream through HBM
// sequentially.  The converted weights never go back to shared memory: the
// converters store them into tensor memory (tcgen05.st), and the MMA takes
// its A operand from there, so shared memory only carries the copies, the
// converters' int8 reads and the MMA's B reads.
//
// Work split (stream-K).  A unit is one (batch chunk, m tile, k tile).  The
// grid has at most one CTA per SM, G = the fewest that keep each CTA at
// ceil(U / SMs) units; CTA c takes the contiguous unit range
// [c*U/G, (c+1)*U/G), so all CTAs get (nearly) the same number of units
// whatever the tile count.  A range covers the tail of one m tile and the
// head of the next (a "segment" each); two TMEM accumulators alternate
// between segments.
// Every segment's partial sums go to a slot of a partial buffer (schedule in
// dn_sched.cuh); the consumer sums a tile's slots in slot order (the state
// kernel for the in_proj, splitk_reduce_kernel for the out_proj), so
// results do not depend on scheduling and no CTA waits on another.
//
// A unit is one or two row tiles (TP) x 128 k: per row tile 16 KB of int8
// weights, one bulk copy (copies this size keep the per-copy hand-off cost
// small against the HBM time).
// Weights and activations stream through separate shared-memory rings: the
// converters free a weight stage as soon as they hold its bytes in
// registers, so up to six weight copies are in flight per SM however long
// the MMAs of a unit take; activation stages are freed by the MMAs.
// Roles (28 warps): warp 0 copies weights, warp 26 copies activations,
// warps 1 and 27 (one thread each) issue the MMAs of the first and second
// row tile of a unit (two issuers: in this kernel a single thread issuing
// both tiles' MMAs paces the whole pipeline), warps 2-17 convert the int8
// unit to bf16 into one of two tensor-memory A buffers (warp w owns lane
// quarter w % 4 and 64 k of one row tile: one row per lane), warps 18-25
// read the accumulators (tcgen05.ld) and write results.  Tensor memory (all
// 512 columns): the two row tiles' accumulators in columns 0-255, A buffers
// in 256-511.  The weight producer does not wait for the previous kernel of
// the step (programmatic dependent launch): weights are read-only, the
// activations and the partial buffers are not.
// Every wait is bounded (about one second of the global timer): on timeout
// the kernel records an error in `err`, waits (bounded) for its own copies
// and MMAs in flight, frees its tensor memory and returns.
#include <cuda_bf16.h>

#include <algorithm>

#include "dn_device.cuh"
#include "dn_internal.cuh"
#include "dn_sched.cuh"

namespace dn {
namespace {

using dev::bulk_g2s;
using dev::global_ns;
using dev::mbar_arrive;
using dev::mbar_arrive_expect_tx;
using dev::mbar_init;
using dev::instr_desc;
using dev::mma_bf16_ts_x4;
using dev::mma_commit;
using dev::smem_desc_sw128;
using dev::smem_u32;
using dev::tc_fence_after;
using dev::tc_fence_before;
using dev::tmem_ld16;
using dev::tmem_st32;

constexpr int BM = 128;          // weight rows per tile (MMA M)
constexpr int BK = 64;           // k per weight tile
constexpr int KU = 2;            // k tiles per unit (128 k)
constexpr int AST = 3;           // int8 weight stages (2 row tiles x 16 KB)
constexpr int BST = 3;           // bf16 activation stages (32 KB)
constexpr int NB_CHUNK = 64;     // sequences per batch chunk (MMA N <= 128)
constexpr int kConvWarps = 16;
constexpr int kEpiWarps = 8;
constexpr int kEpiWarp0 = 2 + kConvWarps;
constexpr int kBProdWarp = kEpiWarp0 + kEpiWarps;
constexpr int kMma1Warp = kBProdWarp + 1;            // the second row tile's MMA issuer
constexpr int kThreads = 32 * (kMma1Warp + 1);       // 28 warps
constexpr int NABUF = 2;                             // tensor-memory A buffers (one pair unit each)
constexpr uint32_t kATileBytes = BM * BK;            // 8 KB int8
constexpr uint32_t kAUnitBytes = KU * kATileBytes;   // 16 KB: one row tile of a unit
constexpr uint32_t kOpTileBytes = 128 * BK * 2;      // 16 KB bf16
constexpr uint32_t kTmemCols = 512;                  // 2 accumulators x 128 + 2 A buffers x 128
constexpr uint32_t kTmemA = 256;                     // first column of the A buffers
constexpr uint32_t kACols = 2 * KU * BK / 2;         // 128: bf16 pairs of two 128-k row tiles
constexpr uint64_t kWaitLimitNs = 1000000000ull;
// A waiting thread is suspended until the phase completes or this many ns
// pass, so waiting warps leave the issue slots to the working ones (the
// single MMA-issuing thread above all).
constexpr uint32_t kSuspendHintNs = 20000;

// A unit is 2 row tiles x 128 k: 2 x 16 KB of int8 weights and one 32 KB
// activation tile that both row tiles use.
struct __align__(1024) GemmSmem {
    uint8_t b16[BST][KU * kOpTileBytes];     // bf16 B operand as copied (3 x 32 KB)
    uint8_t a8[AST][2][kAUnitBytes];         // int8 A as copied (3 x 2 x 16 KB)
    uint64_t a_full[AST];                    // weight copies of the stage landed
    uint64_t a_empty[AST];                   // converters done reading the stage (one arrival per warp)
    uint64_t b_full[BST];                    // activation copies of the stage landed
    uint64_t b_empty[BST];                   // MMAs done reading the stage
    uint64_t conv[NABUF];                    // A converted into tensor-memory buffer i (one arrival per converter warp)
    uint64_t a_free[NABUF];                  // MMAs done reading tensor-memory A buffer i
    uint64_t acc_full;                       // accumulators ready for the epilogue (one commit per issuer)
    uint64_t acc_empty;                      // epilogue done reading the accumulators (one arrival per warp)
    uint64_t drain[2];                       // all MMAs of an issuer completed
    uint32_t tmem_base;
    int abort_flag;
};

struct GemmParams {
    const uint8_t *Wt;   // int8 weight tiles
    const uint8_t *xb;   // bf16 B tiles [nchunks][KT][16 KB]
    float *part;         // [tiles][max_seg][64][128] segment partials (unscaled)
    int *nseg;           // [tiles] segment count, written by each tile's last segment
    int *err;
    int M, MT, MP, TP, KT, UT, B, nchunks, U, G, max_seg;  // MP row-tile groups of TP (1 or 2) tiles;
                                                          // KT: k tiles; UT: units per group
};

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `bar` with the given parity; false after about one
// second, or at once when another role has aborted (unless ignore_abort).
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

// 4 int8 -> 4 bf16, exact, without float conversions: 0x43 above the low
// 7 bits of a byte is the bf16 128 + (b & 127); 0x43 above its sign bit
// (b & 0x80) is the bf16 128 or 256.  Their difference is the signed byte
// b = (b & 127) - (b & 128), an integer of at most 8 significant bits that
// bf16 holds exactly, so the packed subtraction is exact.
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
    __nv_bfloat162 r = __hsub2(*reinterpret_cast<__nv_bfloat162 *>(&a),
                               *reinterpret_cast<__nv_bfloat162 *>(&b));
    return *reinterpret_cast<uint32_t *>(&r);
}
__device__ __forceinline__ uint2 i8x4_to_bf16x4(uint32_t w) {
    const uint32_t mag = w & 0x7F7F7F7Fu, sgn = w & 0x80808080u;
    const uint32_t a01 = __byte_perm(mag, 0x43u, 0x4140), a23 = __byte_perm(mag, 0x43u, 0x4342);
    const uint32_t s01 = __byte_perm(sgn, 0x43u, 0x4140), s23 = __byte_perm(sgn, 0x43u, 0x4342);
    return make_uint2(bf16x2_sub(a01, s01), bf16x2_sub(a23, s23));
}

__device__ __forceinline__ int unit_start(int c, const GemmParams &p) {
    return (int)(((unsigned)c * (unsigned)p.U) / (unsigned)p.G);
}

__device__ __forceinline__ int chunk_rows(int chunk, const GemmParams &p) {
    return min(NB_CHUNK, p.B - chunk * NB_CHUNK);
}

__global__ void __launch_bounds__(kThreads, 1) gemm_i8_tc_kernel(const GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    GemmSmem &sm = *reinterpret_cast<GemmSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    const int u0 = unit_start(c, p), u1 = unit_start(c + 1, p);

    if (tid == 0) {
        for (int s = 0; s < AST; ++s) {
            mbar_init(&sm.a_full[s], 1);
            mbar_init(&sm.a_empty[s], kConvWarps);
        }
        for (int s = 0; s < BST; ++s) {
            mbar_init(&sm.b_full[s], 1);
            mbar_init(&sm.b_empty[s], 2);  // both issuers' commits
        }
        for (int a = 0; a < NABUF; ++a) {
            mbar_init(&sm.conv[a], kConvWarps);
            mbar_init(&sm.a_free[a], 2);
        }
        mbar_init(&sm.acc_full, 2);
        mbar_init(&sm.acc_empty, kEpiWarps);
        mbar_init(&sm.drain[0], 1);
        mbar_init(&sm.drain[1], 1);
        sm.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&sm.tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    volatile int *abort_flag = &sm.abort_flag;

    // unit u: row-tile pair pi = u / UT (pi = chunk * MP + pair: tiles 2 pair,
    // 2 pair + 1), k tiles (u % UT) * KU ...
    if (warp == 0) {
        // ---- weight producer: read-only data, so it runs ahead of the previous
        //      kernel of the step (no wait on it) ------------------------------
        if (lane == 0) {
            int issued = 0;  // copies issued; the last AST may still be in flight
            for (int u = u0; u < u1; ++u) {
                const int it = u - u0, sa = it % AST;
                const int pi = u / p.UT, kt0 = (u % p.UT) * KU;
                const int mt0 = p.TP * (pi % p.MP), ntl = min(p.TP, p.MT - mt0);
                const int nk = min(KU, p.KT - kt0);
                if (it >= AST && !mbar_wait(&sm.a_empty[sa], ((it / AST) - 1) & 1, abort_flag)) {
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive_expect_tx(&sm.a_full[sa], (uint32_t)(ntl * nk) * kATileBytes);
                for (int tp = 0; tp < ntl; ++tp)
                    bulk_g2s(smem_u32(sm.a8[sa][tp]), p.Wt + ((size_t)(mt0 + tp) * p.KT + kt0) * kATileBytes,
                             (uint32_t)nk * kATileBytes, &sm.a_full[sa]);
                issued = it + 1;
            }
            if (*abort_flag) {  // let every copy still in flight land before exiting
                for (int it = max(0, issued - AST); it < issued; ++it)
                    mbar_wait(&sm.a_full[it % AST], (it / AST) & 1, abort_flag, true);
            }
        }
    } else if (warp == kBProdWarp) {
        // ---- activation producer: after the previous kernel (which may write them)
        if (lane == 0) {
            pdl_wait();
            pdl_trigger();
            int issued = 0;
            for (int u = u0; u < u1; ++u) {
                const int it = u - u0, sb = it % BST;
                const int chunk = (u / p.UT) / p.MP, kt0 = (u % p.UT) * KU;
                const int nk = min(KU, p.KT - kt0);
                const int N = 2 * ((chunk_rows(chunk, p) + 7) & ~7);
                if (it >= BST && !mbar_wait(&sm.b_empty[sb], ((it / BST) - 1) & 1, abort_flag)) {
                    *abort_flag = 1;
                    break;
                }
                mbar_arrive_expect_tx(&sm.b_full[sb], (uint32_t)nk * (uint32_t)N * 128u);
                for (int i = 0; i < nk; ++i)
                    bulk_g2s(smem_u32(sm.b16[sb]) + (uint32_t)i * kOpTileBytes,
                             p.xb + ((size_t)chunk * p.KT + kt0 + i) * kOpTileBytes, (uint32_t)N * 128u,
                             &sm.b_full[sb]);
                issued = it + 1;
            }
            if (*abort_flag) {
                for (int it = max(0, issued - BST); it < issued; ++it)
                    mbar_wait(&sm.b_full[it % BST], (it / BST) & 1, abort_flag, true);
            }
        }
    } else if (warp == 1 || warp == kMma1Warp) {
        // ---- MMA issuers: row tile tp of the pair, its own accumulator (columns
        //      128 tp); both follow every unit's barriers, so with a single row
        //      tile the second one only commits -------------------------------------
        if (lane == 0) {
            const int tp = warp == 1 ? 0 : 1;
            int it = 0, seg = 0;
            bool ok = true;
            for (int u = u0; u < u1 && ok; ++seg) {
                const int pi = u / p.UT;
                const int ue = min(u1, (pi + 1) * p.UT);
                const int chunk = pi / p.MP, mt0 = p.TP * (pi % p.MP), ntl = min(p.TP, p.MT - mt0);
                const int N = 2 * ((chunk_rows(chunk, p) + 7) & ~7);
                const uint32_t idesc = instr_desc(BM, N);
                // the accumulators are free once the epilogue has read the last segment's
                if (seg >= 1 && !mbar_wait(&sm.acc_empty, (seg - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int useg = u;  // first unit of this segment: overwrite the accumulator
                for (; u < ue; ++u, ++it) {
                    const int sb = it % BST, ab = it % NABUF;
                    if (!mbar_wait(&sm.conv[ab], (it / NABUF) & 1, abort_flag) ||
                        !mbar_wait(&sm.b_full[sb], (it / BST) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // K steps of 16: 8 tensor-memory columns of A and 32 bytes of
                    // B's rows (+2 in the descriptor's address field) each; the
                    // second 64-k tile's B starts 16 KB (+1024) further.  Row tile
                    // tp: accumulator columns 128 tp, A columns 64 tp of the buffer.
                    if (tp < ntl) {
                        const uint32_t ta = tmem + kTmemA + (uint32_t)ab * kACols + (uint32_t)tp * 64u;
                        const uint32_t dt = tmem + (uint32_t)tp * 128u;
                        const uint64_t bd = smem_desc_sw128(smem_u32(sm.b16[sb]));
                        mma_bf16_ts_x4(dt, ta, bd, idesc, u == useg ? 0u : 1u);
                        if ((u % p.UT) * KU + 1 < p.KT) mma_bf16_ts_x4(dt, ta + 32u, bd + 1024u, idesc, 1u);
                    }
                    mma_commit(&sm.b_empty[sb]);
                    mma_commit(&sm.a_free[ab]);
                }
                if (!ok) break;
                mma_commit(&sm.acc_full);
            }
            if (!ok) *abort_flag = 1;
            mma_commit(&sm.drain[tp]);  // arrives once every MMA issued above has completed
            mbar_wait(&sm.drain[tp], 0, abort_flag, true);
        }
    } else if (warp < kEpiWarp0) {
        // ---- int8 -> bf16 converters: lane = row; warp group g = (w - 2) / 4
        //      takes k tile g % 2 of row tile g / 2 of the pair ---------------------
        const int quarter = warp & 3, g = (warp - 2) >> 2, tp = g >> 1, kh = g & 1;
        const int row = quarter * 32 + lane;
        const uint32_t tlane = (uint32_t)(quarter * 32) << 16;
        for (int u = u0; u < u1; ++u) {
            const int it = u - u0, sa = it % AST, ab = it % NABUF;
            if (!mbar_wait(&sm.a_full[sa], (it / AST) & 1, abort_flag) ||
                (it >= NABUF && !mbar_wait(&sm.a_free[ab], ((it / NABUF) - 1) & 1, abort_flag))) {
                *abort_flag = 1;
                break;
            }
            const int mt0 = p.TP * ((u / p.UT) % p.MP);
            const bool mine = tp < min(p.TP, p.MT - mt0) && kh < min(KU, p.KT - (u % p.UT) * KU);  // warp-uniform
            uint4 w[4];
#pragma unroll
            for (int kp = 0; kp < 4; ++kp) w[kp] = make_uint4(0, 0, 0, 0);
            if (mine) {
                // the row's 4 k parts: 16 bytes each, 2 KB apart (the lanes read 512
                // contiguous bytes per part)
                const uint8_t *src = sm.a8[sa][tp] + kh * kATileBytes + row * 16;
#pragma unroll
                for (int kp = 0; kp < 4; ++kp) w[kp] = *reinterpret_cast<const uint4 *>(src + kp * 2048);
            }
            // the weight stage is free once every warp has its bytes in registers
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.a_empty[sa]);
            if (mine) {
                uint32_t v[32];  // bf16 pairs (k even, k odd) of the row's 64 k, in k order
#pragma unroll
                for (int kp = 0; kp < 4; ++kp) {
                    uint2 e;
                    e = i8x4_to_bf16x4(w[kp].x);
                    v[kp * 8 + 0] = e.x;
                    v[kp * 8 + 1] = e.y;
                    e = i8x4_to_bf16x4(w[kp].y);
                    v[kp * 8 + 2] = e.x;
                    v[kp * 8 + 3] = e.y;
                    e = i8x4_to_bf16x4(w[kp].z);
                    v[kp * 8 + 4] = e.x;
                    v[kp * 8 + 5] = e.y;
                    e = i8x4_to_bf16x4(w[kp].w);
                    v[kp * 8 + 6] = e.x;
                    v[kp * 8 + 7] = e.y;
                }
                tmem_st32(tmem + tlane + kTmemA + (uint32_t)ab * kACols + (uint32_t)(tp * 64 + kh * 32), v);
            }
            // one arrival per warp: every lane's stores are complete (wait::st)
            // and fenced before the warp converges and lane 0 arrives
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.conv[ab]);
        }
    } else {
        // ---- epilogue: warps 18..25; warp w reads lane quarter w % 4 of the
        //      accumulator of row tile (w - 18) / 4 --------------------------------
        pdl_wait();  // the partial buffers may still be read by the previous kernel
        const int quarter = warp & 3, tp = (warp - kEpiWarp0) >> 2;
        const int r = quarter * 32 + lane;
        const SchedView sv{p.U, p.G, p.UT, p.MP, p.max_seg};
        int seg = 0;
        for (int u = u0; u < u1; ++seg) {
            const int pi = u / p.UT;
            u = min(u1, (pi + 1) * p.UT);
            const int chunk = pi / p.MP, mt0 = p.TP * (pi % p.MP), ntl = min(p.TP, p.MT - mt0);
            const int Bc = chunk_rows(chunk, p);
            const int N = 2 * ((Bc + 7) & ~7);
            const int slot = c - sched_cta_of_unit(pi * p.UT, sv);
            bool ok = mbar_wait(&sm.acc_full, seg & 1, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            if (tp < ntl) {
                const int tile = chunk * p.MT + mt0 + tp;
                if (quarter == 0 && lane == 0 && u1 >= (pi + 1) * p.UT) p.nseg[tile] = slot + 1;
                const uint32_t trow = tmem + (uint32_t)(tp * 128) + ((uint32_t)(quarter * 32) << 16);
                float *pslot = p.part + ((size_t)tile * p.max_seg + slot) * (NB_CHUNK * BM);
#pragma unroll
                for (int c16 = 0; c16 < 8; ++c16) {
                    if (c16 * 16 < N) {  // warp-uniform
                        float v[16];
                        tmem_ld16(trow + c16 * 16, v);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const int b = c16 * 8 + j;
                            if (b < Bc) pslot[b * BM + r] = v[2 * j] + v[2 * j + 1];
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.acc_empty);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
    if (tid == 0 && sm.abort_flag) atomicOr(p.err, 1);
}

// Activations fp32 [B][K] -> bf16 B-operand tiles [chunk][kt][16 KB]: rows
// 2b (hi) and 2b+1 (lo) of sequence b; k >= K and b in [Bc, Bpad) are zero.
__global__ void pack_b_kernel(const float *__restrict__ x, uint8_t *__restrict__ xb, int B, int K,
                              int KT) {
    pdl_trigger();  // the projection after this kernel may start streaming its weights
    pdl_wait();
    const int kt = blockIdx.x, chunk = blockIdx.y;
    const int Bc = min(NB_CHUNK, B - chunk * NB_CHUNK);
    const int Bpad = (Bc + 7) & ~7;
    uint8_t *tile = xb + ((size_t)chunk * KT + kt) * kOpTileBytes;
    for (int idx = blockIdx.z * blockDim.x + threadIdx.x; idx < Bpad * 8; idx += blockDim.x * gridDim.z) {
        const int b = idx >> 3, kc = idx & 7;
        const int k0 = kt * BK + kc * 8;
        float v[8];
        if (b < Bc && k0 < K) {
            const float4 *src = reinterpret_cast<const float4 *>(x + (size_t)(chunk * NB_CHUNK + b) * K + k0);
            const float4 a0 = src[0], a1 = src[1];
            v[0] = a0.x; v[1] = a0.y; v[2] = a0.z; v[3] = a0.w;
            v[4] = a1.x; v[5] = a1.y; v[6] = a1.z; v[7] = a1.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.f;
        }
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
            const float2 hf = __bfloat1622float2(h);
            __nv_bfloat162 l = __floats2bfloat162_rn(v[2 * j] - hf.x, v[2 * j + 1] - hf.y);
            hi[j] = *reinterpret_cast<uint32_t *>(&h);
            lo[j] = *reinterpret_cast<uint32_t *>(&l);
        }
        const int rh = 2 * b, rl = 2 * b + 1;
        *reinterpret_cast<uint4 *>(tile + op_chunk_offset(rh, kc)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(tile + op_chunk_offset(rl, kc)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// y[row(j)][m] = s[m] * (sum of the tile's segment partials, in slot order)
// for column j of the projection; row(j) = (j / T) * Sr + t0 + j % T (a
// decode step: T = Sr = 1, t0 = 0, row(j) = j; a block of T prompt tokens
// of each sequence: the token's row of the [sequence][token] output).
// Also advances the ring positions of `rpos` by `adv` (block 0) for the
// B / T sequences of the launch.
__global__ void splitk_reduce_kernel(const float *__restrict__ part, const int *__restrict__ nseg_tab,
                                     const float *__restrict__ s, float *__restrict__ y,
                                     SchedView sv, int M, int B, int32_t *__restrict__ rpos,
                                     int conv_k, int T, int Sr, int t0, int adv, int *__restrict__ pool_reset) {
    pdl_trigger();  // the next step's first kernels may be launched already
    pdl_wait();
    // the state kernel's item pool, for the next step (that kernel has completed)
    if (pool_reset != nullptr && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *pool_reset = 0;
    if (rpos != nullptr && blockIdx.x == 0 && blockIdx.y == 0) {
        for (int b = threadIdx.x; b < B / T; b += blockDim.x) {
            int2 q = reinterpret_cast<int2 *>(rpos)[b];
            q.x = (q.x + adv) % conv_k;
            q.y = (q.y + adv) % (conv_k - 1);
            reinterpret_cast<int2 *>(rpos)[b] = q;
        }
    }
    const int tile = blockIdx.x;             // chunk * MT + mt
    const int chunk = tile / sv.MT, mt = tile % sv.MT;
    const int Bc = min(NB_CHUNK, B - chunk * NB_CHUNK);
    const int r = threadIdx.x & (BM - 1);
    const int b = blockIdx.y * 2 + (threadIdx.x >> 7);
    const int m = mt * BM + r;
    if (m >= M || b >= Bc) return;
    const int nseg = nseg_tab[tile];
    const float *pt = part + (size_t)tile * sv.max_seg * (NB_CHUNK * BM) + b * BM + r;
    float acc = 0.f;
#pragma unroll 8
    for (int k = 0; k < nseg; ++k) acc += __ldcg(pt + (size_t)k * (NB_CHUNK * BM));
    const int j = chunk * NB_CHUNK + b;
    y[(size_t)((j / T) * Sr + t0 + j % T) * M + m] = s[m] * acc;
}

}  // namespace

GemmPlan plan_tc_gemm(int M, int K, int B) {
    GemmPlan g;
    // (unit counts stay far below 2^31 / num_sms for every accepted config)
    g.MT = (M + BM - 1) / BM;
    g.KT = (K + kTileK - 1) / kTileK;
    g.KU = B >= kTcMinBatch ? KU : 4;
    g.UT = (g.KT + g.KU - 1) / g.KU;
    g.nchunks = (B + NB_CHUNK - 1) / NB_CHUNK;
    // tensor-core units cover a pair of row tiles (the activation operand is
    // then read once per two weight tiles) when that still leaves every SM
    // several units; otherwise, and for the CUDA-core kernel, one row tile
    g.TP = (B >= kTcMinBatch && g.nchunks * ((g.MT + 1) / 2) * g.UT >= 4 * num_sms()) ? 2 : 1;
    g.MP = (g.MT + g.TP - 1) / g.TP;
    g.U = g.nchunks * g.MP * g.UT;
    // one CTA per SM, two for the CUDA-core kernel at batch 1 (dn_gemv.cu)
    g.G = std::min((B == 1 ? 2 : 1) * num_sms(), g.U);
    // then the fewest CTAs that still take no more than ceil(U / G) units
    // each: every CTA gets the same count (the step waits on the slowest one),
    // segments are longer, and the SMs left over take the next kernel's CTAs
    // early
    const int per = (g.U + g.G - 1) / g.G;
    g.G = (g.U + per - 1) / per;
    // segments per tile (pair): UT units meet at most ceil(UT / min_range) + 1 ranges
    const int min_range = g.U / g.G;
    g.max_seg = (g.UT + min_range - 1) / min_range + 1;
    g.tiles = g.nchunks * g.MT;
    return g;
}

size_t tc_gemm_smem_bytes() { return sizeof(GemmSmem) + 1024; }

cudaError_t launch_pack_b(const float *x, uint8_t *xb, int B, int K, cudaStream_t st) {
    const int KT = (K + BK - 1) / BK;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)KT, (unsigned)((B + NB_CHUNK - 1) / NB_CHUNK), 4);
    cfg.blockDim = dim3(128);
    cfg.stream = st;
    PdlAttr pdl;
    pdl.apply(cfg);
    return cudaLaunchKernelEx(&cfg, pack_b_kernel, x, xb, B, K, KT);
}

cudaError_t launch_gemm_i8_tc(const uint8_t *Wt, const uint8_t *xb, float *part, int *nseg, int *err,
                              int M, int K, int B, cudaStream_t st) {
    static std::atomic<uint64_t> attr_done{0};
    const size_t smem = tc_gemm_smem_bytes();
    const cudaError_t e = once_per_device(attr_done, [&](int) {
        return cudaFuncSetAttribute(gemm_i8_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    });
    if (e != cudaSuccess) return e;
    const GemmPlan g = plan_tc_gemm(M, K, B);
    GemmParams p;
    p.Wt = Wt;
    p.xb = xb;
    p.part = part;
    p.nseg = nseg;
    p.err = err;
    p.M = M;
    p.MT = g.MT;
    p.MP = g.MP;
    p.TP = g.TP;
    p.KT = g.KT;
    p.UT = g.UT;
    p.B = B;
    p.nchunks = g.nchunks;
    p.U = g.U;
    p.G = g.G;
    p.max_seg = g.max_seg;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)g.G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    PdlAttr pdl;
    pdl.apply(cfg);
    return cudaLaunchKernelEx(&cfg, gemm_i8_tc_kernel, p);
}

cudaError_t launch_splitk_reduce(const float *part, const int *nseg, const float *s, float *y, int M,
                                 int K, int B, int32_t *rpos_advance, int conv_k, cudaStream_t st, int T,
                                 int Sr, int t0, int adv, int *pool_reset) {
    const GemmPlan g = plan_tc_gemm(M, K, B);
    const SchedView sv{g.U, g.G, g.UT, g.MT, g.max_seg};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)g.tiles, (unsigned)((std::min(B, NB_CHUNK) + 1) / 2));
    cfg.blockDim = dim3(2 * BM);
    cfg.stream = st;
    PdlAttr pdl;
    pdl.apply(cfg);
    return cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, part, nseg, s, y, sv, M, B, rpos_advance,
                              conv_k, T, Sr, t0, adv, pool_reset);
}

}  // namespace dn
