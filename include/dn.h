/*
 * dn.h — C ABI of the gated-DeltaNet decode-step library (libdn.so, sm_103a).
 *
 * One dn_layer is one gated-DeltaNet layer for up to max_batch independent
 * sequences.  It follows the layer object of the page "qwen36: run the
 * DeltaNet layer end to end on the card (Q36_DN_GPU=1): conv, recurrence and
 * gated norm join the two projections", section "What the PR does": one
 * object per layer holds the short-conv ring, the recurrent state
 * [n_v_heads x dk x dv], the conv and norm weights, the two int8 projections
 * and one token's scratch in device memory, behind five entry points
 * (create / set_state / get_state / step / destroy).  The gates stay outside
 * and arrive per head with every step.
 *
 * Conventions for every call:
 *   - Return value: DN_OK (0) or a negative DN_E* code.  Argument checks run
 *     on the host before any device work; a call that fails them returns
 *     DN_EINVAL and leaves the layer and its state untouched.
 *   - A CUDA error seen by a call marks the layer failed (sticky): afterwards
 *     dn_step and dn_set_state return DN_EFAILED, while dn_get_state still
 *     copies out what the device holds and dn_destroy still frees it (the
 *     page lets the state be read back after a step has failed).
 *   - Device work is enqueued on a CUDA stream and is asynchronous unless a
 *     call says otherwise; errors of asynchronous work surface at a later
 *     call on the same layer.
 *   - Arrays are dense, row-major (last index fastest), fp32 unless stated.
 *   - The library keeps no pointer to caller memory after a call returns.
 *   - Threads: calls on one layer must not overlap (a layer holds one step's
 *     scratch); different layers may be driven from different host threads
 *     and devices at the same time.
 */
#ifndef DN_H
#define DN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------- */
#define DN_OK         0
#define DN_EINVAL    -1  /* bad argument: nothing was done */
#define DN_ENOMEM    -2  /* device allocation failed */
#define DN_ECUDA     -3  /* a CUDA call failed; the layer is now failed */
#define DN_EFAILED   -4  /* the layer failed earlier; only get_state/destroy work */
#define DN_EINJECTED -5  /* failure injected with dn_debug_fail_next */

/* ---- dn_config.flags ----------------------------------------------------- */
/* per-key-channel decay: g carries one log-decay per key index of each head
 * (g[b][h][i] scales row i of that head's state), the gate of the page's
 * KDA engines; without it one log-decay per head scales the whole state */
#define DN_FLAG_KEY_GATE 1
/* device-side gates: the layer holds the a/b gate projections as int8 rows
 * (dn_weights.w_ab / s_ab / gate_A) and computes g = -A[h] * softplus(a) and
 * beta = sigmoid(b) itself from each step's x, so dn_step and dn_stack_step
 * take no g or beta (pass NULL); the page keeps these two small projections
 * on the host and passes their values to the kernels */
#define DN_FLAG_DEVICE_GATES 2
/* int4 projection weights (the page's model is a per-row int4 container):
 * w_in, w_out and w_ab hold two weights per byte, [rows][K/2]; byte i of a
 * row holds k = 2i in its low and k = 2i + 1 in its high four bits, two's
 * complement (values -8 .. 7), with one fp32 scale per row as for int8 */
#define DN_FLAG_INT4_WEIGHTS 4

/* ---- where a pointer argument lives ------------------------------------ */
#define DN_PTR_HOST   0
#define DN_PTR_DEVICE 1

typedef struct dn_layer dn_layer; /* opaque; owns all of its device memory */

/*
 * Layer dimensions.  The page's backend object is parameterised by them, up
 * to 64 value heads and key/value head sizes up to 256 (section "Where this
 * goes next").
 * This build accepts:
 *   hidden      multiple of 16, 16 .. 16384
 *   n_qk_heads  >= 1, divides n_v_heads; n_v_heads <= 64
 *   dk, dv      each one of 32, 64, 128, 256
 *   conv_k      2 .. 8 (taps of the causal short conv; the ring keeps conv_k-1)
 *   max_batch   1 .. 1024 (sequences the layer holds state for)
 *   l2_eps      eps inside the square root of the q/k L2 norms (> 0)
 *   norm_eps    eps of the gated RMSNorm (> 0)
 *   q_scale     multiplies the normalised q (e.g. 1/sqrt(dk))
 *   flags       any combination of DN_FLAG_KEY_GATE, DN_FLAG_DEVICE_GATES,
 *               DN_FLAG_INT4_WEIGHTS
 * Derived: conv_ch = 2*n_qk_heads*dk + n_v_heads*dv,
 *          in_rows = conv_ch + n_v_heads*dv, v_dim = n_v_heads*dv.
 */
typedef struct dn_config {
    int32_t hidden, n_qk_heads, n_v_heads, dk, dv, conv_k, max_batch;
    float l2_eps, norm_eps, q_scale;
    int32_t flags;
} dn_config;

/*
 * Layer weights, host pointers, copied by dn_create (the caller may free
 * them afterwards).  The in_proj fuses the q, k, v rows and the z rows into
 * one matrix (one GEMV where there were two), int8 rows with one fp32 scale
 * per row (page "feat(qwen36): the
 * dense trunk places itself", section "What this adds", item 1):
 *   w_in   int8 [in_rows][hidden]; rows are q | k | v | z, head h of a block
 *          is the contiguous slice h*d .. (h+1)*d; y[o] = s_in[o]*sum_i w_in[o][i]*x[i]
 *   s_in   [in_rows]
 *   w_conv [conv_ch][conv_k]; tap conv_k-1 meets the newest input
 *   w_norm [dv]; one gated-RMSNorm weight vector shared by all value heads
 *   w_out  int8 [hidden][v_dim]; out[o] = s_out[o]*sum_i w_out[o][i]*n[i]
 *   s_out  [hidden]
 *   w_ab   (DN_FLAG_DEVICE_GATES only, else NULL) int8 [gate_rows][hidden]:
 *          the a rows (n_v_heads * gw, gw = dk with DN_FLAG_KEY_GATE, else
 *          1; head-major) then the b rows (n_v_heads);
 *          a = s_ab * (w_ab x), b likewise
 *   s_ab   [gate_rows] row scales, gate_rows = n_v_heads * (gw + 1)
 *   gate_A [n_v_heads] decay coefficients: g = -gate_A[h] * softplus(a)
 * Value head h reads q/k head h / (n_v_heads / n_qk_heads).
 */
typedef struct dn_weights {
    const int8_t *w_in;
    const float  *s_in;
    const float  *w_conv;
    const float  *w_norm;
    const int8_t *w_out;
    const float  *s_out;
    const int8_t *w_ab;
    const float  *s_ab;
    const float  *gate_A;
} dn_weights;

/*
 * dn_create — allocate a layer on the current CUDA device, upload its
 * weights and zero its state (S = 0, ring = 0, ring_pos = 0 for every
 * sequence).  `stream` (a cudaStream_t, NULL for the legacy default stream)
 * becomes the layer's stream for state copies and for dn_step calls that
 * pass no stream.  Synchronous: the layer is ready when the call returns.
 * On success *out receives the layer; on failure *out is set to NULL and
 * nothing stays allocated.  Errors: DN_EINVAL, DN_ENOMEM, DN_ECUDA.
 */
int dn_create(const dn_config *cfg, const dn_weights *w, void *stream, dn_layer **out);

/*
 * dn_set_state — overwrite the state of sequences [seq0, seq0+n):
 *   S        [n][n_v_heads][dk][dv]   recurrent state, row = key index
 *   ring     [n][conv_k-1][conv_ch]   the last conv_k-1 conv inputs
 *   ring_pos [n] int32 in [0, conv_k-2], the ring slot of the oldest input
 * ptr_kind (DN_PTR_HOST or DN_PTR_DEVICE) says where all three live.  This
 * is the push half of the page's state hand-over: the engine keeps the
 * canonical copy of the state and moves it in and out of the layer with
 * set/get.  The copy is ordered after every dn_step already enqueued on this
 * layer, on whatever stream (the layer waits for the last step's completion
 * event), and the call returns after the copy has completed (it synchronises
 * the layer's stream).  Errors: DN_EINVAL (range, pointer or ring_pos out of
 * range, or a device other than the layer's is current), DN_EFAILED,
 * DN_ECUDA.
 */
int dn_set_state(dn_layer *layer, int seq0, int n, const float *S, const float *ring,
                 const int32_t *ring_pos, int ptr_kind);

/*
 * dn_get_state — copy out the state of sequences [seq0, seq0+n) in the same
 * layout as dn_set_state.  Any of S, ring, ring_pos may be NULL to skip it.
 * Works on a failed layer (returns what the device holds).  The copy is
 * ordered after every dn_step already enqueued on this layer, whichever
 * stream it was enqueued on (the layer's stream waits for the last step's
 * completion event), and the call synchronises the layer's stream before it
 * returns.  Errors: DN_EINVAL (including a device other than the layer's
 * being current), DN_ECUDA.
 */
int dn_get_state(dn_layer *layer, int seq0, int n, float *S, float *ring, int32_t *ring_pos,
                 int ptr_kind);

/*
 * dn_step — advance sequences [0, batch) by one decode token, the whole
 * step on the device: in_proj GEMV, causal conv + SiLU with the ring
 * advancing, per value head the L2 norms of q and k, the decay, the delta
 * against the decayed state, the write-back, out = q^T S over the updated
 * state, the gated RMSNorm with silu(z), out_proj GEMV):
 *   x    [batch][hidden]     layer input
 *   g    [batch][n_v_heads]  log-decay per head (the state is scaled by exp(g));
 *        [batch][n_v_heads][dk] with DN_FLAG_KEY_GATE (row i of a head's
 *        state is scaled by exp(g[b][h][i]))
 *   beta [batch][n_v_heads]  write strength per head
 *   out  [batch][hidden]     layer output (written)
 * With DN_FLAG_DEVICE_GATES, g and beta must be NULL (the layer computes
 * them from x).
 * ptr_kind DN_PTR_DEVICE: all four are device pointers (x 16-byte aligned); the call only
 *   enqueues kernels on `stream` (NULL: the layer's stream) and returns; it
 *   allocates nothing and does not synchronise, so it can be captured in a
 *   CUDA graph.  x/g/beta must stay valid until the work has run.
 * ptr_kind DN_PTR_HOST: all four are host pointers; the call uploads x, g
 *   and beta, runs the step, downloads out and synchronises `stream` before
 *   returning (the page's one upload of x and one download of out per
 *   token).  Pinned host memory makes the copies asynchronous DMA.
 * Steps of one layer on different streams must be ordered by the caller
 * (events); dn_get_state and dn_set_state order themselves after the last
 * step, whatever its stream.  The layer's device must be current.
 * Sequences >= batch are untouched.  Errors: DN_EINVAL (batch < 1 or >
 * max_batch, NULL pointer, bad ptr_kind, another device current),
 * DN_EFAILED, DN_EINJECTED, DN_ECUDA.
 */
int dn_step(dn_layer *layer, int batch, const float *x, const float *g, const float *beta,
            float *out, int ptr_kind, void *stream);

/*
 * dn_prefill — advance sequences [0, batch) by n_tokens tokens each (a
 * prompt), with the result of n_tokens successive dn_step calls: every
 * token's output, the state, the conv ring and ring_pos end as they would.
 * (The page, section "What the PR does", keeps prompts on its batched CPU
 * path; this is the same step on the card.)
 *   x    [batch][n_tokens][hidden]          device, 16-byte aligned
 *   g    [batch][n_tokens][n_v_heads](gw)   device (NULL with device gates)
 *   beta [batch][n_tokens][n_v_heads]       device (NULL with device gates)
 *   out  [batch][n_tokens][hidden]          device (written)
 * The prompt runs in blocks of up to 512 token columns (sequences x
 * tokens): per block the in_proj and the out_proj run once over all of its
 * columns (tensor cores from 2 columns), and each head's state stays on chip
 * for all of the block's tokens.  With one decay per head (no
 * DN_FLAG_KEY_GATE) and 128-wide keys the recurrence takes its chunked form
 * (32-token chunks; on the tensor cores for 128 x 128 heads when the block
 * holds a (head, sequence) pair per SM): the same algebra in another
 * summation order, so the results equal those of the dn_step calls up to
 * rounding (within the decode step's tolerance), not bit for bit.
 * Device pointers only; the call enqueues on
 * `stream` (NULL: the layer's stream) and returns.  The first call on a layer
 * allocates its scratch (about 140 MB for the 35B shape; counted by
 * dn_device_bytes, freed by dn_destroy), so make it before any stream
 * capture.  Errors: DN_EINVAL (sizes, NULL or misaligned pointers, gates
 * against the layer's flags, another device current), DN_ENOMEM,
 * DN_EFAILED, DN_EINJECTED, DN_ECUDA.
 */
int dn_prefill(dn_layer *layer, int batch, int n_tokens, const float *x, const float *g, const float *beta,
               float *out, void *stream);

/* dn_destroy — free the layer and all its device memory.  NULL-safe.  Waits
 * for the layer's outstanding work first. */
void dn_destroy(dn_layer *layer);

/*
 * dn_stack_step — one decode token through a stack of layers, the residual
 * stream h carried between them (the pages' model runs 30 DeltaNet layers per
 * token, page "qwen36: run the DeltaNet layer end to end on the card
 * (Q36_DN_GPU=1)", section "Measured"):
 *   for l = 0 .. n_layers-1:  h <- h + layer_l( h / sqrt(mean(h^2) + eps) )
 * with an unweighted RMS pre-norm per sequence over `hidden`.
 *   layers  n_layers layer handles with equal hidden and n_v_heads, on the
 *           current device, each with max_batch >= batch
 *   h       [batch][hidden] device, read and overwritten
 *   g, beta [n_layers][batch][n_v_heads] device, each layer's gates (g has a
 *           trailing [dk] with DN_FLAG_KEY_GATE; all layers then share it);
 *           both NULL when the layers have DN_FLAG_DEVICE_GATES (all or none)
 * Device pointers only; the call enqueues on `stream` (NULL: the first
 * layer's stream) and uses the first layer's staging buffers for the
 * normalised input and each layer's output.  Errors: DN_EINVAL (NULL, bad
 * sizes, mismatched layers, eps < 0), DN_EFAILED (a failed layer), and the
 * errors of dn_step; on an error the layers before the failing one have
 * already advanced.
 */
int dn_stack_step(dn_layer *const *layers, int n_layers, int batch, float *h, const float *g,
                  const float *beta, float eps, void *stream);

/*
 * dn_debug_fail_next — failure injection for tests: the next dn_step on this
 * layer returns `code` (a negative DN_E* value) before any device work and
 * marks the layer failed, like the page's fake backend, whose steps can be
 * made to fail and whose failure switches the layer off.  code = 0 cancels a
 * pending injection.  Errors: DN_EINVAL.
 */
int dn_debug_fail_next(dn_layer *layer, int code);

/*
 * dn_debug_expire_wait — device-side failure detection for tests: the next
 * dn_step on this layer first launches one thread that waits for a flag
 * nothing sets, gives up after `limit_us` microseconds (global timer) and
 * records the give-up in the layer's device error word, as every bounded wait
 * of the step's kernels does when it runs out (about one second).  The step
 * itself then runs normally; the next dn_get_state finds the error word set,
 * still copies the state out, returns DN_ECUDA and marks the layer failed,
 * so later steps return DN_EFAILED.  No trap, fault or unbounded wait is
 * involved.  limit_us in 1 .. 1000000; 0 cancels a pending request.
 * Errors: DN_EINVAL.
 */
int dn_debug_expire_wait(dn_layer *layer, int limit_us);

/*
 * dn_profile_next_step — instrumentation for benchmarks: the next dn_step on
 * this layer records, on its stream, events[0] before its first kernel,
 * events[1] after the in_proj (activation packing + projection),
 * events[2] after the per-sequence preparation kernel (conv, norms, gates;
 * recorded right after events[1] when the step fuses it into the state
 * kernel), events[3] after the state kernel (recurrence, readout, gated
 * norm) and events[4] after the out_proj (projection + reduction), so that
 * cudaEventElapsedTime gives each stage's device time.  `events` points to
 * five cudaEvent_t created by the caller (timing enabled); it is used by that
 * one dn_step call only (one-shot).  NULL cancels.  Errors: DN_EINVAL.
 */
int dn_profile_next_step(dn_layer *layer, void *const *events);

/*
 * dn_step_kernels — the number of kernels one dn_step of `batch` sequences
 * launches on this layer (for launch accounting in benchmarks); 0 when
 * `batch` is out of range.  Not part of the page's layer: instrumentation.
 */
int dn_step_kernels(const dn_layer *layer, int batch);

/*
 * dn_proj_i8_noalloc — the int8 row-scaled projection used inside dn_step,
 * offered on its own for callers that must not allocate device memory:
 *   y[b][o] = s[o] * sum_i W[o][i] * x[b][i],  b < B, o < M
 * The pages have no counterpart of this call; it exists for code that runs
 * where it does not own the device allocator (a plug-in inside another
 * runtime's memory pool, a loop with a memory budget fixed in advance) and
 * so can call neither cudaMalloc nor dn_create.  Its scratch (split-K
 * partial sums) lives in one static device array of the library, about
 * 4 MiB, that every GPU which loads the library holds until the process
 * exits; the call itself allocates nothing.
 *   W  int8 [M][K] row-major, device, 16-byte aligned
 *   s  [M] row scales, device
 *   x  [B][K] activations, device, 16-byte aligned
 *   y  [B][M] output, device (written)
 * Limits: 1 <= B <= 8, 1 <= M <= 16384, 16 <= K <= 16384, K a multiple of
 * 16, and the split-K scratch of the shape must fit the static array (it
 * does for every M, K within the limits on a 152-SM GPU); anything else
 * returns DN_EINVAL before any device work.
 * Work is enqueued on `stream` (NULL: the legacy default stream) and the
 * call returns without synchronising.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture.  The address is
 * kept for the life of the process, so a device reset (cudaDeviceReset) while
 * the library stays loaded is not supported by this call.  Every call on a
 * device shares the one array: nothing in it needs to start at zero (a call
 * writes every scratch value it reads before reading it), but calls whose
 * work overlaps on the GPU (other streams, other threads) race on it.
 * Errors: DN_EINVAL, DN_ECUDA (launch failure).
 */
int dn_proj_i8_noalloc(const int8_t *W, const float *s, const float *x, float *y, int M, int K,
                       int B, void *stream);

/* dn_device_bytes — device bytes currently held by all live layers of this
 * process (leak accounting: 0 once every layer is destroyed). */
int64_t dn_device_bytes(void);

/* dn_strerror — a static string naming a status code. */
const char *dn_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* DN_H */
