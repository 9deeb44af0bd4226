// C ABI of libdn: the five layer calls of the page "qwen36: run the DeltaNet
// layer end to end on the card (Q36_DN_GPU=1)" (section "What the PR does":
// create / set_state / get_state / step / destroy on one object per layer),
// plus failure injection and device-memory accounting for tests.  See
// include/dn.h for the contract of every call.
#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "dn_internal.cuh"

#define DN_API extern "C" __attribute__((visibility("default")))

struct dn_layer {
    dn::Dims d;
    dn::LayerDev L;
    cudaStream_t stream;
    int device;
    int failed;
    int fail_next;
    int expire_us_next;  // dn_debug_expire_wait: bounded device wait before the next step
    cudaEvent_t prof[5];  // one-shot per-stage events for the next step
    int prof_armed;
    // completion of the last step enqueued on a stream other than `stream`
    // (state copies wait for it); not recorded while that stream captures
    cudaEvent_t step_done;
    int step_done_pending;
    dn::PrefillDev P;  // dn_prefill's scratch (allocated on its first call)
    int prefill_ready;
    size_t bytes;
    std::vector<void *> allocs;
};

namespace {

std::atomic<int64_t> g_device_bytes{0};

int layer_alloc(dn_layer *l, void **p, size_t n) {
    *p = nullptr;
    if (n == 0) return DN_OK;
    cudaError_t e = cudaMalloc(p, n);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();  // allocation failures are not sticky; clear it
        *p = nullptr;
        return e == cudaErrorMemoryAllocation ? DN_ENOMEM : DN_ECUDA;
    }
    l->allocs.push_back(*p);
    l->bytes += n;
    g_device_bytes += (int64_t)n;
    return DN_OK;
}

void layer_free_all(dn_layer *l) {
    if (l->step_done != nullptr) cudaEventDestroy(l->step_done);
    l->step_done = nullptr;
    for (void *p : l->allocs) cudaFree(p);
    g_device_bytes -= (int64_t)l->bytes;
    l->allocs.clear();
    l->bytes = 0;
}

bool valid_cfg(const dn_config *c) {
    if (c->hidden < 16 || c->hidden > 16384 || c->hidden % 16 != 0) return false;
    if (c->n_qk_heads < 1 || c->n_v_heads < 1 || c->n_v_heads > 64) return false;
    if (c->n_v_heads % c->n_qk_heads != 0) return false;
    if (!(c->dk == 32 || c->dk == 64 || c->dk == 128 || c->dk == 256)) return false;
    if (!(c->dv == 32 || c->dv == 64 || c->dv == 128 || c->dv == 256)) return false;
    if ((c->flags & ~(DN_FLAG_KEY_GATE | DN_FLAG_DEVICE_GATES | DN_FLAG_INT4_WEIGHTS)) != 0) return false;
    if (c->conv_k < 2 || c->conv_k > 8) return false;
    if (c->max_batch < 1 || c->max_batch > 1024) return false;
    if (!(c->l2_eps > 0.f) || !(c->norm_eps > 0.f)) return false;
    if (c->q_scale != c->q_scale) return false;  // NaN
    return true;
}

// int4 rows packed two per byte ([M][K/2], low nibble first) -> int8 [M][K]
std::vector<int8_t> unpack_int4(const int8_t *W, int M, int K) {
    std::vector<int8_t> out((size_t)M * K);
    for (size_t m = 0; m < (size_t)M; ++m)
        for (int i = 0; i < K / 2; ++i) {
            const uint8_t byte = (uint8_t)W[m * (K / 2) + i];
            // sign-extend each nibble: (n ^ 8) - 8
            out[m * K + 2 * i] = (int8_t)(((byte & 0xF) ^ 8) - 8);
            out[m * K + 2 * i + 1] = (int8_t)(((byte >> 4) ^ 8) - 8);
        }
    return out;
}

// W [M][K] int8 -> [ceil(M/128)][ceil(K/64)][128][64], zero-padded
std::vector<uint8_t> tile_weights(const int8_t *W, int M, int K) {
    const int MT = (M + dn::kTileM - 1) / dn::kTileM, KT = (K + dn::kTileK - 1) / dn::kTileK;
    std::vector<uint8_t> t((size_t)MT * KT * dn::kTileM * dn::kTileK, 0);
    for (int m = 0; m < M; ++m) {
        const int mt = m / dn::kTileM, r = m % dn::kTileM;
        for (int k = 0; k < K; ++k) {
            const int kt = k / dn::kTileK, kk = k % dn::kTileK;
            // [mt][kt][k part (16 k)][row][16 B]
            t[((size_t)mt * KT + kt) * dn::kTileM * dn::kTileK + (size_t)(kk >> 4) * dn::kTileM * 16 + r * 16 +
              (kk & 15)] = (uint8_t)W[(size_t)m * K + k];
        }
    }
    return t;
}

int cuda_fail(dn_layer *l) {
    l->failed = 1;
    return DN_ECUDA;
}

// The layer's device must be current for every call that enqueues work.
bool on_layer_device(const dn_layer *l) {
    int cur = -1;
    return cudaGetDevice(&cur) == cudaSuccess && cur == l->device;
}

// State copies run on the layer's stream; order them after the last step
// that ran on another stream.
cudaError_t order_after_steps(dn_layer *l) {
    if (!l->step_done_pending) return cudaSuccess;
    const cudaError_t e = cudaStreamWaitEvent(l->stream, l->step_done, 0);
    if (e == cudaSuccess) l->step_done_pending = 0;
    return e;
}

#define DN_TRY(layer, expr)                            \
    do {                                               \
        cudaError_t e_ = (expr);                       \
        if (e_ != cudaSuccess) return cuda_fail(layer); \
    } while (0)

}  // namespace

namespace dn {
int num_sms() {
    // per device (ordinals below 64 cached), safe from several host threads
    static std::atomic<int> cached[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();  // no device: the caller's next CUDA call reports it; nothing is cached
        return 1;
    }
    if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}
}  // namespace dn

DN_API const char *dn_strerror(int code) {
    switch (code) {
        case DN_OK: return "ok";
        case DN_EINVAL: return "invalid argument";
        case DN_ENOMEM: return "out of device memory";
        case DN_ECUDA: return "CUDA error (layer is now failed)";
        case DN_EFAILED: return "layer failed earlier";
        case DN_EINJECTED: return "injected failure";
        default: return "unknown status";
    }
}

DN_API int64_t dn_device_bytes(void) { return g_device_bytes.load(); }

DN_API int dn_create(const dn_config *cfg, const dn_weights *w, void *stream, dn_layer **out) {
    if (out == nullptr) return DN_EINVAL;
    *out = nullptr;
    if (cfg == nullptr || w == nullptr || !valid_cfg(cfg)) return DN_EINVAL;
    if (!w->w_in || !w->s_in || !w->w_conv || !w->w_norm || !w->w_out || !w->s_out)
        return DN_EINVAL;
    if ((cfg->flags & DN_FLAG_DEVICE_GATES) && (!w->w_ab || !w->s_ab || !w->gate_A)) return DN_EINVAL;

    dn_layer *l = new (std::nothrow) dn_layer();
    if (l == nullptr) return DN_ENOMEM;
    dn::Dims &d = l->d;
    d.hidden = cfg->hidden;
    d.n_qk = cfg->n_qk_heads;
    d.n_v = cfg->n_v_heads;
    d.dk = cfg->dk;
    d.dv = cfg->dv;
    d.conv_k = cfg->conv_k;
    d.max_batch = cfg->max_batch;
    d.qk_dim = d.n_qk * d.dk;
    d.v_dim = d.n_v * d.dv;
    d.conv_ch = 2 * d.qk_dim + d.v_dim;
    d.in_rows = d.conv_ch + d.v_dim;
    d.l2_eps = cfg->l2_eps;
    d.norm_eps = cfg->norm_eps;
    d.q_scale = cfg->q_scale;
    d.gw = (cfg->flags & DN_FLAG_KEY_GATE) ? d.dk : 1;
    d.dev_gates = (cfg->flags & DN_FLAG_DEVICE_GATES) ? 1 : 0;
    d.proj_rows = d.in_rows + (d.dev_gates ? d.n_v * (d.gw + 1) : 0);
    d.i4 = (cfg->flags & DN_FLAG_INT4_WEIGHTS) ? 1 : 0;
    l->stream = (cudaStream_t)stream;
    cudaGetDevice(&l->device);

    const size_t MB = (size_t)d.max_batch;
    const size_t s_elems = MB * d.n_v * d.dk * d.dv;
    dn::LayerDev &L = l->L;
    int rc = DN_OK;
#define ALLOC(ptr, bytes)                                               \
    if (rc == DN_OK) rc = layer_alloc(l, (void **)&(ptr), (size_t)(bytes));
    // the in_proj's rows, then (device gates) the a/b gate rows, one matrix
    std::vector<int8_t> w_proj;
    std::vector<float> s_proj;
    const int8_t *w_in_all = w->w_in;
    const float *s_in_all = w->s_in;
    const size_t rb = d.i4 ? (size_t)d.hidden / 2 : (size_t)d.hidden;  // bytes per in_proj row as given
    if (d.dev_gates) {
        const size_t n_in = (size_t)d.in_rows * rb, n_ab = (size_t)(d.proj_rows - d.in_rows) * rb;
        w_proj.resize(n_in + n_ab);
        std::memcpy(w_proj.data(), w->w_in, n_in);
        std::memcpy(w_proj.data() + n_in, w->w_ab, n_ab);
        s_proj.resize((size_t)d.proj_rows);
        std::memcpy(s_proj.data(), w->s_in, (size_t)d.in_rows * 4);
        std::memcpy(s_proj.data() + d.in_rows, w->s_ab, (size_t)(d.proj_rows - d.in_rows) * 4);
        w_in_all = w_proj.data();
        s_in_all = s_proj.data();
    }
    // int4: the packed rows tile like int8 rows of K/2 bytes (128 k per 8 KB
    // tile) for the CUDA-core GEMV, and an exact int8 expansion feeds the
    // tensor-core path
    std::vector<uint8_t> wt_in4, wt_out4;
    std::vector<int8_t> w_in8, w_out8;
    const int8_t *w_out_all = w->w_out;
    if (d.i4) {
        wt_in4 = tile_weights(w_in_all, d.proj_rows, d.hidden / 2);
        wt_out4 = tile_weights(w->w_out, d.hidden, d.v_dim / 2);
        w_in8 = unpack_int4(w_in_all, d.proj_rows, d.hidden);
        w_out8 = unpack_int4(w->w_out, d.hidden, d.v_dim);
        w_in_all = w_in8.data();
        w_out_all = w_out8.data();
    }
    const std::vector<uint8_t> wt_in = tile_weights(w_in_all, d.proj_rows, d.hidden);
    const std::vector<uint8_t> wt_out = tile_weights(w_out_all, d.hidden, d.v_dim);
    const size_t kt_in = (size_t)(d.hidden + dn::kTileK - 1) / dn::kTileK;
    const size_t kt_out = (size_t)(d.v_dim + dn::kTileK - 1) / dn::kTileK;
    ALLOC(L.w_in, wt_in.size());
    ALLOC(L.s_in, (size_t)d.proj_rows * 4);
    if (d.dev_gates) ALLOC(L.gate_A, (size_t)d.n_v * 4);
    ALLOC(L.wconv_t, (size_t)d.conv_k * d.conv_ch * 4);
    ALLOC(L.w_norm, (size_t)d.dv * 4);
    ALLOC(L.w_out, wt_out.size());
    if (d.i4) {
        ALLOC(L.w_in4, wt_in4.size());
        ALLOC(L.w_out4, wt_out4.size());
    }
    ALLOC(L.s_out, (size_t)d.hidden * 4);
    ALLOC(L.S, s_elems * 4);
    ALLOC(L.ring, MB * d.conv_k * d.conv_ch * 4);
    ALLOC(L.rpos, MB * 2 * 4);
    ALLOC(L.nrm, MB * d.v_dim * 4);
    ALLOC(L.x_stage, MB * d.hidden * 4);
    ALLOC(L.g_stage, MB * d.n_v * d.gw * 4);
    ALLOC(L.beta_stage, MB * d.n_v * 4);
    ALLOC(L.out_stage, MB * d.hidden * 4);
    ALLOC(L.ring_stage, MB * (d.conv_k - 1) * d.conv_ch * 4);
    ALLOC(L.rp_stage, MB * 4);
    // projections: the largest segment-partial buffer over every batch size
    // the layer accepts (the schedule, hence the segment count, depends on
    // the batch); packed activations for the tensor-core path
    const size_t chunks = (MB + 63) / 64;
    size_t part_in = 0, part_out = 0, tiles_in = 0, tiles_out = 0, xb_bytes_in = 0, xb_bytes_out = 0;
    for (int b = 1; b <= (int)MB; ++b) {
        const dn::GemmPlan gi = dn::plan_tc_gemm(d.proj_rows, dn::plan_k(d, d.hidden, b), b);
        const dn::GemmPlan go = dn::plan_tc_gemm(d.hidden, dn::plan_k(d, d.v_dim, b), b);
        part_in = std::max(part_in, (size_t)gi.tiles * gi.max_seg * 64 * 128);
        part_out = std::max(part_out, (size_t)go.tiles * go.max_seg * 64 * 128);
        tiles_in = std::max(tiles_in, (size_t)gi.tiles);
        tiles_out = std::max(tiles_out, (size_t)go.tiles);
        // the stream-K schedule computes c * U / G in 32 bits
        if ((uint64_t)gi.U * gi.G >= (1ull << 32) || (uint64_t)go.U * go.G >= (1ull << 32)) rc = DN_EINVAL;
    }
    if (d.max_batch >= dn::kTcMinBatch) {
        xb_bytes_in = chunks * kt_in * dn::kOpTile;
        xb_bytes_out = chunks * kt_out * dn::kOpTile;
    }
    ALLOC(L.part_in, part_in * 4);
    ALLOC(L.part_out, part_out * 4);
    ALLOC(L.nseg_in, tiles_in * 4);
    ALLOC(L.nseg_out, tiles_out * 4);
    ALLOC(L.xb_in, xb_bytes_in);
    ALLOC(L.xb_out, xb_bytes_out);
    ALLOC(L.err, 4);
    ALLOC(L.pool, 4);
#undef ALLOC
    if (rc == DN_OK && cudaEventCreateWithFlags(&l->step_done, cudaEventDisableTiming) != cudaSuccess) {
        (void)cudaGetLastError();
        l->step_done = nullptr;
        rc = DN_ECUDA;
    }
    if (rc != DN_OK) {
        layer_free_all(l);
        delete l;
        return rc;
    }

    std::vector<float> wct((size_t)d.conv_k * d.conv_ch);
    for (int c = 0; c < d.conv_ch; ++c)
        for (int t = 0; t < d.conv_k; ++t)
            wct[(size_t)t * d.conv_ch + c] = w->w_conv[(size_t)c * d.conv_k + t];

    cudaStream_t st = l->stream;
    cudaError_t e = cudaSuccess;
    auto H2D = cudaMemcpyHostToDevice;
    if (e == cudaSuccess) e = cudaMemcpyAsync(L.w_in, wt_in.data(), wt_in.size(), H2D, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(L.s_in, s_in_all, (size_t)d.proj_rows * 4, H2D, st);
    if (e == cudaSuccess && d.dev_gates) e = cudaMemcpyAsync(L.gate_A, w->gate_A, (size_t)d.n_v * 4, H2D, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(L.wconv_t, wct.data(), wct.size() * 4, H2D, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(L.w_norm, w->w_norm, (size_t)d.dv * 4, H2D, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(L.w_out, wt_out.data(), wt_out.size(), H2D, st);
    if (e == cudaSuccess && d.i4) e = cudaMemcpyAsync(L.w_in4, wt_in4.data(), wt_in4.size(), H2D, st);
    if (e == cudaSuccess && d.i4) e = cudaMemcpyAsync(L.w_out4, wt_out4.data(), wt_out4.size(), H2D, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(L.s_out, w->s_out, (size_t)d.hidden * 4, H2D, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(L.S, 0, s_elems * 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(L.ring, 0, MB * d.conv_k * d.conv_ch * 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(L.rpos, 0, MB * 2 * 4, st);
    if (e == cudaSuccess && xb_bytes_in) e = cudaMemsetAsync(L.xb_in, 0, xb_bytes_in, st);
    if (e == cudaSuccess && xb_bytes_out) e = cudaMemsetAsync(L.xb_out, 0, xb_bytes_out, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(L.err, 0, 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(L.pool, 0, 4, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        layer_free_all(l);
        delete l;
        return DN_ECUDA;
    }
    *out = l;
    return DN_OK;
}

DN_API void dn_destroy(dn_layer *l) {
    if (l == nullptr) return;
    int cur = 0;
    cudaGetDevice(&cur);
    if (cur != l->device) cudaSetDevice(l->device);
    if (l->step_done_pending) cudaEventSynchronize(l->step_done);
    cudaStreamSynchronize(l->stream);
    layer_free_all(l);
    if (cur != l->device) cudaSetDevice(cur);
    delete l;
}

DN_API int dn_debug_fail_next(dn_layer *l, int code) {
    if (l == nullptr || code > 0) return DN_EINVAL;
    l->fail_next = code;
    return DN_OK;
}

DN_API int dn_debug_expire_wait(dn_layer *l, int limit_us) {
    if (l == nullptr || limit_us < 0 || limit_us > 1000000) return DN_EINVAL;
    l->expire_us_next = limit_us;
    return DN_OK;
}

DN_API int dn_profile_next_step(dn_layer *l, void *const *events) {
    if (l == nullptr) return DN_EINVAL;
    if (events == nullptr) {
        l->prof_armed = 0;
        return DN_OK;
    }
    for (int i = 0; i < 5; ++i) {
        if (events[i] == nullptr) return DN_EINVAL;
        l->prof[i] = (cudaEvent_t)events[i];
    }
    l->prof_armed = 1;
    return DN_OK;
}

DN_API int dn_step_kernels(const dn_layer *l, int batch) {
    if (l == nullptr || batch < 1 || batch > l->d.max_batch) return 0;
    const bool tc = batch >= dn::kTcMinBatch;
    const int in_proj = tc ? 2 : 1;                                // (pack) + projection
    return in_proj + 1 + 1 + 1;  // state kernel, out projection, reduction
}

DN_API int dn_stack_step(dn_layer *const *layers, int n_layers, int batch, float *h, const float *g,
                         const float *beta, float eps, void *stream) {
    if (layers == nullptr || n_layers < 1 || h == nullptr) return DN_EINVAL;
    if (!(eps >= 0.f)) return DN_EINVAL;
    dn_layer *first = layers[0];
    if (first == nullptr) return DN_EINVAL;
    const dn::Dims &d0 = first->d;
    for (int l = 0; l < n_layers; ++l) {
        const dn_layer *L = layers[l];
        if (L == nullptr || L->device != first->device) return DN_EINVAL;
        if (L->d.hidden != d0.hidden || L->d.n_v != d0.n_v || L->d.gw != d0.gw) return DN_EINVAL;
        if (L->d.dev_gates != d0.dev_gates) return DN_EINVAL;
        if (batch < 1 || batch > L->d.max_batch) return DN_EINVAL;
        if (L->failed) return DN_EFAILED;
    }
    // gates: from the caller, or (device gates) from the layers themselves
    if (d0.dev_gates ? (g != nullptr || beta != nullptr) : (g == nullptr || beta == nullptr)) return DN_EINVAL;
    int cur = 0;
    if (cudaGetDevice(&cur) != cudaSuccess || cur != first->device) return DN_EINVAL;
    cudaStream_t st = stream != nullptr ? (cudaStream_t)stream : first->stream;
    // the first layer's staging buffers hold the normalised input and the
    // layer output (dn_step with device pointers does not touch them)
    float *xn = first->L.x_stage, *y = first->L.out_stage;
    const size_t gstride = (size_t)batch * d0.n_v;  // beta; g has gw values per head
    if (dn::launch_residual_prenorm(h, nullptr, xn, batch, d0.hidden, eps, st) != cudaSuccess)
        return cuda_fail(first);
    for (int l = 0; l < n_layers; ++l) {
        const float *gl = d0.dev_gates ? nullptr : g + l * gstride * d0.gw;
        const float *bl = d0.dev_gates ? nullptr : beta + l * gstride;
        const int rc = dn_step(layers[l], batch, xn, gl, bl, y, DN_PTR_DEVICE, st);
        if (rc != DN_OK) return rc;
        // h += y and the next layer's input (after the last layer: only the add matters)
        if (dn::launch_residual_prenorm(h, y, xn, batch, d0.hidden, eps, st) != cudaSuccess)
            return cuda_fail(layers[l]);
    }
    return DN_OK;
}

DN_API int dn_set_state(dn_layer *l, int seq0, int n, const float *S, const float *ring,
                        const int32_t *ring_pos, int ptr_kind) {
    if (l == nullptr) return DN_EINVAL;
    const dn::Dims &d = l->d;
    if (ptr_kind != DN_PTR_HOST && ptr_kind != DN_PTR_DEVICE) return DN_EINVAL;
    if (seq0 < 0 || n < 1 || seq0 + n > d.max_batch) return DN_EINVAL;
    if (S == nullptr || ring == nullptr || ring_pos == nullptr) return DN_EINVAL;
    if (!on_layer_device(l)) return DN_EINVAL;
    if (l->failed) return DN_EFAILED;
    cudaStream_t st = l->stream;
    DN_TRY(l, order_after_steps(l));

    // ring positions are validated on the host before anything is written
    std::vector<int32_t> rp((size_t)n);
    if (ptr_kind == DN_PTR_HOST) {
        std::memcpy(rp.data(), ring_pos, (size_t)n * 4);
    } else {
        DN_TRY(l, cudaMemcpyAsync(rp.data(), ring_pos, (size_t)n * 4, cudaMemcpyDeviceToHost, st));
        DN_TRY(l, cudaStreamSynchronize(st));
    }
    for (int i = 0; i < n; ++i)
        if (rp[i] < 0 || rp[i] > d.conv_k - 2) return DN_EINVAL;

    const size_t tile = (size_t)d.n_v * d.dk * d.dv;
    const size_t ring_n = (size_t)n * (d.conv_k - 1) * d.conv_ch;
    const cudaMemcpyKind kind = ptr_kind == DN_PTR_HOST ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice;
    DN_TRY(l, cudaMemcpyAsync(l->L.S + (size_t)seq0 * tile, S, (size_t)n * tile * 4, kind, st));
    DN_TRY(l, cudaMemcpyAsync(l->L.ring_stage, ring, ring_n * 4, kind, st));
    DN_TRY(l, cudaMemcpyAsync(l->L.rp_stage, rp.data(), (size_t)n * 4, cudaMemcpyHostToDevice, st));
    DN_TRY(l, dn::launch_ring_import(d, l->L, seq0, n, st));
    DN_TRY(l, cudaStreamSynchronize(st));
    return DN_OK;
}

DN_API int dn_get_state(dn_layer *l, int seq0, int n, float *S, float *ring, int32_t *ring_pos,
                        int ptr_kind) {
    if (l == nullptr) return DN_EINVAL;
    const dn::Dims &d = l->d;
    if (ptr_kind != DN_PTR_HOST && ptr_kind != DN_PTR_DEVICE) return DN_EINVAL;
    if (seq0 < 0 || n < 1 || seq0 + n > d.max_batch) return DN_EINVAL;
    if (!on_layer_device(l)) return DN_EINVAL;
    cudaStream_t st = l->stream;
    const size_t tile = (size_t)d.n_v * d.dk * d.dv;
    const size_t ring_n = (size_t)n * (d.conv_k - 1) * d.conv_ch;
    const cudaMemcpyKind kind = ptr_kind == DN_PTR_HOST ? cudaMemcpyDeviceToHost : cudaMemcpyDeviceToDevice;
    cudaError_t e = order_after_steps(l);
    if (S != nullptr)
        e = cudaMemcpyAsync(S, l->L.S + (size_t)seq0 * tile, (size_t)n * tile * 4, kind, st);
    if (e == cudaSuccess && (ring != nullptr || ring_pos != nullptr))
        e = dn::launch_ring_export(d, l->L, seq0, n, st);
    if (e == cudaSuccess && ring != nullptr)
        e = cudaMemcpyAsync(ring, l->L.ring_stage, ring_n * 4, kind, st);
    if (e == cudaSuccess && ring_pos != nullptr)
        e = cudaMemcpyAsync(ring_pos, l->L.rp_stage, (size_t)n * 4, kind, st);
    int dev_err = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&dev_err, l->L.err, 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(l);
    if (dev_err != 0) return cuda_fail(l);  // a kernel gave up on a bounded wait
    return DN_OK;
}

namespace {

// dn_prefill's scratch, for blocks of up to kPrefillCols token columns
int ensure_prefill(dn_layer *l) {
    if (l->prefill_ready) return DN_OK;
    const dn::Dims &d = l->d;
    dn::PrefillDev &P = l->P;
    const size_t C = dn::kPrefillCols;
    size_t part_in = 0, part_out = 0, tiles_in = 0, tiles_out = 0;
    for (int c = 1; c <= (int)C; ++c) {
        const dn::GemmPlan gi = dn::plan_tc_gemm(d.proj_rows, dn::plan_k(d, d.hidden, c), c);
        const dn::GemmPlan go = dn::plan_tc_gemm(d.hidden, dn::plan_k(d, d.v_dim, c), c);
        part_in = std::max(part_in, (size_t)gi.tiles * gi.max_seg * 64 * 128);
        part_out = std::max(part_out, (size_t)go.tiles * go.max_seg * 64 * 128);
        tiles_in = std::max(tiles_in, (size_t)gi.tiles);
        tiles_out = std::max(tiles_out, (size_t)go.tiles);
    }
    const size_t chunks = (C + 63) / 64;
    const size_t kt_in = (size_t)(d.hidden + dn::kTileK - 1) / dn::kTileK;
    const size_t kt_out = (size_t)(d.v_dim + dn::kTileK - 1) / dn::kTileK;
    int rc = DN_OK;
#define PALLOC(ptr, bytes) \
    if (rc == DN_OK) rc = layer_alloc(l, (void **)&(ptr), (size_t)(bytes));
    PALLOC(P.xg, C * d.hidden * 4);
    PALLOC(P.xb_in, chunks * kt_in * dn::kOpTile);
    PALLOC(P.part_in, part_in * 4);
    PALLOC(P.nseg_in, tiles_in * 4);
    PALLOC(P.xin, C * d.proj_rows * 4);
    PALLOC(P.qn, C * d.qk_dim * 4);
    PALLOC(P.kn, C * d.qk_dim * 4);
    PALLOC(P.vv, C * d.v_dim * 4);
    PALLOC(P.zs, C * d.v_dim * 4);
    PALLOC(P.gg, C * d.n_v * d.gw * 4);
    PALLOC(P.bb, C * d.n_v * 4);
    PALLOC(P.o, C * d.v_dim * 4);
    PALLOC(P.nrm, C * d.v_dim * 4);
    PALLOC(P.xb_out, chunks * kt_out * dn::kOpTile);
    PALLOC(P.part_out, part_out * 4);
    PALLOC(P.nseg_out, tiles_out * 4);
#undef PALLOC
    if (rc != DN_OK) return rc;  // (what was allocated stays with the layer and is freed with it)
    // the padded operand rows must read as zero
    if (cudaMemsetAsync(P.xb_in, 0, chunks * kt_in * dn::kOpTile, l->stream) != cudaSuccess ||
        cudaMemsetAsync(P.xb_out, 0, chunks * kt_out * dn::kOpTile, l->stream) != cudaSuccess ||
        cudaStreamSynchronize(l->stream) != cudaSuccess)
        return DN_ECUDA;
    l->prefill_ready = 1;
    return DN_OK;
}

// after work enqueued on a stream other than the layer's: state copies wait
// for it (a stream that captures a graph is ordered by whoever launches it)
cudaError_t note_foreign_stream(dn_layer *l, cudaStream_t st) {
    if (st == l->stream) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(st, &cs);
    if (e == cudaSuccess && cs == cudaStreamCaptureStatusNone) {
        e = cudaEventRecord(l->step_done, st);
        if (e == cudaSuccess) l->step_done_pending = 1;
    }
    return e;
}

}  // namespace

DN_API int dn_prefill(dn_layer *l, int batch, int n_tokens, const float *x, const float *g, const float *beta,
                      float *out, void *stream) {
    if (l == nullptr) return DN_EINVAL;
    const dn::Dims &d = l->d;
    if (batch < 1 || batch > d.max_batch || n_tokens < 1) return DN_EINVAL;
    if (x == nullptr || out == nullptr) return DN_EINVAL;
    if (((uintptr_t)x & 15u) != 0) return DN_EINVAL;  // rows are gathered with 16-byte loads
    if (d.dev_gates ? (g != nullptr || beta != nullptr) : (g == nullptr || beta == nullptr)) return DN_EINVAL;
    if ((size_t)batch * n_tokens > (size_t)INT32_MAX / 4) return DN_EINVAL;
    if (!on_layer_device(l)) return DN_EINVAL;
    if (l->failed) return DN_EFAILED;
    if (l->fail_next != 0) {
        const int code = l->fail_next;
        l->fail_next = 0;
        l->failed = 1;
        return code;
    }
    const int rc = ensure_prefill(l);
    if (rc == DN_ECUDA) return cuda_fail(l);
    if (rc != DN_OK) return rc;
    cudaStream_t st = stream != nullptr ? (cudaStream_t)stream : l->stream;
    for (int b0 = 0; b0 < batch; b0 += dn::kPrefillCols) {
        const int nb = std::min(dn::kPrefillCols, batch - b0);
        const int T = std::max(1, dn::kPrefillCols / nb);
        for (int t0 = 0; t0 < n_tokens; t0 += T) {
            const dn::PrefillBlock blk{b0, nb, t0, std::min(T, n_tokens - t0), n_tokens, x, g, beta, out};
            DN_TRY(l, dn::launch_prefill_block(d, l->L, l->P, blk, st));
        }
    }
    DN_TRY(l, note_foreign_stream(l, st));
    return DN_OK;
}

DN_API int dn_step(dn_layer *l, int batch, const float *x, const float *g, const float *beta,
                   float *out, int ptr_kind, void *stream) {
    if (l == nullptr) return DN_EINVAL;
    const dn::Dims &d = l->d;
    if (ptr_kind != DN_PTR_HOST && ptr_kind != DN_PTR_DEVICE) return DN_EINVAL;
    if (batch < 1 || batch > d.max_batch) return DN_EINVAL;
    if (x == nullptr || out == nullptr) return DN_EINVAL;
    if (ptr_kind == DN_PTR_DEVICE && ((uintptr_t)x & 15u) != 0) return DN_EINVAL;  // read 16 bytes at a time
    if (d.dev_gates ? (g != nullptr || beta != nullptr) : (g == nullptr || beta == nullptr)) return DN_EINVAL;
    if (!on_layer_device(l)) return DN_EINVAL;
    if (l->failed) return DN_EFAILED;
    if (l->fail_next != 0) {
        const int code = l->fail_next;
        l->fail_next = 0;
        l->failed = 1;
        return code;
    }
    cudaStream_t st = stream != nullptr ? (cudaStream_t)stream : l->stream;
    const dn::LayerDev &L = l->L;
    const float *xd = x, *gd = g, *bd = beta;
    float *od = out;
    if (ptr_kind == DN_PTR_HOST) {
        DN_TRY(l, cudaMemcpyAsync(L.x_stage, x, (size_t)batch * d.hidden * 4, cudaMemcpyHostToDevice, st));
        if (!d.dev_gates) {
            DN_TRY(l, cudaMemcpyAsync(L.g_stage, g, (size_t)batch * d.n_v * d.gw * 4, cudaMemcpyHostToDevice, st));
            DN_TRY(l, cudaMemcpyAsync(L.beta_stage, beta, (size_t)batch * d.n_v * 4, cudaMemcpyHostToDevice, st));
            gd = L.g_stage;
            bd = L.beta_stage;
        }
        xd = L.x_stage;
        od = L.out_stage;
    }
    if (l->expire_us_next > 0) {
        const int us = l->expire_us_next;
        l->expire_us_next = 0;
        DN_TRY(l, dn::launch_expire_wait(L.err, us, st));
    }
    const bool prof = l->prof_armed != 0;
    l->prof_armed = 0;
    if (prof) DN_TRY(l, cudaEventRecord(l->prof[0], st));
    const bool tc = batch >= dn::kTcMinBatch;
    if (tc) {
        DN_TRY(l, dn::launch_pack_b(xd, L.xb_in, batch, d.hidden, st));
        DN_TRY(l, dn::launch_gemm_i8_tc(L.w_in, L.xb_in, L.part_in, L.nseg_in, L.err, d.proj_rows,
                                        d.hidden, batch, st));
    } else {
        DN_TRY(l, dn::launch_gemv_i8(d.i4 ? L.w_in4 : L.w_in, xd, L.part_in, L.nseg_in, L.err, d.proj_rows,
                                     d.hidden, batch, st, d.i4 != 0));
    }
    if (prof) DN_TRY(l, cudaEventRecord(l->prof[1], st));
    if (prof) DN_TRY(l, cudaEventRecord(l->prof[2], st));  // no separate preparation kernel
    if (dn::dn_core_stream_ok(d, batch))
        DN_TRY(l, dn::launch_dn_core_stream(d, L, batch, gd, bd, tc, st));
    else
        DN_TRY(l, dn::launch_dn_core(d, L, batch, gd, bd, tc, st));
    if (prof) DN_TRY(l, cudaEventRecord(l->prof[3], st));
    if (tc)
        DN_TRY(l, dn::launch_gemm_i8_tc(L.w_out, L.xb_out, L.part_out, L.nseg_out, L.err, d.hidden,
                                        d.v_dim, batch, st));
    else
        DN_TRY(l, dn::launch_gemv_i8(d.i4 ? L.w_out4 : L.w_out, L.nrm, L.part_out, L.nseg_out, L.err, d.hidden,
                                     d.v_dim, batch, st, d.i4 != 0));
    DN_TRY(l, dn::launch_splitk_reduce(L.part_out, L.nseg_out, L.s_out, od, d.hidden, dn::plan_k(d, d.v_dim, batch), batch,
                                       L.rpos, d.conv_k, st, 1, 1, 0, 1, L.pool));
    if (prof) DN_TRY(l, cudaEventRecord(l->prof[4], st));
    DN_TRY(l, note_foreign_stream(l, st));  // later state copies wait for this step
    if (ptr_kind == DN_PTR_HOST) {
        DN_TRY(l, cudaMemcpyAsync(out, L.out_stage, (size_t)batch * d.hidden * 4, cudaMemcpyDeviceToHost, st));
        DN_TRY(l, cudaStreamSynchronize(st));
    }
    return DN_OK;
}
