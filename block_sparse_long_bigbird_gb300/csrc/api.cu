// Host side of the C ABI: argument validation, kernel selection, the device
// status word, scratch (workspace) management and options.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "internal.h"
#include "tc_sync.cuh"

namespace {

// Per-device latched status (OR of sa::DeviceStatusBits). Every device that
// loads the library holds its own copy of this module variable.
__device__ unsigned int g_device_status;

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    unsigned int *status = nullptr;  // device address of g_device_status
    int cc_major = 0, cc_minor = 0, num_sms = 0;
    void *ws = nullptr;  // library-owned scratch
    size_t ws_bytes = 0;
    size_t ws_clean = 0;  // [0, ws_clean) of `ws` is known to be zero between calls
    void *user_ws = nullptr;  // caller-owned scratch (sa_set_workspace)
    size_t user_ws_bytes = 0;
    size_t user_ws_clean = 0;
    // host-buffer path: copy streams, events and device staging buffers
    bool host_ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t ev_start = nullptr, ev_last = nullptr;
    cudaEvent_t ev_in[2] = {}, ev_done[2] = {}, ev_out[2] = {};
    void *stage = nullptr;
    size_t stage_bytes = 0;
};

std::mutex g_mutex;
// Held while a host-buffer call enqueues its work: calls share the staging
// sets, and the event chain between them is built in enqueue order.
std::mutex g_host_mutex;
DeviceState g_devices[kMaxDevices];
std::atomic<int> g_force_simt{0};
std::atomic<long long> g_wait_limit{2000000};  // microseconds
std::atomic<int> g_max_splits{16};
std::atomic<int> g_grid_ctas{0};
std::atomic<int> g_chunk_keys{0};
thread_local int g_last_launches = 0;

sa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? SA_OK : SA_ERR_CUDA; }

// Returns the state of the current device, initialising it on first use.
sa_status current_device(int *dev_out, DeviceState **st_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return SA_ERR_UNSUPPORTED;
    DeviceState &st = g_devices[dev];
    if (!st.ready) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) return SA_ERR_CUDA;
        st.status = static_cast<unsigned int *>(addr);
        if (cudaDeviceGetAttribute(&st.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&st.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SA_ERR_CUDA;
        st.ready = true;
    }
    *dev_out = dev;
    *st_out = &st;
    return SA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

sa_status check_tensors(const void *Q, const void *K, const void *V, const void *O) {
    if (!Q || !K || !V || !O) return SA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O)) return SA_ERR_INVALID_ARG;
    if (O == Q || O == K || O == V) return SA_ERR_INVALID_ARG;
    return SA_OK;
}

bool size_ok(int B, int H, int n, int d) {
    if (B < 1 || H < 1 || n < 1) return false;
    if (d != 64 && d != 128) return false;
    // Offsets are computed in 64-bit, but per-head row counts and grid sizes are 32-bit.
    if ((long long)B * H > (1ll << 30)) return false;
    return true;
}

size_t bwd_stats_bytes(int B, int H, int n) { return 2 * sizeof(float) * (size_t)B * H * sa::stats_stride(n); }

sa_status bigbird_args_ok(int B, int H, int n, int d, int b, int g, int w, int r, const int32_t *rand_idx) {
    if (!size_ok(B, H, n, d)) return SA_ERR_INVALID_ARG;
    if (b != 64 && b != 128) return SA_ERR_INVALID_ARG;
    if (n % b != 0) return SA_ERR_INVALID_ARG;
    if (g < 0 || g > n / b) return SA_ERR_INVALID_ARG;
    if (w < 1 || (w % 2) == 0) return SA_ERR_INVALID_ARG;
    if (r < 0 || (r > 0 && !rand_idx)) return SA_ERR_INVALID_ARG;
    return SA_OK;
}

sa_status longformer_args_ok(int B, int H, int n, int d, int window, const int32_t *global_idx, int n_global) {
    if (!size_ok(B, H, n, d)) return SA_ERR_INVALID_ARG;
    if (window < 0 || (window % 2) != 0) return SA_ERR_INVALID_ARG;
    if (n_global < 0 || n_global > n || (n_global > 0 && !global_idx)) return SA_ERR_INVALID_ARG;
    return SA_OK;
}

sa::TcConfig tc_config(const DeviceState *st) {
    sa::TcConfig cfg;
    const int grid = g_grid_ctas.load();
    cfg.grid_ctas = grid > 0 ? grid : (st ? st->num_sms : 148);
    cfg.max_splits = g_max_splits.load();
    cfg.chunk_keys = g_chunk_keys.load();
    cfg.wait_limit = g_wait_limit.load();
    return cfg;
}

// Scratch for one call: the caller's region if one is set, else the
// library-owned region, grown (and zeroed) on demand.
sa_status get_workspace(DeviceState &st, size_t need, void **ptr) {
    if (need == 0) {
        *ptr = nullptr;
        return SA_OK;
    }
    if (st.user_ws) {
        if (st.user_ws_bytes < need) return SA_ERR_INVALID_ARG;
        *ptr = st.user_ws;
        return SA_OK;
    }
    if (st.ws_bytes < need) {
        // Every call that used the old region was issued before this one; a
        // device-wide sync makes the free safe whatever streams they ran on.
        if (st.ws) {
            if (cudaDeviceSynchronize() != cudaSuccess) return SA_ERR_CUDA;
            cudaFree(st.ws);
            st.ws = nullptr;
            st.ws_bytes = 0;
        }
        const size_t bytes = (need + 0xFFFFF) & ~(size_t)0xFFFFF;
        if (cudaMalloc(&st.ws, bytes) != cudaSuccess) return SA_ERR_CUDA;
        if (cudaMemset(st.ws, 0, bytes) != cudaSuccess) return SA_ERR_CUDA;
        st.ws_bytes = bytes;
        st.ws_clean = bytes;
    }
    *ptr = st.ws;
    return SA_OK;
}

sa_status run(const sa::Problem &prob_in, sa_dtype dtype, cudaStream_t stream) {
    int dev = 0;
    DeviceState *st = nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    sa_status s = current_device(&dev, &st);
    if (s != SA_OK) return s;
    if (st->cc_major != 10 || st->cc_minor != 3) return SA_ERR_UNSUPPORTED;
    sa::Problem prob = prob_in;
    prob.status = st->status;
    int launches = 0;
    cudaError_t e;
    if (dtype == SA_FP32 || g_force_simt.load()) {
        e = sa::launch_simt(prob, dtype, stream, &launches);
    } else {
        const sa::TcConfig cfg = tc_config(st);
        void *ws = nullptr;
        // Dilated Longformer heads run on residue-class copies of Q, K, V when
        // the call has no global tokens, key mask or separate projections and
        // the scratch can hold the copies (always for the library's own).
        if (prob.kind == sa::kLongformer && prob.dilation && prob.n_global == 0 && !prob.key_mask && !prob.Qg) {
            prob.class_perm = 1;
            if (st->user_ws && st->user_ws_bytes < sa::tc_workspace_bytes(prob, cfg)) prob.class_perm = 0;
        }
        const size_t need = sa::tc_workspace_bytes(prob, cfg);
        s = get_workspace(*st, need, &ws);
        if (s != SA_OK) return s;
        // The kernel needs its counters zero at entry. A call leaves its own
        // counters zero but writes split partials past them, and the next call
        // (another shape) may place counters over those bytes: clear them then.
        size_t *clean = (ws == st->user_ws) ? &st->user_ws_clean : &st->ws_clean;
        const size_t counters = sa::tc_workspace_counter_bytes(prob, cfg);
        if (ws && counters > *clean) {
            if (cudaMemsetAsync(ws, 0, counters, stream) != cudaSuccess) return SA_ERR_CUDA;
            *clean = counters;
        }
        e = sa::launch_tc(prob, cfg, ws, need, stream, &launches);
        if (e == cudaErrorNotSupported) return SA_ERR_UNSUPPORTED;
        if (e == cudaSuccess && need > counters) *clean = counters;  // partials dirty [counters, need)
    }
    if (e != cudaSuccess) return SA_ERR_CUDA;
    g_last_launches = launches;
    return SA_OK;
}

// Backward: scratch holds the per-row statistics (2 * B * H * n floats) at
// offset 0, so the forward's counters must be cleared before its next use.
sa_status run_bwd(const sa::Problem &prob_in, sa_dtype dtype, cudaStream_t stream) {
    int dev = 0;
    DeviceState *st = nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    sa_status s = current_device(&dev, &st);
    if (s != SA_OK) return s;
    if (st->cc_major != 10 || st->cc_minor != 3) return SA_ERR_UNSUPPORTED;
    sa::Problem prob = prob_in;
    prob.status = st->status;
    void *ws = nullptr;
    const size_t need = bwd_stats_bytes(prob.B, prob.H, prob.n);
    s = get_workspace(*st, need, &ws);
    if (s != SA_OK) return s;
    prob.row_stats = static_cast<float *>(ws);
    size_t *clean = (ws == st->user_ws) ? &st->user_ws_clean : &st->ws_clean;
    *clean = 0;
    int launches = 0;
    cudaError_t e;
    if (dtype == SA_FP32 || g_force_simt.load())
        e = sa::launch_simt_bwd(prob, dtype, stream, &launches);
    else
        e = sa::launch_tc_bwd(prob, tc_config(st), stream, &launches);
    if (e == cudaErrorNotSupported) return SA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return SA_ERR_CUDA;
    g_last_launches = launches;
    return SA_OK;
}

sa_status check_bwd_tensors(const void *Q, const void *K, const void *V, const void *dO, const void *dQ,
                            const void *dK, const void *dV) {
    const void *in[4] = {Q, K, V, dO};
    const void *out[3] = {dQ, dK, dV};
    for (const void *t : in)
        if (!t || !aligned16(t)) return SA_ERR_INVALID_ARG;
    for (int a = 0; a < 3; ++a) {
        if (!out[a] || !aligned16(out[a])) return SA_ERR_INVALID_ARG;
        for (const void *t : in)
            if (out[a] == t) return SA_ERR_INVALID_ARG;
        for (int b = 0; b < a; ++b)
            if (out[a] == out[b]) return SA_ERR_INVALID_ARG;
    }
    return SA_OK;
}

// ---------------------------------------------------------------------------
// Host-buffer path: the forward on HOST tensors, pipelined over chunks of heads.
// Chunk k's inputs are copied in on one library stream while chunk k - 1
// computes on the caller's stream and chunk k - 2's output is copied out on a
// second library stream; two device staging sets alternate. Every chunk is an
// ordinary device-side call of the library on a slice of heads of one batch
// entry, so the numerics are those of the device entry points.
constexpr int kHostChunks = 4;  // target number of chunks per call

sa_status host_path_init(DeviceState &st) {
    if (st.host_ready) return SA_OK;
    if (cudaStreamCreateWithFlags(&st.h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&st.d2h, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&st.ev_start, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&st.ev_last, cudaEventDisableTiming) != cudaSuccess)
        return SA_ERR_CUDA;
    for (int i = 0; i < 2; ++i)
        if (cudaEventCreateWithFlags(&st.ev_in[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&st.ev_done[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&st.ev_out[i], cudaEventDisableTiming) != cudaSuccess)
            return SA_ERR_CUDA;
    // the first call waits on ev_last: give it a completed state
    if (cudaEventRecord(st.ev_last, st.d2h) != cudaSuccess) return SA_ERR_CUDA;
    st.host_ready = true;
    return SA_OK;
}

// `hp` carries HOST pointers in Q, K, V, O, rand_idx / global_idx, dilation
// and key_mask. A chunk is `bc` whole batch entries, or (when one batch entry
// is more than a chunk) `hc` consecutive heads of one batch entry; either way
// its rows are one contiguous stretch of the [B][H][n][d] arrays.
sa_status run_host(const sa::Problem &hp, sa_dtype dtype, cudaStream_t s) {
    std::lock_guard<std::mutex> host_lock(g_host_mutex);
    const size_t elem = dtype == SA_FP32 ? 4 : 2;
    const int B = hp.B, H = hp.H, n = hp.n, d = hp.d;
    const size_t head_bytes = (size_t)n * d * elem;
    const int per_chunk = std::max(1, (B * H + kHostChunks - 1) / kHostChunks);  // (batch, head) pairs
    const int bc = per_chunk >= H ? per_chunk / H : 1;   // batch entries per chunk
    const int hc = per_chunk >= H ? H : per_chunk;       // heads per chunk (within one batch entry)
    const size_t set_bytes = 4 * (size_t)bc * hc * head_bytes;  // Q, K, V, O of one chunk
    // small tables, copied once per call
    const bool bb = hp.kind == sa::kBigBird;
    const size_t rand_bytes = bb && hp.rand_idx ? (size_t)H * (n / hp.b) * hp.r * 4 : 0;
    const size_t gidx_bytes = !bb && hp.global_idx ? (size_t)hp.n_global * 4 : 0;
    const size_t dil_bytes = !bb && hp.dilation ? (size_t)H * 4 : 0;
    const size_t km_bytes = hp.key_mask ? (size_t)B * n : 0;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t need = 2 * up(set_bytes) + up(rand_bytes) + up(gidx_bytes) + up(dil_bytes) + up(km_bytes);

    int dev = 0;
    DeviceState *st = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        sa_status e = current_device(&dev, &st);
        if (e != SA_OK) return e;
        if (st->cc_major != 10 || st->cc_minor != 3) return SA_ERR_UNSUPPORTED;
        if ((e = host_path_init(*st)) != SA_OK) return e;
        if (st->stage_bytes < need) {
            if (st->stage) {
                if (cudaDeviceSynchronize() != cudaSuccess) return SA_ERR_CUDA;
                cudaFree(st->stage);
                st->stage = nullptr;
                st->stage_bytes = 0;
            }
            if (cudaMalloc(&st->stage, need) != cudaSuccess) return SA_ERR_CUDA;
            st->stage_bytes = need;
        }
    }
    uint8_t *base = static_cast<uint8_t *>(st->stage);
    uint8_t *sets[2] = {base, base + up(set_bytes)};
    uint8_t *tab = base + 2 * up(set_bytes);
    int32_t *d_rand = rand_bytes ? reinterpret_cast<int32_t *>(tab) : nullptr;
    tab += up(rand_bytes);
    int32_t *d_gidx = gidx_bytes ? reinterpret_cast<int32_t *>(tab) : nullptr;
    tab += up(gidx_bytes);
    int32_t *d_dil = dil_bytes ? reinterpret_cast<int32_t *>(tab) : nullptr;
    tab += up(dil_bytes);
    uint8_t *d_km = km_bytes ? tab : nullptr;

    // order: after earlier work on the caller's stream and the previous host call
    if (cudaEventRecord(st->ev_start, s) != cudaSuccess || cudaStreamWaitEvent(st->h2d, st->ev_start, 0) != cudaSuccess ||
        cudaStreamWaitEvent(st->h2d, st->ev_last, 0) != cudaSuccess)
        return SA_ERR_CUDA;
    // From here on copies may be queued on the library streams. An error exit
    // still closes the chain: the output copies already queued end with
    // ev_last on the output stream (which the copy-in stream also follows), and
    // the caller's stream waits on it, so the caller may free or reuse its host
    // buffers once its stream has drained, even after an error.
    auto fail = [&](sa_status e) {
        cudaEventRecord(st->ev_start, st->h2d);  // everything queued for copy-in so far
        cudaStreamWaitEvent(st->d2h, st->ev_start, 0);
        cudaEventRecord(st->ev_last, st->d2h);
        cudaStreamWaitEvent(s, st->ev_last, 0);
        return e;
    };
    if (rand_bytes && cudaMemcpyAsync(d_rand, hp.rand_idx, rand_bytes, cudaMemcpyHostToDevice, st->h2d) != cudaSuccess)
        return fail(SA_ERR_CUDA);
    if (gidx_bytes && cudaMemcpyAsync(d_gidx, hp.global_idx, gidx_bytes, cudaMemcpyHostToDevice, st->h2d) != cudaSuccess)
        return fail(SA_ERR_CUDA);
    if (dil_bytes && cudaMemcpyAsync(d_dil, hp.dilation, dil_bytes, cudaMemcpyHostToDevice, st->h2d) != cudaSuccess)
        return fail(SA_ERR_CUDA);
    if (km_bytes && cudaMemcpyAsync(d_km, hp.key_mask, km_bytes, cudaMemcpyHostToDevice, st->h2d) != cudaSuccess)
        return fail(SA_ERR_CUDA);

    int launches = 0, k = 0;
    const size_t chunk_cap = (size_t)bc * hc * head_bytes;
    for (int beta = 0; beta < B; beta += bc) {
        const int nb_here = std::min(bc, B - beta);
        for (int h0 = 0; h0 < H; h0 += hc, ++k) {
            const int cnt = std::min(hc, H - h0);
            const int set = k & 1;
            const size_t off = ((size_t)beta * H + h0) * head_bytes;  // byte offset of the slice in [B][H][n][d]
            const size_t bytes = (size_t)nb_here * cnt * head_bytes;
            uint8_t *dq = sets[set], *dk = dq + chunk_cap, *dv = dk + chunk_cap, *dout = dv + chunk_cap;
            // the staging set is free once chunk k - 2's output has been copied out
            if (k >= 2 && cudaStreamWaitEvent(st->h2d, st->ev_out[set], 0) != cudaSuccess) return fail(SA_ERR_CUDA);
            if (cudaMemcpyAsync(dq, static_cast<const uint8_t *>(hp.Q) + off, bytes, cudaMemcpyHostToDevice, st->h2d) !=
                    cudaSuccess ||
                cudaMemcpyAsync(dk, static_cast<const uint8_t *>(hp.K) + off, bytes, cudaMemcpyHostToDevice, st->h2d) !=
                    cudaSuccess ||
                cudaMemcpyAsync(dv, static_cast<const uint8_t *>(hp.V) + off, bytes, cudaMemcpyHostToDevice, st->h2d) !=
                    cudaSuccess ||
                cudaEventRecord(st->ev_in[set], st->h2d) != cudaSuccess || cudaStreamWaitEvent(s, st->ev_in[set], 0) != cudaSuccess)
                return fail(SA_ERR_CUDA);
            sa::Problem p = hp;
            p.Q = dq;
            p.K = dk;
            p.V = dv;
            p.O = dout;
            p.B = nb_here;  // whole batch entries (cnt == H), or one entry's heads [h0, h0 + cnt)
            p.H = cnt;
            p.key_mask = d_km ? d_km + (size_t)beta * n : nullptr;
            if (bb) {
                p.rand_idx = d_rand ? d_rand + (size_t)h0 * (n / hp.b) * hp.r : nullptr;
            } else {
                p.global_idx = d_gidx;
                p.dilation = d_dil ? d_dil + h0 : nullptr;
            }
            const sa_status e = run(p, dtype, s);
            if (e != SA_OK) return fail(e);
            launches += g_last_launches;
            if (cudaEventRecord(st->ev_done[set], s) != cudaSuccess ||
                cudaStreamWaitEvent(st->d2h, st->ev_done[set], 0) != cudaSuccess ||
                cudaMemcpyAsync(static_cast<uint8_t *>(hp.O) + off, dout, bytes, cudaMemcpyDeviceToHost, st->d2h) !=
                    cudaSuccess ||
                cudaEventRecord(st->ev_out[set], st->d2h) != cudaSuccess)
                return fail(SA_ERR_CUDA);
        }
    }
    // the caller's stream completes once the last output copy has (the copies
    // of one stream run in order)
    if (cudaEventRecord(st->ev_last, st->d2h) != cudaSuccess || cudaStreamWaitEvent(s, st->ev_last, 0) != cudaSuccess)
        return SA_ERR_CUDA;
    g_last_launches = launches;
    return SA_OK;
}

}  // namespace

extern "C" {

sa_status bigbird_attn_fwd(const void *Q, const void *K, const void *V, void *O, int B, int H, int n, int d,
                           int b, int g, int w, int r, const int32_t *rand_idx, const uint8_t *key_mask,
                           sa_dtype dtype, sa_stream_t stream) {
    if (dtype != SA_BF16 && dtype != SA_FP32) return SA_ERR_INVALID_ARG;
    sa_status s = check_tensors(Q, K, V, O);
    if (s != SA_OK) return s;
    s = bigbird_args_ok(B, H, n, d, b, g, w, r, rand_idx);
    if (s != SA_OK) return s;
    if (!aligned16(key_mask)) return SA_ERR_INVALID_ARG;
    sa::Problem p = {};
    p.kind = sa::kBigBird;
    p.Q = Q; p.K = K; p.V = V; p.O = O;
    p.B = B; p.H = H; p.n = n; p.d = d;
    p.b = b; p.g = g; p.w = w; p.r = r;
    p.rand_idx = r > 0 ? rand_idx : nullptr;
    p.key_mask = key_mask;
    return run(p, dtype, reinterpret_cast<cudaStream_t>(stream));
}

sa_status longformer_attn_fwd(const void *Q, const void *K, const void *V, void *O, int B, int H, int n, int d,
                              int window, const int32_t *global_idx, int n_global, const uint8_t *key_mask,
                              sa_dtype dtype, sa_stream_t stream) {
    return longformer_attn_fwd_ex(Q, K, V, O, B, H, n, d, window, nullptr, 0, global_idx, n_global, key_mask,
                                  dtype, stream);
}

sa_status longformer_attn_fwd_ex(const void *Q, const void *K, const void *V, void *O, int B, int H, int n, int d,
                                 int window, const int32_t *dilation, int causal, const int32_t *global_idx,
                                 int n_global, const uint8_t *key_mask, sa_dtype dtype, sa_stream_t stream) {
    return longformer_attn_fwd_gproj(Q, K, V, nullptr, nullptr, nullptr, O, B, H, n, d, window, dilation, causal,
                                     global_idx, n_global, key_mask, dtype, stream);
}

sa_status longformer_attn_fwd_gproj(const void *Q, const void *K, const void *V, const void *Qg, const void *Kg,
                                    const void *Vg, void *O, int B, int H, int n, int d, int window,
                                    const int32_t *dilation, int causal, const int32_t *global_idx, int n_global,
                                    const uint8_t *key_mask, sa_dtype dtype, sa_stream_t stream) {
    if (dtype != SA_BF16 && dtype != SA_FP32) return SA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return SA_ERR_INVALID_ARG;
    sa_status s = check_tensors(Q, K, V, O);
    if (s != SA_OK) return s;
    // the separate set: all three or none, aligned, never aliasing O
    const bool sep = Qg || Kg || Vg;
    if (sep) {
        s = check_tensors(Qg, Kg, Vg, O);
        if (s != SA_OK) return s;
    }
    s = longformer_args_ok(B, H, n, d, window, global_idx, n_global);
    if (s != SA_OK) return s;
    sa::Problem p = {};
    p.kind = sa::kLongformer;
    p.Q = Q; p.K = K; p.V = V; p.O = O;
    p.B = B; p.H = H; p.n = n; p.d = d;
    p.window = window;
    p.global_idx = n_global > 0 ? global_idx : nullptr;
    p.n_global = n_global;
    p.dilation = dilation;
    p.causal = causal;
    p.key_mask = key_mask;
    if (sep) {
        p.Qg = Qg;
        p.Kg = Kg;
        p.Vg = Vg;
    }
    return run(p, dtype, reinterpret_cast<cudaStream_t>(stream));
}

sa_status bigbird_attn_bwd(const void *Q, const void *K, const void *V, const void *dO, void *dQ, void *dK,
                           void *dV, int B, int H, int n, int d, int b, int g, int w, int r,
                           const int32_t *rand_idx, const uint8_t *key_mask, sa_dtype dtype, sa_stream_t stream) {
    if (dtype != SA_BF16 && dtype != SA_FP32) return SA_ERR_INVALID_ARG;
    sa_status s = check_bwd_tensors(Q, K, V, dO, dQ, dK, dV);
    if (s != SA_OK) return s;
    s = bigbird_args_ok(B, H, n, d, b, g, w, r, rand_idx);
    if (s != SA_OK) return s;
    if (!aligned16(key_mask)) return SA_ERR_INVALID_ARG;
    sa::Problem p = {};
    p.kind = sa::kBigBird;
    p.Q = Q; p.K = K; p.V = V;
    p.dO = dO; p.dQ = dQ; p.dK = dK; p.dV = dV;
    p.B = B; p.H = H; p.n = n; p.d = d;
    p.b = b; p.g = g; p.w = w; p.r = r;
    p.rand_idx = r > 0 ? rand_idx : nullptr;
    p.key_mask = key_mask;
    return run_bwd(p, dtype, reinterpret_cast<cudaStream_t>(stream));
}

sa_status longformer_attn_bwd(const void *Q, const void *K, const void *V, const void *dO, void *dQ, void *dK,
                              void *dV, int B, int H, int n, int d, int window,
                              const int32_t *dilation, int causal, const int32_t *global_idx, int n_global,
                              const uint8_t *key_mask, sa_dtype dtype, sa_stream_t stream) {
    if (dtype != SA_BF16 && dtype != SA_FP32) return SA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return SA_ERR_INVALID_ARG;
    sa_status s = check_bwd_tensors(Q, K, V, dO, dQ, dK, dV);
    if (s != SA_OK) return s;
    s = longformer_args_ok(B, H, n, d, window, global_idx, n_global);
    if (s != SA_OK) return s;
    sa::Problem p = {};
    p.kind = sa::kLongformer;
    p.Q = Q; p.K = K; p.V = V;
    p.dO = dO; p.dQ = dQ; p.dK = dK; p.dV = dV;
    p.B = B; p.H = H; p.n = n; p.d = d;
    p.window = window;
    p.global_idx = n_global > 0 ? global_idx : nullptr;
    p.n_global = n_global;
    p.dilation = dilation;
    p.causal = causal;
    p.key_mask = key_mask;
    return run_bwd(p, dtype, reinterpret_cast<cudaStream_t>(stream));
}

sa_status longformer_attn_bwd_gproj(const void *Q, const void *K, const void *V, const void *Qg, const void *Kg,
                                    const void *Vg, const void *dO, void *dQ, void *dK, void *dV, void *dQg, void *dKg,
                                    void *dVg, int B, int H, int n, int d, int window, const int32_t *dilation,
                                    int causal, const int32_t *global_idx, int n_global, const uint8_t *key_mask,
                                    sa_dtype dtype, sa_stream_t stream) {
    if (dtype != SA_BF16 && dtype != SA_FP32) return SA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return SA_ERR_INVALID_ARG;
    const void *in[7] = {Q, K, V, Qg, Kg, Vg, dO};
    void *out[6] = {dQ, dK, dV, dQg, dKg, dVg};
    for (const void *t : in)
        if (!t || !aligned16(t)) return SA_ERR_INVALID_ARG;
    for (int a = 0; a < 6; ++a) {
        if (!out[a] || !aligned16(out[a])) return SA_ERR_INVALID_ARG;
        for (const void *t : in)
            if (out[a] == t) return SA_ERR_INVALID_ARG;
        for (int b = 0; b < a; ++b)
            if (out[a] == out[b]) return SA_ERR_INVALID_ARG;
    }
    sa_status s = longformer_args_ok(B, H, n, d, window, global_idx, n_global);
    if (s != SA_OK) return s;
    // the non-global rows against Q, K, V, then the global rows against Qg, Kg, Vg
    for (int set = 1; set <= 2; ++set) {
        sa::Problem p = {};
        p.kind = sa::kLongformer;
        p.Q = set == 1 ? Q : Qg;
        p.K = set == 1 ? K : Kg;
        p.V = set == 1 ? V : Vg;
        p.dO = dO;
        p.dQ = set == 1 ? dQ : dQg;
        p.dK = set == 1 ? dK : dKg;
        p.dV = set == 1 ? dV : dVg;
        p.B = B; p.H = H; p.n = n; p.d = d;
        p.window = window;
        p.global_idx = n_global > 0 ? global_idx : nullptr;
        p.n_global = n_global;
        p.dilation = dilation;
        p.causal = causal;
        p.key_mask = key_mask;
        p.row_set = set;
        s = run_bwd(p, dtype, reinterpret_cast<cudaStream_t>(stream));
        if (s != SA_OK) return s;
    }
    return SA_OK;
}

size_t sa_attn_bwd_workspace_bytes(int B, int H, int n, int d) {
    if (!size_ok(B, H, n, d)) return 0;
    return bwd_stats_bytes(B, H, n);
}

sa_status bigbird_attn_fwd_host(const void *Q, const void *K, const void *V, void *O, int B, int H, int n, int d,
                                int b, int g, int w, int r, const int32_t *rand_idx, const uint8_t *key_mask,
                                sa_dtype dtype, sa_stream_t stream) {
    if (dtype != SA_BF16 && dtype != SA_FP32) return SA_ERR_INVALID_ARG;
    if (!Q || !K || !V || !O || O == Q || O == K || O == V) return SA_ERR_INVALID_ARG;
    sa_status s = bigbird_args_ok(B, H, n, d, b, g, w, r, rand_idx);
    if (s != SA_OK) return s;
    sa::Problem p = {};
    p.kind = sa::kBigBird;
    p.Q = Q; p.K = K; p.V = V; p.O = O;
    p.B = B; p.H = H; p.n = n; p.d = d;
    p.b = b; p.g = g; p.w = w; p.r = r;
    p.rand_idx = r > 0 ? rand_idx : nullptr;
    p.key_mask = key_mask;
    return run_host(p, dtype, reinterpret_cast<cudaStream_t>(stream));
}

sa_status longformer_attn_fwd_host(const void *Q, const void *K, const void *V, void *O, int B, int H, int n, int d,
                                   int window, const int32_t *dilation, int causal, const int32_t *global_idx,
                                   int n_global, const uint8_t *key_mask, sa_dtype dtype, sa_stream_t stream) {
    if (dtype != SA_BF16 && dtype != SA_FP32) return SA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return SA_ERR_INVALID_ARG;
    if (!Q || !K || !V || !O || O == Q || O == K || O == V) return SA_ERR_INVALID_ARG;
    sa_status s = longformer_args_ok(B, H, n, d, window, global_idx, n_global);
    if (s != SA_OK) return s;
    sa::Problem p = {};
    p.kind = sa::kLongformer;
    p.Q = Q; p.K = K; p.V = V; p.O = O;
    p.B = B; p.H = H; p.n = n; p.d = d;
    p.window = window;
    p.global_idx = n_global > 0 ? global_idx : nullptr;
    p.n_global = n_global;
    p.dilation = dilation;
    p.causal = causal;
    p.key_mask = key_mask;
    return run_host(p, dtype, reinterpret_cast<cudaStream_t>(stream));
}

size_t sa_bigbird_workspace_bytes(int B, int H, int n, int d, int b, int g) {
    if (!size_ok(B, H, n, d) || (b != 64 && b != 128) || n % b != 0 || g < 0 || g > n / b) return 0;
    sa::Problem p = {};
    p.kind = sa::kBigBird;
    p.B = B; p.H = H; p.n = n; p.d = d; p.b = b; p.g = g; p.w = 1;
    return sa::tc_workspace_bytes(p, tc_config(nullptr));
}

size_t sa_longformer_workspace_bytes(int B, int H, int n, int d, int n_global) {
    if (!size_ok(B, H, n, d) || n_global < 0 || n_global > n) return 0;
    sa::Problem p = {};
    p.kind = sa::kLongformer;
    p.B = B; p.H = H; p.n = n; p.d = d; p.n_global = n_global;
    return sa::tc_workspace_bytes(p, tc_config(nullptr));
}

sa_status sa_set_workspace(void *dev_ptr, size_t bytes) {
    if ((reinterpret_cast<uintptr_t>(dev_ptr) & 255u) != 0) return SA_ERR_INVALID_ARG;
    if (!dev_ptr && bytes > 0) return SA_ERR_INVALID_ARG;
    int dev = 0;
    DeviceState *st = nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    sa_status s = current_device(&dev, &st);
    if (s != SA_OK) return s;
    st->user_ws = dev_ptr;
    st->user_ws_bytes = dev_ptr ? bytes : 0;
    st->user_ws_clean = st->user_ws_bytes;  // the caller hands it over zeroed
    return SA_OK;
}

sa_status sa_get_last_device_status(sa_stream_t stream) {
    int dev = 0;
    DeviceState *st = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        sa_status s = current_device(&dev, &st);
        if (s != SA_OK) return s;
    }
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return SA_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpy(&word, st->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return SA_ERR_CUDA;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpy(st->status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return SA_ERR_CUDA;
    }
    if (word & sa::kDevTimeout) {
        // An aborted kernel may leave scheduler or split-merge counters set:
        // zero the scratch so the next call starts clean.
        std::lock_guard<std::mutex> lock(g_mutex);
        if (st->ws && cudaMemset(st->ws, 0, st->ws_bytes) != cudaSuccess) return SA_ERR_CUDA;
        if (st->user_ws && cudaMemset(st->user_ws, 0, st->user_ws_bytes) != cudaSuccess) return SA_ERR_CUDA;
        st->ws_clean = st->ws_bytes;
        st->user_ws_clean = st->user_ws_bytes;
        if (cudaDeviceSynchronize() != cudaSuccess) return SA_ERR_CUDA;
        return SA_ERR_TIMEOUT;
    }
    if (word & sa::kDevBadIndex) return SA_ERR_BAD_INDEX;
    return SA_OK;
}

const char *sa_status_string(sa_status status) {
    switch (status) {
        case SA_OK: return "SA_OK";
        case SA_ERR_INVALID_ARG: return "SA_ERR_INVALID_ARG";
        case SA_ERR_UNSUPPORTED: return "SA_ERR_UNSUPPORTED";
        case SA_ERR_CUDA: return "SA_ERR_CUDA";
        case SA_ERR_TIMEOUT: return "SA_ERR_TIMEOUT";
        case SA_ERR_BAD_INDEX: return "SA_ERR_BAD_INDEX";
    }
    return "SA_ERR_UNKNOWN";
}

sa_status sa_set_option(int option, int64_t value) {
    switch (option) {
        case SA_OPT_FORCE_SIMT: g_force_simt = value != 0; return SA_OK;
        case SA_OPT_WAIT_LIMIT: g_wait_limit = value > 0 ? (long long)value : 2000000; return SA_OK;
        case SA_OPT_MAX_SPLITS: g_max_splits = value < 1 ? 1 : (value > 64 ? 64 : (int)value); return SA_OK;
        case SA_OPT_GRID_CTAS: g_grid_ctas = value < 0 ? 0 : (int)value; return SA_OK;
        case SA_OPT_CHUNK_KEYS: g_chunk_keys = value <= 0 ? 0 : (value > (1 << 20) ? (1 << 20) : (int)value); return SA_OK;
    }
    return SA_ERR_INVALID_ARG;
}

int sa_last_launch_count(void) { return g_last_launches; }

}  // extern "C"

// ---------------------------------------------------------------------------
// bigbird_attn_fwd_noalloc: the BigBird forward for callers that may not
// allocate device memory (see sparse_attn.h). Its scratch is the fixed array
// below instead of a cudaMalloc'ed region.
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[SA_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on each device. The array's host-side
// name is only a stand-in: a kernel must be given this address instead.
void *g_noalloc_addr[kMaxDevices];

// Looks the address up once per device, with that device current.
sa_status noalloc_scratch(int dev, void **out) {
    if (!g_noalloc_addr[dev]) {
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr) return SA_ERR_CUDA;
        g_noalloc_addr[dev] = addr;
    }
    *out = g_noalloc_addr[dev];
    return SA_OK;
}

}  // namespace

extern "C" sa_status bigbird_attn_fwd_noalloc(const void *Q, const void *K, const void *V, void *O, int B, int H,
                                              int n, int d, int b, int g, int w, int r, const int32_t *rand_idx,
                                              const uint8_t *key_mask, sa_stream_t stream) {
    sa_status s = check_tensors(Q, K, V, O);
    if (s != SA_OK) return s;
    s = bigbird_args_ok(B, H, n, d, b, g, w, r, rand_idx);
    if (s != SA_OK) return s;
    if (!aligned16(key_mask)) return SA_ERR_INVALID_ARG;
    sa::Problem p = {};
    p.kind = sa::kBigBird;
    p.Q = Q; p.K = K; p.V = V; p.O = O;
    p.B = B; p.H = H; p.n = n; p.d = d;
    p.b = b; p.g = g; p.w = w; p.r = r;
    p.rand_idx = r > 0 ? rand_idx : nullptr;
    p.key_mask = key_mask;
    // One configuration for the size check, the counter clear and the launch
    // (the split option is read once). The scratch need depends only on the
    // sizes and the split option, not on the grid size: reject oversize calls
    // before touching the device.
    sa::TcConfig cfg = tc_config(nullptr);
    const size_t need = sa::tc_workspace_bytes(p, cfg);
    if (need > SA_NOALLOC_SCRATCH_BYTES) return SA_ERR_UNSUPPORTED;

    int dev = 0;
    DeviceState *st = nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    s = current_device(&dev, &st);
    if (s != SA_OK) return s;
    if (st->cc_major != 10 || st->cc_minor != 3) return SA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    s = noalloc_scratch(dev, &scratch);
    if (s != SA_OK) return s;
    p.status = st->status;
    if (g_grid_ctas.load() <= 0) cfg.grid_ctas = st->num_sms;  // grid size only: the scratch need is unchanged
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const size_t zero_bytes = sa::tc_workspace_counter_bytes(p, cfg);
    if (cudaMemsetAsync(scratch, 0, zero_bytes, cs) != cudaSuccess) return SA_ERR_CUDA;
    int launches = 0;
    const cudaError_t e = sa::launch_tc(p, cfg, scratch, need, cs, &launches);
    if (e == cudaErrorNotSupported) return SA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return SA_ERR_CUDA;
    g_last_launches = launches;
    return SA_OK;
}

// ---------------------------------------------------------------------------
// sa_check_wait_expiry: the bounded-wait machinery of the tensor-core kernels,
// exercised without a fault. One warp waits, through the kernels' own wait
// helper, on an mbarrier that nothing ever arrives at; the wait gives up after
// the limit, raises the CTA's abort flag and latches SA_ERR_TIMEOUT in the
// device status word, and the kernel returns.
namespace {

__global__ void __launch_bounds__(32, 1) wait_expiry_kernel(unsigned *status, unsigned long long limit_ns) {
    using namespace sa::tcsync;
    __shared__ __align__(8) uint64_t never;  // phase 0 never completes: its one arrival never comes
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        sa::ptx::mbar_init(sa::ptx::smem_u32(&never), 1);
        abort_flag = 0;
        sa::ptx::fence_mbar_init();
    }
    __syncthreads();
    const Ctl ctl{&abort_flag, status, limit_ns};
    wait_warp(sa::ptx::smem_u32(&never), 0, ctl);
}

}  // namespace

extern "C" sa_status sa_check_wait_expiry(int64_t limit_us, sa_stream_t stream) {
    if (limit_us < 1 || limit_us > 1000000) return SA_ERR_INVALID_ARG;
    int dev = 0;
    DeviceState *st = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        const sa_status s = current_device(&dev, &st);
        if (s != SA_OK) return s;
        if (st->cc_major != 10 || st->cc_minor != 3) return SA_ERR_UNSUPPORTED;
    }
    wait_expiry_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        st->status, (unsigned long long)limit_us * 1000ull);
    if (cudaGetLastError() != cudaSuccess) return SA_ERR_CUDA;
    g_last_launches = 1;
    return SA_OK;
}
