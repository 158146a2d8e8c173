// Longformer host side of the tensor-core forward ("Longformer", Sec. 3.1:
// sliding window of w/2 tokens per side plus symmetric global attention).
// A one-CTA preparation kernel turns the global list into per-block bit masks
// and a compact list of the 64-key blocks holding global keys; the persistent
// kernel then runs the global-row units (split-KV sweeps over all keys) and
// one band unit per 128-row tile.
#include "tc_kernel.cuh"
#include "tc_split.h"

namespace sa {
namespace {

constexpr int kPrepThreads = 1024;

// For every 64-key block kb: gbits[kb] = bits of its global keys, gpre[kb] =
// number of blocks before kb holding a global key (gpre[nkb] = their total),
// glist = those blocks in increasing order. Entries of gidx out of [0, n) or
// not above their predecessor are skipped and latch SA_ERR_BAD_INDEX. Every
// output word is rewritten, so the scratch needs no clearing between calls.
__global__ void __launch_bounds__(kPrepThreads) longformer_prep(const int32_t *gidx, int ng, int n, int nkb,
                                                                unsigned long long *gbits, int *gpre, int *glist,
                                                                unsigned *status) {
    __shared__ int warp_off[kPrepThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    for (int i = tid; i < nkb; i += kPrepThreads) gbits[i] = 0ull;
    __syncthreads();
    bool bad = false;
    for (int t = tid; t < ng; t += kPrepThreads) {
        const int v = global_row(gidx, ng, n, t);
        if (v >= n) {
            bad = true;
            continue;
        }
        atomicOr(gbits + (v >> 6), 1ull << (v & 63));
    }
    if (__syncthreads_or(bad) && tid == 0) atomicOr(status, kDevBadIndex);
    // exclusive prefix count of non-empty blocks; thread tid owns blocks [lo, hi)
    const int seg = (nkb + kPrepThreads - 1) / kPrepThreads;
    const int lo = min(nkb, tid * seg), hi = min(nkb, lo + seg);
    int cnt = 0;
    for (int i = lo; i < hi; ++i) cnt += __ldcg(gbits + i) != 0ull;
    int inc = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += v;
    }
    if (lane == 31) warp_off[wid] = inc;
    __syncthreads();
    if (wid == 0) {
        const int w = warp_off[lane];
        int winc = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(kFull, winc, o);
            if (lane >= o) winc += v;
        }
        warp_off[lane] = winc - w;
    }
    __syncthreads();
    int base = warp_off[wid] + inc - cnt;
    for (int i = lo; i < hi; ++i) {
        gpre[i] = base;
        if (__ldcg(gbits + i) != 0ull) glist[base++] = i;
    }
    if (tid == kPrepThreads - 1) gpre[nkb] = base;
}

// Residue-class gather of the dilated heads ("Longformer", Sec. 3.1: a dilated
// window of stride s = dilation + 1 joins only tokens of one residue class
// mod s). For each (batch, head) whose dilation is in range, nonzero and
// whose stride divides n, row m of class c (token c + s m) is copied to
// position c (n / s) + m of Q, K and V's copies; the attention kernel then runs
// those heads as plain windows on the copies. Other heads are not touched.
constexpr int kGatherThreads = 256;
__global__ void __launch_bounds__(kGatherThreads) longformer_class_gather(const uint4 *Q, const uint4 *K,
                                                                          const uint4 *V, uint4 *Qp, uint4 *Kp,
                                                                          uint4 *Vp, const int32_t *dilation, int BH,
                                                                          int H, int n, int cpr) {
    for (int bh = blockIdx.y; bh < BH; bh += gridDim.y) {
        const int dil = __ldg(dilation + bh % H);
        if (dil <= 0 || dil > kMaxDilation) continue;  // out-of-range values are latched by the attention kernel
        const int s = dil + 1;
        if (n % s != 0) continue;
        const int M = n / s;
        const size_t head = (size_t)bh * n * cpr;
        const long long total = (long long)n * cpr;
        for (long long i = (long long)blockIdx.x * kGatherThreads + threadIdx.x; i < total;
             i += (long long)gridDim.x * kGatherThreads) {
            const int pos = (int)(i / cpr), cq = (int)(i - (long long)pos * cpr);
            const int c = pos / M;
            const size_t src = head + ((size_t)(c + s * (pos - c * M))) * cpr + cq;
            const size_t dst = head + (size_t)pos * cpr + cq;
            Qp[dst] = __ldg(Q + src);
            Kp[dst] = __ldg(K + src);
            Vp[dst] = __ldg(V + src);
        }
    }
}

Geometry longformer_geometry(const Problem &p, const TcConfig &cfg) {
    Geometry G = {};
    G.B = p.B;
    G.H = p.H;
    G.n = p.n;
    G.b = kBM;
    G.half = p.window / 2 < p.n ? p.window / 2 : p.n;  // |i - k| < n always: a wider window changes nothing
    G.tiles = (p.n + kBM - 1) / kBM;
    G.ng = p.n_global;
    G.causal = p.causal;
    G.gtiles = (p.n_global + kBM - 1) / kBM;
    G.nkb = (p.n + 63) / 64;
    const int kb = keys_per_step(p.d);
    G.steps_full = (p.n + kb - 1) / kb;
    {
        // a band tile: its window around 128 rows, plus a step of global keys
        long long keys = 2LL * G.half + kBM;
        if (keys > p.n) keys = p.n;
        const long long per_tile = (keys + kb - 1) / kb + (p.n_global > 0 ? 1 : 0);
        const int nt = p.d == 64 ? Cfg<64>::NT : Cfg<128>::NT;
        choose_splits(G, (long long)p.B * p.H * G.tiles * per_tile, kb, nt, cfg.chunk_keys, cfg.max_splits);
    }
    const long long BH = (long long)p.B * p.H;
    G.n_split_units = (int)(BH * G.gtiles * G.splits);
    G.total_units = G.n_split_units + (int)(BH * G.tiles);
    G.scale_log2 = 1.4426950408889634f / sqrtf((float)p.d);
    G.wait_ns = (unsigned long long)cfg.wait_limit * 1000ull;
    return G;
}

// Scratch: counters and per-row merge counters (zero at entry, left zero),
// then split partials and the prep outputs (rewritten by every call).
struct LfLayout {
    size_t row_cnt, part_o, part_ml, gbits, gpre, glist, perm, total;
};

LfLayout lf_layout(const Geometry &G, int d, bool class_perm) {
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    LfLayout L;
    const size_t tiles = (size_t)G.B * G.H * G.gtiles;
    size_t off = 256;
    L.row_cnt = off;
    off += up(tiles * kBM * sizeof(unsigned));
    if (G.splits > 1 && tiles > 0) {
        L.part_o = off;
        off += up(tiles * G.splits * kBM * d * sizeof(float));
        L.part_ml = off;
        off += up(tiles * G.splits * kBM * sizeof(float2));
    } else {
        L.part_o = L.part_ml = 0;
    }
    L.gbits = off;
    off += up((size_t)G.nkb * sizeof(unsigned long long));
    L.gpre = off;
    off += up(((size_t)G.nkb + 1) * sizeof(int));
    L.glist = off;
    off += up((size_t)G.nkb * sizeof(int));
    L.perm = 0;
    if (class_perm) {  // residue-class copies of Q, K, V (rewritten by every call)
        L.perm = off;
        off += 3 * up((size_t)G.B * G.H * G.n * d * 2);
    }
    L.total = off;
    return L;
}

template <int D>
cudaError_t launch_longformer(const Problem &p, const TcConfig &cfg, void *ws, size_t ws_bytes, cudaStream_t stream,
                              int *launches) {
    Params prm = {};
    prm.geo = longformer_geometry(p, cfg);
    const LfLayout L = lf_layout(prm.geo, D, p.class_perm != 0);
    if (!ws || ws_bytes < L.total) return cudaErrorInvalidValue;
    uint8_t *base = static_cast<uint8_t *>(ws);
    prm.ws.counters = reinterpret_cast<unsigned *>(base);
    prm.ws.row_cnt = reinterpret_cast<unsigned *>(base + L.row_cnt);
    prm.ws.n_row_cnt = (size_t)prm.geo.B * prm.geo.H * prm.geo.gtiles * kBM;
    prm.ws.part_o = L.part_o ? reinterpret_cast<float *>(base + L.part_o) : nullptr;
    prm.ws.part_ml = L.part_ml ? reinterpret_cast<float2 *>(base + L.part_ml) : nullptr;
    prm.key_mask = p.key_mask;
    prm.O = static_cast<__nv_bfloat16 *>(p.O);
    prm.status = p.status;
    prm.Q = static_cast<const __nv_bfloat16 *>(p.Q);
    // separate projections for global attention ("Longformer", Sec. 3.1): the
    // global-row units take their queries, keys and values from Qg, Kg, Vg
    const bool sep = p.Qg != nullptr;
    prm.Qg = static_cast<const __nv_bfloat16 *>(sep ? p.Qg : p.Q);
    prm.gidx = p.global_idx;
    prm.dilation = p.dilation;
    unsigned long long *gbits = reinterpret_cast<unsigned long long *>(base + L.gbits);
    int *gpre = reinterpret_cast<int *>(base + L.gpre);
    int *glist = reinterpret_cast<int *>(base + L.glist);
    prm.gbits = gbits;
    prm.gpre = gpre;
    prm.glist = glist;
    const int BH = p.B * p.H;
    // residue-class copies (no global tokens, so the global-row key and value
    // maps are free to point at them)
    const bool cls = p.class_perm && p.dilation && prm.geo.ng == 0 && !sep && !p.key_mask;
    const size_t tensor_bytes = (size_t)BH * p.n * D * 2;
    const size_t cstride = (tensor_bytes + 255) & ~(size_t)255;
    void *qp = cls ? base + L.perm : nullptr;
    void *kp = cls ? base + L.perm + cstride : nullptr;
    void *vp = cls ? base + L.perm + 2 * cstride : nullptr;
    prm.class_perm = cls ? 1 : 0;
    CUtensorMap mq, mk, mv, mkg, mvg, mqp;
    if (!make_qkv_map(&mq, p.Q, BH, p.n, D) || !make_qkv_map(&mk, p.K, BH, p.n, D) ||
        !make_qkv_map(&mv, p.V, BH, p.n, D) ||
        !make_qkv_map(&mkg, cls ? kp : (sep ? p.Kg : p.K), BH, p.n, D) ||
        !make_qkv_map(&mvg, cls ? vp : (sep ? p.Vg : p.V), BH, p.n, D) ||
        !make_qkv_map(&mqp, cls ? qp : p.Q, BH, p.n, D))
        return cudaErrorInvalidValue;
    auto kern = p.key_mask ? sparse_tc_fwd<D, true, true> : sparse_tc_fwd<D, false, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::ALLOC_BYTES);
    if (e != cudaSuccess) return e;
    if (prm.geo.ng > 0) {
        longformer_prep<<<1, kPrepThreads, 0, stream>>>(p.global_idx, prm.geo.ng, p.n, prm.geo.nkb, gbits, gpre,
                                                        glist, p.status);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        ++*launches;
    }
    if (cls) {
        const int cpr = D / 8;  // 16-byte chunks per row
        long long chunks = ((long long)p.n * cpr + kGatherThreads - 1) / kGatherThreads;
        const dim3 ggrid((unsigned)(chunks < 64 ? chunks : 64), (unsigned)(BH < 65535 ? BH : 65535));
        longformer_class_gather<<<ggrid, kGatherThreads, 0, stream>>>(
            static_cast<const uint4 *>(p.Q), static_cast<const uint4 *>(p.K), static_cast<const uint4 *>(p.V),
            static_cast<uint4 *>(qp), static_cast<uint4 *>(kp), static_cast<uint4 *>(vp), p.dilation, BH, p.H, p.n,
            cpr);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        ++*launches;
    }
    int grid = cfg.grid_ctas;
    if (grid > prm.geo.total_units) grid = prm.geo.total_units;
    if (grid < 1) grid = 1;
    kern<<<grid, Cfg<D>::THREADS, Cfg<D>::ALLOC_BYTES, stream>>>(mq, mk, mv, mkg, mvg, mqp, prm);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    ++*launches;
    return cudaSuccess;
}

}  // namespace

size_t tc_longformer_workspace_bytes(const Problem &p, const TcConfig &cfg) {
    return lf_layout(longformer_geometry(p, cfg), p.d, p.class_perm != 0).total;
}

size_t tc_longformer_counter_bytes(const Problem &p, const TcConfig &cfg) {
    const LfLayout L = lf_layout(longformer_geometry(p, cfg), p.d, p.class_perm != 0);
    return L.part_o ? L.part_o : L.gbits;
}

cudaError_t launch_tc_longformer(const Problem &p, const TcConfig &cfg, void *ws, size_t ws_bytes,
                                 cudaStream_t stream, int *launches) {
    *launches = 0;
    return (p.d == 64) ? launch_longformer<64>(p, cfg, ws, ws_bytes, stream, launches)
                       : launch_longformer<128>(p, cfg, ws, ws_bytes, stream, launches);
}

}  // namespace sa
