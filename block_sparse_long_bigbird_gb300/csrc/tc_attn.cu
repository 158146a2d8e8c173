// BigBird-ITC host side of the tensor-core forward: geometry of the units
// (local 128-row tiles and split global tiles), scratch layout, launch.
#include "tc_kernel.cuh"
#include "tc_split.h"

namespace sa {
namespace {

Geometry bigbird_geometry(const Problem &p, const TcConfig &cfg) {
    Geometry G = {};
    G.B = p.B;
    G.H = p.H;
    G.n = p.n;
    G.b = p.b;
    G.nb = p.n / p.b;
    G.g = p.g;
    G.w = p.w;
    G.r = p.r;
    G.half = p.w / 2;
    G.tiles = (p.n + kBM - 1) / kBM;
    G.gtiles = (p.g * p.b + kBM - 1) / kBM;
    if (G.gtiles > G.tiles) G.gtiles = G.tiles;
    const int kb = keys_per_step(p.d);
    G.steps_full = (p.n + kb - 1) / kb;
    {
        // a local tile walks the union of its query blocks' lists
        const int qb = kBM / p.b > 1 ? kBM / p.b : 1;
        long long blocks = (long long)p.g + (p.w - 1 + qb) + (long long)qb * p.r;
        if (blocks > G.nb) blocks = G.nb;
        const long long per_tile = (blocks * p.b + kb - 1) / kb;
        const int nt = p.d == 64 ? Cfg<64>::NT : Cfg<128>::NT;
        choose_splits(G, (long long)p.B * p.H * (G.tiles - G.gtiles) * per_tile, kb, nt, cfg.chunk_keys,
                      cfg.max_splits);
    }
    const long long BH = (long long)p.B * p.H;
    G.n_split_units = (int)(BH * G.gtiles * G.splits);
    G.total_units = G.n_split_units + (int)(BH * (G.tiles - G.gtiles));
    G.scale_log2 = 1.4426950408889634f / sqrtf((float)p.d);
    G.wait_ns = (unsigned long long)cfg.wait_limit * 1000ull;
    return G;
}

struct WsLayout {
    size_t row_cnt, part_o, part_ml, total;
};

WsLayout ws_layout(const Geometry &G, int d) {
    WsLayout L;
    const size_t tiles = (size_t)G.B * G.H * G.gtiles;
    size_t off = 256;  // scheduler counters
    L.row_cnt = off;
    off += (tiles * kBM * sizeof(unsigned) + 255) & ~(size_t)255;
    if (G.splits > 1) {
        L.part_o = off;
        off += (tiles * G.splits * kBM * d * sizeof(float) + 255) & ~(size_t)255;
        L.part_ml = off;
        off += (tiles * G.splits * kBM * sizeof(float2) + 255) & ~(size_t)255;
    } else {
        L.part_o = L.part_ml = 0;
    }
    L.total = off;
    return L;
}

template <int D>
cudaError_t launch_bigbird(const Problem &p, const TcConfig &cfg, void *ws, size_t ws_bytes, cudaStream_t stream) {
    Params prm = {};
    prm.geo = bigbird_geometry(p, cfg);
    const WsLayout L = ws_layout(prm.geo, D);
    if (!ws || ws_bytes < L.total) return cudaErrorInvalidValue;
    uint8_t *base = static_cast<uint8_t *>(ws);
    prm.ws.counters = reinterpret_cast<unsigned *>(base);
    prm.ws.row_cnt = reinterpret_cast<unsigned *>(base + L.row_cnt);
    prm.ws.n_row_cnt = (size_t)prm.geo.B * prm.geo.H * prm.geo.gtiles * kBM;
    prm.ws.part_o = L.part_o ? reinterpret_cast<float *>(base + L.part_o) : nullptr;
    prm.ws.part_ml = L.part_ml ? reinterpret_cast<float2 *>(base + L.part_ml) : nullptr;
    prm.rand_idx = p.rand_idx;
    prm.key_mask = p.key_mask;
    prm.O = static_cast<__nv_bfloat16 *>(p.O);
    prm.status = p.status;
    const int BH = p.B * p.H;
    CUtensorMap mq, mk, mv;
    if (!make_qkv_map(&mq, p.Q, BH, p.n, D) || !make_qkv_map(&mk, p.K, BH, p.n, D) ||
        !make_qkv_map(&mv, p.V, BH, p.n, D))
        return cudaErrorInvalidValue;
    auto kern = p.key_mask ? sparse_tc_fwd<D, true, false> : sparse_tc_fwd<D, false, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::ALLOC_BYTES);
    if (e != cudaSuccess) return e;
    int grid = cfg.grid_ctas;
    if (grid > prm.geo.total_units) grid = prm.geo.total_units;
    if (grid < 1) grid = 1;
    kern<<<grid, Cfg<D>::THREADS, Cfg<D>::ALLOC_BYTES, stream>>>(mq, mk, mv, mk, mv, mq, prm);
    return cudaGetLastError();
}

}  // namespace

size_t tc_workspace_bytes(const Problem &p, const TcConfig &cfg) {
    if (p.kind != kBigBird) return tc_longformer_workspace_bytes(p, cfg);
    return ws_layout(bigbird_geometry(p, cfg), p.d).total;
}

size_t tc_workspace_counter_bytes(const Problem &p, const TcConfig &cfg) {
    if (p.kind != kBigBird) return tc_longformer_counter_bytes(p, cfg);
    const WsLayout L = ws_layout(bigbird_geometry(p, cfg), p.d);
    return L.part_o ? L.part_o : L.total;
}

cudaError_t launch_tc(const Problem &p, const TcConfig &cfg, void *ws, size_t ws_bytes, cudaStream_t stream,
                      int *launches) {
    *launches = 0;
    if (p.kind != kBigBird) return launch_tc_longformer(p, cfg, ws, ws_bytes, stream, launches);
    cudaError_t e = (p.d == 64) ? launch_bigbird<64>(p, cfg, ws, ws_bytes, stream)
                                : launch_bigbird<128>(p, cfg, ws, ws_bytes, stream);
    if (e == cudaSuccess) *launches = 1;
    return e;
}

}  // namespace sa
