// Exact SIMT sparse-attention backward (fp32 arithmetic, no tensor cores).
//
// The gradient of the forward O = softmax_N(i)(Q K^T / sqrt(d)) V for an
// upstream gradient dO. The pages train through this attention ("Big Bird",
// App. E.1, MLM pretraining; "Longformer", Sec. 5, pretraining with gradient
// updates) without printing the backward; it is the exact derivative:
//
//     P_ij  = 2^(s_ij - lse_i),  s_ij = log2(e) Q_i . K_j / sqrt(d) on N(i), else P_ij = 0
//     D_i   = sum_j P_ij (dO_i . V_j)     (= dO_i . O_i for the exact O)
//     dS_ij = P_ij (dO_i . V_j - D_i)
//     dQ_i  = sum_j dS_ij K_j / sqrt(d)
//     dK_j  = sum_i dS_ij Q_i / sqrt(d)
//     dV_j  = sum_i P_ij dO_i
//
// Two launches, no atomics, every sum in a fixed order (deterministic):
//  * row pass (one CTA per query tile): one online pass over the row's keys
//    gives lse_i and D_i (D is accumulated with the same rescaling as the
//    softmax denominator, so it never depends on how O was rounded), a second
//    pass sums dQ_i; lse and D go to scratch;
//  * key pass (one CTA per key tile): walks the query rows whose
//    neighbourhood holds the tile's keys (the transposed pattern) and sums
//    dK_j and dV_j.
// This is the fp32 path and the exact cross-check of the bf16 tensor-core
// backward.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "internal.h"
#include "simt_common.cuh"

namespace sa {
namespace {

using simt::kFull;
using simt::lower_bound_i32;
using simt::store_val;
using simt::to_f32;
using simt::warp_max;
using simt::warp_sum;

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 64;  // keys (row pass) or query rows (key pass) staged per step
constexpr float kLog2e = 1.4426950408889634f;

// Bits of the sorted global positions that fall in [c0, c0 + 64) -> words[0..1].
// Called by one warp.
__device__ __forceinline__ void global_bits_of_chunk(const int32_t *gidx, int ng, int c0, unsigned *words) {
    const int lane = threadIdx.x & 31;
    if (ng <= 0) return;
    const int pos = lower_bound_i32(gidx, ng, c0);
    for (int t = pos + lane; t < ng && t < pos + kChunk; t += 32) {
        const int gpos = gidx[t];
        if (gpos >= c0 && gpos < c0 + kChunk) atomicOr(&words[(gpos - c0) >> 5], 1u << ((gpos - c0) & 31));
    }
}

// Longformer per-head window geometry ("Longformer", Sec. 3.1: dilated window
// of stride dilation + 1 reaching window / 2 positions on each side).
struct LfGeom {
    int stride, reach;
    bool causal;
};
__device__ __forceinline__ LfGeom lf_geom(const Problem &p, int h, bool latch) {
    int dil = p.dilation ? p.dilation[h] : 0;
    if (dil < 0 || dil > kMaxDilation) {
        if (latch) atomicOr(p.status, kDevBadIndex);
        dil = 0;
    }
    LfGeom g;
    g.stride = dil + 1;
    g.reach = (int)min((long long)(p.window / 2) * g.stride, (long long)p.n);
    g.causal = p.causal != 0;
    return g;
}
__device__ __forceinline__ bool lf_allowed(const LfGeom &g, int i, int j, bool iglob, bool jglob) {
    if (g.causal && j > i) return false;
    const int dk = i - j;
    return iglob || jglob || (abs(dk) <= g.reach && dk % g.stride == 0);
}

// Validates the global list once per launch and marks the 64-position chunks
// that hold a global position; sets tile_bits[0..1] for the positions in
// [t0, t0 + 64).
__device__ void lf_mark_globals(const Problem &p, int t0, unsigned *bmap, unsigned *tile_bits) {
    const int32_t *gidx = p.global_idx;
    for (int t = threadIdx.x; t < p.n_global; t += kThreads) {
        const int gpos = gidx[t];
        if (gpos < 0 || gpos >= p.n || (t > 0 && gidx[t - 1] >= gpos)) {
            if (blockIdx.x == 0 && blockIdx.y == 0) atomicOr(p.status, kDevBadIndex);
            continue;
        }
        atomicOr(&bmap[(gpos / kChunk) >> 5], 1u << ((gpos / kChunk) & 31));
        if (gpos >= t0 && gpos < t0 + kChunk) atomicOr(&tile_bits[(gpos - t0) >> 5], 1u << ((gpos - t0) & 31));
    }
}

__device__ __forceinline__ void mark_range(unsigned *bmap, int lo, int hi) {
    for (int c = lo + threadIdx.x; c <= hi; c += kThreads) atomicOr(&bmap[c >> 5], 1u << (c & 31));
}

// Loads rows [r0, r0 + rows) of one head as fp32 into dst (row stride `ld`
// floats); rows at or past n are zero.
template <typename T, int D>
__device__ void load_rows(const T *src, int r0, int rows, int n, float *dst, int ld) {
    for (int idx = threadIdx.x; idx < rows * D; idx += kThreads) {
        const int rr = idx / D, c = idx - rr * D;
        const int i = r0 + rr;
        dst[rr * ld + c] = (i < n) ? to_f32(src[(size_t)i * D + c]) : 0.f;
    }
}

template <int D>
__device__ __forceinline__ float dot_rows(const float *a, const float *b) {
    float s = 0.f;
#pragma unroll
    for (int c = 0; c < D; c += 4) {
        const float4 x = *reinterpret_cast<const float4 *>(a + c);
        const float4 y = *reinterpret_cast<const float4 *>(b + c);
        s = fmaf(x.x, y.x, s);
        s = fmaf(x.y, y.y, s);
        s = fmaf(x.z, y.z, s);
        s = fmaf(x.w, y.w, s);
    }
    return s;
}

// ======================================================================= row pass
// Shared memory (floats): Q tile [BQ][D], dO tile [BQ][D], K and V chunks
// [64][D + 4] (padded rows: conflict-free per-lane float4 reads), misc words,
// then the bitmap of key blocks (BigBird: blocks of b keys; Longformer: 64-key
// chunks).
template <int D, int BQ>
struct RowLayout {
    static constexpr int kS = D + 4;
    static constexpr int q_off = 0;
    static constexpr int do_off = q_off + BQ * D;
    static constexpr int k_off = do_off + BQ * D;
    static constexpr int v_off = k_off + kChunk * kS;
    static constexpr int misc_off = v_off + kChunk * kS;
    static constexpr int misc_words = 32;  // [0..1] tile globals, [2..3] chunk globals, bytes from [4]: key validity
    static constexpr int map_off = misc_off + misc_words;
};

template <typename T, int D, int BQ, bool LF>
__global__ void __launch_bounds__(kThreads) bwd_rows_kernel(Problem p) {
    using L = RowLayout<D, BQ>;
    constexpr int R = BQ / kWarps;  // rows per warp
    constexpr int DL = D / 32;
    extern __shared__ float sm[];
    const int tile = blockIdx.x;
    const int bh = blockIdx.y;
    const int beta = bh / p.H, h = bh - beta * p.H;
    const int n = p.n;
    const int i0 = tile * BQ;
    const size_t head_off = (size_t)bh * n * D;
    const T *Qh = static_cast<const T *>(p.Q) + head_off;
    const T *Kh = static_cast<const T *>(p.K) + head_off;
    const T *Vh = static_cast<const T *>(p.V) + head_off;
    const T *dOh = static_cast<const T *>(p.dO) + head_off;
    T *dQh = static_cast<T *>(p.dQ) + head_off;
    const size_t sst = (size_t)stats_stride(n);
    float *lse_out = p.row_stats + (size_t)bh * sst;
    float *dl_out = p.row_stats + (size_t)p.B * p.H * sst + (size_t)bh * sst;
    const uint8_t *km = p.key_mask ? p.key_mask + (size_t)beta * n : nullptr;

    unsigned *misc = reinterpret_cast<unsigned *>(sm + L::misc_off);
    unsigned *bmap = reinterpret_cast<unsigned *>(sm + L::map_off);
    const int blk = LF ? kChunk : p.b;  // keys per bitmap bit
    const int nblk = (n + blk - 1) / blk;
    const int words = (nblk + 31) / 32;
    for (int t = threadIdx.x; t < words; t += kThreads) bmap[t] = 0u;
    if (threadIdx.x < 4) misc[threadIdx.x] = 0u;
    __syncthreads();

    LfGeom geo = {1, 0, false};
    if (LF) {
        geo = lf_geom(p, h, tile == 0 && threadIdx.x == 0);
        lf_mark_globals(p, i0, bmap, misc);
        __syncthreads();
        const bool tile_has_global = (misc[0] | misc[1]) != 0u;
        const int lo = tile_has_global ? 0 : max(0, i0 - geo.reach) / kChunk;
        const int hi = geo.causal ? min(n - 1, i0 + BQ - 1) / kChunk
                                  : (tile_has_global ? nblk - 1 : min(n - 1, i0 + BQ - 1 + geo.reach) / kChunk);
        mark_range(bmap, lo, hi);
    } else {
        const int qb = tile;
        if (qb < p.g) {
            mark_range(bmap, 0, nblk - 1);
        } else {
            const int half = p.w / 2;
            mark_range(bmap, 0, p.g - 1);
            mark_range(bmap, max(0, qb - half), min(nblk - 1, qb + half));
            if (p.rand_idx) {
                const int32_t *rr = p.rand_idx + ((size_t)h * nblk + qb) * p.r;
                for (int t = threadIdx.x; t < p.r; t += kThreads) {
                    const int kb = rr[t];
                    if (kb == -1) continue;
                    if (kb < -1 || kb >= nblk) { atomicOr(p.status, kDevBadIndex); continue; }
                    atomicOr(&bmap[kb >> 5], 1u << (kb & 31));
                }
            }
        }
    }
    float *Qs = sm + L::q_off;
    float *dOs = sm + L::do_off;
    float *Ks = sm + L::k_off;
    float *Vs = sm + L::v_off;
    load_rows<T, D>(Qh, i0, BQ, n, Qs, D);
    load_rows<T, D>(dOh, i0, BQ, n, dOs, D);
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = warp * R;
    const float scale_log2 = kLog2e / sqrtf((float)D);
    bool qvalid[R], qglob[R];
    float m[R], l[R], u[R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        const int il = row0 + rr, i = i0 + il;
        qvalid[rr] = (i < n) && (km ? (km[i] != 0) : true);
        qglob[rr] = LF ? (((misc[il >> 5] >> (il & 31)) & 1u) != 0u) : false;
        if (LF && p.row_set != 0 && qglob[rr] != (p.row_set == 2)) qvalid[rr] = false;  // row outside the set
        m[rr] = -CUDART_INF_F;
        l[rr] = 0.f;
        u[rr] = 0.f;
    }
    __syncthreads();
    uint8_t *kvalid = reinterpret_cast<uint8_t *>(misc + 4);
    const int32_t *gidx = p.global_idx;

    // Stages keys [k0, k0 + 64) (K and V), their validity and, for
    // Longformer, their global bits (misc[2..3]).
    auto stage = [&](int k0) {
        load_rows<T, D>(Kh, k0, kChunk, n, Ks, L::kS);
        load_rows<T, D>(Vh, k0, kChunk, n, Vs, L::kS);
        if (threadIdx.x < 2) misc[2 + threadIdx.x] = 0u;
        if (threadIdx.x < kChunk) {
            const int k = k0 + threadIdx.x;
            kvalid[threadIdx.x] = (k < n) && (km ? (km[k] != 0) : true);
        }
        __syncthreads();
        if (LF && threadIdx.x < 32) global_bits_of_chunk(gidx, p.n_global, k0, misc + 2);
        __syncthreads();
    };
    auto allowed = [&](int rr, int k0, int kl) -> bool {
        if (!qvalid[rr] || !kvalid[kl]) return false;
        if (!LF) return true;
        const bool kg = ((misc[2 + (kl >> 5)] >> (kl & 31)) & 1u) != 0u;
        return lf_allowed(geo, i0 + row0 + rr, k0 + kl, qglob[rr], kg);
    };

    // ---- pass 1: row statistics in the log2 domain: running maximum m,
    // l = sum_j 2^(s_ij - m) and u = sum_j 2^(s_ij - m) (dO_i . V_j), both
    // rescaled whenever m grows; then lse = m + log2(l) and D = u / l.
    for (int wd = 0; wd < words; ++wd) {
        unsigned bits = bmap[wd];
        while (bits) {
            const int kb = wd * 32 + __ffs(bits) - 1;
            bits &= bits - 1;
            for (int k0 = kb * blk; k0 < min(n, (kb + 1) * blk); k0 += kChunk) {
                stage(k0);
#pragma unroll 1
                for (int grp = 0; grp < 2; ++grp) {
                    const int kl = grp * 32 + lane;
#pragma unroll 1
                    for (int rr = 0; rr < R; ++rr) {
                        const bool ok = allowed(rr, k0, kl);
                        float sl = -CUDART_INF_F, dp = 0.f;
                        if (ok) {
                            sl = dot_rows<D>(Qs + (row0 + rr) * D, Ks + kl * L::kS) * scale_log2;
                            dp = dot_rows<D>(dOs + (row0 + rr) * D, Vs + kl * L::kS);
                        }
                        const float mnew = fmaxf(m[rr], warp_max(sl));
                        if (mnew == -CUDART_INF_F) continue;
                        const float alpha = exp2f(m[rr] - mnew);
                        const float e = exp2f(sl - mnew);
                        l[rr] = l[rr] * alpha + warp_sum(e);
                        u[rr] = u[rr] * alpha + warp_sum(e * dp);
                        m[rr] = mnew;
                    }
                }
                __syncthreads();
            }
        }
    }
    // lse_i (+inf for a row without keys, so that every P_ij is 0) and D_i.
    float lse[R], dl[R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        const int i = i0 + row0 + rr;
        lse[rr] = l[rr] > 0.f ? m[rr] + log2f(l[rr]) : CUDART_INF_F;
        dl[rr] = l[rr] > 0.f ? u[rr] / l[rr] : 0.f;
        if (lane == 0 && i < n) {
            lse_out[i] = lse[rr];
            dl_out[i] = dl[rr];
        }
    }

    // ---- pass 2: dQ_i = sum_j P_ij (dO_i . V_j - D_i) K_j / sqrt(d)
    float acc[R][DL];
#pragma unroll
    for (int rr = 0; rr < R; ++rr)
#pragma unroll
        for (int j = 0; j < DL; ++j) acc[rr][j] = 0.f;
    for (int wd = 0; wd < words; ++wd) {
        unsigned bits = bmap[wd];
        while (bits) {
            const int kb = wd * 32 + __ffs(bits) - 1;
            bits &= bits - 1;
            for (int k0 = kb * blk; k0 < min(n, (kb + 1) * blk); k0 += kChunk) {
                stage(k0);
#pragma unroll 1
                for (int grp = 0; grp < 2; ++grp) {
                    const int kl = grp * 32 + lane;
#pragma unroll 1
                    for (int rr = 0; rr < R; ++rr) {
                        float ds = 0.f;
                        if (allowed(rr, k0, kl)) {
                            const float s = dot_rows<D>(Qs + (row0 + rr) * D, Ks + kl * L::kS);
                            const float dp = dot_rows<D>(dOs + (row0 + rr) * D, Vs + kl * L::kS);
                            const float pr = exp2f(s * scale_log2 - lse[rr]);
                            ds = pr * (dp - dl[rr]);
                        }
                        if (!__any_sync(kFull, ds != 0.f)) continue;
#pragma unroll 4
                        for (int kk = 0; kk < 32; ++kk) {
                            const float dsk = __shfl_sync(kFull, ds, kk);
                            const float *krow = Ks + (grp * 32 + kk) * L::kS + lane * DL;
#pragma unroll
                            for (int j = 0; j < DL; ++j) acc[rr][j] = fmaf(dsk, krow[j], acc[rr][j]);
                        }
                    }
                }
                __syncthreads();
            }
        }
    }
    const float scale = 1.f / sqrtf((float)D);
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        const int i = i0 + row0 + rr;
        if (i >= n) continue;
#pragma unroll
        for (int j = 0; j < DL; ++j) store_val(dQh + (size_t)i * D + lane * DL + j, acc[rr][j] * scale);
    }
}

// ======================================================================= key pass
// Shared memory (floats): K and V tiles [BK][D], Q and dO row chunks
// [64][D + 4], lse and D of the chunk's rows, misc words, then the bitmap of
// query blocks (BigBird: blocks of b rows; Longformer: 64-row chunks).
template <int D, int BK>
struct ColLayout {
    static constexpr int kS = D + 4;
    static constexpr int k_off = 0;
    static constexpr int v_off = k_off + BK * D;
    static constexpr int q_off = v_off + BK * D;
    static constexpr int do_off = q_off + kChunk * kS;
    static constexpr int lse_off = do_off + kChunk * kS;
    static constexpr int dl_off = lse_off + kChunk;
    static constexpr int misc_off = dl_off + kChunk;
    static constexpr int misc_words = 32;  // [0..1] tile globals, [2..3] chunk globals, bytes from [4]: row validity
    static constexpr int map_off = misc_off + misc_words;
};

template <typename T, int D, int BK, bool LF>
__global__ void __launch_bounds__(kThreads) bwd_cols_kernel(Problem p) {
    using L = ColLayout<D, BK>;
    constexpr int R = BK / kWarps;  // keys per warp
    constexpr int DL = D / 32;
    extern __shared__ float sm[];
    const int tile = blockIdx.x;
    const int bh = blockIdx.y;
    const int beta = bh / p.H, h = bh - beta * p.H;
    const int n = p.n;
    const int j0 = tile * BK;
    const size_t head_off = (size_t)bh * n * D;
    const T *Qh = static_cast<const T *>(p.Q) + head_off;
    const T *Kh = static_cast<const T *>(p.K) + head_off;
    const T *Vh = static_cast<const T *>(p.V) + head_off;
    const T *dOh = static_cast<const T *>(p.dO) + head_off;
    T *dKh = static_cast<T *>(p.dK) + head_off;
    T *dVh = static_cast<T *>(p.dV) + head_off;
    const size_t sst = (size_t)stats_stride(n);
    const float *lse_in = p.row_stats + (size_t)bh * sst;
    const float *dl_in = p.row_stats + (size_t)p.B * p.H * sst + (size_t)bh * sst;
    const uint8_t *km = p.key_mask ? p.key_mask + (size_t)beta * n : nullptr;

    unsigned *misc = reinterpret_cast<unsigned *>(sm + L::misc_off);
    unsigned *bmap = reinterpret_cast<unsigned *>(sm + L::map_off);
    const int blk = LF ? kChunk : p.b;  // query rows per bitmap bit
    const int nblk = (n + blk - 1) / blk;
    const int words = (nblk + 31) / 32;
    for (int t = threadIdx.x; t < words; t += kThreads) bmap[t] = 0u;
    if (threadIdx.x < 4) misc[threadIdx.x] = 0u;
    __syncthreads();

    LfGeom geo = {1, 0, false};
    if (LF) {
        // Rows that see a key of [j0, j0 + 64): the global rows (marked with
        // the global chunks), every row when a key is global, else the rows of
        // the band around the tile (causal: only rows at or after the key).
        geo = lf_geom(p, h, tile == 0 && threadIdx.x == 0);
        lf_mark_globals(p, j0, bmap, misc);
        __syncthreads();
        const bool tile_has_global = (misc[0] | misc[1]) != 0u;
        const int lo = geo.causal ? j0 / kChunk : (tile_has_global ? 0 : max(0, j0 - geo.reach) / kChunk);
        const int hi = tile_has_global ? nblk - 1 : min(n - 1, j0 + BK - 1 + geo.reach) / kChunk;
        mark_range(bmap, lo, hi);
    } else {
        // Query blocks that see key block kb: the global rows, every block when
        // kb is global, the window around kb, and the rows whose random list
        // names kb (the transposed pattern of "Big Bird", App. D).
        const int kb = tile;
        mark_range(bmap, 0, p.g - 1);
        if (kb < p.g) mark_range(bmap, 0, nblk - 1);
        const int half = p.w / 2;
        mark_range(bmap, max(0, kb - half), min(nblk - 1, kb + half));
        if (p.rand_idx && p.r > 0) {
            const int32_t *tab = p.rand_idx + (size_t)h * nblk * p.r;
            const int cnt = (nblk - p.g) * p.r;
            for (int t = threadIdx.x; t < cnt; t += kThreads) {
                const int qb = p.g + t / p.r;
                const int e = tab[(size_t)qb * p.r + (t % p.r)];
                if (e == -1) continue;
                if (e < -1 || e >= nblk) { atomicOr(p.status, kDevBadIndex); continue; }
                if (e == kb) atomicOr(&bmap[qb >> 5], 1u << (qb & 31));
            }
        }
    }
    float *Ks = sm + L::k_off;
    float *Vs = sm + L::v_off;
    float *Qs = sm + L::q_off;
    float *dOs = sm + L::do_off;
    float *lse_s = sm + L::lse_off;
    float *dl_s = sm + L::dl_off;
    load_rows<T, D>(Kh, j0, BK, n, Ks, D);
    load_rows<T, D>(Vh, j0, BK, n, Vs, D);
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int key0 = warp * R;
    const float scale_log2 = kLog2e / sqrtf((float)D);
    bool kvalid[R], kglob[R];
    float dk[R][DL], dv[R][DL];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        const int jl = key0 + rr, j = j0 + jl;
        kvalid[rr] = (j < n) && (km ? (km[j] != 0) : true);
        kglob[rr] = LF ? (((misc[jl >> 5] >> (jl & 31)) & 1u) != 0u) : false;
#pragma unroll
        for (int c = 0; c < DL; ++c) dk[rr][c] = dv[rr][c] = 0.f;
    }
    __syncthreads();
    uint8_t *rvalid = reinterpret_cast<uint8_t *>(misc + 4);
    const int32_t *gidx = p.global_idx;

    for (int wd = 0; wd < words; ++wd) {
        unsigned bits = bmap[wd];
        while (bits) {
            const int qb = wd * 32 + __ffs(bits) - 1;
            bits &= bits - 1;
            for (int c0 = qb * blk; c0 < min(n, (qb + 1) * blk); c0 += kChunk) {
                load_rows<T, D>(Qh, c0, kChunk, n, Qs, L::kS);
                load_rows<T, D>(dOh, c0, kChunk, n, dOs, L::kS);
                if (threadIdx.x < 2) misc[2 + threadIdx.x] = 0u;
                if (threadIdx.x < kChunk) {
                    const int i = c0 + threadIdx.x;
                    const bool ok = (i < n) && (km ? (km[i] != 0) : true);
                    rvalid[threadIdx.x] = ok;
                    lse_s[threadIdx.x] = ok ? lse_in[i] : CUDART_INF_F;
                    dl_s[threadIdx.x] = ok ? dl_in[i] : 0.f;
                }
                __syncthreads();
                if (LF && threadIdx.x < 32) global_bits_of_chunk(gidx, p.n_global, c0, misc + 2);
                __syncthreads();
#pragma unroll 1
                for (int grp = 0; grp < 2; ++grp) {
                    const int il = grp * 32 + lane;
                    const int i = c0 + il;
                    const bool iglob = LF && (((misc[2 + (il >> 5)] >> (il & 31)) & 1u) != 0u);
#pragma unroll 1
                    for (int rr = 0; rr < R; ++rr) {
                        const int j = j0 + key0 + rr;
                        bool ok = rvalid[il] && kvalid[rr];
                        if (LF && p.row_set != 0 && iglob != (p.row_set == 2)) ok = false;  // row outside the set
                        if (LF && ok) ok = lf_allowed(geo, i, j, iglob, kglob[rr]);
                        float pr = 0.f, ds = 0.f;
                        if (ok) {
                            const float s = dot_rows<D>(Qs + il * L::kS, Ks + (key0 + rr) * D);
                            const float dp = dot_rows<D>(dOs + il * L::kS, Vs + (key0 + rr) * D);
                            pr = exp2f(s * scale_log2 - lse_s[il]);
                            ds = pr * (dp - dl_s[il]);
                        }
                        if (!__any_sync(kFull, pr != 0.f || ds != 0.f)) continue;
#pragma unroll 4
                        for (int kk = 0; kk < 32; ++kk) {
                            const float pk = __shfl_sync(kFull, pr, kk);
                            const float dsk = __shfl_sync(kFull, ds, kk);
                            const float *orow = dOs + (grp * 32 + kk) * L::kS + lane * DL;
                            const float *qrow = Qs + (grp * 32 + kk) * L::kS + lane * DL;
#pragma unroll
                            for (int c = 0; c < DL; ++c) {
                                dv[rr][c] = fmaf(pk, orow[c], dv[rr][c]);
                                dk[rr][c] = fmaf(dsk, qrow[c], dk[rr][c]);
                            }
                        }
                    }
                }
                __syncthreads();
            }
        }
    }
    const float scale = 1.f / sqrtf((float)D);
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        const int j = j0 + key0 + rr;
        if (j >= n) continue;
#pragma unroll
        for (int c = 0; c < DL; ++c) {
            store_val(dKh + (size_t)j * D + lane * DL + c, dk[rr][c] * scale);
            store_val(dVh + (size_t)j * D + lane * DL + c, dv[rr][c]);
        }
    }
}

template <class KernelFn>
cudaError_t launch_with_smem(KernelFn kernel, dim3 grid, size_t smem, const Problem &p, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

template <int D, int BQ>
size_t row_smem(int map_bits) {
    return sizeof(float) * (size_t)RowLayout<D, BQ>::map_off + sizeof(unsigned) * (size_t)((map_bits + 31) / 32);
}
template <int D, int BK>
size_t col_smem(int map_bits) {
    return sizeof(float) * (size_t)ColLayout<D, BK>::map_off + sizeof(unsigned) * (size_t)((map_bits + 31) / 32);
}

template <typename T, int D, int TILE, bool LF>
cudaError_t launch_pair(const Problem &p, int tiles, int map_bits, cudaStream_t s) {
    const dim3 grid(tiles, p.B * p.H);
    cudaError_t e = launch_with_smem(bwd_rows_kernel<T, D, TILE, LF>, grid, row_smem<D, TILE>(map_bits), p, s);
    if (e != cudaSuccess) return e;
    return launch_with_smem(bwd_cols_kernel<T, D, TILE, LF>, grid, col_smem<D, TILE>(map_bits), p, s);
}

template <typename T>
cudaError_t launch_typed(const Problem &p, cudaStream_t s) {
    if (p.kind == kBigBird) {
        const int nb = p.n / p.b;
        if (p.d == 64 && p.b == 64) return launch_pair<T, 64, 64, false>(p, nb, nb, s);
        if (p.d == 64 && p.b == 128) return launch_pair<T, 64, 128, false>(p, nb, nb, s);
        if (p.d == 128 && p.b == 64) return launch_pair<T, 128, 64, false>(p, nb, nb, s);
        if (p.d == 128 && p.b == 128) return launch_pair<T, 128, 128, false>(p, nb, nb, s);
        return cudaErrorInvalidValue;
    }
    const int tiles = (p.n + kChunk - 1) / kChunk;
    if (p.d == 64) return launch_pair<T, 64, kChunk, true>(p, tiles, tiles, s);
    if (p.d == 128) return launch_pair<T, 128, kChunk, true>(p, tiles, tiles, s);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_simt_bwd(const Problem &p, sa_dtype dtype, cudaStream_t stream, int *launches) {
    *launches = 2;
    if (dtype == SA_FP32) return launch_typed<float>(p, stream);
    return launch_typed<__nv_bfloat16>(p, stream);
}

}  // namespace sa
