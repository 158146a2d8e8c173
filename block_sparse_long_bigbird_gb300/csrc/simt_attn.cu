// Exact SIMT sparse-attention forward (fp32 arithmetic, no tensor cores).
//
// This is the library's fp32 path (inputs and outputs fp32; TF32's 10-bit
// mantissa could not hold a 1e-4 error bound) and an exact cross-check for
// the bf16 tensor-core path. One CTA handles one tile of query rows of one
// (batch, head): a BigBird query block (b rows) or a 64-row Longformer tile.
// The key positions the tile needs are kept as a bitmap of 64-key chunks;
// chunks are staged in shared memory as fp32 and every warp streams them
// through an online softmax for its rows ("Big Bird", App. D: blockified
// look-ups so that loads are contiguous; "Longformer", Sec. 3.1 pattern).
//
// Online softmax (per row): running maximum m in the log2 domain, running
// denominator l, running numerator acc; each group of 32 keys rescales the
// running terms by 2^(m_old - m_new). Masked keys contribute exactly zero.
#include <cuda_bf16.h>
#include <math_constants.h>

#include "internal.h"
#include "simt_common.cuh"

namespace sa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 64;  // keys staged per step
using simt::kFull;
using simt::lower_bound_i32;
using simt::store_val;
using simt::to_f32;
using simt::warp_max;
using simt::warp_sum;

// Shared-memory layout of one CTA (float offsets).
template <int D, int BQ>
struct Layout {
    static constexpr int kKStride = D + 4;  // padded rows: conflict-free float4 reads
    static constexpr int q_off = 0;                         // [BQ][D]
    static constexpr int k_off = q_off + BQ * D;            // [kChunk][D+4]
    static constexpr int v_off = k_off + kChunk * kKStride;  // [kChunk][D]
    static constexpr int misc_off = v_off + kChunk * D;     // small per-chunk data
    static constexpr int misc_words = 32;  // masks + 64 validity bytes
    static constexpr int map_off = misc_off + misc_words;   // chunk bitmap words
};

// Stage keys [k0, k0 + 64) of one head as fp32; rows outside [0, n) are zero.
template <typename T, int D, int BQ>
__device__ void stage_chunk(const T *Kh, const T *Vh, int k0, int n, float *sm) {
    using L = Layout<D, BQ>;
    float *Ks = sm + L::k_off;
    float *Vs = sm + L::v_off;
    for (int idx = threadIdx.x; idx < kChunk * D; idx += kThreads) {
        const int rr = idx / D, c = idx - rr * D;
        const int k = k0 + rr;
        float kv = 0.f, vv = 0.f;
        if (k >= 0 && k < n) {
            kv = to_f32(Kh[(size_t)k * D + c]);
            vv = to_f32(Vh[(size_t)k * D + c]);
        }
        Ks[rr * L::kKStride + c] = kv;
        Vs[rr * D + c] = vv;
    }
}

// One warp folds a staged 64-key chunk into the running softmax of its R rows.
// allowed(rr, key) decides per (row-in-warp, key); it must be exact, cheap and
// side-effect free.
template <int D, int BQ, int R, class Allowed>
__device__ __forceinline__ void fold_chunk(const float *sm, int row0, int k0, float scale_log2,
                                           float (&m)[R], float (&l)[R], float (&acc)[R][D / 32],
                                           Allowed allowed) {
    using L = Layout<D, BQ>;
    constexpr int DL = D / 32;
    const int lane = threadIdx.x & 31;
    const float *Qs = sm + L::q_off;
    const float *Ks = sm + L::k_off;
    const float *Vs = sm + L::v_off;
#pragma unroll 1
    for (int grp = 0; grp < 2; ++grp) {
        const int kl = grp * 32 + lane;
        const float *krow = Ks + kl * L::kKStride;
#pragma unroll 1
        for (int rr = 0; rr < R; ++rr) {
            const float *q = Qs + (row0 + rr) * D;
            float s = 0.f;
#pragma unroll
            for (int c = 0; c < D; c += 4) {
                const float4 qv = *reinterpret_cast<const float4 *>(q + c);
                const float4 kv = *reinterpret_cast<const float4 *>(krow + c);
                s = fmaf(qv.x, kv.x, s);
                s = fmaf(qv.y, kv.y, s);
                s = fmaf(qv.z, kv.z, s);
                s = fmaf(qv.w, kv.w, s);
            }
            const float sl = allowed(rr, k0 + kl) ? s * scale_log2 : -CUDART_INF_F;
            const float mnew = fmaxf(m[rr], warp_max(sl));
            if (mnew == -CUDART_INF_F) continue;  // nothing allowed yet (warp-uniform)
            const float alpha = exp2f(m[rr] - mnew);
            const float p = exp2f(sl - mnew);
            l[rr] = l[rr] * alpha + warp_sum(p);
#pragma unroll
            for (int j = 0; j < DL; ++j) acc[rr][j] *= alpha;
#pragma unroll 4
            for (int kk = 0; kk < 32; ++kk) {
                const float pk = __shfl_sync(kFull, p, kk);
                const float *vrow = Vs + (grp * 32 + kk) * D + lane * DL;
#pragma unroll
                for (int j = 0; j < DL; ++j) acc[rr][j] = fmaf(pk, vrow[j], acc[rr][j]);
            }
            m[rr] = mnew;
        }
    }
}

template <typename T, int D, int BQ>
__device__ void load_q_tile(const T *Qh, int q0, int n, float *sm) {
    using L = Layout<D, BQ>;
    float *Qs = sm + L::q_off;
    for (int idx = threadIdx.x; idx < BQ * D; idx += kThreads) {
        const int rr = idx / D, c = idx - rr * D;
        const int i = q0 + rr;
        Qs[idx] = (i < n) ? to_f32(Qh[(size_t)i * D + c]) : 0.f;
    }
}

template <typename T, int D, int R>
__device__ void write_rows(T *Oh, int i0, int n, const float (&l)[R], const float (&acc)[R][D / 32]) {
    constexpr int DL = D / 32;
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        const int i = i0 + rr;
        if (i >= n) continue;
        const float inv = l[rr] > 0.f ? 1.f / l[rr] : 0.f;
#pragma unroll
        for (int j = 0; j < DL; ++j) store_val(Oh + (size_t)i * D + lane * DL + j, acc[rr][j] * inv);
    }
}

// ---------------------------------------------------------------- BigBird
// One CTA = query block qb of one (batch, head). Its key blocks: every block
// if qb < g; else global blocks, the clipped window and its random blocks.
template <typename T, int D, int BQ>
__global__ void __launch_bounds__(kThreads) bigbird_simt_kernel(Problem p) {
    using L = Layout<D, BQ>;
    constexpr int R = BQ / kWarps;
    extern __shared__ float sm[];
    const int qb = blockIdx.x;
    const int bh = blockIdx.y;
    const int beta = bh / p.H, h = bh - beta * p.H;
    const int n = p.n, nb = n / BQ;
    const size_t head_off = (size_t)bh * n * D;
    const T *Qh = static_cast<const T *>(p.Q) + head_off;
    const T *Kh = static_cast<const T *>(p.K) + head_off;
    const T *Vh = static_cast<const T *>(p.V) + head_off;
    T *Oh = static_cast<T *>(p.O) + head_off;
    const uint8_t *km = p.key_mask ? p.key_mask + (size_t)beta * n : nullptr;
    unsigned *bmap = reinterpret_cast<unsigned *>(sm + L::map_off);
    const int words = (nb + 31) / 32;

    for (int t = threadIdx.x; t < words; t += kThreads) bmap[t] = 0u;
    __syncthreads();
    if (qb < p.g) {
        for (int kb = threadIdx.x; kb < nb; kb += kThreads) atomicOr(&bmap[kb >> 5], 1u << (kb & 31));
    } else {
        const int half = p.w / 2;
        for (int kb = threadIdx.x; kb < p.g; kb += kThreads) atomicOr(&bmap[kb >> 5], 1u << (kb & 31));
        for (int kb = max(0, qb - half) + threadIdx.x; kb <= min(nb - 1, qb + half); kb += kThreads)
            atomicOr(&bmap[kb >> 5], 1u << (kb & 31));
        if (p.rand_idx) {
            const int32_t *rr = p.rand_idx + ((size_t)h * nb + qb) * p.r;
            for (int t = threadIdx.x; t < p.r; t += kThreads) {
                const int kb = rr[t];
                if (kb == -1) continue;
                if (kb < -1 || kb >= nb) { atomicOr(p.status, kDevBadIndex); continue; }
                atomicOr(&bmap[kb >> 5], 1u << (kb & 31));
            }
        }
    }
    load_q_tile<T, D, BQ>(Qh, qb * BQ, n, sm);
    __syncthreads();

    const int warp = threadIdx.x >> 5;
    const int row0 = warp * R;
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    float m[R], l[R], acc[R][D / 32];
    bool qvalid[R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        m[rr] = -CUDART_INF_F;
        l[rr] = 0.f;
#pragma unroll
        for (int j = 0; j < D / 32; ++j) acc[rr][j] = 0.f;
        const int i = qb * BQ + row0 + rr;
        qvalid[rr] = km ? (km[i] != 0) : true;
    }
    uint8_t *kvalid = reinterpret_cast<uint8_t *>(sm + L::misc_off);  // 64 flags

    for (int wd = 0; wd < words; ++wd) {
        unsigned bits = bmap[wd];
        while (bits) {
            const int kb = wd * 32 + __ffs(bits) - 1;
            bits &= bits - 1;
            for (int sub = 0; sub < BQ / kChunk; ++sub) {
                const int k0 = kb * BQ + sub * kChunk;
                stage_chunk<T, D, BQ>(Kh, Vh, k0, n, sm);
                if (threadIdx.x < kChunk) kvalid[threadIdx.x] = km ? (km[k0 + threadIdx.x] != 0) : 1;
                __syncthreads();
                fold_chunk<D, BQ, R>(sm, row0, k0, scale_log2, m, l, acc,
                                     [&](int rr, int key) { return qvalid[rr] && kvalid[key - k0]; });
                __syncthreads();
            }
        }
    }
    write_rows<T, D, R>(Oh, qb * BQ + row0, n, l, acc);
}

// ---------------------------------------------------------------- Longformer
// One CTA = 64 query rows [i0, i0 + 64) of one (batch, head). Chunks needed:
// all of them if a row is global, else those meeting the clipped band
// [i0 - reach, i0 + 63 + reach] plus those holding a global key, where
// reach = (window / 2) (dilation + 1) ("Longformer", Sec. 3.1: dilated
// window); the causal mode (App. B) drops everything after the query.
// mode: 0 computes every row; with separate projections for global attention
// (Sec. 3.1) the call runs twice, mode 1 (Q, K, V; global rows not stored)
// and mode 2 (Qg, Kg, Vg; only global rows, tiles without one exit early).
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) longformer_simt_kernel(Problem p, int mode) {
    constexpr int BQ = 64;
    using L = Layout<D, BQ>;
    constexpr int R = BQ / kWarps;
    extern __shared__ float sm[];
    const int i0 = blockIdx.x * BQ;
    const int bh = blockIdx.y;
    const int beta = bh / p.H;
    const int n = p.n;
    const int nch = (n + kChunk - 1) / kChunk;
    const int half = p.window / 2;
    // this head's window stride (dilation + 1); out-of-range dilations latch
    int dil = p.dilation ? p.dilation[bh % p.H] : 0;
    if (dil < 0 || dil > kMaxDilation) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.status, kDevBadIndex);
        dil = 0;
    }
    const int stride = dil + 1;
    const int reach = (int)min((long long)half * stride, (long long)n);
    const bool causal = p.causal != 0;
    const size_t head_off = (size_t)bh * n * D;
    const bool gset = (mode == 2);
    const T *Qh = static_cast<const T *>(gset ? p.Qg : p.Q) + head_off;
    const T *Kh = static_cast<const T *>(gset ? p.Kg : p.K) + head_off;
    const T *Vh = static_cast<const T *>(gset ? p.Vg : p.V) + head_off;
    T *Oh = static_cast<T *>(p.O) + head_off;
    const uint8_t *km = p.key_mask ? p.key_mask + (size_t)beta * n : nullptr;
    const int32_t *gidx = p.global_idx;
    const int ng = p.n_global;

    unsigned *misc = reinterpret_cast<unsigned *>(sm + L::misc_off);
    // misc[0..1]: 64-bit global-row mask of this tile; misc[2..3]: 64-bit
    // global-key mask of the current chunk; bytes at misc[4..]: key validity.
    unsigned *bmap = reinterpret_cast<unsigned *>(sm + L::map_off);
    const int words = (nch + 31) / 32;
    for (int t = threadIdx.x; t < words; t += kThreads) bmap[t] = 0u;
    if (threadIdx.x < 4) misc[threadIdx.x] = 0u;
    __syncthreads();

    // Validate the global list and mark the chunks holding global keys.
    for (int t = threadIdx.x; t < ng; t += kThreads) {
        const int gpos = gidx[t];
        if (gpos < 0 || gpos >= n || (t > 0 && gidx[t - 1] >= gpos)) {
            if (blockIdx.x == 0 && blockIdx.y == 0) atomicOr(p.status, kDevBadIndex);
            continue;
        }
        atomicOr(&bmap[(gpos / kChunk) >> 5], 1u << ((gpos / kChunk) & 31));
        if (gpos >= i0 && gpos < i0 + BQ) atomicOr(&misc[(gpos - i0) >> 5], 1u << ((gpos - i0) & 31));
    }
    __syncthreads();
    const bool tile_has_global = (misc[0] | misc[1]) != 0u;
    if (mode == 2 && !tile_has_global) return;  // block-uniform
    {
        const int lo = tile_has_global ? 0 : max(0, i0 - reach) / kChunk;
        const int hi = causal ? min(n - 1, i0 + BQ - 1) / kChunk
                              : (tile_has_global ? nch - 1 : min(n - 1, i0 + BQ - 1 + reach) / kChunk);
        for (int c = lo + threadIdx.x; c <= hi; c += kThreads) atomicOr(&bmap[c >> 5], 1u << (c & 31));
    }
    load_q_tile<T, D, BQ>(Qh, i0, n, sm);
    __syncthreads();

    const int warp = threadIdx.x >> 5;
    const int row0 = warp * R;
    const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    float m[R], l[R], acc[R][D / 32];
    bool qvalid[R], qglobal[R];
#pragma unroll
    for (int rr = 0; rr < R; ++rr) {
        m[rr] = -CUDART_INF_F;
        l[rr] = 0.f;
#pragma unroll
        for (int j = 0; j < D / 32; ++j) acc[rr][j] = 0.f;
        const int il = row0 + rr;
        const int i = i0 + il;
        qvalid[rr] = (i < n) && (km ? (km[i] != 0) : true);
        qglobal[rr] = (misc[il >> 5] >> (il & 31)) & 1u;
    }
    __syncthreads();
    uint8_t *kvalid = reinterpret_cast<uint8_t *>(misc + 4);

    for (int wd = 0; wd < words; ++wd) {
        unsigned bits = bmap[wd];
        while (bits) {
            const int c = wd * 32 + __ffs(bits) - 1;
            bits &= bits - 1;
            const int k0 = c * kChunk;
            stage_chunk<T, D, BQ>(Kh, Vh, k0, n, sm);
            if (threadIdx.x < 2) misc[2 + threadIdx.x] = 0u;
            if (threadIdx.x < kChunk) {
                const int k = k0 + threadIdx.x;
                kvalid[threadIdx.x] = (k < n) && (km ? (km[k] != 0) : true);
            }
            __syncthreads();
            if (threadIdx.x < 32 && ng > 0) {
                const int pos = lower_bound_i32(gidx, ng, k0);
                for (int t = pos + (int)threadIdx.x; t < ng && t < pos + kChunk; t += 32) {
                    const int gpos = gidx[t];
                    if (gpos >= k0 && gpos < k0 + kChunk)
                        atomicOr(&misc[2 + ((gpos - k0) >> 5)], 1u << ((gpos - k0) & 31));
                }
            }
            __syncthreads();
            const unsigned gk0 = misc[2], gk1 = misc[3];
            fold_chunk<D, BQ, R>(sm, row0, k0, scale_log2, m, l, acc, [&](int rr, int key) {
                const int kl = key - k0;
                if (!qvalid[rr] || !kvalid[kl]) return false;
                const unsigned gbit = ((kl < 32 ? gk0 : gk1) >> (kl & 31)) & 1u;
                const int i = i0 + row0 + rr;
                if (causal && key > i) return false;
                const int dk = i - key;
                return qglobal[rr] || gbit != 0u || (abs(dk) <= reach && dk % stride == 0);
            });
            __syncthreads();
        }
    }
    if (mode == 0) {
        write_rows<T, D, R>(Oh, i0 + row0, n, l, acc);
    } else {
        // mode 1 stores the non-global rows, mode 2 the global ones
        constexpr int DL = D / 32;
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int rr = 0; rr < R; ++rr) {
            const int i = i0 + row0 + rr;
            if (i >= n || qglobal[rr] != (mode == 2)) continue;
            const float inv = l[rr] > 0.f ? 1.f / l[rr] : 0.f;
#pragma unroll
            for (int j = 0; j < DL; ++j) store_val(Oh + (size_t)i * D + lane * DL + j, acc[rr][j] * inv);
        }
    }
}

template <class KernelFn, class... Args>
cudaError_t launch_with_smem(KernelFn kernel, dim3 grid, size_t smem, cudaStream_t s, Args... args) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, kThreads, smem, s>>>(args...);
    return cudaGetLastError();
}

template <typename T, int D, int BQ>
size_t smem_bytes(int map_bits) {
    using L = Layout<D, BQ>;
    return sizeof(float) * (size_t)L::map_off + sizeof(unsigned) * (size_t)((map_bits + 31) / 32);
}

template <typename T>
cudaError_t launch_typed(const Problem &p, cudaStream_t s) {
    const int BH = p.B * p.H;
    if (p.kind == kBigBird) {
        const int nb = p.n / p.b;
        dim3 grid(nb, BH);
        if (p.d == 64 && p.b == 64)
            return launch_with_smem(bigbird_simt_kernel<T, 64, 64>, grid, smem_bytes<T, 64, 64>(nb), s, p);
        if (p.d == 64 && p.b == 128)
            return launch_with_smem(bigbird_simt_kernel<T, 64, 128>, grid, smem_bytes<T, 64, 128>(nb), s, p);
        if (p.d == 128 && p.b == 64)
            return launch_with_smem(bigbird_simt_kernel<T, 128, 64>, grid, smem_bytes<T, 128, 64>(nb), s, p);
        if (p.d == 128 && p.b == 128)
            return launch_with_smem(bigbird_simt_kernel<T, 128, 128>, grid, smem_bytes<T, 128, 128>(nb), s, p);
        return cudaErrorInvalidValue;
    }
    const int tiles = (p.n + 63) / 64;
    const int nch = (p.n + kChunk - 1) / kChunk;
    dim3 grid(tiles, BH);
    const bool sep = p.Qg != nullptr && p.n_global > 0;
    for (int mode = sep ? 1 : 0; mode <= (sep ? 2 : 0); ++mode) {
        cudaError_t e = cudaErrorInvalidValue;
        if (p.d == 64) e = launch_with_smem(longformer_simt_kernel<T, 64>, grid, smem_bytes<T, 64, 64>(nch), s, p, mode);
        if (p.d == 128)
            e = launch_with_smem(longformer_simt_kernel<T, 128>, grid, smem_bytes<T, 128, 64>(nch), s, p, mode);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_simt(const Problem &p, sa_dtype dtype, cudaStream_t stream, int *launches) {
    *launches = (p.kind == kLongformer && p.Qg != nullptr && p.n_global > 0) ? 2 : 1;
    if (dtype == SA_FP32) return launch_typed<float>(p, stream);
    return launch_typed<__nv_bfloat16>(p, stream);
}

}  // namespace sa
