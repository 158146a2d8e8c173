// Tensor-core sparse-attention backward for sm_103a (GB300), bf16 in and out,
// fp32 statistics and accumulation.
//
// The gradient of O = softmax_N(i)(Q K^T / sqrt(d)) V (the exact derivative;
// the pages train through this attention, "Big Bird" App. E.1 and
// "Longformer" Sec. 5, without printing it):
//
//     P_ij = 2^(s_ij - lse_i) on N(i), s_ij = log2(e) Q_i . K_j / sqrt(d)
//     D_i  = sum_j P_ij dP_ij,  dP_ij = dO_i . V_j,  dS_ij = P_ij (dP_ij - D_i)
//     dQ = dS K / sqrt(d),  dK = dS^T Q / sqrt(d),  dV = P^T dO
//
// Two launches of one kernel template, no atomics (deterministic):
//   * row pass, one CTA per 128 query rows of one (batch, head): resident
//     A1 = Q and A2 = dO tiles, streamed 64-key chunks B1 = K and B2 = V.
//     Pass 1 over the row's chunks: X = Q K^T, Y = dO V^T (tcgen05, TMEM) and
//     the online statistics m, l = sum 2^(s - m), u = sum 2^(s - m) dP, giving
//     lse = m + log2 l and D = u / l. Pass 2 over the same chunks: X, Y again,
//     dS (bf16) written to TMEM, dQ += dS K (A operand from TMEM, B = the K
//     chunk read as an MN-major operand). lse and D go to scratch.
//   * key pass, one CTA per 128 keys: resident A1 = K and A2 = V, streamed
//     64-row chunks B1 = Q and B2 = dO of the query rows whose neighbourhood
//     holds the tile's keys (the transposed pattern): X = K Q^T = S^T,
//     Y = V dO^T = dP^T, P^T and dS^T (bf16) to TMEM, dV += P^T dO and
//     dK += dS^T Q.
// Roles (384 threads): warp 0 writes per-step records (chunk position, the
// tile halves it is allowed for, validity and global bits) and starts the
// resident tile's copy; warp 1 issues the MMAs (one elected lane); warps 2 and
// 3 stream the two chunk tensors (TMA), warp 3 also the key pass's per-row
// lse and D; warpgroups 1 and 2 (warps 4-7, 8-11) take even and odd
// steps, each thread owning one TMEM lane (one tile row). X and Y rotate
// through NSL TMEM slots (three for d = 64, two for d = 128) and each step's
// accumulate products are issued NSL - 1 steps late, so the MMA issuer runs
// ahead of the elementwise work. Every wait is bounded in time.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <climits>

#include "internal.h"
#include "sm103_ptx.cuh"
#include "tc_sync.cuh"

namespace sa {
namespace {

using namespace ptx;
using namespace tcsync;

constexpr int kTM = 128;    // tile rows = TMEM lanes
constexpr int kCN = 64;     // streamed rows per step (one chunk)
constexpr int kSI = 8;      // step-record ring depth
constexpr int kThreads = 384;
constexpr unsigned kFullMask = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

enum BwdPass { kRowPass = 0, kKeyPass = 1 };

struct BwdStep {
    int y;            // first streamed row of the chunk
    uint32_t allow;   // bit h: tile half h (64 rows) may see the chunk
    uint64_t vbits;   // valid entries of the chunk (position < n and not padded)
    uint64_t gbits;   // Longformer: global positions among the chunk's entries
    uint64_t pad;
};
static_assert(sizeof(BwdStep) == 32, "BwdStep layout");

template <int D>
struct BwdCfg {
    static constexpr int NSTG = (D == 64) ? 6 : 4;  // chunk stages (one K/Q + one V/dO chunk each)
    static constexpr int NSL = (D == 64) ? 3 : 2;   // X/Y slots in TMEM (128 columns each)
    static constexpr int TILE_BYTES = kTM * D * 2;
    static constexpr int CH_BYTES = kCN * D * 2;
    static constexpr int REG_T = kTM * 128;  // one 64-column swizzled region of a tile
    static constexpr int REG_C = kCN * 128;  // one 64-column swizzled region of a chunk
    static constexpr int A1_OFF = 0;
    static constexpr int A2_OFF = TILE_BYTES;
    static constexpr int B1_OFF = 2 * TILE_BYTES;
    static constexpr int B2_OFF = B1_OFF + NSTG * CH_BYTES;
    static constexpr int LS_OFF = B2_OFF + NSTG * CH_BYTES;  // key pass: per stage the chunk rows' lse, D
    static constexpr int BIG = LS_OFF + NSTG * 2 * kCN * 4;
    // barriers
    static constexpr int B_TF = 0, B_F = 1, B_E = B_F + NSTG, B_SF = B_E + NSTG, B_PF = B_SF + NSL,
                         B_IF = B_PF + NSL, B_IE = B_IF + kSI, B_DONE = B_IE + kSI, B_DRAIN = B_DONE + 1,
                         B_COUNT = B_DRAIN + 1;
    static constexpr int BAR_OFF = BIG;
    static constexpr int STEP_OFF = (BAR_OFF + B_COUNT * 8 + 127) & ~127;
    static constexpr int STAT_OFF = STEP_OFF + kSI * (int)sizeof(BwdStep);  // [3][128] floats
    static constexpr int MISC_OFF = STAT_OFF + 3 * kTM * 4;                 // tmem addr, abort, nsteps
    static constexpr int MAP_OFF = MISC_OFF + 16;  // chunk bitmap, then the per-chunk tables (chunk_tables)
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t ACC_COL = NSL * 128;  // accumulators after the X/Y slots
    static_assert(ACC_COL + 2 * D <= TMEM_COLS, "TMEM columns");
    static_assert(LS_OFF % 1024 == 0, "buffers stay 1024-B aligned");
};

struct BwdParams {
    int B, H, n, d;
    int kind;                // kBigBird / kLongformer
    int nb, b, g, w, r, half;  // BigBird
    int window, ng, causal;  // Longformer
    int row_set;             // Longformer: 0 all rows, 1 non-global rows, 2 global rows only
    int nch;                 // 64-row chunks per head, ceil(n / 64)
    float scale_log2, scale;
    unsigned long long wait_ns;
    const int32_t *rand_idx;
    const uint8_t *key_mask;
    const int32_t *gidx;
    const int32_t *dilation;
    __nv_bfloat16 *dQ, *dK, *dV;
    float *lse, *dl;  // [B*H*stats_stride(n)] each, stored negated (-lse, -D)
    unsigned *status;
};

// Per-chunk tables after the chunk bitmap (byte offsets from the bitmap):
// validity bits [nch] (uint64; only with key padding, else computed from n),
// Longformer global bits [nch] (uint64; Longformer only), and the tile halves
// each chunk is marked for [nch] (uint32; bit h: half h).
struct ChunkTables {
    int vb_off, gb_off, hv_off, bytes;
};
__host__ __device__ inline ChunkTables chunk_tables(int nch, bool padded, bool lf) {
    ChunkTables t;
    const int words = (nch + 31) / 32;
    t.vb_off = ((words * 4) + 7) & ~7;
    t.gb_off = t.vb_off + (padded ? 8 * nch : 0);
    t.hv_off = t.gb_off + (lf ? 8 * nch : 0);
    t.bytes = t.hv_off + 4 * nch;
    return t;
}

// ----------------------------------------------------------------- pattern helpers
__device__ __forceinline__ uint64_t bits_below64(int c) {
    return c <= 0 ? 0ull : (c >= 64 ? ~0ull : ((1ull << c) - 1ull));
}

// Random-list entry e of query block qb (INT_MAX for -1 or an out-of-range
// entry, which also latches SA_ERR_BAD_INDEX).
__device__ __forceinline__ int rand_entry(const BwdParams &p, int h, int qb, int e) {
    const int v = __ldg(p.rand_idx + ((size_t)h * p.nb + qb) * p.r + e);
    if (v == -1) return INT_MAX;
    if (v < -1 || v >= p.nb) {
        atomicOr(p.status, kDevBadIndex);
        return INT_MAX;
    }
    return v;
}

// Longformer window geometry of head h: stride dilation + 1 and reach
// (window / 2) * stride ("Longformer", Sec. 3.1); bad dilations count as 0.
__device__ __forceinline__ void lf_geometry(const BwdParams &p, int h, int &stride, int &reach) {
    int dil = p.dilation ? __ldg(p.dilation + h) : 0;
    if (dil < 0 || dil > kMaxDilation) dil = 0;
    stride = dil + 1;
    reach = (int)min((long long)(p.window / 2) * stride, (long long)p.n);
}

// Entries of [y, y + 64) in the dilated band of position i: |i - x| <= reach
// and (i - x) divisible by stride.
__device__ __forceinline__ uint64_t band_bits(int i, int y, int reach, int stride) {
    const int lo = max(y, i - reach), hi = min(y + 63, i + reach);
    if (lo > hi) return 0ull;
    const int r0 = ((i - lo) % stride + stride) % stride;
    const int p0 = lo + r0;
    if (p0 > hi) return 0ull;
    uint64_t pat = 1ull << (p0 - y);
    for (int sh = stride; sh < 64; sh *= 2) pat |= pat << sh;
    return pat & bits_below64(hi - y + 1);
}

// Is position i in the (validated) global list?
__device__ __forceinline__ bool lf_is_global(const BwdParams &p, int i) {
    int lo = 0, hi = p.ng;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(p.gidx + mid) < i) lo = mid + 1; else hi = mid;
    }
    if (lo >= p.ng || __ldg(p.gidx + lo) != i) return false;
    return lo == 0 || __ldg(p.gidx + lo - 1) < i;
}

__device__ __forceinline__ bool pos_valid(const uint8_t *km, int pos, int n) {
    return pos < n && (km == nullptr || km[pos] != 0);
}

// ----------------------------------------------------------------- kernel
template <int D, int PASS>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_tc_bwd(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmA2,
                  const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmB2,
                  const BwdParams p) {
    using C = BwdCfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x, bh = blockIdx.y;
    const int beta = bh / p.H, h = bh - beta * p.H;
    const int n = p.n;
    const int t0 = tile * kTM;  // first tile row
    const bool LF = p.kind == kLongformer;
    const uint8_t *km = p.key_mask ? p.key_mask + (size_t)beta * n : nullptr;

    auto bar = [&](int i) { return sbase + C::BAR_OFF + 8u * (uint32_t)i; };
    BwdStep *steps = reinterpret_cast<BwdStep *>(smem + C::STEP_OFF);
    float *stat = reinterpret_cast<float *>(smem + C::STAT_OFF);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
    int *nsteps_s = reinterpret_cast<int *>(smem + C::MISC_OFF + 8);
    unsigned *bmap = reinterpret_cast<unsigned *>(smem + C::MAP_OFF);
    const int words = (p.nch + 31) / 32;
    const ChunkTables ct = chunk_tables(p.nch, km != nullptr, LF);
    unsigned long long *vbt = reinterpret_cast<unsigned long long *>(smem + C::MAP_OFF + ct.vb_off);
    unsigned long long *gbt = reinterpret_cast<unsigned long long *>(smem + C::MAP_OFF + ct.gb_off);
    unsigned *hvt = reinterpret_cast<unsigned *>(smem + C::MAP_OFF + ct.hv_off);
    const Ctl ctl{abort_flag, p.status, p.wait_ns};
    const int sst = stats_stride(n);

    // ---------------------------------------------------------- setup
    for (int t = threadIdx.x; t < words; t += kThreads) bmap[t] = 0u;
    for (int t = threadIdx.x; t < p.nch; t += kThreads) hvt[t] = 0u;
    if (LF)
        for (int t = threadIdx.x; t < p.nch; t += kThreads) gbt[t] = 0ull;
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        mbar_init(bar(C::B_TF), 1);
        for (int i = 0; i < C::NSTG; ++i) {
            mbar_init(bar(C::B_F + i), 2);  // the two chunk loaders
            mbar_init(bar(C::B_E + i), 1);
        }
        for (int i = 0; i < C::NSL; ++i) {
            mbar_init(bar(C::B_SF + i), 1);
            mbar_init(bar(C::B_PF + i), 4);  // the four warps of the step's warpgroup
        }
        for (int i = 0; i < kSI; ++i) {
            mbar_init(bar(C::B_IF + i), 1);
            mbar_init(bar(C::B_IE + i), 4);
        }
        mbar_init(bar(C::B_DONE), 1);
        mbar_init(bar(C::B_DRAIN), 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    __syncthreads();
    // The resident tile does not depend on the chunk list: start its copy now.
    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tmB1);
            prefetch_tmap(&tmB2);
            mbar_arrive_expect_tx(bar(C::B_TF), 2 * C::TILE_BYTES);
        }
        __syncwarp();
        if (lane < 4 * (D / 64)) {  // 2 tensors x 2 row halves x D/64 column regions
            const int tsel = lane / (2 * (D / 64)), rem = lane % (2 * (D / 64));
            const int rh = rem / (D / 64), dc = rem % (D / 64);
            const uint32_t dst = sbase + (tsel ? C::A2_OFF : C::A1_OFF) + dc * C::REG_T + rh * 8192;
            tma_load_3d(dst, tsel ? &tmA2 : &tmA1, bar(C::B_TF), dc * 64, t0 + rh * 64, bh);
        }
    }

    // Mark the 64-row chunks this tile streams, with the tile halves (64
    // rows each) whose neighbourhood holds them.
    auto mark = [&](int lo, int hi, unsigned halves) {  // chunks [lo, hi]
        for (int c = max(lo, 0) + (int)threadIdx.x; c <= min(hi, p.nch - 1); c += kThreads)
            atomicOr(&hvt[c], halves);
    };
    int lstride = 1, lreach = 0;
    bool tile_global = false;  // Longformer: a global position among the tile's rows or keys
    if (LF) {
        lf_geometry(p, h, lstride, lreach);
        if (tile == 0 && threadIdx.x == 0 && p.dilation) {
            const int dil = __ldg(p.dilation + h);
            if (dil < 0 || dil > kMaxDilation) atomicOr(p.status, kDevBadIndex);
        }
        // chunks holding a global position (validated here once per head)
        for (int t = threadIdx.x; t < p.ng; t += kThreads) {
            const int gp = __ldg(p.gidx + t);
            if (gp < 0 || gp >= n || (t > 0 && __ldg(p.gidx + t - 1) >= gp)) {
                if (tile == 0 && bh == 0) atomicOr(p.status, kDevBadIndex);
                continue;
            }
            atomicOr(&hvt[gp >> 6], 3u);
            atomicOr(&gbt[gp >> 6], 1ull << (gp & 63));
            tile_global |= (gp >= t0 && gp < t0 + kTM);
        }
        tile_global = __syncthreads_or(tile_global);
        const int last = min(n - 1, t0 + kTM - 1);
        if (PASS == kRowPass) {
            // rows see: everything (a global row), else their band; causal: nothing later
            const int lo = tile_global ? 0 : max(0, t0 - lreach) >> 6;
            const int hi = p.causal ? last >> 6 : (tile_global ? p.nch - 1 : min(n - 1, last + lreach) >> 6);
            mark(lo, hi, 3u);
        } else {
            // keys are seen by: every row (a global key), else the rows of their band;
            // causal: only rows at or after the key
            const int lo = p.causal ? (t0 >> 6) : (tile_global ? 0 : max(0, t0 - lreach) >> 6);
            const int hi = tile_global ? p.nch - 1 : min(n - 1, last + lreach) >> 6;
            mark(lo, hi, 3u);
        }
    } else {
        const int cpb = p.b / 64;  // chunks per block
        const int nblk_tile = (p.b == 64) ? 2 : 1;
        for (int hb = 0; hb < nblk_tile; ++hb) {
            const int tb = (p.b == 64) ? 2 * tile + hb : tile;  // tile block (query or key)
            const unsigned bit = (p.b == 64) ? (1u << hb) : 3u;
            if (tb >= p.nb) continue;
            if (PASS == kRowPass) {
                // the key blocks query block tb sees
                if (tb < p.g) {
                    mark(0, p.nch - 1, bit);
                } else {
                    mark(0, p.g * cpb - 1, bit);
                    mark(max(0, tb - p.half) * cpb, (min(p.nb - 1, tb + p.half) + 1) * cpb - 1, bit);
                    if (p.rand_idx)
                        for (int e = threadIdx.x; e < p.r; e += kThreads) {
                            const int kb = rand_entry(p, h, tb, e);
                            if (kb != INT_MAX)
                                for (int c = kb * cpb; c < (kb + 1) * cpb; ++c) atomicOr(&hvt[c], bit);
                        }
                }
            } else {
                // the query blocks that see key block tb
                mark(0, p.g * cpb - 1, bit);                // global rows see everything
                if (tb < p.g) mark(0, p.nch - 1, bit);      // a global key block is seen by all
                mark(max(0, tb - p.half) * cpb, (min(p.nb - 1, tb + p.half) + 1) * cpb - 1, bit);
                if (p.rand_idx) {
                    const int cnt = (p.nb - p.g) * p.r;
                    for (int t = threadIdx.x; t < cnt; t += kThreads) {
                        const int qb = p.g + t / p.r;
                        if (rand_entry(p, h, qb, t % p.r) == tb)
                            for (int c = qb * cpb; c < (qb + 1) * cpb; ++c) atomicOr(&hvt[c], bit);
                    }
                }
            }
        }
    }
    __syncthreads();
    // Per marked chunk: validity bits; a chunk without a valid entry is
    // dropped, the others go into the bitmap the roles walk.
    for (int c = threadIdx.x; c < p.nch; c += kThreads) {
        if (hvt[c] == 0u) continue;
        const int y = c * kCN;
        uint64_t vb = bits_below64(n - y);
        if (km) {
            vb = 0ull;
            for (int e = 0; e < kCN && y + e < n; ++e) vb |= (uint64_t)(km[y + e] != 0) << e;
        }
        if (km) vbt[c] = vb;
        // global rows only: row pass tiles and key pass chunks without a global row have no work
        if (LF && p.row_set == 2 && (PASS == kRowPass ? !tile_global : gbt[c] == 0ull)) vb = 0ull;
        if (vb != 0ull) atomicOr(&bmap[c >> 5], 1u << (c & 31));
    }
    __syncthreads();
    if (warp == 0) {
        int cnt = 0;
        for (int t = lane; t < words; t += 32) cnt += __popc(bmap[t]);
        cnt = __reduce_add_sync(kFullMask, cnt);
        if (lane == 0) *nsteps_s = cnt;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const int nsteps = *nsteps_s;
    const int total = (PASS == kRowPass) ? 2 * nsteps : nsteps;
    const uint32_t tmem = *tmem_holder;

    // Sequential walk over the set bits of the chunk bitmap.
    struct Walk {
        int wd;
        unsigned bits;
    };
    auto walk_next = [&](Walk &wk) -> int {
        while (wk.bits == 0u) {
            ++wk.wd;
            wk.bits = bmap[wk.wd];
        }
        const int c = wk.wd * 32 + __ffs(wk.bits) - 1;
        wk.bits &= wk.bits - 1;
        return c;
    };

    if (warp == 0) {
        // ======================================================== step records
        bool ok = true;
        Walk wk{0, bmap[0]};
        for (int g = 0; g < total && ok; ++g) {
            if (g == nsteps) wk = Walk{0, bmap[0]};  // row pass: second sweep
            const int c = walk_next(wk);
            const uint32_t ii = g % kSI;
            if (g >= kSI && !(ok = wait_warp(bar(C::B_IE + ii), ((g / kSI) - 1) & 1, ctl))) break;
            if (lane == 0) {
                BwdStep &rec = steps[ii];
                rec.y = c * kCN;
                rec.allow = hvt[c];
                rec.vbits = km ? vbt[c] : bits_below64(n - c * kCN);
                rec.gbits = LF ? gbt[c] : 0ull;
                mbar_arrive(bar(C::B_IF + ii));
            }
            __syncwarp();
        }
        // the resident tile copy was issued at start-up; with no steps (or on
        // abort) nothing else waits for it
        if (total == 0 || !ok || *abort_flag) wait_drain(bar(C::B_TF), 0);
    } else if (warp == 2 || warp == 3) {
        // ======================================================== chunk loaders
        // Warp 2 streams B1 (K or Q), warp 3 B2 (V or dO) and, in the key
        // pass, the chunk rows' lse and D: copies issued by one warp complete
        // one after another, so each tensor gets its own warp. Both arrive on
        // the stage's full barrier with their own byte counts.
        const bool second = (warp == 3);
        uint32_t arms[C::NSTG] = {};
        bool ok = true;
        Walk wk{0, bmap[0]};
        for (int g = 0; g < total && ok; ++g) {
            if (g == nsteps) wk = Walk{0, bmap[0]};  // row pass: second sweep
            const int c = walk_next(wk);
            const int y = c * kCN;
            const uint32_t st = g % C::NSTG;
            if (g >= C::NSTG && !(ok = wait_warp(bar(C::B_E + st), ((g / C::NSTG) - 1) & 1, ctl))) break;
            const uint32_t tx = C::CH_BYTES + ((PASS == kKeyPass && second) ? 2 * kCN * 4 : 0);
            if (lane == 0) mbar_arrive_expect_tx(bar(C::B_F + st), tx);
            __syncwarp();
            if (lane < D / 64) {
                const uint32_t dst = sbase + (second ? C::B2_OFF : C::B1_OFF) + st * C::CH_BYTES + lane * C::REG_C;
                tma_load_3d(dst, second ? &tmB2 : &tmB1, bar(C::B_F + st), lane * 64, y, bh);
            } else if (PASS == kKeyPass && second && lane < D / 64 + 2) {
                // the chunk rows' -lse and -D (rows of the padded stride; rows
                // at or past n hold -lse = -inf, -D = 0)
                const int which = lane - D / 64;
                const float *src = (which ? p.dl : p.lse) + (size_t)bh * sst + y;
                bulk_load(sbase + C::LS_OFF + st * (2 * kCN * 4) + which * kCN * 4, src, kCN * 4, bar(C::B_F + st));
            }
            ++arms[st];
        }
        if (!ok || *abort_flag) {
            // drain our copies in flight before the CTA leaves
            for (int i = 0; i < C::NSTG; ++i)
                if (arms[i]) wait_drain(bar(C::B_F + i), (arms[i] - 1) & 1);
        }
    } else if (warp == 1) {
        // ======================================================== MMA issuer
        // The whole warp runs the loop and the waits (so the descriptors and
        // TMEM addresses stay warp-uniform); one elected lane, the same every
        // time, issues the MMAs and the commits that track them.
        if (total > 0) {
            constexpr uint32_t idesc_xy = idesc_bf16(kTM, kCN, false);
            constexpr uint32_t idesc_acc = idesc_bf16(kTM, D, true);
            const bool leader = elect_one();
            bool ok = wait_warp(bar(C::B_TF), 0, ctl);
            auto has_ts = [&](int g) { return PASS == kKeyPass || g >= nsteps; };
            const int first_ts = (PASS == kKeyPass) ? 0 : nsteps;
            // Descriptors: built once, then advanced by the byte offset >> 4
            // (the start-address field; every address stays below 256 KB).
            const uint64_t dA1 = desc_sw128(sbase + C::A1_OFF, 16), dA2 = desc_sw128(sbase + C::A2_OFF, 16);
            const uint64_t dB1 = desc_sw128(sbase + C::B1_OFF, 16), dB2 = desc_sw128(sbase + C::B2_OFF, 16);
            const uint64_t dB1m = desc_sw128(sbase + C::B1_OFF, C::REG_C), dB2m = desc_sw128(sbase + C::B2_OFF, C::REG_C);
            auto issue_ts = [&](int hs) -> bool {
                const uint32_t sl = hs % C::NSL, st = hs % C::NSTG;
                if (!wait_warp(bar(C::B_PF + sl), (hs / C::NSL) & 1, ctl)) return false;
                tc_fence_after();
                const uint32_t x = tmem + sl * 128;
                const uint64_t so = (uint64_t)((st * C::CH_BYTES) >> 4);
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < kCN / 16; ++kk) {
                        const uint32_t acc = (hs == first_ts && kk == 0) ? 0u : 1u;
                        const uint64_t ko = so + (uint64_t)((kk * 2048) >> 4);
                        if (PASS == kRowPass) {
                            mma_bf16_ts(tmem + C::ACC_COL, x + kk * 8, dB1m + ko, idesc_acc, acc);  // dQ += dS K
                        } else {
                            mma_bf16_ts(tmem + C::ACC_COL, x + kk * 8, dB2m + ko, idesc_acc, acc);  // dV += P^T dO
                            mma_bf16_ts(tmem + C::ACC_COL + D, x + 64 + kk * 8, dB1m + ko, idesc_acc,
                                        acc);  // dK += dS^T Q
                        }
                    }
                    mma_commit(bar(C::B_E + st));
                }
                __syncwarp();
                return true;
            };
            // Step g's accumulate products are issued after X and Y of step
            // g + NSL - 1 (in order, so before X of step g + NSL reuses the slot).
            int next_ts = first_ts;  // oldest step whose accumulate products are pending
            for (int g = 0; g < total && ok; ++g) {
                const uint32_t st = g % C::NSTG, sl = g % C::NSL;
                if (!(ok = wait_warp(bar(C::B_F + st), (g / C::NSTG) & 1, ctl))) break;
                // a statistics step's slot is free once its elementwise pass read it
                if (g >= C::NSL && !has_ts(g - C::NSL) &&
                    !(ok = wait_warp(bar(C::B_PF + sl), ((g - C::NSL) / C::NSL) & 1, ctl)))
                    break;
                tc_fence_after();
                const uint64_t so = (uint64_t)((st * C::CH_BYTES) >> 4);
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint64_t to = (uint64_t)(((kk >> 2) * C::REG_T + (kk & 3) * 32) >> 4);
                        const uint64_t co = so + (uint64_t)(((kk >> 2) * C::REG_C + (kk & 3) * 32) >> 4);
                        mma_bf16_ss(tmem + sl * 128, dA1 + to, dB1 + co, idesc_xy, kk > 0 ? 1u : 0u);
                        mma_bf16_ss(tmem + sl * 128 + 64, dA2 + to, dB2 + co, idesc_xy, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(C::B_SF + sl));
                    if (!has_ts(g)) mma_commit(bar(C::B_E + st));
                }
                __syncwarp();
                while (ok && next_ts <= g - (C::NSL - 1)) ok = issue_ts(next_ts++);
            }
            while (ok && next_ts < total) ok = issue_ts(next_ts++);
            if (leader) {
                mma_commit(bar(C::B_DONE));
                mma_commit(bar(C::B_DRAIN));
            }
            __syncwarp();
            wait_drain(bar(C::B_DRAIN), 0);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ======================================================== elementwise warpgroups
        const int wg = (warp - 4) >> 2;          // 0: even steps, 1: odd steps
        const int row = ((warp & 3) << 5) + lane;  // TMEM lane = tile row
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const int pos = t0 + row;                // this thread's query row (row pass) or key (key pass)
        const int hf = row >> 6;                 // tile half
        const bool own_global = LF && p.ng > 0 && pos < n && lf_is_global(p, pos);
        // row pass: a query row outside the row set takes no part
        const bool own_valid = pos_valid(km, pos, n) &&
                               !(PASS == kRowPass && LF && p.row_set != 0 && own_global != (p.row_set == 2));
        const float sl2 = p.scale_log2;
        float m = -CUDART_INF_F, l = 0.f, u = 0.f;  // row pass statistics
        float lse = CUDART_INF_F, dlv = 0.f;
        bool ok = true;

        // allowed columns of one step for this thread
        auto step_mask = [&](const BwdStep &rec) -> uint64_t {
            if (!own_valid) return 0ull;
            uint64_t mk;
            if (LF) {
                mk = own_global ? ~0ull : (band_bits(pos, rec.y, lreach, lstride) | rec.gbits);
                if (p.causal)
                    mk &= (PASS == kRowPass) ? bits_below64(pos - rec.y + 1) : ~bits_below64(pos - rec.y);
            } else {
                mk = ((rec.allow >> hf) & 1u) ? ~0ull : 0ull;
            }
            // key pass: only the rows of the row set (the columns are query rows)
            if (PASS == kKeyPass && LF && p.row_set != 0) mk &= (p.row_set == 2) ? rec.gbits : ~rec.gbits;
            return mk & rec.vbits;
        };

        // One step: wait for its record and its X / Y, then per half of 32
        // columns load X and Y and either fold them into the statistics
        // (row pass, first sweep) or form P and dS (bf16) and write them back
        // over the slot's first columns for the accumulate products.
        auto run_step = [&](int g, bool stats) -> bool {
            const uint32_t ii = g % kSI, sl = g % C::NSL;
            if (!wait_warp(bar(C::B_IF + ii), (g / kSI) & 1, ctl)) return false;
            const BwdStep &rec = steps[ii];
            const uint64_t mk = step_mask(rec);
            if (!wait_warp(bar(C::B_SF + sl), (g / C::NSL) & 1, ctl)) return false;
            tc_fence_after();
            const uint32_t xa = tmem + lane_addr + sl * 128;
            // key pass: the chunk rows' lse and D, landed with the stage (the
            // MMA waited for the stage before X and Y, so SF implies them)
            const float *lsd = reinterpret_cast<const float *>(smem + C::LS_OFF + (g % C::NSTG) * (2 * kCN * 4));
            uint32_t pw[32], dw[32];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float xv[32], yv[32];
                tmem_ld32(xa + 32 * hh, xv);
                tmem_ld32(xa + 64 + 32 * hh, yv);
                tmem_wait_ld();
                const uint32_t mh = (uint32_t)(mk >> (32 * hh));
                const bool full = (mh == 0xffffffffu);
                if (stats) {
                    // scaled scores (masked: -inf), their maximum, then the
                    // rescaled sums l and u in packed fp32 pairs
                    const uint64_t c2 = f2_pack(sl2, sl2);
                    float mx = -CUDART_INF_F;
                    if (full) {
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            f2_unpack(f2_fma(f2_pack(xv[j], xv[j + 1]), c2, 0ull), xv[j], xv[j + 1]);
                            mx = fmax3(mx, xv[j], xv[j + 1]);
                        }
                    } else if (mh != 0u) {
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            float a, b;
                            f2_unpack(f2_fma(f2_pack(xv[j], xv[j + 1]), c2, 0ull), a, b);
                            xv[j] = ((mh >> j) & 1u) ? a : -CUDART_INF_F;
                            xv[j + 1] = ((mh >> (j + 1)) & 1u) ? b : -CUDART_INF_F;
                            mx = fmax3(mx, xv[j], xv[j + 1]);
                        }
                    }
                    const float mn = fmaxf(m, mx);
                    if (mh != 0u && mn != -CUDART_INF_F) {
                        const float alpha = ex2(m - mn);
                        const uint64_t nm2 = f2_pack(-mn, -mn);
                        uint64_t ls2 = 0ull, us2 = 0ull;
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            float a, b;
                            f2_unpack(f2_add(f2_pack(xv[j], xv[j + 1]), nm2), a, b);
                            const uint64_t e2 = f2_pack(ex2(a), ex2(b));
                            ls2 = f2_add(ls2, e2);
                            us2 = f2_fma(e2, f2_pack(yv[j], yv[j + 1]), us2);
                        }
                        float la, lb, ua, ub;
                        f2_unpack(ls2, la, lb);
                        f2_unpack(us2, ua, ub);
                        l = fmaf(l, alpha, la + lb);
                        u = fmaf(u, alpha, ua + ub);
                        m = mn;
                    }
                } else if (mh == 0u) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) pw[16 * hh + j] = dw[16 * hh + j] = 0u;
                } else {
                    // P = 2^(s c - lse) on the allowed columns, dS = P (dP - D);
                    // the statistics arrive negated (-lse, -D) as packed pairs
                    const uint64_t c2 = f2_pack(sl2, sl2);
                    const uint64_t nl_row = f2_pack(-lse, -lse), nd_row = f2_pack(-dlv, -dlv);
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        const int c = 32 * hh + j;
                        uint64_t nl = nl_row, nd = nd_row;
                        if (PASS == kKeyPass) {
                            nl = *reinterpret_cast<const uint64_t *>(lsd + c);
                            nd = *reinterpret_cast<const uint64_t *>(lsd + kCN + c);
                        }
                        float ta, tb;
                        f2_unpack(f2_fma(f2_pack(xv[j], xv[j + 1]), c2, nl), ta, tb);
                        float p0 = ex2(ta), p1 = ex2(tb);
                        if (!full) {
                            p0 = ((mh >> j) & 1u) ? p0 : 0.f;
                            p1 = ((mh >> (j + 1)) & 1u) ? p1 : 0.f;
                        }
                        const uint64_t p2 = f2_pack(p0, p1);
                        float da, db;
                        f2_unpack(f2_fma(p2, f2_add(f2_pack(yv[j], yv[j + 1]), nd), 0ull), da, db);
                        __nv_bfloat162 pp = __floats2bfloat162_rn(p0, p1);
                        __nv_bfloat162 dd = __floats2bfloat162_rn(da, db);
                        pw[c >> 1] = *reinterpret_cast<uint32_t *>(&pp);
                        dw[c >> 1] = *reinterpret_cast<uint32_t *>(&dd);
                    }
                }
            }
            if (!stats) {
                if (PASS == kRowPass) {
                    tmem_st32u(xa, dw);  // dS over X's first 32 columns
                } else {
                    tmem_st32u(xa, pw);       // P^T over X's first 32 columns
                    tmem_st32u(xa + 64, dw);  // dS^T over Y's first 32 columns
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(C::B_PF + sl));
                mbar_arrive(bar(C::B_IE + ii));
            }
            return true;
        };

        if (PASS == kRowPass) {
            for (int g = wg; g < nsteps && ok; g += 2) ok = run_step(g, true);
            if (nsteps > 0) {
                // Merge the two warpgroups' (m, l, u) into lse and D. Every
                // elementwise thread reaches both barriers (all waits above
                // are bounded), aborted or not.
                if (wg == 1) {
                    stat[row] = m;
                    stat[kTM + row] = l;
                    stat[2 * kTM + row] = u;
                }
                named_bar_sync(1, 256);
                if (wg == 0) {
                    const float m1 = stat[row], l1 = stat[kTM + row], u1 = stat[2 * kTM + row];
                    const float mm = fmaxf(m, m1);
                    float lt = 0.f, ut = 0.f;
                    if (mm != -CUDART_INF_F) {
                        const float a0 = ex2(m - mm), a1 = ex2(m1 - mm);
                        lt = l * a0 + l1 * a1;
                        ut = u * a0 + u1 * a1;
                    }
                    lse = lt > 0.f ? mm + log2f(lt) : CUDART_INF_F;
                    dlv = lt > 0.f ? ut / lt : 0.f;
                    stat[row] = lse;
                    stat[kTM + row] = dlv;
                    if (pos < sst) {  // stored negated: the key pass adds them
                        p.lse[(size_t)bh * sst + pos] = -lse;
                        p.dl[(size_t)bh * sst + pos] = -dlv;
                    }
                }
                named_bar_sync(1, 256);
                if (wg == 1) {
                    lse = stat[row];
                    dlv = stat[kTM + row];
                }
            }
            for (int g = nsteps + ((wg + nsteps) & 1); g < total && ok; g += 2) ok = run_step(g, false);
        } else {
            for (int g = wg; g < total && ok; g += 2) ok = run_step(g, false);
        }
        // ---- epilogue: accumulators to global memory
        if (ok && !*abort_flag) {
            bool have = total > 0;
            if (have && !(ok = wait_warp(bar(C::B_DONE), 0, ctl))) have = false;
            tc_fence_after();
            if (ok) {
                // row pass: dQ columns [32 wg, 32 wg + 32) (d = 64) or [64 wg, 64 wg + 64)
                // key pass: warpgroup 0 writes dV, warpgroup 1 dK
                constexpr int COLS = (PASS == kRowPass) ? D / 2 : D;
                const uint32_t col0 = (PASS == kRowPass) ? C::ACC_COL + wg * (D / 2) : C::ACC_COL + wg * D;
                __nv_bfloat16 *dst_base = (PASS == kRowPass) ? p.dQ : (wg == 0 ? p.dV : p.dK);
                const float mul = (PASS == kRowPass || wg == 1) ? p.scale : 1.f;
                const int cbase = (PASS == kRowPass) ? wg * (D / 2) : 0;
                __nv_bfloat16 *dst = dst_base + ((size_t)bh * n + pos) * D + cbase;
#pragma unroll
                for (int c0 = 0; c0 < COLS; c0 += 32) {
                    float v[32];
                    if (have) {
                        tmem_ld32(tmem + lane_addr + col0 + c0, v);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = 0.f;
                    }
                    if (pos < n) {
                        uint4 out[4];
                        uint32_t *ow = reinterpret_cast<uint32_t *>(out);
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            __nv_bfloat162 t = __floats2bfloat162_rn(v[j] * mul, v[j + 1] * mul);
                            ow[j >> 1] = *reinterpret_cast<uint32_t *>(&t);
                        }
                        uint4 *dp4 = reinterpret_cast<uint4 *>(dst + c0);
#pragma unroll
                        for (int q = 0; q < 4; ++q) dp4[q] = out[q];
                    }
                }
            }
        }
        if (PASS == kRowPass && nsteps == 0 && pos < sst && wg == 0) {
            p.lse[(size_t)bh * sst + pos] = -CUDART_INF_F;  // negated, as above
            p.dl[(size_t)bh * sst + pos] = 0.f;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(*tmem_holder, C::TMEM_COLS);
}

// ----------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// [B*H][n][d] bf16 viewed as {d, n, B*H}; 64 x 64 boxes with the 128-B swizzle.
bool make_map(CUtensorMap *m, const void *base, int BH, int n, int d) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)n, (cuuint64_t)BH};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)n * d * 2};
    const cuuint32_t box[3] = {64, 64, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
size_t bwd_smem_bytes(int nch, bool padded, bool lf) {
    return (size_t)BwdCfg<D>::MAP_OFF + (size_t)chunk_tables(nch, padded, lf).bytes + 1024;  // + alignment slack
}

template <int D>
cudaError_t launch_d(const Problem &pr, const BwdParams &bp, cudaStream_t s) {
    CUtensorMap mQ, mK, mV, mdO;
    const int BH = pr.B * pr.H;
    if (!make_map(&mQ, pr.Q, BH, pr.n, D) || !make_map(&mK, pr.K, BH, pr.n, D) || !make_map(&mV, pr.V, BH, pr.n, D) ||
        !make_map(&mdO, pr.dO, BH, pr.n, D))
        return cudaErrorInvalidValue;
    const size_t smem = bwd_smem_bytes<D>(bp.nch, bp.key_mask != nullptr, bp.kind == kLongformer);
    if (smem > 232448) return cudaErrorNotSupported;
    const dim3 grid((pr.n + kTM - 1) / kTM, BH);
    auto rows = sparse_tc_bwd<D, kRowPass>;
    auto keys = sparse_tc_bwd<D, kKeyPass>;
    cudaError_t e = cudaFuncSetAttribute(rows, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(keys, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    rows<<<grid, kThreads, smem, s>>>(mQ, mdO, mK, mV, bp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    keys<<<grid, kThreads, smem, s>>>(mK, mV, mQ, mdO, bp);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_bwd(const Problem &pr, const TcConfig &cfg, cudaStream_t stream, int *launches) {
    BwdParams bp = {};
    bp.B = pr.B;
    bp.H = pr.H;
    bp.n = pr.n;
    bp.d = pr.d;
    bp.kind = pr.kind;
    if (pr.kind == kBigBird) {
        bp.b = pr.b;
        bp.nb = pr.n / pr.b;
        bp.g = pr.g;
        bp.w = pr.w;
        bp.r = pr.r;
        bp.half = pr.w / 2;
        bp.rand_idx = pr.r > 0 ? pr.rand_idx : nullptr;
    } else {
        bp.window = pr.window;
        bp.ng = pr.n_global;
        bp.causal = pr.causal;
        bp.gidx = pr.global_idx;
        bp.dilation = pr.dilation;
    }
    bp.nch = (pr.n + kCN - 1) / kCN;
    bp.row_set = pr.row_set;
    bp.scale_log2 = kLog2e / sqrtf((float)pr.d);
    bp.scale = 1.f / sqrtf((float)pr.d);
    bp.wait_ns = (unsigned long long)cfg.wait_limit * 1000ull;
    bp.key_mask = pr.key_mask;
    bp.dQ = static_cast<__nv_bfloat16 *>(pr.dQ);
    bp.dK = static_cast<__nv_bfloat16 *>(pr.dK);
    bp.dV = static_cast<__nv_bfloat16 *>(pr.dV);
    bp.lse = pr.row_stats;
    bp.dl = pr.row_stats + (size_t)pr.B * pr.H * stats_stride(pr.n);
    bp.status = pr.status;
    *launches = 2;
    if (pr.d == 64) return launch_d<64>(pr, bp, stream);
    if (pr.d == 128) return launch_d<128>(pr, bp, stream);
    return cudaErrorInvalidValue;
}

}  // namespace sa
