// Tensor-core sparse-attention forward for sm_103a (GB300): TMA gathers of
// key/value blocks into shared memory, tcgen05 MMAs with TMEM accumulators,
// fp32 online softmax, persistent CTAs fed by a device-side work counter.
// One kernel template serves both patterns; the BigBird and Longformer host
// sides instantiate it in their own translation units.
//
// The BigBird method ("Big Bird", App. D; blog summary Sec. 4) packs each
// query block's global, window and random key blocks into one dense product.
// Here the same block lists drive a flash-style pipeline instead: no key
// tensor is materialised and no score matrix leaves the SM.
//
// Work unit = one 128-row query tile of one (batch, head):
//   * BigBird, b = 64: query blocks (2t, 2t+1); the unit walks the union of
//     their key-block lists (blocks both see first, then one-half blocks
//     alternating halves), one 64-key block per step for d = 64 and two for
//     d = 128, and each 64-row half masks the blocks outside its own list.
//   * BigBird, b = 128: query block t; one key block per step.
//   * Tiles that contain a global query block (attends all n keys) are split
//     into `splits` chunks of steps (split-KV); each chunk writes an fp32
//     partial (m, l, O) and the last chunk to finish a row merges the
//     partials of that row in chunk order (deterministic, no float atomics).
//   * Longformer ("Longformer", Sec. 3.1), band unit: query rows
//     [128t, 128t + 128); the unit walks the 64-key blocks that meet the
//     band [128t - w/2, 128t + 127 + w/2], plus every other 64-key block that
//     holds a global key. Each row masks keys outside its own window that are
//     not global. Global rows of the tile are computed but not stored.
//   * Longformer, global-row unit: up to 128 global query rows, gathered into
//     the Q tile by the producer warp; they sweep all keys with split-KV as
//     BigBird's global tiles do.
//   * Longformer, residue-class band unit: a dilated head (stride s) of a
//     call without global tokens or padding, whose rows the host-side launch
//     gathered by residue class mod s; in that order its window is a plain
//     window, so the unit is a band unit over the copies with each row's mask
//     clipped to its class and its output stored back at its own token.
// Roles (256 threads for one tile in flight, 384 for two): per tile, one warp
// claims and decodes units, builds the key-block lists, writes the step
// records and loads Q (for d = 64 it also issues the K and V copies; for
// d = 128 two loader warps do); one warp runs the MMA loop converged, one
// elected lane issuing the tcgen05 MMAs and commits; a warpgroup runs the
// softmax (thread t owns query row t = TMEM lane t), the lazy O rescale and
// the epilogue, and releases K/V stages once the S of a later step shows
// the MMAs that read them complete (MMAs of one thread complete in order). The softmax writes P (bf16) over the first half
// of its S buffer and the PV product reads A straight from TMEM. O is double
// buffered in TMEM so a unit's epilogue runs while the next unit computes.
// Every wait is bounded in time: on expiry the CTA records SA_ERR_TIMEOUT,
// drains its in-flight copies and MMAs, frees TMEM and exits.
#pragma once

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

constexpr int kBM = 128;           // query rows per tile = TMEM lanes
constexpr int kNU = 4;             // unit-info ring depth
constexpr float kRescaleLog2 = 8.0f;  // lazy O rescale threshold (factor 256)
constexpr unsigned kFull = 0xffffffffu;
constexpr int kRegionBytes = 128 * 128;  // 128 rows x 128 B (64 bf16) swizzled region

enum UnitKind { kUnitEnd = 0, kUnitDirect = 1, kUnitSplit = 2 };

struct UnitInfo {
    int kind, bh, q0, n_steps;
    int tile_slot, chunk, nchunks, step0;  // split bookkeeping; first sweep step (-1: block list)
    int j0, j1, pad0, pad1;                // BigBird query blocks of the halves (-1: none); pad0: list length
    int pad[4];
};
static_assert(sizeof(UnitInfo) == 64, "UnitInfo layout");

struct StepInfo {
    int y[2];          // first key row of each 64-key sub-slot (n: empty, reads zeros)
    uint32_t allow;    // bit (2*s + hf): sub-slot s is in query half hf's neighbourhood
    uint32_t masked;   // nonzero: kmask holds per-key validity (key padding)
    uint64_t kmask[2];
};
static_assert(sizeof(StepInfo) == 32, "StepInfo layout");

// Keys per pipeline step (= S columns of one step): 64 for d = 64, where
// two query tiles share the SM and each tile's TMEM share (256 columns) holds
// two 64-column S slots and two O buffers; 128 for d = 128 (one tile, two
// 128-column S slots, two O buffers). Host and device both use this.
__host__ __device__ constexpr int keys_per_step(int d) { return d == 64 ? 64 : 128; }

template <int D>
struct Cfg {
    // Query tiles in flight per CTA: two independent pipelines for d = 64
    // (one tile's softmax overlaps the other's waits and MMAs), one for d = 128.
    static constexpr int NT = (D == 64) ? 2 : 1;
    static constexpr int THREADS = 128 + 128 * NT;  // control warps + one softmax warpgroup per tile
    // With one tile the spare control warps 2 and 3 issue the V and K copies:
    // a thread's bulk copies complete one after another (a few hundred cycles
    // each), so a producer that also decodes units cannot keep d = 128 fed.
    static constexpr bool LOADERS = (NT == 1);
    static constexpr int KB = keys_per_step(D);     // keys per step
    static constexpr int SUB = KB / 64;             // 64-key sub-blocks per step
    static constexpr int NS = 2;                    // S slots per tile (QK^T of step g+1 overlaps softmax g)
    static constexpr int KST = (KB == 64) ? 5 : 3;  // K / V stages per tile
    // Q buffers per tile pipeline (two let the next unit's Q load while the
    // current unit runs; measured no faster for d = 64 than a fifth K/V stage)
    static constexpr int VST = KST, NQ = 1;
    static constexpr int SI = (KB == 64) ? 8 : 6;   // step-info ring depth
    static constexpr int Q_BYTES = kBM * D * 2;     // Q tile
    static constexpr int KV_BYTES = KB * D * 2;     // K or V stage
    static constexpr int KV_REGION = KB * 128;      // one 64-column swizzled region of a K/V stage
    // per-tile big buffers (1024-B aligned), then per-tile small areas
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + NQ * Q_BYTES;
    static constexpr int V_OFF = K_OFF + KST * KV_BYTES;
    static constexpr int BIG = V_OFF + VST * KV_BYTES;
    // barrier slots within a tile's small area
    static constexpr int B_QF = 0, B_QE = B_QF + NQ, B_KF = B_QE + NQ, B_KE = B_KF + KST, B_VF = B_KE + KST, B_VE = B_VF + VST,
                         B_IF = B_VE + VST, B_IE = B_IF + SI, B_SF = B_IE + SI, B_PF = B_SF + NS, B_PV = B_PF + NS,
                         B_UF = B_PV + NS, B_UE = B_UF + kNU, B_DRAIN = B_UE + kNU, B_COUNT = B_DRAIN + 1;
    static constexpr int BAR_OFF = 0;
    static constexpr int UNIT_OFF = (B_COUNT * 8 + 15) & ~15;
    static constexpr int STEP_OFF = UNIT_OFF + kNU * 64;
    static constexpr int LIST_OFF = STEP_OFF + SI * 32;  // two lists: the next unit is decoded early
    // key-validity bits of each list entry (two 64-key words; with a key mask),
    // kept for d = 64 only (d = 128 has no shared memory left for them and
    // reads the key mask per step)
    static constexpr bool KBITS = (D == 64);
    static constexpr int KBITS_OFF = LIST_OFF + 2 * 32 * 4;
    static constexpr int SMALL = KBITS_OFF + (KBITS ? 2 * 32 * 16 : 0);
    static constexpr int SMALL_OFF = NT * BIG;
    static constexpr int MISC_OFF = SMALL_OFF + NT * SMALL;  // TMEM address, abort flag, last-CTA flag
    static constexpr int SMEM_BYTES = MISC_OFF + 16;
    static constexpr int ALLOC_BYTES = SMEM_BYTES + 1024;  // slack for 1024-B alignment
    // TMEM: each tile owns TILE_COLS columns: NS S slots of KB, then two O buffers of D
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t TILE_COLS = TMEM_COLS / NT;
    static constexpr uint32_t O_COL = NS * KB;

    static_assert(O_COL + 2 * D <= TILE_COLS, "TMEM columns per tile");
    static_assert(BIG % 1024 == 0, "tile buffers stay 1024-B aligned");
};
static_assert(Cfg<128>::ALLOC_BYTES <= 232448, "d=128 shared memory budget");
static_assert(Cfg<64>::ALLOC_BYTES <= 232448, "d=64 shared memory budget");

// Host-computed geometry of one call.
struct Geometry {
    int B, H, n, nb, b, g, w, r, half;
    int tiles;            // query tiles per head
    int gtiles;           // tiles holding a global query block
    int splits;           // chunks per global tile
    int steps_full;       // steps of a full key sweep
    int steps_per_chunk;
    int n_split_units;    // B*H*gtiles*splits
    int total_units;
    int ng;               // Longformer: entries of the global list
    int nkb;              // Longformer: 64-key blocks, ceil(n / 64)
    int causal;           // Longformer: autoregressive mode
    float scale_log2;
    unsigned long long wait_ns;
};

struct Workspace {
    unsigned *counters;   // [0] next unit, [1] finished CTAs
    unsigned *row_cnt;    // [B*H*gtiles][128] arrivals per split row
    size_t n_row_cnt;     // entries of row_cnt
    float *part_o;        // [B*H*gtiles][splits][128][D]
    float2 *part_ml;      // [B*H*gtiles][splits][128] (m, l)
};

struct Params {
    Geometry geo;
    Workspace ws;
    const int32_t *rand_idx;
    const uint8_t *key_mask;
    // Longformer: the global list, and per 64-key block kb the bits of its
    // global keys (gbits[kb]), the number of blocks before kb holding a
    // global key (gpre[kb], gpre[nkb] = total) and those blocks in order
    // (glist); all three written by longformer_prep before the main kernel.
    const __nv_bfloat16 *Q;
    const __nv_bfloat16 *Qg;  // Longformer: queries of the global-row units (Q, or the separate Qg)
    const int32_t *dilation;  // Longformer: per-head dilation [H] or NULL
    // Longformer: dilated heads with n a multiple of their stride were gathered
    // by residue class (class c's rows c, c + s, c + 2s, ... contiguous) into
    // the copies tmQp / tmKg / tmVg read; their band units run on those copies
    int class_perm;
    const int32_t *gidx;
    const unsigned long long *gbits;
    const int *gpre;
    const int *glist;
    __nv_bfloat16 *O;
    unsigned *status;
};

// ---------------------------------------------------------------- producer helpers
// Longformer global list entry t as a token position, or n when t is past the
// list or the entry is out of [0, n) or not above its predecessor (such
// entries are skipped everywhere and latch SA_ERR_BAD_INDEX in the prep pass).
__device__ __forceinline__ int global_row(const int32_t *gidx, int ng, int n, int t) {
    if (t >= ng) return n;
    const int v = __ldg(gidx + t);
    if (v < 0 || v >= n) return n;
    if (t > 0 && __ldg(gidx + t - 1) >= v) return n;
    return v;
}

// Bits [0, c) of a 64-bit word, c clamped to [0, 64].
__device__ __forceinline__ uint64_t bits_below(int c) {
    return c <= 0 ? 0ull : (c >= 64 ? ~0ull : ((1ull << c) - 1ull));
}

__device__ __forceinline__ int load_rand(const Params &p, const int32_t *row, int e, int nb) {
    int v = row ? __ldg(row + e) : -1;
    if (v == -1) return INT_MAX;
    if (v < -1 || v >= nb) {
        atomicOr(p.status, kDevBadIndex);
        return INT_MAX;
    }
    return v;
}

// Is key block kb among the random blocks of `row` (warp-uniform answer)?
__device__ __forceinline__ bool rand_has(const Params &p, const int32_t *row, int kb) {
    bool hit = false;
    if (row)
        for (int e = threadIdx.x & 31; e < p.geo.r; e += 32) hit |= load_rand(p, row, e, p.geo.nb) == kb;
    return __any_sync(kFull, hit);
}

// Does query block j (>= 0) see key block kb? `row`: j's random list.
__device__ __forceinline__ bool block_allowed(const Params &p, const int32_t *row, int j, int kb) {
    const Geometry &G = p.geo;
    if (j < 0) return false;
    if (j < G.g || kb < G.g) return true;
    if (abs(kb - j) <= G.half) return true;
    return rand_has(p, row, kb);
}

// Any valid key in block kb (per-lane check, 16-byte loads; key_mask is
// 16-byte aligned and every block starts on a multiple of 64 bytes).
__device__ __forceinline__ bool block_has_valid_lane(const uint8_t *km, int kb, int b) {
    const uint4 *src = reinterpret_cast<const uint4 *>(km + (size_t)kb * b);
    uint32_t any = 0;
    for (int i = 0; i < b / 16; ++i) {
        const uint4 v = __ldg(src + i);
        any |= v.x | v.y | v.z | v.w;
    }
    return any != 0;
}

// Validity bits of the keys of block kb (per lane, 16-byte loads): bit i of
// word h is key kb * b + 64 h + i. Blocks lie inside [0, n) (n is a multiple
// of b), so no bound check is needed.
__device__ __forceinline__ void block_key_bits_lane(const uint8_t *km, int kb, int b, uint64_t (&bits)[2]) {
    const uint4 *src = reinterpret_cast<const uint4 *>(km + (size_t)kb * b);
    bits[0] = bits[1] = 0ull;
    for (int i = 0; i < b / 16; ++i) {
        const uint4 v = __ldg(src + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t m = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int j = 0; j < 4; ++j) m |= (((w[k] >> (8 * j)) & 0xFFu) != 0u ? 1u : 0u) << (4 * k + j);
        bits[i >> 2] |= (uint64_t)m << (16 * (i & 3));
    }
}

// Validity bits of the 64 keys [y, y + 64) (per lane, 16-byte loads; y is a
// multiple of 64 inside [0, n), n a multiple of 64).
__device__ __forceinline__ uint64_t key_bits64_lane(const uint8_t *km, int y) {
    const uint4 *src = reinterpret_cast<const uint4 *>(km + y);
    uint64_t bits = 0ull;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = __ldg(src + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t m = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int j = 0; j < 4; ++j) m |= (((w[k] >> (8 * j)) & 0xFFu) != 0u ? 1u : 0u) << (4 * k + j);
        bits |= (uint64_t)m << (16 * i);
    }
    return bits;
}

// Any valid key in block kb (warp-uniform answer).
__device__ __forceinline__ bool block_has_valid_warp(const uint8_t *km, int kb, int b) {
    const int lane = threadIdx.x & 31;
    bool any = false;
    if (lane < b / 16) {
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(km + (size_t)kb * b) + lane);
        any = (v.x | v.y | v.z | v.w) != 0;
    }
    return __any_sync(kFull, any);
}

// 64-bit validity of keys [k0, k0 + 64) (warp-uniform).
__device__ __forceinline__ uint64_t key_bits64(const uint8_t *km, int k0, int n) {
    const int lane = threadIdx.x & 31;
    const int a = k0 + lane, b = k0 + 32 + lane;
    const unsigned lo = __ballot_sync(kFull, a < n && km[a] != 0);
    const unsigned hi = __ballot_sync(kFull, b < n && km[b] != 0);
    return ((uint64_t)hi << 32) | lo;
}

// Sorted, de-duplicated key-block list of a local tile, built by the whole
// producer warp: each lane holds one candidate (global block, window block or
// random block), duplicates and padded blocks drop out, and each survivor's
// rank among the survivors is its position. list[pos] = block | allow bits
// (bit 30: query block j0 sees it, bit 31: j1 sees it). Returns the number of
// blocks, or -1 when the candidates do not fit in one warp. With a key mask,
// kbits[2 pos + h] receives the validity bits of the entry's keys (word h),
// so the per-step records need no global loads.
__device__ __forceinline__ int build_local_list(const Params &p, int j0, int j1, const int32_t *r0,
                                                const int32_t *r1, const uint8_t *km, uint32_t *list,
                                                uint64_t *kbits) {
    const Geometry &G = p.geo;
    const int lane = threadIdx.x & 31;
    const int nglob = min(G.g, G.nb);
    const int jl = j1 >= 0 ? j1 : j0;
    const int wlo = max(max(0, j0 - G.half), nglob);
    const int whi = min(G.nb - 1, jl + G.half);
    const int wcount = max(0, whi - wlo + 1);
    const int nr0 = r0 ? G.r : 0, nr1 = r1 ? G.r : 0;
    const int total = nglob + wcount + nr0 + nr1;
    if (total > 32) return -1;
    int v = INT_MAX, src = 0;
    if (lane < nglob) {
        v = lane;
        src = 1;
    } else if (lane < nglob + wcount) {
        v = wlo + (lane - nglob);
        src = 2;
    } else if (lane < nglob + wcount + nr0) {
        v = load_rand(p, r0, lane - nglob - wcount, G.nb);
        src = 3;
    } else if (lane < total) {
        v = load_rand(p, r1, lane - nglob - wcount - nr0, G.nb);
        src = 4;
    }
    const unsigned same = __match_any_sync(kFull, v);
    const bool in_r0 = (__ballot_sync(kFull, src == 3) & same) != 0;
    const bool in_r1 = (__ballot_sync(kFull, src == 4) & same) != 0;
    bool valid = v < G.nb && (same & ((1u << lane) - 1u)) == 0;  // first lane holding this block
    uint64_t kb2[2] = {~0ull, ~0ull};
    if (valid && km) {
        block_key_bits_lane(km, v, G.b, kb2);
        valid = (kb2[0] | kb2[1]) != 0ull;
    }
    const bool a0 = valid && (j0 < G.g || v < G.g || abs(v - j0) <= G.half || in_r0);
    const bool a1 = valid && j1 >= 0 && (j1 < G.g || v < G.g || abs(v - j1) <= G.half || in_r1);
    const unsigned vm = __ballot_sync(kFull, valid);
    // Order for steps of two 64-key sub-slots: blocks both query halves see
    // first, then blocks of one half only, alternating half 0 / half 1, so a
    // step's two sub-slots give both halves' warps work where possible (a
    // sub-slot masked for a half costs that half's warps nothing). The rest of
    // the longer one-half run follows. Within a class, lane order.
    const unsigned below = (1u << lane) - 1u;
    const unsigned m_both = __ballot_sync(kFull, valid && a0 && a1);
    const unsigned m_0 = __ballot_sync(kFull, valid && a0 && !a1);
    const unsigned m_1 = __ballot_sync(kFull, valid && a1 && !a0);
    const int nboth = __popc(m_both), n0 = __popc(m_0), n1 = __popc(m_1), k = min(n0, n1);
    int pos;
    if (a0 && a1) {
        pos = __popc(m_both & below);
    } else {
        const int i = __popc((a0 ? m_0 : m_1) & below);
        pos = nboth + (i < k ? 2 * i + (a0 ? 0 : 1) : 2 * k + (i - k));
    }
    // survivors that no query half sees (possible only with a key mask) go last
    if (!a0 && !a1) pos = nboth + n0 + n1 + __popc(vm & ~(m_both | m_0 | m_1) & below);
    if (valid) {
        list[pos] = (uint32_t)v | (a0 ? (1u << 30) : 0u) | (a1 ? (1u << 31) : 0u);
        if (km && kbits) {
            kbits[2 * pos] = kb2[0];
            kbits[2 * pos + 1] = kb2[1];
        }
    }
    __syncwarp();
    return __popc(vm);
}

// Fallback for very wide patterns: smallest union block > x (warp-uniform).
__device__ __forceinline__ int union_next_slow(const Params &p, const int32_t *r0, const int32_t *r1, int lo, int hi,
                                               int x) {
    const Geometry &G = p.geo;
    int best = G.nb;
    if (x + 1 < G.g) best = x + 1;
    const int c = max(x + 1, lo);
    if (c <= hi && c < best) best = c;
    int cand = INT_MAX;
    for (int e = threadIdx.x & 31; e < 2 * G.r; e += 32) {
        const int v = e < G.r ? load_rand(p, r0, e, G.nb) : load_rand(p, r1, e - G.r, G.nb);
        if (v > x && v < cand) cand = v;
    }
    cand = __reduce_min_sync(kFull, cand);
    return cand < best ? cand : best;
}

struct UnitPtrs {
    const uint8_t *km;
    const int32_t *r0, *r1;
    int wlo, whi;
};
// Key mask row, random lists of the tile's query blocks, and the merged window range.
__device__ __forceinline__ UnitPtrs unit_ptrs(const Params &p, const UnitInfo &ui) {
    const Geometry &G = p.geo;
    UnitPtrs u;
    const int beta = ui.bh / G.H, h = ui.bh - beta * G.H;
    u.km = p.key_mask ? p.key_mask + (size_t)beta * G.n : nullptr;
    u.r0 = (p.rand_idx && G.r > 0) ? p.rand_idx + ((size_t)h * G.nb + ui.j0) * G.r : nullptr;
    u.r1 = (p.rand_idx && G.r > 0 && ui.j1 >= 0) ? p.rand_idx + ((size_t)h * G.nb + ui.j1) * G.r : nullptr;
    const int jl = ui.j1 >= 0 ? ui.j1 : ui.j0;
    u.wlo = max(0, ui.j0 - G.half);
    u.whi = min(G.nb - 1, jl + G.half);
    return u;
}

// ---------------------------------------------------------------- kernel
// PADDED: a key mask is present. The unpadded BigBird instantiation carries
// no per-key or per-row masking code at all (rows past n are never stored).
// LF: Longformer units (band and global-row) instead of BigBird units.
template <int D, bool PADDED, bool LF>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1)
    sparse_tc_fwd(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmKg,
                   const __grid_constant__ CUtensorMap tmVg, const __grid_constant__ CUtensorMap tmQp,
                   const Params p) {
    using C = Cfg<D>;
    static_assert(C::SI * 2 * 8 <= 2 * 32 * 4, "Longformer global-key masks fit the list area");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);

    const Geometry &G = p.geo;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Ctl ctl{abort_flag, p.status, G.wait_ns};

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int x = 0; x < C::NT; ++x) {
            const uint32_t bb = sbase + C::SMALL_OFF + x * C::SMALL + C::BAR_OFF;
            auto bar = [&](int i) { return bb + 8u * (uint32_t)i; };
            for (int i = 0; i < C::NQ; ++i) {
                mbar_init(bar(C::B_QF + i), 1);
                mbar_init(bar(C::B_QE + i), 1);
            }
            for (int i = 0; i < C::KST; ++i) {
                mbar_init(bar(C::B_KF + i), 1);
                mbar_init(bar(C::B_KE + i), 1);
            }
            for (int i = 0; i < C::VST; ++i) {
                mbar_init(bar(C::B_VF + i), 1);
                mbar_init(bar(C::B_VE + i), 1);
            }
            for (int i = 0; i < C::SI; ++i) {
                mbar_init(bar(C::B_IF + i), 1);
                mbar_init(bar(C::B_IE + i), 4 + (C::LOADERS ? 2 : 0));  // softmax warps (+ loaders)
            }
            for (int i = 0; i < C::NS; ++i) {
                mbar_init(bar(C::B_SF + i), 1);
                mbar_init(bar(C::B_PF + i), 128);
                mbar_init(bar(C::B_PV + i), 1);
            }
            for (int i = 0; i < kNU; ++i) {
                mbar_init(bar(C::B_UF + i), 1);
                mbar_init(bar(C::B_UE + i), 1 + 128 + (C::LOADERS ? 2 : 0));  // MMA, softmax (+ loaders)
            }
            mbar_init(bar(C::B_DRAIN), 1);
        }
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        if (LF) {
            prefetch_tmap(&tmKg);
            prefetch_tmap(&tmVg);
            prefetch_tmap(&tmQp);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // Role and tile of this warp: warps 2x and 2x+1 are tile x's producer and
    // MMA issuer (with one tile, warps 2 and 3 load V and K); warps
    // 4 + 4x .. 7 + 4x its softmax warpgroup.
    int role = -1, x = 0;  // 0 producer, 1 MMA, 2 softmax, 3 V loader, 4 K loader
    if (warp < 4) {
        if (C::LOADERS) {
            role = (warp < 2) ? warp : (warp == 2 ? 3 : 4);
        } else if ((warp >> 1) < C::NT) {
            role = warp & 1;
            x = warp >> 1;
        }
    } else {
        role = 2;
        x = (warp - 4) >> 2;
    }
    const uint32_t tbase = sbase + x * C::BIG;  // this tile's Q/K/V buffers
    uint8_t *small = smem + C::SMALL_OFF + x * C::SMALL;
    const uint32_t bars = sbase + C::SMALL_OFF + x * C::SMALL + C::BAR_OFF;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    UnitInfo *ring = reinterpret_cast<UnitInfo *>(small + C::UNIT_OFF);
    StepInfo *steps = reinterpret_cast<StepInfo *>(small + C::STEP_OFF);
    uint32_t *list = reinterpret_cast<uint32_t *>(small + C::LIST_OFF);
    uint64_t *kbits = C::KBITS ? reinterpret_cast<uint64_t *>(small + C::KBITS_OFF) : nullptr;  // [2][32][2]
    const uint32_t tmem = *tmem_holder + x * C::TILE_COLS;  // this tile's TMEM columns

    if (role == 0) {
        // ================================================================ producer (tile x)
        // Units are decoded one unit ahead of the TMA loads that consume them.
        uint32_t g = 0, qcnt = 0;
        uint32_t issued = 0;  // steps whose K and V copies are out (drained on abort)
        bool q_tma_last = false;  // the latest Q fill was a TMA copy (drained on abort)
        uint64_t *gmk = reinterpret_cast<uint64_t *>(list);  // Longformer: global-key bits per step
        bool ok = true;
        unsigned u_next = 0;
        // decode the next unit from the work counter into ring slot `slot`
        // and list buffer `lb`; returns its info (kind kUnitEnd when done).
        // The unit is claimed here, not earlier: a claim made ahead of need
        // holds the unit back from a tile slot that may free sooner, which
        // lengthens the call's tail (measured: the n = 4096 Longformer call 7%)
        // more than the counter's latency costs off the critical path.
        auto decode_next = [&](uint32_t ui_idx, uint32_t *lbuf, bool &slow_out) -> UnitInfo {
            UnitInfo ui = {};
            slow_out = false;
            // A tile slot's first unit is fixed by the slot's index (the call's
            // first copies wait for no counter round trip); later claims count
            // on from there.
            const unsigned slots = gridDim.x * C::NT;
            if (lane == 0) u_next = ui_idx == 0 ? blockIdx.x * C::NT + x : atomicAdd(p.ws.counters, 1u) + slots;
            int u = (int)__shfl_sync(kFull, u_next, 0);
            const uint32_t slot = ui_idx % kNU;
            if (ui_idx >= kNU && !(ok = wait_warp(bar(C::B_UE + slot), ((ui_idx / kNU) - 1) & 1, ctl))) {
                ui.kind = kUnitEnd;
                return ui;
            }
            if (u >= G.total_units) {
                ui.kind = kUnitEnd;
                if (lane == 0) {
                    ring[slot] = ui;
                    mbar_arrive(bar(C::B_UF + slot));
                }
                return ui;
            }
            int tile;
            if (u < G.n_split_units) {
                const int per = G.gtiles * G.splits;
                ui.bh = u / per;
                const int rem = u - ui.bh * per;
                tile = rem / G.splits;
                ui.chunk = rem - tile * G.splits;
                ui.nchunks = G.splits;
                ui.tile_slot = ui.bh * G.gtiles + tile;
                ui.kind = G.splits > 1 ? kUnitSplit : kUnitDirect;
                ui.step0 = ui.chunk * G.steps_per_chunk;
                ui.n_steps = max(0, min(G.steps_per_chunk, G.steps_full - ui.step0));
            } else {
                const int t0 = LF ? 0 : G.gtiles;  // Longformer: every tile has a band unit
                const int per = G.tiles - t0;
                const int v = u - G.n_split_units;
                ui.bh = v / per;
                tile = t0 + (v - ui.bh * per);
                ui.kind = kUnitDirect;
                ui.step0 = -1;
            }
            ui.q0 = tile * kBM;  // Longformer global-row unit: first entry of the global list
            if constexpr (LF) {
                ui.j0 = ui.j1 = -1;
                if (ui.step0 < 0) {
                    // band unit: 64-key blocks [blo, bhi] meet the band of rows
                    // [q0, q0 + 128); global-key blocks outside it come from
                    // glist[0, pad0) (before) and glist[pad1, ...) (after)
                    bool any_row = true;
                    if (PADDED) {
                        const uint8_t *km = p.key_mask + (size_t)(ui.bh / G.H) * G.n;
                        bool a = false;
                        for (int t = lane; t < kBM; t += 32) a |= (ui.q0 + t < G.n) && km[ui.q0 + t] != 0;
                        any_row = __any_sync(kFull, a);
                    }
                    // this head's window stride (dilation + 1) and reach
                    int dil = p.dilation ? __ldg(p.dilation + ui.bh % G.H) : 0;
                    if (dil < 0 || dil > kMaxDilation) {
                        if (lane == 0) atomicOr(p.status, kDevBadIndex);
                        dil = 0;
                    }
                    // residue-class unit: the head's rows were gathered by class, so
                    // the dilated window is a plain window (stride 1, reach w/2) in
                    // the gathered order, each row clipped to its own class
                    const int cls = (p.class_perm && dil > 0 && G.n % (dil + 1) == 0) ? dil + 1 : 0;
                    const int reach = cls ? G.half : (int)min((long long)G.half * (dil + 1), (long long)G.n);
                    ui.pad[1] = cls ? 1 : dil + 1;
                    ui.pad[2] = reach;
                    ui.pad[3] = cls;
                    const int blo = max(0, ui.q0 - reach) >> 6;
                    const int bhi = min(G.n - 1, ui.q0 + kBM - 1 + (G.causal ? 0 : reach)) >> 6;
                    int before = 0, after0 = 0, after = 0;
                    if (G.ng > 0) {
                        before = __ldg(p.gpre + blo);
                        after0 = __ldg(p.gpre + bhi + 1);
                        // causal: blocks after the band hold only keys after every row
                        after = G.causal ? 0 : __ldg(p.gpre + G.nkb) - after0;
                    }
                    ui.j0 = blo;
                    ui.j1 = bhi;
                    ui.pad0 = before;
                    ui.pad1 = after0;
                    ui.pad[0] = before + (bhi - blo + 1) + after;
                    if (before < 0 || after < 0 || ui.pad[0] > G.nkb) {  // prep tables out of step
                        if (lane == 0) atomicOr(p.status, kDevBadIndex);
                        ui.pad0 = ui.pad1 = 0;
                        ui.pad[0] = bhi - blo + 1;
                    }
                    ui.n_steps = any_row ? (ui.pad[0] + C::SUB - 1) / C::SUB : 0;
                }
                if (lane == 0) {
                    ring[slot] = ui;
                    mbar_arrive(bar(C::B_UF + slot));
                }
                return ui;
            }
            if (G.b == 64) {
                ui.j0 = 2 * tile;
                ui.j1 = (2 * tile + 1 < G.nb) ? 2 * tile + 1 : -1;
            } else {
                ui.j0 = tile;
                ui.j1 = -1;
            }
            const UnitPtrs up = unit_ptrs(p, ui);
            // steps covering `nlist` key blocks of b keys, KB keys per step
            auto list_steps = [&](int nlist) {
                return G.b == 64 ? (nlist + C::SUB - 1) / C::SUB : nlist * (2 / C::SUB);
            };
            // with a key mask, the validity of the tile's 128 query rows as four
            // 32-bit words in pad[] (the softmax reads them from the ring instead
            // of loading the mask at the start of every unit)
            bool any_row = true;
            if (up.km) {
                uint32_t any = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int t = ui.q0 + 32 * k + lane;
                    const uint32_t w = __ballot_sync(kFull, t < G.n && up.km[t] != 0);
                    ui.pad[k] = (int)w;
                    any |= w;
                }
                any_row = any != 0;
            }
            if (ui.step0 < 0) {
                int nlist = 0;
                if (any_row) {
                    nlist = build_local_list(p, ui.j0, ui.j1, up.r0, up.r1, up.km, lbuf,
                                             C::KBITS ? kbits + (lbuf - list) * 2 : nullptr);
                    if (nlist < 0) {  // wide pattern: the union is generated block by block later
                        slow_out = true;
                        nlist = 0;
                        for (int xb = union_next_slow(p, up.r0, up.r1, up.wlo, up.whi, -1); xb < G.nb;
                             xb = union_next_slow(p, up.r0, up.r1, up.wlo, up.whi, xb))
                            if (!up.km || block_has_valid_warp(up.km, xb, G.b)) ++nlist;
                    }
                }
                ui.pad0 = nlist;
                ui.n_steps = list_steps(nlist);
            }

            if (lane == 0) {
                ring[slot] = ui;
                mbar_arrive(bar(C::B_UF + slot));
            }
            return ui;
        };

        bool slow_cur = false, slow_nxt = false;
        UnitInfo cur = decode_next(0, list, slow_cur);
        for (uint32_t ui_idx = 0; ok && cur.kind != kUnitEnd; ++ui_idx) {
            uint32_t *lcur = list + (ui_idx & 1) * 32;
            uint64_t *kcur = C::KBITS ? kbits + (ui_idx & 1) * 64 : nullptr;
            // The next unit is decoded one unit ahead. With loader warps it is
            // decoded once this unit's first steps are out (the loaders then
            // run ahead meanwhile); otherwise first, because this warp's own
            // copies and step records must not pause mid-unit (decoding after
            // the second step measured +3-5% for long units but -9% for the
            // short units of the autoregressive char-LM call). A BigBird call's
            // first unit is the exception: nothing is in flight yet, so its
            // first copies go out before the second unit's list is built
            // (measured: padded n = 16384 +4%; the same order for Longformer,
            // whose units need no list, cost the char-LM call 12%).
            UnitInfo nxt;
            bool have_nxt = false;
            auto decode_ahead = [&]() {
                if (!have_nxt) {
                    nxt = decode_next(ui_idx + 1, list + ((ui_idx + 1) & 1) * 32, slow_nxt);
                    have_nxt = true;
                }
            };
            if (!C::LOADERS && (LF || ui_idx > 0)) {
                decode_ahead();
                if (!ok) break;
            }
            if (cur.n_steps > 0) {
                const UnitPtrs up = unit_ptrs(p, cur);
                const int nlist = cur.pad0;
                // ---- Q tile
                const uint32_t qs = qcnt % C::NQ;  // Q buffer of this unit
                if (qcnt >= (uint32_t)C::NQ && !(ok = wait_warp(bar(C::B_QE + qs), ((qcnt / C::NQ) - 1) & 1, ctl)))
                    break;
                if (LF && cur.step0 >= 0) {
                    // Longformer global rows: gather them with plain loads into
                    // the 128-B swizzled K-major layout the TMA would produce
                    // (16-B chunk c of row r lands at chunk c ^ (r & 7)).
                    constexpr int CPR = D / 8;  // 16-B chunks per row
                    int pr[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) pr[k] = global_row(p.gidx, G.ng, G.n, cur.q0 + lane + 32 * k);
                    const uint4 *qh = reinterpret_cast<const uint4 *>(p.Qg + (size_t)cur.bh * G.n * D);
                    uint8_t *qsm = smem + x * C::BIG + C::Q_OFF + qs * C::Q_BYTES;
#pragma unroll 8
                    for (int it = 0; it < kBM * CPR / 32; ++it) {
                        const int idx = it * 32 + lane;
                        const int r = idx / CPR, cq = idx % CPR;
                        const int grp = r >> 5;  // warp-uniform
                        const int src = grp == 0 ? pr[0] : grp == 1 ? pr[1] : grp == 2 ? pr[2] : pr[3];
                        const int pos = __shfl_sync(kFull, src, r & 31);
                        const uint4 v = pos < G.n ? __ldg(qh + (size_t)pos * CPR + cq) : make_uint4(0u, 0u, 0u, 0u);
                        *reinterpret_cast<uint4 *>(qsm + (cq >> 3) * kRegionBytes + r * 128 +
                                                   (((cq & 7) ^ (r & 7)) << 4)) = v;
                    }
                    fence_proxy_async_smem();  // generic-proxy writes -> tcgen05 operand reads
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(C::B_QF + qs));
                    q_tma_last = false;
                } else {
                    if (lane == 0) {
                        const uint32_t dst = tbase + C::Q_OFF + qs * C::Q_BYTES;
                        mbar_arrive_expect_tx(bar(C::B_QF + qs), C::Q_BYTES);
                        for (int dc = 0; dc < D / 64; ++dc)
                            for (int rh = 0; rh < 2; ++rh)
                                tma_load_3d(dst + dc * kRegionBytes + rh * 8192, (LF && cur.pad[3] > 0) ? &tmQp : &tmQ,
                                            bar(C::B_QF + qs), dc * 64,
                                            cur.q0 + rh * 64, cur.bh);
                    }
                    q_tma_last = true;
                }
                ++qcnt;
                // ---- key steps
                int xs = -1;  // wide patterns: last block emitted
                for (int t = 0; t < cur.n_steps; ++t, ++g) {
                    if (!LF && C::KBITS && up.km && cur.step0 >= 0 && (t & 31) == 0) {
                        // a global tile's sweep with a key mask: the validity bits of
                        // the next 32 steps' keys, one step per lane (one global round
                        // trip per 32 steps instead of one per step), in this unit's
                        // key-bit buffer (a sweep has no block list)
                        static_assert(!C::KBITS || C::SUB == 1, "one 64-key block per step");
                        const int yy = (cur.step0 + t + lane) * 64;
                        kcur[lane] = (t + lane < cur.n_steps && yy < G.n) ? key_bits64_lane(up.km, yy) : 0ull;
                        __syncwarp();
                    }
                    StepInfo si;
                    si.masked = up.km ? 1u : 0u;
                    si.allow = 0;
                    si.kmask[0] = si.kmask[1] = ~0ull;
                    uint64_t gm2[2] = {~0ull, ~0ull};
                    if constexpr (LF) {
                        // sub-slot s of step t is entry 2t + s of: global-key blocks
                        // before the band, the band blocks, global-key blocks after;
                        // a global-row unit sweeps every block.
                        // kmask: valid keys; gm2: global keys; masked bit s: band block
                        si.masked = 0;
                        const int nband = cur.j1 - cur.j0 + 1;
#pragma unroll
                        for (int s = 0; s < C::SUB; ++s) {
                            const int li = C::SUB * t + s;
                            int kb = -1;
                            bool band = false;
                            if (cur.step0 >= 0) {
                                kb = C::SUB * (cur.step0 + t) + s;
                                if (kb >= G.nkb) kb = -1;
                            } else if (li < cur.pad0) {
                                kb = __ldg(p.glist + li);
                            } else if (li < cur.pad0 + nband) {
                                kb = cur.j0 + (li - cur.pad0);
                                band = true;
                            } else if (li < cur.pad[0]) {
                                kb = __ldg(p.glist + cur.pad1 + (li - cur.pad0 - nband));
                            }
                            if (kb >= G.nkb) {  // prep tables out of step with this call
                                if (lane == 0) atomicOr(p.status, kDevBadIndex);
                                kb = -1;
                            }
                            const int y = kb >= 0 ? kb * 64 : G.n;
                            uint64_t kv = 0ull, gm = 0ull;
                            if (kb >= 0) {
                                kv = PADDED ? key_bits64(up.km, y, G.n) : bits_below(G.n - y);
                                gm = cur.step0 >= 0 ? ~0ull : (G.ng > 0 ? __ldg(p.gbits + kb) : 0ull);
                            }
                            si.y[s] = y;
                            si.kmask[s] = kv;
                            gm2[s] = gm;
                            if (kv & gm) {
                                si.allow |= 3u << (2 * s);  // global keys: every row sees them
                            } else if (band && kv) {
                                // a 64-row half sees a band block only when the block
                                // meets its rows' windows [i - reach, i + reach]
                                const int reach = cur.pad[2];
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    const int lo = cur.q0 + 64 * h - reach;
                                    const int hi = cur.q0 + 64 * h + 63 + (G.causal ? 0 : reach);
                                    if (y + 63 >= lo && y <= hi) si.allow |= 1u << (2 * s + h);
                                }
                            }
                            if (band) si.masked |= 1u << s;
                        }
                    } else {
#pragma unroll
                    for (int s = 0; s < C::SUB; ++s) {
                        // sub-slot u (64 keys) of the unit; a b = 128 block spans two
                        const int u = C::SUB * t + s;
                        const int part = (G.b == 64) ? 0 : (u & 1);
                        int kb = -1, y = G.n;
                        bool a0 = false, a1 = false;
                        bool have_bits = false;  // list entry: its key bits were taken at decode
                        uint64_t lbits = 0ull;
                        if (cur.step0 >= 0) {  // full sweep of a global tile
                            const int yy = (C::SUB * cur.step0) * 64 + u * 64;
                            if (yy < G.n) {
                                y = yy;
                                kb = (G.b == 64) ? (yy >> 6) : (yy >> 7);
                                a0 = block_allowed(p, up.r0, cur.j0, kb);
                                a1 = (G.b == 64) ? block_allowed(p, up.r1, cur.j1, kb) : a0;
                                if (C::KBITS && up.km) {
                                    lbits = kcur[t & 31];
                                    have_bits = true;
                                }
                            }
                        } else if (!slow_cur) {
                            const int li = (G.b == 64) ? u : (u >> 1);
                            if (li < nlist) {
                                const uint32_t e = lcur[li];
                                kb = (int)(e & 0x3FFFFFFFu);
                                a0 = (e >> 30) & 1u;
                                a1 = (G.b == 64) ? ((e >> 31) & 1u) : a0;
                                y = kb * G.b + part * 64;
                                if (C::KBITS && up.km) {
                                    lbits = kcur[2 * li + part];
                                    have_bits = true;
                                }
                            }
                        } else {
                            if (part == 0) {
                                do {
                                    xs = union_next_slow(p, up.r0, up.r1, up.wlo, up.whi, xs);
                                } while (xs < G.nb && up.km && !block_has_valid_warp(up.km, xs, G.b));
                            }
                            if (xs < G.nb) {
                                kb = xs;
                                a0 = block_allowed(p, up.r0, cur.j0, kb);
                                a1 = (G.b == 64) ? block_allowed(p, up.r1, cur.j1, kb) : a0;
                                y = kb * G.b + part * 64;
                            }
                        }
                        si.y[s] = y;
                        if (kb < 0) continue;
                        if (up.km) {
                            const uint64_t bits = have_bits ? lbits : key_bits64(up.km, y, G.n);
                            si.kmask[s] = bits;
                            if (bits == 0) continue;
                        }
                        si.allow |= (a0 ? 1u : 0u) << (2 * s);
                        si.allow |= (a1 ? 1u : 0u) << (2 * s + 1);
                    }
                    }
                    // step info -> softmax
                    const uint32_t ii = g % C::SI;
                    const uint32_t sk = g % C::KST;
                    if constexpr (!C::LOADERS) {
                        // One wait per step. Stage sk is released once PV of step
                        // g - KST has completed. PV of a step is issued only after
                        // every softmax thread published its P, and each softmax
                        // warp releases its step record before that, so the
                        // record slot of step g - SI (<= g - KST) is free as well.
                        static_assert(C::SI >= C::KST && C::KST == C::VST, "record ring covers the stage ring");
                        if (g >= C::KST && !(ok = wait_warp(bar(C::B_KE + sk), ((g / C::KST) - 1) & 1, ctl))) break;
                    } else {
                        if (g >= C::SI && !(ok = wait_warp(bar(C::B_IE + ii), ((g / C::SI) - 1) & 1, ctl))) break;
                    }
                    if constexpr (!C::LOADERS) {
                        // Branch-free: every lane stores the same record, lane 0
                        // publishes it, and two lanes arm the K and V stages and
                        // issue their copies (one box each). A thread's bulk copies
                        // complete one after another, so the issuing pair moves on
                        // by two lanes every step: consecutive steps' copies overlap.
                        static_assert(D == 64 && C::SUB == 1, "one 64-key box per K or V step");
                        steps[ii] = si;
                        if (LF) {
                            gmk[2 * ii] = gm2[0];
                            gmk[2 * ii + 1] = gm2[1];
                        }
                        mbar_arrive_if(bar(C::B_IF + ii), lane == 0);
                        const int kl = (int)((2u * g) & 31u);  // this step's K lane; V: the next one
                        const bool is_v = lane == kl + 1;
                        // global-row units read the global projections' keys and values
                        // (and residue-class units the gathered copies, passed in the same slots)
                        const bool gsel = LF && (cur.step0 >= 0 || cur.pad[3] > 0);
                        const CUtensorMap *tm = is_v ? (gsel ? &tmVg : &tmV) : (gsel ? &tmKg : &tmK);
                        tma_load_3d_if(lane == kl || is_v, tbase + (is_v ? C::V_OFF : C::K_OFF) + sk * C::KV_BYTES, tm,
                                       bar((is_v ? C::B_VF : C::B_KF) + sk), 0, si.y[0], cur.bh, C::KV_BYTES);
                        ++issued;
                    } else if (lane == 0) {
                        steps[ii] = si;
                        if (LF) {
                            gmk[2 * ii] = gm2[0];
                            gmk[2 * ii + 1] = gm2[1];
                        }
                        mbar_arrive(bar(C::B_IF + ii));
                    }
                    if (t == 1) {
                        decode_ahead();
                        if (!ok) break;
                    }
                }
            }
            if (!ok) break;
            decode_ahead();
            if (!ok) break;
            cur = nxt;
            slow_cur = slow_nxt;
        }
        if (!ok && lane == 0) {  // abort: wait for the copies this tile still has in flight
            for (uint32_t i = 0; i < (uint32_t)C::KST && i < issued; ++i) {
                const uint32_t arms = (issued - 1 - i) / C::KST + 1;  // copies into stage i
                wait_drain(bar(C::B_KF + i), (arms - 1) & 1);
                wait_drain(bar(C::B_VF + i), (arms - 1) & 1);
            }
            if (qcnt && q_tma_last) wait_drain(bar(C::B_QF + (qcnt - 1) % C::NQ), ((qcnt - 1) / C::NQ) & 1);
        }
    } else if (role == 1) {
        // ================================================================ MMA issuer (tile x)
        // The whole warp runs the loop and the waits, so descriptors and TMEM
        // addresses stay warp-uniform; one elected lane, the same every time,
        // issues the MMAs and the commits that track them.
        {
            constexpr uint32_t idesc_qk = idesc_bf16(128, C::KB, false);
            constexpr uint32_t idesc_pv = idesc_bf16(128, D, true);
            const bool leader = elect_one();
            uint32_t g = 0, qcnt = 0;
            int pend = -1;
            bool pend_first = false;
            uint32_t pend_ob = 0;
            bool ok = true;
            // descriptors built once and advanced by (byte offset >> 4): the
            // start-address field, every address below 256 KB
            const uint64_t dQ0 = desc_sw128(tbase + C::Q_OFF, 16);
            const uint64_t dK0 = desc_sw128(tbase + C::K_OFF, 16);
            const uint64_t dV0 = desc_sw128(tbase + C::V_OFF, C::KV_REGION);
            // O_ob (+)= P_h V_h; P_h is read from TMEM over S buffer h % NS
            auto issue_pv = [&](uint32_t h, bool first, uint32_t ob) -> bool {
                const uint32_t sv = h % C::VST, sb = h % C::NS;
                if (!wait_warp(bar(C::B_PF + sb), (h / C::NS) & 1, ctl)) return false;
                if (!wait_warp(bar(C::B_VF + sv), (h / C::VST) & 1, ctl)) return false;
                tc_fence_after();
                const uint32_t pt = tmem + sb * C::KB;
                const uint64_t vo = (uint64_t)((sv * C::KV_BYTES) >> 4);
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < C::KB / 16; ++kk)
                        mma_bf16_ts(tmem + C::O_COL + ob * D, pt + kk * 8, dV0 + vo + (uint64_t)((kk * 2048) >> 4),
                                    idesc_pv, (first && kk == 0) ? 0u : 1u);
                    mma_commit(bar(C::B_PV + sb));
                }
                __syncwarp();
                return true;
            };
            for (uint32_t ui_idx = 0; ok; ++ui_idx) {
                const uint32_t slot = ui_idx % kNU;
                if (!(ok = wait_warp(bar(C::B_UF + slot), (ui_idx / kNU) & 1, ctl))) break;
                const int kind = ring[slot].kind;
                const int n_steps = ring[slot].n_steps;
                __syncwarp();
                if (leader) mbar_arrive(bar(C::B_UE + slot));
                if (kind == kUnitEnd) break;
                if (n_steps == 0) {
                    // The softmax writes the previous unit's epilogue while it handles
                    // this empty unit, and that needs the held-back PV: issue it now
                    // rather than after a later unit's first QK^T (which may wait on
                    // ring slots the softmax has not released yet).
                    if (pend >= 0 && !(ok = issue_pv((uint32_t)pend, pend_first, pend_ob))) break;
                    pend = -1;
                    continue;
                }
                const uint32_t ob = qcnt & 1, qs = qcnt % C::NQ;
                if (!(ok = wait_warp(bar(C::B_QF + qs), (qcnt / C::NQ) & 1, ctl))) break;
                const uint64_t dQ = dQ0 + (uint64_t)((qs * C::Q_BYTES) >> 4);
                tc_fence_after();
                for (int t = 0; t < n_steps; ++t, ++g) {
                    const uint32_t sk = g % C::KST, sb = g % C::NS;
                    if (!(ok = wait_warp(bar(C::B_KF + sk), (g / C::KST) & 1, ctl))) break;
                    tc_fence_after();
                    const uint64_t ko = (uint64_t)((sk * C::KV_BYTES) >> 4);
                    if (leader) {
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint64_t qoff = (uint64_t)(((kk >> 2) * kRegionBytes + (kk & 3) * 32) >> 4);
                            const uint64_t koff = ko + (uint64_t)(((kk >> 2) * C::KV_REGION + (kk & 3) * 32) >> 4);
                            mma_bf16_ss(tmem + sb * C::KB, dQ + qoff, dK0 + koff, idesc_qk, kk > 0 ? 1u : 0u);
                        }
                        mma_commit(bar(C::B_SF + sb));
                        if (t == n_steps - 1) mma_commit(bar(C::B_QE + qs));
                    }
                    __syncwarp();
                    // two S slots: S_g overlaps the softmax of step g-1, then PV_{g-1}
                    if (pend >= 0 && !(ok = issue_pv((uint32_t)pend, pend_first, pend_ob))) break;
                    pend = (int)g;
                    pend_first = (t == 0);
                    pend_ob = ob;
                }
                ++qcnt;
            }
            if (ok && pend >= 0) issue_pv((uint32_t)pend, pend_first, pend_ob);
            // drain: every MMA issued by the leader has completed once this arrives
            if (leader) mma_commit(bar(C::B_DRAIN));
            __syncwarp();
            wait_drain(bar(C::B_DRAIN), 0);
        }
    } else if (role == 3 || role == 4) {
        // ================================================================ V (3) / K (4) loader
        // Follows the unit ring and the step records; one box per lane.
        const bool is_k = (role == 4);
        const uint32_t buf0 = tbase + (is_k ? C::K_OFF : C::V_OFF);
        const int bf = is_k ? C::B_KF : C::B_VF, be = is_k ? C::B_KE : C::B_VE;
        static_assert(C::KST == C::VST, "one stage count for both loaders");
        uint32_t arms[C::KST] = {};
        uint32_t g = 0;
        bool ok = true;
        for (uint32_t ui_idx = 0; ok; ++ui_idx) {
            const uint32_t slot = ui_idx % kNU;
            if (!(ok = wait_warp(bar(C::B_UF + slot), (ui_idx / kNU) & 1, ctl))) break;
            const int kind = ring[slot].kind, n_steps = ring[slot].n_steps, bh = ring[slot].bh;
            // global-row units read the global projections' keys and values
            const bool gsel = LF && (ring[slot].step0 >= 0 || ring[slot].pad[3] > 0);
            const CUtensorMap *tmap = is_k ? (gsel ? &tmKg : &tmK) : (gsel ? &tmVg : &tmV);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_UE + slot));
            if (kind == kUnitEnd) break;
            for (int t = 0; t < n_steps; ++t, ++g) {
                const uint32_t ii = g % C::SI;
                if (!(ok = wait_warp(bar(C::B_IF + ii), (g / C::SI) & 1, ctl))) break;
                const int y0 = steps[ii].y[0], y1 = steps[ii].y[1];
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_IE + ii));
                const uint32_t st = g % C::KST;
                if (g >= (uint32_t)C::KST && !(ok = wait_warp(bar(be + st), ((g / C::KST) - 1) & 1, ctl))) break;
                const uint32_t dst = buf0 + st * C::KV_BYTES;
                if (lane == 0) mbar_arrive_expect_tx(bar(bf + st), C::KV_BYTES);
                __syncwarp();
                if (lane < C::SUB * (D / 64)) {
                    const int s = lane / (D / 64), dc = lane % (D / 64);
                    tma_load_3d(dst + dc * C::KV_REGION + s * 8192, tmap, bar(bf + st), dc * 64, s ? y1 : y0, bh);
                }
                ++arms[st];
            }
        }
        if (!ok && lane == 0)  // abort: wait for the copies still in flight
            for (int i = 0; i < C::KST; ++i)
                if (arms[i]) wait_drain(bar(bf + i), (arms[i] - 1) & 1);
    } else if (role == 2) {
        // ================================================================ softmax / epilogue (tile x)
        const int tid = (warp & 3) * 32 + lane;  // query row within the tile = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        // 64-row half of this thread's row: BigBird b = 64 tiles hold two query
        // blocks; Longformer band units skip band blocks a half's windows miss
        const int hf = (LF || G.b == 64) ? (tid >> 6) : 0;
        const uint64_t *gmk = reinterpret_cast<const uint64_t *>(list);  // Longformer: global-key bits per step
        const float sl2 = G.scale_log2;

        // State of the unit whose epilogue is deferred until the next unit's
        // first step has been handed to the MMA warp.
        struct Pend {
            int kind, bh, row, tile_slot, chunk, nchunks, have;  // row: output row of this thread (n: none)
            bool row_valid;
            float m, l;
            uint32_t ob, g_last;
        };
        Pend pe = {};  // every field defined: the epilogue reads them all
        pe.kind = kUnitEnd;

        // `wait_pv` false: the caller already saw PV of step g_last complete.
        auto epilogue = [&](const Pend &e, bool wait_pv) -> bool {
            const int row = e.row;
            const uint32_t oaddr = tmem + lane_base + C::O_COL + e.ob * D;
            if (e.have) {
                if (wait_pv &&
                    !wait_warp(bar(C::B_PV + (e.g_last % C::NS)), (e.g_last / C::NS) & 1, ctl))
                    return false;
                tc_fence_after();
            }
            if (e.kind == kUnitDirect) {
                const float inv = (e.row_valid && e.l > 0.f) ? 1.f / e.l : 0.f;
                __nv_bfloat16 *orow = p.O + ((size_t)e.bh * G.n + (row < G.n ? row : 0)) * D;
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    float o[32];
                    if (e.have) {
                        tmem_ld32(oaddr + cc * 32, o);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = 0.f;
                    }
                    if (row < G.n) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint32_t w4[4];
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                __nv_bfloat162 b2 =
                                    __floats2bfloat162_rn(o[q * 8 + 2 * k] * inv, o[q * 8 + 2 * k + 1] * inv);
                                w4[k] = *reinterpret_cast<uint32_t *>(&b2);
                            }
                            *reinterpret_cast<uint4 *>(orow + cc * 32 + q * 8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        }
                    }
                }
                return true;
            }
            // split chunk: publish this row's partial; the last arrival merges the row
            const size_t prow = ((size_t)e.tile_slot * G.splits + e.chunk) * kBM + tid;
            float *po = p.ws.part_o + prow * D;
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
                float o[32];
                if (e.have) {
                    tmem_ld32(oaddr + cc * 32, o);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = 0.f;
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    __stcg(reinterpret_cast<float4 *>(po + cc * 32 + q * 4),
                           make_float4(o[q * 4], o[q * 4 + 1], o[q * 4 + 2], o[q * 4 + 3]));
            }
            __stcg(p.ws.part_ml + prow, make_float2(e.row_valid ? e.m : -CUDART_INF_F, e.row_valid ? e.l : 0.f));
            __threadfence();
            unsigned *cnt = p.ws.row_cnt + (size_t)e.tile_slot * kBM + tid;
            const unsigned prev = atomicAdd(cnt, 1u);
            if (prev != (unsigned)(e.nchunks - 1)) return true;
            __threadfence();
            float M = -CUDART_INF_F;
            for (int c = 0; c < e.nchunks; ++c) {
                const float2 ml = __ldcg(p.ws.part_ml + ((size_t)e.tile_slot * G.splits + c) * kBM + tid);
                M = fmaxf(M, ml.x);
            }
            float L = 0.f;
            for (int c = 0; c < e.nchunks; ++c) {
                const float2 ml = __ldcg(p.ws.part_ml + ((size_t)e.tile_slot * G.splits + c) * kBM + tid);
                if (ml.y > 0.f) L += ex2(ml.x - M) * ml.y;
            }
            const float inv = (e.row_valid && L > 0.f) ? 1.f / L : 0.f;
            // merge 32 columns at a time, chunks in fixed order
#pragma unroll 1
            for (int cc = 0; cc < D / 32; ++cc) {
                float acc[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) acc[i] = 0.f;
                for (int c = 0; c < e.nchunks; ++c) {
                    const float2 ml = __ldcg(p.ws.part_ml + ((size_t)e.tile_slot * G.splits + c) * kBM + tid);
                    if (!(ml.y > 0.f)) continue;
                    const float wk = ex2(ml.x - M);
                    const float *src = p.ws.part_o + (((size_t)e.tile_slot * G.splits + c) * kBM + tid) * D + cc * 32;
#pragma unroll
                    for (int i = 0; i < 32; i += 4) {
                        const float4 v = __ldcg(reinterpret_cast<const float4 *>(src + i));
                        acc[i] = fmaf(wk, v.x, acc[i]);
                        acc[i + 1] = fmaf(wk, v.y, acc[i + 1]);
                        acc[i + 2] = fmaf(wk, v.z, acc[i + 2]);
                        acc[i + 3] = fmaf(wk, v.w, acc[i + 3]);
                    }
                }
                if (row < G.n) {
                    __nv_bfloat16 *orow = p.O + ((size_t)e.bh * G.n + row) * D + cc * 32;
#pragma unroll
                    for (int i = 0; i < 32; i += 8) {
                        uint32_t w4[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[i + 2 * k] * inv, acc[i + 2 * k + 1] * inv);
                            w4[k] = *reinterpret_cast<uint32_t *>(&b2);
                        }
                        *reinterpret_cast<uint4 *>(orow + i) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                    }
                }
            }
            atomicExch(cnt, 0u);  // ready for the next call
            return true;
        };

        uint32_t g = 0, qcnt = 0;
        bool ok = true;
        for (uint32_t ui_idx = 0; ok; ++ui_idx) {
            const uint32_t slot = ui_idx % kNU;
            if (!(ok = wait_warp(bar(C::B_UF + slot), (ui_idx / kNU) & 1, ctl))) break;
            const UnitInfo ui = ring[slot];
            // BigBird with a key mask: this thread's query-row validity word
            // (read from shared memory before the slot is released)
            const uint32_t rowbits = (PADDED && !LF) ? (uint32_t)ring[slot].pad[tid >> 5] : 0u;
            mbar_arrive(bar(C::B_UE + slot));
            if (ui.kind == kUnitEnd) break;
            const int beta = ui.bh / G.H;
            // qpos: the query token of this thread's row; srow: where it is stored
            int qpos = ui.q0 + tid, srow = qpos;
            // residue-class unit: qpos is a position in the gathered order; the
            // row's class occupies [clo, chi] there, and its token is stored at
            // c + s (qpos - clo)
            bool cls_unit = false;
            int clo = 0, chi = G.n - 1;
            if constexpr (LF) {
                if (ui.step0 >= 0) {
                    qpos = srow = global_row(p.gidx, G.ng, G.n, ui.q0 + tid);
                } else if (qpos < G.n && G.ng > 0 && ((__ldg(p.gbits + (qpos >> 6)) >> (qpos & 63)) & 1ull)) {
                    srow = G.n;  // a global row: its global-row unit stores it
                }
                if (ui.step0 < 0 && ui.pad[3] > 0) {
                    const int s = ui.pad[3], M = G.n / s;
                    const int c = min(qpos, G.n - 1) / M;
                    cls_unit = true;
                    clo = c * M;
                    chi = clo + M - 1;
                    srow = qpos < G.n ? c + s * (qpos - clo) : G.n;
                }
            }
            bool row_valid = qpos < G.n;
            if constexpr (PADDED) {
                if constexpr (LF)
                    row_valid = row_valid && p.key_mask[(size_t)beta * G.n + qpos] != 0;
                else  // BigBird: the producer's row bits (qpos = q0 + tid)
                    row_valid = row_valid && ((rowbits >> (tid & 31)) & 1u);
            }
            // Longformer band units: window stride, reach and the stride pattern
            // (bits 0, s, 2s, ... of a 64-key block)
            int lstride = 1, lreach = G.half;
            uint64_t lpat = ~0ull;
            if (LF && ui.step0 < 0) {
                lstride = ui.pad[1];
                lreach = ui.pad[2];
                lpat = 1ull;  // bits 0, s, 2s, ...: doubled until the word is full
                for (int sh = lstride; sh < 64; sh *= 2) lpat |= lpat << sh;
            }
            Pend cur = {};
            cur.kind = ui.kind;
            cur.bh = ui.bh;
            cur.row = srow;
            cur.tile_slot = ui.tile_slot;
            cur.chunk = ui.chunk;
            cur.nchunks = ui.nchunks;
            cur.have = ui.n_steps > 0;
            cur.row_valid = row_valid;
            // a warp none of whose rows is valid (rows past n, padded rows, the
            // unused rows of a Longformer global-row unit) writes zero P and skips
            // the step's arithmetic
            const bool warp_rows = __any_sync(kFull, row_valid);
            cur.ob = qcnt & 1;
            if (ui.n_steps == 0) {
                if (pe.kind != kUnitEnd && !(ok = epilogue(pe, true))) break;
                pe.kind = kUnitEnd;
                cur.m = -CUDART_INF_F;
                cur.l = 0.f;
                cur.g_last = 0;
                if (!(ok = epilogue(cur, true))) break;
                continue;
            }
            ++qcnt;
            float m_ref = -CUDART_INF_F, l = 0.f;
            const uint32_t obase = tmem + lane_base + C::O_COL + cur.ob * D;
            for (int t = 0; t < ui.n_steps; ++t, ++g) {
                const uint32_t ii = g % C::SI, sb = g % C::NS;
                if (!(ok = wait_warp(bar(C::B_IF + ii), (g / C::SI) & 1, ctl))) break;
                const uint32_t allow = steps[ii].allow;
                uint64_t km0 = ~0ull, km1 = ~0ull, gm0 = 0ull, gm1 = 0ull;
                int y0 = 0, y1 = 0;
                uint32_t bandb = 0;
                if (PADDED || LF) {
                    km0 = steps[ii].kmask[0];
                    km1 = steps[ii].kmask[1];
                }
                if (LF) {
                    gm0 = gmk[2 * ii];
                    gm1 = gmk[2 * ii + 1];
                    y0 = steps[ii].y[0];
                    y1 = steps[ii].y[1];
                    bandb = steps[ii].masked;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::B_IE + ii));
                if (!(ok = wait_warp(bar(C::B_SF + sb), (g / C::NS) & 1, ctl))) break;
                tc_fence_after();
                // MMAs of one thread complete in issue order (S_g, PV_{g-1},
                // S_{g+1}, ...), so S_g complete means: K_g is consumed, PV_{g-2}
                // has read the P that S_g's slot held and its V stage is free.
                // The stage releases go out from here rather than as tensor-core
                // commits, each of which costs the shared MMA front end about as
                // much as an MMA. With separate K and V loaders K_g and V_{g-2} are
                // released on their own barriers; with one producer both halves of
                // stage g-2 are released at once, so the producer waits once.
                if (tid == 0) {
                    if constexpr (C::LOADERS) {
                        mbar_arrive(bar(C::B_KE + g % C::KST));
                        if (g >= 2) mbar_arrive(bar(C::B_VE + (g - 2) % C::VST));
                    } else {
                        if (g >= 2) mbar_arrive(bar(C::B_KE + (g - 2) % C::KST));
                    }
                }
                const uint32_t sa = tmem + lane_base + sb * C::KB;
                // Stream the step's 64-key sub-blocks ("halves"; one for d = 64):
                // each is loaded, reduced and exponentiated against the running
                // reference m_ref, then written back as bf16 P over the first
                // KB / 2 columns of S_g.
                float alpha = 1.f;
                bool resc = false;  // O needs a rescale by alpha
                float lsum = 0.f;
#pragma unroll 1
                for (int half = 0; half < C::SUB; ++half) {
                    const bool w_ok = warp_rows && ((allow >> (2 * half + hf)) & 1u);  // warp-uniform
                    uint32_t pk[32];
                    if (w_ok) {
                        float s0[32], s1[32];
                        tmem_ld32(sa + half * 64, s0);
                        tmem_ld32(sa + half * 64 + 32, s1);
                        tmem_wait_ld();
                        if constexpr (LF) {
                            // valid key and (global key, or inside this row's window
                            // [qpos - w/2, qpos + w/2] on a band block); else -inf
                            uint64_t kmh = 0ull;
                            if (row_valid) {
                                const int yh = half ? y1 : y0;
                                uint64_t bandm = 0ull;
                                if ((bandb >> half) & 1u) {
                                    bandm = bits_below(qpos + (G.causal ? 0 : lreach) - yh + 1) &
                                            ~bits_below(qpos - lreach - yh);
                                    if (lstride > 1) {  // dilated: keys k with k = qpos (mod stride)
                                        const int c0 = ((qpos - yh) % lstride + lstride) % lstride;
                                        bandm &= lpat << c0;
                                    }
                                    if (cls_unit)  // gathered order: keys of the row's own class only
                                        bandm &= bits_below(chi - yh + 1) & ~bits_below(clo - yh);
                                }
                                kmh = (half ? km1 : km0) & ((half ? gm1 : gm0) | bandm);
                                if (G.causal) kmh &= bits_below(qpos - yh + 1);  // nothing after the query
                            }
                            if (!__all_sync(kFull, kmh == ~0ull)) {
                                const uint32_t lo = (uint32_t)kmh, hi = (uint32_t)(kmh >> 32);
#pragma unroll
                                for (int i = 0; i < 32; ++i) {
                                    s0[i] = ((lo >> i) & 1u) ? s0[i] : -CUDART_INF_F;
                                    s1[i] = ((hi >> i) & 1u) ? s1[i] : -CUDART_INF_F;
                                }
                            }
                        } else if (PADDED) {
                            // padded row: nothing allowed; padded keys: -inf (skipped
                            // when the whole warp keeps every key, the common case
                            // for prefix masks)
                            const uint64_t kmh = row_valid ? (half ? km1 : km0) : 0ull;
                            if (!__all_sync(kFull, kmh == ~0ull)) {
                                const uint32_t lo = (uint32_t)kmh, hi = (uint32_t)(kmh >> 32);
#pragma unroll
                                for (int i = 0; i < 32; ++i) {
                                    s0[i] = ((lo >> i) & 1u) ? s0[i] : -CUDART_INF_F;
                                    s1[i] = ((hi >> i) & 1u) ? s1[i] : -CUDART_INF_F;
                                }
                            }
                        }
                        float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            mx0 = fmax3(mx0, s0[i], s0[i + 1]);
                            mx1 = fmax3(mx1, s1[i], s1[i + 1]);
                        }
                        const float m_new = fmaxf(m_ref, fmaxf(mx0, mx1) * sl2);
                        float fix = 1.f;  // factor for this row's first-half P (second half only)
                        if (m_new > m_ref + kRescaleLog2) {
                            const float a = ex2(m_ref - m_new);  // 0 when m_ref was -inf
                            if (m_ref != -CUDART_INF_F) {
                                if (t > 0) resc = true;
                                alpha *= a;
                                fix = a;
                            }
                            l *= a;
                            lsum *= a;
                            m_ref = m_new;
                        }
                        // The first half's P already used the old reference. tcgen05.ld/st
                        // are warp-collective (.sync.aligned): the whole warp takes the
                        // round trip when any row needs it, each row scaling by its own
                        // factor (1 leaves a bf16 value unchanged).
                        if (half == 1 && ((allow >> hf) & 1u) && __any_sync(kFull, fix != 1.f)) {
                            uint32_t q[32];
                            tmem_ld32u(sa, q);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                __nv_bfloat162 b2 = *reinterpret_cast<__nv_bfloat162 *>(&q[i]);
                                float2 f = __bfloat1622float2(b2);
                                b2 = __floats2bfloat162_rn(f.x * fix, f.y * fix);
                                q[i] = *reinterpret_cast<uint32_t *>(&b2);
                            }
                            tmem_st32u(sa, q);
                        }
                        const float neg_m = (m_ref == -CUDART_INF_F) ? 0.f : -m_ref;
                        // s * scale - m on element pairs, exponentials, pair sums
                        const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(neg_m, neg_m);
                        uint64_t acc0 = f2_pack(0.f, 0.f), acc1 = f2_pack(0.f, 0.f);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            float p0, p1, p2, p3;
                            f2_unpack(f2_fma(f2_pack(s0[i], s0[i + 1]), sc2, nm2), p0, p1);
                            f2_unpack(f2_fma(f2_pack(s1[i], s1[i + 1]), sc2, nm2), p2, p3);
                            p0 = ex2(p0);
                            p1 = ex2(p1);
                            p2 = ex2(p2);
                            p3 = ex2(p3);
                            acc0 = f2_add(acc0, f2_pack(p0, p1));
                            acc1 = f2_add(acc1, f2_pack(p2, p3));
                            __nv_bfloat162 b01 = __floats2bfloat162_rn(p0, p1);
                            __nv_bfloat162 b23 = __floats2bfloat162_rn(p2, p3);
                            pk[i >> 1] = *reinterpret_cast<uint32_t *>(&b01);
                            pk[16 + (i >> 1)] = *reinterpret_cast<uint32_t *>(&b23);
                        }
                        float a0x, a0y, a1x, a1y;
                        f2_unpack(acc0, a0x, a0y);
                        f2_unpack(acc1, a1x, a1y);
                        lsum += (a0x + a0y) + (a1x + a1y);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) pk[i] = 0u;
                    }
                    tmem_st32u(sa + half * 32, pk);
                }
                l += lsum;
                tmem_wait_st();
                if (__any_sync(kFull, resc)) {
                    // O must hold PV of step g-1 before it is rescaled
                    const uint32_t h = g - 1;
                    if (!(ok = wait_warp(bar(C::B_PV + (h % C::NS)), (h / C::NS) & 1, ctl))) break;
                    tc_fence_after();
                    const float a = resc ? alpha : 1.f;
#pragma unroll 1
                    for (int cc = 0; cc < D / 32; ++cc) {
                        float o[32];
                        tmem_ld32(obase + cc * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= a;
                        tmem_st32(obase + cc * 32, o);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                mbar_arrive(bar(C::B_PF + sb));
                if (t == 0 && pe.kind != kUnitEnd) {  // previous unit's epilogue, now off the critical path
                    if (!(ok = epilogue(pe, true))) break;
                    pe.kind = kUnitEnd;
                }
            }
            if (!ok) break;
            cur.m = m_ref;
            cur.l = l;
            cur.g_last = g - 1;
            pe = cur;
        }
        if (ok && pe.kind != kUnitEnd) epilogue(pe, true);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(*tmem_holder, C::TMEM_COLS);
    // The last CTA to finish resets the scheduler for the next call. Every
    // other CTA has finished all its work (merges included) by then. After a
    // timeout some split rows may not have been merged and their arrival
    // counters are left non-zero: the last CTA zeroes them as well, so the
    // next call starts from a clean scratch whether or not the caller has
    // read the status word in between.
    volatile int *last_flag = abort_flag + 1;
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned done = atomicAdd(p.ws.counters + 1, 1u);
        const bool last = done == gridDim.x - 1;
        *last_flag = last ? 1 + ((atomicOr(p.status, 0u) & kDevTimeout) ? 1 : 0) : 0;
    }
    __syncthreads();
    const int last = *last_flag;
    if (last == 2) {
        for (size_t i = threadIdx.x; i < p.ws.n_row_cnt; i += blockDim.x) p.ws.row_cnt[i] = 0u;
        __threadfence();
        __syncthreads();
    }
    if (last && threadIdx.x == 0) {
        atomicExch(p.ws.counters, 0u);
        atomicExch(p.ws.counters + 1, 0u);
    }
}

// ---------------------------------------------------------------- host side
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

// [B*H][n][d] bf16 viewed as a 3-D tensor {d, n, B*H}; 64 x 64 boxes, 128-B swizzle.
bool make_qkv_map(CUtensorMap *m, const void *base, int BH, int n, int d) {
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

}  // namespace
}  // namespace sa
