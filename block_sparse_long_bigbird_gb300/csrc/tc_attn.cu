// Tensor-core sparse-attention forward for sm_103a (GB300): TMA gathers of
// key/value blocks into shared memory, tcgen05 MMAs with TMEM accumulators,
// fp32 online softmax, persistent CTAs fed by a device-side work counter.
//
// The method ("Big Bird", App. D; blog summary Sec. 4) packs each query
// block's global, window and random key blocks into one dense product. Here
// the same block lists drive a flash-style pipeline instead: no key tensor is
// materialised and no score matrix leaves the SM.
//
// Work unit = one 128-row query tile of one (batch, head):
//   * BigBird, b = 64: query blocks (2t, 2t+1); the unit walks the sorted
//     union of their key-block lists, two 64-key blocks per 128-key step, and
//     each 64-row half masks the blocks outside its own list.
//   * BigBird, b = 128: query block t; one key block per step.
//   * Tiles that contain a global query block (attends all n keys) are split
//     into `splits` chunks of steps (split-KV); each chunk writes an fp32
//     partial (m, l, O) and the last chunk to finish a row merges the
//     partials of that row in chunk order (deterministic, no float atomics).
// Roles (256 threads): warp 0 schedules units, builds the step lists and
// issues TMA loads; warp 1 allocates TMEM and issues tcgen05 MMAs (lane 0);
// warps 4-7 run the softmax (thread t owns query row t = TMEM lane t), the
// O rescale and the epilogue. Every wait is bounded: on expiry the CTA
// records SA_ERR_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM
// and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>

#include <climits>

#include "internal.h"
#include "sm103_ptx.cuh"

namespace sa {
namespace {

using namespace ptx;

constexpr int kBM = 128;           // query rows per tile = TMEM lanes
constexpr int kBN = 128;           // keys per step = S tile columns
constexpr int kThreads = 256;
constexpr int kNU = 4;             // unit-info ring depth
constexpr int kSoftmaxThread0 = 128;
constexpr int kTargetChunkSteps = 64;
constexpr float kRescaleLog2 = 8.0f;  // lazy O rescale threshold (factor 256)
constexpr unsigned kFull = 0xffffffffu;
constexpr int kRegionBytes = 128 * 128;  // 128 rows x 128 B (64 bf16) swizzled region

enum UnitKind { kUnitEnd = 0, kUnitDirect = 1, kUnitSplit = 2 };

struct UnitInfo {
    int kind, bh, q0, n_steps;
    int tile_slot, chunk, nchunks, step0;  // split bookkeeping; first sweep step
    int j0, j1, pad0, pad1;                // BigBird query blocks of the two halves (-1: none)
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

template <int D>
struct Cfg {
    static constexpr int STAGES = (D == 64) ? 3 : 2;
    static constexpr int NQ = (D == 64) ? 2 : 1;
    static constexpr int TILE_BYTES = 128 * D * 2;  // Q tile / K step / V step
    static constexpr int P_BYTES = 128 * 128 * 2;
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + NQ * TILE_BYTES;
    static constexpr int V_OFF = K_OFF + STAGES * TILE_BYTES;
    static constexpr int P_OFF = V_OFF + STAGES * TILE_BYTES;
    static constexpr int SMALL_OFF = P_OFF + 2 * P_BYTES;
    // small area: barriers, TMEM address, abort flag, unit ring, step ring
    static constexpr int BAR_OFF = SMALL_OFF;
    static constexpr int MISC_OFF = SMALL_OFF + 512;
    static constexpr int UNIT_OFF = SMALL_OFF + 576;
    static constexpr int STEP_OFF = UNIT_OFF + kNU * 64;
    static constexpr int SMEM_BYTES = STEP_OFF + STAGES * 32;
    static constexpr int ALLOC_BYTES = SMEM_BYTES + 1024;  // slack for 1024-B alignment
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t O_COL = 256;
};
static_assert(Cfg<128>::ALLOC_BYTES <= 232448, "d=128 shared memory budget");

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
    float scale_log2;
    long long wait_limit;
};

struct Workspace {
    unsigned *counters;   // [0] next unit, [1] finished CTAs
    unsigned *row_cnt;    // [B*H*gtiles][128] arrivals per split row
    float *part_o;        // [B*H*gtiles][splits][128][D]
    float2 *part_ml;      // [B*H*gtiles][splits][128] (m, l)
};

struct Params {
    Geometry geo;
    Workspace ws;
    const int32_t *rand_idx;
    const uint8_t *key_mask;
    __nv_bfloat16 *O;
    unsigned *status;
};

// Barrier slots (8 B each) in the small area.
enum Bar {
    B_QFULL = 0, B_QEMPTY = 2, B_KFULL = 4, B_VFULL = 7, B_SEMPTY = 10, B_SFULL = 13, B_PFULL = 15,
    B_PVDONE = 17, B_UFULL = 19, B_UEMPTY = 23, B_DRAIN = 27, B_COUNT = 28
};

struct Ctl {
    volatile int *abort;
    unsigned *status;
    long long limit;
};

// Single-thread bounded wait. Returns false (and leaves) once the CTA aborts.
__device__ __noinline__ bool wait_one(uint32_t bar, uint32_t parity, const Ctl &c) {
    if (mbar_try_wait(bar, parity)) return true;
    for (long long it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if (it >= c.limit) {
            *c.abort = 1;
            atomicOr(c.status, kDevTimeout);
            return false;
        }
        if ((it & 63) == 0 && *c.abort) return false;
    }
}
// Warp-uniform bounded wait: lane 0 waits, every lane gets the same answer.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const Ctl &c) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = wait_one(bar, parity, c) ? 1 : 0;
    return __shfl_sync(kFull, ok, 0) != 0;
}
// Drain wait used on the abort path (ignores the abort flag, still bounded).
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity, long long limit) {
    for (long long it = 0; it < limit; ++it)
        if (mbar_try_wait(bar, parity)) return;
}

// ---------------------------------------------------------------- producer helpers
// Per-lane cache of a local tile's random blocks: entries e = lane, lane + 32
// of the concatenation rand[h][j0][:] ++ rand[h][j1][:]; invalid -> INT_MAX.
struct RandCache {
    int v0, v1;
    int e0, e1;
};

__device__ __forceinline__ int load_rand(const Params &p, const int32_t *r0, const int32_t *r1, int e, int nb) {
    const int r = p.geo.r;
    int v = INT_MAX;
    if (e < r) v = r0 ? __ldg(r0 + e) : -1;
    else if (e < 2 * r) v = r1 ? __ldg(r1 + (e - r)) : -1;
    else return INT_MAX;
    if (v == -1) return INT_MAX;
    if (v < -1 || v >= nb) {
        atomicOr(p.status, kDevBadIndex);
        return INT_MAX;
    }
    return v;
}

// Smallest random block > x over both query blocks (warp-uniform result).
__device__ __forceinline__ int rand_next(const Params &p, const RandCache &rc, const int32_t *r0,
                                         const int32_t *r1, int x, int nb) {
    int cand = INT_MAX;
    if (rc.v0 > x) cand = rc.v0;
    if (rc.v1 > x && rc.v1 < cand) cand = rc.v1;
    for (int e = 64 + (threadIdx.x & 31); e < 2 * p.geo.r; e += 32) {
        const int v = load_rand(p, r0, r1, e, nb);
        if (v > x && v < cand) cand = v;
    }
    return __reduce_min_sync(kFull, cand);
}

// Is key block kb among the random blocks of query block `which` (0: j0, 1: j1)?
__device__ __forceinline__ bool rand_has(const Params &p, const RandCache &rc, const int32_t *r0,
                                         const int32_t *r1, int kb, int which, int nb) {
    const int r = p.geo.r;
    const int lo = which * r, hi = lo + r;
    bool hit = (rc.e0 >= lo && rc.e0 < hi && rc.v0 == kb) || (rc.e1 >= lo && rc.e1 < hi && rc.v1 == kb);
    for (int e = 64 + (threadIdx.x & 31); e < 2 * r; e += 32)
        if (e >= lo && e < hi && load_rand(p, r0, r1, e, nb) == kb) hit = true;
    return __any_sync(kFull, hit);
}

// Does query block j (>= 0) see key block kb? `which` selects its random list.
__device__ __forceinline__ bool block_allowed(const Params &p, const RandCache &rc, const int32_t *r0,
                                              const int32_t *r1, int j, int which, int kb) {
    const Geometry &G = p.geo;
    if (j < 0) return false;
    if (j < G.g || kb < G.g) return true;
    if (abs(kb - j) <= G.half) return true;
    return rand_has(p, rc, r0, r1, kb, which, G.nb);
}

// Smallest block > x in the union of the tile's key-block lists.
__device__ __forceinline__ int union_next(const Params &p, const RandCache &rc, const int32_t *r0,
                                          const int32_t *r1, int lo, int hi, int x) {
    const Geometry &G = p.geo;
    int best = G.nb;
    if (x + 1 < G.g) best = x + 1;
    const int c = max(x + 1, lo);
    if (c <= hi && c < best) best = c;
    const int rn = rand_next(p, rc, r0, r1, x, G.nb);
    return rn < best ? rn : best;
}

// 64-bit validity of keys [k0, k0 + 64) of sequence `beta` (warp-uniform).
__device__ __forceinline__ uint64_t key_bits64(const uint8_t *km, int k0, int n) {
    const int lane = threadIdx.x & 31;
    const int a = k0 + lane, b = k0 + 32 + lane;
    const unsigned lo = __ballot_sync(kFull, a < n && km[a] != 0);
    const unsigned hi = __ballot_sync(kFull, b < n && km[b] != 0);
    return ((uint64_t)hi << 32) | lo;
}

// Any valid key in block kb?
__device__ __forceinline__ bool block_has_valid(const Params &p, const uint8_t *km, int kb) {
    const int b = p.geo.b;
    bool any = false;
    for (int t = threadIdx.x & 31; t < b; t += 32) any |= km[kb * b + t] != 0;
    return __any_sync(kFull, any);
}

// ---------------------------------------------------------------- kernel
template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bigbird_tc_fwd(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const Params p) {
    using C = Cfg<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + C::BAR_OFF;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + C::MISC_OFF);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::MISC_OFF + 4);
    UnitInfo *ring = reinterpret_cast<UnitInfo *>(smem + C::UNIT_OFF);
    StepInfo *steps = reinterpret_cast<StepInfo *>(smem + C::STEP_OFF);

    const Geometry &G = p.geo;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Ctl ctl{abort_flag, p.status, G.wait_limit};

    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int i = 0; i < C::NQ; ++i) {
            mbar_init(bar(B_QFULL + i), 1);
            mbar_init(bar(B_QEMPTY + i), 1);
        }
        for (int i = 0; i < C::STAGES; ++i) {
            mbar_init(bar(B_KFULL + i), 1);
            mbar_init(bar(B_VFULL + i), 1);
            mbar_init(bar(B_SEMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_SFULL + i), 1);
            mbar_init(bar(B_PFULL + i), 128);
            mbar_init(bar(B_PVDONE + i), 1);
        }
        for (int i = 0; i < kNU; ++i) {
            mbar_init(bar(B_UFULL + i), 1);
            mbar_init(bar(B_UEMPTY + i), 1 + 128);
        }
        mbar_init(bar(B_DRAIN), 1);
        fence_mbar_init();
        if ((sbase & 1023u) != 0) atomicOr(p.status, kDevTimeout);  // cannot happen: aligned above
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_holder), C::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ================================================================ producer
        uint32_t g = 0, qcnt = 0;
        uint32_t kv_arms[C::STAGES] = {};
        uint32_t q_arms[C::NQ] = {};
        bool ok = true;
        for (uint32_t ui_idx = 0; ok; ++ui_idx) {
            int u = 0;
            if (lane == 0) u = (int)atomicAdd(p.ws.counters, 1u);
            u = __shfl_sync(kFull, u, 0);
            const uint32_t slot = ui_idx % kNU;
            if (ui_idx >= kNU && !(ok = wait_warp(bar(B_UEMPTY + slot), ((ui_idx / kNU) - 1) & 1, ctl))) break;
            UnitInfo ui = {};
            if (u >= G.total_units) {
                ui.kind = kUnitEnd;
                if (lane == 0) {
                    ring[slot] = ui;
                    mbar_arrive(bar(B_UFULL + slot));
                }
                break;
            }
            // ---- decode the unit
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
                const int per = G.tiles - G.gtiles;
                const int v = u - G.n_split_units;
                ui.bh = v / per;
                tile = G.gtiles + (v - ui.bh * per);
                ui.kind = kUnitDirect;
                ui.step0 = -1;  // local: sorted union of block lists
            }
            ui.q0 = tile * kBM;
            if (G.b == 64) {
                ui.j0 = 2 * tile;
                ui.j1 = (2 * tile + 1 < G.nb) ? 2 * tile + 1 : -1;
            } else {
                ui.j0 = tile;
                ui.j1 = -1;
            }
            const int beta = ui.bh / G.H, h = ui.bh - beta * G.H;
            const uint8_t *km = p.key_mask ? p.key_mask + (size_t)beta * G.n : nullptr;
            const int32_t *r0 = (p.rand_idx && G.r > 0) ? p.rand_idx + ((size_t)h * G.nb + ui.j0) * G.r : nullptr;
            const int32_t *r1 =
                (p.rand_idx && G.r > 0 && ui.j1 >= 0) ? p.rand_idx + ((size_t)h * G.nb + ui.j1) * G.r : nullptr;
            RandCache rc;
            rc.e0 = lane;
            rc.e1 = lane + 32;
            rc.v0 = load_rand(p, r0, r1, rc.e0, G.nb);
            rc.v1 = load_rand(p, r0, r1, rc.e1, G.nb);
            // union window range of the (one or two) query blocks
            const int jl = ui.j1 >= 0 ? ui.j1 : ui.j0;
            const int wlo = max(0, ui.j0 - G.half), whi = min(G.nb - 1, jl + G.half);
            const int bps = (G.b == 64) ? 2 : 1;  // key blocks per step

            if (ui.step0 < 0) {
                bool any_row = true;
                if (km) {
                    bool a = false;
                    for (int t = lane; t < kBM; t += 32) a |= (ui.q0 + t < G.n) && km[ui.q0 + t] != 0;
                    any_row = __any_sync(kFull, a);
                }
                int cnt = 0;
                if (any_row) {
                    for (int x = union_next(p, rc, r0, r1, wlo, whi, -1); x < G.nb;
                         x = union_next(p, rc, r0, r1, wlo, whi, x))
                        if (!km || block_has_valid(p, km, x)) ++cnt;
                }
                ui.n_steps = (cnt + bps - 1) / bps;
            }
            if (lane == 0) {
                ring[slot] = ui;
                mbar_arrive(bar(B_UFULL + slot));
            }
            if (ui.n_steps == 0) continue;

            // ---- Q tile
            const uint32_t qb = qcnt % C::NQ;
            if (qcnt >= C::NQ && !(ok = wait_warp(bar(B_QEMPTY + qb), ((qcnt / C::NQ) - 1) & 1, ctl))) break;
            if (lane == 0) {
                const uint32_t dst = sbase + C::Q_OFF + qb * C::TILE_BYTES;
                mbar_arrive_expect_tx(bar(B_QFULL + qb), C::TILE_BYTES);
                for (int dc = 0; dc < D / 64; ++dc)
                    for (int rh = 0; rh < 2; ++rh)
                        tma_load_3d(dst + dc * kRegionBytes + rh * 8192, &tmQ, bar(B_QFULL + qb), dc * 64,
                                    ui.q0 + rh * 64, ui.bh);
            }
            ++q_arms[qb];
            ++qcnt;

            // ---- key steps
            int x = -1;  // last block emitted (local units)
            for (int t = 0; t < ui.n_steps; ++t, ++g) {
                const uint32_t st = g % C::STAGES;
                if (g >= C::STAGES && !(ok = wait_warp(bar(B_SEMPTY + st), ((g / C::STAGES) - 1) & 1, ctl)))
                    break;
                StepInfo si;
                si.masked = 0;
                si.allow = 0;
                si.kmask[0] = si.kmask[1] = ~0ull;
                for (int s = 0; s < 2; ++s) {
                    int kb, y;
                    if (ui.step0 >= 0) {  // full sweep
                        if (G.b == 64) {
                            kb = 2 * (ui.step0 + t) + s;
                            y = kb < G.nb ? kb * 64 : G.n;
                        } else {
                            kb = ui.step0 + t;
                            y = kb * 128 + s * 64;
                        }
                        if (kb >= G.nb) kb = -1;
                    } else if (G.b == 64) {
                        do {
                            x = union_next(p, rc, r0, r1, wlo, whi, x);
                        } while (x < G.nb && km && !block_has_valid(p, km, x));
                        kb = x < G.nb ? x : -1;
                        y = kb >= 0 ? kb * 64 : G.n;
                    } else {
                        if (s == 0) {
                            do {
                                x = union_next(p, rc, r0, r1, wlo, whi, x);
                            } while (x < G.nb && km && !block_has_valid(p, km, x));
                        }
                        kb = x < G.nb ? x : -1;
                        y = kb >= 0 ? kb * 128 + s * 64 : G.n;
                    }
                    si.y[s] = y;
                    if (kb < 0) continue;
                    uint64_t bits = ~0ull;
                    if (km) {
                        bits = key_bits64(km, y, G.n);
                        si.masked = 1;
                        si.kmask[s] = bits;
                    }
                    if (bits == 0) continue;
                    const bool a0 = block_allowed(p, rc, r0, r1, ui.j0, 0, kb);
                    const bool a1 = (G.b == 64) ? block_allowed(p, rc, r0, r1, ui.j1, 1, kb) : a0;
                    si.allow |= (a0 ? 1u : 0u) << (2 * s);
                    si.allow |= (a1 ? 1u : 0u) << (2 * s + 1);
                }
                if (lane == 0) {
                    steps[st] = si;
                    const uint32_t kdst = sbase + C::K_OFF + st * C::TILE_BYTES;
                    const uint32_t vdst = sbase + C::V_OFF + st * C::TILE_BYTES;
                    mbar_arrive_expect_tx(bar(B_KFULL + st), C::TILE_BYTES);
                    for (int s = 0; s < 2; ++s)
                        for (int dc = 0; dc < D / 64; ++dc)
                            tma_load_3d(kdst + dc * kRegionBytes + s * 8192, &tmK, bar(B_KFULL + st), dc * 64,
                                        si.y[s], ui.bh);
                    mbar_arrive_expect_tx(bar(B_VFULL + st), C::TILE_BYTES);
                    for (int s = 0; s < 2; ++s)
                        for (int dc = 0; dc < D / 64; ++dc)
                            tma_load_3d(vdst + dc * kRegionBytes + s * 8192, &tmV, bar(B_VFULL + st), dc * 64,
                                        si.y[s], ui.bh);
                }
                ++kv_arms[st];
            }
        }
        if (!ok && lane == 0) {  // abort: wait for the copies this CTA still has in flight
            for (int i = 0; i < C::STAGES; ++i)
                if (kv_arms[i]) {
                    wait_drain(bar(B_KFULL + i), (kv_arms[i] - 1) & 1, G.wait_limit);
                    wait_drain(bar(B_VFULL + i), (kv_arms[i] - 1) & 1, G.wait_limit);
                }
            for (int i = 0; i < C::NQ; ++i)
                if (q_arms[i]) wait_drain(bar(B_QFULL + i), (q_arms[i] - 1) & 1, G.wait_limit);
        }
    } else if (warp == 1) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = idesc_bf16(128, kBN, false);
            constexpr uint32_t idesc_pv = idesc_bf16(128, D, true);
            uint32_t g = 0, qcnt = 0;
            int pend = -1;
            bool pend_first = false;
            bool ok = true;
            auto issue_pv = [&](uint32_t h, bool first) -> bool {
                const uint32_t st = h % C::STAGES, pb = h & 1;
                if (!wait_one(bar(B_PFULL + pb), (h >> 1) & 1, ctl)) return false;
                if (!wait_one(bar(B_VFULL + st), (h / C::STAGES) & 1, ctl)) return false;
                tc_fence_after();
                const uint32_t pa = sbase + C::P_OFF + pb * C::P_BYTES;
                const uint32_t va = sbase + C::V_OFF + st * C::TILE_BYTES;
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t a = desc_sw128(pa + (kk >> 2) * kRegionBytes + (kk & 3) * 32, 16);
                    const uint64_t b = desc_sw128(va + kk * 2048, kRegionBytes);
                    mma_bf16_ss(tmem + C::O_COL, a, b, idesc_pv, (first && kk == 0) ? 0u : 1u);
                }
                mma_commit(bar(B_SEMPTY + st));
                mma_commit(bar(B_PVDONE + pb));
                return true;
            };
            for (uint32_t ui_idx = 0; ok; ++ui_idx) {
                const uint32_t slot = ui_idx % kNU;
                if (!(ok = wait_one(bar(B_UFULL + slot), (ui_idx / kNU) & 1, ctl))) break;
                const int kind = ring[slot].kind;
                const int n_steps = ring[slot].n_steps;
                mbar_arrive(bar(B_UEMPTY + slot));
                if (kind == kUnitEnd) break;
                if (n_steps == 0) continue;
                const uint32_t qb = qcnt % C::NQ;
                if (!(ok = wait_one(bar(B_QFULL + qb), (qcnt / C::NQ) & 1, ctl))) break;
                tc_fence_after();
                const uint32_t qa = sbase + C::Q_OFF + qb * C::TILE_BYTES;
                for (int t = 0; t < n_steps; ++t, ++g) {
                    const uint32_t st = g % C::STAGES, sb = g & 1;
                    if (!(ok = wait_one(bar(B_KFULL + st), (g / C::STAGES) & 1, ctl))) break;
                    tc_fence_after();
                    const uint32_t ka = sbase + C::K_OFF + st * C::TILE_BYTES;
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kRegionBytes + (kk & 3) * 32;
                        mma_bf16_ss(tmem + sb * kBN, desc_sw128(qa + off, 16), desc_sw128(ka + off, 16), idesc_qk,
                                    kk > 0 ? 1u : 0u);
                    }
                    mma_commit(bar(B_SFULL + sb));
                    if (t == n_steps - 1) mma_commit(bar(B_QEMPTY + qb));
                    if (pend >= 0 && !(ok = issue_pv((uint32_t)pend, pend_first))) break;
                    pend = (int)g;
                    pend_first = (t == 0);
                }
                ++qcnt;
            }
            if (ok && pend >= 0) issue_pv((uint32_t)pend, pend_first);
            // drain: every MMA issued by this thread has completed once this arrives
            mma_commit(bar(B_DRAIN));
            wait_drain(bar(B_DRAIN), 0, G.wait_limit);
        }
    } else if (warp >= 4) {
        // ================================================================ softmax / epilogue
        const int tid = threadIdx.x - kSoftmaxThread0;  // query row within the tile
        const uint32_t lane_base = (uint32_t)((warp - 4) * 32) << 16;
        const int hf = (G.b == 64) ? (tid >> 6) : 0;
        const float sl2 = G.scale_log2;
        uint32_t g = 0;
        for (uint32_t ui_idx = 0;; ++ui_idx) {
            const uint32_t slot = ui_idx % kNU;
            if (!wait_warp(bar(B_UFULL + slot), (ui_idx / kNU) & 1, ctl)) break;
            const UnitInfo ui = ring[slot];
            mbar_arrive(bar(B_UEMPTY + slot));
            if (ui.kind == kUnitEnd) break;
            const int beta = ui.bh / G.H;
            const int row = ui.q0 + tid;
            const bool row_valid = row < G.n && (!p.key_mask || p.key_mask[(size_t)beta * G.n + row] != 0);
            float m_ref = -CUDART_INF_F, l = 0.f;
            bool ok = true;
            for (int t = 0; t < ui.n_steps; ++t, ++g) {
                const uint32_t st = g % C::STAGES, sb = g & 1, pb = g & 1;
                if (!(ok = wait_warp(bar(B_KFULL + st), (g / C::STAGES) & 1, ctl))) break;
                if (!(ok = wait_warp(bar(B_SFULL + sb), (g >> 1) & 1, ctl))) break;
                tc_fence_after();
                const StepInfo si = steps[st];
                const bool w0 = (si.allow >> (0 + hf)) & 1u;  // warp-uniform
                const bool w1 = (si.allow >> (2 + hf)) & 1u;
                float s[4][32];
                const uint32_t sa = tmem + lane_base + sb * kBN;
                if (w0) {
                    tmem_ld32(sa + 0, s[0]);
                    tmem_ld32(sa + 32, s[1]);
                }
                if (w1) {
                    tmem_ld32(sa + 64, s[2]);
                    tmem_ld32(sa + 96, s[3]);
                }
                tmem_wait_ld();
                const bool u0 = w0 && row_valid, u1 = w1 && row_valid;
                if (si.masked) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        if (!((si.kmask[0] >> c) & 1ull)) s[c >> 5][c & 31] = -CUDART_INF_F;
                        if (!((si.kmask[1] >> c) & 1ull)) s[2 + (c >> 5)][c & 31] = -CUDART_INF_F;
                    }
                }
                float mx = -CUDART_INF_F;
                if (u0) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) mx = fmaxf(mx, fmaxf(s[0][c], s[1][c]));
                }
                if (u1) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) mx = fmaxf(mx, fmaxf(s[2][c], s[3][c]));
                }
                const float m_new = fmaxf(m_ref, mx * sl2);
                bool resc = false;
                float alpha = 1.f;
                if (m_new > m_ref + kRescaleLog2) {
                    alpha = ex2(m_ref - m_new);
                    resc = (m_ref != -CUDART_INF_F) && t > 0;
                    l *= alpha;
                    m_ref = m_new;
                }
                const float neg_m = (m_ref == -CUDART_INF_F) ? 0.f : -m_ref;
                uint32_t pk[64];
                float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const bool use = half == 0 ? u0 : u1;
#pragma unroll
                    for (int c = 0; c < 64; c += 2) {
                        float p0 = 0.f, p1 = 0.f;
                        if (use) {
                            p0 = ex2(fmaf(s[2 * half + (c >> 5)][c & 31], sl2, neg_m));
                            p1 = ex2(fmaf(s[2 * half + (c >> 5)][(c & 31) + 1], sl2, neg_m));
                        }
                        ls0 += p0;
                        ls1 += p1;
                        __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
                        pk[half * 32 + (c >> 1)] = *reinterpret_cast<uint32_t *>(&b2);
                    }
                }
                l += ls0 + ls1;
                // P buffer pb is free once PV of step g-2 completed
                if (g >= 2 && !(ok = wait_warp(bar(B_PVDONE + pb), ((g - 2) >> 1) & 1, ctl))) break;
                uint8_t *pbuf = smem + C::P_OFF + pb * C::P_BYTES;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        uint4 v = make_uint4(pk[half * 32 + ch * 4 + 0], pk[half * 32 + ch * 4 + 1],
                                             pk[half * 32 + ch * 4 + 2], pk[half * 32 + ch * 4 + 3]);
                        *reinterpret_cast<uint4 *>(pbuf + half * kRegionBytes + tid * 128 +
                                                   ((ch ^ (tid & 7)) << 4)) = v;
                    }
                }
                fence_proxy_async_smem();
                if (__any_sync(kFull, resc)) {
                    if (!(ok = wait_warp(bar(B_PVDONE + ((g - 1) & 1)), ((g - 1) >> 1) & 1, ctl))) break;
                    tc_fence_after();
                    const float a = resc ? alpha : 1.f;
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) {
                        float o[32];
                        tmem_ld32(tmem + lane_base + C::O_COL + cc * 32, o);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= a;
                        tmem_st32(tmem + lane_base + C::O_COL + cc * 32, o);
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                mbar_arrive(bar(B_PFULL + pb));
            }
            if (!ok) break;
            // ---------------------------------------------------- epilogue
            if (ui.n_steps > 0) {
                const uint32_t gl = g - 1;
                if (!wait_warp(bar(B_PVDONE + (gl & 1)), (gl >> 1) & 1, ctl)) break;
                tc_fence_after();
            }
            const bool have = ui.n_steps > 0;
            if (ui.kind == kUnitDirect) {
                const float inv = (row_valid && l > 0.f) ? 1.f / l : 0.f;
                __nv_bfloat16 *orow = p.O + ((size_t)ui.bh * G.n + (row < G.n ? row : 0)) * D;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    float o[32];
                    if (have) {
                        tmem_ld32(tmem + lane_base + C::O_COL + cc * 32, o);
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
                            for (int e = 0; e < 4; ++e) {
                                __nv_bfloat162 b2 =
                                    __floats2bfloat162_rn(o[q * 8 + 2 * e] * inv, o[q * 8 + 2 * e + 1] * inv);
                                w4[e] = *reinterpret_cast<uint32_t *>(&b2);
                            }
                            *reinterpret_cast<uint4 *>(orow + cc * 32 + q * 8) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        }
                    }
                }
            } else {
                // split chunk: publish this row's partial, last arrival merges the row
                const size_t prow = ((size_t)ui.tile_slot * G.splits + ui.chunk) * kBM + tid;
                float *po = p.ws.part_o + prow * D;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    float o[32];
                    if (have) {
                        tmem_ld32(tmem + lane_base + C::O_COL + cc * 32, o);
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
                __stcg(p.ws.part_ml + prow, make_float2(row_valid ? m_ref : -CUDART_INF_F, row_valid ? l : 0.f));
                __threadfence();
                unsigned *cnt = p.ws.row_cnt + (size_t)ui.tile_slot * kBM + tid;
                const unsigned prev = atomicAdd(cnt, 1u);
                if (prev == (unsigned)(ui.nchunks - 1)) {
                    __threadfence();
                    float M = -CUDART_INF_F;
                    for (int c = 0; c < ui.nchunks; ++c) {
                        const float2 ml = __ldcg(p.ws.part_ml + ((size_t)ui.tile_slot * G.splits + c) * kBM + tid);
                        M = fmaxf(M, ml.x);
                    }
                    float acc[D];
#pragma unroll
                    for (int i = 0; i < D; ++i) acc[i] = 0.f;
                    float L = 0.f;
                    for (int c = 0; c < ui.nchunks; ++c) {
                        const size_t pr = ((size_t)ui.tile_slot * G.splits + c) * kBM + tid;
                        const float2 ml = __ldcg(p.ws.part_ml + pr);
                        if (ml.y == 0.f || M == -CUDART_INF_F) continue;
                        const float wgt = ex2(ml.x - M);
                        L += wgt * ml.y;
                        const float *src = p.ws.part_o + pr * D;
#pragma unroll
                        for (int i = 0; i < D; i += 4) {
                            const float4 v = __ldcg(reinterpret_cast<const float4 *>(src + i));
                            acc[i] = fmaf(wgt, v.x, acc[i]);
                            acc[i + 1] = fmaf(wgt, v.y, acc[i + 1]);
                            acc[i + 2] = fmaf(wgt, v.z, acc[i + 2]);
                            acc[i + 3] = fmaf(wgt, v.w, acc[i + 3]);
                        }
                    }
                    const float inv = (row_valid && L > 0.f) ? 1.f / L : 0.f;
                    if (row < G.n) {
                        __nv_bfloat16 *orow = p.O + ((size_t)ui.bh * G.n + row) * D;
#pragma unroll
                        for (int i = 0; i < D; i += 8) {
                            uint32_t w4[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[i + 2 * e] * inv, acc[i + 2 * e + 1] * inv);
                                w4[e] = *reinterpret_cast<uint32_t *>(&b2);
                            }
                            *reinterpret_cast<uint4 *>(orow + i) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                        }
                    }
                    atomicExch(cnt, 0u);  // ready for the next call
                }
            }
            tc_fence_before();
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned done = atomicAdd(p.ws.counters + 1, 1u);
        if (done == gridDim.x - 1) {  // last CTA: reset the scheduler for the next call
            atomicExch(p.ws.counters, 0u);
            atomicExch(p.ws.counters + 1, 0u);
        }
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
    G.steps_full = (p.n + kBN - 1) / kBN;
    int s0 = (G.steps_full + kTargetChunkSteps - 1) / kTargetChunkSteps;
    if (s0 > cfg.max_splits) s0 = cfg.max_splits;
    if (s0 < 1) s0 = 1;
    G.steps_per_chunk = (G.steps_full + s0 - 1) / s0;
    G.splits = (G.steps_full + G.steps_per_chunk - 1) / G.steps_per_chunk;
    const long long BH = (long long)p.B * p.H;
    G.n_split_units = (int)(BH * G.gtiles * G.splits);
    G.total_units = G.n_split_units + (int)(BH * (G.tiles - G.gtiles));
    G.scale_log2 = 1.4426950408889634f / sqrtf((float)p.d);
    G.wait_limit = cfg.wait_limit;
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
    auto kern = bigbird_tc_fwd<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::ALLOC_BYTES);
    if (e != cudaSuccess) return e;
    int grid = cfg.grid_ctas;
    if (grid > prm.geo.total_units) grid = prm.geo.total_units;
    if (grid < 1) grid = 1;
    kern<<<grid, kThreads, Cfg<D>::ALLOC_BYTES, stream>>>(mq, mk, mv, prm);
    return cudaGetLastError();
}

}  // namespace

size_t tc_workspace_bytes(const Problem &p, const TcConfig &cfg) {
    if (p.kind != kBigBird) return 256;
    return ws_layout(bigbird_geometry(p, cfg), p.d).total;
}

size_t tc_workspace_counter_bytes(const Problem &p, const TcConfig &cfg) {
    if (p.kind != kBigBird) return 256;
    const WsLayout L = ws_layout(bigbird_geometry(p, cfg), p.d);
    return L.part_o ? L.part_o : L.total;
}

cudaError_t launch_tc(const Problem &p, const TcConfig &cfg, void *ws, size_t ws_bytes, cudaStream_t stream,
                      int *launches) {
    *launches = 0;
    if (p.kind != kBigBird) return cudaErrorNotSupported;
    cudaError_t e = (p.d == 64) ? launch_bigbird<64>(p, cfg, ws, ws_bytes, stream)
                                : launch_bigbird<128>(p, cfg, ws, ws_bytes, stream);
    if (e == cudaSuccess) *launches = 1;
    return e;
}

}  // namespace sa
