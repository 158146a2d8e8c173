// Host-side choice of the split-KV chunking of global tiles, shared by the
// BigBird and Longformer launchers (kept apart from the kernel source: it
// decides how work is cut, not what a launch computes).
#pragma once

#include "tc_kernel.cuh"

namespace sa {
namespace {

constexpr int kSplitRefSms = 152;  // GB300 SMs: the split choice assumes a full-chip grid

// Split-KV chunks of a global tile. A global tile sweeps every key in one unit,
// so unsplit it can outlast the rest of the call; it is cut into chunks when
// its sweep is longer than three quarters of the average work of one tile
// slot (tiles in flight on a full-chip grid), each chunk about half of it.
// (Measured: the n = 4096 Longformer call, whose 64-step sweeps are 0.97 of a
// slot's work, gains 19% from two chunks; the BigBird-ETC n = 4352 call at
// 0.55 loses 13% from them.) `local_steps`:
// estimated steps of all other units. The choice depends only on the sizes and
// the options (not on the grid actually launched), so the scratch a call needs
// is known before the device is queried. SA_OPT_CHUNK_KEYS overrides the
// chunk length, SA_OPT_MAX_SPLITS bounds the count.
inline void choose_splits(Geometry &G, long long local_steps, int kb, int tiles_per_cta, int chunk_keys,
                          int max_splits) {
    const long long BH = (long long)G.B * G.H;
    int target = G.steps_full;
    if (chunk_keys > 0) {
        target = chunk_keys / kb;
    } else {
        const long long avg = (local_steps + BH * G.gtiles * G.steps_full) / ((long long)kSplitRefSms * tiles_per_cta);
        if (4LL * G.steps_full > 3LL * avg) target = (int)(avg / 2);
    }
    if (target < 8) target = 8;
    int s0 = (G.steps_full + target - 1) / target;
    if (s0 > max_splits) s0 = max_splits;
    if (s0 < 1) s0 = 1;
    G.steps_per_chunk = (G.steps_full + s0 - 1) / s0;
    G.splits = (G.steps_full + G.steps_per_chunk - 1) / G.steps_per_chunk;
}

}  // namespace
}  // namespace sa
