// Host pattern builder: BigBird's per-head random key blocks.
//
// "Big Bird", Sec. 2 and App. E Tab. 8 say each query block sees r = 3 random
// key blocks; the blog summary (Sec. 2.1, Sec. 4.2(3)) adds that these are
// gathered. No generator is named, so the draw is fixed as: SplitMix64
// (Steele, Lea & Flood, OOPSLA 2014) as one sequential stream from `seed`,
// rows h-major then query block; candidates are the ascending non-global,
// non-window key blocks; partial Fisher-Yates draws; chosen blocks sorted,
// -1 padded. Global query blocks draw nothing.
#include <stdint.h>

#include <algorithm>
#include <vector>

#include "sparse_attn.h"

namespace {

struct SplitMix64 {
    uint64_t state;
    explicit SplitMix64(uint64_t seed) : state(seed) {}
    uint64_t next() {
        state += 0x9E3779B97F4A7C15ull;
        uint64_t z = state;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
        return z ^ (z >> 31);
    }
};

}  // namespace

extern "C" sa_status build_bigbird_pattern(uint64_t seed, int H, int n, int b, int g, int w, int r,
                                           int32_t *out_host) {
    if ((!out_host && r > 0) || H < 1 || b < 1 || n < b || n % b != 0 || g < 0 || w < 1 || (w % 2) == 0 || r < 0)
        return SA_ERR_INVALID_ARG;
    const int nb = n / b;
    if (g > nb) return SA_ERR_INVALID_ARG;
    const int half = w / 2;
    SplitMix64 gen(seed);
    std::vector<int32_t> cand;
    cand.reserve(nb);
    for (int h = 0; h < H; ++h) {
        for (int j = 0; j < nb; ++j) {
            int32_t *row = out_host + ((size_t)h * nb + j) * r;
            for (int t = 0; t < r; ++t) row[t] = -1;
            if (j < g) continue;
            cand.clear();
            for (int kb = g; kb < nb; ++kb) {
                const int dist = kb > j ? kb - j : j - kb;
                if (dist > half) cand.push_back(kb);
            }
            const int m = (int)cand.size();
            const int k = std::min(r, m);
            for (int t = 0; t < k; ++t) {
                const uint64_t u = gen.next();
                const int idx = t + (int)(u % (uint64_t)(m - t));
                std::swap(cand[t], cand[idx]);
            }
            std::sort(cand.begin(), cand.begin() + k);
            for (int t = 0; t < k; ++t) row[t] = cand[t];
        }
    }
    return SA_OK;
}
