// Small helpers shared by the exact SIMT kernels (forward and backward).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace sa {
namespace simt {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void store_val(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_val(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// First index t in sorted idx[0..cnt) with idx[t] >= key.
__device__ __forceinline__ int lower_bound_i32(const int32_t *idx, int cnt, int key) {
    int lo = 0, hi = cnt;
    while (lo < hi) {
        int mid = (lo + hi) >> 1;
        if (idx[mid] < key) lo = mid + 1; else hi = mid;
    }
    return lo;
}

}  // namespace simt
}  // namespace sa
