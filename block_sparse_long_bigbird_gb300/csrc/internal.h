// Internal declarations shared by the host API and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "sparse_attn.h"

namespace sa {

enum PatternKind { kBigBird = 0, kLongformer = 1 };

// Device status bits latched by kernels (OR-ed into the per-device word).
// Largest accepted Longformer dilation (window stride dilation + 1 <= 64).
constexpr int kMaxDilation = 63;

enum DeviceStatusBits : unsigned int {
    kDevTimeout = 1u << 0,
    kDevBadIndex = 1u << 1,
};

// One attention call, as validated by the host API.
struct Problem {
    int kind;
    const void *Q, *K, *V;
    void *O;
    int B, H, n, d;
    // BigBird-ITC
    int b, g, w, r;
    const int32_t *rand_idx;
    // Longformer
    int window;
    const int32_t *global_idx;
    int n_global;
    const int32_t *dilation;  // device [H] or NULL (dilated sliding window)
    int causal;               // autoregressive mode
    // separate projections for global attention (NULL: global rows use Q, K, V)
    const void *Qg, *Kg, *Vg;
    // both
    const uint8_t *key_mask;
    unsigned int *status;  // device status word
    // backward only: dO is the upstream gradient; row_stats holds
    // 2 * B * H * stats_stride(n) floats of scratch (per-row log2-domain
    // log-sum-exp, then per-row D = sum_j P_ij dO_i . V_j), rows of each head
    // stats_stride(n) apart.
    const void *dO;
    void *dQ, *dK, *dV;
    float *row_stats;
    // Longformer backward with separate global projections: which query rows
    // take part (0 all, 1 the non-global rows, 2 the global rows only)
    int row_set;
    // Longformer forward: the scratch holds room for residue-class copies of
    // Q, K and V (3 * B * H * n * d elements), so dilated heads whose stride
    // divides n run as plain windows on those copies
    int class_perm;
};

// Row stride of the backward's per-row statistics: n rounded up to 64, so that
// every 64-row chunk of them starts 256-B aligned.
__host__ __device__ inline int stats_stride(int n) { return (n + 63) & ~63; }

// Exact SIMT kernels (fp32 arithmetic; bf16 or fp32 storage).
cudaError_t launch_simt(const Problem &p, sa_dtype dtype, cudaStream_t stream, int *launches);

// Exact SIMT backward (two launches: row pass for dQ and the row statistics,
// then key pass for dK and dV).
cudaError_t launch_simt_bwd(const Problem &p, sa_dtype dtype, cudaStream_t stream, int *launches);

// Tensor-core (tcgen05/TMEM/TMA) kernels for bf16.
struct TcConfig {
    int grid_ctas;     // persistent grid size
    int max_splits;    // split-KV upper bound for global row tiles
    int chunk_keys;    // split-KV target keys per chunk (0: the kernel's default)
    long long wait_limit;
};
// Tensor-core backward (bf16): row pass then key pass, two launches.
cudaError_t launch_tc_bwd(const Problem &p, const TcConfig &cfg, cudaStream_t stream, int *launches);
size_t tc_workspace_bytes(const Problem &p, const TcConfig &cfg);
// Leading bytes of the tensor-core scratch that must be zero when a call
// starts (scheduler and merge counters).
size_t tc_workspace_counter_bytes(const Problem &p, const TcConfig &cfg);
cudaError_t launch_tc(const Problem &p, const TcConfig &cfg, void *workspace, size_t ws_bytes,
                      cudaStream_t stream, int *launches);
// Longformer parts of the above (tensor-core Longformer translation unit).
size_t tc_longformer_workspace_bytes(const Problem &p, const TcConfig &cfg);
size_t tc_longformer_counter_bytes(const Problem &p, const TcConfig &cfg);
cudaError_t launch_tc_longformer(const Problem &p, const TcConfig &cfg, void *workspace, size_t ws_bytes,
                                 cudaStream_t stream, int *launches);

}  // namespace sa
