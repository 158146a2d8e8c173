/*
 * sparse_attn.h - C ABI of the GB300 (sm_103a) sparse long-sequence attention
 * forward library: BigBird-ITC block-sparse attention and Longformer
 * sliding-window + global attention.
 *
 * What is computed (both patterns), per batch entry beta and head h:
 *
 *     O[i,:] = sum_{j in N(i)} softmax_j( Q[i,:] . K[j,:] / sqrt(d) ) V[j,:]
 *
 * i.e. the generalised attention Attn_D of "Big Bird: Transformers for
 * Longer Sequences", Sec. 2, Eq. (AT), for one head and without the residual
 * term, with the scaled dot-product form of "Longformer: The Long-Document
 * Transformer", Sec. 3.1, Eq. (1). N(i) is the pattern's neighbourhood of
 * query i intersected with the valid (unpadded) keys. A padded query row, or
 * a row whose neighbourhood holds no valid key, is written as zeros.
 *
 * Conventions shared by every entry point:
 *  - Tensors Q, K, V, O are device pointers to contiguous row-major
 *    [B][H][n][d] arrays, d innermost, 16-byte aligned, all of the same dtype
 *    (sa_dtype). O must not alias Q, K or V.
 *  - The caller owns every buffer it passes; the library never frees caller
 *    memory and keeps no pointer to it after the call returns.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream). The returned status reports argument errors found on the host
 *    before anything is launched, and launch errors. Conditions the device
 *    detects (an out-of-range index in a table, a pipeline wait that ran past
 *    its bound) are latched in a per-device status word; read and clear it
 *    with sa_get_last_device_status().
 *  - Results are deterministic: identical inputs give bitwise-identical O
 *    (no floating-point atomics; split reductions merge in a fixed order).
 *  - The device that runs a call is the calling thread's current CUDA device.
 *  - Scratch is per device, not per stream: every tensor-core call on a
 *    device (forward and backward, whatever its stream) uses the same
 *    scratch region (library-owned, or the one set with sa_set_workspace).
 *    Calls on one device must therefore be stream-ordered: issue them on one
 *    stream, or order the streams with events. Two calls that run at the same
 *    time on unordered streams race on the scheduler and merge counters and
 *    give wrong outputs (or a bounded wait expires: SA_ERR_TIMEOUT). The same
 *    holds for the host-buffer entry points, which run each chunk as an
 *    ordinary device call on the caller's stream.
 */
#ifndef SPARSE_ATTN_H
#define SPARSE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque stream handle, ABI-identical to cudaStream_t. */
typedef struct CUstream_st *sa_stream_t;

typedef enum {
    SA_OK = 0,
    SA_ERR_INVALID_ARG = 1, /* a size, a flag or a pointer is outside the contract */
    SA_ERR_UNSUPPORTED = 2, /* valid arguments this build does not run (e.g. no sm_103a device) */
    SA_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a kernel launch failed */
    SA_ERR_TIMEOUT = 4,     /* device: a bounded pipeline wait expired; the kernel exited cleanly */
    SA_ERR_BAD_INDEX = 5    /* device: rand_idx / global_idx held an out-of-range or unsorted entry */
} sa_status;

typedef enum {
    SA_BF16 = 0, /* bf16 inputs/outputs; fp32 softmax and accumulation (tensor cores) */
    SA_FP32 = 1  /* fp32 inputs/outputs; fp32 arithmetic throughout (no TF32) */
} sa_dtype;

/*
 * build_bigbird_pattern - host-only. Draw BigBird's per-head random key blocks.
 *
 * Source: "Big Bird", Sec. 2 (random attention: each query attends r random
 * keys) and App. E Tab. 8 (r = 3b tokens, i.e. r blocks of size b); the blog
 * summary of BigBird, Sec. 2.1 and Sec. 4.2(3). The pages name no generator,
 * so the draw is fixed here: one SplitMix64 stream (Steele, Lea & Flood 2014)
 * started at `seed`; rows visited h = 0..H-1, then j = g..nb-1 (nb = n / b);
 * the candidates of row j are the ascending key blocks kb in [0, nb) with
 * kb >= g and |kb - j| > w / 2 (m of them); k = min(r, m) partial
 * Fisher-Yates draws, draw t swapping position t with t + (u mod (m - t));
 * the k chosen blocks are stored sorted ascending, then -1 up to r. Global
 * rows (j < g) hold -1 only.
 *
 * out_host: caller-owned HOST buffer of H * (n / b) * r int32, layout [H][nb][r]
 *   (may be NULL when r == 0: there is nothing to write).
 * Errors: SA_ERR_INVALID_ARG if out_host is NULL with r > 0, H < 1, b < 1, n < b,
 * n % b != 0, g < 0, g > nb, w < 1, w even, or r < 0.
 */
sa_status build_bigbird_pattern(uint64_t seed, int H, int n, int b, int g, int w, int r,
                                int32_t *out_host);

/*
 * bigbird_attn_fwd - BigBird-ITC block-sparse attention forward.
 *
 * Source: "Big Bird", Sec. 2 (Eq. AT; random, window and global components),
 * App. D (blockified pattern on blocks of b tokens, Eq. 13 and Fig. 6: the
 * block-sparse product equals the sparse matrix of Fig. 3(d)), App. E Tab. 8
 * (ITC: g = 2b, w = 3b, r = 3b tokens); blog summary Sec. 2.1-2.3.
 *
 * Query block qb = i / b sees key block kb = j / b iff qb < g (global rows
 * attend everything), or kb < g (everyone attends the global blocks), or
 * |qb - kb| <= w / 2 (window of w blocks, clipped at the sequence ends), or kb
 * is listed in rand_idx[h][qb][:].
 *
 * BigBird-ETC ("Big Bird", Sec. 2: g added global tokens such as CLS; App. E:
 * r = 0) runs through this call: place the added tokens first, pad them to
 * ceil(g_tokens / b) whole blocks with tokens that key_mask marks invalid, and
 * pass g = ceil(g_tokens / b), r = 0. The padding rows come out zero.
 *
 * Sizes: B, H >= 1; d in {64, 128}; b in {64, 128}; n a multiple of b;
 * 0 <= g <= n / b; w odd and >= 1; r >= 0.
 * rand_idx: DEVICE int32 [H][n/b][r] (e.g. from build_bigbird_pattern, copied
 *   to the device), shared by all batch entries; -1 entries are ignored. May
 *   be NULL when r == 0. An entry outside [-1, n/b) is skipped and latches
 *   SA_ERR_BAD_INDEX.
 * key_mask: DEVICE uint8 [B][n], nonzero = valid token, or NULL (all valid);
 *   16-byte aligned.
 * dtype: SA_BF16 (tensor-core path) or SA_FP32 (exact fp32 SIMT path).
 * Scratch: global query blocks may be split across CTAs (split-KV) with a
 *   fixed-order merge; their partials live in the workspace (see
 *   sa_bigbird_workspace_bytes / sa_set_workspace).
 * Errors: SA_ERR_INVALID_ARG for any size or pointer outside the contract,
 *   SA_ERR_UNSUPPORTED if the current device is not sm_103, SA_ERR_CUDA if a
 *   launch fails.
 */
sa_status bigbird_attn_fwd(const void *Q, const void *K, const void *V, void *O,
                           int B, int H, int n, int d, int b, int g, int w, int r,
                           const int32_t *rand_idx, const uint8_t *key_mask,
                           sa_dtype dtype, sa_stream_t stream);

/*
 * longformer_attn_fwd - Longformer sliding-window + symmetric global attention.
 *
 * Source: "Longformer", Sec. 3.1 (sliding window: window / 2 tokens on each
 * side; global attention is symmetric: a global token attends every token and
 * every token attends it) and Eq. (1); Sec. 3.2 / App. A (banded product).
 *
 * Token i sees token j iff i or j is global, or |i - j| <= window / 2.
 *
 * Sizes: B, H >= 1; n >= 1; d in {64, 128}; window even and >= 0.
 * global_idx: DEVICE int32 [n_global], strictly increasing positions in
 *   [0, n); may be NULL when n_global == 0. Entries that break the order or
 *   the range are skipped and latch SA_ERR_BAD_INDEX.
 * n_global: 0 <= n_global <= n.
 * key_mask: DEVICE uint8 [B][n] or NULL, as for bigbird_attn_fwd.
 * Errors: as for bigbird_attn_fwd.
 */
sa_status longformer_attn_fwd(const void *Q, const void *K, const void *V, void *O,
                              int B, int H, int n, int d, int window,
                              const int32_t *global_idx, int n_global,
                              const uint8_t *key_mask, sa_dtype dtype, sa_stream_t stream);

/*
 * longformer_attn_fwd_ex - longformer_attn_fwd with the dilated sliding window
 * and the autoregressive mode.
 *
 * Source: "Longformer", Sec. 3.1 and Fig. 2(c) (dilated sliding window: gaps
 * of size `dilation` between the window positions; per-head dilation as in
 * Tab. 12, where dilation 0 is the plain window) and App. B (autoregressive
 * mode: each token attends to previous tokens only).
 *
 * Token i sees token j iff (i or j is global, or j = i + k (dilation[h] + 1)
 * for some |k| <= window / 2) and, when `causal` is nonzero, j <= i (global
 * tokens included: nothing after the query is ever seen).
 *
 * dilation: DEVICE int32 [H] or NULL (all heads 0). Values outside [0, 63]
 *   latch SA_ERR_BAD_INDEX and are taken as 0.
 * causal: 0 or 1.
 * Scratch: with dilation set and no global tokens, key mask or separate
 *   projections, the bf16 call also uses 3 * B * H * n * d elements of scratch
 *   for residue-class copies of Q, K and V (a dilated head whose stride
 *   dilation + 1 divides n then runs as a plain window on its copies). The
 *   library-owned scratch grows to hold them; a caller-owned region
 *   (sa_set_workspace) too small for them is used without them, at the cost of
 *   computing those heads over their whole dilated reach. The result does not
 *   depend on which is taken beyond rounding order.
 * Other arguments, layout, ownership and errors: as for longformer_attn_fwd,
 * which is this call with dilation NULL and causal 0.
 */
sa_status longformer_attn_fwd_ex(const void *Q, const void *K, const void *V, void *O,
                                 int B, int H, int n, int d, int window,
                                 const int32_t *dilation, int causal,
                                 const int32_t *global_idx, int n_global,
                                 const uint8_t *key_mask, sa_dtype dtype, sa_stream_t stream);

/*
 * longformer_attn_fwd_gproj - longformer_attn_fwd_ex with separate projections
 * for global attention.
 *
 * Source: "Longformer", Sec. 3.1, "Linear Projections for Global Attention":
 * one set of projections (Q, K, V) computes the sliding-window attention and a
 * second set (Qg, Kg, Vg) the global attention. Reading taken here: the row of
 * a global token is computed from Qg against Kg and Vg over every key it may
 * see; every other row uses Q, K and V throughout, its scores against global
 * keys included. With Qg = Q, Kg = K, Vg = V the result is that of
 * longformer_attn_fwd_ex.
 *
 * Qg, Kg, Vg: DEVICE [B][H][n][d], same dtype and alignment as Q, K, V; all
 *   three NULL (then this is longformer_attn_fwd_ex) or all three set; none may
 *   alias O.
 * Other arguments, layout, ownership and errors: as for longformer_attn_fwd_ex.
 */
sa_status longformer_attn_fwd_gproj(const void *Q, const void *K, const void *V,
                                    const void *Qg, const void *Kg, const void *Vg, void *O,
                                    int B, int H, int n, int d, int window,
                                    const int32_t *dilation, int causal,
                                    const int32_t *global_idx, int n_global,
                                    const uint8_t *key_mask, sa_dtype dtype, sa_stream_t stream);

/*
 * bigbird_attn_fwd_host / longformer_attn_fwd_host - the forward on HOST
 * buffers, with the host<->device copies pipelined against the computation.
 * (The pages have no counterpart: this is a deployment variant of the same
 * computation for inputs that live in host memory.)
 *
 * The (batch, head) pairs are processed in about four chunks per call: whole
 * batch entries, or consecutive heads of one batch entry when an entry is
 * more than a chunk. Chunk k's Q, K, V are copied to the device on a
 * library-owned stream while chunk k - 1 computes on `stream` and chunk k - 2's
 * O is copied back on a second library-owned stream; two device staging sets
 * alternate. Each chunk is an ordinary device-side call
 * (bigbird_attn_fwd / longformer_attn_fwd_ex) on a slice, so results are
 * bitwise those of the device entry points.
 *
 * Q, K, V, O: HOST [B][H][n][d] arrays of the dtype. Page-locked memory
 *   (cudaHostAlloc, cudaHostRegister) is needed for the copies to overlap;
 *   pageable memory works but the copies then run one after another.
 * rand_idx, global_idx, dilation, key_mask: HOST arrays with the layouts of
 *   the device entry points (copied once per call).
 * Completion: asynchronous on `stream`; O is complete once `stream` has
 *   completed the work issued by this call. The caller must not modify Q, K,
 *   V or read O before then.
 * Scratch: device staging of 2 x 4 x (heads per chunk) x n x d elements plus
 *   the tables, allocated by the library on first use and grown on demand;
 *   plus the device entry points' own workspace.
 * Concurrency: calls from several host threads are serialised while they
 *   enqueue (they share the staging sets); on the device each call's copies
 *   wait for the previous call's last output copy.
 * Errors: as for bigbird_attn_fwd / longformer_attn_fwd_ex (NULL or aliasing
 *   tensors are SA_ERR_INVALID_ARG).
 */
sa_status bigbird_attn_fwd_host(const void *Q, const void *K, const void *V, void *O,
                                int B, int H, int n, int d, int b, int g, int w, int r,
                                const int32_t *rand_idx, const uint8_t *key_mask,
                                sa_dtype dtype, sa_stream_t stream);
sa_status longformer_attn_fwd_host(const void *Q, const void *K, const void *V, void *O,
                                   int B, int H, int n, int d, int window,
                                   const int32_t *dilation, int causal,
                                   const int32_t *global_idx, int n_global,
                                   const uint8_t *key_mask, sa_dtype dtype, sa_stream_t stream);

/*
 * bigbird_attn_bwd - gradients of bigbird_attn_fwd.
 *
 * Source: the pages train through this attention ("Big Bird", App. E.1, MLM
 * pretraining; "Longformer", Sec. 5, pretraining with gradient updates) but
 * print no backward formulas; this is the exact derivative of the forward
 * above at (Q, K, V). With P the forward's masked softmax (P_ij = 0 outside
 * N(i)) and dO the upstream gradient dL/dO:
 *
 *     D_i = sum_j P_ij (dO_i . V_j),   dS_ij = P_ij (dO_i . V_j - D_i),
 *     dQ = dS K / sqrt(d),   dK = dS^T Q / sqrt(d),   dV = P^T dO.
 *
 * P and D are recomputed from Q, K, V and dO in fp32, so the forward's
 * output O is not an argument: the result does not depend on how O was
 * rounded.
 *
 * Q, K, V, dO: DEVICE [B][H][n][d] inputs; dQ, dK, dV: DEVICE [B][H][n][d]
 *   outputs, all of one dtype, contiguous, 16-byte aligned. The outputs must
 *   not alias an input or each other. Every element of the outputs is
 *   written: padded queries get dQ = 0, padded keys dK = dV = 0.
 * Other arguments: as for bigbird_attn_fwd (same pattern, same rand_idx and
 *   key_mask as the forward call).
 * Arithmetic: fp32 softmax statistics and accumulation (bf16 inputs are
 *   widened exactly; outputs are rounded to the storage dtype).
 *   Deterministic: no atomics; every sum runs in a fixed order.
 * Scratch: 2 * B * H * n64 floats of per-row statistics in the workspace,
 *   n64 = n rounded up to a multiple of 64 (sa_attn_bwd_workspace_bytes).
 * Limits: the bf16 tensor-core kernels keep per-64-row tables in shared
 *   memory, which bounds n (d = 64: about 1.4M tokens, 500K with key padding;
 *   d = 128: about 470K, 160K with key padding; the Longformer call with
 *   padding about 300K / 97K). Beyond that the call returns
 *   SA_ERR_UNSUPPORTED before any work is queued; SA_OPT_FORCE_SIMT runs the
 *   SIMT backward, which has no such bound.
 * Errors: as for bigbird_attn_fwd, plus SA_ERR_INVALID_ARG when an output
 *   aliases an input or another output.
 */
sa_status bigbird_attn_bwd(const void *Q, const void *K, const void *V, const void *dO,
                           void *dQ, void *dK, void *dV,
                           int B, int H, int n, int d, int b, int g, int w, int r,
                           const int32_t *rand_idx, const uint8_t *key_mask,
                           sa_dtype dtype, sa_stream_t stream);

/*
 * longformer_attn_bwd - gradients of longformer_attn_fwd_ex (sliding window,
 * dilation, autoregressive mode, symmetric global attention).
 *
 * Formulas, tensors, numerics, scratch and errors as for bigbird_attn_bwd;
 * the pattern arguments (window, dilation, causal, global_idx, n_global,
 * key_mask) are those of longformer_attn_fwd_ex and must match the forward
 * call.
 */
sa_status longformer_attn_bwd(const void *Q, const void *K, const void *V, const void *dO,
                              void *dQ, void *dK, void *dV,
                              int B, int H, int n, int d, int window,
                              const int32_t *dilation, int causal,
                              const int32_t *global_idx, int n_global,
                              const uint8_t *key_mask, sa_dtype dtype, sa_stream_t stream);

/*
 * longformer_attn_bwd_gproj - gradients of longformer_attn_fwd_gproj.
 *
 * With separate projections for global attention the rows of global tokens
 * depend only on Qg, Kg, Vg and the other rows only on Q, K, V, so the six
 * gradients split by rows: dQ, dK, dV sum over the non-global rows (dQ is 0
 * on global rows), dQg, dKg, dVg over the global rows (dQg is 0 elsewhere).
 * Formulas, layouts, numerics and scratch as for longformer_attn_bwd; two
 * backward runs (four launches).
 * Errors: as for longformer_attn_bwd; every pointer is required, and no output
 *   may alias an input or another output.
 */
sa_status longformer_attn_bwd_gproj(const void *Q, const void *K, const void *V,
                                    const void *Qg, const void *Kg, const void *Vg, const void *dO,
                                    void *dQ, void *dK, void *dV, void *dQg, void *dKg, void *dVg,
                                    int B, int H, int n, int d, int window,
                                    const int32_t *dilation, int causal,
                                    const int32_t *global_idx, int n_global,
                                    const uint8_t *key_mask, sa_dtype dtype, sa_stream_t stream);

/*
 * Scratch (workspace) sizing. The split-KV partials of the global rows and the
 * kernel's work counters need device scratch. By default the library allocates
 * it once per device (cudaMalloc, zeroed) and grows it on demand; a caller that
 * manages memory itself passes a region with sa_set_workspace instead. Either
 * way one region serves every call on the device, so the calls must be
 * stream-ordered (see the conventions above). A call leaves the counters at
 * zero when it completes, also after a wait expired (the last CTA to finish
 * clears the split-merge counters an aborted CTA left set).
 * Returns the bytes one call with these sizes needs (0 if the sizes are invalid):
 * an upper bound over the window and random-block counts for BigBird. For a
 * dilated Longformer call it is the need without the optional residue-class
 * copies (see longformer_attn_fwd_ex), which add 3 * B * H * n * d elements.
 */
size_t sa_bigbird_workspace_bytes(int B, int H, int n, int d, int b, int g);
size_t sa_longformer_workspace_bytes(int B, int H, int n, int d, int n_global);
/* Scratch bytes of one bigbird_attn_bwd / longformer_attn_bwd call (both patterns). */
size_t sa_attn_bwd_workspace_bytes(int B, int H, int n, int d);

/*
 * sa_set_workspace - use a caller-owned, device-resident scratch region on the
 * current device (dev_ptr 256-byte aligned, `bytes` large enough for the
 * calls that follow). The region must start zeroed; the library leaves its
 * counters at zero after every call that completes. Pass NULL/0 to go back to
 * the library-owned scratch. Calls sharing one region must be stream-ordered.
 * Errors: SA_ERR_INVALID_ARG for a misaligned pointer or NULL with bytes > 0.
 */
sa_status sa_set_workspace(void *dev_ptr, size_t bytes);

/*
 * sa_get_last_device_status - synchronise `stream`, then read and clear the
 * current device's latched device status (SA_OK, SA_ERR_TIMEOUT or
 * SA_ERR_BAD_INDEX). Returns SA_ERR_CUDA if the synchronisation fails.
 */
sa_status sa_get_last_device_status(sa_stream_t stream);

/* Human-readable name of a status code (static string). */
const char *sa_status_string(sa_status status);

/*
 * Options (process-wide; set them before issuing calls):
 *  SA_OPT_FORCE_SIMT   value != 0: run bf16 calls on the exact SIMT kernels
 *                      instead of the tensor-core kernels (a cross-check path).
 *  SA_OPT_WAIT_LIMIT   time bound, in microseconds, of every pipeline wait
 *                      in the tensor-core kernels (default 2000000 = 2 s);
 *                      value <= 0 restores the default. A wait that runs
 *                      past it aborts its CTA: the CTA latches
 *                      SA_ERR_TIMEOUT, waits for its own copies and MMAs in
 *                      flight (a separate fixed bound of 1 s, whatever this
 *                      option says), frees its tensor memory and exits. The
 *                      outputs of such a call are unspecified.
 *  SA_OPT_MAX_SPLITS   upper bound on split-KV chunks per global row tile
 *                      (default 16, 1 disables splitting).
 *  SA_OPT_GRID_CTAS    persistent-grid size (0 = one CTA per SM).
 *  SA_OPT_CHUNK_KEYS   keys per split-KV chunk of a global row tile, before
 *                      the SA_OPT_MAX_SPLITS bound (at most 2^20; chunks are
 *                      at least 8 steps). value <= 0 restores the default: a
 *                      tile's sweep is cut only when it exceeds three quarters
 *                      of the call's average work per tile in flight on a
 *                      full GB300 (estimated from the sizes and the pattern),
 *                      into chunks of about half that work. Shorter chunks
 *                      shorten the longest unit of a call (a global row
 *                      sweeps every key) at the cost of more partial results
 *                      to merge. The output does not depend on it beyond
 *                      rounding order.
 * Returns SA_ERR_INVALID_ARG for an unknown option.
 */
enum { SA_OPT_FORCE_SIMT = 1, SA_OPT_WAIT_LIMIT = 2, SA_OPT_MAX_SPLITS = 3, SA_OPT_GRID_CTAS = 4,
       SA_OPT_CHUNK_KEYS = 5 };
sa_status sa_set_option(int option, int64_t value);

/* Number of kernel launches issued by the calling thread's last successful
 * attention call (for launch accounting). */
int sa_last_launch_count(void);

/*
 * sa_check_wait_expiry - self-check of failure detection on the current
 * device, without a fault. It launches one warp that waits, through the same
 * bounded-wait helper every tensor-core kernel uses, on a barrier that nothing
 * ever arrives at. After `limit_us` microseconds (1 .. 1000000) the wait gives
 * up and latches SA_ERR_TIMEOUT in the device status word, exactly as an
 * expired pipeline wait would, and the kernel returns: the next
 * sa_get_last_device_status() on `stream` must report SA_ERR_TIMEOUT, and the
 * context stays usable. (The pages have no counterpart: this checks the
 * library's boundary contract for deferred device errors.)
 * Errors: SA_ERR_INVALID_ARG for a limit out of range; SA_ERR_UNSUPPORTED
 * without an sm_103a device; SA_ERR_CUDA if the launch fails.
 */
sa_status sa_check_wait_expiry(int64_t limit_us, sa_stream_t stream);

/*
 * bigbird_attn_fwd_noalloc - bigbird_attn_fwd for callers that must not
 * allocate device memory. (The pages have no counterpart: this is a
 * deployment variant of the same computation.)
 *
 * Who needs it: bigbird_attn_fwd sizes its scratch on the first call and
 * grows it with cudaMalloc later, and cudaMalloc may synchronise the whole
 * device and can fail once memory is fragmented. Some callers cannot accept
 * that: serving processes that reserve device memory at start-up and forbid
 * allocation on the request path, and plugins hosted by a framework that owns
 * the device's memory and does not let extensions allocate. This entry point
 * never calls cudaMalloc, cudaFree or any allocating routine. Its scratch is
 * one array of SA_NOALLOC_SCRATCH_BYTES compiled into the library; every GPU
 * that loads the library holds that array until the process exits.
 *
 * Arguments, layout, numerics and results are those of bigbird_attn_fwd with
 * dtype SA_BF16 (the tensor-core path); there is no dtype argument.
 * Set-up: the first call on a device looks up the array's device address on
 * that device (cudaGetSymbolAddress), so make that first call before any
 * stream capture begins. Each call first clears the array's counters with
 * cudaMemsetAsync on `stream`.
 * Sharing: all calls on a device share the one array, which keeps the last
 * call's contents. Calls ordered on one stream are safe; calls that overlap
 * on the GPU (different streams without ordering, or several host threads)
 * race on the array and give wrong results.
 * Errors: as bigbird_attn_fwd, plus SA_ERR_UNSUPPORTED, before any work is
 * queued, when the call needs more scratch than SA_NOALLOC_SCRATCH_BYTES
 * (sa_bigbird_workspace_bytes gives the need; it grows with B*H*g*b*d*n).
 */
#define SA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)
sa_status bigbird_attn_fwd_noalloc(const void *Q, const void *K, const void *V, void *O,
                                   int B, int H, int n, int d, int b, int g, int w, int r,
                                   const int32_t *rand_idx, const uint8_t *key_mask,
                                   sa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_ATTN_H */
