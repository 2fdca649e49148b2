/*
 * mse.h -- C ABI of the GB300 (sm_103a) shared-expert SwiGLU MLP library.
 *
 * The library computes, on one GPU:
 *   - the Kimi-K3 shared-expert / dense SwiGLU MLP
 *       y = W_down . ( SiLU(W_gate . x) * (W_up . x) )
 *     with a merged gate_up weight (gate rows first), hidden 7168 and
 *     intermediate 6144 in bf16
 *     ("[Kimi-K3] Add option to shard the shared expert instead of replicating",
 *      sections "Problem" and "Change");
 *   - the tensor-parallel sharded form of that MLP: shard r of tp owns the
 *     intermediate slice [r*s, (r+1)*s), s = I/tp, computes a partial output over
 *     it for all gathered tokens, and the partials are summed -- the sum half of
 *     the reduce-scatter; rank r keeps token rows [r*T/tp, (r+1)*T/tp)
 *     (same page, section "Change"; prhub analysis of vllm PR #50656, sections
 *      "实现拆解" and "关键源码片段");
 *   - the merged MLA q_a/kv_a latent projection stored as tensor-parallel
 *     column shards, whose gathered output is rank-major and is restored to the
 *     logical [q_a | kv_a] layout
 *     ("[II] TP-shard Kimi MLA latent projections", sections "Behavior",
 *      "Technical reason" and "Compatibility").
 *
 * Conventions (every entry point):
 *   - bf16 tensors are uint16_t bit patterns; all tensors are dense row-major.
 *   - Every tensor pointer is a DEVICE pointer owned by the caller.  The library
 *     allocates no device memory; scratch comes from the caller's workspace.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Launches are asynchronous on it; nothing synchronises.
 *   - The return value reports host-side validation and launch errors.  Errors
 *     raised on the device (a bounded wait that ran out) are reported later by
 *     mse_poll_device_error().
 *   - Arguments are validated before any CUDA call, so invalid calls fail the
 *     same way with or without a GPU.  There is no CPU fallback: on a device
 *     other than sm_103 the calls return MSE_ERR_UNSUPPORTED_DEVICE.
 *   - "capacity" arguments are element counts of the caller's buffer; a buffer
 *     smaller than the geometry needs is rejected as MSE_ERR_GEOMETRY (the
 *     truncated-geometry rejection of the MLA page, section "Validation").
 *   - The library is thread-safe; calls on the same stream are ordered.
 */
#ifndef MSE_H
#define MSE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported symbols (the library is built with hidden default visibility). */
#if defined(__GNUC__)
#define MSE_API __attribute__((visibility("default")))
#else
#define MSE_API
#endif

typedef uint16_t mse_bf16;

typedef enum {
    MSE_OK = 0,
    MSE_ERR_INVALID_ARG = 1,        /* null pointer, non-positive size, bad enum      */
    MSE_ERR_NOT_DIVISIBLE = 2,      /* I, H, q or kv not divisible by tp; T by parts  */
    MSE_ERR_GEOMETRY = 3,           /* capacity too small, rank range outside [0,tp)  */
    MSE_ERR_WORKSPACE = 4,          /* workspace missing, too small or misaligned     */
    MSE_ERR_UNSUPPORTED_DEVICE = 5, /* no CUDA device, or not compute capability 10.3 */
    MSE_ERR_CUDA = 6,               /* a CUDA runtime call failed                      */
    MSE_ERR_TIMEOUT = 7,            /* a device-side bounded wait ran out              */
    MSE_ERR_UNSUPPORTED_SHAPE = 8   /* kernel path forced by mse_set_kernel_path()
                                       cannot serve this shape/alignment               */
} mse_status;

typedef enum { MSE_BF16 = 0, MSE_F32 = 1 } mse_dtype;

/* Kernel path selection (process-wide; default MSE_PATH_AUTO).
 *   AUTO:        tensor-core (tcgen05/TMA) kernels where the shape and the
 *                16-byte alignment allow, else the generic CUDA-core kernels.
 *   GENERIC:     always the generic CUDA-core kernels (any shape).
 *   TENSORCORE:  always tcgen05 kernels; calls they cannot serve return
 *                MSE_ERR_UNSUPPORTED_SHAPE. */
typedef enum { MSE_PATH_AUTO = 0, MSE_PATH_GENERIC = 1, MSE_PATH_TENSORCORE = 2 } mse_kernel_path;

/* Tensor-core kernel for the token counts the decode-size kernels do not serve
 * (MSE_TUNE_SWAPAB_MAX_T), process-wide.
 *   AUTO:   CTA-pair kernel (two SMs share one 256 x 256 tile) up to 256 tokens and from
 *           512 on, single-CTA 128 x 256 kernel between.
 *   SINGLE: always the single-CTA kernel.   PAIR: always the CTA-pair kernel. */
typedef enum { MSE_PREFILL_AUTO = 0, MSE_PREFILL_SINGLE = 1, MSE_PREFILL_PAIR = 2 } mse_prefill_kernel;

/* ---------------------------------------------------------------------------
 * Workspace sizing.  The workspace holds the bf16 intermediate h [T x I] and,
 * for the tensor-core path, fp32 split-K partial tiles and the sync words (tile
 * counters and flags).  It must be 256-byte aligned and ZERO-FILLED before its
 * first use.  The sync words sit at the END of the buffer (their size depends on
 * H and I, or on q_dim + kv_dim, only); h and the partial tiles are laid out from
 * its start.  Every call that completes leaves the sync words zero again, so a
 * workspace of mlp_swiglu_workspace_bytes(T, H, I) bytes serves any sequence of
 * calls on one stream with at most T tokens and the same H and I (likewise for
 * the merged projection).  A call with another H or I needs a freshly zeroed
 * workspace.  Calls that run concurrently (different streams) need different
 * workspaces.  After MSE_ERR_TIMEOUT the caller must zero the workspace again.
 * A call accepts any workspace at least as large as its own minimal need, which
 * can be smaller than the size query's answer (the query covers all smaller T).
 * ------------------------------------------------------------------------- */

/* Bytes of a workspace that serves mlp_swiglu_forward, mlp_swiglu_shard_partial
 * and mlp_swiglu_shard_forward for every token count up to T (tp does not change
 * it).  Returns 0 on invalid arguments. */
MSE_API size_t mlp_swiglu_workspace_bytes(int64_t T, int64_t H, int64_t I);

/* Bytes of a workspace that serves merged_proj_forward for every token count up
 * to T with the same q_dim + kv_dim.  Returns 0 on invalid arguments. */
MSE_API size_t merged_proj_workspace_bytes(int64_t T, int64_t H, int64_t q_dim, int64_t kv_dim);

/* Byte range [*offset, *offset + *bytes) of the sync words (tile counters and
 * flags) inside a workspace of workspace_bytes for calls with at most T tokens
 * and this H and I.  Only this range must be zero before a call: after
 * MSE_ERR_TIMEOUT, zeroing it is enough to reuse the workspace.  Returns
 * MSE_ERR_WORKSPACE when workspace_bytes is below the call's minimal need,
 * MSE_ERR_INVALID_ARG on invalid sizes or null pointers.  Host only. */
MSE_API mse_status mlp_swiglu_workspace_sync_range(int64_t T, int64_t H, int64_t I, size_t workspace_bytes,
                                                   size_t *offset, size_t *bytes);

/* The same for a merged-projection workspace (the tile counters). */
MSE_API mse_status merged_proj_workspace_sync_range(int64_t T, int64_t H, int64_t q_dim, int64_t kv_dim,
                                                    size_t workspace_bytes, size_t *offset, size_t *bytes);

/* ---------------------------------------------------------------------------
 * Replicated SwiGLU MLP ("[Kimi-K3] Add option to shard the shared expert
 * instead of replicating", section "Change": gate_up projection, SiluAndMul,
 * down projection; the replicated path when the flag is off).
 *
 *   x          [T x H]    bf16 tokens
 *   w_gate_up  [2I x H]   bf16; rows [0, I) = W_gate, rows [I, 2I) = W_up
 *   w_down     [H x I]    bf16 (out x in)
 *   y          [T x H]    bf16 output, y_capacity >= T*H elements
 *
 *   g = x W_gate^T, u = x W_up^T accumulate in fp32 and are not rounded;
 *   h = bf16_rne(silu(g) * u) is rounded once and kept in the workspace;
 *   y = bf16_rne(h W_down^T) with fp32 accumulation.
 * ------------------------------------------------------------------------- */
MSE_API mse_status mlp_swiglu_forward(const mse_bf16 *x, int64_t T, int64_t H, int64_t I,
                              const mse_bf16 *w_gate_up, const mse_bf16 *w_down,
                              mse_bf16 *y, int64_t y_capacity,
                              void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * Partial outputs of shards [rank_first, rank_first + rank_count) of a tp-way
 * shard of the MLP over the intermediate dimension (prhub analysis of vllm
 * PR #50656, section "关键源码片段": shard r uses gate rows and up rows
 * [r*s, (r+1)*s) and down columns [r*s, (r+1)*s); the down projection is
 * RowParallel and partial over the intermediate dimension per the Kimi-K3 PR,
 * section "Change").  All T tokens are the gathered token set.
 *
 *   partials   [rank_count x T x H], partial_dtype MSE_BF16 or MSE_F32;
 *              partials[i] is the partial of rank rank_first + i, rounded once
 *              from its fp32 accumulator; partials_capacity >= rank_count*T*H.
 *
 * Errors: MSE_ERR_NOT_DIVISIBLE if I % tp or H % tp (the divisibility rule of
 * the sharding gate, prhub section "实现拆解"); MSE_ERR_GEOMETRY if
 * rank_first < 0, rank_count < 1 or rank_first + rank_count > tp.
 * ------------------------------------------------------------------------- */
MSE_API mse_status mlp_swiglu_shard_partial(const mse_bf16 *x, int64_t T, int64_t H, int64_t I,
                                    const mse_bf16 *w_gate_up, const mse_bf16 *w_down,
                                    int tp, int rank_first, int rank_count,
                                    void *partials, mse_dtype partial_dtype,
                                    int64_t partials_capacity,
                                    void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * The partials of shards [rank_first, rank_first + rank_count) summed inside the
 * down projection: a GEMM whose epilogue does the reduce-scatter's sum (Kimi-K3
 * PR, section "Change": the block-end reduce-scatter sums across TP and restores
 * the sequence sharding; prhub analysis of vllm PR #50656, section "关键源码片段":
 * per-shard partials, then stack(partials).sum(0)).  No partial is rounded or
 * stored: the down projection accumulates the group's intermediate columns
 * [rank_first*s, (rank_first + rank_count)*s), s = I/tp, in fp32 (split across
 * CTAs in ascending k order), and the sum is rounded once.
 *
 *   out   [T x H], out_dtype MSE_BF16 or MSE_F32, out_capacity >= T*H.
 *         rank_count = tp: the whole TP group's reduced output; rank r's scatter
 *         share is the row block [r*T/tp, (r+1)*T/tp) (a view; nothing is copied).
 *         rank_count < tp: the group's pre-reduced partial, which a cross-GPU
 *         reduce-scatter would sum with the other groups'.
 *   Same inputs, workspace and stream rules as mlp_swiglu_shard_partial.
 *
 * Errors: MSE_ERR_NOT_DIVISIBLE if I % tp or H % tp; MSE_ERR_GEOMETRY if
 * rank_first < 0, rank_count < 1, rank_first + rank_count > tp or
 * out_capacity < T*H; MSE_ERR_INVALID_ARG for an unknown out_dtype.
 * ------------------------------------------------------------------------- */
MSE_API mse_status mlp_swiglu_shard_forward(const mse_bf16 *x, int64_t T, int64_t H, int64_t I,
                                    const mse_bf16 *w_gate_up, const mse_bf16 *w_down,
                                    int tp, int rank_first, int rank_count,
                                    void *out, mse_dtype out_dtype, int64_t out_capacity,
                                    void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * Whether a dense or shared-expert MLP is to be TP-sharded under sequence
 * parallelism rather than replicated on every rank (prhub analysis of vllm PR
 * #50656, section "实现拆解", item 2; Kimi-K3 PR, sections "Change" and "Trade-off
 * and why it is opt-in"): 1
 * when all of
 *   - enabled: the opt-in switch is on (it is off by default);
 *   - use_sequence_parallel: the model runs with sequence parallelism;
 *   - eligible: the call site may shard (shared experts only on the path whose
 *     MoE block hands them the tokens directly; dense MLPs always);
 *   - tp_size > 1, and hidden_size % tp_size == 0 and
 *     intermediate_size % tp_size == 0;
 * hold, else 0: the MLP stays replicated (the conservative fallback, never an
 * error).  A pure host function: it touches no GPU and needs no device.
 * ------------------------------------------------------------------------- */
MSE_API int mse_shard_sequence_parallel_mlp(int enabled, int use_sequence_parallel, int eligible,
                                            int tp_size, int64_t hidden_size, int64_t intermediate_size);

/* ---------------------------------------------------------------------------
 * Sum of partials: the reduction half of the block-end reduce-scatter
 * (Kimi-K3 PR, section "Change": it sums across TP and restores the sequence
 * sharding).  out[t, n] = bf16_rne( sum_{r ascending} partials[r, t, n] ) with
 * fp32 accumulation.  Rank r's scatter share is the row block
 * [r*T/n_parts, (r+1)*T/n_parts) of `out` (a view; nothing is copied).
 *
 *   partials   [n_parts x T x H] of partial_dtype
 *   out        [T x H] bf16, out_capacity >= T*H
 *
 * Errors: MSE_ERR_NOT_DIVISIBLE if T % n_parts != 0 (token rows cannot be
 * scattered evenly).
 * ------------------------------------------------------------------------- */
MSE_API mse_status shard_sum(const void *partials, mse_dtype partial_dtype, int n_parts,
                     int64_t T, int64_t H, mse_bf16 *out, int64_t out_capacity, void *stream);

/* ---------------------------------------------------------------------------
 * Merged MLA q_a/kv_a latent projection ("[II] TP-shard Kimi MLA latent
 * projections", section "Behavior").  C = q_dim + kv_dim.
 *
 *   x            [T x H] bf16
 *   w            [C x H] bf16, logical row order: q_a rows then kv_a rows
 *   out_logical    nullable, [T x C] bf16 in logical column order [q_a | kv_a]
 *   out_rank_major nullable, [T x C] bf16 in gathered order: for each rank r
 *                  ascending, its q_a columns [r*q/tp, (r+1)*q/tp) then its kv_a
 *                  columns [r*kv/tp, (r+1)*kv/tp)  (the layout a tensor-parallel
 *                  gather of merged column shards produces)
 *   At least one output must be non-null; out_capacity >= T*C.
 *   out = bf16_rne(x w^T) with fp32 accumulation.
 *
 * Errors: MSE_ERR_NOT_DIVISIBLE if q_dim % tp or kv_dim % tp (every merged
 * output size must be divisible by tp, section "Compatibility").
 * ------------------------------------------------------------------------- */
MSE_API mse_status merged_proj_forward(const mse_bf16 *x, int64_t T, int64_t H, const mse_bf16 *w,
                               int64_t q_dim, int64_t kv_dim, int tp,
                               mse_bf16 *out_logical, mse_bf16 *out_rank_major,
                               int64_t out_capacity,
                               void *workspace, size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * Rank-major -> logical reorder alone (MLA page, sections "Behavior" and
 * "Technical reason": the merged-column gather is rank-major and the logical
 * q_a-then-kv_a ranges are restored explicitly).  A pure permutation of 16-bit
 * words: gathered column g = r*(qs+ks) + l maps to logical column
 * r*qs + l (l < qs) or q_dim + r*ks + (l - qs) (l >= qs), qs = q/tp, ks = kv/tp.
 *
 *   rank_major, logical: [T x C] bf16, capacity >= T*C each; must not overlap.
 * ------------------------------------------------------------------------- */
MSE_API mse_status merged_proj_reorder(const mse_bf16 *rank_major, mse_bf16 *logical, int64_t T,
                               int64_t q_dim, int64_t kv_dim, int tp, int64_t capacity,
                               void *stream);

/* ---------------------------------------------------------------------------
 * mlp_swiglu_forward for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is a deployment convenience of this library.
 *
 * Some callers hold only their input and output buffers and have no way to
 * obtain scratch memory: custom-operator interfaces of inference runtimes that
 * pass tensors but no workspace, or code that must not call the CUDA allocator
 * at all (cudaMalloc can synchronise the device and fail under memory pressure).
 * This entry point computes exactly what mlp_swiglu_forward computes, with the
 * same arguments minus the workspace: its scratch (h, split-K partial tiles,
 * tile counters) is a fixed 32 MiB file-scope device array inside the library,
 * which every device that loads the library holds until the process exits.
 *
 *  - Limit: mlp_swiglu_workspace_bytes(T, H, I) <= 32 MiB, e.g. T <= 64 tokens
 *    at hidden 7168 / intermediate 6144.  Larger calls return MSE_ERR_WORKSPACE
 *    and launch nothing.
 *  - It calls no cudaMalloc, cudaFree or allocating library routine.
 *  - The first call on a device performs a one-time set-up on that device
 *    (it looks up the array's device address with cudaGetSymbolAddress); make
 *    that first call before any stream capture.
 *  - Every call on a device shares the one array, and the array keeps the last
 *    call's contents (each call clears the tile counters it needs on `stream`).
 *    Calls whose executions overlap on the GPU (different streams, or several
 *    host threads without ordering) race on the array and give wrong results;
 *    order them on one stream.
 * ------------------------------------------------------------------------- */
MSE_API mse_status mlp_swiglu_forward_static_scratch(const mse_bf16 *x, int64_t T, int64_t H, int64_t I,
                                                     const mse_bf16 *w_gate_up, const mse_bf16 *w_down,
                                                     mse_bf16 *y, int64_t y_capacity, void *stream);

/* ---------------------------------------------------------------------------
 * The replicated SwiGLU MLP with its activations in host memory: the same layer as
 * mlp_swiglu_forward ("[Kimi-K3] Add option to shard the shared expert instead of
 * replicating", section "Change"), for callers whose tokens arrive in, and whose output
 * goes back to, page-locked host memory.
 *
 *   x_host  [T x H] bf16, page-locked host memory mapped into the device's address space
 *           (cudaHostAlloc, or cudaHostRegister with cudaHostRegisterMapped); on systems
 *           whose GPU reaches pageable host memory (cudaDevAttrPageableMemoryAccess, e.g.
 *           Grace-based ones) any host memory
 *   y_host  [T x H] bf16, the same kind of memory, y_capacity >= T*H elements
 *   w_gate_up, w_down  device memory, as for mlp_swiglu_forward
 *   workspace  device memory of mlp_swiglu_host_workspace_bytes(T, H, I) bytes, 256-byte
 *           aligned, zero before first use: 256 bytes of copy counts, two device copies of
 *           x, then the workspace of mlp_swiglu_forward (same rules for reuse)
 *
 * The kernels are launched on `stream` with programmatic dependent launch, so that none of
 * them cuts the overlap of consecutive calls; the down projection writes y straight into
 * y_host.  On the decode-size (swap-AB) kernels the gate_up launch copies x itself: the
 * CTAs that start first (on the SMs the previous layer's down projection leaves free; at
 * most MSE_TUNE_HOST_X_COPIERS) copy one slice each into one of the two device copies, the
 * other one than the previous call on this workspace, and every CTA's token loads wait for
 * all slices.  Elsewhere a copy kernel into the first device copy runs before the layer.
 * x is read while the previous work on the stream still runs, unless x overlaps the y_host
 * of the previous call of this entry point on the same stream (layers chained through host
 * memory), or the previous call on this workspace is unknown (the first, one with another T
 * or H, one on another path, or one captured into a CUDA graph; calls during capture always
 * wait): then it is read once that work is complete.  y_host holds the result once the
 * stream has reached the end of the call (e.g. after cudaStreamSynchronize); the host must
 * not modify x or read y before then.  MSE_ERR_INVALID_ARG if a host pointer is not mapped
 * page-locked memory or the two buffers overlap.
 * ------------------------------------------------------------------------- */
MSE_API size_t mlp_swiglu_host_workspace_bytes(int64_t T, int64_t H, int64_t I);
MSE_API mse_status mlp_swiglu_forward_host(const mse_bf16 *x_host, int64_t T, int64_t H, int64_t I,
                                           const mse_bf16 *w_gate_up, const mse_bf16 *w_down, mse_bf16 *y_host,
                                           int64_t y_capacity, void *workspace, size_t workspace_bytes,
                                           void *stream);

/* ---------------------------------------------------------------------------
 * Errors raised on the device and process-wide settings.
 * ------------------------------------------------------------------------- */

/* Synchronises `stream`, then reads and clears the library's device error word
 * on the current device: MSE_OK, MSE_ERR_TIMEOUT, or MSE_ERR_CUDA if the
 * synchronisation itself failed. */
MSE_API mse_status mse_poll_device_error(void *stream);

/* Upper bound, in nanoseconds, of every device-side wait of later launches
 * (default 2e9 = 2 s).  A wait that runs out sets the device error word, the
 * kernel drains its in-flight copies, frees its tensor memory and returns. */
MSE_API void mse_set_wait_limit_ns(uint64_t ns);
MSE_API uint64_t mse_get_wait_limit_ns(void);

/* Kernel path selection, see mse_kernel_path.  Returns the previous value. */
MSE_API int mse_set_kernel_path(int path);

/* Prefill kernel selection, see mse_prefill_kernel.  Returns the previous value. */
MSE_API int mse_set_prefill_kernel(int kind);

/* Tuning of the decode-size (swap-AB) kernels, process-wide, for later launches.
 *   MSE_TUNE_ISSUE_GROUP  consecutive 64-wide k-blocks per pipeline stage, i.e. each weight row
 *                         is fetched in runs of 128 x value contiguous bytes (1..4); 0 (default)
 *                         = 3 for launches of at most 64 tokens, 2 above
 *   MSE_TUNE_STAGES       shared-memory pipeline depth (0 = as many as fit, default)
 *   MSE_TUNE_CACHE_HINTS  1 = weights evict-first / tokens evict-last in L2 (default), 0 = none
 *   MSE_TUNE_GRID         CTAs of the stream-K grid (at most 160).  0 (default) = chosen per shape:
 *                         among 90-100% of the SMs the count that splits tiles into the fewest
 *                         parts when that is at most three, else one per SM; MLP launches with
 *                         little work (one shard's narrow slice) then at most one CTA per 16
 *                         k-blocks, but not fewer than half of the SMs
 *   MSE_TUNE_SPIN_WAIT    1 = pipeline waits poll (mbarrier.test_wait) instead of suspending
 *   MSE_TUNE_ONE_LAUNCH   decode token counts (T <= 256): 0 = gate_up + SiluAndMul and the down
 *                         projection as two launches (default: with programmatic dependent
 *                         launch this measured fastest); 1 = as passes of one launch, the down
 *                         weights streaming while the last gate_up tiles finish; 2 = one
 *                         launch with the gate_up tiles in two halves, the down pass taking
 *                         the first half's k-blocks first (replicated layer, else as 1)
 *   MSE_TUNE_PDL          1 = kernels are launched with programmatic dependent launch: a kernel
 *                         starts while the previous one in the stream drains and fetches its
 *                         first weight tiles before waiting for it (default); 0 = plain
 *                         stream order
 *   MSE_TUNE_COOP_FINISH  decode token counts: a tile whose reduction is split between at least
 *                         this many CTAs (0..128; 0 = never) is finished jointly by the CTAs for
 *                         which it is the final segment: each waits (bounded) for all parts,
 *                         then sums and writes one slice of the tile's token columns.  Other
 *                         split tiles are finished by the CTA arriving last.  Applies to the
 *                         merged projection and to MLP launches with some tile split this many
 *                         ways (one shard's narrow gate_up slice); same results bit for bit.
 *                         Default 6
 *   MSE_TUNE_PAIR_MIN_T   token counts from which the decode-size kernels run as CTA pairs: one
 *                         256-row weight tile per pair (one M = 256 MMA over both CTAs), each
 *                         CTA holding half of the token rows, so that more weight bytes are in
 *                         flight per SM (0 = never, the default: at 64 and 128 tokens it
 *                         measured no faster than single CTAs)
 *   MSE_TUNE_GRID_DOWN    CTAs of the down-projection swap-AB kernel (0 = as MSE_TUNE_GRID)
 *   MSE_TUNE_CLUSTER_FINISH  1 = when three CTAs of a decode-size kernel cover two tiles exactly
 *                         (gate_up at 64 tokens on 144 CTAs), launch clusters of three and finish
 *                         each two-part tile inside its cluster (same results bit for bit;
 *                         measured within 0.1 us); 0 = through L2 only (default)
 *   MSE_TUNE_L2_PREFETCH  decode token counts: 64-wide k-blocks of weight tiles beyond the
 *                         pipeline that a CTA prefetches into L2 before waiting for the previous
 *                         kernel, if it was not placed on an SM idle at launch: such CTAs start
 *                         while the previous kernel's split-K tail leaves HBM underused.  Applied
 *                         to launches of at most 64 tokens with at least 32 k-blocks per CTA
 *                         (default 8: the decode layer measured 54.2 against 54.35 us with none,
 *                         56.0 with 16; 0 = none)
 *   MSE_TUNE_SWAPAB_MAX_T launches over at least 4096 weight rows (the full layer) take the
 *                         decode-size (swap-AB) kernels up to this token count and the prefill
 *                         kernels above it (0 .. 256, default 160: at 176-256 tokens the full
 *                         layer measured 73 us on the CTA-pair kernel against 80-93 us); narrower
 *                         launches take the swap-AB kernels up to 256 tokens
 *   MSE_TUNE_X_EARLY      1 = mlp_swiglu_forward, mlp_swiglu_shard_partial, mlp_swiglu_shard_forward
 *                         and merged_proj_forward (decode-size kernels) read their x without
 *                         waiting for the previous kernel on the stream when x overlaps neither
 *                         this call's workspace nor anything the previous call on that stream
 *                         writes (its outputs and workspace), the previous call being one of
 *                         these four (independent layers, ranks or requests streamed back to
 *                         back): the first kernel's weight stream then runs during the previous
 *                         call's split-K tail.  Only for callers whose x is not written by a
 *                         kernel of their own that lets its dependents start early
 *                         (programmatic dependent launch) while still writing x.  0 = always
 *                         wait (default).
 *   MSE_TUNE_DOWN_FLAGS   decode token counts, two launches per layer: 1 = the gate_up kernel sets
 *                         a flag per finished 64-column block of h, and each CTA of the down
 *                         kernel, instead of waiting for the gate_up grid to complete, waits
 *                         until the flags of every h block it reads are set (its epilogue still
 *                         waits for the gate_up grid before any store); 0 = off (default)
 *   MSE_TUNE_HOST_X_COPIERS mlp_swiglu_forward_host on the decode-size kernels: the number of
 *                         CTAs of the gate_up launch that copy a slice of x each from host memory
 *                         (the first to start; 1 .. 1024, at most the launch's CTAs; default 16);
 *                         0 = a separate copy kernel before the layer
 *   MSE_TUNE_PAIR_SPLIT   1 = CTA-pair kernel launches of an MLP call at 129-256 tokens with at
 *                         most half as many tiles as clusters split the k-blocks of their tiles
 *                         over more clusters, at most two parts per tile (default); 0 = whole
 *                         tiles only
 * Returns the previous value, or -1 for an unknown key or out-of-range value.
 * Results do not depend on these settings beyond floating-point summation order. */
typedef enum {
    MSE_TUNE_ISSUE_GROUP = 1,
    MSE_TUNE_STAGES = 2,
    MSE_TUNE_CACHE_HINTS = 3,
    MSE_TUNE_GRID = 4,
    MSE_TUNE_SPIN_WAIT = 6,
    MSE_TUNE_ONE_LAUNCH = 7,
    MSE_TUNE_PDL = 8,
    MSE_TUNE_COOP_FINISH = 9,
    MSE_TUNE_PAIR_MIN_T = 10,
    MSE_TUNE_GRID_DOWN = 11,
    MSE_TUNE_CLUSTER_FINISH = 12,
    MSE_TUNE_L2_PREFETCH = 14,
    MSE_TUNE_SWAPAB_MAX_T = 15,
    MSE_TUNE_X_EARLY = 16,
    MSE_TUNE_DOWN_FLAGS = 17,
    MSE_TUNE_HOST_X_COPIERS = 18,
    MSE_TUNE_PAIR_SPLIT = 19
} mse_tune_key;
MSE_API int mse_set_tuning(int key, int value);

/* Launch plan of the decode-size (swap-AB) kernels of an MLP call, computed on the host
 * without a GPU: the CTA counts that mlp_swiglu_forward (tp = 1, rank_count = 1) or a
 * group of rank_count consecutive ranks of a tp-way split (mlp_swiglu_shard_partial /
 * mlp_swiglu_shard_forward, slices of I / tp intermediate columns; pages P1 "Change",
 * P2 "关键源码片段") would launch for T tokens on a device with sm_count SMs, with the
 * tuning keys as currently set; x_early = 1 when the call's early token loads apply (a
 * streamed call whose x the previous call does not write, MSE_TUNE_X_EARLY).
 * out[8] (host memory, written): [0] 1 when the call takes the swap-AB kernels, 0 when it
 * takes the prefill or the generic kernels (shapes off the 64-column grid, or
 * mse_set_kernel_path(MSE_PATH_GENERIC); then [1..7] are 0); [1] gate_up CTAs; [2] down
 * CTAs; [3] / [4] the largest number of CTAs a gate_up / down tile is split between;
 * [5] token tile width (T rounded up to 16); [6] k-blocks per pipeline stage; [7] stages.
 * Returns MSE_OK; MSE_ERR_INVALID_ARG (null out, non-positive size, rank_count outside
 * [1, tp]); MSE_ERR_NOT_DIVISIBLE (I by tp); MSE_ERR_UNSUPPORTED_SHAPE when a tuning key
 * makes the shape depend on the device's occupancy (MSE_TUNE_ONE_LAUNCH,
 * MSE_TUNE_PAIR_MIN_T, MSE_TUNE_CLUSTER_FINISH). */
MSE_API int mse_mlp_launch_plan(int64_t T, int64_t H, int64_t I, int tp, int rank_count, int x_early,
                                int sm_count, int32_t *out);

/* The same for merged_proj_forward (page P4 "Behavior": the 2112 x 7168 merged q_a / kv_a
 * projection).  out[8]: [0] 1 when the call takes the swap-AB kernel (0: the prefill or the
 * generic kernels, then [1..7] are 0); [1] CTAs; [2] the largest number of CTAs a 128-row
 * weight tile is split between; [3] 1 when the tiles' parts are finished jointly (every part's
 * CTA sums a slice of the token columns, MSE_TUNE_COOP_FINISH); [4] token tile width;
 * [5] k-blocks per pipeline stage; [6] stages; [7] 0.  Errors as mse_mlp_launch_plan (q_dim
 * and kv_dim by tp for MSE_ERR_NOT_DIVISIBLE). */
MSE_API int mse_merged_launch_plan(int64_t T, int64_t H, int64_t q_dim, int64_t kv_dim, int tp, int sm_count,
                                   int32_t *out);

/* Failure-detection self test: launches one CTA that waits on a barrier no one
 * arrives on, bounded by `limit_ns`.  The wait runs out by design; the kernel
 * records MSE_ERR_TIMEOUT in the device error word and returns, leaving the
 * context usable.  Read the result with mse_poll_device_error(). */
MSE_API mse_status mse_selftest_wait_timeout(uint64_t limit_ns, void *stream);

/* Timing hook for profiling harnesses.  While set, every mlp_swiglu_forward,
 * mlp_swiglu_shard_partial and mlp_swiglu_shard_forward call on the tensor-core
 * path records ev_begin before its first kernel, ev_mid between the gate_up and
 * the down kernel, and ev_end after the down kernel, on its stream (cudaEvent_t
 * handles passed as void*; all three non-null, or all null to clear).  The
 * records separate the two kernels, so launches made while the hook is set do
 * not overlap them. Process-wide; not meant for concurrent callers. */
MSE_API void mse_set_phase_events(void *ev_begin, void *ev_mid, void *ev_end);

/* Human-readable name of a status code (static string). */
MSE_API const char *mse_status_string(mse_status s);

/* Library version string, e.g. "mse 0.1 sm_103a". */
MSE_API const char *mse_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MSE_H */
