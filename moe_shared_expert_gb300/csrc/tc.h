// Internal interface of the tensor-core (tcgen05 + TMA) kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mse {
namespace tc {

enum Epi : int {
    EPI_SWIGLU = 0,      // h[t, j] = bf16(silu(g) * u)
    EPI_BF16 = 1,        // out[t, n] = bf16(acc)
    EPI_F32 = 2,         // out[t, n] = acc (fp32)
    EPI_MERGED = 3,      // logical and/or rank-major bf16 outputs
};

// Work of one launch of the swap-AB kernel (weights on the 128-row MMA side,
// tokens on the N side), decomposed stream-K over (group, m-tile, k-block).
struct SwapAbParams {
    int n_mtiles;          // 128-row A tiles per group (pair kernel: pairs of them, 256 rows)
    int n_mtiles_real;     // pair kernel: 128-row A tiles per group
    int n_groups;          // independent outputs (shards); 1 when replicated
    int kb_per_tile;       // units per tile: 64-wide k-blocks (halves = 1) or pairs of them (halves = 2)
    int halves;            // 2: unit u of a tile stands for k-blocks u and kb_per_tile + u
    int kb_first;          // k-block index of group 0's first block
    int kb_group_stride;   // k-block offset between groups
    int total_units;       // n_groups * n_mtiles * kb_per_tile
    int bn;                // MMA N (tokens, padded to a multiple of 16), <= 256
    int stages;            // smem pipeline depth
    int tmem_cols;         // allocated TMEM columns (power of two >= 2*bn)
    int a_row_base;        // SWIGLU: first intermediate index j of tile 0 (multiple of 64); the
                           // weight operand is W_gate_up viewed as (k, row, gate/up, 16-row
                           // block), so that rows 32b .. 32b+15 of a tile are gate rows and
                           // rows 32b+16 .. 32b+31 the up rows of the same j
    int kbs;               // consecutive k-blocks per pipeline stage (each weight row is fetched
                           // kbs x 128 contiguous bytes at a time; DRAM row-buffer locality)
    int cache_hints;       // 1: weights evict_first, tokens evict_last in L2; 0: no hints
    int spin_wait;         // 1: pipeline waits poll without suspending the thread
    int cluster_finish;    // 1: launched in clusters of three CTAs that cover two tiles exactly; the
                           // two-part tiles of the final segments are finished inside the cluster
    int coop_finish;       // > 0: a tile split into at least this many parts, in the CTAs' final
                           // segments, is finished jointly (each part's CTA sums one slice of
                           // token columns) when the ring is idle; 0: never
    int l2_prefetch_kb;    // k-blocks of weight tiles beyond the ring prefetched into L2 before the
                           // wait for the previous kernel, by CTAs with blockIdx >= l2_prefetch_from
    int l2_prefetch_from;  // (CTAs dispatched after the SMs that were idle at launch: they start
                           // while the previous kernel's tail leaves HBM underused)
    int x_early;           // gate_up: the token operand is not written by the previous kernel on the
                           // stream, so the producer requests it without waiting for that kernel
                           // (the epilogue still waits before any store)
    int T;                 // valid tokens
    int64_t m_valid;       // valid output features (A rows) for masking
    void *out; int64_t ldo; int64_t o_group_stride;
    uint16_t *out_rm; int64_t q_dim, kv_dim; int tp;   // EPI_MERGED
    float *slots;          // split-K partial tiles: 2 per CTA, 128 x bn fp32 each
    int *counters;         // one per tile; zero on entry, left zero on exit
    // h handed between the two launches of a layer by per-block flags (null: not used).
    // gate_up (EPI_SWIGLU): the flag of h column block a_row_base / 64 + m is set to
    //   hflag_epoch once that tile is written; the launch lets its dependent grid start only
    //   after waiting for the previous grid on the stream (the previous call's down kernel,
    //   which clears the flags), so the down kernel never sees the previous call's flags.
    // down: its epilogue warps poll, once, the flags of every h block the CTA reads until they
    //   equal hflag_epoch, and then release the producer's token loads (instead of waiting for
    //   the gate_up grid to complete); the last CTA past its poll (exit_count) clears the
    //   flags [hflag_first, hflag_first + hflag_n) and exit_count.  The epoch also differs between
    //   consecutive calls made outside graphs.
    int *hflags;
    int *exit_count;
    int hflag_first, hflag_n, hflag_epoch;
    // gate_up with x in host memory (null: x is already in device memory).  The first
    // x_copiers CTAs to start (those on SMs the previous kernel leaves free) copy one slice
    // of x each from x_host into x_copy, the buffer the token operand's tensor map reads, and
    // count it in x_sync[1]; every CTA's token loads wait until all slices are counted.
    // x_sync = [tickets taken, slices copied, CTAs past the wait]: the last CTA past the wait
    // zeroes all three.  x_copy_early = 0: the copiers wait for the previous grid first.
    const uint4 *x_host;
    uint4 *x_copy;
    int64_t x_vecs;        // 16-byte words of x
    int *x_sync;
    int x_copiers;
    int x_copy_early;
    uint64_t wait_limit_ns;
    uint32_t *err;
};

// The decode-size shared-expert layer in one launch: one or two gate_up + SiluAndMul
// passes into h (EPI_SWIGLU; ph[0], ph[1]), then the down projection of h (ph[2];
// EPI_BF16 or EPI_F32, groups = shards).  All passes use the same bn, stages and kbs.
struct SwapAbMlpParams {
    SwapAbParams ph[3];
    int n_gate_up_passes;   // 1 or 2
    int *hflags;            // per 64-column block of h: 1 once its gate_up tile is written
    int hflag_first;        // first flag index of this launch's h columns
    int n_htiles;           // gate_up tiles (flags) of this launch
    int *hcount;            // [2]: tiles published so far by gate_up pass 0 / pass 1
    int *exit_count;        // CTAs done; the last one clears hflags, hcount and this word
};

// Persistent standard-orientation kernel (tokens on the 128-row MMA side,
// weights on N = 256), one tile = 128 tokens x 256 output columns, full K.
struct StdParams {
    int n_mtiles;          // token tiles of 128
    int n_ntiles;          // 256-wide column tiles (SWIGLU: 128 j's of gate + 128 of up)
    int n_groups;
    int kb_per_tile;
    int kb_first;
    int kb_group_stride;
    int stages;
    int T;
    int64_t n_valid;       // valid output columns (I, H or C)
    int n_base;            // SWIGLU: first j of column tile 0
    void *out; int64_t ldo; int64_t o_group_stride;
    uint16_t *out_rm; int64_t q_dim, kv_dim; int tp;
    // CTA-pair kernel only: B row coordinate = b_base + n * b_n_stride + rank * b_rank_stride
    int b_base, b_n_stride, b_rank_stride;
    // CTA-pair kernel only: split_k = 1 splits the (tile, k-block) units evenly over the
    // clusters (stream-K; the host picks a cluster count that splits no tile into more than
    // two parts).  A split tile's parts are parked in slots (2 per CTA, 128 rows x 256
    // columns fp32, [column][row]) and counted in counters[tile * 2 + rank] (zero on entry,
    // left zero); the CTA arriving last sums them in part order and runs the epilogue.
    int split_k;
    float *slots;
    int *counters;
    int cache_hints;       // CTA-pair kernel: 1 = B (weights) evict_first, A (tokens) evict_last in L2
    int x_early;           // CTA-pair kernel: the A operand (tokens) is not written by the previous
                           // kernel on the stream, so the producer does not wait for that kernel
                           // (the epilogue still waits before any store)
    uint64_t wait_limit_ns;
    uint32_t *err;
};

constexpr int kSwapAbThreads = 192;   // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kStdThreads = 192;
constexpr int kMaxStages = 12;
constexpr int kMaxKbs = 4;            // k-blocks per pipeline stage (issue group)
constexpr int kMaxGrid = 160;         // cap on stream-K grids (one CTA per SM)
constexpr int kMaxPersistentGrid = 160; // cap on the persistent prefill grids

// Dynamic shared memory of the kernels.
size_t swapab_smem_bytes(int bn, int stages, int kbs);
size_t std_smem_bytes(int stages);
size_t pair_smem_bytes(int stages);
int pair_stages(bool one_token_tile);
int swapab_stages_for(int bn, int kbs);
int std_stages();

// grid = workers: CTAs, or CTA pairs (clusters of two) when `pair`.
cudaError_t launch_swapab(int epi, const CUtensorMap &ta, const CUtensorMap &tb, const SwapAbParams &p, int grid,
                          bool pdl, bool pair, cudaStream_t s);
int swapab_pair_max_clusters(int bn, int stages, int kbs);
// Largest number of CTAs any tile of a single-CTA stream-K launch of `grid` CTAs is split
// between (the launch takes the joint-finish kernel from coop_finish parts on).
int swapab_max_parts(const SwapAbParams &p, int grid);
// clusters of three single CTAs of the swap-AB kernel resident at once (0 on failure)
int swapab_trio_max_clusters(int bn, int stages, int kbs);
// The one-launch decode layer (grid <= SMs, one CTA per SM).
cudaError_t launch_swapab_mlp(int epi1, const CUtensorMap &ta0, const CUtensorMap &tb0, const CUtensorMap &ta1,
                              const CUtensorMap &tb1, const SwapAbMlpParams &fp, int grid, bool pdl, cudaStream_t s);
cudaError_t launch_std(int epi, const CUtensorMap &ta, const CUtensorMap &tb, const StdParams &p, int grid, bool pdl,
                       cudaStream_t s);
// CTA-pair kernel: 256 tokens x 256 columns per tile, grid = 2 x clusters.
cudaError_t launch_pair(int epi, const CUtensorMap &ta, const CUtensorMap &tb, const StdParams &p, int clusters,
                        bool pdl, cudaStream_t s);

}  // namespace tc
}  // namespace mse
