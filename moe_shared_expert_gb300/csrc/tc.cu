// Tensor-core kernels for sm_103a: TMA-fed, mbarrier-pipelined tcgen05 MMA with
// fp32 accumulators in tensor memory, warp-specialised:
//   warp 0      TMA producer (one elected lane)
//   warp 1      TMEM allocator + MMA issuer (one elected lane)
//   warps 2..5  epilogue (tcgen05.ld of the warp's 32-lane quarter)
//
// swapab_kernel: decode-sized token counts.  The weight rows fill the 128-row
//   MMA M side and the tokens form N (<= 256), so each CTA streams weight tiles
//   through a deep TMA ring, requesting several consecutive k-blocks back to back
//   so that DRAM sees runs of >= 512 contiguous bytes per weight row.  Work is
//   split stream-K over (group, m-tile,
//   k-block) units so that every SM streams the same number of weight bytes;
//   a tile cut between CTAs is finished by whichever CTA arrives last on the
//   tile's counter (fp32 partial tiles in the workspace, summed in a fixed
//   order, so results do not depend on arrival order).  No CTA ever waits on
//   another one.
// std_kernel: prefill-sized token counts.  Persistent CTAs walk 128-token x
//   256-column tiles over the full reduction with two TMEM accumulators, so the
//   epilogue of one tile overlaps the MMA of the next.
// pair_kernel: the same with a CTA pair (cta_group::2) per 256 x 256 tile.
#include <atomic>

#include "common.cuh"
#include "tc.h"

namespace mse {
namespace tc {
namespace {

constexpr uint32_t kATileBytes = 128 * 64 * 2;   // 128 rows x 64 bf16

struct Ctrl {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint64_t fixbar;         // swap-AB finisher: bulk copies of partial tiles into shared memory
    uint32_t tmem_base;
    int abort_flag;
    int fin_flag;
    float xbuf[4][16][32];   // swap-AB SwiGLU epilogue: g/u exchange between lane quarters
    int seg_slot[128];       // swap-AB split-K finisher: slot index of each part of the tile
};

__device__ __forceinline__ uint32_t bar_addr(const uint64_t *b) { return smem_u32(b); }

__device__ __forceinline__ int64_t logical_to_gathered(int64_t c, int64_t q_dim, int64_t kv_dim, int tp) {
    const int64_t qs = q_dim / tp, ks = kv_dim / tp, w = qs + ks;
    if (c < q_dim) return (c / qs) * w + (c % qs);
    const int64_t c2 = c - q_dim;
    return (c2 / ks) * w + qs + (c2 % ks);
}

__device__ __forceinline__ void load_tmem_chunk(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    tmem_ld16(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------------------
// swap-AB stream-K kernel
// ---------------------------------------------------------------------------

struct StreamK {
    int64_t U, G;
    __device__ __forceinline__ int64_t begin(int64_t c) const { return c * U / G; }
    __device__ __forceinline__ int64_t owner(int64_t u) const { return ((u + 1) * G - 1) / U; }
};

// Epilogue of one 16-token chunk of a swap-AB tile.  Thread `lane` of epilogue
// warp quarter `q` holds accumulator row r = 32q + lane for tokens c*16 .. c*16+15.
// All 128 epilogue threads call it together (it contains named barriers).
template <int EPI>
__device__ __forceinline__ void swapab_epilogue_chunk(const SwapAbParams &p, Ctrl *ctl, int group, int m, int q,
                                                      int lane, int c, const float (&v)[16]) {
    // Results are computed for every token before any store (branch-free, so the
    // independent chains interleave); the stores are unpredicated when the whole
    // chunk is inside T.
    if constexpr (EPI == EPI_SWIGLU) {
        // Rows 0-63 are gate rows j = j0 + r, rows 64-127 the up rows of the same j, so
        // quarter q (gate) pairs with quarter q ^ 2 (up).  The gate warp computes tokens
        // 0-7 of the chunk and the up warp tokens 8-15, each reading its partner's half
        // from shared memory.
#pragma unroll
        for (int i = 0; i < 16; ++i) ctl->xbuf[q][i][lane] = v[i];
        named_barrier_sync(1, 128);
        const bool is_gate = q < 2;
        const int pq = q ^ 2;
        const int64_t j = (int64_t)p.a_row_base + (int64_t)m * 64 + 32 * (q & 1) + lane;
        const int t0 = c * 16 + (is_gate ? 0 : 8);
        uint16_t hv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float g = is_gate ? v[i] : ctl->xbuf[pq][8 + i][lane];
            const float u = is_gate ? ctl->xbuf[pq][i][lane] : v[8 + i];
            hv[i] = f32_to_bf16_bits(silu_f32(g) * u);
        }
        named_barrier_sync(1, 128);   // xbuf is rewritten by the next chunk
        uint16_t *h = static_cast<uint16_t *>(p.out) + (int64_t)t0 * p.ldo + j;
        if (t0 + 8 <= p.T) {
#pragma unroll
            for (int i = 0; i < 8; ++i) h[(int64_t)i * p.ldo] = hv[i];
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (t0 + i < p.T) h[(int64_t)i * p.ldo] = hv[i];
        }
    } else {
        const int64_t n = (int64_t)m * 128 + q * 32 + lane;
        if (n >= p.m_valid) return;
        const int t0 = c * 16;
        const int nt = min(16, p.T - t0);
        if constexpr (EPI == EPI_F32) {
            float *o = static_cast<float *>(p.out) + group * p.o_group_stride + (int64_t)t0 * p.ldo + n;
            if (nt == 16) {
#pragma unroll
                for (int i = 0; i < 16; ++i) o[(int64_t)i * p.ldo] = v[i];
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (i < nt) o[(int64_t)i * p.ldo] = v[i];
            }
        } else {
            uint16_t b[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) b[i] = f32_to_bf16_bits(v[i]);
            if constexpr (EPI == EPI_BF16) {
                uint16_t *o = static_cast<uint16_t *>(p.out) + group * p.o_group_stride + (int64_t)t0 * p.ldo + n;
                if (nt == 16) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) o[(int64_t)i * p.ldo] = b[i];
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (i < nt) o[(int64_t)i * p.ldo] = b[i];
                }
            } else {  // EPI_MERGED
                uint16_t *lo = static_cast<uint16_t *>(p.out);
                const int64_t gcol = logical_to_gathered(n, p.q_dim, p.kv_dim, p.tp);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    if (i < nt) {
                        if (lo) lo[(int64_t)(t0 + i) * p.ldo + n] = b[i];
                        if (p.out_rm) p.out_rm[(int64_t)(t0 + i) * p.ldo + gcol] = b[i];
                    }
                }
            }
        }
    }
}

// Epilogue of a whole swap-AB tile held in shared memory as fp32 [token][row]
// (row = accumulator row, 128 per token).  All 128 epilogue threads (tid 0..127)
// work element-wise: a fixed row per thread, tokens strided, so shared reads are
// conflict-free and the 32 lanes of a warp store 32 consecutive outputs.
template <int EPI>
__device__ __forceinline__ void swapab_epilogue_smem(const SwapAbParams &p, const float *tilebuf, int group, int m,
                                                     int tid) {
    if constexpr (EPI == EPI_SWIGLU) {
        // rows 0-63: g of j = j0 + r; rows 64-127: u of the same j
        const int jr = tid & 63;
        uint16_t *h = static_cast<uint16_t *>(p.out) + (int64_t)p.a_row_base + (int64_t)m * 64 + jr;
        int t = tid >> 6;
        for (; t + 6 < p.T; t += 8) {   // 4 tokens per step, computed before storing
            uint16_t hv[4];
#pragma unroll
            for (int r = 0; r < 4; ++r)
                hv[r] = f32_to_bf16_bits(silu_f32(tilebuf[(t + 2 * r) * 128 + jr]) * tilebuf[(t + 2 * r) * 128 + 64 + jr]);
#pragma unroll
            for (int r = 0; r < 4; ++r) h[(int64_t)(t + 2 * r) * p.ldo] = hv[r];
        }
        for (; t < p.T; t += 2)
            h[(int64_t)t * p.ldo] = f32_to_bf16_bits(silu_f32(tilebuf[t * 128 + jr]) * tilebuf[t * 128 + 64 + jr]);
    } else {
        const int64_t n = (int64_t)m * 128 + tid;
        if (n >= p.m_valid) return;
        if constexpr (EPI == EPI_F32) {
            float *o = static_cast<float *>(p.out) + group * p.o_group_stride + n;
            for (int t = 0; t < p.T; ++t) o[(int64_t)t * p.ldo] = tilebuf[t * 128 + tid];
        } else if constexpr (EPI == EPI_BF16) {
            uint16_t *o = static_cast<uint16_t *>(p.out) + group * p.o_group_stride + n;
            int t = 0;
            for (; t + 3 < p.T; t += 4) {
                uint16_t b[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) b[r] = f32_to_bf16_bits(tilebuf[(t + r) * 128 + tid]);
#pragma unroll
                for (int r = 0; r < 4; ++r) o[(int64_t)(t + r) * p.ldo] = b[r];
            }
            for (; t < p.T; ++t) o[(int64_t)t * p.ldo] = f32_to_bf16_bits(tilebuf[t * 128 + tid]);
        } else {
            uint16_t *lo = static_cast<uint16_t *>(p.out);
            const int64_t gcol = logical_to_gathered(n, p.q_dim, p.kv_dim, p.tp);
            for (int t = 0; t < p.T; ++t) {
                const uint16_t b = f32_to_bf16_bits(tilebuf[t * 128 + tid]);
                if (lo) lo[(int64_t)t * p.ldo + n] = b;
                if (p.out_rm) p.out_rm[(int64_t)t * p.ldo + gcol] = b;
            }
        }
    }
}

template <int EPI>
__global__ void __launch_bounds__(kSwapAbThreads, 1)
    swapab_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const SwapAbParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int S = p.stages, bn = p.bn;
    const int KBS = p.kbs;                                     // k-blocks per pipeline stage
    const uint32_t b_tile_bytes = (uint32_t)bn * 128u;         // one k-block of tokens
    const uint32_t a_stage_bytes = (uint32_t)KBS * kATileBytes;
    const uint32_t stage_bytes = a_stage_bytes + (uint32_t)KBS * b_tile_bytes;
    // stage s: [KBS weight tiles of 128 x 64][KBS token tiles of bn x 64]
    auto sA = [&](int st) { return base + (uint32_t)st * stage_bytes; };
    auto sB = [&](int st) { return base + (uint32_t)st * stage_bytes + a_stage_bytes; };
    Ctrl *ctl = reinterpret_cast<Ctrl *>(smem_raw + (base - raw) + (uint32_t)S * stage_bytes);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const StreamK sk{p.total_units, gridDim.x};
    const int64_t ub = sk.begin(blockIdx.x), ue = sk.begin(blockIdx.x + 1);
    const int kbp = p.kb_per_tile;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_addr(&ctl->full[s]), 1);
            mbar_init(bar_addr(&ctl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_addr(&ctl->tfull[b]), 1);
            mbar_init(bar_addr(&ctl->tempty[b]), 128);
        }
        mbar_init(bar_addr(&ctl->drain), 1);
        mbar_init(bar_addr(&ctl->fixbar), 1);
        ctl->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), (uint32_t)p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    volatile int *abort_flag = &ctl->abort_flag;
    pdl_launch_dependents();

    // The CTA's units [ub, ue) form segments (one per tile touched); each segment is cut
    // into stages of up to KBS consecutive k-blocks.  Producer and MMA walk the same
    // sequence with incremental counters (no divisions inside the loops).
    struct Walk {
        int64_t u, ue;
        int kbp, n_mtiles;
        int kb, kb_end, m, group;     // current stage starts at k-block kb of tile (group, m)
        int seg;                      // segment index within this CTA
        __device__ void init(int64_t ub_, int64_t ue_, int kbp_, int n_mtiles_) {
            u = ub_; ue = ue_; kbp = kbp_; n_mtiles = n_mtiles_; seg = 0;
            const int64_t tile = ub_ / kbp_;
            kb = (int)(ub_ - tile * kbp_);
            group = (int)(tile / n_mtiles_);
            m = (int)(tile - (int64_t)group * n_mtiles_);
            set_end();
        }
        __device__ void set_end() {
            const int64_t rem = ue - u;
            kb_end = (kbp - kb) < rem ? kbp : kb + (int)rem;
        }
        __device__ bool done() const { return u >= ue; }
        // k-blocks of the current stage
        __device__ int count(int kbs) const { return (kb_end - kb) < kbs ? (kb_end - kb) : kbs; }
        // advance past a stage of n k-blocks; returns true when that stage ended its segment
        __device__ bool advance(int n) {
            kb += n;
            u += n;
            if (kb < kb_end) return false;
            kb = 0;
            ++seg;
            if (++m == n_mtiles) { m = 0; ++group; }
            set_end();
            return true;
        }
    };

    int issued = 0;   // producer: stages whose loads were issued

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_x = l2_policy_evict_last();
            const bool hints = p.cache_hints != 0;
            auto kglob = [&](const Walk &w, int i) { return p.kb_first + w.group * p.kb_group_stride + w.kb + i; };
            auto load_a = [&](const Walk &w, int n, int st) {
                const uint32_t fb = bar_addr(&ctl->full[st]);
                for (int i = 0; i < n; ++i) {
                    const int k = kglob(w, i) * 64;
                    const uint32_t dst = sA(st) + (uint32_t)i * kATileBytes;
                    if constexpr (EPI == EPI_SWIGLU) {
                        // rows 0-63: gate rows j0..j0+63; rows 64-127: the up rows of the same j
                        const int j0 = p.a_row_base + w.m * 64;
                        if (hints) {
                            tma_load_2d(dst, &tmA, fb, k, j0, pol_w);
                            tma_load_2d(dst + 8192u, &tmA, fb, k, p.a_up_offset + j0, pol_w);
                        } else {
                            tma_load_2d_nohint(dst, &tmA, fb, k, j0);
                            tma_load_2d_nohint(dst + 8192u, &tmA, fb, k, p.a_up_offset + j0);
                        }
                    } else {
                        if (hints) tma_load_2d(dst, &tmA, fb, k, w.m * 128, pol_w);
                        else tma_load_2d_nohint(dst, &tmA, fb, k, w.m * 128);
                    }
                }
            };
            auto load_b = [&](const Walk &w, int n, int st) {
                const uint32_t fb = bar_addr(&ctl->full[st]);
                for (int i = 0; i < n; ++i) {
                    const int k = kglob(w, i) * 64;
                    const uint32_t dst = sB(st) + (uint32_t)i * b_tile_bytes;
                    if (hints) tma_load_2d(dst, &tmB, fb, k, 0, pol_x);
                    else tma_load_2d_nohint(dst, &tmB, fb, k, 0);
                }
            };
            Walk w;
            w.init(ub, ue, kbp, p.n_mtiles);
            // Prologue: weight tiles do not depend on the previous kernel, so they are
            // requested before waiting for it; the token tiles follow the wait.
            {
                Walk a = w;
                int st = 0;
                for (; st < S && !a.done(); ++st) {
                    const int n = a.count(KBS);
                    mbar_arrive_expect_tx(bar_addr(&ctl->full[st]), (uint32_t)n * (kATileBytes + b_tile_bytes));
                    load_a(a, n, st);
                    a.advance(n);
                }
                pdl_wait();
                for (int t = 0; t < st; ++t) {
                    const int n = w.count(KBS);
                    load_b(w, n, t);
                    w.advance(n);
                }
                issued = st;
            }
            int stage = issued == S ? 0 : issued;
            uint32_t phase = issued == S ? 1u : 0u;
            while (!w.done()) {
                if (!mbar_wait_bounded(bar_addr(&ctl->empty[stage]), phase ^ 1u, abort_flag, p.wait_limit_ns, p.err,
                                       p.spin_wait != 0))
                    break;
                const int n = w.count(KBS);
                mbar_arrive_expect_tx(bar_addr(&ctl->full[stage]), (uint32_t)n * (kATileBytes + b_tile_bytes));
                load_a(w, n, stage);
                load_b(w, n, stage);
                w.advance(n);
                ++issued;
                if (++stage == S) { stage = 0; phase ^= 1u; }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, (uint32_t)bn);
            int stage = 0;
            uint32_t phase = 0;
            Walk w;
            w.init(ub, ue, kbp, p.n_mtiles);
            bool ok = true;
            while (!w.done() && ok) {
                const int buf = w.seg & 1;
                const uint32_t use = (uint32_t)(w.seg >> 1);
                if (!mbar_wait_bounded(bar_addr(&ctl->tempty[buf]), (use & 1u) ^ 1u, abort_flag, p.wait_limit_ns,
                                       p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(buf * (p.tmem_cols / 2));
                bool first = true, seg_end = false;
                while (!seg_end) {
                    if (!mbar_wait_bounded(bar_addr(&ctl->full[stage]), phase, abort_flag, p.wait_limit_ns, p.err,
                                           p.spin_wait != 0)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int n = w.count(KBS);
                    for (int i = 0; i < n; ++i) {
                        const uint64_t ad = smem_desc_sw128(sA(stage) + (uint32_t)i * kATileBytes);
                        const uint64_t bd = smem_desc_sw128(sB(stage) + (uint32_t)i * b_tile_bytes);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            tc_mma_bf16(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, first ? 0u : 1u);
                            first = false;
                        }
                    }
                    tc_commit(bar_addr(&ctl->empty[stage]));
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                    seg_end = w.advance(n);
                }
                if (!ok) break;
                tc_commit(bar_addr(&ctl->tfull[buf]));
            }
        }
    } else {
        // epilogue warps 2..5
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        pdl_wait();
        int seg = 0;
        uint32_t fix_round = 0;   // completed phases of fixbar
        for (int64_t u = ub; u < ue; ++seg) {
            const int64_t tile = u / kbp;
            const int kb0 = (int)(u % kbp);
            const int64_t rem = ue - u;
            const int kb1 = (int)((kbp - kb0) < rem ? kbp : kb0 + rem);
            const int buf = seg & 1;
            const uint32_t use = (uint32_t)(seg >> 1);
            const int group = (int)(tile / p.n_mtiles);
            const int m = (int)(tile % p.n_mtiles);
            u = tile * kbp + kb1;
            const bool got = mbar_wait_bounded(bar_addr(&ctl->tfull[buf]), use & 1u, abort_flag, p.wait_limit_ns, p.err);
            if (!named_barrier_and(1, 128, got)) break;   // all epilogue warps take the same branch
            tc_fence_after();
            const uint32_t tacc = tmem_base + (uint32_t)(buf * (p.tmem_cols / 2)) + lane_off;
            const int nchunks = bn / 16;
            if (kb0 == 0 && kb1 == kbp) {
                for (int c = 0; c < nchunks; ++c) {
                    float v[16];
                    load_tmem_chunk(tacc + (uint32_t)(c * 16), v);
                    swapab_epilogue_chunk<EPI>(p, ctl, group, m, q, lane, c, v);
                }
                tc_fence_before();
                mbar_arrive(bar_addr(&ctl->tempty[buf]));
                continue;
            }
            // Tile shared with other CTAs: park the fp32 partial in this CTA's slot, laid
            // out [token column][accumulator row] (each warp store is a 128-byte run).
            const int which = (sk.begin(blockIdx.x) / kbp == tile) ? 0 : 1;
            float *slot = p.slots + ((size_t)blockIdx.x * 2 + which) * (size_t)(128 * bn);
            for (int c = 0; c < nchunks; ++c) {
                float v[16];
                load_tmem_chunk(tacc + (uint32_t)(c * 16), v);
#pragma unroll
                for (int i = 0; i < 16; ++i) __stcg(slot + (size_t)(c * 16 + i) * 128 + row, v[i]);
            }
            tc_fence_before();
            mbar_arrive(bar_addr(&ctl->tempty[buf]));
            fence_proxy_async_global();   // a finisher may fetch this slot with a bulk copy
            named_barrier_sync(1, 128);
            const int64_t c_first = sk.owner(tile * kbp), c_last = sk.owner(tile * kbp + kbp - 1);
            const int nseg = (int)(c_last - c_first + 1);
            if (threadIdx.x == 64) {
                // release: the barrier above orders every epilogue thread's slot stores
                // before this atomic; acquire: the finisher then sees all other parts
                const int prev = atomic_add_acq_rel_gpu(p.counters + tile, 1);
                ctl->fin_flag = (prev == nseg - 1) ? 1 : 0;
            }
            named_barrier_sync(1, 128);
            if (ctl->fin_flag) {
                // slot of each part: CTA cc's first segment uses slot 2cc, its last one 2cc+1
                for (int k = threadIdx.x - 64; k < nseg && k < 128; k += 128) {
                    const int64_t cc = c_first + k;
                    ctl->seg_slot[k] = (int)(cc * 2 + ((sk.begin(cc) >= tile * kbp) ? 0 : 1));
                }
                named_barrier_sync(1, 128);
                const size_t slot_floats = (size_t)128 * bn;
                const uint32_t slot_bytes = (uint32_t)(slot_floats * 4);
                const int per_round = (int)(((size_t)S * stage_bytes) / slot_bytes);
                const int tid = threadIdx.x - 64;
                if (u == ue && per_round >= 2 && nseg <= 128) {
                    // Last segment of this CTA: the pipeline's shared memory is idle, so the
                    // parts are bulk-copied into it (buffer 0 keeps the running sum) and summed
                    // element-wise in ascending part order starting from 0, as the fallback does.
                    fence_proxy_async_global();
                    float *buf0 = reinterpret_cast<float *>(smem_raw + (base - raw));
                    bool fix_ok = true;
                    int k0 = 0;
                    while (k0 < nseg) {
                        const int first_buf = k0 == 0 ? 0 : 1;
                        const int nload = min(nseg - k0, per_round - first_buf);
                        if (threadIdx.x == 64) {
                            mbar_arrive_expect_tx(bar_addr(&ctl->fixbar), (uint32_t)nload * slot_bytes);
                            for (int i = 0; i < nload; ++i)
                                bulk_load(base + (uint32_t)(first_buf + i) * slot_bytes,
                                          p.slots + (size_t)ctl->seg_slot[k0 + i] * slot_floats, slot_bytes,
                                          bar_addr(&ctl->fixbar));
                        }
                        const bool got_fix = mbar_wait_bounded(bar_addr(&ctl->fixbar), fix_round & 1u, abort_flag,
                                                               p.wait_limit_ns, p.err);
                        ++fix_round;
                        if (!named_barrier_and(1, 128, got_fix)) { fix_ok = false; break; }
                        const int nsum = first_buf + nload;
                        float4 *b0 = reinterpret_cast<float4 *>(buf0);
                        const int n4 = (int)(slot_floats / 4);   // a multiple of 512
                        for (int e = tid; e < n4; e += 512) {    // 4 independent float4 per thread per step
                            float4 a[4];
#pragma unroll
                            for (int r = 0; r < 4; ++r) {
                                a[r] = b0[e + r * 128];
                                if (k0 == 0) a[r] = make_float4(0.f + a[r].x, 0.f + a[r].y, 0.f + a[r].z, 0.f + a[r].w);
                            }
                            for (int bb = 1; bb < nsum; ++bb) {
                                const float4 *src = reinterpret_cast<const float4 *>(buf0 + (size_t)bb * slot_floats);
                                float4 t4[4];
#pragma unroll
                                for (int r = 0; r < 4; ++r) t4[r] = src[e + r * 128];
#pragma unroll
                                for (int r = 0; r < 4; ++r) {
                                    a[r].x += t4[r].x; a[r].y += t4[r].y; a[r].z += t4[r].z; a[r].w += t4[r].w;
                                }
                            }
#pragma unroll
                            for (int r = 0; r < 4; ++r) b0[e + r * 128] = a[r];
                        }
                        k0 += nload;
                        named_barrier_sync(1, 128);   // buffers 1.. are refilled by the next round
                    }
                    if (fix_ok) swapab_epilogue_smem<EPI>(p, buf0, group, m, tid);
                } else {
                    for (int c = 0; c < nchunks; ++c) {
                        float v[16] = {};
                        for (int k = 0; k < nseg; ++k) {
                            const int sl = k < 128 ? ctl->seg_slot[k]
                                                   : (int)((c_first + k) * 2 + ((sk.begin(c_first + k) >= tile * kbp) ? 0 : 1));
                            const float *src = p.slots + (size_t)sl * slot_floats + (size_t)(c * 16) * 128 + row;
                            float t16[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) t16[i] = __ldcg(src + (size_t)i * 128);
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] += t16[i];
                        }
                        swapab_epilogue_chunk<EPI>(p, ctl, group, m, q, lane, c, v);
                    }
                }
                if (threadIdx.x == 64) p.counters[tile] = 0;
            }
            named_barrier_sync(1, 128);   // fin_flag is reused by the next tile
        }
    }

    // ---- teardown: drain in-flight copies and MMAs, then free tensor memory ----
    if (warp == 0 && lane == 0) {
        const int first = issued > S ? issued - S : 0;
        for (int i = first; i < issued; ++i)
            (void)mbar_wait_drain(bar_addr(&ctl->full[i % S]), (uint32_t)((i / S) & 1), p.wait_limit_ns);
    }
    if (warp == 1 && lane == 0) {
        tc_commit(bar_addr(&ctl->drain));
        (void)mbar_wait_drain(bar_addr(&ctl->drain), 0, p.wait_limit_ns);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, (uint32_t)p.tmem_cols);
}

// ---------------------------------------------------------------------------
// persistent standard-orientation kernel
// ---------------------------------------------------------------------------
constexpr uint32_t kStdBTileBytes = 256 * 64 * 2;   // 256 rows x 64 bf16
constexpr int kStdBandM = 16;                       // m-tiles per raster band

struct StdTile { int group, m, n; };

__device__ __forceinline__ StdTile std_tile(const StdParams &p, int64_t id) {
    const int64_t per_group = (int64_t)p.n_mtiles * p.n_ntiles;
    StdTile t;
    t.group = (int)(id / per_group);
    const int64_t r = id % per_group;
    const int64_t per_band = (int64_t)kStdBandM * p.n_ntiles;
    const int band = (int)(r / per_band);
    const int first_m = band * kStdBandM;
    const int band_m = min(kStdBandM, p.n_mtiles - first_m);
    const int64_t in_band = r % per_band;
    t.m = first_m + (int)(in_band % band_m);
    t.n = (int)(in_band / band_m);
    return t;
}

template <int EPI>
__global__ void __launch_bounds__(kStdThreads, 1)
    std_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const StdParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int S = p.stages;
    const uint32_t sA = base;
    const uint32_t sB = base + (uint32_t)S * kATileBytes;
    Ctrl *ctl = reinterpret_cast<Ctrl *>(smem_raw + (base - raw) + (uint32_t)S * (kATileBytes + kStdBTileBytes));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int64_t n_tiles = (int64_t)p.n_groups * p.n_mtiles * p.n_ntiles;
    const int kbp = p.kb_per_tile;
    constexpr uint32_t kTmemCols = 512;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_addr(&ctl->full[s]), 1);
            mbar_init(bar_addr(&ctl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_addr(&ctl->tfull[b]), 1);
            mbar_init(bar_addr(&ctl->tempty[b]), 128);
        }
        mbar_init(bar_addr(&ctl->drain), 1);
        ctl->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    volatile int *abort_flag = &ctl->abort_flag;
    pdl_launch_dependents();

    int64_t issued = 0;
    if (warp == 0) {
        if (lane == 0) {
            pdl_wait();
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int64_t id = blockIdx.x; id < n_tiles && ok; id += gridDim.x) {
                const StdTile t = std_tile(p, id);
                for (int kb = 0; kb < kbp; ++kb) {
                    if (!mbar_wait_bounded(bar_addr(&ctl->empty[stage]), phase ^ 1u, abort_flag, p.wait_limit_ns,
                                           p.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = bar_addr(&ctl->full[stage]);
                    mbar_arrive_expect_tx(fb, kATileBytes + kStdBTileBytes);
                    const int k = (p.kb_first + t.group * p.kb_group_stride + kb) * 64;
                    tma_load_2d_nohint(sA + stage * kATileBytes, &tmA, fb, k, t.m * 128);
                    if constexpr (EPI == EPI_SWIGLU)
                        tma_load_3d_nohint(sB + stage * kStdBTileBytes, &tmB, fb, k, p.n_base + t.n * 128, 0);
                    else
                        tma_load_2d_nohint(sB + stage * kStdBTileBytes, &tmB, fb, k, t.n * 256);
                    ++issued;
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, 256);
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int64_t id = blockIdx.x; id < n_tiles && ok; id += gridDim.x, ++it) {
                const int buf = it & 1;
                const uint32_t use = (uint32_t)(it >> 1);
                if (!mbar_wait_bounded(bar_addr(&ctl->tempty[buf]), (use & 1u) ^ 1u, abort_flag, p.wait_limit_ns,
                                       p.err))
                    break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(buf * 256);
                for (int kb = 0; kb < kbp; ++kb) {
                    if (!mbar_wait_bounded(bar_addr(&ctl->full[stage]), phase, abort_flag, p.wait_limit_ns, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = smem_desc_sw128(sA + stage * kATileBytes);
                    const uint64_t bd = smem_desc_sw128(sB + stage * kStdBTileBytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_bf16(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc,
                                    (kb > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(bar_addr(&ctl->empty[stage]));
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit(bar_addr(&ctl->tfull[buf]));
            }
        }
    } else {
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        pdl_wait();
        int it = 0;
        for (int64_t id = blockIdx.x; id < n_tiles; id += gridDim.x, ++it) {
            const StdTile t = std_tile(p, id);
            const int buf = it & 1;
            const uint32_t use = (uint32_t)(it >> 1);
            const bool got = mbar_wait_bounded(bar_addr(&ctl->tfull[buf]), use & 1u, abort_flag, p.wait_limit_ns, p.err);
            if (!named_barrier_and(1, 128, got)) break;
            tc_fence_after();
            const uint32_t tacc = tmem_base + (uint32_t)(buf * 256) + lane_off;
            const int64_t tok = (int64_t)t.m * 128 + row;
            const bool tok_ok = tok < p.T;
            if constexpr (EPI == EPI_SWIGLU) {
                uint16_t *h = static_cast<uint16_t *>(p.out);
                const int64_t j0 = (int64_t)p.n_base + (int64_t)t.n * 128;
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                    float g[16], u[16];
                    load_tmem_chunk(tacc + (uint32_t)(c * 16), g);
                    load_tmem_chunk(tacc + (uint32_t)(128 + c * 16), u);
                    const int64_t j = j0 + c * 16;
                    if (tok_ok && j < p.n_valid) {
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            w[i] = (uint32_t)f32_to_bf16_bits(silu_f32(g[2 * i]) * u[2 * i]) |
                                   ((uint32_t)f32_to_bf16_bits(silu_f32(g[2 * i + 1]) * u[2 * i + 1]) << 16);
                        uint4 *dst = reinterpret_cast<uint4 *>(h + tok * p.ldo + j);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < 16; ++c) {
                    float v[16];
                    load_tmem_chunk(tacc + (uint32_t)(c * 16), v);
                    const int64_t n = (int64_t)t.n * 256 + c * 16;
                    if (!tok_ok || n >= p.n_valid) continue;
                    if constexpr (EPI == EPI_F32) {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) +
                                                                 t.group * p.o_group_stride + tok * p.ldo + n);
#pragma unroll
                        for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    } else if constexpr (EPI == EPI_BF16) {
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            w[i] = (uint32_t)f32_to_bf16_bits(v[2 * i]) | ((uint32_t)f32_to_bf16_bits(v[2 * i + 1]) << 16);
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) +
                                                               t.group * p.o_group_stride + tok * p.ldo + n);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    } else {  // EPI_MERGED
                        uint16_t *lo = static_cast<uint16_t *>(p.out);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int64_t col = n + i;
                            if (col >= p.n_valid) break;
                            const uint16_t b = f32_to_bf16_bits(v[i]);
                            if (lo) lo[tok * p.ldo + col] = b;
                            if (p.out_rm) p.out_rm[tok * p.ldo + logical_to_gathered(col, p.q_dim, p.kv_dim, p.tp)] = b;
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar_addr(&ctl->tempty[buf]));
        }
    }

    if (warp == 0 && lane == 0) {
        const int64_t first = issued > S ? issued - S : 0;
        for (int64_t i = first; i < issued; ++i)
            (void)mbar_wait_drain(bar_addr(&ctl->full[i % S]), (uint32_t)((i / S) & 1), p.wait_limit_ns);
    }
    if (warp == 1 && lane == 0) {
        tc_commit(bar_addr(&ctl->drain));
        (void)mbar_wait_drain(bar_addr(&ctl->drain), 0, p.wait_limit_ns);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}


// ---------------------------------------------------------------------------
// CTA-pair persistent kernel (cta_group::2): tile = 256 tokens x 256 columns.
// Each CTA of a cluster pair loads its own 128 token rows (A) and its own half of
// the 256 B rows, and holds the accumulator rows of its tokens in its own TMEM;
// the even CTA issues the MMAs for both.  Per SM this halves the operand bytes
// per FLOP against the single-CTA 128 x 256 tile.
// ---------------------------------------------------------------------------
constexpr uint32_t kPairBTileBytes = 128 * 64 * 2;
constexpr int kPairBandM = 8;

template <int EPI>
__global__ void __launch_bounds__(kStdThreads, 1)
    pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const StdParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int S = p.stages;
    const uint32_t sA = base;
    const uint32_t sB = base + (uint32_t)S * kATileBytes;
    Ctrl *ctl = reinterpret_cast<Ctrl *>(smem_raw + (base - raw) + (uint32_t)S * (kATileBytes + kPairBTileBytes));
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int64_t cluster = blockIdx.x / 2, n_clusters = gridDim.x / 2;
    const int64_t n_tiles = (int64_t)p.n_groups * p.n_mtiles * p.n_ntiles;
    const int kbp = p.kb_per_tile;
    constexpr uint32_t kTmemCols = 512;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_addr(&ctl->full[s]), 1);
            mbar_init(bar_addr(&ctl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_addr(&ctl->tfull[b]), 1);
            mbar_init(bar_addr(&ctl->tempty[b]), 8);   // 4 epilogue warps x 2 CTAs
        }
        mbar_init(bar_addr(&ctl->drain), 1);
        ctl->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(&ctl->tmem_base), kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();        // the peer's barriers are initialised before any remote use
    tc_fence_after();
    const uint32_t tmem_base = ctl->tmem_base;
    volatile int *abort_flag = &ctl->abort_flag;
    pdl_launch_dependents();

    auto tile_of = [&](int64_t id) {
        StdTile t;
        const int64_t per_group = (int64_t)p.n_mtiles * p.n_ntiles;
        t.group = (int)(id / per_group);
        const int64_t r = id % per_group;
        const int64_t per_band = (int64_t)kPairBandM * p.n_ntiles;
        const int band = (int)(r / per_band);
        const int first_m = band * kPairBandM;
        const int band_m = min(kPairBandM, p.n_mtiles - first_m);
        const int64_t in_band = r % per_band;
        t.m = first_m + (int)(in_band % band_m);
        t.n = (int)(in_band / band_m);
        return t;
    };

    int64_t issued = 0;
    if (warp == 0) {
        if (lane == 0) {
            pdl_wait();
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int64_t id = cluster; id < n_tiles && ok; id += n_clusters) {
                const StdTile t = tile_of(id);
                for (int kb = 0; kb < kbp; ++kb) {
                    if (!mbar_wait_bounded(bar_addr(&ctl->empty[stage]), phase ^ 1u, abort_flag, p.wait_limit_ns,
                                           p.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = map_to_rank(bar_addr(&ctl->full[stage]), 0);
                    if (leader) mbar_arrive_expect_tx(bar_addr(&ctl->full[stage]), 2u * (kATileBytes + kPairBTileBytes));
                    const int k = (p.kb_first + t.group * p.kb_group_stride + kb) * 64;
                    tma_load_2d_pair(sA + stage * kATileBytes, &tmA, fb, k, t.m * 256 + (int)rank * 128);
                    tma_load_2d_pair(sB + stage * kPairBTileBytes, &tmB, fb, k,
                                     p.b_base + t.n * p.b_n_stride + (int)rank * p.b_rank_stride);
                    ++issued;
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            const uint32_t idesc = idesc_bf16_f32(256, 256);
            int stage = 0;
            uint32_t phase = 0;
            int it = 0;
            bool ok = true;
            for (int64_t id = cluster; id < n_tiles && ok; id += n_clusters, ++it) {
                const int buf = it & 1;
                const uint32_t use = (uint32_t)(it >> 1);
                if (!mbar_wait_bounded(bar_addr(&ctl->tempty[buf]), (use & 1u) ^ 1u, abort_flag, p.wait_limit_ns,
                                       p.err))
                    break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(buf * 256);
                for (int kb = 0; kb < kbp; ++kb) {
                    if (!mbar_wait_bounded(bar_addr(&ctl->full[stage]), phase, abort_flag, p.wait_limit_ns, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = smem_desc_sw128(sA + stage * kATileBytes);
                    const uint64_t bd = smem_desc_sw128(sB + stage * kPairBTileBytes);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_bf16_pair(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc,
                                         (kb > 0 || kk > 0) ? 1u : 0u);
                    tc_commit_pair_multicast(bar_addr(&ctl->empty[stage]), (uint16_t)0x3);
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                tc_commit_pair_multicast(bar_addr(&ctl->tfull[buf]), (uint16_t)0x3);
            }
        }
    } else {
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t lane_off = (uint32_t)(q * 32) << 16;
        pdl_wait();
        int it = 0;
        for (int64_t id = cluster; id < n_tiles; id += n_clusters, ++it) {
            const StdTile t = tile_of(id);
            const int buf = it & 1;
            const uint32_t use = (uint32_t)(it >> 1);
            const bool got = mbar_wait_bounded(bar_addr(&ctl->tfull[buf]), use & 1u, abort_flag, p.wait_limit_ns, p.err);
            if (!named_barrier_and(1, 128, got)) break;
            tc_fence_after();
            const uint32_t tacc = tmem_base + (uint32_t)(buf * 256) + lane_off;
            const int64_t tok = (int64_t)t.m * 256 + rank * 128 + row;
            const bool tok_ok = tok < p.T;
            if constexpr (EPI == EPI_SWIGLU) {
                uint16_t *h = static_cast<uint16_t *>(p.out);
                const int64_t j0 = (int64_t)p.n_base + (int64_t)t.n * 128;
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {
                    float g[16], u[16];
                    load_tmem_chunk(tacc + (uint32_t)(c * 16), g);
                    load_tmem_chunk(tacc + (uint32_t)(128 + c * 16), u);
                    const int64_t j = j0 + c * 16;
                    if (tok_ok && j < p.n_valid) {
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            w[i] = (uint32_t)f32_to_bf16_bits(silu_f32(g[2 * i]) * u[2 * i]) |
                                   ((uint32_t)f32_to_bf16_bits(silu_f32(g[2 * i + 1]) * u[2 * i + 1]) << 16);
                        uint4 *dst = reinterpret_cast<uint4 *>(h + tok * p.ldo + j);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < 16; ++c) {
                    float v[16];
                    load_tmem_chunk(tacc + (uint32_t)(c * 16), v);
                    const int64_t n = (int64_t)t.n * 256 + c * 16;
                    if (!tok_ok || n >= p.n_valid) continue;
                    if constexpr (EPI == EPI_F32) {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) +
                                                                 t.group * p.o_group_stride + tok * p.ldo + n);
#pragma unroll
                        for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    } else if constexpr (EPI == EPI_BF16) {
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            w[i] = (uint32_t)f32_to_bf16_bits(v[2 * i]) | ((uint32_t)f32_to_bf16_bits(v[2 * i + 1]) << 16);
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) +
                                                               t.group * p.o_group_stride + tok * p.ldo + n);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    } else {  // EPI_MERGED
                        uint16_t *lo = static_cast<uint16_t *>(p.out);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int64_t col = n + i;
                            if (col >= p.n_valid) break;
                            const uint16_t b = f32_to_bf16_bits(v[i]);
                            if (lo) lo[tok * p.ldo + col] = b;
                            if (p.out_rm) p.out_rm[tok * p.ldo + logical_to_gathered(col, p.q_dim, p.kv_dim, p.tp)] = b;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_rank(bar_addr(&ctl->tempty[buf]), 0));
        }
    }

    // ---- teardown ----
    if (warp == 0 && lane == 0) {
        // every issued stage is released by the leader's MMA commit once its bytes
        // (from both CTAs) have landed and been consumed
        const int64_t first = issued > S ? issued - S : 0;
        for (int64_t i = first; i < issued; ++i) {
            const bool done = mbar_wait_drain(bar_addr(&ctl->empty[i % S]), (uint32_t)((i / S) & 1), p.wait_limit_ns);
            if (!done) __nanosleep(200000);   // abort path: let in-flight copies land
        }
    }
    if (warp == 1 && lane == 0 && leader) {
        tc_commit_pair_multicast(bar_addr(&ctl->drain), (uint16_t)0x1);
        (void)mbar_wait_drain(bar_addr(&ctl->drain), 0, p.wait_limit_ns);
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

// Opt the kernel into the largest dynamic shared memory once per device.
template <typename Kern>
cudaError_t ensure_smem_attr(Kern kern, int slot) {
    static std::atomic<uint64_t> done[16];   // bit per device, per kernel slot
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = 1ull << (dev & 63);
    if (done[slot].load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e == cudaSuccess) done[slot].fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

}  // namespace

size_t swapab_smem_bytes(int bn, int stages, int kbs) {
    return (size_t)stages * kbs * (kATileBytes + (size_t)bn * 128) + 1024 + sizeof(Ctrl);
}
size_t std_smem_bytes(int stages) { return (size_t)stages * (kATileBytes + kStdBTileBytes) + 1024 + sizeof(Ctrl); }

int swapab_stages_for(int bn, int kbs) {
    const size_t budget = 227 * 1024 - 1024 - sizeof(Ctrl) - 64;
    int st = (int)(budget / ((size_t)kbs * (kATileBytes + (size_t)bn * 128)));
    return st > kMaxStages ? kMaxStages : st;
}
int std_stages() { return 4; }

cudaError_t launch_swapab(int epi, const CUtensorMap &ta, const CUtensorMap &tb, const SwapAbParams &p, int grid,
                          bool pdl, cudaStream_t s) {
    const size_t smem = swapab_smem_bytes(p.bn, p.stages, p.kbs);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)kSwapAbThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e;
    switch (epi) {
        case EPI_SWIGLU:
            e = ensure_smem_attr(swapab_kernel<EPI_SWIGLU>, 0);
            if (e != cudaSuccess) return e;
            return cudaLaunchKernelEx(&cfg, swapab_kernel<EPI_SWIGLU>, ta, tb, p);
        case EPI_BF16:
            e = ensure_smem_attr(swapab_kernel<EPI_BF16>, 1);
            if (e != cudaSuccess) return e;
            return cudaLaunchKernelEx(&cfg, swapab_kernel<EPI_BF16>, ta, tb, p);
        case EPI_F32:
            e = ensure_smem_attr(swapab_kernel<EPI_F32>, 2);
            if (e != cudaSuccess) return e;
            return cudaLaunchKernelEx(&cfg, swapab_kernel<EPI_F32>, ta, tb, p);
        default:
            e = ensure_smem_attr(swapab_kernel<EPI_MERGED>, 3);
            if (e != cudaSuccess) return e;
            return cudaLaunchKernelEx(&cfg, swapab_kernel<EPI_MERGED>, ta, tb, p);
    }
}

cudaError_t launch_std(int epi, const CUtensorMap &ta, const CUtensorMap &tb, const StdParams &p, int grid, bool pdl,
                       cudaStream_t s) {
    const size_t smem = std_smem_bytes(p.stages);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)kStdThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e;
    switch (epi) {
        case EPI_SWIGLU:
            e = ensure_smem_attr(std_kernel<EPI_SWIGLU>, 4);
            if (e != cudaSuccess) return e;
            return cudaLaunchKernelEx(&cfg, std_kernel<EPI_SWIGLU>, ta, tb, p);
        case EPI_BF16:
            e = ensure_smem_attr(std_kernel<EPI_BF16>, 5);
            if (e != cudaSuccess) return e;
            return cudaLaunchKernelEx(&cfg, std_kernel<EPI_BF16>, ta, tb, p);
        case EPI_F32:
            e = ensure_smem_attr(std_kernel<EPI_F32>, 6);
            if (e != cudaSuccess) return e;
            return cudaLaunchKernelEx(&cfg, std_kernel<EPI_F32>, ta, tb, p);
        default:
            e = ensure_smem_attr(std_kernel<EPI_MERGED>, 7);
            if (e != cudaSuccess) return e;
            return cudaLaunchKernelEx(&cfg, std_kernel<EPI_MERGED>, ta, tb, p);
    }
}


size_t pair_smem_bytes(int stages) { return (size_t)stages * (kATileBytes + kPairBTileBytes) + 1024 + sizeof(Ctrl); }
int pair_stages() { return 6; }

cudaError_t launch_pair(int epi, const CUtensorMap &ta, const CUtensorMap &tb, const StdParams &p, int clusters,
                        bool pdl, cudaStream_t s) {
    const size_t smem = pair_smem_bytes(p.stages);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * clusters));
    cfg.blockDim = dim3((unsigned)kStdThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    cudaError_t e;
    // one wave: no more clusters than can be resident at once
    {
        static std::atomic<int> max_clusters[64];
        int dev = 0;
        if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
        int mc = max_clusters[dev & 63].load();
        if (mc == 0) {
            if ((e = ensure_smem_attr(pair_kernel<EPI_BF16>, 9)) != cudaSuccess) return e;
            cudaLaunchConfig_t q = cfg;
            q.numAttrs = 1;
            q.gridDim = dim3(2);
            if ((e = cudaOccupancyMaxActiveClusters(&mc, pair_kernel<EPI_BF16>, &q)) != cudaSuccess) return e;
            if (mc < 1) mc = 1;
            max_clusters[dev & 63].store(mc);
        }
        if (clusters > mc) cfg.gridDim = dim3((unsigned)(2 * mc));
    }
    switch (epi) {
        case EPI_SWIGLU:
            e = ensure_smem_attr(pair_kernel<EPI_SWIGLU>, 8);
            if (e != cudaSuccess) return e;
            return cudaLaunchKernelEx(&cfg, pair_kernel<EPI_SWIGLU>, ta, tb, p);
        case EPI_BF16:
            e = ensure_smem_attr(pair_kernel<EPI_BF16>, 9);
            if (e != cudaSuccess) return e;
            return cudaLaunchKernelEx(&cfg, pair_kernel<EPI_BF16>, ta, tb, p);
        case EPI_F32:
            e = ensure_smem_attr(pair_kernel<EPI_F32>, 10);
            if (e != cudaSuccess) return e;
            return cudaLaunchKernelEx(&cfg, pair_kernel<EPI_F32>, ta, tb, p);
        default:
            e = ensure_smem_attr(pair_kernel<EPI_MERGED>, 11);
            if (e != cudaSuccess) return e;
            return cudaLaunchKernelEx(&cfg, pair_kernel<EPI_MERGED>, ta, tb, p);
    }
}

}  // namespace tc
}  // namespace mse
