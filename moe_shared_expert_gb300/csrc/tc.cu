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
    uint64_t go_bar;         // swap-AB cluster finish: the receiving CTA's ring is free
    uint64_t recv_bar;       // swap-AB cluster finish: the sending CTA's part has landed
    uint64_t hready_bar;     // swap-AB down with h flags: every h block the CTA reads is published
    uint32_t tmem_base;
    int abort_flag;
    int fin_flag;
    int x_ticket;            // swap-AB gate_up with x in host memory: this CTA's copy ticket
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
        // Rows 32q .. 32q+15 are the gate rows of j = j0 + 16q + (lane & 15), rows 32q+16 ..
        // 32q+31 the up rows of the same j, so lane l < 16 pairs with lane l + 16 of the same
        // warp.  The gate lane computes tokens 0-7 of the chunk and the up lane tokens 8-15,
        // each taking its partner's half by a register shuffle.
        (void)ctl;
        const bool is_gate = lane < 16;
        float other[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) other[i] = __shfl_xor_sync(0xffffffffu, is_gate ? v[8 + i] : v[i], 16);
        const int64_t j = (int64_t)p.a_row_base + (int64_t)m * 64 + 16 * q + (lane & 15);
        const int t0 = c * 16 + (is_gate ? 0 : 8);
        uint16_t hv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float g = is_gate ? v[i] : other[i];
            const float u = is_gate ? other[i] : v[8 + i];
            hv[i] = f32_to_bf16_bits(silu_f32(g) * u);
        }
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

// Epilogue of token columns [t0, t1) of a swap-AB tile held in shared memory as fp32
// [token][row] (row = accumulator row, 128 per token; tilebuf starts at column t0).
// All 128 epilogue threads (tid 0..127) work element-wise: a fixed row per thread,
// tokens strided, so shared reads are conflict-free and the 32 lanes of a warp store
// 32 consecutive outputs.
template <int EPI>
__device__ __forceinline__ void swapab_epilogue_smem(const SwapAbParams &p, const float *tilebuf, int group, int m,
                                                     int tid, int t0, int t1) {
    if (t1 > p.T) t1 = p.T;
    if constexpr (EPI == EPI_SWIGLU) {
        // j = j0 + jr: its gate row is 32 (jr / 16) + jr % 16, its up row 16 further
        const int jr = tid & 63;
        const int gr = 32 * (jr >> 4) + (jr & 15);
        uint16_t *h = static_cast<uint16_t *>(p.out) + (int64_t)p.a_row_base + (int64_t)m * 64 + jr;
        int t = t0 + (tid >> 6);
        for (; t + 6 < t1; t += 8) {   // 4 tokens per step, computed before storing
            uint16_t hv[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const float *c = tilebuf + (t + 2 * r - t0) * 128;
                hv[r] = f32_to_bf16_bits(silu_f32(c[gr]) * c[gr + 16]);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) h[(int64_t)(t + 2 * r) * p.ldo] = hv[r];
        }
        for (; t < t1; t += 2) {
            const float *c = tilebuf + (t - t0) * 128;
            h[(int64_t)t * p.ldo] = f32_to_bf16_bits(silu_f32(c[gr]) * c[gr + 16]);
        }
    } else {
        const int64_t n = (int64_t)m * 128 + tid;
        if (n >= p.m_valid) return;
        if constexpr (EPI == EPI_F32) {
            float *o = static_cast<float *>(p.out) + group * p.o_group_stride + n;
            for (int t = t0; t < t1; ++t) o[(int64_t)t * p.ldo] = tilebuf[(t - t0) * 128 + tid];
        } else if constexpr (EPI == EPI_BF16) {
            uint16_t *o = static_cast<uint16_t *>(p.out) + group * p.o_group_stride + n;
            int t = t0;
            for (; t + 3 < t1; t += 4) {
                uint16_t b[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) b[r] = f32_to_bf16_bits(tilebuf[(t + r - t0) * 128 + tid]);
#pragma unroll
                for (int r = 0; r < 4; ++r) o[(int64_t)(t + r) * p.ldo] = b[r];
            }
            for (; t < t1; ++t) o[(int64_t)t * p.ldo] = f32_to_bf16_bits(tilebuf[(t - t0) * 128 + tid]);
        } else {
            uint16_t *lo = static_cast<uint16_t *>(p.out);
            const int64_t gcol = logical_to_gathered(n, p.q_dim, p.kv_dim, p.tp);
            for (int t = t0; t < t1; ++t) {
                const uint16_t b = f32_to_bf16_bits(tilebuf[(t - t0) * 128 + tid]);
                if (lo) lo[(int64_t)t * p.ldo + n] = b;
                if (p.out_rm) p.out_rm[(int64_t)t * p.ldo + gcol] = b;
            }
        }
    }
}

// Teardown waits for copies and MMAs that were issued and will complete; they get at
// least 100 ms even when the wait limit of the pipeline is set shorter.
__device__ __forceinline__ uint64_t drain_limit_ns(uint64_t limit) {
    return limit > 100000000ull ? limit : 100000000ull;
}

// Position in the shared-memory ring (stage index and the parity of its current use).
struct RingPos {
    int stage = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next(int S) {
        if (++stage == S) { stage = 0; phase ^= 1u; }
    }
};

// Shared-memory layout of the swap-AB ring: stage s holds [kbs weight tiles of
// 128 x 64][kbs token tiles of bn x 64], 1024-byte aligned (128-byte swizzle atoms).
struct SwapAbSmem {
    uint32_t base, stage_bytes, a_stage_bytes, b_tile_bytes;
    __device__ __forceinline__ SwapAbSmem(uint32_t base_, int bn, int kbs) {
        base = base_;
        b_tile_bytes = (uint32_t)bn * 128u;
        a_stage_bytes = (uint32_t)kbs * kATileBytes;
        stage_bytes = a_stage_bytes + (uint32_t)kbs * b_tile_bytes;
    }
    __device__ __forceinline__ uint32_t a(int st) const { return base + (uint32_t)st * stage_bytes; }
    __device__ __forceinline__ uint32_t b(int st) const { return a(st) + a_stage_bytes; }
};

// The work of one CTA in one pass.  The pass's units are (tile, u), u in [0, kbu), split
// stream-K over the grid; the CTA's range [ub, ue) touches `nseg` consecutive tiles (its
// segments).  With halves == 1 unit u is k-block u of the tile and a segment is one run
// of k-blocks.  With halves == 2 unit u stands for the two k-blocks u and kbu + u: each
// segment is processed as two runs (first halves, then second halves), and when the CTA
// touches at most two tiles the first halves of all its segments come before the second
// halves, so that both of its accumulators are open at once.
struct Plan {
    int64_t ub, ue, tile0;
    int kbu, halves, n_mtiles, nseg;
    bool inter;
    // worker w of nw: a CTA, or a CTA pair (both CTAs of a pair share the plan)
    __device__ void init(const SwapAbParams &p, int64_t w, int64_t nw) {
        const StreamK sk{p.total_units, nw};
        ub = sk.begin(w);
        ue = sk.begin(w + 1);
        kbu = p.kb_per_tile;
        halves = p.halves;
        n_mtiles = p.n_mtiles;
        tile0 = ub / kbu;
        nseg = ue > ub ? (int)((ue - 1) / kbu - tile0 + 1) : 0;
        inter = halves == 2 && nseg <= 2;
    }
    __device__ int nruns() const { return nseg * halves; }
    __device__ void run(int r, int &seg, int &half) const {
        if (halves == 1) { seg = r; half = 0; }
        else if (inter) { half = r >= nseg ? 1 : 0; seg = r - half * nseg; }
        else { seg = r >> 1; half = r & 1; }
    }
    // tile of segment s and its unit range [kb0, kb1) within the tile
    __device__ void seg_range(int s, int64_t &tile, int &kb0, int &kb1) const {
        tile = tile0 + s;
        const int64_t t0 = tile * kbu;
        kb0 = (int)(ub > t0 ? ub - t0 : 0);
        kb1 = (int)(ue < t0 + kbu ? ue - t0 : kbu);
    }
};

// The stream-K worker of this CTA: the CTA itself, or its pair (clusters of two CTAs,
// both take the same units, each its own 128-row half of the 256-row weight tile).
template <bool PAIR>
__device__ __forceinline__ int64_t worker_index() { return PAIR ? blockIdx.x / 2 : blockIdx.x; }
template <bool PAIR>
__device__ __forceinline__ int64_t worker_count() { return PAIR ? gridDim.x / 2 : gridDim.x; }
template <bool PAIR>
__device__ __forceinline__ uint32_t pair_rank() { return PAIR ? cluster_ctarank() : 0u; }

// Stages of a Plan in order: runs cut into stages of up to kbs k-blocks.
struct StageIter {
    const Plan *pl;
    int r, nr;            // current run, number of runs
    int kb, kb1;          // stage start and run end (units within the tile)
    int half, group, m;   // of the current run
    __device__ void start(const Plan &p) {
        pl = &p;
        nr = p.nruns();
        r = -1;
        kb = kb1 = 0;
        next_run();
    }
    __device__ void next_run() {
        while (kb >= kb1 && ++r < nr) {
            int seg;
            pl->run(r, seg, half);
            int64_t tile;
            pl->seg_range(seg, tile, kb, kb1);
            group = (int)(tile / pl->n_mtiles);
            m = (int)(tile - (int64_t)group * pl->n_mtiles);
        }
    }
    __device__ bool done() const { return r >= nr; }
    __device__ int count(int kbs) const { return (kb1 - kb) < kbs ? (kb1 - kb) : kbs; }
    __device__ void advance(int n) {
        kb += n;
        if (kb >= kb1) next_run();
    }
    // k-block index, within the group's reduction, of the i-th k-block of the stage
    __device__ int kblock(int i) const { return half * pl->kbu + kb + i; }
};

// ---- producer (one elected thread of warp 0) ----
// pdl_prologue: the weight tiles of the first stages are requested before waiting for
//   the previous kernel of the stream, the token tiles after that wait (first pass).
// hflags: the token operand is the intermediate h written earlier in this launch; a
//   stage's token tiles are requested once every gate_up tile they read has been
//   published there, while weight tiles keep filling the free stages meanwhile.
// `issued` counts stages whose loads were requested.  Returns false after an abort.
// The h flags of a launch: flags[first + t] is set once the gate_up tile writing h
// columns 64 (first + t) .. is published; tiles t < n0 belong to gate_up pass 0, the
// next n1 to pass 1, and counts[k] is the number of tiles pass k has published.
struct HFlags {
    const int *flags;
    const int *counts;
    int first, n0, n1;
};

// PAIR: each CTA of the pair loads its own weight rows (m-tile 2 m' + rank of pair tile
// m') and its half of the token rows; both signal the first CTA's full barriers, which
// expect the bytes of both.
template <int EPI, bool PAIR = false>
__device__ bool swapab_produce(const SwapAbParams &p, const CUtensorMap *tmA, const CUtensorMap *tmB, Ctrl *ctl,
                               const SwapAbSmem &sm, RingPos &r, int &issued, bool pdl_prologue, const HFlags *hf,
                               volatile int *abort_flag) {
    const int S = p.stages, KBS = p.kbs;
    const uint32_t rank = pair_rank<PAIR>();
    const bool leader = rank == 0;
    const uint32_t kb_tx = (PAIR ? 2u : 1u) * (kATileBytes + sm.b_tile_bytes);   // per k-block, both CTAs
    const int b_row0 = PAIR ? (int)rank * (p.bn / 2) : 0;
    auto mreal = [&](int m) { return PAIR ? 2 * m + (int)rank : m; };
    auto fbar = [&](int st) {
        return PAIR ? map_to_rank(bar_addr(&ctl->full[st]), 0) : bar_addr(&ctl->full[st]);
    };
    auto expect = [&](int st, int n) {
        if (!PAIR || leader) mbar_arrive_expect_tx(bar_addr(&ctl->full[st]), (uint32_t)n * kb_tx);
    };
    auto tma2d = [&](uint32_t dst, const CUtensorMap *map, uint32_t fb, int c0, int c1, uint64_t pol, bool hint) {
        if constexpr (PAIR) {
            tma_load_2d_pair_hint(dst, map, fb, c0, c1, pol);
            (void)hint;
        } else {
            if (hint) tma_load_2d(dst, map, fb, c0, c1, pol);
            else tma_load_2d_nohint(dst, map, fb, c0, c1);
        }
    };
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_x = l2_policy_evict_last();
    const bool hints = p.cache_hints != 0;
    auto kglob = [&](const StageIter &w, int i) { return p.kb_first + w.group * p.kb_group_stride + w.kblock(i); };
    auto load_a = [&](const StageIter &w, int n, int st) {
        const uint32_t fb = fbar(st);
        for (int i = 0; i < n; ++i) {
            const int k = kglob(w, i) * 64;
            const uint32_t dst = sm.a(st) + (uint32_t)i * kATileBytes;
            if constexpr (EPI == EPI_SWIGLU) {
                // one box of the (k, row, gate/up, 16-row block) view of W_gate_up: rows
                // 32b .. 32b+15 are the gate rows of j = j0 + 16b .., rows 32b+16 .. 32b+31
                // the up rows of the same j (b = 0..3)
                const int jb0 = (p.a_row_base + mreal(w.m) * 64) / 16;
                if constexpr (PAIR) {
                    tma_load_4d_pair_hint(dst, tmA, fb, k, 0, 0, jb0, pol_w);
                } else {
                    if (hints) tma_load_4d(dst, tmA, fb, k, 0, 0, jb0, pol_w);
                    else tma_load_4d_nohint(dst, tmA, fb, k, 0, 0, jb0);
                }
            } else {
                tma2d(dst, tmA, fb, k, mreal(w.m) * 128, pol_w, hints);
            }
        }
    };
    auto load_b = [&](const StageIter &w, int n, int st) {
        const uint32_t fb = fbar(st);
        for (int i = 0; i < n; ++i) {
            const int k = kglob(w, i) * 64;
            const uint32_t dst = sm.b(st) + (uint32_t)i * sm.b_tile_bytes;
            tma2d(dst, tmB, fb, k, b_row0, pol_x, hints);
        }
    };
    Plan pl;
    pl.init(p, worker_index<PAIR>(), worker_count<PAIR>());
    StageIter w;
    w.start(pl);
    if (pdl_prologue && !p.x_early) {
        // the ring is fresh: stages 0.. in their first use
        StageIter a = w;
        int st = 0;
        for (; st < S && !a.done(); ++st) {
            const int n = a.count(KBS);
            expect(st, n);
            load_a(a, n, st);
            a.advance(n);
        }
        if (!PAIR && p.l2_prefetch_kb > 0 && (int)blockIdx.x >= p.l2_prefetch_from) {
            // the next weight tiles into L2 while the previous kernel finishes
            int left = p.l2_prefetch_kb;
            while (left > 0 && !a.done()) {
                const int n = a.count(KBS) < left ? a.count(KBS) : left;
                for (int i = 0; i < n; ++i) {
                    const int k = kglob(a, i) * 64;
                    if constexpr (EPI == EPI_SWIGLU)
                        tma_prefetch_l2_4d(tmA, k, 0, 0, (p.a_row_base + a.m * 64) / 16);
                    else
                        tma_prefetch_l2_2d(tmA, k, a.m * 128);
                }
                a.advance(n);
                left -= n;
            }
        }
        bool flags_ok = true;
        if ((EPI != EPI_SWIGLU && p.hflags) || (EPI == EPI_SWIGLU && p.x_host)) {
            // the epilogue warps poll the flags of every h block this CTA reads (no wait for
            // the gate_up grid to complete), or the count of copied slices of x, and arrive
            // here once the token operand is complete
            flags_ok = mbar_wait_bounded(bar_addr(&ctl->hready_bar), 0u, abort_flag, p.wait_limit_ns, p.err);
            fence_proxy_async_global();   // written through the generic proxy
        } else {
            pdl_wait();
        }
        for (int t = 0; t < st; ++t) {
            const int n = w.count(KBS);
            load_b(w, n, t);
            w.advance(n);
        }
        if (!flags_ok) {
            issued += st;
            return false;
        }
        issued += st;
        r.stage = st == S ? 0 : st;
        r.phase = st == S ? 1u : 0u;
    }
    if (!hf) {
        while (!w.done()) {
            if (!mbar_wait_bounded(bar_addr(&ctl->empty[r.stage]), r.phase ^ 1u, abort_flag, p.wait_limit_ns, p.err,
                                   p.spin_wait != 0))
                return false;
            const int n = w.count(KBS);
            expect(r.stage, n);
            load_a(w, n, r.stage);
            load_b(w, n, r.stage);
            w.advance(n);
            ++issued;
            r.next(S);
        }
        return true;
    }
    // Two cursors over the same stages: `w` requests weight tiles into free stages, `wb`
    // follows with the token tiles once their h columns are published.  After an abort
    // the pending token tiles are still requested (without waiting) so that every
    // issued stage completes and the teardown drain ends.
    // Readiness is read with relaxed loads, at most every 256 ns (polling harder slows the
    // publishers): first the published counts of the passes the stage reads; a pass
    // found complete is never read again; while one is not, the stage's flags of that
    // pass.  One fence follows the poll that finds the stage ready.
    StageIter wb = w;
    RingPos rb = r;
    int pending = 0;
    bool aborted = false;
    bool done0 = hf->n0 == 0, done1 = hf->n1 == 0;   // pass complete
    uint64_t next_poll = 0;
    uint64_t idle_since = 0;
    while (true) {
        bool progress = false;
        if (!aborted && !w.done() && mbar_test_wait(bar_addr(&ctl->empty[r.stage]), r.phase ^ 1u)) {
            const int n = w.count(KBS);
            expect(r.stage, n);
            load_a(w, n, r.stage);
            w.advance(n);
            ++issued;
            r.next(S);
            ++pending;
            progress = true;
        }
        if (pending > 0) {
            const int n = wb.count(KBS);
            bool ready = true;
            if (!aborted) {
                int fi[kMaxKbs];
                bool in1[kMaxKbs];
                bool need0 = false, need1 = false;
#pragma unroll
                for (int i = 0; i < kMaxKbs; ++i) {
                    fi[i] = i < n ? kglob(wb, i) : hf->first;
                    in1[i] = fi[i] >= hf->first + hf->n0;
                    if (i < n) {
                        if (in1[i]) need1 = need1 || !done1;
                        else need0 = need0 || !done0;
                    }
                }
                if (need0 || need1) {
                    ready = false;
                    const uint64_t now = global_timer_ns();
                    if (now >= next_poll) {
                        const int c0 = need0 ? ld_relaxed_gpu(hf->counts) : 0;
                        const int c1 = need1 ? ld_relaxed_gpu(hf->counts + 1) : 0;
                        if (need0 && c0 >= hf->n0) done0 = true;
                        if (need1 && c1 >= hf->n1) done1 = true;
                        bool all = true;
#pragma unroll
                        for (int i = 0; i < kMaxKbs; ++i)
                            if (i < n && !(in1[i] ? done1 : done0)) all = all && ld_relaxed_gpu(hf->flags + fi[i]) != 0;
                        if (all) {
                            fence_acq_rel_gpu();   // acquire the publishers' h stores
                            ready = true;
                        } else {
                            next_poll = now + 256;
                        }
                    }
                }
            }
            if (ready) {
                fence_proxy_async_global();   // h was written through the generic proxy
                load_b(wb, n, rb.stage);
                wb.advance(n);
                rb.next(S);
                --pending;
                progress = true;
            }
        } else if (w.done() || aborted) {
            break;
        }
        if (progress) {
            idle_since = 0;
            continue;
        }
        if (*abort_flag) {
            aborted = true;
            continue;
        }
        const uint64_t now = global_timer_ns();
        if (idle_since == 0) {
            idle_since = now;
        } else if (now - idle_since > p.wait_limit_ns) {
            *abort_flag = 1;
            raise_device_error(p.err, DEV_ERR_TIMEOUT);
            aborted = true;
        }
    }
    return !aborted;
}

// ---- MMA issuer (one elected thread of warp 1) ----
// Segment s of the pass accumulates in TMEM buffer (gseg + s) & 1, gseg counting the
// segments of earlier passes; its first run starts the accumulator, its last run
// hands it to the epilogue.
// PAIR: run by the first CTA of the pair only; each MMA covers both CTAs' weight rows
// (M = 256) and both token halves, and the commits reach both CTAs' barriers.
template <bool PAIR = false>
__device__ bool swapab_mma(const SwapAbParams &p, Ctrl *ctl, const SwapAbSmem &sm, RingPos &r, int &gseg,
                           uint32_t tmem_base, volatile int *abort_flag) {
    const int S = p.stages, KBS = p.kbs;
    const uint32_t idesc = idesc_bf16_f32(PAIR ? 256 : 128, (uint32_t)p.bn);
    Plan pl;
    pl.init(p, worker_index<PAIR>(), worker_count<PAIR>());
    const int nr = pl.nruns();
    for (int rr = 0; rr < nr; ++rr) {
        int seg, half;
        pl.run(rr, seg, half);
        int64_t tile;
        int kb0, kb1;
        pl.seg_range(seg, tile, kb0, kb1);
        const int g = gseg + seg;
        const int buf = g & 1;
        const uint32_t use = (uint32_t)(g >> 1);
        if (half == 0) {
            if (!mbar_wait_bounded(bar_addr(&ctl->tempty[buf]), (use & 1u) ^ 1u, abort_flag, p.wait_limit_ns, p.err))
                return false;
            tc_fence_after();
        }
        const uint32_t d = tmem_base + (uint32_t)(buf * (p.tmem_cols / 2));
        bool first = half == 0;
        for (int kb = kb0; kb < kb1;) {
            const int n = (kb1 - kb) < KBS ? (kb1 - kb) : KBS;
            if (!mbar_wait_bounded(bar_addr(&ctl->full[r.stage]), r.phase, abort_flag, p.wait_limit_ns, p.err,
                                   p.spin_wait != 0))
                return false;
            tc_fence_after();
            for (int i = 0; i < n; ++i) {
                const uint64_t ad = smem_desc_sw128(sm.a(r.stage) + (uint32_t)i * kATileBytes);
                const uint64_t bd = smem_desc_sw128(sm.b(r.stage) + (uint32_t)i * sm.b_tile_bytes);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    if constexpr (PAIR)
                        tc_mma_bf16_pair(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, first ? 0u : 1u);
                    else
                        tc_mma_bf16(d, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, first ? 0u : 1u);
                    first = false;
                }
            }
            if constexpr (PAIR) tc_commit_pair_multicast(bar_addr(&ctl->empty[r.stage]), (uint16_t)0x3);
            else tc_commit(bar_addr(&ctl->empty[r.stage]));
            r.next(S);
            kb += n;
        }
        if (half == pl.halves - 1) {
            if constexpr (PAIR) tc_commit_pair_multicast(bar_addr(&ctl->tfull[buf]), (uint16_t)0x3);
            else tc_commit(bar_addr(&ctl->tfull[buf]));
        }
    }
    gseg += pl.nseg;
    return true;
}

// Sum, in ascending part order starting from 0, token columns [c0, c1) of the nseg parts
// listed in ctl->seg_slot (nseg <= 128), staged in the idle ring's shared memory by bulk
// copies (buffer 0 keeps the running sum; each round refills buffers 1..), then run the
// epilogue on those columns.  All 128 epilogue threads call it; false after an abort.
template <int EPI>
__device__ bool finish_cols_smem(const SwapAbParams &p, Ctrl *ctl, float *ring, uint32_t ring_base,
                                 uint32_t ring_bytes, uint32_t &fix_round, int nseg, int c0, int c1, int group,
                                 int m, int tid, volatile int *abort_flag) {
    const size_t slot_floats = (size_t)128 * p.bn;
    const uint32_t sl_bytes = (uint32_t)(c1 - c0) * 512u;   // 128 fp32 rows per token column
    const int n4 = (c1 - c0) * 32;                           // float4 of the slice
    const int per_round = (int)(ring_bytes / sl_bytes);
    fence_proxy_async_global();
    int k0 = 0;
    while (k0 < nseg) {
        const int first_buf = k0 == 0 ? 0 : 1;
        const int nload = min(nseg - k0, per_round - first_buf);
        if (threadIdx.x == 64) {
            mbar_arrive_expect_tx(bar_addr(&ctl->fixbar), (uint32_t)nload * sl_bytes);
            for (int i = 0; i < nload; ++i)
                bulk_load(ring_base + (uint32_t)(first_buf + i) * sl_bytes,
                          p.slots + (size_t)ctl->seg_slot[k0 + i] * slot_floats + (size_t)c0 * 128, sl_bytes,
                          bar_addr(&ctl->fixbar));
        }
        const bool got_fix =
            mbar_wait_bounded(bar_addr(&ctl->fixbar), fix_round & 1u, abort_flag, p.wait_limit_ns, p.err);
        ++fix_round;
        if (!named_barrier_and(1, 128, got_fix)) {
            // copies into the ring may still be in flight: let them land first
            if (threadIdx.x == 64)
                (void)mbar_wait_drain(bar_addr(&ctl->fixbar), (fix_round - 1) & 1u, drain_limit_ns(p.wait_limit_ns));
            return false;
        }
        const int nsum = first_buf + nload;
        float4 *b0 = reinterpret_cast<float4 *>(ring);
        const size_t bstride = sl_bytes / 16;   // float4 per buffer
        int e = tid;
        for (; e + 384 < n4; e += 512) {   // 4 independent float4 per thread per step
            float4 a[4];
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                a[rr] = b0[e + rr * 128];
                if (k0 == 0) a[rr] = make_float4(0.f + a[rr].x, 0.f + a[rr].y, 0.f + a[rr].z, 0.f + a[rr].w);
            }
            for (int bb = 1; bb < nsum; ++bb) {
                const float4 *src = b0 + (size_t)bb * bstride;
                float4 t4[4];
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) t4[rr] = src[e + rr * 128];
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    a[rr].x += t4[rr].x; a[rr].y += t4[rr].y; a[rr].z += t4[rr].z; a[rr].w += t4[rr].w;
                }
            }
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) b0[e + rr * 128] = a[rr];
        }
        for (; e < n4; e += 128) {
            float4 a = b0[e];
            if (k0 == 0) a = make_float4(0.f + a.x, 0.f + a.y, 0.f + a.z, 0.f + a.w);
            for (int bb = 1; bb < nsum; ++bb) {
                const float4 t4 = b0[(size_t)bb * bstride + e];
                a.x += t4.x; a.y += t4.y; a.z += t4.z; a.w += t4.w;
            }
            b0[e] = a;
        }
        k0 += nload;
        named_barrier_sync(1, 128);   // buffers 1.. are refilled by the next round
    }
    swapab_epilogue_smem<EPI>(p, ring, group, m, tid, c0, c1);
    return true;
}

// Publication of a finished gate_up tile (m) for readers of h in the same launch: every
// epilogue thread's h stores, then GPU-scope releases of the tile's flag and of the
// pass's count of published tiles.
__device__ __forceinline__ void publish_h_tile(const SwapAbParams &p, int *hflags, int *hcount, int m,
                                               int epoch = 1) {
    fence_proxy_async_global();
    named_barrier_sync(1, 128);
    if (threadIdx.x == 64) {
        st_release_gpu(hflags + p.a_row_base / 64 + m, epoch);
        if (hcount) red_add_release_gpu(hcount, 1);
    }
}

// ---- epilogue (warps 2..5, 128 threads) ----
// ring_idle_at_end: after this pass's last MMA the ring is idle, so a split tile
//   finished in the CTA's last segment may stage the parts in the ring's memory.
// hflags: publish each completed tile (gate_up passes of the fused layer).
// PAIR: each CTA finishes its own 128-row half (m-tile 2 m' + rank) of the pair tile;
// the parts of a split tile are the same halves of the pairs sharing it.
template <int EPI, bool PAIR = false, bool COOP = false>
__device__ bool swapab_epilogue(const SwapAbParams &p, Ctrl *ctl, uint8_t *ring, uint32_t ring_base,
                                uint32_t ring_bytes, int &gseg, uint32_t &fix_round, uint32_t tmem_base,
                                bool ring_idle_at_end, int *hflags, int *hcount, volatile int *abort_flag) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int tid = threadIdx.x - 64;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int bn = p.bn, kbp = p.kb_per_tile;
    const int nchunks = bn / 16;
    const StreamK sk{p.total_units, worker_count<PAIR>()};
    const uint32_t rank = pair_rank<PAIR>();
    const int n_real = PAIR ? p.n_mtiles_real : p.n_mtiles;   // m-tiles of 128 rows
    Plan pl;
    pl.init(p, worker_index<PAIR>(), worker_count<PAIR>());
    // slot index of the part of worker cc (a CTA, or this CTA's counterpart in pair cc)
    auto part_slot = [&](int64_t cc, int64_t tile) -> int {
        const int64_t cta = PAIR ? cc * 2 + rank : cc;
        return (int)(cta * 2 + ((sk.begin(cc) >= tile * kbp) ? 0 : 1));
    };
    auto release = [&](int buf) {   // hand the accumulator back to the MMA issuer
        tc_fence_before();
        if constexpr (PAIR) {
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_rank(bar_addr(&ctl->tempty[buf]), 0));
        } else {
            mbar_arrive(bar_addr(&ctl->tempty[buf]));
        }
    };
    const size_t slot_floats = (size_t)128 * bn;
    const int gbase = gseg;
    gseg += pl.nseg;
    for (int s = 0; s < pl.nseg; ++s) {
        int64_t tile;
        int kb0, kb1;
        pl.seg_range(s, tile, kb0, kb1);
        const int g = gbase + s;
        const int buf = g & 1;
        const uint32_t use = (uint32_t)(g >> 1);
        const int group = (int)(tile / p.n_mtiles);
        const int mp = (int)(tile - (int64_t)group * p.n_mtiles);
        const int m = PAIR ? 2 * mp + (int)rank : mp;         // this CTA's m-tile
        const int64_t ctile = (int64_t)group * n_real + m;    // its counter
        const bool got = mbar_wait_bounded(bar_addr(&ctl->tfull[buf]), use & 1u, abort_flag, p.wait_limit_ns, p.err);
        if (!named_barrier_and(1, 128, got)) return false;   // all epilogue warps take the same branch
        tc_fence_after();
        if (PAIR && m >= n_real) {   // the second half of a pair tile past the last m-tile
            release(buf);
            continue;
        }
        const uint32_t tacc = tmem_base + (uint32_t)(buf * (p.tmem_cols / 2)) + lane_off;
        if (kb0 == 0 && kb1 == kbp) {
            for (int c = 0; c < nchunks; ++c) {
                float v[16];
                load_tmem_chunk(tacc + (uint32_t)(c * 16), v);
                swapab_epilogue_chunk<EPI>(p, ctl, group, m, q, lane, c, v);
            }
            release(buf);
            if (hflags) publish_h_tile(p, hflags, hcount, m, p.hflag_epoch > 0 ? p.hflag_epoch : 1);
            continue;
        }
        // Clustered finish of two-part tiles (clusters of three CTAs covering two tiles
        // exactly; the pass's final segments; the ring idle).  Parts are summed in CTA
        // order from 0 like every other path, so results are identical.
        //  - the other part is the next CTA's first segment (finished long before): this
        //    CTA finishes the tile without publishing its own part: it waits for the
        //    other part's count, fetches that part and adds its own from tensor memory;
        //  - both parts are final segments: the first CTA writes its part straight into
        //    the second one's idle ring (distributed shared memory) once that ring is
        //    free, and the second CTA finishes the tile.
        if (!PAIR && p.cluster_finish && ring_idle_at_end && s == pl.nseg - 1) {
            const int64_t cf = sk.owner(tile * kbp), cl = sk.owner(tile * kbp + kbp - 1);
            const int64_t me = blockIdx.x;
            const bool cl_early = cl == cf + 1 && sk.begin(cl + 1) > (tile + 1) * kbp;
            const bool both_final = cl == cf + 1 && !cl_early && cf / 3 == cl / 3;
            const uint32_t slot_bytes1 = (uint32_t)(slot_floats * 4);
            const float *other = reinterpret_cast<const float *>(ring);
            if (cl_early && me == cf) {
                if (threadIdx.x == 64) {
                    bool ok = true;
                    const uint64_t t0 = global_timer_ns();
                    while (ld_acquire_gpu(p.counters + ctile) < 1) {
                        if (*abort_flag) { ok = false; break; }
                        if (global_timer_ns() - t0 > p.wait_limit_ns) {
                            *abort_flag = 1;
                            raise_device_error(p.err, DEV_ERR_TIMEOUT);
                            ok = false;
                            break;
                        }
                    }
                    if (ok) {
                        fence_proxy_async_global();
                        mbar_arrive_expect_tx(bar_addr(&ctl->fixbar), slot_bytes1);
                        bulk_load(ring_base, p.slots + (size_t)part_slot(cl, tile) * slot_floats, slot_bytes1,
                                  bar_addr(&ctl->fixbar));
                    }
                    ctl->fin_flag = ok ? 1 : 0;
                }
                named_barrier_sync(1, 128);
                if (!ctl->fin_flag) return false;
                const bool got_fix =
                    mbar_wait_bounded(bar_addr(&ctl->fixbar), fix_round & 1u, abort_flag, p.wait_limit_ns, p.err);
                ++fix_round;
                if (!named_barrier_and(1, 128, got_fix)) {
                    if (threadIdx.x == 64)
                        (void)mbar_wait_drain(bar_addr(&ctl->fixbar), (fix_round - 1) & 1u,
                                              drain_limit_ns(p.wait_limit_ns));
                    return false;
                }
                for (int c = 0; c < nchunks; ++c) {
                    float own[16], v[16];
                    load_tmem_chunk(tacc + (uint32_t)(c * 16), own);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = (0.f + own[i]) + other[(c * 16 + i) * 128 + row];
                    swapab_epilogue_chunk<EPI>(p, ctl, group, m, q, lane, c, v);
                }
                release(buf);
                if (threadIdx.x == 64) p.counters[ctile] = 0;
                named_barrier_sync(1, 128);   // fin_flag is reused by the next tile
                continue;
            }
            if (both_final && me == cf) {
                const uint32_t peer = (uint32_t)(cl % 3);
                bool ok = true;
                if (threadIdx.x == 64)
                    ok = mbar_wait_bounded(bar_addr(&ctl->go_bar), 0u, abort_flag, p.wait_limit_ns, p.err);
                if (!named_barrier_and(1, 128, ok)) return false;
                const uint32_t remote = map_to_rank(ring_base, peer);
                for (int c = 0; c < nchunks; ++c) {
                    float v[16];
                    load_tmem_chunk(tacc + (uint32_t)(c * 16), v);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        st_cluster_f32(remote + (uint32_t)(((c * 16 + i) * 128 + row) * 4), v[i]);
                }
                release(buf);
                named_barrier_sync(1, 128);   // every thread's stores precede the arrive
                if (threadIdx.x == 64) mbar_arrive_cluster(map_to_rank(bar_addr(&ctl->recv_bar), peer));
                continue;
            }
            if (both_final && me == cl) {
                const uint32_t peer = (uint32_t)(cf % 3);
                bool ok = true;
                if (threadIdx.x == 64) {
                    mbar_arrive_cluster(map_to_rank(bar_addr(&ctl->go_bar), peer));   // this ring is free
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait_acq_cluster(bar_addr(&ctl->recv_bar), 0u)) {
                        if (*abort_flag) { ok = false; break; }
                        if (global_timer_ns() - t0 > p.wait_limit_ns) {
                            *abort_flag = 1;
                            raise_device_error(p.err, DEV_ERR_TIMEOUT);
                            ok = false;
                            break;
                        }
                    }
                }
                if (!named_barrier_and(1, 128, ok)) return false;
                for (int c = 0; c < nchunks; ++c) {
                    float own[16], v[16];
                    load_tmem_chunk(tacc + (uint32_t)(c * 16), own);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = (0.f + other[(c * 16 + i) * 128 + row]) + own[i];
                    swapab_epilogue_chunk<EPI>(p, ctl, group, m, q, lane, c, v);
                }
                release(buf);
                continue;
            }
        }
        // Tile shared with other CTAs: park the fp32 partial in this CTA's slot, laid
        // out [token column][accumulator row] (each warp store is a 128-byte run).
        // A CTA's first segment uses its slot 0, a later one its slot 1.
        const int which = s == 0 ? 0 : 1;
        float *slot = p.slots + ((size_t)blockIdx.x * 2 + which) * slot_floats;
        for (int c = 0; c < nchunks; ++c) {
            float v[16];
            load_tmem_chunk(tacc + (uint32_t)(c * 16), v);
#pragma unroll
            for (int i = 0; i < 16; ++i) __stcg(slot + (size_t)(c * 16 + i) * 128 + row, v[i]);
        }
        release(buf);
        if (ring_idle_at_end) fence_proxy_async_global();   // a finisher may fetch this slot with a bulk copy
        named_barrier_sync(1, 128);
        const int64_t c_first = sk.owner(tile * kbp), c_last = sk.owner(tile * kbp + kbp - 1);
        const int nseg = (int)(c_last - c_first + 1);
        // Cooperative finish (the ring is idle after the pass, the tile has at least
        // coop_finish parts): every part for which the tile is its CTA's final segment
        // waits for all parts, then sums and finishes its own slice of token columns.
        // Only the last CTA's part can be a non-final segment (the tile is that CTA's
        // first); it hands its part over and goes on.  All parts of the tile take the
        // same decision.
        // (compiled into the merged-projection kernel, whose tiles are split about nine
        // ways, and into the COOP kernels the host picks when some tile is split at least
        // coop_finish ways, e.g. one shard's narrow gate_up slice; the replicated layer's
        // tiles are split two to four ways, where the CTA arriving last finishing alone
        // measured faster and even the untaken branch cost time)
        int n_fin = 0;   // parts that finish jointly; 0: the CTA arriving last finishes alone
        if constexpr (EPI == EPI_MERGED || COOP) {
            if (ring_idle_at_end && p.coop_finish > 0 && nseg >= p.coop_finish && nseg <= 128) {
                n_fin = nseg - (sk.begin(c_last + 1) <= (tile + 1) * kbp ? 0 : 1);
                if (ring_bytes / ((uint32_t)((bn + n_fin - 1) / n_fin) * 512u) < 2) n_fin = 0;
            }
        }
        if (n_fin > 0) {
            if (s != pl.nseg - 1) {
                if (threadIdx.x == 64) (void)atomic_add_acq_rel_gpu(p.counters + ctile, 1);
                continue;
            }
            if (threadIdx.x == 64) {
                (void)atomic_add_acq_rel_gpu(p.counters + ctile, 1);
                bool ok = true;
                const uint64_t t0 = global_timer_ns();
                while (ld_acquire_gpu(p.counters + ctile) < nseg) {
                    if (*abort_flag) { ok = false; break; }
                    if (global_timer_ns() - t0 > p.wait_limit_ns) {
                        *abort_flag = 1;
                        raise_device_error(p.err, DEV_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                }
                ctl->fin_flag = ok ? 1 : 0;
            }
            named_barrier_sync(1, 128);
            if (!ctl->fin_flag) return false;
            for (int k = tid; k < nseg; k += 128) ctl->seg_slot[k] = part_slot(c_first + k, tile);
            named_barrier_sync(1, 128);
            const int idx = (int)(worker_index<PAIR>() - c_first);
            const int col0 = idx * bn / n_fin, col1 = (idx + 1) * bn / n_fin;
            if (col1 > col0 && !finish_cols_smem<EPI>(p, ctl, reinterpret_cast<float *>(ring), ring_base, ring_bytes,
                                                       fix_round, nseg, col0, col1, group, m, tid, abort_flag))
                return false;
            if (hflags) {
                // every epilogue thread's h stores precede this CTA's count below
                fence_proxy_async_global();
                named_barrier_sync(1, 128);
            }
            if (threadIdx.x == 64) {
                // every finisher is past its wait once all have counted themselves here; the
                // last one to count (acquiring every other finisher's slice) publishes the tile
                if (atomic_add_acq_rel_gpu(p.counters + ctile, 1) == nseg + n_fin - 1) {
                    p.counters[ctile] = 0;
                    if (hflags) {
                        st_release_gpu(hflags + p.a_row_base / 64 + m, p.hflag_epoch > 0 ? p.hflag_epoch : 1);
                        if (hcount) red_add_release_gpu(hcount, 1);
                    }
                }
            }
            named_barrier_sync(1, 128);   // fin_flag is reused by the next tile
            continue;
        }
        if (threadIdx.x == 64) {
            // release: the barrier above orders every epilogue thread's slot stores
            // before this atomic; acquire: the finisher then sees all other parts
            const int prev = atomic_add_acq_rel_gpu(p.counters + ctile, 1);
            ctl->fin_flag = (prev == nseg - 1) ? 1 : 0;
        }
        named_barrier_sync(1, 128);
        if (!ctl->fin_flag) {
            named_barrier_sync(1, 128);   // fin_flag is reused by the next tile
            continue;
        }
        // This CTA arrived last: sum the parts in ascending part (CTA) order starting
        // from 0, so the result does not depend on which CTA finishes the tile.
        // Slot of each part: CTA cc's first segment uses slot 2cc, a later one 2cc+1.
        for (int k = tid; k < nseg && k < 128; k += 128) ctl->seg_slot[k] = part_slot(c_first + k, tile);
        named_barrier_sync(1, 128);
        auto slot_of = [&](int k) -> int { return k < 128 ? ctl->seg_slot[k] : part_slot(c_first + k, tile); };
        const uint32_t slot_bytes = (uint32_t)(slot_floats * 4);
        if (ring_idle_at_end && s == pl.nseg - 1 && ring_bytes / slot_bytes >= 2 && nseg <= 128) {
            // Last segment of the pass with the ring idle: the parts are staged in the
            // ring's memory and summed there.
            if (!finish_cols_smem<EPI>(p, ctl, reinterpret_cast<float *>(ring), ring_base, ring_bytes, fix_round,
                                       nseg, 0, bn, group, m, tid, abort_flag))
                return false;
        } else {
            // In registers, every part from its slot in L2: two chunks of 16 tokens x two
            // parts per round keep 64 loads per thread in flight.
            constexpr int NB = 2, NP = 2;
            for (int c0 = 0; c0 < nchunks; c0 += NB) {
                float acc[NB][16];
#pragma unroll
                for (int b = 0; b < NB; ++b)
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[b][i] = 0.f;
                for (int k0 = 0; k0 < nseg; k0 += NP) {
                    float t[NP][NB][16];
#pragma unroll
                    for (int sp = 0; sp < NP; ++sp) {
                        if (k0 + sp < nseg) {
                            const float *src = p.slots + (size_t)slot_of(k0 + sp) * slot_floats + row;
#pragma unroll
                            for (int b = 0; b < NB; ++b) {
                                if (c0 + b < nchunks) {
#pragma unroll
                                    for (int i = 0; i < 16; ++i)
                                        t[sp][b][i] = __ldcg(src + (size_t)((c0 + b) * 16 + i) * 128);
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int sp = 0; sp < NP; ++sp) {
                        if (k0 + sp < nseg) {
#pragma unroll
                            for (int b = 0; b < NB; ++b)
#pragma unroll
                                for (int i = 0; i < 16; ++i) acc[b][i] += t[sp][b][i];
                        }
                    }
                }
#pragma unroll
                for (int b = 0; b < NB; ++b)
                    if (c0 + b < nchunks) swapab_epilogue_chunk<EPI>(p, ctl, group, m, q, lane, c0 + b, acc[b]);
            }
        }
        if (threadIdx.x == 64) p.counters[ctile] = 0;
        if (hflags) publish_h_tile(p, hflags, hcount, m, p.hflag_epoch > 0 ? p.hflag_epoch : 1);
        named_barrier_sync(1, 128);   // fin_flag is reused by the next tile
    }
    return true;
}

// ---- gate_up with x in host memory (epilogue warps, before their first tile) ----
// Each CTA takes a ticket; the first x_copiers tickets copy one slice of x each (16-byte
// words, sixteen loads in flight per thread), make the stores visible to the tensor-memory
// copies' proxy and count the slice (release).  One thread per CTA then waits for every
// slice (acquire), releases the producer's token loads, and counts itself past the wait;
// the last CTA past it zeroes the three words.  Without x_copy_early every CTA first waits
// for the previous grid (then every earlier user of the buffer and of the words is done).
// Every wait is bounded.
__device__ __noinline__ void swapab_copy_x(const SwapAbParams &p, Ctrl *ctl, volatile int *abort_flag) {
    const int tid = threadIdx.x - 64;
    if (!p.x_copy_early) pdl_wait();
    if (tid == 0) ctl->x_ticket = atomicAdd(p.x_sync, 1);
    named_barrier_sync(1, 128);
    const int ticket = ctl->x_ticket;
    if (ticket < p.x_copiers) {
        const int64_t v0 = p.x_vecs * ticket / p.x_copiers, v1 = p.x_vecs * (ticket + 1) / p.x_copiers;
        constexpr int kIn = 16;   // 32 KB of host reads in flight per CTA
        for (int64_t v = v0 + tid; v < v1; v += 128 * kIn) {
            uint4 r[kIn];
#pragma unroll
            for (int k = 0; k < kIn; ++k)
                if (v + k * 128 < v1) r[k] = p.x_host[v + k * 128];
#pragma unroll
            for (int k = 0; k < kIn; ++k)
                if (v + k * 128 < v1) p.x_copy[v + k * 128] = r[k];
        }
        fence_proxy_async_global();
        named_barrier_sync(1, 128);
        if (tid == 0) red_add_release_gpu(p.x_sync + 1, 1);
    }
    if (tid == 0) {
        const uint64_t t0 = global_timer_ns();
        bool ok = true;
        while (ld_acquire_gpu(p.x_sync + 1) < p.x_copiers) {
            if (*abort_flag || global_timer_ns() - t0 > p.wait_limit_ns) { ok = false; break; }
            __nanosleep(100);
        }
        if (ok) {
            mbar_arrive(bar_addr(&ctl->hready_bar));
            if (atomic_add_acq_rel_gpu(p.x_sync + 2, 1) == (int)gridDim.x - 1) {
                p.x_sync[0] = 0;
                p.x_sync[1] = 0;
                p.x_sync[2] = 0;
            }
        } else if (!*abort_flag) {
            *abort_flag = 1;
            raise_device_error(p.err, DEV_ERR_TIMEOUT);
        }
    }
}

// ---- set-up and teardown shared by the swap-AB kernels ----
// PAIR: the second CTA's full barriers are unused (its copies signal the first CTA's),
// the first CTA's tempty barriers count one arrival per epilogue warp of both CTAs, and
// tensor memory is allocated for the pair.
template <bool PAIR = false>
__device__ __forceinline__ void swapab_setup(Ctrl *ctl, int S, int tmem_cols, const CUtensorMap *const *maps,
                                             int n_maps, bool clustered = false) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(bar_addr(&ctl->full[s]), 1);
            mbar_init(bar_addr(&ctl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar_addr(&ctl->tfull[b]), 1);
            mbar_init(bar_addr(&ctl->tempty[b]), PAIR ? 8 : 128);
        }
        mbar_init(bar_addr(&ctl->drain), 1);
        mbar_init(bar_addr(&ctl->fixbar), 1);
        mbar_init(bar_addr(&ctl->go_bar), 1);
        mbar_init(bar_addr(&ctl->recv_bar), 1);
        mbar_init(bar_addr(&ctl->hready_bar), 1);
        ctl->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0)
        for (int i = 0; i < n_maps; ++i) tma_prefetch_desc(maps[i]);
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_u32(&ctl->tmem_base), (uint32_t)tmem_cols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(&ctl->tmem_base), (uint32_t)tmem_cols);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR || clustered) cluster_sync();   // the peers' barriers are initialised before any remote use
    tc_fence_after();
}

// Drain in-flight copies and MMAs, then free tensor memory (all threads).  PAIR: each
// CTA's issued stages are drained through its empty barriers, which the first CTA's
// MMA commits release once both CTAs' bytes have landed and been consumed.
template <bool PAIR = false>
__device__ __forceinline__ void swapab_teardown(Ctrl *ctl, int S, int issued, uint32_t tmem_base, int tmem_cols,
                                                uint64_t limit_ns, bool clustered = false) {
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (warp == 0 && lane == 0) {
        const int first = issued > S ? issued - S : 0;
        for (int i = first; i < issued; ++i) {
            if constexpr (PAIR) {
                const bool done =
                    mbar_wait_drain(bar_addr(&ctl->empty[i % S]), (uint32_t)((i / S) & 1), drain_limit_ns(limit_ns));
                if (!done) __nanosleep(200000);   // abort path: let in-flight copies land
            } else {
                (void)mbar_wait_drain(bar_addr(&ctl->full[i % S]), (uint32_t)((i / S) & 1), drain_limit_ns(limit_ns));
            }
        }
    }
    if (warp == 1 && lane == 0 && (!PAIR || cluster_ctarank() == 0)) {
        if constexpr (PAIR) tc_commit_pair_multicast(bar_addr(&ctl->drain), (uint16_t)0x1);
        else tc_commit(bar_addr(&ctl->drain));
        (void)mbar_wait_drain(bar_addr(&ctl->drain), 0, drain_limit_ns(limit_ns));
    }
    tc_fence_before();
    __syncthreads();
    if (PAIR || clustered) cluster_sync();   // no CTA leaves while a peer may still use its memory
    tc_fence_after();
    if (warp == 1) {
        if constexpr (PAIR) tmem_dealloc_pair(tmem_base, (uint32_t)tmem_cols);
        else tmem_dealloc(tmem_base, (uint32_t)tmem_cols);
    }
}

// One stream-K pass: out = epilogue(A . B^T) over p's (group, m-tile, k-block) units.
// PAIR: clusters of two CTAs take (group, pair of m-tiles, k-block) units; one M = 256
// MMA per k-block covers both CTAs' weight rows, each CTA holding half of the tokens.
template <int EPI, bool PAIR, bool COOP = false>
__global__ void __launch_bounds__(kSwapAbThreads, 1)
    swapab_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const SwapAbParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const SwapAbSmem sm(base, PAIR ? p.bn / 2 : p.bn, p.kbs);
    const int S = p.stages;
    uint8_t *ring = smem_raw + (base - raw);
    Ctrl *ctl = reinterpret_cast<Ctrl *>(ring + (uint32_t)S * sm.stage_bytes);
    const CUtensorMap *maps[2] = {&tmA, &tmB};
    const bool clustered = !PAIR && p.cluster_finish != 0;
    swapab_setup<PAIR>(ctl, S, p.tmem_cols, maps, 2, clustered);
    const uint32_t tmem_base = ctl->tmem_base;
    volatile int *abort_flag = &ctl->abort_flag;
    // gate_up that publishes h flags lets the down grid launch only once the previous grid on
    // the stream (the previous call's down kernel, which clears the flags) is complete: no down
    // CTA can see a flag that the previous call left behind.  gate_up that copies x from host
    // memory does the same, so that every grid before it is complete once the next call's
    // gate_up starts (that one may write the other x buffer, which this call's predecessors read)
    const bool late_trigger = EPI == EPI_SWIGLU && (p.hflags != nullptr || p.x_host != nullptr);
    if (!late_trigger) pdl_launch_dependents();

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    int issued = 0;
    if (warp == 0) {
        if (lane == 0) {
            RingPos r;
            (void)swapab_produce<EPI, PAIR>(p, &tmA, &tmB, ctl, sm, r, issued, true, nullptr, abort_flag);
        }
    } else if (warp == 1) {
        if (lane == 0 && pair_rank<PAIR>() == 0) {
            RingPos r;
            int gseg = 0;
            (void)swapab_mma<PAIR>(p, ctl, sm, r, gseg, tmem_base, abort_flag);
        }
    } else {
        if (EPI == EPI_SWIGLU && p.x_host) swapab_copy_x(p, ctl, abort_flag);
        if (EPI != EPI_SWIGLU && p.hflags) {
            // the h blocks of every stage of this CTA: one flag per thread per round (an acquire
            // load at most every 0.2 us), a CTA barrier once every flag is seen, then one arrival
            // releases the producer's token loads
            const int tid = threadIdx.x - 64;
            Plan pl;
            pl.init(p, worker_index<PAIR>(), worker_count<PAIR>());
            const uint64_t t0 = global_timer_ns();
            bool ok = true;
            while (true) {
                bool mine = true;
                int base = 0;
                for (int sg = 0; sg < pl.nseg; ++sg) {
                    int64_t tile;
                    int kb0, kb1;
                    pl.seg_range(sg, tile, kb0, kb1);
                    const int group = (int)(tile / p.n_mtiles);
                    for (int kb = kb0 + ((tid - base) % 128 + 128) % 128; kb < kb1; kb += 128)
                        mine &= ld_acquire_gpu(p.hflags + p.kb_first + group * p.kb_group_stride + kb) ==
                                p.hflag_epoch;
                    base += kb1 - kb0;
                }
                const bool timed_out = global_timer_ns() - t0 > p.wait_limit_ns || *abort_flag;
                if (named_barrier_and(1, 128, mine)) break;
                if (named_barrier_and(1, 128, !timed_out) == false) { ok = false; break; }
                __nanosleep(200);
            }
            if (threadIdx.x == 64) {
                if (ok) {
                    mbar_arrive(bar_addr(&ctl->hready_bar));
                    // Every flag is read by some CTA, so once all CTAs are past their polls the
                    // gate_up grid has published every flag and no one reads them any more:
                    // the last CTA here clears them (while the grid still runs, not at its end)
                    if (atomic_add_acq_rel_gpu(p.exit_count, 1) == (int)gridDim.x - 1) {
                        for (int t = 0; t < p.hflag_n; ++t) p.hflags[p.hflag_first + t] = 0;
                        *p.exit_count = 0;
                    }
                } else if (!*abort_flag) {
                    *abort_flag = 1;
                    raise_device_error(p.err, DEV_ERR_TIMEOUT);
                }
            }
        }
        pdl_wait();
        if (late_trigger && threadIdx.x == 64) pdl_launch_dependents();
        int gseg = 0;
        uint32_t fix_round = 0;
        // (the epilogue waits for the previous grid even where the producer does not: no output or
        // split-K slot is written before the gate_up grid is complete)
        (void)swapab_epilogue<EPI, PAIR, COOP>(p, ctl, ring, base, (uint32_t)S * sm.stage_bytes, gseg, fix_round,
                                               tmem_base, true, EPI == EPI_SWIGLU ? p.hflags : nullptr, nullptr,
                                               abort_flag);
    }
    swapab_teardown<PAIR>(ctl, S, issued, tmem_base, p.tmem_cols, p.wait_limit_ns, clustered);
}

// The whole shared-expert layer at decode token counts in one launch:
//   gate_up passes  h = silu(x W_gate^T) * (x W_up^T)   (stream-K over gate_up tiles)
//   down pass       out = h W_down^T                     (stream-K over down tiles)
// Every CTA runs its share of each pass in turn through the same ring.  Down weight
// tiles stream into stages as soon as gate_up MMAs free them; their token tiles (h)
// wait for the flag of the gate_up tile that writes them.  With two gate_up passes
// (the first and the second half of the tiles) the first half's tiles are finished
// while the second half streams, and the down pass takes its units as pairs of
// k-blocks from the two halves, the first-half k-blocks first: the second half's
// split-K tail then overlaps down work.  One CTA per SM and grid <= SMs: every CTA is
// resident once the previous work on the stream leaves, and every wait is bounded.
// The last CTA to leave clears the flags and counts, so the sync words are zero again.
template <int EPI1>
__global__ void __launch_bounds__(kSwapAbThreads, 1)
    swapab_mlp_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
                      const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                      const SwapAbMlpParams fp) {
    const SwapAbParams &p0 = fp.ph[0];
    const SwapAbParams &pd = fp.ph[2];
    const int n_gu = fp.n_gate_up_passes;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const SwapAbSmem sm(base, p0.bn, p0.kbs);
    const int S = p0.stages;
    uint8_t *ring = smem_raw + (base - raw);
    Ctrl *ctl = reinterpret_cast<Ctrl *>(ring + (uint32_t)S * sm.stage_bytes);
    const CUtensorMap *maps[4] = {&tmA0, &tmB0, &tmA1, &tmB1};
    swapab_setup(ctl, S, p0.tmem_cols, maps, 4);
    const uint32_t tmem_base = ctl->tmem_base;
    volatile int *abort_flag = &ctl->abort_flag;
    pdl_launch_dependents();

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    int issued = 0;
    if (warp == 0) {
        if (lane == 0) {
            RingPos r;
            bool ok = true;
            for (int ph = 0; ph < n_gu && ok; ++ph)
                ok = swapab_produce<EPI_SWIGLU>(fp.ph[ph], &tmA0, &tmB0, ctl, sm, r, issued, ph == 0, nullptr,
                                                abort_flag);
            const HFlags hf = {fp.hflags, fp.hcount, fp.hflag_first, fp.ph[0].n_mtiles,
                               n_gu == 2 ? fp.ph[1].n_mtiles : 0};
            if (ok) (void)swapab_produce<EPI1>(pd, &tmA1, &tmB1, ctl, sm, r, issued, false, &hf, abort_flag);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            RingPos r;
            int gseg = 0;
            bool ok = true;
            for (int ph = 0; ph < n_gu && ok; ++ph) ok = swapab_mma(fp.ph[ph], ctl, sm, r, gseg, tmem_base, abort_flag);
            if (ok) (void)swapab_mma(pd, ctl, sm, r, gseg, tmem_base, abort_flag);
        }
    } else {
        pdl_wait();
        int gseg = 0;
        uint32_t fix_round = 0;
        const uint32_t ring_bytes = (uint32_t)S * sm.stage_bytes;
        bool ok = true;
        for (int ph = 0; ph < n_gu && ok; ++ph)
            ok = swapab_epilogue<EPI_SWIGLU>(fp.ph[ph], ctl, ring, base, ring_bytes, gseg, fix_round, tmem_base, false,
                                             fp.hflags, fp.hcount + ph, abort_flag);
        if (ok)
            (void)swapab_epilogue<EPI1>(pd, ctl, ring, base, ring_bytes, gseg, fix_round, tmem_base, true, nullptr,
                                        nullptr, abort_flag);
    }
    swapab_teardown(ctl, S, issued, tmem_base, p0.tmem_cols, p0.wait_limit_ns);
    if (threadIdx.x == 0 && !*abort_flag) {
        // every flag read of this CTA precedes this increment; the last CTA clears them
        if (atomic_add_acq_rel_gpu(fp.exit_count, 1) == (int)gridDim.x - 1) {
            for (int t = 0; t < fp.n_htiles; ++t) fp.hflags[fp.hflag_first + t] = 0;
            fp.hcount[0] = 0;
            fp.hcount[1] = 0;
            *fp.exit_count = 0;
        }
    }
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
            const bool got =
                mbar_wait_bounded(bar_addr(&ctl->tfull[buf]), use & 1u, abort_flag, p.wait_limit_ns, p.err);
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
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    } else if constexpr (EPI == EPI_BF16) {
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            w[i] = (uint32_t)f32_to_bf16_bits(v[2 * i]) |
                                   ((uint32_t)f32_to_bf16_bits(v[2 * i + 1]) << 16);
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
            (void)mbar_wait_drain(bar_addr(&ctl->full[i % S]), (uint32_t)((i / S) & 1),
                                  drain_limit_ns(p.wait_limit_ns));
    }
    if (warp == 1 && lane == 0) {
        tc_commit(bar_addr(&ctl->drain));
        (void)mbar_wait_drain(bar_addr(&ctl->drain), 0, drain_limit_ns(p.wait_limit_ns));
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

// Epilogue stores of the pair kernel for one CTA's token row `tok`: SwiGLU chunk c (gate
// columns 16c .., up columns 128 + 16c ..) or 16 output columns 16c .. of the tile.
__device__ __forceinline__ void pair_store_swiglu(const StdParams &p, const StdTile &t, int64_t tok, bool tok_ok,
                                                  int c, const float (&g)[16], const float (&u)[16]) {
    uint16_t *h = static_cast<uint16_t *>(p.out);
    const int64_t j = (int64_t)p.n_base + (int64_t)t.n * 128 + c * 16;
    if (!tok_ok || j >= p.n_valid) return;
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        w[i] = (uint32_t)f32_to_bf16_bits(silu_f32(g[2 * i]) * u[2 * i]) |
               ((uint32_t)f32_to_bf16_bits(silu_f32(g[2 * i + 1]) * u[2 * i + 1]) << 16);
    uint4 *dst = reinterpret_cast<uint4 *>(h + tok * p.ldo + j);
    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

template <int EPI>
__device__ __forceinline__ void pair_store_cols(const StdParams &p, const StdTile &t, int64_t tok, bool tok_ok, int c,
                                                const float (&v)[16]) {
    const int64_t n = (int64_t)t.n * 256 + c * 16;
    if (!tok_ok || n >= p.n_valid) return;
    if constexpr (EPI == EPI_F32) {
        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + t.group * p.o_group_stride +
                                                 tok * p.ldo + n);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else if constexpr (EPI == EPI_BF16) {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            w[i] = (uint32_t)f32_to_bf16_bits(v[2 * i]) | ((uint32_t)f32_to_bf16_bits(v[2 * i + 1]) << 16);
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + t.group * p.o_group_stride +
                                               tok * p.ldo + n);
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

constexpr int kPairSlotFloats = 128 * 256;

// The units of one cluster of the pair kernel, as segments (tile, k-blocks [kb0, kb1)):
// whole tiles cluster, cluster + n_clusters, ..., or with split_k the cluster's share
// [ub, ue) of the (tile, k-block) units.
struct PairWork {
    int64_t cluster, n_clusters, n_tiles, ub, ue;
    int kbp;
    bool split;
    __device__ bool seg(int64_t i, int64_t &tile, int &kb0, int &kb1) const {
        if (!split) {
            tile = cluster + i * n_clusters;
            kb0 = 0;
            kb1 = kbp;
            return tile < n_tiles;
        }
        tile = ub / kbp + i;
        if (tile * kbp >= ue) return false;
        kb0 = (int)(ub > tile * kbp ? ub - tile * kbp : 0);
        kb1 = (int)(ue < (tile + 1) * kbp ? ue - tile * kbp : kbp);
        return true;
    }
};

template <int EPI>
__global__ void __launch_bounds__(kStdThreads, 1)
    pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const StdParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const int S = p.stages;
    const uint32_t sA = base;
    const uint32_t sB = base + (uint32_t)S * kATileBytes;
    uint8_t *ring = smem_raw + (base - raw);
    const uint32_t ring_bytes = (uint32_t)S * (kATileBytes + kPairBTileBytes);
    Ctrl *ctl = reinterpret_cast<Ctrl *>(ring + ring_bytes);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int64_t cluster = blockIdx.x / 2, n_clusters = gridDim.x / 2;
    const int64_t n_tiles = (int64_t)p.n_groups * p.n_mtiles * p.n_ntiles;
    const int kbp = p.kb_per_tile;
    constexpr uint32_t kTmemCols = 512;
    const StreamK sk{n_tiles * kbp, n_clusters};
    const PairWork work{cluster, n_clusters, n_tiles, sk.begin(cluster), sk.begin(cluster + 1), kbp, p.split_k != 0};

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
        mbar_init(bar_addr(&ctl->fixbar), 1);
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
            // (token tiles are read by every tile of a column band, weight tiles once when the
            // launch has one token tile)
            const uint64_t pol_a = l2_policy_evict_last(), pol_b = l2_policy_evict_first();
            auto rows = [&](const StdTile &t, int kb, int &k, int &a_row, int &b_row) {
                k = (p.kb_first + t.group * p.kb_group_stride + kb) * 64;
                a_row = t.m * 256 + (int)rank * 128;
                b_row = p.b_base + t.n * p.b_n_stride + (int)rank * p.b_rank_stride;
            };
            int64_t id;
            int kb0, kb1;
            // Launches with one token tile stream their weights once: the weight tiles of the
            // first stages (a fresh ring) are requested before the wait for the previous
            // kernel, whose results only the token tiles can depend on.
            int pre = 0;
            if (p.cache_hints) {
                for (int64_t i = 0; pre < S && work.seg(i, id, kb0, kb1); ++i) {
                    const StdTile t = tile_of(id);
                    for (int kb = kb0; kb < kb1 && pre < S; ++kb, ++pre) {
                        int k, a_row, b_row;
                        rows(t, kb, k, a_row, b_row);
                        if (leader)
                            mbar_arrive_expect_tx(bar_addr(&ctl->full[pre]), 2u * (kATileBytes + kPairBTileBytes));
                        tma_load_2d_pair_hint(sB + pre * kPairBTileBytes, &tmB,
                                              map_to_rank(bar_addr(&ctl->full[pre]), 0), k, b_row, pol_b);
                    }
                }
            }
            if (!p.x_early) pdl_wait();
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int64_t i = 0; ok && work.seg(i, id, kb0, kb1); ++i) {
                const StdTile t = tile_of(id);
                for (int kb = kb0; kb < kb1; ++kb) {
                    const uint32_t fb = map_to_rank(bar_addr(&ctl->full[stage]), 0);
                    int k, a_row, b_row;
                    rows(t, kb, k, a_row, b_row);
                    if (issued < pre) {   // its weight tile is requested already
                        tma_load_2d_pair_hint(sA + stage * kATileBytes, &tmA, fb, k, a_row, pol_a);
                    } else {
                        if (!mbar_wait_bounded(bar_addr(&ctl->empty[stage]), phase ^ 1u, abort_flag,
                                               p.wait_limit_ns, p.err)) {
                            ok = false;
                            break;
                        }
                        if (leader)
                            mbar_arrive_expect_tx(bar_addr(&ctl->full[stage]), 2u * (kATileBytes + kPairBTileBytes));
                        if (p.cache_hints) {
                            tma_load_2d_pair_hint(sA + stage * kATileBytes, &tmA, fb, k, a_row, pol_a);
                            tma_load_2d_pair_hint(sB + stage * kPairBTileBytes, &tmB, fb, k, b_row, pol_b);
                        } else {
                            tma_load_2d_pair(sA + stage * kATileBytes, &tmA, fb, k, a_row);
                            tma_load_2d_pair(sB + stage * kPairBTileBytes, &tmB, fb, k, b_row);
                        }
                    }
                    ++issued;
                    if (++stage == S) { stage = 0; phase ^= 1u; }
                }
            }
            if (issued < pre) {
                // (only after an abort: the token tiles of the stages whose weight tiles were
                // requested, so that every expected byte lands before the teardown drains)
                for (int64_t i = 0, u = 0; work.seg(i, id, kb0, kb1); ++i) {
                    const StdTile t = tile_of(id);
                    for (int kb = kb0; kb < kb1; ++kb, ++u) {
                        if (u < issued || u >= pre) continue;
                        int k, a_row, b_row;
                        rows(t, kb, k, a_row, b_row);
                        tma_load_2d_pair_hint(sA + (int)u * kATileBytes, &tmA, map_to_rank(bar_addr(&ctl->full[u]), 0),
                                              k, a_row, pol_a);
                    }
                }
                issued = pre;
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            const uint32_t idesc = idesc_bf16_f32(256, 256);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int64_t id;
            int kb0, kb1;
            for (int64_t i = 0; ok && work.seg(i, id, kb0, kb1); ++i) {
                const int buf = (int)(i & 1);
                const uint32_t use = (uint32_t)(i >> 1);
                if (!mbar_wait_bounded(bar_addr(&ctl->tempty[buf]), (use & 1u) ^ 1u, abort_flag, p.wait_limit_ns,
                                       p.err))
                    break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(buf * 256);
                for (int kb = kb0; kb < kb1; ++kb) {
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
                                         (kb > kb0 || kk > 0) ? 1u : 0u);
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
        auto release = [&](int buf) {   // hand the accumulator back to the MMA issuer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_rank(bar_addr(&ctl->tempty[buf]), 0));
        };
        pdl_wait();
        uint32_t fix_round = 0;
        int64_t id;
        int kb0, kb1;
        for (int64_t i = 0; work.seg(i, id, kb0, kb1); ++i) {
            const StdTile t = tile_of(id);
            const int buf = (int)(i & 1);
            const uint32_t use = (uint32_t)(i >> 1);
            const bool got =
                mbar_wait_bounded(bar_addr(&ctl->tfull[buf]), use & 1u, abort_flag, p.wait_limit_ns, p.err);
            if (!named_barrier_and(1, 128, got)) break;
            tc_fence_after();
            const uint32_t tacc = tmem_base + (uint32_t)(buf * 256) + lane_off;
            const int64_t tok = (int64_t)t.m * 256 + rank * 128 + row;
            const bool tok_ok = tok < p.T;
            if (kb0 == 0 && kb1 == kbp) {   // the whole tile: straight from tensor memory
                if constexpr (EPI == EPI_SWIGLU) {
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {
                        float g[16], u[16];
                        load_tmem_chunk(tacc + (uint32_t)(c * 16), g);
                        load_tmem_chunk(tacc + (uint32_t)(128 + c * 16), u);
                        pair_store_swiglu(p, t, tok, tok_ok, c, g, u);
                    }
                } else {
#pragma unroll 1
                    for (int c = 0; c < 16; ++c) {
                        float v[16];
                        load_tmem_chunk(tacc + (uint32_t)(c * 16), v);
                        pair_store_cols<EPI>(p, t, tok, tok_ok, c, v);
                    }
                }
                release(buf);
                continue;
            }
            // A part of a split tile (at most two parts: the host's choice of clusters).  Park
            // it in this CTA's slot (0 for the cluster's first segment, 1 for its last), count
            // it, and if it arrived last, sum both parts in part order and finish the tile.
            int64_t id_next;
            int nb0, nb1;
            const bool final_seg = !work.seg(i + 1, id_next, nb0, nb1);
            float *slot = p.slots + ((size_t)blockIdx.x * 2 + (work.ub >= id * kbp ? 0 : 1)) * kPairSlotFloats;
#pragma unroll 1
            for (int c = 0; c < 16; ++c) {
                float v[16];
                load_tmem_chunk(tacc + (uint32_t)(c * 16), v);
#pragma unroll
                for (int k = 0; k < 16; ++k) __stcg(slot + (size_t)(c * 16 + k) * 128 + row, v[k]);
            }
            fence_proxy_async_global();   // a finisher may fetch this slot with a bulk copy
            named_barrier_sync(1, 128);
            const int64_t c_first = sk.owner(id * kbp), c_last = sk.owner(id * kbp + kbp - 1);
            const int nparts = (int)(c_last - c_first + 1);
            int *ctr = p.counters + id * 2 + rank;
            if (threadIdx.x == 64) ctl->fin_flag = atomic_add_acq_rel_gpu(ctr, 1) == nparts - 1 ? 1 : 0;
            named_barrier_sync(1, 128);
            const bool finisher = ctl->fin_flag != 0;
            auto part = [&](int64_t cc) -> const float * {   // part of cluster cc (this CTA's rank)
                return p.slots + ((size_t)(cc * 2 + rank) * 2 + (sk.begin(cc) >= id * kbp ? 0 : 1)) * kPairSlotFloats;
            };
            if (finisher && nparts == 2 && final_seg && ring_bytes >= kPairSlotFloats * 4u) {
                // the ring is idle after this cluster's last MMA: the other part goes into it
                // with one bulk copy; this CTA's own part is still in tensor memory
                const bool own_first = c_first == cluster;
                bool ok = true;
                if (threadIdx.x == 64) {
                    fence_proxy_async_global();
                    mbar_arrive_expect_tx(bar_addr(&ctl->fixbar), kPairSlotFloats * 4u);
                    bulk_load(base, part(own_first ? c_last : c_first), kPairSlotFloats * 4u, bar_addr(&ctl->fixbar));
                    ok = mbar_wait_bounded(bar_addr(&ctl->fixbar), fix_round & 1u, abort_flag, p.wait_limit_ns, p.err);
                }
                ++fix_round;
                if (!named_barrier_and(1, 128, ok)) {
                    if (threadIdx.x == 64)
                        (void)mbar_wait_drain(bar_addr(&ctl->fixbar), (fix_round - 1) & 1u,
                                              drain_limit_ns(p.wait_limit_ns));
                    release(buf);
                    break;
                }
                const float *other = reinterpret_cast<const float *>(ring);
                auto sum2 = [&](int col0, float (&v)[16]) {   // (0 + first part) + second part
                    float own[16];
                    load_tmem_chunk(tacc + (uint32_t)col0, own);
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float o = other[(col0 + k) * 128 + row];
                        v[k] = own_first ? (0.f + own[k]) + o : (0.f + o) + own[k];
                    }
                };
                if constexpr (EPI == EPI_SWIGLU) {
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {
                        float g[16], u[16];
                        sum2(c * 16, g);
                        sum2(128 + c * 16, u);
                        pair_store_swiglu(p, t, tok, tok_ok, c, g, u);
                    }
                } else {
#pragma unroll 1
                    for (int c = 0; c < 16; ++c) {
                        float v[16];
                        sum2(c * 16, v);
                        pair_store_cols<EPI>(p, t, tok, tok_ok, c, v);
                    }
                }
                release(buf);
            } else {
                release(buf);
                if (finisher) {
                    // from L2, every part in cluster order (first to arrive finishing early, or
                    // more than two parts)
                    auto sumk = [&](int col0, float (&v)[16]) {
#pragma unroll
                        for (int k = 0; k < 16; ++k) v[k] = 0.f;
                        for (int64_t cc = c_first; cc <= c_last; ++cc) {
                            const float *src = part(cc) + row;
                            float w[16];
#pragma unroll
                            for (int k = 0; k < 16; ++k) w[k] = __ldcg(src + (size_t)(col0 + k) * 128);
#pragma unroll
                            for (int k = 0; k < 16; ++k) v[k] += w[k];
                        }
                    };
                    if constexpr (EPI == EPI_SWIGLU) {
#pragma unroll 1
                        for (int c = 0; c < 8; ++c) {
                            float g[16], u[16];
                            sumk(c * 16, g);
                            sumk(128 + c * 16, u);
                            pair_store_swiglu(p, t, tok, tok_ok, c, g, u);
                        }
                    } else {
#pragma unroll 1
                        for (int c = 0; c < 16; ++c) {
                            float v[16];
                            sumk(c * 16, v);
                            pair_store_cols<EPI>(p, t, tok, tok_ok, c, v);
                        }
                    }
                }
            }
            if (finisher && threadIdx.x == 64) *ctr = 0;
            named_barrier_sync(1, 128);   // fin_flag is reused by the next segment
        }
    }

    // ---- teardown ----
    if (warp == 0 && lane == 0) {
        // every issued stage is released by the leader's MMA commit once its bytes
        // (from both CTAs) have landed and been consumed
        const int64_t first = issued > S ? issued - S : 0;
        for (int64_t i = first; i < issued; ++i) {
            const bool done = mbar_wait_drain(bar_addr(&ctl->empty[i % S]), (uint32_t)((i / S) & 1),
                                              drain_limit_ns(p.wait_limit_ns));
            if (!done) __nanosleep(200000);   // abort path: let in-flight copies land
        }
    }
    if (warp == 1 && lane == 0 && leader) {
        tc_commit_pair_multicast(bar_addr(&ctl->drain), (uint16_t)0x1);
        (void)mbar_wait_drain(bar_addr(&ctl->drain), 0, drain_limit_ns(p.wait_limit_ns));
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

// Opt the kernel into the largest dynamic shared memory once per device.
constexpr int kSmemAttrSlots = 32;   // one per kernel instantiation (slots 0..20 in use)

template <typename Kern>
cudaError_t ensure_smem_attr(Kern kern, int slot) {
    static std::atomic<uint64_t> done[kSmemAttrSlots];   // bit per device, per kernel slot
    if (slot < 0 || slot >= kSmemAttrSlots) return cudaErrorInvalidValue;
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

// Largest number of CTAs any tile of a single-CTA stream-K launch is split between.
int swapab_max_parts(const SwapAbParams &p, int grid) {
    const int64_t U = p.total_units, kbp = p.kb_per_tile;
    if (U <= 0 || kbp <= 0 || grid <= 0) return 1;
    const int64_t n_tiles = U / kbp;
    auto owner = [&](int64_t u) { return ((u + 1) * grid - 1) / U; };
    int worst = 1;
    for (int64_t t = 0; t < n_tiles && t < 65536; ++t)
        worst = std::max(worst, (int)(owner(t * kbp + kbp - 1) - owner(t * kbp) + 1));
    return worst;
}

cudaError_t launch_swapab(int epi, const CUtensorMap &ta, const CUtensorMap &tb, const SwapAbParams &p, int grid,
                          bool pdl, bool pair, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3((unsigned)kSwapAbThreads);
    cfg.dynamicSmemBytes = swapab_smem_bytes(pair ? p.bn / 2 : p.bn, p.stages, p.kbs);
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (pair || p.cluster_finish) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = pair ? 2 : 3;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    cfg.gridDim = dim3((unsigned)(pair ? 2 * grid : grid));   // grid: workers (CTAs or pairs)
    cudaError_t e;
#define MSE_LAUNCH_SWAPAB(E, PR, SLOT)                                  \
    e = ensure_smem_attr(swapab_kernel<E, PR>, SLOT);                   \
    if (e != cudaSuccess) return e;                                     \
    return cudaLaunchKernelEx(&cfg, swapab_kernel<E, PR>, ta, tb, p);
#define MSE_LAUNCH_SWAPAB_COOP(E, SLOT)                                 \
    e = ensure_smem_attr(swapab_kernel<E, false, true>, SLOT);          \
    if (e != cudaSuccess) return e;                                     \
    return cudaLaunchKernelEx(&cfg, swapab_kernel<E, false, true>, ta, tb, p);
    if (!pair && epi != EPI_MERGED && !p.cluster_finish && swapab_max_parts(p, grid) >= p.coop_finish &&
        p.coop_finish > 0) {
        switch (epi) {
            case EPI_SWIGLU: MSE_LAUNCH_SWAPAB_COOP(EPI_SWIGLU, 18)
            case EPI_BF16: MSE_LAUNCH_SWAPAB_COOP(EPI_BF16, 19)
            default: MSE_LAUNCH_SWAPAB_COOP(EPI_F32, 20)
        }
    }
    if (!pair) {
        switch (epi) {
            case EPI_SWIGLU: MSE_LAUNCH_SWAPAB(EPI_SWIGLU, false, 0)
            case EPI_BF16: MSE_LAUNCH_SWAPAB(EPI_BF16, false, 1)
            case EPI_F32: MSE_LAUNCH_SWAPAB(EPI_F32, false, 2)
            default: MSE_LAUNCH_SWAPAB(EPI_MERGED, false, 3)
        }
    }
    switch (epi) {
        case EPI_SWIGLU: MSE_LAUNCH_SWAPAB(EPI_SWIGLU, true, 14)
        case EPI_BF16: MSE_LAUNCH_SWAPAB(EPI_BF16, true, 15)
        case EPI_F32: MSE_LAUNCH_SWAPAB(EPI_F32, true, 16)
        default: MSE_LAUNCH_SWAPAB(EPI_MERGED, true, 17)
    }
#undef MSE_LAUNCH_SWAPAB
#undef MSE_LAUNCH_SWAPAB_COOP
}

// Clusters of three single CTAs of the swap-AB kernel that can be resident at once.
int swapab_trio_max_clusters(int bn, int stages, int kbs) {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    int mc = cache[dev & 63].load();
    if (mc > 0) return mc;
    if (ensure_smem_attr(swapab_kernel<EPI_SWIGLU, false>, 0) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t q = {};
    q.gridDim = dim3(3);
    q.blockDim = dim3((unsigned)kSwapAbThreads);
    q.dynamicSmemBytes = swapab_smem_bytes(bn, stages, kbs);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 3;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    q.attrs = attr;
    q.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&mc, swapab_kernel<EPI_SWIGLU, false>, &q) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cache[dev & 63].store(mc);
    return mc;
}

// Pairs of the swap-AB kernel that can be resident at once (one wave).
int swapab_pair_max_clusters(int bn, int stages, int kbs) {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    int mc = cache[dev & 63].load();
    if (mc > 0) return mc;
    if (ensure_smem_attr(swapab_kernel<EPI_BF16, true>, 15) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t q = {};
    q.gridDim = dim3(2);
    q.blockDim = dim3((unsigned)kSwapAbThreads);
    q.dynamicSmemBytes = swapab_smem_bytes(bn / 2, stages, kbs);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    q.attrs = attr;
    q.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&mc, swapab_kernel<EPI_BF16, true>, &q) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cache[dev & 63].store(mc);
    return mc;
}

// One CTA per SM (the ring takes most of the shared memory) and grid <= SMs, so every
// CTA of the launch is resident once the previous work on the stream has left its SM;
// phase 1's waits on other CTAs are bounded like every other wait.
cudaError_t launch_swapab_mlp(int epi1, const CUtensorMap &ta0, const CUtensorMap &tb0, const CUtensorMap &ta1,
                              const CUtensorMap &tb1, const SwapAbMlpParams &fp, int grid, bool pdl, cudaStream_t s) {
    const SwapAbParams &p0 = fp.ph[0];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)kSwapAbThreads);
    cfg.dynamicSmemBytes = swapab_smem_bytes(p0.bn, p0.stages, p0.kbs);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e;
    switch (epi1) {
        case EPI_BF16:
            e = ensure_smem_attr(swapab_mlp_kernel<EPI_BF16>, 12);
            if (e != cudaSuccess) return e;
            return cudaLaunchKernelEx(&cfg, swapab_mlp_kernel<EPI_BF16>, ta0, tb0, ta1, tb1, fp);
        case EPI_F32:
            e = ensure_smem_attr(swapab_mlp_kernel<EPI_F32>, 13);
            if (e != cudaSuccess) return e;
            return cudaLaunchKernelEx(&cfg, swapab_mlp_kernel<EPI_F32>, ta0, tb0, ta1, tb1, fp);
        default:
            return cudaErrorInvalidValue;
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
// one token tile (up to 256 tokens, weights streamed once): seven stages of 32 KB (the
// 256-token layer 65.1 against 66.3 us with six); prefill keeps six (1,939 against
// 1,946-1,972 TFLOP/s with seven)
int pair_stages(bool one_token_tile) { return one_token_tile ? 7 : 6; }

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
