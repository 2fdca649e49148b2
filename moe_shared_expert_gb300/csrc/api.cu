// C-ABI entry points: argument validation (before any CUDA call), device
// check, workspace carving, tensor-map encoding and kernel dispatch.
#include <atomic>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "common.cuh"
#include "kernels.h"
#include "tc.h"

namespace mse {

__device__ uint32_t g_device_error_word;

namespace {

std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_path{MSE_PATH_AUTO};
std::atomic<int> g_prefill{MSE_PREFILL_AUTO};
std::atomic<int> g_tune_issue_group{0}, g_tune_stages{0}, g_tune_cache_hints{1}, g_tune_grid{0},
    g_tune_spin_wait{0}, g_tune_one_launch{0}, g_tune_pdl{1},
    g_tune_coop_finish{6}, g_tune_pair_min_t{0}, g_tune_grid_down{0}, g_tune_cluster_finish{0},
    g_tune_l2_prefetch{8}, g_tune_swapab_max_t{160}, g_tune_x_early{0}, g_tune_down_flags{0},
    g_tune_host_x_copiers{16}, g_tune_pair_split{1};
std::atomic<void *> g_ev_begin{nullptr}, g_ev_mid{nullptr}, g_ev_end{nullptr};

struct DeviceInfo {
    bool init = false;
    bool supported = false;
    int sm_count = 0;
    uint32_t *err = nullptr;
};
constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

mse_status current_device(DeviceInfo **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return MSE_ERR_UNSUPPORTED_DEVICE;
    }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.init) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return MSE_ERR_CUDA;
        }
        d.supported = (major == 10 && minor == 3);
        d.sm_count = sms;
        if (d.supported) {
            void *p = nullptr;
            if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) {
                cudaGetLastError();
                return MSE_ERR_CUDA;
            }
            d.err = static_cast<uint32_t *>(p);
        }
        d.init = true;
    }
    if (!d.supported) return MSE_ERR_UNSUPPORTED_DEVICE;
    *out = &d;
    return MSE_OK;
}

mse_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MSE_OK : MSE_ERR_CUDA; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int round_up16(int64_t v) { return (int)((v + 15) / 16 * 16); }

int pow2_at_least(int v) {
    int p = 64;   // two accumulator buffers of >= 32 columns each
    while (p < v) p <<= 1;
    return p;
}

// ----------------------------------------------------------------- workspace
// h | split-K slots of the (first) gate_up pass | of the down pass | of the second gate_up
// pass ... and, at the END of the caller's buffer, the sync words: counters of the gate_up
// tiles | counters of the down tiles | h-tile flags | exit and published-tile counts.  The
// sync words must be zero before a call and every call that completes leaves them zero.
// Their size depends on H and I only and they sit at the buffer's end whatever T is, while
// h and the slots grow from its start: so a workspace sized for T tokens serves every call
// with at most T tokens and the same H and I, in any order, and each call finds the sync
// words the previous one left at zero (the T-dependent h and slot regions never reach
// them).  Calls with token counts above the swap-AB range use no sync words but keep the
// room for them, so they do not overwrite them either.
struct MlpWs {
    size_t h_off = 0, slots_off = 0, slots_dn_off = 0, slots_gu2_off = 0, cnt_gu_off = 0, cnt_dn_off = 0,
           flags_off = 0, exit_off = 0, sync_off = 0, sync_bytes = 0, total = 0;
};

constexpr int64_t kSwapAbMaxT = 256;   // token counts the swap-AB kernels can serve (workspace layout)

size_t align_down(size_t v, size_t a) { return v / a * a; }

// Minimal layout for (T, H, I): the sync words directly after the slots.
MlpWs mlp_ws_layout(int64_t T, int64_t H, int64_t I) {
    MlpWs w;
    size_t off = 0;
    w.h_off = off;
    off = align_up(off + (size_t)T * (size_t)I * 2, 256);
    if (T <= kSwapAbMaxT) {
        // 2 slots per CTA of 128 rows x bn tokens (swap-AB), or of 128 tokens x 256 columns
        // (the CTA-pair kernel's split tiles, from 129 tokens on)
        const int bn = T > 128 ? 256 : round_up16(T);
        const size_t slot_region = (size_t)tc::kMaxGrid * 2 * 128 * (size_t)bn * 4;
        w.slots_off = off;
        off = align_up(off + slot_region, 256);
        w.slots_dn_off = off;
        off = align_up(off + slot_region, 256);
        w.slots_gu2_off = off;
        off = align_up(off + slot_region, 256);
    }
    w.sync_off = off;
    w.cnt_gu_off = off;
    off = align_up(off + (size_t)((I + 63) / 64) * 4, 256);
    w.cnt_dn_off = off;
    off = align_up(off + (size_t)((I + 63) / 64) * (size_t)((H + 127) / 128) * 4, 256);
    w.flags_off = off;
    off = align_up(off + (size_t)((I + 63) / 64) * 4, 256);
    w.exit_off = off;   // exit count, then the published-tile counts of the two gate_up passes
    off = align_up(off + 12, 256);
    w.sync_bytes = off - w.sync_off;
    w.total = off;
    return w;
}

// The layout inside a caller buffer of workspace_bytes (>= the minimal total): the sync
// words moved to the buffer's last 256-aligned sync_bytes.
MlpWs mlp_ws_place(int64_t T, int64_t H, int64_t I, size_t workspace_bytes) {
    MlpWs w = mlp_ws_layout(T, H, I);
    if (workspace_bytes < w.total) return w;
    const size_t base = align_down(workspace_bytes - w.sync_bytes, 256);
    const size_t delta = base - w.sync_off;
    w.sync_off += delta;
    w.cnt_gu_off += delta;
    w.cnt_dn_off += delta;
    w.flags_off += delta;
    w.exit_off += delta;
    return w;
}

// merged projection: split-K slots from the start, the tile counters at the end of the
// caller's buffer (their size depends on C only), as for the MLP workspace.
struct MergedWs {
    size_t slots_off = 0, cnt_off = 0, cnt_bytes = 0, total = 0;
};

MergedWs merged_ws_layout(int64_t T, int64_t C) {
    MergedWs w;
    size_t off = 0;
    if (T <= kSwapAbMaxT) {
        const int bn = round_up16(T);
        w.slots_off = off;
        off = align_up(off + (size_t)tc::kMaxGrid * 2 * 128 * (size_t)bn * 4, 256);
    }
    w.cnt_off = off;
    w.cnt_bytes = align_up((size_t)((C + 127) / 128) * 4, 256);
    off += w.cnt_bytes;
    w.total = off;
    return w;
}

MergedWs merged_ws_place(int64_t T, int64_t C, size_t workspace_bytes) {
    MergedWs w = merged_ws_layout(T, C);
    if (workspace_bytes >= w.total) w.cnt_off = align_down(workspace_bytes - w.cnt_bytes, 256);
    return w;
}

// ----------------------------------------------------------------- tensor maps
mse_status encoder(EncodeTiledFn *fn) {
    std::call_once(g_encode_once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(p);
        cudaGetLastError();
    });
    if (!g_encode) return MSE_ERR_CUDA;
    *fn = g_encode;
    return MSE_OK;
}

// Encoded descriptors are cached by their full argument list (they are plain host
// data; the driver call costs more than a lookup).
struct MapKey {
    uint64_t base;
    uint64_t dims[5];
    uint64_t strides[4];
    uint32_t box[5];
    int rank;
    bool operator==(const MapKey &o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};
struct MapKeyHash {
    size_t operator()(const MapKey &k) const {
        const unsigned char *p = reinterpret_cast<const unsigned char *>(&k);
        uint64_t h = 1469598103934665603ull;
        for (size_t i = 0; i < sizeof(MapKey); ++i) h = (h ^ p[i]) * 1099511628211ull;
        return (size_t)h;
    }
};
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_map_cache;
constexpr size_t kMapCacheMax = 4096;

// bf16 tensor map with 128-byte swizzle; dims/strides innermost first, strides in bytes.
mse_status make_map(CUtensorMap *m, const void *base, int rank, const uint64_t *dims, const uint64_t *strides,
                    const uint32_t *box) {
    MapKey key;
    std::memset(&key, 0, sizeof key);
    key.base = reinterpret_cast<uint64_t>(base);
    key.rank = rank;
    for (int i = 0; i < rank; ++i) { key.dims[i] = dims[i]; key.box[i] = box[i]; }
    for (int i = 0; i < rank - 1; ++i) key.strides[i] = strides[i];
    {
        std::lock_guard<std::mutex> lk(g_map_mu);
        auto it = g_map_cache.find(key);
        if (it != g_map_cache.end()) { *m = it->second; return MSE_OK; }
    }
    EncodeTiledFn fn;
    mse_status st = encoder(&fn);
    if (st != MSE_OK) return st;
    cuuint64_t d[5], s[4];
    cuuint32_t b[5], e[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
    }
    for (int i = 0; i < rank - 1; ++i) s[i] = strides[i];
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(base), d, s, b, e,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return MSE_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_map_mu);
    if (g_map_cache.size() >= kMapCacheMax) g_map_cache.clear();
    g_map_cache.emplace(key, *m);
    return MSE_OK;
}

// [rows x cols] row-major bf16 (row pitch ld elements), box 64 cols x box_rows rows.
mse_status map_2d(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
    const uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
    const uint64_t strides[1] = {(uint64_t)ld * 2};
    const uint32_t box[2] = {64u, (uint32_t)box_rows};
    return make_map(m, base, 2, dims, strides, box);
}

// W_gate_up [2I x H] viewed as (k, j, half): one box = `rows` gate rows followed by
// the `rows` up rows of the same j (rows = 128: the 256-row operand of the
// single-CTA prefill kernel).
mse_status map_gate_up_halves(CUtensorMap *m, const void *w, int64_t H, int64_t I, int rows) {
    const uint64_t dims[3] = {(uint64_t)H, (uint64_t)I, 2};
    const uint64_t strides[2] = {(uint64_t)H * 2, (uint64_t)I * H * 2};
    const uint32_t box[3] = {64, (uint32_t)rows, 2};
    return make_map(m, w, 3, dims, strides, box);
}

// W_gate_up [2I x H] viewed as (k, row r < 16, gate/up, 16-row block b): one box of
// 64 k x 16 rows x 2 halves x 4 blocks is the 128-row operand of a decode-size gate_up tile
// of 64 j, in which rows 32b .. 32b+15 are gate rows and rows 32b+16 .. 32b+31 the up rows of
// the same j, so that a warp's 32 accumulator lanes hold both factors of 16 j.
mse_status map_gate_up_interleaved(CUtensorMap *m, const void *w, int64_t H, int64_t I) {
    const uint64_t dims[4] = {(uint64_t)H, 16, 2, (uint64_t)(I / 16)};
    const uint64_t strides[3] = {(uint64_t)H * 2, (uint64_t)I * H * 2, (uint64_t)16 * H * 2};
    const uint32_t box[4] = {64, 16, 2, 4};
    return make_map(m, w, 4, dims, strides, box);
}

// ----------------------------------------------------------------- launch helpers
// pair: the CTA-pair kernel, whose CTAs each hold half of the token rows
tc::SwapAbParams swapab_base(int64_t T, int total_units, bool pair = false) {
    tc::SwapAbParams p;
    std::memset(&p, 0, sizeof p);
    p.bn = round_up16(T);
    // k-blocks per stage: 3 for token tiles of at most 64 (the full layer at 64 tokens measured
    // 53.8 against 55.0 us with the library's defaults, 16 tokens 50.7 against 52.2), 2 above
    // (128 tokens 63.1 against 65.0)
    const int ig = g_tune_issue_group.load();
    p.kbs = ig > 0 ? ig : (p.bn <= 64 ? 3 : 2);
    const int b_rows = pair ? p.bn / 2 : p.bn;
    int max_stages = tc::swapab_stages_for(b_rows, p.kbs);
    while (max_stages < 2 && p.kbs > 1) max_stages = tc::swapab_stages_for(b_rows, --p.kbs);
    const int want = g_tune_stages.load();
    p.stages = (want >= 2 && want < max_stages) ? want : max_stages;
    p.halves = 1;
    p.cache_hints = g_tune_cache_hints.load();
    p.spin_wait = g_tune_spin_wait.load();
    p.coop_finish = g_tune_coop_finish.load();
    p.tmem_cols = pow2_at_least(2 * p.bn);
    p.T = (int)T;
    p.total_units = total_units;
    p.wait_limit_ns = g_wait_limit_ns.load();
    return p;
}

bool use_pdl() { return g_tune_pdl.load() != 0; }

// Whether a launch of T tokens over `rows` weight rows takes the swap-AB kernels (else the
// prefill kernels).  Up to 256 tokens (the split-K slots the workspace layout provides),
// except that launches over at least 4096 weight rows switch at MSE_TUNE_SWAPAB_MAX_T
// (default 160): the full layer measured 80-93 us at 176-256 tokens on the swap-AB kernels,
// whose ring holds two stages there, and 72.6-73.2 us on the CTA-pair prefill kernel (68.3
// against 72.8 us at 160 tokens).  Narrow launches (a shard's slice) would leave most SMs
// idle on the prefill kernels.
bool use_swapab(int64_t T, int64_t rows) {
    if (T > kSwapAbMaxT) return false;
    return rows < 4096 || T <= g_tune_swapab_max_t.load();
}

// Stream-K grid for `units` units of `kbp` per tile.  Among CTA counts from 90% of the
// SMs up to all of them, the largest one that minimises the largest number of CTAs any
// tile is split between, if that is at most three: each extra part lengthens the tile's
// split-K tail, which the whole launch waits for (gate_up at T = 64: 144 CTAs split every
// tile in two, 152 split some in three; measured 54.9 against 56.2 us per layer, and the
// T = 128 sharded layer 67.6 against 71.7 us).  Cached per shape.
int stream_k_grid(int units, int kbp, int g_max) {
    static std::mutex mu;
    static std::unordered_map<uint64_t, int> cache;
    const uint64_t key = ((uint64_t)(uint32_t)units << 32) ^ ((uint64_t)(uint32_t)kbp << 12) ^ (uint64_t)g_max;
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    const int64_t U = units;
    const int64_t n_tiles = U / kbp;
    int best = g_max, best_parts = INT32_MAX;
    const int g_min = std::max(1, (g_max * 9 + 9) / 10);
    for (int G = g_max; G >= g_min; --G) {
        if (n_tiles > 65536) break;   // very large shapes: keep g_max
        auto owner = [&](int64_t u) { return ((u + 1) * G - 1) / U; };
        int worst = 1;
        for (int64_t t = 0; t < n_tiles && worst < best_parts; ++t)
            worst = std::max(worst, (int)(owner(t * kbp + kbp - 1) - owner(t * kbp) + 1));
        if (worst < best_parts) {
            best_parts = worst;
            best = G;
        }
    }
    // Fewer CTAs pay where tiles end up split in at most three parts.  Tiles split more ways
    // (the merged projection's 17 tiles of 112 k-blocks) take the grid that puts every tile in
    // the same number of parts, one part per CTA, when it keeps at least 80% of the SMs: 136
    // CTAs measured 14.8 against 16.3 us (13.9 against 16.1 with early token loads), where 138
    // or 152 CTAs leave parts straddling tiles.
    if (best_parts > 3) {
        const int64_t per = n_tiles > 0 ? g_max / n_tiles : 0;
        const int64_t aligned = n_tiles * per;
        best = (per >= 2 && kbp >= per && 5 * aligned >= 4LL * g_max) ? (int)aligned : g_max;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (cache.size() > 4096) cache.clear();
    cache.emplace(key, best);
    return best;
}

// kbp = 0: no tile-aware choice (all SMs).  override: a CTA count for this kernel that
// takes precedence over MSE_TUNE_GRID (0 = none).
int swapab_grid(const DeviceInfo &d, int total_units, int kbp, int override = 0) {
    int g = d.sm_count < tc::kMaxGrid ? d.sm_count : tc::kMaxGrid;
    const int want = override > 0 ? override : g_tune_grid.load();
    if (want > 0) {
        if (want < g) g = want;
    } else if (kbp > 0 && total_units > g) {
        g = stream_k_grid(total_units, kbp, g);
    }
    return g < total_units ? g : total_units;
}

// Swap-AB launch shape for n_real 128-row weight tiles per group: CTA pairs (each CTA
// one 128-row half of a 256-row tile, half of the tokens) from MSE_TUNE_PAIR_MIN_T tokens
// on, when the device can hold the clusters; single CTAs otherwise.  grid = workers.
struct SwapAbShape {
    tc::SwapAbParams p;
    bool pair;
    int grid;
    int b_box_rows;   // token rows of one B copy (each CTA's half for pairs)
};
// narrow: an MLP launch whose CTAs may be fewer than the SMs when its work is small (see below).
SwapAbShape swapab_shape(const DeviceInfo &d, int64_t T, int n_real, int groups, int kbp, bool down = false,
                         bool narrow = false) {
    SwapAbShape r;
    const int pmin = g_tune_pair_min_t.load();
    if (pmin > 0 && T >= pmin) {
        const int n_mt = (n_real + 1) / 2;
        r.p = swapab_base(T, groups * n_mt * kbp, true);
        const int mc = tc::swapab_pair_max_clusters(r.p.bn, r.p.stages, r.p.kbs);
        if (mc > 0) {
            r.pair = true;
            r.p.n_mtiles = n_mt;
            r.p.n_mtiles_real = n_real;
            int g = std::min(d.sm_count, tc::kMaxGrid) / 2;
            const int want = g_tune_grid.load() / 2;
            if (want > 0 && want < g) g = want;
            g = std::min(g, mc);
            r.grid = std::max(1, std::min(g, r.p.total_units));
            r.b_box_rows = r.p.bn / 2;
            return r;
        }
    }
    r.pair = false;
    r.p = swapab_base(T, groups * n_real * kbp, false);
    r.p.n_mtiles = n_real;
    r.p.n_mtiles_real = n_real;
    r.grid = swapab_grid(d, r.p.total_units, kbp, down ? g_tune_grid_down.load() : 0);
    // Small work (one shard's narrow slice): at least 16 k-blocks per CTA, but never fewer
    // CTAs than half of the SMs.  Such launches are bound by their split-K tails and
    // stragglers, not by bytes, and fewer CTAs split each tile into fewer parts (one rank's
    // TP8 / TP16 step measured 1-3 us faster on 76-120 CTAs than on 152).  Not applied when
    // a grid is set through the tuning keys.
    if (narrow && g_tune_grid.load() == 0 && (!down || g_tune_grid_down.load() == 0)) {
        const int cap = std::max((r.p.total_units + 15) / 16, std::min(d.sm_count, tc::kMaxGrid) / 2);
        if (cap < r.grid) {
            r.grid = cap;
            // gate_up slices: every tile in the same number of parts, one part per CTA, on
            // about two thirds of the SMs (TP8's 12 tiles and TP16's 6 on 96 CTAs: one rank's
            // step 19.5 against 20.2 us and 16.0 against 17.4, with early token loads 15.9
            // against 16.4 and 13.8 against 15.6)
            const int n_tiles = groups * n_real;
            const int target = std::min(d.sm_count, tc::kMaxGrid) * 2 / 3;
            if (!down && n_tiles <= target && kbp >= 2 * (target / n_tiles)) r.grid = n_tiles * (target / n_tiles);
        }
    }
    // gate_up launches of at least 128 tokens over at least half as many tiles as SMs (the
    // full layer's 96): one CTA per whole tile, no split-K finish (the layer at 128 / 160
    // tokens 62.3 / 66.5 against 63.1 / 68.7 us, 59.3 / 61.6 against 60.8 / 66.4 with early
    // token loads and h flags; TP8 as partials at 128 tokens 65.9 against 68.0); at 80-96
    // tokens the stream-K split stays ahead by 0.3-1 us.
    {
        const int n_tiles = groups * n_real, g_cap = std::min(d.sm_count, tc::kMaxGrid);
        if (!down && g_tune_grid.load() == 0 && r.p.bn >= 128 && 2 * n_tiles >= g_cap && n_tiles <= g_cap)
            r.grid = n_tiles;
    }
    // Down projections of a narrow slice (at most 24 k-blocks per tile, one shard's or a few
    // shards' columns): one CTA per whole tile when every tile has an SM, so no tile is split
    // and no split-K finish runs (one rank's step at 64 tokens: TP8 20.3 against 27.1 us,
    // TP16 17.4 against 23.7, TP4 26.6 against 29.9).  The replicated layer's down projection
    // (96 k-blocks per tile) keeps the stream-K split, whose finish costs less than streaming
    // whole tiles on 56 SMs.
    if (down && narrow && g_tune_grid.load() == 0 && g_tune_grid_down.load() == 0 && kbp <= 24 &&
        (int64_t)groups * n_real <= std::min(d.sm_count, tc::kMaxGrid))
        r.grid = groups * n_real;
    r.b_box_rows = r.p.bn;
    // L2 prefetch beyond the ring by the CTAs that start during the previous kernel's tail,
    // for launches of at most 64 tokens whose CTAs stream at least 32 k-blocks each (the full
    // decode layer: 54.2 against 54.35 us per layer, its gate_up kernel alone 39.8 against
    // 40.9 us).  At 128 tokens (a shallower ring) it measured slower (the TP8 workload 69.4
    // against 66.8 us), and the narrow launches' ranges are mostly covered by the ring.
    if (r.p.bn <= 64 && r.p.total_units >= 32LL * r.grid) {
        r.p.l2_prefetch_kb = g_tune_l2_prefetch.load();
        r.p.l2_prefetch_from = std::max(0, d.sm_count - r.grid);
    }
    // clusters of three when three CTAs cover two tiles exactly (every tile in two parts)
    if (g_tune_cluster_finish.load() != 0 && r.grid % 3 == 0 &&
        3LL * r.p.total_units == 2LL * kbp * r.grid &&
        tc::swapab_trio_max_clusters(r.p.bn, r.p.stages, r.p.kbs) >= r.grid / 3)
        r.p.cluster_finish = 1;
    return r;
}

tc::StdParams std_base(int64_t T) {
    tc::StdParams p;
    std::memset(&p, 0, sizeof p);
    p.stages = tc::std_stages();
    p.T = (int)T;
    p.wait_limit_ns = g_wait_limit_ns.load();
    return p;
}

// Prefill-kernel choice (MSE_PREFILL_AUTO): the CTA pair up to 256 tokens (one 256-token
// tile: the full layer measured 73 us against 89 on single CTAs at 192-256 tokens) and from
// 512 on; single CTAs between (at 320 tokens 90 against 103 us for the pair, whose second
// token tile is mostly padding).
bool use_pair(int64_t T) {
    const int k = g_prefill.load();
    if (k == MSE_PREFILL_SINGLE) return false;
    if (k == MSE_PREFILL_PAIR) return true;
    return T <= 256 || T >= 512;
}

// Split-K for the CTA-pair kernel (MSE_TUNE_PAIR_SPLIT): when a launch has at most half as
// many tiles as clusters (up to 256 tokens: one token tile), the largest cluster count that
// splits no tile into more than two parts (the finisher then adds one other part); 0
// otherwise.  At 256 tokens the down projection's 28 tiles of 96 k-blocks run on 56 clusters
// (34.8 against 38.9 us alone); gate_up's 48 tiles stay whole: on 72 clusters it measured
// 47.1 against 43.3 us (the launch's operand stream does not grow with more SMs).
int pair_split_clusters(const DeviceInfo &d, int64_t n_tiles, int kbp) {
    const int64_t max_c = (d.sm_count < tc::kMaxPersistentGrid ? d.sm_count : tc::kMaxPersistentGrid) / 2;
    if (g_tune_pair_split.load() == 0 || 2 * n_tiles > max_c || kbp < 2) return 0;
    const int64_t U = n_tiles * kbp;
    for (int64_t C = max_c; C > n_tiles; --C) {
        int worst = 1;
        for (int64_t t = 0; t < n_tiles && worst <= 2; ++t) {
            const int64_t c0 = ((t * kbp + 1) * C - 1) / U, c1 = ((t * kbp + kbp) * C - 1) / U;
            worst = std::max(worst, (int)(c1 - c0 + 1));
        }
        if (worst <= 2) return (int)C;
    }
    return 0;
}

int pair_clusters(const DeviceInfo &d, int64_t n_tiles) {
    int64_t c = (d.sm_count < tc::kMaxPersistentGrid ? d.sm_count : tc::kMaxPersistentGrid) / 2;
    return (int)(c < n_tiles ? c : n_tiles);
}

int std_grid(const DeviceInfo &d, int64_t n_tiles) {
    int64_t g = d.sm_count < tc::kMaxPersistentGrid ? d.sm_count : tc::kMaxPersistentGrid;
    return (int)(g < n_tiles ? g : n_tiles);
}

// x of a replicated layer in host memory, copied by the gate_up launch itself
// (mlp_swiglu_forward_host on the decode-size kernels): the device view of the caller's x,
// the three copy-count words of this call's buffer, and whether the copy may run before
// the previous grid on the stream is complete.
struct HostX {
    const void *x_host;
    int *sync;
    bool early;
};

// gate_up + SiluAndMul over intermediate columns [j_begin, j_begin + width) into h [T x I].
// Whether the two swap-AB launches of a decode-size layer hand h over by per-block flags
// (MSE_TUNE_DOWN_FLAGS): both launches single-CTA and the gate_up launch without cluster
// finish (every other way of finishing a gate_up tile publishes it: the CTA that owns it
// whole, the last of its parts to arrive, or the last of its joint finishers).  Returns the
// epoch the flags of this call carry, or 0 for no flags.
int down_flags_epoch(const DeviceInfo &d, int64_t T, int64_t H, int64_t width, int64_t s_width, int groups);

// Early token loads: a gate_up grid streams while the previous call's down kernel (of the
// same shape as this call's, down_grid CTAs) finishes.  When that kernel leaves at least a
// third of the SMs free, as a shard's narrow down projection does, the grid takes those SMs,
// every tile in the same number of parts and one part per CTA, so that the two kernels run
// side by side (one rank's step at 64 tokens, TP4: 19.8 against 25.4 us).  n_gt: gate_up
// tiles; kbp: their k-blocks.
void coreside_gate_up_grid(const DeviceInfo &d, int n_gt, int kbp, int down_grid, SwapAbShape &sh) {
    const int free_sms = std::min(d.sm_count, tc::kMaxGrid) - down_grid;
    if (down_grid > 0 && !sh.pair && g_tune_grid.load() == 0 && 3 * free_sms >= d.sm_count && n_gt <= free_sms &&
        kbp >= 2 * (free_sms / n_gt)) {
        sh.grid = n_gt * (free_sms / n_gt);
        if (sh.p.total_units < 32LL * sh.grid) sh.p.l2_prefetch_kb = 0;
        sh.p.l2_prefetch_from = std::max(0, d.sm_count - sh.grid);
    }
}

mse_status tc_gate_up(const DeviceInfo &d, const uint16_t *x, int64_t T, int64_t H, int64_t I,
                      const uint16_t *w_gate_up, int64_t j_begin, int64_t width, uint16_t *h, char *ws,
                      const MlpWs &L, cudaStream_t s, bool x_early = false, int flags = 0,
                      const HostX *hx = nullptr, int down_grid = 0) {
    CUtensorMap ta, tb;
    mse_status st;
    if (use_swapab(T, 2 * width)) {
        const int kbp = (int)(H / 64);
        SwapAbShape sh = swapab_shape(d, T, (int)(width / 64), 1, kbp, false, true);
        tc::SwapAbParams &p = sh.p;
        if (x_early) coreside_gate_up_grid(d, (int)(width / 64), kbp, down_grid, sh);
        if ((st = map_gate_up_interleaved(&ta, w_gate_up, H, I)) != MSE_OK) return st;
        if ((st = map_2d(&tb, x, T, H, H, sh.b_box_rows)) != MSE_OK) return st;
        p.n_groups = 1;
        p.kb_per_tile = kbp;
        p.kb_first = 0;
        p.kb_group_stride = 0;
        p.a_row_base = (int)j_begin;
        p.m_valid = 2 * width;
        p.out = h;
        p.ldo = I;
        p.slots = reinterpret_cast<float *>(ws + L.slots_off);
        p.counters = reinterpret_cast<int *>(ws + L.cnt_gu_off);
        p.x_early = x_early ? 1 : 0;
        if (flags) {
            p.hflags = reinterpret_cast<int *>(ws + L.flags_off);
            p.hflag_epoch = flags;
        }
        if (hx) {
            if (sh.pair) return MSE_ERR_UNSUPPORTED_SHAPE;
            p.x_host = static_cast<const uint4 *>(hx->x_host);
            p.x_copy = reinterpret_cast<uint4 *>(const_cast<uint16_t *>(x));
            p.x_vecs = T * H * 2 / 16;
            p.x_sync = hx->sync;
            // the copiers should be CTAs that start while the previous layer's down kernel
            // still runs: at most the SMs that launch leaves free (its shape is this layer's)
            const SwapAbShape dn = swapab_shape(d, T, (int)((H + 127) / 128), 1, (int)(I / 64), true, true);
            const int free_sms = std::max(1, d.sm_count - dn.grid * (dn.pair ? 2 : 1));
            p.x_copiers = std::min({sh.grid, g_tune_host_x_copiers.load(), free_sms});
            p.x_copy_early = hx->early ? 1 : 0;
        }
        p.err = d.err;
        return from_cuda(tc::launch_swapab(tc::EPI_SWIGLU, ta, tb, p, sh.grid, use_pdl(), sh.pair, s));
    }
    if (hx) return MSE_ERR_UNSUPPORTED_SHAPE;
    tc::StdParams p = std_base(T);
    if (use_pair(T)) {
        p.stages = tc::pair_stages(T <= 256);
        if ((st = map_2d(&ta, x, T, H, H, 128)) != MSE_OK) return st;
        if ((st = map_2d(&tb, w_gate_up, 2 * I, H, H, 128)) != MSE_OK) return st;
        p.n_mtiles = (int)((T + 255) / 256);
        p.n_ntiles = (int)((width + 127) / 128);
        p.n_groups = 1;
        p.kb_per_tile = (int)(H / 64);
        p.n_valid = j_begin + width;
        p.n_base = (int)j_begin;
        p.b_base = (int)j_begin;
        p.b_n_stride = 128;
        p.b_rank_stride = (int)I;     // CTA 0 loads the gate rows, CTA 1 the up rows
        p.out = h;
        p.ldo = I;
        p.err = d.err;
        int clusters = pair_clusters(d, (int64_t)p.n_mtiles * p.n_ntiles);
        p.cache_hints = T <= 256 ? g_tune_cache_hints.load() : 0;   // weights streamed once
        p.x_early = x_early && T <= 256 ? 1 : 0;
        if (T <= kSwapAbMaxT && T > 128) {
            const int c = pair_split_clusters(d, (int64_t)p.n_mtiles * p.n_ntiles, p.kb_per_tile);
            if (c > 0) {
                p.split_k = 1;
                p.slots = reinterpret_cast<float *>(ws + L.slots_off);
                p.counters = reinterpret_cast<int *>(ws + L.cnt_gu_off);
                clusters = c;
            }
        }
        return from_cuda(tc::launch_pair(tc::EPI_SWIGLU, ta, tb, p, clusters, use_pdl(), s));
    }
    if ((st = map_2d(&ta, x, T, H, H, 128)) != MSE_OK) return st;
    if ((st = map_gate_up_halves(&tb, w_gate_up, H, I, 128)) != MSE_OK) return st;
    p.n_mtiles = (int)((T + 127) / 128);
    p.n_ntiles = (int)((width + 127) / 128);
    p.n_groups = 1;
    p.kb_per_tile = (int)(H / 64);
    p.n_valid = j_begin + width;
    p.n_base = (int)j_begin;
    p.out = h;
    p.ldo = I;
    p.err = d.err;
    const int64_t n_tiles = (int64_t)p.n_mtiles * p.n_ntiles;
    return from_cuda(tc::launch_std(tc::EPI_SWIGLU, ta, tb, p, std_grid(d, n_tiles), use_pdl(), s));
}

// out[g] = h[:, slice g] . W_down[:, slice g]^T for groups g, slices of `s_width`
// intermediate columns starting at column kcol0 + g * s_width.
mse_status tc_down(const DeviceInfo &d, const uint16_t *h, int64_t T, int64_t H, int64_t I, const uint16_t *w_down,
                   int64_t kcol0, int64_t s_width, int groups, void *out, int epi, char *ws, const MlpWs &L,
                   cudaStream_t s, int flags = 0, bool coreside = false) {
    CUtensorMap ta, tb;
    mse_status st;
    // the same choice as the layer's gate_up launch (its rows: 2 x the intermediate columns)
    if (use_swapab(T, 2 * (int64_t)groups * s_width)) {
        const int kbp = (int)(s_width / 64);
        SwapAbShape sh = swapab_shape(d, T, (int)((H + 127) / 128), groups, kbp, true, true);
        tc::SwapAbParams &p = sh.p;
        if ((st = map_2d(&ta, w_down, H, I, I, 128)) != MSE_OK) return st;
        if ((st = map_2d(&tb, h, T, I, I, sh.b_box_rows)) != MSE_OK) return st;
        p.n_groups = groups;
        p.kb_per_tile = kbp;
        p.kb_first = (int)(kcol0 / 64);
        p.kb_group_stride = kbp;
        p.m_valid = H;
        p.out = out;
        p.ldo = H;
        p.o_group_stride = T * H;
        p.slots = reinterpret_cast<float *>(ws + L.slots_dn_off);
        p.counters = reinterpret_cast<int *>(ws + L.cnt_dn_off);
        if (flags) {
            p.hflags = reinterpret_cast<int *>(ws + L.flags_off);
            p.exit_count = reinterpret_cast<int *>(ws + L.exit_off);
            p.hflag_first = (int)(kcol0 / 64);
            p.hflag_n = (int)((int64_t)groups * s_width / 64);
            p.hflag_epoch = flags;
        }
        p.err = d.err;
        return from_cuda(tc::launch_swapab(epi, ta, tb, p, sh.grid, use_pdl(), sh.pair, s));
    }
    tc::StdParams p = std_base(T);
    if (use_pair(T)) {
        p.stages = tc::pair_stages(T <= 256);
        if ((st = map_2d(&ta, h, T, I, I, 128)) != MSE_OK) return st;
        if ((st = map_2d(&tb, w_down, H, I, I, 128)) != MSE_OK) return st;
        p.n_mtiles = (int)((T + 255) / 256);
        p.n_ntiles = (int)((H + 255) / 256);
        p.n_groups = groups;
        p.kb_per_tile = (int)(s_width / 64);
        p.kb_first = (int)(kcol0 / 64);
        p.kb_group_stride = p.kb_per_tile;
        p.n_valid = H;
        p.b_base = 0;
        p.b_n_stride = 256;
        p.b_rank_stride = 128;
        p.out = out;
        p.ldo = H;
        p.o_group_stride = T * H;
        p.err = d.err;
        const int64_t n_tiles = (int64_t)groups * p.n_mtiles * p.n_ntiles;
        int clusters = pair_clusters(d, n_tiles);
        p.cache_hints = T <= 256 ? g_tune_cache_hints.load() : 0;   // weights streamed once
        // coreside (calls streamed with early token loads): whole tiles, so that the next
        // call's gate_up grid fits on the SMs this launch leaves free and streams beside it
        if (T <= kSwapAbMaxT && T > 128 && !coreside) {
            const int c = pair_split_clusters(d, n_tiles, p.kb_per_tile);
            if (c > 0) {
                p.split_k = 1;
                p.slots = reinterpret_cast<float *>(ws + L.slots_dn_off);
                p.counters = reinterpret_cast<int *>(ws + L.cnt_dn_off);
                clusters = c;
            }
        }
        return from_cuda(tc::launch_pair(epi, ta, tb, p, clusters, use_pdl(), s));
    }
    if ((st = map_2d(&ta, h, T, I, I, 128)) != MSE_OK) return st;
    if ((st = map_2d(&tb, w_down, H, I, I, 256)) != MSE_OK) return st;
    p.n_mtiles = (int)((T + 127) / 128);
    p.n_ntiles = (int)((H + 255) / 256);
    p.n_groups = groups;
    p.kb_per_tile = (int)(s_width / 64);
    p.kb_first = (int)(kcol0 / 64);
    p.kb_group_stride = p.kb_per_tile;
    p.n_valid = H;
    p.out = out;
    p.ldo = H;
    p.o_group_stride = T * H;
    p.err = d.err;
    const int64_t n_tiles = (int64_t)groups * p.n_mtiles * p.n_ntiles;
    return from_cuda(tc::launch_std(epi, ta, tb, p, std_grid(d, n_tiles), use_pdl(), s));
}

// The decode-size layer in one launch: gate_up + SiluAndMul over intermediate columns
// [j0, j0 + width) into h, then `groups` down projections of `s_width` columns each
// (group g reads h columns j0 + g * s_width ..) into out[g].
mse_status tc_mlp_one_launch(const DeviceInfo &d, const uint16_t *x, int64_t T, int64_t H, int64_t I,
                             const uint16_t *w_gate_up, const uint16_t *w_down, int64_t j0, int64_t width,
                             int64_t s_width, int groups, void *out, int epi1, char *ws, const MlpWs &L,
                             cudaStream_t s) {
    uint16_t *h = reinterpret_cast<uint16_t *>(ws + L.h_off);
    CUtensorMap ta0, tb0, ta1, tb1;
    mse_status st;
    const int n0 = (int)(width / 64), kbp0 = (int)(H / 64);
    const int n1 = (int)((H + 127) / 128), kbp1 = (int)(s_width / 64);
    // two gate_up passes (first and second half of the tiles) when the down pass can take
    // its k-blocks in matching halves
    const bool two = g_tune_one_launch.load() == 2 && groups == 1 && n0 >= 2 && n0 % 2 == 0 && kbp1 == n0;
    const int n0a = two ? n0 / 2 : n0;
    tc::SwapAbMlpParams fp;
    std::memset(&fp, 0, sizeof fp);
    tc::SwapAbParams &p0 = fp.ph[0];
    tc::SwapAbParams &p1 = fp.ph[2];
    p0 = swapab_base(T, n0a * kbp0);
    p1 = swapab_base(T, groups * n1 * (two ? kbp1 / 2 : kbp1));
    if ((st = map_gate_up_interleaved(&ta0, w_gate_up, H, I)) != MSE_OK) return st;
    if ((st = map_2d(&tb0, x, T, H, H, p0.bn)) != MSE_OK) return st;
    if ((st = map_2d(&ta1, w_down, H, I, I, 128)) != MSE_OK) return st;
    if ((st = map_2d(&tb1, h, T, I, I, p1.bn)) != MSE_OK) return st;
    p0.n_mtiles = n0a;
    p0.n_groups = 1;
    p0.kb_per_tile = kbp0;
    p0.a_row_base = (int)j0;
    p0.m_valid = 2 * width;
    p0.out = h;
    p0.ldo = I;
    p0.slots = reinterpret_cast<float *>(ws + L.slots_off);
    p0.counters = reinterpret_cast<int *>(ws + L.cnt_gu_off);
    p0.err = d.err;
    p1.n_mtiles = n1;
    p1.n_groups = groups;
    p1.kb_per_tile = two ? kbp1 / 2 : kbp1;
    p1.halves = two ? 2 : 1;
    p1.kb_first = (int)(j0 / 64);
    p1.kb_group_stride = kbp1;
    p1.m_valid = H;
    p1.out = out;
    p1.ldo = H;
    p1.o_group_stride = T * H;
    p1.slots = reinterpret_cast<float *>(ws + L.slots_dn_off);
    p1.counters = reinterpret_cast<int *>(ws + L.cnt_dn_off);
    p1.err = d.err;
    fp.n_gate_up_passes = 1;
    if (two) {
        tc::SwapAbParams &pb = fp.ph[1];
        pb = p0;
        pb.a_row_base = (int)j0 + n0a * 64;
        pb.n_mtiles = n0 - n0a;
        pb.total_units = pb.n_mtiles * kbp0;
        pb.slots = reinterpret_cast<float *>(ws + L.slots_gu2_off);
        pb.counters = p0.counters + n0a;
        fp.n_gate_up_passes = 2;
    }
    fp.hflags = reinterpret_cast<int *>(ws + L.flags_off);
    fp.hflag_first = (int)(j0 / 64);
    fp.n_htiles = n0;
    fp.hcount = reinterpret_cast<int *>(ws + L.exit_off) + 1;
    fp.exit_count = reinterpret_cast<int *>(ws + L.exit_off);
    // every CTA needs units in every pass: a split tile counts one part per CTA in the
    // range of its owners
    int units = p0.total_units < p1.total_units ? p0.total_units : p1.total_units;
    if (two && fp.ph[1].total_units < units) units = fp.ph[1].total_units;
    const int grid = swapab_grid(d, units, 0);   // one launch: every pass needs units on every CTA
    return from_cuda(tc::launch_swapab_mlp(epi1, ta0, tb0, ta1, tb1, fp, grid, use_pdl(), s));
}

bool one_launch_enabled(int64_t T) { return T <= kSwapAbMaxT && g_tune_one_launch.load() != 0; }

// Whether the gate_up launch of a replicated layer of T tokens copies x from host memory
// itself: the single-CTA swap-AB kernels of the two-launch layer.
bool hostx_supported(const DeviceInfo &d, int64_t T, int64_t H, int64_t I) {
    if (one_launch_enabled(T) || !use_swapab(T, 2 * I)) return false;
    return !swapab_shape(d, T, (int)(I / 64), 1, (int)(H / 64), false, true).pair;
}

std::atomic<uint32_t> g_epoch{0};

int down_flags_epoch(const DeviceInfo &d, int64_t T, int64_t H, int64_t width, int64_t s_width, int groups) {
    if (g_tune_down_flags.load() == 0 || !use_pdl() || !use_swapab(T, 2 * width)) return 0;
    SwapAbShape gu = swapab_shape(d, T, (int)(width / 64), 1, (int)(H / 64), false, true);
    if (gu.pair || gu.p.cluster_finish) return 0;
    const SwapAbShape dn = swapab_shape(d, T, (int)((H + 127) / 128), groups, (int)(s_width / 64), true, true);
    if (dn.pair) return 0;
    // positive, and different from the previous call's
    return (int)(g_epoch.fetch_add(1) % 0x7ffffffeu) + 1;
}

// CTAs of the swap-AB down launch of a layer call (0 when it does not take the swap-AB kernels).
int swapab_down_grid(const DeviceInfo &d, int64_t T, int64_t H, int64_t s_width, int groups) {
    if (!use_swapab(T, 2 * (int64_t)groups * s_width)) return 0;
    const SwapAbShape dn = swapab_shape(d, T, (int)((H + 127) / 128), groups, (int)(s_width / 64), true, true);
    return dn.pair ? 2 * dn.grid : dn.grid;
}

// ----------------------------------------------------------------- path choice
enum Path { PATH_GENERIC, PATH_TC };

mse_status choose(bool tc_ok, Path *out) {
    const int pol = g_path.load();
    if (pol == MSE_PATH_GENERIC) { *out = PATH_GENERIC; return MSE_OK; }
    if (pol == MSE_PATH_TENSORCORE) {
        if (!tc_ok) return MSE_ERR_UNSUPPORTED_SHAPE;
        *out = PATH_TC;
        return MSE_OK;
    }
    *out = tc_ok ? PATH_TC : PATH_GENERIC;
    return MSE_OK;
}

bool mlp_tc_ok(const void *x, int64_t H, int64_t I, int64_t slice, const void *wgu, const void *wd, const void *out,
               const void *ws) {
    return H % 64 == 0 && I % 64 == 0 && slice % 64 == 0 && aligned16(x) && aligned16(wgu) && aligned16(wd) &&
           aligned16(out) && aligned16(ws) && H <= (int64_t)1 << 20 && I <= (int64_t)1 << 20;
}

void record(std::atomic<void *> &ev, cudaStream_t s) {
    void *e = ev.load();
    if (e) cudaEventRecord(static_cast<cudaEvent_t>(e), s);
}

}  // namespace

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(); }

// Byte range of the sync words (tile counters, h flags, exit counts) inside an mlp
// workspace of workspace_bytes (they must be zero before a call).
void mlp_workspace_counter_range(int64_t T, int64_t H, int64_t I, size_t workspace_bytes, size_t *off,
                                 size_t *bytes) {
    const MlpWs L = mlp_ws_place(T, H, I, workspace_bytes);
    *off = L.sync_off;
    *bytes = L.sync_bytes;
}

}  // namespace mse

using namespace mse;

// =============================================================================
// exported C ABI
// =============================================================================
namespace mse {
namespace {
// The host range that the last mlp_swiglu_forward_host call on each stream writes (its
// y).  A call whose x overlaps it must not read x before that call's kernels are done;
// any other host range may be read while the previous work on the stream still runs
// (kernels of other libraries do not start this library's kernels early, and copies
// complete before a kernel after them starts).  Recorded in call order, so also right
// for calls captured into a CUDA graph.
struct HostOutput {
    void *stream;
    uintptr_t lo, hi;
};
std::mutex g_hostout_mu;
HostOutput g_hostout[64];
int g_hostout_n = 0;

// The device ranges that the last mlp_swiglu_forward call on each stream writes (y, its
// workspace), for MSE_TUNE_X_EARLY: the next call on the stream may read its x before the
// previous kernel completes when x overlaps neither.  Any other call of this library on the
// stream forgets the record (its kernels write other ranges).
struct StreamWrites {
    void *stream;
    uintptr_t lo[3], hi[3];
    bool known;
};
StreamWrites g_writes[64];
int g_writes_n = 0;

StreamWrites *stream_writes(void *stream) {   // caller holds g_hostout_mu
    for (int i = 0; i < g_writes_n; ++i)
        if (g_writes[i].stream == stream) return &g_writes[i];
    if (g_writes_n == 64) g_writes_n = 0;
    StreamWrites *w = &g_writes[g_writes_n++];
    w->stream = stream;
    w->known = false;
    return w;
}

bool x_independent_of_last_forward(void *stream, uintptr_t lo, uintptr_t hi) {
    std::lock_guard<std::mutex> lk(g_hostout_mu);
    const StreamWrites *w = stream_writes(stream);
    if (!w->known) return false;
    for (int k = 0; k < 3; ++k)
        if (lo < w->hi[k] && w->lo[k] < hi) return false;
    return true;
}

// The device ranges a call's kernels write (outputs and workspace; empty ranges allowed).
void record_forward_writes(void *stream, uintptr_t y_lo, uintptr_t y_hi, uintptr_t ws_lo, uintptr_t ws_hi,
                           uintptr_t z_lo = 0, uintptr_t z_hi = 0) {
    std::lock_guard<std::mutex> lk(g_hostout_mu);
    StreamWrites *w = stream_writes(stream);
    w->lo[0] = y_lo; w->hi[0] = y_hi; w->lo[1] = ws_lo; w->hi[1] = ws_hi; w->lo[2] = z_lo; w->hi[2] = z_hi;
    w->known = true;
}

// MSE_TUNE_X_EARLY for a call reading x [x, x + x_bytes) with workspace [ws, ws + ws_bytes):
// x overlaps neither this call's workspace nor anything the previous call on the stream
// writes (recorded in call order; no other call of this library came between).
bool x_early_for(void *stream, const void *x, size_t x_bytes, const void *ws, size_t ws_bytes) {
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x), wa = reinterpret_cast<uintptr_t>(ws);
    return g_tune_x_early.load() != 0 && !(xa < wa + ws_bytes && wa < xa + x_bytes) &&
           x_independent_of_last_forward(stream, xa, xa + x_bytes);
}

void forget_writes(void *stream) {
    std::lock_guard<std::mutex> lk(g_hostout_mu);
    stream_writes(stream)->known = false;
}

bool host_range_overlaps_last_output(void *stream, uintptr_t lo, uintptr_t hi) {
    std::lock_guard<std::mutex> lk(g_hostout_mu);
    for (int i = 0; i < g_hostout_n; ++i)
        if (g_hostout[i].stream == stream) return lo < g_hostout[i].hi && g_hostout[i].lo < hi;
    return false;
}

void record_host_output(void *stream, uintptr_t lo, uintptr_t hi) {
    std::lock_guard<std::mutex> lk(g_hostout_mu);
    for (int i = 0; i < g_hostout_n; ++i)
        if (g_hostout[i].stream == stream) { g_hostout[i].lo = lo; g_hostout[i].hi = hi; return; }
    if (g_hostout_n == 64) g_hostout_n = 0;   // forget the oldest streams (only makes copies wait)
    g_hostout[g_hostout_n++] = {stream, lo, hi};
}
}  // namespace
}  // namespace mse

// Workspace of mlp_swiglu_forward_host: the copy-count words of the two x buffers (fixed
// place, whatever T), the two device copies of x, then the workspace of the layer.
struct HostWs {
    size_t sync_off, x_off[2], mlp_off;
};
HostWs host_ws_layout(int64_t T, int64_t H) {
    const size_t act = align_up((size_t)T * (size_t)H * 2, 256);
    HostWs w;
    w.sync_off = 0;
    w.x_off[0] = 256;
    w.x_off[1] = 256 + act;
    w.mlp_off = 256 + 2 * act;
    return w;
}

// Which x buffer each host workspace used last (per workspace, in call order; a small table).
// A call takes the other buffer, and may copy early, only when the previous call on that
// workspace is known, had the same T and H, and was not captured into a graph.
struct XBufState {
    const void *ws;
    int64_t T, H;
    int buffer;
};
std::mutex g_xbuf_mu;
XBufState g_xbuf[16];
int g_xbuf_next = 0;

int next_x_buffer(const void *ws, int64_t T, int64_t H, bool capturing, bool *alternate) {
    std::lock_guard<std::mutex> lk(g_xbuf_mu);
    *alternate = false;
    XBufState *e = nullptr;
    for (auto &x : g_xbuf)
        if (x.ws == ws) e = &x;
    if (capturing) {
        if (e) e->ws = nullptr;
        return 0;
    }
    if (e && e->T == T && e->H == H) {
        e->buffer ^= 1;
        *alternate = true;
        return e->buffer;
    }
    if (!e) {
        e = &g_xbuf[g_xbuf_next];
        g_xbuf_next = (g_xbuf_next + 1) % 16;
    }
    *e = {ws, T, H, 0};
    return 0;
}

void forget_x_buffer(const void *ws) {
    std::lock_guard<std::mutex> lk(g_xbuf_mu);
    for (auto &x : g_xbuf)
        if (x.ws == ws) x.ws = nullptr;
}

// The replicated layer (mlp_swiglu_forward); hx: gate_up copies x from host memory into
// the device buffer x (mlp_swiglu_forward_host, decode-size kernels only).
mse_status forward_impl(const mse_bf16 *x, int64_t T, int64_t H, int64_t I, const mse_bf16 *w_gate_up,
                        const mse_bf16 *w_down, mse_bf16 *y, int64_t y_capacity, void *workspace,
                        size_t workspace_bytes, void *stream, const HostX *hx) {
    if (!x || !w_gate_up || !w_down || !y || T <= 0 || H <= 0 || I <= 0) return MSE_ERR_INVALID_ARG;
    if (y_capacity < T * H) return MSE_ERR_GEOMETRY;
    const MlpWs L = mlp_ws_place(T, H, I, workspace_bytes);
    if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MSE_ERR_WORKSPACE;
    DeviceInfo *d = nullptr;
    mse_status st = current_device(&d);
    if (st != MSE_OK) return st;
    Path path;
    if ((st = choose(mlp_tc_ok(x, H, I, I, w_gate_up, w_down, y, workspace), &path)) != MSE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    uint16_t *h = reinterpret_cast<uint16_t *>(ws + L.h_off);
    // MSE_TUNE_X_EARLY: x overlaps nothing the previous call on this stream writes (nor this
    // call's workspace); the record is forgotten until this call's launches succeed
    const uintptr_t wa = reinterpret_cast<uintptr_t>(workspace);
    const bool x_early = !hx && x_early_for(stream, x, (size_t)(T * H * 2), workspace, workspace_bytes);
    if (hx && (path != PATH_TC || !hostx_supported(*d, T, H, I))) return MSE_ERR_UNSUPPORTED_SHAPE;
    forget_writes(stream);

    record(g_ev_begin, s);
    if (path == PATH_GENERIC) {
        SimtGemmArgs a = {};
        a.A = x; a.lda = H; a.B = w_gate_up; a.B2 = w_gate_up + I * H; a.ldb = H;
        a.M = T; a.N = I; a.K = H; a.groups = 1; a.out = h; a.ldo = I; a.mode = SIMT_SWIGLU;
        if ((st = from_cuda(launch_simt_gemm(a, s))) != MSE_OK) return st;
        record(g_ev_mid, s);
        SimtGemmArgs b = {};
        b.A = h; b.lda = I; b.B = w_down; b.ldb = I;
        b.M = T; b.N = H; b.K = I; b.groups = 1; b.out = y; b.ldo = H; b.mode = SIMT_BF16;
        if ((st = from_cuda(launch_simt_gemm(b, s))) != MSE_OK) return st;
    } else {
        if (one_launch_enabled(T)) {
            if ((st = tc_mlp_one_launch(*d, x, T, H, I, w_gate_up, w_down, 0, I, I, 1, y, tc::EPI_BF16, ws, L, s)) !=
                MSE_OK)
                return st;
            record(g_ev_mid, s);   // one launch: no boundary between the passes
        } else {
            const int fl = down_flags_epoch(*d, T, H, I, I, 1);
            if ((st = tc_gate_up(*d, x, T, H, I, w_gate_up, 0, I, h, ws, L, s, x_early, fl, hx,
                                 x_early ? swapab_down_grid(*d, T, H, I, 1) : 0)) != MSE_OK)
                return st;
            record(g_ev_mid, s);
            if ((st = tc_down(*d, h, T, H, I, w_down, 0, I, 1, y, tc::EPI_BF16, ws, L, s, fl, x_early)) != MSE_OK)
                return st;
        }
    }
    record(g_ev_end, s);
    const uintptr_t ya = reinterpret_cast<uintptr_t>(y);
    record_forward_writes(stream, ya, ya + (uintptr_t)(T * H * 2), wa, wa + workspace_bytes);
    return MSE_OK;
}

extern "C" {

size_t mlp_swiglu_workspace_bytes(int64_t T, int64_t H, int64_t I) {
    if (T <= 0 || H <= 0 || I <= 0) return 0;
    // the largest need of any call with at most T tokens (the split-K slots of the swap-AB
    // range can outweigh h of a few hundred tokens more), so that the buffer serves them all
    const size_t n = mlp_ws_layout(T, H, I).total;
    const size_t m = mlp_ws_layout(T < kSwapAbMaxT ? T : kSwapAbMaxT, H, I).total;
    return n > m ? n : m;
}

size_t merged_proj_workspace_bytes(int64_t T, int64_t H, int64_t q_dim, int64_t kv_dim) {
    if (T <= 0 || H <= 0 || q_dim < 0 || kv_dim < 0 || q_dim + kv_dim <= 0) return 0;
    const size_t n = merged_ws_layout(T, q_dim + kv_dim).total;
    const size_t m = merged_ws_layout(T < kSwapAbMaxT ? T : kSwapAbMaxT, q_dim + kv_dim).total;
    return n > m ? n : m;
}

mse_status mlp_swiglu_workspace_sync_range(int64_t T, int64_t H, int64_t I, size_t workspace_bytes, size_t *offset,
                                          size_t *bytes) {
    if (T <= 0 || H <= 0 || I <= 0 || !offset || !bytes) return MSE_ERR_INVALID_ARG;
    const MlpWs L = mlp_ws_place(T, H, I, workspace_bytes);
    if (workspace_bytes < L.total) return MSE_ERR_WORKSPACE;
    *offset = L.sync_off;
    *bytes = L.sync_bytes;
    return MSE_OK;
}

mse_status merged_proj_workspace_sync_range(int64_t T, int64_t H, int64_t q_dim, int64_t kv_dim,
                                           size_t workspace_bytes, size_t *offset, size_t *bytes) {
    if (T <= 0 || H <= 0 || q_dim < 0 || kv_dim < 0 || q_dim + kv_dim <= 0 || !offset || !bytes)
        return MSE_ERR_INVALID_ARG;
    const MergedWs L = merged_ws_place(T, q_dim + kv_dim, workspace_bytes);
    if (workspace_bytes < L.total) return MSE_ERR_WORKSPACE;
    *offset = L.cnt_off;
    *bytes = L.cnt_bytes;
    return MSE_OK;
}

mse_status mlp_swiglu_forward(const mse_bf16 *x, int64_t T, int64_t H, int64_t I, const mse_bf16 *w_gate_up,
                              const mse_bf16 *w_down, mse_bf16 *y, int64_t y_capacity, void *workspace,
                              size_t workspace_bytes, void *stream) {
    return forward_impl(x, T, H, I, w_gate_up, w_down, y, y_capacity, workspace, workspace_bytes, stream, nullptr);
}

mse_status mlp_swiglu_shard_partial(const mse_bf16 *x, int64_t T, int64_t H, int64_t I, const mse_bf16 *w_gate_up,
                                    const mse_bf16 *w_down, int tp, int rank_first, int rank_count, void *partials,
                                    mse_dtype partial_dtype, int64_t partials_capacity, void *workspace,
                                    size_t workspace_bytes, void *stream) {
    if (!x || !w_gate_up || !w_down || !partials || T <= 0 || H <= 0 || I <= 0 || tp <= 0)
        return MSE_ERR_INVALID_ARG;
    if (partial_dtype != MSE_BF16 && partial_dtype != MSE_F32) return MSE_ERR_INVALID_ARG;
    if (I % tp != 0 || H % tp != 0) return MSE_ERR_NOT_DIVISIBLE;
    if (rank_first < 0 || rank_count < 1 || (int64_t)rank_first + rank_count > tp) return MSE_ERR_GEOMETRY;
    if (partials_capacity < (int64_t)rank_count * T * H) return MSE_ERR_GEOMETRY;
    const MlpWs L = mlp_ws_place(T, H, I, workspace_bytes);
    if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MSE_ERR_WORKSPACE;
    DeviceInfo *d = nullptr;
    mse_status st = current_device(&d);
    if (st != MSE_OK) return st;
    const size_t out_bytes = (size_t)rank_count * T * H * (partial_dtype == MSE_F32 ? 4 : 2);
    const bool x_early = x_early_for(stream, x, (size_t)(T * H * 2), workspace, workspace_bytes);
    forget_writes(stream);
    const int64_t sw = I / tp;
    Path path;
    if ((st = choose(mlp_tc_ok(x, H, I, sw, w_gate_up, w_down, partials, workspace), &path)) != MSE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    uint16_t *h = reinterpret_cast<uint16_t *>(ws + L.h_off);
    const int64_t j0 = (int64_t)rank_first * sw, width = (int64_t)rank_count * sw;

    if (path == PATH_GENERIC) {
        // the shards' gate rows [j0, j0 + width) and up rows I + [j0, j0 + width)
        SimtGemmArgs a = {};
        a.A = x; a.lda = H; a.B = w_gate_up + j0 * H; a.B2 = w_gate_up + (I + j0) * H; a.ldb = H;
        a.M = T; a.N = width; a.K = H; a.groups = 1; a.out = h + j0; a.ldo = I; a.mode = SIMT_SWIGLU;
        if ((st = from_cuda(launch_simt_gemm(a, s))) != MSE_OK) return st;
        // per shard: its h columns times its W_down columns
        SimtGemmArgs b = {};
        b.A = h + j0; b.lda = I; b.a_gstride = sw;
        b.B = w_down + j0; b.ldb = I; b.b_gstride = sw;
        b.M = T; b.N = H; b.K = sw; b.groups = rank_count;
        b.out = partials; b.ldo = H; b.o_gstride = T * H;
        b.mode = partial_dtype == MSE_F32 ? SIMT_F32 : SIMT_BF16;
        return from_cuda(launch_simt_gemm(b, s));
    }
    const int epi = partial_dtype == MSE_F32 ? tc::EPI_F32 : tc::EPI_BF16;
    record(g_ev_begin, s);
    if (one_launch_enabled(T)) {
        st = tc_mlp_one_launch(*d, x, T, H, I, w_gate_up, w_down, j0, width, sw, rank_count, partials, epi, ws, L, s);
        if (st != MSE_OK) return st;
        record(g_ev_mid, s);
    } else {
        const int fl = down_flags_epoch(*d, T, H, width, sw, rank_count);
        if ((st = tc_gate_up(*d, x, T, H, I, w_gate_up, j0, width, h, ws, L, s, x_early, fl, nullptr,
                             x_early ? swapab_down_grid(*d, T, H, sw, rank_count) : 0)) != MSE_OK)
            return st;
        record(g_ev_mid, s);
        if ((st = tc_down(*d, h, T, H, I, w_down, j0, sw, rank_count, partials, epi, ws, L, s, fl)) != MSE_OK)
            return st;
    }
    record(g_ev_end, s);
    const uintptr_t pa = reinterpret_cast<uintptr_t>(partials), wa = reinterpret_cast<uintptr_t>(workspace);
    record_forward_writes(stream, pa, pa + out_bytes, wa, wa + workspace_bytes);
    return MSE_OK;
}

mse_status mlp_swiglu_shard_forward(const mse_bf16 *x, int64_t T, int64_t H, int64_t I, const mse_bf16 *w_gate_up,
                                    const mse_bf16 *w_down, int tp, int rank_first, int rank_count, void *out,
                                    mse_dtype out_dtype, int64_t out_capacity, void *workspace,
                                    size_t workspace_bytes, void *stream) {
    if (!x || !w_gate_up || !w_down || !out || T <= 0 || H <= 0 || I <= 0 || tp <= 0)
        return MSE_ERR_INVALID_ARG;
    if (out_dtype != MSE_BF16 && out_dtype != MSE_F32) return MSE_ERR_INVALID_ARG;
    if (I % tp != 0 || H % tp != 0) return MSE_ERR_NOT_DIVISIBLE;
    if (rank_first < 0 || rank_count < 1 || (int64_t)rank_first + rank_count > tp) return MSE_ERR_GEOMETRY;
    if (out_capacity < T * H) return MSE_ERR_GEOMETRY;
    const MlpWs L = mlp_ws_place(T, H, I, workspace_bytes);
    if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MSE_ERR_WORKSPACE;
    DeviceInfo *d = nullptr;
    mse_status st = current_device(&d);
    if (st != MSE_OK) return st;
    const size_t out_bytes = (size_t)T * H * (out_dtype == MSE_F32 ? 4 : 2);
    const bool x_early = x_early_for(stream, x, (size_t)(T * H * 2), workspace, workspace_bytes);
    forget_writes(stream);
    const int64_t sw = I / tp;
    Path path;
    if ((st = choose(mlp_tc_ok(x, H, I, sw, w_gate_up, w_down, out, workspace), &path)) != MSE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    uint16_t *h = reinterpret_cast<uint16_t *>(ws + L.h_off);
    // the group's intermediate columns form one contiguous range: one reduction over it
    const int64_t j0 = (int64_t)rank_first * sw, width = (int64_t)rank_count * sw;

    if (path == PATH_GENERIC) {
        SimtGemmArgs a = {};
        a.A = x; a.lda = H; a.B = w_gate_up + j0 * H; a.B2 = w_gate_up + (I + j0) * H; a.ldb = H;
        a.M = T; a.N = width; a.K = H; a.groups = 1; a.out = h + j0; a.ldo = I; a.mode = SIMT_SWIGLU;
        if ((st = from_cuda(launch_simt_gemm(a, s))) != MSE_OK) return st;
        SimtGemmArgs b = {};
        b.A = h + j0; b.lda = I;
        b.B = w_down + j0; b.ldb = I;
        b.M = T; b.N = H; b.K = width; b.groups = 1;
        b.out = out; b.ldo = H;
        b.mode = out_dtype == MSE_F32 ? SIMT_F32 : SIMT_BF16;
        return from_cuda(launch_simt_gemm(b, s));
    }
    const int epi = out_dtype == MSE_F32 ? tc::EPI_F32 : tc::EPI_BF16;
    record(g_ev_begin, s);
    if (one_launch_enabled(T)) {
        if ((st = tc_mlp_one_launch(*d, x, T, H, I, w_gate_up, w_down, j0, width, width, 1, out, epi, ws, L, s)) !=
            MSE_OK)
            return st;
        record(g_ev_mid, s);
    } else {
        const int fl = down_flags_epoch(*d, T, H, width, width, 1);
        if ((st = tc_gate_up(*d, x, T, H, I, w_gate_up, j0, width, h, ws, L, s, x_early, fl, nullptr,
                             x_early ? swapab_down_grid(*d, T, H, width, 1) : 0)) != MSE_OK)
            return st;
        record(g_ev_mid, s);
        if ((st = tc_down(*d, h, T, H, I, w_down, j0, width, 1, out, epi, ws, L, s, fl)) != MSE_OK) return st;
    }
    record(g_ev_end, s);
    const uintptr_t oa = reinterpret_cast<uintptr_t>(out), wa = reinterpret_cast<uintptr_t>(workspace);
    record_forward_writes(stream, oa, oa + out_bytes, wa, wa + workspace_bytes);
    return MSE_OK;
}

size_t mlp_swiglu_host_workspace_bytes(int64_t T, int64_t H, int64_t I) {
    const size_t n = mlp_swiglu_workspace_bytes(T, H, I);
    if (n == 0) return 0;
    return host_ws_layout(T, H).mlp_off + n;
}

mse_status mlp_swiglu_forward_host(const mse_bf16 *x_host, int64_t T, int64_t H, int64_t I,
                                   const mse_bf16 *w_gate_up, const mse_bf16 *w_down, mse_bf16 *y_host,
                                   int64_t y_capacity, void *workspace, size_t workspace_bytes, void *stream) {
    if (!x_host || !w_gate_up || !w_down || !y_host || T <= 0 || H <= 0 || I <= 0) return MSE_ERR_INVALID_ARG;
    if (y_capacity < T * H) return MSE_ERR_GEOMETRY;
    const HostWs hw = host_ws_layout(T, H);
    if (!workspace || workspace_bytes < hw.mlp_off || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MSE_ERR_WORKSPACE;
    const MlpWs L = mlp_ws_place(T, H, I, workspace_bytes - hw.mlp_off);
    if (workspace_bytes - hw.mlp_off < L.total) return MSE_ERR_WORKSPACE;
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x_host), ya = reinterpret_cast<uintptr_t>(y_host);
    const uintptr_t nb = (uintptr_t)(T * H * 2);
    if (xa < ya + nb && ya < xa + nb) return MSE_ERR_INVALID_ARG;   // x and y overlap
    DeviceInfo *d = nullptr;
    mse_status st = current_device(&d);
    if (st != MSE_OK) return st;
    // the device's view of the caller's page-locked buffers
    void *xh = nullptr, *yh = nullptr;
    if (cudaHostGetDevicePointer(&xh, const_cast<mse_bf16 *>(x_host), 0) != cudaSuccess ||
        cudaHostGetDevicePointer(&yh, y_host, 0) != cudaSuccess) {
        cudaGetLastError();
        return MSE_ERR_INVALID_ARG;
    }
    char *ws = static_cast<char *>(workspace);
    char *wsm = ws + hw.mlp_off;
    const size_t wsm_bytes = workspace_bytes - hw.mlp_off;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // x may be read before the previous work on the stream is done unless the previous call
    // of this entry point on the stream writes it
    const bool read_early = !host_range_overlaps_last_output(stream, xa, xa + nb);
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
        cudaGetLastError();
        cap = cudaStreamCaptureStatusActive;   // unknown: take the waiting copy
    }
    const bool hostx = g_tune_host_x_copiers.load() > 0 && g_path.load() != MSE_PATH_GENERIC && aligned16(xh) &&
                       mlp_tc_ok(ws + hw.x_off[0], H, I, I, w_gate_up, w_down, yh, wsm) &&
                       hostx_supported(*d, T, H, I);
    record_host_output(stream, ya, ya + nb);
    forget_writes(stream);
    if (hostx) {
        // the gate_up launch copies x into one of two buffers, the other one than the
        // previous call on this workspace: the copy may then run before the previous grid
        // is complete, since every reader of this buffer is an earlier call's gate_up
        bool alternate = false;
        const int b = next_x_buffer(workspace, T, H, cap != cudaStreamCaptureStatusNone, &alternate);
        const HostX hx = {xh, reinterpret_cast<int *>(ws + hw.sync_off) + 4 * b, alternate && read_early};
        st = forward_impl(reinterpret_cast<const mse_bf16 *>(ws + hw.x_off[b]), T, H, I, w_gate_up, w_down,
                          static_cast<mse_bf16 *>(yh), y_capacity, wsm, wsm_bytes, stream, &hx);
        if (st != MSE_OK) forget_x_buffer(workspace);
        return st;
    }
    // otherwise a copy kernel into buffer 0, which writes once the previous work is complete
    forget_x_buffer(workspace);
    mse_bf16 *xd = reinterpret_cast<mse_bf16 *>(ws + hw.x_off[0]);
    forget_writes(stream);   // the copy kernel writes this call's x
    if ((st = from_cuda(launch_copy_in(xh, xd, T * H * 2, read_early, d->sm_count, s))) != MSE_OK) return st;
    // the down projection writes y straight into the caller's host buffer
    return forward_impl(xd, T, H, I, w_gate_up, w_down, static_cast<mse_bf16 *>(yh), y_capacity, wsm, wsm_bytes,
                        stream, nullptr);
}

int mse_shard_sequence_parallel_mlp(int enabled, int use_sequence_parallel, int eligible, int tp_size,
                                    int64_t hidden_size, int64_t intermediate_size) {
    if (!enabled || !use_sequence_parallel || !eligible || tp_size <= 1) return 0;
    return hidden_size % tp_size == 0 && intermediate_size % tp_size == 0 ? 1 : 0;
}

mse_status shard_sum(const void *partials, mse_dtype partial_dtype, int n_parts, int64_t T, int64_t H,
                     mse_bf16 *out, int64_t out_capacity, void *stream) {
    if (!partials || !out || n_parts <= 0 || T <= 0 || H <= 0) return MSE_ERR_INVALID_ARG;
    if (partial_dtype != MSE_BF16 && partial_dtype != MSE_F32) return MSE_ERR_INVALID_ARG;
    if (T % n_parts != 0) return MSE_ERR_NOT_DIVISIBLE;
    if (out_capacity < T * H) return MSE_ERR_GEOMETRY;
    DeviceInfo *d = nullptr;
    mse_status st = current_device(&d);
    if (st != MSE_OK) return st;
    forget_writes(stream);
    return from_cuda(launch_shard_sum(partials, partial_dtype == MSE_F32, n_parts, T * H, out, d->sm_count,
                                      use_pdl(), static_cast<cudaStream_t>(stream)));
}

mse_status merged_proj_forward(const mse_bf16 *x, int64_t T, int64_t H, const mse_bf16 *w, int64_t q_dim,
                               int64_t kv_dim, int tp, mse_bf16 *out_logical, mse_bf16 *out_rank_major,
                               int64_t out_capacity, void *workspace, size_t workspace_bytes, void *stream) {
    if (!x || !w || (!out_logical && !out_rank_major) || T <= 0 || H <= 0 || q_dim <= 0 || kv_dim <= 0 || tp <= 0)
        return MSE_ERR_INVALID_ARG;
    if (q_dim % tp != 0 || kv_dim % tp != 0) return MSE_ERR_NOT_DIVISIBLE;
    const int64_t C = q_dim + kv_dim;
    if (out_capacity < T * C) return MSE_ERR_GEOMETRY;
    const MergedWs L = merged_ws_place(T, C, workspace_bytes);
    if (!workspace || workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MSE_ERR_WORKSPACE;
    DeviceInfo *d = nullptr;
    mse_status st = current_device(&d);
    if (st != MSE_OK) return st;
    const bool x_early = x_early_for(stream, x, (size_t)(T * H * 2), workspace, workspace_bytes);
    forget_writes(stream);
    const bool tc_ok = H % 64 == 0 && aligned16(x) && aligned16(w) && aligned16(workspace);
    Path path;
    if ((st = choose(tc_ok, &path)) != MSE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (path == PATH_GENERIC) {
        SimtGemmArgs a = {};
        a.A = x; a.lda = H; a.B = w; a.ldb = H; a.M = T; a.N = C; a.K = H; a.groups = 1;
        a.out = out_logical; a.ldo = C; a.out_rm = out_rank_major; a.q_dim = q_dim; a.kv_dim = kv_dim; a.tp = tp;
        a.mode = SIMT_MERGED;
        return from_cuda(launch_simt_gemm(a, s));
    }
    CUtensorMap ta, tb;
    char *ws = static_cast<char *>(workspace);
    if (use_swapab(T, C)) {
        const int kbp = (int)(H / 64);
        SwapAbShape sh = swapab_shape(*d, T, (int)((C + 127) / 128), 1, kbp);
        tc::SwapAbParams &p = sh.p;
        if ((st = map_2d(&ta, w, C, H, H, 128)) != MSE_OK) return st;
        if ((st = map_2d(&tb, x, T, H, H, sh.b_box_rows)) != MSE_OK) return st;
        p.n_groups = 1;
        p.kb_per_tile = kbp;
        p.m_valid = C;
        p.out = out_logical;
        p.ldo = C;
        p.out_rm = out_rank_major;
        p.q_dim = q_dim; p.kv_dim = kv_dim; p.tp = tp;
        p.slots = reinterpret_cast<float *>(ws + L.slots_off);
        p.counters = reinterpret_cast<int *>(ws + L.cnt_off);
        p.x_early = x_early ? 1 : 0;
        p.err = d->err;
        if ((st = from_cuda(tc::launch_swapab(tc::EPI_MERGED, ta, tb, p, sh.grid, use_pdl(), sh.pair, s))) !=
            MSE_OK)
            return st;
        // what this call writes, for the next call's MSE_TUNE_X_EARLY
        const uintptr_t la = reinterpret_cast<uintptr_t>(out_logical), ra = reinterpret_cast<uintptr_t>(out_rank_major);
        const uintptr_t wa = reinterpret_cast<uintptr_t>(workspace), ob = (uintptr_t)(T * C * 2);
        record_forward_writes(stream, la, la ? la + ob : 0, wa, wa + workspace_bytes, ra, ra ? ra + ob : 0);
        return MSE_OK;
    }
    tc::StdParams p = std_base(T);
    if (use_pair(T)) {
        p.stages = tc::pair_stages(T <= 256);
        if ((st = map_2d(&ta, x, T, H, H, 128)) != MSE_OK) return st;
        if ((st = map_2d(&tb, w, C, H, H, 128)) != MSE_OK) return st;
        p.n_mtiles = (int)((T + 255) / 256);
        p.n_ntiles = (int)((C + 255) / 256);
        p.n_groups = 1;
        p.kb_per_tile = (int)(H / 64);
        p.n_valid = C;
        p.b_base = 0;
        p.b_n_stride = 256;
        p.b_rank_stride = 128;
        p.out = out_logical;
        p.ldo = C;
        p.out_rm = out_rank_major;
        p.q_dim = q_dim; p.kv_dim = kv_dim; p.tp = tp;
        p.err = d->err;
        return from_cuda(tc::launch_pair(tc::EPI_MERGED, ta, tb, p,
                                         pair_clusters(*d, (int64_t)p.n_mtiles * p.n_ntiles), use_pdl(), s));
    }
    if ((st = map_2d(&ta, x, T, H, H, 128)) != MSE_OK) return st;
    if ((st = map_2d(&tb, w, C, H, H, 256)) != MSE_OK) return st;
    p.n_mtiles = (int)((T + 127) / 128);
    p.n_ntiles = (int)((C + 255) / 256);
    p.n_groups = 1;
    p.kb_per_tile = (int)(H / 64);
    p.n_valid = C;
    p.out = out_logical;
    p.ldo = C;
    p.out_rm = out_rank_major;
    p.q_dim = q_dim; p.kv_dim = kv_dim; p.tp = tp;
    p.err = d->err;
    return from_cuda(
        tc::launch_std(tc::EPI_MERGED, ta, tb, p, std_grid(*d, (int64_t)p.n_mtiles * p.n_ntiles), use_pdl(), s));
}

mse_status merged_proj_reorder(const mse_bf16 *rank_major, mse_bf16 *logical, int64_t T, int64_t q_dim,
                               int64_t kv_dim, int tp, int64_t capacity, void *stream) {
    if (!rank_major || !logical || T <= 0 || q_dim <= 0 || kv_dim <= 0 || tp <= 0) return MSE_ERR_INVALID_ARG;
    if (q_dim % tp != 0 || kv_dim % tp != 0) return MSE_ERR_NOT_DIVISIBLE;
    const int64_t C = q_dim + kv_dim;
    if (capacity < T * C) return MSE_ERR_GEOMETRY;
    const uintptr_t a = reinterpret_cast<uintptr_t>(rank_major), b = reinterpret_cast<uintptr_t>(logical);
    const uintptr_t n = (uintptr_t)(T * C * 2);
    if (a < b + n && b < a + n) return MSE_ERR_INVALID_ARG;   // buffers overlap
    DeviceInfo *d = nullptr;
    mse_status st = current_device(&d);
    if (st != MSE_OK) return st;
    forget_writes(stream);
    return from_cuda(
        launch_reorder(rank_major, logical, T, q_dim, kv_dim, tp, use_pdl(), static_cast<cudaStream_t>(stream)));
}

mse_status mse_poll_device_error(void *stream) {
    DeviceInfo *d = nullptr;
    mse_status st = current_device(&d);
    if (st != MSE_OK) return st;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return MSE_ERR_CUDA;
    }
    uint32_t word = 0;
    if (cudaMemcpy(&word, d->err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) return MSE_ERR_CUDA;
    if (word != 0) {
        const uint32_t zero = 0;
        if (cudaMemcpy(d->err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) return MSE_ERR_CUDA;
    }
    return (word & DEV_ERR_TIMEOUT) ? MSE_ERR_TIMEOUT : MSE_OK;
}

void mse_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns); }
uint64_t mse_get_wait_limit_ns(void) { return g_wait_limit_ns.load(); }

int mse_set_kernel_path(int path) {
    if (path < MSE_PATH_AUTO || path > MSE_PATH_TENSORCORE) return g_path.load();
    return g_path.exchange(path);
}

int mse_set_prefill_kernel(int kind) {
    if (kind < MSE_PREFILL_AUTO || kind > MSE_PREFILL_PAIR) return g_prefill.load();
    return g_prefill.exchange(kind);
}

int mse_mlp_launch_plan(int64_t T, int64_t H, int64_t I, int tp, int rank_count, int x_early, int sm_count,
                        int32_t *out) {
    if (!out || T < 1 || H < 1 || I < 1 || tp < 1 || rank_count < 1 || rank_count > tp || sm_count < 1)
        return MSE_ERR_INVALID_ARG;
    for (int i = 0; i < 8; ++i) out[i] = 0;
    if (I % tp != 0) return MSE_ERR_NOT_DIVISIBLE;
    const int64_t sw = I / tp, width = (int64_t)rank_count * sw;
    // the generic kernels (shapes off the 64-column grid, or that path forced)
    if (H % 64 != 0 || sw % 64 != 0 || g_path.load() == MSE_PATH_GENERIC) return MSE_OK;
    // options whose shapes depend on occupancy queries of a device
    if (one_launch_enabled(T) || g_tune_pair_min_t.load() > 0 || g_tune_cluster_finish.load() != 0)
        return MSE_ERR_UNSUPPORTED_SHAPE;
    if (!use_swapab(T, 2 * width)) return MSE_OK;    // the prefill kernels
    DeviceInfo d;
    d.init = true;
    d.supported = true;
    d.sm_count = sm_count;
    const int kbp = (int)(H / 64);
    SwapAbShape gu = swapab_shape(d, T, (int)(width / 64), 1, kbp, false, true);
    gu.p.kb_per_tile = kbp;
    if (x_early) coreside_gate_up_grid(d, (int)(width / 64), kbp, swapab_down_grid(d, T, H, sw, rank_count), gu);
    SwapAbShape dn = swapab_shape(d, T, (int)((H + 127) / 128), rank_count, (int)(sw / 64), true, true);
    dn.p.kb_per_tile = (int)(sw / 64);
    out[0] = 1;
    out[1] = gu.grid;
    out[2] = dn.grid;
    out[3] = tc::swapab_max_parts(gu.p, gu.grid);
    out[4] = tc::swapab_max_parts(dn.p, dn.grid);
    out[5] = gu.p.bn;
    out[6] = gu.p.kbs;
    out[7] = gu.p.stages;
    return MSE_OK;
}

int mse_merged_launch_plan(int64_t T, int64_t H, int64_t q_dim, int64_t kv_dim, int tp, int sm_count, int32_t *out) {
    if (!out || T < 1 || H < 1 || q_dim < 1 || kv_dim < 1 || tp < 1 || sm_count < 1) return MSE_ERR_INVALID_ARG;
    for (int i = 0; i < 8; ++i) out[i] = 0;
    if (q_dim % tp != 0 || kv_dim % tp != 0) return MSE_ERR_NOT_DIVISIBLE;
    if (H % 64 != 0 || g_path.load() == MSE_PATH_GENERIC) return MSE_OK;   // the generic kernels
    const int64_t C = q_dim + kv_dim;
    if (!use_swapab(T, C)) return MSE_OK;   // the prefill kernels
    if (g_tune_pair_min_t.load() > 0 || g_tune_cluster_finish.load() != 0) return MSE_ERR_UNSUPPORTED_SHAPE;
    DeviceInfo d;
    d.init = true;
    d.supported = true;
    d.sm_count = sm_count;
    const int kbp = (int)(H / 64);
    SwapAbShape sh = swapab_shape(d, T, (int)((C + 127) / 128), 1, kbp);
    sh.p.kb_per_tile = kbp;
    const int parts = tc::swapab_max_parts(sh.p, sh.grid);
    out[0] = 1;
    out[1] = sh.grid;
    out[2] = parts;
    out[3] = sh.p.coop_finish > 0 && parts >= sh.p.coop_finish ? 1 : 0;
    out[4] = sh.p.bn;
    out[5] = sh.p.kbs;
    out[6] = sh.p.stages;
    return MSE_OK;
}

int mse_set_tuning(int key, int value) {
    std::atomic<int> *slot = nullptr;
    bool ok = false;
    switch (key) {
        case MSE_TUNE_ISSUE_GROUP: slot = &g_tune_issue_group; ok = value >= 0 && value <= 4; break;
        case MSE_TUNE_STAGES: slot = &g_tune_stages; ok = value == 0 || (value >= 2 && value <= tc::kMaxStages); break;
        case MSE_TUNE_CACHE_HINTS: slot = &g_tune_cache_hints; ok = value == 0 || value == 1; break;
        case MSE_TUNE_GRID: slot = &g_tune_grid; ok = value >= 0 && value <= tc::kMaxGrid; break;
        case MSE_TUNE_SPIN_WAIT: slot = &g_tune_spin_wait; ok = value == 0 || value == 1; break;
        case MSE_TUNE_ONE_LAUNCH: slot = &g_tune_one_launch; ok = value >= 0 && value <= 2; break;
        case MSE_TUNE_PDL: slot = &g_tune_pdl; ok = value == 0 || value == 1; break;
        case MSE_TUNE_COOP_FINISH: slot = &g_tune_coop_finish; ok = value >= 0 && value <= 128; break;
        case MSE_TUNE_PAIR_MIN_T: slot = &g_tune_pair_min_t; ok = value >= 0 && value <= 100000; break;
        case MSE_TUNE_GRID_DOWN: slot = &g_tune_grid_down; ok = value >= 0 && value <= tc::kMaxGrid; break;
        case MSE_TUNE_CLUSTER_FINISH: slot = &g_tune_cluster_finish; ok = value == 0 || value == 1; break;
        case MSE_TUNE_L2_PREFETCH: slot = &g_tune_l2_prefetch; ok = value >= 0 && value <= 256; break;
        case MSE_TUNE_SWAPAB_MAX_T: slot = &g_tune_swapab_max_t; ok = value >= 0 && value <= kSwapAbMaxT; break;
        case MSE_TUNE_X_EARLY: slot = &g_tune_x_early; ok = value == 0 || value == 1; break;
        case MSE_TUNE_DOWN_FLAGS: slot = &g_tune_down_flags; ok = value == 0 || value == 1; break;
        case MSE_TUNE_HOST_X_COPIERS: slot = &g_tune_host_x_copiers; ok = value >= 0 && value <= 1024; break;
        case MSE_TUNE_PAIR_SPLIT: slot = &g_tune_pair_split; ok = value == 0 || value == 1; break;
        default: return -1;
    }
    if (!ok) return -1;
    return slot->exchange(value);
}

void mse_set_phase_events(void *ev_begin, void *ev_mid, void *ev_end) {
    const bool all = ev_begin && ev_mid && ev_end;
    g_ev_begin.store(all ? ev_begin : nullptr);
    g_ev_mid.store(all ? ev_mid : nullptr);
    g_ev_end.store(all ? ev_end : nullptr);
}

mse_status mse_selftest_wait_timeout(uint64_t limit_ns, void *stream) {
    DeviceInfo *d = nullptr;
    mse_status st = current_device(&d);
    if (st != MSE_OK) return st;
    return from_cuda(launch_wait_selftest(limit_ns, d->err, static_cast<cudaStream_t>(stream)));
}

const char *mse_status_string(mse_status s) {
    switch (s) {
        case MSE_OK: return "MSE_OK";
        case MSE_ERR_INVALID_ARG: return "MSE_ERR_INVALID_ARG";
        case MSE_ERR_NOT_DIVISIBLE: return "MSE_ERR_NOT_DIVISIBLE";
        case MSE_ERR_GEOMETRY: return "MSE_ERR_GEOMETRY";
        case MSE_ERR_WORKSPACE: return "MSE_ERR_WORKSPACE";
        case MSE_ERR_UNSUPPORTED_DEVICE: return "MSE_ERR_UNSUPPORTED_DEVICE";
        case MSE_ERR_CUDA: return "MSE_ERR_CUDA";
        case MSE_ERR_TIMEOUT: return "MSE_ERR_TIMEOUT";
        case MSE_ERR_UNSUPPORTED_SHAPE: return "MSE_ERR_UNSUPPORTED_SHAPE";
    }
    return "MSE_ERR_UNKNOWN";
}

const char *mse_version(void) { return "mse 0.1 sm_103a"; }

}  // extern "C"
