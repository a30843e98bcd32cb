// gsa_api.cu -- the C ABI of libgsa (declared in include/gsa.h): argument
// validation, layout queries, the work schedule (built on the host, or by the
// one-CTA plan kernel for the graph-safe calls), TMA descriptors and the
// launches: one fused kernel per call (plus the plan kernel when graph-safe).
// No allocation, no synchronization (except gsa_workspace_status), every
// launch on the caller's stream.  Also the wait self-test kernel.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "gsa.h"
#include "gsa_kernel.cuh"

namespace {

using namespace gsa;

thread_local int32_t g_last_launches = 0;

struct Plan {
    int64_t M = 0;
    int W = 0, W_in = 0, E = 0, B = 0;
    bool glu = false;
    std::vector<int64_t> row_off, pad_off;
    std::vector<int> band_start;
    std::vector<int> sc_row, sc_col;   // tiled scale layout: prefixes of ceil(M_e / 128), ceil(M_e / (4 B))
    int n_bands = 0, n_slabs = 0, tiles_per_slab = 0;
    int n_slabs2 = 0, tiles_per_slab2 = 0;   // encode (P2) items
};

bool is_glu(int act) { return act == ACT_SWIGLU || act == ACT_CLAMPED_SWIGLU; }

// Tiles per work item for a call (see make_plan; NVFP4 amax items are then
// fitted to the launch's grid by fit_items_to_grid).  Larger items mean fewer
// item epilogues, dprobs slab merges and scheduling rounds, smaller ones a
// finer-grained schedule with more items per CTA.  Measured (same box):
//  * NVFP4 (65536 x 2048 + RHT), amax items with 8 / 16 / 32 tiles and 8-tile
//    encode items (kEncodeItemTileCap): SReLU forward 188.0 / 191.6 / 202.3 us,
//    SReLU backward 286.2 / 281.3 / 289.4, TanhSReLU forward 237.2 / 233.6 /
//    229.6, TanhSReLU backward 327.8 / 303.9 / 303.4;
//  * MXFP8 (one pass): 2-tile items forward and 4-tile items backward against
//    8 for both: 8192 x 1024 TanhSReLU 35.0 -> 24.6 / 52.6 -> 41.1 us, SwiGLU
//    32768 x 2 x 2048 130.5 -> 120.9 / 315.7 -> 308.4 us, routed SwiGLU
//    262144 x 2 x 4096 1444 -> 1440 / 5175 -> 5048 us.
// The workspace is sized with the smallest cap any call of the recipe uses
// (the most slabs): for NVFP4 the floor of the grid fit (fit_items_to_grid).
bool costly_act(int act) { return act != GSA_ACT_SRELU && act != GSA_ACT_IDENTITY; }
constexpr int kNvMinItemTiles = 4;
int min_item_tile_cap(int recipe) { return recipe == GSA_MXFP8 ? 2 : kNvMinItemTiles; }
// NVFP4 encode items take at most 8 tiles whatever the amax items take: they run
// last, so smaller ones even out the end of the launch (the TanhSReLU backward,
// 32-tile amax items: 317.3 us with 32-tile encode items, 306.1 with 16, 303.4
// with 8, 314.9 with 4; same box).
constexpr int kEncodeItemTileCap = 8;
int item_tile_cap(int act, int recipe, bool bwd, bool two_pass) {
    if (recipe == GSA_MXFP8) return bwd ? 4 : 2;
    if (!two_pass) return 8;
    if (costly_act(act)) return 32;
    return bwd ? 16 : 8;
}

// Shape checks shared by every entry point.

// tile_cap: most tiles (of 64 columns) per work item, a power of two up to
// kMaxItemTiles; items take the largest power of two that divides the
// tiles of a row and does not exceed it -- or, where a band would then have
// more than kMaxSlabs slabs, the smallest larger one that avoids it (a row
// whose tile count has too few factors of two is unsupported).
gsa_status make_plan(int64_t E, const int64_t *split, int64_t W_in, int act, int recipe, Plan &pl,
                     int tile_cap) {
    if (E <= 0 || split == nullptr || W_in <= 0) return GSA_ERR_INVALID_ARG;
    if (act < 0 || act > ACT_IDENTITY || (recipe != GSA_MXFP8 && recipe != GSA_NVFP4)) return GSA_ERR_INVALID_ARG;
    pl.glu = is_glu(act);
    if (pl.glu && (W_in & 1)) return GSA_ERR_INVALID_ARG;
    const int64_t W = pl.glu ? W_in / 2 : W_in;
    pl.B = recipe == GSA_MXFP8 ? 32 : 16;
    if (W % pl.B != 0) return GSA_ERR_INVALID_ARG;
    if (E > kMaxExperts) return GSA_ERR_UNSUPPORTED;
    if (W % kCols != 0 || W_in > (int64_t(1) << 30)) return GSA_ERR_UNSUPPORTED;
    pl.E = static_cast<int>(E);
    pl.W = static_cast<int>(W);
    pl.W_in = static_cast<int>(W_in);
    pl.row_off.assign(E + 1, 0);
    pl.pad_off.assign(E + 1, 0);
    pl.band_start.assign(E + 1, 0);
    pl.sc_row.assign(E + 1, 0);
    pl.sc_col.assign(E + 1, 0);
    for (int64_t e = 0; e < E; ++e) {
        if (split[e] < 0) return GSA_ERR_INVALID_ARG;
        pl.row_off[e + 1] = pl.row_off[e] + split[e];
        pl.pad_off[e + 1] = pl.pad_off[e] + (split[e] + pl.B - 1) / pl.B * pl.B;
        if (split[e] >= (int64_t(1) << 31)) return GSA_ERR_UNSUPPORTED;
        pl.sc_row[e + 1] = pl.sc_row[e] + static_cast<int>((split[e] + 127) / 128);
        pl.sc_col[e + 1] = pl.sc_col[e] + static_cast<int>((split[e] + 4 * pl.B - 1) / (4 * pl.B));
        const int64_t nb = (split[e] + kRows - 1) / kRows;
        if (pl.band_start[e] + nb > (int64_t(1) << 30)) return GSA_ERR_UNSUPPORTED;
        pl.band_start[e + 1] = pl.band_start[e] + static_cast<int>(nb);
    }
    pl.M = pl.row_off[E];
    if (pl.M >= (int64_t(1) << 31) - kRows || pl.pad_off[E] >= (int64_t(1) << 31)) return GSA_ERR_UNSUPPORTED;
    pl.n_bands = pl.band_start[E];
    const int nct = pl.W / kCols;
    int t = 1;
    while (t < tile_cap && t < kMaxItemTiles && nct % (2 * t) == 0) t *= 2;
    // wide rows: larger items than the cap where the slabs of a band would
    // exceed what the dprobs slab merge holds
    while (nct / t > kMaxSlabs && t < kMaxItemTiles && nct % (2 * t) == 0) t *= 2;
    pl.tiles_per_slab = t;
    pl.n_slabs = nct / t;
    if (pl.n_slabs > kMaxSlabs) return GSA_ERR_UNSUPPORTED;
    int t2 = 1;
    while (t2 < kEncodeItemTileCap && t2 < t && nct % (2 * t2) == 0) t2 *= 2;
    pl.tiles_per_slab2 = t2;
    pl.n_slabs2 = nct / t2;
    return GSA_OK;
}

size_t ws_counter_bytes(const Plan &pl) {
    const size_t words = WS_HDR + 5 * static_cast<size_t>(pl.E) + static_cast<size_t>(pl.n_bands);
    return (words * 4 + 255) / 256 * 256;
}

size_t ws_partial_bytes(const Plan &pl) {
    return pl.n_slabs > 1 ? (static_cast<size_t>(pl.M) * pl.n_slabs * 4 + 255) / 256 * 256 : 0;
}

// NVFP4: a BF16 staging copy of Y, written by the forward's amax pass and
// read back (from L2) by its encode pass: one 128-row x 64-column image
// (16 KiB, rows of 128 bytes) per band and column tile.
int64_t stash_rows(const Plan &pl) { return static_cast<int64_t>(pl.n_bands) * (pl.W / kCols) * kRows; }

size_t ws_stash_bytes(const Plan &pl, int recipe) {
    return recipe == GSA_NVFP4 ? static_cast<size_t>(stash_rows(pl)) * kCols * 2 : 0;
}

size_t ws_total_bytes(const Plan &pl, int recipe) {
    return ws_counter_bytes(pl) + ws_partial_bytes(pl) + ws_stash_bytes(pl, recipe);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

gsa_status check_act_params(int act, const gsa_act_params *ap) {
    if (act == GSA_ACT_TANH_SRELU) {
        if (!ap || !(ap->s > 0.0f) || !std::isfinite(ap->s)) return GSA_ERR_INVALID_ARG;
    }
    if (act == GSA_ACT_CLAMPED_SWIGLU) {
        if (!ap || !(ap->limit > 0.0f) || !std::isfinite(ap->limit) || !std::isfinite(ap->alpha) ||
            !std::isfinite(ap->glu_linear_offset))
            return GSA_ERR_INVALID_ARG;
    }
    return GSA_OK;
}

// A quantized output: both halves of each copy or neither; alignment; NVFP4 amax.
gsa_status check_qout(const gsa_qout *q, int recipe, bool need_row_amax, bool allow_row) {
    if (!q) return GSA_OK;
    if ((q->row_data == nullptr) != (q->row_scale == nullptr)) return GSA_ERR_INVALID_ARG;
    if ((q->col_data == nullptr) != (q->col_scale == nullptr)) return GSA_ERR_INVALID_ARG;
    if (!allow_row && q->row_data) return GSA_ERR_INVALID_ARG;
    if (q->row_data && (!aligned16(q->row_data) || !aligned16(q->row_scale))) return GSA_ERR_ALIGNMENT;
    if (q->col_data && (!aligned16(q->col_data) || !aligned16(q->col_scale))) return GSA_ERR_ALIGNMENT;
    if (recipe == GSA_NVFP4) {
        if (q->row_data && need_row_amax && !q->amax_row) return GSA_ERR_INVALID_ARG;
        if (q->col_data && !q->amax_col) return GSA_ERR_INVALID_ARG;
    }
    if ((q->amax_row && !aligned4(q->amax_row)) || (q->amax_col && !aligned4(q->amax_col))) return GSA_ERR_ALIGNMENT;
    return GSA_OK;
}

bool has_row(const gsa_qout *q) { return q && q->row_data; }
bool has_col(const gsa_qout *q) { return q && q->col_data; }

// An NVFP4 backward with a quantized copy (dX, or the regenerated Y) needs
// the amax pass before the encode pass.
bool bwd_two_pass(int recipe, const gsa_qout *dx_q, const gsa_qout *y_regen) {
    return recipe == GSA_NVFP4 && (has_row(dx_q) || has_col(dx_q) || has_col(y_regen));
}
bool fwd_two_pass(int recipe, const gsa_qout *y_q) { return recipe == GSA_NVFP4 && (has_row(y_q) || has_col(y_q)); }

QDev to_dev(const gsa_qout *q) {
    QDev d{};
    if (q) {
        d.row_data = static_cast<uint8_t *>(q->row_data);
        d.row_scale = static_cast<uint8_t *>(q->row_scale);
        d.col_data = static_cast<uint8_t *>(q->col_data);
        d.col_scale = static_cast<uint8_t *>(q->col_scale);
        d.amax_row = q->amax_row;
        d.amax_col = q->amax_col;
    }
    return d;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [rows, cols] BF16 row-major tensor, box 64 columns x 128 rows, 128-byte swizzle,
// zero fill outside the tensor.
bool make_tmap(CUtensorMap *tm, const void *ptr, int64_t rows, int64_t cols) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kCols), static_cast<cuuint32_t>(kRows)};
    cuuint32_t es[2] = {1, 1};
    CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

launch_fn pick(int act) {
    switch (act) {
    case ACT_SRELU: return launch_srelu;
    case ACT_TANH_SRELU: return launch_tanh_srelu;
    case ACT_SWIGLU: return launch_swiglu;
    case ACT_CLAMPED_SWIGLU: return launch_clamped_swiglu;
    case ACT_GELU: return launch_gelu;
    case ACT_SIGMOID: return launch_sigmoid;
    default: return launch_identity;
    }
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// NVFP4 amax items are halved (down to kNvMinItemTiles tiles; the encode
// items follow below 8) while `bands` bands would give fewer items than the
// launch has resident CTAs (3/4 of them for the static interleave of the cheap
// activations, whose crossover measured lower): with too few items SMs idle
// through the amax pass, and an expert's encode items wait longer for its
// amax.  Same box, NVFP4 + RHT, width 2048, 32 experts, 304 resident CTAs,
// rows (bands): us with the policy's cap against the halved caps --
//   TanhSReLU fwd / bwd, 32 / 16 / 8 / 4 tiles:
//     2048 (36): 8 tiles 55.9 / 59.1, 4 tiles 51.2 / 52.7
//     4096 (50): 109.5 / 130.8, 73.4 / 82.7, 65.4 / 69.5, 55.1 / 56.6
//     6144 (64): 8 tiles 68.1 / 73.4, 4 tiles 59.6 / 63.6
//     16384 (147): 114.7 / 137.0, 94.8 / 108.4, 87.5 / 106.2
//     24576 (208): 141.5 / 171.3, 112.8 / 135.2, 125.0 / 146.1
//     32768 (275): 149.0 / 180.0, 134.0 / 169.0, 143.5 / 177.6
//     40960 (339): 164.9 / 204.3, 185.7 / 235.0, 161.5 / 223.2
//   SReLU bwd, 16 / 8 / 4 tiles: 2048: 8 tiles 47.0, 4 tiles 33.0; 4096:
//     63.7 / 48.9 / 41.7; 6144: 8 tiles 51.5, 4 tiles 53.5; 12288 (112):
//     81.1 / 72.6; 16384: 87.2 / 95.0; 24576: 120.4 / 125.4.
//   SReLU fwd, 8 / 4 tiles: 2048: 38.3 / 30.6; 4096: 38.4 / 35.7; 6144:
//     39.0 / 40.6.
// Where the occupancy query fails the plan is left as it is (the launch then
// reports the error).
void fit_items_to_grid(Plan &pl, int64_t bands, int act, int recipe, bool bwd) {
    if (recipe != GSA_NVFP4 || pl.tiles_per_slab <= kNvMinItemTiles) return;
    KParams P;
    std::memset(&P, 0, sizeof(P));
    int per_sm = 0;
    if (pick(act)(recipe, bwd, P, 0, nullptr, &per_sm) != cudaSuccess || per_sm <= 0) return;
    int64_t slots = static_cast<int64_t>(per_sm) * sm_count();
    if (!costly_act(act)) slots = slots * 3 / 4;
    const int nct = pl.W / kCols;
    int t = pl.tiles_per_slab;
    while (t > kNvMinItemTiles && nct / (t / 2) <= kMaxSlabs && bands * (nct / t) < slots) t /= 2;
    pl.tiles_per_slab = t;
    pl.n_slabs = nct / t;
    if (pl.tiles_per_slab2 > t) {   // encode items no larger than the amax items
        pl.tiles_per_slab2 = t;
        pl.n_slabs2 = nct / t;
    }
}

// Activation constants, sizes and pointers common to both ways of building
// the tables.
void fill_common(const Plan &pl, KParams &P, const gsa_act_params *ap, void *ws) {
    const gsa_act_params zero{};
    const gsa_act_params &a = ap ? *ap : zero;
    P.M = static_cast<int>(pl.M);
    P.W = pl.W;
    P.W_in = pl.W_in;
    P.E = pl.E;
    P.n_slabs = pl.n_slabs;
    P.tiles_per_slab = pl.tiles_per_slab;
    P.n_slabs2 = pl.n_slabs2;
    P.tiles_per_slab2 = pl.tiles_per_slab2;
    P.s = a.s;
    P.s2 = a.s * a.s;
    P.two_s = 2.0f * a.s;
    {
        int ex = 0;
        const float m = std::frexp(a.s, &ex);   // s = m * 2^ex, m in [0.5, 1)
        P.s_pow2 = (a.s > 0.0f && m == 0.5f && std::isfinite(1.0f / a.s) && 1.0f / a.s >= 1.17549435e-38f) ? 1 : 0;
        P.inv_s = P.s_pow2 ? 1.0f / a.s : 0.0f;
    }
    P.limit = a.limit;
    P.alpha = a.alpha;
    P.off = a.glu_linear_offset;
    P.ws = static_cast<uint32_t *>(ws);
    P.partial = pl.n_slabs > 1 ? reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + ws_counter_bytes(pl)) : nullptr;
}

// activations as cheap as SReLU keep the static interleave; costly ones go ready-first
bool ready_first_for(int act, bool two_pass) { return two_pass && costly_act(act); }

// Fill schedule, expert tables and activation constants from the host split;
// then clear the workspace counters and launch.
gsa_status run(const Plan &pl, KParams &P, int act, int recipe, bool bwd, bool two_pass, const gsa_act_params *ap,
               void *ws, cudaStream_t stream) {
    launch_fn fn = pick(act);
    int per_sm = 0;
    if (fn(recipe, bwd, P, 0, stream, &per_sm) != cudaSuccess || per_sm <= 0) return GSA_ERR_CUDA;
    const int grid_hint = per_sm * sm_count();
    if (grid_hint <= 0) return GSA_ERR_CUDA;
    fill_common(pl, P, ap, ws);
    P.dtab = nullptr;
    for (int e = 0; e <= pl.E; ++e) {
        P.tab.row_off[e] = pl.row_off[e];
        P.tab.pad_off[e] = pl.pad_off[e];
        P.tab.band_start[e] = pl.band_start[e];
        P.tab.sc_row[e] = pl.sc_row[e];
        P.tab.sc_col[e] = pl.sc_col[e];
    }
    std::vector<int> order;
    for (int e = 0; e < pl.E; ++e)
        if (pl.row_off[e + 1] > pl.row_off[e]) order.push_back(e);
    if (two_pass)
        std::stable_sort(order.begin(), order.end(), [&](int x, int y) {
            return pl.row_off[x + 1] - pl.row_off[x] > pl.row_off[y + 1] - pl.row_off[y];
        });
    std::vector<int> pend_e(order.size() + 1), pend_pos(order.size() + 1);
    // lookahead: one wave of items (measured best for 8-tile items)
    build_queues(P.tab, order.data(), static_cast<int>(order.size()), pl.n_slabs, pl.n_slabs2, two_pass,
                 ready_first_for(act, two_pass), grid_hint, pend_e.data(), pend_pos.data());

    cudaError_t err = cudaMemsetAsync(ws, 0, ws_counter_bytes(pl), stream);
    if (err != cudaSuccess) return GSA_ERR_CUDA;
    g_last_launches = 0;
    if (P.tab.n_items == 0) {  // no rows at all: only the per-expert amax outputs need values
        for (int i = 0; i < 2; ++i) {
            if (P.q[i].amax_row && recipe == NVFP4)
                if (cudaMemsetAsync(P.q[i].amax_row, 0, sizeof(float) * pl.E, stream) != cudaSuccess) return GSA_ERR_CUDA;
            if (P.q[i].amax_col && recipe == NVFP4)
                if (cudaMemsetAsync(P.q[i].amax_col, 0, sizeof(float) * pl.E, stream) != cudaSuccess) return GSA_ERR_CUDA;
        }
        return GSA_OK;
    }
    const int grid = std::min(P.tab.n_items, grid_hint);
    if (grid <= 0) return GSA_ERR_CUDA;
    if (fn(recipe, bwd, P, grid, stream, &per_sm) != cudaSuccess) return GSA_ERR_CUDA;
    g_last_launches = 1;
    return GSA_OK;
}

// ------------------------------------------------------ graph-safe calls
//
// The split lives on the device, so nothing the host does depends on it: the
// plan kernel (one CTA) checks it, builds the tables with the same
// build_queues as the host path, and the fused kernel reads them through
// KParams::dtab.  Sizes are bounded by (E, M): at most M / 128 + E bands and
// M + E (B - 1) padded rows.

int64_t bands_bound(int64_t E, int64_t M) { return (M + (kRows - 1) * E) / kRows; }

// Plan for the graph-safe calls: everything but the split-dependent tables.
gsa_status make_plan_bound(int64_t E, int64_t M, int64_t W_in, int act, int recipe, Plan &pl,
                           int tile_cap) {
    if (M < 0) return GSA_ERR_INVALID_ARG;
    std::vector<int64_t> one(static_cast<size_t>(std::max<int64_t>(E, 1)), 0);
    if (E > 0) one[0] = M;
    gsa_status st = make_plan(E, one.data(), W_in, act, recipe, pl, tile_cap);   // shape checks with M rows in one expert
    if (st != GSA_OK) return st;
    const int64_t nb = bands_bound(E, M);
    if (nb > (int64_t(1) << 30) || M + E * pl.B >= (int64_t(1) << 31)) return GSA_ERR_UNSUPPORTED;
    pl.n_bands = static_cast<int>(nb);
    return GSA_OK;
}

size_t plan_tab_offset(const Plan &pl, int recipe) {
    return (ws_counter_bytes(pl) + ws_partial_bytes(pl) + ws_stash_bytes(pl, recipe) + 255) / 256 * 256;
}

size_t ws_graph_safe_bytes(const Plan &pl, int recipe) { return plan_tab_offset(pl, recipe) + sizeof(PlanTab); }

// One thread per expert and one more (the queue builder's tail position).
constexpr int kPlanThreads = kMaxExperts + 32;

// Inclusive prefix sums over the block of the K values each thread holds
// (Hillis-Steele in shared memory); every thread receives its prefixes in v.
template <int K>
__device__ void plan_block_scan(int64_t (&v)[K], int64_t (*buf)[kPlanThreads]) {
    const int t = threadIdx.x;
#pragma unroll
    for (int k = 0; k < K; ++k) buf[k][t] = v[k];
    __syncthreads();
    for (int d = 1; d < kPlanThreads; d <<= 1) {
        int64_t a[K];
#pragma unroll
        for (int k = 0; k < K; ++k) a[k] = t >= d ? buf[k][t - d] : 0;
        __syncthreads();
#pragma unroll
        for (int k = 0; k < K; ++k) buf[k][t] += a[k];
        __syncthreads();
    }
#pragma unroll
    for (int k = 0; k < K; ++k) v[k] = buf[k][t];
    __syncthreads();   // buf may be reused at once
}

__global__ void __launch_bounds__(kPlanThreads) gsa_plan_kernel(const int64_t *split, int E, int64_t M, int B,
                                                                int n_slabs, int n_slabs2, int two_pass, int ready_first,
                                                                int lookahead, PlanTab *T, uint32_t *ws,
                                                                int ctr_words, int64_t *pad_out) {
    // Per-expert prefixes and the queues by block-wide scans (thread t =
    // expert t, then position t of the order); only the filled part of the
    // tables goes out.
    __shared__ PlanTab S;
    __shared__ QueueScan Q;
    __shared__ int64_t buf[6][kPlanThreads];
    __shared__ int64_t sz[kMaxExperts];
    __shared__ int order[kMaxExperts];
    __shared__ int bad;
    const int t = threadIdx.x;
    for (int i = t; i < ctr_words; i += blockDim.x) ws[i] = 0u;   // the call's counters
    if (t == 0) bad = 0;
    __syncthreads();
    int64_t m = 0;
    if (t < E) {
        m = split[t];
        if (m < 0 || m > M) atomicOr(&bad, 1);
    }
    const int bsh = B == 32 ? 5 : 4;   // B is 16 or 32
    int64_t x[6], v[6];
    auto fill = [&](int64_t r) {   // r >= 0
        x[0] = r;
        x[1] = ((r + B - 1) >> bsh) << bsh;
        x[2] = (r + kRows - 1) >> 7;
        x[3] = (r + 127) >> 7;
        x[4] = (r + 4 * B - 1) >> (bsh + 2);
        x[5] = r > 0 ? 1 : 0;
#pragma unroll
        for (int k = 0; k < 6; ++k) v[k] = x[k];
    };
    fill(m < 0 ? 0 : m);   // a negative entry is already flagged
    plan_block_scan(v, buf);   // each term <= M: no overflow
    if (t == E - 1 && v[0] != M) bad = 1;
    __syncthreads();
    if (bad) {   // an invalid split is not processed: every expert empty
        if (t == 0) atomicOr(ws + WS_ERR, ERR_BAD_SPLIT);
        m = 0;
        fill(m);
        plan_block_scan(v, buf);
    }
    if (t < kMaxExperts) sz[t] = t < E ? m : 0;
    if (t < E) {
        S.row_off[t] = v[0] - x[0];
        S.pad_off[t] = v[1] - x[1];
        S.band_start[t] = static_cast<int>(v[2] - x[2]);
        S.sc_row[t] = static_cast<int>(v[3] - x[3]);
        S.sc_col[t] = static_cast<int>(v[4] - x[4]);
    }
    if (t == E - 1) {
        S.row_off[E] = v[0];
        S.pad_off[E] = v[1];
        S.band_start[E] = static_cast<int>(v[2]);
        S.sc_row[E] = static_cast<int>(v[3]);
        S.sc_col[E] = static_cast<int>(v[4]);
        buf[0][0] = v[5];
    }
    __syncthreads();
    const int n_order = static_cast<int>(buf[0][0]);
    if (t < E && sz[t] > 0) {   // rank among the non-empty experts: by size (two-pass, stable) or by index
        const int64_t mt = sz[t];
        int rank = 0;
        for (int e = 0; e < E; ++e)
            if (sz[e] > 0 && (two_pass ? (sz[e] > mt || (sz[e] == mt && e < t)) : e < t)) ++rank;
        order[rank] = t;
    }
    __syncthreads();

    // the queues (thread t = position t of the order, t = n_order the tail)
    const bool tp = two_pass != 0, rf = ready_first != 0;
    int c1, c2;
    queue_counts(S, order, n_order, n_slabs, n_slabs2, t, c1, c2);
    int64_t w[2] = {c1, c2};
    plan_block_scan(w, buf);
    if (t <= n_order) {
        Q.c[t] = static_cast<int>(w[0]) - c1;
        Q.c2[t] = static_cast<int>(w[1]) - c2;
    }
    __syncthreads();
    int ns = 0, ni = 0;
    if (t <= n_order) queue1_part<false>(S, Q, order, n_order, tp, rf, lookahead, t, ns, ni);
    int64_t u[2] = {ns, ni};
    plan_block_scan(u, buf);
    if (t <= n_order) {
        Q.so[t] = static_cast<int>(u[0]) - ns;
        Q.io[t] = static_cast<int>(u[1]) - ni;
    }
    if (t == n_order) buf[0][0] = u[0], buf[1][0] = u[1];   // totals: the tail is the last contributor
    __syncthreads();
    const int n_segs1 = static_cast<int>(buf[0][0]), n_items = static_cast<int>(buf[1][0]);
    if (t <= n_order) {
        queue1_part<true>(S, Q, order, n_order, tp, rf, lookahead, t, ns, ni);
        queue2_part(S, Q, order, n_order, tp, rf, n_items, n_segs1, t);
    }
    __syncthreads();

    // the filled part: counts, the per-expert prefixes (E + 1 entries), the segments
    if (t == 0) {
        T->n_items = S.n_items;
        T->n_items2 = S.n_items2;
        T->n_segs1 = S.n_segs1;
        T->n_segs = S.n_segs;
    }
    for (int e = t; e <= E; e += blockDim.x) {
        T->row_off[e] = S.row_off[e];
        T->pad_off[e] = S.pad_off[e];
        T->band_start[e] = S.band_start[e];
        T->sc_row[e] = S.sc_row[e];
        T->sc_col[e] = S.sc_col[e];
        if (pad_out) pad_out[e] = S.pad_off[e];
    }
    for (int i = t; i <= S.n_segs; i += blockDim.x) {
        T->seg_start[i] = S.seg_start[i];
        if (i < S.n_segs) {
            T->seg_info[i] = S.seg_info[i];
            T->seg_first[i] = S.seg_first[i];
        }
    }
}

// Failure-detection self-test: the library's bounded waits on something no
// one signals -- a workspace counter (which = 0, the dependency wait) or a
// fresh mbarrier (which = 1, the stage waits) -- so they run out, record
// their error code and return.
__global__ void gsa_selftest_kernel(uint32_t *ws, int which, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    if (which == 0) {
        wait_count(ws + WS_SELFTEST, 1u, ws, limit_ns);
    } else {
        const uint32_t b = smem_addr(&bar);
        mbar_init(b, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_wait_slow(b, 0u, ws, ERR_TIMEOUT_FULL, limit_ns);
    }
}

// Build the tables on the device (the plan kernel also clears the call's
// counters), then launch the fused kernel over the full persistent grid (CTAs
// without items leave at once).
gsa_status run_graph_safe(const Plan &pl, KParams &P, const int64_t *split_dev, int act, int recipe, bool bwd,
                          bool two_pass, const gsa_act_params *ap, void *ws, int64_t *pad_out, cudaStream_t stream) {
    launch_fn fn = pick(act);
    int per_sm = 0;
    if (fn(recipe, bwd, P, 0, stream, &per_sm) != cudaSuccess || per_sm <= 0) return GSA_ERR_CUDA;
    const int grid = per_sm * sm_count();
    if (grid <= 0) return GSA_ERR_CUDA;
    fill_common(pl, P, ap, ws);
    PlanTab *tab = reinterpret_cast<PlanTab *>(static_cast<uint8_t *>(ws) + plan_tab_offset(pl, recipe));
    P.dtab = tab;
    g_last_launches = 0;
    gsa_plan_kernel<<<1, kPlanThreads, 0, stream>>>(split_dev, pl.E, pl.M, pl.B, pl.n_slabs, pl.n_slabs2, two_pass ? 1 : 0,
                                                   ready_first_for(act, two_pass) ? 1 : 0, grid, tab,
                                                   static_cast<uint32_t *>(ws),
                                                   static_cast<int>(ws_counter_bytes(pl) / 4), pad_out);
    if (cudaGetLastError() != cudaSuccess) return GSA_ERR_CUDA;
    if (fn(recipe, bwd, P, grid, stream, &per_sm) != cudaSuccess) return GSA_ERR_CUDA;
    g_last_launches = 2;
    return GSA_OK;
}

// Scratch for gsa_fwd_noalloc: a fixed device array in this library's own
// image, so that the call needs no allocation.  Every device that loads the
// library holds it until the process exits.  Host code may not use the
// symbol as a device address; the address is looked up per device.
constexpr size_t kNoAllocScratchBytes = 64 * 1024;
static __device__ __align__(256) uint32_t g_noalloc_scratch[kNoAllocScratchBytes / 4];

struct NoAllocSetup {
    std::mutex mu;
    void *ptr[64] = {};
};
NoAllocSetup g_noalloc;

// Device address of the scratch array on the current device (looked up on
// the first call per device).  nullptr if the lookup fails.
void *noalloc_scratch_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(g_noalloc.mu);
    if (!g_noalloc.ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_noalloc.ptr[dev] = p;
    }
    return g_noalloc.ptr[dev];
}

// The recipe's RHT signs and scale layout into the kernel parameters.
gsa_status set_recipe(KParams &P, const gsa_recipe *recipe) {
    if (recipe->scale_layout != GSA_SCALES_COMPACT && recipe->scale_layout != GSA_SCALES_TILED)
        return GSA_ERR_INVALID_ARG;
    P.scale_tiled = recipe->scale_layout == GSA_SCALES_TILED ? 1 : 0;
    P.rht = (recipe->kind == GSA_NVFP4 && recipe->rht_colwise) ? 1 : 0;
    P.rht_mask = recipe->rht_sign_mask & 0xFFFFu;
    for (int i = 0; i < 16; ++i) {
        const bool flip = P.rht && ((P.rht_mask >> i) & 1u);
        P.rht_sgn[i] = flip ? 0x80008000u : 0u;
        P.rht_sgnlo[i] = flip ? 0x80000000u : 0u;
    }
    return GSA_OK;
}

// Argument checks and kernel parameters of a forward call; `need` is the
// workspace the call's plan requires.
gsa_status setup_fwd(const Plan &pl, const void *x_bf16, const float *probs, int32_t act_kind,
                     const gsa_act_params *act_params, const gsa_recipe *recipe, const gsa_qout *y_q, void *y_bf16_opt,
                     void *workspace, size_t workspace_bytes, size_t need, KParams &P, bool &two_pass) {
    gsa_status st;
    if ((st = check_act_params(act_kind, act_params)) != GSA_OK) return st;
    if (!has_row(y_q) && !has_col(y_q) && !y_bf16_opt) return GSA_ERR_INVALID_ARG;
    if (pl.M > 0 && !x_bf16) return GSA_ERR_INVALID_ARG;
    if ((st = check_qout(y_q, recipe->kind, true, true)) != GSA_OK) return st;
    if ((x_bf16 && !aligned16(x_bf16)) || (probs && !aligned4(probs)) || (y_bf16_opt && !aligned16(y_bf16_opt)))
        return GSA_ERR_ALIGNMENT;
    if (!workspace || workspace_bytes < need) return GSA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return GSA_ERR_ALIGNMENT;

    std::memset(&P, 0, sizeof(P));
    if (pl.M > 0 && !make_tmap(&P.tm_x, x_bf16, pl.M, pl.W_in)) return GSA_ERR_CUDA;
    P.probs = probs;
    P.y_bf16 = static_cast<uint16_t *>(y_bf16_opt);
    P.q[0] = to_dev(y_q);
    if ((st = set_recipe(P, recipe)) != GSA_OK) return st;
    two_pass = recipe->kind == GSA_NVFP4 && (has_row(y_q) || has_col(y_q));
    if (two_pass && pl.M > 0) P.stash = static_cast<uint8_t *>(workspace) + ws_counter_bytes(pl) + ws_partial_bytes(pl);
    return GSA_OK;
}

// Argument checks and kernel parameters of a backward call.
gsa_status setup_bwd(const Plan &pl, const void *dy_bf16, const void *x_bf16, const float *probs, int32_t act_kind,
                     const gsa_act_params *act_params, const gsa_recipe *recipe, void *dx_bf16_opt,
                     const gsa_qout *dx_q_opt, float *dprobs_opt, const gsa_qout *y_regen_col_opt, void *workspace,
                     size_t workspace_bytes, size_t need, KParams &P, bool &two_pass) {
    gsa_status st;
    if ((st = check_act_params(act_kind, act_params)) != GSA_OK) return st;
    const bool dxq = has_row(dx_q_opt) || has_col(dx_q_opt);
    const bool regen = has_col(y_regen_col_opt);
    if (!dx_bf16_opt && !dxq && !dprobs_opt && !regen) return GSA_ERR_INVALID_ARG;
    if (pl.M > 0 && (!x_bf16 || !dy_bf16)) return GSA_ERR_INVALID_ARG;
    if ((st = check_qout(dx_q_opt, recipe->kind, true, true)) != GSA_OK) return st;
    if ((st = check_qout(y_regen_col_opt, recipe->kind, false, false)) != GSA_OK) return st;
    if ((x_bf16 && !aligned16(x_bf16)) || (dy_bf16 && !aligned16(dy_bf16)) || (probs && !aligned4(probs)) ||
        (dx_bf16_opt && !aligned16(dx_bf16_opt)) || (dprobs_opt && !aligned4(dprobs_opt)))
        return GSA_ERR_ALIGNMENT;
    if (recipe->kind == GSA_NVFP4 && dxq && !dx_bf16_opt) return GSA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < need) return GSA_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return GSA_ERR_ALIGNMENT;

    std::memset(&P, 0, sizeof(P));
    two_pass = recipe->kind == GSA_NVFP4 && (dxq || regen);
    if (pl.M > 0) {
        if (!make_tmap(&P.tm_x, x_bf16, pl.M, pl.W_in)) return GSA_ERR_CUDA;
        if (!make_tmap(&P.tm_dy, dy_bf16, pl.M, pl.W)) return GSA_ERR_CUDA;
        if (two_pass && dx_bf16_opt && !make_tmap(&P.tm_dx, dx_bf16_opt, pl.M, pl.W_in)) return GSA_ERR_CUDA;
    }
    P.probs = probs;
    P.dx_bf16 = static_cast<uint16_t *>(dx_bf16_opt);
    P.dprobs = dprobs_opt;
    P.q[0] = to_dev(dx_q_opt);
    P.q[1] = to_dev(y_regen_col_opt);
    if ((st = set_recipe(P, recipe)) != GSA_OK) return st;
    return GSA_OK;
}

}  // namespace

extern "C" {

gsa_status gsa_layout(int64_t E, const int64_t *split_sizes, int64_t width, int32_t recipe_kind,
                      gsa_layout_info *out, int64_t *col_data_offsets, int64_t *col_scale_offsets) {
    if (E <= 0 || !split_sizes || width <= 0 || !out) return GSA_ERR_INVALID_ARG;
    if (recipe_kind != GSA_MXFP8 && recipe_kind != GSA_NVFP4) return GSA_ERR_INVALID_ARG;
    const int64_t B = recipe_kind == GSA_MXFP8 ? 32 : 16;
    if (width % B != 0) return GSA_ERR_INVALID_ARG;
    int64_t M = 0, Mp = 0;
    for (int64_t e = 0; e < E; ++e) {
        if (split_sizes[e] < 0) return GSA_ERR_INVALID_ARG;
        if (col_data_offsets) col_data_offsets[e] = recipe_kind == GSA_MXFP8 ? width * Mp : width * Mp / 2;
        if (col_scale_offsets) col_scale_offsets[e] = width * Mp / B;
        M += split_sizes[e];
        Mp += (split_sizes[e] + B - 1) / B * B;
    }
    if (col_data_offsets) col_data_offsets[E] = recipe_kind == GSA_MXFP8 ? width * Mp : width * Mp / 2;
    if (col_scale_offsets) col_scale_offsets[E] = width * Mp / B;
    out->rows = M;
    out->row_data_bytes = recipe_kind == GSA_MXFP8 ? M * width : M * width / 2;
    out->row_scale_bytes = M * width / B;
    out->col_data_bytes = recipe_kind == GSA_MXFP8 ? Mp * width : Mp * width / 2;
    out->col_scale_bytes = Mp * width / B;
    out->amax_floats = recipe_kind == GSA_NVFP4 ? E : 0;
    return GSA_OK;
}

gsa_status gsa_layout_ex(int64_t E, const int64_t *split_sizes, int64_t width, const gsa_recipe *recipe,
                         gsa_layout_info *out, int64_t *col_data_offsets, int64_t *col_scale_offsets,
                         int64_t *row_scale_offsets) {
    if (!recipe) return GSA_ERR_INVALID_ARG;
    if (recipe->scale_layout != GSA_SCALES_COMPACT && recipe->scale_layout != GSA_SCALES_TILED)
        return GSA_ERR_INVALID_ARG;
    const bool tiled = recipe->scale_layout == GSA_SCALES_TILED;
    gsa_status st = gsa_layout(E, split_sizes, width, recipe->kind, out, col_data_offsets, tiled ? nullptr : col_scale_offsets);
    if (st != GSA_OK) return st;
    const int64_t B = recipe->kind == GSA_MXFP8 ? 32 : 16;
    const int64_t c4 = (width / B + 3) / 4, rt = (width + 127) / 128;
    int64_t rows = 0, tr = 0, tc = 0;
    for (int64_t e = 0; e <= E; ++e) {
        if (row_scale_offsets) row_scale_offsets[e] = tiled ? tr * 512 * c4 : rows * (width / B);
        if (tiled && col_scale_offsets) col_scale_offsets[e] = tc * 512 * rt;
        if (e == E) break;
        rows += split_sizes[e];
        tr += (split_sizes[e] + 127) / 128;
        tc += (split_sizes[e] + 4 * B - 1) / (4 * B);
    }
    if (tiled) {
        out->row_scale_bytes = tr * 512 * c4;
        out->col_scale_bytes = tc * 512 * rt;
    }
    return GSA_OK;
}

size_t gsa_workspace_size(int64_t E, const int64_t *split_sizes, int64_t W_in, int32_t act_kind,
                          int32_t recipe_kind) {
    Plan pl;
    if (make_plan(E, split_sizes, W_in, act_kind, recipe_kind, pl, min_item_tile_cap(recipe_kind)) != GSA_OK) return 0;
    return ws_total_bytes(pl, recipe_kind);
}

gsa_status grouped_scaled_act_fwd(const void *x_bf16, const float *probs, const int64_t *split_sizes, int64_t E,
                                  int64_t W_in, int32_t act_kind, const gsa_act_params *act_params,
                                  const gsa_recipe *recipe, const gsa_qout *y_q, void *y_bf16_opt, void *workspace,
                                  size_t workspace_bytes, gsa_stream_t stream) {
    if (!recipe) return GSA_ERR_INVALID_ARG;
    Plan pl;
    gsa_status st = make_plan(E, split_sizes, W_in, act_kind, recipe->kind, pl, item_tile_cap(act_kind, recipe->kind, false, fwd_two_pass(recipe->kind, y_q)));
    if (st != GSA_OK) return st;
    fit_items_to_grid(pl, pl.n_bands, act_kind, recipe->kind, false);
    KParams P;
    bool two_pass = false;
    st = setup_fwd(pl, x_bf16, probs, act_kind, act_params, recipe, y_q, y_bf16_opt, workspace, workspace_bytes,
                   ws_total_bytes(pl, recipe->kind), P, two_pass);
    if (st != GSA_OK) return st;
    return run(pl, P, act_kind, recipe->kind, false, two_pass, act_params, workspace,
               reinterpret_cast<cudaStream_t>(stream));
}

gsa_status grouped_scaled_act_bwd(const void *dy_bf16, const void *x_bf16, const float *probs,
                                  const int64_t *split_sizes, int64_t E, int64_t W_in, int32_t act_kind,
                                  const gsa_act_params *act_params, const gsa_recipe *recipe, void *dx_bf16_opt,
                                  const gsa_qout *dx_q_opt, float *dprobs_opt, const gsa_qout *y_regen_col_opt,
                                  void *workspace, size_t workspace_bytes, gsa_stream_t stream) {
    if (!recipe) return GSA_ERR_INVALID_ARG;
    Plan pl;
    gsa_status st = make_plan(E, split_sizes, W_in, act_kind, recipe->kind, pl, item_tile_cap(act_kind, recipe->kind, true, bwd_two_pass(recipe->kind, dx_q_opt, y_regen_col_opt)));
    if (st != GSA_OK) return st;
    fit_items_to_grid(pl, pl.n_bands, act_kind, recipe->kind, true);
    KParams P;
    bool two_pass = false;
    st = setup_bwd(pl, dy_bf16, x_bf16, probs, act_kind, act_params, recipe, dx_bf16_opt, dx_q_opt, dprobs_opt,
                   y_regen_col_opt, workspace, workspace_bytes, ws_total_bytes(pl, recipe->kind), P, two_pass);
    if (st != GSA_OK) return st;
    return run(pl, P, act_kind, recipe->kind, true, two_pass, act_params, workspace,
               reinterpret_cast<cudaStream_t>(stream));
}

gsa_status gsa_layout_bound(int64_t E, int64_t M, int64_t width, int32_t recipe_kind, gsa_layout_info *out) {
    if (E <= 0 || M < 0 || width <= 0 || !out) return GSA_ERR_INVALID_ARG;
    if (recipe_kind != GSA_MXFP8 && recipe_kind != GSA_NVFP4) return GSA_ERR_INVALID_ARG;
    const int64_t B = recipe_kind == GSA_MXFP8 ? 32 : 16;
    if (width % B != 0) return GSA_ERR_INVALID_ARG;
    const int64_t Mp = (M + E * (B - 1)) / B * B;   // sum over experts of ceil(M_e / B) B is at most this
    out->rows = M;
    out->row_data_bytes = recipe_kind == GSA_MXFP8 ? M * width : M * width / 2;
    out->row_scale_bytes = M * width / B;
    out->col_data_bytes = recipe_kind == GSA_MXFP8 ? Mp * width : Mp * width / 2;
    out->col_scale_bytes = Mp * width / B;
    out->amax_floats = recipe_kind == GSA_NVFP4 ? E : 0;
    return GSA_OK;
}

gsa_status gsa_layout_bound_ex(int64_t E, int64_t M, int64_t width, const gsa_recipe *recipe, gsa_layout_info *out) {
    if (!recipe) return GSA_ERR_INVALID_ARG;
    if (recipe->scale_layout != GSA_SCALES_COMPACT && recipe->scale_layout != GSA_SCALES_TILED)
        return GSA_ERR_INVALID_ARG;
    gsa_status st = gsa_layout_bound(E, M, width, recipe->kind, out);
    if (st != GSA_OK || recipe->scale_layout == GSA_SCALES_COMPACT) return st;
    const int64_t B = recipe->kind == GSA_MXFP8 ? 32 : 16;
    out->row_scale_bytes = (M + 127 * E) / 128 * 512 * ((width / B + 3) / 4);
    out->col_scale_bytes = (M + (4 * B - 1) * E) / (4 * B) * 512 * ((width + 127) / 128);
    return GSA_OK;
}

size_t gsa_workspace_size_graph_safe(int64_t E, int64_t M, int64_t W_in, int32_t act_kind, int32_t recipe_kind) {
    Plan pl;
    if (make_plan_bound(E, M, W_in, act_kind, recipe_kind, pl, min_item_tile_cap(recipe_kind)) != GSA_OK) return 0;
    return ws_graph_safe_bytes(pl, recipe_kind);
}

gsa_status grouped_scaled_act_fwd_graph_safe(const void *x_bf16, const float *probs, const int64_t *split_sizes_dev,
                                             int64_t E, int64_t M, int64_t W_in, int32_t act_kind,
                                             const gsa_act_params *act_params, const gsa_recipe *recipe,
                                             const gsa_qout *y_q, void *y_bf16_opt, int64_t *padded_row_offsets_opt,
                                             void *workspace, size_t workspace_bytes, gsa_stream_t stream) {
    if (!recipe || !split_sizes_dev) return GSA_ERR_INVALID_ARG;
    if (padded_row_offsets_opt && (reinterpret_cast<uintptr_t>(padded_row_offsets_opt) & 7u)) return GSA_ERR_ALIGNMENT;
    if (reinterpret_cast<uintptr_t>(split_sizes_dev) & 7u) return GSA_ERR_ALIGNMENT;
    Plan pl;
    gsa_status st = make_plan_bound(E, M, W_in, act_kind, recipe->kind, pl, item_tile_cap(act_kind, recipe->kind, false, fwd_two_pass(recipe->kind, y_q)));
    if (st != GSA_OK) return st;
    fit_items_to_grid(pl, (M + kRows - 1) / kRows, act_kind, recipe->kind, false);   // the fewest bands of M rows
    KParams P;
    bool two_pass = false;
    st = setup_fwd(pl, x_bf16, probs, act_kind, act_params, recipe, y_q, y_bf16_opt, workspace, workspace_bytes,
                   ws_graph_safe_bytes(pl, recipe->kind), P, two_pass);
    if (st != GSA_OK) return st;
    return run_graph_safe(pl, P, split_sizes_dev, act_kind, recipe->kind, false, two_pass, act_params, workspace,
                          padded_row_offsets_opt, reinterpret_cast<cudaStream_t>(stream));
}

gsa_status grouped_scaled_act_bwd_graph_safe(const void *dy_bf16, const void *x_bf16, const float *probs,
                                             const int64_t *split_sizes_dev, int64_t E, int64_t M, int64_t W_in,
                                             int32_t act_kind, const gsa_act_params *act_params,
                                             const gsa_recipe *recipe, void *dx_bf16_opt, const gsa_qout *dx_q_opt,
                                             float *dprobs_opt, const gsa_qout *y_regen_col_opt,
                                             int64_t *padded_row_offsets_opt, void *workspace, size_t workspace_bytes,
                                             gsa_stream_t stream) {
    if (!recipe || !split_sizes_dev) return GSA_ERR_INVALID_ARG;
    if (padded_row_offsets_opt && (reinterpret_cast<uintptr_t>(padded_row_offsets_opt) & 7u)) return GSA_ERR_ALIGNMENT;
    if (reinterpret_cast<uintptr_t>(split_sizes_dev) & 7u) return GSA_ERR_ALIGNMENT;
    Plan pl;
    gsa_status st = make_plan_bound(E, M, W_in, act_kind, recipe->kind, pl, item_tile_cap(act_kind, recipe->kind, true, bwd_two_pass(recipe->kind, dx_q_opt, y_regen_col_opt)));
    if (st != GSA_OK) return st;
    fit_items_to_grid(pl, (M + kRows - 1) / kRows, act_kind, recipe->kind, true);   // the fewest bands of M rows
    KParams P;
    bool two_pass = false;
    st = setup_bwd(pl, dy_bf16, x_bf16, probs, act_kind, act_params, recipe, dx_bf16_opt, dx_q_opt, dprobs_opt,
                   y_regen_col_opt, workspace, workspace_bytes, ws_graph_safe_bytes(pl, recipe->kind), P, two_pass);
    if (st != GSA_OK) return st;
    return run_graph_safe(pl, P, split_sizes_dev, act_kind, recipe->kind, true, two_pass, act_params, workspace,
                          padded_row_offsets_opt, reinterpret_cast<cudaStream_t>(stream));
}

gsa_status gsa_selftest_wait_timeout(void *workspace, int32_t which, uint32_t limit_ms, gsa_stream_t stream) {
    if (!workspace || (which != 0 && which != 1) || limit_ms == 0 || limit_ms > 2000) return GSA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return GSA_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    g_last_launches = 0;
    if (cudaMemsetAsync(workspace, 0, WS_HDR * sizeof(uint32_t), s) != cudaSuccess) return GSA_ERR_CUDA;
    gsa_selftest_kernel<<<1, 32, 0, s>>>(static_cast<uint32_t *>(workspace), which,
                                         static_cast<uint64_t>(limit_ms) * 1000000ull);
    if (cudaGetLastError() != cudaSuccess) return GSA_ERR_CUDA;
    g_last_launches = 1;
    return GSA_OK;
}

gsa_status gsa_workspace_status(const void *workspace, gsa_stream_t stream) {
    if (!workspace) return GSA_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return GSA_ERR_CUDA;
    uint32_t err = 0;
    if (cudaMemcpy(&err, static_cast<const uint32_t *>(workspace) + WS_ERR, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        return GSA_ERR_CUDA;
    if (err & ERR_BAD_SPLIT) return GSA_ERR_INVALID_ARG;
    return err ? GSA_ERR_DEVICE_TIMEOUT : GSA_OK;
}

int32_t gsa_last_launch_count(void) { return g_last_launches; }

const char *gsa_status_string(gsa_status s) {
    switch (s) {
    case GSA_OK: return "ok";
    case GSA_ERR_INVALID_ARG: return "invalid argument";
    case GSA_ERR_UNSUPPORTED: return "unsupported shape or option";
    case GSA_ERR_ALIGNMENT: return "pointer not aligned";
    case GSA_ERR_WORKSPACE: return "workspace missing or too small";
    case GSA_ERR_CUDA: return "CUDA call failed";
    case GSA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

int32_t gsa_version(void) { return (1 << 16) | 1; }

gsa_status gsa_fwd_noalloc(const void *x_bf16, const float *probs, const int64_t *split_sizes, int64_t E,
                           int64_t W_in, int32_t act_kind, const gsa_act_params *act_params,
                           const gsa_recipe *recipe, const gsa_qout *y_q, void *y_bf16_opt, gsa_stream_t stream) {
    if (!recipe) return GSA_ERR_INVALID_ARG;
    Plan pl;
    gsa_status st = make_plan(E, split_sizes, W_in, act_kind, recipe->kind, pl, item_tile_cap(act_kind, recipe->kind, false, fwd_two_pass(recipe->kind, y_q)));
    if (st != GSA_OK) return st;
    if ((st = check_act_params(act_kind, act_params)) != GSA_OK) return st;
    if (!has_row(y_q) && !has_col(y_q) && !y_bf16_opt) return GSA_ERR_INVALID_ARG;
    if (pl.M > 0 && !x_bf16) return GSA_ERR_INVALID_ARG;
    if ((st = check_qout(y_q, recipe->kind, true, true)) != GSA_OK) return st;
    if ((x_bf16 && !aligned16(x_bf16)) || (probs && !aligned4(probs)) || (y_bf16_opt && !aligned16(y_bf16_opt)))
        return GSA_ERR_ALIGNMENT;
    // the forward uses only the counter part of the workspace
    if (ws_counter_bytes(pl) > kNoAllocScratchBytes) return GSA_ERR_WORKSPACE;
    void *scratch = noalloc_scratch_ptr();
    if (!scratch) return GSA_ERR_CUDA;

    KParams P;
    std::memset(&P, 0, sizeof(P));
    if (pl.M > 0 && !make_tmap(&P.tm_x, x_bf16, pl.M, pl.W_in)) return GSA_ERR_CUDA;
    P.probs = probs;
    P.y_bf16 = static_cast<uint16_t *>(y_bf16_opt);
    P.q[0] = to_dev(y_q);
    if ((st = set_recipe(P, recipe)) != GSA_OK) return st;
    const bool two_pass = recipe->kind == GSA_NVFP4 && (has_row(y_q) || has_col(y_q));
    return run(pl, P, act_kind, recipe->kind, false, two_pass, act_params, scratch,
               reinterpret_cast<cudaStream_t>(stream));
}

gsa_status gsa_fwd_noalloc_status(gsa_stream_t stream) {
    uint32_t *scratch = static_cast<uint32_t *>(noalloc_scratch_ptr());
    if (!scratch) return GSA_ERR_CUDA;
    return gsa_workspace_status(scratch, stream);
}

}  // extern "C"
