// gsa_kernel.cuh -- the fused grouped scaled activation + block-scaled
// quantization kernel for sm_103a (forward and backward, MXFP8 and NVFP4).
//
// What it computes ("Activation + GroupedLinear Fusion for MOE", Greptile
// Summary: per-row scale x activation x grouped quantization in one kernel
// dispatch, forward and backward; "Enable fused activation recompute for
// ScaledTanhSReLU", Description: backward regenerates FC2's input from the
// saved FC1 output, MXFP8 and NVFP4-with-RHT recipes):
//   forward : Y = bf16(p * act(X)); Y rowwise + columnwise quantized.
//   backward: dX = bf16(dY * p * act'(X)); dprobs = sum_j dY * act(X);
//             dX rowwise + columnwise quantized; optionally Y's columnwise
//             copy regenerated bit-for-bit.
//
// Activations: SReLU, TanhSReLU, SwiGLU, clamped SwiGLU, and the further
// unary GeLU, sigmoid and identity (the recompute page's review thread: the
// kernel is not specific to the SReLU family).
//
// Structure (one persistent launch per call):
//   * Work item = (band of 128 rows inside one expert) x (slab of up to 8
//     tiles of 64 columns).  Items are handed out from work queues built by
//     build_queues (segments of items per expert), on the host from a host
//     split or by the plan kernel from a device split (graph-safe calls).
//   * NVFP4 needs each expert's tensor amax before any of its blocks can be
//     encoded.  Items therefore come in two kinds: P1 (amax only) and P2
//     (encode).  Queue 1 (atomic ticket) holds the P1 items; the P2 items of
//     an expert either follow in queue 1 after a lookahead of further P1
//     items, their producer waiting (bounded) for the expert's P1 count, or
//     sit in queue 2, taken only once the expert's amax pass is complete.
//     Tickets are taken in order, so the holder of any earlier ticket is
//     already running: no wait can deadlock.  The encode pass of the forward
//     reads Y back from a staging image that the amax pass wrote (meant to
//     hit L2).
//   * Warp 8 is the producer: it takes tickets and streams 128 x 64 BF16
//     tiles into a ring of shared-memory stages with TMA (128-byte swizzle),
//     signalling full/empty mbarriers.  Warps 0-7 consume each tile in two
//     steps: (A) thread = (row, 32-column half): activation, rowwise blocks,
//     dense stores, in-place write-back of the values to quantize; (B) warp =
//     row block, lane = column pair: columnwise blocks (NVFP4: the 16-point
//     RHT in registers, two columns per packed-FP32 op) and transposed stores.
//   * dprobs: each thread sums its 32-column block serially, pairs of blocks
//     combine through a shuffle, tiles merge through a binary-counter stack,
//     and slabs merge in the last-arriving item of the band (a counter per
//     band, no waiting).
//
// All floating-point arithmetic is IEEE binary32 with round-to-nearest-even
// and no contraction (the translation unit is compiled with -fmad=false).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gsa {

enum { ACT_SRELU = 0, ACT_TANH_SRELU = 1, ACT_SWIGLU = 2, ACT_CLAMPED_SWIGLU = 3, ACT_GELU = 4, ACT_SIGMOID = 5,
       ACT_IDENTITY = 6 };
enum { MXFP8 = 0, NVFP4 = 1 };
enum { K_SINGLE = 0, K_P1 = 1, K_P2 = 2, K_END = 3 };

constexpr int kMaxExperts = 256;
constexpr int kMaxSlabs = 64;
constexpr int kMaxItemTiles = 32;         // tiles of one item (a power of two)
constexpr int kStackLevels = 6;            // log2(kMaxItemTiles) + 1 levels of the dprobs binary counter
constexpr int kMaxSegs = 4 * kMaxExperts;
constexpr int kRows = 128;                 // rows per band
constexpr int kCols = 64;                  // Y columns per tile
constexpr int kCons = 256;                 // consumer threads (warps 0-7)
constexpr int kThreads = kCons + 32;       // + producer warp
constexpr int kSlotBytes = kRows * kCols * 2;

// Workspace layout, in 32-bit words.
constexpr int WS_TICKET = 0;                 // next item of queue 1 (amax-pass or single-pass items)
constexpr int WS_ERR = 1;
constexpr int WS_ERRINFO = 2;
constexpr int WS_SELFTEST = 3;               // a word nothing signals (the wait self-test)
constexpr int WS_HDR = 64;                 // done[E], amax[3E], taken2[E], band_cnt[n_bands] follow
constexpr uint32_t ERR_TIMEOUT_FULL = 1u, ERR_TIMEOUT_EMPTY = 2u, ERR_TIMEOUT_DEP = 4u;
constexpr uint32_t ERR_BAD_SPLIT = 8u;     // graph-safe call: the device split was negative or did not sum to M

struct QDev {
    uint8_t *row_data;
    uint8_t *row_scale;
    uint8_t *col_data;
    uint8_t *col_scale;
    float *amax_row;
    float *amax_col;
};

// Byte offset of entry (r, c) of a scale matrix in the tiled layout of the
// block-scaled GEMM operands: 512-byte tiles of 128 rows x 4 columns, tiles in
// row-major order with c4 tiles per tile row; inside a tile, row r at
// 16 (r mod 32) + 4 floor((r mod 128) / 32) and column c at + (c mod 4).
__host__ __device__ inline int64_t tiled_scale_off(int64_t r, int64_t c, int64_t c4) {
    return ((r >> 7) * c4 + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}

// Schedule and expert tables of one call: built on the host from a host
// split (passed inside the kernel parameters), or on the device by the plan
// kernel from a device split (graph-safe calls; read through a pointer).
struct PlanTab {
    int n_items, n_items2;              // items of queue 1 (P1 / single pass) and queue 2 (P2)
    int n_segs1, n_segs;                // segments [0, n_segs1) list queue 1, [n_segs1, n_segs) queue 2
    int64_t row_off[kMaxExperts + 1];
    int64_t pad_off[kMaxExperts + 1];   // prefix of Mp_e (rows padded to the block)
    int band_start[kMaxExperts + 1];
    int seg_start[kMaxSegs + 1];        // first item of the segment within its queue
    int seg_info[kMaxSegs];             // (kind << 16) | expert
    int seg_first[kMaxSegs];            // first item of the segment inside the expert's items
    // tiled scale layout: prefixes over the experts of ceil(M_e / 128) (128-row tiles of the
    // rowwise scales) and of ceil(M_e / (4 B)) (4-column tile groups of the columnwise scales)
    int sc_row[kMaxExperts + 1];
    int sc_col[kMaxExperts + 1];
};

struct KParams {
    CUtensorMap tm_x;       // X  [M, W_in] BF16, box 64 x 128, 128B swizzle
    CUtensorMap tm_dy;      // dY [M, W]
    CUtensorMap tm_dx;      // dX [M, W_in] (NVFP4 backward encode pass)
    const float *probs;
    uint16_t *y_bf16;
    uint16_t *dx_bf16;
    uint8_t *stash;         // NVFP4 forward: BF16 Y of each (band, tile), 128 rows x 128 bytes, written by
                            // the amax pass and read back by the encode pass
    float *dprobs;
    QDev q[2];              // [0] Y (fwd) or dX (bwd); [1] regenerated Y columnwise (bwd)
    uint32_t *ws;
    float *partial;         // [M, n_slabs] dprobs slab partials
    int M, W, W_in, E;
    int n_slabs, tiles_per_slab;   // single-pass and amax items: slabs per band, tiles per slab
    float s, s2, two_s, limit, alpha, off, inv_s;
    int s_pow2;
    uint32_t rht_mask;
    int rht;
    uint32_t rht_sgn[16];   // row i of a 16-row block: 0x80008000 where the RHT flips its sign, else 0
    uint32_t rht_sgnlo[16]; // the same sign as 0x80000000 (added to the low half moved up 16 bits)
    const PlanTab *dtab;    // device-built tables (graph-safe calls), else nullptr and `tab` holds them
    PlanTab tab;
    // last, so the fields above keep their offsets (moving the RHT sign arrays off their
    // 8-byte alignment changed the kernels' register allocation and cost 1-2 %)
    int scale_tiled;        // the scale layout, for the launcher (the kernels take it as TILED)
    int n_slabs2, tiles_per_slab2;   // encode (P2) items: slabs per band and tiles per slab
};

__device__ __forceinline__ const PlanTab &plan_of(const KParams &P) { return P.dtab ? *P.dtab : P.tab; }


// Work queues from the order of the non-empty experts (two-pass: by
// decreasing size).  Queue 1: the single-pass items of the experts in order,
// or the amax items (P1).  The encode items (P2) of expert e need its complete
// amax:
//  * ready-first (queue 2, one segment per expert in the same order): the
//    kernel takes an expert's encode items as soon as its amax items are all
//    done, before further amax items -- best when the amax pass is the costly
//    part (a transcendental activation), as no CTA then waits;
//  * static interleave (ready_first false): the encode items of e follow in
//    queue 1 once `lookahead` further amax items have been queued after e's
//    last one, keeping DRAM-heavy amax items and compute-heavy encode items
//    mixed and the staging data's stay in L2 short.
// An expert has (its bands) x n_slabs single-pass or amax items and (its
// bands) x n_slabs2 encode items; the lookahead counts amax items.
// T.band_start must be filled.  pend_e / pend_pos: scratch of n_order ints.
// The same function builds the tables on the host and in the plan kernel.
__host__ __device__ inline void build_queues(PlanTab &T, const int *order, int n_order, int n_slabs, int n_slabs2,
                                             bool two_pass, bool ready_first, int lookahead, int *pend_e,
                                             int *pend_pos) {
    int nseg = 0, start = 0;
    auto items_of = [&](int e) { return (T.band_start[e + 1] - T.band_start[e]) * n_slabs; };
    auto items2_of = [&](int e) { return (T.band_start[e + 1] - T.band_start[e]) * n_slabs2; };
    auto add = [&](int kind, int e, int first, int count) {
        if (count <= 0) return;
        T.seg_start[nseg] = start;
        T.seg_info[nseg] = (kind << 16) | e;
        T.seg_first[nseg] = first;
        start += count;
        ++nseg;
    };
    if (!two_pass) {
        for (int i = 0; i < n_order; ++i) add(K_SINGLE, order[i], 0, items_of(order[i]));
    } else if (ready_first) {
        for (int i = 0; i < n_order; ++i) add(K_P1, order[i], 0, items_of(order[i]));
    } else {
        int n_pend = 0, head = 0, p1_done = 0;
        for (int i = 0; i < n_order; ++i) {
            const int e = order[i];
            int first = 0, n = items_of(e);
            while (n > 0) {
                int take = n;
                if (head < n_pend) take = min(take, max(0, pend_pos[head] - p1_done));
                add(K_P1, e, first, take);
                first += take;
                n -= take;
                p1_done += take;
                while (head < n_pend && pend_pos[head] <= p1_done) {
                    add(K_P2, pend_e[head], 0, items2_of(pend_e[head]));
                    ++head;
                }
            }
            pend_e[n_pend] = e;
            pend_pos[n_pend] = p1_done + lookahead;
            ++n_pend;
        }
        for (; head < n_pend; ++head) add(K_P2, pend_e[head], 0, items2_of(pend_e[head]));
    }
    T.n_items = start;
    T.n_segs1 = nseg;
    start = 0;
    if (two_pass && ready_first)
        for (int i = 0; i < n_order; ++i) add(K_P2, order[i], 0, items2_of(order[i]));
    T.n_items2 = start;
    T.seg_start[nseg] = start;
    T.n_segs = nseg;
}

// The same queues built in parallel (the graph-safe plan kernel): one thread
// per position t of the order, position n_order the tail.  Between the steps
// the caller forms exclusive prefix sums over t = 0 .. n_order:
//   1. queue_counts: the items of position t (amax / single-pass, encode) ->
//      QueueScan::c, c2 (c[n_order], c2[n_order]: the totals);
//   2. queue1_part<false>: the queue-1 segments and items thread t adds ->
//      QueueScan::so, io;
//   3. queue1_part<true> and queue2_part write them.
// Static interleave: the encode items of position j go in at queue-1 amax
// position q_j = c[j + 1] + lookahead (the end when past it), the serial
// builder's pend_pos; q is increasing, so the insertion points inside the
// amax run [c[t], c[t + 1]) of position t are a range of j found by binary
// search, and thread t adds that run's chunks and those encode segments in
// the serial order.  Thread n_order adds the encode segments at or past the
// last amax item.
struct QueueScan {
    int c[kMaxExperts + 1];    // amax / single-pass items before position t
    int c2[kMaxExperts + 1];   // encode items before position t
    int so[kMaxExperts + 1];   // queue-1 segments before thread t's
    int io[kMaxExperts + 1];   // queue-1 items before thread t's
};

__host__ __device__ inline void queue_counts(const PlanTab &T, const int *order, int n_order, int n_slabs, int n_slabs2,
                                             int t, int &items, int &items2) {
    items = items2 = 0;
    if (t < n_order) {
        const int nb = T.band_start[order[t] + 1] - T.band_start[order[t]];
        items = nb * n_slabs;
        items2 = nb * n_slabs2;
    }
}

// First j in [0, n) with c[j + 1] + lookahead >= v (n when none).
__host__ __device__ inline int first_insert_at_or_after(const QueueScan &Q, int n, int lookahead, int v) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (Q.c[mid + 1] + lookahead >= v) hi = mid;
        else lo = mid + 1;
    }
    return lo;
}

template <bool EMIT>
__host__ __device__ inline void queue1_part(PlanTab &T, const QueueScan &Q, const int *order, int n_order, bool two_pass,
                                            bool ready_first, int lookahead, int t, int &segs, int &items) {
    segs = items = 0;
    int s = 0, at = 0;
    if constexpr (EMIT) {
        s = Q.so[t];
        at = Q.io[t];
    }
    auto put = [&](int kind, int e, int first, int count) {
        if constexpr (EMIT) {
            T.seg_start[s] = at;
            T.seg_info[s] = (kind << 16) | e;
            T.seg_first[s] = first;
        }
        ++s;
        at += count;
        ++segs;
        items += count;
    };
    if (!two_pass || ready_first) {
        if (t < n_order) put(two_pass ? K_P1 : K_SINGLE, order[t], 0, Q.c[t + 1] - Q.c[t]);
        return;
    }
    const int a = Q.c[t];
    const int j0 = first_insert_at_or_after(Q, n_order, lookahead, a);
    const int j1 = t < n_order ? first_insert_at_or_after(Q, n_order, lookahead, Q.c[t + 1]) : n_order;
    int cur = a;
    for (int j = j0; j < j1; ++j) {
        const int q = Q.c[j + 1] + lookahead;
        if (t < n_order && q > cur) {
            put(K_P1, order[t], cur - a, q - cur);
            cur = q;
        }
        put(K_P2, order[j], 0, Q.c2[j + 1] - Q.c2[j]);
    }
    if (t < n_order) put(K_P1, order[t], cur - a, Q.c[t + 1] - cur);
}

// Queue 2 (ready-first: one encode segment per position, after queue 1's
// n_segs1 segments) and the counts; thread t < n_order writes its segment,
// thread n_order the counts and the end marker.
__host__ __device__ inline void queue2_part(PlanTab &T, const QueueScan &Q, const int *order, int n_order, bool two_pass,
                                            bool ready_first, int n_items, int n_segs1, int t) {
    const bool q2 = two_pass && ready_first;
    if (q2 && t < n_order) {
        T.seg_start[n_segs1 + t] = Q.c2[t];
        T.seg_info[n_segs1 + t] = (K_P2 << 16) | order[t];
        T.seg_first[n_segs1 + t] = 0;
    }
    if (t == n_order) {
        T.n_items = n_items;
        T.n_segs1 = n_segs1;
        T.n_items2 = q2 ? Q.c2[n_order] : 0;
        T.n_segs = n_segs1 + (q2 ? n_order : 0);
        T.seg_start[T.n_segs] = T.n_items2;
    }
}

// Per-stage tile descriptor written by the producer warp next to the TMA
// data: item, expert constants and (P2) the expert's amax values.
struct TileHdr {
    int kind, e, row0, nrows;
    int col0, tile, slab, gband;
    float amax[3];
    int lr0;            // band's first row inside the expert
    int Me, Mp;         // expert rows, padded to the block
    int pad_off;        // padded rows of the experts before e
    int pnn;            // every p of the band is >= 0 (so p * act keeps one sign for a non-negative act)
};
static_assert(sizeof(TileHdr) == 64, "tile header is 64 bytes");

// Scale byte of scale column c (block size B) of row lr of expert e in a
// rowwise copy of width `width`; grow is the row's index in the whole tensor.
// Compact: [M, width / B] row-major.  Tiled: expert e's [M_e, width / B]
// matrix in 128 x 4 tiles, the experts' tile blocks one after another.
template <int B, bool TILED>
__device__ __forceinline__ uint8_t *row_scale_ptr(const KParams &P, uint8_t *base, int e, int64_t grow, int64_t lr,
                                                  int c, int width) {
    if constexpr (!TILED) {
        return base + grow * (width / B) + c;
    } else {
        const int64_t c4 = (width / B + 3) >> 2;
        return base + static_cast<int64_t>(plan_of(P).sc_row[e]) * 512 * c4 + tiled_scale_off(lr, c, c4);
    }
}

// Scale byte of block `blk` (rows B blk .. B blk + B - 1 of expert e) of column
// `col` in a columnwise copy of width `width`.  Compact: per expert
// [width, Mp_e / B] row-major after the experts before it.  Tiled: expert e's
// [width, Mp_e / B] matrix in 128 x 4 tiles, the experts' tile blocks one after
// another.
template <int B, bool TILED>
__device__ __forceinline__ uint8_t *col_scale_ptr(const KParams &P, uint8_t *base, const TileHdr &hd, int64_t col,
                                                  int blk, int width) {
    if constexpr (!TILED) {
        return base + static_cast<int64_t>(width) * (hd.pad_off / B) + col * (hd.Mp / B) + blk;
    } else {
        const int64_t c4 = (hd.Mp / B + 3) >> 2;
        return base + static_cast<int64_t>(plan_of(P).sc_col[hd.e]) * 512 * ((width + 127) >> 7) +
               tiled_scale_off(col, blk, c4);
    }
}
// Per-stage area: header (64 B), encode scales S[3] at 64, p of the band
// (128 floats) at 128, and for NVFP4 the multiplier tables rtab[3][128] at 640.
constexpr int kMetaS = 64;
constexpr int kMetaP = 128;
constexpr int kMetaT = 640;
constexpr int kMetaBytesMX = 640;
constexpr int kMetaBytesNV = 640 + 3 * 128 * 4;

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// One wait attempt; the thread may be suspended up to ~1 ms inside it until
// the phase completes, so a waiting warp issues almost nothing.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, 1000000;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: gives up after ~2 s of wall time, records `code` in the
// workspace error word and returns false.
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;

static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, uint32_t *ws, uint32_t code,
                                                   uint64_t limit_ns = kWaitLimitNs) {
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) {
            atomicOr(ws + WS_ERR, code);
            return false;
        }
    }
}

// Same, for a waiter that is not latency-critical (the producer waiting for a
// free stage): polls with a short sleep in between, leaving issue slots to the
// consumer warps.
static __device__ __noinline__ bool mbar_wait_backoff(uint32_t bar, uint32_t parity, uint32_t *ws, uint32_t code) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        __nanosleep(100);
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > kWaitLimitNs) {
            atomicOr(ws + WS_ERR, code);
            return false;
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t *ws, uint32_t code) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, ws, code);
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Plain bulk copy global -> shared (both 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap *tm, int c, int r, uint32_t bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(tm), "r"(c), "r"(r), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void named_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kCons) : "memory");
}

// Barrier of the two consumer warps 2k and 2k+1 (ids 2..5).
__device__ __forceinline__ void pair_sync(int k) {
    asm volatile("bar.sync %0, 64;" ::"r"(2 + k) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Bounded wait for a counter in global memory to reach `target` (acquire
// order): polls with a short sleep, gives up after limit_ns or once another
// wait of the call has failed, records ERR_TIMEOUT_DEP and returns false.
__device__ __forceinline__ bool wait_count(const uint32_t *cnt, uint32_t target, uint32_t *ws,
                                           uint64_t limit_ns = kWaitLimitNs) {
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0;; ++i) {
        __nanosleep(64);
        if (ld_acquire_gpu(cnt) >= target) return true;
        if ((i & 63u) == 63u && (global_ns() - t0 > limit_ns || ld_relaxed_gpu(ws + WS_ERR))) {
            atomicOr(ws + WS_ERR, ERR_TIMEOUT_DEP);
            return false;
        }
    }
}

// Shared-memory tile: 128 rows x 128 bytes, 16-byte chunk c of row r stored
// at chunk position c ^ (r & 7) (the TMA 128-byte swizzle).
__device__ __forceinline__ uint32_t swz_chunk(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t swz_word(int r, int word) {  // word = 32-bit column pair 0..31
    return swz_chunk(r, word >> 2) + ((word & 3) << 2);
}

// Plain typed accesses (not inline asm), so the compiler can overlap the loads
// of one chunk with the arithmetic and stores of the previous one.
__device__ __forceinline__ uint4 lds128(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }

__device__ __forceinline__ void sts128(uint8_t *p, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(x, y, z, w);
}

__device__ __forceinline__ uint32_t lds32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }

// Streaming stores (evict-first) for outputs nothing in the call reads back.
__device__ __forceinline__ void stg128(void *p, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    __stcs(reinterpret_cast<uint4 *>(p), make_uint4(x, y, z, w));
}

__device__ __forceinline__ void stg64(void *p, uint32_t x, uint32_t y) {
    __stcs(reinterpret_cast<uint2 *>(p), make_uint2(x, y));
}

// Plain (write-back) stores for data the encode pass reads back from L2.
__device__ __forceinline__ void stg32(void *p, uint32_t x) { *reinterpret_cast<uint32_t *>(p) = x; }

__device__ __forceinline__ void stg128_wb(void *p, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
    *reinterpret_cast<uint4 *>(p) = make_uint4(x, y, z, w);
}

// --------------------------------------------------------- number formats

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// a - b on both lanes of a packed FP32 pair, each rounded to nearest even.
__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
    float2 r;
    asm("{\n .reg .b64 ra, rb, rr;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
        " sub.rn.f32x2 rr, ra, rb;\n mov.b64 {%0, %1}, rr;\n}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {  // per-half max of BF16 pairs
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Per-half sum of BF16 pairs, rounded to nearest even.
__device__ __forceinline__ uint32_t badd2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Per-half max of |a|, |b| (the sign bit of the result is the xor of the
// operands' signs and is masked off by the caller).
__device__ __forceinline__ uint32_t babsmax2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Four floats -> four E4M3 bytes (v0 in the lowest byte), RNE, satfinite.
__device__ __forceinline__ uint32_t e4m3x4(float v0, float v1, float v2, float v3) {
    uint32_t out;
    asm("{\n .reg .b16 lo, hi;\n"
        " cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n"
        " cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n"
        " mov.b32 %0, {lo, hi};\n}"
        : "=r"(out)
        : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
    return out;
}

__device__ __forceinline__ uint32_t e4m3_byte(float v) {
    uint32_t out;
    asm("{\n .reg .b16 t;\n cvt.rn.satfinite.e4m3x2.f32 t, 0f00000000, %1;\n cvt.u32.u16 %0, t;\n}"
        : "=r"(out)
        : "f"(v));
    return out & 0xFFu;
}

// Value of a non-negative E4M3 code (0..126), exactly.
__device__ __forceinline__ float e4m3_value(uint32_t c) {
    const uint32_t e = (c >> 3) & 15u, m = c & 7u;
    if (e == 0) return static_cast<float>(m) * 0.001953125f;  // m * 2^-9
    return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// Eight floats -> eight E2M1 codes packed in 32 bits (v0 in the lowest nibble).
__device__ __forceinline__ uint32_t e2m1x8(float v0, float v1, float v2, float v3, float v4, float v5, float v6,
                                          float v7) {
    uint32_t out;
    asm("{\n .reg .b8 b0, b1, b2, b3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
        " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
        " mov.b32 %0, {b0, b1, b2, b3};\n}"
        : "=r"(out)
        : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
    return out;
}

// MXFP8 shared exponent: the smallest e with amax <= 448 * 2^e, clamped to
// [-127, 127].  With amax = (1 + m / 2^23) * 2^E, that is E - 8 when the
// mantissa is at most 0.75 (448 = 1.75 * 2^8), else E - 7.
__device__ __forceinline__ int mx_exp(float amax) {
    const uint32_t b = __float_as_uint(amax);
    int e = static_cast<int>((b >> 23) & 0xFFu) - 127 - 8 + (((b & 0x7FFFFFu) > 0x600000u) ? 1 : 0);
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

__device__ __forceinline__ float pow2i(int k) {  // 2^k for k in [-126, 127]
    return __uint_as_float(static_cast<uint32_t>(k + 127) << 23);
}

// NVFP4 per-expert encode scale: 2688 / amax (1 for amax 0), capped at FLT_MAX.
__device__ __forceinline__ float nv_tensor_scale(float amax) {
    if (amax == 0.0f) return 1.0f;
    float s = __fdiv_rn(2688.0f, amax);
    if (!(s <= 3.402823466e38f)) s = 3.402823466e38f;
    return s;
}

// a / 6 rounded to nearest even, for a >= 0.  Above 2^-118 the quotient is
// q = a * RN(1/6) corrected once with the exact remainder a - 6 q (an FMA):
// Markstein's correction step for a quotient from a reciprocal (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990).  For the constant divisor 6 it
// returns the correctly rounded quotient for every binary32 a >= 2^-119
// (checked exhaustively against the IEEE division).  Smaller a divide.
__device__ __forceinline__ float div6(float a) {
    if (a < 0x1p-118f) return __fdiv_rn(a, 6.0f);
    const float y = 0.16666667163372040f;                          // RN(1/6)
    const float q = __fmul_rn(a, y);
    const float r = __fmaf_rn(-q, 6.0f, a);
    return __fmaf_rn(r, y, q);
}

// NVFP4 block: block scale code sb = E4M3((amax_b / 6) * S) and the
// per-element multiplier S / E4M3(sb) looked up from the per-expert table
// rtab[c] = S / value(c) (rtab[0] = 0).
// SMALL_S: the caller knows S <= 2^100.  Then an amax_b below 2^-118 gives
// (amax_b / 6) S < 2^-20, whose E4M3 code is 0 whatever the last bits of the
// quotient, so the corrected product serves every amax_b without the divide.
template <bool SMALL_S = false>
__device__ __forceinline__ float nv_block_mult(float amax_b, float S, const float *rtab, uint32_t &sb) {
    float q;
    if constexpr (SMALL_S) {
        const float y = 0.16666667163372040f;                          // RN(1/6)
        const float q0 = __fmul_rn(amax_b, y);
        q = __fmaf_rn(__fmaf_rn(-q0, 6.0f, amax_b), y, q0);
    } else {
        q = div6(amax_b);
    }
    sb = e4m3_byte(__fmul_rn(q, S));
    return rtab[sb];
}

// Per-expert multiplier table entry (c in 0..127; 0 and the NaN code give 0):
// S / value(c), capped at FLT_MAX as S itself is.  The quotient overflows only
// for S > 2^100 (an expert amax below ~2^-116); capped, every product v * r is
// finite and a zero element stays a zero of its own sign.
__device__ __forceinline__ float nv_table_entry(float S, uint32_t c) {
    return (c == 0 || c >= 127) ? 0.0f : fminf(__fdiv_rn(S, e4m3_value(c)), 3.402823466e38f);
}

// ------------------------------------------------------------ activations

// tanh(u) for 0 <= u <= 1 as u + (u z) Q(z), z = u^2, Q of degree 5 in z.  The
// coefficients are a weighted least-squares fit, reweighted towards minimax
// (Lawson), of (tanh(u)/u - 1)/z on [2^-12, 1] for the relative error of tanh,
// rounded to FP32 (nvfp4_quantization_grouped_gb300/fit_tanh.py prints them);
// evaluated with fused multiply-adds the result stays within 1.7 ulp of tanh(u)
// (checked on the CPU against the exact function).
constexpr float kTanhQ0 = -0x1.555464p-2f, kTanhQ1 = 0x1.10eb8cp-3f, kTanhQ2 = -0x1.b629e6p-5f,
                kTanhQ3 = 0x1.4d2576p-6f, kTanhQ4 = -0x1.988a16p-8f, kTanhQ5 = 0x1.13036ep-10f;

__device__ __forceinline__ float2 tanh01x2(float2 u) {
    const float2 z = __fmul2_rn(u, u);
    float2 q = __ffma2_rn(make_float2(kTanhQ5, kTanhQ5), z, make_float2(kTanhQ4, kTanhQ4));
    q = __ffma2_rn(q, z, make_float2(kTanhQ3, kTanhQ3));
    q = __ffma2_rn(q, z, make_float2(kTanhQ2, kTanhQ2));
    q = __ffma2_rn(q, z, make_float2(kTanhQ1, kTanhQ1));
    q = __ffma2_rn(q, z, make_float2(kTanhQ0, kTanhQ0));
    return __ffma2_rn(__fmul2_rn(u, z), q, u);
}

// tanh of two arguments u >= 0: the polynomial on [0, 1], the library tanhf
// above.  The choice is per element, so a value does not depend on its
// neighbours; callers that know every u <= 1 (a warp vote on X) use
// tanh01x2 alone.  Out of line: the exact form is rare, and inlining the
// library tanhf into every unrolled loop made the kernels' code large enough
// to stall on instruction fetch.
static __device__ __noinline__ float2 tanh_sel2(float2 u) {
    float2 t = tanh01x2(u);
    if (u.x > 1.0f) t.x = tanhf(u.x);
    if (u.y > 1.0f) t.y = tanhf(u.y);
    return t;
}

// x / s for a non-power-of-two s, out of line so that the power-of-two case
// (a product) stays a plain uniform branch.
static __device__ __noinline__ float2 div2_rn(float2 r, float s) {
    return make_float2(__fdiv_rn(r.x, s), __fdiv_rn(r.y, s));
}

struct ActP {
    float s, s2, two_s, limit, alpha, off, inv_s;
    int s_pow2;   // s is a power of two: x / s == x * inv_s exactly
};

// relu on both halves of a BF16 pair.  The sign of a zero may survive; every
// use of the result squares it or divides it and then squares, so the
// activation value is the same as with relu(x) = x > 0 ? x : +0.
__device__ __forceinline__ float2 relu_pair(uint32_t w) {
    const uint32_t r = bmax2(w, 0u);
    return make_float2(bf_lo(r), bf_hi(r));
}

// relu on both halves of a BF16 pair with +0 for every non-positive input
// (including -0), as the derivative needs: halves whose sign bit is set are
// cleared.  The byte permute replicates each half's sign into a 16-bit mask.
__device__ __forceinline__ float2 relu_pair_exact(uint32_t w) {
    uint32_t m;
    asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(m) : "r"(w));   // sign of byte 1 into bytes 0-1, of byte 3 into 2-3
    const uint32_t r = w & ~m;
    return make_float2(bf_lo(r), bf_hi(r));
}

template <int ACT>
struct Act;

template <>
struct Act<ACT_SRELU> {
    static constexpr bool glu = false;
    static constexpr bool ranged = false;
    __device__ __forceinline__ static bool out_of_range(uint32_t, const ActP &) { return false; }
    static constexpr bool nonneg = true;   // act(x) >= 0
    // p * act for the two values of a BF16 pair (packed FP32 products)
    template <bool EXACT = false>
    __device__ __forceinline__ static float2 val2p(uint32_t a, uint32_t, const ActP &, float p) {
        const float2 r = relu_pair(a);
        return __fmul2_rn(__fmul2_rn(r, r), make_float2(p, p));
    }
    __device__ __forceinline__ static float val(float a, float, const ActP &) {
        const float r = a > 0.0f ? a : 0.0f;
        return r * r;
    }
    __device__ __forceinline__ static void grad(float a, float, const ActP &, float &v, float &da, float &db) {
        const float r = a > 0.0f ? a : 0.0f;
        v = r * r;
        da = a > 0.0f ? r + r : 0.0f;
        db = 0.0f;
    }
    // both values of a BF16 pair: relu r (+0 when x <= 0), v = r r, da = r + r
    template <bool EXACT = false>
    __device__ __forceinline__ static void grad2(uint32_t a, uint32_t, const ActP &, float2 &v, float2 &da,
                                                 float2 &db) {
        const float2 r = relu_pair_exact(a);
        v = __fmul2_rn(r, r);
        da = __fadd2_rn(r, r);
        db = make_float2(0.0f, 0.0f);
    }
};

template <>
struct Act<ACT_TANH_SRELU> {  // s^2 tanh^2(relu(x) / s)
    static constexpr bool glu = false;
    static constexpr bool nonneg = true;
    static constexpr bool ranged = true;   // fast tanh needs u <= 1, i.e. x <= s
    __device__ __forceinline__ static float2 arg(float2 r, const ActP &P) {
        if (P.s_pow2) return __fmul2_rn(r, make_float2(P.inv_s, P.inv_s));   // exact
        return div2_rn(r, P.s);
    }
    // some half of BF16 pair m (a running max of X) lies above s, or s is not
    // a power of two (the fast forms compute u = x / s as a product)
    __device__ __forceinline__ static bool out_of_range(uint32_t m, const ActP &P) {
        return fmaxf(bf_lo(m), bf_hi(m)) > P.s || !P.s_pow2;
    }
    // EXACT: any u and s; otherwise every u of the warp's call is <= 1 and s is a
    // power of two, so u is a product and there is no branch
    template <bool EXACT>
    __device__ __forceinline__ static float2 val2p(uint32_t a, uint32_t, const ActP &P, float p) {
        const float2 r = relu_pair(a);
        const float2 u = EXACT ? arg(r, P) : __fmul2_rn(r, make_float2(P.inv_s, P.inv_s));
        const float2 t = EXACT ? tanh_sel2(u) : tanh01x2(u);
        const float2 v = __fmul2_rn(make_float2(P.s2, P.s2), __fmul2_rn(t, t));
        return __fmul2_rn(v, make_float2(p, p));
    }
    // both values of a BF16 pair; for x <= 0, r = +0, t = +0 and da = +0
    template <bool EXACT>
    __device__ __forceinline__ static void grad2(uint32_t a, uint32_t, const ActP &P, float2 &v, float2 &da,
                                                 float2 &db) {
        const float2 r = relu_pair_exact(a);
        const float2 u = EXACT ? arg(r, P) : __fmul2_rn(r, make_float2(P.inv_s, P.inv_s));
        const float2 t = EXACT ? tanh_sel2(u) : tanh01x2(u);
        const float2 tt = __fmul2_rn(t, t);
        v = __fmul2_rn(make_float2(P.s2, P.s2), tt);
        const float2 omt = __ffma2_rn(tt, make_float2(-1.0f, -1.0f), make_float2(1.0f, 1.0f));   // 1 - tt
        da = __fmul2_rn(__fmul2_rn(make_float2(P.two_s, P.two_s), t), omt);
        db = make_float2(0.0f, 0.0f);
    }
};

// e^-t for t >= 0 as 2^(-t log2 e) by the hardware's approximate base-2
// exponential, without flush to zero (results below 2^-126 stay subnormal
// as the exact function's do).  Its relative error is that of the
// exponential (a few units in the last place) plus the rounding of the
// product -t log2(e), which grows with t: at most (4 + 1.25 t) 2^-24, checked
// at every BF16 t on the GPU against the exact function.  t is capped at 200
// (e^-200 is 0 in FP32), so an infinite or huge t gives 0, not 0 * inf.
constexpr float kLog2E = 0x1.715476p+0f;   // RN(log2 e)
__device__ __forceinline__ float exp_neg(float t) {
    const float y = -fminf(t, 200.0f) * kLog2E;
    float e;
    asm("ex2.approx.f32 %0, %1;" : "=f"(e) : "f"(y));
    return e;
}

// sigmoid(a) = 1 / (1 + e^-a) for a >= 0 and e^a / (1 + e^a) for a < 0, with
// E = e^-|a|: the divisor 1 + E stays in [1, 2], where the hardware's
// approximate reciprocal is within an ulp or so.  Both approximations are
// single instructions in inline PTX, so every inlined copy (the forward and
// the backward's regenerated Y) computes the same value.  Below -88.72283...,
// where e^-a overflows FP32, the value is 0, as 1 / (1 + e^-a) evaluated in
// FP32 gives (the defining form of the activation; the exact sigmoid there is
// a subnormal near 1e-39).
constexpr float kExpOverflow = 0x1.62e42ep+6f;   // largest x with e^x finite in FP32
__device__ __forceinline__ float sigmoid_fast(float a) {
    const float e = exp_neg(fabsf(a));
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
    return a >= 0.0f ? r : (a < -kExpOverflow ? 0.0f : e * r);
}

// The same sigmoid for the SwiGLU values (the forward's Y and its
// regeneration, which both take it), with the approximate divide
// __fdividef(1, 1 + E) in place of the reciprocal instruction: it compiled to
// the same value in every case compared (all outputs bitwise equal), and the
// forward kernels schedule it better (MXFP8 SwiGLU forward 104.3 -> 98.5 us).
__device__ __forceinline__ float sigmoid_val(float a) {
    const float e = exp_neg(fabsf(a));
    const float r = __fdividef(1.0f, 1.0f + e);
    return a >= 0.0f ? r : (a < -kExpOverflow ? 0.0f : e * r);
}

template <>
struct Act<ACT_SWIGLU> {  // silu(a) * b
    static constexpr bool glu = true;
    static constexpr bool ranged = false;
    __device__ __forceinline__ static bool out_of_range(uint32_t, const ActP &) { return false; }
    static constexpr bool nonneg = false;
    template <bool EXACT = false>
    __device__ __forceinline__ static float2 val2p(uint32_t a, uint32_t b, const ActP &P, float p) {
        return make_float2(val(bf_lo(a), bf_lo(b), P) * p, val(bf_hi(a), bf_hi(b), P) * p);
    }
    template <bool EXACT = false>
    __device__ __forceinline__ static void grad2(uint32_t a, uint32_t b, const ActP &P, float2 &v, float2 &da,
                                                 float2 &db) {
        grad(bf_lo(a), bf_lo(b), P, v.x, da.x, db.x);
        grad(bf_hi(a), bf_hi(b), P, v.y, da.y, db.y);
    }
    __device__ __forceinline__ static float val(float a, float b, const ActP &) {
        const float sg = sigmoid_val(a);
        const float si = a * sg;
        return si * b;
    }
    __device__ __forceinline__ static void grad(float a, float b, const ActP &, float &v, float &da, float &db) {
        const float sg = sigmoid_fast(a);
        const float si = a * sg;
        v = si * b;
        da = b * (sg + si * (1.0f - sg));
        db = si;
    }
};

template <>
struct Act<ACT_CLAMPED_SWIGLU> {  // min(a,L) sigmoid(alpha min(a,L)) (clamp(b,-L,L) + off)
    static constexpr bool glu = true;
    static constexpr bool ranged = false;
    __device__ __forceinline__ static bool out_of_range(uint32_t, const ActP &) { return false; }
    static constexpr bool nonneg = false;
    template <bool EXACT = false>
    __device__ __forceinline__ static float2 val2p(uint32_t a, uint32_t b, const ActP &P, float p) {
        return make_float2(val(bf_lo(a), bf_lo(b), P) * p, val(bf_hi(a), bf_hi(b), P) * p);
    }
    template <bool EXACT = false>
    __device__ __forceinline__ static void grad2(uint32_t a, uint32_t b, const ActP &P, float2 &v, float2 &da,
                                                 float2 &db) {
        grad(bf_lo(a), bf_lo(b), P, v.x, da.x, db.x);
        grad(bf_hi(a), bf_hi(b), P, v.y, da.y, db.y);
    }
    __device__ __forceinline__ static float val(float a, float b, const ActP &P) {
        const float ac = fminf(a, P.limit);
        const float bc = fminf(fmaxf(b, -P.limit), P.limit);
        const float sg = sigmoid_val(P.alpha * ac);
        const float gl = ac * sg;
        return gl * (bc + P.off);
    }
    __device__ __forceinline__ static void grad(float a, float b, const ActP &P, float &v, float &da, float &db) {
        const float ac = fminf(a, P.limit);
        const float bc = fminf(fmaxf(b, -P.limit), P.limit);
        const float z = P.alpha * ac;
        const float sg = sigmoid_fast(z);
        const float gl = ac * sg;
        const float lin = bc + P.off;
        v = gl * lin;
        da = (a <= P.limit) ? lin * (sg + (z * sg) * (1.0f - sg)) : 0.0f;
        db = (b >= -P.limit && b <= P.limit) ? gl : 0.0f;
    }
};

// Further unary activations (GeLU, sigmoid, identity): the fused kernel and
// its recompute are not specific to the SReLU family.  Each element is
// evaluated on its own in FP32 (GeLU with the library erfcf / expf, sigmoid
// with sigmoid_fast); the packed forms just apply the scalar one to both
// halves of a BF16 pair.
template <int ACT>
struct UnaryAct {
    static constexpr bool glu = false;
    static constexpr bool ranged = false;
    __device__ __forceinline__ static bool out_of_range(uint32_t, const ActP &) { return false; }
    template <bool EXACT = false>
    __device__ __forceinline__ static float2 val2p(uint32_t a, uint32_t, const ActP &P, float p) {
        return make_float2(Act<ACT>::val(bf_lo(a), 0.0f, P) * p, Act<ACT>::val(bf_hi(a), 0.0f, P) * p);
    }
    template <bool EXACT = false>
    __device__ __forceinline__ static void grad2(uint32_t a, uint32_t, const ActP &P, float2 &v, float2 &da,
                                                 float2 &db) {
        float d;
        Act<ACT>::grad(bf_lo(a), 0.0f, P, v.x, da.x, d);
        Act<ACT>::grad(bf_hi(a), 0.0f, P, v.y, da.y, d);
        db = make_float2(0.0f, 0.0f);
    }
};

// GeLU in its defining form x Phi(x), Phi(x) = erfc(-x / sqrt 2) / 2: the
// complementary function keeps the relative accuracy for negative x, where
// 1 + erf(x / sqrt 2) would cancel.  Derivative Phi(x) + x phi(x).
constexpr float kRSqrt2 = 0x1.6a09e6p-1f;      // RN(1 / sqrt 2)
constexpr float kRSqrt2Pi = 0x1.988454p-2f;    // RN(1 / sqrt(2 pi))

template <>
struct Act<ACT_GELU> : UnaryAct<ACT_GELU> {
    static constexpr bool nonneg = false;
    __device__ __forceinline__ static float val(float a, float, const ActP &) {
        const float c = erfcf(-(a * kRSqrt2));
        return (0.5f * a) * c;
    }
    __device__ __forceinline__ static void grad(float a, float, const ActP &, float &v, float &da, float &db) {
        const float c = erfcf(-(a * kRSqrt2));
        v = (0.5f * a) * c;
        const float phi = expf(-((0.5f * a) * a)) * kRSqrt2Pi;
        da = 0.5f * c + a * phi;
        db = 0.0f;
    }
};

template <>
struct Act<ACT_SIGMOID> : UnaryAct<ACT_SIGMOID> {  // 1 / (1 + exp(-x)), derivative s (1 - s)
    static constexpr bool nonneg = true;
    __device__ __forceinline__ static float val(float a, float, const ActP &) {
        return sigmoid_fast(a);
    }
    __device__ __forceinline__ static void grad(float a, float, const ActP &, float &v, float &da, float &db) {
        const float sg = sigmoid_fast(a);
        v = sg;
        da = sg * (1.0f - sg);
        db = 0.0f;
    }
};

template <>
struct Act<ACT_IDENTITY> {   // x: with p = 1 the kernel is a plain grouped quantizer
    static constexpr bool glu = false;
    static constexpr bool ranged = false;
    static constexpr bool nonneg = false;
    __device__ __forceinline__ static bool out_of_range(uint32_t, const ActP &) { return false; }
    template <bool EXACT = false>
    __device__ __forceinline__ static float2 val2p(uint32_t a, uint32_t, const ActP &, float p) {
        return __fmul2_rn(make_float2(bf_lo(a), bf_hi(a)), make_float2(p, p));
    }
    template <bool EXACT = false>
    __device__ __forceinline__ static void grad2(uint32_t a, uint32_t, const ActP &, float2 &v, float2 &da,
                                                 float2 &db) {
        v = make_float2(bf_lo(a), bf_hi(a));
        da = make_float2(1.0f, 1.0f);
        db = make_float2(0.0f, 0.0f);
    }
};

// ------------------------------------------------------ rowwise quantizers

// Pairwise (tree) |max| of n = 8 or 16 packed BF16 pairs; the result's sign
// bits are cleared.  Returns the packed per-half maxima.
__device__ __forceinline__ uint32_t absmax_pairs(const uint32_t *w, int n) {
    uint32_t t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (2 * i < n) t[i] = babsmax2(w[2 * i], w[2 * i + 1]);
#pragma unroll
    for (int s = 1; s < 8; s <<= 1)
#pragma unroll
        for (int i = 0; i < 8; i += 2 * s)
            if (2 * (i + s) < n) t[i] = babsmax2(t[i], t[i + s]);
    return t[0] & 0x7FFF7FFFu;
}

// n packed BF16 pairs -> absolute max.
__device__ __forceinline__ float absmax_words(const uint32_t *w, int n) {
    const uint32_t m = absmax_pairs(w, n);
    return fmaxf(bf_lo(m), bf_hi(m));
}

// MXFP8 rowwise: one 32-value block (16 words) -> 32 bytes + 1 scale byte.
__device__ __forceinline__ void mx_row_block(const uint32_t *w, uint8_t *data, uint8_t *scale) {
    const float amax = absmax_words(w, 16);
    const int e = mx_exp(amax);
    const float2 sc = make_float2(pow2i(-e), pow2i(-e));
    uint32_t o[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const float2 a = __fmul2_rn(make_float2(bf_lo(w[2 * q]), bf_hi(w[2 * q])), sc);
        const float2 b = __fmul2_rn(make_float2(bf_lo(w[2 * q + 1]), bf_hi(w[2 * q + 1])), sc);
        o[q] = e4m3x4(a.x, a.y, b.x, b.y);
    }
    stg128(data, o[0], o[1], o[2], o[3]);
    stg128(data + 16, o[4], o[5], o[6], o[7]);
    *scale = static_cast<uint8_t>(e + 127);
}

// NVFP4 rowwise: two 16-value blocks (16 words) -> 16 bytes + 2 scale bytes.
template <bool SMALL_S = false>
__device__ __forceinline__ void nv_row_blocks(const uint32_t *w, float S, const float *rtab, uint8_t *data,
                                              uint8_t *scale, bool store = true, uint32_t perm = 0) {
    uint32_t o[4], sbs[2];
#pragma unroll
    for (int b = 0; b < 2; ++b) {
        const uint32_t *x = w + 8 * b;
        const float amax = absmax_words(x, 8);
        const float r = nv_block_mult<SMALL_S>(amax, S, rtab, sbs[b]);
        const float2 r2 = make_float2(r, r);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint32_t *y = x + 4 * q;
            float2 t[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) t[u] = __fmul2_rn(make_float2(bf_lo(y[u]), bf_hi(y[u])), r2);
            o[2 * b + q] = e2m1x8(t[0].x, t[0].y, t[1].x, t[1].y, t[2].x, t[2].y, t[3].x, t[3].y);
        }
    }
    // perm: w holds the 16-byte chunks of the 32 values in the order q ^ perm
    // (chunk q = values 8q .. 8q+7): the block amax does not depend on the order,
    // and the encoded words are put back in place
    if (perm & 1u) {
        uint32_t t = o[0]; o[0] = o[1]; o[1] = t;
        t = o[2]; o[2] = o[3]; o[3] = t;
    }
    if (perm & 2u) {
        uint32_t t = o[0]; o[0] = o[2]; o[2] = t;
        t = o[1]; o[1] = o[3]; o[3] = t;
        t = sbs[0]; sbs[0] = sbs[1]; sbs[1] = t;
    }
    if (store) {
        stg128(data, o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint16_t *>(scale) = static_cast<uint16_t>(sbs[0] | (sbs[1] << 8));
    }
}

// --------------------------------------------------------- the kernel body

// YCOL (backward): the instantiation can write the regenerated columnwise copy
// of Y.  The costly activations have a second NVFP4 backward without it.
template <int ACT, int RECIPE, bool BWD, bool YCOL = true, bool TILED = false>
struct Cfg {
    static constexpr bool GLU = Act<ACT>::glu;
    static constexpr bool BWD_ = BWD;
    static constexpr int RECIPE_ = RECIPE;
    static constexpr int B = RECIPE == MXFP8 ? 32 : 16;
    // stage slots: fwd X(a)[, X(b)]; bwd X(a)[, X(b)], dY (+1 for the NVFP4 GLU encode pass)
    static constexpr int NSLOT = BWD ? (GLU ? (RECIPE == NVFP4 ? 4 : 3) : 2) : (GLU ? 2 : 1);
    static constexpr int STAGE_BYTES = NSLOT * kSlotBytes;
    static constexpr int CTAS = NSLOT >= 4 ? 1 : 2;
    static constexpr int STAGES = NSLOT == 1 ? 6 : (NSLOT == 2 ? 3 : (NSLOT == 3 ? 2 : 3));
    static constexpr int META = RECIPE == NVFP4 ? kMetaBytesNV : kMetaBytesMX;
    static constexpr int SEED = RECIPE == NVFP4 ? 2 * kMaxExperts * 4 : 0;
    static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 + STAGES * (META + 16) + 512 + SEED;
    // slot indices
    static constexpr int S_DX_A = GLU ? 0 : 1;  // bwd: where dX (a half) lives after step A
    static constexpr int S_DX_B = 1;            // bwd GLU: dX b half
    static constexpr int S_Y = BWD ? (GLU ? 2 : 0) : 0;  // where Y lives after step A
    static constexpr int S_DY = GLU ? 2 : 1;
    static constexpr bool CHEAP = ACT == ACT_SRELU || ACT == ACT_IDENTITY;
    static constexpr bool YCOL_ = YCOL;
    static constexpr bool TILED_ = TILED;   // block scales in the 128 x 4 tiled layout
    // NVFP4 backward encode pass: the columnwise codes come from warps that each own
    // whole 16-row blocks of a column (no staged codes, no CTA barrier).  A costly
    // activation that regenerates Y keeps the staged-code form: recomputing Y in the
    // column view made its kernel spill and measured slower.
    static constexpr bool COL_OWN = BWD && RECIPE == NVFP4 && (CHEAP || !YCOL);
};

// Dynamic shared memory.  Every pointer into it is formed from this symbol
// plus an offset (never stored in a struct), so the compiler keeps the shared
// address space and emits shared-memory loads and stores.
extern __shared__ __align__(1024) uint8_t gsa_dyn_smem[];

struct Smem {
    uint32_t base;       // offset of the 1024-aligned stage ring
    uint32_t meta_off;   // [STAGES][meta bytes]: TileHdr, S[3], p[128], NVFP4 tables
    uint32_t bar_off;    // full[STAGES], empty[STAGES]
    uint32_t red_off;    // [2][8][3] per-warp partial amax, flag
    uint32_t seed_off;   // NVFP4: [2][kMaxExperts] lower bounds of the columnwise amax (float bits)
    int meta_bytes, stage_bytes, stages;
    __device__ __forceinline__ uint8_t *stage(int s) const { return gsa_dyn_smem + base + s * stage_bytes; }
    __device__ __forceinline__ TileHdr *hdr(int s) const {
        return reinterpret_cast<TileHdr *>(gsa_dyn_smem + meta_off + s * meta_bytes);
    }
    __device__ __forceinline__ float *sbuf(int s) const {
        return reinterpret_cast<float *>(gsa_dyn_smem + meta_off + s * meta_bytes + kMetaS);
    }
    __device__ __forceinline__ float *pbuf(int s) const {
        return reinterpret_cast<float *>(gsa_dyn_smem + meta_off + s * meta_bytes + kMetaP);
    }
    __device__ __forceinline__ float *tbuf(int s) const {
        return reinterpret_cast<float *>(gsa_dyn_smem + meta_off + s * meta_bytes + kMetaT);
    }
    __device__ __forceinline__ uint64_t *full(int s) const {
        return reinterpret_cast<uint64_t *>(gsa_dyn_smem + bar_off) + s;
    }
    __device__ __forceinline__ uint64_t *empty(int s) const {
        return reinterpret_cast<uint64_t *>(gsa_dyn_smem + bar_off) + stages + s;
    }
    __device__ __forceinline__ float *red() const { return reinterpret_cast<float *>(gsa_dyn_smem + red_off); }
    __device__ __forceinline__ int *flag() const { return reinterpret_cast<int *>(gsa_dyn_smem + red_off) + 48; }
    __device__ __forceinline__ uint32_t *seed(int k) const {
        return reinterpret_cast<uint32_t *>(gsa_dyn_smem + seed_off) + k * kMaxExperts;
    }
};

template <class C>
__device__ __forceinline__ Smem carve() {
    Smem s;
    s.base = (1024u - (smem_addr(gsa_dyn_smem) & 1023u)) & 1023u;
    s.stage_bytes = C::STAGE_BYTES;
    s.stages = C::STAGES;
    s.meta_bytes = C::META;
    s.meta_off = s.base + C::STAGES * C::STAGE_BYTES;
    s.bar_off = s.meta_off + C::STAGES * C::META;
    s.red_off = s.bar_off + 16 * C::STAGES;
    s.seed_off = s.red_off + 512;
    return s;
}

// ----------------------------------------------------------------- producer

// One work item as the producer sees it: the tile header fields, the band's
// probabilities and what lane 0 read of the expert's counters when the item
// was decoded.  Those loads are issued one item ahead, so their latency (and
// the ticket's) hides behind the previous item's tile issue.
struct PItem {
    TileHdr h;
    float pv[4];        // p of rows lane + 32 j
    uint32_t am[3];     // lane 0: amax words of the expert (P1 seeds; P2 final once dep >= target)
    uint32_t dep;       // lane 0, P2: done count observed with acquire order
    uint32_t target;    // P2: items of the expert's amax pass
};

// Segment of queue item `item` within segments [seg_lo, seg_hi); a CTA takes
// the items of one queue in increasing order, so the search resumes from seg.
__device__ __forceinline__ int find_seg(const PlanTab &T, uint32_t item, int seg, int seg_hi) {
    if (seg + 1 < seg_hi && T.seg_start[seg + 1] <= static_cast<int>(item)) {
        int lo = seg + 1, hi = seg_hi;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (T.seg_start[mid] <= static_cast<int>(item)) lo = mid; else hi = mid;
        }
        seg = lo;
    }
    return seg;
}

// Decode item `item` of segment seg (K_END when seg < 0) and issue its loads.
__device__ __forceinline__ void decode_item(const KParams &P, uint32_t item, int lane, int seg, PItem &it) {
    it.h.kind = K_END;
    if (seg < 0) return;
    const PlanTab &T = plan_of(P);
    const int info = T.seg_info[seg];
    TileHdr &h = it.h;
    h.kind = info >> 16;
    h.e = info & 0xFFFF;
    const int local = static_cast<int>(item) - T.seg_start[seg] + T.seg_first[seg];
    const int ns = h.kind == K_P2 ? P.n_slabs2 : P.n_slabs;
    const int band = local / ns;
    h.slab = local - band * ns;
    const int64_t ro = T.row_off[h.e];
    h.Me = static_cast<int>(T.row_off[h.e + 1] - ro);
    h.pad_off = static_cast<int>(T.pad_off[h.e]);
    h.Mp = static_cast<int>(T.pad_off[h.e + 1] - T.pad_off[h.e]);
    h.pnn = 0;
    h.lr0 = band * kRows;
    h.row0 = static_cast<int>(ro) + h.lr0;
    h.nrows = min(kRows, h.Me - h.lr0);
    h.gband = T.band_start[h.e] + band;
    h.amax[0] = h.amax[1] = h.amax[2] = 0.0f;
    it.target = static_cast<uint32_t>((T.band_start[h.e + 1] - T.band_start[h.e]) * P.n_slabs);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int r = lane + 32 * j;
        it.pv[j] = r < h.nrows ? (P.probs ? __ldg(P.probs + h.row0 + r) : 1.0f) : 0.0f;
    }
    it.dep = 0;
    it.am[0] = it.am[1] = it.am[2] = 0u;
    if (lane == 0 && h.kind != K_SINGLE) {
        const uint32_t *done = P.ws + WS_HDR;
        const uint32_t *amax_ws = done + P.E;
        // acquire first: amax words read after a complete count are final
        if (h.kind == K_P2) it.dep = ld_acquire_gpu(done + h.e);
#pragma unroll
        for (int k = 0; k < 3; ++k) it.am[k] = ld_relaxed_gpu(amax_ws + 3 * h.e + k);
    }
}

// Scheduler (the producer warp): the next item for this CTA.  An encode item
// (queue 2: one segment per expert, in the amax order) is taken first, from an
// expert whose amax pass is complete, so that it reads that expert's staging
// data while it is in L2; lanes 0-7 look at the next eight experts that still
// have encode items (cursor seg2) at once, and the item comes from a per-expert
// counter (taken2[e]), so a CTA never holds an encode item it would have to
// wait for.  Otherwise the next amax item (queue 1) is taken.  Once queue 1 is
// empty the CTA waits, holding nothing, for an expert to complete (bounded).
// Returns the item (its index within its queue) and sets seg to its segment,
// -1 when no items are left.  Uniform over the warp.
// Queue 1 may also hold encode items, placed by the host after a lookahead of
// further amax items (static interleave, queue 2 empty): such an item is taken
// in ticket order and its producer waits, bounded, for the expert's amax pass.
static __device__ __noinline__ uint32_t next_item(const KParams &P, int lane, bool &q1_left, int &seg1, int &seg2,
                                                  int &seg) {
    uint32_t *ws = P.ws;
    const uint32_t *done = ws + WS_HDR;
    uint32_t *taken2 = ws + WS_HDR + 4 * P.E;
    const PlanTab &T = plan_of(P);
    uint64_t t0 = 0;
    for (uint32_t spin = 0;; ++spin) {
        bool q2_left = false;
        if (seg2 < T.n_segs) {
            const int k = seg2 + lane;
            bool have = false, ready = false;
            uint32_t cnt = 0;
            int e = 0;
            if (lane < 8 && k < T.n_segs) {
                e = T.seg_info[k] & 0xFFFF;
                const uint32_t nb = static_cast<uint32_t>(T.band_start[e + 1] - T.band_start[e]);
                cnt = nb * static_cast<uint32_t>(P.n_slabs2);   // encode items of e
                const uint32_t tk = ld_relaxed_gpu(taken2 + e);
                const uint32_t dn = ld_acquire_gpu(done + e);
                have = tk < cnt;
                ready = have && dn >= nb * static_cast<uint32_t>(P.n_slabs);   // every amax item of e done
            }
            const uint32_t hv = __ballot_sync(0xFFFFFFFFu, have);
            const uint32_t rd = __ballot_sync(0xFFFFFFFFu, ready);
            const int base = seg2;
            if (hv == 0) {
                seg2 = min(seg2 + 8, T.n_segs);   // all eight exhausted: move on
                if (seg2 < T.n_segs) continue;
            } else {
                seg2 += __ffs(hv) - 1;            // skip exhausted experts
                q2_left = true;
            }
            if (rd != 0) {
                const int l = __ffs(rd) - 1;
                uint32_t u = 0;
                if (lane == l) u = atomicAdd(taken2 + e, 1u);
                u = __shfl_sync(0xFFFFFFFFu, u, l);
                const uint32_t c = __shfl_sync(0xFFFFFFFFu, cnt, l);
                if (u < c) {
                    seg = base + l;
                    return static_cast<uint32_t>(T.seg_start[seg]) + u;
                }
                continue;   // that expert ran out meanwhile
            }
        }
        if (q1_left) {
            uint32_t v1 = 0;
            if (lane == 0) v1 = atomicAdd(ws + WS_TICKET, 1u);
            v1 = __shfl_sync(0xFFFFFFFFu, v1, 0);
            if (v1 < static_cast<uint32_t>(T.n_items)) {
                seg1 = find_seg(T, v1, seg1, T.n_segs1);
                seg = seg1;
                return v1;
            }
            q1_left = false;
            continue;
        }
        if (!q2_left) {
            seg = -1;
            return 0;
        }
        // every amax item is taken; no expert with encode items left is complete yet
        if (t0 == 0) t0 = global_ns();
        __nanosleep(200);
        if ((spin & 63u) == 63u) {
            int bad = 0;
            if (lane == 0) bad = (global_ns() - t0 > kWaitLimitNs || ld_relaxed_gpu(ws + WS_ERR)) ? 1 : 0;
            if (__shfl_sync(0xFFFFFFFFu, bad, 0)) {
                if (lane == 0) atomicOr(ws + WS_ERR, ERR_TIMEOUT_DEP);
                seg = -1;
                return 0;
            }
        }
    }
}

template <class C>
__device__ void producer(const KParams &P, const Smem &sm, int lane) {
    uint32_t *ws = P.ws;
    uint32_t *done = ws + WS_HDR;
    uint32_t *amax_ws = done + P.E;
    const uint64_t pol_keep = policy_evict_last();
    const uint64_t pol_stream = policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    bool q1_left = plan_of(P).n_items > 0;
    int seg1 = 0, seg2 = plan_of(P).n_segs1;
    PItem cur;
    {
        int seg = -1;
        const uint32_t item = next_item(P, lane, q1_left, seg1, seg2, seg);
        decode_item(P, item, lane, seg, cur);
    }
    for (;;) {
        TileHdr &h = cur.h;
        float Sk[3] = {1.0f, 1.0f, 1.0f};
        float tab[3][4];
        if (h.kind == K_P1 || h.kind == K_P2) {
            if (h.kind == K_P2 && lane == 0) {
                if (cur.dep < cur.target) {
                    wait_count(done + h.e, cur.target, ws);
#pragma unroll
                    for (int k = 0; k < 3; ++k) cur.am[k] = ld_relaxed_gpu(amax_ws + 3 * h.e + k);
                }
                // what the amax pass wrote (staging copy, dense dX) is read below through the async proxy
                asm volatile("fence.proxy.async.global;" ::: "memory");
            }
#pragma unroll
            for (int k = 0; k < 3; ++k) h.amax[k] = __uint_as_float(__shfl_sync(0xFFFFFFFFu, cur.am[k], 0));
            if constexpr (C::RECIPE_ == NVFP4) {
                if (h.kind == K_P2) {
#pragma unroll
                    for (int k = 0; k < 3; ++k) {
                        Sk[k] = nv_tensor_scale(h.amax[k]);
#pragma unroll
                        for (int j = 0; j < 4; ++j) tab[k][j] = nv_table_entry(Sk[k], static_cast<uint32_t>(lane + 32 * j));
                    }
                }
            }
        }
        h.pnn = __all_sync(0xFFFFFFFFu, !(cur.pv[0] < 0.0f) && !(cur.pv[1] < 0.0f) && !(cur.pv[2] < 0.0f) &&
                                            !(cur.pv[3] < 0.0f)) ? 1 : 0;
        const int tps = (h.kind == K_P2) ? P.tiles_per_slab2 : P.tiles_per_slab;
        const int ntiles = (h.kind == K_END) ? 1 : tps;
        for (int t = 0; t < ntiles; ++t) {
            const uint32_t full = smem_addr(sm.full(stage));
            int ok = 1;
            if (lane == 0) ok = mbar_wait_backoff(smem_addr(sm.empty(stage)), phase ^ 1u, ws, ERR_TIMEOUT_EMPTY) ? 1 : 0;
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) return;
            float *pb = sm.pbuf(stage);
#pragma unroll
            for (int j = 0; j < 4; ++j) pb[lane + 32 * j] = cur.pv[j];
            if constexpr (C::RECIPE_ == NVFP4) {
                if (h.kind == K_P2) {
                    float *tb = sm.tbuf(stage);
#pragma unroll
                    for (int k = 0; k < 3; ++k)
#pragma unroll
                        for (int j = 0; j < 4; ++j) tb[128 * k + lane + 32 * j] = tab[k][j];
                    if (lane < 3) sm.sbuf(stage)[lane] = lane == 0 ? Sk[0] : (lane == 1 ? Sk[1] : Sk[2]);
                }
            }
            if (lane == 0) {
                TileHdr hh = h;
                hh.tile = t;
                hh.col0 = (h.slab * tps + t) * kCols;
                *sm.hdr(stage) = hh;
            }
            __syncwarp();
            if (lane == 0) {
                if (h.kind == K_END) {
                    mbar_arrive(full);
                } else {
                    const uint32_t dst = smem_addr(sm.stage(stage));
                    const int c = (h.slab * tps + t) * kCols, r = h.row0;
                    // L2 priority: keep (evict_last) only what the encode pass reads again --
                    // X in the forward without a staging copy, X in the backward when Y
                    // is regenerated; everything else streams (evict_first).
                    const bool regen_x = C::BWD_ && P.q[1].col_data != nullptr;
                    const bool x_again = (h.kind == K_P1) && (C::BWD_ ? regen_x : !P.stash);
                    const uint64_t pol = x_again ? pol_keep : pol_stream;
                    if constexpr (!C::BWD_) {
                        if (h.kind == K_P2 && P.stash) {
                            // the (band, tile) staging image, byte for byte (its layout is the one
                            // the encode pass reads)
                            const int64_t img = static_cast<int64_t>(h.gband) * (P.W / kCols) + h.slab * tps + t;
                            mbar_expect_tx(full, kSlotBytes);
                            bulk_load(dst, P.stash + img * kSlotBytes, kSlotBytes, full, pol);
                        } else {
                            mbar_expect_tx(full, (C::GLU ? 2 : 1) * kSlotBytes);
                            tma_load(dst, &P.tm_x, c, r, full, pol);
                            if constexpr (C::GLU) tma_load(dst + kSlotBytes, &P.tm_x, P.W + c, r, full, pol);
                        }
                    } else {
                        if (h.kind != K_P2) {
                            mbar_expect_tx(full, (C::GLU ? 3 : 2) * kSlotBytes);
                            tma_load(dst, &P.tm_x, c, r, full, pol);
                            if constexpr (C::GLU) tma_load(dst + kSlotBytes, &P.tm_x, P.W + c, r, full, pol);
                            tma_load(dst + C::S_DY * kSlotBytes, &P.tm_dy, c, r, full, pol_stream);
                        } else {
                            // encode pass: the dense dX when its quantized copy is requested (the
                            // host then requires the dense dX, so tm_dx is encoded), X when Y is
                            // regenerated
                            const bool regen = P.q[1].col_data != nullptr;
                            const bool dxq = P.q[0].row_data != nullptr || P.q[0].col_data != nullptr;
                            const int n = (C::GLU ? 2 : 1) * ((dxq ? 1 : 0) + (regen ? 1 : 0));
                            mbar_expect_tx(full, n * kSlotBytes);
                            if (dxq) {
                                tma_load(dst + C::S_DX_A * kSlotBytes, &P.tm_dx, c, r, full, pol_stream);
                                if constexpr (C::GLU)
                                    tma_load(dst + C::S_DX_B * kSlotBytes, &P.tm_dx, P.W + c, r, full, pol_stream);
                            }
                            if (regen) {
                                if constexpr (C::GLU) {
                                    tma_load(dst + 2 * kSlotBytes, &P.tm_x, c, r, full, pol);
                                    tma_load(dst + 3 * kSlotBytes, &P.tm_x, P.W + c, r, full, pol);
                                } else {
                                    tma_load(dst, &P.tm_x, c, r, full, pol);
                                }
                            }
                        }
                    }
                }
            }
            if (h.kind == K_END) return;
            if (++stage == C::STAGES) {
                stage = 0;
                phase ^= 1u;
            }
        }
        // the next item: chosen and decoded while the consumers work on this one's tiles
        // the next item, chosen once this one's tiles are out (so a CTA that waits
        // for an expert holds nothing that expert could need); its loads overlap the
        // consumers' work on the tiles just issued
        int seg = -1;
        const uint32_t item = next_item(P, lane, q1_left, seg1, seg2, seg);
        decode_item(P, item, lane, seg, cur);
    }
}

// ---------------------------------------------------------------- consumers

// NVFP4 columnwise amax of one 16-row x 2-column block held as 16 packed
// BF16 words (rows in order), folded into the running maximum acc.  With the
// RHT, a warp first tests a rigorous upper bound of every output,
// |w| <= (1/4) sum |v| (1 + 20 * 2^-24), with the sum taken in BF16 from
// above (tree depth 4, margin 1.02), and skips the transform when no lane could
// raise max(acc, seed).
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

// Per-half sum of |v| over 16 packed BF16 words, in BF16 (tree of depth 4,
// each sum rounded to nearest: within 2% of the exact sum).
__device__ __forceinline__ uint32_t sum_abs_pairs(const uint32_t (&wd)[16]) {
    uint32_t t[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) t[i] = badd2(wd[2 * i] & 0x7FFF7FFFu, wd[2 * i + 1] & 0x7FFF7FFFu);
#pragma unroll
    for (int s = 1; s < 8; s <<= 1)
#pragma unroll
        for (int i = 0; i < 8; i += 2 * s) t[i] = badd2(t[i], t[i + s]);
    return t[0];
}

// The two values of BF16 pair w as FP32 with the RHT sign of row i applied:
// lo = (w << 16) with bit 31 flipped by adding sgnlo (0x80000000 or 0),
// hi = (w ^ sgn) with the low half cleared.
__device__ __forceinline__ float2 unpack_signed(uint32_t w, uint32_t sgn, uint32_t sgnlo) {
    return make_float2(__uint_as_float(w * 65536u + sgnlo), __uint_as_float((w ^ sgn) & 0xFFFF0000u));
}

// 16-point FWHT (stride 1, 2, 4, 8) of 16 rows of two columns, in place.
__device__ __forceinline__ void fwht16(float2 (&v)[16]) {
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (i & h) continue;
            const float2 a = v[i], c = v[i + h];
            v[i] = __fadd2_rn(a, c);
            v[i + h] = fsub2(a, c);
        }
    }
}

// max(|a|, |b|, |c|) in one instruction (the three-input max of sm_100 and later).
__device__ __forceinline__ float absmax3(float a, float b, float c) {
    float r;
    asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
// Per-column maximum |v| over 16 rows (x: first column, y: second): a tree of
// three-input maxima, 8 per column.
__device__ __forceinline__ float2 absmax16(const float2 (&v)[16]) {
    float a[5], b[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) {
        a[i] = absmax3(v[3 * i].x, v[3 * i + 1].x, v[3 * i + 2].x);
        b[i] = absmax3(v[3 * i].y, v[3 * i + 1].y, v[3 * i + 2].y);
    }
    const float a5 = absmax3(a[0], a[1], v[15].x), b5 = absmax3(b[0], b[1], v[15].y);
    return make_float2(absmax3(a[2], a[3], absmax3(a[4], a5, 0.0f)), absmax3(b[2], b[3], absmax3(b[4], b5, 0.0f)));
}

// Largest |H D v| (before the 1/4) of the lane's two RHT blocks (16 rows x 2 columns).
__device__ __forceinline__ float rht_absmax_words(const uint32_t (&wd)[16], const KParams &P) {
    float2 v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = unpack_signed(wd[i], P.rht_sgn[i], P.rht_sgnlo[i]);
    fwht16(v);
    const float2 m = absmax16(v);
    return fmaxf(m.x, m.y);
}

// NVFP4 amax pass, columnwise copy with the RHT, for one warp's 16-row block.
//   bound: per lane, an upper bound of every |w| of its two blocks
//   lower: per lane, a lower bound of the expert's final columnwise amax
//   seed : the CTA's best lower bound for this expert (shared, raised with atomicMax)
//   pub  : what earlier items published for this expert
// The transform runs only when some lane's bound exceeds every known lower
// bound; the final amax is the largest computed value, so a block whose
// values cannot exceed a lower bound of it leaves it unchanged.  acc takes
// computed values only; the seed takes both kinds.
__device__ __forceinline__ void p1_col_rht_amax(const uint32_t (&wd)[16], const KParams &P, float bound, float lower,
                                                uint32_t *seed, float pub, float &acc, int lane) {
    const float lw = warp_max(lower);
    const float s = fmaxf(fmaxf(lw, __uint_as_float(*reinterpret_cast<volatile uint32_t *>(seed))), fmaxf(pub, acc));
    float known = s;
    if (__any_sync(0xFFFFFFFFu, bound > s)) {
        const float m = rht_absmax_words(wd, P) * 0.25f;   // max |RN(x / 4)| = RN(max |x| / 4)
        acc = fmaxf(acc, m);
        known = fmaxf(known, warp_max(m));
    }
    if (lane == 0 && known > __uint_as_float(*reinterpret_cast<volatile uint32_t *>(seed)))
        atomicMax(seed, __float_as_uint(known));
}

// NVFP4 columnwise amax of one 16-row x 2-column block held as 16 packed
// BF16 words (rows in order), folded into the running maximum acc.  With the
// RHT, a warp first tests a rigorous upper bound of every output,
// |w| <= (1/4) sum |v| (1 + 20 * 2^-24), with the sum taken in BF16 (tree
// depth 4, margin 1.02), and skips the transform when no lane could raise
// max(acc, seed).
__device__ __forceinline__ void nv_col_amax_words(const uint32_t (&wd)[16], const KParams &P, float &acc, float seed) {
    if (P.rht) {
        const uint32_t t = sum_abs_pairs(wd);
        const float bound = fmaxf(bf_lo(t), bf_hi(t)) * 0.255f + 1e-36f;
        // any value already computed for this expert (by any lane, any item) is a
        // lower bound of its final amax: a chunk that cannot exceed it changes nothing
        if (__all_sync(0xFFFFFFFFu, bound <= warp_max(fmaxf(acc, seed)))) return;
        acc = fmaxf(acc, rht_absmax_words(wd, P) * 0.25f);   // max |RN(x / 4)| = RN(max |x| / 4)
        return;
    }
    const uint32_t m = absmax_pairs(wd, 16);
    acc = fmaxf(acc, fmaxf(bf_lo(m), bf_hi(m)));
}

// NVFP4 columnwise codes of one lane's two 16-row blocks (16 packed BF16
// words, rows in order; a column pair of the tile): sign flips and FWHT when
// the RHT is on, block amax, scale codes sb0/sb1 and multipliers, E2M1 codes
// (o0: first column's 16 rows, o1: second's).
// With the RHT the 1/4 is folded into the multiplier, RN(RN(w / 4) k) ==
// RN(w (k / 4)), when k / 4 is exact and the block amax is at least 2^-100
// (then an element whose w / 4 would round, |w| < 2^-124, gives a code 0 of
// the same sign either way); otherwise the warp takes the two products.
template <bool SMALL_S = false>
__device__ __forceinline__ void nv_col_block_codes(const uint32_t (&wd)[16], const KParams &P, float S,
                                                   const float *rtab, uint32_t (&o0)[2], uint32_t (&o1)[2],
                                                   uint32_t &sb0, uint32_t &sb1) {
    float2 v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = unpack_signed(wd[i], P.rht_sgn[i], P.rht_sgnlo[i]);   // signs 0 without the RHT
    float2 k;
    if (P.rht) {
        fwht16(v);
        const float2 m = absmax16(v);
        const float c0 = m.x * 0.25f, c1 = m.y * 0.25f;   // max |RN(x / 4)| = RN(max |x| / 4)
        k = make_float2(nv_block_mult<SMALL_S>(c0, S, rtab, sb0), nv_block_mult<SMALL_S>(c1, S, rtab, sb1));
        const bool ok = (k.x == 0.0f || (k.x >= 0x1p-122f && c0 >= 0x1p-100f)) &&
                        (k.y == 0.0f || (k.y >= 0x1p-122f && c1 >= 0x1p-100f));
        if (__all_sync(0xFFFFFFFFu, ok)) {
            k = __fmul2_rn(k, make_float2(0.25f, 0.25f));
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __fmul2_rn(v[i], make_float2(0.25f, 0.25f));
        }
    } else {
        const float2 m = absmax16(v);
        k = make_float2(nv_block_mult<SMALL_S>(m.x, S, rtab, sb0), nv_block_mult<SMALL_S>(m.y, S, rtab, sb1));
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __fmul2_rn(v[i], k);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const float2 *x = v + 8 * j;
        o0[j] = e2m1x8(x[0].x, x[1].x, x[2].x, x[3].x, x[4].x, x[5].x, x[6].x, x[7].x);
        o1[j] = e2m1x8(x[0].y, x[1].y, x[2].y, x[3].y, x[4].y, x[5].y, x[6].y, x[7].y);
    }
}

// The same, staged in the warp's own 16-row region of `slot` (which it has
// finished reading) for nv_col_flush.
template <bool SMALL_S = false>
__device__ __forceinline__ void nv_col_block_encode(const uint32_t (&wd)[16], const KParams &P, float S,
                                                    const float *rtab, uint8_t *slot, int warp, int lane) {
    uint32_t o0[2], o1[2], sb0, sb1;
    nv_col_block_codes<SMALL_S>(wd, P, S, rtab, o0, o1, sb0, sb1);
    // Staging of the warp's block (row block w of the tile) in its region
    // slot + 2048 w: the 8 code bytes of column c at 8 (c ^ 2w) -- the lane's two
    // columns as one 16-byte store at 16 (lane ^ w) -- and the scale code of
    // column c at byte 512 + c.  The swizzle keeps both this store and the
    // flush's reads at the minimum number of shared-memory wavefronts.
    uint8_t *region = slot + warp * 2048;
    __syncwarp();   // every lane has read its words from the region
    sts128(region + 16 * (lane ^ warp), o0[0], o0[1], o1[0], o1[1]);
    *reinterpret_cast<uint16_t *>(region + 512 + 2 * lane) = static_cast<uint16_t>(sb0 | (sb1 << 8));
}

// Store a tile's staged NVFP4 columnwise codes (64 columns x 8 row blocks) once
// every consumer warp has staged its block: each column's 64 code bytes of the
// band go out as one run written by 8 lanes, its 8 scale bytes by 4 lanes.
// Row blocks at or past the expert's end are not stored.
template <bool TILED>
__device__ __forceinline__ void nv_col_flush(const KParams &P, const uint8_t *slot, const QDev &q, int colbase,
                                             int width, const TileHdr &hd, int tid) {
    const int64_t Mp = hd.Mp;
    const int64_t rowbytes = Mp / 2;
    uint8_t *dbase = q.col_data + static_cast<int64_t>(width) * (hd.pad_off / 2);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const int u = tid + kCons * k;
        const int c = u >> 3, w = u & 7;
        const int lrb = hd.lr0 + 16 * w;
        const uint2 d = *reinterpret_cast<const uint2 *>(slot + w * 2048 + 8 * (c ^ (2 * w)));
        const int64_t col = colbase + hd.col0 + c;
        if (lrb < hd.Me) stg64(dbase + col * rowbytes + lrb / 2, d.x, d.y);
    }
    const int c = tid >> 2, w = 2 * (tid & 3);
    const int64_t col = colbase + hd.col0 + c;
    const uint8_t a = slot[w * 2048 + 512 + c], b = slot[(w + 1) * 2048 + 512 + c];
    // blocks w, w + 1 (w even, lr0 a multiple of 128) sit in adjacent bytes in both layouts
    uint8_t *sp = col_scale_ptr<16, TILED>(P, q.col_scale, hd, col, hd.lr0 / 16 + w, width);
    if (hd.lr0 + 16 * w < hd.Me) sp[0] = a;
    if (hd.lr0 + 16 * (w + 1) < hd.Me) sp[1] = b;
}

// Columnwise pass over one 128 x 64 value slot for output q.
//   colbase: first output column of this slot's columns (GLU dX b half: W)
//   width  : output tensor width (sets the columnwise layout)
//   mode   : 0 encode, 1 amax only (into acc)
template <int RECIPE, bool TILED>
__device__ __forceinline__ void col_pass(const KParams &P, const TileHdr &hd, const uint8_t *slot, const QDev &q,
                                         int colbase, int width, int mode, float S, const float *rtab, float &acc,
                                         int warp, int lane, float seed = 0.0f) {
    const int64_t Me = hd.Me;
    const int64_t Mp = hd.Mp;
    const int lr0 = hd.lr0;   // band's first row inside the expert
    // Word (column pair) p of tile row r sits at r*128 + (((p>>2) ^ (r&7)) << 4) + (p&3)*4.
    // With xo = ((p>>2) << 4) | ((p&3) << 2) that is r*128 + (xo ^ ((r&7) << 4)).
    if constexpr (RECIPE == MXFP8) {
        const int b = warp >> 1;
        const int hb = lane >> 4;
        const int p = 16 * (warp & 1) + (lane & 15);
        const int lrb = lr0 + 32 * b;
        if (lrb >= Me) return;
        // rows 32b + 16hb + ((i + 4hb) & 15): rotated for the two half-warps so that
        // they hit disjoint banks; (i + 4hb) & 7 == (i & 7) ^ 4hb.
        const uint32_t xo = ((static_cast<uint32_t>(p) >> 2) << 4) | ((static_cast<uint32_t>(p) & 3u) << 2);
        const uint32_t xh = xo ^ (static_cast<uint32_t>(hb) << 6);
        const uint8_t *sb = slot + (32 * b + 16 * hb) * 128;
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t roff = ((static_cast<uint32_t>(i) * 128u + static_cast<uint32_t>(hb) * 512u) & 2047u);
            w[i] = lds32(sb + roff + (xh ^ ((static_cast<uint32_t>(i) & 7u) << 4)));
        }
        uint32_t m = absmax_pairs(w, 16);
        m = bmax2(m, __shfl_xor_sync(0xFFFFFFFFu, m, 16));
        const int e0 = mx_exp(bf_lo(m)), e1 = mx_exp(bf_hi(m));
        const float2 sc = make_float2(pow2i(-e0), pow2i(-e1));
        uint32_t c0[4], c1[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float2 t[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) t[u] = __fmul2_rn(make_float2(bf_lo(w[4 * j + u]), bf_hi(w[4 * j + u])), sc);
            c0[j] = e4m3x4(t[0].x, t[1].x, t[2].x, t[3].x);
            c1[j] = e4m3x4(t[0].y, t[1].y, t[2].y, t[3].y);
        }
        // iteration i holds row (i + 4 hb) & 15: rotate words back into row order
        uint32_t r0[4], r1[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            r0[k] = hb ? c0[(k + 3) & 3] : c0[k];
            r1[k] = hb ? c1[(k + 3) & 3] : c1[k];
        }
        const int64_t col = colbase + hd.col0 + 2 * p;
        uint8_t *base = q.col_data + static_cast<int64_t>(width) * hd.pad_off;
        uint8_t *d0 = base + col * Mp + lrb + 16 * hb;
        stg128(d0, r0[0], r0[1], r0[2], r0[3]);
        stg128(d0 + Mp, r1[0], r1[1], r1[2], r1[3]);
        if (hb == 0) {
            *col_scale_ptr<32, TILED>(P, q.col_scale, hd, col, lrb / 32, width) = static_cast<uint8_t>(e0 + 127);
            *col_scale_ptr<32, TILED>(P, q.col_scale, hd, col + 1, lrb / 32, width) = static_cast<uint8_t>(e1 + 127);
        }
    } else {
        const int b = warp;
        const int p = lane;
        const int lrb = lr0 + 16 * b;
        if (lrb >= Me) return;
        const uint32_t xo = ((static_cast<uint32_t>(p) >> 2) << 4) | ((static_cast<uint32_t>(p) & 3u) << 2);
        const uint8_t *sb = slot + 16 * b * 128;
        if (mode == 1) {
            uint32_t wd[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) wd[i] = lds32(sb + i * 128 + (xo ^ ((static_cast<uint32_t>(i) & 7u) << 4)));
            nv_col_amax_words(wd, P, acc, seed);
            return;
        }
        uint32_t wd[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) wd[i] = lds32(sb + i * 128 + (xo ^ ((static_cast<uint32_t>(i) & 7u) << 4)));
        nv_col_block_encode(wd, P, S, rtab, const_cast<uint8_t *>(slot), warp, lane);   // flushed after the tile
    }
}

// Rowwise pass of 32 values (16 words) of row `grow` starting at column gc of a
// width-`width` tensor.  mode 0 encode, 1 amax only.
template <int RECIPE, bool TILED>
__device__ __forceinline__ void row_pass(const KParams &P, const TileHdr &hd, const QDev &q, const uint32_t *w,
                                         int64_t grow, int gc, int width, int mode, float S, const float *rtab,
                                         float &acc) {
    if (mode == 1) {
        acc = fmaxf(acc, absmax_words(w, 16));
        return;
    }
    const int64_t lr = hd.lr0 + (grow - hd.row0);
    if constexpr (RECIPE == MXFP8) {
        mx_row_block(w, q.row_data + grow * width + gc, row_scale_ptr<32, TILED>(P, q.row_scale, hd.e, grow, lr, gc / 32, width));
    } else {
        nv_row_blocks(w, S, rtab, q.row_data + grow * (width / 2) + gc / 2,
                      row_scale_ptr<16, TILED>(P, q.row_scale, hd.e, grow, lr, gc / 16, width));
    }
}

// NVFP4 forward amax pass over one warp's 16-row block of a tile, in the
// column layout (lane = column pair): Y = p * act(X) row by row from the
// swizzled X tile at sa, the packed words into wd[] and, when img is set, into
// the staging image (row i of the block at img + 32 i words).  Returns the
// per-half maximum |Y| of the lane's 16 rows.  FULL: all 16 rows are valid;
// otherwise rows from nvalid on give Y = 0.  SUMS: vs receives the per-column
// sums of the FP32 values (before rounding to BF16).  An activation with a
// restricted fast range runs the block again exactly (EXACT) when some X of
// the warp lies outside it.
template <class A, bool GLU, bool FULL, bool SUMS, bool EXACT = false>
__device__ __forceinline__ uint32_t p1_rows(const uint8_t *sa, const float4 *pq, uint32_t xo, const ActP &ap,
                                            int nvalid, uint32_t *img, uint32_t (&wd)[16], float2 &vs) {
    uint32_t rm = 0u, xm = 0u;
    vs = make_float2(0.0f, 0.0f);
    float4 p4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t off = static_cast<uint32_t>(i) * 128u + (xo ^ ((static_cast<uint32_t>(i) & 7u) << 4));
        const uint32_t a = lds32(sa + off);
        uint32_t bw = 0u;
        if constexpr (GLU) bw = lds32(sa + kSlotBytes + off);
        if ((i & 3) == 0) p4 = pq[i >> 2];   // p of rows i..i+3 (broadcast load)
        const float pr = (i & 3) == 0 ? p4.x : ((i & 3) == 1 ? p4.y : ((i & 3) == 2 ? p4.z : p4.w));
        if constexpr (A::ranged && !EXACT) xm = bmax2(xm, a);
        const float2 v = A::template val2p<EXACT>(a, bw, ap, pr);
        if constexpr (SUMS) vs = __fadd2_rn(vs, v);
        uint32_t y = pack_bf16x2(v.x, v.y);
        if constexpr (!FULL) y = i < nvalid ? y : 0u;
        wd[i] = y;
        rm = babsmax2(rm, y);
        if (img) stg32(img + 32 * i, y);   // row i of the block: 128 bytes on
    }
    if constexpr (A::ranged && !EXACT) {
        if (__any_sync(0xFFFFFFFFu, A::out_of_range(xm, ap)))
            return p1_rows<A, GLU, FULL, SUMS, true>(sa, pq, xo, ap, nvalid, img, wd, vs);
    }
    return rm & 0x7FFF7FFFu;
}

// Whether some X of the warp's four words lies outside the activation's fast range.
template <class A>
__device__ __forceinline__ bool need_exact4(const uint32_t (&aw)[4], const ActP &ap) {
    if constexpr (!A::ranged) return false;
    const uint32_t m = bmax2(bmax2(aw[0], aw[1]), bmax2(aw[2], aw[3]));
    return __any_sync(0xFFFFFFFFu, A::out_of_range(m, ap));
}

// NVFP4 forward encode pass over a tile whose Y came back from its staging
// image.  Image layout: row r at r * 128, its 16-byte chunk c (columns 8c ..
// 8c+7) at position c ^ (r >> 4) -- the 16-row block index.  Two views, both
// at the minimum number of shared-memory wavefronts:
//  * rowwise copy, thread = (row 16 warp + j, 32-column half h): the four
//    chunks of the half are read in the order q ^ (j & 3), which spreads a
//    warp's 16 rows over all chunk positions, and encoded with that permutation;
//  * columnwise copy, warp = 8 columns (chunk `warp`) x all 128 rows, lane =
//    (16-row block b, column pair): the block's chunk sits at warp ^ b, distinct
//    across the 8 blocks.  Each column's 64 code bytes of the band (8 blocks)
//    then come from 8 lanes of one warp and are stored directly, with no
//    exchange between warps.
// Only stores depend on whether a row (or a block) lies inside the expert.
template <bool ROW, bool COL, bool SMALL_S, bool TILED>
__device__ __forceinline__ void p2_stash_tile(const KParams &P, const TileHdr &hd, const uint8_t *st, int warp, int lane,
                                              float Srow, const float *rt_row, float Scol, const float *rt_col) {
    const int j = lane >> 1, h = lane & 1;
    const int r = 16 * warp + j;
    const bool vrow = r < hd.nrows;
    const int64_t grow = static_cast<int64_t>(hd.row0) + r;
    const uint32_t perm = static_cast<uint32_t>(j) & 3u;
    uint32_t yw[16];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t c = 4u * h + (static_cast<uint32_t>(k) ^ perm);
        const uint4 y4 = lds128(st + r * 128 + (((c ^ static_cast<uint32_t>(warp)) & 7u) << 4));
        yw[4 * k] = y4.x; yw[4 * k + 1] = y4.y; yw[4 * k + 2] = y4.z; yw[4 * k + 3] = y4.w;
    }
    const int b = lane >> 2, cp = lane & 3;
    uint32_t wd[16];
    if constexpr (COL) {
        const uint8_t *sb = st + 16 * b * 128 + ((((warp ^ b) & 7)) << 4) + cp * 4;
#pragma unroll
        for (int i = 0; i < 16; ++i) wd[i] = lds32(sb + i * 128);
    }
    if (h == 0) {
        // row r of the staging image (128 bytes) is dead after this read
        const uint8_t *line =
            P.stash + (static_cast<int64_t>(hd.gband) * (P.W / kCols) + hd.col0 / kCols) * kSlotBytes + r * 128;
        asm volatile("discard.global.L2 [%0], 128;" ::"l"(line) : "memory");
    }
    if (P.y_bf16 && vrow) {
        uint16_t *dst = P.y_bf16 + grow * P.W + hd.col0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int c = 4 * h + (k ^ static_cast<int>(perm));
            stg128(dst + 8 * c, yw[4 * k], yw[4 * k + 1], yw[4 * k + 2], yw[4 * k + 3]);
        }
    }
    const int gc = hd.col0 + 32 * h;
    if constexpr (ROW)
        nv_row_blocks<SMALL_S>(yw, Srow, rt_row, P.q[0].row_data + grow * (P.W / 2) + gc / 2,
                               row_scale_ptr<16, TILED>(P, P.q[0].row_scale, hd.e, grow, hd.lr0 + r, gc / 16, P.W), vrow,
                               perm);
    if constexpr (COL) {
        uint32_t o0[2], o1[2], sb0, sb1;
        nv_col_block_codes<SMALL_S>(wd, P, Scol, rt_col, o0, o1, sb0, sb1);
        const int lrb = hd.lr0 + 16 * b;
        if (lrb < hd.Me) {
            const int64_t Mp = hd.Mp;
            const int64_t rowbytes = Mp / 2;
            const int64_t col = hd.col0 + 8 * warp + 2 * cp;
            uint8_t *d0 = P.q[0].col_data + static_cast<int64_t>(P.W) * (hd.pad_off / 2) + col * rowbytes + lrb / 2;
            stg64(d0, o0[0], o0[1]);
            stg64(d0 + rowbytes, o1[0], o1[1]);
            // col is even: column col + 1 is the next scale row (16 bytes on in the tiled layout)
            uint8_t *s0 = col_scale_ptr<16, TILED>(P, P.q[0].col_scale, hd, col, lrb / 16, P.W);
            s0[0] = static_cast<uint8_t>(sb0);
            s0[TILED ? 16 : Mp / 16] = static_cast<uint8_t>(sb1);
        }
    }
}

// Column codes of one lane's two 16-row blocks and their direct stores (blocks
// at or past the expert's end are not stored).
template <bool SMALL_S, bool TILED>
__device__ __forceinline__ void nv_col_store_pair(const uint32_t (&wd)[16], const KParams &P, const QDev &q, float S,
                                                  const float *rtab, int width, int64_t col, int lrb,
                                                  const TileHdr &hd) {
    uint32_t o0[2], o1[2], sb0, sb1;
    nv_col_block_codes<SMALL_S>(wd, P, S, rtab, o0, o1, sb0, sb1);
    if (lrb < hd.Me) {
        const int64_t Mp = hd.Mp;
        const int64_t rowbytes = Mp / 2;
        uint8_t *d0 = q.col_data + static_cast<int64_t>(width) * (hd.pad_off / 2) + col * rowbytes + lrb / 2;
        stg64(d0, o0[0], o0[1]);
        stg64(d0 + rowbytes, o1[0], o1[1]);
        uint8_t *s0 = col_scale_ptr<16, TILED>(P, q.col_scale, hd, col, lrb / 16, width);   // col even, as above
        s0[0] = static_cast<uint8_t>(sb0);
        s0[TILED ? 16 : Mp / 16] = static_cast<uint8_t>(sb1);
    }
}

template <class A, bool GLU, bool EXACT>
__device__ __forceinline__ void regen_y_words(uint32_t (&a)[16], const uint32_t (&b)[GLU ? 16 : 1], const float *pr,
                                              const ActP &ap, int nv) {
    const float4 *pq = reinterpret_cast<const float4 *>(pr);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
        const float4 p4 = pq[q4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = 4 * q4 + u;
            const float p = u == 0 ? p4.x : (u == 1 ? p4.y : (u == 2 ? p4.z : p4.w));
            uint32_t bw = 0u;
            if constexpr (GLU) bw = b[i];
            const float2 v = A::template val2p<EXACT>(a[i], bw, ap, p);
            a[i] = (i < nv) ? pack_bf16x2(v.x, v.y) : 0u;
        }
    }
}

// NVFP4 backward encode pass of the cheap activations, columnwise copies, with
// no exchange between warps: warp = 4 row blocks (64 rows) x 2 chunks (16 columns), lane = (block,
// chunk, column pair).  The four blocks read the same chunk positions of the
// TMA-swizzled tile (a 4-way bank conflict); each column's 32 code bytes of the
// four blocks are one full sector written by 4 lanes.
template <class A, class C, bool SMALL_S>
__device__ __forceinline__ void bwd_p2_cols(const KParams &P, const TileHdr &hd, const uint8_t *st, const float *pb,
                                            int warp, int lane, const ActP &ap, float Scol, const float *rt_col,
                                            float Sy, const float *rt_y) {
    const int bq = lane >> 3, k = (lane >> 2) & 1, cp = lane & 3;
    const int b = 4 * (warp >> 2) + bq;
    const int chunk = 2 * (warp & 3) + k;
    const int lrb = hd.lr0 + 16 * b;
    const int nv = hd.nrows - 16 * b;
    const int64_t col = hd.col0 + 8 * chunk + 2 * cp;
    const uint32_t base = static_cast<uint32_t>(16 * b * 128 + 4 * cp);
    const uint32_t cx = static_cast<uint32_t>(chunk) << 4;
    auto load16 = [&](const uint8_t *slot, uint32_t (&wd)[16]) {
#pragma unroll
        for (int i = 0; i < 16; ++i)
            wd[i] = lds32(slot + base + static_cast<uint32_t>(i) * 128u + (cx ^ ((static_cast<uint32_t>(i) & 7u) << 4)));
        if (nv < 16) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (i >= nv) wd[i] = 0u;
        }
    };
    if (P.q[0].col_data) {
        uint32_t wd[16];
        load16(st + C::S_DX_A * kSlotBytes, wd);
        nv_col_store_pair<SMALL_S, C::TILED_>(wd, P, P.q[0], Scol, rt_col, P.W_in, col, lrb, hd);
        if constexpr (C::GLU) {
            load16(st + C::S_DX_B * kSlotBytes, wd);
            nv_col_store_pair<SMALL_S, C::TILED_>(wd, P, P.q[0], Scol, rt_col, P.W_in, P.W + col, lrb, hd);
        }
    }
    if (C::YCOL_ && P.q[1].col_data) {
        constexpr int SXA = C::GLU ? 2 : 0;
        uint32_t av[16];
        uint32_t bv[C::GLU ? 16 : 1];
        load16(st + SXA * kSlotBytes, av);
        if constexpr (C::GLU) load16(st + (SXA + 1) * kSlotBytes, bv);
        bool exact = false;
        if constexpr (A::ranged) {
            uint32_t m = 0u;
#pragma unroll
            for (int i = 0; i < 16; ++i) m = bmax2(m, av[i]);
            exact = __any_sync(0xFFFFFFFFu, A::out_of_range(m, ap));
        }
        if (exact) regen_y_words<A, C::GLU, true>(av, bv, pb + 16 * b, ap, nv);
        else regen_y_words<A, C::GLU, false>(av, bv, pb + 16 * b, ap, nv);
        nv_col_store_pair<SMALL_S, C::TILED_>(av, P, P.q[1], Sy, rt_y, P.W, col, lrb, hd);
    }
}


template <int ACT, int RECIPE, bool BWD, bool YCOL, bool TILED>
struct Consumer {
    using C = Cfg<ACT, RECIPE, BWD, YCOL, TILED>;
    using A = Act<ACT>;

    __device__ static void run(const KParams &P, const Smem &sm) {
        const int tid = threadIdx.x;
        const int warp = tid >> 5, lane = tid & 31;
        const int r = tid >> 1, h = tid & 1;
        const ActP ap{P.s, P.s2, P.two_s, P.limit, P.alpha, P.off, P.inv_s, P.s_pow2};
        float acc[3] = {0.0f, 0.0f, 0.0f};   // P1 running amax: [0] rowwise, [1] columnwise, [2] regen columnwise
        uint32_t red_par = 0;
        int kn_e = -1;            // expert of the known columnwise maxima below
        float kn = 0.0f;          // largest columnwise value this thread computed for expert kn_e
        float kn2 = 0.0f;         // same for the regenerated Y copy (backward)
        float stk[kStackLevels] = {};
        int stage = 0;
        uint32_t phase = 0;
        for (;;) {
            if (!mbar_wait(smem_addr(sm.full(stage)), phase, P.ws, ERR_TIMEOUT_FULL)) return;
            const TileHdr hd = *sm.hdr(stage);
            if (hd.kind == K_END) return;
            uint8_t *st = sm.stage(stage);
            const bool vrow = r < hd.nrows;
            const int64_t grow = static_cast<int64_t>(hd.row0) + r;
            const float p = sm.pbuf(stage)[r];
            const int gc = hd.col0 + 32 * h;
            const int qmode = (hd.kind == K_P1) ? 1 : 0;
            const float *rt_row = nullptr, *rt_col = nullptr, *rt_y = nullptr;
            float Srow = 1.0f, Scol = 1.0f, Sy = 1.0f;
            if constexpr (RECIPE == NVFP4) {
                if (hd.kind == K_P2) {
                    const float *sv = sm.sbuf(stage);
                    Srow = sv[0];
                    Scol = sv[1];
                    Sy = sv[2];
                    const float *tb = sm.tbuf(stage);
                    rt_row = tb;
                    rt_col = tb + 128;
                    rt_y = tb + 256;
                }
            }
            if (hd.kind == K_P2 && hd.tile == 0 && hd.slab == 0 && hd.lr0 == 0 && tid == 0) {
                if (P.q[0].amax_row) P.q[0].amax_row[hd.e] = hd.amax[0];
                if (P.q[0].amax_col) P.q[0].amax_col[hd.e] = hd.amax[1];
                if (BWD && P.q[1].amax_col) P.q[1].amax_col[hd.e] = hd.amax[2];
            }

            // NVFP4 forward amax pass: directly in the column layout (warp = 16-row
            // block, lane = column pair), with no write-back of Y to shared memory.
            bool fast = false;
            if constexpr (!BWD && RECIPE == NVFP4) {
                if (hd.kind == K_P1) {
                    fast = true;
                    const uint32_t xo = ((static_cast<uint32_t>(lane) >> 2) << 4) | ((static_cast<uint32_t>(lane) & 3u) << 2);
                    const uint8_t *sa = st + 16 * warp * 128;
                    const float4 *pq = reinterpret_cast<const float4 *>(sm.pbuf(stage) + 16 * warp);
                    // staging image of (band, tile): 128 rows of 128 bytes; in the rows of 16-row
                    // block b the 16-byte chunk c sits at position c ^ b (see p2_stash_tile)
                    uint32_t *img = P.stash ? reinterpret_cast<uint32_t *>(
                                                  P.stash + (static_cast<int64_t>(hd.gband) * (P.W / kCols) + hd.col0 / kCols) * kSlotBytes +
                                                  16 * warp * 128 + ((((lane >> 2) ^ warp) & 7) << 4) + (lane & 3) * 4)
                                            : nullptr;
                    uint32_t wd[16];
                    float2 vs;
                    const int nvalid = hd.nrows - 16 * warp;
                    const bool sums = A::nonneg && hd.pnn && nvalid >= 16;
                    // a non-negative activation takes the column sums whenever the band's p are >= 0,
                    // so its remaining blocks (ragged, or some p < 0) share the general form
                    const uint32_t rm = sums ? p1_rows<A, C::GLU, true, A::nonneg>(sa, pq, xo, ap, nvalid, img, wd, vs)
                                        : ((!A::nonneg && nvalid >= 16)
                                               ? p1_rows<A, C::GLU, true, false>(sa, pq, xo, ap, nvalid, img, wd, vs)
                                               : p1_rows<A, C::GLU, false, false>(sa, pq, xo, ap, nvalid, img, wd, vs));
                    const float rmax = fmaxf(bf_lo(rm), bf_hi(rm));
                    if (P.q[0].row_data) acc[0] = fmaxf(acc[0], rmax);
                    if (P.q[0].col_data && hd.lr0 + 16 * warp < hd.Me) {
                        if (P.rht) {
                            // Upper bound of every |w| = |(H D v)_j| / 4 of the lane's blocks:
                            // sum |v| / 4, inflated for the transform's rounding and (FP32 sums) for
                            // the BF16 rounding of v; with p >= 0 a non-negative act gives Y >= 0, so the FP32
                            // column sums are the sums of |v|.
                            float bound;
                            if (sums) {
                                bound = fmaxf(vs.x, vs.y) * 0.2512f + 1e-36f;
                            } else {
                                const uint32_t t = sum_abs_pairs(wd);
                                bound = fmaxf(bf_lo(t), bf_hi(t)) * 0.255f + 1e-36f;
                            }
                            // one of the lane's two blocks holds max|v| = rmax, and |H D v / 4| of that
                            // block reaches rmax / 4 (H D / 4 orthogonal); less the transform's
                            // rounding (< 2^-20 rmax), 0.2499 rmax stays below the expert's final maximum
                            p1_col_rht_amax(wd, P, bound, rmax * 0.2499f, sm.seed(0) + hd.e,
                                            fmaxf(hd.amax[1], 0.2499f * hd.amax[0]), acc[1], lane);
                        } else {
                            acc[1] = fmaxf(acc[1], rmax);   // no transform: the columnwise values are Y itself
                        }
                    }
                } else if (hd.kind == K_P2 && P.stash) {
                    fast = true;
                    // an expert's tensor scale S above 2^100 (amax below ~2^-90) takes the exact divides
                    const bool small_s = Srow <= 0x1p100f && Scol <= 0x1p100f;
                    if (P.q[0].row_data && P.q[0].col_data) {
                        if (small_s) p2_stash_tile<true, true, true, C::TILED_>(P, hd, st, warp, lane, Srow, rt_row, Scol, rt_col);
                        else p2_stash_tile<true, true, false, C::TILED_>(P, hd, st, warp, lane, Srow, rt_row, Scol, rt_col);
                    } else if (P.q[0].row_data) {
                        p2_stash_tile<true, false, false, C::TILED_>(P, hd, st, warp, lane, Srow, rt_row, Scol, rt_col);
                    } else {
                        p2_stash_tile<false, true, false, C::TILED_>(P, hd, st, warp, lane, Srow, rt_row, Scol, rt_col);
                    }
                }
            }
            if constexpr (C::COL_OWN) {
                // encode pass: rowwise codes per thread, columnwise codes per warp (no CTA barrier)
                if (hd.kind == K_P2) {
                    fast = true;
                    if (vrow && P.q[0].row_data) {
                        uint32_t w[16];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint4 v = lds128(st + C::S_DX_A * kSlotBytes + swz_chunk(r, 4 * h + k));
                            w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
                        }
                        row_pass<RECIPE, C::TILED_>(P, hd, P.q[0], w, grow, gc, P.W_in, 0, Srow, rt_row, acc[0]);
                        if constexpr (C::GLU) {
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const uint4 v = lds128(st + C::S_DX_B * kSlotBytes + swz_chunk(r, 4 * h + k));
                                w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
                            }
                            row_pass<RECIPE, C::TILED_>(P, hd, P.q[0], w, grow, P.W + gc, P.W_in, 0, Srow, rt_row, acc[0]);
                        }
                    }
                    const float *pb = sm.pbuf(stage);
                    if (fmaxf(Srow, fmaxf(Scol, Sy)) <= 0x1p100f)
                        bwd_p2_cols<A, C, true>(P, hd, st, pb, warp, lane, ap, Scol, rt_col, Sy, rt_y);
                    else
                        bwd_p2_cols<A, C, false>(P, hd, st, pb, warp, lane, ap, Scol, rt_col, Sy, rt_y);
                }
            }
            if (!fast) {
                // ---------------- step A: thread = (row r, 32-column half h)
                if constexpr (!BWD) {
                    uint32_t yw[16];
                    if (hd.kind == K_P2 && P.stash) {
                        // encode pass: Y comes back from the staging copy (an L2 hit), no activation
    #pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t off = swz_chunk(r, 4 * h + k);
                            uint4 y4 = lds128(st + off);
                            if (!vrow) {
                                y4 = make_uint4(0, 0, 0, 0);
                                sts128(st + off, 0, 0, 0, 0);
                            }
                            yw[4 * k] = y4.x; yw[4 * k + 1] = y4.y; yw[4 * k + 2] = y4.z; yw[4 * k + 3] = y4.w;
                        }
                        if (h == 0) {
                            // row r of the staging image (128 bytes, written for every row) is dead
                            // after this read
                            const uint8_t *line = P.stash +
                                                  (static_cast<int64_t>(hd.gband) * (P.W / kCols) + hd.col0 / kCols) * kSlotBytes +
                                                  r * 128;
                            asm volatile("discard.global.L2 [%0], 128;" ::"l"(line) : "memory");
                        }
                    } else {
    #pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t off = swz_chunk(r, 4 * h + k);
                            const uint4 a4 = lds128(st + off);
                            uint4 b4 = make_uint4(0, 0, 0, 0);
                            if constexpr (C::GLU) b4 = lds128(st + kSlotBytes + off);
                            const uint32_t aw[4] = {a4.x, a4.y, a4.z, a4.w};
                            const uint32_t bw[4] = {b4.x, b4.y, b4.z, b4.w};
                            float2 v4[4];
                            if (need_exact4<A>(aw, ap)) {
    #pragma unroll
                                for (int j = 0; j < 4; ++j) v4[j] = A::template val2p<true>(aw[j], bw[j], ap, p);
                            } else {
    #pragma unroll
                                for (int j = 0; j < 4; ++j) v4[j] = A::template val2p<false>(aw[j], bw[j], ap, p);
                            }
    #pragma unroll
                            for (int j = 0; j < 4; ++j) yw[4 * k + j] = vrow ? pack_bf16x2(v4[j].x, v4[j].y) : 0u;
                            sts128(st + off, yw[4 * k], yw[4 * k + 1], yw[4 * k + 2], yw[4 * k + 3]);
                        }
                    }
                    if (vrow) {
                        if (P.y_bf16 && hd.kind != K_P1) {
                            uint16_t *dst = P.y_bf16 + grow * P.W + gc;
    #pragma unroll
                            for (int k = 0; k < 4; ++k)
                                stg128(dst + 8 * k, yw[4 * k], yw[4 * k + 1], yw[4 * k + 2], yw[4 * k + 3]);
                        }
                        if (P.q[0].row_data) row_pass<RECIPE, C::TILED_>(P, hd, P.q[0], yw, grow, gc, P.W, qmode, Srow, rt_row, acc[0]);
                    }
                } else if (hd.kind != K_P2) {
                    const bool regen = P.q[1].col_data != nullptr;
                    // MXFP8 encodes each row's 32-value block after the loop; NVFP4 only
                    // needs the running rowwise amax here, so it keeps no block in registers.
                    constexpr bool kKeep = (RECIPE == MXFP8);
                    uint32_t dxa[kKeep ? 16 : 4], dxb[kKeep ? 16 : 4];
                    uint32_t rmax = 0u;
                    uint16_t *dst = P.dx_bf16 ? P.dx_bf16 + grow * P.W_in + gc : nullptr;
                    const bool row_amax = !kKeep && vrow && P.q[0].row_data != nullptr && qmode == 1;
                    float bsum = 0.0f;
    #pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t off = swz_chunk(r, 4 * h + k);
                        const uint4 a4 = lds128(st + off);
                        uint4 b4 = make_uint4(0, 0, 0, 0);
                        if constexpr (C::GLU) b4 = lds128(st + kSlotBytes + off);
                        const uint4 d4 = lds128(st + C::S_DY * kSlotBytes + off);
                        const uint32_t aw[4] = {a4.x, a4.y, a4.z, a4.w};
                        const uint32_t bw[4] = {b4.x, b4.y, b4.z, b4.w};
                        const uint32_t dw[4] = {d4.x, d4.y, d4.z, d4.w};
                        uint32_t xa4[4], xb4[4], y4[4];
                        // ranged activations: one warp vote per four words picks the fast or exact form
                        float2 v4[4], da4[4], db4[4];
                        if constexpr (A::ranged) {
                            if (need_exact4<A>(aw, ap)) {
    #pragma unroll
                                for (int j = 0; j < 4; ++j) A::template grad2<true>(aw[j], bw[j], ap, v4[j], da4[j], db4[j]);
                            } else {
    #pragma unroll
                                for (int j = 0; j < 4; ++j) A::template grad2<false>(aw[j], bw[j], ap, v4[j], da4[j], db4[j]);
                            }
                        }
    #pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            float2 v, da, db;
                            if constexpr (A::ranged) {
                                v = v4[j];
                                da = da4[j];
                                db = db4[j];
                            } else {
                                A::template grad2<false>(aw[j], bw[j], ap, v, da, db);
                            }
                            const float2 d = make_float2(bf_lo(dw[j]), bf_hi(dw[j]));
                            const float2 g = __fmul2_rn(d, make_float2(p, p));
                            const float2 xa = __fmul2_rn(g, da);
                            xa4[j] = vrow ? pack_bf16x2(xa.x, xa.y) : 0u;
                            if constexpr (C::GLU) {
                                const float2 xb = __fmul2_rn(g, db);
                                xb4[j] = vrow ? pack_bf16x2(xb.x, xb.y) : 0u;
                            }
                            const float2 tm = __fmul2_rn(d, v);   // dprobs terms, summed in column order
                            bsum = bsum + tm.x;
                            bsum = bsum + tm.y;
                            if (regen) {
                                const float2 yv = __fmul2_rn(v, make_float2(p, p));
                                y4[j] = vrow ? pack_bf16x2(yv.x, yv.y) : 0u;
                            }
                        }
                        sts128(st + C::S_DX_A * kSlotBytes + off, xa4[0], xa4[1], xa4[2], xa4[3]);
                        if constexpr (C::GLU) sts128(st + C::S_DX_B * kSlotBytes + off, xb4[0], xb4[1], xb4[2], xb4[3]);
                        if (regen) sts128(st + C::S_Y * kSlotBytes + off, y4[0], y4[1], y4[2], y4[3]);
                        if (vrow && dst) {
                            stg128_wb(dst + 8 * k, xa4[0], xa4[1], xa4[2], xa4[3]);
                            if constexpr (C::GLU) stg128_wb(dst + P.W + 8 * k, xb4[0], xb4[1], xb4[2], xb4[3]);
                        }
                        if constexpr (kKeep) {
    #pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                dxa[4 * k + j] = xa4[j];
                                if constexpr (C::GLU) dxb[4 * k + j] = xb4[j];
                            }
                        } else if (row_amax) {
    #pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                rmax = babsmax2(rmax, xa4[j]);
                                if constexpr (C::GLU) rmax = babsmax2(rmax, xb4[j]);
                            }
                        }
                    }
                    if constexpr (kKeep) {
                        if (vrow && P.q[0].row_data) {
                            row_pass<RECIPE, C::TILED_>(P, hd, P.q[0], dxa, grow, gc, P.W_in, qmode, Srow, rt_row, acc[0]);
                            if constexpr (C::GLU) row_pass<RECIPE, C::TILED_>(P, hd, P.q[0], dxb, grow, P.W + gc, P.W_in, qmode, Srow, rt_row, acc[0]);
                        }
                    } else if (row_amax) {
                        rmax &= 0x7FFF7FFFu;
                        acc[0] = fmaxf(acc[0], fmaxf(bf_lo(rmax), bf_hi(rmax)));
                    }
                    if (P.dprobs) {
                        // pair of 32-blocks (2t, 2t+1) of this tile, then the in-slab binary-counter merge
                        float node = bsum + __shfl_xor_sync(0xFFFFFFFFu, bsum, 1);
                        const int t = hd.tile;
    #pragma unroll
                        for (int i = 0; i < kStackLevels; ++i) {
                            if ((t >> i) & 1) {
                                node = stk[i] + node;
                            } else {
                                stk[i] = node;
                                break;
                            }
                        }
                    }
                } else {
                    // NVFP4 backward encode pass: dX from the dense copy, Y recomputed on request
                    uint32_t dxa[16], dxb[16];
    #pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t off = swz_chunk(r, 4 * h + k);
                        uint4 a4 = lds128(st + C::S_DX_A * kSlotBytes + off);
                        if (!vrow) {
                            a4 = make_uint4(0, 0, 0, 0);
                            sts128(st + C::S_DX_A * kSlotBytes + off, 0, 0, 0, 0);
                        }
                        dxa[4 * k] = a4.x; dxa[4 * k + 1] = a4.y; dxa[4 * k + 2] = a4.z; dxa[4 * k + 3] = a4.w;
                        if constexpr (C::GLU) {
                            uint4 b4 = lds128(st + C::S_DX_B * kSlotBytes + off);
                            if (!vrow) {
                                b4 = make_uint4(0, 0, 0, 0);
                                sts128(st + C::S_DX_B * kSlotBytes + off, 0, 0, 0, 0);
                            }
                            dxb[4 * k] = b4.x; dxb[4 * k + 1] = b4.y; dxb[4 * k + 2] = b4.z; dxb[4 * k + 3] = b4.w;
                        }
                    }
                    if (vrow && P.q[0].row_data) {
                        row_pass<RECIPE, C::TILED_>(P, hd, P.q[0], dxa, grow, gc, P.W_in, 0, Srow, rt_row, acc[0]);
                        if constexpr (C::GLU) row_pass<RECIPE, C::TILED_>(P, hd, P.q[0], dxb, grow, P.W + gc, P.W_in, 0, Srow, rt_row, acc[0]);
                    }
                    if (P.q[1].col_data) {
                        constexpr int SXA = C::GLU ? 2 : 0;
    #pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const uint32_t off = swz_chunk(r, 4 * h + k);
                            const uint4 a4 = lds128(st + SXA * kSlotBytes + off);
                            uint4 b4 = make_uint4(0, 0, 0, 0);
                            if constexpr (C::GLU) b4 = lds128(st + 3 * kSlotBytes + off);
                            const uint32_t aw[4] = {a4.x, a4.y, a4.z, a4.w};
                            const uint32_t bw[4] = {b4.x, b4.y, b4.z, b4.w};
                            uint32_t y4[4];
                            float2 v4[4];
                            if (need_exact4<A>(aw, ap)) {
    #pragma unroll
                                for (int j = 0; j < 4; ++j) v4[j] = A::template val2p<true>(aw[j], bw[j], ap, p);
                            } else {
    #pragma unroll
                                for (int j = 0; j < 4; ++j) v4[j] = A::template val2p<false>(aw[j], bw[j], ap, p);
                            }
    #pragma unroll
                            for (int j = 0; j < 4; ++j) y4[j] = vrow ? pack_bf16x2(v4[j].x, v4[j].y) : 0u;
                            sts128(st + C::S_Y * kSlotBytes + off, y4[0], y4[1], y4[2], y4[3]);
                        }
                    }
                }
                // Step B of warp w reads only rows that step A of the same warp wrote
                // (NVFP4: one 16-row block) or of warps w and w^1 (MXFP8: one 32-row block).
                if constexpr (RECIPE == NVFP4) __syncwarp();
                else pair_sync(warp >> 1);

                // ---------------- step B: warp = row block, lane = column pair
                const int cmode = (hd.kind == K_P1) ? 1 : 0;
            if (BWD && hd.kind == K_P1 && hd.e != kn_e) {
                kn_e = hd.e;
                kn = kn2 = 0.0f;
            }
                if constexpr (!BWD) {
                    if (P.q[0].col_data)
                        col_pass<RECIPE, C::TILED_>(P, hd, st, P.q[0], 0, P.W, cmode, Scol, rt_col, acc[1], warp, lane, hd.amax[1]);
                } else {
                    if (P.q[0].col_data) {
                        col_pass<RECIPE, C::TILED_>(P, hd, st + C::S_DX_A * kSlotBytes, P.q[0], 0, P.W_in, cmode, Scol, rt_col, acc[1],
                                         warp, lane, fmaxf(hd.amax[1], kn));
                        if constexpr (C::GLU)
                            col_pass<RECIPE, C::TILED_>(P, hd, st + C::S_DX_B * kSlotBytes, P.q[0], P.W, P.W_in, cmode, Scol, rt_col, acc[1],
                                             warp, lane, fmaxf(hd.amax[1], kn));
                        kn = fmaxf(kn, acc[1]);
                    }
                    if (P.q[1].col_data) {
                        col_pass<RECIPE, C::TILED_>(P, hd, st + C::S_Y * kSlotBytes, P.q[1], 0, P.W, cmode, Sy, rt_y, acc[2], warp,
                                         lane, fmaxf(hd.amax[2], kn2));
                        kn2 = fmaxf(kn2, acc[2]);
                    }
                }
            }
            if constexpr (RECIPE == NVFP4) {
                // encode pass: store the columnwise codes every warp staged in its slot region
                // (the forward's staging-image path stores its columnwise codes directly)
                if (hd.kind == K_P2 && (P.q[0].col_data || (BWD && P.q[1].col_data)) && (BWD || !P.stash) &&
                    !C::COL_OWN) {
                    named_sync();
                    if constexpr (!BWD) {
                        nv_col_flush<C::TILED_>(P, st, P.q[0], 0, P.W, hd, tid);
                    } else {
                        if (P.q[0].col_data) {
                            nv_col_flush<C::TILED_>(P, st + C::S_DX_A * kSlotBytes, P.q[0], 0, P.W_in, hd, tid);
                            if constexpr (C::GLU) nv_col_flush<C::TILED_>(P, st + C::S_DX_B * kSlotBytes, P.q[0], P.W, P.W_in, hd, tid);
                        }
                        if (P.q[1].col_data) nv_col_flush<C::TILED_>(P, st + C::S_Y * kSlotBytes, P.q[1], 0, P.W, hd, tid);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(sm.empty(stage)));
            if (++stage == C::STAGES) {
                stage = 0;
                phase ^= 1u;
            }

            // ---------------- item epilogue
            if (hd.tile == P.tiles_per_slab - 1) {
                const bool need_dp = BWD && hd.kind != K_P2 && P.dprobs != nullptr;
                const bool multi = need_dp && P.n_slabs > 1;
                if (need_dp && h == 0 && vrow) {
                    const int lvl = 31 - __clz(P.tiles_per_slab);   // tiles_per_slab is a power of two
                    float node = stk[0];
#pragma unroll
                    for (int i = 1; i < kStackLevels; ++i)
                        if (i == lvl) node = stk[i];
                    if (P.n_slabs == 1) P.dprobs[grow] = node;
                    else P.partial[grow * P.n_slabs + hd.slab] = node;
                }
                if (hd.kind == K_P1 || multi) {
                    // per-warp partial amax, double-buffered: warps may reach the next
                    // item's reduction while thread 0 still reads this one
                    float *red = sm.red() + 24 * (red_par & 1);
                    if (hd.kind == K_P1) {
                        ++red_par;
#pragma unroll
                        for (int k = 0; k < 3; ++k) {
                            float v = acc[k];
#pragma unroll
                            for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
                            if (lane == 0) red[warp * 3 + k] = v;
                            acc[k] = 0.0f;
                        }
                    }
                    // Every consumer's stores of this item (dense dX, dprobs partials)
                    // precede the barrier; thread 0 then publishes them device-wide with
                    // a fence before it bumps the counters others acquire.
                    named_sync();
                    if (tid == 0) {
                        __threadfence();
                        if (hd.kind == K_P1) {
                            uint32_t *amax_ws = P.ws + WS_HDR + P.E;
                            for (int k = 0; k < 3; ++k) {
                                float v = 0.0f;
                                for (int w = 0; w < 8; ++w) v = fmaxf(v, red[w * 3 + k]);
                                atomicMax(amax_ws + 3 * hd.e + k, __float_as_uint(v));
                            }
                            __threadfence();
                            atomicAdd(P.ws + WS_HDR + hd.e, 1u);
                        }
                        if (multi) {
                            uint32_t *band_cnt = P.ws + WS_HDR + 5 * P.E;
                            const uint32_t old = atomicAdd(band_cnt + hd.gband, 1u);
                            const int last = (old == static_cast<uint32_t>(P.n_slabs - 1)) ? 1 : 0;
                            if (last) __threadfence();   // acquire the other slabs' partials
                            *sm.flag() = last;
                        }
                    }
                    if (multi) {
                        named_sync();
                        if (*sm.flag() && h == 0 && vrow) {
                            float buf[kMaxSlabs];
                            int n = P.n_slabs;
                            for (int i = 0; i < n; ++i) buf[i] = __ldcg(P.partial + grow * P.n_slabs + i);
                            while (n > 1) {
                                const int half = n >> 1;
                                for (int j = 0; j < half; ++j) buf[j] = buf[2 * j] + buf[2 * j + 1];
                                if (n & 1) buf[half] = buf[n - 1];
                                n = half + (n & 1);
                            }
                            P.dprobs[grow] = buf[0];
                        }
                    }
                }
            }
        }
    }
};

template <int ACT, int RECIPE, bool BWD, bool YCOL, bool TILED>
__global__ void __launch_bounds__(kThreads, Cfg<ACT, RECIPE, BWD, YCOL, TILED>::CTAS) gsa_kernel(const __grid_constant__ KParams P) {
    using C = Cfg<ACT, RECIPE, BWD, YCOL, TILED>;
    const Smem sm = carve<C>();
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(smem_addr(sm.full(s)), 1);
            mbar_init(smem_addr(sm.empty(s)), kCons / 32);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if constexpr (RECIPE == NVFP4)
        for (int i = threadIdx.x; i < 2 * kMaxExperts; i += kThreads) sm.seed(0)[i] = 0u;
    if (RECIPE == NVFP4 && blockIdx.x == 0 && threadIdx.x < 32) {
        // experts without rows never get an encode item: report amax 0 for them
        for (int e = threadIdx.x; e < P.E; e += 32) {
            if (plan_of(P).row_off[e + 1] != plan_of(P).row_off[e]) continue;
            if (P.q[0].amax_row) P.q[0].amax_row[e] = 0.0f;
            if (P.q[0].amax_col) P.q[0].amax_col[e] = 0.0f;
            if (BWD && P.q[1].amax_col) P.q[1].amax_col[e] = 0.0f;
        }
    }
    __syncthreads();
    if (threadIdx.x >= kCons) {
        producer<C>(P, sm, threadIdx.x - kCons);
        return;
    }
    Consumer<ACT, RECIPE, BWD, YCOL, TILED>::run(P, sm);
}

// Launch (grid > 0) or occupancy query (grid == 0: *ctas_per_sm receives the
// resident CTAs per SM) of one variant.  Defined once per activation.
template <int ACT, int RECIPE, bool BWD, bool YCOL, bool TILED>
cudaError_t launch_variant(const KParams &P, int grid, cudaStream_t stream, int *ctas_per_sm) {
    using C = Cfg<ACT, RECIPE, BWD, YCOL, TILED>;
    auto *k = gsa_kernel<ACT, RECIPE, BWD, YCOL, TILED>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    static int configured[64] = {0};
    static int occupancy[64] = {0};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (err != cudaSuccess) return err;
        int n = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kThreads, C::SMEM);
        if (err != cudaSuccess) return err;
        occupancy[dev] = n;
        configured[dev] = 1;
    }
    if (grid == 0) {
        *ctas_per_sm = occupancy[dev];
        return cudaSuccess;
    }
    k<<<grid, kThreads, C::SMEM, stream>>>(P);
    return cudaGetLastError();
}

typedef cudaError_t (*launch_fn)(int recipe, bool bwd, const KParams &P, int grid, cudaStream_t stream,
                                 int *ctas_per_sm);

// The variant of one call: recipe and direction; the NVFP4 backward of a costly
// activation takes the variant without the regenerated copy of Y when the call
// does not request it; the scale layout picks the TILED instantiations.
template <int ACT, bool TILED>
cudaError_t launch_layout(int recipe, bool bwd, const KParams &P, int grid, cudaStream_t stream, int *ctas_per_sm) {
    if (recipe == MXFP8)
        return bwd ? launch_variant<ACT, MXFP8, true, true, TILED>(P, grid, stream, ctas_per_sm)
                   : launch_variant<ACT, MXFP8, false, true, TILED>(P, grid, stream, ctas_per_sm);
    if (!bwd) return launch_variant<ACT, NVFP4, false, true, TILED>(P, grid, stream, ctas_per_sm);
    if constexpr (!Cfg<ACT, NVFP4, true>::CHEAP) {
        if (P.q[1].col_data == nullptr) return launch_variant<ACT, NVFP4, true, false, TILED>(P, grid, stream, ctas_per_sm);
    }
    return launch_variant<ACT, NVFP4, true, true, TILED>(P, grid, stream, ctas_per_sm);
}

#define GSA_DEFINE_ACT(ACT, NAME)                                                                         \
    cudaError_t launch_##NAME(int recipe, bool bwd, const KParams &P, int grid, cudaStream_t stream,     \
                              int *ctas_per_sm) {                                                         \
        return P.scale_tiled ? launch_layout<ACT, true>(recipe, bwd, P, grid, stream, ctas_per_sm)       \
                             : launch_layout<ACT, false>(recipe, bwd, P, grid, stream, ctas_per_sm);     \
    }

cudaError_t launch_srelu(int, bool, const KParams &, int, cudaStream_t, int *);
cudaError_t launch_tanh_srelu(int, bool, const KParams &, int, cudaStream_t, int *);
cudaError_t launch_swiglu(int, bool, const KParams &, int, cudaStream_t, int *);
cudaError_t launch_clamped_swiglu(int, bool, const KParams &, int, cudaStream_t, int *);
cudaError_t launch_gelu(int, bool, const KParams &, int, cudaStream_t, int *);
cudaError_t launch_sigmoid(int, bool, const KParams &, int, cudaStream_t, int *);
cudaError_t launch_identity(int, bool, const KParams &, int, cudaStream_t, int *);

}  // namespace gsa
