// The hot path: a persistent, warp-specialised TMA pipeline that moves boxes
// between global memory and a ring of shared-memory stages.
//
//   warp 0, lane 0  producer: for its k-th box, waits until stage k mod N is
//                   free, arms the stage's "full" mbarrier with
//                   arrive.expect_tx(box_bytes) and issues one bulk copy into
//                   it (a tensor-map load, or a 1-D bulk load of a packed
//                   image).
//   warp 1          consumer: waits on the stage's phase, then lane 0 issues
//                   the drain (a tensor-map store, or a 1-D bulk store of the
//                   image), commits it as a bulk async group and, once
//                   wait_group.read shows the group has finished reading the
//                   stage, arrives on the stage's "empty" mbarrier.  Boxes a
//                   tensor store may not write (a negative origin, or a ragged
//                   row end) are written by the whole warp with plain clipped
//                   stores, and their stages are freed at once.
//
// tile_wide_kernel runs the same ring with four consumer warps, for the fp32
// update and for launches that write listed boxes into a tensor.
//
// Sources: "lesson 04: TMA - the async bulk copy engine" ("What the issuing
// thread actually does", "Load completion - the mbarrier and the byte budget",
// "Store completion - commit group and wait group", "Why this only pays off
// inside a pipeline"); "GPU TMA tensor memory accelerator" ("The architecture:
// every piece explained": warp specialisation and the multi-stage ring);
// "Day 76: The Tensor Memory Accelerator (TMA)" ("An exact round trip",
// "Exercise", "Hint 2", "Pitfalls"); "Understanding TMA loads in CuTe DSL"
// ("Initialize the barrier before using it", "Issue the load and wait for its
// phase": parity starts at 0 and flips on every reuse of a barrier).
//
// Every mbarrier wait is bounded by the global timer.  On expiry the kernel
// records ATB_ERR_TIMEOUT in the device status block, tells the other role to
// stop through a shared flag, waits (again bounded) for the copies it already
// started, and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "atb_internal.h"
#include "ptx.cuh"

namespace atb {
namespace {

enum Mode : int { kRoundtrip = 0, kLoad = 1, kStore = 2, kRoundtripAddF32 = 3 };

struct PipeArgs {
    const int32_t* coords;  // n_tiles * rank origins, or null for the tile grid
    uint8_t* packed;        // kLoad: destination images; kStore: source images
    DeviceStatus* status;
    uint8_t* dst_base;      // destination tensor (plain stores)
    const uint8_t* src_base;  // source tensor (plain loads of boxes the engine may not start)
    uint64_t timeout_ns;
    uint64_t dst_dims[ATB_MAX_RANK];
    uint64_t dst_strides[ATB_MAX_RANK];
    uint64_t src_dims[ATB_MAX_RANK];
    uint64_t src_strides[ATB_MAX_RANK];
    uint32_t fill[4];       // one 16-byte chunk of out-of-bounds fill (zero bytes, or the NaN pattern)
    uint32_t wide_box0;     // box[0] of the one-chunk-wider map, 0 = none
    uint32_t wide_pitch;    // bytes of one row of its image
    uint32_t wide_bytes;    // bytes of its image
    uint32_t grid[ATB_MAX_RANK];  // boxes along each dimension (tile grid)
    uint32_t box[ATB_MAX_RANK];
    uint32_t visits[ATB_MAX_RANK];  // elements a box visits per dimension: ceil(box / step)
    uint32_t step[ATB_MAX_RANK];    // traversal step per dimension
    uint32_t n_tiles;       // boxes in this launch
    uint32_t tile_begin;    // index of its first box in the list or grid
    uint32_t esize;
    uint32_t box_bytes;
    uint32_t stage_bytes;
    uint32_t stages;
    uint32_t store_lag;     // groups left reading after each commit
    uint32_t early_release; // one-thread drain: free a stage before the next store
    uint32_t contiguous;    // 1: CTA b takes a contiguous run of boxes
    uint32_t swizzle_bits;  // 0 none, 1 32B, 2 64B, 3 128B
    uint32_t dst_ragged_x;  // destination rows end inside a 16-byte chunk
    uint32_t l2_hints;      // ATB_HINT_* bits
    uint32_t suspend_ns;    // mbarrier poll suspend-time hint, 0 = hardware default
    uint32_t prefetch;      // boxes ahead to prefetch into L2 (tensor loads), 0 = off
    uint32_t checks;        // ATB_CHECK_* bits
};

// Shared-memory control words after the stage ring and the barriers.
struct Control {
    uint32_t abort;
    uint32_t issued;         // boxes whose stage the producer has armed
    uint32_t producer_done;
    uint32_t pad;
    // ATB_CHECK_RING shadows, per stage: 1 + the CTA-local number of the box
    // the producer last armed it for, and 1 + (the number of the box the
    // consumer last released it from, modulo 256); 0 = not used yet.
    uint32_t filled[kMaxStages];
    uint32_t freed[kMaxStages];
    // Listed boxes: the origin of the box each stage holds, written by the
    // producer before it arms the stage, so that consumers never read the
    // coordinate list in global memory.
    int32_t origin[kMaxStages][ATB_MAX_RANK];
};

__device__ __forceinline__ void record_error(DeviceStatus* st, int32_t code, int32_t tile, int32_t where)
{
    atomicAdd(&st->errors, 1u);
    if (atomicCAS(&st->code, 0, code) == 0) {
        st->block = static_cast<int32_t>(blockIdx.x);
        st->tile = tile;
        st->where = where;
    }
}

// Waits for the phase of `bar` with the given parity for at most `timeout_ns`.
// Returns false on expiry or, when `abort` is non-null, once another role
// has raised it.  The timer is read only after the first poll fails.
// Each poll may suspend the thread until the phase completes (for a
// hardware-chosen time, or at most `suspend_ns` when that is non-zero).
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                             const volatile uint32_t* abort, uint32_t suspend_ns = 0)
{
    auto poll = [&]() {
        return suspend_ns ? ptx::mbar_try_wait_suspend(bar, parity, suspend_ns) : ptx::mbar_try_wait(bar, parity);
    };
    if (poll()) return true;
    const uint64_t t0 = ptx::global_timer_ns();
    for (;;) {
        if (poll()) return true;
        if (abort && *abort) return false;
        if (ptx::global_timer_ns() - t0 > timeout_ns) return false;
    }
}

// Same, against an absolute deadline of the global timer.
__device__ __forceinline__ bool wait_until(uint32_t bar, uint32_t parity, uint64_t deadline)
{
    for (;;) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (ptx::global_timer_ns() > deadline) return false;
    }
}

// Box t -> CTA-local iteration and back.
__device__ __forceinline__ uint32_t my_tile_count(const PipeArgs& a)
{
    const uint32_t G = gridDim.x, b = blockIdx.x;
    if (a.contiguous) {
        const uint32_t per = (a.n_tiles + G - 1) / G;
        const uint64_t lo = static_cast<uint64_t>(b) * per;
        if (lo >= a.n_tiles) return 0;
        const uint64_t hi = lo + per < a.n_tiles ? lo + per : a.n_tiles;
        return static_cast<uint32_t>(hi - lo);
    }
    return b < a.n_tiles ? (a.n_tiles - b + G - 1) / G : 0;
}

// Index (in the list or grid) of this CTA's k-th box.
__device__ __forceinline__ uint32_t tile_of(const PipeArgs& a, uint32_t k)
{
    if (a.contiguous) return a.tile_begin + blockIdx.x * ((a.n_tiles + gridDim.x - 1) / gridDim.x) + k;
    return a.tile_begin + blockIdx.x + k * gridDim.x;
}

// Origin of box t, innermost first: from the list, or from the row-major tile
// grid (innermost tile index fastest).
template <int R>
__device__ __forceinline__ void tile_origin(const PipeArgs& a, uint32_t t, int32_t (&c)[R])
{
    if (a.coords) {
        const int32_t* p = a.coords + static_cast<size_t>(t) * R;
#pragma unroll
        for (int d = 0; d < R; ++d) c[d] = __ldg(p + d);
    } else {
        uint32_t rest = t;
#pragma unroll
        for (int d = 0; d < R - 1; ++d) {
            const uint32_t q = rest / a.grid[d];
            c[d] = static_cast<int32_t>((rest - q * a.grid[d]) * a.box[d]);
            rest = q;
        }
        c[R - 1] = static_cast<int32_t>(rest * a.box[R - 1]);
    }
}

// Walks one CTA's boxes in order with additions only: the ring stage and the
// parity of its current use, the box's index in the list or grid and, for the
// grid, its tile coordinates.  The step between consecutive boxes (gridDim.x,
// or 1 for contiguous runs) is kept in the grid's mixed radix and added digit
// by digit, with at most one carry per dimension.
template <int R>
struct BoxCursor {
    uint32_t stage = 0;
    uint32_t parity = 0;
    uint32_t t = 0;   // index in the list or grid
    uint32_t g[R];    // tile coordinates (grid)
    uint32_t dg[R];   // the step, digit by digit

    __device__ __forceinline__ void init(const PipeArgs& a)
    {
        t = tile_of(a, 0);
        uint32_t rest = t, rstep = a.contiguous ? 1u : gridDim.x;
#pragma unroll
        for (int d = 0; d < R - 1; ++d) {
            g[d] = rest % a.grid[d];
            rest /= a.grid[d];
            dg[d] = rstep % a.grid[d];
            rstep /= a.grid[d];
        }
        g[R - 1] = rest;
        dg[R - 1] = rstep;
    }

    __device__ __forceinline__ void origin(const PipeArgs& a, int32_t (&c)[R]) const
    {
        if (a.coords) {
            const int32_t* p = a.coords + static_cast<size_t>(t) * R;
#pragma unroll
            for (int d = 0; d < R; ++d) c[d] = __ldg(p + d);
        } else {
            grid_origin(a, c);
        }
    }

    // The origin of the current box of the tile grid.
    __device__ __forceinline__ void grid_origin(const PipeArgs& a, int32_t (&c)[R]) const
    {
#pragma unroll
        for (int d = 0; d < R; ++d) c[d] = static_cast<int32_t>(g[d] * a.box[d]);
    }

    __device__ __forceinline__ void advance(const PipeArgs& a, uint32_t stages)
    {
        if (++stage == stages) {
            stage = 0;
            parity ^= 1u;
        }
        step(a);
    }

    // To the next box: its index and tile coordinates only.
    __device__ __forceinline__ void step(const PipeArgs& a)
    {
        t += a.contiguous ? 1u : gridDim.x;
        uint32_t carry = 0;
#pragma unroll
        for (int d = 0; d < R - 1; ++d) {
            g[d] += dg[d] + carry;
            carry = g[d] >= a.grid[d] ? 1u : 0u;
            if (carry) g[d] -= a.grid[d];
        }
        g[R - 1] += dg[R - 1] + carry;
    }
};

// The origin of a CTA's current box of the tile grid, stepped by additions
// only: the step between consecutive boxes (gridDim.x boxes, or one for
// contiguous runs) is kept per dimension in elements, and every coordinate
// but the outermost wraps at most once per step.  The host runs this walk only
// where every grid extent but the outermost is at most 2^31 elements, so no
// sum overflows.  INDEX = true also keeps the box's index.
template <int R, bool INDEX>
struct GridWalk {
    uint32_t c[R];   // origin, elements
    uint32_t dc[R];  // the step, per dimension, in elements
    uint32_t t = 0;  // index in the grid (INDEX)

    __device__ __forceinline__ void init(const PipeArgs& a)
    {
        const uint32_t t0 = tile_of(a, 0);
        if (INDEX) t = t0;
        uint32_t rest = t0, rstep = a.contiguous ? 1u : gridDim.x;
#pragma unroll
        for (int d = 0; d < R - 1; ++d) {
            c[d] = rest % a.grid[d] * a.box[d];
            rest /= a.grid[d];
            dc[d] = rstep % a.grid[d] * a.box[d];
            rstep /= a.grid[d];
        }
        c[R - 1] = rest * a.box[R - 1];
        dc[R - 1] = rstep * a.box[R - 1];
    }

    __device__ __forceinline__ void step(const PipeArgs& a)
    {
        if (INDEX) t += a.contiguous ? 1u : gridDim.x;
        bool carry = false;
#pragma unroll
        for (int d = 0; d < R - 1; ++d) {
            c[d] += dc[d] + (carry ? a.box[d] : 0u);
            const uint32_t extent = a.grid[d] * a.box[d];
            carry = c[d] >= extent;
            if (carry) c[d] -= extent;
        }
        c[R - 1] += dc[R - 1] + (carry ? a.box[R - 1] : 0u);
    }

    __device__ __forceinline__ const int32_t* origin() const { return reinterpret_cast<const int32_t*>(c); }
};

// A listed origin the engine must not be given: beyond +-2^30 along any
// dimension.  Such a box is refused (recorded, not moved).
template <int R>
__device__ __forceinline__ int32_t origin_error(const PipeArgs& a, const int32_t (&c)[R])
{
    if (!a.coords) return 0;
#pragma unroll
    for (int d = 0; d < R; ++d)
        if (c[d] > (1 << 30) || c[d] < -(1 << 30)) return ATB_ERR_COORD_RANGE;
    return 0;
}

// A tensor-map copy must start on a 16-byte boundary along the contiguous
// dimension: x * element size a multiple of 16.  Tile-grid origins always
// are (the box row is a multiple of 16 bytes); a listed origin off that grid
// is moved by the consumer threads instead, with plain loads and stores.
template <int R>
__device__ __forceinline__ bool off_grid(const PipeArgs& a, const int32_t (&c)[R])
{
    return ((static_cast<uint32_t>(c[0]) * a.esize) & 15u) != 0;
}

// How a box gets into its stage: one engine copy through the map (the origin
// is on the 16-byte grid); one engine copy through the one-chunk-wider map
// from the origin rounded down to the grid (off the grid, the map has one);
// plain loads by the consumer threads (off the grid, no wider map); or not at
// all (a refused origin).
enum LoadKind : int { kLoadEngine = 0, kLoadWide = 1, kLoadThreads = 2, kLoadRefused = 3 };

template <int R>
__device__ __forceinline__ int load_kind(const PipeArgs& a, const int32_t (&c)[R])
{
    if (origin_error<R>(a, c)) return kLoadRefused;
    if (!off_grid<R>(a, c)) return kLoadEngine;
    return a.wide_box0 ? kLoadWide : kLoadThreads;
}

// x * element size mod 16: how far a box row starts past a 16-byte boundary.
template <int R>
__device__ __forceinline__ uint32_t row_phase(const PipeArgs& a, const int32_t (&c)[R])
{
    return (static_cast<uint32_t>(c[0]) * a.esize) & 15u;
}

enum StoreKind : int { kStoreTensor = 0, kStorePlain = 1, kStoreNothing = 2 };

// How a box reaches the destination tensor: nothing when it misses the tensor
// entirely; plain stores when it starts before the tensor (a tensor store may
// not start at a negative coordinate), when its x origin is off the 16-byte
// grid, or when it crosses the end of a row whose byte length is not a
// multiple of 16 (the engine writes such a row's last 16-byte chunk whole,
// past the row's end); a tensor store otherwise.
template <int R>
__device__ __forceinline__ int store_kind(const PipeArgs& a, const int32_t (&c)[R])
{
    bool plain = false;
#pragma unroll
    for (int d = 0; d < R; ++d) {
        if (static_cast<int64_t>(c[d]) >= static_cast<int64_t>(a.dst_dims[d]) ||
            static_cast<int64_t>(c[d]) + a.box[d] <= 0)
            return kStoreNothing;
        if (c[d] < 0) plain = true;
    }
    if (a.dst_ragged_x && static_cast<int64_t>(c[0]) + a.box[0] > static_cast<int64_t>(a.dst_dims[0])) plain = true;
    if (off_grid<R>(a, c)) plain = true;
    return plain ? kStorePlain : kStoreTensor;
}

// Bytes rb .. rb + 15 of the 32 little-endian bytes A then B (rb in 0..15).
__device__ __forceinline__ uint4 bytes_from_pair(const uint4& A, const uint4& B, uint32_t rb)
{
    const uint32_t w[8] = {A.x, A.y, A.z, A.w, B.x, B.y, B.z, B.w};
    const uint32_t s = rb >> 2, sh = 8 * (rb & 3u);
    uint32_t t[5];
#pragma unroll
    for (int i = 0; i < 5; ++i) t[i] = s == 0 ? w[i] : s == 1 ? w[i + 1] : s == 2 ? w[i + 2] : w[i + 3];
    return make_uint4(__funnelshift_r(t[0], t[1], sh), __funnelshift_r(t[1], t[2], sh),
                      __funnelshift_r(t[2], t[3], sh), __funnelshift_r(t[3], t[4], sh));
}

// Bytes 4 S + b / 8 ... of the 32 bytes A then B (b = 8 x the shift's byte
// part, 0..24), for a shift whose word part S is known at compile time: four
// funnel shifts and no selects.
template <int S>
__device__ __forceinline__ uint4 shift_pair(const uint4& A, const uint4& B, uint32_t b)
{
    const uint32_t w[8] = {A.x, A.y, A.z, A.w, B.x, B.y, B.z, B.w};
    return make_uint4(__funnelshift_r(w[S], w[S + 1], b), __funnelshift_r(w[S + 1], w[S + 2], b),
                      __funnelshift_r(w[S + 2], w[S + 3], b), __funnelshift_r(w[S + 3], w[S + 4], b));
}

// Keeps bytes [lo, hi) of v (0 <= lo <= hi <= 16) and puts the fill's bytes
// elsewhere.  Element boundaries are multiples of the element size and the
// fill repeats every element, so the result is whole elements of either.
__device__ __forceinline__ uint4 keep_bytes(const uint4& v, const uint4& fill, uint32_t lo, uint32_t hi)
{
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const uint32_t f[4] = {fill.x, fill.y, fill.z, fill.w};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int32_t a = static_cast<int32_t>(lo) - 4 * i, b = static_cast<int32_t>(hi) - 4 * i;
        const uint32_t from = a <= 0 ? 0u : a >= 4 ? 32u : 8u * a;  // first kept bit
        const uint32_t to = b <= 0 ? 0u : b >= 4 ? 32u : 8u * b;    // one past the last kept bit
        const uint32_t below_to = to >= 32 ? 0xFFFFFFFFu : (1u << to) - 1u;
        const uint32_t below_from = from >= 32 ? 0xFFFFFFFFu : (1u << from) - 1u;
        const uint32_t m = below_to & ~below_from;
        out[i] = (w[i] & m) | (f[i] & ~m);
    }
    return make_uint4(out[0], out[1], out[2], out[3]);
}

// Gathers one box image into a stage with plain loads, for a box whose x
// origin is off the 16-byte grid; `nthreads` threads, 16-byte image chunks.
// Chunk (row, column j) holds elements x0 = c0 + j q ... x0 + q - 1 (q = 16 /
// element size) of that box row and lands at its swizzled place in the stage
// (the swizzle moves whole 16-byte chunks).  It is read as the two aligned
// 16-byte words of the row that cover it, shifted into place.  A word is read
// only when it holds at least one byte of the row, so it lies in the memory
// page of that byte; elements outside the row (a chunk cut by the row's start
// or end) then take the fill value, and a row outside the tensor is all fill.
// Threads are laid out as `group` rows of `cols` columns and each issues the
// loads of four rows before it stores any of them, so one memory latency is
// paid per four rows.
template <int R>
__device__ void thread_load_box(const PipeArgs& a, const int32_t (&c)[R], uint32_t stage, uint32_t tid,
                                uint32_t nthreads)
{
    constexpr int U = 4;
    const uint32_t es = a.esize;
    const uint32_t row_bytes = a.box[0] * es;  // the innermost step is always 1
    const uint32_t cpr = row_bytes / 16;
    const uint32_t rows1 = R > 1 ? a.visits[1] : 1;
    const uint32_t planes = a.box_bytes / (row_bytes * rows1);
    const uint32_t q = 16 / es;
    const uint32_t rb = (static_cast<uint32_t>(c[0]) * es) & 15u;
    const uint32_t line_mask = (1u << a.swizzle_bits) - 1u;
    const int64_t dims0 = static_cast<int64_t>(a.src_dims[0]);
    const int64_t dims1 = R > 1 ? static_cast<int64_t>(a.src_dims[1]) : 1;
    const uint64_t stride1 = R > 1 ? a.src_strides[1] : 0;
    const int64_t step1 = R > 1 ? a.step[1] : 0;
    const int64_t c1 = R > 1 ? c[1] : 0;
    const uint4 fill = make_uint4(a.fill[0], a.fill[1], a.fill[2], a.fill[3]);
    const uint32_t cols = cpr < nthreads ? cpr : nthreads;
    const uint32_t group = nthreads / cols;
    const uint32_t first_row = tid / cols;
    if (first_row >= group) return;  // threads beyond group * cols have no chunk
    const uint32_t j0 = tid - first_row * cols;

    for (uint32_t plane = 0; plane < planes; ++plane) {
        uint32_t rest = plane;
        bool plane_in = true;
        uint64_t plane_off = 0;
#pragma unroll
        for (int d = 2; d < R; ++d) {
            const uint32_t k = rest % a.visits[d];
            rest /= a.visits[d];
            const int64_t g = static_cast<int64_t>(c[d]) + static_cast<int64_t>(k) * a.step[d];
            if (g < 0 || g >= static_cast<int64_t>(a.src_dims[d])) plane_in = false;
            else plane_off += static_cast<uint64_t>(g) * a.src_strides[d];
        }
        for (uint32_t j = j0; j < cpr; j += cols) {
            const int64_t x0 = static_cast<int64_t>(c[0]) + static_cast<int64_t>(j) * q;
            // bytes of the chunk inside the row, and the row bytes of its two aligned words
            const int64_t xb = x0 * static_cast<int64_t>(es);  // row byte of the chunk's first element
            const int64_t row_end = dims0 * static_cast<int64_t>(es);
            const int64_t lo_b = xb < 0 ? -xb : 0;
            const int64_t hi_b = row_end - xb < 16 ? row_end - xb : 16;
            const bool any_x = lo_b < hi_b;
            const int64_t wa = xb - static_cast<int64_t>(rb);  // first aligned word (row bytes)
            const bool load_a = any_x && wa >= 0 && wa < row_end;
            const bool load_b = any_x && rb != 0 && wa + 16 >= 0 && wa + 16 < row_end;
            const uint32_t keep_lo = any_x ? static_cast<uint32_t>(lo_b) : 16u;
            const uint32_t keep_hi = any_x ? static_cast<uint32_t>(hi_b) : 16u;
            for (uint32_t k1 = first_row; k1 < rows1; k1 += U * group) {
                uint4 A[U], B[U];
                bool row_in[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint32_t kk = k1 + u * group;
                    const int64_t g1 = c1 + static_cast<int64_t>(kk) * step1;
                    row_in[u] = plane_in && kk < rows1 && g1 >= 0 && g1 < dims1;
                    A[u] = make_uint4(0, 0, 0, 0);
                    B[u] = make_uint4(0, 0, 0, 0);
                    if (row_in[u]) {
                        const uint8_t* row = a.src_base + plane_off + static_cast<uint64_t>(g1) * stride1;
                        if (load_a) A[u] = ptx::ld_global_nc_v4(row + wa);
                        if (load_b) B[u] = ptx::ld_global_nc_v4(row + wa + 16);
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const uint32_t kk = k1 + u * group;
                    if (kk >= rows1) continue;
                    const uint32_t o = (plane * rows1 + kk) * row_bytes + 16 * j;
                    const uint32_t dst = stage + (o ^ (((o >> 7) & line_mask) << 4));
                    uint4 v = fill;
                    if (row_in[u]) {
                        v = bytes_from_pair(A[u], B[u], rb);
                        if (keep_lo != 0 || keep_hi != 16) v = keep_bytes(v, fill, keep_lo, keep_hi);
                    }
                    ptx::st_shared_v4_u32(dst, v);
                }
            }
        }
    }
}

// Clipped store of one box image whose x origin is on the 16-byte grid (every
// tile-grid box, and listed boxes on that grid) from shared memory by
// `nthreads` threads, 16 bytes at a time.  The swizzle moves whole 16-byte chunks (the chunk
// number, bits 4..6 of the image offset, is XORed with the low swizzle bits of
// the 128-byte line number, bits 7..9), and a box row starts on a 16-byte
// boundary in both spaces (the origin's x is 16-byte aligned, strides are
// multiples of 16), so a chunk that lies wholly inside the tensor moves as one
// vector; only a chunk cut by the end of a row moves element by element.
//
// Threads are laid out as `group` rows of `cpr` chunks (or, for rows wider
// than the thread count, one row at a time).  The box is walked plane by plane
// (dimensions 2..R-1, decomposed once per plane) and, inside a plane, row by
// row along dimension 1 with additions only: in the warp consumer a single
// warp runs this loop alone, so short dependency chains matter more than
// instruction counts.
template <int R>
__device__ void plain_store_grid_box(const PipeArgs& a, const int32_t (&c)[R], uint32_t stage, uint32_t tid,
                                uint32_t nthreads)
{
    const uint32_t row_bytes = a.box[0] * a.esize;  // the innermost step is always 1
    const uint32_t cpr = row_bytes / 16;             // 16-byte chunks per row
    const uint32_t rows = a.box_bytes / row_bytes;
    const uint32_t group = cpr < nthreads ? nthreads / cpr : 1;  // rows in flight per pass
    const uint32_t jstep = cpr < nthreads ? cpr : nthreads;
    const uint32_t first_row = tid / cpr;
    if (first_row >= group) return;  // threads beyond group * cpr have no chunk
    const uint32_t j0 = tid - first_row * cpr;
    const uint32_t q = 16 / a.esize;  // elements per chunk
    const uint32_t line_mask = (1u << a.swizzle_bits) - 1u;
    const int64_t dims0 = static_cast<int64_t>(a.dst_dims[0]);
    const uint32_t rows1 = R > 1 ? a.visits[1] : 1;  // rows per plane
    const uint32_t planes = rows / rows1;
    const int64_t dims1 = R > 1 ? static_cast<int64_t>(a.dst_dims[1]) : 1;
    const int64_t gstep1 = R > 1 ? static_cast<int64_t>(group) * a.step[1] : 0;
    const uint64_t stride1 = R > 1 ? a.dst_strides[1] : 0;

    // One 16-byte column per thread (the usual case: a row fits in the thread
    // group): the column's x offset, bounds and swizzle-free part are fixed,
    // so each row costs a bounds check, two address additions and the copy.
    const bool one_column = cpr <= nthreads;
    const int64_t xc = static_cast<int64_t>(c[0]) + static_cast<int64_t>(j0) * q;
    if (one_column && (xc < 0 || xc >= dims0)) return;  // this column lies outside every row
    const bool xc_whole = xc + q <= dims0;

    for (uint32_t plane = 0; plane < planes; ++plane) {
        uint32_t rest = plane;
        bool inside = true;
        uint64_t plane_addr = 0;
#pragma unroll
        for (int d = 2; d < R; ++d) {
            const uint32_t k = rest % a.visits[d];
            rest /= a.visits[d];
            const int64_t g = static_cast<int64_t>(c[d]) + static_cast<int64_t>(k) * a.step[d];
            if (g < 0 || g >= static_cast<int64_t>(a.dst_dims[d])) inside = false;
            else plane_addr += static_cast<uint64_t>(g) * a.dst_strides[d];
        }
        if (!inside) continue;
        int64_t g1 = R > 1 ? static_cast<int64_t>(c[1]) + static_cast<int64_t>(first_row) * a.step[1] : 0;
        uint32_t o_row = (plane * rows1 + first_row) * row_bytes;
        if (one_column) {
            uint8_t* col = a.dst_base + plane_addr + static_cast<uint64_t>(xc) * a.esize;
            const uint32_t row_step = group * row_bytes;
#pragma unroll 4
            for (uint32_t k1 = first_row; k1 < rows1; k1 += group, g1 += gstep1, o_row += row_step) {
                if (g1 < 0 || g1 >= dims1) continue;
                const uint32_t o = o_row + 16 * j0;
                const uint32_t src = stage + (o ^ (((o >> 7) & line_mask) << 4));
                uint8_t* dst = col + static_cast<uint64_t>(g1) * stride1;
                if (xc_whole) {
                    *reinterpret_cast<uint4*>(dst) = ptx::ld_shared_v4_u32(src);
                } else {
                    for (uint32_t b = 0; b < static_cast<uint32_t>(dims0 - xc) * a.esize; ++b)
                        dst[b] = ptx::ld_shared_u8(src + b);
                }
            }
            continue;
        }
        for (uint32_t k1 = first_row; k1 < rows1; k1 += group, g1 += gstep1, o_row += group * row_bytes) {
            if (g1 < 0 || g1 >= dims1) continue;
            const uint64_t addr = plane_addr + static_cast<uint64_t>(g1) * stride1;
            for (uint32_t j = j0; j < cpr; j += jstep) {
                const int64_t x0 = static_cast<int64_t>(c[0]) + static_cast<int64_t>(j) * q;
                if (x0 < 0 || x0 >= dims0) continue;
                const uint32_t o = o_row + 16 * j;
                const uint32_t src = stage + (o ^ (((o >> 7) & line_mask) << 4));
                uint8_t* dst = a.dst_base + addr + static_cast<uint64_t>(x0) * a.esize;
                if (x0 + q <= dims0) {
                    *reinterpret_cast<uint4*>(dst) = ptx::ld_shared_v4_u32(src);
                } else {
                    for (uint32_t b = 0; b < static_cast<uint32_t>(dims0 - x0) * a.esize; ++b)
                        dst[b] = ptx::ld_shared_u8(src + b);
                }
            }
        }
    }
}

// Where a plain store finds the box in shared memory: the box image (rows of
// box[0] elements, swizzled like the map), or the one-chunk-wider unswizzled
// image that the wider map loads from the origin rounded down to the grid.
enum StoreSource : int { kFromImage = 0, kFromWide = 1 };

// A box whose first row byte is off the 16-byte grid, written into the
// tensor with aligned stores of U bytes.  U (1, 2 or 4) is the largest power
// of two up to 4 that divides both that row byte and the tensor row's byte
// length, so every U-byte unit lies wholly inside or wholly outside the
// tensor and no store reaches a byte outside the box.  Each consumer warp
// takes whole box rows and its lanes the row's units: one store instruction
// writes 32 U contiguous bytes of a row.  A unit's place in the stage follows
// from its byte offset in the row: in the box image (swizzled like the map)
// or in the wider unswizzled image, where the box's row starts rb bytes in.
constexpr uint32_t kRowsInFlight = 4;

template <int R, uint32_t U>
__device__ void store_units(const PipeArgs& a, const int32_t (&c)[R], uint32_t stage, int source, uint32_t tid,
                            uint32_t nthreads)
{
    const uint32_t es = a.esize;
    const uint32_t row_bytes = a.box[0] * es;  // the innermost step is always 1
    const uint32_t upr = row_bytes / U;        // units per box row
    const uint32_t rows1 = R > 1 ? a.visits[1] : 1;
    uint32_t planes = 1;
#pragma unroll
    for (int d = 2; d < R; ++d) planes *= a.visits[d];
    const uint32_t pitch = source == kFromWide ? a.wide_pitch : row_bytes;
    const uint32_t src0 = source == kFromWide ? row_phase<R>(a, c) : 0u;
    const uint32_t line_mask = source == kFromWide ? 0u : (1u << a.swizzle_bits) - 1u;
    const int64_t gx0 = static_cast<int64_t>(c[0]) * es;
    const int64_t row_end = static_cast<int64_t>(a.dst_dims[0]) * es;
    const int64_t dims1 = R > 1 ? static_cast<int64_t>(a.dst_dims[1]) : 1;
    const uint64_t stride1 = R > 1 ? a.dst_strides[1] : 0;
    const uint32_t warp = tid >> 5, lane = tid & 31, nwarps = nthreads >> 5;

    for (uint32_t plane = 0; plane < planes; ++plane) {
        uint32_t rest = plane;
        bool inside = true;
        uint64_t plane_addr = 0;
#pragma unroll
        for (int d = 2; d < R; ++d) {
            const uint32_t k = planes == 1 ? 0u : rest % a.visits[d];
            if (planes != 1) rest /= a.visits[d];
            const int64_t g = static_cast<int64_t>(c[d]) + static_cast<int64_t>(k) * a.step[d];
            if (g < 0 || g >= static_cast<int64_t>(a.dst_dims[d])) inside = false;
            else plane_addr += static_cast<uint64_t>(g) * a.dst_strides[d];
        }
        if (!inside) continue;
        uint8_t* const plane_dst = a.dst_base + plane_addr;
        const uint32_t plane_off = plane * rows1 * pitch + src0;
        // kRowsInFlight rows of the warp at a time: their shared loads are all
        // issued before the first global store (one load latency per batch).
        if (upr <= 32) {  // one unit per lane: its place in the row is fixed for the box
            const uint32_t k = lane;
            const int64_t x = gx0 + static_cast<int64_t>(k * U);
            const bool x_in = k < upr && x >= 0 && x < row_end;
            const uint32_t o_k = plane_off + k * U;
            for (uint32_t k1 = warp; k1 < rows1; k1 += kRowsInFlight * nwarps) {
                uint32_t v[kRowsInFlight];
                uint8_t* dst[kRowsInFlight];
                bool in[kRowsInFlight];
#pragma unroll
                for (uint32_t u = 0; u < kRowsInFlight; ++u) {
                    const uint32_t kk = k1 + u * nwarps;
                    const int64_t g1 = R > 1 ? static_cast<int64_t>(c[1]) + static_cast<int64_t>(kk) * a.step[1] : 0;
                    in[u] = x_in && kk < rows1 && g1 >= 0 && g1 < dims1;
                    dst[u] = plane_dst + static_cast<uint64_t>(in[u] ? g1 : 0) * stride1 + x;
                    const uint32_t o = o_k + kk * pitch;
                    const uint32_t p = stage + (o ^ (((o >> 7) & line_mask) << 4));
                    v[u] = 0;
                    if (in[u]) v[u] = U == 4 ? ptx::ld_shared_u32(p) : U == 2 ? ptx::ld_shared_u16(p) : ptx::ld_shared_u8(p);
                }
#pragma unroll
                for (uint32_t u = 0; u < kRowsInFlight; ++u) {
                    if (!in[u]) continue;
                    if (U == 4) *reinterpret_cast<uint32_t*>(dst[u]) = v[u];
                    else if (U == 2) *reinterpret_cast<uint16_t*>(dst[u]) = static_cast<uint16_t>(v[u]);
                    else *dst[u] = static_cast<uint8_t>(v[u]);
                }
            }
            continue;
        }
        for (uint32_t k1 = warp; k1 < rows1; k1 += kRowsInFlight * nwarps) {
            for (uint32_t k = lane; k < upr; k += 32) {
                const int64_t x = gx0 + static_cast<int64_t>(k * U);
                const bool x_in = x >= 0 && x < row_end;
                uint32_t v[kRowsInFlight];
                uint8_t* dst[kRowsInFlight];
                bool in[kRowsInFlight];
#pragma unroll
                for (uint32_t u = 0; u < kRowsInFlight; ++u) {
                    const uint32_t kk = k1 + u * nwarps;
                    const int64_t g1 = R > 1 ? static_cast<int64_t>(c[1]) + static_cast<int64_t>(kk) * a.step[1] : 0;
                    in[u] = x_in && kk < rows1 && g1 >= 0 && g1 < dims1;
                    dst[u] = plane_dst + static_cast<uint64_t>(in[u] ? g1 : 0) * stride1 + x;
                    const uint32_t o = plane_off + kk * pitch + k * U;
                    const uint32_t p = stage + (o ^ (((o >> 7) & line_mask) << 4));
                    v[u] = 0;
                    if (in[u]) v[u] = U == 4 ? ptx::ld_shared_u32(p) : U == 2 ? ptx::ld_shared_u16(p) : ptx::ld_shared_u8(p);
                }
#pragma unroll
                for (uint32_t u = 0; u < kRowsInFlight; ++u) {
                    if (!in[u]) continue;
                    if (U == 4) *reinterpret_cast<uint32_t*>(dst[u]) = v[u];
                    else if (U == 2) *reinterpret_cast<uint16_t*>(dst[u]) = static_cast<uint16_t>(v[u]);
                    else *dst[u] = static_cast<uint8_t>(v[u]);
                }
            }
        }
    }
}

template <int R>
__device__ __forceinline__ void store_off_grid_box(const PipeArgs& a, const int32_t (&c)[R], uint32_t stage,
                                                   int source, uint32_t tid, uint32_t nthreads)
{
    const uint32_t bits = static_cast<uint32_t>(c[0]) * a.esize | a.dst_dims[0] * a.esize | 4u;
    switch (bits & (~bits + 1u)) {  // the lowest set bit: 1, 2 or 4
    case 1: store_units<R, 1>(a, c, stage, source, tid, nthreads); break;
    case 2: store_units<R, 2>(a, c, stage, source, tid, nthreads); break;
    default: store_units<R, 4>(a, c, stage, source, tid, nthreads); break;
    }
}

// A gather's packed image of a box that the wider map loaded: image chunk
// (row, j) is bytes rb + 16 j ... rb + 16 j + 15 of the wider row, shifted
// out of two aligned chunks, and goes to its swizzled place in the box's slot
// of the packed buffer.  `nthreads` threads as `group` rows of `cols` chunks;
// the shift is the same for the whole box, and its word part S is fixed at
// compile time (pack_from_wide dispatches once per box).
template <int R, int S>
__device__ void pack_from_wide_s(const PipeArgs& a, uint32_t rb, uint32_t stage, uint8_t* slot, uint32_t tid,
                                 uint32_t nthreads)
{
    const uint32_t row_bytes = a.box[0] * a.esize;
    const uint32_t cpr = row_bytes / 16;
    const uint32_t rows = a.box_bytes / row_bytes;
    const uint32_t line_mask = (1u << a.swizzle_bits) - 1u;
    const uint32_t bits = 8 * (rb & 3u);
    const uint32_t cols = cpr < nthreads ? cpr : nthreads;
    const uint32_t group = nthreads / cols;
    const uint32_t first_row = tid / cols;
    if (first_row >= group) return;
    const uint32_t j0 = tid - first_row * cols;
    // one row at a time: two rows in flight took the kernel over its register
    // budget (spills) and measured 13 % slower
    for (uint32_t j = j0; j < cpr; j += cols) {
        for (uint32_t r = first_row; r < rows; r += group) {
            const uint32_t w = stage + r * a.wide_pitch + 16 * j;
            const uint4 A = ptx::ld_shared_v4_u32(w);
            const uint4 B = ptx::ld_shared_v4_u32(w + 16);
            const uint32_t o = r * row_bytes + 16 * j;
            *reinterpret_cast<uint4*>(slot + (o ^ (((o >> 7) & line_mask) << 4))) = shift_pair<S>(A, B, bits);
        }
    }
}

template <int R>
__device__ void pack_from_wide(const PipeArgs& a, const int32_t (&c)[R], uint32_t stage, uint8_t* slot, uint32_t tid,
                               uint32_t nthreads)
{
    const uint32_t rb = row_phase<R>(a, c);
    switch (rb >> 2) {
    case 0: pack_from_wide_s<R, 0>(a, rb, stage, slot, tid, nthreads); break;
    case 1: pack_from_wide_s<R, 1>(a, rb, stage, slot, tid, nthreads); break;
    case 2: pack_from_wide_s<R, 2>(a, rb, stage, slot, tid, nthreads); break;
    default: pack_from_wide_s<R, 3>(a, rb, stage, slot, tid, nthreads); break;
    }
}

// Shared-memory layout of one CTA: the stage ring (aligned to the swizzle
// period), full[] and empty[] mbarriers, then the control words.
struct Ring {
    uint32_t base;      // shared address of stage 0
    uint8_t* base_ptr;  // generic pointer to stage 0
    uint32_t stages;
    uint32_t stage_bytes;
    uint32_t full0;     // full[s]  at full0 + 8 s
    uint32_t empty0;    // empty[s] at empty0 + 8 s
    Control* ctl;

    __device__ uint32_t stage(uint32_t s) const { return base + s * stage_bytes; }
    __device__ uint32_t full(uint32_t s) const { return full0 + 8 * s; }
    __device__ uint32_t empty(uint32_t s) const { return empty0 + 8 * s; }
    __device__ volatile uint32_t* abort_flag() const { return &ctl->abort; }
};

// A CTA's walk round the ring: the current stage's index and the parity of
// its current use; the stage's and its barriers' shared addresses follow from
// the index.
struct StageWalk {
    uint32_t s = 0, parity = 0;

    __device__ __forceinline__ void next(const Ring& r)
    {
        if (++s == r.stages) {
            s = 0;
            parity ^= 1u;
        }
    }
};

__device__ __forceinline__ Ring ring_layout(const PipeArgs& a, uint8_t* smem_raw)
{
    Ring r;
    const uint32_t raw = ptx::smem_addr(smem_raw);
    r.base = (raw + (kStageAlignSwizzled - 1)) & ~(kStageAlignSwizzled - 1);
    r.base_ptr = smem_raw + (r.base - raw);
    r.stages = a.stages;
    r.stage_bytes = a.stage_bytes;
    r.full0 = r.base + a.stages * a.stage_bytes;
    r.empty0 = r.full0 + 8 * a.stages;
    r.ctl = reinterpret_cast<Control*>(r.base_ptr + a.stages * a.stage_bytes + 16 * a.stages);
    return r;
}

// Thread 0 initialises every barrier (one arrival each) and publishes the
// initialisation to the async proxy; the caller follows with a block barrier.
__device__ __forceinline__ void init_ring(const Ring& r)
{
    for (uint32_t s = 0; s < r.stages; ++s) {
        ptx::mbar_init(r.full(s), 1);
        ptx::mbar_init(r.empty(s), 1);
    }
    r.ctl->abort = 0;
    r.ctl->issued = 0;
    r.ctl->producer_done = 0;
    for (uint32_t s = 0; s < r.stages; ++s) {
        r.ctl->filled[s] = 0;
        r.ctl->freed[s] = 0;
    }
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
}

__device__ __forceinline__ void raise_abort(const PipeArgs& a, const Ring& r, uint32_t tile, int32_t where)
{
    if (!*r.abort_flag()) {
        record_error(a.status, ATB_ERR_TIMEOUT, static_cast<int32_t>(tile), where);
        *r.abort_flag() = 1;
    }
}

// ATB_CHECK_RING: the releasing consumer thread records which box it is done
// with before arriving on the stage's empty barrier (whose release order
// publishes the write to the producer's acquiring wait) ...
__device__ __forceinline__ void ring_note_freed(const PipeArgs& a, const Ring& r, uint32_t stage, uint32_t box)
{
    if (a.checks & ATB_CHECK_RING)
        *reinterpret_cast<volatile uint32_t*>(&r.ctl->freed[stage]) = (box & 255u) + 1u;
}

// ... and the producer, after that wait, checks it was the stage's previous box.
__device__ __forceinline__ void ring_check_freed(const PipeArgs& a, const Ring& r, uint32_t stage, uint32_t k,
                                                 uint32_t tile)
{
    if (!(a.checks & ATB_CHECK_RING) || k < r.stages) return;
    const uint32_t want = ((k - r.stages) & 255u) + 1u;
    if (*reinterpret_cast<volatile uint32_t*>(&r.ctl->freed[stage]) != want)
        record_error(a.status, ATB_ERR_RING_CHECK, static_cast<int32_t>(tile), kWhereProducerRing);
}

// After its full-barrier wait, the consumer checks the stage holds its k-th box.
__device__ __forceinline__ void ring_check_filled(const PipeArgs& a, const Ring& r, uint32_t stage, uint32_t k,
                                                  uint32_t tile)
{
    if ((a.checks & ATB_CHECK_RING) && *reinterpret_cast<volatile uint32_t*>(&r.ctl->filled[stage]) != k + 1u)
        record_error(a.status, ATB_ERR_RING_CHECK, static_cast<int32_t>(tile), kWhereConsumerRing);
}

// Origin of the box that landed in stage s: from the cursor for the tile grid,
// from the stage's origin slot for listed boxes.  Read after the stage's
// full-barrier wait, which orders it after the producer's write.
template <int R>
__device__ __forceinline__ void landed_origin(const PipeArgs& a, const Ring& r, uint32_t s, const BoxCursor<R>& cur,
                                              int32_t (&c)[R])
{
    if (a.coords) {
        const volatile int32_t* slot = r.ctl->origin[s];
#pragma unroll
        for (int d = 0; d < R; ++d) c[d] = slot[d];
    } else {
        cur.origin(a, c);
    }
}

// One producer thread: for its k-th box, wait until stage k mod N is free,
// arm the stage's full barrier with the box's byte count and issue the copy.
// A listed box whose x origin is off the 16-byte grid gets a plain arrival
// instead: the consumer threads load it themselves.  LISTED = false compiles
// the coordinate-list handling out (tile-grid launches).
template <int MODE, int R, bool LISTED>
__device__ void producer_loop(const PipeArgs& a, const CUtensorMap& src_map, const CUtensorMap& wide_map,
                              const Ring& r, uint32_t count)
{
    const bool hint = (a.l2_hints & ATB_HINT_LOAD_EVICT_FIRST) != 0;
    const uint64_t policy = hint ? ptx::policy_evict_first() : 0;
    const uint32_t S = r.stages;
    const bool listed = LISTED && a.coords != nullptr;
    if (MODE != kStore && a.prefetch) {  // warm L2 with the first boxes
        for (uint32_t k = 0; k < a.prefetch && k < count; ++k) {
            int32_t c[R];
            tile_origin<R>(a, tile_of(a, k), c);
            if (!listed || (!origin_error<R>(a, c) && !off_grid<R>(a, c))) ptx::tma_prefetch_l2<R>(&src_map, c);
        }
    }
    BoxCursor<R> cur;
    cur.init(a);
    for (uint32_t k = 0; k < count; ++k, cur.advance(a, S)) {
        const uint32_t s = cur.stage;
        if (MODE != kStore && a.prefetch && k + a.prefetch < count) {
            int32_t c[R];
            tile_origin<R>(a, tile_of(a, k + a.prefetch), c);
            if (!listed || (!origin_error<R>(a, c) && !off_grid<R>(a, c))) ptx::tma_prefetch_l2<R>(&src_map, c);
        }
        // The origin first: for listed boxes it is a load from the coordinate
        // list, whose latency then overlaps the wait for the stage.
        int32_t c[R];
        if (listed) cur.origin(a, c);
        else cur.grid_origin(a, c);
        // the stage's previous use completed the empty phase of the other parity
        if (k >= S && !wait_bounded(r.empty(s), cur.parity ^ 1u, a.timeout_ns, r.abort_flag(), a.suspend_ns)) {
            raise_abort(a, r, cur.t, kWhereProducerWait);
            break;
        }
        const uint32_t t = cur.t;
        ring_check_freed(a, r, s, k, t);
        if (a.checks & ATB_CHECK_RING)  // published by the arrive below (release order)
            *reinterpret_cast<volatile uint32_t*>(&r.ctl->filled[s]) = k + 1u;
        if (listed) {  // hand the origin over with the stage (published by the arrive below)
            volatile int32_t* slot = r.ctl->origin[s];
#pragma unroll
            for (int d = 0; d < R; ++d) slot[d] = c[d];
        }
        const int32_t bad = listed ? origin_error<R>(a, c) : 0;
        if (bad) {
            record_error(a.status, bad, static_cast<int32_t>(t), kWhereProducerIssue);
            ptx::mbar_arrive(r.full(s));  // completes the phase with no bytes; consumers skip the box
        } else if (MODE != kStore && listed && off_grid<R>(a, c)) {
            if (a.wide_box0) {
                // the wider box from the origin rounded down to the 16-byte grid
                int32_t cw[R];
#pragma unroll
                for (int d = 0; d < R; ++d) cw[d] = c[d];
                cw[0] -= static_cast<int32_t>(row_phase<R>(a, c) / a.esize);
                ptx::mbar_arrive_expect_tx(r.full(s), a.wide_bytes);
                ptx::tma_load<R>(r.stage(s), &wide_map, cw, r.full(s));
            } else {
                ptx::mbar_arrive(r.full(s));  // completes the phase with no bytes; consumers load the box
            }
        } else {
            ptx::mbar_arrive_expect_tx(r.full(s), a.box_bytes);
            if (MODE == kStore)
                ptx::bulk_load(r.stage(s), a.packed + static_cast<size_t>(t) * a.box_bytes, a.box_bytes, r.full(s));
            else if (hint)
                ptx::tma_load_hint<R>(r.stage(s), &src_map, c, r.full(s), policy);
            else
                ptx::tma_load<R>(r.stage(s), &src_map, c, r.full(s));
        }
        *reinterpret_cast<volatile uint32_t*>(&r.ctl->issued) = k + 1;
    }
    *reinterpret_cast<volatile uint32_t*>(&r.ctl->producer_done) = 1;
}

// After a failed wait at box k: stop the producer, then wait (bounded) for
// every load it already started so that no copy lands in shared memory after
// the CTA exits.  Called by one thread, after bulk_wait_all().  The drain has
// its own budget of at least one second, so that a very short wait limit
// still leaves time for copies that are merely slow.
constexpr uint64_t kMinDrainNs = 1000000000ull;

__device__ void drain_after_failure(const PipeArgs& a, const Ring& r, uint32_t k)
{
    raise_abort(a, r, tile_of(a, k), kWhereConsumerWait);
    const uint64_t deadline = ptx::global_timer_ns() + (a.timeout_ns > kMinDrainNs ? a.timeout_ns : kMinDrainNs);
    while (!*reinterpret_cast<volatile uint32_t*>(&r.ctl->producer_done) && ptx::global_timer_ns() < deadline) {
    }
    const uint32_t issued = *reinterpret_cast<volatile uint32_t*>(&r.ctl->issued);
    for (uint32_t j = k; j < issued; ++j) wait_until(r.full(j % r.stages), (j / r.stages) & 1, deadline);
}

// Store groups that may still be reading their stages, oldest first: the
// stage index (4 bits, stages <= 16) and the consumer's box counter modulo 256
// (8 bits) of each, at most 8 in flight.  Only boxes the engine stores have a
// group; a box written by threads, or dropped, frees its stage as soon as its
// readers are done.  After every box k, each group started at least `lag`
// boxes earlier is retired, so a stage is always free again by the time the
// producer comes back to it (lag < stages).
struct PendingStores {
    uint64_t stages = 0;
    uint64_t boxes = 0;
    uint32_t count = 0;

    __device__ __forceinline__ void push(uint32_t stage, uint32_t box)
    {
        stages |= static_cast<uint64_t>(stage) << (4 * count);
        boxes |= static_cast<uint64_t>(box & 255u) << (8 * count);
        ++count;
    }

    __device__ __forceinline__ void retire(const PipeArgs& a, const Ring& r, uint32_t k, uint32_t lag)
    {
        uint32_t keep = 0;  // groups younger than `lag` boxes may stay in flight
        for (uint32_t i = 0; i < count; ++i)
            if (((k - static_cast<uint32_t>((boxes >> (8 * i)) & 255u)) & 255u) < lag) ++keep;
        if (keep == count) return;
        ptx::bulk_wait_read_le(keep);
        for (; count > keep; --count) {
            ring_note_freed(a, r, static_cast<uint32_t>(stages & 15u), static_cast<uint32_t>(boxes & 255u));
            ptx::mbar_arrive(r.empty(static_cast<uint32_t>(stages & 15u)));
            stages >>= 4;
            boxes >>= 8;
        }
    }
};

// The one-thread drain's producer: one thread walks the CTA's boxes of the
// tile grid, waits until each box's stage is free, arms the stage's full
// barrier with the box's byte count and issues the box's load (a tensor load,
// or a 1-D bulk load of a packed image for stores).  OPTS = false compiles the
// ring check and the L2 hint out.
template <int MODE, int R, bool OPTS>
__device__ __forceinline__ void grid_producer(const PipeArgs& a, const CUtensorMap& src_map, const Ring& r,
                                              uint32_t count)
{
    const bool hint = OPTS && (a.l2_hints & ATB_HINT_LOAD_EVICT_FIRST) != 0;
    const uint64_t policy = hint ? ptx::policy_evict_first() : 0;
    const bool check = OPTS && (a.checks & ATB_CHECK_RING) != 0;
    const uint32_t S = r.stages, bytes = a.box_bytes;
    volatile uint32_t* issued = &r.ctl->issued;
    GridWalk<R, MODE == kStore> g;
    g.init(a);
    StageWalk w;
    for (uint32_t k = 0; k < count; ++k, g.step(a), w.next(r)) {
        // the stage's previous use completed the empty phase of the other parity
        if (k >= S && !wait_bounded(r.empty(w.s), w.parity ^ 1u, a.timeout_ns, r.abort_flag())) {
            raise_abort(a, r, tile_of(a, k), kWhereProducerWait);
            break;
        }
        if (check) {
            ring_check_freed(a, r, w.s, k, tile_of(a, k));
            *reinterpret_cast<volatile uint32_t*>(&r.ctl->filled[w.s]) = k + 1u;  // published by the arrive
        }
        const uint32_t full = r.full(w.s), stage = r.stage(w.s);
        ptx::mbar_arrive_expect_tx(full, bytes);
        if (MODE == kStore) ptx::bulk_load(stage, a.packed + static_cast<size_t>(g.t) * bytes, bytes, full);
        else if (hint) ptx::tma_load_hint<R>(stage, &src_map, g.origin(), full, policy);
        else ptx::tma_load<R>(stage, &src_map, g.origin(), full);
        *issued = k + 1;
    }
    *reinterpret_cast<volatile uint32_t*>(&r.ctl->producer_done) = 1;
}

// One consumer thread drains every box of the tile grid with one engine copy:
// a 1-D bulk store of the image into the packed buffer (gathers), or a tensor
// store into the destination (round trips and stores whose destination holds
// the whole grid and whose rows end on 16-byte boundaries).  Every box opens a
// bulk group and at most L + 1 groups read their stages at once (L, the
// launch's store lag, is fixed at compile time up to 2; LAG < 0 reads it from
// the launch).  A stage is released once its group has finished reading:
//   EARLY = false  after committing box k the thread waits until at most L
//                  groups still read and frees the stage of box k - L;
//   EARLY = true   before storing box k the thread waits until at most L
//                  groups still read and frees the stage of box k - L - 1,
//                  so that the load into that stage is issued ahead of the
//                  store of box k (needs L + 1 < stages).  The thread first
//                  pauses for about kEarlyReleasePauseNs after each box lands.
// Measured on GB300 (512 MiB fp16 round trip, 16 KiB boxes, seven stages, one
// CTA per SM, three store groups): early release with the pause sustained
// 6,786-6,799 GB/s, early release without it 6,694-6,716, and the late order
// 6,627-6,633; a pause of the same length in the producer did not help.
constexpr unsigned kEarlyReleasePauseNs = 64;

template <int MODE, int R, int LAG, bool EARLY, bool OPTS>
__device__ __forceinline__ void grid_drain(const PipeArgs& a, const CUtensorMap& dst_map, const Ring& r,
                                           uint32_t count)
{
    const uint32_t S = r.stages, L = LAG >= 0 ? static_cast<uint32_t>(LAG) : a.store_lag;
    const uint32_t lag = EARLY ? L + 1 : L;  // boxes between a box and the release of its stage
    const bool check = OPTS && (a.checks & ATB_CHECK_RING) != 0;
    const bool store_hint =
        OPTS && (a.l2_hints & (ATB_HINT_STORE_EVICT_FIRST | ATB_HINT_STORE_EVICT_LAST)) != 0;
    const uint64_t store_policy = !store_hint ? 0
                                  : (a.l2_hints & ATB_HINT_STORE_EVICT_FIRST) ? ptx::policy_evict_first()
                                                                               : ptx::policy_evict_last();
    auto release = [&](const StageWalk& w, uint32_t k) {  // the stage of box k - lag
        if (LAG >= 0) ptx::bulk_wait_read<(LAG >= 0 ? LAG : 0)>();
        else ptx::bulk_wait_read_le(L);
        uint32_t sf = w.s + S - lag;  // lag < S
        if (sf >= S) sf -= S;
        if (check) ring_note_freed(a, r, sf, k - lag);
        ptx::mbar_arrive(r.empty(sf));
    };
    GridWalk<R, MODE == kLoad> g;
    g.init(a);
    StageWalk w;
    uint32_t k = 0;
    bool failed = false;
    for (; k < count; ++k, g.step(a), w.next(r)) {
        if (!wait_bounded(r.full(w.s), w.parity, a.timeout_ns, r.abort_flag())) {
            failed = true;
            break;
        }
        if (EARLY) __nanosleep(kEarlyReleasePauseNs);
        if (check) ring_check_filled(a, r, w.s, k, tile_of(a, k));
        if (EARLY && k + 1 > lag) release(w, k);
        ptx::fence_proxy_async_smem();
        const uint32_t stage = r.stage(w.s);
        if (MODE == kLoad) ptx::bulk_store(a.packed + static_cast<size_t>(g.t) * a.box_bytes, stage, a.box_bytes);
        else if (store_hint) ptx::tma_store_hint<R>(&dst_map, g.origin(), stage, store_policy);
        else ptx::tma_store<R>(&dst_map, g.origin(), stage);
        ptx::bulk_commit();
        if (!EARLY && k + 1 > lag) release(w, k);
    }
    ptx::bulk_wait_all();
    if (failed) drain_after_failure(a, r, k);
}

// The tile-grid pipeline, 64 threads: warp 0 lane 0 produces, warp 1
// consumes.
//   kConsumerDrain      every box is drained by one engine copy: thread 0
//                       is the producer (grid_producer) and thread 32 the
//                       whole consumer (grid_drain);
//   kConsumerDrainOpts  the same with the ring check and L2 hints compiled in;
//   kConsumerWarp       warp 1 follows every box; lane 0 issues the engine's
//                       drain copies, and boxes that miss the destination or
//                       cross the end of a row whose byte length is not a
//                       multiple of 16 are written by the warp with plain
//                       clipped stores.
constexpr int kConsumerWarp = 0;
constexpr int kConsumerDrain = 1;
constexpr int kConsumerDrainOpts = 2;

template <int MODE, int R, int CONSUMER>
__global__ void __launch_bounds__(kPipelineThreads, 1)
    tile_pipeline_kernel(const __grid_constant__ CUtensorMap src_map, const __grid_constant__ CUtensorMap dst_map,
                         const PipeArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    const Ring r = ring_layout(a, smem_raw);
    const uint32_t S = r.stages;
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) init_ring(r);
    if (threadIdx.x == 32) {
        if (MODE != kStore) ptx::prefetch_tensor_map(&src_map);
        if (MODE != kLoad) ptx::prefetch_tensor_map(&dst_map);
    }
    // Let the next launch on the stream be scheduled now; it sets up its own
    // shared memory and then waits, as this grid does here, for the grids
    // before it to complete before touching global memory.
    ptx::launch_dependents();
    __syncthreads();
    ptx::wait_prerequisite_grids();

    const uint32_t count = my_tile_count(a);

    if (CONSUMER != kConsumerWarp) {
        constexpr bool O = CONSUMER == kConsumerDrainOpts;
        if (threadIdx.x == 0) {
            grid_producer<MODE, R, O>(a, src_map, r, count);
        } else if (threadIdx.x == 32) {
            if (a.early_release) {
                switch (a.store_lag) {
                case 1: grid_drain<MODE, R, 1, true, O>(a, dst_map, r, count); break;
                case 2: grid_drain<MODE, R, 2, true, O>(a, dst_map, r, count); break;
                default: grid_drain<MODE, R, -1, true, O>(a, dst_map, r, count); break;
                }
            } else {
                switch (a.store_lag) {
                case 0: grid_drain<MODE, R, 0, false, O>(a, dst_map, r, count); break;
                case 1: grid_drain<MODE, R, 1, false, O>(a, dst_map, r, count); break;
                case 2: grid_drain<MODE, R, 2, false, O>(a, dst_map, r, count); break;
                default: grid_drain<MODE, R, -1, false, O>(a, dst_map, r, count); break;
                }
            }
        }
        return;
    }
    if (warp == 0) {
        if (lane == 0) producer_loop<MODE, R, false>(a, src_map, src_map, r, count);
        return;
    }

    // ---------------------------------------------------------------- consumer
    const bool store_hint = (a.l2_hints & (ATB_HINT_STORE_EVICT_FIRST | ATB_HINT_STORE_EVICT_LAST)) != 0;
    const uint64_t store_policy = !store_hint ? 0
                                  : (a.l2_hints & ATB_HINT_STORE_EVICT_FIRST) ? ptx::policy_evict_first()
                                                                               : ptx::policy_evict_last();
    PendingStores pending;  // lane 0's store groups still reading their stages
    BoxCursor<R> cur;
    cur.init(a);
    uint32_t k = 0;
    bool failed = false;
    for (; k < count; ++k, cur.advance(a, S)) {
        const uint32_t s = cur.stage;
        const bool ok = wait_bounded(r.full(s), cur.parity, a.timeout_ns, r.abort_flag(), a.suspend_ns);
        if (!__all_sync(0xffffffffu, ok)) {
            failed = true;
            break;
        }
        const uint32_t t = cur.t;
        if (lane == 0) {
            ring_check_filled(a, r, s, k, t);
            if (a.early_release)  // free the stage of every box stored at least store_groups boxes back
                pending.retire(a, r, k, a.store_lag + 1);
        }
        int32_t c[R];
        cur.grid_origin(a, c);  // every lane follows the same cursor
        // kLoad: kStoreTensor means "drain the image to the packed buffer"
        const int kind = MODE == kLoad ? kStoreTensor : store_kind<R>(a, c);
        if (MODE != kLoad && kind == kStorePlain) {
            // boxes the engine may not store: the warp writes them itself
            plain_store_grid_box<R>(a, c, r.stage(s), lane, 32);
            __syncwarp();
        }
        if (lane == 0) {
            if (kind == kStoreTensor) {
                ptx::fence_proxy_async_smem();
                if (MODE == kLoad)
                    ptx::bulk_store(a.packed + static_cast<size_t>(t) * a.box_bytes, r.stage(s), a.box_bytes);
                else if (store_hint) ptx::tma_store_hint<R>(&dst_map, c, r.stage(s), store_policy);
                else ptx::tma_store<R>(&dst_map, c, r.stage(s));
                ptx::bulk_commit();
                pending.push(s, k);
            } else {
                ring_note_freed(a, r, s, k);
                ptx::mbar_arrive(r.empty(s));  // written by the warp, or nothing to write
            }
            if (!a.early_release) pending.retire(a, r, k, a.store_lag);
        }
    }

    if (lane != 0) return;
    ptx::bulk_wait_all();
    if (failed) drain_after_failure(a, r, k);
}

// The pipeline with several consumer warps: warp 0 lane 0 produces, the
// consumer warps share each landed stage, and consumer thread 0 issues the
// engine's drain copy (a tensor store, or for gathers the 1-D bulk store of
// the image into the packed buffer).  Launches with a coordinate list run
// here: their boxes may start before the tensor or off the 16-byte grid along
// x, and the consumer threads share the plain loads and clipped stores of
// such boxes.
//   ADD   round trip with an elementwise fp32 update in shared memory between
//         the load and the store ("Day 76: The Tensor Memory Accelerator
//         (TMA)", "Exercise" and "Solution": the threads change the tile in
//         shared memory, every writer publishes its writes across the proxy
//         line with fence.proxy.async, the group meets at a barrier, and one
//         thread issues the tensor store).  Each element becomes x + addend in
//         round-to-nearest fp32.  Two consumer warps.
//   !ADD  gathers, stores and round trips over a coordinate list: four
//         consumer warps.
//   LISTED  launched with a coordinate list; false (the fp32 update over the
//         tile grid) compiles the listed-box paths out: grid origins are
//         always on the 16-byte grid and never refused.
template <int MODE, int R, bool ADD, bool LISTED>
__global__ void __launch_bounds__(32 + (ADD ? kUpdateConsumerThreads : kConsumerThreads), ADD ? 1 : (MODE == kLoad ? 3 : 4))
    tile_wide_kernel(const __grid_constant__ CUtensorMap src_map, const __grid_constant__ CUtensorMap dst_map,
                     const __grid_constant__ CUtensorMap wide_map, const PipeArgs a, float addend)
{
    extern __shared__ uint8_t smem_raw[];
    const Ring r = ring_layout(a, smem_raw);
    const uint32_t S = r.stages;
    const uint32_t warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) init_ring(r);
    if (threadIdx.x == 32) {
        if (MODE != kStore) ptx::prefetch_tensor_map(&src_map);
        if (MODE != kLoad) ptx::prefetch_tensor_map(&dst_map);
        if (MODE != kStore && a.wide_box0) ptx::prefetch_tensor_map(&wide_map);
    }
    ptx::launch_dependents();
    __syncthreads();
    ptx::wait_prerequisite_grids();

    const uint32_t count = my_tile_count(a);
    if (warp == 0) {
        if (threadIdx.x == 0) producer_loop<MODE, R, LISTED>(a, src_map, wide_map, r, count);
        return;
    }

    // consumer threads: fewer for the update (measured faster), more for clipped stores
    constexpr uint32_t CT = ADD ? kUpdateConsumerThreads : kConsumerThreads;
    const uint32_t ct = threadIdx.x - 32;  // consumer thread 0 .. CT-1
    const bool store_hint = MODE != kLoad && (a.l2_hints & (ATB_HINT_STORE_EVICT_FIRST | ATB_HINT_STORE_EVICT_LAST));
    const uint64_t store_policy = !store_hint ? 0
                                  : (a.l2_hints & ATB_HINT_STORE_EVICT_FIRST) ? ptx::policy_evict_first()
                                                                               : ptx::policy_evict_last();
    PendingStores pending;  // consumer thread 0's store groups still reading their stages
    BoxCursor<R> cur;
    cur.init(a);
    uint32_t k = 0;
    bool failed = false;
    for (; k < count; ++k, cur.advance(a, S)) {
        const uint32_t s = cur.stage;
        const bool ok = wait_bounded(r.full(s), cur.parity, a.timeout_ns, r.abort_flag(), a.suspend_ns);
        if (!__all_sync(0xffffffffu, ok)) {
            failed = true;
        }
        // Every consumer thread reads the origin slot before the barrier
        // below; consumer thread 0 frees the stage only after that barrier, so
        // no thread can see the slot refilled for a later box.
        int32_t c[R];
        landed_origin<R>(a, r, s, cur, c);
        // every consumer warp must agree before any of them leaves the loop
        if (ptx::named_barrier_or(1, CT, failed)) {
            failed = true;
            break;
        }
        if (ct == 0) {
            ring_check_filled(a, r, s, k, cur.t);
            if (a.early_release)  // free the stage of every box stored at least store_groups boxes back
                pending.retire(a, r, k, a.store_lag + 1);
        }
        const int lk = !LISTED          ? kLoadEngine
                       : MODE == kStore ? (origin_error<R>(a, c) ? kLoadRefused : kLoadEngine)
                                        : load_kind<R>(a, c);
        const bool tload = lk == kLoadThreads;  // arrived with no bytes: the consumer threads load it
        const bool wide = lk == kLoadWide;      // the wider image from the origin rounded down to the grid
        // How the box leaves.  Gathers: kStoreTensor = one bulk store of the
        // image into the packed buffer, kStorePlain = the threads write the
        // packed image out of the wider image.  Stores and round trips: as
        // store_kind says (an origin off the grid always takes plain stores).
        int kind;
        if (lk == kLoadRefused) kind = kStoreNothing;
        else if (MODE == kLoad) kind = wide ? kStorePlain : kStoreTensor;
        else kind = store_kind<R>(a, c);
        if (tload) {
            thread_load_box<R>(a, c, r.stage(s), ct, CT);
            if (kind == kStoreTensor) ptx::fence_proxy_async_smem();  // each writer, before the engine reads
            ptx::named_barrier_sync(1, CT);  // the whole image is in the stage before anyone reads it
        }
        const uint32_t chunks = (wide ? a.wide_bytes : a.box_bytes) / 16;
        if (ADD && kind != kStoreNothing) {
            // generic-proxy update of the landed box; element order is irrelevant.
            // Sixteen 16-byte chunks per thread at a time (with two consumer
            // warps a 16 KiB box is exactly one such pass), all loads issued
            // before the first add, so one shared-memory latency is paid per
            // pass instead of one per chunk.
            const uint32_t base = r.stage(s);
            uint32_t j = ct;
            for (; j + 15 * CT < chunks; j += 16 * CT) {
                float v[16][4];
#pragma unroll
                for (int u = 0; u < 16; ++u) ptx::ld_shared_v4_f32(base + 16 * (j + u * CT), v[u]);
#pragma unroll
                for (int u = 0; u < 16; ++u) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[u][e] = __fadd_rn(v[u][e], addend);
                }
#pragma unroll
                for (int u = 0; u < 16; ++u) ptx::st_shared_v4_f32(base + 16 * (j + u * CT), v[u]);
            }
            for (; j < chunks; j += CT) {  // the rest of a box that is not a multiple of 16 x 16 x CT bytes
                float v[4];
                ptx::ld_shared_v4_f32(base + 16 * j, v);
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] = __fadd_rn(v[e], addend);
                ptx::st_shared_v4_f32(base + 16 * j, v);
            }
            ptx::fence_proxy_async_smem();  // each writer publishes its own writes to the async proxy
        }
        if (ADD) ptx::named_barrier_sync(1, CT);  // the update is complete and fenced before any store
        if (kind == kStorePlain) {
            if (MODE == kLoad)
                pack_from_wide<R>(a, c, r.stage(s), a.packed + static_cast<size_t>(cur.t) * a.box_bytes, ct, CT);
            else if (LISTED && row_phase<R>(a, c))  // off the 16-byte grid: aligned stores of up to 4 bytes
                store_off_grid_box<R>(a, c, r.stage(s), wide ? kFromWide : kFromImage, ct, CT);
            else  // on the 16-byte grid: 16-byte chunks
                plain_store_grid_box<R>(a, c, r.stage(s), ct, CT);
            ptx::named_barrier_sync(1, CT);  // every reader is done with the stage
        }
        if (ct == 0) {
            if (kind == kStoreTensor) {
                if (!ADD && !tload) ptx::fence_proxy_async_smem();  // (writers of the stage fenced already)
                if (MODE == kLoad)
                    ptx::bulk_store(a.packed + static_cast<size_t>(cur.t) * a.box_bytes, r.stage(s), a.box_bytes);
                else if (store_hint)
                    ptx::tma_store_hint<R>(&dst_map, c, r.stage(s), store_policy);
                else
                    ptx::tma_store<R>(&dst_map, c, r.stage(s));
                ptx::bulk_commit();
                pending.push(s, k);
            } else {
                ring_note_freed(a, r, s, k);
                ptx::mbar_arrive(r.empty(s));  // written by the threads, or nothing to write
            }
            if (!a.early_release) pending.retire(a, r, k, a.store_lag);
        }
    }

    if (ct != 0) return;
    ptx::bulk_wait_all();
    if (failed) drain_after_failure(a, r, k);
}

// Self-test of the bounded wait: nothing ever completes this barrier.
__global__ void wait_timeout_selftest_kernel(DeviceStatus* st, uint64_t timeout_ns)
{
    __shared__ alignas(8) uint64_t bar;
    const uint32_t b = ptx::smem_addr(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        ptx::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0 && !wait_bounded(b, 0, timeout_ns, nullptr))
        record_error(st, ATB_ERR_TIMEOUT, -1, kWhereSelftest);
}

using KernelFn = void (*)(const CUtensorMap, const CUtensorMap, const PipeArgs);
using WideKernelFn = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const PipeArgs, float);

template <int MODE, int CONSUMER>
KernelFn kernel_for_rank(uint32_t rank)
{
    switch (rank) {
    case 1: return tile_pipeline_kernel<MODE, 1, CONSUMER>;
    case 2: return tile_pipeline_kernel<MODE, 2, CONSUMER>;
    case 3: return tile_pipeline_kernel<MODE, 3, CONSUMER>;
    case 4: return tile_pipeline_kernel<MODE, 4, CONSUMER>;
    default: return tile_pipeline_kernel<MODE, 5, CONSUMER>;
    }
}

template <int MODE>
KernelFn grid_kernel(uint32_t rank, bool drain, bool opts)
{
    if (!drain) return kernel_for_rank<MODE, kConsumerWarp>(rank);
    return opts ? kernel_for_rank<MODE, kConsumerDrainOpts>(rank) : kernel_for_rank<MODE, kConsumerDrain>(rank);
}

template <int MODE, bool ADD, bool LISTED>
WideKernelFn wide_kernel_for_rank(uint32_t rank)
{
    switch (rank) {
    case 1: return tile_wide_kernel<MODE, 1, ADD, LISTED>;
    case 2: return tile_wide_kernel<MODE, 2, ADD, LISTED>;
    case 3: return tile_wide_kernel<MODE, 3, ADD, LISTED>;
    case 4: return tile_wide_kernel<MODE, 4, ADD, LISTED>;
    default: return tile_wide_kernel<MODE, 5, ADD, LISTED>;
    }
}

uint32_t swizzle_bits(uint32_t sw) { return sw <= ATB_SWIZZLE_128B ? sw : 0; }

// Bytes of one stage: the box image, or (launches that may load through the
// one-chunk-wider map) the larger of that and the wider image, rounded up to
// the stage alignment.
uint32_t stage_bytes_for(const atb_tensor_map* m, bool wide_loads = false)
{
    const uint32_t align = m->swizzle != ATB_SWIZZLE_NONE ? kStageAlignSwizzled : kStageAlignPlain;
    uint32_t bytes = m->box_bytes;
    if (wide_loads && m->wide_box0) {
        const uint32_t wide = m->box_bytes / m->box[0] * m->wide_box0;
        if (wide > bytes) bytes = wide;
    }
    return (bytes + align - 1) / align * align;
}

size_t smem_bytes_for(const atb_tensor_map* m, uint32_t stages, bool wide_loads = false)
{
    return kStageAlignSwizzled + static_cast<size_t>(stages) * stage_bytes_for(m, wide_loads) + 16u * stages +
           sizeof(Control);
}

// Default pipeline shape, measured on GB300 round trips of a 512 MiB fp16
// tensor (8, 16 and 32 KiB boxes, every cell of stages x CTAs per SM x store
// groups, strided and contiguous schedules): three stages per CTA, two store
// groups in flight, and about 96 KiB of stages per SM (one CTA of 32 KiB
// boxes, two of 16 KiB, four of 8 KiB).  A stage is then busy for one load and
// one store read, and the ring always has a free stage for the next load.
constexpr uint32_t kDefaultStages = 3;
constexpr uint32_t kDefaultStoreGroups = 2;
constexpr uint64_t kStageBytesPerSm = 96u * 1024u;
constexpr uint64_t kMaxDefaultCtasPerSm = 8;
constexpr uint32_t kDrainStageBytes = 32u * 1024u;

// The one-thread drain's own default ring for stages of 8 to 32 KiB, measured
// on GB300 (16 KiB boxes of a 512 MiB fp16 round trip, one CTA per SM, rings
// of 6 to 12 stages with every store-group count, stages released before or
// after the next store): about 64 KiB of stages waiting for or holding landed
// boxes plus 48 KiB of store groups in flight, one CTA per SM, each stage
// freed before the next store is issued so that the load into it goes out
// first.  Every ring with four stages on the load side and three to six
// store groups sustained 6,786-6,796 GB/s; three or five load-side stages
// fell to 6,190-6,240.  Stages of 4 to 8 KiB would need more stages than a
// ring holds; they run two CTAs per SM, each with 32 KiB of stages on the load
// side (64 KiB per SM again) and 16 KiB of store groups (4 KiB boxes: 6,297-
// 6,341 GB/s against 6,199-6,291 for the warp consumer, the step-2 gather
// 5,552 -> 6,355; 24 KiB of store groups per CTA measured 5,984-6,162).
constexpr uint32_t kDrainMinStageBytes = 4u * 1024u;
constexpr uint32_t kDrainLoadSideBytes = 64u * 1024u;
constexpr uint32_t kDrainStoreSideBytes = 48u * 1024u;
constexpr uint32_t kDrainSmallStageBytes = 8u * 1024u;  // below: two CTAs per SM
constexpr uint32_t kDrainSmallLoadSideBytes = 32u * 1024u;
constexpr uint32_t kDrainSmallStoreSideBytes = 16u * 1024u;

// The several-warp kernel's own ring (coordinate lists and the fp32 update) for
// stages of 16 to 32 KiB, measured the same way: two CTAs per SM (its consumer
// warps' per-box work needs another CTA's boxes to hide behind), each with
// 32 KiB of stages for boxes being loaded or landed (64 KiB per SM again) and
// 48 KiB of store groups, stages freed before the next store.  16 KiB boxes:
// fp32 update 6,343 -> 6,564 GB/s and listed gather 6,344 -> 6,644 against the
// common ring (same GPU); 48 KiB per CTA on the load side fell to 5,870-6,160.
constexpr uint32_t kWideDeepMinStageBytes = 16u * 1024u;
constexpr uint32_t kWideLoadSideBytes = 32u * 1024u;
constexpr uint32_t kWideStoreSideBytes = 48u * 1024u;
constexpr uint32_t kWideDeepCtasPerSm = 2;

uint32_t default_stages(const atb_tensor_map* m, const DeviceInfo& dev, bool wide_loads)
{
    uint32_t s = kDefaultStages;
    while (s > 1 && smem_bytes_for(m, s, wide_loads) > static_cast<size_t>(dev.smem_optin)) --s;
    return s;
}

std::mutex g_attr_mutex;

atb_status prepare_kernel(const void* fn, const DeviceInfo& dev)
{
    // Opt every instantiation into the full per-block shared memory once per device.
    static const void* done[64][64];
    static int n_done[64];
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    for (int i = 0; i < n_done[dev.device]; ++i)
        if (done[dev.device][i] == fn) return ATB_OK;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, dev.smem_optin);
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute");
    if (n_done[dev.device] < 64) done[dev.device][n_done[dev.device]++] = fn;
    return ATB_OK;
}

// CTAs of `fn` that fit on one SM with `threads` threads and `smem` bytes of
// dynamic shared memory, after opting the kernel into the full per-block
// shared memory.  Each host thread keeps the answers of its last sixteen
// launch shapes, so that a repeated launch asks the runtime nothing and takes
// no lock.
atb_status kernel_fit(const void* fn, const DeviceInfo& dev, uint32_t threads, size_t smem, int* fit)
{
    struct Shape {
        const void* fn;
        int device;
        uint32_t threads;
        size_t smem;
        int fit;
    };
    thread_local Shape cache[16] = {};
    thread_local uint32_t next = 0;
    for (const Shape& c : cache) {
        if (c.fn == fn && c.device == dev.device && c.threads == threads && c.smem == smem) {
            *fit = c.fit;
            return ATB_OK;
        }
    }
    atb_status st = prepare_kernel(fn, dev);
    if (st != ATB_OK) return st;
    int f = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&f, fn, static_cast<int>(threads), smem);
    if (e != cudaSuccess) return cuda_error(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    cache[next++ % 16] = Shape{fn, dev.device, threads, smem, f};
    *fit = f;
    return ATB_OK;
}

// `caller_status`, when given, receives the kernel's error record instead of
// the device's lazily allocated status block.
// Launches one pipeline over boxes [first, first + count) of the list or grid
// (count = UINT64_MAX: all of them).
// The shape of this host thread's most recent pipeline launch (atb_last_launch).
thread_local atb_launch_shape g_last_shape = {};

template <int MODE>
atb_status launch_pipeline(const atb_tensor_map* src, const atb_tensor_map* dst, const int32_t* coords, uint64_t n,
                           void* packed, const atb_launch* cfg, cudaStream_t stream,
                           DeviceStatus* caller_status = nullptr, float addend = 0.0f, uint64_t first = 0,
                           uint64_t count = UINT64_MAX)
{
    clear_error();
    g_last_shape = atb_launch_shape{};
    const atb_tensor_map* shape = MODE == kStore ? dst : src;
    if ((MODE != kStore && !map_is_valid(src)) || (MODE != kLoad && !map_is_valid(dst)))
        return set_error(ATB_ERR_ARG, "tensor map is NULL or was not produced by atb_encode_tiled");
    if (MODE == kRoundtripAddF32 && (src->dtype != ATB_F32 || dst->dtype != ATB_F32))
        return set_error(ATB_ERR_DTYPE, "the fp32 update needs ATB_F32 maps (got types %u and %u)", src->dtype,
                         dst->dtype);
    if (MODE == kRoundtrip || MODE == kRoundtripAddF32) {
        bool same = src->rank == dst->rank && src->esize == dst->esize && src->swizzle == dst->swizzle;
        for (uint32_t d = 0; same && d < src->rank; ++d)
            same = src->box[d] == dst->box[d] && src->elem_strides[d] == dst->elem_strides[d];
        if (!same)
            return set_error(ATB_ERR_ARG,
                             "source and destination maps differ in rank, element size, box, steps or swizzle");
    }
    if (cfg && (cfg->checks & ~ATB_CHECK_RING))
        return set_error(ATB_ERR_ARG, "unknown check bits 0x%x", cfg->checks & ~ATB_CHECK_RING);
    if (cfg && cfg->consumer > ATB_CONSUMER_WARP)
        return set_error(ATB_ERR_ARG, "unknown consumer %u", cfg->consumer);
    if (cfg && cfg->release > ATB_RELEASE_BEFORE_STORE)
        return set_error(ATB_ERR_ARG, "unknown release %u", cfg->release);
    if (MODE == kLoad || MODE == kStore) {
        if (!packed) return set_error(ATB_ERR_ARG, "packed buffer is NULL");
        if (reinterpret_cast<uintptr_t>(packed) % 16)
            return set_error(ATB_ERR_SMEM_ALIGN, "packed buffer %p is not 16-byte aligned", packed);
    }
    const uint32_t rank = shape->rank;
    uint64_t n_tiles = coords ? n : atb_grid_tiles(shape);
    if (!coords) {
        for (uint32_t d = 0; d < rank; ++d) {
            const uint64_t tiles = (shape->dims[d] + shape->box[d] - 1) / shape->box[d];
            if ((tiles - 1) * shape->box[d] > 0x7FFFFFFFull)
                return set_error(ATB_ERR_DIM_RANGE, "tile grid origin along dimension %u exceeds int32", d);
        }
    }
    if (n_tiles >= 0x80000000ull)
        return set_error(ATB_ERR_ARG, "%llu boxes in one call; the limit is 2^31 - 1",
                         static_cast<unsigned long long>(n_tiles));
    if (first > n_tiles) return set_error(ATB_ERR_ARG, "box range starts past the last box");
    const uint64_t all_tiles = n_tiles;
    n_tiles = count < all_tiles - first ? count : all_tiles - first;

    DeviceInfo dev;
    atb_status st = current_device(&dev);
    if (st != ATB_OK) return st;
    // listed boxes off the 16-byte grid load the wider image into their stage
    const bool wide_loads = coords && MODE != kStore && shape->wide_box0;
    const uint32_t stage_b = stage_bytes_for(shape, wide_loads);

    // Launches over a coordinate list (whose boxes may start before the tensor
    // or off the 16-byte grid along x) and the fp32 update run the kernel with
    // several consumer warps; tile-grid launches run the 64-thread kernel.
    constexpr int kBase = MODE == kRoundtripAddF32 ? kRoundtrip : MODE;
    const bool wide = MODE == kRoundtripAddF32 || coords != nullptr;
    // Tile grid: where every box leaves through one engine copy (no box misses
    // the destination or crosses a ragged row end) either consumer serves.
    // The library takes the one-thread drain for stages of 32 KiB and more,
    // and for stages of 4 to 32 KiB when the caller leaves the ring's shape to
    // it (the drain then runs its own deeper ring, one CTA per SM, two below
    // 8 KiB); the warp
    // consumer otherwise (measured on GB300: each was the faster there).  The
    // warp consumer, which can also write plain clipped stores, serves the
    // rest.  The drain's producer neither prefetches nor suspends its polls:
    // launches asking for either take the warp consumer, as do grids wider
    // than 2^31 elements along a dimension below the outermost.
    bool plain = false;
    if (!wide && MODE != kLoad) {
        plain = (dst->dims[0] * dst->esize) % 16 != 0;
        if (MODE == kRoundtrip)
            for (uint32_t d = 0; d < rank; ++d) plain = plain || dst->dims[d] < src->dims[d];
    }
    const uint32_t consumer = cfg ? cfg->consumer : ATB_CONSUMER_AUTO;
    bool drain_fits = !wide && !plain && !(cfg && (cfg->prefetch_boxes || cfg->poll_suspend_ns));
    for (uint32_t d = 0; d + 1 < rank; ++d)  // the drain's origin walk: extents of at most 2^31 elements
        drain_fits = drain_fits && (shape->dims[d] + shape->box[d] - 1) / shape->box[d] * shape->box[d] <= (1ull << 31);
    const bool shape_given = cfg && (cfg->stages || cfg->store_groups || cfg->ctas_per_sm);
    const bool deep_fits = !shape_given && stage_b >= kDrainMinStageBytes && stage_b < kDrainStageBytes;
    const bool drain = drain_fits && (consumer == ATB_CONSUMER_DRAIN ||
                                      (consumer == ATB_CONSUMER_AUTO && (stage_b >= kDrainStageBytes || deep_fits)));
    const bool deep = drain && deep_fits;  // the drain's own ring
    // the several-warp kernel's own ring (coordinate lists and the fp32 update, 16 to 32 KiB stages)
    // (sized on the box image: off-grid listed boxes load a wider image into the same number of stages)
    const uint32_t image_b = stage_bytes_for(shape);
    const bool wide_deep = wide && !shape_given && image_b >= kWideDeepMinStageBytes && image_b < kDrainStageBytes;
    const bool deep_small = deep && stage_b < kDrainSmallStageBytes;
    const uint32_t deep_groups = deep_small ? kDrainSmallStoreSideBytes / stage_b
                                 : deep     ? kDrainStoreSideBytes / stage_b
                                 : wide_deep ? kWideStoreSideBytes / image_b
                                             : 0u;
    const uint32_t stages = cfg && cfg->stages ? cfg->stages
                            : deep_small       ? kDrainSmallLoadSideBytes / stage_b + deep_groups
                            : deep             ? kDrainLoadSideBytes / stage_b + deep_groups
                            : wide_deep        ? kWideLoadSideBytes / image_b + deep_groups
                                               : default_stages(shape, dev, wide_loads);
    if (stages < 1 || stages > kMaxStages)
        return set_error(ATB_ERR_ARG, "stages = %u is outside 1..%u", stages, kMaxStages);
    const size_t smem = smem_bytes_for(shape, stages, wide_loads);
    if (smem > static_cast<size_t>(dev.smem_optin))
        return set_error(ATB_ERR_SMEM_BUDGET,
                         "%u stages of %u bytes need %zu bytes of shared memory; a block may have at most %d",
                         stages, stage_b, smem, dev.smem_optin);
    uint32_t groups = cfg && cfg->store_groups ? cfg->store_groups
                      : deep || wide_deep        ? deep_groups
                                                 : kDefaultStoreGroups;
    if (groups > stages) groups = stages;
    if (groups > 8) groups = 8;
    const uint32_t release = cfg ? cfg->release : ATB_RELEASE_AUTO;
    if (release == ATB_RELEASE_BEFORE_STORE && groups >= stages)
        return set_error(ATB_ERR_ARG, "releasing before the next store needs store_groups (%u) < stages (%u)", groups,
                         stages);
    const bool early =
        groups < stages && (release == ATB_RELEASE_BEFORE_STORE || (release == ATB_RELEASE_AUTO && (deep || wide_deep)));
    if (n_tiles == 0) return ATB_OK;

    DeviceStatus* status = caller_status;
    if (!status) {
        st = device_status_block(&status);
        if (st != ATB_OK) return st;
    }

    WideKernelFn wide_fn = nullptr;
    KernelFn grid_fn = nullptr;
    if (MODE == kRoundtripAddF32)
        wide_fn = coords ? wide_kernel_for_rank<kRoundtrip, true, true>(rank)
                         : wide_kernel_for_rank<kRoundtrip, true, false>(rank);
    else if (wide) wide_fn = wide_kernel_for_rank<kBase, false, true>(rank);
    else grid_fn = grid_kernel<kBase>(rank, drain, cfg && (cfg->checks || cfg->l2_hints));
    const void* fn = wide ? reinterpret_cast<const void*>(wide_fn) : reinterpret_cast<const void*>(grid_fn);
    const uint32_t threads = MODE == kRoundtripAddF32 ? 32 + kUpdateConsumerThreads
                             : wide                     ? kTransformThreads
                                                        : kPipelineThreads;
    int fit = 0;
    st = kernel_fit(fn, dev, threads, smem, &fit);
    if (st != ATB_OK) return st;

    uint32_t per_sm = cfg && cfg->ctas_per_sm ? cfg->ctas_per_sm
                      : deep_small               ? 2u
                      : deep                     ? 1u
                      : wide_deep                ? kWideDeepCtasPerSm
                                                 : 0u;
    if (!per_sm) {
        // sized on the box image: a wider stage for off-grid loads does not cut the CTA count
        uint64_t want = kStageBytesPerSm / (static_cast<uint64_t>(stages) * stage_bytes_for(shape));
        want = want < 1 ? 1 : (want > kMaxDefaultCtasPerSm ? kMaxDefaultCtasPerSm : want);
        // A short launch, whose CTAs would each see no more than four ring-fulls
        // of boxes, spreads them over as many CTAs per SM as fit, up to one
        // ring-full each, so that more of its boxes are in flight from the start
        // (workload 2, 924 boxes of 32 KiB, two CTAs per SM instead of one: 9.3
        // -> 6.1 us back to back, 13.0 -> 12.5 us after an L2 flush, on GB300).
        const uint64_t sms = static_cast<uint64_t>(dev.sm_count);
        if (n_tiles <= 4 * sms * want * stages) {
            const uint64_t spread = (n_tiles + sms * stages - 1) / (sms * stages);
            if (spread > want) want = spread > kMaxDefaultCtasPerSm ? kMaxDefaultCtasPerSm : spread;
        }
        per_sm = static_cast<uint32_t>(fit < 1 ? 1 : (static_cast<uint64_t>(fit) < want ? fit : want));
    }
    uint64_t grid = cfg && cfg->ctas ? cfg->ctas : static_cast<uint64_t>(dev.sm_count) * per_sm;
    if (grid > n_tiles) grid = n_tiles;
    if (grid > 0x7FFFFFFFull) grid = 0x7FFFFFFFull;

    PipeArgs a{};
    a.coords = coords;
    a.packed = static_cast<uint8_t*>(packed);
    a.status = status;
    a.timeout_ns = wait_timeout_ns();
    a.n_tiles = static_cast<uint32_t>(n_tiles);
    a.tile_begin = static_cast<uint32_t>(first);
    a.esize = shape->esize;
    a.box_bytes = shape->box_bytes;
    a.stage_bytes = stage_b;
    a.stages = stages;
    a.store_lag = groups - 1;
    a.early_release = early ? 1u : 0u;
    a.contiguous = cfg && cfg->schedule == 1 ? 1u : 0u;
    a.l2_hints = cfg ? cfg->l2_hints : 0u;
    a.suspend_ns = cfg ? cfg->poll_suspend_ns : 0u;
    a.prefetch = cfg ? cfg->prefetch_boxes : 0u;
    a.checks = cfg ? cfg->checks : 0u;
    a.swizzle_bits = swizzle_bits(shape->swizzle);
    for (uint32_t d = 0; d < rank; ++d) {
        a.box[d] = shape->box[d];
        a.step[d] = shape->elem_strides[d] ? shape->elem_strides[d] : 1;
        a.visits[d] = (shape->box[d] + a.step[d] - 1) / a.step[d];
        a.grid[d] = static_cast<uint32_t>((shape->dims[d] + shape->box[d] - 1) / shape->box[d]);
    }
    if (MODE != kLoad) {  // every mode that writes a tensor
        a.dst_base = reinterpret_cast<uint8_t*>(dst->base);
        for (uint32_t d = 0; d < rank; ++d) {
            a.dst_dims[d] = dst->dims[d];
            a.dst_strides[d] = dst->strides[d];
        }
        a.dst_ragged_x = (dst->dims[0] * dst->esize) % 16 != 0;
    }
    if (MODE != kStore) {  // every mode that reads a tensor: plain loads of off-grid boxes
        a.src_base = reinterpret_cast<const uint8_t*>(src->base);
        for (uint32_t d = 0; d < rank; ++d) {
            a.src_dims[d] = src->dims[d];
            a.src_strides[d] = src->strides[d];
        }
        // the bytes the engine writes for out-of-bounds elements: zero, or
        // the NaN request's fill, 0x7FF7 in every 16-bit half (as measured on
        // GB300 for f16, bf16, f32 and f64 maps)
        const uint32_t fill = src->oob_fill == ATB_OOB_NAN ? kNanFillWord : 0u;
        for (int i = 0; i < 4; ++i) a.fill[i] = fill;
    }
    if (wide_loads) {
        a.wide_box0 = src->wide_box0;
        a.wide_pitch = src->wide_box0 * src->esize;
        a.wide_bytes = src->box_bytes / src->box[0] * src->wide_box0;
    }

    alignas(64) CUtensorMap src_map;
    alignas(64) CUtensorMap dst_map;
    alignas(64) CUtensorMap wide_map;
    memcpy(&src_map, (MODE == kStore ? dst : src)->map, sizeof src_map);
    memcpy(&dst_map, (MODE == kLoad ? src : dst)->map, sizeof dst_map);
    memcpy(&wide_map, wide_loads ? src->map_wide : (MODE == kStore ? dst : src)->map, sizeof wide_map);

    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(static_cast<unsigned>(grid));
    lc.blockDim = dim3(threads);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = cfg && cfg->no_pdl ? 0 : 1;
    cudaError_t e;
    if (wide)
        e = cudaLaunchKernelEx(&lc, wide_fn, src_map, dst_map, wide_map, a, addend);
    else
        e = cudaLaunchKernelEx(&lc, grid_fn, src_map, dst_map, a);
    if (e != cudaSuccess) return cuda_error(e, "kernel launch");
    atb_launch_shape& ls = g_last_shape;
    ls.consumer = wide ? ATB_CONSUMER_WARPS : drain ? ATB_CONSUMER_DRAIN : ATB_CONSUMER_WARP;
    ls.release = a.early_release ? ATB_RELEASE_BEFORE_STORE : ATB_RELEASE_AFTER_STORE;
    ls.stages = stages;
    ls.store_groups = groups;
    ls.ctas_per_sm = per_sm;
    ls.ctas = static_cast<uint32_t>(grid);
    ls.threads = threads;
    ls.smem_bytes = static_cast<uint32_t>(smem);
    ls.boxes = a.n_tiles;
    return ATB_OK;
}

// ---- allocation-free round trip ---------------------------------------------
// Scratch of atb_tile_roundtrip_noalloc: the kernel's error record lives in
// this file-scope device array instead of a block obtained from cudaMalloc.
// The module loader reserves it on every GPU that loads the library, and it
// stays reserved until the process exits.  All calls on one device share it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[ATB_NOALLOC_SCRATCH_BYTES];
static_assert(sizeof(DeviceStatus) <= ATB_NOALLOC_SCRATCH_BYTES, "status record must fit the static scratch");

std::mutex g_noalloc_mutex;
void* g_noalloc_address[64];

// Device address of the array on the current device.  In host code the
// array's name stands for a host-side shadow, never for device memory, so the
// address must come from the runtime, once per device, with that device current.
atb_status noalloc_scratch_address(const DeviceInfo& dev, void** out)
{
    if (dev.device < 0 || dev.device >= 64) return set_error(ATB_ERR_ARG, "device ordinal %d out of range", dev.device);
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_address[dev.device]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_error(e, "cudaGetSymbolAddress(no-allocation scratch)");
        if (!p) return set_error(ATB_ERR_CUDA, "cudaGetSymbolAddress returned a null scratch address");
        g_noalloc_address[dev.device] = p;
    }
    *out = g_noalloc_address[dev.device];
    return ATB_OK;
}

// ---- host-resident round trip ------------------------------------------------
// Per-device streams and events that overlap the host-to-device copies, the
// round trips and the device-to-host copies of atb_tile_roundtrip_host.
constexpr uint32_t kMaxHostSlabs = 64;
constexpr uint32_t kDefaultHostSlabs = 12;

struct HostPipe {
    bool ready;
    cudaStream_t in, out;
    cudaEvent_t start, end;
    cudaEvent_t landed[kMaxHostSlabs], moved[kMaxHostSlabs];
};

std::mutex g_host_mutex;
HostPipe g_host_pipe[64];

atb_status host_pipe(int device, HostPipe** out)
{
    if (device < 0 || device >= 64) return set_error(ATB_ERR_ARG, "device ordinal %d out of range", device);
    HostPipe& p = g_host_pipe[device];
    if (!p.ready) {
        cudaError_t e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.end, cudaEventDisableTiming);
        for (uint32_t j = 0; e == cudaSuccess && j < kMaxHostSlabs; ++j) {
            e = cudaEventCreateWithFlags(&p.landed[j], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.moved[j], cudaEventDisableTiming);
        }
        if (e != cudaSuccess) return cuda_error(e, "creating the host-transfer streams and events");
        p.ready = true;
    }
    *out = &p;
    return ATB_OK;
}

// Bytes of dimensions 0..d-1 of a map, from element 0 to one past the last.
uint64_t inner_span(const atb_tensor_map* m, uint32_t d)
{
    uint64_t span = m->esize;
    for (uint32_t i = 1; i < d; ++i) span += (m->dims[i] - 1) * m->strides[i];
    return span + (d > 0 ? (m->dims[0] - 1) * m->esize : 0);
}

// Byte range [lo, hi) that holds rows [r0, r1) of the outermost dimension.
void slab_bytes(const atb_tensor_map* m, uint64_t r0, uint64_t r1, uint64_t* lo, uint64_t* hi)
{
    const uint32_t L = m->rank - 1;
    const uint64_t stride = L ? m->strides[L] : m->esize;
    const uint64_t inner = L ? inner_span(m, L) : m->esize;
    *lo = r0 * stride;
    *hi = (r1 - 1) * stride + inner;
}

}  // namespace
}  // namespace atb

using namespace atb;

extern "C" {

atb_status atb_tile_roundtrip_host(const atb_tensor_map* src, const atb_tensor_map* dst, const void* h_src,
                                   void* h_dst, uint32_t slabs, const atb_launch* launch, atb_stream_t stream)
{
    clear_error();
    if (!map_is_valid(src) || !map_is_valid(dst))
        return set_error(ATB_ERR_ARG, "tensor map is NULL or was not produced by atb_encode_tiled");
    if (!h_src || !h_dst) return set_error(ATB_ERR_ARG, "host source or destination is NULL");
    if (src->rank != dst->rank) return set_error(ATB_ERR_ARG, "source and destination ranks differ");
    for (uint32_t d = 0; d < src->rank; ++d)
        if (src->dims[d] != dst->dims[d])
            return set_error(ATB_ERR_ARG, "source and destination extents differ along dimension %u", d);
    DeviceInfo dev;
    atb_status st = current_device(&dev);
    if (st != ATB_OK) return st;

    const uint32_t L = src->rank - 1;
    const uint64_t tiles_l = (src->dims[L] + src->box[L] - 1) / src->box[L];
    const uint64_t per_row = atb_grid_tiles(src) / tiles_l;
    // Slabs are contiguous byte ranges only when the outermost dimension
    // steps over everything inside it.
    const bool nested = L == 0 || (src->strides[L] >= inner_span(src, L) && dst->strides[L] >= inner_span(dst, L));
    uint64_t n = slabs ? slabs : kDefaultHostSlabs;
    if (n > kMaxHostSlabs) n = kMaxHostSlabs;
    if (n > tiles_l) n = tiles_l;
    if (!nested) n = 1;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(g_host_mutex);
    HostPipe* p = nullptr;
    st = host_pipe(dev.device, &p);
    if (st != ATB_OK) return st;
    cudaError_t e = cudaEventRecord(p->start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->in, p->start, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(p->out, p->start, 0);
    if (e != cudaSuccess) return cuda_error(e, "ordering the transfer streams after the caller's stream");

    const uint8_t* hs = static_cast<const uint8_t*>(h_src);
    uint8_t* hd = static_cast<uint8_t*>(h_dst);
    uint8_t* ds = reinterpret_cast<uint8_t*>(src->base);
    uint8_t* dd = reinterpret_cast<uint8_t*>(dst->base);
    for (uint64_t j = 0; j < n; ++j) {  // host -> device, slab by slab
        const uint64_t t0 = tiles_l * j / n, t1 = tiles_l * (j + 1) / n;
        uint64_t lo, hi;
        if (n == 1) {
            lo = 0;
            hi = inner_span(src, src->rank);
        } else {
            const uint64_t r1 = t1 * src->box[L] < src->dims[L] ? t1 * src->box[L] : src->dims[L];
            slab_bytes(src, t0 * src->box[L], r1, &lo, &hi);
        }
        e = cudaMemcpyAsync(ds + lo, hs + lo, hi - lo, cudaMemcpyHostToDevice, p->in);
        if (e == cudaSuccess) e = cudaEventRecord(p->landed[j], p->in);
        if (e != cudaSuccess) return cuda_error(e, "host-to-device slab copy");
    }
    for (uint64_t j = 0; j < n; ++j) {  // round trip of each slab's boxes once its rows have landed
        const uint64_t t0 = tiles_l * j / n, t1 = tiles_l * (j + 1) / n;
        e = cudaStreamWaitEvent(s, p->landed[j], 0);
        if (e != cudaSuccess) return cuda_error(e, "cudaStreamWaitEvent");
        st = launch_pipeline<kRoundtrip>(src, dst, nullptr, 0, nullptr, launch, s, nullptr, 0.0f, t0 * per_row,
                                         (t1 - t0) * per_row);
        if (st != ATB_OK) return st;
        e = cudaEventRecord(p->moved[j], s);
        if (e != cudaSuccess) return cuda_error(e, "cudaEventRecord");
    }
    for (uint64_t j = 0; j < n; ++j) {  // device -> host of each slab once its boxes are stored
        const uint64_t t0 = tiles_l * j / n, t1 = tiles_l * (j + 1) / n;
        uint64_t lo, hi;
        if (n == 1) {
            lo = 0;
            hi = inner_span(dst, dst->rank);
        } else {
            const uint64_t r1 = t1 * dst->box[L] < dst->dims[L] ? t1 * dst->box[L] : dst->dims[L];
            slab_bytes(dst, t0 * dst->box[L], r1, &lo, &hi);
        }
        e = cudaStreamWaitEvent(p->out, p->moved[j], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(hd + lo, dd + lo, hi - lo, cudaMemcpyDeviceToHost, p->out);
        if (e != cudaSuccess) return cuda_error(e, "device-to-host slab copy");
    }
    e = cudaEventRecord(p->end, p->out);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, p->end, 0);
    if (e != cudaSuccess) return cuda_error(e, "ordering the caller's stream after the transfers");
    return ATB_OK;
}

atb_status atb_tile_roundtrip_noalloc(const atb_tensor_map* src, const atb_tensor_map* dst, const int32_t* d_coords,
                                      uint64_t n, const atb_launch* launch, atb_stream_t stream,
                                      atb_device_report* report)
{
    clear_error();
    DeviceInfo dev;
    atb_status st = current_device(&dev);
    if (st != ATB_OK) return st;
    const size_t needed = sizeof(DeviceStatus);  // this kernel's scratch does not grow with the problem
    if (needed > ATB_NOALLOC_SCRATCH_BYTES)
        return set_error(ATB_ERR_ARG, "the round trip needs %zu bytes of scratch; the static array holds %d",
                         needed, ATB_NOALLOC_SCRATCH_BYTES);
    void* scratch = nullptr;
    st = noalloc_scratch_address(dev, &scratch);
    if (st != ATB_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The array keeps the previous call's record: start this one from zero.
    cudaError_t e = cudaMemsetAsync(scratch, 0, needed, s);
    if (e != cudaSuccess) return cuda_error(e, "cudaMemsetAsync(no-allocation scratch)");
    st = launch_pipeline<kRoundtrip>(src, dst, d_coords, n, nullptr, launch, s, static_cast<DeviceStatus*>(scratch));
    if (st != ATB_OK) return st;
    if (!report) return ATB_OK;
    e = cudaMemcpyAsync(report, scratch, needed, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_error(e, "cudaMemcpyAsync(no-allocation report)");
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_error(e, "cudaStreamSynchronize");
    return static_cast<atb_status>(report->code);
}

atb_status atb_last_launch(atb_launch_shape* out)
{
    if (!out) return set_error(ATB_ERR_ARG, "out is NULL");
    *out = g_last_shape;
    return ATB_OK;
}

atb_status atb_pipeline_smem_bytes(const atb_tensor_map* map, uint32_t stages, size_t* bytes)
{
    clear_error();
    if (!map_is_valid(map) || !bytes) return set_error(ATB_ERR_ARG, "map or bytes is NULL");
    if (stages < 1 || stages > kMaxStages)
        return set_error(ATB_ERR_ARG, "stages = %u is outside 1..%u", stages, kMaxStages);
    *bytes = smem_bytes_for(map, stages);
    DeviceInfo dev;
    atb_status st = current_device(&dev);
    if (st != ATB_OK) return st;
    if (*bytes > static_cast<size_t>(dev.smem_optin))
        return set_error(ATB_ERR_SMEM_BUDGET, "%zu bytes exceed the per-block limit of %d", *bytes, dev.smem_optin);
    return ATB_OK;
}

atb_status atb_tile_load(const atb_tensor_map* src, const int32_t* d_coords, uint64_t n, void* d_packed,
                         const atb_launch* launch, atb_stream_t stream)
{
    return launch_pipeline<kLoad>(src, nullptr, d_coords, n, d_packed, launch,
                                  reinterpret_cast<cudaStream_t>(stream));
}

atb_status atb_tile_store(const atb_tensor_map* dst, const int32_t* d_coords, uint64_t n, const void* d_packed,
                          const atb_launch* launch, atb_stream_t stream)
{
    return launch_pipeline<kStore>(nullptr, dst, d_coords, n, const_cast<void*>(d_packed), launch,
                                   reinterpret_cast<cudaStream_t>(stream));
}

atb_status atb_tile_roundtrip(const atb_tensor_map* src, const atb_tensor_map* dst, const int32_t* d_coords,
                              uint64_t n, const atb_launch* launch, atb_stream_t stream)
{
    return launch_pipeline<kRoundtrip>(src, dst, d_coords, n, nullptr, launch,
                                       reinterpret_cast<cudaStream_t>(stream));
}

atb_status atb_tile_roundtrip_add_f32(const atb_tensor_map* src, const atb_tensor_map* dst, const int32_t* d_coords,
                                      uint64_t n, float addend, const atb_launch* launch, atb_stream_t stream)
{
    return launch_pipeline<kRoundtripAddF32>(src, dst, d_coords, n, nullptr, launch,
                                             reinterpret_cast<cudaStream_t>(stream), nullptr, addend);
}

atb_status atb_selftest_wait_timeout(uint64_t timeout_ns, atb_stream_t stream)
{
    clear_error();
    DeviceStatus* status = nullptr;
    atb_status st = device_status_block(&status);
    if (st != ATB_OK) return st;
    wait_timeout_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status, timeout_ns);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "kernel launch");
    return ATB_OK;
}

}  // extern "C"
