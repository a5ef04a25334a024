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
    uint8_t* dst_base;      // destination tensor (ragged plain stores)
    uint64_t timeout_ns;
    uint64_t dst_dims[ATB_MAX_RANK];
    uint64_t dst_strides[ATB_MAX_RANK];
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
#pragma unroll
            for (int d = 0; d < R; ++d) c[d] = static_cast<int32_t>(g[d] * a.box[d]);
        }
    }

    __device__ __forceinline__ void advance(const PipeArgs& a, uint32_t stages)
    {
        if (++stage == stages) {
            stage = 0;
            parity ^= 1u;
        }
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

// A listed origin the engine must not be given: beyond +-2^30, or not on a
// 16-byte boundary along the contiguous dimension.
template <int R>
__device__ __forceinline__ int32_t origin_error(const PipeArgs& a, const int32_t (&c)[R])
{
    if (!a.coords) return 0;
#pragma unroll
    for (int d = 0; d < R; ++d)
        if (c[d] > (1 << 30) || c[d] < -(1 << 30)) return ATB_ERR_COORD_RANGE;
    if ((static_cast<int64_t>(c[0]) * a.esize) & 15) return ATB_ERR_COORD_ALIGN;
    return 0;
}

enum StoreKind : int { kStoreTensor = 0, kStorePlain = 1, kStoreNothing = 2 };

// How a box reaches the destination tensor: nothing when it misses the tensor
// entirely; plain stores when it starts before the tensor (a tensor store may
// not start at a negative coordinate) or when it crosses the end of a row whose
// byte length is not a multiple of 16 (the engine writes such a row's last
// 16-byte chunk whole, past the row's end); a tensor store otherwise.
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
    return plain ? kStorePlain : kStoreTensor;
}

// Clipped store of one box image from shared memory by `nthreads` threads,
// 16 bytes at a time.  The swizzle moves whole 16-byte chunks (the chunk
// number, bits 4..6 of the image offset, is XORed with the low swizzle bits of
// the 128-byte line number, bits 7..9), and a box row starts on a 16-byte
// boundary in both spaces (the origin's x is 16-byte aligned, strides are
// multiples of 16), so a chunk that lies wholly inside the tensor moves as one
// vector; only a chunk cut by the end of a row moves element by element.
//
// Threads are laid out as `group` rows of `cpr` chunks (or, for rows wider
// than the thread count, one row at a time).  The box is walked plane by plane
// (dimensions 2..R-1, decomposed once per plane) and, inside a plane, row by
// row along dimension 1 with additions only: a single warp runs this loop
// alone, so short dependency chains matter more than instruction counts.
template <int R>
__device__ void plain_store_box(const PipeArgs& a, const int32_t (&c)[R], uint32_t stage, uint32_t tid,
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
template <int MODE, int R>
__device__ void producer_loop(const PipeArgs& a, const CUtensorMap& src_map, const Ring& r, uint32_t count)
{
    const bool hint = (a.l2_hints & ATB_HINT_LOAD_EVICT_FIRST) != 0;
    const uint64_t policy = hint ? ptx::policy_evict_first() : 0;
    const uint32_t S = r.stages;
    if (MODE != kStore && a.prefetch) {  // warm L2 with the first boxes
        for (uint32_t k = 0; k < a.prefetch && k < count; ++k) {
            int32_t c[R];
            tile_origin<R>(a, tile_of(a, k), c);
            if (!origin_error<R>(a, c)) ptx::tma_prefetch_l2<R>(&src_map, c);
        }
    }
    BoxCursor<R> cur;
    cur.init(a);
    for (uint32_t k = 0; k < count; ++k, cur.advance(a, S)) {
        const uint32_t s = cur.stage;
        if (MODE != kStore && a.prefetch && k + a.prefetch < count) {
            int32_t c[R];
            tile_origin<R>(a, tile_of(a, k + a.prefetch), c);
            if (!origin_error<R>(a, c)) ptx::tma_prefetch_l2<R>(&src_map, c);
        }
        // The origin first: for listed boxes it is a load from the coordinate
        // list, whose latency then overlaps the wait for the stage.
        int32_t c[R];
        cur.origin(a, c);
        // the stage's previous use completed the empty phase of the other parity
        if (k >= S && !wait_bounded(r.empty(s), cur.parity ^ 1u, a.timeout_ns, r.abort_flag(), a.suspend_ns)) {
            raise_abort(a, r, cur.t, kWhereProducerWait);
            break;
        }
        const uint32_t t = cur.t;
        ring_check_freed(a, r, s, k, t);
        if (a.checks & ATB_CHECK_RING)  // published by the arrive below (release order)
            *reinterpret_cast<volatile uint32_t*>(&r.ctl->filled[s]) = k + 1u;
        if (a.coords) {  // hand the origin over with the stage (published by the arrive below)
            volatile int32_t* slot = r.ctl->origin[s];
#pragma unroll
            for (int d = 0; d < R; ++d) slot[d] = c[d];
        }
        const int32_t bad = origin_error<R>(a, c);
        if (bad) {
            record_error(a.status, bad, static_cast<int32_t>(t), kWhereProducerIssue);
            ptx::mbar_arrive(r.full(s));  // completes the phase with no bytes; consumers skip the box
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

template <int MODE, int R>
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

    if (warp == 0) {
        if (lane == 0) producer_loop<MODE, R>(a, src_map, r, count);
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
        if (lane == 0) ring_check_filled(a, r, s, k, t);
        int32_t c[R] = {};
        if (!a.coords) {
            cur.origin(a, c);  // the tile grid: every lane follows the same cursor
        } else if (MODE == kLoad) {
            // a gathered box is drained by lane 0 alone; no other lane needs it
            if (lane == 0) landed_origin<R>(a, r, s, cur, c);
        } else {
            // Lane 0 reads the slot and the warp takes its copy: a lane that
            // ran late could otherwise read the slot after lane 0 has freed
            // the stage and the producer has refilled it.
            if (lane == 0) landed_origin<R>(a, r, s, cur, c);
#pragma unroll
            for (int d = 0; d < R; ++d) c[d] = __shfl_sync(0xffffffffu, c[d], 0);
        }
        const bool skip = origin_error<R>(a, c) != 0;
        // kLoad: kStoreTensor means "drain the image to the packed buffer"
        const int kind = skip ? kStoreNothing : (MODE == kLoad ? kStoreTensor : store_kind<R>(a, c));

        if (kind == kStorePlain) {
            // boxes the engine may not store: the warp writes them itself
            plain_store_box<R>(a, c, r.stage(s), lane, 32);
            __syncwarp();
        }
        if (lane == 0) {
            if (kind == kStoreTensor) {
                ptx::fence_proxy_async_smem();
                if (MODE == kLoad)
                    ptx::bulk_store(a.packed + static_cast<size_t>(t) * a.box_bytes, r.stage(s), a.box_bytes);
                else if (store_hint)
                    ptx::tma_store_hint<R>(&dst_map, c, r.stage(s), store_policy);
                else
                    ptx::tma_store<R>(&dst_map, c, r.stage(s));
                ptx::bulk_commit();
                pending.push(s, k);
            } else {
                ring_note_freed(a, r, s, k);
                ptx::mbar_arrive(r.empty(s));  // written by the warp, or nothing to write
            }
            pending.retire(a, r, k, a.store_lag);
        }
    }

    if (lane != 0) return;
    ptx::bulk_wait_all();
    if (failed) drain_after_failure(a, r, k);
}

// The pipeline with several consumer warps: warp 0 lane 0 produces, the
// consumer warps share each landed stage, and consumer thread 0 issues the
// tensor store.
//   ADD   round trip with an elementwise fp32 update in shared memory between
//         the load and the store ("Day 76: The Tensor Memory Accelerator
//         (TMA)", "Exercise" and "Solution": the threads change the tile in
//         shared memory, every writer publishes its writes across the proxy
//         line with fence.proxy.async, the group meets at a barrier, and one
//         thread issues the tensor store).  Each element becomes x + addend in
//         round-to-nearest fp32.  Two consumer warps.
//   !ADD  a plain round trip or store whose boxes come from a list, where
//         boxes that start before the tensor are common: four consumer warps
//         share the clipped stores of such boxes instead of one warp.
template <int MODE, int R, bool ADD>
__global__ void __launch_bounds__(32 + (ADD ? kUpdateConsumerThreads : kConsumerThreads), 1)
    tile_wide_kernel(const __grid_constant__ CUtensorMap src_map, const __grid_constant__ CUtensorMap dst_map,
                     const PipeArgs a, float addend)
{
    extern __shared__ uint8_t smem_raw[];
    const Ring r = ring_layout(a, smem_raw);
    const uint32_t S = r.stages;
    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) init_ring(r);
    if (threadIdx.x == 32) {
        if (MODE != kStore) ptx::prefetch_tensor_map(&src_map);
        ptx::prefetch_tensor_map(&dst_map);
    }
    ptx::launch_dependents();
    __syncthreads();
    ptx::wait_prerequisite_grids();

    const uint32_t count = my_tile_count(a);
    if (warp == 0) {
        if (lane == 0) producer_loop<MODE, R>(a, src_map, r, count);
        return;
    }

    // consumer threads: fewer for the update (measured faster), more for clipped stores
    constexpr uint32_t CT = ADD ? kUpdateConsumerThreads : kConsumerThreads;
    const uint32_t ct = threadIdx.x - 32;  // consumer thread 0 .. CT-1
    const uint32_t chunks = a.box_bytes / 16;
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
        if (ct == 0) ring_check_filled(a, r, s, k, cur.t);
        const int kind = origin_error<R>(a, c) != 0 ? kStoreNothing : store_kind<R>(a, c);
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
            plain_store_box<R>(a, c, r.stage(s), ct, CT);
            ptx::named_barrier_sync(1, CT);  // every reader is done with the stage
        }
        if (ct == 0) {
            if (kind == kStoreTensor) {
                if (!ADD) ptx::fence_proxy_async_smem();  // (with ADD every writer fenced already)
                ptx::tma_store<R>(&dst_map, c, r.stage(s));
                ptx::bulk_commit();
                pending.push(s, k);
            } else {
                ring_note_freed(a, r, s, k);
                ptx::mbar_arrive(r.empty(s));  // written by the threads, or nothing to write
            }
            pending.retire(a, r, k, a.store_lag);
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
using WideKernelFn = void (*)(const CUtensorMap, const CUtensorMap, const PipeArgs, float);

template <int MODE>
KernelFn kernel_for_rank(uint32_t rank)
{
    switch (rank) {
    case 1: return tile_pipeline_kernel<MODE, 1>;
    case 2: return tile_pipeline_kernel<MODE, 2>;
    case 3: return tile_pipeline_kernel<MODE, 3>;
    case 4: return tile_pipeline_kernel<MODE, 4>;
    default: return tile_pipeline_kernel<MODE, 5>;
    }
}

template <int MODE, bool ADD>
WideKernelFn wide_kernel_for_rank(uint32_t rank)
{
    switch (rank) {
    case 1: return tile_wide_kernel<MODE, 1, ADD>;
    case 2: return tile_wide_kernel<MODE, 2, ADD>;
    case 3: return tile_wide_kernel<MODE, 3, ADD>;
    case 4: return tile_wide_kernel<MODE, 4, ADD>;
    default: return tile_wide_kernel<MODE, 5, ADD>;
    }
}

uint32_t swizzle_bits(uint32_t sw) { return sw <= ATB_SWIZZLE_128B ? sw : 0; }

uint32_t stage_bytes_for(const atb_tensor_map* m)
{
    const uint32_t align = m->swizzle != ATB_SWIZZLE_NONE ? kStageAlignSwizzled : kStageAlignPlain;
    return (m->box_bytes + align - 1) / align * align;
}

size_t smem_bytes_for(const atb_tensor_map* m, uint32_t stages)
{
    return kStageAlignSwizzled + static_cast<size_t>(stages) * stage_bytes_for(m) + 16u * stages + sizeof(Control);
}

// Default pipeline shape, measured on GB300 round trips of a 512 MiB fp16
// tensor (32 KiB and 16 KiB boxes): three stages per CTA, two store groups in
// flight, and about 96 KiB of stages per SM (one CTA of 32 KiB boxes, two of
// 16 KiB boxes).  A stage is then busy for one load and one store read, and
// the ring always has a free stage for the next load.
constexpr uint32_t kDefaultStages = 3;
constexpr uint32_t kDefaultStoreGroups = 2;
constexpr uint64_t kStageBytesPerSm = 96u * 1024u;
constexpr uint64_t kMaxDefaultCtasPerSm = 8;

uint32_t default_stages(const atb_tensor_map* m, const DeviceInfo& dev)
{
    uint32_t s = kDefaultStages;
    while (s > 1 && smem_bytes_for(m, s) > static_cast<size_t>(dev.smem_optin)) --s;
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

// `caller_status`, when given, receives the kernel's error record instead of
// the device's lazily allocated status block.
// Launches one pipeline over boxes [first, first + count) of the list or grid
// (count = UINT64_MAX: all of them).
template <int MODE>
atb_status launch_pipeline(const atb_tensor_map* src, const atb_tensor_map* dst, const int32_t* coords, uint64_t n,
                           void* packed, const atb_launch* cfg, cudaStream_t stream,
                           DeviceStatus* caller_status = nullptr, float addend = 0.0f, uint64_t first = 0,
                           uint64_t count = UINT64_MAX)
{
    clear_error();
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
    const uint32_t stages = cfg && cfg->stages ? cfg->stages : default_stages(shape, dev);
    if (stages < 1 || stages > kMaxStages)
        return set_error(ATB_ERR_ARG, "stages = %u is outside 1..%u", stages, kMaxStages);
    const size_t smem = smem_bytes_for(shape, stages);
    if (smem > static_cast<size_t>(dev.smem_optin))
        return set_error(ATB_ERR_SMEM_BUDGET,
                         "%u stages of %u bytes need %zu bytes of shared memory; a block may have at most %d",
                         stages, stage_bytes_for(shape), smem, dev.smem_optin);
    if (n_tiles == 0) return ATB_OK;

    DeviceStatus* status = caller_status;
    if (!status) {
        st = device_status_block(&status);
        if (st != ATB_OK) return st;
    }

    // Listed boxes written to a tensor often start before it and need clipped
    // thread stores: those launches (and the fp32 update) use four consumer warps.
    constexpr int kBase = MODE == kRoundtripAddF32 ? kRoundtrip : MODE;
    const bool wide = MODE == kRoundtripAddF32 || (MODE != kLoad && coords != nullptr);
    WideKernelFn wide_fn = nullptr;
    if (MODE == kRoundtripAddF32) wide_fn = wide_kernel_for_rank<kRoundtrip, true>(rank);
    else if (wide) wide_fn = wide_kernel_for_rank<kBase == kLoad ? kRoundtrip : kBase, false>(rank);
    const void* fn = wide ? reinterpret_cast<const void*>(wide_fn) : reinterpret_cast<const void*>(kernel_for_rank<kBase>(rank));
    const uint32_t threads = MODE == kRoundtripAddF32 ? 32 + kUpdateConsumerThreads
                             : wide                     ? kTransformThreads
                                                        : kPipelineThreads;
    st = prepare_kernel(fn, dev);
    if (st != ATB_OK) return st;

    uint32_t per_sm = cfg && cfg->ctas_per_sm ? cfg->ctas_per_sm : 0;
    if (!per_sm) {
        int fit = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, fn, threads, smem);
        if (e != cudaSuccess) return cuda_error(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
        uint64_t want = kStageBytesPerSm / (static_cast<uint64_t>(stages) * stage_bytes_for(shape));
        want = want < 1 ? 1 : (want > kMaxDefaultCtasPerSm ? kMaxDefaultCtasPerSm : want);
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
    a.stage_bytes = stage_bytes_for(shape);
    a.stages = stages;
    uint32_t groups = cfg && cfg->store_groups ? cfg->store_groups : kDefaultStoreGroups;
    if (groups > stages) groups = stages;
    if (groups > 8) groups = 8;
    a.store_lag = groups - 1;
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

    alignas(64) CUtensorMap src_map;
    alignas(64) CUtensorMap dst_map;
    memcpy(&src_map, (MODE == kStore ? dst : src)->map, sizeof src_map);
    memcpy(&dst_map, (MODE == kLoad ? src : dst)->map, sizeof dst_map);

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
        e = cudaLaunchKernelEx(&lc, wide_fn, src_map, dst_map, a, addend);
    else
        e = cudaLaunchKernelEx(&lc, kernel_for_rank<kBase>(rank), src_map, dst_map, a);
    if (e != cudaSuccess) return cuda_error(e, "kernel launch");
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
