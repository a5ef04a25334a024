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
//                   tensor store may not start (a negative origin) are written
//                   by the whole warp with plain clipped stores.
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

enum Mode : int { kRoundtrip = 0, kLoad = 1, kStore = 2 };

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
    uint32_t n_tiles;
    uint32_t esize;
    uint32_t box_bytes;
    uint32_t stage_bytes;
    uint32_t stages;
    uint32_t store_lag;     // groups left reading after each commit
    uint32_t contiguous;    // 1: CTA b takes a contiguous run of boxes
    uint32_t swizzle_bits;  // 0 none, 1 32B, 2 64B, 3 128B
    uint32_t dst_ragged_x;  // destination rows end inside a 16-byte chunk
    uint32_t l2_hints;      // ATB_HINT_* bits
};

// Shared-memory control words after the stage ring and the barriers.
struct Control {
    uint32_t abort;
    uint32_t issued;         // boxes whose stage the producer has armed
    uint32_t producer_done;
    uint32_t pad;
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
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                             const volatile uint32_t* abort)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::global_timer_ns();
    for (;;) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
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

__device__ __forceinline__ uint32_t tile_of(const PipeArgs& a, uint32_t k)
{
    if (a.contiguous) return blockIdx.x * ((a.n_tiles + gridDim.x - 1) / gridDim.x) + k;
    return blockIdx.x + k * gridDim.x;
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

// Whole-warp clipped store of one box image from shared memory.  The image
// byte at offset o lives at o with its 16-byte chunk number (bits 4..6) XORed
// by the low swizzle bits of its 128-byte line number (bits 7..9).
template <int R>
__device__ void plain_store_box(const PipeArgs& a, const int32_t (&c)[R], const uint8_t* stage, uint32_t lane)
{
    const uint32_t elems = a.box_bytes / a.esize;
    const uint32_t line_mask = (1u << a.swizzle_bits) - 1u;
    for (uint32_t e = lane; e < elems; e += 32) {
        uint32_t rest = e;
        bool inside = true;
        uint64_t addr = 0;
#pragma unroll
        for (int d = 0; d < R; ++d) {
            const uint32_t k = rest % a.box[d];
            rest /= a.box[d];
            const int64_t g = static_cast<int64_t>(c[d]) + k;
            if (g < 0 || g >= static_cast<int64_t>(a.dst_dims[d])) inside = false;
            else addr += static_cast<uint64_t>(g) * a.dst_strides[d];
        }
        if (!inside) continue;
        const uint32_t o = e * a.esize;
        const uint32_t so = o ^ (((o >> 7) & line_mask) << 4);
        uint8_t* dst = a.dst_base + addr;
        const uint8_t* src = stage + so;
        switch (a.esize) {
        case 1: *dst = *src; break;
        case 2: *reinterpret_cast<uint16_t*>(dst) = *reinterpret_cast<const uint16_t*>(src); break;
        case 4: *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(src); break;
        default: *reinterpret_cast<uint64_t*>(dst) = *reinterpret_cast<const uint64_t*>(src); break;
        }
    }
}

template <int MODE, int R>
__global__ void __launch_bounds__(kPipelineThreads, 1)
    tile_pipeline_kernel(const __grid_constant__ CUtensorMap src_map, const __grid_constant__ CUtensorMap dst_map,
                         const PipeArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t ring = (raw + (kStageAlignSwizzled - 1)) & ~(kStageAlignSwizzled - 1);
    uint8_t* const ring_ptr = smem_raw + (ring - raw);
    const uint32_t S = a.stages;
    const uint32_t full0 = ring + S * a.stage_bytes;  // full[s]  at full0 + 8 s
    const uint32_t empty0 = full0 + 8 * S;            // empty[s] at empty0 + 8 s
    Control* ctl = reinterpret_cast<Control*>(ring_ptr + S * a.stage_bytes + 16 * S);
    volatile uint32_t* abort_flag = &ctl->abort;

    const uint32_t warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (uint32_t s = 0; s < S; ++s) {
            ptx::mbar_init(full0 + 8 * s, 1);
            ptx::mbar_init(empty0 + 8 * s, 1);
        }
        ctl->abort = 0;
        ctl->issued = 0;
        ctl->producer_done = 0;
        ptx::fence_barrier_init();
        ptx::fence_proxy_async_smem();
    }
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
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        const bool hint = (a.l2_hints & ATB_HINT_LOAD_EVICT_FIRST) != 0;
        const uint64_t policy = hint ? ptx::policy_evict_first() : 0;
        for (uint32_t k = 0; k < count; ++k) {
            const uint32_t s = k % S, use = k / S;
            if (k >= S) {
                if (!wait_bounded(empty0 + 8 * s, (use - 1) & 1, a.timeout_ns, abort_flag)) {
                    if (!*abort_flag) {
                        record_error(a.status, ATB_ERR_TIMEOUT, static_cast<int32_t>(tile_of(a, k)),
                                     kWhereProducerWait);
                        *abort_flag = 1;
                    }
                    break;
                }
            }
            const uint32_t t = tile_of(a, k);
            const uint32_t full = full0 + 8 * s;
            const uint32_t dst = ring + s * a.stage_bytes;
            int32_t c[R];
            tile_origin<R>(a, t, c);
            const int32_t bad = origin_error<R>(a, c);
            if (bad) {
                record_error(a.status, bad, static_cast<int32_t>(t), kWhereProducerIssue);
                ptx::mbar_arrive(full);  // completes the phase with no bytes; the consumer skips the box
            } else {
                ptx::mbar_arrive_expect_tx(full, a.box_bytes);
                if (MODE == kStore)
                    ptx::bulk_load(dst, a.packed + static_cast<size_t>(t) * a.box_bytes, a.box_bytes, full);
                else if (hint)
                    ptx::tma_load_hint<R>(dst, &src_map, c, full, policy);
                else
                    ptx::tma_load<R>(dst, &src_map, c, full);
            }
            *reinterpret_cast<volatile uint32_t*>(&ctl->issued) = k + 1;
        }
        *reinterpret_cast<volatile uint32_t*>(&ctl->producer_done) = 1;
        return;
    }

    // ---------------------------------------------------------------- consumer
    const bool store_hint = (a.l2_hints & (ATB_HINT_STORE_EVICT_FIRST | ATB_HINT_STORE_EVICT_LAST)) != 0;
    const uint64_t store_policy = !store_hint ? 0
                                  : (a.l2_hints & ATB_HINT_STORE_EVICT_FIRST) ? ptx::policy_evict_first()
                                                                               : ptx::policy_evict_last();
    uint32_t next_release = 0;  // boxes [next_release, k) still have a group reading their stage
    uint32_t k = 0;
    bool failed = false;
    for (; k < count; ++k) {
        const uint32_t s = k % S, parity = (k / S) & 1;
        const uint32_t full = full0 + 8 * s;
        const bool ok = wait_bounded(full, parity, a.timeout_ns, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
            failed = true;
            break;
        }
        const uint32_t t = tile_of(a, k);
        int32_t c[R];
        tile_origin<R>(a, t, c);
        const bool skip = origin_error<R>(a, c) != 0;
        const int kind = MODE == kLoad ? kStoreTensor : (skip ? kStoreNothing : store_kind<R>(a, c));
        const uint32_t src = ring + s * a.stage_bytes;

        if (MODE != kLoad && kind != kStoreTensor) {
            // Rare path: retire every pending group so that stage bookkeeping
            // stays in order, then write (or drop) this box without the engine.
            if (lane == 0) {
                ptx::bulk_wait_read<0>();
                for (; next_release < k; ++next_release) ptx::mbar_arrive(empty0 + 8 * (next_release % S));
            }
            __syncwarp();
            if (kind == kStorePlain) plain_store_box<R>(a, c, ring_ptr + s * a.stage_bytes, lane);
            __syncwarp();
            if (lane == 0) {
                ptx::mbar_arrive(empty0 + 8 * s);
                next_release = k + 1;
            }
            continue;
        }
        if (MODE == kLoad && skip) {
            if (lane == 0) {
                ptx::bulk_wait_read<0>();
                for (; next_release < k; ++next_release) ptx::mbar_arrive(empty0 + 8 * (next_release % S));
                ptx::mbar_arrive(empty0 + 8 * s);
                next_release = k + 1;
            }
            continue;
        }
        if (lane == 0) {
            ptx::fence_proxy_async_smem();
            if (MODE == kLoad)
                ptx::bulk_store(a.packed + static_cast<size_t>(t) * a.box_bytes, src, a.box_bytes);
            else if (store_hint)
                ptx::tma_store_hint<R>(&dst_map, c, src, store_policy);
            else
                ptx::tma_store<R>(&dst_map, c, src);
            ptx::bulk_commit();
            ptx::bulk_wait_read_le(a.store_lag);
            for (; next_release + a.store_lag <= k; ++next_release)
                ptx::mbar_arrive(empty0 + 8 * (next_release % S));
        }
    }

    if (lane != 0) return;
    ptx::bulk_wait_all();
    if (!failed) return;

    // Failure: stop the producer, then wait (bounded) for every load it
    // already started so that no copy lands in shared memory after exit.
    if (!*abort_flag) {
        record_error(a.status, ATB_ERR_TIMEOUT, static_cast<int32_t>(tile_of(a, k)), kWhereConsumerWait);
        *abort_flag = 1;
    }
    const uint64_t deadline = ptx::global_timer_ns() + a.timeout_ns;
    while (!*reinterpret_cast<volatile uint32_t*>(&ctl->producer_done) && ptx::global_timer_ns() < deadline) {
    }
    const uint32_t issued = *reinterpret_cast<volatile uint32_t*>(&ctl->issued);
    for (uint32_t j = k; j < issued; ++j) wait_until(full0 + 8 * (j % S), (j / S) & 1, deadline);
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

atb_status prepare_kernel(KernelFn fn, const DeviceInfo& dev)
{
    // Opt every instantiation into the full per-block shared memory once per device.
    static const void* done[64][64];
    static int n_done[64];
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    for (int i = 0; i < n_done[dev.device]; ++i)
        if (done[dev.device][i] == reinterpret_cast<const void*>(fn)) return ATB_OK;
    cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, dev.smem_optin);
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute");
    if (n_done[dev.device] < 64) done[dev.device][n_done[dev.device]++] = reinterpret_cast<const void*>(fn);
    return ATB_OK;
}

// `caller_status`, when given, receives the kernel's error record instead of
// the device's lazily allocated status block.
template <int MODE>
atb_status launch_pipeline(const atb_tensor_map* src, const atb_tensor_map* dst, const int32_t* coords, uint64_t n,
                           void* packed, const atb_launch* cfg, cudaStream_t stream,
                           DeviceStatus* caller_status = nullptr)
{
    clear_error();
    const atb_tensor_map* shape = MODE == kStore ? dst : src;
    if ((MODE != kStore && !map_is_valid(src)) || (MODE != kLoad && !map_is_valid(dst)))
        return set_error(ATB_ERR_ARG, "tensor map is NULL or was not produced by atb_encode_tiled");
    if (MODE == kRoundtrip) {
        bool same = src->rank == dst->rank && src->esize == dst->esize && src->swizzle == dst->swizzle;
        for (uint32_t d = 0; same && d < src->rank; ++d) same = src->box[d] == dst->box[d];
        if (!same)
            return set_error(ATB_ERR_ARG,
                             "source and destination maps differ in rank, element size, box or swizzle");
    }
    if (MODE != kRoundtrip) {
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

    KernelFn fn = kernel_for_rank<MODE>(rank);
    st = prepare_kernel(fn, dev);
    if (st != ATB_OK) return st;

    uint32_t per_sm = cfg && cfg->ctas_per_sm ? cfg->ctas_per_sm : 0;
    if (!per_sm) {
        int fit = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&fit, fn, kPipelineThreads, smem);
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
    a.swizzle_bits = swizzle_bits(shape->swizzle);
    for (uint32_t d = 0; d < rank; ++d) {
        a.box[d] = shape->box[d];
        a.grid[d] = static_cast<uint32_t>((shape->dims[d] + shape->box[d] - 1) / shape->box[d]);
    }
    if (MODE != kLoad) {
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
    lc.blockDim = dim3(kPipelineThreads);
    lc.dynamicSmemBytes = smem;
    lc.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = attr;
    lc.numAttrs = cfg && cfg->no_pdl ? 0 : 1;
    cudaError_t e = cudaLaunchKernelEx(&lc, fn, src_map, dst_map, a);
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

}  // namespace
}  // namespace atb

using namespace atb;

extern "C" {

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
