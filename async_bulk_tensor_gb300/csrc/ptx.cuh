// Hand-written PTX for the async proxy on sm_103a: mbarriers with transaction
// counts, tensor-map (TMA) and 1-D bulk copies, bulk async groups, proxy
// fences.  Nothing here depends on libcu++ so that every wait can be bounded.
//
// Instruction forms follow the pages' description of the mechanism:
//   "lesson 04: TMA - the async bulk copy engine", sections "Load completion -
//   the mbarrier and the byte budget", "Store completion - commit group and
//   wait group" and "The real toolchain - PTX and the descriptor object";
//   "Day 76: The Tensor Memory Accelerator (TMA)", "Hint 2" (fence, store,
//   commit, wait_group.read) and "Pitfalls" (fence after barrier init).
#pragma once

#include <cstdint>

namespace atb {
namespace ptx {

__device__ __forceinline__ uint32_t smem_addr(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier --------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t arrivals)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(arrivals) : "memory");
}

// Makes barrier initialisation visible to the async proxy (the engine's
// complete_tx updates) and to the rest of the CTA after the block barrier.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (bulk copy engine) accesses.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One arrival plus a byte budget for the current phase.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// True once the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Same, letting the hardware suspend the thread for up to `suspend_ns` while
// the phase is incomplete (it resumes as soon as the phase completes).
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t suspend_ns)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity), "r"(suspend_ns)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- named barriers and shared-memory vectors -------------------------------
__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Barrier over `nthreads` threads that also ORs a predicate across them.
__device__ __forceinline__ bool named_barrier_or(uint32_t id, uint32_t nthreads, bool pred)
{
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred pin, pout;\n\t"
        "setp.ne.u32 pin, %1, 0;\n\t"
        "bar.red.or.pred pout, %2, %3, pin;\n\t"
        "selp.u32 %0, 1, 0, pout;\n\t}"
        : "=r"(out)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
        : "memory");
    return out != 0;
}

__device__ __forceinline__ uint4 ld_shared_v4_u32(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint8_t ld_shared_u8(uint32_t addr)
{
    uint16_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
    return static_cast<uint8_t>(v);
}

__device__ __forceinline__ uint16_t ld_shared_u16(uint32_t addr)
{
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_shared_v4_u32(uint32_t addr, const uint4& v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// ---- plain global loads through the read-only path ---------------------------
// Used only on tensors no thread of the launch writes.  Volatile, so that a
// batch of them stays ahead of the shared-memory stores that consume it.
__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(reinterpret_cast<uint64_t>(p)));
    return v;
}

__device__ __forceinline__ void ld_shared_v4_f32(uint32_t addr, float (&v)[4])
{
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void st_shared_v4_f32(uint32_t addr, const float (&v)[4])
{
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3])
                 : "memory");
}

// ---- programmatic dependent launch -------------------------------------------
// Lets the next grid on the stream be scheduled while this one finishes.
__device__ __forceinline__ void launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Blocks until every grid this one depends on has completed and its memory
// operations are visible; returns at once when there is no such grid.
__device__ __forceinline__ void wait_prerequisite_grids()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---- L2 cache policies -----------------------------------------------------
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---- tensor-map copies -----------------------------------------------------
__device__ __forceinline__ void prefetch_tensor_map(const void* map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Global -> shared box load, completion counted in bytes on `bar`.
template <int R>
__device__ __forceinline__ void tma_load(uint32_t dst, const void* map, const int32_t* c, uint32_t bar);

template <>
__device__ __forceinline__ void tma_load<1>(uint32_t dst, const void* map, const int32_t* c, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.1d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2}], [%3];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(bar)
        : "memory");
}
template <>
__device__ __forceinline__ void tma_load<2>(uint32_t dst, const void* map, const int32_t* c, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(c[1]), "r"(bar)
        : "memory");
}
template <>
__device__ __forceinline__ void tma_load<3>(uint32_t dst, const void* map, const int32_t* c, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(bar)
        : "memory");
}
template <>
__device__ __forceinline__ void tma_load<4>(uint32_t dst, const void* map, const int32_t* c, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(bar)
        : "memory");
}
template <>
__device__ __forceinline__ void tma_load<5>(uint32_t dst, const void* map, const int32_t* c, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4]),
        "r"(bar)
        : "memory");
}

// Shared -> global box store, completion tracked by the bulk async group.
template <int R>
__device__ __forceinline__ void tma_store(const void* map, const int32_t* c, uint32_t src);

template <>
__device__ __forceinline__ void tma_store<1>(const void* map, const int32_t* c, uint32_t src)
{
    asm volatile("cp.async.bulk.tensor.1d.global.shared::cta.tile.bulk_group [%0, {%1}], [%2];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c[0]), "r"(src)
                 : "memory");
}
template <>
__device__ __forceinline__ void tma_store<2>(const void* map, const int32_t* c, uint32_t src)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c[0]), "r"(c[1]), "r"(src)
                 : "memory");
}
template <>
__device__ __forceinline__ void tma_store<3>(const void* map, const int32_t* c, uint32_t src)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(src)
        : "memory");
}
template <>
__device__ __forceinline__ void tma_store<4>(const void* map, const int32_t* c, uint32_t src)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(src)
        : "memory");
}
template <>
__device__ __forceinline__ void tma_store<5>(const void* map, const int32_t* c, uint32_t src)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3, %4, %5}], [%6];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4]), "r"(src)
        : "memory");
}

// Same copies with an L2 cache-eviction policy from createpolicy.
template <int R>
__device__ __forceinline__ void tma_load_hint(uint32_t dst, const void* map, const int32_t* c, uint32_t bar,
                                              uint64_t policy);
template <>
__device__ __forceinline__ void tma_load_hint<1>(uint32_t dst, const void* map, const int32_t* c, uint32_t bar,
                                                 uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.1d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2}], [%3], %4;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(bar), "l"(policy)
        : "memory");
}
template <>
__device__ __forceinline__ void tma_load_hint<2>(uint32_t dst, const void* map, const int32_t* c, uint32_t bar,
                                                 uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(c[1]), "r"(bar), "l"(policy)
        : "memory");
}
template <>
__device__ __forceinline__ void tma_load_hint<3>(uint32_t dst, const void* map, const int32_t* c, uint32_t bar,
                                                 uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(bar), "l"(policy)
        : "memory");
}
template <>
__device__ __forceinline__ void tma_load_hint<4>(uint32_t dst, const void* map, const int32_t* c, uint32_t bar,
                                                 uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(bar), "l"(policy)
        : "memory");
}
template <>
__device__ __forceinline__ void tma_load_hint<5>(uint32_t dst, const void* map, const int32_t* c, uint32_t bar,
                                                 uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4]), "r"(bar), "l"(policy)
        : "memory");
}

template <int R>
__device__ __forceinline__ void tma_store_hint(const void* map, const int32_t* c, uint32_t src, uint64_t policy);
template <>
__device__ __forceinline__ void tma_store_hint<1>(const void* map, const int32_t* c, uint32_t src, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.1d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%1}], [%2], %3;"
        ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(src), "l"(policy)
        : "memory");
}
template <>
__device__ __forceinline__ void tma_store_hint<2>(const void* map, const int32_t* c, uint32_t src, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%1, %2}], [%3], %4;"
        ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(c[1]), "r"(src), "l"(policy)
        : "memory");
}
template <>
__device__ __forceinline__ void tma_store_hint<3>(const void* map, const int32_t* c, uint32_t src, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%1, %2, %3}], [%4], %5;"
        ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(src), "l"(policy)
        : "memory");
}
template <>
__device__ __forceinline__ void tma_store_hint<4>(const void* map, const int32_t* c, uint32_t src, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%1, %2, %3, %4}], [%5], %6;"
        ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(src), "l"(policy)
        : "memory");
}
template <>
__device__ __forceinline__ void tma_store_hint<5>(const void* map, const int32_t* c, uint32_t src, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.global.shared::cta.tile.bulk_group.L2::cache_hint [%0, {%1, %2, %3, %4, %5}], [%6], %7;"
        ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4]), "r"(src), "l"(policy)
        : "memory");
}

// Brings a box into L2 ahead of its load; no completion to wait for.
template <int R>
__device__ __forceinline__ void tma_prefetch_l2(const void* map, const int32_t* c);
template <>
__device__ __forceinline__ void tma_prefetch_l2<1>(const void* map, const int32_t* c)
{
    asm volatile("cp.async.bulk.prefetch.tensor.1d.L2.global.tile [%0, {%1}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c[0])
                 : "memory");
}
template <>
__device__ __forceinline__ void tma_prefetch_l2<2>(const void* map, const int32_t* c)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c[0]), "r"(c[1])
                 : "memory");
}
template <>
__device__ __forceinline__ void tma_prefetch_l2<3>(const void* map, const int32_t* c)
{
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c[0]), "r"(c[1]), "r"(c[2])
                 : "memory");
}
template <>
__device__ __forceinline__ void tma_prefetch_l2<4>(const void* map, const int32_t* c)
{
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3])
                 : "memory");
}
template <>
__device__ __forceinline__ void tma_prefetch_l2<5>(const void* map, const int32_t* c)
{
    asm volatile("cp.async.bulk.prefetch.tensor.5d.L2.global.tile [%0, {%1, %2, %3, %4, %5}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]), "r"(c[4])
                 : "memory");
}

// ---- 1-D bulk copies (contiguous byte ranges, 16-byte aligned, size % 16 == 0)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void bulk_store(void* dst, uint32_t src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
                 "r"(src), "r"(bytes)
                 : "memory");
}

// ---- bulk async groups -----------------------------------------------------
__device__ __forceinline__ void bulk_commit()
{
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N committed groups still read their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Runtime-depth variant (0..7); larger values clamp to 7.
__device__ __forceinline__ void bulk_wait_read_le(uint32_t n)
{
    switch (n) {
    case 0: bulk_wait_read<0>(); break;
    case 1: bulk_wait_read<1>(); break;
    case 2: bulk_wait_read<2>(); break;
    case 3: bulk_wait_read<3>(); break;
    case 4: bulk_wait_read<4>(); break;
    case 5: bulk_wait_read<5>(); break;
    case 6: bulk_wait_read<6>(); break;
    default: bulk_wait_read<7>(); break;
    }
}

// Wait until every committed group has fully completed (writes included).
__device__ __forceinline__ void bulk_wait_all()
{
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

}  // namespace ptx
}  // namespace atb
