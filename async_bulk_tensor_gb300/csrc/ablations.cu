// Bandwidth ablations beside the TMA pipeline: the thread-issued copies the
// engine replaces.
//
//   copy_cpasync_kernel  every lane issues its own 16-byte cp.async (LDGSTS)
//                        into a shared-memory ring, then moves its bytes on
//                        with ld.shared.v4 / st.global.v4 -- "lesson 04: TMA -
//                        the async bulk copy engine", "What the issuing thread
//                        actually does" (Ampere's thread-issued async copy:
//                        registers bypassed, addresses still per lane).
//   copy_ldst_v4_kernel  coalesced ld.global.v4 / st.global.v4 through
//                        registers -- "Day 76: The Tensor Memory Accelerator
//                        (TMA)", the per-thread loads of the diagram in "The
//                        address arithmetic moves into a descriptor".
//   atb_copy_memcpy      cudaMemcpyAsync device to device -- the same page,
//                        "The copy does not use lane-level loads".
#include <cuda_runtime.h>

#include "atb_internal.h"

namespace atb {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kUnroll = 4;  // 16-byte pieces per lane per stage / iteration

__device__ __forceinline__ void ld_global_v4(const void* p, uint32_t (&r)[4])
{
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "l"(p));
}

__device__ __forceinline__ void st_global_v4(void* p, const uint32_t (&r)[4])
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
}

__device__ __forceinline__ void ld_shared_v4(uint32_t a, uint32_t (&r)[4])
{
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a)
                 : "memory");
}

__device__ __forceinline__ void cp_async_16(uint32_t smem, const void* gmem)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Grid-stride copy of n16 16-byte pieces; each lane keeps kUnroll loads in flight.
__global__ void __launch_bounds__(kCopyThreads) copy_ldst_v4_kernel(const uint8_t* __restrict__ src,
                                                                    uint8_t* __restrict__ dst, uint64_t n16)
{
    const uint64_t stride = static_cast<uint64_t>(gridDim.x) * kCopyThreads;
    uint64_t i = static_cast<uint64_t>(blockIdx.x) * kCopyThreads + threadIdx.x;
    for (; i + (kUnroll - 1) * stride < n16; i += kUnroll * stride) {
        uint32_t r[kUnroll][4];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) ld_global_v4(src + (i + u * stride) * 16, r[u]);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) st_global_v4(dst + (i + u * stride) * 16, r[u]);
    }
    for (; i < n16; i += stride) {
        uint32_t r[4];
        ld_global_v4(src + i * 16, r);
        st_global_v4(dst + i * 16, r);
    }
}

// Each CTA walks chunks of kCopyThreads * kUnroll * 16 bytes (16 KiB) with a
// STAGES-deep cp.async ring.  A lane only ever reads back the bytes its own
// cp.async wrote, so cp.async.wait_group alone orders the ring.
template <int STAGES>
__global__ void __launch_bounds__(kCopyThreads) copy_cpasync_kernel(const uint8_t* __restrict__ src,
                                                                    uint8_t* __restrict__ dst, uint64_t n16)
{
    extern __shared__ __align__(16) uint8_t ring[];
    constexpr uint64_t kChunk16 = static_cast<uint64_t>(kCopyThreads) * kUnroll;  // pieces per chunk
    const uint64_t n_chunks = (n16 + kChunk16 - 1) / kChunk16;
    const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(ring));

    auto issue = [&](uint64_t j, int stage) {
        const uint64_t chunk = blockIdx.x + j * gridDim.x;
        if (chunk < n_chunks) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const uint64_t piece = chunk * kChunk16 + u * kCopyThreads + threadIdx.x;
                if (piece < n16)
                    cp_async_16(base + (stage * kChunk16 + u * kCopyThreads + threadIdx.x) * 16, src + piece * 16);
            }
        }
        cp_async_commit();  // empty groups keep the count uniform at the tail
    };

    const uint64_t my_chunks = blockIdx.x < n_chunks ? (n_chunks - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
#pragma unroll
    for (int s = 0; s < STAGES - 1; ++s) issue(s, s);
    for (uint64_t j = 0; j < my_chunks; ++j) {
        issue(j + STAGES - 1, static_cast<int>((j + STAGES - 1) % STAGES));
        cp_async_wait<STAGES - 1>();
        const int stage = static_cast<int>(j % STAGES);
        const uint64_t chunk = blockIdx.x + j * gridDim.x;
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const uint64_t piece = chunk * kChunk16 + u * kCopyThreads + threadIdx.x;
            if (piece < n16) {
                uint32_t r[4];
                ld_shared_v4(base + (stage * kChunk16 + u * kCopyThreads + threadIdx.x) * 16, r);
                st_global_v4(dst + piece * 16, r);
            }
        }
    }
    cp_async_wait<0>();
}

atb_status check_flat(const void* src, void* dst, size_t bytes)
{
    if (!src || !dst) return set_error(ATB_ERR_ARG, "source or destination is NULL");
    if (reinterpret_cast<uintptr_t>(src) % 16 || reinterpret_cast<uintptr_t>(dst) % 16)
        return set_error(ATB_ERR_BASE_ALIGN, "source and destination must be 16-byte aligned");
    if (bytes % 16) return set_error(ATB_ERR_ARG, "bytes = %zu is not a multiple of 16", bytes);
    return ATB_OK;
}

unsigned flat_grid(const DeviceInfo& dev, const atb_launch* cfg, uint32_t default_per_sm, uint64_t work_items)
{
    uint64_t g = cfg && cfg->ctas ? cfg->ctas
                                  : static_cast<uint64_t>(dev.sm_count) *
                                        (cfg && cfg->ctas_per_sm ? cfg->ctas_per_sm : default_per_sm);
    if (g > work_items) g = work_items;
    if (g < 1) g = 1;
    if (g > 0x7FFFFFFFull) g = 0x7FFFFFFFull;
    return static_cast<unsigned>(g);
}

}  // namespace
}  // namespace atb

using namespace atb;

extern "C" {

atb_status atb_copy_ldst_v4(const void* d_src, void* d_dst, size_t bytes, const atb_launch* launch,
                            atb_stream_t stream)
{
    clear_error();
    atb_status st = check_flat(d_src, d_dst, bytes);
    if (st != ATB_OK) return st;
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != ATB_OK) return st;
    if (!bytes) return ATB_OK;
    const uint64_t n16 = bytes / 16;
    const unsigned grid = flat_grid(dev, launch, 8, (n16 + kCopyThreads - 1) / kCopyThreads);
    copy_ldst_v4_kernel<<<grid, kCopyThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(d_src), static_cast<uint8_t*>(d_dst), n16);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ATB_OK : cuda_error(e, "kernel launch");
}

atb_status atb_copy_cpasync(const void* d_src, void* d_dst, size_t bytes, const atb_launch* launch,
                            atb_stream_t stream)
{
    clear_error();
    atb_status st = check_flat(d_src, d_dst, bytes);
    if (st != ATB_OK) return st;
    DeviceInfo dev;
    st = current_device(&dev);
    if (st != ATB_OK) return st;
    if (!bytes) return ATB_OK;
    const uint32_t stages = launch && launch->stages ? launch->stages : 4;
    const uint64_t n16 = bytes / 16;
    const uint64_t chunk16 = static_cast<uint64_t>(kCopyThreads) * kUnroll;
    const size_t smem = static_cast<size_t>(stages) * chunk16 * 16;
    const unsigned grid = flat_grid(dev, launch, 2, (n16 + chunk16 - 1) / chunk16);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const void* fn = nullptr;
    switch (stages) {
    case 2: fn = reinterpret_cast<const void*>(copy_cpasync_kernel<2>); break;
    case 3: fn = reinterpret_cast<const void*>(copy_cpasync_kernel<3>); break;
    case 4: fn = reinterpret_cast<const void*>(copy_cpasync_kernel<4>); break;
    case 6: fn = reinterpret_cast<const void*>(copy_cpasync_kernel<6>); break;
    case 8: fn = reinterpret_cast<const void*>(copy_cpasync_kernel<8>); break;
    default: return set_error(ATB_ERR_ARG, "cp.async ablation supports 2, 3, 4, 6 or 8 stages, not %u", stages);
    }
    if (smem > static_cast<size_t>(dev.smem_optin))
        return set_error(ATB_ERR_SMEM_BUDGET, "%u stages need %zu bytes of shared memory", stages, smem);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute");
    const uint8_t* src8 = static_cast<const uint8_t*>(d_src);
    uint8_t* dst8 = static_cast<uint8_t*>(d_dst);
    switch (stages) {
    case 2: copy_cpasync_kernel<2><<<grid, kCopyThreads, smem, s>>>(src8, dst8, n16); break;
    case 3: copy_cpasync_kernel<3><<<grid, kCopyThreads, smem, s>>>(src8, dst8, n16); break;
    case 4: copy_cpasync_kernel<4><<<grid, kCopyThreads, smem, s>>>(src8, dst8, n16); break;
    case 6: copy_cpasync_kernel<6><<<grid, kCopyThreads, smem, s>>>(src8, dst8, n16); break;
    default: copy_cpasync_kernel<8><<<grid, kCopyThreads, smem, s>>>(src8, dst8, n16); break;
    }
    e = cudaGetLastError();
    return e == cudaSuccess ? ATB_OK : cuda_error(e, "kernel launch");
}

atb_status atb_copy_memcpy(const void* d_src, void* d_dst, size_t bytes, atb_stream_t stream)
{
    clear_error();
    if (!d_src || !d_dst) return set_error(ATB_ERR_ARG, "source or destination is NULL");
    DeviceInfo dev;
    atb_status st = current_device(&dev);
    if (st != ATB_OK) return st;
    if (!bytes) return ATB_OK;
    cudaError_t e =
        cudaMemcpyAsync(d_dst, d_src, bytes, cudaMemcpyDeviceToDevice, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATB_OK : cuda_error(e, "cudaMemcpyAsync");
}

}  // extern "C"
