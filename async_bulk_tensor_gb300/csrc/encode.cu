// Host side of libatb: error reporting, device checks, the status block, and
// the tensor-map encoder with one check per rule.
//
// The encoder follows "Day 76: The Tensor Memory Accelerator (TMA)", sections
// "The address arithmetic moves into a descriptor" (element type, rank, base,
// dimensions, byte strides, box; box extents at most 256, strides multiples of
// 16 bytes, base 16-byte aligned) and "Pitfalls" (the driver's encoder answers
// every broken rule with the same invalid-value code, so each rule is checked
// here first and reported on its own), plus "lesson 04: TMA - the async bulk
// copy engine", "The real toolchain - PTX and the descriptor object" (the map
// is encoded once on the host and passed to kernels as a grid constant).  The
// driver function is fetched through the runtime's entry-point query, so the
// library needs no link against the driver library.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "atb_internal.h"

namespace atb {

namespace {
thread_local char g_last_error[512] = "";
std::atomic<uint64_t> g_timeout_ns{1000000000ull};

std::mutex g_dev_mutex;
constexpr int kMaxDevices = 64;
DeviceInfo g_dev_info[kMaxDevices];
bool g_dev_known[kMaxDevices];
DeviceStatus* g_status[kMaxDevices];
}  // namespace

atb_status set_error(atb_status code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return code;
}

void clear_error() { g_last_error[0] = '\0'; }

atb_status cuda_error(int err, const char* what)
{
    return set_error(ATB_ERR_CUDA, "%s failed: %s", what, cudaGetErrorString(static_cast<cudaError_t>(err)));
}

uint64_t wait_timeout_ns() { return g_timeout_ns.load(std::memory_order_relaxed); }

atb_status current_device(DeviceInfo* info)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return set_error(ATB_ERR_ARG, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_dev_known[dev]) {
        DeviceInfo d{};
        d.device = dev;
        int* fields[] = {&d.sm_count, &d.cc_major, &d.cc_minor, &d.smem_optin, &d.smem_per_sm};
        cudaDeviceAttr attrs[] = {cudaDevAttrMultiProcessorCount, cudaDevAttrComputeCapabilityMajor,
                                  cudaDevAttrComputeCapabilityMinor, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                  cudaDevAttrMaxSharedMemoryPerMultiprocessor};
        for (int i = 0; i < 5; ++i) {
            e = cudaDeviceGetAttribute(fields[i], attrs[i], dev);
            if (e != cudaSuccess) return cuda_error(e, "cudaDeviceGetAttribute");
        }
        g_dev_info[dev] = d;
        g_dev_known[dev] = true;
    }
    *info = g_dev_info[dev];
    if (info->cc_major != 10 || info->cc_minor != 3)
        return set_error(ATB_ERR_UNSUPPORTED_DEVICE,
                         "device %d has compute capability %d.%d; this library carries sm_103a code only", dev,
                         info->cc_major, info->cc_minor);
    return ATB_OK;
}

atb_status device_status_block(DeviceStatus** out)
{
    DeviceInfo info;
    atb_status s = current_device(&info);
    if (s != ATB_OK) return s;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_status[info.device]) {
        void* p = nullptr;
        cudaError_t e = cudaMalloc(&p, sizeof(DeviceStatus));
        if (e != cudaSuccess) return cuda_error(e, "cudaMalloc(status block)");
        e = cudaMemset(p, 0, sizeof(DeviceStatus));
        if (e != cudaSuccess) {
            cudaFree(p);
            return cuda_error(e, "cudaMemset(status block)");
        }
        e = cudaDeviceSynchronize();
        if (e != cudaSuccess) {
            cudaFree(p);
            return cuda_error(e, "cudaDeviceSynchronize");
        }
        g_status[info.device] = static_cast<DeviceStatus*>(p);
    }
    *out = g_status[info.device];
    return ATB_OK;
}

bool map_is_valid(const atb_tensor_map* m)
{
    return m && m->magic == kMapMagic && m->rank >= 1 && m->rank <= ATB_MAX_RANK;
}

namespace {

uint32_t dtype_size(uint32_t dt)
{
    switch (dt) {
    case ATB_U8: return 1;
    case ATB_U16: case ATB_F16: case ATB_BF16: return 2;
    case ATB_U32: case ATB_I32: case ATB_F32: return 4;
    case ATB_U64: case ATB_I64: case ATB_F64: return 8;
    default: return 0;
    }
}

bool dtype_is_float(uint32_t dt)
{
    return dt == ATB_F16 || dt == ATB_BF16 || dt == ATB_F32 || dt == ATB_F64;
}

CUtensorMapDataType dtype_to_cu(uint32_t dt)
{
    switch (dt) {
    case ATB_U8: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
    case ATB_U16: return CU_TENSOR_MAP_DATA_TYPE_UINT16;
    case ATB_U32: return CU_TENSOR_MAP_DATA_TYPE_UINT32;
    case ATB_I32: return CU_TENSOR_MAP_DATA_TYPE_INT32;
    case ATB_U64: return CU_TENSOR_MAP_DATA_TYPE_UINT64;
    case ATB_I64: return CU_TENSOR_MAP_DATA_TYPE_INT64;
    case ATB_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    case ATB_F32: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    case ATB_F64: return CU_TENSOR_MAP_DATA_TYPE_FLOAT64;
    default: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    }
}

uint32_t swizzle_span(uint32_t sw)
{
    switch (sw) {
    case ATB_SWIZZLE_32B: return 32;
    case ATB_SWIZZLE_64B: return 64;
    case ATB_SWIZZLE_128B: return 128;
    default: return 0;
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn(atb_status* status)
{
    static std::mutex m;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::lock_guard<std::mutex> lock(m);
    if (fn) return fn;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !p) {
        *status = set_error(ATB_ERR_DRIVER, "cuTensorMapEncodeTiled is unavailable (%s, query result %d)",
                            cudaGetErrorString(e), static_cast<int>(q));
        cudaGetLastError();
        return nullptr;
    }
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return fn;
}

}  // namespace
}  // namespace atb

using namespace atb;

extern "C" {

int atb_version(void) { return ATB_VERSION; }

size_t atb_tensor_map_size(void) { return sizeof(atb_tensor_map); }

const char* atb_last_error(void) { return g_last_error; }

const char* atb_status_string(atb_status s)
{
    switch (s) {
    case ATB_OK: return "ATB_OK";
    case ATB_ERR_RANK: return "ATB_ERR_RANK";
    case ATB_ERR_BOX_DIM: return "ATB_ERR_BOX_DIM";
    case ATB_ERR_STRIDE_ALIGN: return "ATB_ERR_STRIDE_ALIGN";
    case ATB_ERR_BASE_ALIGN: return "ATB_ERR_BASE_ALIGN";
    case ATB_ERR_SMEM_ALIGN: return "ATB_ERR_SMEM_ALIGN";
    case ATB_ERR_SWIZZLE: return "ATB_ERR_SWIZZLE";
    case ATB_ERR_SWIZZLE_SPAN: return "ATB_ERR_SWIZZLE_SPAN";
    case ATB_ERR_INNER_BYTES: return "ATB_ERR_INNER_BYTES";
    case ATB_ERR_DTYPE: return "ATB_ERR_DTYPE";
    case ATB_ERR_DRIVER: return "ATB_ERR_DRIVER";
    case ATB_ERR_UNSUPPORTED_DEVICE: return "ATB_ERR_UNSUPPORTED_DEVICE";
    case ATB_ERR_SMEM_BUDGET: return "ATB_ERR_SMEM_BUDGET";
    case ATB_ERR_ARG: return "ATB_ERR_ARG";
    case ATB_ERR_TIMEOUT: return "ATB_ERR_TIMEOUT";
    case ATB_ERR_CUDA: return "ATB_ERR_CUDA";
    case ATB_ERR_COORD_ALIGN: return "ATB_ERR_COORD_ALIGN";
    case ATB_ERR_COORD_RANGE: return "ATB_ERR_COORD_RANGE";
    case ATB_ERR_STRIDE_RANGE: return "ATB_ERR_STRIDE_RANGE";
    case ATB_ERR_DIM_RANGE: return "ATB_ERR_DIM_RANGE";
    case ATB_ERR_RING_CHECK: return "ATB_ERR_RING_CHECK";
    }
    return "ATB_ERR_UNKNOWN";
}

void atb_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1000000000ull); }

atb_status atb_encode_tiled(atb_tensor_map* out, atb_dtype dtype, uint32_t rank, void* gbase,
                            const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                            const uint32_t* elem_strides, atb_swizzle swizzle, atb_l2_promotion l2_promotion,
                            atb_oob_fill oob_fill)
{
    clear_error();
    if (!out) return set_error(ATB_ERR_ARG, "out is NULL");
    memset(out, 0, sizeof *out);
    if (rank < 1 || rank > ATB_MAX_RANK)
        return set_error(ATB_ERR_RANK, "rank %u is outside 1..%d", rank, ATB_MAX_RANK);
    const uint32_t esize = dtype_size(static_cast<uint32_t>(dtype));
    if (!esize) return set_error(ATB_ERR_DTYPE, "unknown element type %d", static_cast<int>(dtype));
    if (!gbase) return set_error(ATB_ERR_ARG, "global base address is NULL");
    if (reinterpret_cast<uintptr_t>(gbase) % 16)
        return set_error(ATB_ERR_BASE_ALIGN, "global base address %p is not 16-byte aligned", gbase);
    if (!dims || !box) return set_error(ATB_ERR_ARG, "dims or box is NULL");
    if (rank > 1 && !strides_bytes) return set_error(ATB_ERR_ARG, "strides_bytes is NULL for rank %u", rank);
    for (uint32_t d = 0; d < rank; ++d)
        if (dims[d] == 0 || dims[d] > (1ull << 32))
            return set_error(ATB_ERR_DIM_RANGE, "dims[%u] = %llu is outside 1..2^32", d,
                             static_cast<unsigned long long>(dims[d]));
    for (uint32_t d = 1; d < rank; ++d) {
        const uint64_t s = strides_bytes[d];
        if (s % 16)
            return set_error(ATB_ERR_STRIDE_ALIGN, "strides_bytes[%u] = %llu is not a multiple of 16", d,
                             static_cast<unsigned long long>(s));
        if (s == 0 || s >= (1ull << 40))
            return set_error(ATB_ERR_STRIDE_RANGE, "strides_bytes[%u] = %llu is outside 16..2^40-16", d,
                             static_cast<unsigned long long>(s));
    }
    for (uint32_t d = 0; d < rank; ++d)
        if (box[d] == 0 || box[d] > 256)
            return set_error(ATB_ERR_BOX_DIM, "box[%u] = %u is outside 1..256", d, box[d]);
    const uint64_t inner_bytes = static_cast<uint64_t>(box[0]) * esize;
    if (inner_bytes % 16)
        return set_error(ATB_ERR_INNER_BYTES, "inner box bytes %llu (box[0] = %u x %u) are not a multiple of 16",
                         static_cast<unsigned long long>(inner_bytes), box[0], esize);
    if (static_cast<uint32_t>(swizzle) > ATB_SWIZZLE_128B)
        return set_error(ATB_ERR_SWIZZLE, "unknown swizzle mode %d", static_cast<int>(swizzle));
    const uint32_t span_bytes = swizzle_span(swizzle);
    if (span_bytes && inner_bytes != span_bytes)
        return set_error(ATB_ERR_SWIZZLE_SPAN, "inner box bytes %llu must equal the %u-byte swizzle span",
                         static_cast<unsigned long long>(inner_bytes), span_bytes);
    uint32_t steps[ATB_MAX_RANK] = {1, 1, 1, 1, 1};
    if (elem_strides) {
        if (elem_strides[0] != 1)
            return set_error(ATB_ERR_ARG, "elem_strides[0] = %u; the innermost traversal step must be 1",
                             elem_strides[0]);
        for (uint32_t d = 1; d < rank; ++d) {
            if (elem_strides[d] < 1 || elem_strides[d] > 8)
                return set_error(ATB_ERR_ARG, "elem_strides[%u] = %u is outside 1..8", d, elem_strides[d]);
            steps[d] = elem_strides[d];
        }
    }
    if (static_cast<uint32_t>(l2_promotion) > ATB_L2_PROMO_256B)
        return set_error(ATB_ERR_ARG, "unknown L2 promotion %d", static_cast<int>(l2_promotion));
    if (oob_fill != ATB_OOB_ZERO && oob_fill != ATB_OOB_NAN)
        return set_error(ATB_ERR_ARG, "unknown out-of-bounds fill %d", static_cast<int>(oob_fill));
    if (oob_fill == ATB_OOB_NAN && !dtype_is_float(static_cast<uint32_t>(dtype)))
        return set_error(ATB_ERR_DTYPE, "NaN out-of-bounds fill needs a floating-point element type, not dtype %d",
                         static_cast<int>(dtype));

    uint64_t box_bytes = esize;
    for (uint32_t d = 0; d < rank; ++d) box_bytes *= (box[d] + steps[d] - 1) / steps[d];
    if (box_bytes > 0xFFFFFFFFull) return set_error(ATB_ERR_BOX_DIM, "box of %llu bytes is too large",
                                                    static_cast<unsigned long long>(box_bytes));

    atb_status st = ATB_OK;
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn(&st);
    if (!fn) return st;

    cuuint64_t gdim[ATB_MAX_RANK];
    cuuint64_t gstride[ATB_MAX_RANK] = {0, 0, 0, 0, 0};
    cuuint32_t bdim[ATB_MAX_RANK];
    cuuint32_t estr[ATB_MAX_RANK];
    for (uint32_t d = 0; d < rank; ++d) {
        gdim[d] = dims[d];
        bdim[d] = box[d];
        estr[d] = steps[d];
        if (d + 1 < rank) gstride[d] = strides_bytes[d + 1];
    }
    alignas(64) CUtensorMap map;
    CUresult r = fn(&map, dtype_to_cu(dtype), rank, gbase, gdim, gstride, bdim, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, static_cast<CUtensorMapSwizzle>(swizzle),
                    static_cast<CUtensorMapL2promotion>(l2_promotion),
                    oob_fill == ATB_OOB_NAN ? CU_TENSOR_MAP_FLOAT_OOB_FILL_NAN_REQUEST_ZERO_FMA
                                            : CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return set_error(ATB_ERR_DRIVER, "cuTensorMapEncodeTiled refused the map (CUresult %d)", static_cast<int>(r));

    static_assert(sizeof(CUtensorMap) == sizeof(out->map), "tensor map size");
    memcpy(out->map, &map, sizeof map);

    // The second descriptor: box[0] widened by one 16-byte chunk, no swizzle,
    // everything else the same.  A box starting off the 16-byte grid along x
    // lies inside the wider box that starts at the origin rounded down to the
    // grid, which the engine may copy.
    const uint32_t wide0 = box[0] + 16 / esize;
    if (wide0 <= 256) {
        cuuint32_t wdim[ATB_MAX_RANK];
        for (uint32_t d = 0; d < rank; ++d) wdim[d] = d == 0 ? wide0 : box[d];
        alignas(64) CUtensorMap wmap;
        r = fn(&wmap, dtype_to_cu(dtype), rank, gbase, gdim, gstride, wdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, static_cast<CUtensorMapL2promotion>(l2_promotion),
               oob_fill == ATB_OOB_NAN ? CU_TENSOR_MAP_FLOAT_OOB_FILL_NAN_REQUEST_ZERO_FMA
                                       : CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r == CUDA_SUCCESS) {
            memcpy(out->map_wide, &wmap, sizeof wmap);
            out->wide_box0 = wide0;
        }
    }
    out->base = reinterpret_cast<uint64_t>(gbase);
    for (uint32_t d = 0; d < rank; ++d) {
        out->dims[d] = dims[d];
        out->strides[d] = d == 0 ? esize : strides_bytes[d];
        out->box[d] = box[d];
        out->elem_strides[d] = steps[d];
    }
    out->rank = rank;
    out->esize = esize;
    out->dtype = static_cast<uint32_t>(dtype);
    out->swizzle = static_cast<uint32_t>(swizzle);
    out->l2_promotion = static_cast<uint32_t>(l2_promotion);
    out->oob_fill = static_cast<uint32_t>(oob_fill);
    out->box_bytes = static_cast<uint32_t>(box_bytes);
    out->magic = kMapMagic;
    return ATB_OK;
}

size_t atb_box_bytes(const atb_tensor_map* map) { return map_is_valid(map) ? map->box_bytes : 0; }

uint64_t atb_grid_tiles(const atb_tensor_map* map)
{
    if (!map_is_valid(map)) return 0;
    uint64_t n = 1;
    for (uint32_t d = 0; d < map->rank; ++d) n *= (map->dims[d] + map->box[d] - 1) / map->box[d];
    return n;
}

atb_status atb_init_device(void)
{
    clear_error();
    DeviceStatus* st = nullptr;
    return device_status_block(&st);
}

int atb_status_block_allocated(void)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return -1;
    }
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    return g_status[dev] != nullptr ? 1 : 0;
}

atb_status atb_device_status(atb_stream_t stream, atb_device_report* report)
{
    clear_error();
    DeviceStatus* st = nullptr;
    atb_status rc = device_status_block(&st);
    if (rc != ATB_OK) return rc;
    // Read and clear the record in stream order, after everything already
    // queued on `stream`; work on other streams is not waited for.
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    DeviceStatus host{};
    cudaError_t e = cudaMemcpyAsync(&host, st, sizeof host, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return cuda_error(e, "cudaMemcpyAsync(status block)");
    e = cudaMemsetAsync(st, 0, sizeof host, s);
    if (e != cudaSuccess) return cuda_error(e, "cudaMemsetAsync(status block)");
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_error(e, "cudaStreamSynchronize");
    if (report) memcpy(report, &host, sizeof host);
    return static_cast<atb_status>(host.code);
}

}  // extern "C"
