// Internal declarations shared by the translation units of libatb.
#pragma once

#include <cstddef>
#include <cstdint>

#include "atb.h"

namespace atb {

constexpr uint32_t kMapMagic = 0x31425441u;  // "ATB1"
constexpr uint32_t kMaxStages = 16;
constexpr uint32_t kPipelineThreads = 64;    // warp 0 producer, warp 1 consumer
constexpr uint32_t kConsumerThreads = 128;   // wide kernel, listed stores: warps 1..4 share clipped stores
constexpr uint32_t kTransformThreads = 32 + kConsumerThreads;
constexpr uint32_t kUpdateConsumerThreads = 64;  // wide kernel, fp32 update: warps 1..2 update the stage
constexpr uint32_t kStageAlignSwizzled = 1024;  // one period of the 128-byte swizzle
constexpr uint32_t kStageAlignPlain = 128;
// The engine's out-of-bounds NaN fill: 0x7FF7 in every 16-bit half (a NaN of
// f16, bf16, f32 and f64 alike).
constexpr uint32_t kNanFillWord = 0x7FF77FF7u;

// Device status block: the first error wins the code/block/tile/where slots,
// `errors` counts all of them.
struct DeviceStatus {
    int32_t code;
    int32_t block;
    int32_t tile;
    int32_t where;
    uint32_t errors;
    uint32_t reserved[3];
};
static_assert(sizeof(DeviceStatus) == sizeof(atb_device_report), "status layout");

enum Where : int32_t {
    kWhereProducerWait = 1,
    kWhereConsumerWait = 2,
    kWhereProducerIssue = 3,
    kWhereConsumerIssue = 4,
    kWhereSelftest = 5,
    kWhereProducerRing = 6,
    kWhereConsumerRing = 7,
};

// ---- host helpers (defined in encode.cu) -----------------------------------
atb_status set_error(atb_status code, const char* fmt, ...);
void clear_error();
atb_status cuda_error(int err, const char* what);

struct DeviceInfo {
    int device;
    int sm_count;
    int cc_major;
    int cc_minor;
    int smem_optin;   // max dynamic shared memory per block (opt-in)
    int smem_per_sm;  // shared memory per SM
};

// Current device's properties; ATB_ERR_UNSUPPORTED_DEVICE unless it is CC 10.3.
atb_status current_device(DeviceInfo* info);

// Lazily allocated status block of the current device.
atb_status device_status_block(DeviceStatus** out);

uint64_t wait_timeout_ns();

bool map_is_valid(const atb_tensor_map* m);

}  // namespace atb
