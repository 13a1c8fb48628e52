// Internal helpers shared by the library's translation units (not part of the ABI).
#pragma once

#include <cstdarg>
#include <cstdint>

#include "ddp_bucket.h"

namespace ddp {

// Record the calling thread's error message and return `code`.
ddp_status fail(ddp_status code, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
// Clear the calling thread's message and return DDP_OK.
ddp_status ok();

constexpr int32_t kMaxReplicas = 64;

// Launch caches (occupancy, SM counts, function attributes, symbol addresses)
// are kept per device index below this bound, in atomics, so that several host
// threads and several devices in one process each see their own values.
constexpr int kMaxDevices = 64;
// The current device's index, or -1 when it cannot be read or is >= kMaxDevices
// (such a device is served without caching).
int current_device();
// Multiprocessors of the current device (cached per device; 132 if unknown).
int device_sm_count();

// Device data-path launchers (kernels.cu); arguments are already validated.
ddp_status launch_pack(const ddp_bucket_desc& b, const void* const* grads, const uint8_t* used, int32_t ld,
                       int32_t W, float* main_grad, int64_t stride, int32_t accumulate, void* stream);
ddp_status launch_allreduce(float* replicas, int64_t stride, int64_t n, int32_t W, int32_t mode, void* stream,
                            int32_t wire = DDP_F32);
ddp_status launch_unpack(const ddp_bucket_desc& b, const float* main_grad, int64_t stride, int32_t W,
                         int32_t mode, void* const* grads_out, int32_t ld, const uint8_t* global_used,
                         void* stream);
ddp_status launch_fused(const ddp_bucket_desc& b, const void* const* grads, const uint8_t* used, int32_t ld,
                        int32_t W, int32_t mode, int32_t accumulate, float* main_grad, int64_t stride,
                        void* const* grads_out, const uint8_t* global_used, void* stream, int32_t wire = DDP_F32);
ddp_status launch_pack_plain(const ddp_bucket_desc& b, const void* const* grads, const uint8_t* used, int32_t ld,
                             int32_t W, float* main_grad, int64_t stride, int32_t accumulate, void* stream);
ddp_status launch_pack_group(const ddp_bucket_desc* bs, float* const* mgs, int32_t nb, const void* const* grads,
                             const uint8_t* used, int32_t ld, int32_t W, int32_t accumulate, int64_t stride,
                             void* stream);
// Several buckets (bs[i] with main_grad copy mgs[i], may be null) in as few launches as possible.
ddp_status launch_fused_group(const ddp_bucket_desc* bs, float* const* mgs, int32_t nb, const void* const* grads,
                              const uint8_t* used, int32_t ld, int32_t W, int32_t mode, int32_t accumulate,
                              int64_t stride, void* const* grads_out, const uint8_t* global_used, void* stream,
                              int32_t wire = DDP_F32);

// Replicas and bucket size a PowerSGD state was planned for (powersgd.cu).
int32_t powersgd_replicas(const ddp_powersgd* h);
int64_t powersgd_numel(const ddp_powersgd* h);

}  // namespace ddp
