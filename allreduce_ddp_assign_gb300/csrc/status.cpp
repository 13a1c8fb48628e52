// Status strings and the per-thread last-error message.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <cstring>

#include "common.h"

namespace {
thread_local char g_message[1024] = "";
}

namespace ddp {

ddp_status fail(ddp_status code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_message, sizeof(g_message), fmt, ap);
    va_end(ap);
    return code;
}

ddp_status ok()
{
    g_message[0] = '\0';
    return DDP_OK;
}

int current_device()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

int device_sm_count()
{
    static std::atomic<int> cached[kMaxDevices] = {};
    const int dev = current_device();
    int v = dev >= 0 ? cached[dev].load(std::memory_order_relaxed) : 0;
    if (!v) {
        int d = 0;
        if (cudaGetDevice(&d) != cudaSuccess || cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d) != cudaSuccess ||
            v <= 0)
            v = 132;
        if (dev >= 0) cached[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

}  // namespace ddp

extern "C" const char* ddp_status_str(ddp_status s)
{
    switch (s) {
    case DDP_OK: return "DDP_OK";
    case DDP_E_INVAL: return "DDP_E_INVAL";
    case DDP_E_ALIGN: return "DDP_E_ALIGN";
    case DDP_E_CUDA: return "DDP_E_CUDA";
    case DDP_E_STATE: return "DDP_E_STATE";
    case DDP_E_INCOMPLETE: return "DDP_E_INCOMPLETE";
    case DDP_E_TIMEOUT: return "DDP_E_TIMEOUT";
    case DDP_E_CAPACITY: return "DDP_E_CAPACITY";
    default: return "DDP_E_UNKNOWN";
    }
}

extern "C" const char* ddp_last_error_message(void) { return g_message; }

extern "C" int32_t ddp_version(void) { return 100; }
