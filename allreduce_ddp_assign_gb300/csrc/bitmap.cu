// The local-used bitmap all-reduce of find_unused_parameters.
//
// "Lecture 15: PyTorch DDP" section 4.2 and "DDP: PyTorch Distributed-
// Experiences on Accelerating Data Parallel Training" sections 2.2 and 3.2:
// one byte per parameter and replica says whether the replica used the
// parameter; the replicas' bitmaps are summed, and a parameter whose sum is
// zero was used by nobody.
//
// The work is a column count over a W x P byte matrix: HBM-bound, W*P bytes
// read and 5*P written per call.  Each thread owns 16 consecutive parameters:
// one 16-byte load per replica, the bytes turned into 0/1 four at a time in
// 32-bit words and added lane-wise (a byte lane holds at most 64, so no carry
// crosses lanes), then the four words are spread into 16 int32 counts and 16
// flag bytes.  Rows that are not 16-byte aligned, and the ragged tail, take
// a per-byte path.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include "common.h"

namespace {

constexpr int kThreads = 256;
constexpr int kGroup = 16;  // parameters per thread

// Per byte lane of x: 1 if the byte is nonzero, else 0.  (b & 0x7f) + 0x7f sets
// bit 7 exactly when the low seven bits are not all zero and cannot carry out
// of the lane; or-ing b itself covers a set top bit.
__device__ __forceinline__ uint32_t nonzero_lanes(uint32_t x)
{
    return ((x | ((x & 0x7f7f7f7fu) + 0x7f7f7f7fu)) >> 7) & 0x01010101u;
}

__global__ void __launch_bounds__(kThreads)
used_allreduce_kernel(const uint8_t* __restrict__ local, int64_t ld, int W, int64_t nparams, bool vec_rows,
                      int32_t* __restrict__ count, uint8_t* __restrict__ flag)
{
    const int64_t groups = (nparams + kGroup - 1) / kGroup;
    const int64_t step = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const bool vec_count = count && (reinterpret_cast<uintptr_t>(count) & 15) == 0;
    const bool vec_flag = flag && (reinterpret_cast<uintptr_t>(flag) & 15) == 0;
    for (int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < groups; g += step) {
        const int64_t p0 = g * kGroup;
        if (vec_rows && p0 + kGroup <= nparams) {
            uint32_t acc[4] = {0u, 0u, 0u, 0u};
            const uint8_t* src = local + p0;
#pragma unroll 4
            for (int w = 0; w < W; ++w) {
                const uint4 v = __ldcs(reinterpret_cast<const uint4*>(src + w * ld));
                acc[0] += nonzero_lanes(v.x);
                acc[1] += nonzero_lanes(v.y);
                acc[2] += nonzero_lanes(v.z);
                acc[3] += nonzero_lanes(v.w);
            }
            if (count) {
                int32_t c[kGroup];
#pragma unroll
                for (int j = 0; j < kGroup; ++j) c[j] = static_cast<int32_t>((acc[j >> 2] >> (8 * (j & 3))) & 0xffu);
                if (vec_count) {
                    int4* dst = reinterpret_cast<int4*>(count + p0);
#pragma unroll
                    for (int q = 0; q < 4; ++q) dst[q] = make_int4(c[4 * q], c[4 * q + 1], c[4 * q + 2], c[4 * q + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < kGroup; ++j) count[p0 + j] = c[j];
                }
            }
            if (flag) {
                const uint4 f = make_uint4(nonzero_lanes(acc[0]), nonzero_lanes(acc[1]), nonzero_lanes(acc[2]),
                                           nonzero_lanes(acc[3]));
                if (vec_flag) {
                    *reinterpret_cast<uint4*>(flag + p0) = f;
                } else {
                    const uint32_t fw[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                    for (int j = 0; j < kGroup; ++j) flag[p0 + j] = static_cast<uint8_t>(fw[j >> 2] >> (8 * (j & 3)));
                }
            }
        } else {
            const int64_t p1 = p0 + kGroup < nparams ? p0 + kGroup : nparams;
            for (int64_t p = p0; p < p1; ++p) {
                int32_t c = 0;
                for (int w = 0; w < W; ++w) c += local[w * ld + p] != 0;
                if (count) count[p] = c;
                if (flag) flag[p] = c > 0;
            }
        }
    }
}

// Blocks that are resident at once: SMs x blocks per SM (a grid of one wave).
int resident_blocks()
{
    static std::atomic<int> cached[ddp::kMaxDevices] = {};
    const int dev = ddp::current_device();
    int n = dev >= 0 ? cached[dev].load(std::memory_order_relaxed) : 0;
    if (!n) {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, used_allreduce_kernel, kThreads, 0) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
        n = ddp::device_sm_count() * per_sm;
        if (dev >= 0) cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

}  // namespace

extern "C" ddp_status ddp_used_allreduce(const uint8_t* local_used, int32_t ld, int32_t W, int32_t nparams,
                                         int32_t* global_count, uint8_t* global_used, void* stream)
{
    using ddp::fail;
    const char* fn = "ddp_used_allreduce";
    if (W < 1 || W > ddp::kMaxReplicas) return fail(DDP_E_INVAL, "%s: W = %d outside [1, %d]", fn, W, ddp::kMaxReplicas);
    if (nparams < 0) return fail(DDP_E_INVAL, "%s: nparams = %d < 0", fn, nparams);
    if (ld < nparams) return fail(DDP_E_INVAL, "%s: ld = %d < nparams = %d", fn, ld, nparams);
    if (!global_count && !global_used) return fail(DDP_E_INVAL, "%s: both outputs are NULL", fn);
    if (nparams == 0) return ddp::ok();
    if (!local_used) return fail(DDP_E_INVAL, "%s: local_used is NULL", fn);

    const bool vec_rows = (reinterpret_cast<uintptr_t>(local_used) & 15) == 0 && (ld & 15) == 0;
    const int64_t groups = (static_cast<int64_t>(nparams) + kGroup - 1) / kGroup;
    const int64_t want = (groups + kThreads - 1) / kThreads;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, resident_blocks())));
    used_allreduce_kernel<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        local_used, ld, W, nparams, vec_rows, global_count, global_used);
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return fail(DDP_E_CUDA, "%s: kernel launch failed: %s", fn, cudaGetErrorString(err));
    return ddp::ok();
}
