// The streaming kernel's ring instantiation, the per-operation dispatch, and
// the device status word the streaming kernels report wait timeouts in.
#include <mutex>

#include "stream_impl.cuh"

namespace ddpk {

ddp_status launch_stream_fused(StreamArgs& a, int dtype, void* stream);  // stream_fused.cu
ddp_status launch_stream_pack(StreamArgs& a, int dtype, void* stream);   // stream_pack.cu

namespace {
// bit 0: a streaming kernel gave up on an mbarrier wait
__device__ int g_device_status = 0;

// The status word's address on the current device, looked up once per device.
int* status_word()
{
    static std::atomic<int*> cached[ddp::kMaxDevices] = {};
    const int dev = ddp::current_device();
    int* p = dev >= 0 ? cached[dev].load(std::memory_order_acquire) : nullptr;
    if (!p) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, g_device_status) != cudaSuccess) return nullptr;
        p = static_cast<int*>(a);
        if (dev >= 0) cached[dev].store(p, std::memory_order_release);
    }
    return p;
}
}  // namespace

bool stream_supported(int op, int W, int dtype, bool acc, int mode)
{
    if (W < 2 || W > 16) return false;
    // the W copies of an allreduce result leave through bulk stores; a pack writes W different values
    const bool sbulk = op != OP_PACK && mode == DDP_ALLREDUCE;
    const int gb = (op == OP_RING || dtype == DDP_F32) ? 4 : 2;
    StagePlan p{};
    if (op == OP_RING) return plan_for(W, tile_for_w<OP_RING, false>(W), 4, false, sbulk, &p);
    const int tile = acc ? tile_for_w<OP_FUSED, true>(W) : tile_for_w<OP_FUSED, false>(W);
    return plan_for(W, tile, gb, acc, sbulk, &p);
}

namespace {

// Counters of the streaming kernels' work pools.  A launch with a pool owns one
// slot (claimed, finished; 128 bytes apart) for its lifetime: the last of its CTAs
// to stop claiming clears the slot.  Slots are handed out round robin per device,
// and a launch waits, on its stream, for the event recorded after the slot's
// previous launch, so two launches never share a slot at the same time whatever
// streams they run on.
constexpr int kPoolSlots = 64;
constexpr int kSlotWords = 32;
__device__ uint32_t g_pool_counters[kPoolSlots * kSlotWords];

// A launch moving at least this many operand elements (numel x W) gets a pool
// under DDP_KERNEL_AUTO: below it the static split's tail is short.
constexpr int64_t kPoolMinElems = int64_t{1} << 23;

struct PoolSlots {
    std::mutex mu;
    uint32_t next = 0;
    uint32_t* base = nullptr;
    cudaEvent_t done[kPoolSlots] = {};
    bool pending[kPoolSlots] = {};
};
PoolSlots g_pools[ddp::kMaxDevices];

bool wants_pool(const StreamArgs& a, void* stream)
{
    const int v = kernel_variant();
    if (v == DDP_KERNEL_STREAM) return false;
    if (v != DDP_KERNEL_STREAM_DYNAMIC && a.total * a.W < kPoolMinElems) return false;
    // a captured launch would replay with the slot it was captured with, outside the
    // event chain: captured launches keep the static split
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return cs == cudaStreamCaptureStatusNone;
}

}  // namespace

ddp_status launch_stream(int op, StreamArgs& a, int dtype, void* stream)
{
    a.status = status_word();
    if (!a.status) return ddp::fail(DDP_E_CUDA, "stream kernel: device status word unavailable");
    a.store_bulk = op != OP_PACK && a.mode == DDP_ALLREDUCE;
    a.dyn = nullptr;
    auto launch = [&]() -> ddp_status {
        if (op == OP_RING)
            return a.wire == DDP_F32 ? launch_op<OP_RING, false>(a, dtype, stream)
                                     : launch_op<OP_RING, true>(a, dtype, stream);
        if (op == OP_PACK) return launch_stream_pack(a, dtype, stream);
        return launch_stream_fused(a, dtype, stream);
    };
    const int dev = ddp::current_device();
    if (dev < 0 || !wants_pool(a, stream)) return launch();

    PoolSlots& P = g_pools[dev];
    std::lock_guard<std::mutex> lock(P.mu);
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!P.base) {
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_pool_counters) != cudaSuccess) {
            cudaGetLastError();
            return launch();   // no pool: the static split
        }
        P.base = static_cast<uint32_t*>(addr);
    }
    const uint32_t k = P.next % kPoolSlots;
    if (!P.done[k] && cudaEventCreateWithFlags(&P.done[k], cudaEventDisableTiming) != cudaSuccess) {
        cudaGetLastError();
        P.done[k] = nullptr;
        return launch();
    }
    if (P.pending[k]) {
        const cudaError_t e = cudaStreamWaitEvent(s, P.done[k], 0);
        if (e != cudaSuccess) return ddp::fail(DDP_E_CUDA, "cudaStreamWaitEvent: %s", cudaGetErrorString(e));
    }
    ++P.next;
    a.dyn = P.base + k * kSlotWords;
    const ddp_status st = launch();
    const cudaError_t e = cudaEventRecord(P.done[k], s);
    if (e != cudaSuccess) return ddp::fail(DDP_E_CUDA, "cudaEventRecord: %s", cudaGetErrorString(e));
    P.pending[k] = true;
    return st;
}

ddp_status read_device_status(void* stream, int32_t* out, int reset)
{
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_device_status, sizeof(int), 0, cudaMemcpyDeviceToHost,
                                              static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess && reset && v != 0) {
        const int zero = 0;
        e = cudaMemcpyToSymbolAsync(g_device_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                                    static_cast<cudaStream_t>(stream));
        if (e == cudaSuccess) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    }
    if (e != cudaSuccess) return ddp::fail(DDP_E_CUDA, "ddp_device_status: %s", cudaGetErrorString(e));
    *out = v;
    return ddp::ok();
}

namespace {

// The failure path of the streaming kernels' waits, on its own: one block waits
// (bounded by limit_ns) on an mbarrier that expects one arrival, which a thread
// makes only when `arrive` is set.  A thread that gives up records the timeout
// in the status word as the streaming kernels do; the block then invalidates
// the barrier and returns.
__global__ void wait_selftest_kernel(int* status, int arrive, uint64_t limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
    const bool got = wait_bounded(&bar, 0, limit_ns);
    if (!got) record_error(status, kErrWaitTimeout);
    __syncthreads();
    if (threadIdx.x == 0) asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(su32(&bar)) : "memory");
}

}  // namespace

ddp_status wait_selftest(int32_t arrive, int64_t limit_ns, void* stream)
{
    if (limit_ns < 1000 || limit_ns > static_cast<int64_t>(kWaitNs))
        return ddp::fail(DDP_E_INVAL, "ddp_wait_selftest: limit_ns = %lld outside [1000, %llu]",
                         static_cast<long long>(limit_ns), static_cast<unsigned long long>(kWaitNs));
    int* status = status_word();
    if (!status) return ddp::fail(DDP_E_CUDA, "ddp_wait_selftest: device status word unavailable");
    wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, arrive != 0,
                                                                          static_cast<uint64_t>(limit_ns));
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return ddp::fail(DDP_E_CUDA, "ddp_wait_selftest: launch failed: %s", cudaGetErrorString(err));
    return ddp::ok();
}

}  // namespace ddpk

extern "C" ddp_status ddp_wait_selftest(int32_t arrive, int64_t limit_ns, void* stream)
{
    return ddpk::wait_selftest(arrive, limit_ns, stream);
}

extern "C" ddp_status ddp_device_status(void* stream, int32_t* status, int32_t reset)
{
    if (!status) return ddp::fail(DDP_E_INVAL, "ddp_device_status: status is NULL");
    return ddpk::read_device_status(stream, status, reset);
}
