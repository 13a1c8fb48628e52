// The streaming kernel's ring instantiation, the per-operation dispatch, and
// the device status word the streaming kernels report wait timeouts in.
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

ddp_status launch_stream(int op, StreamArgs& a, int dtype, void* stream)
{
    a.status = status_word();
    if (!a.status) return ddp::fail(DDP_E_CUDA, "stream kernel: device status word unavailable");
    a.store_bulk = op != OP_PACK && a.mode == DDP_ALLREDUCE;
    if (op == OP_RING)
        return a.wire == DDP_F32 ? launch_op<OP_RING, false>(a, dtype, stream) : launch_op<OP_RING, true>(a, dtype, stream);
    if (op == OP_PACK) return launch_stream_pack(a, dtype, stream);
    return launch_stream_fused(a, dtype, stream);
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
