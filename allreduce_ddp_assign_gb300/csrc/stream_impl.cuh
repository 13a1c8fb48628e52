// TMA-pipelined streaming kernel: definitions shared by stream_ring.cu,
// stream_fused.cu and stream_pack.cu, each of which instantiates one operation.
#pragma once
// TMA-pipelined streaming kernel for the three hot operations: the ring-ordered
// reduction of packed replicas (ddp_bucket_allreduce) and the fused
// pack + reduce (+ unpack) pass over one bucket or a group of buckets
// (ddp_fused_bucket, ddp_fused_bucket_group, and the reducer's coalesced issue),
// and the no_sync pack of a bucket group (ddp_pack, ddp_pack_group).
//
// Arithmetic and decomposition are those of the plain kernels in kernels.cu:
// the buckets of a launch are laid end to end, each CTA takes an equal
// contiguous slice, and walks it in pieces cut wherever a bucket, a ring chunk
// or a parameter segment ends, so that inside a piece the ring order (chunk c:
// replicas c+1, ..., c) and the source tensors are fixed; every term is
// scaled with __fmul_rn and summed with __fadd_rn in that order.
//
// What differs is how bytes move:
//   warp 0      producer.  All 32 lanes walk the pieces together; lane w loads
//               replica w's pointers (one round trip per piece) and issues
//               replica w's cp.async.bulk copy into a ring of shared-memory
//               stages, completing on the stage's "full" mbarrier (expect-tx).
//               Misaligned heads, tails and pieces become scalar tiles that
//               carry only a descriptor.
//   warps 1..8  consumers.  Wait on "full", sum the tile in ring order from
//               shared memory (scalar tiles: from global memory), write the
//               result -- allreduce: staged once in shared memory and written to
//               every replica by TMA bulk stores; reduce-scatter: plain 16-byte
//               stores to the owning replica -- and release the stage on its
//               "empty" mbarrier.
// Several stages stay in flight per CTA, so HBM stays busy with few registers.
//
// Every mbarrier wait is bounded (iteration count and %globaltimer).  On
// expiry the kernel records an error bit in a device status word, all
// consumers leave together (a barrier vote), the producer waits (bounded) for
// the copies it issued, and the CTA returns with its outputs incomplete.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "common.h"
#include "device_common.cuh"

#ifndef DDP_STREAM_TILE_W
#define DDP_STREAM_TILE_W 16384    // tile elements x W (tiles are clamped to 1024..4096 elements)
#endif
#ifndef DDP_STREAM_TILE_MAX
#define DDP_STREAM_TILE_MAX 4096   // largest tile (elements)
#endif
#ifndef DDP_STREAM_L2_HINT
#define DDP_STREAM_L2_HINT 0       // 1: stream operands in with an L2 evict-first policy
#endif
#ifndef DDP_STREAM_TAPER
#define DDP_STREAM_TAPER 2         // > 1: the pool's last stretch in units of unit / DDP_STREAM_TAPER
#endif
#ifndef DDP_STREAM_BUDGET2_KB
#define DDP_STREAM_BUDGET2_KB 110  // shared memory per CTA when two CTAs share an SM
#endif

namespace ddpk {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreadsTma = 32 + kConsumers;
constexpr int kResDepth = 2;                 // result buffers for bulk stores
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s: a wait that long means something is broken
constexpr int kErrWaitTimeout = 1;
constexpr unsigned kFull = 0xffffffffu;

// elements per tile: DDP_STREAM_TILE_W / W, between 1024 and 4096, so each
// consumer thread owns 1, 2 or 4 vectors (W = 8: 2048 elements, 64 KB of fp32
// or 32 KB of bf16 staged per stage)
template <int OP, int WT, int DT, bool ACC>
__host__ __device__ constexpr int tile_of()
{
    constexpr int w = WT ? WT : 8;
    // staging main_grad as well (accumulating) doubles a stage: halve the tile
    constexpr int t = DDP_STREAM_TILE_W / w / (ACC ? 2 : 1);
    return (t >= 4096 && DDP_STREAM_TILE_MAX >= 4096) ? 4096 : ((t >= 2048 && DDP_STREAM_TILE_MAX >= 2048) ? 2048 : 1024);
}

struct TileDesc {
    float* mg;          // the tile's bucket in main_grad, replica 0 (nullptr: none)
    int64_t e0;         // first element, bucket-local
    int64_t off;        // first element of the tile's segment, bucket-local (gradient index = e - off)
    uint32_t src_mask;  // replicas with a gradient source
    int32_t len;        // elements
    int32_t c;          // ring chunk
    int32_t bulk;       // 1: operands staged in shared memory; 0: read from global memory
    int32_t stop;       // 1: no more tiles
    int32_t pad_;
};

// -- PTX wrappers ------------------------------------------------------------
__device__ __forceinline__ uint32_t su32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* b, uint32_t tx)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(tx) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return done != 0;
}
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol)
{
    if (DDP_STREAM_L2_HINT)
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
            "%4;" ::"r"(su32(dst)),
            "l"(src), "r"(bytes), "r"(su32(bar)), "l"(pol)
            : "memory");
    else
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         su32(dst)),
                     "l"(src), "r"(bytes), "r"(su32(bar))
                     : "memory");
}
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(su32(src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"r"(kConsumers) : "memory"); }
// barrier over the consumer warps that also ANDs a flag: every consumer takes the same branch after it
__device__ __forceinline__ bool consumers_all(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.and.pred po, 1, %2, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(kConsumers)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity; false after about limit_ns.
__device__ __forceinline__ bool wait_bounded(uint64_t* b, uint32_t parity, uint64_t limit_ns = kWaitNs)
{
    if (mbar_try_wait(b, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1; i < (1u << 28); ++i) {
        if (mbar_try_wait(b, parity)) return true;
        if ((i & 255u) == 0 && globaltimer() - t0 > limit_ns) break;
    }
    return false;
}

__device__ __forceinline__ void record_error(int* status, int code) { atomicOr(status, code); }

// -- shared-memory layout (dynamic) -------------------------------------------
struct Layout {
    uint32_t full, empty, desc, src, dst, res, data, mgd, cache, total;
};

// seg_cached: segment-table entries copied into shared memory (8 bytes of offset
// and 4 of parameter index each), placed after everything else
__host__ __device__ inline Layout layout_for(int ns, int W, int tile, int gb, bool acc, bool store_bulk,
                                             int seg_cached = 0)
{
    Layout L{};
    uint32_t o = 0;
    L.full = o;
    o += 8u * ns;
    L.empty = o;
    o += 8u * ns;
    L.desc = o;
    o += static_cast<uint32_t>(sizeof(TileDesc)) * ns;
    o = (o + 15u) & ~15u;
    L.src = o;
    o += 8u * ns * W;
    L.dst = o;
    o += 8u * ns * W;
    o = (o + 127u) & ~127u;
    L.res = o;
    if (store_bulk) o += kResDepth * static_cast<uint32_t>(tile) * 4u;
    L.data = o;
    o += static_cast<uint32_t>(ns) * W * tile * gb;
    o = (o + 127u) & ~127u;
    L.mgd = o;
    if (acc) o += static_cast<uint32_t>(ns) * W * tile * 4;
    L.cache = o;
    o += static_cast<uint32_t>(seg_cached) * 12u;
    L.total = o;
    return L;
}

// Last s in [0, nseg] with seg_offset[s] <= x, found by the whole warp
// (every lane gets the result); 32 probes per round.
__device__ __forceinline__ int warp_find_segment(const int64_t* seg_offset, int nseg, int64_t x, int lane)
{
    int lo = 0, hi = nseg + 1;
    while (hi - lo > 1) {
        const int step = (hi - lo + 31) / 32;
        const int idx = lo + step * (lane + 1);
        const bool le = idx < hi && seg_offset[idx] <= x;
        const int t = __popc(__ballot_sync(kFull, le));
        const int nlo = lo + step * t;
        int nhi = lo + step * (t + 1);
        if (nhi > hi) nhi = hi;
        lo = nlo;
        hi = nhi;
    }
    return lo;
}

// -- consumer arithmetic --------------------------------------------------------
template <int DT>
__device__ __forceinline__ float4 lds_grad4(const unsigned char* base, int i)
{
    if constexpr (DT == DDP_F32) {
        return *reinterpret_cast<const float4*>(base + 4 * i);
    } else {
        const uint2 u = *reinterpret_cast<const uint2*>(base + 2 * i);
        if constexpr (DT == DDP_BF16) {
            return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                               __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
        } else {
            const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
            const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
            return make_float4(lo.x, lo.y, hi.x, hi.y);
        }
    }
}

// WR: the instantiations that round the ring's arithmetic to a 16-bit wire type
// (the compression hook).  The others carry the plain fp32 multiply and add,
// with no wire test in the loop: there the test's predicated rounding path cost
// the 16-bit-input fused launches 35% (GPT-2's bf16 buckets: the consumer warps
// became ALU-bound) and an isolated 1 GiB ring launch 7%.  The fused fp32-input
// instantiations are the exception: they keep the runtime test on a.wire (and
// so serve every wire type), because back to back on ResNet-50's buckets they
// measured 4.5% faster with it (an isolated launch under ncu is 2.5% slower:
// the gain is in consecutive launches).
template <int OP, int WT, int DT, bool ACC, bool WR>
__global__ void __launch_bounds__(kThreadsTma) stream_kernel(const StreamArgs a)
{
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int kTile = tile_of<OP, WT, DT, ACC>();
    constexpr int kVpt = kTile / (4 * kConsumers);
    constexpr int gb = (OP == OP_RING) ? 4 : elem_bytes<DT>();
    const int W = WT ? WT : a.W;
    const int ns = a.ns;
    constexpr bool acc = ACC;
    const bool sbulk = a.store_bulk != 0;
    const Layout L = layout_for(ns, W, kTile, gb, acc, sbulk, a.seg_cached);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.full);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + L.empty);
    TileDesc* desc = reinterpret_cast<TileDesc*>(smem + L.desc);
    const void** srcp = reinterpret_cast<const void**>(smem + L.src);
    float** dstp = reinterpret_cast<float**>(smem + L.dst);
    float* res = reinterpret_cast<float*>(smem + L.res);
    unsigned char* data = smem + L.data;
    unsigned char* mgd = smem + L.mgd;
    int64_t* cache_off = reinterpret_cast<int64_t*>(smem + L.cache);
    int32_t* cache_par = reinterpret_cast<int32_t*>(smem + L.cache + 8u * static_cast<uint32_t>(a.seg_cached));
    __shared__ int abort_flag;

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < ns; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        abort_flag = 0;
        fence_mbar_init();
    }
    // every thread copies a share of the launch's segment tables: one round of
    // independent loads, after which finding a piece's segment, offset and
    // parameter reads shared memory only
    if (a.seg_cached) {
        for (int b = 0; b < a.nb; ++b) {
            const StreamSpan& S = a.span[b];
            if (!S.seg_offset) continue;
            for (int i = tid; i <= S.nseg; i += kThreadsTma) {
                cache_off[S.cache_base + i] = S.seg_offset[i];
                if (i < S.nseg) cache_par[S.cache_base + i] = S.seg_param[i];
            }
        }
    }
    __syncthreads();

    // this CTA's static slice of the head [0, a.head)
    const int64_t G = gridDim.x;
    const int64_t blk = blockIdx.x;
    const int64_t lo = (blk * a.head / G) & ~int64_t(15);
    const int64_t hi = (blk + 1 == G) ? a.head : (((blk + 1) * a.head / G) & ~int64_t(15));

    if (tid < 32) {
        // ===================== producer warp =====================
        int64_t k = 0;  // tiles emitted
        bool ok = true;
        const uint64_t pol = policy_evict_first();
        const void* my_src = nullptr;  // lane w: replica w's operands for the current piece
        float* my_dst = nullptr;

        auto claim = [&]() -> int {
            const int st = static_cast<int>(k % ns);
            bool good = true;
            if (k >= ns && lane == 0) good = wait_bounded(&empty[st], static_cast<uint32_t>(((k / ns) - 1) & 1));
            good = __shfl_sync(kFull, good, 0);
            if (!good) {
                if (lane == 0) {
                    record_error(a.status, kErrWaitTimeout);
                    atomicExch(&abort_flag, 1);
                }
                ok = false;
            }
            __syncwarp();
            fence_proxy_async();  // consumers' reads of the stage come before this warp's copies into it
            return st;
        };
        auto emit = [&](float* mgb, int c, int64_t off, int64_t e0, int32_t len, bool bulk, uint32_t mask) {
            const int st = claim();
            if (!ok) return;
            if (lane < W) {
                srcp[st * W + lane] = my_src;
                dstp[st * W + lane] = my_dst;
            }
            if (lane == 0) {
                TileDesc& d = desc[st];
                d.mg = mgb;
                d.e0 = e0;
                d.off = off;
                d.src_mask = mask;
                d.len = len;
                d.c = c;
                d.bulk = bulk ? 1 : 0;
                d.stop = 0;
            }
            __syncwarp();  // descriptor and pointers are written before the arrive publishes them
            uint32_t tx = 0;
            if (bulk)
                tx = static_cast<uint32_t>(__popc(mask)) * len * gb + (acc ? static_cast<uint32_t>(W) * len * 4 : 0);
            if (lane == 0) {
                if (tx) mbar_arrive_expect_tx(&full[st], tx);
                else mbar_arrive(&full[st]);
            }
            if (bulk && lane < W) {
                if (my_src)
                    bulk_g2s(data + (static_cast<size_t>(st) * W + lane) * kTile * gb,
                             static_cast<const unsigned char*>(my_src) + (e0 - off) * gb,
                             static_cast<uint32_t>(len) * gb, &full[st], pol);
                if (acc)
                    bulk_g2s(mgd + (static_cast<size_t>(st) * W + lane) * kTile * 4, mgb + lane * a.stride + e0,
                             static_cast<uint32_t>(len) * 4, &full[st], pol);
            }
            ++k;
        };

        // tiles of the element range [lo, hi), in order
        auto walk = [&](const int64_t lo, const int64_t hi) {
            int b = 0;
            int64_t x = lo;  // position in the launch's element space
            while (x < hi && ok) {
                while (b + 1 < a.nb && a.span[b].base + a.span[b].numel <= x) ++b;
                const StreamSpan& S = a.span[b];
                // the span's segment tables: the shared-memory copy when there is one
                const int64_t* const seg_off = (a.seg_cached && S.seg_offset) ? cache_off + S.cache_base : S.seg_offset;
                const int32_t* const seg_par = (a.seg_cached && S.seg_offset) ? cache_par + S.cache_base : S.seg_param;
                const int64_t end = lmin(hi, S.base + S.numel) - S.base;  // bucket-local end of this CTA's part
                const int64_t chunk = (OP == OP_PACK) ? lmax(1, S.numel) : lmax(1, (S.numel + W - 1) / W);
                int64_t e = x - S.base;
                int c = static_cast<int>(e / chunk);
                if (c >= W) c = W - 1;
                int s = seg_off ? warp_find_segment(seg_off, S.nseg, e, lane) : 0;
                while (e < end && ok) {
                    const int64_t c_end = (c + 1 >= W) ? S.numel : lmin(static_cast<int64_t>(c + 1) * chunk, S.numel);
                    int64_t s_off = 0, s_end = S.numel;
                    int p = -1;
                    if (seg_off) {
                        s_off = seg_off[s];
                        if (s < S.nseg) {
                            s_end = seg_off[s + 1];
                            p = seg_par[s];
                        }
                    }
                    const int64_t y = lmin(end, lmin(c_end, s_end));
                    if (y > e) {
                        my_src = nullptr;
                        my_dst = nullptr;
                        if (lane < W) {
                            if constexpr (OP == OP_RING) {
                                my_src = S.mg + lane * a.stride;
                            } else if (p >= 0 && p < a.ld) {
                                // flags and pointers read side by side: one round trip, not two
                                const int64_t slot = static_cast<int64_t>(lane) * a.ld + p;
                                const uint8_t u = a.used ? a.used[slot] : uint8_t{1};
                                const void* g = a.grads[slot];
                                const uint8_t gu = (a.grads_out && a.global_used) ? a.global_used[p] : uint8_t{1};
                                void* d = a.grads_out ? a.grads_out[slot] : nullptr;
                                my_src = u ? g : nullptr;
                                my_dst = gu ? static_cast<float*>(d) : nullptr;
                            }
                        }
                        bool lane_ok = true;
                        if (my_src && (reinterpret_cast<uintptr_t>(my_src) - static_cast<uintptr_t>(s_off * gb)) % 16 != 0)
                            lane_ok = false;
                        if (my_dst && (reinterpret_cast<uintptr_t>(my_dst) - static_cast<uintptr_t>(s_off * 4)) % 16 != 0)
                            lane_ok = false;
                        const bool aligned = __all_sync(kFull, lane_ok) && (S.mg == nullptr || S.mg_vec);
                        const uint32_t mask = __ballot_sync(kFull, my_src != nullptr);
                        // bulk tiles start and end on 16-byte multiples of every operand
                        constexpr int64_t gran = 16 / gb;
                        int64_t t = e;
                        if (aligned) {
                            const int64_t va = lmin(y, (e + gran - 1) / gran * gran);
                            const int64_t vb = lmax(va, y / gran * gran);
                            if (va > e) emit(S.mg, c, s_off, e, static_cast<int32_t>(va - e), false, mask);
                            for (t = va; t < vb && ok; t += kTile)
                                emit(S.mg, c, s_off, t, static_cast<int32_t>(lmin(kTile, vb - t)), true, mask);
                            t = vb;
                        }
                        for (; t < y && ok; t += kTile)
                            emit(S.mg, c, s_off, t, static_cast<int32_t>(lmin(kTile, y - t)), false, mask);
                    }
                    e = lmax(e, y);
                    while (c + 1 < W && static_cast<int64_t>(c + 1) * chunk <= e) ++c;
                    if (seg_off)
                        while (s < S.nseg && seg_off[s + 1] <= e) ++s;
                }
                x = S.base + e;
                if (b + 1 >= a.nb && e >= S.numel) break;  // past the last bucket
            }
        };
        walk(lo, hi);
        if (a.dyn) {
            // the pool: claim a unit after the previous one's tiles are issued (the
            // claim's round trip overlaps the stages still queued), until none is left.
            // The last stretch, one unit per CTA, goes out in units of unit / d
            // (d = DDP_STREAM_TAPER) where those are still whole tiles, so that the
            // last claimers finish closer together.
            const bool taper = DDP_STREAM_TAPER > 1 && a.unit / DDP_STREAM_TAPER >= kTile;
            const int64_t small = taper ? (a.unit / DDP_STREAM_TAPER) & ~int64_t(15) : a.unit;
            const int64_t z2 = taper ? lmax(a.head, (a.total - G * a.unit) & ~int64_t(15)) : a.total;
            const int64_t n1 = (z2 - a.head + a.unit - 1) / a.unit;
            const int64_t nunits = n1 + (a.total - z2 + small - 1) / small;
            while (ok) {
                uint32_t u = 0;
                if (lane == 0) u = atomicAdd(&a.dyn[0], 1u);
                u = __shfl_sync(kFull, u, 0);
                if (static_cast<int64_t>(u) >= nunits) break;
                if (static_cast<int64_t>(u) < n1) {
                    const int64_t x0 = a.head + static_cast<int64_t>(u) * a.unit;
                    walk(x0, lmin(z2, x0 + a.unit));
                } else {
                    const int64_t x0 = z2 + (static_cast<int64_t>(u) - n1) * small;
                    walk(x0, lmin(a.total, x0 + small));
                }
            }
            // the last CTA to stop claiming clears both counters for the slot's next
            // launch (which the launcher orders after this one)
            if (lane == 0 && atomicAdd(&a.dyn[1], 1u) == gridDim.x - 1) {
                atomicExch(&a.dyn[0], 0u);
                atomicExch(&a.dyn[1], 0u);
            }
        }
        // sentinel
        const int st = claim();
        if (ok) {
            if (lane == 0) {
                desc[st].stop = 1;
                mbar_arrive(&full[st]);
            }
            ++k;
        }
        // leave only when every copy this warp issued has landed
        if (lane == 0) {
            const int64_t first = lmax(0, k - ns);
            for (int64_t kk = first; kk < k; ++kk)
                wait_bounded(&full[static_cast<int>(kk % ns)], static_cast<uint32_t>((kk / ns) & 1));
        }
        return;
    }

    // ===================== consumers =====================
    const int ct = tid - 32;
    for (int64_t k = 0;; ++k) {
        const int st = static_cast<int>(k % ns);
        const bool got = wait_bounded(&full[st], static_cast<uint32_t>((k / ns) & 1));
        if (!got) record_error(a.status, kErrWaitTimeout);
        if (sbulk && ct == 0) bulk_wait_read<kResDepth - 1>();  // result buffer k % kResDepth is free again
        // one decision for all consumers (this barrier also publishes the line above)
        if (!consumers_all(got && !*static_cast<volatile int*>(&abort_flag))) break;
        const TileDesc d = desc[st];
        if (d.stop) break;
        const int c = d.c;
        float* const mgb = d.mg;
        const void* const* srcs = srcp + st * W;
        float* const* dsts = dstp + st * W;
        const bool early = (OP == OP_RING) || a.grads_out == nullptr;  // nothing else is read from the stage
        if constexpr (OP == OP_PACK) {
            // every replica keeps its own value: copy (or add) the staged gradient into main_grad
            if (d.bulk) {
#pragma unroll
                for (int v = 0; v < kVpt; ++v) {
                    const int i = 4 * (ct + v * kConsumers);
                    if (i >= d.len) continue;
                    const int64_t e = d.e0 + i;
                    for (int w = 0; w < W; ++w) {
                        const bool has = (d.src_mask >> w) & 1;
                        if (acc && !has) continue;  // no gradient: the bucket keeps its sum
                        float4 t = has ? lds_grad4<DT>(data + (static_cast<size_t>(st) * W + w) * kTile * gb, i)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                        if (acc)
                            t = Lane<4>::add(*reinterpret_cast<const float4*>(
                                                 mgd + (static_cast<size_t>(st) * W + w) * kTile * 4 + 4 * i),
                                             t);
                        Lane<4>::st(mgb + w * a.stride + e, t);
                    }
                }
            } else {
                for (int i = ct; i < d.len; i += kConsumers) {
                    const int64_t e = d.e0 + i;
                    for (int w = 0; w < W; ++w) {
                        const void* src = srcs[w];
                        if (acc && !src) continue;
                        float t = src ? Lane<1>::template ldg<DT>(src, e - d.off) : 0.f;
                        if (acc) t = Lane<1>::add(Lane<1>::ld(mgb + w * a.stride + e), t);
                        Lane<1>::st(mgb + w * a.stride + e, t);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            continue;
        }
        if (d.bulk) {
            float4 sum[kVpt];
#pragma unroll
            for (int v = 0; v < kVpt; ++v) {
                const int i = 4 * (ct + v * kConsumers);
                if (i >= d.len) continue;
                auto term = [&](int kk) {
                    int r = c + 1 + kk;
                    if (r >= W) r -= W;
                    float4 t;
                    if constexpr (OP == OP_RING) {
                        t = lds_grad4<DDP_F32>(data + (static_cast<size_t>(st) * W + r) * kTile * 4, i);
                    } else {
                        const bool has = (d.src_mask >> r) & 1;
                        t = has ? lds_grad4<DT>(data + (static_cast<size_t>(st) * W + r) * kTile * gb, i)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
                        if (acc) {
                            const float4 m = *reinterpret_cast<const float4*>(
                                mgd + (static_cast<size_t>(st) * W + r) * kTile * 4 + 4 * i);
                            t = has ? Lane<4>::add(m, t) : m;
                        }
                    }
                    if constexpr (WR || (DT == DDP_F32 && OP != OP_RING)) {
                        t = ring_term(t, a.inv_w, static_cast<float>(W), a.wire);
                        sum[v] = (kk == 0) ? t : ring_add(sum[v], t, a.wire);
                    } else {
                        t = Lane<4>::mul(t, a.inv_w);
                        sum[v] = (kk == 0) ? t : Lane<4>::add(sum[v], t);
                    }
                };
                if constexpr (WT > 0) {
#pragma unroll
                    for (int kk = 0; kk < WT; ++kk) term(kk);
                } else {
                    for (int kk = 0; kk < W; ++kk) term(kk);
                }
            }
            if (early) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
            }
            if (sbulk) {
                float* rb = res + (k % kResDepth) * kTile;
#pragma unroll
                for (int v = 0; v < kVpt; ++v) {
                    const int i = 4 * (ct + v * kConsumers);
                    if (i < d.len) *reinterpret_cast<float4*>(rb + i) = sum[v];
                }
                consumers_sync();
                if (ct == 0) {
                    fence_proxy_async();  // the tile's shared-memory writes, seen by the bulk copies
                    const uint32_t bytes = static_cast<uint32_t>(d.len) * 4;
                    if (mgb) {
                        if (a.mode == DDP_ALLREDUCE) {
                            for (int w = 0; w < W; ++w) bulk_s2g(mgb + w * a.stride + d.e0, rb, bytes);
                        } else {
                            bulk_s2g(mgb + c * a.stride + d.e0, rb, bytes);
                        }
                    }
                    if constexpr (OP == OP_FUSED) {
                        if (a.mode == DDP_ALLREDUCE) {
                            for (int w = 0; w < W; ++w)
                                if (dsts[w]) bulk_s2g(dsts[w] + (d.e0 - d.off), rb, bytes);
                        } else if (dsts[c]) {
                            bulk_s2g(dsts[c] + (d.e0 - d.off), rb, bytes);
                        }
                    }
                    bulk_commit();
                }
            } else {
#pragma unroll
                for (int v = 0; v < kVpt; ++v) {
                    const int i = 4 * (ct + v * kConsumers);
                    if (i >= d.len) continue;
                    const int64_t e = d.e0 + i;
                    if (mgb) {
                        if (a.mode == DDP_ALLREDUCE) {
                            for (int w = 0; w < W; ++w) Lane<4>::st(mgb + w * a.stride + e, sum[v]);
                        } else {
                            Lane<4>::st(mgb + c * a.stride + e, sum[v]);
                        }
                    }
                    if constexpr (OP == OP_FUSED) {
                        if (a.mode == DDP_ALLREDUCE) {
                            for (int w = 0; w < W; ++w)
                                if (dsts[w]) Lane<4>::st(dsts[w] + (e - d.off), sum[v]);
                        } else if (dsts[c]) {
                            Lane<4>::st(dsts[c] + (e - d.off), sum[v]);
                        }
                    }
                }
            }
            if (!early) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
            }
            continue;
        }
        // scalar tile: same arithmetic, operands straight from global memory
        for (int i = ct; i < d.len; i += kConsumers) {
            const int64_t e = d.e0 + i;
            float sum = 0.f;
            for (int kk = 0; kk < W; ++kk) {
                int r = c + 1 + kk;
                if (r >= W) r -= W;
                float t;
                if constexpr (OP == OP_RING) {
                    t = Lane<1>::ld(mgb + r * a.stride + e);
                } else {
                    const void* src = srcs[r];
                    t = src ? Lane<1>::template ldg<DT>(src, e - d.off) : 0.f;
                    if (acc) {
                        const float m = Lane<1>::ld(mgb + r * a.stride + e);
                        t = src ? Lane<1>::add(m, t) : m;
                    }
                }
                if constexpr (WR || (DT == DDP_F32 && OP != OP_RING)) {
                    t = ring_term(t, a.inv_w, static_cast<float>(W), a.wire);
                    sum = (kk == 0) ? t : ring_add(sum, t, a.wire);
                } else {
                    t = Lane<1>::mul(t, a.inv_w);
                    sum = (kk == 0) ? t : Lane<1>::add(sum, t);
                }
            }
            if (mgb) {
                if (a.mode == DDP_ALLREDUCE) {
                    for (int w = 0; w < W; ++w) Lane<1>::st(mgb + w * a.stride + e, sum);
                } else {
                    Lane<1>::st(mgb + c * a.stride + e, sum);
                }
            }
            if constexpr (OP == OP_FUSED) {
                if (a.mode == DDP_ALLREDUCE) {
                    for (int w = 0; w < W; ++w)
                        if (dsts[w]) Lane<1>::st(dsts[w] + (e - d.off), sum);
                } else if (dsts[c]) {
                    Lane<1>::st(dsts[c] + (e - d.off), sum);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (sbulk && ct == 0) bulk_wait_all();  // every bulk store of this CTA has completed
}

// -- host side ------------------------------------------------------------------
constexpr uint32_t kSmemBudget2 = DDP_STREAM_BUDGET2_KB * 1024;  // two CTAs per SM
constexpr uint32_t kSmemBudget1 = 220 * 1024;                    // one CTA per SM: the stage ring
// Fraction of a launch with a pool that is split statically (in 1/16ths), and the
// operand bytes staged per pool unit (whole tiles, at least one).  Measured on
// GB300: the ring reduction of packed replicas does best with the larger pool of
// smaller units (its units cost the producer no table reads), the launches that
// read gradients through the segment tables with the smaller pool of larger units
// (ResNet-50 W = 8, coalesced: 6.01 TB/s at 10/16 and 64 KB, 6.22 at 12/16 and
// 128 KB, 6.12 at 12/16 and 256 KB; the 64 MiB x 2 ring: 5.62 against 5.39).
#ifndef DDP_STREAM_HEAD_16THS
#define DDP_STREAM_HEAD_16THS 12
#endif
#ifndef DDP_STREAM_UNIT_KB
#define DDP_STREAM_UNIT_KB 128
#endif
#ifndef DDP_STREAM_RING_HEAD_16THS
#define DDP_STREAM_RING_HEAD_16THS 10
#endif
#ifndef DDP_STREAM_RING_UNIT_KB
#define DDP_STREAM_RING_UNIT_KB 64
#endif
template <int OP> constexpr int64_t head_sixteenths()
{
    return OP == OP_RING ? DDP_STREAM_RING_HEAD_16THS : DDP_STREAM_HEAD_16THS;
}
template <int OP> constexpr int64_t unit_bytes()
{
    return (OP == OP_RING ? DDP_STREAM_RING_UNIT_KB : DDP_STREAM_UNIT_KB) * 1024;
}

// stages that fit the budget (0 if fewer than two)
inline int stages_for(int W, int tile, int gb, bool acc, bool sbulk, uint32_t budget)
{
    for (int ns = 8; ns >= 2; --ns)
        if (layout_for(ns, W, tile, gb, acc, sbulk).total <= budget) return ns;
    return 0;
}

struct StagePlan {
    int ns;
    uint32_t bytes, budget;
};

inline bool plan_for(int W, int tile, int gb, bool acc, bool sbulk, StagePlan* p)
{
    int ns = stages_for(W, tile, gb, acc, sbulk, kSmemBudget2);
    uint32_t budget = kSmemBudget2;
    if (ns < 3) {
        ns = stages_for(W, tile, gb, acc, sbulk, kSmemBudget1);
        budget = kSmemBudget1;
    }
    if (ns < 2) return false;
    *p = StagePlan{ns, layout_for(ns, W, tile, gb, acc, sbulk).total, budget};
    return true;
}

// The most dynamic shared memory a CTA of the current device may use (per device).
inline uint32_t smem_optin_limit()
{
    static std::atomic<uint32_t> cached[ddp::kMaxDevices] = {};
    const int dev = ddp::current_device();
    uint32_t v = dev >= 0 ? cached[dev].load(std::memory_order_relaxed) : 0;
    if (!v) {
        int x = 0, d = 0;
        if (cudaGetDevice(&d) != cudaSuccess ||
            cudaDeviceGetAttribute(&x, cudaDevAttrMaxSharedMemoryPerBlockOptin, d) != cudaSuccess || x <= 0)
            x = static_cast<int>(kSmemBudget1);
        v = static_cast<uint32_t>(x);
        if (dev >= 0) cached[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

template <int OP, int WT, int DT, bool ACC, bool WR>
ddp_status launch_instance(StreamArgs& a, void* stream)
{
    auto kern = stream_kernel<OP, WT, DT, ACC, WR>;
    constexpr int tile = tile_of<OP, WT, DT, ACC>();
    constexpr int gb = (OP == OP_RING) ? 4 : elem_bytes<DT>();
    StagePlan p{};
    if (!plan_for(a.W, tile, gb, ACC, a.store_bulk, &p))
        return ddp::fail(DDP_E_INVAL, "stream kernel: no stage layout fits for W = %d", a.W);
    a.ns = p.ns;
    // the segment tables go into shared memory when they fit beside the stages
    // without costing a CTA per SM: up to the device's limit for one CTA per SM, up
    // to the two-CTA budget otherwise
    int64_t entries = 0;
    for (int b = 0; b < a.nb; ++b) {
        a.span[b].cache_base = static_cast<int32_t>(entries);
        if (a.span[b].seg_offset) entries += a.span[b].nseg + 1;
    }
    const uint32_t room = (p.budget == kSmemBudget1) ? smem_optin_limit() : kSmemBudget2;
    a.seg_cached = (entries > 0 && p.bytes + 12 * entries <= room) ? static_cast<int32_t>(entries) : 0;
    const uint32_t bytes = layout_for(p.ns, a.W, tile, gb, ACC, a.store_bulk, a.seg_cached).total;
    // the pool: whole tiles of about kUnitBytes of staged operands
    if (a.dyn) {
        const int64_t stage = static_cast<int64_t>(a.W) * tile * (gb + (ACC ? 4 : 0));
        a.unit = static_cast<int32_t>(tile * lmax(1, unit_bytes<OP>() / stage));
        a.head = (a.total * head_sixteenths<OP>() / 16) & ~int64_t(15);
    } else {
        a.unit = 0;
        a.head = a.total;
    }
    // Per device: the dynamic shared memory this instantiation may use (a function
    // attribute, set once per device and raised when a launch needs more), and the
    // resident CTAs per SM at the last stage-ring size asked for, packed as
    // (bytes << 32 | CTAs) so that the pair is read and written as one value.
    static std::atomic<uint32_t> configured[ddp::kMaxDevices] = {};
    static std::atomic<uint64_t> occupancy[ddp::kMaxDevices] = {};
    const int dev = ddp::current_device();
    const uint32_t want_attr = bytes > p.budget ? bytes : p.budget;
    if (dev < 0 || configured[dev].load(std::memory_order_acquire) < want_attr) {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, want_attr);
        if (e != cudaSuccess) return ddp::fail(DDP_E_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
        if (dev >= 0) {
            uint32_t cur = configured[dev].load(std::memory_order_relaxed);
            while (cur < want_attr && !configured[dev].compare_exchange_weak(cur, want_attr, std::memory_order_release)) {
            }
        }
    }
    const uint64_t packed = dev >= 0 ? occupancy[dev].load(std::memory_order_relaxed) : 0;
    int occ = static_cast<int>(packed & 0xffffffffu);
    if (packed == 0 || (packed >> 32) != p.bytes) {
        int v = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, kThreadsTma, p.bytes) != cudaSuccess || v < 1) v = 1;
        occ = v;
        if (dev >= 0) occupancy[dev].store((static_cast<uint64_t>(p.bytes) << 32) | static_cast<uint32_t>(v),
                                           std::memory_order_relaxed);
    }
    // small launches: spread down to 16-element slices so that the pieces (one per ring
    // chunk, at least) run in parallel CTAs rather than through one CTA's pipeline
    const int64_t want = (a.total + 15) / 16;
    const int grid = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, int64_t(ddp::device_sm_count()) * occ)));
    kern<<<grid, kThreadsTma, bytes, static_cast<cudaStream_t>(stream)>>>(a);
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return ddp::fail(DDP_E_CUDA, "stream kernel launch failed: %s", cudaGetErrorString(err));
    return ddp::ok();
}

template <int OP, int DT, bool ACC, bool WR>
ddp_status dispatch_w(StreamArgs& a, void* stream)
{
    switch (a.W) {
    case 2: return launch_instance<OP, 2, DT, ACC, WR>(a, stream);
    case 4: return launch_instance<OP, 4, DT, ACC, WR>(a, stream);
    case 8: return launch_instance<OP, 8, DT, ACC, WR>(a, stream);
    case 16: return launch_instance<OP, 16, DT, ACC, WR>(a, stream);
    default: return launch_instance<OP, 0, DT, ACC, WR>(a, stream);
    }
}

template <int OP, bool ACC>
int tile_for_w(int W)
{
    switch (W) {
    case 2: return tile_of<OP, 2, DDP_F32, ACC>();
    case 4: return tile_of<OP, 4, DDP_F32, ACC>();
    case 8: return tile_of<OP, 8, DDP_F32, ACC>();
    case 16: return tile_of<OP, 16, DDP_F32, ACC>();
    default: return tile_of<OP, 0, DDP_F32, ACC>();
    }
}

// the operations a launch of one TU covers.  WR selects the instantiations with
// wire rounding (ring launches, and fused launches of 16-bit gradients); fused
// launches of fp32 gradients always take the instantiations with the runtime
// wire test.
template <int OP, bool WR>
ddp_status launch_op(StreamArgs& a, int dtype, void* stream)
{
    if constexpr (OP == OP_RING) {
        return dispatch_w<OP_RING, DDP_F32, false, WR>(a, stream);
    } else {
        const bool acc = a.accumulate != 0;
        switch (dtype) {
        case DDP_BF16:
            return acc ? dispatch_w<OP, DDP_BF16, true, WR>(a, stream) : dispatch_w<OP, DDP_BF16, false, WR>(a, stream);
        case DDP_F16:
            return acc ? dispatch_w<OP, DDP_F16, true, WR>(a, stream) : dispatch_w<OP, DDP_F16, false, WR>(a, stream);
        default:
            if constexpr (WR) {
                return ddp::fail(DDP_E_INVAL, "stream kernel: wire instantiations exist for 16-bit inputs only");
            } else {
                return acc ? dispatch_w<OP, DDP_F32, true, false>(a, stream) : dispatch_w<OP, DDP_F32, false, false>(a, stream);
            }
        }
    }
}

}  // namespace
}  // namespace ddpk
