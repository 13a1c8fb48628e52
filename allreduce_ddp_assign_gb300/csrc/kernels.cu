// Steps 2-4 of the path on the GPU: pack, ring-ordered reduction with the 1/W
// scale, unpack, and the three fused into one pass.
//
// Sources: "DDP: ring AllReduce and gradient buckets" sections 17.4 (ring
// allreduce = reduce-scatter then all-gather, 1/N of the data per step), 17.9
// (each contribution multiplied by 1/world_size), 17.12 (copy into the
// bucket); "Megatron DDP: contiguous buffer and overlap" sections 1 (fp32
// main_grad, bf16 gradients widened) and 3 (reduce_scatter leaves shard r on
// rank r).
//
// Every kernel is one template, bucket_kernel<OP, WT, DT>: the grid splits
// the bucket's elements into equal contiguous slices, one per CTA.  A CTA
// walks its slice in "pieces", cut wherever a ring chunk or a parameter
// segment ends, so that within a piece the chunk c (hence the ring order) and
// the source tensors are fixed.  The W replicas' pointers of the piece are
// staged in shared memory.  Aligned pieces stream 16-byte vectors
// (ld/st.global.cs: each byte is touched once); the rest takes scalar,
// still coalesced, accesses.  HBM-bound: no tensor cores (nothing is a
// contraction).
//
// Bit-exactness: for an element of chunk c the W scaled values are summed in
// ring order c+1, c+2, ..., c with __fmul_rn / __fadd_rn (no FMA
// contraction), the first term taken as is -- the additions the ring's
// reduce-scatter performs, in its order.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <type_traits>
#include <vector>

#include "common.h"
#include "device_common.cuh"

namespace ddpk {

// ---------------------------------------------------------------------------
// main_grad access of VEC consecutive elements whose address is aligned to MGA
// floats: a 16-byte vector (MGA 4), two 8-byte halves (2) or four words (1).
// A segment whose bucket offset is not a multiple of 4 (a 10-element bias ahead
// of it, say) keeps 16-byte gradient and output accesses this way, with only
// its main_grad accesses split.
// ---------------------------------------------------------------------------
template <int VEC, int MGA> struct MgLane {
    __device__ __forceinline__ static float ld(const float* p) { return __ldcs(p); }
    __device__ __forceinline__ static void st(float* p, float v) { __stcs(p, v); }
};
template <int MGA> struct MgLane<4, MGA> {
    __device__ __forceinline__ static float4 ld(const float* p)
    {
        if constexpr (MGA == 4) {
            return __ldcs(reinterpret_cast<const float4*>(p));
        } else if constexpr (MGA == 2) {
            const float2 x = __ldcs(reinterpret_cast<const float2*>(p));
            const float2 y = __ldcs(reinterpret_cast<const float2*>(p + 2));
            return make_float4(x.x, x.y, y.x, y.y);
        } else {
            return make_float4(__ldcs(p), __ldcs(p + 1), __ldcs(p + 2), __ldcs(p + 3));
        }
    }
    __device__ __forceinline__ static void st(float* p, float4 v)
    {
        if constexpr (MGA == 4) {
            __stcs(reinterpret_cast<float4*>(p), v);
        } else if constexpr (MGA == 2) {
            __stcs(reinterpret_cast<float2*>(p), make_float2(v.x, v.y));
            __stcs(reinterpret_cast<float2*>(p + 2), make_float2(v.z, v.w));
        } else {
            __stcs(p, v.x);
            __stcs(p + 1, v.y);
            __stcs(p + 2, v.z);
            __stcs(p + 3, v.w);
        }
    }
};

// ---------------------------------------------------------------------------
// one piece: elements [a, b) of chunk c, inside one segment (or the padding)
// ---------------------------------------------------------------------------
// Processes elements e0 + VEC*v, v in [0, count).  `off` is the segment's
// first bucket element (gradient index i = e - off).  With VEC = 4 the
// gradient and output vectors are 16-byte aligned and main_grad's are aligned
// to MGA floats.
template <int OP, int WT, int DT, int VEC, int U, int MGA = 4>
__device__ __forceinline__ void run_range(const Ctx& cx, const PieceShared& sh, int c, int64_t e0, int64_t count,
                                          int64_t off)
{
    using L = Lane<VEC>;
    using M = MgLane<VEC, MGA>;
    using T = typename L::T;
    const int W = WT ? WT : cx.W;
    const int64_t step = static_cast<int64_t>(kThreads) * U;
    for (int64_t v0 = threadIdx.x; v0 < count; v0 += step) {
        int64_t e[U];
        bool live[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = v0 + static_cast<int64_t>(u) * kThreads;
            live[u] = v < count;
            e[u] = e0 + static_cast<int64_t>(VEC) * v;
        }

        if constexpr (OP == OP_RING || OP == OP_FUSED) {
            T acc[U];
            // value of replica r at element x (before scaling)
            auto value = [&](int r, int64_t x) -> T {
                if constexpr (OP == OP_RING) {
                    return M::ld(cx.mg + r * cx.stride + x);
                } else {
                    const void* src = sh.src[r];
                    if (cx.accumulate) {
                        const T m = M::ld(cx.mg + r * cx.stride + x);
                        return src ? L::add(m, L::template ldg<DT>(src, x - off)) : m;
                    }
                    return src ? L::template ldg<DT>(src, x - off) : L::zero();
                }
            };
            auto term = [&](int k) {
                int r = c + 1 + k;  // ring order: c+1, c+2, ..., c
                if (r >= W) r -= W;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (!live[u]) continue;
                    const T t = ring_term(value(r, e[u]), cx.inv_w, static_cast<float>(W), cx.wire);
                    acc[u] = (k == 0) ? t : ring_add(acc[u], t, cx.wire);
                }
            };
            if constexpr (WT > 0 && OP == OP_FUSED) {
                // every replica's values first, then the ring's arithmetic: the W x U
                // loads are all in flight together instead of one replica's at a time
                T val[WT][U];
                auto load_all = [&](auto accumulate) {
#pragma unroll
                    for (int k = 0; k < WT; ++k) {
                        int r = c + 1 + k;
                        if (r >= WT) r -= WT;
                        const void* src = sh.src[r];
#pragma unroll
                        for (int u = 0; u < U; ++u) {
                            if (!live[u]) {
                                val[k][u] = L::zero();
                                continue;
                            }
                            if constexpr (decltype(accumulate)::value) {
                                const T m = M::ld(cx.mg + r * cx.stride + e[u]);
                                val[k][u] = src ? L::add(m, L::template ldg<DT>(src, e[u] - off)) : m;
                            } else {
                                val[k][u] = src ? L::template ldg<DT>(src, e[u] - off) : L::zero();
                            }
                        }
                    }
                };
                if (cx.accumulate)
                    load_all(std::true_type{});
                else
                    load_all(std::false_type{});
#pragma unroll
                for (int k = 0; k < WT; ++k)
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const T t = ring_term(val[k][u], cx.inv_w, static_cast<float>(WT), cx.wire);
                        acc[u] = (k == 0) ? t : ring_add(acc[u], t, cx.wire);
                    }
            } else if constexpr (WT > 0) {
#pragma unroll
                for (int k = 0; k < WT; ++k) term(k);
            } else {
#pragma unroll 4
                for (int k = 0; k < W; ++k) term(k);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (!live[u]) continue;
                if (cx.mg) {
                    if (cx.mode == DDP_ALLREDUCE) {
                        for (int w = 0; w < W; ++w) M::st(cx.mg + w * cx.stride + e[u], acc[u]);
                    } else {
                        M::st(cx.mg + c * cx.stride + e[u], acc[u]);
                    }
                }
                if constexpr (OP == OP_FUSED) {
                    if (cx.mode == DDP_ALLREDUCE) {
                        for (int w = 0; w < W; ++w)
                            if (sh.dst[w]) L::st(sh.dst[w] + (e[u] - off), acc[u]);
                    } else if (sh.dst[c]) {
                        L::st(sh.dst[c] + (e[u] - off), acc[u]);
                    }
                }
            }
        } else if constexpr (OP == OP_PACK) {
            for (int w = 0; w < W; ++w) {
                const void* src = sh.src[w];
                if (cx.accumulate && !src) continue;  // no gradient: the bucket keeps its sum
                float* row = cx.mg + w * cx.stride;
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (!live[u]) continue;
                    T t = src ? L::template ldg<DT>(src, e[u] - off) : L::zero();
                    if (cx.accumulate) t = L::add(M::ld(row + e[u]), t);
                    M::st(row + e[u], t);
                }
            }
        } else {  // OP_UNPACK
            for (int w = 0; w < W; ++w) {
                if (cx.mode == DDP_REDUCE_SCATTER && w != c) continue;
                float* dst = sh.dst[w];
                if (!dst) continue;
                const float* row = cx.mg + w * cx.stride;
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (live[u]) L::st(dst + (e[u] - off), M::ld(row + e[u]));
            }
        }
    }
}

// Stage the piece's pointers (parameter p, or -1 for padding).  Returns, on
// every thread: 2 when every operand allows 16-byte vectors at bucket elements
// e = 0 mod 4; 1 when the gradients and outputs allow them at gradient index
// 0 mod 4 (bucket elements e = off mod 4) and main_grad is vector-aligned, so
// that only main_grad's accesses there are narrower; 0 otherwise (scalars).  The
// flag and pointer tables are read side by side, not one after the other: one
// round trip to memory instead of two.  Contains three block-wide barriers.
template <int OP, int DT>
__device__ __forceinline__ int piece_setup(const Ctx& cx, PieceShared& sh, int p, int64_t off)
{
    __syncthreads();  // the previous piece is done reading sh
    int ok = 1, okg = 1;
    const int t = threadIdx.x;
    if (t < cx.W) {
        const void* src = nullptr;
        float* dst = nullptr;
        if (p >= 0 && p < cx.ld) {
            const int64_t slot = static_cast<int64_t>(t) * cx.ld + p;
            if constexpr (OP == OP_PACK || OP == OP_FUSED) {
                const uint8_t u = cx.used ? cx.used[slot] : uint8_t{1};
                const void* g = cx.grads[slot];
                src = u ? g : nullptr;
            }
            if constexpr (OP == OP_UNPACK || OP == OP_FUSED) {
                if (cx.grads_out) {
                    const uint8_t gu = cx.global_used ? cx.global_used[p] : uint8_t{1};
                    void* d = cx.grads_out[slot];
                    dst = gu ? static_cast<float*>(d) : nullptr;
                }
            }
        }
        sh.src[t] = src;
        sh.dst[t] = dst;
        // vectors at bucket elements e = 0 mod 4 read gradient index e - off
        constexpr int64_t gb = elem_bytes<DT>();
        if (src && ((reinterpret_cast<uintptr_t>(src) - static_cast<uintptr_t>(off * gb)) % (4 * gb)) != 0) ok = 0;
        if (dst && ((reinterpret_cast<uintptr_t>(dst) - static_cast<uintptr_t>(off * 4)) % 16) != 0) ok = 0;
        if (src && (reinterpret_cast<uintptr_t>(src) % (4 * gb)) != 0) okg = 0;
        if (dst && (reinterpret_cast<uintptr_t>(dst) % 16) != 0) okg = 0;
    }
    const bool all = __syncthreads_and(ok) != 0;
    const bool shifted = __syncthreads_and(okg) != 0;
    if (!(cx.mg == nullptr || cx.mg_vec)) return 0;
    return all ? 2 : (shifted ? 1 : 0);
}

template <int OP, int WT, int DT>
__device__ __forceinline__ void process_piece(const Ctx& cx, PieceShared& sh, int c, int p, int64_t off, int64_t a,
                                              int64_t b)
{
    constexpr int U = unroll_for<WT>();
    const int al = piece_setup<OP, DT>(cx, sh, p, off);
    if (al == 2 || (al == 1 && off % 4 == 0)) {
        const int64_t va = lmin(b, (a + 3) & ~int64_t(3));
        const int64_t vb = lmax(va, b & ~int64_t(3));
        run_range<OP, WT, DT, 1, 1>(cx, sh, c, a, va - a, off);
        run_range<OP, WT, DT, 4, U>(cx, sh, c, va, (vb - va) >> 2, off);
        run_range<OP, WT, DT, 1, 1>(cx, sh, c, vb, b - vb, off);
    } else if (al == 1) {
        // vectors on the gradient's grid: bucket elements e = off mod 4
        const int64_t va = lmin(b, a + (((off - a) % 4) + 4) % 4);
        const int64_t nv = (b - va) >> 2;
        const int64_t vb = va + 4 * nv;
        run_range<OP, WT, DT, 1, 1>(cx, sh, c, a, va - a, off);
        if (off % 2 == 0)
            run_range<OP, WT, DT, 4, U, 2>(cx, sh, c, va, nv, off);
        else
            run_range<OP, WT, DT, 4, U, 1>(cx, sh, c, va, nv, off);
        run_range<OP, WT, DT, 1, 1>(cx, sh, c, vb, b - vb, off);
    } else {
        run_range<OP, WT, DT, 1, 4>(cx, sh, c, a, b - a, off);
    }
}

// A bucket's segment table, copied into shared memory by every CTA when it has at
// most kSegCache segments: all entries are read at once (one round trip) instead
// of a binary search of dependent loads followed by a load per piece.  Buckets
// with more segments read the table in global memory as they go.
constexpr int kSegCache = 256;
struct SegCache {
    int64_t off[kSegCache + 1];
    int32_t par[kSegCache];
};

// Exclusive prefix sum over the block's threads (one value each); *total gets the sum.
// Contains two block-wide barriers.
__device__ __forceinline__ int block_exclusive_scan(int v, int* total)
{
    __shared__ int warp_sum[kThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sum[warp] = x;
    __syncthreads();
    int base = 0, all = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
        base += (w < warp) ? warp_sum[w] : 0;
        all += warp_sum[w];
    }
    __syncthreads();
    *total = all;
    return base + x - v;
}

template <int OP, int WT, int DT>
__global__ void __launch_bounds__(kThreads) bucket_kernel(const Ctx cx)
{
    __shared__ PieceShared sh;
    __shared__ SegCache sc;
    const int64_t G = gridDim.x;
    const int64_t blk = blockIdx.x;
    // uniform split: this CTA's slice of the bucket, boundaries on 16-element multiples
    const int64_t lo = (blk * cx.n / G) & ~int64_t(15);
    const int64_t hi = (blk + 1 == G) ? cx.n : (((blk + 1) * cx.n / G) & ~int64_t(15));
    if (cx.per_cta == 0 && lo >= hi) return;  // whole CTA: no barrier is skipped by part of it

    const bool cached = cx.seg_offset && cx.nseg <= kSegCache;
    if (cached) {
        for (int i = threadIdx.x; i <= cx.nseg; i += kThreads) {
            sc.off[i] = cx.seg_offset[i];
            if (i < cx.nseg) sc.par[i] = cx.seg_param[i];
        }
        __syncthreads();
    }
    auto seg_off = [&](int i) -> int64_t { return cached ? sc.off[i] : cx.seg_offset[i]; };
    auto seg_par = [&](int i) -> int { return cached ? sc.par[i] : cx.seg_param[i]; };

    if (cx.per_cta > 0 && cached) {
        // One piece part per CTA: interval s (segment s, or s == nseg: the padding
        // after the last gradient) is cut at ring-chunk ends into pieces, and piece
        // i gets ceil(len_i / per_cta) CTAs.  A CTA then waits on one round of pointer
        // loads and one of data, never on a second piece's.
        __shared__ int first_cta[kSegCache + 2];
        const int nint = cx.nseg + 1;
        // visit(s, f): the pieces of interval s in order, f(chunk, start, end, ctas)
        // returning true to stop
        auto visit = [&](int s, auto&& f) {
            const int64_t lo_s = seg_off(s), hi_s = (s < cx.nseg) ? seg_off(s + 1) : cx.n;
            for (int64_t x = lo_s; x < hi_s;) {
                int c = static_cast<int>(x / cx.chunk);
                if (c >= cx.nchunks) c = cx.nchunks - 1;
                const int64_t y = (c + 1 < cx.nchunks) ? lmin(hi_s, static_cast<int64_t>(c + 1) * cx.chunk) : hi_s;
                if (f(c, x, y, static_cast<int>((y - x + cx.per_cta - 1) / cx.per_cta))) return;
                x = y;
            }
        };
        int count = 0;
        if (static_cast<int>(threadIdx.x) < nint)
            visit(threadIdx.x, [&](int, int64_t, int64_t, int k) { count += k; return false; });
        int total = 0;
        const int first = block_exclusive_scan(count, &total);
        if (static_cast<int>(threadIdx.x) < nint) first_cta[threadIdx.x] = first;
        __syncthreads();
        const int b = blockIdx.x;
        if (b >= total) return;  // whole CTA: a spare one
        int lo_i = 0, hi_i = nint;  // last interval whose first CTA is <= b
        while (hi_i - lo_i > 1) {
            const int mid = (lo_i + hi_i) >> 1;
            if (first_cta[mid] <= b) lo_i = mid; else hi_i = mid;
        }
        const int s = lo_i;
        int j = b - first_cta[s];
        int pc = 0;
        int64_t pa = 0, pb = 0;
        visit(s, [&](int c, int64_t x, int64_t y, int k) {
            if (j >= k) {
                j -= k;
                return false;
            }
            pc = c;
            pa = x + static_cast<int64_t>(j) * cx.per_cta;
            pb = lmin(y, pa + cx.per_cta);
            return true;
        });
        if (pb > pa)
            process_piece<OP, WT, DT>(cx, sh, pc, (s < cx.nseg) ? seg_par(s) : -1, seg_off(s), pa, pb);
        return;
    }

    int c = static_cast<int>(lo / cx.chunk);
    if (c >= cx.nchunks) c = cx.nchunks - 1;
    int s = 0;
    if (cx.seg_offset) {  // segment holding lo: last s with seg_offset[s] <= lo (s == nseg: padding)
        int lo_i = 0, hi_i = cx.nseg + 1;
        while (hi_i - lo_i > 1) {
            const int mid = (lo_i + hi_i) >> 1;
            if (seg_off(mid) <= lo) lo_i = mid; else hi_i = mid;
        }
        s = lo_i;
    }
    int64_t a = lo;
    while (a < hi) {
        const int64_t c_end = (c + 1 >= cx.nchunks) ? cx.n : lmin(static_cast<int64_t>(c + 1) * cx.chunk, cx.n);
        int64_t s_off = 0, s_end = cx.n;
        int p = -1;
        if (cx.seg_offset) {
            s_off = seg_off(s);
            if (s < cx.nseg) {
                s_end = seg_off(s + 1);
                p = seg_par(s);
            }
        }
        const int64_t b = lmin(hi, lmin(c_end, s_end));
        if (b > a) process_piece<OP, WT, DT>(cx, sh, c, p, s_off, a, b);
        a = lmax(a, b);
        while (c + 1 < cx.nchunks && static_cast<int64_t>(c + 1) * cx.chunk <= a) ++c;
        if (cx.seg_offset)
            while (s < cx.nseg && seg_off(s + 1) <= a) ++s;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int OP, int WT, int DT>
ddp_status launch_instance(const Ctx& cx, void* stream)
{
    // resident CTAs per SM of this instantiation, per device (0: not asked yet)
    static std::atomic<int> occupancy[ddp::kMaxDevices] = {};
    auto kern = bucket_kernel<OP, WT, DT>;
    const int dev = ddp::current_device();
    int blocks_per_sm = dev >= 0 ? occupancy[dev].load(std::memory_order_relaxed) : 0;
    if (!blocks_per_sm) {
        int v = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kern, kThreads, 0) != cudaSuccess || v < 1) v = 1;
        blocks_per_sm = v;
        if (dev >= 0) occupancy[dev].store(v, std::memory_order_relaxed);
    }
    // at least a CTA per ring chunk (down to 16-element slices): on a small bucket the
    // pieces then run side by side instead of one after another in one CTA
    int64_t want = (cx.n + kMinElemsPerCta - 1) / kMinElemsPerCta;
    if (cx.nchunks > 1) want = std::max<int64_t>(want, std::min<int64_t>(cx.nchunks, (cx.n + 15) / 16));
    const int64_t room = static_cast<int64_t>(ddp::device_sm_count()) * blocks_per_sm;
    int grid = static_cast<int>(std::max<int64_t>(1, std::min(want, room)));
    Ctx c = cx;
    c.per_cta = 0;
    // a bucket whose segment table the CTAs copy into shared memory gets one piece
    // part per CTA, when a wave has room for a CTA per piece besides the elements:
    // the pieces number at most nseg + 1 (the padding) + nchunks - 1, and each adds
    // at most one partly filled CTA to ceil(n / per_cta)
    const int64_t extra = static_cast<int64_t>(cx.nseg) + cx.nchunks;
    if (cx.seg_offset && cx.nseg < kSegCache && cx.n > 0 && room > 2 * extra) {
        int64_t per = std::max<int64_t>(kMinElemsPerCta, (cx.n + room - extra - 1) / (room - extra));
        per = (per + 15) & ~int64_t(15);
        c.per_cta = per;
        grid = static_cast<int>(std::min<int64_t>(room, (cx.n + per - 1) / per + extra));
    }
    kern<<<grid, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(c);
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return ddp::fail(DDP_E_CUDA, "kernel launch failed: %s", cudaGetErrorString(err));
    return ddp::ok();
}

template <int OP, int DT>
ddp_status dispatch_w(const Ctx& cx, void* stream)
{
    switch (cx.W) {
    case 2: return launch_instance<OP, 2, DT>(cx, stream);
    case 4: return launch_instance<OP, 4, DT>(cx, stream);
    case 8: return launch_instance<OP, 8, DT>(cx, stream);
    case 16: return launch_instance<OP, 16, DT>(cx, stream);
    default: return launch_instance<OP, 0, DT>(cx, stream);
    }
}

template <int OP>
ddp_status dispatch(const Ctx& cx, int32_t dtype, void* stream)
{
    if constexpr (OP == OP_RING || OP == OP_UNPACK) {
        return dispatch_w<OP, DDP_F32>(cx, stream);  // no gradient is read
    } else {
        switch (dtype) {
        case DDP_BF16: return dispatch_w<OP, DDP_BF16>(cx, stream);
        case DDP_F16: return dispatch_w<OP, DDP_F16>(cx, stream);
        default: return dispatch_w<OP, DDP_F32>(cx, stream);
        }
    }
}

Ctx base_ctx(int64_t n, int32_t W, bool ring_order, int32_t mode)
{
    Ctx cx{};
    cx.n = n;
    cx.W = W;
    cx.mode = mode;
    cx.inv_w = 1.0f / static_cast<float>(W);
    if (ring_order) {
        cx.nchunks = W;
        cx.chunk = std::max<int64_t>(1, (n + W - 1) / W);
    } else {
        cx.nchunks = 1;
        cx.chunk = std::max<int64_t>(1, n);
    }
    return cx;
}

void set_segments(Ctx& cx, const ddp_bucket_desc& b)
{
    cx.nseg = b.nseg;
    cx.seg_offset = b.nseg > 0 ? b.seg_offset : nullptr;
    cx.seg_param = b.seg_param;
}

void set_mg(Ctx& cx, float* mg, int64_t stride)
{
    cx.mg = mg;
    cx.stride = stride;
    cx.mg_vec = mg && (reinterpret_cast<uintptr_t>(mg) % 16 == 0) && (stride % 4 == 0);
}

std::atomic<int> g_variant{DDP_KERNEL_AUTO};
int kernel_variant() { return g_variant.load(std::memory_order_relaxed); }

// Under DDP_KERNEL_AUTO, a launch of one bucket with at most this many elements over
// all replicas (numel x W) goes to the plain kernel: the streaming kernel's fixed
// cost (a CTA per SM, barrier set-up, filling the stage ring) outweighs its higher
// bandwidth there.  Measured on GB300: a 0.2M-element bucket at W = 4 takes 8.2 us
// plain against 11.8 us streaming; the crossover lies between 2^21 and 2^22.
constexpr int64_t kSmallLaunch = int64_t{1} << 21;

bool use_stream(int op, int32_t W, int32_t dtype, bool acc, int32_t mode, int64_t numel, int32_t nbuckets)
{
    const int v = kernel_variant();
    if (v == DDP_KERNEL_PLAIN) return false;
    if (v == DDP_KERNEL_AUTO && nbuckets == 1 && numel * W <= kSmallLaunch) return false;
    return stream_supported(op, W, dtype, acc, mode);
}

}  // namespace ddpk

extern "C" ddp_status ddp_set_kernel_variant(int32_t variant)
{
    if (variant != DDP_KERNEL_AUTO && variant != DDP_KERNEL_PLAIN && variant != DDP_KERNEL_STREAM &&
        variant != DDP_KERNEL_STREAM_DYNAMIC)
        return ddp::fail(DDP_E_INVAL, "ddp_set_kernel_variant: unknown variant %d", variant);
    ddpk::g_variant.store(variant, std::memory_order_relaxed);
    return ddp::ok();
}

namespace ddp {

using namespace ddpk;

ddp_status launch_allreduce(float* replicas, int64_t stride, int64_t n, int32_t W, int32_t mode, void* stream,
                            int32_t wire)
{
    // the fp32 mean of one replica is the replica (x * 1 is exact); a 16-bit wire still rounds
    if (n == 0 || (W == 1 && wire == DDP_F32)) return ok();
    Ctx cx = base_ctx(n, W, true, mode);
    set_mg(cx, replicas, stride);
    cx.wire = wire;
    if (cx.mg_vec && use_stream(OP_RING, W, DDP_F32, false, mode, n, 1)) {
        StreamArgs a{};
        a.total = n;
        a.stride = stride;
        a.inv_w = cx.inv_w;
        a.W = W;
        a.mode = mode;
        a.wire = wire;
        a.nb = 1;
        a.span[0] = StreamSpan{n, 0, replicas, nullptr, nullptr, 0, 1};
        return launch_stream(OP_RING, a, DDP_F32, stream);
    }
    return dispatch<OP_RING>(cx, DDP_F32, stream);
}

ddp_status launch_pack(const ddp_bucket_desc& b, const void* const* grads, const uint8_t* used, int32_t ld,
                       int32_t W, float* main_grad, int64_t stride, int32_t accumulate, void* stream)
{
    if (b.numel == 0) return ok();
    if (use_stream(OP_PACK, W, b.dtype, accumulate != 0, DDP_ALLREDUCE, b.numel, 1)) {
        float* mgs[1] = {main_grad};
        return launch_pack_group(&b, mgs, 1, grads, used, ld, W, accumulate, stride, stream);
    }
    return launch_pack_plain(b, grads, used, ld, W, main_grad, stride, accumulate, stream);
}

ddp_status launch_pack_plain(const ddp_bucket_desc& b, const void* const* grads, const uint8_t* used, int32_t ld,
                             int32_t W, float* main_grad, int64_t stride, int32_t accumulate, void* stream)
{
    if (b.numel == 0) return ok();
    Ctx cx = base_ctx(b.numel, W, false, DDP_ALLREDUCE);
    set_segments(cx, b);
    set_mg(cx, main_grad, stride);
    cx.ld = ld;
    cx.grads = grads;
    cx.used = used;
    cx.accumulate = accumulate != 0;
    return dispatch<OP_PACK>(cx, b.dtype, stream);
}

ddp_status launch_unpack(const ddp_bucket_desc& b, const float* main_grad, int64_t stride, int32_t W,
                         int32_t mode, void* const* grads_out, int32_t ld, const uint8_t* global_used,
                         void* stream)
{
    if (b.numel == 0 || b.nseg == 0) return ok();
    Ctx cx = base_ctx(b.numel, W, mode == DDP_REDUCE_SCATTER, mode);
    set_segments(cx, b);
    set_mg(cx, const_cast<float*>(main_grad), stride);
    cx.ld = ld;
    cx.grads_out = grads_out;
    cx.global_used = global_used;
    return dispatch<OP_UNPACK>(cx, DDP_F32, stream);
}

ddp_status launch_fused(const ddp_bucket_desc& b, const void* const* grads, const uint8_t* used, int32_t ld,
                        int32_t W, int32_t mode, int32_t accumulate, float* main_grad, int64_t stride,
                        void* const* grads_out, const uint8_t* global_used, void* stream, int32_t wire)
{
    if (b.numel == 0) return ok();
    Ctx cx = base_ctx(b.numel, W, true, mode);
    set_segments(cx, b);
    set_mg(cx, main_grad, stride);
    cx.ld = ld;
    cx.grads = grads;
    cx.used = used;
    cx.grads_out = grads_out;
    cx.global_used = global_used;
    cx.accumulate = accumulate != 0;
    cx.wire = wire;
    if (use_stream(OP_FUSED, W, b.dtype, cx.accumulate, mode, b.numel, 1)) {
        float* mgs[1] = {main_grad};
        return launch_fused_group(&b, mgs, 1, grads, used, ld, W, mode, accumulate, stride, grads_out, global_used,
                                  stream, wire);
    }
    return dispatch<OP_FUSED>(cx, b.dtype, stream);
}

// One streaming launch per run of same-dtype buckets (at most kMaxBatch); buckets the
// streaming kernel cannot take go one by one through `single`.
template <typename Single>
ddp_status launch_group(int op, const ddp_bucket_desc* bs, float* const* mgs, int32_t nb, const void* const* grads,
                        const uint8_t* used, int32_t ld, int32_t W, int32_t mode, int32_t accumulate, int64_t stride,
                        void* const* grads_out, const uint8_t* global_used, void* stream, int32_t wire, Single single)
{
    const bool acc = accumulate != 0;
    int32_t i = 0;
    while (i < nb) {
        const int32_t dt = bs[i].dtype;
        int32_t run = 0;
        int64_t run_numel = 0;
        while (i + run < nb && run < kMaxBatch && bs[i + run].dtype == dt) run_numel += bs[i + run++].numel;
        if (!use_stream(op, W, dt, acc, mode, run_numel, run)) {
            for (const int32_t end = i + run; i < end; ++i) {
                const ddp_status st = single(i);
                if (st != DDP_OK) return st;
            }
            continue;
        }
        StreamArgs a{};
        a.stride = stride;
        a.grads = grads;
        a.used = used;
        a.grads_out = grads_out;
        a.global_used = global_used;
        a.inv_w = 1.0f / static_cast<float>(W);
        a.W = W;
        a.mode = mode;
        a.accumulate = acc;
        a.ld = ld;
        a.wire = wire;
        int64_t total = 0;
        int32_t n = 0;
        while (i < nb && n < kMaxBatch && bs[i].dtype == dt) {
            const ddp_bucket_desc& d = bs[i];
            float* mg = mgs[i];
            const int32_t vec = mg && (reinterpret_cast<uintptr_t>(mg) % 16 == 0) && (stride % 4 == 0);
            a.span[n] = StreamSpan{d.numel, total, mg, d.nseg > 0 ? d.seg_offset : nullptr, d.seg_param, d.nseg, vec};
            total += d.numel;
            ++n;
            ++i;
        }
        a.nb = n;
        a.total = total;
        if (total == 0) continue;
        const ddp_status st = launch_stream(op, a, dt, stream);
        if (st != DDP_OK) return st;
    }
    return ok();
}

ddp_status launch_fused_group(const ddp_bucket_desc* bs, float* const* mgs, int32_t nb, const void* const* grads,
                              const uint8_t* used, int32_t ld, int32_t W, int32_t mode, int32_t accumulate,
                              int64_t stride, void* const* grads_out, const uint8_t* global_used, void* stream,
                              int32_t wire)
{
    return launch_group(OP_FUSED, bs, mgs, nb, grads, used, ld, W, mode, accumulate, stride, grads_out, global_used,
                        stream, wire, [&](int32_t i) {
                            return launch_fused(bs[i], grads, used, ld, W, mode, accumulate, mgs[i], stride,
                                                grads_out, global_used, stream, wire);
                        });
}

ddp_status launch_pack_group(const ddp_bucket_desc* bs, float* const* mgs, int32_t nb, const void* const* grads,
                             const uint8_t* used, int32_t ld, int32_t W, int32_t accumulate, int64_t stride,
                             void* stream)
{
    return launch_group(OP_PACK, bs, mgs, nb, grads, used, ld, W, DDP_ALLREDUCE, accumulate, stride, nullptr,
                        nullptr, stream, DDP_F32, [&](int32_t i) {
                            return launch_pack_plain(bs[i], grads, used, ld, W, mgs[i], stride, accumulate, stream);
                        });
}

}  // namespace ddp

// ---------------------------------------------------------------------------
// C ABI: validation, then launch
// ---------------------------------------------------------------------------
namespace {

ddp_status check_w(const char* fn, int32_t W)
{
    if (W < 1 || W > ddp::kMaxReplicas)
        return ddp::fail(DDP_E_INVAL, "%s: W = %d outside [1, %d]", fn, W, ddp::kMaxReplicas);
    return DDP_OK;
}

ddp_status check_mode(const char* fn, int32_t mode, int64_t n, int32_t W)
{
    if (mode != DDP_ALLREDUCE && mode != DDP_REDUCE_SCATTER)
        return ddp::fail(DDP_E_INVAL, "%s: unknown mode %d", fn, mode);
    if (mode == DDP_REDUCE_SCATTER && n % W != 0)
        return ddp::fail(DDP_E_INVAL, "%s: reduce_scatter needs numel %% W == 0 (numel %lld, W %d)", fn,
                         static_cast<long long>(n), W);
    return DDP_OK;
}

ddp_status check_desc(const char* fn, const ddp_bucket_desc* b, int32_t ld, bool need_tables)
{
    if (!b) return ddp::fail(DDP_E_INVAL, "%s: bucket descriptor is NULL", fn);
    if (b->numel < 0 || b->nseg < 0)
        return ddp::fail(DDP_E_INVAL, "%s: negative size (numel %lld, nseg %d)", fn,
                         static_cast<long long>(b->numel), b->nseg);
    if (b->dtype != DDP_F32 && b->dtype != DDP_BF16 && b->dtype != DDP_F16)
        return ddp::fail(DDP_E_INVAL, "%s: unknown dtype %d", fn, b->dtype);
    if (b->nseg > 0 && (!b->seg_offset || !b->seg_param))
        return ddp::fail(DDP_E_INVAL, "%s: segment tables are NULL with nseg = %d", fn, b->nseg);
    if (need_tables && b->nseg > 0 && ld < 1) return ddp::fail(DDP_E_INVAL, "%s: ld = %d < 1", fn, ld);
    return DDP_OK;
}

ddp_status check_mg(const char* fn, const float* mg, int64_t stride, int64_t n, int32_t W)
{
    if (!mg && n > 0) return ddp::fail(DDP_E_INVAL, "%s: main_grad is NULL", fn);
    if (W > 1 && stride < n)
        return ddp::fail(DDP_E_INVAL, "%s: replica_stride %lld < numel %lld", fn, static_cast<long long>(stride),
                         static_cast<long long>(n));
    return DDP_OK;
}

#define DDP_TRY(x)                          \
    do {                                    \
        const ddp_status st_ = (x);         \
        if (st_ != DDP_OK) return st_;      \
    } while (0)

ddp_status check_wire(const char* fn, int32_t wire)
{
    if (wire != DDP_F32 && wire != DDP_BF16 && wire != DDP_F16)
        return ddp::fail(DDP_E_INVAL, "%s: unknown wire dtype %d", fn, wire);
    return DDP_OK;
}

ddp_status allreduce_checked(const char* fn, float* replicas, int64_t replica_stride, int64_t numel, int32_t W,
                             int32_t mode, int32_t wire, void* stream)
{
    DDP_TRY(check_w(fn, W));
    DDP_TRY(check_wire(fn, wire));
    if (numel < 0) return ddp::fail(DDP_E_INVAL, "%s: numel < 0", fn);
    DDP_TRY(check_mode(fn, mode, numel, W));
    DDP_TRY(check_mg(fn, replicas, replica_stride, numel, W));
    return ddp::launch_allreduce(replicas, replica_stride, numel, W, mode, stream, wire);
}

}  // namespace

extern "C" ddp_status ddp_bucket_allreduce(float* replicas, int64_t replica_stride, int64_t numel, int32_t W,
                                           int32_t mode, void* stream)
{
    return allreduce_checked("ddp_bucket_allreduce", replicas, replica_stride, numel, W, mode, DDP_F32, stream);
}

extern "C" ddp_status ddp_bucket_allreduce_wire(float* replicas, int64_t replica_stride, int64_t numel, int32_t W,
                                                int32_t mode, int32_t wire_dtype, void* stream)
{
    return allreduce_checked("ddp_bucket_allreduce_wire", replicas, replica_stride, numel, W, mode, wire_dtype, stream);
}

extern "C" ddp_status ddp_pack(const ddp_bucket_desc* bucket, const void* const* grads, const uint8_t* used,
                               int32_t ld, int32_t W, float* main_grad, int64_t replica_stride, int32_t accumulate,
                               void* stream)
{
    const char* fn = "ddp_pack";
    DDP_TRY(check_w(fn, W));
    DDP_TRY(check_desc(fn, bucket, ld, true));
    if (bucket->nseg > 0 && !grads) return ddp::fail(DDP_E_INVAL, "%s: grads table is NULL", fn);
    DDP_TRY(check_mg(fn, main_grad, replica_stride, bucket->numel, W));
    return ddp::launch_pack(*bucket, grads, used, ld, W, main_grad, replica_stride, accumulate, stream);
}

extern "C" ddp_status ddp_unpack(const ddp_bucket_desc* bucket, const float* main_grad, int64_t replica_stride,
                                 int32_t W, int32_t mode, void* const* grads_out, int32_t ld,
                                 const uint8_t* global_used, void* stream)
{
    const char* fn = "ddp_unpack";
    DDP_TRY(check_w(fn, W));
    DDP_TRY(check_desc(fn, bucket, ld, true));
    DDP_TRY(check_mode(fn, mode, bucket->numel, W));
    if (bucket->nseg > 0 && !grads_out) return ddp::fail(DDP_E_INVAL, "%s: grads_out table is NULL", fn);
    DDP_TRY(check_mg(fn, main_grad, replica_stride, bucket->numel, W));
    return ddp::launch_unpack(*bucket, main_grad, replica_stride, W, mode, grads_out, ld, global_used, stream);
}

extern "C" ddp_status ddp_pack_group(const ddp_bucket_desc* buckets, const int64_t* bucket_start, int32_t nbuckets,
                                     const void* const* grads, const uint8_t* used, int32_t ld, int32_t W,
                                     float* main_grad, int64_t replica_stride, int32_t accumulate, void* stream)
{
    const char* fn = "ddp_pack_group";
    DDP_TRY(check_w(fn, W));
    if (nbuckets < 0 || (nbuckets > 0 && (!buckets || !bucket_start)))
        return ddp::fail(DDP_E_INVAL, "%s: bad bucket list", fn);
    std::vector<float*> mgs(static_cast<size_t>(nbuckets), nullptr);
    for (int32_t b = 0; b < nbuckets; ++b) {
        DDP_TRY(check_desc(fn, &buckets[b], ld, true));
        if (buckets[b].nseg > 0 && !grads) return ddp::fail(DDP_E_INVAL, "%s: grads table is NULL", fn);
        DDP_TRY(check_mg(fn, main_grad, replica_stride, buckets[b].numel, W));
        if (bucket_start[b] < 0 || (W > 1 && bucket_start[b] + buckets[b].numel > replica_stride))
            return ddp::fail(DDP_E_INVAL, "%s: bucket %d [%lld, +%lld) exceeds replica_stride %lld", fn, b,
                             static_cast<long long>(bucket_start[b]), static_cast<long long>(buckets[b].numel),
                             static_cast<long long>(replica_stride));
        mgs[b] = main_grad ? main_grad + bucket_start[b] : nullptr;
    }
    return ddp::launch_pack_group(buckets, mgs.data(), nbuckets, grads, used, ld, W, accumulate, replica_stride,
                                  stream);
}

namespace {

ddp_status fused_group_checked(const char* fn, const ddp_bucket_desc* buckets, const int64_t* bucket_start,
                               int32_t nbuckets, const void* const* grads, const uint8_t* used, int32_t ld, int32_t W,
                               int32_t mode, int32_t accumulate, float* main_grad, int64_t replica_stride,
                               void* const* grads_out, const uint8_t* global_used, int32_t wire, void* stream)
{
    DDP_TRY(check_w(fn, W));
    DDP_TRY(check_wire(fn, wire));
    if (nbuckets < 0 || (nbuckets > 0 && (!buckets || (main_grad && !bucket_start))))
        return ddp::fail(DDP_E_INVAL, "%s: bad bucket list", fn);
    std::vector<float*> mgs(static_cast<size_t>(nbuckets), nullptr);
    for (int32_t b = 0; b < nbuckets; ++b) {
        DDP_TRY(check_desc(fn, &buckets[b], ld, true));
        DDP_TRY(check_mode(fn, mode, buckets[b].numel, W));
        if (buckets[b].nseg > 0 && !grads) return ddp::fail(DDP_E_INVAL, "%s: grads table is NULL", fn);
        if (!main_grad && !grads_out && buckets[b].numel > 0)
            return ddp::fail(DDP_E_INVAL, "%s: main_grad and grads_out are both NULL", fn);
        if (accumulate && !main_grad && buckets[b].numel > 0)
            return ddp::fail(DDP_E_INVAL, "%s: accumulate needs main_grad", fn);
        if (main_grad) {
            if (bucket_start[b] < 0 || (W > 1 && bucket_start[b] + buckets[b].numel > replica_stride))
                return ddp::fail(DDP_E_INVAL, "%s: bucket %d [%lld, +%lld) exceeds replica_stride %lld", fn, b,
                                 static_cast<long long>(bucket_start[b]), static_cast<long long>(buckets[b].numel),
                                 static_cast<long long>(replica_stride));
            mgs[b] = main_grad + bucket_start[b];
        }
    }
    return ddp::launch_fused_group(buckets, mgs.data(), nbuckets, grads, used, ld, W, mode, accumulate,
                                   replica_stride, grads_out, global_used, stream, wire);
}

}  // namespace

extern "C" ddp_status ddp_fused_bucket_group(const ddp_bucket_desc* buckets, const int64_t* bucket_start,
                                             int32_t nbuckets, const void* const* grads, const uint8_t* used,
                                             int32_t ld, int32_t W, int32_t mode, int32_t accumulate, float* main_grad,
                                             int64_t replica_stride, void* const* grads_out,
                                             const uint8_t* global_used, void* stream)
{
    return fused_group_checked("ddp_fused_bucket_group", buckets, bucket_start, nbuckets, grads, used, ld, W, mode,
                               accumulate, main_grad, replica_stride, grads_out, global_used, DDP_F32, stream);
}

extern "C" ddp_status ddp_fused_bucket_group_wire(const ddp_bucket_desc* buckets, const int64_t* bucket_start,
                                                  int32_t nbuckets, const void* const* grads, const uint8_t* used,
                                                  int32_t ld, int32_t W, int32_t mode, int32_t accumulate,
                                                  float* main_grad, int64_t replica_stride, void* const* grads_out,
                                                  const uint8_t* global_used, int32_t wire_dtype, void* stream)
{
    return fused_group_checked("ddp_fused_bucket_group_wire", buckets, bucket_start, nbuckets, grads, used, ld, W,
                               mode, accumulate, main_grad, replica_stride, grads_out, global_used, wire_dtype, stream);
}

extern "C" ddp_status ddp_fused_bucket(const ddp_bucket_desc* bucket, const void* const* grads,
                                       const uint8_t* used, int32_t ld, int32_t W, int32_t mode,
                                       int32_t accumulate, float* main_grad, int64_t replica_stride,
                                       void* const* grads_out, const uint8_t* global_used, void* stream)
{
    const char* fn = "ddp_fused_bucket";
    DDP_TRY(check_w(fn, W));
    DDP_TRY(check_desc(fn, bucket, ld, true));
    DDP_TRY(check_mode(fn, mode, bucket->numel, W));
    if (bucket->nseg > 0 && !grads) return ddp::fail(DDP_E_INVAL, "%s: grads table is NULL", fn);
    if (!main_grad && !grads_out && bucket->numel > 0)
        return ddp::fail(DDP_E_INVAL, "%s: main_grad and grads_out are both NULL", fn);
    if (accumulate && !main_grad && bucket->numel > 0)
        return ddp::fail(DDP_E_INVAL, "%s: accumulate needs main_grad", fn);
    if (main_grad) DDP_TRY(check_mg(fn, main_grad, replica_stride, bucket->numel, W));
    return ddp::launch_fused(*bucket, grads, used, ld, W, mode, accumulate, main_grad, replica_stride, grads_out,
                             global_used, stream);
}
