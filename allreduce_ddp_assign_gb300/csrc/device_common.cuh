// Device-side definitions shared by the kernel translation units (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "common.h"

namespace ddpk {

constexpr int kThreads = 256;
// The plain kernel's smallest slice a CTA: on small buckets more CTAs win (a 0.2M-
// element bucket at W = 4 took 23 us a launch with 4096-element slices, 8.2 us
// with 512); from about 0.6M elements the grid is capped at one wave anyway.
constexpr int64_t kMinElemsPerCta = 512;

enum Op { OP_RING = 0, OP_PACK = 1, OP_FUSED = 2, OP_UNPACK = 3 };

struct Ctx {
    int64_t n;          // bucket elements, padding included
    int64_t chunk;      // ring chunk length (n when the op has no ring order)
    int32_t nchunks;    // W for ring-ordered ops, 1 otherwise
    int32_t W;
    int32_t mode;
    int32_t accumulate;
    float inv_w;
    int32_t nseg;       // 0 with seg_offset == nullptr: the whole bucket is one piece
    const int64_t* seg_offset;
    const int32_t* seg_param;
    int32_t ld;
    const void* const* grads;
    const uint8_t* used;
    void* const* grads_out;
    const uint8_t* global_used;
    float* mg;          // replica 0 of the bucket (main_grad), may be null for OP_FUSED
    int64_t stride;     // elements between replicas of mg
    int32_t mg_vec;     // every replica of mg is 16-byte aligned
    int32_t wire;       // ring arithmetic type: DDP_F32, or DDP_BF16 / DDP_F16 (compression hook)
    int64_t per_cta;    // > 0: every CTA takes at most this many elements of one piece (set by the launcher)
};

struct PieceShared {
    const void* src[ddp::kMaxReplicas];  // replica w's gradient of the piece's parameter, or null
    float* dst[ddp::kMaxReplicas];       // replica w's output of that parameter, or null
};

// ---------------------------------------------------------------------------
// element access
// ---------------------------------------------------------------------------
template <int VEC> struct Lane;

template <> struct Lane<4> {
    using T = float4;
    __device__ __forceinline__ static T zero() { return make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ __forceinline__ static T ld(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
    __device__ __forceinline__ static void st(float* p, T v) { __stcs(reinterpret_cast<float4*>(p), v); }
    __device__ __forceinline__ static T mul(T a, float s)
    {
        return make_float4(__fmul_rn(a.x, s), __fmul_rn(a.y, s), __fmul_rn(a.z, s), __fmul_rn(a.w, s));
    }
    __device__ __forceinline__ static T add(T a, T b)
    {
        return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
    }
    template <int DT> __device__ __forceinline__ static T ldg(const void* base, int64_t i);
};

template <> __device__ __forceinline__ float4 Lane<4>::ldg<DDP_F32>(const void* base, int64_t i)
{
    return __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(base) + i));
}
template <> __device__ __forceinline__ float4 Lane<4>::ldg<DDP_BF16>(const void* base, int64_t i)
{
    // bf16 -> fp32 widening is exact: the bf16 bits become the upper half
    const uint2 u = __ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + i));
    return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                       __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}
template <> __device__ __forceinline__ float4 Lane<4>::ldg<DDP_F16>(const void* base, int64_t i)
{
    const uint2 u = __ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(base) + i));
    const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

template <> struct Lane<1> {
    using T = float;
    __device__ __forceinline__ static T zero() { return 0.f; }
    __device__ __forceinline__ static T ld(const float* p) { return __ldcs(p); }
    __device__ __forceinline__ static void st(float* p, T v) { __stcs(p, v); }
    __device__ __forceinline__ static T mul(T a, float s) { return __fmul_rn(a, s); }
    __device__ __forceinline__ static T add(T a, T b) { return __fadd_rn(a, b); }
    template <int DT> __device__ __forceinline__ static T ldg(const void* base, int64_t i);
};

template <> __device__ __forceinline__ float Lane<1>::ldg<DDP_F32>(const void* base, int64_t i)
{
    return __ldcs(static_cast<const float*>(base) + i);
}
template <> __device__ __forceinline__ float Lane<1>::ldg<DDP_BF16>(const void* base, int64_t i)
{
    return __uint_as_float(static_cast<uint32_t>(__ldcs(static_cast<const unsigned short*>(base) + i)) << 16);
}
template <> __device__ __forceinline__ float Lane<1>::ldg<DDP_F16>(const void* base, int64_t i)
{
    return __half2float(__ushort_as_half(__ldcs(static_cast<const unsigned short*>(base) + i)));
}

__host__ __device__ __forceinline__ int64_t lmin(int64_t a, int64_t b) { return a < b ? a : b; }
__host__ __device__ __forceinline__ int64_t lmax(int64_t a, int64_t b) { return a > b ? a : b; }

template <int DT> __host__ __device__ constexpr int elem_bytes() { return DT == DDP_F32 ? 4 : 2; }

// ---------------------------------------------------------------------------
// one ring term and one ring addition
// ---------------------------------------------------------------------------
// wire == DDP_F32: the contribution is t * fp32(1/W) and partial sums are fp32.
// wire == DDP_BF16 / DDP_F16 (the compression hook, "DDP: ring AllReduce and
// gradient buckets" 17.9, 17.20): t is rounded to the wire type, divided by W
// and rounded again, and every partial sum is rounded to the wire type.  Each
// step is computed in fp32 and then rounded: for 16-bit wire types (8- and
// 11-bit significands) an fp32 sum or quotient of two wire values rounded to
// the wire type equals the correctly rounded result (24 >= 2q + 2).
__device__ __forceinline__ float wire_round(float x, int wire)
{
    return wire == DDP_BF16 ? __bfloat162float(__float2bfloat16_rn(x)) : __half2float(__float2half_rn(x));
}
__device__ __forceinline__ float ring_term(float t, float inv_w, float fw, int wire)
{
    if (wire == DDP_F32) return __fmul_rn(t, inv_w);
    return wire_round(__fdiv_rn(wire_round(t, wire), fw), wire);
}
__device__ __forceinline__ float ring_add(float acc, float t, int wire)
{
    const float s = __fadd_rn(acc, t);
    return wire == DDP_F32 ? s : wire_round(s, wire);
}
__device__ __forceinline__ float4 ring_term(float4 t, float inv_w, float fw, int wire)
{
    return make_float4(ring_term(t.x, inv_w, fw, wire), ring_term(t.y, inv_w, fw, wire),
                       ring_term(t.z, inv_w, fw, wire), ring_term(t.w, inv_w, fw, wire));
}
__device__ __forceinline__ float4 ring_add(float4 acc, float4 t, int wire)
{
    return make_float4(ring_add(acc.x, t.x, wire), ring_add(acc.y, t.y, wire), ring_add(acc.z, t.z, wire),
                       ring_add(acc.w, t.w, wire));
}

// Loads per thread kept in flight: about 16 vectors whatever W is.
template <int WT> __host__ __device__ constexpr int unroll_for()
{
    return WT == 2 ? 4 : (WT == 4 ? 2 : 1);
}

// streaming (TMA-pipelined) kernel, stream.cu: one launch covers up to
// kMaxBatch buckets laid end to end in a single element space
constexpr int kMaxBatch = 32;

struct StreamSpan {
    int64_t numel;               // bucket elements, padding included
    int64_t base;                // first element of the bucket in the launch's element space
    float* mg;                   // the bucket in main_grad, replica 0 (ring op: the replicas); may be null
    const int64_t* seg_offset;   // nullptr: the whole bucket is one piece without gradient source
    const int32_t* seg_param;
    int32_t nseg;
    int32_t mg_vec;              // every replica of mg is 16-byte aligned
    int32_t cache_base;          // first entry of this span's tables in the shared-memory copy (set by the launcher)
    int32_t pad_;
};

struct StreamArgs {
    int64_t total;               // sum of the spans' numel
    int64_t stride;              // elements between main_grad replicas
    const void* const* grads;
    const uint8_t* used;
    void* const* grads_out;
    const uint8_t* global_used;
    float inv_w;
    int32_t W, mode, accumulate, ld, nb;
    int32_t ns;                  // pipeline stages (set by the launcher)
    int32_t store_bulk;          // results leave through TMA bulk stores (set by the launcher)
    int* status;                 // device status word (set by the launcher)
    int32_t wire;                // ring arithmetic type: DDP_F32, DDP_BF16, DDP_F16
    // Work split (set by the launcher).  Elements [0, head) of the launch are cut
    // into equal static slices, one per CTA; elements [head, total) form a pool of
    // `unit`-element units that CTAs claim one at a time from the counters at
    // `dyn` (claimed, finished) once their slice is done.  dyn == nullptr: no
    // pool (head == total).
    uint32_t* dyn;
    int64_t head;
    int32_t unit;
    int32_t seg_cached;          // segment-table entries copied into shared memory (0: read from global memory)
    StreamSpan span[kMaxBatch];
};

bool stream_supported(int op, int W, int dtype, bool acc, int mode);
ddp_status launch_stream(int op, StreamArgs& a, int dtype, void* stream);
ddp_status read_device_status(void* stream, int32_t* out, int reset);

// kernel variant chosen by ddp_set_kernel_variant (kernels.cu)
int kernel_variant();

}  // namespace ddpk
