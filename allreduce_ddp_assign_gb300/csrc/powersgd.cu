// The PowerSGD communication hook on one bucket of W replicas.
//
// "DDP: ring AllReduce and gradient buckets" section 17.27: every tensor of
// two or more dimensions, viewed as M x N, is replaced by a rank-R
// approximation computed with one step of a warm-started power iteration --
// P = M Q, all-reduce P, orthonormalise P, Q = M^T P, all-reduce Q and divide
// by the world size, reconstruct P Q^T -- with error feedback (M = G + E,
// E <- M - P Q^T); 1-D tensors take a plain all-reduce; the first
// start_powerSGD_iter iterations take a plain all-reduce of the whole bucket.
//
// Kernels per compressed iteration (one launch each, over every tensor of the
// bucket through tile tables built on the host):
//   psgd_p_kernel       per (row, group of replicas, column split): M = G + E
//                       (stored back into E), P_w[row] = M[row, split] Q[split];
//                       the sum over replicas, one partial P per split.  Extra
//                       blocks take the 1-D tensors: ring-ordered mean over
//                       their concatenation
//   psgd_orth_kernel    per tensor: P = the splits' partials added in order,
//                       P^T P in float pairs (compensated), its Cholesky factor
//                       R in fp64, and P <- P R^-1
//   psgd_qpart_kernel   per (column block, row split, replica): partial M^T P,
//                       the split's rows shared by the block's warps; the last
//                       block of a column block sums the partials in a fixed
//                       order into Q = (sum_w M_w^T P) / W
//   psgd_out_kernel     G^ = P Q^T written to every replica, E = M - G^: flat
//                       tiles of 16-byte quads over the matrix's rows laid end to
//                       end (a warp per row where rows are not 16-byte multiples),
//                       one wave of blocks looping over the tiles
// Every kernel streams its matrix once: the contraction is rank R (1..8)
// against a row or column of M, R fused multiply-adds per element and 4 to 12
// bytes per element, far below the CUDA cores' arithmetic ridge, so the work is
// HBM-bound and stays on the CUDA cores in fp32.
//
// Rank is padded to RP in {1, 2, 4, 8}: Q and P carry RP columns, those past a
// tensor's effective rank min(R, M, N) are zero and stay zero.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <vector>

#include "common.h"

namespace {

#ifndef DDP_PSGD_P_BLOCKS
#define DDP_PSGD_P_BLOCKS 1   // resident blocks per SM the P pass is compiled for
#endif
#ifndef DDP_PSGD_Q_BLOCKS
#define DDP_PSGD_Q_BLOCKS 3   // resident blocks per SM the Q pass is compiled for
#endif
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRowsOut = kWarps;       // rows per output tile: one per warp
#ifndef DDP_PSGD_Q_WAVE
#define DDP_PSGD_Q_WAVE 0   // 1: the Q launch is one wave of blocks looping over the tiles (0: a block per tile)
#endif
#ifndef DDP_PSGD_QROWS
#define DDP_PSGD_QROWS 256
#endif
constexpr int kRowsPerSplit = DDP_PSGD_QROWS;   // rows of one partial M^T P
constexpr int kMaxPairs = 256;         // (row, replica) pairs per P tile
constexpr int kMaxRowsP = 16;          // rows per P tile
#ifndef DDP_PSGD_PCOLS
#define DDP_PSGD_PCOLS 1024
#endif
constexpr int kPCols = DDP_PSGD_PCOLS;  // longest column split of a P tile (a multiple of 128)
// Rank 8 holds 148 registers a thread in the P pass (one block per SM): twice the split
// there, so that a matrix's tiles still fit the fewer resident blocks.
constexpr int p_cols(int rp) { return rp >= 8 ? 2 * kPCols : kPCols; }
// The Q pass at rank 8 needs more than the 80 registers three blocks per SM allow.
constexpr int q_min_blocks(int rp) { return rp >= 8 ? 2 : DDP_PSGD_Q_BLOCKS; }
#ifndef DDP_PSGD_GW
#define DDP_PSGD_GW 4
#endif
constexpr int kGW = DDP_PSGD_GW;       // replicas a warp carries at once in the P pass
constexpr int kOutBatch = 8;           // replicas whose error loads the output pass issues together
#ifndef DDP_PSGD_OUTQ
#define DDP_PSGD_OUTQ 2048
#endif
constexpr int kOutQuads = DDP_PSGD_OUTQ;   // 16-byte quads per flat output tile
constexpr int64_t kVecPiece = 16384;   // elements of a 1-D tensor per block

struct PsgdMat {
    int64_t off;     // element offset of the tensor in the bucket
    int64_t p_off;   // into P: M x RP
    int64_t q_off;   // into the Q state: N x RP
    int64_t qp_off;  // into the partial sums: S x W x N x RP
    int32_t M, N;
    int32_t r;       // effective rank
    int32_t vec;     // offset and N are multiples of 4 (16-byte rows when the buffers are aligned)
    int32_t S;       // row splits of M^T P
    int32_t cbw;     // column block width of M^T P (128 on the 16-byte path, 32 otherwise)
    int32_t psp;     // column splits of the P pass (their partial sums of P follow in split order)
    int32_t pcw;     // columns of one split (a multiple of 128 unless the split is the whole row)
    int64_t ps_off;  // into the partial sums of P: psp x M x RP
    int32_t cnt0;    // first completion counter (one per column block)
    int32_t pad;
};

struct PsgdVec {
    int64_t off;     // element offset in the bucket
    int64_t vpos;    // position in the concatenation of the 1-D tensors
    int64_t len;
};

struct PsgdArgs {
    float* mg;
    int64_t stride;
    float* err;
    int64_t estride;
    float* P;
    float* Q;
    float* QP;
    float* PS;        // per tensor and column split: the replica-summed partial P
    int* CNT;         // per column block: blocks of the Q pass finished
    const PsgdMat* mats;
    const int4* tiles;
    const PsgdVec* vecs;
    int32_t n_ptiles; // blocks of the P launch past this take the 1-D tensors
    int32_t n_otiles; // output tiles (the output launch's blocks loop over them)
    int32_t n_qtiles; // Q-pass tiles (the Q launch's blocks loop over them)
    int32_t ncnt;
    int32_t W;
    int32_t ef;
    int32_t vec_ok;
    float inv_w;
    int64_t nvec;     // length of the concatenation of the 1-D tensors
};

template <int RP>
__device__ __forceinline__ void load_row(const float* __restrict__ src, float (&v)[RP])
{
    if constexpr (RP % 4 == 0) {
#pragma unroll
        for (int k = 0; k < RP; k += 4) {
            const float4 x = __ldg(reinterpret_cast<const float4*>(src + k));
            v[k] = x.x;
            v[k + 1] = x.y;
            v[k + 2] = x.z;
            v[k + 3] = x.w;
        }
    } else if constexpr (RP == 2) {
        const float2 x = __ldg(reinterpret_cast<const float2*>(src));
        v[0] = x.x;
        v[1] = x.y;
    } else {
        v[0] = __ldg(src);
    }
}

__device__ __forceinline__ float comp(const float4& v, int c) { return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w; }

// ---------------------------------------------------------------------------
// 1-D tensors: the ring mean over the concatenation (chunk c summed from
// replica c+1 round to replica c, each term scaled by fp32(1/W))
// ---------------------------------------------------------------------------
__device__ void vec_piece(const PsgdArgs& a, const PsgdVec v)
{
    const int64_t L = (a.nvec + a.W - 1) / a.W;
    for (int64_t i = threadIdx.x; i < v.len; i += kThreads) {
        const int64_t e = v.off + i;
        const int c = static_cast<int>((v.vpos + i) / L);
        float acc = 0.f;
        for (int k = 0; k < a.W; ++k) {
            int w = c + 1 + k;
            w -= (w >= a.W) ? a.W : 0;
            const float t = __fmul_rn(a.mg[w * a.stride + e], a.inv_w);
            acc = k == 0 ? t : __fadd_rn(acc, t);
        }
        for (int w = 0; w < a.W; ++w) a.mg[w * a.stride + e] = acc;
    }
}

// ---------------------------------------------------------------------------
// P = sum_w (G_w + E_w) Q  (tile: {mat, row0, nrows, column split}; one warp per
// row and group of up to kGW replicas, which share the loads of Q).  A tile sums
// its columns [split * pcw, +pcw) into the split's partial P; the
// orthonormalisation adds the splits.
// ---------------------------------------------------------------------------
template <int RP>
__global__ void __launch_bounds__(kThreads, DDP_PSGD_P_BLOCKS) psgd_p_kernel(const PsgdArgs a)
{
    __shared__ float part[kMaxPairs][RP];
    if (static_cast<int>(blockIdx.x) >= a.n_ptiles) {
        vec_piece(a, a.vecs[blockIdx.x - a.n_ptiles]);
        return;
    }
    if (blockIdx.x == 0)   // the Q pass's completion counters start each call at zero
        for (int k = threadIdx.x; k < a.ncnt; k += kThreads) a.CNT[k] = 0;
    const int4 t = a.tiles[blockIdx.x];
    const PsgdMat m = a.mats[t.x];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ngroups = (a.W + kGW - 1) / kGW;
    const int units = t.z * ngroups;
    const bool vec = m.vec && a.vec_ok;
    const float* q = a.Q + m.q_off;
    const int c0 = t.w * m.pcw, c1 = min(m.N, c0 + m.pcw);
    for (int u = warp; u < units; u += kWarps) {
        const int rl = u / ngroups, w0 = (u % ngroups) * kGW;
        const int gw = min(kGW, a.W - w0);
        const int64_t rowoff = m.off + static_cast<int64_t>(t.y + rl) * m.N;
        float* g[kGW];
        float* e[kGW];
#pragma unroll
        for (int k = 0; k < kGW; ++k) {
            const int w = w0 + (k < gw ? k : 0);
            g[k] = a.mg + w * a.stride + rowoff;
            e[k] = a.ef ? a.err + w * a.estride + rowoff : nullptr;
        }
        float acc[kGW][RP];
#pragma unroll
        for (int k = 0; k < kGW; ++k)
#pragma unroll
            for (int r = 0; r < RP; ++r) acc[k][r] = 0.f;
        if (vec) {
            for (int j = c0 + 4 * lane; j < c1; j += 128) {
                // every load of the step first (stores to E would otherwise keep the
                // next replica's loads from being issued early), then the sums
                float4 x[kGW], y[kGW];
#pragma unroll
                for (int k = 0; k < kGW; ++k) {
                    if (k >= gw) continue;
                    x[k] = __ldcs(reinterpret_cast<const float4*>(g[k] + j));
                    if (a.ef) y[k] = __ldcs(reinterpret_cast<const float4*>(e[k] + j));
                }
                if (a.ef) {
#pragma unroll
                    for (int k = 0; k < kGW; ++k) {
                        if (k >= gw) continue;
                        x[k] = make_float4(__fadd_rn(x[k].x, y[k].x), __fadd_rn(x[k].y, y[k].y), __fadd_rn(x[k].z, y[k].z),
                                           __fadd_rn(x[k].w, y[k].w));
                        __stcs(reinterpret_cast<float4*>(e[k] + j), x[k]);
                    }
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float qv[RP];
                    load_row<RP>(q + static_cast<int64_t>(j + c) * RP, qv);
#pragma unroll
                    for (int k = 0; k < kGW; ++k) {
                        if (k >= gw) continue;
                        const float xc = comp(x[k], c);
#pragma unroll
                        for (int r = 0; r < RP; ++r) acc[k][r] = fmaf(xc, qv[r], acc[k][r]);
                    }
                }
            }
        } else {
            for (int j = c0 + lane; j < c1; j += 32) {
                float qv[RP];
                load_row<RP>(q + static_cast<int64_t>(j) * RP, qv);
#pragma unroll
                for (int k = 0; k < kGW; ++k) {
                    if (k >= gw) continue;
                    float x = g[k][j];
                    if (a.ef) {
                        x = __fadd_rn(x, e[k][j]);
                        e[k][j] = x;
                    }
#pragma unroll
                    for (int r = 0; r < RP; ++r) acc[k][r] = fmaf(x, qv[r], acc[k][r]);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < kGW; ++k)
#pragma unroll
            for (int r = 0; r < RP; ++r)
#pragma unroll
                for (int o = 16; o; o >>= 1) acc[k][r] += __shfl_xor_sync(0xffffffffu, acc[k][r], o);
        if (lane == 0)
#pragma unroll
            for (int k = 0; k < kGW; ++k)
                if (k < gw)
#pragma unroll
                    for (int r = 0; r < RP; ++r) part[rl * a.W + w0 + k][r] = acc[k][r];
    }
    __syncthreads();
    // the all-reduce of P: replicas summed in order 0 .. W-1
    float* ps = a.PS + m.ps_off + (static_cast<int64_t>(t.w) * m.M + t.y) * RP;
    for (int k = threadIdx.x; k < t.z * RP; k += kThreads) {
        const int rl = k / RP, r = k % RP;
        float s = 0.f;
        for (int w = 0; w < a.W; ++w) s = __fadd_rn(s, part[rl * a.W + w][r]);
        ps[k] = s;
    }
}

// ---------------------------------------------------------------------------
// P^T P in pairs of floats (this GPU's fp64 rate is a small fraction of its fp32
// rate): each sum is carried as hi + lo with the error-free transformations
// TwoSum (Knuth) and TwoProduct (one fused multiply-add), the compensated dot
// product Dot2 of Ogita, Rump and Oishi ("Accurate sum and dot product", SIAM
// J. Sci. Comput. 26(6), 2005), which is as accurate as a sum in twice the
// working precision; partial pairs are merged the same way.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// (hi, lo) += x * y
__device__ __forceinline__ void dot2_add(float& hi, float& lo, float x, float y)
{
    const float h = __fmul_rn(x, y);
    const float r = __fmaf_rn(x, y, -h);   // x * y = h + r exactly
    float s, q;
    two_sum(hi, h, s, q);
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(q, r));
}

// (hi, lo) += (hi2, lo2)
__device__ __forceinline__ void dot2_merge(float& hi, float& lo, float hi2, float lo2)
{
    float s, q;
    two_sum(hi, hi2, s, q);
    hi = s;
    lo = __fadd_rn(__fadd_rn(lo, lo2), q);
}

// ---------------------------------------------------------------------------
// orthonormal columns of P (one block per tensor): P from the column splits'
// partial sums, P^T P summed over its rows in a fixed order, its Cholesky factor
// R (upper triangular, positive diagonal) and R^-1 on one thread, then P <- P R^-1 -- the
// orthonormal basis whose triangle has a positive diagonal.  A column whose
// pivot is not positive (zero, or in the span of the earlier columns) becomes 0.
// ---------------------------------------------------------------------------
template <int RP>
__global__ void __launch_bounds__(kThreads) psgd_orth_kernel(const PsgdArgs a)
{
    constexpr int NG = RP * (RP + 1) / 2;
    __shared__ float2 red[kWarps][NG];
    __shared__ double gsum[NG];
    __shared__ float rinv[RP][RP];
    const PsgdMat m = a.mats[blockIdx.x];
    float* p = a.P + m.p_off;
    {   // P = the column splits' partial sums added in split order; P^T P from the rows
        // as float pairs: thread i takes rows i, i + 256, ..., then a fixed tree over
        // the block (lanes, then warps in order)
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const float* ps = a.PS + m.ps_off;
        const int64_t plane = static_cast<int64_t>(m.M) * RP;
        float ghi[NG], glo[NG];
#pragma unroll
        for (int k = 0; k < NG; ++k) ghi[k] = glo[k] = 0.f;
        for (int i = threadIdx.x; i < m.M; i += kThreads) {
            float x[RP];
#pragma unroll
            for (int r = 0; r < RP; ++r) x[r] = ps[static_cast<int64_t>(i) * RP + r];
            for (int c = 1; c < m.psp; ++c)
#pragma unroll
                for (int r = 0; r < RP; ++r) x[r] = __fadd_rn(x[r], ps[c * plane + static_cast<int64_t>(i) * RP + r]);
#pragma unroll
            for (int r = 0; r < RP; ++r) p[static_cast<int64_t>(i) * RP + r] = x[r];
            int k = 0;
#pragma unroll
            for (int c = 0; c < RP; ++c)
#pragma unroll
                for (int d = c; d < RP; ++d, ++k) dot2_add(ghi[k], glo[k], x[c], x[d]);
        }
#pragma unroll
        for (int k = 0; k < NG; ++k) {
#pragma unroll
            for (int o = 16; o; o >>= 1)
                dot2_merge(ghi[k], glo[k], __shfl_xor_sync(0xffffffffu, ghi[k], o), __shfl_xor_sync(0xffffffffu, glo[k], o));
            if (lane == 0) red[warp][k] = make_float2(ghi[k], glo[k]);
        }
        __syncthreads();
        if (threadIdx.x < NG) {
            float hi = red[0][threadIdx.x].x, lo = red[0][threadIdx.x].y;
            for (int w = 1; w < kWarps; ++w) dot2_merge(hi, lo, red[w][threadIdx.x].x, red[w][threadIdx.x].y);
            gsum[threadIdx.x] = static_cast<double>(hi) + static_cast<double>(lo);
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {   // every loop unrolled: the small matrices stay in registers
        double G[RP][RP], R[RP][RP], X[RP][RP];
        bool ok[RP];
        {
            int k = 0;
#pragma unroll
            for (int c = 0; c < RP; ++c)
#pragma unroll
                for (int d = c; d < RP; ++d) {
                    G[c][d] = G[d][c] = gsum[k];
                    ++k;
                }
        }
#pragma unroll
        for (int c = 0; c < RP; ++c)
#pragma unroll
            for (int d = 0; d < RP; ++d) R[c][d] = X[c][d] = 0.0;
#pragma unroll
        for (int c = 0; c < RP; ++c) {
            double d = G[c][c];
#pragma unroll
            for (int q = 0; q < c; ++q)
                if (ok[q]) d -= R[q][c] * R[q][c];
            ok[c] = c < m.r && d > 0.0;
            const double inv = ok[c] ? rsqrt(d) : 1.0;
            const double rc = ok[c] ? d * inv : 1.0;
            R[c][c] = ok[c] ? rc : 0.0;
#pragma unroll
            for (int e = c + 1; e < RP; ++e) {
                double s = G[c][e];
#pragma unroll
                for (int q = 0; q < c; ++q)
                    if (ok[q]) s -= R[q][c] * R[q][e];
                R[c][e] = ok[c] ? s * inv : 0.0;
            }
            X[c][c] = ok[c] ? inv : 0.0;
        }
#pragma unroll
        for (int c = 0; c < RP; ++c) {   // column c of R^-1 (zero for a dropped column)
#pragma unroll
            for (int r = c - 1; r >= 0; --r) {
                double s = 0.0;
#pragma unroll
                for (int q = r + 1; q <= c; ++q) s += R[r][q] * X[q][c];
                X[r][c] = (ok[c] && ok[r]) ? -s * X[r][r] : 0.0;
            }
        }
#pragma unroll
        for (int c = 0; c < RP; ++c)
#pragma unroll
            for (int d = 0; d < RP; ++d) rinv[c][d] = static_cast<float>(X[c][d]);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < m.M; i += kThreads) {
        float* row = p + static_cast<int64_t>(i) * RP;
        float x[RP], y[RP];
#pragma unroll
        for (int c = 0; c < RP; ++c) x[c] = row[c];
#pragma unroll
        for (int c = 0; c < RP; ++c) {
            float s = 0.f;
#pragma unroll
            for (int q = 0; q <= c; ++q) s = fmaf(x[q], rinv[q][c], s);
            y[c] = s;
        }
#pragma unroll
        for (int c = 0; c < RP; ++c) row[c] = y[c];
    }
}

// ---------------------------------------------------------------------------
// partial Q_w = M_w^T P over one row split and one column block (tile: {mat,
// column block, unit}; unit = split * W + replica): the 8 warps take every 8th
// row of the split and their sums are added in warp order in shared memory.
// The last block of a column block to finish (a completion counter) adds the
// partials in the order (replica, split) and writes Q = sum / W.
// ---------------------------------------------------------------------------
template <int RP>
__device__ __forceinline__ void qpart_tile(const PsgdArgs& a, const int4 t, float (&red)[kWarps][128 * RP], int& last)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const PsgdMat m = a.mats[t.x];
    const int u = t.z;
    const int s = u / a.W, w = u % a.W;
    const int i0 = s * kRowsPerSplit, i1 = min(m.M, i0 + kRowsPerSplit);
    const float* src = (a.ef ? a.err + w * a.estride : a.mg + w * a.stride) + m.off;
    const float* p = a.P + m.p_off;
    float* out = a.QP + m.qp_off + static_cast<int64_t>(u) * m.N * RP;
    const int c0 = t.y * m.cbw;
    const int ncol = min(m.cbw, m.N - c0);
    const bool vec = m.vec && a.vec_ok;
    if (vec) {
        const int c = 4 * lane;
        float acc[4][RP];
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int r = 0; r < RP; ++r) acc[k][r] = 0.f;
        if (c < ncol) {
#pragma unroll 4
            for (int i = i0 + warp; i < i1; i += kWarps) {
                const float4 x = __ldcs(reinterpret_cast<const float4*>(src + static_cast<int64_t>(i) * m.N + c0 + c));
                float pv[RP];
                load_row<RP>(p + static_cast<int64_t>(i) * RP, pv);
#pragma unroll
                for (int r = 0; r < RP; ++r) {
                    acc[0][r] = fmaf(x.x, pv[r], acc[0][r]);
                    acc[1][r] = fmaf(x.y, pv[r], acc[1][r]);
                    acc[2][r] = fmaf(x.z, pv[r], acc[2][r]);
                    acc[3][r] = fmaf(x.w, pv[r], acc[3][r]);
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int r = 0; r < RP; ++r) red[warp][(c + k) * RP + r] = acc[k][r];
    } else {
        for (int c = lane; c < m.cbw; c += 32) {
            float acc[RP];
#pragma unroll
            for (int r = 0; r < RP; ++r) acc[r] = 0.f;
            if (c < ncol) {
#pragma unroll 4
                for (int i = i0 + warp; i < i1; i += kWarps) {
                    const float x = src[static_cast<int64_t>(i) * m.N + c0 + c];
                    float pv[RP];
                    load_row<RP>(p + static_cast<int64_t>(i) * RP, pv);
#pragma unroll
                    for (int r = 0; r < RP; ++r) acc[r] = fmaf(x, pv[r], acc[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < RP; ++r) red[warp][c * RP + r] = acc[r];
        }
    }
    __syncthreads();
    for (int k = threadIdx.x; k < ncol * RP; k += kThreads) {
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < kWarps; ++q) v = __fadd_rn(v, red[q][k]);
        out[static_cast<int64_t>(c0) * RP + k] = v;
    }
    // completion: the partial is published before the count (threadFenceReduction pattern)
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(a.CNT + m.cnt0 + t.y, 1) == m.S * a.W - 1;
    __syncthreads();
    if (!last) return;   // uniform over the block
    __threadfence();
    const int64_t plane = static_cast<int64_t>(m.N) * RP;
    const float wf = static_cast<float>(a.W);
    for (int k = threadIdx.x; k < ncol * RP; k += kThreads) {
        const int64_t el = static_cast<int64_t>(c0) * RP + k;
        // partial (replica ww, split s) is term ww * S + s: sixteen loads in flight,
        // each replica's splits added in order, then the replicas in order
        float tot = 0.f, qw = 0.f;
        const int nterm = a.W * m.S;
        for (int j0 = 0; j0 < nterm; j0 += 16) {
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int tj = j0 + j;
                v[j] = tj < nterm
                           ? __ldcg(a.QP + m.qp_off + (static_cast<int64_t>(tj % m.S) * a.W + tj / m.S) * plane + el)
                           : 0.f;
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int tj = j0 + j;
                if (tj < nterm) {
                    qw = __fadd_rn(qw, v[j]);
                    if (tj % m.S == m.S - 1) {
                        tot = __fadd_rn(tot, qw);
                        qw = 0.f;
                    }
                }
            }
        }
        a.Q[m.q_off + el] = __fdiv_rn(tot, wf);
    }
}

// One wave of blocks looping over the tiles (in table order: a block's next tile
// is gridDim.x further on).  The block-wide barriers inside a tile order the
// reuse of red and last across tiles.
template <int RP>
__global__ void __launch_bounds__(kThreads, q_min_blocks(RP)) psgd_qpart_kernel(const PsgdArgs a)
{
    __shared__ float red[kWarps][128 * RP];
    __shared__ int last;
    for (int i = blockIdx.x; i < a.n_qtiles; i += gridDim.x) qpart_tile<RP>(a, a.tiles[i], red, last);
}

// ---------------------------------------------------------------------------
// G^ = P Q^T on every replica, E = M - G^  (tile: {mat, row0, nrows}; one warp per row)
// ---------------------------------------------------------------------------
// Output rows of a row tile {mat, row0, rows, 0}: a warp per row (matrices whose
// rows are not 16-byte multiples).
template <int RP>
__device__ void out_rows(const PsgdArgs& a, const int4 t)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp >= t.z) return;
    const PsgdMat m = a.mats[t.x];
    const int row = t.y + warp;
    float pr[RP];
    load_row<RP>(a.P + m.p_off + static_cast<int64_t>(row) * RP, pr);
    const float* q = a.Q + m.q_off;
    const int64_t base = m.off + static_cast<int64_t>(row) * m.N;
    for (int j = lane; j < m.N; j += 32) {
        float qv[RP];
        load_row<RP>(q + static_cast<int64_t>(j) * RP, qv);
        float h = 0.f;
#pragma unroll
        for (int r = 0; r < RP; ++r) h = fmaf(pr[r], qv[r], h);
        for (int w = 0; w < a.W; ++w) {
            if (a.ef) {
                float* e = a.err + w * a.estride + base + j;
                *e = __fsub_rn(*e, h);
            }
            a.mg[w * a.stride + base + j] = h;
        }
    }
}

// Output of a flat tile {mat, quad0, quads, 1}: the matrix's rows laid end to end
// as 16-byte quads (N a multiple of 4), thread i taking quads i, i + 256, ...  Each
// quad's error loads for a batch of replicas are issued before the reads of P and
// Q that give G^ = P Q^T, then G^ goes to every replica and E - G^ back into E.
template <int RP>
__device__ void out_quads(const PsgdArgs& a, const int4 t)
{
    const PsgdMat m = a.mats[t.x];
    const int64_t n4 = m.N >> 2;
    const float* q = a.Q + m.q_off;
    const float* p = a.P + m.p_off;
    for (int k = threadIdx.x; k < t.z; k += kThreads) {
        const int64_t quad = static_cast<int64_t>(t.y) + k;
        const int64_t row = quad / n4;
        const int64_t col = (quad - row * n4) * 4;
        const int64_t e = m.off + quad * 4;
        float h[4];
        auto compute_h = [&]() {
            float pr[RP];
            load_row<RP>(p + row * RP, pr);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float qv[RP];
                load_row<RP>(q + (col + c) * RP, qv);
                float v = 0.f;
#pragma unroll
                for (int r = 0; r < RP; ++r) v = fmaf(pr[r], qv[r], v);
                h[c] = v;
            }
        };
        if (a.vec_ok) {
            for (int w0 = 0; w0 < a.W; w0 += kOutBatch) {
                const int nb = min(kOutBatch, a.W - w0);
                float4 x[kOutBatch];
                if (a.ef) {
#pragma unroll
                    for (int b = 0; b < kOutBatch; ++b)
                        if (b < nb) x[b] = __ldcs(reinterpret_cast<const float4*>(a.err + (w0 + b) * a.estride + e));
                }
                if (w0 == 0) compute_h();
                const float4 hv = make_float4(h[0], h[1], h[2], h[3]);
#pragma unroll
                for (int b = 0; b < kOutBatch; ++b) {
                    if (b >= nb) continue;
                    if (a.ef)
                        __stcs(reinterpret_cast<float4*>(a.err + (w0 + b) * a.estride + e),
                               make_float4(__fsub_rn(x[b].x, h[0]), __fsub_rn(x[b].y, h[1]), __fsub_rn(x[b].z, h[2]),
                                           __fsub_rn(x[b].w, h[3])));
                    __stcs(reinterpret_cast<float4*>(a.mg + (w0 + b) * a.stride + e), hv);
                }
            }
        } else {
            compute_h();
            for (int w = 0; w < a.W; ++w)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (a.ef) {
                        float* ep = a.err + w * a.estride + e + c;
                        *ep = __fsub_rn(*ep, h[c]);
                    }
                    a.mg[w * a.stride + e + c] = h[c];
                }
        }
    }
}

// ---------------------------------------------------------------------------
// G^ = P Q^T written to every replica, E <- M - G^ (the blocks loop over the
// output tiles)
// ---------------------------------------------------------------------------
template <int RP>
__global__ void __launch_bounds__(kThreads, 3) psgd_out_kernel(const PsgdArgs a)
{
    for (int i = blockIdx.x; i < a.n_otiles; i += gridDim.x) {
        const int4 t = a.tiles[i];
        if (t.w) out_quads<RP>(a, t);
        else out_rows<RP>(a, t);
    }
}

int round_rank(int r) { return r <= 1 ? 1 : r <= 2 ? 2 : r <= 4 ? 4 : 8; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int64_t align4(int64_t x) { return (x + 3) & ~static_cast<int64_t>(3); }

}  // namespace

struct ddp_powersgd {
    int32_t W = 1, rank = 1, RP = 1, ef = 1, start_iter = 0, iter = 0;
    int64_t bucket_numel = 0;
    int32_t nseg = 0;
    std::vector<int32_t> seg_mat;   // matrix index of each segment, -1 for 1-D
    std::vector<PsgdMat> mats;
    std::vector<PsgdVec> vecs;
    int64_t nvec = 0;
    std::vector<int4> t_p, t_q, t_o;
    int32_t rows_p = 1, ncnt = 0;
    int64_t q_elems = 0, p_elems = 0, qp_elems = 0, ps_elems = 0;
    // workspace: the tables, then the scratch (offsets from the scratch's start)
    size_t off_mats = 0, off_tp = 0, off_tq = 0, off_to = 0, off_vecs = 0, off_scratch = 0;
    size_t s_P = 0, s_QP = 0, s_PS = 0, s_CNT = 0, scratch_bytes = 0;
    size_t ws_bytes = 0;
    // bound buffers
    uint8_t* ws = nullptr;
    float* q = nullptr;
    float* err = nullptr;
    int64_t estride = 0;
};

namespace {

// The kernels' arguments over the bound buffers, with the scratch at `scratch`.
PsgdArgs make_args(const ddp_powersgd& h, uint8_t* scratch, float* main_grad, int64_t replica_stride)
{
    PsgdArgs a{};
    a.mg = main_grad;
    a.stride = replica_stride;
    a.err = h.err;
    a.estride = h.estride;
    a.P = reinterpret_cast<float*>(scratch + h.s_P);
    a.QP = reinterpret_cast<float*>(scratch + h.s_QP);
    a.PS = reinterpret_cast<float*>(scratch + h.s_PS);
    a.CNT = reinterpret_cast<int*>(scratch + h.s_CNT);
    a.Q = h.q;
    a.mats = reinterpret_cast<const PsgdMat*>(h.ws + h.off_mats);
    a.vecs = reinterpret_cast<const PsgdVec*>(h.ws + h.off_vecs);
    a.n_ptiles = static_cast<int32_t>(h.t_p.size());
    a.ncnt = h.ncnt;
    a.W = h.W;
    a.ef = h.ef && h.err;
    auto al16 = [](const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
    a.vec_ok = al16(main_grad) && replica_stride % 4 == 0 && (!a.ef || (al16(h.err) && h.estride % 4 == 0));
    a.inv_w = 1.0f / static_cast<float>(h.W);
    a.nvec = h.nvec;
    return a;
}

// Blocks of one wave of a kernel (SMs x its resident blocks), cached per device
// and kernel (`cached` is the kernel's own array).
template <typename Kernel>
size_t wave_blocks(Kernel kernel, std::atomic<int> (&cached)[ddp::kMaxDevices])
{
    const int dev = ddp::current_device();
    int n = dev >= 0 ? cached[dev].load(std::memory_order_relaxed) : 0;
    if (!n) {
        int v = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, kernel, kThreads, 0) != cudaSuccess || v < 1) v = 1;
        n = ddp::device_sm_count() * v;
        if (dev >= 0) cached[dev].store(n, std::memory_order_relaxed);
    }
    return static_cast<size_t>(n);
}

template <int RP>
size_t out_blocks()
{
    static std::atomic<int> cached[ddp::kMaxDevices] = {};
    return wave_blocks(psgd_out_kernel<RP>, cached);
}

template <int RP>
size_t q_blocks()
{
    static std::atomic<int> cached[ddp::kMaxDevices] = {};
    return wave_blocks(psgd_qpart_kernel<RP>, cached);
}

template <int RP>
ddp_status launch_all(const ddp_powersgd& h, const PsgdArgs& base, cudaStream_t s)
{
    PsgdArgs a = base;
    const unsigned nblocks_p = static_cast<unsigned>(h.t_p.size() + h.vecs.size());
    if (nblocks_p > 0) {
        a.tiles = reinterpret_cast<const int4*>(h.ws + h.off_tp);
        psgd_p_kernel<RP><<<nblocks_p, kThreads, 0, s>>>(a);
    }
    if (!h.mats.empty()) {
        psgd_orth_kernel<RP><<<static_cast<unsigned>(h.mats.size()), kThreads, 0, s>>>(a);
        a.tiles = reinterpret_cast<const int4*>(h.ws + h.off_tq);
        a.n_qtiles = static_cast<int32_t>(h.t_q.size());
        const size_t qgrid = DDP_PSGD_Q_WAVE ? std::min<size_t>(h.t_q.size(), q_blocks<RP>()) : h.t_q.size();
        psgd_qpart_kernel<RP><<<static_cast<unsigned>(qgrid), kThreads, 0, s>>>(a);
        a.tiles = reinterpret_cast<const int4*>(h.ws + h.off_to);
        a.n_otiles = static_cast<int32_t>(h.t_o.size());
        psgd_out_kernel<RP><<<static_cast<unsigned>(std::min<size_t>(h.t_o.size(), out_blocks<RP>())), kThreads, 0, s>>>(a);
    }
    const cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return ddp::fail(DDP_E_CUDA, "ddp_powersgd_reduce: kernel launch failed: %s", cudaGetErrorString(err));
    return DDP_OK;
}

ddp_status launch_rank(const ddp_powersgd& h, const PsgdArgs& a, cudaStream_t s)
{
    switch (h.RP) {
    case 1: return launch_all<1>(h, a, s);
    case 2: return launch_all<2>(h, a, s);
    case 4: return launch_all<4>(h, a, s);
    default: return launch_all<8>(h, a, s);
    }
}

}  // namespace

extern "C" ddp_status ddp_powersgd_create(int32_t W, int32_t rank, int32_t nseg, const int64_t* seg_offset,
                                          const int64_t* seg_numel, const int64_t* seg_rows, int64_t bucket_numel,
                                          int32_t error_feedback, int32_t start_iter, ddp_powersgd** out)
{
    using ddp::fail;
    const char* fn = "ddp_powersgd_create";
    if (!out) return fail(DDP_E_INVAL, "%s: out is NULL", fn);
    *out = nullptr;
    if (W < 1 || W > ddp::kMaxReplicas) return fail(DDP_E_INVAL, "%s: W = %d outside [1, %d]", fn, W, ddp::kMaxReplicas);
    if (rank < 1 || rank > 8) return fail(DDP_E_INVAL, "%s: rank = %d outside [1, 8]", fn, rank);
    if (nseg < 0 || bucket_numel < 0 || start_iter < 0) return fail(DDP_E_INVAL, "%s: negative size", fn);
    if (nseg > 0 && (!seg_offset || !seg_numel || !seg_rows)) return fail(DDP_E_INVAL, "%s: a segment array is NULL", fn);
    auto h = new ddp_powersgd();
    auto reject = [&](ddp_status s) {
        delete h;
        return s;
    };
    h->W = W;
    h->rank = rank;
    h->RP = round_rank(rank);
    h->ef = error_feedback != 0;
    h->start_iter = start_iter;
    h->bucket_numel = bucket_numel;
    h->nseg = nseg;
    h->seg_mat.assign(nseg, -1);
    {   // P tiles: about two warp units per warp, at most kMaxPairs (row, replica) pairs
        const int ngroups = (W + kGW - 1) / kGW;
        h->rows_p = std::max(1, std::min({kMaxPairs / W, 16 / ngroups, kMaxRowsP}));
    }
    const int RP = h->RP;
    for (int32_t t = 0; t < nseg; ++t) {
        const int64_t off = seg_offset[t], n = seg_numel[t], rows = seg_rows[t];
        if (off < 0 || n < 0 || off + n > bucket_numel)
            return reject(fail(DDP_E_INVAL, "%s: segment %d [%lld, +%lld) outside the bucket of %lld", fn, t,
                               static_cast<long long>(off), static_cast<long long>(n),
                               static_cast<long long>(bucket_numel)));
        if (rows < 0) return reject(fail(DDP_E_INVAL, "%s: segment %d has %lld rows", fn, t, static_cast<long long>(rows)));
        if (rows == 0) {
            for (int64_t i = 0; i < n; i += kVecPiece)   // pieces of at most kVecPiece elements, one block each
                h->vecs.push_back(PsgdVec{off + i, h->nvec + i, std::min<int64_t>(kVecPiece, n - i)});
            h->nvec += n;
            continue;
        }
        if (n % rows != 0 || n == 0)
            return reject(fail(DDP_E_INVAL, "%s: segment %d: %lld elements are not %lld rows", fn, t,
                               static_cast<long long>(n), static_cast<long long>(rows)));
        const int64_t cols = n / rows;
        if (rows > (1LL << 30) || cols * RP > (1LL << 30))
            return reject(fail(DDP_E_INVAL, "%s: segment %d: %lld x %lld too large", fn, t, static_cast<long long>(rows),
                               static_cast<long long>(cols)));
        PsgdMat m{};
        m.off = off;
        m.M = static_cast<int32_t>(rows);
        m.N = static_cast<int32_t>(cols);
        m.r = static_cast<int32_t>(std::min<int64_t>({rank, rows, cols}));
        m.vec = (off % 4 == 0) && (cols % 4 == 0);
        m.cbw = m.vec ? 128 : 32;
        m.S = static_cast<int32_t>((rows + kRowsPerSplit - 1) / kRowsPerSplit);
        m.p_off = h->p_elems;
        h->p_elems += align4(rows * RP);
        m.q_off = h->q_elems;
        h->q_elems += align4(cols * RP);
        m.qp_off = h->qp_elems;
        h->qp_elems += align4(static_cast<int64_t>(m.S) * W * cols * RP);
        const int32_t mi = static_cast<int32_t>(h->mats.size());
        // P tiles: rows_p rows by one column split; rows longer than p_cols(RP)
        // columns are cut into equal splits of whole 128-column blocks
        m.psp = 1;
        m.pcw = m.N;
        const int pcols = p_cols(RP);
        if (cols > pcols) {
            const int64_t parts = (cols + pcols - 1) / pcols;
            m.pcw = static_cast<int32_t>(((cols + parts - 1) / parts + 127) / 128 * 128);
            m.psp = static_cast<int32_t>((cols + m.pcw - 1) / m.pcw);
        }
        m.ps_off = h->ps_elems;
        h->ps_elems += align4(static_cast<int64_t>(m.psp) * rows * RP);
        for (int32_t cs = 0; cs < m.psp; ++cs)
            for (int32_t r0 = 0; r0 < m.M; r0 += h->rows_p)
                h->t_p.push_back(make_int4(mi, r0, std::min(h->rows_p, m.M - r0), cs));
        const int64_t quads = rows * cols / 4;
        if (m.vec && quads < (int64_t{1} << 31) - kOutQuads) {
            for (int64_t q0 = 0; q0 < quads; q0 += kOutQuads)
                h->t_o.push_back(make_int4(mi, static_cast<int32_t>(q0),
                                           static_cast<int32_t>(std::min<int64_t>(kOutQuads, quads - q0)), 1));
        } else {
            for (int32_t r0 = 0; r0 < m.M; r0 += kRowsOut)
                h->t_o.push_back(make_int4(mi, r0, std::min(kRowsOut, m.M - r0), 0));
        }
        const int32_t ncb = (m.N + m.cbw - 1) / m.cbw, units = m.S * W;
        m.cnt0 = h->ncnt;
        h->ncnt += ncb;
        for (int32_t cb = 0; cb < ncb; ++cb)
            for (int32_t u = 0; u < units; ++u) h->t_q.push_back(make_int4(mi, cb, u, 0));
        h->seg_mat[t] = mi;
        h->mats.push_back(m);
    }
    size_t o = 0;
    h->off_mats = o;
    o = align256(o + h->mats.size() * sizeof(PsgdMat));
    h->off_tp = o;
    o = align256(o + h->t_p.size() * sizeof(int4));
    h->off_tq = o;
    o = align256(o + h->t_q.size() * sizeof(int4));
    h->off_to = o;
    o = align256(o + h->t_o.size() * sizeof(int4));
    h->off_vecs = o;
    o = align256(o + h->vecs.size() * sizeof(PsgdVec));
    h->off_scratch = o;
    size_t sc = 0;
    h->s_P = sc;
    sc = align256(sc + static_cast<size_t>(h->p_elems) * sizeof(float));
    h->s_QP = sc;
    sc = align256(sc + static_cast<size_t>(h->qp_elems) * sizeof(float));
    h->s_PS = sc;
    sc = align256(sc + static_cast<size_t>(h->ps_elems) * sizeof(float));
    h->s_CNT = sc;
    sc = align256(sc + static_cast<size_t>(h->ncnt) * sizeof(int));
    h->scratch_bytes = sc;
    h->ws_bytes = std::max<size_t>(o + sc, 256);
    *out = h;
    return ddp::ok();
}

extern "C" ddp_status ddp_powersgd_sizes(const ddp_powersgd* h, int64_t* workspace_bytes, int64_t* q_elems,
                                         int32_t* nmatrices)
{
    if (!h) return ddp::fail(DDP_E_INVAL, "ddp_powersgd_sizes: handle is NULL");
    if (workspace_bytes) *workspace_bytes = static_cast<int64_t>(h->ws_bytes);
    if (q_elems) *q_elems = h->q_elems;
    if (nmatrices) *nmatrices = static_cast<int32_t>(h->mats.size());
    return ddp::ok();
}

extern "C" ddp_status ddp_powersgd_matrix(const ddp_powersgd* h, int32_t seg, int64_t* q_offset, int32_t* rows,
                                          int32_t* cols, int32_t* rank_eff, int32_t* rank_pad)
{
    const char* fn = "ddp_powersgd_matrix";
    if (!h) return ddp::fail(DDP_E_INVAL, "%s: handle is NULL", fn);
    if (seg < 0 || seg >= h->nseg) return ddp::fail(DDP_E_INVAL, "%s: segment %d outside [0, %d)", fn, seg, h->nseg);
    const int32_t mi = h->seg_mat[seg];
    if (mi < 0) return ddp::fail(DDP_E_INVAL, "%s: segment %d is a 1-D tensor", fn, seg);
    const PsgdMat& m = h->mats[mi];
    if (q_offset) *q_offset = m.q_off;
    if (rows) *rows = m.M;
    if (cols) *cols = m.N;
    if (rank_eff) *rank_eff = m.r;
    if (rank_pad) *rank_pad = h->RP;
    return ddp::ok();
}

extern "C" ddp_status ddp_powersgd_bind(ddp_powersgd* h, void* workspace, int64_t workspace_bytes, float* q_state,
                                        float* error, int64_t error_stride, void* stream)
{
    using ddp::fail;
    const char* fn = "ddp_powersgd_bind";
    if (!h) return fail(DDP_E_INVAL, "%s: handle is NULL", fn);
    if (!workspace || workspace_bytes < static_cast<int64_t>(h->ws_bytes))
        return fail(DDP_E_INVAL, "%s: workspace of %lld bytes, %lld needed", fn, static_cast<long long>(workspace_bytes),
                    static_cast<long long>(h->ws_bytes));
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return fail(DDP_E_INVAL, "%s: workspace not 256-byte aligned", fn);
    if (h->q_elems > 0 && (!q_state || reinterpret_cast<uintptr_t>(q_state) % 16 != 0))
        return fail(DDP_E_INVAL, "%s: q_state is NULL or not 16-byte aligned", fn);
    if (h->ef && !h->mats.empty() && (!error || error_stride < h->bucket_numel))
        return fail(DDP_E_INVAL, "%s: error feedback needs an error buffer with stride >= %lld", fn,
                    static_cast<long long>(h->bucket_numel));
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    auto put = [&](size_t off, const void* src, size_t bytes) {
        return bytes == 0 ? cudaSuccess : cudaMemcpyAsync(ws + off, src, bytes, cudaMemcpyHostToDevice, s);
    };
    cudaError_t e = put(h->off_mats, h->mats.data(), h->mats.size() * sizeof(PsgdMat));
    if (e == cudaSuccess) e = put(h->off_tp, h->t_p.data(), h->t_p.size() * sizeof(int4));
    if (e == cudaSuccess) e = put(h->off_tq, h->t_q.data(), h->t_q.size() * sizeof(int4));
    if (e == cudaSuccess) e = put(h->off_to, h->t_o.data(), h->t_o.size() * sizeof(int4));
    if (e == cudaSuccess) e = put(h->off_vecs, h->vecs.data(), h->vecs.size() * sizeof(PsgdVec));
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(DDP_E_CUDA, "%s: %s", fn, cudaGetErrorString(e));
    h->ws = ws;
    h->q = q_state;
    h->err = h->ef ? error : nullptr;
    h->estride = error_stride;
    return ddp::ok();
}

extern "C" ddp_status ddp_powersgd_set_q(ddp_powersgd* h, int32_t seg, const float* q, void* stream)
{
    using ddp::fail;
    const char* fn = "ddp_powersgd_set_q";
    if (!h) return fail(DDP_E_INVAL, "%s: handle is NULL", fn);
    if (!h->q) return fail(DDP_E_STATE, "%s: call ddp_powersgd_bind first", fn);
    if (seg < 0 || seg >= h->nseg || h->seg_mat[seg] < 0)
        return fail(DDP_E_INVAL, "%s: segment %d is not a matrix of this bucket", fn, seg);
    if (!q) return fail(DDP_E_INVAL, "%s: q is NULL", fn);
    const PsgdMat& m = h->mats[h->seg_mat[seg]];
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* dst = h->q + m.q_off;
    const size_t pitch = static_cast<size_t>(h->RP) * sizeof(float);
    cudaError_t e = cudaMemsetAsync(dst, 0, static_cast<size_t>(m.N) * pitch, s);
    if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(dst, pitch, q, static_cast<size_t>(m.r) * sizeof(float), static_cast<size_t>(m.r) * sizeof(float),
                              static_cast<size_t>(m.N), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(DDP_E_CUDA, "%s: %s", fn, cudaGetErrorString(e));
    return ddp::ok();
}

extern "C" ddp_status ddp_powersgd_reduce(ddp_powersgd* h, float* main_grad, int64_t replica_stride, void* stream)
{
    using ddp::fail;
    const char* fn = "ddp_powersgd_reduce";
    if (!h) return fail(DDP_E_INVAL, "%s: handle is NULL", fn);
    if (!main_grad) return fail(DDP_E_INVAL, "%s: main_grad is NULL", fn);
    if (h->W > 1 && replica_stride < h->bucket_numel)
        return fail(DDP_E_INVAL, "%s: replica_stride %lld < bucket numel %lld", fn, static_cast<long long>(replica_stride),
                    static_cast<long long>(h->bucket_numel));
    if (h->iter < h->start_iter) {
        const ddp_status st = ddp::launch_allreduce(main_grad, replica_stride, h->bucket_numel, h->W, DDP_ALLREDUCE, stream);
        if (st == DDP_OK) ++h->iter;
        return st;
    }
    if (!h->ws) return fail(DDP_E_STATE, "%s: call ddp_powersgd_bind first", fn);
    const ddp_status st = launch_rank(*h, make_args(*h, h->ws + h->off_scratch, main_grad, replica_stride),
                                      static_cast<cudaStream_t>(stream));
    if (st != DDP_OK) return st;
    ++h->iter;
    return ddp::ok();
}

extern "C" ddp_status ddp_powersgd_iter(const ddp_powersgd* h, int32_t* iter)
{
    if (!h || !iter) return ddp::fail(DDP_E_INVAL, "ddp_powersgd_iter: NULL argument");
    *iter = h->iter;
    return ddp::ok();
}

extern "C" void ddp_powersgd_destroy(ddp_powersgd* h) { delete h; }

int32_t ddp::powersgd_replicas(const ddp_powersgd* h) { return h->W; }
int64_t ddp::powersgd_numel(const ddp_powersgd* h) { return h->bucket_numel; }

// ---------------------------------------------------------------------------
// ddp_powersgd_reduce_static: the same kernels with their scratch (the summed
// P, the partial sums of Q, the shares of P^T P and the completion counters)
// in a fixed device array of this library instead of the caller's workspace.
// Within one call every part of that scratch is written before it is read
// (the counters are zeroed by the first kernel), so nothing needs clearing.
// ---------------------------------------------------------------------------
namespace {

constexpr int64_t kStaticScratchBytes = DDP_POWERSGD_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_psgd_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
uint8_t* g_static_ptr[kMaxDevices] = {};

// The array's address on the current device, looked up once per device and
// kept for the life of the process.  cudaDeviceReset on a device unloads the
// library's module there, so the kept address is then stale: this entry point
// must not be called again on that device in the same process.
ddp_status static_scratch(uint8_t** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return ddp::fail(DDP_E_CUDA, "ddp_powersgd_reduce_static: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return ddp::fail(DDP_E_INVAL, "ddp_powersgd_reduce_static: device %d beyond the %d supported", dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_psgd_static_scratch);
        if (e != cudaSuccess)
            return ddp::fail(DDP_E_CUDA, "ddp_powersgd_reduce_static: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
        g_static_ptr[dev] = static_cast<uint8_t*>(p);
    }
    *out = g_static_ptr[dev];
    return DDP_OK;
}

}  // namespace

extern "C" ddp_status ddp_powersgd_reduce_static(ddp_powersgd* h, float* main_grad, int64_t replica_stride,
                                                 void* stream)
{
    using ddp::fail;
    const char* fn = "ddp_powersgd_reduce_static";
    if (!h) return fail(DDP_E_INVAL, "%s: handle is NULL", fn);
    if (!main_grad) return fail(DDP_E_INVAL, "%s: main_grad is NULL", fn);
    if (h->W > 1 && replica_stride < h->bucket_numel)
        return fail(DDP_E_INVAL, "%s: replica_stride %lld < bucket numel %lld", fn, static_cast<long long>(replica_stride),
                    static_cast<long long>(h->bucket_numel));
    if (h->iter < h->start_iter) {  // warm-up: the plain all-reduce, which uses no scratch
        const ddp_status st = ddp::launch_allreduce(main_grad, replica_stride, h->bucket_numel, h->W, DDP_ALLREDUCE, stream);
        if (st == DDP_OK) ++h->iter;
        return st;
    }
    if (static_cast<int64_t>(h->scratch_bytes) > kStaticScratchBytes)
        return fail(DDP_E_CAPACITY, "%s: this bucket needs %lld bytes of scratch, the static array holds %lld "
                    "(use ddp_powersgd_reduce with a workspace)", fn, static_cast<long long>(h->scratch_bytes),
                    static_cast<long long>(kStaticScratchBytes));
    if (!h->ws) return fail(DDP_E_STATE, "%s: call ddp_powersgd_bind first", fn);
    uint8_t* scratch = nullptr;
    const ddp_status sst = static_scratch(&scratch);
    if (sst != DDP_OK) return sst;
    const ddp_status st = launch_rank(*h, make_args(*h, scratch, main_grad, replica_stride), static_cast<cudaStream_t>(stream));
    if (st != DDP_OK) return st;
    ++h->iter;
    return ddp::ok();
}
