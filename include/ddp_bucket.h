/*
 * ddp_bucket.h -- C ABI of libddpbucket, the gradient-bucket reduction of
 * data-parallel training on one GB300 (sm_103a).
 *
 * The path has five steps, each an entry point below:
 *   assign    parameters -> size-capped buckets          (host)
 *   pack      per-parameter gradients -> fp32 bucket      (device kernel)
 *   reduce    W replicas of a bucket, ring order, 1/W     (device kernel)
 *   unpack    reduced bucket -> per-parameter gradients   (device kernel)
 *   schedule  in-order bucket issue gated by events       (host + device)
 * plus ddp_fused_bucket, which does pack + reduce + unpack in one pass.
 *
 * The W data-parallel ranks are W replica buffers in this GPU's memory; the
 * ring's summation order is reproduced element by element inside the kernels.
 *
 * Sources (page title, section):
 *   "DDP: ring AllReduce and gradient buckets" (PyTorch internals book, ch. 17)
 *     -- the DDP chapter below;
 *   "Lecture 15: PyTorch DDP" (CMU 11-868 notes) -- the lecture;
 *   "Megatron DDP: contiguous buffer and overlap" -- the Megatron page.
 *
 * Conventions for every call:
 *   - Status: every call returns a ddp_status (int32_t).  Nothing is thrown
 *     across the ABI.  On failure ddp_last_error_message() (per thread) says
 *     why, naming the parameter or bucket involved.  Arguments are validated on
 *     the host before anything is launched; a failed call launches nothing.
 *   - Memory: the caller owns all host and device memory.  The library
 *     allocates no device memory; its own device data are three small static
 *     arrays of the module (the status word of ddp_device_status, the
 *     streaming kernels' pool counters, and the scratch of
 *     ddp_powersgd_reduce_static).  A reducer owns host bookkeeping and the
 *     CUDA events it creates, released by ddp_reducer_destroy; a host front end
 *     owns two copy streams, one gate stream and its events, released by
 *     ddp_host_front_destroy; the library keeps up to 64 events per device for
 *     the pool counters until exit.
 *   - Streams: `stream` arguments are cudaStream_t handles passed as void*
 *     (NULL = the legacy default stream).  Data-path calls are asynchronous on
 *     that stream; only ddp_reducer_finalize with a timeout waits on the host.
 *   - Pointers marked DEVICE must be device (or managed) memory of the current
 *     device; HOST pointers are ordinary host memory read during the call.
 *   - Element types: DDP_F32, DDP_BF16, DDP_F16 gradients; buckets
 *     (main_grad) are always fp32 (the Megatron page, section 1: main_grad in
 *     fp32, grad_reduce_in_fp32).
 *   - Sizes are element counts unless a name ends in _bytes.
 *   - Alignment: no alignment is required.  16-byte-aligned buffers whose
 *     offsets keep that alignment take the vector path; the rest is done with
 *     scalar accesses on the GPU (there is no CPU fallback).
 *   - Threads and devices: every entry point may be called from several host
 *     threads at once and for several devices in one process (the launch
 *     caches -- occupancy, function attributes, symbol addresses -- are kept
 *     per device, in atomics), with these exceptions: a reducer, a plan
 *     under construction, a PowerSGD state and a host front end (with its
 *     reducer) are used by one thread at a time, and ddp_set_kernel_variant is
 *     process-wide.  Kernels launch on the
 *     device that is current in the calling thread; pointers must belong to it.
 */
#ifndef DDP_BUCKET_H
#define DDP_BUCKET_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t ddp_status;
enum {
    DDP_OK = 0,
    DDP_E_INVAL = 1,      /* bad argument (null pointer, size, range, mode) */
    DDP_E_ALIGN = 2,      /* reserved: a layout no kernel path accepts */
    DDP_E_CUDA = 3,       /* a CUDA runtime call failed (message has the CUDA error) */
    DDP_E_STATE = 4,      /* call out of order, e.g. a parameter marked ready twice */
    DDP_E_INCOMPLETE = 5, /* buckets not all reduced: some parameters never marked ready */
    DDP_E_TIMEOUT = 6,    /* ddp_reducer_finalize's deadline passed before the GPU finished */
    DDP_E_CAPACITY = 7    /* an output array is too small */
};

enum { DDP_F32 = 0, DDP_BF16 = 1, DDP_F16 = 2 };

/* Bucket assignment orders. */
enum {
    /* Rebuilt DDP buckets: parameters in reverse model.parameters() order
     * (approximately the order backward produces gradients); bucket 0 gets
     * first_cap_bytes, the rest cap_bytes; issued 0, 1, 2, ...
     * (DDP chapter, sections 17.2 and 17.13; lecture, section 2.2). */
    DDP_ORDER_REVERSE = 0,
    /* Initial DDP buckets (also find_unused_parameters=True): computed over
     * forward order with caps [first, cap, cap, ...], then the bucket list is
     * reversed, so the first-cap bucket comes last (DDP chapter, 17.13). */
    DDP_ORDER_FWD_THEN_REVERSE = 1,
    /* Megatron contiguous buffer: forward layout, bucket 0 holds p0, every
     * bucket capped at cap_bytes (first_cap_bytes ignored), numel padded to a
     * multiple of pad_multiple; issued from the last bucket to the first,
     * the order backward fills them (Megatron page, sections 1-2). */
    DDP_ORDER_MEGATRON = 2
};

/* Reduction modes (Megatron page, section 3, start_grad_sync). */
enum {
    DDP_ALLREDUCE = 0,      /* every replica ends with the mean of the bucket */
    DDP_REDUCE_SCATTER = 1  /* replica r ends with the mean of shard r only */
};

/* ------------------------------------------------------------------------ */
/* Step 1: bucket assignment (host)                                          */
/* ------------------------------------------------------------------------ */
/*
 * ddp_assign_buckets -- map parameters to size-capped buckets.
 *
 * Defined by: DDP chapter 17.2 (a bucket is closed once its bytes reach the
 * cap, so it may overshoot; default cap 25 MiB; the rebuilt first bucket uses
 * 1 MiB) and 17.13 (reversed order, the rebuilt and the initial assignment);
 * lecture 2.2 (fill in reverse parameter order, close at the cap) and exercise
 * 3; lecture answer 9 and the Megatron page 1 (one dtype per bucket buffer;
 * max(40 MB, 1 MB x DP) buckets over a contiguous fp32 buffer).
 *
 * Rule: walk the parameters in the order's iteration order; append each to the
 * open bucket of its dtype; after appending, if that bucket's bytes >= its cap,
 * close it.  Each dtype group keeps its own cap sequence (first cap for its
 * first bucket, except DDP_ORDER_MEGATRON).  At the end the still-open buckets
 * are closed in order of their dtype's first appearance.  Offsets are tight
 * (no gaps) in append order; bucket_numel is rounded up to pad_multiple.
 * Bucket bytes count 4 bytes per element when grad_reduce_in_fp32 != 0 (the
 * bucket is fp32 main_grad), else the dtype's own size.
 *
 * HOST in:  numels[nparams] (>= 0), dtypes[nparams] (DDP_F32/BF16/F16),
 *           cap_bytes > 0, first_cap_bytes > 0, order (DDP_ORDER_*),
 *           pad_multiple >= 1.
 * HOST out (caller-allocated): bucket_of[nparams], offset_of[nparams]
 *           (elements from the bucket's start), members[nparams] (bucket 0's
 *           parameters in layout order, then bucket 1's, ...), and per bucket
 *           (max_buckets entries): bucket_numel (padded), bucket_bytes
 *           (unpadded), bucket_dtype, bucket_order (bucket_order[k] = bucket
 *           issued k-th); *nbuckets.
 * Errors: DDP_E_INVAL (null pointer, bad value, nparams < 0);
 *         DDP_E_CAPACITY if more than max_buckets buckets are needed
 *         (*nbuckets then holds the count needed).  nparams + 2 always suffices.
 */
ddp_status ddp_assign_buckets(const int64_t* numels, const int32_t* dtypes, int32_t nparams,
                              int64_t cap_bytes, int64_t first_cap_bytes, int32_t order,
                              int32_t pad_multiple, int32_t grad_reduce_in_fp32,
                              int32_t* bucket_of, int64_t* offset_of, int32_t* members,
                              int64_t* bucket_numel, int64_t* bucket_bytes, int32_t* bucket_dtype,
                              int32_t* bucket_order, int32_t max_buckets, int32_t* nbuckets);

/*
 * ddp_assign_buckets_ordered -- rebuilt buckets: the same rule as
 * ddp_assign_buckets, walking the parameters in `sequence` (the order their
 * gradients were observed in; see ddp_reducer_ready_order).
 *
 * Defined by: DDP chapter 17.13 (the first backward records the order
 * gradients arrive in; the next forward re-buckets in that order, the earliest
 * gradients into bucket 0 under the 1 MiB first cap, the rest under
 * bucket_cap_mb).  Issue order is bucket index order (bucket_order[k] = k).
 * Each dtype group keeps its own cap sequence, as in ddp_assign_buckets.
 *
 * HOST in: sequence[nparams], a permutation of 0..nparams-1; the rest and the
 * outputs as ddp_assign_buckets (without `order`).
 * Errors: as ddp_assign_buckets; DDP_E_INVAL if sequence is not a permutation.
 */
ddp_status ddp_assign_buckets_ordered(const int64_t* numels, const int32_t* dtypes, int32_t nparams,
                                      const int32_t* sequence, int64_t cap_bytes, int64_t first_cap_bytes,
                                      int32_t pad_multiple, int32_t grad_reduce_in_fp32, int32_t* bucket_of,
                                      int64_t* offset_of, int32_t* members, int64_t* bucket_numel,
                                      int64_t* bucket_bytes, int32_t* bucket_dtype, int32_t* bucket_order,
                                      int32_t max_buckets, int32_t* nbuckets);

/*
 * ddp_overlap_timeline -- the overlap model of the lecture (section 3.1,
 * exercises 4 and 5), on the host.  Gradient p appears at ready_ms[p]; bucket
 * b (of bucket_bytes[b] bytes) is reduced as soon as its last gradient exists
 * and the bucket issued before it (bucket_order) is done, taking
 * alpha_ms + ms_per_byte * bucket_bytes[b].  (A ring over K ranks with latency
 * alpha and bandwidth beta: alpha_ms = 2(K-1)alpha, ms_per_byte = 2(K-1)/(K beta).)
 *
 * HOST out: start_ms[b], end_ms[b] (indexed by bucket id); *step_ms = when the
 * gradients and every reduction are done; *serial_ms = the step without
 * overlap (every reduction after the last gradient).
 * Errors: DDP_E_INVAL (NULL array, negative size or cost, bucket_of out of
 * range, bucket_order not a permutation).
 */
ddp_status ddp_overlap_timeline(int32_t nparams, const double* ready_ms, int32_t nbuckets, const int32_t* bucket_of,
                                const int32_t* bucket_order, const int64_t* bucket_bytes, double alpha_ms,
                                double ms_per_byte, double* start_ms, double* end_ms, double* step_ms,
                                double* serial_ms);

/* ------------------------------------------------------------------------ */
/* Bucket descriptor used by the device steps                                */
/* ------------------------------------------------------------------------ */
/*
 * One bucket as the kernels see it (DDP chapter 17.2: a bucket has an index,
 * a flat buffer and a parameter list; lecture 2.2, GradBucket).  The struct is
 * HOST memory passed by pointer; its two tables are DEVICE arrays that the
 * caller fills once from ddp_assign_buckets's output and keeps alive while
 * kernels that use them run.
 *
 *   numel       elements of the bucket, padding included (bucket_numel[b]).
 *   nseg        parameters in the bucket (>= 0).
 *   dtype       gradient dtype of every segment (bucket_dtype[b]).
 *   seg_offset  DEVICE int64[nseg + 1], ascending: segment s covers bucket
 *               elements [seg_offset[s], seg_offset[s+1]); seg_offset[0] == 0;
 *               [seg_offset[nseg], numel) is padding.
 *   seg_param   DEVICE int32[nseg]: the parameter (column of the pointer
 *               tables below) of segment s.
 *
 * Pointer tables (DEVICE arrays of device pointers, replica-major, leading
 * dimension ld >= 1 + the largest seg_param):
 *   grads[w * ld + p]      replica w's gradient of parameter p (dtype, numel
 *                          elements); may be NULL where used[] says unused.
 *   grads_out[w * ld + p]  fp32 destination of the reduced gradient.
 *   used[w * ld + p]       uint8, nonzero if replica w produced a gradient
 *                          for p this iteration (NULL: all used).
 *   global_used[p]         uint8, nonzero if any replica used p (NULL: all).
 *
 * Replicated buckets: main_grad points at replica 0's copy of the bucket;
 * replica w's copy starts replica_stride elements after replica w-1's
 * (replica_stride >= numel).
 */
typedef struct ddp_bucket_desc {
    int64_t numel;
    int32_t nseg;
    int32_t dtype;
    const int64_t* seg_offset;
    const int32_t* seg_param;
} ddp_bucket_desc;

/* ------------------------------------------------------------------------ */
/* Step 2: pack (device)                                                     */
/* ------------------------------------------------------------------------ */
/*
 * ddp_pack -- copy (or accumulate) per-parameter gradients into the bucket.
 *
 * Defined by: DDP chapter 17.12 (mark_variable_ready copies the gradient into
 * the bucket's flat buffer) and 17.5; Megatron page 1 (fp32 main_grad, bf16
 * gradients widened); lecture 4.1 and the summary of Li et al. 2020 section
 * 2.2.4 (no_sync: gradients accumulate locally and the next synchronised
 * backward reduces the sum); DDP chapter 17.33 (an unused parameter's segment
 * is zero).
 *
 * For every replica w and bucket element e in segment s (parameter p, index
 * i = e - seg_offset[s]):
 *   accumulate == 0:  main_grad[w][e] = used ? (float)grads[w][p][i] : 0
 *   accumulate != 0:  main_grad[w][e] = main_grad[w][e] + (float)grads[w][p][i]
 *                     (unchanged where unused)
 * Padding elements are set to 0 when accumulate == 0 and left alone otherwise.
 * No 1/W scaling here: the scale is fused into the reduction.
 *
 * Errors: DDP_E_INVAL (W outside [1, 64], null desc/tables/main_grad,
 * replica_stride < numel, ld < 1, negative sizes); DDP_E_CUDA (launch failure).
 */
ddp_status ddp_pack(const ddp_bucket_desc* bucket, const void* const* grads, const uint8_t* used,
                    int32_t ld, int32_t W, float* main_grad, int64_t replica_stride,
                    int32_t accumulate, void* stream);

/*
 * ddp_pack_group -- ddp_pack over several buckets in as few kernel launches as
 * possible (one per run of up to 32 buckets of one dtype): a no_sync
 * micro-step's local accumulation over the whole model in one call.  Results
 * are those of ddp_pack on each bucket in turn.
 *   buckets[nbuckets], bucket_start[nbuckets]  HOST, as ddp_fused_bucket_group;
 *   main_grad   DEVICE start of the per-replica buffer holding all buckets.
 * Errors: as ddp_pack for any bucket; DDP_E_INVAL if a bucket does not fit in
 * replica_stride.  Nothing is launched when a bucket is rejected.
 */
ddp_status ddp_pack_group(const ddp_bucket_desc* buckets, const int64_t* bucket_start, int32_t nbuckets,
                          const void* const* grads, const uint8_t* used, int32_t ld, int32_t W, float* main_grad,
                          int64_t replica_stride, int32_t accumulate, void* stream);

/* ------------------------------------------------------------------------ */
/* Step 3: reduce (device)                                                   */
/* ------------------------------------------------------------------------ */
/*
 * ddp_bucket_allreduce -- average W replicas of one fp32 bucket in place, in
 * the ring allreduce's summation order.
 *
 * Defined by: DDP chapter 17.4 (ring: reduce-scatter in N-1 steps, each rank
 * sending 1/N to the next and adding what arrives, then all-gather in N-1
 * steps) and 17.1, 17.9 (every rank ends with the average; each contribution is
 * multiplied by 1/world_size); Megatron page 3 (reduce_scatter leaves shard r
 * on rank r; scaling by 1/DP before the collective).
 *
 * With chunk length L = ceil(n / W), chunk c = [c*L, min((c+1)*L, n)).  For an
 * element e of chunk c, with x_w = replicas[w*replica_stride + e] * fp32(1/W)
 * (each product rounded to fp32):
 *   s = x_{(c+1)%W}; then s = s + x_{(c+k)%W} for k = 2..W (fp32, in order)
 * i.e. the order in which the ring's reduce-scatter visits ranks, ending on
 * rank c.  No fused multiply-add is used.
 *   DDP_ALLREDUCE:       s is written to element e of every replica.
 *   DDP_REDUCE_SCATTER:  s is written to element e of replica c only (shard c
 *                        of replica c); every other element is left as is.
 *                        Requires n % W == 0.
 * W == 1 leaves the bucket unchanged; n == 0 does nothing.
 *
 * replicas: DEVICE fp32, W copies, replica_stride >= n apart.
 * Errors: DDP_E_INVAL (W outside [1, 64], null pointer with n > 0, stride < n,
 * bad mode, reduce-scatter with n % W != 0); DDP_E_CUDA.
 */
ddp_status ddp_bucket_allreduce(float* replicas, int64_t replica_stride, int64_t numel, int32_t W,
                                int32_t mode, void* stream);

/*
 * ddp_bucket_allreduce_wire -- ddp_bucket_allreduce through a compression hook:
 * the allreduce runs in a 16-bit wire type.
 *
 * Defined by: DDP chapter 17.9 and 17.20 (bf16_compress_hook /
 * fp16_compress_hook: the fp32 bucket is converted to bf16 (fp16) and divided
 * by the world size, the converted tensor is allreduced with a sum, and the
 * result is copied back into the fp32 bucket).
 *
 * For an element of chunk c: z_w = wire(wire(x_w) / W) for every replica w,
 * where wire() rounds to the wire type, to nearest with ties to even; then
 * s = z_{c+1}; s = wire(s + z_{c+k}) for k = 2..W (the ring's order, every
 * partial sum a wire value, as the messages are); the result is s widened to
 * fp32.  Output placement as for ddp_bucket_allreduce.  W == 1 still rounds to
 * the wire type.  fp16 saturates to infinity beyond 65504.
 *
 * wire_dtype: DDP_BF16 or DDP_F16 (DDP_F32 gives ddp_bucket_allreduce).
 * Errors: as ddp_bucket_allreduce; DDP_E_INVAL for another wire_dtype.
 */
ddp_status ddp_bucket_allreduce_wire(float* replicas, int64_t replica_stride, int64_t numel, int32_t W,
                                     int32_t mode, int32_t wire_dtype, void* stream);

/* ------------------------------------------------------------------------ */
/* Step 4: unpack (device)                                                   */
/* ------------------------------------------------------------------------ */
/*
 * ddp_unpack -- copy the reduced bucket back into per-parameter gradients.
 *
 * Defined by: DDP chapter 17.5 and 17.12 (without gradient_as_bucket_view the
 * reduced bucket is copied back to each .grad; with it .grad is a view of the
 * bucket and nothing moves -- use offset_of/bucket_numel as views instead of
 * calling this); DDP chapter 17.33 and lecture 4.2 (a parameter no rank used
 * keeps its .grad untouched); Megatron page 3 (after reduce_scatter a rank only
 * holds its own shard).
 *
 *   grads_out[w][p][i] = main_grad[w][seg_offset[s] + i]
 * for every segment whose global_used[p] is nonzero (all if NULL).  In
 * DDP_REDUCE_SCATTER mode replica w writes only the elements inside shard w
 * (bucket elements [w*numel/W, (w+1)*numel/W)).
 *
 * Errors: as ddp_pack, plus bad mode / reduce-scatter with numel % W != 0.
 */
ddp_status ddp_unpack(const ddp_bucket_desc* bucket, const float* main_grad, int64_t replica_stride,
                      int32_t W, int32_t mode, void* const* grads_out, int32_t ld,
                      const uint8_t* global_used, void* stream);

/* ------------------------------------------------------------------------ */
/* The local-used bitmap all-reduce (device)                                 */
/* ------------------------------------------------------------------------ */
/*
 * ddp_used_allreduce -- sum the replicas' local-used bitmaps into the global
 * one that decides which gradients unpack may write.
 *
 * Defined by: lecture 4.2 (with find_unused_parameters each rank records in a
 * bitmap which parameters it used and the ranks all-reduce it in one extra
 * collective, kept apart from the gradient buckets because its element type
 * differs; a parameter no rank used keeps its .grad untouched, one that some
 * ranks used is reduced with zeros from the others); the summary of Li et
 * al. 2020, sections 2.2 and 3.2 (one bitmap for the whole model, kept on the
 * host, copied to the device without blocking, then all-reduced).
 *
 *   global_count[p] = number of replicas w with local_used[w * ld + p] != 0
 *   global_used[p]  = global_count[p] > 0 ? 1 : 0
 * for p in [0, nparams).  Any nonzero byte counts as one use.  Integer sums do
 * not depend on the order of the additions, so the ring's order needs no
 * reproduction: every rank of an all-reduce ends with these values, and they
 * are written once.
 *
 *   local_used     DEVICE uint8[W * ld], replica-major (row w = replica w).
 *   ld             row stride in bytes, >= nparams.
 *   W              replicas, 1..64.
 *   global_count   DEVICE int32[nparams], or NULL.
 *   global_used    DEVICE uint8[nparams], or NULL (not both NULL).
 * nparams == 0 launches nothing.  16-byte-aligned local_used with ld a
 * multiple of 16 takes the vector path (16 parameters per thread).
 *
 * Errors: DDP_E_INVAL (W outside [1, 64], nparams < 0, ld < nparams, null
 * local_used, both outputs NULL); DDP_E_CUDA (launch failure).
 */
ddp_status ddp_used_allreduce(const uint8_t* local_used, int32_t ld, int32_t W, int32_t nparams,
                              int32_t* global_count, uint8_t* global_used, void* stream);

/* ------------------------------------------------------------------------ */
/* The PowerSGD communication hook (device)                                  */
/* ------------------------------------------------------------------------ */
/*
 * A PowerSGD state object for one bucket: the hook of DDP chapter 17.27
 * (Vogels et al., PowerSGD), applied in place to the W replicas of the
 * bucket's fp32 main_grad in place of ddp_bucket_allreduce.
 *
 * Per iteration, after start_iter plain all-reduces of the whole bucket:
 *   - every 1-D tensor (seg_rows == 0) gets the ring mean of the concatenation
 *     of the bucket's 1-D tensors (same arithmetic as ddp_bucket_allreduce);
 *   - every tensor with seg_rows = M > 0, viewed as M x N (N = numel / M, the
 *     tensor's shape[0] x the rest), rank R' = min(rank, M, N):
 *       M_w = G_w + E_w              (error feedback; E_w = 0 without it)
 *       P   = sum_w M_w Q            (Q: N x R', the warm-started state)
 *       P   = P R^-1, R the Cholesky factor of P^T P (the orthonormal
 *             basis with a positive-diagonal triangle; a column with no
 *             positive pivot becomes 0)
 *       Q   = (sum_w M_w^T P) / W    (kept as the next iteration's Q)
 *       every replica's tensor = P Q^T;  E_w = M_w - P Q^T
 * The bucket's padding is left alone once compression starts.  Sums over
 * replicas are taken in replica order; P and Q products accumulate in fp32
 * with fused multiply-adds (P^T P as compensated float pairs, its Cholesky
 * factor in fp64), so
 * results match an exact evaluation to within rounding, not bit for bit.
 *
 * Memory (all the caller's; the library allocates none):
 *   workspace  DEVICE, ddp_powersgd_sizes bytes, 256-byte aligned: tile
 *              tables (written by ddp_powersgd_bind) and the scratch: P, the
 *              column splits' partial sums of P, the partial sums of Q and
 *              completion counters (all rewritten by every reduce).
 *   q_state    DEVICE fp32, q_elems: every matrix's Q as N rows of rank_pad
 *              floats (ddp_powersgd_matrix gives the offset); columns past
 *              the effective rank must be 0.  ddp_powersgd_set_q writes one
 *              matrix's initial Q (the hook's random draw is the caller's).
 *   error      DEVICE fp32, W replicas of the bucket layout with stride
 *              error_stride >= bucket_numel; must start at 0; only the
 *              matrices' elements are used.  NULL without error feedback.
 */
typedef struct ddp_powersgd ddp_powersgd;

/*
 * ddp_powersgd_create -- plan the hook for one bucket (HOST only).
 *   W                 replicas, 1..64.
 *   rank              1..8 (padded internally to 1, 2, 4 or 8).
 *   nseg              tensors in the bucket.
 *   seg_offset, seg_numel  HOST int64[nseg]: element offset and size of each
 *                     tensor in the bucket (as from ddp_assign_buckets).
 *   seg_rows          HOST int64[nseg]: the matrix view's rows (shape[0]) of a
 *                     tensor of two or more dimensions, 0 for a 1-D tensor.
 *   bucket_numel      elements of the bucket, padding included.
 *   error_feedback    0/1.   start_iter  plain all-reduce iterations first.
 * Errors: DDP_E_INVAL (ranges; a segment outside the bucket; numel not a
 * multiple of rows; N x rank_pad above 2^30).
 */
ddp_status ddp_powersgd_create(int32_t W, int32_t rank, int32_t nseg, const int64_t* seg_offset,
                               const int64_t* seg_numel, const int64_t* seg_rows, int64_t bucket_numel,
                               int32_t error_feedback, int32_t start_iter, ddp_powersgd** out);

/* Sizes of the caller's buffers (any output may be NULL); nmatrices = tensors compressed. */
ddp_status ddp_powersgd_sizes(const ddp_powersgd* h, int64_t* workspace_bytes, int64_t* q_elems,
                              int32_t* nmatrices);

/* Layout of segment seg's Q inside q_state.  DDP_E_INVAL for a 1-D segment. */
ddp_status ddp_powersgd_matrix(const ddp_powersgd* h, int32_t seg, int64_t* q_offset, int32_t* rows,
                               int32_t* cols, int32_t* rank_eff, int32_t* rank_pad);

/*
 * ddp_powersgd_bind -- attach the caller's buffers and copy the tile tables
 * into the workspace on `stream` (waits for the copy).  The buffers must stay
 * valid while reductions use them.
 * Errors: DDP_E_INVAL (workspace too small or unaligned, q_state NULL or not
 * 16-byte aligned, error buffer missing with error feedback); DDP_E_CUDA.
 */
ddp_status ddp_powersgd_bind(ddp_powersgd* h, void* workspace, int64_t workspace_bytes, float* q_state,
                             float* error, int64_t error_stride, void* stream);

/*
 * ddp_powersgd_set_q -- write segment seg's initial Q from HOST q[N x R']
 * (row-major), zeroing the padding columns; waits for the copy on `stream`.
 * Errors: DDP_E_INVAL (not a matrix segment, q NULL); DDP_E_STATE (not bound).
 */
ddp_status ddp_powersgd_set_q(ddp_powersgd* h, int32_t seg, const float* q, void* stream);

/*
 * ddp_powersgd_reduce -- one iteration of the hook on the bucket's W replicas:
 * main_grad (DEVICE) is replica 0's bucket, replica w starts replica_stride
 * elements later.  Asynchronous on `stream`; advances the iteration count.
 * Two reductions with the same state must not overlap.
 * Errors: DDP_E_INVAL (NULL main_grad, stride < bucket_numel); DDP_E_STATE
 * (compressing before ddp_powersgd_bind); DDP_E_CUDA.
 */
ddp_status ddp_powersgd_reduce(ddp_powersgd* h, float* main_grad, int64_t replica_stride, void* stream);

/*
 * ddp_powersgd_reduce_static -- ddp_powersgd_reduce, allocating nothing and
 * using no caller scratch: the kernels' scratch (the summed P, the partial
 * sums of P and of Q and the Q pass's completion counters) lives in a fixed device array of DDP_POWERSGD_STATIC_SCRATCH_BYTES
 * (8 MiB) inside the library.  The pages have no counterpart: this is an
 * entry point of this library for callers that want no scratch allocation at
 * all.  The workspace bound by ddp_powersgd_bind still supplies the tile
 * tables; its scratch part is not used.
 *
 * Set-up: the first compressing call on each device, with that device
 * current, looks up the array's address (cudaGetSymbolAddress) and keeps it
 * for the life of the process; make that first call before any stream
 * capture.  cudaDeviceReset on a device makes the kept address stale: do not
 * call this entry point on that device again in the same process.  Nothing of the scratch is read before the
 * same call writes it (the first kernel zeroes the counters), so nothing needs
 * clearing beforehand.  Calls that overlap in time
 * (any state objects, any streams, on one device) share the array and race:
 * serialise them.  Results are identical to ddp_powersgd_reduce's.
 * Errors: as ddp_powersgd_reduce; DDP_E_CAPACITY when a compressing call's
 * scratch (ddp_powersgd_sizes minus the tables) exceeds the array (the plain
 * warm-up iterations use no scratch and are never refused for size), checked
 * before anything is launched; DDP_E_CUDA if the address lookup fails.
 */
#define DDP_POWERSGD_STATIC_SCRATCH_BYTES (8ll << 20)
ddp_status ddp_powersgd_reduce_static(ddp_powersgd* h, float* main_grad, int64_t replica_stride, void* stream);

/* Iterations done so far (plain and compressed). */
ddp_status ddp_powersgd_iter(const ddp_powersgd* h, int32_t* iter);

void ddp_powersgd_destroy(ddp_powersgd* h);

/* ------------------------------------------------------------------------ */
/* Steps 2-4 fused (device)                                                  */
/* ------------------------------------------------------------------------ */
/*
 * ddp_fused_bucket -- pack, reduce and unpack one bucket in a single pass: the
 * gradients are read once, summed in ring order with the 1/W scale, and the
 * result is written where the staged calls would put it.
 *
 * Results are bit-identical to ddp_pack (same accumulate, used) followed by
 * ddp_bucket_allreduce (same mode) and, when grads_out != NULL, ddp_unpack,
 * with one difference in reduce-scatter mode: main_grad is written only inside
 * shard w of replica w (the staged ddp_pack would also have written the packed
 * local gradients elsewhere).
 *
 *   main_grad     DEVICE fp32 bucket replicas; may be NULL when accumulate == 0
 *                 and grads_out != NULL (the bucket then never materialises).
 *   grads_out     DEVICE pointer table or NULL (gradient_as_bucket_view: the
 *                 caller reads main_grad through views).  May alias grads
 *                 when the gradients are fp32 (reduce in place).
 *
 * Errors: DDP_E_INVAL as the staged calls, and if both main_grad and grads_out
 * are NULL, or accumulate != 0 with main_grad NULL; DDP_E_CUDA.
 */
ddp_status ddp_fused_bucket(const ddp_bucket_desc* bucket, const void* const* grads,
                            const uint8_t* used, int32_t ld, int32_t W, int32_t mode,
                            int32_t accumulate, float* main_grad, int64_t replica_stride,
                            void* const* grads_out, const uint8_t* global_used, void* stream);

/*
 * ddp_fused_bucket_group -- ddp_fused_bucket over several buckets in as few
 * kernel launches as possible (one per run of up to 32 buckets of one dtype):
 * the collectives of a bucket group coalesced into one call (Megatron page,
 * section 3, _coalescing_manager).  Results are those of calling
 * ddp_fused_bucket on each bucket in turn.
 *
 *   buckets[nbuckets]       HOST descriptors.
 *   bucket_start[nbuckets]  HOST: bucket b occupies main_grad + bucket_start[b]
 *                           in every replica (ignored when main_grad is NULL).
 *   other arguments         as ddp_fused_bucket; main_grad is the start of the
 *                           per-replica buffer holding all the buckets.
 * Errors: as ddp_fused_bucket, for any bucket; DDP_E_INVAL if a bucket does
 * not fit in replica_stride.  Nothing is launched when a bucket is rejected.
 */
ddp_status ddp_fused_bucket_group(const ddp_bucket_desc* buckets, const int64_t* bucket_start, int32_t nbuckets,
                                  const void* const* grads, const uint8_t* used, int32_t ld, int32_t W,
                                  int32_t mode, int32_t accumulate, float* main_grad, int64_t replica_stride,
                                  void* const* grads_out, const uint8_t* global_used, void* stream);

/*
 * ddp_fused_bucket_group_wire -- ddp_fused_bucket_group with the reduction
 * through a compression hook (wire_dtype as for ddp_bucket_allreduce_wire):
 * the packed value of each replica goes through wire(wire(.) / W) and the ring
 * sums in the wire type.  Errors: as ddp_fused_bucket_group; DDP_E_INVAL for an
 * unknown wire_dtype.
 */
ddp_status ddp_fused_bucket_group_wire(const ddp_bucket_desc* buckets, const int64_t* bucket_start,
                                       int32_t nbuckets, const void* const* grads, const uint8_t* used, int32_t ld,
                                       int32_t W, int32_t mode, int32_t accumulate, float* main_grad,
                                       int64_t replica_stride, void* const* grads_out, const uint8_t* global_used,
                                       int32_t wire_dtype, void* stream);

/* ------------------------------------------------------------------------ */
/* Step 5: the reducer -- in-order bucket issue on a side stream             */
/* ------------------------------------------------------------------------ */
/*
 * Models DDP's Reducer (DDP chapter 17.2, 17.12, 17.16, 17.41; lecture 2.3;
 * the summary of Li et al. section 2.2.3; Megatron page 2): each bucket has a
 * pending count; marking a parameter ready decrements it; a bucket whose count
 * reaches 0 is ready, and buckets are issued strictly in issue order starting
 * from the next unissued one (bucket k+1 waits for bucket k even if it filled
 * first).  Each issue makes the side stream wait for the streams that produced
 * the bucket's gradients (CUDA events) and launches that bucket's reduction on
 * the side stream; finalize makes the consumer stream wait for all of them.
 */
typedef struct ddp_reducer ddp_reducer;

enum {
    DDP_R_FUSED = 1,     /* issue ddp_fused_bucket per bucket (else pack + allreduce [+ unpack]) */
    DDP_R_COPY_BACK = 2, /* write reduced gradients to grads_out (else main_grad views only) */
    DDP_R_TIMING = 4,    /* record CUDA events around each bucket's kernels (ddp_reducer_bucket_ms) */
    DDP_R_DRY_RUN = 8,   /* schedule only: no CUDA call at all; issues are logged, not launched */
    DDP_R_COALESCE = 16, /* buckets that become issuable together go out in one launch
                            (ddp_fused_bucket_group); needs DDP_R_FUSED */
    DDP_R_WIRE_BF16 = 32, /* reduce through the bf16 compression hook (ddp_bucket_allreduce_wire) */
    DDP_R_WIRE_F16 = 64,  /* reduce through the fp16 compression hook */
    DDP_R_BUCKET_DONE = 128 /* record an event after each bucket's reduction (ddp_reducer_wait_bucket) */
};

/*
 * ddp_reducer_create
 *   nparams, nbuckets     sizes of the plan from ddp_assign_buckets.
 *   bucket_of             HOST int32[nparams].
 *   bucket_order          HOST int32[nbuckets] (issue order).
 *   buckets               HOST ddp_bucket_desc[nbuckets] (device tables inside),
 *                         copied into the reducer.
 *   bucket_start          HOST int64[nbuckets]: element offset of bucket b inside
 *                         each main_grad replica (main_grad + w*replica_stride +
 *                         bucket_start[b] is replica w's copy of bucket b).
 *   W, mode, flags        replicas (1..64), DDP_ALLREDUCE/DDP_REDUCE_SCATTER, DDP_R_*.
 *   grads, used, ld       DEVICE pointer table / flags as for ddp_pack.
 *   main_grad, replica_stride   DEVICE fp32 buffer holding every bucket per replica.
 *   grads_out, global_used      as for ddp_unpack (used with DDP_R_COPY_BACK).
 *   side_stream           the stream the reductions run on.
 * The pointers are kept and used by later calls; they must stay valid until
 * ddp_reducer_destroy.  With DDP_R_DRY_RUN the device pointers may be NULL.
 * Errors: DDP_E_INVAL; DDP_E_CUDA (event creation).
 */
ddp_status ddp_reducer_create(int32_t nparams, int32_t nbuckets, const int32_t* bucket_of,
                              const int32_t* bucket_order, const ddp_bucket_desc* buckets,
                              const int64_t* bucket_start, int32_t W, int32_t mode, int32_t flags,
                              const void* const* grads, const uint8_t* used, int32_t ld,
                              float* main_grad, int64_t replica_stride, void* const* grads_out,
                              const uint8_t* global_used, void* side_stream, ddp_reducer** out);

/*
 * ddp_reducer_prepare -- start an iteration (prepare_for_backward, DDP chapter
 * 17.16): reset every pending count, the ready marks and the issue position.
 * accumulate != 0 means main_grad already holds gradients accumulated locally
 * during no_sync micro-steps and this backward adds to them (lecture 4.1).
 * Errors: DDP_E_INCOMPLETE if the previous iteration marked some parameters
 * but never finished (the DDP chapter 17.6 error "Expected to have finished
 * reduction in the prior iteration"); the message lists the parameter indices
 * that did not receive a gradient.  The reducer is reset anyway.
 * With find_unused on (ddp_reducer_find_unused) it also uploads the bitmap,
 * launches the bitmap all-reduce on the side stream and marks ready the
 * parameters no replica used; buckets made only of those are issued here.
 */
ddp_status ddp_reducer_prepare(ddp_reducer* r, int32_t accumulate);

/*
 * ddp_reducer_find_unused -- turn on find_unused_parameters (lecture 4.2; the
 * summary of Li et al. 2020, sections 2.2 and 3.2; DDP chapter 17.33).
 *
 * From then on the reducer keeps a HOST bitmap, W rows of nparams bytes (row
 * w = replica w's local use, all 1 at first), set by ddp_reducer_set_local_used.
 * Every ddp_reducer_prepare then, on the side stream:
 *   1. copies the host bitmap into local_used (rows of stride ld);
 *   2. runs ddp_used_allreduce(local_used, ld, W, nparams, global_count,
 *      global_used) -- the extra all-reduce;
 * and on the host marks ready, without a producer stream, every parameter
 * that no replica used (the backward will not produce it), so that its
 * bucket can complete.  Unpack and copy-back then skip the globally unused
 * parameters (they read global_used), and a replica that did not use a
 * parameter contributes zero to its bucket: the packs read local_used as
 * their `used` flags when ddp_reducer_create was given none.
 *
 *   local_used    DEVICE uint8[W * ld] (ld from ddp_reducer_create, >= nparams),
 *                 written by the reducer.
 *   global_used   DEVICE uint8[nparams], written by the reducer.
 *   global_count  DEVICE int32[nparams] or NULL, written by the reducer.
 * With DDP_R_DRY_RUN all three may be NULL (the host marking still happens).
 * Call outside an iteration, once per reducer.  The host bitmap is pinned
 * host memory owned by the reducer.
 * Errors: DDP_E_INVAL (null reducer or pointers, ld < nparams, or the reducer
 * was created with its own global_used); DDP_E_STATE (inside an iteration, or
 * already on); DDP_E_CUDA (host allocation or event creation).
 */
ddp_status ddp_reducer_find_unused(ddp_reducer* r, uint8_t* local_used, uint8_t* global_used,
                                   int32_t* global_count);

/*
 * ddp_reducer_set_local_used -- this iteration's local-used bitmap: HOST
 * flags[w * ld + p] nonzero if replica w used parameter p (for a no_sync
 * window, whether it used p in any of the window's micro-steps).  Copied into
 * the reducer's host bitmap; if the copy to the device issued by the last
 * prepare has not finished, waits for it first.  Call before the prepare of
 * the iteration it describes.
 * Errors: DDP_E_INVAL (null reducer or flags, ld < nparams); DDP_E_STATE
 * (find_unused is off, or inside an iteration); DDP_E_CUDA.
 */
ddp_status ddp_reducer_set_local_used(ddp_reducer* r, const uint8_t* flags, int32_t ld);

/*
 * ddp_reducer_register_powersgd -- register the PowerSGD hook (DDP chapter
 * 17.27, register_comm_hook) for bucket `bucket`: from then on its issue is
 * pack, ddp_powersgd_reduce on the side stream, and the copy-back when
 * DDP_R_COPY_BACK is set (never coalesced with other buckets).  NULL removes
 * the hook.  The state object stays the caller's and must be bound.
 * Errors: DDP_E_INVAL (bucket out of range, a reduce_scatter reducer, no
 * main_grad, a state planned for another W); DDP_E_STATE (inside an iteration).
 */
ddp_status ddp_reducer_register_powersgd(ddp_reducer* r, int32_t bucket, ddp_powersgd* h);

/*
 * ddp_reducer_mark_ready -- the autograd hook of parameter `param` fired: its
 * gradient has been (or is being) produced on `producer_stream`
 * (mark_variable_ready, DDP chapter 17.12; lecture 2.3).
 * The producer is given as a stream, not as an event the caller recorded:
 * when the bucket's last parameter is marked, the reducer records one event of
 * its own on each distinct producer stream of the bucket, at that moment, and
 * the bucket's issue waits for those.  A caller-recorded event per parameter
 * would cost an event record per gradient (161 for ResNet-50) where this costs
 * one per bucket and stream, and would leave the caller to keep every event
 * alive until the side stream has waited on it.  A caller that holds an event
 * instead can make a stream of its own wait on it and pass that stream.
 * Errors: DDP_E_INVAL (param out of range); DDP_E_STATE if param was already
 * marked in this iteration (DDP chapter 17.16: "Expected to mark a variable
 * ready only once") or prepare was not called; DDP_E_CUDA (event/launch).
 */
ddp_status ddp_reducer_mark_ready(ddp_reducer* r, int32_t param, void* producer_stream);

/*
 * ddp_reducer_mark_ready_many -- ddp_reducer_mark_ready for params[0..n-1], in
 * that order, all produced on producer_stream (one backward layer's weight and
 * bias, or a whole backward pass, in one call).  HOST params[n].  The buckets
 * the list completes are issued after the whole list is marked, in issue order
 * (with DDP_R_COALESCE, consecutive ones in one launch).  Stops marking at the
 * first failing parameter and returns its status; the earlier ones stay marked
 * and their complete buckets are still issued.
 */
ddp_status ddp_reducer_mark_ready_many(ddp_reducer* r, const int32_t* params, int32_t n, void* producer_stream);

/*
 * ddp_reducer_finalize -- end of backward (finalize_backward, DDP chapter
 * 17.41; Megatron finish_grad_sync): makes consumer_stream (NULL: the legacy
 * default stream) wait for every issued reduction.  With timeout_us > 0 it also waits on the
 * host, polling, until the reductions finish or the deadline passes.
 * Errors: DDP_E_INCOMPLETE if some bucket was never issued (message lists the
 * unmarked parameters); DDP_E_TIMEOUT if the deadline passed (the work stays
 * queued; call again or synchronise); DDP_E_CUDA.
 */
ddp_status ddp_reducer_finalize(ddp_reducer* r, void* consumer_stream, int64_t timeout_us);

/*
 * ddp_reducer_wait_bucket -- make consumer_stream wait for bucket `bucket`'s
 * reduction in this iteration (Megatron page 3: finish_grad_sync per bucket;
 * a consumer such as an optimizer or a copy to the host can start on the
 * early buckets while later ones are still reducing).  Needs DDP_R_BUCKET_DONE.
 * Errors: DDP_E_INVAL (bucket out of range); DDP_E_STATE (flag not set, or
 * the bucket was not issued in this iteration); DDP_E_CUDA.
 */
ddp_status ddp_reducer_wait_bucket(ddp_reducer* r, int32_t bucket, void* consumer_stream);

/* Buckets issued in this iteration, in issue order (HOST out[cap]); *n = count. */
ddp_status ddp_reducer_issue_log(const ddp_reducer* r, int32_t* out, int32_t cap, int32_t* n);

/*
 * ddp_reducer_ready_order -- the order in which the last finalized iteration
 * marked its parameters ready (the gradient-ready order DDP records for the
 * bucket rebuild, DDP chapter 17.13).  HOST out[cap]; *n = nparams marked.
 * Parameters marked by prepare under find_unused come first.
 * Errors: DDP_E_STATE if no iteration was finalized; DDP_E_CAPACITY.
 */
ddp_status ddp_reducer_ready_order(const ddp_reducer* r, int32_t* out, int32_t cap, int32_t* n);

/*
 * Per-bucket GPU time in milliseconds of the last finalized iteration (needs
 * DDP_R_TIMING; waits for those events).  HOST out[cap], indexed by bucket id.
 * Buckets issued together in one coalesced launch each report that launch's time.
 */
ddp_status ddp_reducer_bucket_ms(ddp_reducer* r, float* out, int32_t cap);

void ddp_reducer_destroy(ddp_reducer* r);

/* ------------------------------------------------------------------------ */
/* The bucket plan as an object (host)                                       */
/* ------------------------------------------------------------------------ */
/*
 * A ddp_plan holds step 1's result and everything derived from it that a C
 * caller needs to run the path without re-deriving it: the buckets' places in
 * one fp32 main_grad buffer per replica, the segment tables the kernels read
 * (to be copied to the device by the caller: the library allocates no device
 * memory), the bucket descriptors over those device copies, and the
 * description DDP's logging data reports -- every bucket's bytes, padded
 * elements, dtype, parameters and issue position (bucket_sizes), and the sizes
 * of the buckets a rebuild over an observed gradient-ready order would form
 * (rebuilt_bucket_sizes) ("DDP: ring AllReduce and gradient buckets" 17.13;
 * 17.12: a bucket is a flat buffer with its parameters at fixed offsets;
 * Megatron page 1: the buckets are slices of one contiguous main_grad buffer).
 * A plan is immutable after creation and may be read from several threads.
 */
typedef struct ddp_plan ddp_plan;

typedef struct ddp_plan_info {
    int32_t nparams, nbuckets;
    int32_t order, pad_multiple, grad_reduce_in_fp32, reserved_;
    int64_t cap_bytes, first_cap_bytes;
    int64_t align_elems;     /* every bucket starts on a multiple of this in main_grad */
    int64_t replica_stride;  /* fp32 elements of one main_grad replica (all buckets) */
    int64_t seg_offset_len;  /* entries of the segment-offset table: nparams + nbuckets */
    int64_t seg_param_len;   /* entries of the segment-parameter table: nparams */
} ddp_plan_info;

/*
 * ddp_plan_create -- run ddp_assign_buckets (same arguments and rules; dtypes
 * NULL = every parameter fp32) and lay the buckets out: bucket b occupies
 * elements [bucket_start[b], bucket_start[b] + bucket_numel[b]) of each
 * replica, bucket_start[0] = 0 and every later start the previous bucket's end
 * rounded up to a multiple of align_elems (64 makes every replica of every
 * bucket 256-byte aligned when main_grad is).  HOST in; *out owns host memory
 * only, released by ddp_plan_destroy.
 * Errors: those of ddp_assign_buckets; DDP_E_INVAL (out NULL, align_elems
 * outside [1, 2^20]).
 */
ddp_status ddp_plan_create(const int64_t* numels, const int32_t* dtypes, int32_t nparams, int64_t cap_bytes,
                           int64_t first_cap_bytes, int32_t order, int32_t pad_multiple,
                           int32_t grad_reduce_in_fp32, int64_t align_elems, ddp_plan** out);

/*
 * ddp_plan_describe -- the plan's sizes into *info and, for every output that
 * is not NULL, its tables (HOST, caller-allocated): per bucket (nbuckets
 * entries) bucket_numel (padded), bucket_bytes (unpadded, the logging data's
 * bucket_sizes), bucket_dtype, bucket_order (bucket_order[k] = bucket issued
 * k-th), bucket_start; member_start[nbuckets + 1] with members[nparams]
 * (bucket b's parameters, in layout order, are members[member_start[b]] ..
 * members[member_start[b + 1] - 1]); per parameter bucket_of and offset_of
 * (elements from its bucket's start).  Same values as ddp_assign_buckets.
 * Errors: DDP_E_INVAL (plan NULL).
 */
ddp_status ddp_plan_describe(const ddp_plan* plan, ddp_plan_info* info, int64_t* bucket_numel, int64_t* bucket_bytes,
                             int32_t* bucket_dtype, int32_t* bucket_order, int64_t* bucket_start,
                             int32_t* member_start, int32_t* members, int32_t* bucket_of, int64_t* offset_of);

/*
 * ddp_plan_tables -- the kernels' segment tables, HOST out: seg_offset
 * int64[info.seg_offset_len], seg_param int32[info.seg_param_len].  Bucket by
 * bucket: its parameters' offsets in layout order followed by the end of its
 * last gradient (nseg + 1 entries), and its parameters' indices (nseg).  Copy
 * both to the device and pass the device copies to ddp_plan_bucket_descs.
 * Errors: DDP_E_INVAL (NULL plan or output).
 */
ddp_status ddp_plan_tables(const ddp_plan* plan, int64_t* seg_offset, int32_t* seg_param);

/*
 * ddp_plan_bucket_descs -- the descriptors of every bucket (HOST out
 * ddp_bucket_desc[nbuckets]) pointing into the DEVICE copies of the tables of
 * ddp_plan_tables.  Errors: DDP_E_INVAL (NULL argument).
 */
ddp_status ddp_plan_bucket_descs(const ddp_plan* plan, const int64_t* seg_offset_dev, const int32_t* seg_param_dev,
                                 ddp_bucket_desc* out);

/*
 * ddp_plan_rebuilt -- the buckets a rebuild over `sequence` (HOST
 * int32[nparams], a permutation: the gradient-ready order, e.g. from
 * ddp_reducer_ready_order) would form with the plan's caps and dtypes
 * (ddp_assign_buckets_ordered; DDP chapter 17.13, rebuilt_bucket_sizes):
 * HOST out bucket_bytes and bucket_numel (either may be NULL), max_buckets
 * entries; *nbuckets = their count.
 * Errors: as ddp_assign_buckets_ordered; DDP_E_CAPACITY if more than
 * max_buckets (nparams + 2 always suffices).
 */
ddp_status ddp_plan_rebuilt(const ddp_plan* plan, const int32_t* sequence, int64_t* bucket_bytes,
                            int64_t* bucket_numel, int32_t max_buckets, int32_t* nbuckets);

/*
 * ddp_reducer_create_from_plan -- ddp_reducer_create with the plan's
 * bucket_of, bucket_order, bucket_start and replica_stride; buckets are the
 * descriptors from ddp_plan_bucket_descs.  The plan may be destroyed after
 * the call (the reducer copies what it needs); the device tables may not.
 */
ddp_status ddp_reducer_create_from_plan(const ddp_plan* plan, const ddp_bucket_desc* buckets, int32_t W, int32_t mode,
                                        int32_t flags, const void* const* grads, const uint8_t* used, int32_t ld,
                                        float* main_grad, void* const* grads_out, const uint8_t* global_used,
                                        void* side_stream, ddp_reducer** out);

void ddp_plan_destroy(ddp_plan* plan);

/* ------------------------------------------------------------------------ */
/* Kernel variants and device status                                         */
/* ------------------------------------------------------------------------ */
/*
 * Two implementations compute every data-path call with identical results:
 * the TMA-pipelined streaming kernel (it takes a launch when its shared-memory
 * stage ring fits: 2 <= W <= 16, and a vector-aligned main_grad for the
 * allreduce) and the plain kernel (16-byte loads straight into registers).
 * The streaming kernel splits a launch between its CTAs in one of two ways with
 * identical results: a static split (equal slices), or a static head (5/8 of
 * the elements for the ring reduction, 3/4 for the launches that read
 * gradients) followed by a pool of units (about 64 KB and 128 KB of staged
 * operands; the pool's last stretch, one unit per CTA, in half units where
 * those are whole tiles) that CTAs claim one at a time when their slice is
 * done, so that CTAs on faster SMs take more of the tail.  A launch with a pool uses one of 64
 * counter slots in the library's own device memory and waits, on its stream,
 * for the previous launch that used the same slot (an event the library
 * records); launches made during stream capture keep the static split.
 *   DDP_KERNEL_AUTO   (default) a launch of a single bucket with numel x W <=
 *                     2^21 elements takes the plain kernel, which finishes such
 *                     small launches first; the rest take the streaming kernel,
 *                     with a pool when numel x W >= 2^23.
 *   DDP_KERNEL_STREAM every launch the streaming kernel can take uses it, with
 *                     the static split; the rest use the plain kernel.
 *   DDP_KERNEL_STREAM_DYNAMIC  as DDP_KERNEL_STREAM, with a pool on every
 *                     streaming launch outside stream capture.
 *   DDP_KERNEL_PLAIN  every call uses the plain kernel.
 * The choice is process-wide and applies to calls made after it.
 * Errors: DDP_E_INVAL for an unknown variant.
 */
enum { DDP_KERNEL_AUTO = 0, DDP_KERNEL_PLAIN = 1, DDP_KERNEL_STREAM = 2, DDP_KERNEL_STREAM_DYNAMIC = 3 };
ddp_status ddp_set_kernel_variant(int32_t variant);

/*
 * ddp_device_status -- the library's device status word: 0 normally; bit 0
 * set if a streaming kernel gave up on an mbarrier wait (about 2 s), recorded
 * the failure and returned early, leaving its outputs incomplete.  Reads the
 * word on `stream` (synchronising that stream); reset != 0 clears it.
 * HOST out: *status.  Errors: DDP_E_INVAL (NULL status); DDP_E_CUDA.
 */
ddp_status ddp_device_status(void* stream, int32_t* status, int32_t reset);

/*
 * ddp_wait_selftest -- exercise the streaming kernels' failure path without a
 * fault: one block waits, bounded by limit_ns (1 us .. 2 s), on an mbarrier
 * that completes only if arrive != 0.  When nothing arrives the wait gives up,
 * bit 0 of the device status word is set exactly as a streaming kernel sets it,
 * and the block returns; the context stays usable.  Asynchronous on `stream`;
 * read the result with ddp_device_status.  The pages have no counterpart: this
 * is the library's own check of its failure detection.
 * Errors: DDP_E_INVAL (limit out of range); DDP_E_CUDA.
 */
ddp_status ddp_wait_selftest(int32_t arrive, int64_t limit_ns, void* stream);

/*
 * ddp_copy_rows -- copy `rows` rows of `row_bytes` bytes each, row i from
 * src + i * src_pitch to dst + i * dst_pitch, as one copy command on `stream`
 * (cudaMemcpy2DAsync, direction inferred from the pointers; host memory must be
 * pinned for the copy to be asynchronous).  A host-buffer front end moves a
 * bucket's W replica slices, which are one pitch apart on both sides, with one
 * call instead of W.  The pages have no counterpart: this is plumbing for callers
 * whose gradients live in host memory.
 * Errors: DDP_E_INVAL (negative sizes, a pitch below row_bytes, a NULL pointer
 * with rows and row_bytes > 0); DDP_E_CUDA (the copy was refused).
 */
ddp_status ddp_copy_rows(void* dst, int64_t dst_pitch, const void* src, int64_t src_pitch, int64_t row_bytes,
                         int64_t rows, void* stream);

/*
 * The host-buffer front end of a reducer: per step, every replica's gradients
 * from pinned host memory to the device, the reducer's iteration (all
 * parameters marked ready as their bucket's copies land), and each reduced
 * bucket back to pinned host memory as soon as that bucket is done ("Megatron
 * DDP: contiguous buffer and overlap" section 3: a consumer may start on a
 * bucket once its reduction finishes).  The three run as a pipeline over the
 * buckets in issue order on two copy streams of the front end's own, and
 * consecutive steps overlap bucket by bucket: step k + 1's copies into bucket
 * b's gradients wait for step k's reduction of b, and its reduction of b waits
 * for step k's copy of b to the host.  The pages have no counterpart (their
 * gradients are on the device already); this is the library's entry for
 * callers whose data lives in host memory.
 *
 * ddp_host_front_create
 *   r            a reducer built with DDP_R_BUCKET_DONE and a main_grad, not a
 *                dry run.  The front end must be destroyed before it.
 *   dev_in       DEVICE: the gradient buffer the reducer's pointer table points
 *                into, W rows `dev_pitch` bytes apart; parameter p occupies
 *                elements [param_offset[p], param_offset[p + 1]) of each row.
 *   param_offset HOST int64[nparams + 1], non-decreasing, param_offset[0] = 0.
 *   elem_bytes   the gradients' element size (4: fp32; 2: bf16 or fp16).
 *   Errors: DDP_E_INVAL (a NULL or inconsistent argument, a dry-run reducer,
 *   no DDP_R_BUCKET_DONE, no main_grad); DDP_E_CUDA (streams or events).
 *
 * ddp_host_front_step -- one step, enqueued (nothing waits on the host).
 *   host_in      HOST, pinned: W rows `host_pitch` bytes apart in dev_in's layout.
 *   host_out     HOST, pinned fp32, W x replica_stride elements in main_grad's
 *                layout.  Allreduce: every bucket's elements are written (the
 *                alignment gaps between buckets are not); reduce_scatter: row w
 *                receives only shard w of each bucket.
 *   stream       waits for the whole step (the last copy to the host); the
 *                host buffers must stay untouched until then.  The first step
 *                also waits for what `stream` holds when it is called.
 *   Errors: DDP_E_INVAL (a NULL buffer, a pitch below a row); the reducer's
 *   errors (a parameter marked twice, DDP_E_STATE); DDP_E_CUDA.
 */
typedef struct ddp_host_front ddp_host_front;
ddp_status ddp_host_front_create(ddp_reducer* r, void* dev_in, int64_t dev_pitch, const int64_t* param_offset,
                                 int32_t elem_bytes, ddp_host_front** out);
ddp_status ddp_host_front_step(ddp_host_front* h, const void* host_in, int64_t host_pitch, float* host_out,
                               void* stream);
void ddp_host_front_destroy(ddp_host_front* h);

/* ------------------------------------------------------------------------ */
/* Errors and version                                                        */
/* ------------------------------------------------------------------------ */
const char* ddp_status_str(ddp_status s);
/* Message of the calling thread's last failed call ("" if none). */
const char* ddp_last_error_message(void);
/* Library ABI version (major * 10000 + minor * 100 + patch). */
int32_t ddp_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DDP_BUCKET_H */
