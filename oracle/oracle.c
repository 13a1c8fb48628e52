/*
 * oracle.c -- plain, slow CPU statement of the DDP gradient-bucket path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library imports, links or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header or constant with the CUDA library.
 *
 * Build: cc -std=c99 -O2 -ffp-contract=off -fPIC -shared  (no FMA contraction,
 * so every fp32 multiply and add rounds once, on x86-64 and on aarch64 alike).
 *
 * Sources (page title, section):
 *   [P1] "DDP: ring AllReduce and gradient buckets" (PyTorch internals book,
 *        chapter 17): §17.2 bucket cap / 1 MiB first bucket / close-on-reach,
 *        §17.4 ring AllReduce, §17.9 pre-scaling by 1/world_size,
 *        §17.12 mark_variable_ready copy into the bucket,
 *        §17.13 reversed bucket order and the rebuilt/initial byte lists,
 *        §17.33 unused parameters (zero segment, untouched .grad).
 *   [P2] "Lecture 15: PyTorch DDP" (CMU 11-868 notes): §2.2 buckets filled in
 *        reverse parameter order and closed once the cap is reached,
 *        §4.1 no_sync accumulation, §4.2 unused parameters, exercise 3.
 *   [P3] "Megatron DDP: contiguous buffer and overlap": §1 contiguous fp32
 *        main_grad buffer and max(40MB, 1MB x DP) buckets, §3 start_grad_sync
 *        (all_reduce or reduce_scatter with rank r keeping shard r, scaling by
 *        1/DP before the collective).
 *   [P4] "DDP: PyTorch Distributed-Experiences on Accelerating Data Parallel
 *        Training" (a summary of the DDP paper): §2.2 unused parameters and
 *        the global bitmap, §3.2 the bitmap kept on the host, copied to the
 *        device and all-reduced once per iteration.
 *
 * Readings taken where the pages leave a step open (each is a parameter or a
 * documented convention):
 *   - caps are bytes; bucket bytes count fp32 when grad_reduce_in_fp32 is set
 *     (Megatron's main_grad), else the gradient's own element size;
 *   - one open bucket per dtype with its own cap sequence; open buckets are
 *     flushed at the end in order of the dtype's first appearance;
 *   - Megatron layout: forward parameter order, bucket 0 holds p0, one cap for
 *     every bucket, numel padded to a multiple of pad_multiple, issue order
 *     from the last bucket to the first;
 *   - ring chunk c = [c*ceil(n/W), min((c+1)*ceil(n/W), n)); at step s rank r
 *     sends chunk (r-s-1) mod W to rank r+1, which adds received + local;
 *     rank r ends the reduce-scatter holding chunk r (Megatron's shard r);
 *   - each rank's contribution is multiplied by fp32(1/W) before the ring;
 *   - reduce_scatter writes only shard r of rank r; the rest is unchanged;
 *   - a compressed ring (the bf16/fp16 compression hook of [P1 §17.9, §17.20])
 *     rounds every message and every partial sum to the wire type, to nearest
 *     with ties to even, and divides by W in the wire type before the ring.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORDER_REVERSE 0          /* rebuilt buckets: reversed parameters, first cap on bucket 0 */
#define ORDER_FWD_THEN_REVERSE 1 /* initial buckets: forward parameters, then the list reversed */
#define ORDER_MEGATRON 2         /* contiguous forward layout, issued last to first */

#define MODE_ALLREDUCE 0
#define MODE_REDUCE_SCATTER 1

#define DT_F32 0
#define DT_BF16 1
#define DT_F16 2

static int64_t dtype_size(int32_t dt) { return dt == DT_F32 ? 4 : 2; }

/* bf16 -> fp32 is exact: the bf16 bits are the upper half of the fp32 bits. */
static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* IEEE binary16 -> fp32 (exact), written out from the format definition. */
static float f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h >> 15) << 31;
    uint32_t ex = (h >> 10) & 0x1f, man = h & 0x3ff, u;
    if (ex == 0x1f) {
        u = sign | 0x7f800000u | (man << 13);
    } else if (ex == 0) {
        if (man == 0) {
            u = sign;
        } else { /* subnormal: renormalise */
            int e = -1;
            do { man <<= 1; e++; } while (!(man & 0x400));
            u = sign | ((uint32_t)(127 - 15 - e) << 23) | ((man & 0x3ff) << 13);
        }
    } else {
        u = sign | ((ex + 112) << 23) | (man << 13);
    }
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static float load_as_f32(const void* p, int32_t dt, int64_t i)
{
    if (dt == DT_F32) return ((const float*)p)[i];
    if (dt == DT_BF16) return bf16_to_f32(((const uint16_t*)p)[i]);
    return f16_to_f32(((const uint16_t*)p)[i]);
}

/* ------------------------------------------------------------------------ */
/* 1. bucket assignment                                                     */
/* ------------------------------------------------------------------------ */
/*
 * Walk the parameters in iteration order and append each one to the open
 * bucket of its dtype; after appending, close that bucket as soon as its bytes
 * reach the current cap (so a bucket may overshoot).  The first bucket closed
 * in a dtype group uses first_cap_bytes, every later one cap_bytes [P1 §17.2,
 * §17.13; P2 §2.2 and exercise 3].  Megatron uses cap_bytes throughout [P3 §1].
 *
 * Outputs (caller-allocated):
 *   bucket_of[p], offset_of[p] (elements from the bucket start),
 *   bucket_numel[b] (padded), bucket_bytes[b] (unpadded, counted as above),
 *   bucket_dtype[b], bucket_order[b] (issue order: position k -> bucket id),
 *   members[nparams]: the parameters of bucket 0 in layout order, then bucket 1's, ...
 * Returns 0, or -1 on bad arguments, -2 if more than max_buckets are needed.
 */
static int assign_impl(const int64_t* numels, const int32_t* dtypes, int32_t nparams,
                       int64_t cap_bytes, int64_t first_cap_bytes, int32_t order, const int32_t* given,
                       int32_t pad_multiple, int32_t grad_reduce_in_fp32,
                       int32_t* bucket_of, int64_t* offset_of,
                       int64_t* bucket_numel, int64_t* bucket_bytes, int32_t* bucket_dtype,
                       int32_t* bucket_order, int32_t* members_out, int32_t max_buckets,
                       int32_t* nbuckets);

int oracle_assign(const int64_t* numels, const int32_t* dtypes, int32_t nparams,
                  int64_t cap_bytes, int64_t first_cap_bytes, int32_t order,
                  int32_t pad_multiple, int32_t grad_reduce_in_fp32,
                  int32_t* bucket_of, int64_t* offset_of,
                  int64_t* bucket_numel, int64_t* bucket_bytes, int32_t* bucket_dtype,
                  int32_t* bucket_order, int32_t* members_out, int32_t max_buckets,
                  int32_t* nbuckets)
{
    if (order < ORDER_REVERSE || order > ORDER_MEGATRON) return -1;
    return assign_impl(numels, dtypes, nparams, cap_bytes, first_cap_bytes, order, NULL, pad_multiple,
                       grad_reduce_in_fp32, bucket_of, offset_of, bucket_numel, bucket_bytes, bucket_dtype,
                       bucket_order, members_out, max_buckets, nbuckets);
}

/*
 * Rebuilt buckets [P1 §17.13]: the order in which the first backward produced
 * the gradients is recorded, and the next forward re-buckets the parameters in
 * that order -- the earliest gradients into bucket 0 under the 1 MiB first cap,
 * the rest under bucket_cap_mb -- issued 0, 1, 2, ...  `sequence` is that
 * recorded order (a permutation of 0..nparams-1).
 */
int oracle_assign_sequence(const int64_t* numels, const int32_t* dtypes, int32_t nparams, const int32_t* sequence,
                           int64_t cap_bytes, int64_t first_cap_bytes, int32_t pad_multiple,
                           int32_t grad_reduce_in_fp32, int32_t* bucket_of, int64_t* offset_of,
                           int64_t* bucket_numel, int64_t* bucket_bytes, int32_t* bucket_dtype,
                           int32_t* bucket_order, int32_t* members_out, int32_t max_buckets, int32_t* nbuckets)
{
    if (nparams < 0 || (nparams > 0 && !sequence)) return -1;
    /* the sequence must name every parameter once */
    uint8_t* seen = (uint8_t*)calloc((size_t)(nparams > 0 ? nparams : 1), 1);
    for (int32_t k = 0; k < nparams; k++) {
        if (sequence[k] < 0 || sequence[k] >= nparams || seen[sequence[k]]) { free(seen); return -1; }
        seen[sequence[k]] = 1;
    }
    free(seen);
    return assign_impl(numels, dtypes, nparams, cap_bytes, first_cap_bytes, ORDER_REVERSE, sequence, pad_multiple,
                       grad_reduce_in_fp32, bucket_of, offset_of, bucket_numel, bucket_bytes, bucket_dtype,
                       bucket_order, members_out, max_buckets, nbuckets);
}

static int assign_impl(const int64_t* numels, const int32_t* dtypes, int32_t nparams,
                       int64_t cap_bytes, int64_t first_cap_bytes, int32_t order, const int32_t* given,
                       int32_t pad_multiple, int32_t grad_reduce_in_fp32,
                       int32_t* bucket_of, int64_t* offset_of,
                       int64_t* bucket_numel, int64_t* bucket_bytes, int32_t* bucket_dtype,
                       int32_t* bucket_order, int32_t* members_out, int32_t max_buckets,
                       int32_t* nbuckets)
{
    if (nparams < 0 || cap_bytes <= 0 || first_cap_bytes <= 0 || pad_multiple < 1) return -1;

    /* iteration order: the given sequence, reversed parameters, or forward parameters */
    int32_t* seq = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nparams > 0 ? nparams : 1));
    for (int32_t k = 0; k < nparams; k++)
        seq[k] = given ? given[k] : ((order == ORDER_REVERSE) ? nparams - 1 - k : k);

    /* per-dtype open bucket: its members in append order, bytes, caps used */
    int32_t* open_list[3];
    int32_t open_len[3] = {0, 0, 0};
    int64_t open_bytes[3] = {0, 0, 0};
    int32_t closed_count[3] = {0, 0, 0};
    int32_t first_seen[3] = {-1, -1, -1};
    for (int g = 0; g < 3; g++)
        open_list[g] = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nparams > 0 ? nparams : 1));

    /* buckets in the order they are closed: member lists kept in one array */
    int32_t* members = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nparams > 0 ? nparams : 1));
    int32_t* b_first = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nparams + 3));
    int32_t* b_len = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nparams + 3));
    int32_t* b_dt = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nparams + 3));
    int64_t* b_bytes = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nparams + 3));
    int32_t nb = 0, nmem = 0, rc = 0;

    for (int32_t k = 0; k < nparams; k++) {
        int32_t p = seq[k];
        int32_t g = dtypes[p];
        if (g < 0 || g > 2 || numels[p] < 0) { rc = -1; goto done; }
        if (first_seen[g] < 0) first_seen[g] = k;
        int64_t esize = grad_reduce_in_fp32 ? 4 : dtype_size(g);
        open_list[g][open_len[g]++] = p;
        open_bytes[g] += numels[p] * esize;
        int64_t cap = (order != ORDER_MEGATRON && closed_count[g] == 0) ? first_cap_bytes : cap_bytes;
        if (open_bytes[g] >= cap) {
            b_first[nb] = nmem;
            b_len[nb] = open_len[g];
            b_dt[nb] = g;
            b_bytes[nb] = open_bytes[g];
            for (int32_t j = 0; j < open_len[g]; j++) members[nmem++] = open_list[g][j];
            nb++;
            closed_count[g]++;
            open_len[g] = 0;
            open_bytes[g] = 0;
        }
    }
    /* flush the buckets still open, dtype groups in order of first appearance */
    for (int pass = 0; pass < 3; pass++) {
        int best = -1;
        for (int g = 0; g < 3; g++)
            if (open_len[g] > 0 && (best < 0 || first_seen[g] < first_seen[best])) best = g;
        if (best < 0) break;
        b_first[nb] = nmem;
        b_len[nb] = open_len[best];
        b_dt[nb] = best;
        b_bytes[nb] = open_bytes[best];
        for (int32_t j = 0; j < open_len[best]; j++) members[nmem++] = open_list[best][j];
        nb++;
        open_len[best] = 0;
    }
    if (nb > max_buckets) { rc = -2; goto done; }

    /* the initial assignment hands the bucket list to the reducer reversed [P1 §17.13] */
    int32_t nout = 0;
    for (int32_t b = 0; b < nb; b++) {
        int32_t src = (order == ORDER_FWD_THEN_REVERSE) ? nb - 1 - b : b;
        int64_t off = 0;
        for (int32_t j = 0; j < b_len[src]; j++) {
            int32_t p = members[b_first[src] + j];
            members_out[nout++] = p;
            bucket_of[p] = b;
            offset_of[p] = off;
            off += numels[p];
        }
        int64_t padded = ((off + pad_multiple - 1) / pad_multiple) * pad_multiple;
        bucket_numel[b] = padded;
        bucket_bytes[b] = b_bytes[src];
        bucket_dtype[b] = b_dt[src];
        /* Megatron's layout puts p0 in bucket 0, but backward fills the last bucket first */
        bucket_order[b] = (order == ORDER_MEGATRON) ? nb - 1 - b : b;
    }
    *nbuckets = nb;

done:
    free(seq);
    for (int g = 0; g < 3; g++) free(open_list[g]);
    free(members); free(b_first); free(b_len); free(b_dt); free(b_bytes);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* 2. pack: per-parameter gradients -> the bucket's flat fp32 buffer        */
/* ------------------------------------------------------------------------ */
/*
 * For replica w and every parameter segment s of the bucket [P1 §17.12; P3 §1]:
 *   bucket[w][off_s + i] = (float) grad[w][s][i]                  (copy), or
 *   bucket[w][off_s + i] = bucket[w][off_s + i] + (float) grad     (no_sync accumulation, P2 §4.1)
 * A parameter that replica w did not use (used[w*nseg+s] == 0) has no gradient:
 * its segment is written as 0 when copying and left alone when accumulating
 * [P1 §17.33].  Padding past the last segment is 0 after a copy.
 * grads[w*nseg + s] points at replica w's gradient of segment s (may be NULL if unused).
 */
void oracle_pack(int32_t W, int32_t nseg, const int64_t* seg_offset, const int64_t* seg_numel,
                 const int32_t* seg_dtype, const void* const* grads, const uint8_t* used,
                 int32_t accumulate, float* const* bucket, int64_t bucket_numel)
{
    for (int32_t w = 0; w < W; w++) {
        float* out = bucket[w];
        if (!accumulate)
            for (int64_t e = 0; e < bucket_numel; e++) out[e] = 0.0f;
        for (int32_t s = 0; s < nseg; s++) {
            int is_used = used ? used[(int64_t)w * nseg + s] != 0 : 1;
            if (!is_used) continue; /* copy: stays 0; accumulate: unchanged */
            const void* g = grads[(int64_t)w * nseg + s];
            for (int64_t i = 0; i < seg_numel[s]; i++) {
                float v = load_as_f32(g, seg_dtype[s], i);
                if (accumulate)
                    out[seg_offset[s] + i] = out[seg_offset[s] + i] + v;
                else
                    out[seg_offset[s] + i] = v;
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* 3. ring allreduce / reduce-scatter over W rank buffers                    */
/* ------------------------------------------------------------------------ */
static int64_t chunk_begin(int64_t n, int32_t W, int32_t c)
{
    int64_t len = (n + W - 1) / W;
    int64_t b = (int64_t)c * len;
    return b < n ? b : n;
}

static int64_t chunk_end(int64_t n, int32_t W, int32_t c) { return chunk_begin(n, W, c + 1); }

static int32_t mod(int32_t a, int32_t W) { return ((a % W) + W) % W; }

/*
 * The ring of [P1 §17.4]: W ranks, reduce-scatter in W-1 steps (each rank sends
 * one chunk to the next rank and adds the chunk arriving from the previous
 * one), then, for allreduce, all-gather in W-1 steps (each rank forwards a
 * finished chunk).  Every rank's buffer is first multiplied by fp32(1/W) [P1
 * §17.9, P3 §3].  The ranks' memories and the messages are kept apart: each
 * step first copies every outgoing chunk into a message buffer, then every
 * rank applies what it received.  bytes_sent[r] counts the payload rank r put
 * on the wire.
 *
 * rank_buf[r] is rank r's bucket (n floats), replaced in place:
 *   allreduce       -> every element of every rank holds the mean;
 *   reduce_scatter  -> chunk r of rank r holds the mean of chunk r; the rest of
 *                      rank r's buffer is left as it was (requires n % W == 0).
 * Returns 0, or -1 on bad arguments.
 */
int oracle_ring_allreduce(float* const* rank_buf, int32_t W, int64_t n, int32_t mode,
                          uint64_t* bytes_sent)
{
    if (W < 1 || n < 0) return -1;
    if (mode == MODE_REDUCE_SCATTER && n % W != 0) return -1;
    for (int32_t r = 0; r < W; r++) bytes_sent[r] = 0;
    if (n == 0) return 0;

    const float inv_w = 1.0f / (float)W;
    float** local = (float**)malloc(sizeof(float*) * (size_t)W);
    float** msg = (float**)malloc(sizeof(float*) * (size_t)W);
    int64_t maxchunk = (n + W - 1) / W;
    for (int32_t r = 0; r < W; r++) {
        local[r] = (float*)malloc(sizeof(float) * (size_t)n);
        msg[r] = (float*)malloc(sizeof(float) * (size_t)maxchunk);
        for (int64_t e = 0; e < n; e++) local[r][e] = rank_buf[r][e] * inv_w;
    }

    /* reduce-scatter */
    for (int32_t s = 0; s < W - 1; s++) {
        for (int32_t r = 0; r < W; r++) { /* everybody sends ... */
            int32_t c = mod(r - s - 1, W);
            int64_t b = chunk_begin(n, W, c), e = chunk_end(n, W, c);
            for (int64_t i = b; i < e; i++) msg[r][i - b] = local[r][i];
            bytes_sent[r] += (uint64_t)(e - b) * sizeof(float);
        }
        for (int32_t r = 0; r < W; r++) { /* ... then everybody receives from r-1 */
            int32_t from = mod(r - 1, W);
            int32_t c = mod(from - s - 1, W);
            int64_t b = chunk_begin(n, W, c), e = chunk_end(n, W, c);
            for (int64_t i = b; i < e; i++) local[r][i] = msg[from][i - b] + local[r][i];
        }
    }

    if (mode == MODE_ALLREDUCE) {
        /* all-gather: at step s rank r forwards chunk (r - s) mod W */
        for (int32_t s = 0; s < W - 1; s++) {
            for (int32_t r = 0; r < W; r++) {
                int32_t c = mod(r - s, W);
                int64_t b = chunk_begin(n, W, c), e = chunk_end(n, W, c);
                for (int64_t i = b; i < e; i++) msg[r][i - b] = local[r][i];
                bytes_sent[r] += (uint64_t)(e - b) * sizeof(float);
            }
            for (int32_t r = 0; r < W; r++) {
                int32_t from = mod(r - 1, W);
                int32_t c = mod(from - s, W);
                int64_t b = chunk_begin(n, W, c), e = chunk_end(n, W, c);
                for (int64_t i = b; i < e; i++) local[r][i] = msg[from][i - b];
            }
        }
        for (int32_t r = 0; r < W; r++)
            for (int64_t e = 0; e < n; e++) rank_buf[r][e] = local[r][e];
    } else {
        for (int32_t r = 0; r < W; r++) {
            int64_t b = chunk_begin(n, W, r), e = chunk_end(n, W, r);
            for (int64_t i = b; i < e; i++) rank_buf[r][i] = local[r][i];
        }
    }

    for (int32_t r = 0; r < W; r++) { free(local[r]); free(msg[r]); }
    free(local);
    free(msg);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* 4. unpack: bucket -> per-parameter gradients                              */
/* ------------------------------------------------------------------------ */
/*
 * Copy each segment of the reduced bucket back into replica w's gradient of
 * that parameter [P1 §17.5, §17.12].  Parameters that no replica used keep
 * their gradient untouched [P1 §17.33; P2 §4.2].  In reduce_scatter mode rank w
 * holds only shard w, so only the elements of the segment that fall inside
 * shard w are written.
 */
void oracle_unpack(int32_t W, int32_t nseg, const int64_t* seg_offset, const int64_t* seg_numel,
                   const float* const* bucket, int64_t bucket_numel, int32_t mode,
                   const uint8_t* global_used, float* const* grads_out)
{
    for (int32_t w = 0; w < W; w++) {
        int64_t lo = 0, hi = bucket_numel;
        if (mode == MODE_REDUCE_SCATTER) {
            lo = chunk_begin(bucket_numel, W, w);
            hi = chunk_end(bucket_numel, W, w);
        }
        for (int32_t s = 0; s < nseg; s++) {
            if (global_used && !global_used[s]) continue;
            float* g = grads_out[(int64_t)w * nseg + s];
            for (int64_t i = 0; i < seg_numel[s]; i++) {
                int64_t e = seg_offset[s] + i;
                if (e >= lo && e < hi) g[i] = bucket[w][e];
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* 4b. the local-used bitmap all-reduce                                      */
/* ------------------------------------------------------------------------ */
/*
 * [P2 §4.2], [P4 §2.2, §3.2]: every rank records, one integer per parameter of
 * the whole model, whether it used the parameter this iteration (1) or not
 * (0), and the ranks sum these bitmaps in one extra all-reduce.  A parameter
 * whose sum is 0 was used by no rank: it is globally unused and its .grad is
 * left alone; any other parameter is reduced as usual, the ranks that did not
 * use it contributing zeros.  A sum of integers does not depend on the order
 * of its additions, so the ring's order is not reproduced here; every rank
 * ends with the same sums, written once.
 *
 * local_used[w * nparams + p]: rank w's byte for p, nonzero meaning used.
 * global_count[p]  (may be NULL): number of ranks that used p.
 * global_used[p]   (may be NULL): 1 if at least one rank used p, else 0.
 * Returns 0, or -1 on bad arguments.
 */
int oracle_used_allreduce(int32_t W, int32_t nparams, const uint8_t* local_used, int32_t* global_count,
                          uint8_t* global_used)
{
    if (W < 1 || nparams < 0 || (nparams > 0 && !local_used)) return -1;
    for (int32_t p = 0; p < nparams; p++) {
        int32_t sum = 0;
        for (int32_t w = 0; w < W; w++) {
            int32_t bit = local_used[(int64_t)w * nparams + p] != 0 ? 1 : 0;
            sum += bit;
        }
        if (global_count) global_count[p] = sum;
        if (global_used) global_used[p] = sum > 0 ? 1 : 0;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* 5. compressed ring: the bf16 / fp16 compression hook                      */
/* ------------------------------------------------------------------------ */
/*
 * The hook of [P1 §17.9, §17.20]: the fp32 bucket is converted to the wire
 * type and divided by the world size (in the wire type), the converted tensor
 * is allreduced with a sum (every partial sum is a value of the wire type),
 * and the result is copied back into the fp32 bucket.
 *
 * Rounding to a binary format with p significand bits, exponent range
 * [emin, emax], to nearest with ties to even, written from the format's
 * definition: scale |x| by the quantum of its binade (or of the subnormal
 * range), round the integer to nearest even, and encode; a result at or past
 * 2^(emax+1) becomes infinity.  Inputs are doubles, so every wire value and
 * every exact sum or quotient of two of them used below is rounded once.
 */
static uint16_t encode_rounded(double x, int p, int emin, int emax, int mbits)
{
    const int bias = -emin + 1;
    const uint16_t exp_mask = (uint16_t)(((1u << (15 - mbits)) - 1) << mbits);
    uint16_t sign = signbit(x) ? (uint16_t)(1u << 15) : 0;
    if (isnan(x)) return (uint16_t)(exp_mask | (1u << (mbits - 1)));  /* a quiet NaN */
    double ax = fabs(x);
    uint16_t inf = sign | exp_mask;
    if (isinf(ax)) return inf;
    if (ax == 0.0) return sign;
    int k;
    frexp(ax, &k);            /* ax = m * 2^k with m in [0.5, 1): binade exponent k - 1 */
    int e = k - 1;
    if (e < emin) e = emin;   /* subnormal range: fixed quantum */
    double quantum = ldexp(1.0, e - p + 1);
    double q = rint(ax / quantum);  /* exact scaling by a power of two, then nearest-even */
    if (q >= ldexp(1.0, p)) {       /* rounded up into the next binade */
        q = ldexp(1.0, p - 1);
        e += 1;
    }
    if (e > emax) return inf;
    uint32_t mant = (uint32_t)q;
    if (mant < (1u << (p - 1))) return sign | (uint16_t)mant;  /* subnormal (exponent field 0) */
    uint32_t ef = (uint32_t)(e + bias);
    return sign | (uint16_t)(ef << mbits) | (uint16_t)(mant - (1u << (p - 1)));
}

static double decode_wire(uint16_t h, int p, int emin, int mbits)
{
    const int bias = -emin + 1;
    int sign = h >> 15;
    uint32_t ef = (h >> mbits) & ((1u << (15 - mbits)) - 1);
    uint32_t mant = h & ((1u << mbits) - 1);
    double v;
    if (ef == ((1u << (15 - mbits)) - 1)) v = mant ? NAN : INFINITY;
    else if (ef == 0) v = ldexp((double)mant, emin - p + 1);
    else v = ldexp((double)(mant | (1u << mbits)), (int)ef - bias - p + 1);
    return sign ? -v : v;
}

/* wire formats: bf16 (8-bit significand, exponents -126..127), fp16 (11-bit, -14..15) */
uint16_t oracle_round_wire(double x, int32_t wire)
{
    return wire == DT_BF16 ? encode_rounded(x, 8, -126, 127, 7) : encode_rounded(x, 11, -14, 15, 10);
}

double oracle_wire_value(uint16_t h, int32_t wire)
{
    return wire == DT_BF16 ? decode_wire(h, 8, -126, 7) : decode_wire(h, 11, -14, 10);
}

/*
 * Same ring as oracle_ring_allreduce, over wire-typed messages.  bytes_sent
 * counts 2 bytes per element.  rank_buf is replaced as there (allreduce: all;
 * reduce_scatter: shard r of rank r) with the widened wire result.
 */
int oracle_ring_allreduce_wire(float* const* rank_buf, int32_t W, int64_t n, int32_t mode, int32_t wire,
                               uint64_t* bytes_sent)
{
    if (W < 1 || n < 0 || (wire != DT_BF16 && wire != DT_F16)) return -1;
    if (mode == MODE_REDUCE_SCATTER && n % W != 0) return -1;
    for (int32_t r = 0; r < W; r++) bytes_sent[r] = 0;
    if (n == 0) return 0;

    uint16_t** local = (uint16_t**)malloc(sizeof(uint16_t*) * (size_t)W);
    uint16_t** msg = (uint16_t**)malloc(sizeof(uint16_t*) * (size_t)W);
    int64_t maxchunk = (n + W - 1) / W;
    for (int32_t r = 0; r < W; r++) {
        local[r] = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)n);
        msg[r] = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)maxchunk);
        for (int64_t e = 0; e < n; e++) {
            uint16_t c = oracle_round_wire((double)rank_buf[r][e], wire);              /* compress */
            local[r][e] = oracle_round_wire(oracle_wire_value(c, wire) / (double)W, wire); /* divide by W */
        }
    }
    for (int32_t s = 0; s < W - 1; s++) {
        for (int32_t r = 0; r < W; r++) {
            int32_t c = mod(r - s - 1, W);
            int64_t b = chunk_begin(n, W, c), e = chunk_end(n, W, c);
            for (int64_t i = b; i < e; i++) msg[r][i - b] = local[r][i];
            bytes_sent[r] += (uint64_t)(e - b) * sizeof(uint16_t);
        }
        for (int32_t r = 0; r < W; r++) {
            int32_t from = mod(r - 1, W);
            int32_t c = mod(from - s - 1, W);
            int64_t b = chunk_begin(n, W, c), e = chunk_end(n, W, c);
            for (int64_t i = b; i < e; i++)
                local[r][i] = oracle_round_wire(oracle_wire_value(msg[from][i - b], wire) +
                                                    oracle_wire_value(local[r][i], wire), wire);
        }
    }
    if (mode == MODE_ALLREDUCE) {
        for (int32_t s = 0; s < W - 1; s++) {
            for (int32_t r = 0; r < W; r++) {
                int32_t c = mod(r - s, W);
                int64_t b = chunk_begin(n, W, c), e = chunk_end(n, W, c);
                for (int64_t i = b; i < e; i++) msg[r][i - b] = local[r][i];
                bytes_sent[r] += (uint64_t)(e - b) * sizeof(uint16_t);
            }
            for (int32_t r = 0; r < W; r++) {
                int32_t from = mod(r - 1, W);
                int32_t c = mod(from - s, W);
                int64_t b = chunk_begin(n, W, c), e = chunk_end(n, W, c);
                for (int64_t i = b; i < e; i++) local[r][i] = msg[from][i - b];
            }
        }
        for (int32_t r = 0; r < W; r++)
            for (int64_t e = 0; e < n; e++) rank_buf[r][e] = (float)oracle_wire_value(local[r][e], wire);
    } else {
        for (int32_t r = 0; r < W; r++) {
            int64_t b = chunk_begin(n, W, r), e = chunk_end(n, W, r);
            for (int64_t i = b; i < e; i++) rank_buf[r][i] = (float)oracle_wire_value(local[r][i], wire);
        }
    }
    for (int32_t r = 0; r < W; r++) { free(local[r]); free(msg[r]); }
    free(local);
    free(msg);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* 6. overlap timeline (the lecture's alpha-beta model)                      */
/* ------------------------------------------------------------------------ */
/*
 * [P2 §3.1, exercises 4 and 5]: one compute stream produces the gradients
 * (parameter p at ready_ms[p]); one communication stream reduces the buckets
 * one at a time in issue order, each as soon as its last gradient exists and
 * the previous bucket is done; a bucket of n bytes takes alpha_ms +
 * ms_per_byte * n.  Outputs per bucket (indexed by bucket id): start_ms,
 * end_ms; step_ms = when both streams are done; serial_ms = the step with no
 * overlap (all communication after the last gradient).
 */
int oracle_overlap_timeline(int32_t nparams, const double* ready_ms, int32_t nbuckets, const int32_t* bucket_of,
                            const int32_t* bucket_order, const int64_t* bucket_bytes, double alpha_ms,
                            double ms_per_byte, double* start_ms, double* end_ms, double* step_ms,
                            double* serial_ms)
{
    if (nparams < 0 || nbuckets < 0) return -1;
    double backward_end = 0.0;
    for (int32_t p = 0; p < nparams; p++)
        if (ready_ms[p] > backward_end) backward_end = ready_ms[p];
    double comm_total = 0.0, comm_free = 0.0;
    for (int32_t k = 0; k < nbuckets; k++) {
        int32_t b = bucket_order[k];
        double ready = 0.0;
        for (int32_t p = 0; p < nparams; p++)
            if (bucket_of[p] == b && ready_ms[p] > ready) ready = ready_ms[p];
        double t = alpha_ms + ms_per_byte * (double)bucket_bytes[b];
        start_ms[b] = ready > comm_free ? ready : comm_free;
        end_ms[b] = start_ms[b] + t;
        comm_free = end_ms[b];
        comm_total += t;
    }
    *step_ms = comm_free > backward_end ? comm_free : backward_end;
    *serial_ms = backward_end + comm_total;
    return 0;
}
