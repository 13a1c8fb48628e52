// Step 1 of the path: parameters -> size-capped buckets (host only).
//
// "DDP: ring AllReduce and gradient buckets", sections 17.2 and 17.13: a
// bucket is sealed as soon as its byte count reaches the cap, so it may
// overshoot; the rebuilt buckets follow reversed parameter order with a 1 MiB
// first bucket, the initial ones are computed in forward order and then handed
// over reversed.  "Lecture 15: PyTorch DDP", section 2.2 and exercise 3.
// "Megatron DDP: contiguous buffer and overlap", section 1: one contiguous
// buffer per dtype cut into max(40 MB, 1 MB x DP) buckets.
#include <algorithm>
#include <array>
#include <vector>

#include "common.h"

namespace {

struct Filling {                 // the open bucket of one dtype group
    std::vector<int32_t> params;
    int64_t bytes = 0;
    int32_t sealed = 0;          // buckets this group has sealed so far
    int32_t first_step = -1;     // iteration step at which the group first appeared
};

struct Sealed {
    std::vector<int32_t> params;
    int64_t bytes;
    int32_t dtype;
};

int64_t bytes_per_element(int32_t dtype, bool fp32_buffer)
{
    if (fp32_buffer) return 4;
    return dtype == DDP_F32 ? 4 : 2;
}

// `walk`: the parameters in iteration order (nullptr: derived from `order`).
ddp_status assign(const int64_t* numels, const int32_t* dtypes, int32_t nparams, const int32_t* walk,
                  int64_t cap_bytes, int64_t first_cap_bytes, int32_t order, int32_t pad_multiple,
                  int32_t grad_reduce_in_fp32, int32_t* bucket_of, int64_t* offset_of, int32_t* members,
                  int64_t* bucket_numel, int64_t* bucket_bytes, int32_t* bucket_dtype, int32_t* bucket_order,
                  int32_t max_buckets, int32_t* nbuckets)
{
    using ddp::fail;
    if (!nbuckets) return fail(DDP_E_INVAL, "ddp_assign_buckets: nbuckets is NULL");
    if (nparams < 0) return fail(DDP_E_INVAL, "ddp_assign_buckets: nparams = %d < 0", nparams);
    if (nparams > 0 && (!numels || !dtypes || !bucket_of || !offset_of || !members))
        return fail(DDP_E_INVAL, "ddp_assign_buckets: a per-parameter array is NULL");
    if (cap_bytes <= 0 || first_cap_bytes <= 0)
        return fail(DDP_E_INVAL, "ddp_assign_buckets: caps must be positive (cap %lld, first %lld)",
                    (long long)cap_bytes, (long long)first_cap_bytes);
    if (order != DDP_ORDER_REVERSE && order != DDP_ORDER_FWD_THEN_REVERSE && order != DDP_ORDER_MEGATRON)
        return fail(DDP_E_INVAL, "ddp_assign_buckets: unknown order %d", order);
    if (pad_multiple < 1) return fail(DDP_E_INVAL, "ddp_assign_buckets: pad_multiple %d < 1", pad_multiple);
    if (max_buckets < 0) return fail(DDP_E_INVAL, "ddp_assign_buckets: max_buckets < 0");
    for (int32_t p = 0; p < nparams; ++p) {
        if (numels[p] < 0) return fail(DDP_E_INVAL, "ddp_assign_buckets: parameter %d has numel %lld", p,
                                       (long long)numels[p]);
        if (dtypes[p] != DDP_F32 && dtypes[p] != DDP_BF16 && dtypes[p] != DDP_F16)
            return fail(DDP_E_INVAL, "ddp_assign_buckets: parameter %d has dtype code %d", p, dtypes[p]);
    }

    const bool fp32_buffer = grad_reduce_in_fp32 != 0;
    const bool megatron = order == DDP_ORDER_MEGATRON;
    std::array<Filling, 3> open;
    std::vector<Sealed> sealed;
    sealed.reserve(static_cast<size_t>(nparams) + 3);

    auto seal = [&](Filling& f, int32_t dtype) {
        sealed.push_back(Sealed{std::move(f.params), f.bytes, dtype});
        f.params.clear();
        f.bytes = 0;
        ++f.sealed;
    };

    for (int32_t step = 0; step < nparams; ++step) {
        const int32_t p = walk ? walk[step] : ((order == DDP_ORDER_REVERSE) ? (nparams - 1 - step) : step);
        const int32_t dt = dtypes[p];
        Filling& f = open[dt];
        if (f.first_step < 0) f.first_step = step;
        f.params.push_back(p);
        f.bytes += numels[p] * bytes_per_element(dt, fp32_buffer);
        const int64_t limit = (!megatron && f.sealed == 0) ? first_cap_bytes : cap_bytes;
        if (f.bytes >= limit) seal(f, dt);
    }

    // buckets still filling are sealed last, groups in order of first appearance
    std::array<int32_t, 3> groups = {0, 1, 2};
    std::stable_sort(groups.begin(), groups.end(),
                     [&](int32_t a, int32_t b) { return open[a].first_step < open[b].first_step; });
    for (int32_t dt : groups)
        if (!open[dt].params.empty()) seal(open[dt], dt);

    if (order == DDP_ORDER_FWD_THEN_REVERSE) std::reverse(sealed.begin(), sealed.end());

    const int32_t count = static_cast<int32_t>(sealed.size());
    *nbuckets = count;
    if (count > max_buckets)
        return fail(DDP_E_CAPACITY, "ddp_assign_buckets: %d buckets needed, room for %d", count, max_buckets);
    if (count > 0 && (!bucket_numel || !bucket_bytes || !bucket_dtype || !bucket_order))
        return fail(DDP_E_INVAL, "ddp_assign_buckets: a per-bucket array is NULL");

    int32_t k = 0;
    for (int32_t b = 0; b < count; ++b) {
        int64_t used = 0;
        for (int32_t p : sealed[b].params) {
            bucket_of[p] = b;
            offset_of[p] = used;
            members[k++] = p;
            used += numels[p];
        }
        const int64_t rem = used % pad_multiple;
        bucket_numel[b] = rem ? used + (pad_multiple - rem) : used;
        bucket_bytes[b] = sealed[b].bytes;
        bucket_dtype[b] = sealed[b].dtype;
        bucket_order[b] = megatron ? (count - 1 - b) : b;
    }
    return ddp::ok();
}

}  // namespace

extern "C" ddp_status ddp_assign_buckets(const int64_t* numels, const int32_t* dtypes, int32_t nparams,
                                         int64_t cap_bytes, int64_t first_cap_bytes, int32_t order,
                                         int32_t pad_multiple, int32_t grad_reduce_in_fp32,
                                         int32_t* bucket_of, int64_t* offset_of, int32_t* members,
                                         int64_t* bucket_numel, int64_t* bucket_bytes, int32_t* bucket_dtype,
                                         int32_t* bucket_order, int32_t max_buckets, int32_t* nbuckets)
{
    return assign(numels, dtypes, nparams, nullptr, cap_bytes, first_cap_bytes, order, pad_multiple,
                  grad_reduce_in_fp32, bucket_of, offset_of, members, bucket_numel, bucket_bytes, bucket_dtype,
                  bucket_order, max_buckets, nbuckets);
}

// Rebuilt buckets over the order the gradients were observed in ("DDP: ring
// AllReduce and gradient buckets" 17.13): the first gradients to arrive fill
// bucket 0 under first_cap_bytes, the rest follow under cap_bytes; issue order
// is bucket index order.
extern "C" ddp_status ddp_assign_buckets_ordered(const int64_t* numels, const int32_t* dtypes, int32_t nparams,
                                                 const int32_t* sequence, int64_t cap_bytes, int64_t first_cap_bytes,
                                                 int32_t pad_multiple, int32_t grad_reduce_in_fp32,
                                                 int32_t* bucket_of, int64_t* offset_of, int32_t* members,
                                                 int64_t* bucket_numel, int64_t* bucket_bytes, int32_t* bucket_dtype,
                                                 int32_t* bucket_order, int32_t max_buckets, int32_t* nbuckets)
{
    using ddp::fail;
    if (nparams > 0 && !sequence) return fail(DDP_E_INVAL, "ddp_assign_buckets_ordered: sequence is NULL");
    if (nparams > 0) {
        std::vector<uint8_t> seen(static_cast<size_t>(nparams), 0);
        for (int32_t k = 0; k < nparams; ++k) {
            const int32_t p = sequence[k];
            if (p < 0 || p >= nparams || seen[p])
                return fail(DDP_E_INVAL, "ddp_assign_buckets_ordered: sequence is not a permutation (position %d)", k);
            seen[p] = 1;
        }
    }
    return assign(numels, dtypes, nparams, sequence, cap_bytes, first_cap_bytes, DDP_ORDER_REVERSE, pad_multiple,
                  grad_reduce_in_fp32, bucket_of, offset_of, members, bucket_numel, bucket_bytes, bucket_dtype,
                  bucket_order, max_buckets, nbuckets);
}
