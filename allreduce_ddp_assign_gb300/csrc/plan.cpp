// The bucket plan as an object of the C ABI (host only): the assignment of step
// 1, the buckets' places in one fp32 main_grad buffer per replica, the segment
// tables the kernels read, and the description DDP's logging data reports.
//
// "DDP: ring AllReduce and gradient buckets", section 17.13: the reducer's
// logging data lists every bucket's size (bucket_sizes) and, once the first
// iteration has recorded the order gradients became ready, the sizes of the
// buckets rebuilt over that order (rebuilt_bucket_sizes); section 17.12: each
// bucket is a flat buffer with its parameters' gradients at fixed offsets.
// "Megatron DDP: contiguous buffer and overlap", section 1: the buckets are
// slices of one contiguous main_grad buffer.
#include <cstring>
#include <vector>

#include "common.h"

struct ddp_plan {
    int32_t nparams = 0, nbuckets = 0;
    int64_t cap_bytes = 0, first_cap_bytes = 0;
    int32_t order = 0, pad_multiple = 1, fp32_buffer = 1;
    int64_t align = 1, replica_stride = 0;
    std::vector<int64_t> numels;
    std::vector<int32_t> dtypes;
    std::vector<int32_t> bucket_of, members;
    std::vector<int64_t> offset_of;
    std::vector<int64_t> bucket_numel, bucket_bytes, bucket_start;
    std::vector<int32_t> bucket_dtype, bucket_order;
    std::vector<int32_t> member_start;   // [nbuckets + 1]: bucket b's parameters are members[member_start[b] ..]
    std::vector<int64_t> seg_offset;     // per bucket nseg + 1 entries (the last: the end of its gradients)
    std::vector<int32_t> seg_param;      // per bucket nseg entries
    std::vector<int64_t> seg_offset_base, seg_param_base;
};

namespace {

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

}  // namespace

extern "C" ddp_status ddp_plan_create(const int64_t* numels, const int32_t* dtypes, int32_t nparams,
                                      int64_t cap_bytes, int64_t first_cap_bytes, int32_t order,
                                      int32_t pad_multiple, int32_t grad_reduce_in_fp32, int64_t align_elems,
                                      ddp_plan** out)
{
    using ddp::fail;
    const char* fn = "ddp_plan_create";
    if (!out) return fail(DDP_E_INVAL, "%s: out is NULL", fn);
    *out = nullptr;
    if (nparams < 0) return fail(DDP_E_INVAL, "%s: nparams = %d < 0", fn, nparams);
    if (nparams > 0 && !numels) return fail(DDP_E_INVAL, "%s: numels is NULL", fn);
    if (align_elems < 1 || align_elems > (int64_t{1} << 20))
        return fail(DDP_E_INVAL, "%s: align_elems = %lld outside [1, 2^20]", fn, static_cast<long long>(align_elems));
    auto p = new ddp_plan();
    p->nparams = nparams;
    p->cap_bytes = cap_bytes;
    p->first_cap_bytes = first_cap_bytes;
    p->order = order;
    p->pad_multiple = pad_multiple;
    p->fp32_buffer = grad_reduce_in_fp32 != 0;
    p->align = align_elems;
    p->numels.assign(numels, numels + nparams);
    p->dtypes = dtypes ? std::vector<int32_t>(dtypes, dtypes + nparams) : std::vector<int32_t>(nparams, DDP_F32);
    const size_t np = static_cast<size_t>(nparams);
    p->bucket_of.assign(np, 0);
    p->offset_of.assign(np, 0);
    p->members.assign(np, 0);
    const int32_t room = nparams + 2;   // enough for any assignment (ddp_assign_buckets)
    p->bucket_numel.assign(room, 0);
    p->bucket_bytes.assign(room, 0);
    p->bucket_dtype.assign(room, 0);
    p->bucket_order.assign(room, 0);
    int32_t nb = 0;
    const ddp_status st = ddp_assign_buckets(p->numels.data(), p->dtypes.data(), nparams, cap_bytes, first_cap_bytes,
                                             order, pad_multiple, grad_reduce_in_fp32, p->bucket_of.data(),
                                             p->offset_of.data(), p->members.data(), p->bucket_numel.data(),
                                             p->bucket_bytes.data(), p->bucket_dtype.data(), p->bucket_order.data(),
                                             room, &nb);
    if (st != DDP_OK) {
        delete p;
        return st;   // the assignment's own message stands
    }
    p->nbuckets = nb;
    for (auto* v : {&p->bucket_numel, &p->bucket_bytes}) v->resize(nb);
    for (auto* v : {&p->bucket_dtype, &p->bucket_order}) v->resize(nb);

    // members are grouped by bucket in layout order; place the buckets end to end,
    // each starting on a multiple of align_elems
    p->member_start.assign(static_cast<size_t>(nb) + 1, 0);
    for (int32_t q = 0; q < nparams; ++q) ++p->member_start[p->bucket_of[q] + 1];
    for (int32_t b = 0; b < nb; ++b) p->member_start[b + 1] += p->member_start[b];
    p->bucket_start.assign(nb, 0);
    int64_t pos = 0;
    for (int32_t b = 0; b < nb; ++b) {
        p->bucket_start[b] = pos;
        pos = round_up(pos + p->bucket_numel[b], align_elems);
    }
    p->replica_stride = pos > align_elems ? pos : align_elems;

    // segment tables: bucket b's parameters in layout order, then the end of its gradients
    p->seg_offset_base.assign(nb, 0);
    p->seg_param_base.assign(nb, 0);
    for (int32_t b = 0; b < nb; ++b) {
        p->seg_offset_base[b] = static_cast<int64_t>(p->seg_offset.size());
        p->seg_param_base[b] = static_cast<int64_t>(p->seg_param.size());
        int64_t end = 0;
        for (int32_t k = p->member_start[b]; k < p->member_start[b + 1]; ++k) {
            const int32_t q = p->members[k];
            p->seg_offset.push_back(p->offset_of[q]);
            p->seg_param.push_back(q);
            end = p->offset_of[q] + p->numels[q];
        }
        p->seg_offset.push_back(end);
    }
    *out = p;
    return ddp::ok();
}

extern "C" ddp_status ddp_plan_describe(const ddp_plan* p, ddp_plan_info* info, int64_t* bucket_numel,
                                        int64_t* bucket_bytes, int32_t* bucket_dtype, int32_t* bucket_order,
                                        int64_t* bucket_start, int32_t* member_start, int32_t* members,
                                        int32_t* bucket_of, int64_t* offset_of)
{
    if (!p) return ddp::fail(DDP_E_INVAL, "ddp_plan_describe: plan is NULL");
    if (info) {
        std::memset(info, 0, sizeof(*info));
        info->nparams = p->nparams;
        info->nbuckets = p->nbuckets;
        info->order = p->order;
        info->pad_multiple = p->pad_multiple;
        info->grad_reduce_in_fp32 = p->fp32_buffer;
        info->cap_bytes = p->cap_bytes;
        info->first_cap_bytes = p->first_cap_bytes;
        info->align_elems = p->align;
        info->replica_stride = p->replica_stride;
        info->seg_offset_len = static_cast<int64_t>(p->seg_offset.size());
        info->seg_param_len = static_cast<int64_t>(p->seg_param.size());
    }
    auto put = [](auto* dst, const auto& src) {
        if (dst && !src.empty()) std::memcpy(dst, src.data(), src.size() * sizeof(src[0]));
    };
    put(bucket_numel, p->bucket_numel);
    put(bucket_bytes, p->bucket_bytes);
    put(bucket_dtype, p->bucket_dtype);
    put(bucket_order, p->bucket_order);
    put(bucket_start, p->bucket_start);
    put(member_start, p->member_start);
    put(members, p->members);
    put(bucket_of, p->bucket_of);
    put(offset_of, p->offset_of);
    return ddp::ok();
}

extern "C" ddp_status ddp_plan_tables(const ddp_plan* p, int64_t* seg_offset, int32_t* seg_param)
{
    if (!p) return ddp::fail(DDP_E_INVAL, "ddp_plan_tables: plan is NULL");
    if ((!p->seg_offset.empty() && !seg_offset) || (!p->seg_param.empty() && !seg_param))
        return ddp::fail(DDP_E_INVAL, "ddp_plan_tables: an output table is NULL");
    if (!p->seg_offset.empty()) std::memcpy(seg_offset, p->seg_offset.data(), p->seg_offset.size() * sizeof(int64_t));
    if (!p->seg_param.empty()) std::memcpy(seg_param, p->seg_param.data(), p->seg_param.size() * sizeof(int32_t));
    return ddp::ok();
}

extern "C" ddp_status ddp_plan_bucket_descs(const ddp_plan* p, const int64_t* seg_offset_dev,
                                            const int32_t* seg_param_dev, ddp_bucket_desc* out)
{
    using ddp::fail;
    const char* fn = "ddp_plan_bucket_descs";
    if (!p) return fail(DDP_E_INVAL, "%s: plan is NULL", fn);
    if (p->nbuckets > 0 && (!out || !seg_offset_dev || (p->nparams > 0 && !seg_param_dev)))
        return fail(DDP_E_INVAL, "%s: NULL argument", fn);
    for (int32_t b = 0; b < p->nbuckets; ++b) {
        ddp_bucket_desc& d = out[b];
        d.numel = p->bucket_numel[b];
        d.nseg = p->member_start[b + 1] - p->member_start[b];
        d.dtype = p->bucket_dtype[b];
        d.seg_offset = seg_offset_dev + p->seg_offset_base[b];
        d.seg_param = seg_param_dev ? seg_param_dev + p->seg_param_base[b] : nullptr;
    }
    return ddp::ok();
}

extern "C" ddp_status ddp_plan_rebuilt(const ddp_plan* p, const int32_t* sequence, int64_t* bucket_bytes,
                                       int64_t* bucket_numel, int32_t max_buckets, int32_t* nbuckets)
{
    using ddp::fail;
    const char* fn = "ddp_plan_rebuilt";
    if (!p || !nbuckets) return fail(DDP_E_INVAL, "%s: NULL argument", fn);
    const size_t np = static_cast<size_t>(p->nparams);
    std::vector<int32_t> bucket_of(np), members(np);
    std::vector<int64_t> offset_of(np);
    const int32_t room = p->nparams + 2;
    std::vector<int64_t> numel(room), bytes(room);
    std::vector<int32_t> dtype(room), order(room);
    const ddp_status st = ddp_assign_buckets_ordered(
        p->numels.data(), p->dtypes.data(), p->nparams, sequence, p->cap_bytes, p->first_cap_bytes, p->pad_multiple,
        p->fp32_buffer, bucket_of.data(), offset_of.data(), members.data(), numel.data(), bytes.data(), dtype.data(),
        order.data(), room, nbuckets);
    if (st != DDP_OK) return st;
    if (*nbuckets > max_buckets)
        return fail(DDP_E_CAPACITY, "%s: %d buckets, room for %d", fn, *nbuckets, max_buckets);
    for (int32_t b = 0; b < *nbuckets; ++b) {
        if (bucket_bytes) bucket_bytes[b] = bytes[b];
        if (bucket_numel) bucket_numel[b] = numel[b];
    }
    return ddp::ok();
}

extern "C" ddp_status ddp_reducer_create_from_plan(const ddp_plan* p, const ddp_bucket_desc* buckets, int32_t W,
                                                   int32_t mode, int32_t flags, const void* const* grads,
                                                   const uint8_t* used, int32_t ld, float* main_grad,
                                                   void* const* grads_out, const uint8_t* global_used,
                                                   void* side_stream, ddp_reducer** out)
{
    if (!p) return ddp::fail(DDP_E_INVAL, "ddp_reducer_create_from_plan: plan is NULL");
    return ddp_reducer_create(p->nparams, p->nbuckets, p->bucket_of.data(), p->bucket_order.data(), buckets,
                              p->bucket_start.data(), W, mode, flags, grads, used, ld, main_grad, p->replica_stride,
                              grads_out, global_used, side_stream, out);
}

extern "C" void ddp_plan_destroy(ddp_plan* p) { delete p; }
