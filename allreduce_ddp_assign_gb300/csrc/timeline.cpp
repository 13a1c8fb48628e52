// The overlap model of "Lecture 15: PyTorch DDP" section 3.1 and exercises 4-5
// (host only): backward produces gradients on one stream, the reducer reduces
// buckets one after another on a second stream, each as soon as its last
// gradient exists and the previous bucket is done.  A bucket of n bytes costs
// alpha_ms + ms_per_byte * n (the ring's 2(K-1)alpha + 2(K-1)/K n/beta is this
// form with alpha_ms = 2(K-1)alpha and ms_per_byte = 2(K-1)/(K beta)).
#include <algorithm>
#include <vector>

#include "common.h"

extern "C" ddp_status ddp_overlap_timeline(int32_t nparams, const double* ready_ms, int32_t nbuckets,
                                           const int32_t* bucket_of, const int32_t* bucket_order,
                                           const int64_t* bucket_bytes, double alpha_ms, double ms_per_byte,
                                           double* start_ms, double* end_ms, double* step_ms, double* serial_ms)
{
    using ddp::fail;
    const char* fn = "ddp_overlap_timeline";
    if (nparams < 0 || nbuckets < 0) return fail(DDP_E_INVAL, "%s: negative size", fn);
    if ((nparams > 0 && (!ready_ms || !bucket_of)) ||
        (nbuckets > 0 && (!bucket_order || !bucket_bytes || !start_ms || !end_ms)) || !step_ms || !serial_ms)
        return fail(DDP_E_INVAL, "%s: NULL array", fn);
    if (alpha_ms < 0 || ms_per_byte < 0) return fail(DDP_E_INVAL, "%s: negative cost", fn);
    // when each bucket's last gradient appears
    std::vector<double> ready(static_cast<size_t>(nbuckets), 0.0);
    double backward_done = 0.0;
    for (int32_t p = 0; p < nparams; ++p) {
        const int32_t b = bucket_of[p];
        if (b < 0 || b >= nbuckets) return fail(DDP_E_INVAL, "%s: parameter %d in bucket %d of %d", fn, p, b, nbuckets);
        ready[b] = std::max(ready[b], ready_ms[p]);
        backward_done = std::max(backward_done, ready_ms[p]);
    }
    std::vector<uint8_t> seen(static_cast<size_t>(nbuckets), 0);
    double comm_free = 0.0, comm_sum = 0.0;
    for (int32_t k = 0; k < nbuckets; ++k) {
        const int32_t b = bucket_order[k];
        if (b < 0 || b >= nbuckets || seen[b]) return fail(DDP_E_INVAL, "%s: bucket_order is not a permutation", fn);
        seen[b] = 1;
        const double cost = alpha_ms + ms_per_byte * static_cast<double>(bucket_bytes[b]);
        start_ms[b] = std::max(ready[b], comm_free);
        end_ms[b] = start_ms[b] + cost;
        comm_free = end_ms[b];
        comm_sum += cost;
    }
    *step_ms = std::max(backward_done, comm_free);
    *serial_ms = backward_done + comm_sum;
    return ddp::ok();
}
