// Step 5 of the path: the reducer -- per-bucket pending counts, strictly
// in-order issue on a side stream, and the end-of-backward wait.
//
// "DDP: ring AllReduce and gradient buckets" sections 17.2 (pending count per
// bucket), 17.12 (mark_variable_ready; mark_bucket_ready issues buckets in
// index order from next_bucket_), 17.16 (prepare_for_backward resets the
// counts; marking a variable twice is an error), 17.41 (finalize_backward waits
// on every bucket; on CUDA the wait is a stream wait); "Lecture 15: PyTorch
// DDP" section 2.3 (bucket i+1 waits for bucket i even if it filled first; all
// ranks must issue in the same order); "Megatron DDP: contiguous buffer and
// overlap" sections 2-3 (grad-ready hook, start_grad_sync / finish_grad_sync on
// a separate stream).
//
// GPU side: when a bucket's count reaches zero, an event is recorded on every
// stream that produced one of its gradients; when the bucket's turn comes the
// side stream waits for those events and the bucket's kernels are launched on
// it.  Finalize records one event on the side stream and makes the consumer
// wait for it; with a timeout it also polls that event on the host.
//
// find_unused_parameters ("Lecture 15: PyTorch DDP" section 4.2; "DDP: PyTorch
// Distributed-Experiences on Accelerating Data Parallel Training" sections 2.2
// and 3.2): the local-used bitmap lives in pinned host memory; prepare copies
// it to the device and runs the bitmap all-reduce on the side stream ahead of
// every bucket, and marks ready on the host the parameters no replica used.
#include <cuda_runtime.h>

#include <algorithm>
#include <chrono>
#include <string>
#include <thread>
#include <vector>

#include "common.h"

namespace {

enum class Phase { Idle, Backward, Finalized };

bool cuda_ok(cudaError_t e, const char* what, ddp_status* st)
{
    if (e == cudaSuccess) return true;
    *st = ddp::fail(DDP_E_CUDA, "%s failed: %s", what, cudaGetErrorString(e));
    return false;
}

}  // namespace

struct ddp_reducer {
    int32_t nparams = 0, nbuckets = 0, W = 1, mode = DDP_ALLREDUCE, flags = 0;
    std::vector<int32_t> bucket_of, order, bucket_params;
    std::vector<ddp_bucket_desc> buckets;
    std::vector<int64_t> start;
    const void* const* grads = nullptr;
    const uint8_t* used = nullptr;
    int32_t ld = 0;
    float* mg = nullptr;
    int64_t stride = 0;
    void* const* grads_out = nullptr;
    const uint8_t* global_used = nullptr;
    cudaStream_t side = nullptr;

    // one iteration
    Phase phase = Phase::Idle;
    int32_t accumulate = 0;
    std::vector<int32_t> pending;
    std::vector<uint8_t> marked;
    int32_t next = 0;
    std::vector<std::vector<cudaStream_t>> producers;
    std::vector<int32_t> log;

    // CUDA events (none in dry-run mode)
    std::vector<std::vector<cudaEvent_t>> ready;
    std::vector<cudaEvent_t> t_begin, t_end;
    cudaEvent_t done = nullptr;
    bool timing_valid = false;
    std::vector<ddp_bucket_desc> group_descs;  // scratch for coalesced issue
    std::vector<float*> group_mgs;
    std::vector<int32_t> seq_now, seq_last;        // gradient-ready order: this iteration, last finalized one
    std::vector<std::vector<cudaEvent_t>> gates;  // per bucket: the events its issue waits for
    std::vector<int32_t> batch_done;               // buckets completed in the current batch of marks
    std::vector<cudaStream_t> batch_streams;
    std::vector<cudaEvent_t> batch_events;
    std::vector<cudaEvent_t> waited;

    // find_unused_parameters
    bool find_unused = false;
    uint8_t* fu_local = nullptr;     // DEVICE W x ld: the copied local-used bitmap
    uint8_t* fu_global = nullptr;    // DEVICE nparams: the all-reduced flags
    int32_t* fu_count = nullptr;     // DEVICE nparams or null: the all-reduced counts
    uint8_t* fu_host = nullptr;      // HOST W x nparams, pinned (dry-run: fu_host_dry)
    std::vector<uint8_t> fu_host_dry;
    cudaEvent_t fu_copied = nullptr; // the last host-to-device copy of the bitmap has been read
    bool fu_copy_pending = false;

    std::vector<ddp_powersgd*> hooks;  // per bucket: the PowerSGD hook, or null
    std::vector<cudaEvent_t> bdone;    // per bucket: recorded after its reduction (DDP_R_BUCKET_DONE)
    // per bucket: one more event its issue waits for, or null (the host front end's
    // copy of the bucket's previous result to the host; owned by the front end)
    std::vector<cudaEvent_t> extra_gate;

    bool dry() const { return flags & DDP_R_DRY_RUN; }
    uint8_t* host_bitmap() { return dry() ? fu_host_dry.data() : fu_host; }
    // flags the packs read (replica w used p) and the ones unpack reads (anyone used p)
    const uint8_t* pack_used() const { return used ? used : (find_unused ? fu_local : nullptr); }
    const uint8_t* unpack_used() const { return find_unused ? fu_global : global_used; }

    std::string unmarked_list() const
    {
        std::string s;
        int shown = 0;
        for (int32_t p = 0; p < nparams; ++p) {
            if (marked[p]) continue;
            if (shown == 64) {
                s += " ...";
                break;
            }
            s += " " + std::to_string(p);
            ++shown;
        }
        return s;
    }

    int32_t wire() const
    {
        return (flags & DDP_R_WIRE_BF16) ? DDP_BF16 : ((flags & DDP_R_WIRE_F16) ? DDP_F16 : DDP_F32);
    }

    ddp_status launch_bucket(int32_t b)
    {
        const ddp_bucket_desc& d = buckets[b];
        float* mgb = mg ? mg + start[b] : nullptr;
        void* st = static_cast<void*>(side);
        const bool copy_back = flags & DDP_R_COPY_BACK;
        if (hooks[b]) {   // communication hook: pack, the hook's reduction, copy-back
            ddp_status s = ddp::launch_pack(d, grads, pack_used(), ld, W, mgb, stride, accumulate, st);
            if (s == DDP_OK) s = ddp_powersgd_reduce(hooks[b], mgb, stride, st);
            if (s == DDP_OK && copy_back)
                s = ddp::launch_unpack(d, mgb, stride, W, mode, grads_out, ld, unpack_used(), st);
            return s;
        }
        if (flags & DDP_R_FUSED)
            return ddp::launch_fused(d, grads, pack_used(), ld, W, mode, accumulate, mgb, stride,
                                     copy_back ? grads_out : nullptr, unpack_used(), st, wire());
        ddp_status s = ddp::launch_pack(d, grads, pack_used(), ld, W, mgb, stride, accumulate, st);
        if (s == DDP_OK) s = ddp::launch_allreduce(mgb, stride, d.numel, W, mode, st, wire());
        if (s == DDP_OK && copy_back)
            s = ddp::launch_unpack(d, mgb, stride, W, mode, grads_out, ld, unpack_used(), st);
        return s;
    }

    // Issue the buckets order[pos .. pos+count-1] (all ready) on the side stream,
    // then (DDP_R_BUCKET_DONE) record each bucket's completion event after them.
    ddp_status issue(int32_t pos, int32_t count)
    {
        ddp_status st = issue_launches(pos, count);
        if (st != DDP_OK || dry() || !(flags & DDP_R_BUCKET_DONE)) return st;
        for (int32_t i = 0; i < count; ++i)
            if (!cuda_ok(cudaEventRecord(bdone[order[pos + i]], side), "cudaEventRecord", &st)) return st;
        return DDP_OK;
    }

    // Wait for the buckets' producers, then one launch per bucket, or one coalesced launch.
    ddp_status issue_launches(int32_t pos, int32_t count)
    {
        for (int32_t i = 0; i < count; ++i) log.push_back(order[pos + i]);
        if (dry()) return DDP_OK;
        ddp_status st = DDP_OK;
        // wait once for every distinct gating event of the buckets going out
        waited.clear();
        for (int32_t i = 0; i < count; ++i) {
            for (cudaEvent_t e : gates[order[pos + i]]) {
                bool seen = false;
                for (cudaEvent_t x : waited) seen = seen || x == e;
                if (seen) continue;
                waited.push_back(e);
                if (!cuda_ok(cudaStreamWaitEvent(side, e, 0), "cudaStreamWaitEvent", &st)) return st;
            }
        }
        for (int32_t i = 0; i < count; ++i) {
            const cudaEvent_t e = extra_gate[order[pos + i]];
            if (e && !cuda_ok(cudaStreamWaitEvent(side, e, 0), "cudaStreamWaitEvent", &st)) return st;
        }
        const bool timing = flags & DDP_R_TIMING;
        bool hooked = false;
        for (int32_t i = 0; i < count; ++i) hooked = hooked || hooks[order[pos + i]];
        if (hooked && count > 1) {   // hooked buckets go out one by one
            for (int32_t i = 0; i < count; ++i) {
                const int32_t b = order[pos + i];
                if (timing && !cuda_ok(cudaEventRecord(t_begin[b], side), "cudaEventRecord", &st)) return st;
                if ((st = launch_bucket(b)) != DDP_OK) return st;
                if (timing && !cuda_ok(cudaEventRecord(t_end[b], side), "cudaEventRecord", &st)) return st;
            }
            return DDP_OK;
        }
        if (count > 1) {
            if (timing)
                for (int32_t i = 0; i < count; ++i)
                    if (!cuda_ok(cudaEventRecord(t_begin[order[pos + i]], side), "cudaEventRecord", &st)) return st;
            group_descs.clear();
            group_mgs.clear();
            for (int32_t i = 0; i < count; ++i) {
                const int32_t b = order[pos + i];
                group_descs.push_back(buckets[b]);
                group_mgs.push_back(mg ? mg + start[b] : nullptr);
            }
            st = ddp::launch_fused_group(group_descs.data(), group_mgs.data(), count, grads, pack_used(), ld, W,
                                         mode, accumulate, stride, (flags & DDP_R_COPY_BACK) ? grads_out : nullptr,
                                         unpack_used(), static_cast<void*>(side), wire());
            if (st != DDP_OK) return st;
            if (timing)
                for (int32_t i = 0; i < count; ++i)
                    if (!cuda_ok(cudaEventRecord(t_end[order[pos + i]], side), "cudaEventRecord", &st)) return st;
            return DDP_OK;
        }
        const int32_t b = order[pos];
        if (timing)
            if (!cuda_ok(cudaEventRecord(t_begin[b], side), "cudaEventRecord", &st)) return st;
        st = launch_bucket(b);
        if (st != DDP_OK) return st;
        if (timing)
            if (!cuda_ok(cudaEventRecord(t_end[b], side), "cudaEventRecord", &st)) return st;
        return DDP_OK;
    }

    ddp_status ensure_events(int32_t b)
    {
        ddp_status st = DDP_OK;
        auto& evs = ready[b];
        while (evs.size() < producers[b].size()) {
            cudaEvent_t e = nullptr;
            if (!cuda_ok(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "cudaEventCreate", &st)) return st;
            evs.push_back(e);
        }
        return DDP_OK;
    }

    // Bucket b's count reached zero: record the events that gate it (one per
    // stream that produced its gradients).  With `defer` the recording waits for
    // the end of the batch (gate_batch), which records one event per stream for
    // every bucket the batch completed.
    ddp_status bucket_ready(int32_t b, bool defer)
    {
        if (dry()) return DDP_OK;
        if (defer) {
            batch_done.push_back(b);
            return DDP_OK;
        }
        ddp_status st = ensure_events(b);
        if (st != DDP_OK) return st;
        gates[b].clear();
        for (size_t i = 0; i < producers[b].size(); ++i) {
            if (!cuda_ok(cudaEventRecord(ready[b][i], producers[b][i]), "cudaEventRecord", &st)) return st;
            gates[b].push_back(ready[b][i]);
        }
        return DDP_OK;
    }

    // End of a batch of marks: one event per producer stream gates all the buckets
    // the batch completed (events on one stream are ordered, so the last suffices).
    ddp_status gate_batch()
    {
        if (dry() || batch_done.empty()) return DDP_OK;
        ddp_status st = DDP_OK;
        batch_streams.clear();
        batch_events.clear();
        for (int32_t b : batch_done) {
            if ((st = ensure_events(b)) != DDP_OK) return st;
            gates[b].clear();
            for (size_t i = 0; i < producers[b].size(); ++i) {
                const cudaStream_t s = producers[b][i];
                size_t j = 0;
                while (j < batch_streams.size() && batch_streams[j] != s) ++j;
                if (j == batch_streams.size()) {  // first bucket of the batch on this stream: record its event
                    if (!cuda_ok(cudaEventRecord(ready[b][i], s), "cudaEventRecord", &st)) return st;
                    batch_streams.push_back(s);
                    batch_events.push_back(ready[b][i]);
                }
                gates[b].push_back(batch_events[j]);
            }
        }
        batch_done.clear();
        return DDP_OK;
    }

    // Issue, in order, every bucket from `next` on whose count has reached zero.
    ddp_status issue_ready()
    {
        if (phase != Phase::Backward) return DDP_OK;  // counts are only meaningful inside an iteration
        const bool coalesce = flags & DDP_R_COALESCE;
        while (next < nbuckets && pending[order[next]] == 0) {
            int32_t count = 1;
            if (coalesce)
                while (next + count < nbuckets && pending[order[next + count]] == 0) ++count;
            const ddp_status st = issue(next, count);
            next += count;
            if (st != DDP_OK) return st;
        }
        return DDP_OK;
    }

    ddp_status start_find_unused();

    void destroy_events()
    {
        if (dry()) return;
        for (auto& v : ready)
            for (cudaEvent_t e : v) cudaEventDestroy(e);
        for (cudaEvent_t e : t_begin) cudaEventDestroy(e);
        for (cudaEvent_t e : t_end) cudaEventDestroy(e);
        if (done) cudaEventDestroy(done);
        if (fu_copied) cudaEventDestroy(fu_copied);
        for (cudaEvent_t e : bdone) cudaEventDestroy(e);
        if (fu_host) cudaFreeHost(fu_host);
    }
};

extern "C" ddp_status ddp_reducer_create(int32_t nparams, int32_t nbuckets, const int32_t* bucket_of,
                                         const int32_t* bucket_order, const ddp_bucket_desc* buckets,
                                         const int64_t* bucket_start, int32_t W, int32_t mode, int32_t flags,
                                         const void* const* grads, const uint8_t* used, int32_t ld,
                                         float* main_grad, int64_t replica_stride, void* const* grads_out,
                                         const uint8_t* global_used, void* side_stream, ddp_reducer** out)
{
    using ddp::fail;
    const char* fn = "ddp_reducer_create";
    if (!out) return fail(DDP_E_INVAL, "%s: out is NULL", fn);
    *out = nullptr;
    if (nparams < 0 || nbuckets < 0) return fail(DDP_E_INVAL, "%s: negative size", fn);
    if (nparams > 0 && !bucket_of) return fail(DDP_E_INVAL, "%s: bucket_of is NULL", fn);
    if (nbuckets > 0 && (!bucket_order || !buckets || !bucket_start))
        return fail(DDP_E_INVAL, "%s: a per-bucket array is NULL", fn);
    if (W < 1 || W > ddp::kMaxReplicas) return fail(DDP_E_INVAL, "%s: W = %d outside [1, %d]", fn, W, ddp::kMaxReplicas);
    if (mode != DDP_ALLREDUCE && mode != DDP_REDUCE_SCATTER) return fail(DDP_E_INVAL, "%s: unknown mode %d", fn, mode);
    if (flags & ~(DDP_R_FUSED | DDP_R_COPY_BACK | DDP_R_TIMING | DDP_R_DRY_RUN | DDP_R_COALESCE | DDP_R_WIRE_BF16 |
                  DDP_R_WIRE_F16 | DDP_R_BUCKET_DONE))
        return fail(DDP_E_INVAL, "%s: unknown flag bits 0x%x", fn, flags);
    if ((flags & DDP_R_WIRE_BF16) && (flags & DDP_R_WIRE_F16))
        return fail(DDP_E_INVAL, "%s: DDP_R_WIRE_BF16 and DDP_R_WIRE_F16 exclude each other", fn);
    if ((flags & DDP_R_COALESCE) && !(flags & DDP_R_FUSED))
        return fail(DDP_E_INVAL, "%s: DDP_R_COALESCE needs DDP_R_FUSED", fn);
    const bool dry = flags & DDP_R_DRY_RUN;

    auto r = new ddp_reducer();
    r->nparams = nparams;
    r->nbuckets = nbuckets;
    r->W = W;
    r->mode = mode;
    r->flags = flags;
    r->bucket_of.assign(bucket_of, bucket_of + nparams);
    r->order.assign(bucket_order, bucket_order + nbuckets);
    r->buckets.assign(buckets, buckets + nbuckets);
    r->start.assign(bucket_start, bucket_start + nbuckets);
    r->bucket_params.assign(nbuckets, 0);
    auto reject = [&](ddp_status s) {
        delete r;
        return s;
    };
    for (int32_t p = 0; p < nparams; ++p) {
        if (bucket_of[p] < 0 || bucket_of[p] >= nbuckets)
            return reject(fail(DDP_E_INVAL, "%s: parameter %d maps to bucket %d of %d", fn, p, bucket_of[p], nbuckets));
        ++r->bucket_params[bucket_of[p]];
    }
    std::vector<uint8_t> seen(nbuckets, 0);
    for (int32_t k = 0; k < nbuckets; ++k) {
        const int32_t b = bucket_order[k];
        if (b < 0 || b >= nbuckets || seen[b])
            return reject(fail(DDP_E_INVAL, "%s: bucket_order is not a permutation (position %d)", fn, k));
        seen[b] = 1;
        if (r->bucket_params[b] == 0)
            return reject(fail(DDP_E_INVAL, "%s: bucket %d has no parameter", fn, b));
        const ddp_bucket_desc& d = buckets[b];
        if (d.numel < 0 || d.nseg < 0 || (d.nseg > 0 && (!d.seg_offset || !d.seg_param)))
            return reject(fail(DDP_E_INVAL, "%s: bad descriptor for bucket %d", fn, b));
        if (mode == DDP_REDUCE_SCATTER && d.numel % W != 0)
            return reject(fail(DDP_E_INVAL, "%s: bucket %d numel %lld not a multiple of W = %d", fn, b,
                               static_cast<long long>(d.numel), W));
        if (bucket_start[b] < 0 || (W > 1 && bucket_start[b] + d.numel > replica_stride))
            return reject(fail(DDP_E_INVAL, "%s: bucket %d [%lld, +%lld) exceeds replica_stride %lld", fn, b,
                               static_cast<long long>(bucket_start[b]), static_cast<long long>(d.numel),
                               static_cast<long long>(replica_stride)));
    }
    if (!dry) {
        if (nparams > 0 && (!grads || ld < 1)) return reject(fail(DDP_E_INVAL, "%s: grads table is NULL or ld < 1", fn));
        if (!(flags & DDP_R_FUSED) && !main_grad)
            return reject(fail(DDP_E_INVAL, "%s: staged issue (no DDP_R_FUSED) needs main_grad", fn));
        if (!main_grad && !(flags & DDP_R_COPY_BACK))
            return reject(fail(DDP_E_INVAL, "%s: without main_grad the results need DDP_R_COPY_BACK", fn));
        if ((flags & DDP_R_COPY_BACK) && !grads_out)
            return reject(fail(DDP_E_INVAL, "%s: DDP_R_COPY_BACK needs grads_out", fn));
    }
    r->grads = grads;
    r->used = used;
    r->ld = ld;
    r->mg = main_grad;
    r->stride = replica_stride;
    r->grads_out = grads_out;
    r->global_used = global_used;
    r->side = static_cast<cudaStream_t>(side_stream);
    r->extra_gate.assign(nbuckets, nullptr);
    r->pending.assign(nbuckets, 0);
    r->marked.assign(nparams, 0);
    r->producers.resize(nbuckets);
    r->ready.resize(nbuckets);
    r->gates.resize(nbuckets);
    r->hooks.assign(nbuckets, nullptr);

    if (!dry) {
        ddp_status st = DDP_OK;
        auto mk = [&](cudaEvent_t* e, unsigned fl) {
            return cuda_ok(cudaEventCreateWithFlags(e, fl), "cudaEventCreate", &st);
        };
        if (!mk(&r->done, cudaEventDisableTiming)) return reject(st);
        for (int32_t b = 0; b < nbuckets; ++b) {
            cudaEvent_t e = nullptr;
            if (!mk(&e, cudaEventDisableTiming)) return reject(st);
            r->ready[b].push_back(e);
        }
        if (flags & DDP_R_BUCKET_DONE) {
            r->bdone.assign(nbuckets, nullptr);
            for (int32_t b = 0; b < nbuckets; ++b)
                if (!mk(&r->bdone[b], cudaEventDisableTiming)) return reject(st);
        }
        if (flags & DDP_R_TIMING) {
            r->t_begin.assign(nbuckets, nullptr);
            r->t_end.assign(nbuckets, nullptr);
            for (int32_t b = 0; b < nbuckets; ++b)
                if (!mk(&r->t_begin[b], cudaEventDefault) || !mk(&r->t_end[b], cudaEventDefault)) return reject(st);
        }
    }
    *out = r;
    return ddp::ok();
}

extern "C" ddp_status ddp_reducer_prepare(ddp_reducer* r, int32_t accumulate)
{
    if (!r) return ddp::fail(DDP_E_INVAL, "ddp_reducer_prepare: reducer is NULL");
    if (accumulate && !r->mg && !r->dry())
        return ddp::fail(DDP_E_INVAL, "ddp_reducer_prepare: accumulate needs main_grad");
    ddp_status st = DDP_OK;
    if (r->phase == Phase::Backward && r->next < r->nbuckets) {
        bool any = false;
        for (uint8_t m : r->marked) any = any || m;
        if (any)
            st = ddp::fail(DDP_E_INCOMPLETE,
                           "ddp_reducer_prepare: the previous iteration did not finish reducing its buckets "
                           "(%d of %d issued); parameters never marked ready:%s",
                           r->next, r->nbuckets, r->unmarked_list().c_str());
    }
    for (int32_t b = 0; b < r->nbuckets; ++b) {
        r->pending[b] = r->bucket_params[b];
        r->producers[b].clear();
        r->gates[b].clear();
    }
    r->batch_done.clear();
    std::fill(r->marked.begin(), r->marked.end(), 0);
    r->seq_now.clear();
    r->next = 0;
    r->log.clear();
    r->accumulate = accumulate != 0;
    r->phase = Phase::Backward;
    if (r->find_unused) {
        const ddp_status s2 = r->start_find_unused();
        if (s2 != DDP_OK) return s2;
    }
    return st == DDP_OK ? ddp::ok() : st;
}

namespace {

// Mark one parameter; with defer the issue pass is left to the caller.  A
// parameter marked without a producer (has_producer false) gates nothing.
ddp_status mark_one(ddp_reducer* r, int32_t param, void* producer_stream, bool defer, bool has_producer)
{
    if (!r) return ddp::fail(DDP_E_INVAL, "ddp_reducer_mark_ready: reducer is NULL");
    if (param < 0 || param >= r->nparams)
        return ddp::fail(DDP_E_INVAL, "ddp_reducer_mark_ready: parameter %d outside [0, %d)", param, r->nparams);
    if (r->phase != Phase::Backward)
        return ddp::fail(DDP_E_STATE, "ddp_reducer_mark_ready: parameter %d marked outside an iteration "
                                      "(call ddp_reducer_prepare first)", param);
    if (r->marked[param])
        return ddp::fail(DDP_E_STATE, "ddp_reducer_mark_ready: parameter %d was marked ready twice in one iteration",
                         param);
    r->marked[param] = 1;
    r->seq_now.push_back(param);
    const int32_t b = r->bucket_of[param];
    if (!r->dry() && has_producer) {
        auto& ps = r->producers[b];
        const cudaStream_t s = static_cast<cudaStream_t>(producer_stream);
        bool have = false;
        for (cudaStream_t x : ps) have = have || x == s;
        if (!have) ps.push_back(s);
    }
    if (--r->pending[b] == 0) {
        ddp_status st = r->bucket_ready(b, defer);
        if (st == DDP_OK && !defer) st = r->issue_ready();
        if (st != DDP_OK) return st;
    }
    return ddp::ok();
}

}  // namespace

// prepare's find_unused steps: copy the host bitmap to the device and all-reduce
// it on the side stream (ahead of every bucket of the iteration), then mark
// ready, without a producer, every parameter no replica used.
ddp_status ddp_reducer::start_find_unused()
{
    ddp_status st = DDP_OK;
    const uint8_t* host = host_bitmap();
    if (!dry() && nparams > 0) {
        if (!cuda_ok(cudaMemcpy2DAsync(fu_local, static_cast<size_t>(ld), host, static_cast<size_t>(nparams),
                                       static_cast<size_t>(nparams), static_cast<size_t>(W), cudaMemcpyHostToDevice,
                                       side),
                     "cudaMemcpy2DAsync", &st))
            return st;
        if (!cuda_ok(cudaEventRecord(fu_copied, side), "cudaEventRecord", &st)) return st;
        fu_copy_pending = true;
        st = ddp_used_allreduce(fu_local, ld, W, nparams, fu_count, fu_global, static_cast<void*>(side));
        if (st != DDP_OK) return st;
    }
    for (int32_t p = 0; p < nparams && st == DDP_OK; ++p) {
        bool any = false;
        for (int32_t w = 0; w < W && !any; ++w) any = host[static_cast<int64_t>(w) * nparams + p] != 0;
        if (!any) st = mark_one(this, p, nullptr, true, false);
    }
    const ddp_status s2 = gate_batch();
    if (st != DDP_OK) return st;
    if (s2 != DDP_OK) return s2;
    return issue_ready();
}

extern "C" ddp_status ddp_reducer_find_unused(ddp_reducer* r, uint8_t* local_used, uint8_t* global_used,
                                              int32_t* global_count)
{
    using ddp::fail;
    const char* fn = "ddp_reducer_find_unused";
    if (!r) return fail(DDP_E_INVAL, "%s: reducer is NULL", fn);
    if (r->phase == Phase::Backward) return fail(DDP_E_STATE, "%s: called inside an iteration", fn);
    if (r->find_unused) return fail(DDP_E_STATE, "%s: already on", fn);
    if (r->global_used)
        return fail(DDP_E_INVAL, "%s: the reducer was created with its own global_used flags", fn);
    const size_t bytes = static_cast<size_t>(r->W) * static_cast<size_t>(r->nparams);
    if (r->dry()) {
        r->fu_host_dry.assign(bytes > 0 ? bytes : 1, 1);
    } else {
        if (r->nparams > 0 && (!local_used || !global_used))
            return fail(DDP_E_INVAL, "%s: local_used or global_used is NULL", fn);
        if (r->ld < r->nparams) return fail(DDP_E_INVAL, "%s: ld = %d < nparams = %d", fn, r->ld, r->nparams);
        ddp_status st = DDP_OK;
        if (!cuda_ok(cudaEventCreateWithFlags(&r->fu_copied, cudaEventDisableTiming), "cudaEventCreate", &st))
            return st;
        void* h = nullptr;
        if (!cuda_ok(cudaHostAlloc(&h, bytes > 0 ? bytes : 1, cudaHostAllocDefault), "cudaHostAlloc", &st)) {
            cudaEventDestroy(r->fu_copied);
            r->fu_copied = nullptr;
            return st;
        }
        r->fu_host = static_cast<uint8_t*>(h);
        std::fill(r->fu_host, r->fu_host + bytes, static_cast<uint8_t>(1));
    }
    r->fu_local = local_used;
    r->fu_global = global_used;
    r->fu_count = global_count;
    r->find_unused = true;
    return ddp::ok();
}

extern "C" ddp_status ddp_reducer_register_powersgd(ddp_reducer* r, int32_t bucket, ddp_powersgd* h)
{
    using ddp::fail;
    const char* fn = "ddp_reducer_register_powersgd";
    if (!r) return fail(DDP_E_INVAL, "%s: reducer is NULL", fn);
    if (bucket < 0 || bucket >= r->nbuckets) return fail(DDP_E_INVAL, "%s: bucket %d outside [0, %d)", fn, bucket, r->nbuckets);
    if (r->phase == Phase::Backward) return fail(DDP_E_STATE, "%s: called inside an iteration", fn);
    if (h) {
        if (r->mode != DDP_ALLREDUCE) return fail(DDP_E_INVAL, "%s: the hook replaces an allreduce, not a reduce_scatter", fn);
        if (!r->mg && !r->dry()) return fail(DDP_E_INVAL, "%s: the hook works on main_grad; the reducer has none", fn);
        if (ddp::powersgd_replicas(h) != r->W)
            return fail(DDP_E_INVAL, "%s: state planned for W = %d, reducer has W = %d", fn, ddp::powersgd_replicas(h), r->W);
        if (ddp::powersgd_numel(h) != r->buckets[bucket].numel)
            return fail(DDP_E_INVAL, "%s: state planned for %lld elements, bucket %d has %lld", fn,
                        static_cast<long long>(ddp::powersgd_numel(h)), bucket,
                        static_cast<long long>(r->buckets[bucket].numel));
    }
    r->hooks[bucket] = h;
    return ddp::ok();
}

extern "C" ddp_status ddp_reducer_set_local_used(ddp_reducer* r, const uint8_t* flags, int32_t ld)
{
    using ddp::fail;
    const char* fn = "ddp_reducer_set_local_used";
    if (!r) return fail(DDP_E_INVAL, "%s: reducer is NULL", fn);
    if (!r->find_unused) return fail(DDP_E_STATE, "%s: find_unused is off (call ddp_reducer_find_unused)", fn);
    if (r->phase == Phase::Backward) return fail(DDP_E_STATE, "%s: called inside an iteration", fn);
    if (r->nparams > 0 && !flags) return fail(DDP_E_INVAL, "%s: flags is NULL", fn);
    if (ld < r->nparams) return fail(DDP_E_INVAL, "%s: ld = %d < nparams = %d", fn, ld, r->nparams);
    ddp_status st = DDP_OK;
    if (r->fu_copy_pending) {
        if (!cuda_ok(cudaEventSynchronize(r->fu_copied), "cudaEventSynchronize", &st)) return st;
        r->fu_copy_pending = false;
    }
    uint8_t* host = r->host_bitmap();
    for (int32_t w = 0; w < r->W; ++w)
        for (int32_t p = 0; p < r->nparams; ++p)
            host[static_cast<int64_t>(w) * r->nparams + p] = flags[static_cast<int64_t>(w) * ld + p] != 0;
    return ddp::ok();
}

extern "C" ddp_status ddp_reducer_mark_ready(ddp_reducer* r, int32_t param, void* producer_stream)
{
    return mark_one(r, param, producer_stream, false, true);
}

extern "C" ddp_status ddp_reducer_mark_ready_many(ddp_reducer* r, const int32_t* params, int32_t n,
                                                  void* producer_stream)
{
    if (n < 0 || (n > 0 && !params)) return ddp::fail(DDP_E_INVAL, "ddp_reducer_mark_ready_many: bad list");
    ddp_status st = DDP_OK;
    for (int32_t i = 0; i < n && st == DDP_OK; ++i) st = mark_one(r, params[i], producer_stream, true, true);
    // one issue pass for everything the list completed (coalesced when enabled),
    // also after a failure so that the parameters already marked are not stranded
    ddp_status st2 = r ? r->gate_batch() : DDP_OK;
    if (st2 == DDP_OK && r) st2 = r->issue_ready();
    if (st != DDP_OK) return st;
    return st2 == DDP_OK ? ddp::ok() : st2;
}

extern "C" ddp_status ddp_reducer_finalize(ddp_reducer* r, void* consumer_stream, int64_t timeout_us)
{
    const char* fn = "ddp_reducer_finalize";
    if (!r) return ddp::fail(DDP_E_INVAL, "%s: reducer is NULL", fn);
    if (r->phase == Phase::Idle) return ddp::fail(DDP_E_STATE, "%s: no iteration in progress", fn);
    if (r->phase == Phase::Backward) {
        if (r->next < r->nbuckets)
            return ddp::fail(DDP_E_INCOMPLETE, "%s: %d of %d buckets issued; parameters never marked ready:%s", fn,
                             r->next, r->nbuckets, r->unmarked_list().c_str());
        if (!r->dry()) {
            ddp_status st = DDP_OK;
            if (!cuda_ok(cudaEventRecord(r->done, r->side), "cudaEventRecord", &st)) return st;
            if (!cuda_ok(cudaStreamWaitEvent(static_cast<cudaStream_t>(consumer_stream), r->done, 0),
                         "cudaStreamWaitEvent", &st))
                return st;
        }
        r->phase = Phase::Finalized;
        r->timing_valid = (r->flags & DDP_R_TIMING) != 0;
        r->seq_last = r->seq_now;
    }
    if (timeout_us > 0 && !r->dry()) {
        const auto deadline = std::chrono::steady_clock::now() + std::chrono::microseconds(timeout_us);
        for (;;) {
            const cudaError_t q = cudaEventQuery(r->done);
            if (q == cudaSuccess) break;
            if (q != cudaErrorNotReady) return ddp::fail(DDP_E_CUDA, "%s: %s", fn, cudaGetErrorString(q));
            if (std::chrono::steady_clock::now() >= deadline)
                return ddp::fail(DDP_E_TIMEOUT, "%s: reductions still running after %lld us", fn,
                                 static_cast<long long>(timeout_us));
            std::this_thread::sleep_for(std::chrono::microseconds(20));
        }
    }
    return ddp::ok();
}

extern "C" ddp_status ddp_reducer_wait_bucket(ddp_reducer* r, int32_t bucket, void* consumer_stream)
{
    using ddp::fail;
    const char* fn = "ddp_reducer_wait_bucket";
    if (!r) return fail(DDP_E_INVAL, "%s: reducer is NULL", fn);
    if (bucket < 0 || bucket >= r->nbuckets) return fail(DDP_E_INVAL, "%s: bucket %d outside [0, %d)", fn, bucket, r->nbuckets);
    if (!(r->flags & DDP_R_BUCKET_DONE)) return fail(DDP_E_STATE, "%s: reducer built without DDP_R_BUCKET_DONE", fn);
    if (r->phase == Phase::Idle || std::find(r->log.begin(), r->log.end(), bucket) == r->log.end())
        return fail(DDP_E_STATE, "%s: bucket %d has not been issued in this iteration", fn, bucket);
    if (r->dry()) return ddp::ok();
    ddp_status st = DDP_OK;
    if (!cuda_ok(cudaStreamWaitEvent(static_cast<cudaStream_t>(consumer_stream), r->bdone[bucket], 0),
                 "cudaStreamWaitEvent", &st))
        return st;
    return ddp::ok();
}

extern "C" ddp_status ddp_reducer_issue_log(const ddp_reducer* r, int32_t* out, int32_t cap, int32_t* n)
{
    if (!r || !n) return ddp::fail(DDP_E_INVAL, "ddp_reducer_issue_log: NULL argument");
    *n = static_cast<int32_t>(r->log.size());
    if (cap < *n || (!out && *n > 0))
        return ddp::fail(DDP_E_CAPACITY, "ddp_reducer_issue_log: %d entries, room for %d", *n, cap);
    for (int32_t i = 0; i < *n; ++i) out[i] = r->log[i];
    return ddp::ok();
}

extern "C" ddp_status ddp_reducer_ready_order(const ddp_reducer* r, int32_t* out, int32_t cap, int32_t* n)
{
    if (!r || !n) return ddp::fail(DDP_E_INVAL, "ddp_reducer_ready_order: NULL argument");
    *n = static_cast<int32_t>(r->seq_last.size());
    if (*n == 0) return ddp::fail(DDP_E_STATE, "ddp_reducer_ready_order: no finalized iteration");
    if (cap < *n || !out) return ddp::fail(DDP_E_CAPACITY, "ddp_reducer_ready_order: %d entries, room for %d", *n, cap);
    for (int32_t i = 0; i < *n; ++i) out[i] = r->seq_last[i];
    return ddp::ok();
}

extern "C" ddp_status ddp_reducer_bucket_ms(ddp_reducer* r, float* out, int32_t cap)
{
    const char* fn = "ddp_reducer_bucket_ms";
    if (!r || !out) return ddp::fail(DDP_E_INVAL, "%s: NULL argument", fn);
    if (!(r->flags & DDP_R_TIMING) || r->dry()) return ddp::fail(DDP_E_STATE, "%s: reducer built without timing", fn);
    if (!r->timing_valid) return ddp::fail(DDP_E_STATE, "%s: no finalized iteration", fn);
    if (cap < r->nbuckets) return ddp::fail(DDP_E_CAPACITY, "%s: %d buckets, room for %d", fn, r->nbuckets, cap);
    ddp_status st = DDP_OK;
    for (int32_t b = 0; b < r->nbuckets; ++b) {
        if (!cuda_ok(cudaEventSynchronize(r->t_end[b]), "cudaEventSynchronize", &st)) return st;
        float ms = 0.f;
        if (!cuda_ok(cudaEventElapsedTime(&ms, r->t_begin[b], r->t_end[b]), "cudaEventElapsedTime", &st)) return st;
        out[b] = ms;
    }
    return ddp::ok();
}

extern "C" void ddp_reducer_destroy(ddp_reducer* r)
{
    if (!r) return;
    r->destroy_events();
    delete r;
}

extern "C" ddp_status ddp_copy_rows(void* dst, int64_t dst_pitch, const void* src, int64_t src_pitch,
                                    int64_t row_bytes, int64_t rows, void* stream)
{
    const char* fn = "ddp_copy_rows";
    if (row_bytes < 0 || rows < 0)
        return ddp::fail(DDP_E_INVAL, "%s: negative size (row_bytes %lld, rows %lld)", fn,
                         static_cast<long long>(row_bytes), static_cast<long long>(rows));
    if (row_bytes == 0 || rows == 0) return ddp::ok();
    if (!dst || !src) return ddp::fail(DDP_E_INVAL, "%s: NULL pointer", fn);
    if (dst_pitch < row_bytes || src_pitch < row_bytes)
        return ddp::fail(DDP_E_INVAL, "%s: pitch below the row (dst %lld, src %lld, row %lld bytes)", fn,
                         static_cast<long long>(dst_pitch), static_cast<long long>(src_pitch),
                         static_cast<long long>(row_bytes));
    ddp_status st = DDP_OK;
    if (!cuda_ok(cudaMemcpy2DAsync(dst, static_cast<size_t>(dst_pitch), src, static_cast<size_t>(src_pitch),
                                   static_cast<size_t>(row_bytes), static_cast<size_t>(rows), cudaMemcpyDefault,
                                   static_cast<cudaStream_t>(stream)),
                 "cudaMemcpy2DAsync", &st))
        return st;
    return ddp::ok();
}

// ---------------------------------------------------------------------------
// The host-buffer front end: every replica's gradients from pinned host memory
// to the device, the reducer's iteration, each reduced bucket back to pinned
// host memory -- as a pipeline over the buckets in issue order ("Megatron DDP:
// contiguous buffer and overlap" section 3: a consumer starts on a bucket as
// soon as its reduction is done).  Bucket b's copies to the device go out on
// one stream and mark its parameters ready; its copy back waits for that
// bucket alone on a second stream.  Consecutive steps overlap bucket by
// bucket: step k + 1's copies into bucket b's gradients wait for step k's
// reduction of bucket b, and its reduction of bucket b for step k's copy of
// bucket b to the host (a gate the reducer waits for when it issues b).
// ---------------------------------------------------------------------------
struct ddp_host_front {
    ddp_reducer* r = nullptr;
    uint8_t* dev_in = nullptr;
    int64_t dev_pitch = 0;
    int32_t elem = 4;
    int64_t row_elems = 0;
    struct Bucket {
        int32_t b = 0;
        std::vector<std::pair<int64_t, int64_t>> runs;   // element ranges of a row, contiguous in the host layout
        std::vector<int32_t> params;                     // in backward order (last parameter first)
    };
    std::vector<Bucket> issue;   // in issue order
    cudaStream_t h2d = nullptr, d2h = nullptr, gate = nullptr;
    std::vector<cudaEvent_t> reduced, downloaded;   // per issue position
    cudaEvent_t join = nullptr;
    bool first = true;
    std::vector<int32_t> ready;   // scratch: a bucket's parameters still to mark

    void release()
    {
        if (r)
            for (cudaEvent_t& e : r->extra_gate) e = nullptr;
        for (cudaEvent_t e : reduced)
            if (e) cudaEventDestroy(e);
        for (cudaEvent_t e : downloaded)
            if (e) cudaEventDestroy(e);
        if (join) cudaEventDestroy(join);
        if (h2d) cudaStreamDestroy(h2d);
        if (d2h) cudaStreamDestroy(d2h);
        if (gate) cudaStreamDestroy(gate);
    }
};

namespace {

// `waiter` waits for everything queued on `waited` so far
bool join_streams(cudaStream_t waiter, cudaStream_t waited, cudaEvent_t ev, ddp_status* st)
{
    return cuda_ok(cudaEventRecord(ev, waited), "cudaEventRecord", st) &&
           cuda_ok(cudaStreamWaitEvent(waiter, ev, 0), "cudaStreamWaitEvent", st);
}

}  // namespace

extern "C" ddp_status ddp_host_front_create(ddp_reducer* r, void* dev_in, int64_t dev_pitch, const int64_t* param_offset,
                                            int32_t elem_bytes, ddp_host_front** out)
{
    using ddp::fail;
    const char* fn = "ddp_host_front_create";
    if (!out) return fail(DDP_E_INVAL, "%s: out is NULL", fn);
    *out = nullptr;
    if (!r || !param_offset) return fail(DDP_E_INVAL, "%s: NULL argument", fn);
    if (r->dry()) return fail(DDP_E_INVAL, "%s: the reducer is a dry run", fn);
    if (!(r->flags & DDP_R_BUCKET_DONE)) return fail(DDP_E_INVAL, "%s: the reducer needs DDP_R_BUCKET_DONE", fn);
    if (!r->mg) return fail(DDP_E_INVAL, "%s: the reducer has no main_grad", fn);
    if (elem_bytes != 2 && elem_bytes != 4) return fail(DDP_E_INVAL, "%s: elem_bytes = %d, not 2 or 4", fn, elem_bytes);
    if (param_offset[0] != 0) return fail(DDP_E_INVAL, "%s: param_offset[0] = %lld, not 0", fn,
                                          static_cast<long long>(param_offset[0]));
    for (int32_t p = 0; p < r->nparams; ++p)
        if (param_offset[p + 1] < param_offset[p])
            return fail(DDP_E_INVAL, "%s: param_offset decreases at parameter %d", fn, p);
    const int64_t row = param_offset[r->nparams];
    if (row > 0 && !dev_in) return fail(DDP_E_INVAL, "%s: dev_in is NULL", fn);
    if (r->W > 1 && dev_pitch < row * elem_bytes)
        return fail(DDP_E_INVAL, "%s: dev_pitch %lld bytes below a row of %lld", fn, static_cast<long long>(dev_pitch),
                    static_cast<long long>(row * elem_bytes));
    auto* h = new ddp_host_front();
    auto reject = [&](ddp_status st) {
        h->release();
        delete h;
        return st;
    };
    h->r = r;
    h->dev_in = static_cast<uint8_t*>(dev_in);
    h->dev_pitch = dev_pitch;
    h->elem = elem_bytes;
    h->row_elems = row;
    std::vector<std::vector<int32_t>> members(r->nbuckets);
    for (int32_t p = 0; p < r->nparams; ++p) members[r->bucket_of[p]].push_back(p);
    for (int32_t k = 0; k < r->nbuckets; ++k) {
        ddp_host_front::Bucket B;
        B.b = r->order[k];
        const std::vector<int32_t>& mem = members[B.b];   // ascending
        for (size_t i = 0; i < mem.size();) {
            size_t j = i + 1;
            while (j < mem.size() && mem[j] == mem[j - 1] + 1) ++j;
            const int64_t lo = param_offset[mem[i]], hi = param_offset[mem[j - 1] + 1];
            if (hi > lo) B.runs.emplace_back(lo, hi);
            i = j;
        }
        B.params.assign(mem.rbegin(), mem.rend());
        h->issue.push_back(std::move(B));
    }
    ddp_status st = DDP_OK;
    if (!cuda_ok(cudaStreamCreateWithFlags(&h->h2d, cudaStreamNonBlocking), "cudaStreamCreateWithFlags", &st) ||
        !cuda_ok(cudaStreamCreateWithFlags(&h->d2h, cudaStreamNonBlocking), "cudaStreamCreateWithFlags", &st) ||
        !cuda_ok(cudaStreamCreateWithFlags(&h->gate, cudaStreamNonBlocking), "cudaStreamCreateWithFlags", &st) ||
        !cuda_ok(cudaEventCreateWithFlags(&h->join, cudaEventDisableTiming), "cudaEventCreateWithFlags", &st))
        return reject(st);
    h->reduced.assign(r->nbuckets, nullptr);
    h->downloaded.assign(r->nbuckets, nullptr);
    for (int32_t k = 0; k < r->nbuckets; ++k)
        if (!cuda_ok(cudaEventCreateWithFlags(&h->reduced[k], cudaEventDisableTiming), "cudaEventCreateWithFlags", &st) ||
            !cuda_ok(cudaEventCreateWithFlags(&h->downloaded[k], cudaEventDisableTiming), "cudaEventCreateWithFlags", &st))
            return reject(st);
    *out = h;
    return ddp::ok();
}

extern "C" ddp_status ddp_host_front_step(ddp_host_front* h, const void* host_in, int64_t host_pitch, float* host_out,
                                          void* stream)
{
    using ddp::fail;
    const char* fn = "ddp_host_front_step";
    if (!h) return fail(DDP_E_INVAL, "%s: handle is NULL", fn);
    ddp_reducer* r = h->r;
    if (h->row_elems > 0 && !host_in) return fail(DDP_E_INVAL, "%s: host_in is NULL", fn);
    if (!host_out) return fail(DDP_E_INVAL, "%s: host_out is NULL", fn);
    if (r->W > 1 && host_pitch < h->row_elems * h->elem)
        return fail(DDP_E_INVAL, "%s: host_pitch %lld bytes below a row of %lld", fn, static_cast<long long>(host_pitch),
                    static_cast<long long>(h->row_elems * h->elem));
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    ddp_status st = DDP_OK;
    const int32_t nb = r->nbuckets;
    if (h->first) {
        if (!join_streams(h->h2d, s, h->join, &st) || !join_streams(r->side, s, h->join, &st)) return st;
    } else {
        // the previous step's reduction of each bucket, taken before prepare can
        // issue this step's (its gradients may be overwritten after it)
        for (int32_t k = 0; k < nb; ++k)
            if (!cuda_ok(cudaStreamWaitEvent(h->gate, r->bdone[h->issue[k].b], 0), "cudaStreamWaitEvent", &st) ||
                !cuda_ok(cudaEventRecord(h->reduced[k], h->gate), "cudaEventRecord", &st))
                return st;
        // and each bucket's reduction waits for the previous step's copy of it to the host
        for (int32_t k = 0; k < nb; ++k) r->extra_gate[h->issue[k].b] = h->downloaded[k];
    }
    if (!join_streams(h->d2h, s, h->join, &st)) return st;
    st = ddp_reducer_prepare(r, 0);
    if (st != DDP_OK) return st;
    for (int32_t k = 0; k < nb; ++k) {
        const ddp_host_front::Bucket& B = h->issue[k];
        if (!h->first && !cuda_ok(cudaStreamWaitEvent(h->h2d, h->reduced[k], 0), "cudaStreamWaitEvent", &st)) return st;
        for (const auto& run : B.runs) {   // the W replicas' slices of a run, one pitch apart: one copy
            const int64_t bytes = (run.second - run.first) * h->elem;
            st = ddp_copy_rows(h->dev_in + run.first * h->elem, h->dev_pitch,
                               static_cast<const uint8_t*>(host_in) + run.first * h->elem, host_pitch, bytes, r->W, h->h2d);
            if (st != DDP_OK) return st;
        }
        h->ready.clear();
        for (int32_t p : B.params)   // parameters prepare marked (unused everywhere) are not marked again
            if (!r->marked[p]) h->ready.push_back(p);
        if (!h->ready.empty()) {
            st = ddp_reducer_mark_ready_many(r, h->ready.data(), static_cast<int32_t>(h->ready.size()), h->h2d);
            if (st != DDP_OK) return st;
        }
    }
    const int64_t stride = r->stride;
    for (int32_t k = 0; k < nb; ++k) {
        const int32_t b = h->issue[k].b;
        st = ddp_reducer_wait_bucket(r, b, h->d2h);
        if (st != DDP_OK) return st;
        const int64_t lo = r->start[b], n = r->buckets[b].numel;
        int64_t pitch = stride * 4, row = n * 4;
        if (r->mode == DDP_REDUCE_SCATTER) {   // replica w's shard w: elements [w n / W, (w + 1) n / W) of the bucket
            const int64_t kk = n / r->W;
            pitch = (stride + kk) * 4;
            row = kk * 4;
        }
        st = ddp_copy_rows(host_out + lo, pitch, r->mg + lo, pitch, row, r->W, h->d2h);
        if (st != DDP_OK) return st;
        if (!cuda_ok(cudaEventRecord(h->downloaded[k], h->d2h), "cudaEventRecord", &st)) return st;
    }
    st = ddp_reducer_finalize(r, stream, 0);
    if (st != DDP_OK) return st;
    if (!join_streams(s, h->d2h, h->join, &st)) return st;
    h->first = false;
    return ddp::ok();
}

extern "C" void ddp_host_front_destroy(ddp_host_front* h)
{
    if (!h) return;
    h->release();
    delete h;
}
