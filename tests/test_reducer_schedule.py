"""The reducer's schedule (pending counts, in-order issue, errors) on the host,
in dry-run mode: no CUDA call is made (CPU only)."""
import pytest

import allreduce_ddp_assign_gb300 as D


def make(bucket_of, order=None, nb=None):
    nb = nb if nb is not None else max(bucket_of) + 1
    order = list(range(nb)) if order is None else order
    descs = [D.BucketDesc(8, 0, 0, None, None) for _ in range(nb)]
    return D.ddp_reducer_create(len(bucket_of), bucket_of, order, descs, [0] * nb, 2, D.DDP_ALLREDUCE,
                                D.DDP_R_DRY_RUN | D.DDP_R_FUSED, replica_stride=8)


def test_in_order_issue_when_ready_out_of_order():
    # params 0,1 -> bucket 0; 2 -> bucket 1; 3,4 -> bucket 2 (lecture, section 2.3)
    r = make([0, 0, 1, 2, 2])
    D.ddp_reducer_prepare(r)
    for p in (3, 4):             # bucket 2 fills first: nothing may be issued
        D.ddp_reducer_mark_ready(r, p)
    assert D.ddp_reducer_issue_log(r) == []
    D.ddp_reducer_mark_ready(r, 2)        # bucket 1 ready, bucket 0 still pending
    assert D.ddp_reducer_issue_log(r) == []
    D.ddp_reducer_mark_ready(r, 0)
    assert D.ddp_reducer_issue_log(r) == []
    D.ddp_reducer_mark_ready(r, 1)        # bucket 0 completes: 0, 1, 2 go out in order
    assert D.ddp_reducer_issue_log(r) == [0, 1, 2]
    D.ddp_reducer_finalize(r)
    D.ddp_reducer_destroy(r)


def test_issue_as_soon_as_prefix_ready():
    r = make([0, 1, 2])
    D.ddp_reducer_prepare(r)
    D.ddp_reducer_mark_ready(r, 0)
    assert D.ddp_reducer_issue_log(r) == [0]
    D.ddp_reducer_mark_ready(r, 1)
    assert D.ddp_reducer_issue_log(r) == [0, 1]
    D.ddp_reducer_mark_ready(r, 2)
    D.ddp_reducer_finalize(r)
    D.ddp_reducer_destroy(r)


def test_megatron_issue_order_is_last_to_first():
    plan = D.ddp_assign_buckets([10] * 6, None, 80, 80, D.DDP_ORDER_MEGATRON)
    assert plan["nbuckets"] == 3
    r = make(plan["bucket_of"], list(plan["bucket_order"]))
    D.ddp_reducer_prepare(r)
    for p in range(5, -1, -1):  # backward produces the last parameters first
        D.ddp_reducer_mark_ready(r, p)
    assert D.ddp_reducer_issue_log(r) == [2, 1, 0]
    D.ddp_reducer_finalize(r)
    D.ddp_reducer_destroy(r)


def test_double_mark_is_a_state_error():
    r = make([0, 0])
    D.ddp_reducer_prepare(r)
    D.ddp_reducer_mark_ready(r, 1)
    with pytest.raises(D.DdpError) as e:
        D.ddp_reducer_mark_ready(r, 1)
    assert e.value.status == D.DDP_E_STATE and "parameter 1" in str(e.value)
    D.ddp_reducer_destroy(r)


def test_missing_mark_reported_at_finalize_and_next_prepare():
    r = make([0, 0, 1, 1])
    D.ddp_reducer_prepare(r)
    D.ddp_reducer_mark_ready(r, 0)
    D.ddp_reducer_mark_ready(r, 1)
    with pytest.raises(D.DdpError) as e:
        D.ddp_reducer_finalize(r)
    assert e.value.status == D.DDP_E_INCOMPLETE and e.value.args[0].endswith(": 2 3")
    with pytest.raises(D.DdpError) as e:            # next iteration starts: same complaint
        D.ddp_reducer_prepare(r)
    assert e.value.status == D.DDP_E_INCOMPLETE and "2 3" in str(e.value)
    # the reducer was reset anyway: a full iteration now works
    for p in range(4):
        D.ddp_reducer_mark_ready(r, p)
    D.ddp_reducer_finalize(r)
    assert D.ddp_reducer_issue_log(r) == [0, 1]
    D.ddp_reducer_destroy(r)


def test_mark_outside_iteration_and_bad_index():
    r = make([0])
    with pytest.raises(D.DdpError) as e:
        D.ddp_reducer_mark_ready(r, 0)
    assert e.value.status == D.DDP_E_STATE
    D.ddp_reducer_prepare(r)
    with pytest.raises(D.DdpError) as e:
        D.ddp_reducer_mark_ready(r, 7)
    assert e.value.status == D.DDP_E_INVAL
    D.ddp_reducer_destroy(r)


def test_create_validation():
    descs = [D.BucketDesc(8, 0, 0, None, None)]
    with pytest.raises(D.DdpError):    # bucket_of points past the buckets
        D.ddp_reducer_create(2, [0, 1], [0], descs, [0], 2, 0, D.DDP_R_DRY_RUN, replica_stride=8)
    with pytest.raises(D.DdpError):    # order not a permutation
        D.ddp_reducer_create(2, [0, 1], [1, 1], descs * 2, [0, 0], 2, 0, D.DDP_R_DRY_RUN, replica_stride=8)
    with pytest.raises(D.DdpError):    # a bucket without parameters
        D.ddp_reducer_create(2, [0, 0], [0, 1], descs * 2, [0, 0], 2, 0, D.DDP_R_DRY_RUN, replica_stride=8)
    with pytest.raises(D.DdpError):    # reduce_scatter needs numel % W == 0
        D.ddp_reducer_create(1, [0], [0], [D.BucketDesc(7, 0, 0, None, None)], [0], 2, 1, D.DDP_R_DRY_RUN,
                             replica_stride=8)
    with pytest.raises(D.DdpError):    # bucket past the replica stride
        D.ddp_reducer_create(1, [0], [0], descs, [4], 2, 0, D.DDP_R_DRY_RUN, replica_stride=8)
    with pytest.raises(D.DdpError):    # coalescing is a property of the fused issue
        D.ddp_reducer_create(1, [0], [0], descs, [0], 2, 0, D.DDP_R_DRY_RUN | D.DDP_R_COALESCE, replica_stride=8)


def test_repeated_iterations_and_timing_refused_in_dry_run():
    r = make([0, 1, 1])
    for _ in range(3):
        D.ddp_reducer_prepare(r)
        for p in (2, 1, 0):
            D.ddp_reducer_mark_ready(r, p)
        D.ddp_reducer_finalize(r)
        assert D.ddp_reducer_issue_log(r) == [0, 1]
    with pytest.raises(D.DdpError) as e:
        D.ddp_reducer_bucket_ms(r, 2)
    assert e.value.status == D.DDP_E_STATE
    D.ddp_reducer_destroy(r)


def test_coalesced_issue_order_dry_run():
    """Coalescing changes how many launches go out, not the order of buckets."""
    nb = 4
    descs = [D.BucketDesc(8, 0, 0, None, None) for _ in range(nb)]
    r = D.ddp_reducer_create(4, [0, 1, 2, 3], [0, 1, 2, 3], descs, [0] * nb, 2, D.DDP_ALLREDUCE,
                             D.DDP_R_DRY_RUN | D.DDP_R_FUSED | D.DDP_R_COALESCE, replica_stride=8)
    D.ddp_reducer_prepare(r)
    D.ddp_reducer_mark_ready_many(r, [3, 2, 1])
    assert D.ddp_reducer_issue_log(r) == []
    D.ddp_reducer_mark_ready(r, 0)
    assert D.ddp_reducer_issue_log(r) == [0, 1, 2, 3]
    D.ddp_reducer_finalize(r)
    D.ddp_reducer_destroy(r)


def test_mark_many_outside_iteration_issues_nothing():
    r = make([0, 1])
    with pytest.raises(D.DdpError) as e:
        D.ddp_reducer_mark_ready_many(r, [1, 0])
    assert e.value.status == D.DDP_E_STATE
    assert D.ddp_reducer_issue_log(r) == []
    D.ddp_reducer_prepare(r)
    D.ddp_reducer_mark_ready_many(r, [1, 0])
    assert D.ddp_reducer_issue_log(r) == [0, 1]
    D.ddp_reducer_finalize(r)
    D.ddp_reducer_destroy(r)


def test_mark_many_stops_at_the_duplicate_but_issues_completed_buckets():
    r = make([0, 1, 1])
    D.ddp_reducer_prepare(r)
    with pytest.raises(D.DdpError) as e:
        D.ddp_reducer_mark_ready_many(r, [0, 0, 1])
    assert e.value.status == D.DDP_E_STATE
    assert D.ddp_reducer_issue_log(r) == [0]      # bucket 0 was complete before the duplicate
    D.ddp_reducer_mark_ready_many(r, [1, 2])
    assert D.ddp_reducer_issue_log(r) == [0, 1]
    D.ddp_reducer_finalize(r)
    D.ddp_reducer_destroy(r)


def test_ready_order_recorded_for_rebuild():
    """The reducer keeps the order gradients arrived in; re-bucketing over it puts the
    first arrivals in bucket 0 (DDP chapter 17.13)."""
    r = make([0, 0, 1, 1, 2])
    with pytest.raises(D.DdpError) as e:
        D.ddp_reducer_ready_order(r)
    assert e.value.status == D.DDP_E_STATE
    D.ddp_reducer_prepare(r)
    order = [4, 2, 3, 0, 1]
    for p in order:
        D.ddp_reducer_mark_ready(r, p)
    D.ddp_reducer_finalize(r)
    assert D.ddp_reducer_ready_order(r) == order
    plan = D.ddp_assign_buckets_ordered([10, 10, 10, 10, 10], order, None, 80, 40)
    assert [int(p) for p in plan["members"]][:1] == [4]
    D.ddp_reducer_destroy(r)


# ---------------------------------------------------------------------------
# find_unused_parameters (dry run: the host side of the bitmap path)
# ---------------------------------------------------------------------------
def make_fu(bucket_of, W=2, **kw):
    nb = max(bucket_of) + 1
    descs = [D.BucketDesc(8, 0, 0, None, None) for _ in range(nb)]
    return D.ddp_reducer_create(len(bucket_of), bucket_of, list(range(nb)), descs, [0] * nb, W, D.DDP_ALLREDUCE,
                                D.DDP_R_DRY_RUN | D.DDP_R_FUSED, replica_stride=8, ld=len(bucket_of), **kw)


def test_find_unused_marks_parameters_no_replica_used():
    """Lecture 15 section 4.2: parameters nobody used are marked ready at the start of
    the backward, so a bucket made only of them goes out at once and the others
    complete without their marks; a parameter one replica used still needs its mark."""
    r = make_fu([0, 0, 1, 2, 2])
    D.ddp_reducer_find_unused(r, None, None)
    D.ddp_reducer_set_local_used(r, [[1, 0, 0, 1, 0], [1, 0, 0, 0, 0]])
    D.ddp_reducer_prepare(r)
    assert D.ddp_reducer_issue_log(r) == []          # bucket 0 still waits for parameter 0
    D.ddp_reducer_mark_ready(r, 3)                    # used by replica 0 only
    D.ddp_reducer_mark_ready(r, 0)                    # bucket 0, then 1 (p2 unused) and 2 (p4 unused)
    assert D.ddp_reducer_issue_log(r) == [0, 1, 2]
    D.ddp_reducer_finalize(r)
    # an automatically marked parameter marked again is the double-mark error
    D.ddp_reducer_set_local_used(r, [[1, 1, 1, 1, 0], [1, 1, 1, 1, 0]])
    D.ddp_reducer_prepare(r)
    with pytest.raises(D.DdpError, match="twice"):
        D.ddp_reducer_mark_ready(r, 4)
    D.ddp_reducer_destroy(r)


def test_find_unused_all_unused_bucket_issued_at_prepare():
    r = make_fu([0, 1, 1])
    D.ddp_reducer_find_unused(r, None, None)
    D.ddp_reducer_set_local_used(r, [[0, 1, 1], [0, 0, 1]])
    D.ddp_reducer_prepare(r)
    assert D.ddp_reducer_issue_log(r) == [0]
    D.ddp_reducer_mark_ready_many(r, [2, 1])
    assert D.ddp_reducer_issue_log(r) == [0, 1]
    D.ddp_reducer_finalize(r)
    # the ready order seen by a rebuild starts with the parameters marked at prepare
    assert D.ddp_reducer_ready_order(r) == [0, 2, 1]
    D.ddp_reducer_destroy(r)


def test_find_unused_default_bitmap_is_all_used():
    r = make_fu([0, 1])
    D.ddp_reducer_find_unused(r, None, None)
    D.ddp_reducer_prepare(r)
    assert D.ddp_reducer_issue_log(r) == []
    D.ddp_reducer_mark_ready_many(r, [1, 0])
    assert D.ddp_reducer_issue_log(r) == [0, 1]
    D.ddp_reducer_finalize(r)
    D.ddp_reducer_destroy(r)


def test_find_unused_state_and_argument_errors():
    r = make_fu([0, 1])
    with pytest.raises(D.DdpError, match="find_unused is off"):
        D.ddp_reducer_set_local_used(r, [[1, 1], [1, 1]])
    D.ddp_reducer_find_unused(r, None, None)
    with pytest.raises(D.DdpError, match="already on"):
        D.ddp_reducer_find_unused(r, None, None)
    with pytest.raises(D.DdpError, match="ld = 1 < nparams = 2"):
        D.ddp_reducer_set_local_used(r, [[1], [1]])
    D.ddp_reducer_prepare(r)
    with pytest.raises(D.DdpError, match="inside an iteration"):
        D.ddp_reducer_set_local_used(r, [[1, 1], [1, 1]])
    D.ddp_reducer_destroy(r)
    r = make_fu([0, 1], global_used=0x1000)   # dry run: the address is never dereferenced
    with pytest.raises(D.DdpError, match="its own global_used"):
        D.ddp_reducer_find_unused(r, None, None)
    D.ddp_reducer_destroy(r)


def test_used_allreduce_validation_without_launch():
    """Argument errors are found on the host, before anything is launched; an empty
    bitmap launches nothing (so this runs without a GPU)."""
    with pytest.raises(D.DdpError, match="W = 0"):
        D.ddp_used_allreduce(None, 4, 0, 4, None, 0x1000, stream=0)
    with pytest.raises(D.DdpError, match="W = 65"):
        D.ddp_used_allreduce(None, 4, 65, 4, None, 0x1000, stream=0)
    with pytest.raises(D.DdpError, match="ld = 3 < nparams = 4"):
        D.ddp_used_allreduce(0x1000, 3, 2, 4, None, 0x1000, stream=0)
    with pytest.raises(D.DdpError, match="both outputs"):
        D.ddp_used_allreduce(0x1000, 4, 2, 4, None, None, stream=0)
    with pytest.raises(D.DdpError, match="local_used is NULL"):
        D.ddp_used_allreduce(None, 4, 2, 4, None, 0x1000, stream=0)
    D.ddp_used_allreduce(None, 0, 2, 0, None, 0x1000, stream=0)


def test_wait_bucket_needs_flag_and_issue():
    descs = [D.BucketDesc(8, 0, 0, None, None) for _ in range(2)]
    r = D.ddp_reducer_create(2, [0, 1], [0, 1], descs, [0, 0], 2, D.DDP_ALLREDUCE,
                             D.DDP_R_DRY_RUN | D.DDP_R_FUSED | D.DDP_R_BUCKET_DONE, replica_stride=8)
    D.ddp_reducer_prepare(r)
    D.ddp_reducer_mark_ready(r, 0)
    D.ddp_reducer_wait_bucket(r, 0)
    with pytest.raises(D.DdpError, match="not been issued"):
        D.ddp_reducer_wait_bucket(r, 1)
    with pytest.raises(D.DdpError, match="outside"):
        D.ddp_reducer_wait_bucket(r, 2)
    D.ddp_reducer_destroy(r)
    r = make([0, 1])
    D.ddp_reducer_prepare(r)
    D.ddp_reducer_mark_ready(r, 0)
    with pytest.raises(D.DdpError, match="DDP_R_BUCKET_DONE"):
        D.ddp_reducer_wait_bucket(r, 0)
    D.ddp_reducer_destroy(r)
