"""The boundary from C: a C99 program that includes only include/ddp_bucket.h and
links libddpbucket.so compiles warning-free and runs the host-side entry points
(CPU only: nothing here reaches a kernel).  Its bucket assignment and plan layout
must equal the Python binding's for the same parameters."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import allreduce_ddp_assign_gb300 as D
import workloads as WL

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include "ddp_bucket.h"

int main(int argc, char** argv)
{
    int32_t n = argc - 1, nb = 0, i;
    int64_t* numels = malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    int32_t* bucket_of = malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    int64_t* offset_of = malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    int32_t* members = malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
    int32_t* dtypes = calloc((size_t)(n > 0 ? n : 1), sizeof(int32_t));   /* DDP_F32 */
    int64_t bucket_numel[256], bucket_bytes[256], bucket_start[256];
    int32_t bucket_dtype[256], bucket_order[256], member_start[257];
    ddp_plan* plan = NULL;
    ddp_plan_info info;
    ddp_status st;
    for (i = 0; i < n; ++i) numels[i] = atoll(argv[i + 1]);
    printf("version %d %s\n", ddp_version(), ddp_status_str(DDP_E_CAPACITY));
    st = ddp_assign_buckets(numels, dtypes, n, 25 << 20, 1 << 20, DDP_ORDER_REVERSE, 1, 1, bucket_of, offset_of,
                            members, bucket_numel, bucket_bytes, bucket_dtype, bucket_order, 256, &nb);
    if (st != DDP_OK) {
        printf("error %s: %s\n", ddp_status_str(st), ddp_last_error_message());
        return 1;
    }
    printf("nbuckets %d\nbucket_of", nb);
    for (i = 0; i < n; ++i) printf(" %d", bucket_of[i]);
    printf("\noffset_of");
    for (i = 0; i < n; ++i) printf(" %lld", (long long)offset_of[i]);
    printf("\n");
    st = ddp_plan_create(numels, NULL, n, 25 << 20, 1 << 20, DDP_ORDER_REVERSE, 1, 1, 64, &plan);
    if (st == DDP_OK)
        st = ddp_plan_describe(plan, &info, bucket_numel, bucket_bytes, bucket_dtype, bucket_order, bucket_start,
                               member_start, members, bucket_of, offset_of);
    if (st != DDP_OK) {
        printf("error %s: %s\n", ddp_status_str(st), ddp_last_error_message());
        return 1;
    }
    printf("replica_stride %lld\nbucket_start", (long long)info.replica_stride);
    for (i = 0; i < info.nbuckets; ++i) printf(" %lld", (long long)bucket_start[i]);
    printf("\n");
    ddp_plan_destroy(plan);
    st = ddp_bucket_allreduce(NULL, 16, 16, 2, DDP_ALLREDUCE, NULL);   /* refused on the host */
    printf("null_allreduce %s\n", ddp_status_str(st));
    free(numels);
    free(bucket_of);
    free(offset_of);
    free(members);
    free(dtypes);
    return 0;
}
"""


def test_c99_program_runs_the_host_entry_points(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from allreduce_ddp_assign_gb300 import _build

    _build.build()
    src = tmp_path / "caller.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "caller"
    libdir = os.path.dirname(D.library_path())
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(exe), "-L", libdir, "-lddpbucket", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    wl = WL.c2_resnet50()
    run = subprocess.run([str(exe)] + [str(v) for v in wl.numels], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stdout + run.stderr
    out = dict(line.split(" ", 1) for line in run.stdout.strip().splitlines())
    assert out["version"] == f"{D.ddp_version()} DDP_E_CAPACITY"
    a = D.ddp_assign_buckets(wl.numels, None, 25 << 20, 1 << 20, D.DDP_ORDER_REVERSE)
    assert int(out["nbuckets"]) == a["nbuckets"]
    assert [int(v) for v in out["bucket_of"].split()] == [int(v) for v in a["bucket_of"]]
    assert [int(v) for v in out["offset_of"].split()] == [int(v) for v in a["offset_of"]]
    h = D.ddp_plan_create(wl.numels, None, 25 << 20, 1 << 20, D.DDP_ORDER_REVERSE, 1, 1, 64)
    try:
        d = D.ddp_plan_describe(h)
    finally:
        D.ddp_plan_destroy(h)
    assert int(out["replica_stride"]) == d["replica_stride"]
    assert [int(v) for v in out["bucket_start"].split()] == [int(v) for v in np.asarray(d["bucket_start"])]
    assert out["null_allreduce"] == "DDP_E_INVAL"
