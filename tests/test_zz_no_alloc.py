"""ddp_powersgd_reduce_static: the PowerSGD hook with its scratch in the library's
fixed device array, against ddp_powersgd_reduce (caller workspace) on the same
inputs.  Same kernels, same order: the two must agree bit for bit."""
import numpy as np
import pytest

import allreduce_ddp_assign_gb300 as D
import workloads as WL


def _plan(W, rank):
    shapes = [(64, 3, 7, 7), (8,), (256, 64), (3, 5), (130, 2, 3), (512, 64), (40,)]
    offs, pos = [], 0
    for s in shapes:
        pos = -(-pos // 4) * 4
        offs.append(pos)
        pos += int(np.prod(s))
    numel = pos + 4
    q0 = [None if len(s) < 2 else WL.powersgd_q0_np(31, t, int(np.prod(s[1:])), min(rank, s[0], int(np.prod(s[1:]))))
          for t, s in enumerate(shapes)]
    return shapes, offs, numel, q0


@pytest.mark.gpu
def test_static_scratch_matches_workspace_two_calls_in_a_row():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():  # pragma: no cover
        pytest.skip("no CUDA device")
    from allreduce_ddp_assign_gb300.powersgd import PowerSGDBucket

    dev = torch.device("cuda:0")
    W, rank = 4, 4
    shapes, offs, numel, q0 = _plan(W, rank)
    seg_numel = [int(np.prod(s)) for s in shapes]
    a = PowerSGDBucket(W, rank, offs, seg_numel, shapes, numel, lambda k, n, r: q0[k])
    b = PowerSGDBucket(W, rank, offs, seg_numel, shapes, numel, lambda k, n, r: q0[k])
    rng = np.random.default_rng(8)
    for call in range(2):
        host = rng.standard_normal((W, numel)).astype(np.float32)
        xa = torch.from_numpy(host).to(dev)
        xb = torch.from_numpy(host).to(dev)
        a.reduce(xa, numel)
        D.ddp_powersgd_reduce_static(b.handle, xb, numel)
        torch.cuda.synchronize()
        assert torch.equal(xa.view(torch.int32), xb.view(torch.int32)), f"call {call}: outputs differ"
        assert torch.equal(a.q_state.view(torch.int32), b.q_state.view(torch.int32)), f"call {call}: Q differs"
        assert torch.equal(a.error.view(torch.int32), b.error.view(torch.int32)), f"call {call}: error differs"
    assert b.iteration == 2
    a.close()
    b.close()


def test_static_scratch_rejects_oversized_bucket():
    """A 65536 x 4096 matrix needs far more than the 8 MiB array: refused on the host
    before anything is launched.  main_grad is a placeholder address that nothing may
    touch, so the state is made to compress from its first call (start_iter = 0: no
    plain warm-up all-reduce would run on it) and is never bound (the compressed path
    has no tables to launch with); the size check comes first all the same."""
    h = D.ddp_powersgd_create(8, 4, [0], [65536 * 4096], [65536], 65536 * 4096, error_feedback=1, start_iter=0)
    with pytest.raises(D.DdpError, match="static array holds 8388608") as e:
        D.ddp_powersgd_reduce_static(h, 0x1000, 65536 * 4096, stream=0)
    assert e.value.status == D.DDP_E_CAPACITY
    assert D.ddp_powersgd_iter(h) == 0
    D.ddp_powersgd_destroy(h)
