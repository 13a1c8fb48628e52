"""Host-side checks of the PowerSGD hook's C ABI: planning and argument errors
(no CUDA call is made, CPU only)."""
import pytest

import allreduce_ddp_assign_gb300 as D


def test_powersgd_plan_sizes_and_layout():
    # a 64 x 147 conv weight, a 1-D tensor, a 3 x 5 matrix clamped to rank 3
    h = D.ddp_powersgd_create(4, 4, [0, 9408, 9416], [9408, 8, 15], [64, 0, 3], 9432)
    sz = D.ddp_powersgd_sizes(h)
    assert sz["nmatrices"] == 2
    m0 = D.ddp_powersgd_matrix(h, 0)
    assert (m0["rows"], m0["cols"], m0["rank_eff"], m0["rank_pad"]) == (64, 147, 4, 4)
    m2 = D.ddp_powersgd_matrix(h, 2)
    assert (m2["rows"], m2["cols"], m2["rank_eff"], m2["rank_pad"]) == (3, 5, 3, 4)
    assert m2["q_offset"] >= 147 * 4 and m2["q_offset"] % 4 == 0
    assert sz["q_elems"] >= m2["q_offset"] + 5 * 4
    assert sz["workspace_bytes"] % 256 == 0 and sz["workspace_bytes"] > 0
    D.ddp_powersgd_destroy(h)


def test_powersgd_validation():
    with pytest.raises(D.DdpError, match="rank = 9"):
        D.ddp_powersgd_create(2, 9, [0], [4], [2], 4)
    with pytest.raises(D.DdpError, match="not 3 rows"):
        D.ddp_powersgd_create(2, 2, [0], [4], [3], 4)
    with pytest.raises(D.DdpError, match="outside the bucket"):
        D.ddp_powersgd_create(2, 2, [2], [4], [2], 5)
    h = D.ddp_powersgd_create(2, 2, [0, 4], [4, 3], [2, 0], 8)
    with pytest.raises(D.DdpError, match="bind first"):
        D.ddp_powersgd_reduce(h, 0x1000, 8)
    with pytest.raises(D.DdpError, match="1-D"):
        D.ddp_powersgd_matrix(h, 1)
    D.ddp_powersgd_destroy(h)
