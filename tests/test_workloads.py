"""The seeded generators and shape lists (CPU only)."""
import numpy as np
import pytest

import workloads as WL


def test_shape_counts():
    # tensor and parameter counts of the published architectures
    assert (len(WL.mlp3()), sum(WL.numels(WL.mlp3()))) == (6, 199_690)
    assert (len(WL.resnet50()), sum(WL.numels(WL.resnet50()))) == (161, 25_557_032)
    assert (len(WL.gpt2_small()), sum(WL.numels(WL.gpt2_small()))) == (148, 124_439_808)
    assert (len(WL.bert_large()), sum(WL.numels(WL.bert_large()))) == (391, 335_141_888)
    wl = WL.c4_bert_large()
    assert len(wl.unused) == 16 and sum(wl.numels[p] for p in wl.unused) == 12_596_224


def test_splitmix64_reference_values():
    # splitmix64 seeded with 0: first outputs of the published generator
    ref = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    assert [int(v) for v in WL.bits_np(0, 0, 3)] == ref


@pytest.mark.parametrize("name", ["c1", "c2", "c3"])
def test_numpy_and_torch_generators_agree(name):
    wl = WL.ALL[name]()
    for p in (0, 1, wl.nparams - 1):
        a = WL.grad_raw_np(wl, p, 1)
        t = WL.grad_torch(wl, p, 1)
        b = t.view(__import__("torch").int16).numpy().view(np.uint16) if wl.dtype == WL.BF16 else t.numpy()
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
        idx = np.array([0, 3, wl.numels[p] - 1])
        assert np.array_equal(WL.grad_at_np(wl, p, 1, 0, idx), WL.grad_np(wl, p, 1)[idx])


def test_distributions():
    b = WL.bits_np(WL.stream_key(5, 0), 0, 200_000)
    d = WL.values_np(b, "dyadic12")
    assert d.min() >= -1 and d.max() <= 1 and np.all(d * 4096 == np.round(d * 4096))
    u = WL.values_np(b, "uniform")
    assert u.min() >= -1 and u.max() < 1 and abs(u.mean()) < 0.01
    z = WL.values_np(b, "normal", 1e-3)
    assert abs(z.std() / 1e-3 - 1) < 0.01 and abs(z.mean()) < 1e-5
