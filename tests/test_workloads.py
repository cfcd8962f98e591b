"""The seeded synthetic workloads against their stated recipe: value distributions (zeros,
outliers, Laplace / Gaussian scale), the ResNet-152 and BERT-Large shape sets, counter-based
determinism (any sub-range equals the same slice of a full draw), and distinct rank streams."""
import numpy as np

import workloads as wl


def test_headline_bucket_values():
    """Laplace(0, 1e-4) with 30 % exact zeros and 0.1 % of the nonzero values multiplied by 100."""
    n = 2_000_000
    x = wl.fill(2, 0, 0, n).astype(np.float64)
    zero = x == 0.0
    assert abs(zero.mean() - 0.30) < 0.003
    nz = np.abs(x[~zero])
    # |Laplace(0, b)| is exponential with mean b: the non-outlier bulk sets the median b * ln 2
    assert abs(np.median(nz) / (1e-4 * np.log(2)) - 1.0) < 0.01
    # outliers: |x| > 5e-3 is out of reach of the bulk (e^-50) and holds e^-0.5 of the x100 values
    frac = (nz > 5e-3).mean() / np.exp(-0.5)
    assert 0.0007 < frac < 0.0013


def test_small_workload_gaussian():
    x = wl.fill(1, 1, 0, 262144).astype(np.float64)
    assert abs(x.std() / 1e-3 - 1.0) < 0.01
    assert abs(x.mean()) < 1e-5


def test_counter_based_and_rank_streams():
    full = wl.fill(2, 3, 0, 100_000)
    for i0, i1 in ((0, 1), (17, 4099), (65_536, 100_000), (99_999, 100_000)):
        assert np.array_equal(wl.fill(2, 3, i0, i1).view(np.uint32), full[i0:i1].view(np.uint32))
    other = wl.fill(2, 4, 0, 100_000)
    assert not np.array_equal(full, other)


def test_resnet_shape_set():
    sizes, sig = wl.tensor_layout(3)
    assert int(sizes.sum()) == 60_192_808
    assert sizes.min() >= 1 and sizes[:-1].min() >= 64 and sizes.max() <= 2_359_296
    assert 150 <= len(sizes) <= 350
    assert np.all((sig >= 1e-6 * 0.999) & (sig <= 1e-2 * 1.001))


def test_bert_shape_set_and_fp16_values():
    sizes, sig = wl.tensor_layout(4)
    assert int(sizes.sum()) == 335_141_888
    # the embedding table (30,522 x 1024) and the 24 layers' 1024 x 1024 attention matrices
    assert 30522 * 1024 in set(int(s) for s in sizes)
    assert sum(1 for s in sizes if int(s) == 1024 * 1024) >= 24 * 4
    x = wl.fill(4, 0, 0, 1_000_000)
    assert x.dtype == np.float16 and np.all(np.isfinite(x))
