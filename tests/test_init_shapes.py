"""Automatic factorisation and core initialisation (FBTT README, "Parameters":
tt_p_shapes / tt_q_shapes None, weight_dist; "Initialization").  CPU only.

* suggested_tt_shapes: prod(p) >= E, prod(q) == D, and q is the most balanced
  exact factorisation (checked against brute force over every divisor triple).
* tt_init_cores: "normal" / "uniform" cores follow the target distribution
  (Kolmogorov-Smirnov); "approx-normal" / "approx-uniform" give full-table
  entries (expanded by the float64 oracle from one-hot bags) with the target's
  mean and standard deviation; "naive-uniform" splits the target's bound evenly
  over the three cores.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
import tensor_train_compressed_embeddingbag_gb300 as tt
from tt_inputs import TableSpec


@pytest.mark.parametrize("E,D", [(10, 3), (1_000_000, 64), (40_000_000, 128), (11_000_000, 64), (120, 8),
                                 (64, 96), (7, 1), (97, 30), (5000, 17)])
def test_suggested_shapes(E, D):
    p, q = tt.suggested_tt_shapes(E, D)
    assert int(np.prod(p)) >= E and int(np.prod(q)) == D
    assert p[0] == p[1] and all(x >= 1 for x in p) and q == sorted(q)
    # brute force: no exact 3-factorisation of D has a smaller largest factor
    best = min(max(t) for t in itertools.product(range(1, D + 1), repeat=3) if t[0] * t[1] * t[2] == D)
    assert max(q) == best


def test_suggested_shapes_page_examples():
    assert tt.suggested_tt_shapes(10, 3) == ([2, 2, 3], [1, 1, 3])    # TTEmbeddingBag(10, 3, None, None, ...)
    assert tt.suggested_tt_shapes(1_000_000, 64)[1] == [4, 4, 4]      # q of the README's 1e6 x 64 example


def _full_table(spec, cores):
    return oracle.forward([spec], [[np.asarray(c, dtype=np.float64) for c in cores]],
                          np.arange(spec.num_embeddings), np.arange(spec.num_embeddings + 1))


@pytest.mark.parametrize("dist", ["normal", "uniform"])
def test_iid_cores_follow_target(dist):
    from scipy import stats
    g = torch.Generator().manual_seed(1)
    sigma = 0.3
    cores = tt.tt_init_cores([20, 30, 40], [4, 4, 4], [8, 8], dist, sigma, g)
    x = torch.cat([c.reshape(-1) for c in cores]).double().numpy()
    cdf = stats.norm(0, sigma).cdf if dist == "normal" else stats.uniform(-3 ** 0.5 * sigma, 2 * 3 ** 0.5 * sigma).cdf
    assert stats.kstest(x, cdf).pvalue > 1e-3
    assert abs(x.std() / sigma - 1) < 0.03


@pytest.mark.parametrize("dist", ["approx-normal", "approx-uniform"])
def test_approx_dists_match_full_table_moments(dist):
    g = torch.Generator().manual_seed(2)
    sigma = 0.05
    spec = TableSpec(4000, [16, 16, 16], [2, 2, 2], [16, 16])
    cores = tt.tt_init_cores(spec.p, spec.q, spec.ranks, dist, sigma, g)
    W = _full_table(spec, [c.numpy() for c in cores])
    assert abs(W.mean()) < 0.05 * sigma
    assert abs(W.std() / sigma - 1) < 0.05
    if dist == "approx-normal":
        # a single product of three normals has excess kurtosis 24; the 256 summed
        # products (which share core factors) bring the entries close to normal
        from scipy import stats
        assert abs(stats.kurtosis(W.reshape(-1))) < 2.0


def test_naive_uniform_splits_the_bound():
    g = torch.Generator().manual_seed(3)
    sigma = 0.5
    cores = tt.tt_init_cores([30, 30, 30], [2, 2, 2], [4, 4], "naive-uniform", sigma, g)
    b = (3 ** 0.5 * sigma) ** (1 / 3)
    for c in cores:
        m = float(c.abs().max())
        assert m <= b and m > 0.95 * b


def test_unknown_weight_dist_rejected():
    with pytest.raises(ValueError):
        tt.tt_init_cores([2, 2, 2], [2, 2, 2], [2, 2], "xavier")
