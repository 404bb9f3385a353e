"""CPU checks of the parity harness itself (no GPU).

The full-size parity tests take the oracle's gradient of a hot slice as the sum
of the oracle's gradients over ranges of bags (run in parallel threads).  The
gradient of L = sum_g <out[g], grad_out[g]> is a sum over bags, so the split
must reproduce the one-call oracle to float64 rounding, and the slice sampler
must always include the hottest slices of every core.
"""
import numpy as np

import oracle
from _gpu_harness import oracle_grad, sample_slices
from tt_inputs import config


def test_chunked_oracle_gradient_equals_one_call():
    wl = config(3, batch=256)
    i1, i2, i3, _ = oracle.decode(wl.tables, wl.indices, wl.offsets, wl.batch)
    for k, ik in enumerate((i1, i2, i3)):
        u, c = np.unique(ik, return_counts=True)
        sl = np.sort(u[np.argsort(-c)[:3]])
        one = oracle.workload_backward_core(wl, 0, k, sl)
        split = oracle_grad(wl, 0, k, sl, chunks=7)
        np.testing.assert_allclose(split, one, rtol=1e-11, atol=1e-14 * np.abs(one).max())


def test_table_batched_chunks():
    wl = config(5, batch=64)
    for t in (0, 7, 25):
        one = oracle.workload_backward_core(wl, t, 1)
        split = oracle_grad(wl, t, 1, np.arange(wl.tables[t].p[1]), chunks=5)
        np.testing.assert_allclose(split, one, rtol=1e-11, atol=1e-14 * max(np.abs(one).max(), 1e-300))


def test_sampler_includes_hottest_slices():
    wl = config(4, batch=512)
    dec = oracle.decode(wl.tables, wl.indices, wl.offsets, wl.batch)
    pick = sample_slices(wl, dec, np.random.default_rng(0), per_core=4, max_count=3, hot=2)
    for k in range(3):
        u, c = np.unique(dec[k], return_counts=True)
        hottest = u[np.argsort(-c, kind="stable")[:2]]
        assert set(hottest.tolist()) <= set(pick[0][k].tolist())
        assert pick[0][k].size >= 1
