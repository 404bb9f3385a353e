"""GPU: trainable cache rows (FBTT README, "Parameters": sparse, where backward
gives the gradient w.r.t. the TT cores or the cache; "Software Cache": cached
rows are read without decompressing them) against the float64 oracle.

* Forward: hits read the cached values, misses the TT rows (oracle
  ``cached_forward``); checked again after a step, when the cached values no
  longer equal the TT rows.
* Backward: cached values move by the optimizer with the hits' gradient
  (``cache_grad``, ``cache_sgd``, ``cache_adagrad``), untouched slots keep their
  bits; the cores move with the misses' gradient only (plain oracle with the
  hits' weights set to 0).
* TT_OPT_GRAD: the cache gradient equals the oracle's; untouched slots read 0;
  a repeated step gives the same bits (fixed-point sums do not depend on the
  order of the hits, and the accumulators return to zero).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import tensor_train_compressed_embeddingbag_gb300 as tt

from _gpu_harness import GpuRun, assert_rows_close, check_cores, check_decode, dev, sample_slices

pytestmark = pytest.mark.gpu

EPS = 1.0e-10


def _initial_values(wl, rows, cores=None):
    """Cached values at populate time: the TT rows of the slots (0 for empty ways)."""
    s = wl.tables[0]
    live = rows >= 0
    vals = np.zeros((rows.shape[0], s.embedding_dim))
    r = rows[live]
    vals[live] = oracle.forward([s], [(cores or wl.cores)[0]], r, np.arange(r.shape[0] + 1))
    return vals


def _miss_workload(wl, rows):
    """The workload as the cores see it: every cached lookup's weight set to 0."""
    return dataclasses.replace(wl, weights=oracle.cache_miss_weights(rows, wl.indices, wl.offsets, wl.weights))


def _read(run, rows, grads=False):
    t = torch.empty((rows.shape[0], run.wl.embedding_dim), dtype=torch.float32, device="cuda")
    if grads:
        tt.tt_emb_cache_read(run.h, None, t)
    else:
        tt.tt_emb_cache_read(run.h, t)
    return t.cpu().numpy()


def _lfu_run(wl, cache_size=1024):
    """Handle with an LFU cache (set-associative) filled from one counting pass, trainable."""
    run = GpuRun(wl)
    tt.tt_emb_lfu_enable(run.h, cache_size, 1 << 14)
    run.forward()
    tt.tt_emb_lfu_populate(run.h)
    tt.tt_emb_cache_set_trainable(run.h, True)
    return run, tt.tt_emb_lfu_cached_rows(run.h)


def _rows_run(wl):
    """Handle with the workload's 110,000 hot rows cached explicitly (hash index), trainable."""
    run = GpuRun(wl)
    tt.tt_emb_cache_set_trainable(run.h, True)
    tt.tt_emb_cache_populate(run.h, dev(wl.cache_rows))
    rows = tt.tt_emb_lfu_cached_rows(run.h)
    np.testing.assert_array_equal(rows, np.sort(wl.cache_rows))
    return run, rows


@pytest.mark.parametrize("policy,batch", [("lfu", 512), ("rows", 512), ("rows", None)])
def test_two_sgd_steps(workloads, policy, batch):
    """Zipf weighted-mean workload (11M x 64, rank 32): forward, SGD step, forward; an LFU
    cache of 1024 rows or the 110,000 hot rows given explicitly; 512 bags (10k lookups,
    the small grouping path) or all 4096 bags (82k lookups, the large one)."""
    wl = workloads(3, batch)
    run, rows = _lfu_run(wl) if policy == "lfu" else _rows_run(wl)
    live = rows >= 0
    assert np.isin(wl.indices, rows[live]).mean() > 0.3
    vals0 = _initial_values(wl, rows)
    got0 = _read(run, rows)
    assert_rows_close(got0[live], vals0[live], "cached values at populate")
    out1 = run.forward().cpu().numpy()
    assert_rows_close(out1, oracle.cached_forward(wl.tables, wl.cores, rows, vals0, wl.indices, wl.offsets,
                                                  wl.weights, wl.mode), "forward 1")
    dec = check_decode(run, wl)
    run.backward()
    assert run.error() == tt.TT_OK
    d, touched = oracle.cache_grad(rows, wl.indices, wl.offsets, wl.grad_out, wl.weights, wl.mode)
    vals1 = oracle.cache_sgd(vals0, d, touched, wl.lr)
    got1 = _read(run, rows)
    assert_rows_close(got1[touched], vals1[touched], "cached values after SGD")
    np.testing.assert_array_equal(got1[~touched], got0[~touched])
    mwl = _miss_workload(wl, rows)
    rng = np.random.default_rng(1)
    check_cores(run, mwl, dec, sample_slices(wl, dec, rng, 6))
    # second forward on sampled bags: oracle cores after the step on the slices they use
    sel = np.sort(rng.choice(wl.num_bags, 12, replace=False))
    i1, i2, i3, bag = dec
    use = np.isin(bag, sel)
    cores1 = [c.astype(np.float64).copy() for c in wl.cores[0]]
    for k, ik in enumerate((i1, i2, i3)):
        sl = np.unique(ik[use])
        cores1[k][sl] = oracle.workload_sgd_slices(mwl, 0, k, sl)
    out2 = run.forward().cpu().numpy()
    ref2 = oracle.cached_forward(wl.tables, [cores1], rows, vals1, wl.indices, wl.offsets, wl.weights, wl.mode,
                                 bags=sel)
    assert_rows_close(out2[sel], ref2, "forward 2")
    run.close()


def test_gradient_mode_repeatable(workloads):
    """TT_OPT_GRAD: cache and core gradients against the oracle; the same step twice gives the same bits."""
    wl = workloads(3, 256)
    run, rows = _lfu_run(wl, 512)
    aux = [torch.full_like(c, 7.0) for c in run.cores[0]]
    tt.tt_emb_set_optimizer(run.h, tt.TT_OPT_GRAD, 0.0, aux)
    vals0 = _read(run, rows)
    grads = []
    for _ in range(2):
        run.forward()
        run.backward()
        assert run.error() == tt.TT_OK
        grads.append((_read(run, rows, grads=True), [a.cpu().numpy() for a in aux]))
    np.testing.assert_array_equal(_read(run, rows), vals0)  # the gradient mode updates nothing
    d, touched = oracle.cache_grad(rows, wl.indices, wl.offsets, wl.grad_out, wl.weights, wl.mode)
    g = grads[0][0]
    assert touched.sum() > 0
    assert_rows_close(g[touched], d[touched], "cache gradient")
    assert not g[~touched].any()
    np.testing.assert_array_equal(grads[1][0], grads[0][0])
    for k in range(3):
        np.testing.assert_array_equal(grads[1][1][k], grads[0][1][k])
    dec = oracle.decode(wl.tables, wl.indices, wl.offsets, wl.batch)
    mwl = _miss_workload(wl, rows)
    sel = sample_slices(wl, dec, np.random.default_rng(2), 6)
    for k in range(3):
        sl = sel[0][k]
        assert_rows_close(grads[0][1][k][sl], oracle.workload_backward_core(mwl, 0, k, sl), f"core gradient G{k + 1}")
    run.close()


def test_adagrad_two_steps_explicit_rows(workloads):
    """Tiny workload (generic pool path), rows cached by tt_emb_cache_populate, trainable
    before populate; two fused Adagrad steps from zero accumulators, every value checked."""
    wl = workloads(1)
    s = wl.tables[0]
    run = GpuRun(wl)
    state = [torch.zeros_like(c) for c in run.cores[0]]
    tt.tt_emb_set_optimizer(run.h, tt.TT_OPT_ADAGRAD, EPS, state)
    tt.tt_emb_cache_set_trainable(run.h, True)
    uniq = np.unique(wl.indices)
    cached = np.sort(np.concatenate([uniq[::2][:6], [s.num_embeddings - 1]]))  # the last row is never looked up
    cached = np.unique(cached)
    tt.tt_emb_cache_populate(run.h, dev(cached))
    rows = tt.tt_emb_lfu_cached_rows(run.h)
    np.testing.assert_array_equal(rows, cached)
    cores = [c.astype(np.float64) for c in wl.cores[0]]
    st = [np.zeros(c.shape) for c in cores]
    vals = _initial_values(wl, rows)
    cst = np.zeros_like(vals)
    mw = oracle.cache_miss_weights(rows, wl.indices, wl.offsets, wl.weights)
    for step in range(2):
        out = run.forward().cpu().numpy()
        assert_rows_close(out, oracle.cached_forward(wl.tables, [cores], rows, vals, wl.indices, wl.offsets,
                                                     wl.weights, wl.mode), f"forward {step}")
        run.backward()
        assert run.error() == tt.TT_OK
        upd = [oracle.adagrad_slices(wl.tables, [cores], wl.indices, wl.offsets, wl.grad_out, wl.lr, EPS, st[k], 0,
                                     k, mw, wl.mode) for k in range(3)]
        cores, st = [u[0] for u in upd], [u[1] for u in upd]
        d, touched = oracle.cache_grad(rows, wl.indices, wl.offsets, wl.grad_out, wl.weights, wl.mode)
        vals, cst = oracle.cache_adagrad(vals, cst, d, touched, wl.lr, EPS)
        got = run.cores_host()[0]
        for k in range(3):
            assert_rows_close(got[k], cores[k], f"step {step} G{k + 1}")
            assert_rows_close(state[k].cpu().numpy(), st[k], f"step {step} state {k + 1}")
        assert_rows_close(_read(run, rows), vals, f"step {step} cached values")
    run.close()


def test_module_trainable_cache_step(workloads):
    """TTEmbeddingBag(use_cache=True, cache_size, hashtbl_size): count, populate, one
    autograd step with the fused SGD update; cached values against the oracle."""
    wl = workloads(3, 256)
    s = wl.tables[0]
    m = tt.TTEmbeddingBag(s.num_embeddings, s.embedding_dim, s.ranks, s.p, s.q, learning_rate=wl.lr,
                          cores=[torch.from_numpy(c) for c in wl.cores[0]], use_cache=True, cache_size=512,
                          hashtbl_size=4096)
    args = (dev(wl.indices), dev(wl.offsets))
    kw = dict(per_sample_weights=dev(wl.weights), mode=wl.mode, include_last_offset=True)
    with torch.no_grad():
        m(*args, **kw)
    m.cache_populate()
    rows = m.cache_rows()
    vals0 = _initial_values(wl, rows)
    out = m(*args, **kw)
    assert_rows_close(out.detach().cpu().numpy(), oracle.cached_forward(
        wl.tables, wl.cores, rows, vals0, wl.indices, wl.offsets, wl.weights, wl.mode), "module forward")
    out.backward(dev(wl.grad_out))
    d, touched = oracle.cache_grad(rows, wl.indices, wl.offsets, wl.grad_out, wl.weights, wl.mode)
    got = m.cache_values().cpu().numpy()
    assert_rows_close(got[touched], oracle.cache_sgd(vals0, d, touched, wl.lr)[touched], "module cached values")


def test_trainable_cache_argument_and_state_errors(workloads):
    lib = tt.load_library()
    run = GpuRun(workloads(1))
    buf = torch.empty(64, device="cuda")
    assert lib.tt_emb_cache_set_trainable(run.h, 2, None) == tt.TT_ERR_ARG
    assert lib.tt_emb_cache_read(run.h, None, tt._ptr(buf), None) == tt.TT_ERR_STATE  # not trainable
    assert lib.tt_emb_cache_write(run.h, tt._ptr(buf), None) == tt.TT_ERR_STATE
    assert lib.tt_emb_cache_set_trainable(run.h, 1, None) == tt.TT_OK
    assert lib.tt_emb_cache_write(run.h, None, None) == tt.TT_ERR_ARG
    run.close()
    run = GpuRun(workloads(5, 8))
    assert lib.tt_emb_cache_set_trainable(run.h, 1, None) == tt.TT_ERR_STATE  # table-batched handle
    run.close()


def test_trainable_short_bags_rank32():
    """Bags of 1-3 lookups (a warp per bag; the rank-32 pool path) with the 40 most
    frequent rows trainable: three SGD steps, every output, core and cached value
    against the oracle's own chain of steps."""
    from tt_inputs import TableSpec, Workload

    rng = np.random.default_rng(21)
    spec = TableSpec(210, [6, 5, 7], [4, 4, 4], [32, 32])
    cores = [rng.normal(0, 0.3, size=sh).astype(np.float32) for sh in spec.core_shapes()]
    lengths = rng.integers(1, 4, size=300)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    idx = rng.integers(0, spec.num_embeddings, size=int(off[-1]), dtype=np.int64)
    w = rng.random(idx.shape[0], dtype=np.float32)
    go = rng.standard_normal((lengths.shape[0], spec.embedding_dim), dtype=np.float32)
    wl = Workload("short bags", [spec], [cores], idx, off, w, "mean", 0.1, lengths.shape[0], go)
    uniq, counts = np.unique(idx, return_counts=True)
    hot = np.sort(uniq[np.argsort(-counts, kind="stable")[:40]])
    run = GpuRun(wl)
    tt.tt_emb_cache_set_trainable(run.h, True)
    tt.tt_emb_cache_populate(run.h, dev(hot))
    rows = tt.tt_emb_lfu_cached_rows(run.h)
    np.testing.assert_array_equal(rows, hot)
    ref = [c.astype(np.float64) for c in cores]
    vals = _initial_values(wl, rows)
    mw = oracle.cache_miss_weights(rows, idx, off, w)
    for step in range(3):
        out = run.forward().cpu().numpy()
        assert_rows_close(out, oracle.cached_forward(wl.tables, [ref], rows, vals, idx, off, w, "mean"), f"forward {step}")
        run.backward()
        assert run.error() == tt.TT_OK
        ref = oracle.sgd_step(wl.tables, [ref], idx, off, go, wl.lr, mw, "mean")[0]
        d, touched = oracle.cache_grad(rows, idx, off, go, w, "mean")
        vals = oracle.cache_sgd(vals, d, touched, wl.lr)
        got = run.cores_host()[0]
        for k in range(3):
            assert_rows_close(got[k], ref[k], f"step {step} G{k + 1}")
        assert_rows_close(_read(run, rows), vals, f"step {step} cached values")
    run.close()


def test_cache_write_then_forward(workloads):
    """tt_emb_cache_write (an external optimizer's step on the cached values): the values
    read back bit for bit and the next forward pools them (oracle cached_forward)."""
    wl = workloads(1)
    run = GpuRun(wl)
    tt.tt_emb_cache_set_trainable(run.h, True)
    rows = np.unique(wl.indices)[::3]
    tt.tt_emb_cache_populate(run.h, dev(rows))
    vals = np.random.default_rng(3).standard_normal((rows.shape[0], wl.embedding_dim)).astype(np.float32)
    tt.tt_emb_cache_write(run.h, dev(vals))
    np.testing.assert_array_equal(_read(run, rows), vals)
    out = run.forward().cpu().numpy()
    assert_rows_close(out, oracle.cached_forward(wl.tables, wl.cores, rows, vals, wl.indices, wl.offsets,
                                                 wl.weights, wl.mode), "forward after write")
    run.close()
