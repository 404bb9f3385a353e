"""GPU parity of the backward pass's optimizer modes (FBTT README,
"Parameters": sparse, optimizer, learning_rate, eps) against the float64 oracle.

* TT_OPT_GRAD (sparse=False): the gradient buffers hold dL/dG_k; every touched
  slice within the parity tolerance, every untouched slice exactly 0 (the
  buffers start filled with garbage); the cores keep their bits.
* TT_OPT_ADAGRAD: updated cores and accumulators of the touched slices within
  the tolerance; untouched slices keep their bits.  The full-size cases start
  from a warm accumulator (uniform in [0.5, 1.5]).  From a zero accumulator
  the first step is lr g / (|g| + eps): for an element whose exact gradient
  cancels to nearly 0, fp32 rounding noise in g becomes an update of order lr,
  so the cold start is compared on the tiny workload, whose gradients are all
  far from 0.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import tensor_train_compressed_embeddingbag_gb300 as tt

from _gpu_harness import (GpuRun, assert_rows_close, check_decode, check_forward, dev, oracle_grad, sample_slices,
                          touched_slices)

pytestmark = pytest.mark.gpu

EPS = 1.0e-10


def _run(wl, optim, state=None):
    """Forward + backward of `wl` under `optim`; returns (run, aux tensors, cores before, decode, forward out)."""
    run = GpuRun(wl)
    aux = None
    if optim == tt.TT_OPT_ADAGRAD:
        aux = [[dev(s.astype(np.float32)) for s in st] for st in state]
    elif optim == tt.TT_OPT_GRAD:
        aux = [[torch.full_like(c, 7.0) for c in t] for t in run.cores]
    tt.tt_emb_set_optimizer(run.h, optim, EPS, None if aux is None else [a for t in aux for a in t])
    before = run.cores_host()
    out = run.forward().cpu().numpy()
    dec = check_decode(run, wl)
    run.backward()
    assert run.error() == tt.TT_OK
    torch.cuda.synchronize()
    return run, aux, before, dec, out


def _warm_state(wl, seed):
    rng = np.random.default_rng(seed)
    return [[rng.uniform(0.5, 1.5, size=c.shape).astype(np.float32) for c in t] for t in wl.cores]


def _check_grad(wl, slices=None, bags=None, seed=0):
    run, aux, before, dec, out = _run(wl, tt.TT_OPT_GRAD)
    check_forward(out, wl, bags)
    after = run.cores_host()
    touched = touched_slices(wl, dec)
    sel = slices(wl, dec) if slices else None
    for t in range(wl.num_tables):
        for k in range(3):
            np.testing.assert_array_equal(after[t][k], before[t][k], err_msg=f"cores changed t{t} G{k + 1}")
            g = aux[t][k].cpu().numpy()
            un = np.setdiff1d(np.arange(wl.tables[t].p[k]), touched[t][k])
            assert not g[un].any(), f"untouched slices of t{t} G{k + 1} have a nonzero gradient"
            sl = touched[t][k] if sel is None else sel[t][k]
            if len(sl):
                ref = oracle_grad(wl, t, k, sl)
                assert_rows_close(g[sl], ref, f"gradient t{t} G{k + 1}")
    run.close()


def _check_adagrad(wl, state, slices=None, bags=None):
    run, aux, before, dec, out = _run(wl, tt.TT_OPT_ADAGRAD, state)
    check_forward(out, wl, bags)
    after = run.cores_host()
    touched = touched_slices(wl, dec)
    sel = slices(wl, dec) if slices else None
    for t in range(wl.num_tables):
        for k in range(3):
            st = aux[t][k].cpu().numpy()
            un = np.setdiff1d(np.arange(wl.tables[t].p[k]), touched[t][k])
            np.testing.assert_array_equal(after[t][k][un], before[t][k][un], err_msg=f"untouched t{t} G{k + 1}")
            np.testing.assert_array_equal(st[un], state[t][k][un], err_msg=f"untouched state t{t} G{k + 1}")
            sl = touched[t][k] if sel is None else sel[t][k]
            if len(sl):
                ref_g, ref_s = oracle.adagrad_update(wl.cores[t][k][sl], state[t][k][sl], oracle_grad(wl, t, k, sl),
                                                     wl.lr, EPS)
                assert_rows_close(after[t][k][sl], ref_g, f"Adagrad core t{t} G{k + 1}")
                assert_rows_close(st[sl], ref_s, f"Adagrad accumulator t{t} G{k + 1}")
    run.close()


def _sampler(seed, per_core=6, max_count=None):
    rng = np.random.default_rng(seed)
    return lambda wl, dec: sample_slices(wl, dec, rng, per_core, max_count)


def test_gradient_mode_tiny(workloads):
    _check_grad(workloads(1))


def test_gradient_mode_fbtt_sample_sampled(workloads):
    """11M x 64 rank-32, 512 bags: sampled slices; every untouched slice exactly 0."""
    _check_grad(workloads(2), slices=_sampler(1), bags=np.arange(0, 512, 7))


def test_gradient_mode_zipf_weighted_mean_full_sampled(workloads):
    """Zipf weighted mean, 4096 bags (large-path sort): gradients of the hottest,
    the coldest and random slices against the oracle."""
    _check_grad(workloads(3), slices=_sampler(11, per_core=6, max_count=2000), bags=np.arange(0, 4096, 37))


def test_gradient_mode_large_rank64_scaled(workloads):
    """40M x 128 rank 64, Zipf, 512 bags (15k lookups: the large-path sort and the
    rank-64 class): gradients compared directly, not through an update."""
    _check_grad(workloads(4, 512), slices=_sampler(12, per_core=6), bags=np.arange(0, 512, 11))


def test_gradient_mode_table_batched(workloads):
    """26 tables with ranks 16 / 32 / 64: every compiled update site."""
    _check_grad(workloads(5, 96), slices=_sampler(2, per_core=4))


def test_adagrad_tiny_cold_start(workloads):
    wl = workloads(1)
    _check_adagrad(wl, [[np.zeros(c.shape, dtype=np.float32) for c in t] for t in wl.cores])


def test_adagrad_tiny_warm(workloads):
    wl = workloads(1)
    _check_adagrad(wl, _warm_state(wl, 3))


def test_adagrad_fbtt_sample_warm_sampled(workloads):
    wl = workloads(2)
    _check_adagrad(wl, _warm_state(wl, 4), slices=_sampler(5), bags=np.arange(0, 512, 9))


def test_adagrad_table_batched_warm(workloads):
    wl = workloads(5, 96)
    _check_adagrad(wl, _warm_state(wl, 6), slices=_sampler(7, per_core=4))


def test_adagrad_large_rank64_warm_scaled(workloads):
    """40M x 128, rank 64, Zipf: the large-path sort and the rank-64 class."""
    wl = workloads(4, 512)
    _check_adagrad(wl, _warm_state(wl, 8), slices=_sampler(9, per_core=4, max_count=64))


def test_module_sparse_false_returns_gradients(workloads):
    """TTEmbeddingBag(sparse=False): autograd receives dL/dG_k, the cores stay, an external optimizer can step."""
    wl = workloads(1)
    s = wl.tables[0]
    m = tt.TTEmbeddingBag(s.num_embeddings, s.embedding_dim, s.ranks, s.p, s.q, learning_rate=wl.lr,
                          cores=[torch.from_numpy(c) for c in wl.cores[0]], sparse=False)
    out = m(dev(wl.indices), dev(wl.offsets), mode=wl.mode, include_last_offset=True)
    out.backward(dev(wl.grad_out))
    for k, c in enumerate([m.G1, m.G2, m.G3]):
        np.testing.assert_array_equal(c.detach().cpu().numpy(), wl.cores[0][k].astype(np.float32))
        assert_rows_close(c.grad.cpu().numpy(), oracle.workload_backward_core(wl, 0, k), f"grad G{k + 1}")
    opt = torch.optim.SGD(m.parameters(), lr=wl.lr)
    opt.step()
    for k, c in enumerate([m.G1, m.G2, m.G3]):
        assert_rows_close(c.detach().cpu().numpy(), oracle.workload_sgd_slices(wl, 0, k), f"external SGD G{k + 1}")


def test_module_adagrad_two_steps(workloads):
    """TTEmbeddingBag(optimizer='adagrad'): two fused steps against two oracle steps."""
    wl = workloads(1)
    s = wl.tables[0]
    m = tt.TTEmbeddingBag(s.num_embeddings, s.embedding_dim, s.ranks, s.p, s.q, learning_rate=wl.lr,
                          cores=[torch.from_numpy(c) for c in wl.cores[0]], optimizer="adagrad", eps=EPS)
    cur = [[c.astype(np.float64) for c in wl.cores[0]]]
    state = [np.zeros(c.shape) for c in wl.cores[0]]
    for _ in range(2):
        out = m(dev(wl.indices), dev(wl.offsets), mode=wl.mode, include_last_offset=True)
        out.backward(dev(wl.grad_out))
        upd = [oracle.adagrad_slices(wl.tables, cur, wl.indices, wl.offsets, wl.grad_out, wl.lr, EPS, state[k], 0, k,
                                     wl.weights, wl.mode, wl.batch) for k in range(3)]
        cur, state = [[u[0] for u in upd]], [u[1] for u in upd]
    got = [c.detach().cpu().numpy() for c in (m.G1, m.G2, m.G3)]
    for k in range(3):
        assert_rows_close(got[k], cur[0][k], f"Adagrad module G{k + 1}")
        assert_rows_close(m.adagrad_states()[k].cpu().numpy(), state[k], f"Adagrad module state G{k + 1}")


def test_set_optimizer_rejects_bad_arguments(workloads):
    run = GpuRun(workloads(1))
    lib = tt.load_library()
    ok = [torch.zeros_like(c) for c in run.cores[0]]
    arr = lambda ts: (ctypes.c_void_p * 3)(*[t.data_ptr() if isinstance(t, torch.Tensor) else t for t in ts])
    assert lib.tt_emb_set_optimizer(run.h, 3, 0.0, arr(ok)) == tt.TT_ERR_ARG
    assert lib.tt_emb_set_optimizer(run.h, tt.TT_OPT_ADAGRAD, -1.0, arr(ok)) == tt.TT_ERR_ARG
    assert lib.tt_emb_set_optimizer(run.h, tt.TT_OPT_ADAGRAD, float("nan"), arr(ok)) == tt.TT_ERR_ARG
    assert lib.tt_emb_set_optimizer(run.h, tt.TT_OPT_GRAD, 0.0, None) == tt.TT_ERR_ARG
    assert lib.tt_emb_set_optimizer(run.h, tt.TT_OPT_GRAD, 0.0, arr([ok[0], 0, ok[2]])) == tt.TT_ERR_ARG
    assert lib.tt_emb_set_optimizer(run.h, tt.TT_OPT_GRAD, 0.0, arr([ok[0], ok[1].data_ptr() + 4, ok[2]])) == tt.TT_ERR_ARG
    # a rejected call leaves the handle on SGD: one step matches the SGD oracle
    out = run.forward().cpu().numpy()
    dec = check_decode(run, run.wl)
    run.backward()
    check_forward(out, run.wl)
    from _gpu_harness import check_cores
    check_cores(run, run.wl, dec)
    run.close()
