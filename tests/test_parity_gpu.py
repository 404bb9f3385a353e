"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Small cases are compared element by element on every bag and every touched
core slice; the full-size workloads on sampled bags and slices, plus the
properties that hold at any size (decode bit-exact, untouched slices keep
their bits).  Scaled-down cases keep each workload's distributions and table
shapes and still span many tiles and ragged tails.
"""
import numpy as np
import pytest
import torch

import oracle
import tensor_train_compressed_embeddingbag_gb300 as tt
from tt_inputs import TableSpec, Workload, config

from _gpu_harness import (
    GpuRun,
    assert_rows_close,
    check_cores,
    check_decode,
    check_forward,
    dev,
    sample_slices,
)

pytestmark = pytest.mark.gpu


def full_parity(wl, cache=False):
    run = GpuRun(wl, cache=cache)
    out = run.forward().cpu().numpy()
    dec = check_decode(run, wl)
    run.backward()
    assert run.error() == tt.TT_OK
    check_forward(out, wl)
    check_cores(run, wl, dec)
    run.close()


def sampled_parity(wl, nbags=256, per_core=6, max_count=None, cache=False, seed=0):
    rng = np.random.default_rng(seed)
    run = GpuRun(wl, cache=cache)
    out = run.forward().cpu().numpy()
    dec = check_decode(run, wl)
    run.backward()
    assert run.error() == tt.TT_OK
    bags = np.unique(np.concatenate([[0, wl.num_bags - 1], rng.choice(wl.num_bags, nbags, replace=False)]))
    check_forward(out, wl, bags)
    check_cores(run, wl, dec, sample_slices(wl, dec, rng, per_core, max_count))
    run.close()


def test_tiny_workload(workloads):
    full_parity(workloads(1))


def test_fbtt_sample_workload_full(workloads):
    """11M x 64 rank-32, 512 bags x 20 uniform lookups: every bag and slice."""
    full_parity(workloads(2))


@pytest.mark.parametrize("batch", [64, 512])
def test_zipf_weighted_mean_scaled(workloads, batch):
    full_parity(workloads(3, batch))


def test_zipf_weighted_mean_full_sampled(workloads):
    sampled_parity(workloads(3), nbags=256, per_core=6, max_count=2000)


def test_large_rank64_scaled(workloads):
    full_parity(workloads(4, 256))


def test_large_rank64_full_sampled(workloads):
    sampled_parity(workloads(4), nbags=48, per_core=4, max_count=3000)


def test_table_batched_scaled(workloads):
    full_parity(workloads(5, 384))


def test_table_batched_full_sampled(workloads):
    sampled_parity(workloads(5), nbags=256, per_core=2, max_count=2000)


@pytest.mark.parametrize("batch", [64, 4096])
def test_cache_gives_same_results(workloads, batch):
    """With the hot-row cache (Zipf, weighted mean), two steps match the oracle (at 64 bags
    the oracle's own cores after each step, every bag and slice) and the run without cache."""
    wl = workloads(3, batch)
    run = GpuRun(wl, cache=True)
    ref_run = GpuRun(wl, cache=False)
    ref_cores = [c.astype(np.float64) for c in wl.cores[0]]
    for step in range(2):
        out = run.forward().cpu().numpy()
        ref = ref_run.forward().cpu().numpy()
        dec = check_decode(run, wl)
        run.backward()
        ref_run.backward()
        assert run.error() == tt.TT_OK and ref_run.error() == tt.TT_OK
        assert_rows_close(out, ref, f"cache vs no cache, step {step}")
        if batch <= 64:
            assert_rows_close(out, oracle.workload_forward(wl, cores=[ref_cores]), f"forward, step {step}")
        else:
            bags = np.random.default_rng(step).choice(wl.num_bags, 128, replace=False)
            assert_rows_close(out[bags], oracle.workload_forward(wl, bags=bags, cores=[ref_cores]), f"forward, step {step}")
        ref_cores = oracle.sgd_step(wl.tables, [ref_cores], wl.indices, wl.offsets, wl.grad_out, wl.lr,
                                    wl.weights, wl.mode)[0]
        got = run.cores_host()[0]
        for k in range(3):
            assert_rows_close(got[k], ref_cores[k], f"step {step} G{k + 1}")
    run.close()
    ref_run.close()


# ---------------------------------------------------------------- edge cases


def synthetic(p, q, r, lengths, seed=0, E=None, weights=False, mode="sum", lr=0.1, dist="uniform"):
    rng = np.random.default_rng(seed)
    E = E or int(np.prod(p))
    spec = TableSpec(E, list(p), list(q), list(r))
    cores = [rng.normal(0, 0.3, size=s).astype(np.float32) for s in spec.core_shapes()]
    lengths = np.asarray(lengths, dtype=np.int64)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    nnz = int(off[-1])
    if dist == "uniform":
        idx = rng.integers(0, E, size=nnz, dtype=np.int64)
    else:  # few distinct rows: long runs of equal (i1, i2) pairs and rows
        idx = rng.choice(rng.integers(0, E, size=5), size=nnz).astype(np.int64)
    w = rng.random(nnz, dtype=np.float32) if weights else None
    go = rng.standard_normal((lengths.shape[0], spec.embedding_dim), dtype=np.float32)
    return Workload("synthetic", [spec], [cores], idx, off, w, mode, lr, lengths.shape[0], go)


def test_empty_and_single_bags():
    full_parity(synthetic([4, 5, 6], [2, 2, 2], [4, 4], [0, 1, 0, 3, 1, 0, 0, 7, 1], weights=True, mode="mean"))


def test_groups_span_many_tiles():
    """p2 = 2: two (i2) groups of ~1000 lookups, each cut into several tiles;
    pairs and rows split across tile boundaries."""
    rng = np.random.default_rng(1)
    full_parity(synthetic([3, 2, 5], [2, 2, 2], [3, 5], rng.integers(0, 9, size=400), seed=1, weights=True))


@pytest.mark.parametrize("r", [16, 32])
def test_tensor_core_groups_span_many_tiles(r):
    """The tensor-core backward (q = [4, 4, 4], r1 = r2 = 16 or 32) with p2 = 3: three
    (i2) groups of ~300 lookups, each cut into several 64-lookup tiles of up to four
    batches of pairs, tiles launched longest first, every group's dG2 summed by its
    last tile; uniform rows and few distinct rows (long runs of one pair)."""
    rng = np.random.default_rng(11)
    lengths = rng.integers(1, 16, size=110)
    full_parity(synthetic([40, 3, 30], [4, 4, 4], [r, r], lengths, seed=11, weights=True))
    full_parity(synthetic([40, 3, 30], [4, 4, 4], [r, r], lengths, seed=12, dist="few", mode="mean"))


def test_repeated_rows_span_tiles():
    rng = np.random.default_rng(2)
    full_parity(synthetic([7, 3, 4], [2, 4, 1], [6, 2], rng.integers(1, 30, size=100), seed=2, dist="few"))


@pytest.mark.parametrize("q,r", [([1, 1, 1], [1, 1]), ([3, 1, 5], [2, 7]), ([4, 4, 8], [16, 64]), ([2, 8, 4], [64, 8])])
def test_odd_shapes(q, r):
    rng = np.random.default_rng(3)
    full_parity(synthetic([5, 7, 3], q, r, rng.integers(0, 6, size=40), seed=3, E=100, weights=True))


@pytest.mark.parametrize("q,r", [([2, 2, 2], [4, 4]), ([4, 4, 4], [32, 32])])
def test_cache_short_bags(q, r):
    """Bags of 1-3 lookups (a warp per bag in the pool; generic and rank-32 paths) with the
    exact-copy cache of the 40 most frequent rows: three SGD steps, each checked twice
    (stale rows refreshed, then read fresh) against the oracle's own chain of steps."""
    rng = np.random.default_rng(5)
    wl = synthetic([6, 5, 7], q, r, rng.integers(1, 4, size=300), seed=5, weights=True, mode="mean")
    rows, counts = np.unique(wl.indices, return_counts=True)
    hot = rows[np.argsort(-counts, kind="stable")[:40]]
    run = GpuRun(wl)
    tt.tt_emb_cache_populate(run.h, dev(hot))
    ref_cores = [c.astype(np.float64) for c in wl.cores[0]]
    for step in range(3):
        ref = oracle.workload_forward(wl, cores=[ref_cores])
        assert_rows_close(run.forward().cpu().numpy(), ref, f"step {step}, rows refreshed")
        assert_rows_close(run.forward().cpu().numpy(), ref, f"step {step}, rows read")
        run.backward()
        assert run.error() == tt.TT_OK
        ref_cores = oracle.sgd_step(wl.tables, [ref_cores], wl.indices, wl.offsets, wl.grad_out, wl.lr,
                                    wl.weights, wl.mode)[0]
        got = run.cores_host()[0]
        for k in range(3):
            assert_rows_close(got[k], ref_cores[k], f"step {step} G{k + 1}")
    run.close()


def test_padding_rows_and_last_row():
    wl = synthetic([4, 5, 6], [2, 2, 2], [4, 4], [3, 2], E=100)
    wl.indices[:] = [99, 0, 98, 99, 1]
    full_parity(wl)


def test_no_lookups():
    wl = synthetic([4, 5, 6], [2, 2, 2], [4, 4], [0, 0, 0])
    run = GpuRun(wl)
    out = run.forward().cpu().numpy()
    assert out.shape == (3, 8) and not out.any()
    run.backward()
    assert run.error() == tt.TT_OK
    after = run.cores_host()
    for k in range(3):
        np.testing.assert_array_equal(after[0][k], wl.cores[0][k])
    run.close()


def test_index_out_of_range_leaves_cores_unchanged():
    wl = synthetic([4, 5, 6], [2, 2, 2], [4, 4], [3, 3], E=110)
    wl.indices[4] = 110
    run = GpuRun(wl)
    run.forward()
    run.backward()
    assert run.error() == tt.TT_ERR_INDEX
    assert run.error() == tt.TT_OK  # the flag is cleared once read
    after = run.cores_host()
    for k in range(3):
        np.testing.assert_array_equal(after[0][k], wl.cores[0][k])
    run.close()


def test_malformed_offsets_reported():
    wl = synthetic([4, 5, 6], [2, 2, 2], [4, 4], [5, 3])
    wl.offsets = np.array([0, 6, 5], dtype=np.int64)  # decreasing, ends below nnz = 8
    run = GpuRun(wl)
    run.forward()
    run.backward()
    assert run.error() == tt.TT_ERR_ARG
    after = run.cores_host()
    for k in range(3):
        np.testing.assert_array_equal(after[0][k], wl.cores[0][k])
    run.close()


@pytest.mark.parametrize("cid,batch", [(2, None), (1, None)])
def test_tensor_core_wait_give_up(workloads, cid, batch):
    """With a wait bound of 0 polls every tensor-core wait for its own MMAs gives up at
    once: the call reports TT_ERR_TIMEOUT, the backward that follows changes no core,
    and (bound restored) the next step on the same handle matches the oracle.  The
    MMAs in flight are waited for with the full bound before tensor memory is freed,
    so the give-up itself leaves nothing running.  (The tiny workload's shape has no
    tensor-core path: its step must come out clean under the 0 bound.)"""
    wl = workloads(cid, batch)
    run = GpuRun(wl)
    tt.tt_emb_set_wait_limit(run.h, 0)
    run.forward()
    run.backward()
    st = run.error()
    assert st == (tt.TT_ERR_TIMEOUT if cid == 2 else tt.TT_OK)
    if st != tt.TT_OK:
        after = run.cores_host()
        for k in range(3):
            np.testing.assert_array_equal(after[0][k], wl.cores[0][k])
        tt.tt_emb_set_wait_limit(run.h, 1 << 24)
    out = run.forward().cpu().numpy()
    dec = check_decode(run, wl)
    run.backward()
    assert run.error() == tt.TT_OK
    if st != tt.TT_OK:
        check_forward(out, wl)
        check_cores(run, wl, dec)
    run.close()


def test_call_order_errors():
    wl = synthetic([4, 5, 6], [2, 2, 2], [4, 4], [2, 2])
    run = GpuRun(wl)
    with pytest.raises(tt.TTError) as e:
        run.backward()
    assert e.value.code == tt.TT_ERR_STATE
    run.forward()
    run.backward()
    with pytest.raises(tt.TTError) as e:
        run.backward()
    assert e.value.code == tt.TT_ERR_STATE
    run.close()


def test_bitwise_reproducible(workloads):
    wl = workloads(3, 512)
    res = []
    for _ in range(2):
        run = GpuRun(wl)
        out = run.forward().cpu().numpy()
        run.backward()
        res.append((out, run.cores_host()))
        run.close()
    np.testing.assert_array_equal(res[0][0], res[1][0])
    for k in range(3):
        np.testing.assert_array_equal(res[0][1][0][k], res[1][1][0][k])


def test_module_matches_c_abi(workloads):
    """TTEmbeddingBag (autograd, PyTorch-style offsets) gives the C-ABI results."""
    wl = workloads(3, 64)
    s = wl.tables[0]
    m = tt.TTEmbeddingBag(s.num_embeddings, s.embedding_dim, s.ranks, s.p, s.q, learning_rate=wl.lr,
                          cores=[torch.from_numpy(c) for c in wl.cores[0]])
    out = m(dev(wl.indices), dev(wl.offsets[:-1]), per_sample_weights=dev(wl.weights), mode="mean")
    out.backward(dev(wl.grad_out))
    run = GpuRun(wl)
    ref = run.forward()
    run.backward()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.detach().cpu().numpy(), ref.cpu().numpy())
    after = run.cores_host()[0]
    for k, c in enumerate([m.G1, m.G2, m.G3]):
        np.testing.assert_array_equal(c.detach().cpu().numpy(), after[k])
    assert m.G1.grad is None
    run.close()


def test_workspace_reuse_across_sizes(workloads):
    """One handle, calls of growing and shrinking sizes (workspace regrowth)."""
    small, big = workloads(3, 64), workloads(3, 512)
    run = GpuRun(small)
    ref_cores = [c.astype(np.float64) for c in small.cores[0]]
    for i, wl in enumerate((small, big, small)):
        run.wl = wl
        run.idx, run.off, run.w, run.go = dev(wl.indices), dev(wl.offsets), dev(wl.weights), dev(wl.grad_out)
        out = run.forward().cpu().numpy()
        assert_rows_close(out, oracle.workload_forward(wl, cores=[ref_cores]), f"call {i}")
        run.backward()
        assert run.error() == tt.TT_OK
        ref_cores = oracle.sgd_step(wl.tables, [ref_cores], wl.indices, wl.offsets, wl.grad_out, wl.lr,
                                    wl.weights, wl.mode)[0]
    got = run.cores_host()[0]
    for k in range(3):
        assert_rows_close(got[k], ref_cores[k], f"G{k + 1} after three calls")
    run.close()


@pytest.mark.parametrize("q,r", [([4, 4, 4], [32, 32]), ([2, 2, 2], [4, 4])])
def test_consecutive_passes_new_lookups(q, r):
    """Four forward + backward passes on one handle, every pass with new indices, bag
    lengths, weights and upstream gradients (the small path, whose forward T blocks start
    on the decode blocks' per-pass stamps): each pass against the oracle's chain of steps."""
    rng = np.random.default_rng(21)
    spec_wl = synthetic([40, 30, 25], q, r, [1], seed=21)
    spec = spec_wl.tables[0]
    run = GpuRun(spec_wl)
    ref_cores = [c.astype(np.float64) for c in spec_wl.cores[0]]
    for step in range(4):
        lengths = rng.integers(0, 30, size=60)
        wl = synthetic([40, 30, 25], q, r, lengths, seed=100 + step, weights=step % 2 == 0,
                       mode="mean" if step == 1 else "sum")
        out = torch.empty((wl.num_bags, spec.embedding_dim), dtype=torch.float32, device="cuda")
        mode = tt.TT_POOL_MEAN if wl.mode == "mean" else tt.TT_POOL_SUM
        w = None if wl.weights is None else dev(wl.weights)
        tt.tt_emb_forward(run.h, dev(wl.indices), dev(wl.offsets), w, mode, out)
        ref = oracle.forward(wl.tables, [ref_cores], wl.indices, wl.offsets, wl.weights, wl.mode, wl.batch)
        assert_rows_close(out.cpu().numpy(), ref, f"pass {step} forward")
        tt.tt_emb_backward(run.h, dev(wl.grad_out), wl.lr)
        assert run.error() == tt.TT_OK
        ref_cores = oracle.sgd_step(wl.tables, [ref_cores], wl.indices, wl.offsets, wl.grad_out, wl.lr,
                                    wl.weights, wl.mode)[0]
        got = run.cores_host()[0]
        for k in range(3):
            assert_rows_close(got[k], ref_cores[k], f"pass {step} G{k + 1}")
    run.close()


@pytest.mark.parametrize("cid,batch", [(2, 128), (3, 96), (3, 800)])
def test_ffma_backward_on_tensor_core_classes(monkeypatch, cid, batch):
    """TTEMB_BWD_FFMA=1 keeps the rank-16/32 classes on the FFMA backward (k_tile_bwd
    with the column split): full parity on the 11M x 64 workload (small-batch path)
    and the Zipf weighted-mean workload (small path; and at 800 bags, ~16k lookups,
    the large-batch path)."""
    monkeypatch.setenv("TTEMB_BWD_FFMA", "1")
    wl = config(cid, batch=batch)
    if wl.nnz > 12288:
        sampled_parity(wl, nbags=128, per_core=8)
    else:
        full_parity(wl)
