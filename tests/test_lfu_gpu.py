"""GPU: the LFU cache policy (FBTT README, "Software Cache"; "Parameters":
use_cache, cache_size, hashtbl_size) against the oracle.

* Access counts from the forward passes equal the oracle's counts exactly
  (integer, order-independent while the frequency table has room).
* tt_emb_lfu_populate's cache equals the oracle's per-set selection slot by slot.
* With the cache, forward outputs and updated cores stay within the parity
  tolerance of the oracle (cached rows are exact copies of TT rows).
* A full frequency table counts the rows it holds exactly and no others.
"""
import numpy as np
import pytest
import torch

import oracle
import tensor_train_compressed_embeddingbag_gb300 as tt

from _gpu_harness import GpuRun, assert_rows_close, check_cores, check_decode, check_forward, dev, sample_slices

pytestmark = pytest.mark.gpu


def test_counts_and_selection_exact(workloads):
    """Zipf weighted-mean workload (82k lookups): two forward passes, then populate."""
    wl = workloads(3)
    run = GpuRun(wl)
    cache_size = 4000  # 125 sets of 32 ways
    tt.tt_emb_lfu_enable(run.h, cache_size, 1 << 17)
    run.forward()
    run.backward()
    run.forward()
    torch.cuda.synchronize()
    rows, counts = tt.tt_emb_lfu_read(run.h)
    ref_rows, ref_counts = oracle.lfu_counts(wl.indices, wl.indices)
    np.testing.assert_array_equal(rows, ref_rows)
    np.testing.assert_array_equal(counts.astype(np.int64), ref_counts)
    tt.tt_emb_lfu_populate(run.h)
    np.testing.assert_array_equal(tt.tt_emb_lfu_cached_rows(run.h), oracle.lfu_select(ref_rows, ref_counts, cache_size))
    run.close()


def test_forward_backward_with_lfu_cache(workloads):
    """Scaled Zipf workload: count, populate, then a step with the cache against the oracle."""
    wl = workloads(3, 512)
    run = GpuRun(wl)
    tt.tt_emb_lfu_enable(run.h, 1024, 1 << 14)
    run.forward()  # counts only (the cache is empty)
    tt.tt_emb_lfu_populate(run.h)
    cached = tt.tt_emb_lfu_cached_rows(run.h)
    assert np.isin(wl.indices, cached[cached >= 0]).mean() > 0.3  # the hot rows are cached
    out = run.forward().cpu().numpy()
    dec = check_decode(run, wl)
    run.backward()
    assert run.error() == tt.TT_OK
    check_forward(out, wl)
    check_cores(run, wl, dec, sample_slices(wl, dec, np.random.default_rng(0), 6))
    run.close()


def test_full_frequency_table_counts_what_it_holds(workloads):
    wl = workloads(3, 256)
    run = GpuRun(wl)
    tt.tt_emb_lfu_enable(run.h, 64, 32)
    run.forward()
    torch.cuda.synchronize()
    rows, counts = tt.tt_emb_lfu_read(run.h)
    ref_rows, ref_counts = oracle.lfu_counts(wl.indices)
    assert rows.shape[0] == 32  # full: more distinct rows than entries
    idx = np.searchsorted(ref_rows, rows)
    np.testing.assert_array_equal(ref_rows[idx], rows)
    np.testing.assert_array_equal(counts.astype(np.int64), ref_counts[idx])
    run.close()


def test_module_use_cache_lfu(workloads):
    """TTEmbeddingBag(use_cache=True, cache_size, hashtbl_size): forward, cache_populate(), forward."""
    wl = workloads(3, 256)
    s = wl.tables[0]
    m = tt.TTEmbeddingBag(s.num_embeddings, s.embedding_dim, s.ranks, s.p, s.q, learning_rate=wl.lr,
                          cores=[torch.from_numpy(c) for c in wl.cores[0]], use_cache=True, cache_size=512,
                          hashtbl_size=4096)
    args = (dev(wl.indices), dev(wl.offsets))
    kw = dict(per_sample_weights=dev(wl.weights), mode=wl.mode, include_last_offset=True)
    with torch.no_grad():
        first = m(*args, **kw).cpu().numpy()
        m.cache_populate()
        second = m(*args, **kw).cpu().numpy()
    check_forward(first, wl)
    check_forward(second, wl)
    assert (tt.tt_emb_lfu_cached_rows(m._h) >= 0).sum() > 0


def test_lfu_argument_and_state_errors(workloads):
    lib = tt.load_library()
    run = GpuRun(workloads(1))
    assert lib.tt_emb_lfu_populate(run.h, None) == tt.TT_ERR_STATE  # before enable
    assert lib.tt_emb_lfu_enable(run.h, 64, 100) == tt.TT_ERR_ARG    # not a power of two
    assert lib.tt_emb_lfu_enable(run.h, 0, 64) == tt.TT_ERR_ARG
    run.close()
    run = GpuRun(workloads(5, 8))
    assert lib.tt_emb_lfu_enable(run.h, 64, 64) == tt.TT_ERR_STATE   # table-batched handle
    run.close()
