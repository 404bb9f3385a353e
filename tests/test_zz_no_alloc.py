"""The allocation-free forward entry point against the handle-based one and the oracle.

tt_emb_forward_noalloc() serves callers that cannot allocate device memory:
code under a memory manager that owns all of it (a framework's caching
allocator, a serving runtime with a fixed budget), and code that must not
synchronize the device or that runs while a stream is captured into a CUDA
graph.  Its only scratch is a static device array shared by every call.  Two
calls in a row must give the handle path's output and the float64 oracle's
within the parity tolerance: the second call runs on the array as the first
call left it.  The 40M x 128 rank-64 case has more bags than the array has
warp slots, so the grid is clamped and warps take several bags each.  This
file is collected last so that a failure here stops a -x run only after every
other test has run.
"""
import numpy as np
import pytest
import torch

import oracle
import tensor_train_compressed_embeddingbag_gb300 as tt
from tt_inputs import config

from _gpu_harness import GpuRun, assert_rows_close, dev

pytestmark = pytest.mark.gpu


def _noalloc(wl, run, idx, w, err):
    s = wl.tables[0]
    out = torch.full((wl.num_bags, wl.embedding_dim), float("nan"), dtype=torch.float32, device="cuda")
    tt.tt_emb_forward_noalloc(s.num_embeddings, s.p, s.q, s.ranks, run.cores[0], idx, run.off, w, run.mode, out, err)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("cid,batch,sample", [(2, None, None), (3, 256, None), (4, 2560, 160)])
def test_noalloc_forward_matches_handle_forward_and_oracle(cid, batch, sample):
    """(3, 256): Zipf lookups with per-sample weights and mean pooling; (4, 2560): the
    grid clamp of the static array (rank 64: 1024 floats per warp slot)."""
    wl = config(cid, batch=batch)
    run = GpuRun(wl)
    ref = run.forward().cpu().numpy()
    assert run.error() == tt.TT_OK
    bags = None if sample is None else np.unique(
        np.concatenate([[0, wl.num_bags - 1], np.random.default_rng(cid).choice(wl.num_bags, sample, replace=False)]))
    want = oracle.workload_forward(wl, bags=bags)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = _noalloc(wl, run, run.idx, run.w, err)
        assert int(err.item()) == 0
        assert_rows_close(out, ref.astype(np.float64), f"no-alloc vs handle forward, call {call}")
        assert_rows_close(out if bags is None else out[bags], want, f"no-alloc vs oracle, call {call}")
    run.close()


def test_noalloc_out_of_range_index_contributes_nothing():
    """An index outside [0, E) sets bit 1 of the error word and adds nothing; in mean
    mode the bag's other lookups keep the full bag length as divisor."""
    wl = config(3, batch=64)
    run = GpuRun(wl)
    bad = np.array([3, int(wl.offsets[10]), wl.nnz - 1])
    idx = wl.indices.copy()
    idx[bad[0]] = wl.tables[0].num_embeddings
    idx[bad[1]] = -5
    idx[bad[2]] = wl.tables[0].num_embeddings + 1000
    w = wl.weights.copy()
    w[bad] = 0.0
    safe = idx.copy()
    safe[bad] = 0
    want = oracle.forward(wl.tables, wl.cores, safe, wl.offsets, w, wl.mode, wl.batch)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _noalloc(wl, run, dev(idx), run.w, err)
    assert int(err.item()) == 1
    assert_rows_close(out, want, "no-alloc forward with out-of-range indices")
    run.close()
