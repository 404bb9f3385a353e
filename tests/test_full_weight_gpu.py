"""GPU: expanding a TT table to its full weight (FBTT README,
"TableBatchedTTEmbeddingBag": expanding to full weight) and the module's
automatic shapes and weight_dist initialisation, against the float64 oracle
(a row of the table is the forward output of a one-hot bag)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import tensor_train_compressed_embeddingbag_gb300 as tt
from tt_inputs import TableSpec

from _gpu_harness import GpuRun, assert_rows_close

pytestmark = pytest.mark.gpu


def _rows_ref(spec, cores, rows):
    rows = np.asarray(rows, dtype=np.int64)
    return oracle.forward([spec], [cores], rows, np.arange(rows.shape[0] + 1))


def test_full_weight_tiny_every_row(workloads):
    wl = workloads(1)
    run = GpuRun(wl)
    s = wl.tables[0]
    out = torch.empty((s.num_embeddings, s.embedding_dim), device="cuda")
    tt.tt_emb_full_weight(run.h, 0, 0, s.num_embeddings, out)
    assert_rows_close(out.cpu().numpy(), _rows_ref(s, wl.cores[0], np.arange(s.num_embeddings)), "full weight")
    run.close()


def test_full_weight_row_ranges_11m(workloads):
    """11M x 64 rank-32: the first, last and a middle block of rows."""
    wl = workloads(2)
    run = GpuRun(wl)
    s = wl.tables[0]
    for row0 in (0, 5_432_101, s.num_embeddings - 777):
        n = min(777, s.num_embeddings - row0)
        out = torch.empty((n, s.embedding_dim), device="cuda")
        tt.tt_emb_full_weight(run.h, 0, row0, n, out)
        assert_rows_close(out.cpu().numpy(), _rows_ref(s, wl.cores[0], np.arange(row0, row0 + n)), f"rows {row0}+")
    run.close()


def test_full_weight_table_batched(workloads):
    wl = workloads(5, 32)
    run = GpuRun(wl)
    rng = np.random.default_rng(0)
    for t in rng.choice(wl.num_tables, 6, replace=False):
        s = wl.tables[t]
        row0 = int(rng.integers(0, max(1, s.num_embeddings - 64)))
        n = min(64, s.num_embeddings - row0)
        out = torch.empty((n, s.embedding_dim), device="cuda")
        tt.tt_emb_full_weight(run.h, int(t), row0, n, out)
        assert_rows_close(out.cpu().numpy(), _rows_ref(s, wl.cores[t], np.arange(row0, row0 + n)), f"table {t}")
    run.close()


def test_full_weight_rejects_bad_ranges(workloads):
    wl = workloads(1)
    run = GpuRun(wl)
    lib = tt.load_library()
    out = torch.empty((200, 8), device="cuda")
    p = ctypes.c_void_p(out.data_ptr())
    assert lib.tt_emb_full_weight(run.h, 0, -1, 1, p, None) == tt.TT_ERR_ARG
    assert lib.tt_emb_full_weight(run.h, 0, 100, 21, p, None) == tt.TT_ERR_ARG  # past E = 120
    assert lib.tt_emb_full_weight(run.h, 1, 0, 1, p, None) == tt.TT_ERR_ARG     # one table only
    assert lib.tt_emb_full_weight(run.h, 0, 0, 1, None, None) == tt.TT_ERR_ARG
    assert lib.tt_emb_full_weight(run.h, 0, 120, 0, p, None) == tt.TT_OK
    run.close()


@pytest.mark.parametrize("dist", ["uniform", "approx-uniform", "approx-normal"])
def test_module_page_example_auto_shapes(dist):
    """FBTT README "Initialization": TTEmbeddingBag(10, 3, None, None, tt_ranks=[2, 2]) on its bags."""
    g = torch.Generator().manual_seed(0)
    m = tt.TTEmbeddingBag(10, 3, [2, 2], None, None, sparse=False, weight_dist=dist, generator=g)
    assert (m.p, m.q) == ([2, 2, 3], [1, 1, 3])
    inp = torch.tensor([1, 2, 4, 5, 4, 3, 2, 9], device="cuda")
    off = torch.tensor([0, 4], device="cuda")
    out = m(inp, off)
    assert tuple(out.shape) == (2, 3)
    spec = TableSpec(10, m.p, m.q, m.ranks)
    cores = [c.detach().cpu().numpy().astype(np.float64) for c in (m.G1, m.G2, m.G3)]
    ref = oracle.forward([spec], [cores], inp.cpu().numpy(), np.array([0, 4, 8]))
    assert_rows_close(out.detach().cpu().numpy(), ref, "page example")
    full = m.full_weight()
    assert_rows_close(full.cpu().numpy(), _rows_ref(spec, cores, np.arange(10)), "page example full weight")
