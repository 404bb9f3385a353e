"""Helpers for the GPU parity tests: run a seeded workload through the C ABI
and compare with the float64 oracle under the stated tolerance.

Tolerance (the one the TT-EmbeddingBag target states): for every pooled bag,
max_j |gpu - oracle| <= 1e-4 * max_j |oracle|; for every updated core slice,
max |gpu - oracle| <= 1e-4 * max |oracle slice|.  Decoded slice indices and
bag ids must match bit for bit.
"""
import concurrent.futures as cf
import os

import numpy as np
import torch

import oracle
import tensor_train_compressed_embeddingbag_gb300 as tt

RTOL = 1e-4


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


class GpuRun:
    """One handle over a workload's tables, fed the workload's bags."""

    def __init__(self, wl, cache=False, cores=None):
        tt.build()
        self.wl = wl
        src = cores if cores is not None else wl.cores
        self.cores = [[dev(c.astype(np.float32)) for c in t] for t in src]
        if wl.num_tables == 1:
            s = wl.tables[0]
            self.h = tt.tt_emb_create(s.num_embeddings, s.p, s.q, s.ranks, self.cores[0])
        else:
            self.h = tt.tt_emb_batch_create(
                [(s.num_embeddings, s.p, s.q, s.ranks, self.cores[t]) for t, s in enumerate(wl.tables)]
            )
        if cache and wl.cache_rows is not None:
            tt.tt_emb_cache_populate(self.h, dev(wl.cache_rows))
        self.idx = dev(wl.indices)
        self.off = dev(wl.offsets)
        self.w = None if wl.weights is None else dev(wl.weights)
        self.mode = tt.TT_POOL_MEAN if wl.mode == "mean" else tt.TT_POOL_SUM
        self.go = dev(wl.grad_out)

    def forward(self):
        out = torch.empty((self.wl.num_bags, self.wl.embedding_dim), dtype=torch.float32, device="cuda")
        tt.tt_emb_forward(self.h, self.idx, self.off, self.w, self.mode, out)
        return out

    def decoded(self):
        return [x.cpu().numpy().astype(np.int64) for x in tt.tt_emb_get_decoded(self.h, self.wl.nnz, "cuda")]

    def backward(self, lr=None):
        tt.tt_emb_backward(self.h, self.go, self.wl.lr if lr is None else lr)

    def error(self):
        return tt.tt_emb_get_last_error(self.h)

    def cores_host(self):
        torch.cuda.synchronize()
        return [[c.cpu().numpy() for c in t] for t in self.cores]

    def close(self):
        torch.cuda.synchronize()
        tt.tt_emb_destroy(self.h)
        self.h = None


def assert_rows_close(gpu, ref, what, rtol=RTOL):
    gpu = np.asarray(gpu, dtype=np.float64).reshape(ref.shape[0], -1)
    ref = np.asarray(ref, dtype=np.float64).reshape(ref.shape[0], -1)
    err = np.abs(gpu - ref).max(axis=1)
    scale = np.abs(ref).max(axis=1)
    bad = err > rtol * scale
    if bad.any():
        i = int(np.argmax(np.where(scale > 0, err / np.maximum(scale, 1e-300), np.inf)))
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.shape[0]} rows beyond {rtol} x max|row|; "
            f"worst row {i}: err {err[i]:.3e} vs max|ref| {scale[i]:.3e}"
        )


def check_decode(run, wl):
    i1, i2, i3, bag = oracle.decode(wl.tables, wl.indices, wl.offsets, wl.batch)
    t_g, i1_g, i2_g, i3_g, bag_g = run.decoded()
    np.testing.assert_array_equal(i1_g, i1)
    np.testing.assert_array_equal(i2_g, i2)
    np.testing.assert_array_equal(i3_g, i3)
    np.testing.assert_array_equal(bag_g, bag)
    np.testing.assert_array_equal(t_g, bag // wl.batch)
    return i1, i2, i3, bag


def touched_slices(wl, dec):
    """Per table, per core: sorted slice indices that at least one lookup uses."""
    i1, i2, i3, bag = dec
    table = bag // wl.batch
    out = []
    for t in range(wl.num_tables):
        m = table == t
        out.append([np.unique(ik[m]) for ik in (i1, i2, i3)])
    return out


def check_forward(out_gpu, wl, bags=None):
    ref = oracle.workload_forward(wl, bags=bags)
    got = out_gpu if bags is None else out_gpu[np.asarray(bags)]
    assert_rows_close(got, ref, "forward")


def _bag_range(wl, b0, b1):
    """Bags [b0, b1) of every table of `wl` as (indices, offsets, weights, grad_out, batch)."""
    idx, lens, go, w = [], [], [], []
    for t in range(wl.num_tables):
        g0, g1 = t * wl.batch + b0, t * wl.batch + b1
        lo, hi = int(wl.offsets[g0]), int(wl.offsets[g1])
        idx.append(wl.indices[lo:hi])
        lens.append(np.diff(wl.offsets[g0:g1 + 1]))
        go.append(wl.grad_out[g0:g1])
        if wl.weights is not None:
            w.append(wl.weights[lo:hi])
    off = np.concatenate([[0], np.cumsum(np.concatenate(lens))]).astype(np.int64)
    return (np.concatenate(idx), off, None if wl.weights is None else np.concatenate(w),
            np.concatenate(go), b1 - b0)


def oracle_grad(wl, t, k, slices, cores=None, chunks=None):
    """oracle.backward_core of slices `slices` of core k of table t over the whole
    workload.  The gradient is a sum over bags, so for many lookups the oracle runs on
    ranges of bags in parallel threads (the C oracle releases the GIL) and the float64
    partial gradients are added in range order."""
    cores = cores if cores is not None else wl.cores
    sl = np.asarray(slices, dtype=np.int64)
    if chunks is None:
        chunks = 1 if wl.nnz < 40000 else min(wl.batch, 4 * (os.cpu_count() or 4))
    if chunks <= 1:
        return oracle.backward_core(wl.tables, cores, wl.indices, wl.offsets, wl.grad_out, t, k, wl.weights,
                                    wl.mode, wl.batch, sl)
    edges = np.linspace(0, wl.batch, chunks + 1).astype(np.int64)

    def part(c):
        idx, off, w, go, nb = _bag_range(wl, int(edges[c]), int(edges[c + 1]))
        return oracle.backward_core(wl.tables, cores, idx, off, go, t, k, w, wl.mode, nb, sl)

    with cf.ThreadPoolExecutor(max_workers=min(chunks, os.cpu_count() or 4)) as ex:
        parts = list(ex.map(part, range(chunks)))
    total = parts[0]
    for p in parts[1:]:
        total = total + p
    return total


def check_cores(run, wl, dec, slices=None):
    """Updated cores vs oracle on `slices` (per table, per core; None = all) after one
    step from the workload's cores; slices no lookup touched must keep their exact bits."""
    after = run.cores_host()
    touched = touched_slices(wl, dec)
    for t in range(wl.num_tables):
        for k in range(3):
            init = wl.cores[t][k]
            un = np.setdiff1d(np.arange(wl.tables[t].p[k]), touched[t][k])
            np.testing.assert_array_equal(after[t][k][un], init[un], err_msg=f"untouched slices t{t} G{k + 1}")
            sl = touched[t][k] if slices is None else np.asarray(slices[t][k], dtype=np.int64)
            if sl.size == 0:
                continue
            ref = oracle.sgd_update(wl.cores[t][k][sl], oracle_grad(wl, t, k, sl), wl.lr)
            assert_rows_close(after[t][k][sl], ref, f"table {t} core G{k + 1}")


def sample_slices(wl, dec, rng, per_core=6, max_count=None, hot=2):
    """Per table and core: the `hot` touched slices with the most lookups (the longest
    sorted-segment and multi-tile reductions), the touched slices with the fewest
    lookups, and random ones; `max_count` bounds only the cold and random picks.
    Every core with a touched slice gets at least one sampled slice."""
    i1, i2, i3, bag = dec
    table = bag // wl.batch
    out = []
    for t in range(wl.num_tables):
        m = table == t
        row = []
        for k, ik in enumerate((i1[m], i2[m], i3[m])):
            u_all, c_all = np.unique(ik, return_counts=True)
            pick = list(u_all[np.argsort(-c_all, kind="stable")[:hot]])
            u, c = u_all, c_all
            if max_count is not None:
                keep = c <= max_count
                u, c = u[keep], c[keep]
            order = np.argsort(c, kind="stable")
            pick += list(u[order[: per_core // 2]])
            if u.size:
                pick += list(rng.choice(u, size=min(max(per_core - per_core // 2, 0), u.size), replace=False))
            sel = np.unique(np.array(pick, dtype=np.int64))
            assert u_all.size == 0 or sel.size > 0, f"no sampled slice for table {t} core G{k + 1}"
            row.append(sel)
        out.append(row)
    return out
