"""Pins of the float64 oracle against what the pages and the mathematics fix.

None of these checks retypes the oracle's formula: each one compares it with
an independent route to the same numbers.

* TT-SVD: any E x D matrix has an exact tensor-train form at full ranks
  (Oseledets, 2011).  Decomposing a random matrix with numpy's SVD and feeding
  the cores back must reproduce the matrix row for row.  This pins the row
  decode i = i1 p2 p3 + i2 p3 + i3, the column order j = j1 q2 q3 + j2 q3 + j3
  and the [p_k, r_{k-1}, q_k, r_k] core layout.
* Rank 1: with r1 = r2 = 1 a row is the Kronecker product of three vectors.
* Plain EmbeddingBag: p = [E,1,1], q = [D,1,1], r = [1,1] with unit G2, G3
  leaves W = G1, which must match torch.nn.functional.embedding_bag (the
  FBTT README presents the layer as a drop-in for it).
* Finite differences: L = <out, grad_out> is linear in every single core
  element, so a central difference with step 1 is exact up to rounding.
* torch autograd through an einsum of the cores gives the same gradients.
* Invariants: duplicates act as weight 2, order inside a bag does not
  matter, mean = sum / L_b, linearity in grad_out, untouched slices keep
  their exact bits under SGD, batched tables equal separate tables.
* Adagrad: two oracle steps equal torch.optim.Adagrad fed the same
  gradients, from a zero and from a warm accumulator.
* SGD: two oracle steps (sgd_step over every core of two tables, sgd_slices
  on a subset of slices) equal torch.optim.SGD stepping the cores of a torch
  float64 model whose gradients come from autograd through an einsum of the
  cores, in sum mode and in weighted mean mode.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle
from tt_inputs import TableSpec, config

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_cores(rng, spec, sigma=0.5):
    return [rng.normal(0, sigma, size=s) for s in spec.core_shapes()]


def one_hot_rows(spec, cores, rows=None):
    rows = np.arange(spec.num_embeddings) if rows is None else np.asarray(rows)
    off = np.arange(rows.shape[0] + 1)
    return oracle.forward([spec], [cores], rows, off)


def tt_svd(W, p, q):
    """Exact (full-rank) TT decomposition of W[E, D], cores in [p_k, r_{k-1}, q_k, r_k]."""
    p1, p2, p3 = p
    q1, q2, q3 = q
    X = W.reshape(p1, p2, p3, q1, q2, q3).transpose(0, 3, 1, 4, 2, 5)  # (i1,j1,i2,j2,i3,j3)
    U, S, Vt = np.linalg.svd(X.reshape(p1 * q1, -1), full_matrices=False)
    r1 = U.shape[1]
    G1 = U.reshape(p1, q1, r1)[:, None, :, :]
    R = (S[:, None] * Vt).reshape(r1 * p2 * q2, p3 * q3)  # rows (a, i2, j2)
    U2, S2, Vt2 = np.linalg.svd(R, full_matrices=False)
    r2 = U2.shape[1]
    G2 = U2.reshape(r1, p2, q2, r2).transpose(1, 0, 2, 3)
    G3 = (S2[:, None] * Vt2).reshape(r2, p3, q3).transpose(1, 0, 2)[..., None]
    return [np.ascontiguousarray(G1), np.ascontiguousarray(G2), np.ascontiguousarray(G3)], (r1, r2)


@pytest.mark.parametrize("p,q", [([3, 2, 4], [2, 3, 2]), ([2, 5, 3], [4, 1, 3]), ([4, 3, 2], [3, 2, 2])])
def test_tt_svd_reconstructs_arbitrary_matrix(p, q):
    rng = np.random.default_rng(1)
    E, D = int(np.prod(p)), int(np.prod(q))
    W = rng.standard_normal((E, D))
    cores, (r1, r2) = tt_svd(W, p, q)
    spec = TableSpec(E, p, q, [r1, r2])
    got = one_hot_rows(spec, cores)
    np.testing.assert_allclose(got, W, rtol=0, atol=1e-12 * np.abs(W).max())


def test_rank_one_is_kronecker_product():
    rng = np.random.default_rng(2)
    p, q = [3, 4, 5], [2, 3, 2]
    spec = TableSpec(60, p, q, [1, 1])
    cores = rand_cores(rng, spec)
    got = one_hot_rows(spec, cores)
    for i, (a, b, c) in enumerate(itertools.product(range(p[0]), range(p[1]), range(p[2]))):
        want = np.kron(np.kron(cores[0][a, 0, :, 0], cores[1][b, 0, :, 0]), cores[2][c, 0, :, 0])
        np.testing.assert_allclose(got[i], want, rtol=1e-14, atol=1e-15)


def test_decode_follows_enumeration_order():
    p = [3, 4, 5]
    spec = TableSpec(60, p, [1, 1, 1], [1, 1])
    idx = np.arange(60)
    i1, i2, i3, bag = oracle.decode([spec], idx, np.arange(61))
    want = np.array(list(itertools.product(range(p[0]), range(p[1]), range(p[2]))))
    np.testing.assert_array_equal(np.stack([i1, i2, i3], 1), want)
    np.testing.assert_array_equal(bag, idx)


def test_padding_rows_rejected():
    spec = TableSpec(50, [3, 4, 5], [1, 1, 1], [1, 1])  # 60 slots, 50 rows
    cores = rand_cores(np.random.default_rng(0), spec)
    with pytest.raises(IndexError):
        oracle.forward([spec], [cores], np.array([50]), np.array([0, 1]))
    with pytest.raises(IndexError):
        oracle.forward([spec], [cores], np.array([-1]), np.array([0, 1]))


def _plain_bag_case(rng, E=37, D=6, B=9):
    spec = TableSpec(E, [E, 1, 1], [D, 1, 1], [1, 1])
    G1 = rng.standard_normal((E, 1, D, 1))
    cores = [G1, np.ones((1, 1, 1, 1)), np.ones((1, 1, 1, 1))]
    lengths = rng.integers(0, 6, size=B)
    off = np.concatenate([[0], np.cumsum(lengths)])
    idx = rng.integers(0, E, size=int(off[-1]))
    w = rng.random(idx.shape[0])
    return spec, cores, G1[:, 0, :, 0], idx, off, w


@pytest.mark.parametrize("mode", ["sum", "mean"])
def test_plain_embedding_bag_matches_torch(mode):
    rng = np.random.default_rng(3)
    spec, cores, W, idx, off, w = _plain_bag_case(rng)
    got = oracle.forward([spec], [cores], idx, off, mode=mode)
    want = torch.nn.functional.embedding_bag(
        torch.from_numpy(idx), torch.from_numpy(W), torch.from_numpy(off[:-1]), mode=mode
    ).numpy()
    np.testing.assert_allclose(got, want, rtol=1e-14, atol=1e-14)


def test_plain_embedding_bag_weights_and_gradient_match_torch():
    rng = np.random.default_rng(4)
    spec, cores, W, idx, off, w = _plain_bag_case(rng)
    go = rng.standard_normal((off.shape[0] - 1, W.shape[1]))
    Wt = torch.from_numpy(W.copy()).requires_grad_(True)
    out = torch.nn.functional.embedding_bag(
        torch.from_numpy(idx), Wt, torch.from_numpy(off[:-1]), mode="sum",
        per_sample_weights=torch.from_numpy(w),
    )
    (out * torch.from_numpy(go)).sum().backward()
    got = oracle.forward([spec], [cores], idx, off, weights=w)
    np.testing.assert_allclose(got, out.detach().numpy(), rtol=1e-14, atol=1e-14)
    dG1 = oracle.backward_core([spec], [cores], idx, off, go, 0, 0, weights=w)
    np.testing.assert_allclose(dG1[:, 0, :, 0], Wt.grad.numpy(), rtol=1e-13, atol=1e-13)


def _loss(spec, cores, idx, off, go, w, mode):
    return float((oracle.forward([spec], [cores], idx, off, weights=w, mode=mode) * go).sum())


@pytest.mark.parametrize("mode,weighted", [("sum", False), ("mean", True)])
def test_backward_matches_exact_finite_differences(mode, weighted):
    wl = config(1)
    spec, cores = wl.tables[0], [c.astype(np.float64) for c in wl.cores[0]]
    rng = np.random.default_rng(5)
    w = rng.random(wl.nnz) if weighted else None
    go = wl.grad_out.astype(np.float64)
    for k in range(3):
        dG = oracle.backward_core([spec], [cores], wl.indices, wl.offsets, go, 0, k, weights=w, mode=mode)
        fd = np.zeros_like(cores[k])
        flat = cores[k].reshape(-1)
        for e in range(flat.shape[0]):
            keep = flat[e]
            flat[e] = keep + 1.0
            lp = _loss(spec, cores, wl.indices, wl.offsets, go, w, mode)
            flat[e] = keep - 1.0
            lm = _loss(spec, cores, wl.indices, wl.offsets, go, w, mode)
            flat[e] = keep
            fd.reshape(-1)[e] = 0.5 * (lp - lm)
        np.testing.assert_allclose(dG, fd, rtol=1e-10, atol=1e-11)


def test_backward_matches_torch_autograd():
    rng = np.random.default_rng(6)
    spec = TableSpec(100, [5, 4, 6], [2, 3, 2], [3, 5])
    cores = rand_cores(rng, spec)
    B = 7
    lengths = rng.integers(0, 5, size=B)
    off = np.concatenate([[0], np.cumsum(lengths)])
    idx = rng.integers(0, 100, size=int(off[-1]))
    w = rng.random(idx.shape[0])
    go = rng.standard_normal((B, 12))
    gt = [torch.from_numpy(c.copy()).requires_grad_(True) for c in cores]
    full = torch.einsum("xja,yakc,zcl->xyzjkl", gt[0][:, 0], gt[1], gt[2][..., 0]).reshape(120, 12)
    bag = torch.from_numpy(np.repeat(np.arange(B), lengths))
    L = torch.from_numpy(lengths).double()
    s = torch.from_numpy(w) / L[bag]
    out = torch.zeros(B, 12, dtype=torch.float64).index_add_(0, bag, s[:, None] * full[torch.from_numpy(idx)])
    (out * torch.from_numpy(go)).sum().backward()
    np.testing.assert_allclose(
        oracle.forward([spec], [cores], idx, off, weights=w, mode="mean"), out.detach().numpy(), rtol=1e-12, atol=1e-13
    )
    for k in range(3):
        dG = oracle.backward_core([spec], [cores], idx, off, go, 0, k, weights=w, mode="mean")
        np.testing.assert_allclose(dG, gt[k].grad.numpy(), rtol=1e-12, atol=1e-13)


def test_pooling_invariants():
    rng = np.random.default_rng(7)
    spec = TableSpec(100, [5, 4, 5], [2, 2, 2], [3, 4])
    cores = rand_cores(rng, spec)
    # a duplicated index is the same as weight 2
    a = oracle.forward([spec], [cores], np.array([3, 3, 17]), np.array([0, 3]))
    b = oracle.forward([spec], [cores], np.array([3, 17]), np.array([0, 2]), weights=np.array([2.0, 1.0]))
    np.testing.assert_allclose(a, b, rtol=1e-14, atol=1e-15)
    # order inside a bag does not matter
    idx = rng.integers(0, 100, size=9)
    a = oracle.forward([spec], [cores], idx, np.array([0, 9]))
    b = oracle.forward([spec], [cores], idx[::-1].copy(), np.array([0, 9]))
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)
    # mean = sum / L, and an empty bag is a zero row
    off = np.array([0, 4, 4, 9])
    s = oracle.forward([spec], [cores], idx, off)
    m = oracle.forward([spec], [cores], idx, off, mode="mean")
    np.testing.assert_allclose(m[0], s[0] / 4, rtol=1e-14)
    np.testing.assert_allclose(m[2], s[2] / 5, rtol=1e-14)
    assert not s[1].any() and not m[1].any()
    # the selected-bag path gives the same rows
    np.testing.assert_array_equal(oracle.forward([spec], [cores], idx, off, bags=[2, 0]), s[[2, 0]])


def test_backward_invariants():
    wl = config(1)
    spec, cores = wl.tables[0], wl.cores[0]
    rng = np.random.default_rng(8)
    g1 = rng.standard_normal(wl.grad_out.shape)
    g2 = rng.standard_normal(wl.grad_out.shape)
    for k in range(3):
        d1 = oracle.backward_core([spec], [cores], wl.indices, wl.offsets, g1, 0, k)
        d2 = oracle.backward_core([spec], [cores], wl.indices, wl.offsets, g2, 0, k)
        d12 = oracle.backward_core([spec], [cores], wl.indices, wl.offsets, 2 * g1 - 3 * g2, 0, k)
        np.testing.assert_allclose(d12, 2 * d1 - 3 * d2, rtol=1e-12, atol=1e-13)
    # untouched slices keep their exact bits, touched ones move
    i1, i2, i3, _ = oracle.decode([spec], wl.indices, wl.offsets)
    new = oracle.sgd_step([spec], [cores], wl.indices, wl.offsets, wl.grad_out, wl.lr)[0]
    for k, ik in enumerate([i1, i2, i3]):
        untouched = np.setdiff1d(np.arange(spec.p[k]), ik)
        np.testing.assert_array_equal(new[k][untouched], cores[k][untouched].astype(np.float64))
        touched = np.unique(ik)
        assert np.abs(new[k][touched] - cores[k][touched]).max() > 0


def test_batched_tables_equal_separate_tables():
    rng = np.random.default_rng(9)
    specs = [TableSpec(60, [3, 4, 5], [2, 2, 2], [2, 3]), TableSpec(30, [2, 3, 5], [4, 1, 2], [4, 2])]
    cores = [rand_cores(rng, s) for s in specs]
    B = 5
    parts, offs = [], [0]
    for s in specs:
        lengths = rng.integers(0, 4, size=B)
        parts.append(rng.integers(0, s.num_embeddings, size=int(lengths.sum())))
        offs.extend(offs[-1] + np.cumsum(lengths))
    idx, off = np.concatenate(parts), np.array(offs)
    go = rng.standard_normal((2 * B, 8))
    both = oracle.forward(specs, cores, idx, off)
    for t in range(2):
        sub_off = off[t * B : (t + 1) * B + 1] - off[t * B]
        sub_idx = idx[off[t * B] : off[(t + 1) * B]]
        np.testing.assert_array_equal(both[t * B : (t + 1) * B], oracle.forward([specs[t]], [cores[t]], sub_idx, sub_off))
        for k in range(3):
            np.testing.assert_array_equal(
                oracle.backward_core(specs, cores, idx, off, go, t, k),
                oracle.backward_core([specs[t]], [cores[t]], sub_idx, sub_off, go[t * B : (t + 1) * B], 0, k),
            )


def test_page_usage_example_offsets_convention():
    """FBTT README usage example: 10 rows of width 3, two bags of four lookups.

    The page prints values drawn from a random initialisation, so only the
    shape and the bag split given by start-position offsets are pinned.
    """
    with open(os.path.join(GOLDEN, "fbtt_readme_usage_example.json")) as f:
        ex = json.load(f)
    idx = np.array(ex["input"])
    csr = np.concatenate([ex["offsets"], [idx.shape[0]]])
    spec = TableSpec(ex["num_embeddings"], ex["p_shapes_used_here"], ex["q_shapes_used_here"], ex["tt_ranks"])
    cores = rand_cores(np.random.default_rng(10), spec)
    out = oracle.forward([spec], [cores], idx, csr)
    assert list(out.shape) == ex["output_shape"]
    rows = one_hot_rows(spec, cores)
    for b, members in enumerate(ex["bag_members"]):
        np.testing.assert_allclose(out[b], rows[members].sum(0), rtol=1e-14, atol=1e-15)


def test_tiny_workload_golden():
    """Regression fixture written by tests/golden/make_golden.py (oracle only)."""
    with open(os.path.join(GOLDEN, "config1_oracle.json")) as f:
        g = json.load(f)
    wl = config(1)
    np.testing.assert_array_equal(wl.indices, g["indices"])
    np.testing.assert_array_equal(wl.offsets, g["offsets"])
    np.testing.assert_allclose(oracle.workload_forward(wl), np.array(g["out"]), rtol=1e-15, atol=1e-15)
    for k in range(3):
        np.testing.assert_allclose(
            oracle.workload_sgd_slices(wl, 0, k), np.array(g["updated_cores"][k]), rtol=1e-15, atol=1e-15
        )


@pytest.mark.parametrize("init", [0.0, 0.7])
def test_adagrad_matches_torch_optim(init):
    """Two fused element-wise Adagrad steps of the oracle (gradients at the
    pre-update cores of each step) equal torch.optim.Adagrad fed the same
    gradients: the update rule is pinned to an independent implementation."""
    rng = np.random.default_rng(11)
    spec = TableSpec(100, [5, 4, 6], [2, 3, 2], [3, 5])
    cores = rand_cores(rng, spec)
    B = 6
    lengths = rng.integers(1, 5, size=B)
    off = np.concatenate([[0], np.cumsum(lengths)])
    idx = rng.integers(0, 100, size=int(off[-1]))
    go = rng.standard_normal((B, 12))
    lr, eps = 0.05, 1e-10
    params = [torch.from_numpy(c.copy()).requires_grad_(True) for c in cores]
    opt = torch.optim.Adagrad(params, lr=lr, eps=eps, initial_accumulator_value=init)
    cur = [c.copy() for c in cores]
    state = [np.full(c.shape, init) for c in cores]
    for _ in range(2):
        upd = [oracle.adagrad_slices([spec], [cur], idx, off, go, lr, eps, state[k], 0, k) for k in range(3)]
        for k in range(3):
            params[k].grad = torch.from_numpy(oracle.backward_core([spec], [cur], idx, off, go, 0, k))
        opt.step()
        cur, state = [u[0] for u in upd], [u[1] for u in upd]
        for k in range(3):
            np.testing.assert_allclose(cur[k], params[k].detach().numpy(), rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(state[k], opt.state[params[k]]["sum"].numpy(), rtol=1e-12, atol=1e-14)


def _torch_bag_loss(specs, params, idx, off, go, w, mode, batch):
    """<out, grad_out> of a table-batched EmbeddingBag over full tables expanded from
    the cores by einsum (torch float64; autograd gives the core gradients)."""
    loss = 0.0
    for t, spec in enumerate(specs):
        g1, g2, g3 = params[t]
        p1, p2, p3 = spec.p
        D = int(np.prod(spec.q))
        full = torch.einsum("xja,yakc,zcl->xyzjkl", g1[:, 0], g2, g3[..., 0]).reshape(p1 * p2 * p3, D)
        lo, hi = int(off[t * batch]), int(off[(t + 1) * batch])
        lengths = np.diff(off[t * batch:(t + 1) * batch + 1])
        bag = torch.from_numpy(np.repeat(np.arange(batch), lengths))
        s = torch.ones(hi - lo, dtype=torch.float64) if w is None else torch.from_numpy(w[lo:hi]).clone()
        if mode == "mean":
            s = s / torch.from_numpy(np.maximum(lengths, 1)).double()[bag]
        out = torch.zeros(batch, D, dtype=torch.float64).index_add_(
            0, bag, s[:, None] * full[torch.from_numpy(idx[lo:hi])])
        loss = loss + (out * torch.from_numpy(go[t * batch:(t + 1) * batch])).sum()
    return loss


@pytest.mark.parametrize("mode,weighted", [("sum", False), ("mean", True)])
def test_sgd_matches_torch_optim(mode, weighted):
    """Two fused SGD steps of the oracle (every gradient at the pre-update cores of its
    step) equal torch.optim.SGD on a torch model of the same two tables whose gradients
    come from autograd: pins sgd_update, sgd_slices and sgd_step (a sign error or a
    doubled learning rate fails here)."""
    rng = np.random.default_rng(12)
    specs = [TableSpec(100, [5, 4, 6], [2, 3, 2], [3, 5]), TableSpec(60, [3, 4, 5], [3, 2, 2], [2, 4])]
    cores = [rand_cores(rng, s) for s in specs]
    batch = 6
    lengths = rng.integers(0, 5, size=batch * len(specs))
    off = np.concatenate([[0], np.cumsum(lengths)])
    idx = np.concatenate([rng.integers(0, specs[t].num_embeddings, size=int(lengths[t * batch:(t + 1) * batch].sum()))
                          for t in range(len(specs))])
    w = rng.random(idx.shape[0]) if weighted else None
    go = rng.standard_normal((batch * len(specs), 12))
    lr = 0.07
    params = [[torch.from_numpy(c.copy()).requires_grad_(True) for c in cs] for cs in cores]
    opt = torch.optim.SGD([p for ps in params for p in ps], lr=lr)
    cur = [[c.copy() for c in cs] for cs in cores]
    for _ in range(2):
        nxt = oracle.sgd_step(specs, cur, idx, off, go, lr, weights=w, mode=mode, bags_per_table=batch)
        sl = np.array([0, 2, 3])
        part = oracle.sgd_slices(specs, cur, idx, off, go, lr, 1, 1, weights=w, mode=mode, bags_per_table=batch,
                                 slices=sl)
        opt.zero_grad()
        _torch_bag_loss(specs, params, idx, off, go, w, mode, batch).backward()
        opt.step()
        for t in range(len(specs)):
            for k in range(3):
                np.testing.assert_allclose(nxt[t][k], params[t][k].detach().numpy(), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(part, params[1][1].detach().numpy()[sl], rtol=1e-12, atol=1e-14)
        cur = nxt


def test_splitmix64_published_outputs():
    """The row hash of the LFU policy: SplitMix64's published outputs (seed 0; seed 1234567, three steps)."""
    assert oracle.splitmix64(0) == 0xE220A8397B1DCDAF
    golden = 0x9E3779B97F4A7C15
    s, out = 1234567, []
    for _ in range(3):
        out.append(oracle.splitmix64(s))
        s = (s + golden) & ((1 << 64) - 1)
    assert out == [6457827717110365317, 3203168211198807973, 9817491932198370423]


def test_lfu_select_brute_force():
    """Per set, the selection equals a brute-force ranking of that set's rows."""
    rng = np.random.default_rng(9)
    rows = rng.choice(100000, 3000, replace=False)
    counts = rng.integers(1, 6, size=rows.shape[0])  # many ties
    sel = oracle.lfu_select(rows, counts, 40 * 32)
    sets = 40
    for k in range(sets):
        mine = [(-int(c), int(r)) for r, c in zip(rows, counts) if (oracle.splitmix64(int(r)) >> 32) % sets == k]
        want = [r for _, r in sorted(mine)[:32]]
        got = [r for r in sel[k * 32:(k + 1) * 32] if r >= 0]
        assert got == want
    r2, c2 = oracle.lfu_counts([5, 3, 5, 9], np.array([5]))
    assert r2.tolist() == [3, 5, 9] and c2.tolist() == [1, 3, 1]


@pytest.mark.parametrize("mode,weighted", [("sum", True), ("mean", False), ("mean", True)])
def test_trainable_cache_matches_torch_autograd(mode, weighted):
    """Trainable cache rows: a table whose cached rows are separate parameters.  The
    oracle's output, cache gradient and (miss-only) core gradients equal torch
    autograd through the full table with those rows swapped in."""
    rng = np.random.default_rng(13)
    spec = TableSpec(100, [5, 4, 6], [2, 3, 2], [3, 5])
    cores = rand_cores(rng, spec)
    B = 9
    lengths = rng.integers(0, 7, size=B)
    off = np.concatenate([[0], np.cumsum(lengths)])
    hot = np.array([3, 17, 42, 99, 64], dtype=np.int64)
    idx = np.where(rng.random(int(off[-1])) < 0.5, rng.choice(hot, int(off[-1])), rng.integers(0, 100, int(off[-1])))
    w = rng.random(idx.shape[0]) if weighted else None
    go = rng.standard_normal((B, 12))
    cache_rows = np.array([17, -1, 3, 64, 55], dtype=np.int64)  # 55 is never looked up, slot 1 empty
    vals = rng.standard_normal((5, 12))
    gt = [torch.from_numpy(c.copy()).requires_grad_(True) for c in cores]
    cv = torch.from_numpy(vals.copy()).requires_grad_(True)
    full = torch.einsum("xja,yakc,zcl->xyzjkl", gt[0][:, 0], gt[1], gt[2][..., 0]).reshape(120, 12)
    rows = [cv[k] if k >= 0 else full[r] for r, k in
            ((r, list(cache_rows).index(r) if r in cache_rows else -1) for r in range(100))]
    table = torch.stack(rows)
    bag = torch.from_numpy(np.repeat(np.arange(B), lengths))
    wt = torch.ones(idx.shape[0], dtype=torch.float64) if w is None else torch.from_numpy(w)
    if mode == "mean":
        wt = wt / torch.from_numpy(np.maximum(lengths, 1)).double()[bag]
    out = torch.zeros(B, 12, dtype=torch.float64).index_add_(0, bag, wt[:, None] * table[torch.from_numpy(idx)])
    (out * torch.from_numpy(go)).sum().backward()
    np.testing.assert_allclose(oracle.cached_forward([spec], [cores], cache_rows, vals, idx, off, w, mode),
                               out.detach().numpy(), rtol=1e-12, atol=1e-13)
    d, touched = oracle.cache_grad(cache_rows, idx, off, go, w, mode)
    np.testing.assert_allclose(d, cv.grad.numpy(), rtol=1e-12, atol=1e-13)
    assert touched.tolist() == [r in set(idx.tolist()) for r in cache_rows]
    mw = oracle.cache_miss_weights(cache_rows, idx, off, w)
    for k in range(3):
        dG = oracle.backward_core([spec], [cores], idx, off, go, 0, k, weights=mw, mode=mode)
        np.testing.assert_allclose(dG, gt[k].grad.numpy(), rtol=1e-12, atol=1e-13)


def test_trainable_cache_updates_match_torch_optim():
    """The cached values' SGD and Adagrad steps equal torch.optim on a parameter whose
    untouched rows get a zero gradient (with eps > 0 such rows do not move)."""
    rng = np.random.default_rng(14)
    vals = rng.standard_normal((6, 4))
    grad = rng.standard_normal((6, 4))
    touched = np.array([True, False, True, True, False, True])
    grad[~touched] = 0.0
    lr, eps = 0.07, 1e-10
    p = torch.from_numpy(vals.copy()).requires_grad_(True)
    p.grad = torch.from_numpy(grad.copy())
    torch.optim.SGD([p], lr=lr).step()
    np.testing.assert_allclose(oracle.cache_sgd(vals, grad, touched, lr), p.detach().numpy(), rtol=1e-14)
    state0 = rng.uniform(0.0, 1.0, size=vals.shape)
    state0[1] = 0.0  # an untouched row with an empty accumulator stays put
    p = torch.from_numpy(vals.copy()).requires_grad_(True)
    opt = torch.optim.Adagrad([p], lr=lr, eps=eps)
    opt.state[p]["sum"] = torch.from_numpy(state0.copy())
    opt.state[p]["step"] = torch.tensor(0.0)
    p.grad = torch.from_numpy(grad.copy())
    opt.step()
    v, s = oracle.cache_adagrad(vals, state0, grad, touched, lr, eps)
    np.testing.assert_allclose(v, p.detach().numpy(), rtol=1e-13)
    np.testing.assert_allclose(s, opt.state[p]["sum"].numpy(), rtol=1e-13)
