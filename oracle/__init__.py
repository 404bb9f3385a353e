"""Float64 CPU oracle of the TT-EmbeddingBag hot path.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
never loads it, and it imports nothing from the product package.

The TT arithmetic lives in ``tt_oracle.c`` (plain C, float64, definition
written out per lookup, see its header).  This module compiles it with gcc,
promotes the float32 cores to float64 and marshals arrays.  Done here in
numpy: the LFU policy (row hash, counts, per-set selection), the trainable
cache rows (a cached row's value replaces its TT row: the hit terms of the
output and the per-row gradient sums), and the optimizer steps (FBTT README,
"Fused Kernel": the update is applied inside the backward pass; every
gradient is taken at the pre-update cores; "Parameters": optimizer,
learning_rate, eps):

* SGD: ``G <- G - lr dG``;
* Adagrad, element-wise (the pages name the optimizer and its eps but no
  variant; the plainest reading is the textbook one, one accumulator per core
  element): ``s <- s + dG^2``, ``G <- G - lr dG / (sqrt(s) + eps)``.

Tables are any objects with ``num_embeddings``, ``p``, ``q`` and ``ranks``
attributes; cores are ``[p_k, r_{k-1}, q_k, r_k]`` arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tt_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libtt_oracle.so")
_lock = threading.Lock()
_lib = None


class _Table(ctypes.Structure):
    _fields_ = [
        ("E", ctypes.c_int64),
        ("p", ctypes.c_int64 * 3),
        ("q", ctypes.c_int64 * 3),
        ("r", ctypes.c_int64 * 2),
        ("G", ctypes.c_void_p * 3),
    ]


def build(force: bool = False) -> str:
    """Compile ``tt_oracle.c`` into ``oracle/_build/libtt_oracle.so``."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c99", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64p = ctypes.POINTER(ctypes.c_int64)
            lib.tto_num_threads.restype = ctypes.c_int
            lib.tto_decode.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                       i64p, i64p, i64p, i64p, i64p, i64p]
            lib.tto_forward.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                        i64p, i64p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                        ctypes.c_void_p, ctypes.c_void_p]
            lib.tto_backward_core.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                              i64p, i64p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p,
                                              ctypes.c_void_p]
            _lib = lib
    return _lib


def num_threads() -> int:
    """Threads the oracle's OpenMP loops use."""
    return int(_load().tto_num_threads())


def _i64(a):
    return np.ascontiguousarray(a, dtype=np.int64)


def _ptr(a, ctype=ctypes.c_int64):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


class _Tables:
    """ctypes table array with float64 copies of the cores kept alive."""

    def __init__(self, tables, cores):
        if len(tables) != len(cores):
            raise ValueError("one core triple per table")
        self.keep = []
        self.arr = (_Table * len(tables))()
        for t, (spec, cs) in enumerate(zip(tables, cores)):
            tt = self.arr[t]
            tt.E = int(spec.num_embeddings)
            for k in range(3):
                tt.p[k] = int(spec.p[k])
                tt.q[k] = int(spec.q[k])
                g = np.ascontiguousarray(cs[k], dtype=np.float64)
                self.keep.append(g)
                tt.G[k] = g.ctypes.data
            tt.r[0], tt.r[1] = int(spec.ranks[0]), int(spec.ranks[1])


def _bags_per_table(tables, offsets, bags_per_table):
    nb = int(offsets.shape[0] - 1)
    if bags_per_table is None:
        if nb % len(tables):
            raise ValueError("number of bags is not a multiple of the number of tables")
        bags_per_table = nb // len(tables)
    return int(bags_per_table)


def _check(rc, what):
    if rc == 1:
        raise IndexError(f"oracle {what}: index out of range")
    if rc != 0:
        raise ValueError(f"oracle {what}: invalid arguments (code {rc})")


def decode(tables, indices, offsets, bags_per_table=None):
    """(i1, i2, i3, bag) of every lookup, int64 arrays."""
    lib = _load()
    idx, off = _i64(indices), _i64(offsets)
    bpt = _bags_per_table(tables, off, bags_per_table)
    zero = [np.zeros((1, 1, 1, 1)) for _ in range(3)]
    tabs = _Tables(tables, [zero] * len(tables))
    outs = [np.full(idx.shape[0], -1, dtype=np.int64) for _ in range(4)]
    rc = lib.tto_decode(ctypes.byref(tabs.arr), len(tables), bpt, idx.shape[0], _ptr(idx), _ptr(off),
                        *[_ptr(o) for o in outs])
    _check(rc, "decode")
    return tuple(outs)


def forward(tables, cores, indices, offsets, weights=None, mode="sum", bags_per_table=None, bags=None):
    """Pooled output, float64 ``[num_bags or len(bags), D]``."""
    lib = _load()
    idx, off = _i64(indices), _i64(offsets)
    bpt = _bags_per_table(tables, off, bags_per_table)
    tabs = _Tables(tables, cores)
    D = int(np.prod(tables[0].q))
    w = None if weights is None else np.ascontiguousarray(weights, dtype=np.float64)
    sel = None if bags is None else _i64(bags)
    nout = (off.shape[0] - 1) if sel is None else sel.shape[0]
    out = np.zeros((nout, D), dtype=np.float64)
    rc = lib.tto_forward(ctypes.byref(tabs.arr), len(tables), bpt, idx.shape[0], _ptr(idx), _ptr(off),
                         None if w is None else w.ctypes.data, 1 if mode == "mean" else 0,
                         0 if sel is None else sel.shape[0], None if sel is None else sel.ctypes.data,
                         out.ctypes.data)
    _check(rc, "forward")
    return out


def backward_core(tables, cores, indices, offsets, grad_out, table, core, weights=None, mode="sum",
                  bags_per_table=None, slices=None):
    """Gradient of core ``core`` of ``table`` for ``slices`` (default: all).

    Returns float64 ``[len(slices), r_{k-1}, q_k, r_k]``.
    """
    lib = _load()
    idx, off = _i64(indices), _i64(offsets)
    bpt = _bags_per_table(tables, off, bags_per_table)
    tabs = _Tables(tables, cores)
    spec = tables[table]
    rk = [1, int(spec.ranks[0]), int(spec.ranks[1]), 1]
    shape = (rk[core], int(spec.q[core]), rk[core + 1])
    sl = np.arange(int(spec.p[core]), dtype=np.int64) if slices is None else _i64(slices)
    go = np.ascontiguousarray(grad_out, dtype=np.float64)
    w = None if weights is None else np.ascontiguousarray(weights, dtype=np.float64)
    dG = np.zeros((sl.shape[0],) + shape, dtype=np.float64)
    rc = lib.tto_backward_core(ctypes.byref(tabs.arr), len(tables), bpt, idx.shape[0], _ptr(idx), _ptr(off),
                               None if w is None else w.ctypes.data, 1 if mode == "mean" else 0,
                               go.ctypes.data, int(table), int(core), sl.shape[0], sl.ctypes.data,
                               dG.ctypes.data)
    _check(rc, "backward")
    return dG


def sgd_update(G, dG, lr):
    """One SGD step of a block of core elements, float64: ``G - lr dG``."""
    return np.asarray(G, dtype=np.float64) - float(lr) * np.asarray(dG, dtype=np.float64)


def adagrad_update(G, state, dG, lr, eps):
    """One element-wise Adagrad step, float64: ``s + dG^2`` and ``G - lr dG / (sqrt(s + dG^2) + eps)``.

    Returns ``(updated G, updated s)``."""
    dG = np.asarray(dG, dtype=np.float64)
    s_new = np.asarray(state, dtype=np.float64) + dG * dG
    return np.asarray(G, dtype=np.float64) - float(lr) * dG / (np.sqrt(s_new) + float(eps)), s_new


def sgd_slices(tables, cores, indices, offsets, grad_out, lr, table, core, weights=None, mode="sum",
               bags_per_table=None, slices=None):
    """Updated slices ``G_k[s] - lr dG_k[s]`` in float64 (gradients at the pre-update cores)."""
    spec = tables[table]
    sl = np.arange(int(spec.p[core]), dtype=np.int64) if slices is None else _i64(slices)
    dG = backward_core(tables, cores, indices, offsets, grad_out, table, core, weights, mode,
                       bags_per_table, sl)
    return sgd_update(np.asarray(cores[table][core])[sl], dG, lr)


def adagrad_slices(tables, cores, indices, offsets, grad_out, lr, eps, state, table, core, weights=None,
                   mode="sum", bags_per_table=None, slices=None):
    """Element-wise Adagrad on ``slices`` of core ``core`` of ``table``; ``state`` is that core's accumulator.

    Returns float64 ``(updated slices, updated accumulator slices)``.
    """
    spec = tables[table]
    sl = np.arange(int(spec.p[core]), dtype=np.int64) if slices is None else _i64(slices)
    dG = backward_core(tables, cores, indices, offsets, grad_out, table, core, weights, mode,
                       bags_per_table, sl)
    return adagrad_update(np.asarray(cores[table][core])[sl], np.asarray(state)[sl], dG, lr, eps)


def sgd_step(tables, cores, indices, offsets, grad_out, lr, weights=None, mode="sum", bags_per_table=None):
    """Every core of every table after one fused SGD step, float64."""
    return [
        [sgd_slices(tables, cores, indices, offsets, grad_out, lr, t, k, weights, mode, bags_per_table)
         for k in range(3)]
        for t in range(len(tables))
    ]


def workload_forward(w, bags=None, cores=None):
    """``forward`` on a ``tt_inputs.Workload``."""
    return forward(w.tables, cores or w.cores, w.indices, w.offsets, w.weights, w.mode, w.batch, bags)


def workload_backward_core(w, table, core, slices=None, cores=None):
    """``backward_core`` on a ``tt_inputs.Workload``."""
    return backward_core(w.tables, cores or w.cores, w.indices, w.offsets, w.grad_out, table, core,
                         w.weights, w.mode, w.batch, slices)


def workload_adagrad_slices(w, table, core, state, eps, slices=None, cores=None):
    """``adagrad_slices`` on a ``tt_inputs.Workload`` with its learning rate."""
    return adagrad_slices(w.tables, cores or w.cores, w.indices, w.offsets, w.grad_out, w.lr, eps, state, table,
                          core, w.weights, w.mode, w.batch, slices)


def workload_sgd_slices(w, table, core, slices=None, cores=None):
    """``sgd_slices`` on a ``tt_inputs.Workload`` with its learning rate."""
    return sgd_slices(w.tables, cores or w.cores, w.indices, w.offsets, w.grad_out, w.lr, table, core,
                      w.weights, w.mode, w.batch, slices)


# ---------------------------------------------------------------- LFU cache policy
# FBTT README, "Software Cache": access frequencies are counted in a hash table
# during the forward passes; cache_populate() fills a 32-way set-associative
# least-frequently-used cache from them.  Written from those statements and the
# published SplitMix64 definition (the row hash), independently of the library.

_M64 = (1 << 64) - 1
LFU_WAYS = 32


def splitmix64(x: int) -> int:
    """First output of a SplitMix64 generator seeded with x (Steele, Lea and Flood, OOPSLA 2014)."""
    z = (int(x) + 0x9E3779B97F4A7C15) & _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def lfu_counts(*index_arrays):
    """Access count of every row over the given lookups (all forward passes since counting began)."""
    rows, counts = np.unique(np.concatenate([np.asarray(a, dtype=np.int64) for a in index_arrays]),
                             return_counts=True)
    return rows, counts


def lfu_select(rows, counts, cache_size):
    """Cache content per slot (set * 32 + way, -1 = empty): set k holds the 32 most
    frequent rows r with (splitmix64(r) >> 32) mod sets == k, ties to the smaller row."""
    sets = -(-int(cache_size) // LFU_WAYS)
    members = [[] for _ in range(sets)]
    for r, c in zip(np.asarray(rows).tolist(), np.asarray(counts).tolist()):
        members[(splitmix64(r) >> 32) % sets].append((-int(c), int(r)))
    out = np.full(sets * LFU_WAYS, -1, dtype=np.int64)
    for k, m in enumerate(members):
        m.sort()
        for w, (_, r) in enumerate(m[:LFU_WAYS]):
            out[k * LFU_WAYS + w] = r
    return out


# ---------------------------------------------------------------- trainable cache rows
# FBTT README, "Parameters": sparse (backward gives the gradient w.r.t. the TT cores or
# the cache); "Software Cache": a cached row is read from the cache, without
# decompressing it.  Reading: a row that sits in the cache takes the cached value in
# place of its TT row, so the output is linear in the cached values and the cores see
# only the lookups of rows outside the cache.

def _cache_split(cache_rows, indices, offsets, weights, mode):
    """(slot of every lookup or -1, pooling scale, bag) for a single table."""
    idx, off = _i64(indices), _i64(offsets)
    slot_of = {r: k for k, r in enumerate(np.asarray(cache_rows, dtype=np.int64).tolist()) if r >= 0}
    slot = np.array([slot_of.get(r, -1) for r in idx.tolist()], dtype=np.int64)
    lengths = np.diff(off)
    bag = np.repeat(np.arange(lengths.shape[0]), lengths)
    w = np.ones(idx.shape[0]) if weights is None else np.asarray(weights, dtype=np.float64)
    scale = w / np.maximum(lengths[bag], 1) if mode == "mean" else w
    return slot, scale, bag


def cache_miss_weights(cache_rows, indices, offsets, weights=None):
    """Per-sample weights with every cached lookup's weight set to 0: with them the
    plain TT functions give the cores' share of a step (the mean-mode divisor still
    counts every lookup of the bag)."""
    slot, _, _ = _cache_split(cache_rows, indices, offsets, None, "sum")
    w = np.ones(slot.shape[0]) if weights is None else np.asarray(weights, dtype=np.float64)
    return np.where(slot >= 0, 0.0, w)


def cached_forward(tables, cores, cache_rows, cache_vals, indices, offsets, weights=None, mode="sum", bags=None):
    """Pooled output with trainable cache rows, float64 (single table; ``bags``: a subset)."""
    slot, scale, bag = _cache_split(cache_rows, indices, offsets, weights, mode)
    out = forward(tables, cores, indices, offsets, cache_miss_weights(cache_rows, indices, offsets, weights), mode)
    hit = slot >= 0
    np.add.at(out, bag[hit], scale[hit, None] * np.asarray(cache_vals, dtype=np.float64)[slot[hit]])
    return out if bags is None else out[_i64(bags)]


def cache_grad(cache_rows, indices, offsets, grad_out, weights=None, mode="sum"):
    """(dL/d cached value ``[slots, D]``, touched flag per slot): the sum over the lookups
    of each cached row of pooling scale x grad_out of the bag."""
    slot, scale, bag = _cache_split(cache_rows, indices, offsets, weights, mode)
    go = np.asarray(grad_out, dtype=np.float64)
    n = np.asarray(cache_rows).shape[0]
    d = np.zeros((n, go.shape[1]))
    hit = slot >= 0
    np.add.at(d, slot[hit], scale[hit, None] * go[bag[hit]])
    touched = np.zeros(n, dtype=bool)
    touched[slot[hit]] = True
    return d, touched


def cache_sgd(vals, grad, touched, lr):
    """SGD on the touched cached values."""
    v = np.array(vals, dtype=np.float64)
    v[touched] -= float(lr) * grad[touched]
    return v


def cache_adagrad(vals, state, grad, touched, lr, eps):
    """Element-wise Adagrad (the cores' rule) on the touched cached values: (values, state)."""
    v = np.array(vals, dtype=np.float64)
    s = np.array(state, dtype=np.float64)
    s[touched] += grad[touched] ** 2
    v[touched] -= float(lr) * grad[touched] / (np.sqrt(s[touched]) + float(eps))
    return v, s
