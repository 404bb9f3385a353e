"""GB300 (sm_103a) TT-EmbeddingBag: Python binding of libttemb.so.

A drop-in EmbeddingBag whose E x D table is stored as three tensor-train cores
(TT-Rec / FBTT-Embedding pages).  Every step of the computation runs in the
CUDA kernels of ``libttemb.so``; this module only marshals arguments: torch
supplies device memory and the current stream.  There is no CPU fallback:
without the built library every call raises.

Low-level functions carry the C ABI's names (``include/tt_emb.h``):
``tt_emb_create``, ``tt_emb_batch_create``, ``tt_emb_forward``,
``tt_emb_backward``, ``tt_emb_cache_populate`` ...  ``TTEmbeddingBag`` and
``TableBatchedTTEmbeddingBag`` wrap them as ``torch.nn.Module`` s.  With
``sparse=True`` (default) the backward pass applies the fused update (SGD or
Adagrad) to the cores and returns no gradient for them (FBTT README, "Fused
Kernel"); with ``sparse=False`` the cores' gradients are returned to autograd
for an external optimizer (FBTT README, "Parameters": sparse).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import List, Optional, Sequence

import torch

from ._nvcc_build import LIB as _LIB_RELEASE
from ._nvcc_build import LIB_DEBUG as _LIB_DEBUG
from ._nvcc_build import build, build_all

# TTEMB_DEBUG=1 loads the debug library (index checks in the kernels, TT_ERR_BOUNDS)
_LIB_PATH = _LIB_DEBUG if os.environ.get("TTEMB_DEBUG") == "1" else _LIB_RELEASE

__all__ = [
    "TTError",
    "build",
    "build_all",
    "suggested_tt_shapes",
    "tt_init_cores",
    "load_library",
    "library_path",
    "tt_emb_create",
    "tt_emb_batch_create",
    "tt_emb_destroy",
    "tt_emb_reserve",
    "tt_emb_forward",
    "tt_emb_backward",
    "tt_emb_set_optimizer",
    "tt_emb_full_weight",
    "tt_emb_lfu_enable",
    "tt_emb_lfu_populate",
    "tt_emb_lfu_read",
    "tt_emb_lfu_cached_rows",
    "tt_emb_lfu_disable",
    "tt_emb_cache_populate",
    "tt_emb_cache_disable",
    "tt_emb_cache_set_trainable",
    "tt_emb_cache_read",
    "tt_emb_cache_write",
    "tt_emb_get_decoded",
    "tt_emb_get_last_error",
    "tt_emb_set_stage_timing",
    "tt_emb_stage_times",
    "tt_emb_last_launch_count",
    "tt_emb_status_string",
    "tt_emb_forward_noalloc",
    "tt_emb_apply_gradients",
    "tt_emb_set_wait_limit",
    "shard_bags",
    "DataParallelStep",
    "EXPORTED_SYMBOLS",
    "TTEmbeddingBag",
    "TableBatchedTTEmbeddingBag",
]

TT_OK, TT_ERR_ARG, TT_ERR_SHAPE, TT_ERR_INDEX, TT_ERR_CUDA, TT_ERR_STATE, TT_ERR_TIMEOUT, TT_ERR_NOMEM, TT_ERR_BOUNDS = range(9)
TT_POOL_SUM, TT_POOL_MEAN = 0, 1
TT_OPT_SGD, TT_OPT_ADAGRAD, TT_OPT_GRAD = 0, 1, 2

EXPORTED_SYMBOLS = (
    "tt_emb_create",
    "tt_emb_batch_create",
    "tt_emb_destroy",
    "tt_emb_reserve",
    "tt_emb_forward",
    "tt_emb_backward",
    "tt_emb_set_optimizer",
    "tt_emb_full_weight",
    "tt_emb_lfu_enable",
    "tt_emb_lfu_populate",
    "tt_emb_lfu_read",
    "tt_emb_lfu_cached_rows",
    "tt_emb_lfu_disable",
    "tt_emb_cache_populate",
    "tt_emb_cache_disable",
    "tt_emb_cache_set_trainable",
    "tt_emb_cache_read",
    "tt_emb_cache_write",
    "tt_emb_get_decoded",
    "tt_emb_get_last_error",
    "tt_emb_set_stage_timing",
    "tt_emb_stage_times",
    "tt_emb_last_launch_count",
    "tt_emb_status_string",
    "tt_emb_forward_noalloc",
    "tt_emb_apply_gradients",
    "tt_emb_set_wait_limit",
)


class TTError(RuntimeError):
    """A tt_status other than TT_OK."""

    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {tt_emb_status_string(code)} (tt_status {code})")


class _Desc(ctypes.Structure):
    _fields_ = [
        ("num_embeddings", ctypes.c_int64),
        ("p", ctypes.c_int64 * 3),
        ("q", ctypes.c_int32 * 3),
        ("ranks", ctypes.c_int32 * 2),
        ("cores_dev", ctypes.c_void_p * 3),
    ]


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libttemb.so (it must have been built with ``build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build it with "
                "tensor_train_compressed_embeddingbag_gb300.build() (nvcc, sm_103a)"
            )
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        sig = {
            "tt_emb_create": (ctypes.c_int, [i64, ctypes.POINTER(i64), ctypes.POINTER(i32), ctypes.POINTER(i32),
                                             ctypes.POINTER(vp), ctypes.POINTER(vp)]),
            "tt_emb_batch_create": (ctypes.c_int, [i32, ctypes.POINTER(_Desc), ctypes.POINTER(vp)]),
            "tt_emb_destroy": (None, [vp]),
            "tt_emb_reserve": (ctypes.c_int, [vp, i64, i64]),
            "tt_emb_forward": (ctypes.c_int, [vp, vp, i64, vp, i64, vp, ctypes.c_int, vp, vp]),
            "tt_emb_backward": (ctypes.c_int, [vp, vp, f32, vp]),
            "tt_emb_set_optimizer": (ctypes.c_int, [vp, i32, f32, ctypes.POINTER(vp)]),
            "tt_emb_full_weight": (ctypes.c_int, [vp, i32, i64, i64, vp, vp]),
            "tt_emb_lfu_enable": (ctypes.c_int, [vp, i64, i64]),
            "tt_emb_lfu_populate": (ctypes.c_int, [vp, vp]),
            "tt_emb_lfu_read": (ctypes.c_int, [vp, vp, vp, i64, ctypes.POINTER(i64)]),
            "tt_emb_lfu_cached_rows": (ctypes.c_int, [vp, vp, i64, ctypes.POINTER(i64)]),
            "tt_emb_lfu_disable": (ctypes.c_int, [vp]),
            "tt_emb_cache_populate": (ctypes.c_int, [vp, vp, i64, vp]),
            "tt_emb_cache_disable": (ctypes.c_int, [vp]),
            "tt_emb_cache_set_trainable": (ctypes.c_int, [vp, i32, vp]),
            "tt_emb_cache_read": (ctypes.c_int, [vp, vp, vp, vp]),
            "tt_emb_cache_write": (ctypes.c_int, [vp, vp, vp]),
            "tt_emb_get_decoded": (ctypes.c_int, [vp, vp, vp, vp, vp, vp, vp]),
            "tt_emb_get_last_error": (ctypes.c_int, [vp]),
            "tt_emb_set_stage_timing": (ctypes.c_int, [vp, ctypes.c_int]),
            "tt_emb_stage_times": (ctypes.c_int, [vp, ctypes.c_int, ctypes.POINTER(f32),
                                                  ctypes.POINTER(ctypes.c_char_p), ctypes.c_int]),
            "tt_emb_last_launch_count": (ctypes.c_int, [vp, ctypes.c_int]),
            "tt_emb_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "tt_emb_forward_noalloc": (ctypes.c_int, [i64, ctypes.POINTER(i64), ctypes.POINTER(i32),
                                                      ctypes.POINTER(i32), ctypes.POINTER(vp), vp, i64, vp, i64,
                                                      vp, ctypes.c_int, vp, vp, vp]),
            "tt_emb_apply_gradients": (ctypes.c_int, [vp, i32, f32, f32, ctypes.POINTER(vp), ctypes.POINTER(vp), vp]),
            "tt_emb_set_wait_limit": (ctypes.c_int, [vp, ctypes.c_uint32]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(st: int, what: str):
    if st != TT_OK:
        raise TTError(st, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _cuda_f32(t: torch.Tensor, what: str):
    if not (t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()):
        raise TTError(TT_ERR_ARG, f"{what} must be a contiguous float32 CUDA tensor")


def tt_emb_status_string(code: int) -> str:
    return load_library().tt_emb_status_string(int(code)).decode()


def tt_emb_create(num_embeddings: int, p: Sequence[int], q: Sequence[int], ranks: Sequence[int],
                  cores: Sequence[torch.Tensor]) -> ctypes.c_void_p:
    lib = load_library()
    for k, c in enumerate(cores):
        _cuda_f32(c, f"core {k}")
    h = ctypes.c_void_p()
    ptrs = (ctypes.c_void_p * 3)(*[c.data_ptr() for c in cores])
    st = lib.tt_emb_create(int(num_embeddings), (ctypes.c_int64 * 3)(*p), (ctypes.c_int32 * 3)(*q),
                           (ctypes.c_int32 * 2)(*ranks), ptrs, ctypes.byref(h))
    _check(st, "tt_emb_create")
    return h


def tt_emb_batch_create(tables) -> ctypes.c_void_p:
    """tables: sequence of (num_embeddings, p, q, ranks, cores)."""
    lib = load_library()
    arr = (_Desc * len(tables))()
    for i, (E, p, q, r, cores) in enumerate(tables):
        for k, c in enumerate(cores):
            _cuda_f32(c, f"table {i} core {k}")
        arr[i].num_embeddings = int(E)
        for k in range(3):
            arr[i].p[k] = int(p[k])
            arr[i].q[k] = int(q[k])
            arr[i].cores_dev[k] = cores[k].data_ptr()
        arr[i].ranks[0], arr[i].ranks[1] = int(r[0]), int(r[1])
    h = ctypes.c_void_p()
    _check(lib.tt_emb_batch_create(len(tables), arr, ctypes.byref(h)), "tt_emb_batch_create")
    return h


def tt_emb_destroy(h):
    if h:
        load_library().tt_emb_destroy(h)


def tt_emb_reserve(h, max_nnz: int, max_bags: int):
    _check(load_library().tt_emb_reserve(h, int(max_nnz), int(max_bags)), "tt_emb_reserve")


def tt_emb_forward(h, indices: torch.Tensor, offsets: torch.Tensor, weights: Optional[torch.Tensor], mode: int,
                   out: torch.Tensor, stream=None):
    """indices int64 [nnz], offsets int64 [num_bags + 1] (CSR), out float32 [num_bags, D]."""
    nb = offsets.numel() - 1
    st = load_library().tt_emb_forward(h, _ptr(indices), indices.numel(), _ptr(offsets), nb, _ptr(weights),
                                       int(mode), _ptr(out), _stream(stream))
    _check(st, "tt_emb_forward")


def tt_emb_backward(h, grad_out: torch.Tensor, lr: float, stream=None):
    _check(load_library().tt_emb_backward(h, _ptr(grad_out), float(lr), _stream(stream)), "tt_emb_backward")


def tt_emb_set_optimizer(h, optim: int, eps: float = 0.0, aux: Optional[Sequence[torch.Tensor]] = None):
    """What tt_emb_backward does with the core gradients (TT_OPT_SGD / TT_OPT_ADAGRAD / TT_OPT_GRAD).

    aux: 3 * num_tables float32 device tensors shaped like the cores (table-major):
    the Adagrad accumulators, or the gradient buffers for TT_OPT_GRAD.
    """
    arr = None
    if aux is not None:
        for t in aux:
            _cuda_f32(t, "aux")
        arr = (ctypes.c_void_p * len(aux))(*[t.data_ptr() for t in aux])
    _check(load_library().tt_emb_set_optimizer(h, int(optim), float(eps), arr), "tt_emb_set_optimizer")


def tt_emb_full_weight(h, table: int, row0: int, nrows: int, out: torch.Tensor, stream=None):
    """Rows [row0, row0 + nrows) of `table` as dense float [nrows][D] into `out`."""
    _cuda_f32(out, "out")
    if out.numel() < nrows * (out.shape[-1] if out.dim() else 0):
        raise TTError(TT_ERR_ARG, "out is too small")
    _check(load_library().tt_emb_full_weight(h, int(table), int(row0), int(nrows), _ptr(out), _stream(stream)),
           "tt_emb_full_weight")


def tt_emb_lfu_enable(h, cache_size: int, hashtbl_size: int):
    """Count row accesses in every forward pass and size a 32-way set-associative LFU cache."""
    _check(load_library().tt_emb_lfu_enable(h, int(cache_size), int(hashtbl_size)), "tt_emb_lfu_enable")


def tt_emb_lfu_populate(h, stream=None):
    """Rebuild the cache from the access counts (per set: the 32 most frequent rows)."""
    _check(load_library().tt_emb_lfu_populate(h, _stream(stream)), "tt_emb_lfu_populate")


def tt_emb_lfu_read(h):
    """(rows, counts) of the frequency table, sorted by row (numpy int64 / uint32)."""
    import numpy as np
    lib = load_library()
    n = ctypes.c_int64()
    _check(lib.tt_emb_lfu_read(h, None, None, 0, ctypes.byref(n)), "tt_emb_lfu_read")
    rows = np.empty(n.value, dtype=np.int64)
    counts = np.empty(n.value, dtype=np.uint32)
    _check(lib.tt_emb_lfu_read(h, rows.ctypes.data, counts.ctypes.data, n.value, ctypes.byref(n)), "tt_emb_lfu_read")
    return rows, counts


def tt_emb_lfu_cached_rows(h):
    """The cache's row per slot (set * 32 + way; -1 = empty), numpy int64."""
    import numpy as np
    lib = load_library()
    n = ctypes.c_int64()
    _check(lib.tt_emb_lfu_cached_rows(h, None, 0, ctypes.byref(n)), "tt_emb_lfu_cached_rows")
    rows = np.empty(n.value, dtype=np.int64)
    _check(lib.tt_emb_lfu_cached_rows(h, rows.ctypes.data, n.value, ctypes.byref(n)), "tt_emb_lfu_cached_rows")
    return rows


def tt_emb_lfu_disable(h):
    _check(load_library().tt_emb_lfu_disable(h), "tt_emb_lfu_disable")


def tt_emb_cache_populate(h, rows: torch.Tensor, stream=None):
    _check(load_library().tt_emb_cache_populate(h, _ptr(rows), rows.numel(), _stream(stream)), "tt_emb_cache_populate")


def tt_emb_cache_disable(h):
    _check(load_library().tt_emb_cache_disable(h), "tt_emb_cache_disable")


def tt_emb_cache_set_trainable(h, trainable: bool, stream=None):
    _check(load_library().tt_emb_cache_set_trainable(h, 1 if trainable else 0, _stream(stream)),
           "tt_emb_cache_set_trainable")


def tt_emb_cache_read(h, vals: Optional[torch.Tensor], grads: Optional[torch.Tensor] = None, stream=None):
    """Copy the cached values (and, trainable rows, their last gradients) into [slots, D] fp32 CUDA tensors."""
    _check(load_library().tt_emb_cache_read(h, _ptr(vals), _ptr(grads), _stream(stream)), "tt_emb_cache_read")


def tt_emb_cache_write(h, vals: torch.Tensor, stream=None):
    """Overwrite the trainable cached values from a [slots, D] fp32 CUDA tensor."""
    _check(load_library().tt_emb_cache_write(h, _ptr(vals), _stream(stream)), "tt_emb_cache_write")


def tt_emb_get_decoded(h, nnz: int, device, stream=None):
    """(table, i1, i2, i3, bag) int32 CUDA tensors of the last forward pass."""
    outs = [torch.empty(nnz, dtype=torch.int32, device=device) for _ in range(5)]
    _check(load_library().tt_emb_get_decoded(h, *[_ptr(o) for o in outs], _stream(stream)), "tt_emb_get_decoded")
    return tuple(outs)


def tt_emb_get_last_error(h) -> int:
    return int(load_library().tt_emb_get_last_error(h))


def tt_emb_set_stage_timing(h, enable: bool):
    _check(load_library().tt_emb_set_stage_timing(h, 1 if enable else 0), "tt_emb_set_stage_timing")


def tt_emb_stage_times(h, which: int, cap: int = 16):
    """[(kernel name, ms), ...] of the last forward (0) or backward (1) call."""
    ms = (ctypes.c_float * cap)()
    names = (ctypes.c_char_p * cap)()
    n = load_library().tt_emb_stage_times(h, int(which), ms, names, cap)
    if n < 0:
        raise TTError(TT_ERR_CUDA, "tt_emb_stage_times")
    return [(names[i].decode() if names[i] else "?", float(ms[i])) for i in range(min(n, cap)) if names[i]]


def tt_emb_last_launch_count(h, which: int) -> int:
    return int(load_library().tt_emb_last_launch_count(h, int(which)))


def tt_emb_forward_noalloc(num_embeddings: int, p: Sequence[int], q: Sequence[int], ranks: Sequence[int],
                           cores: Sequence[torch.Tensor], indices: torch.Tensor, offsets: torch.Tensor,
                           weights: Optional[torch.Tensor], mode: int, out: torch.Tensor,
                           err: Optional[torch.Tensor] = None, stream=None):
    """Forward pass without a handle that allocates no device memory (see include/tt_emb.h).

    For callers that cannot allocate device memory: every buffer, including
    ``out`` and the optional int32 error word ``err``, is the caller's.
    """
    ptrs = (ctypes.c_void_p * 3)(*[c.data_ptr() for c in cores])
    st = load_library().tt_emb_forward_noalloc(
        int(num_embeddings), (ctypes.c_int64 * 3)(*p), (ctypes.c_int32 * 3)(*q), (ctypes.c_int32 * 2)(*ranks),
        ptrs, _ptr(indices), indices.numel(), _ptr(offsets), offsets.numel() - 1, _ptr(weights), int(mode),
        _ptr(out), _ptr(err), _stream(stream))
    _check(st, "tt_emb_forward_noalloc")


def tt_emb_apply_gradients(h, optim: int, lr: float, grads: Sequence[torch.Tensor],
                           state: Optional[Sequence[torch.Tensor]] = None, eps: float = 0.0, stream=None):
    """The update of the cores from summed gradients (TT_OPT_SGD or TT_OPT_ADAGRAD).

    grads / state: 3 * num_tables float32 device tensors shaped like the cores
    (table-major); elements with a zero summed gradient keep their bits."""
    for t in grads:
        _cuda_f32(t, "grads")
    garr = (ctypes.c_void_p * len(grads))(*[t.data_ptr() for t in grads])
    sarr = None
    if state is not None:
        for t in state:
            _cuda_f32(t, "state")
        sarr = (ctypes.c_void_p * len(state))(*[t.data_ptr() for t in state])
    _check(load_library().tt_emb_apply_gradients(h, int(optim), float(lr), float(eps), garr, sarr, _stream(stream)),
           "tt_emb_apply_gradients")


def tt_emb_set_wait_limit(h, polls: int):
    """Polls before a bounded device wait gives up (default 2^24; 0 exercises the give-up path)."""
    _check(load_library().tt_emb_set_wait_limit(h, int(polls)), "tt_emb_set_wait_limit")


# ---------------------------------------------------------------- data-parallel step


def shard_bags(offsets, num_tables: int, rank: int, world: int):
    """This rank's share of a batch (host arrays, bags table-major).

    Every table's B bags are split into `world` contiguous ranges of near-equal
    size; rank r takes range r of every table.  Returns ``(bag ids, lookup ids,
    rebased CSR offsets)`` as numpy int64 arrays: the rank's bags in table-major
    order, the positions of their lookups in the full batch, and the offsets of
    the rank's own [len(bag ids) + 1] CSR layout.  Slicing indices, weights and
    grad_out with them gives the rank's call arguments."""
    import numpy as np

    off = np.asarray(offsets, dtype=np.int64)
    nb = off.shape[0] - 1
    if num_tables < 1 or nb % num_tables or not (0 <= rank < world):
        raise ValueError("bags must be a multiple of the tables and 0 <= rank < world")
    B = nb // num_tables
    b0, b1 = (B * rank) // world, (B * (rank + 1)) // world
    bags = np.concatenate([np.arange(t * B + b0, t * B + b1, dtype=np.int64) for t in range(num_tables)])
    lens = off[bags + 1] - off[bags]
    look = np.concatenate([np.arange(off[g], off[g + 1], dtype=np.int64) for g in bags]) if bags.size else \
        np.zeros(0, dtype=np.int64)
    return bags, look, np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)


class DataParallelStep:
    """One data-parallel training step of a handle whose cores are replicated on
    every rank: the rank's share of the bags runs forward and backward with the
    gradients written out (TT_OPT_GRAD), one all-reduce (sum) of a flat buffer
    holding every core's gradient goes over ``torch.distributed``, and every
    rank applies the same update (``tt_emb_apply_gradients``).  The cores then
    equal one fused step over the whole batch up to the order of summation.

    optim: TT_OPT_SGD or TT_OPT_ADAGRAD (``state``: the accumulators, shaped like
    the cores, table-major)."""

    def __init__(self, h, cores: Sequence[torch.Tensor], optim: int = TT_OPT_SGD, eps: float = 0.0,
                 state: Optional[Sequence[torch.Tensor]] = None, group=None):
        if optim not in (TT_OPT_SGD, TT_OPT_ADAGRAD):
            raise TTError(TT_ERR_ARG, "DataParallelStep optim")
        self.h, self.optim, self.eps, self.state, self.group = h, optim, float(eps), state, group
        sizes = [c.numel() for c in cores]
        # every gradient view starts 16-byte aligned inside the one flat buffer
        pad = [(-n) % 4 for n in sizes]
        self.flat = torch.zeros(sum(n + p for n, p in zip(sizes, pad)), dtype=torch.float32, device=cores[0].device)
        self.grads, o = [], 0
        for c, n, p in zip(cores, sizes, pad):
            self.grads.append(self.flat[o:o + n].view(c.shape))
            o += n + p
        tt_emb_set_optimizer(h, TT_OPT_GRAD, 0.0, self.grads)

    def __call__(self, indices, offsets, weights, mode: int, out, grad_out, lr: float, stream=None):
        import torch.distributed as dist

        tt_emb_forward(self.h, indices, offsets, weights, mode, out, stream)
        tt_emb_backward(self.h, grad_out, lr, stream)
        if dist.is_available() and dist.is_initialized() and dist.get_world_size(self.group) > 1:
            s = torch.cuda.current_stream() if stream is None else stream
            with torch.cuda.stream(s):
                dist.all_reduce(self.flat, op=dist.ReduceOp.SUM, group=self.group)
        tt_emb_apply_gradients(self.h, self.optim, lr, self.grads, self.state, self.eps, stream)


# ---------------------------------------------------------------- modules


WEIGHT_DISTS = ("uniform", "naive-uniform", "approx-uniform", "normal", "approx-normal")


def suggested_tt_shapes(num_embeddings: int, embedding_dim: int):
    """Factor E and D when tt_p_shapes / tt_q_shapes are None (FBTT README, "Initialization").

    The pages ask only that prod(p) >= E and prod(q) == D.  Read here as the
    balanced choice: p1 = p2 = max(1, round(E^(1/3))), p3 = ceil(E / (p1 p2));
    q = the three factors of D with product exactly D whose largest factor is
    smallest (then whose smallest factor is largest), in ascending order
    (64 -> [4, 4, 4], 128 -> [4, 4, 8]).
    """
    E, D = int(num_embeddings), int(embedding_dim)
    if E < 1 or D < 1:
        raise ValueError("num_embeddings and embedding_dim must be positive")
    c = max(1, int(round(E ** (1.0 / 3.0))))
    p = [c, c, -(-E // (c * c))]
    best = None
    for a in range(1, D + 1):
        if D % a:
            continue
        for b in range(a, D // a + 1):
            if (D // a) % b:
                continue
            cc = D // (a * b)
            if cc < b:
                continue
            key = (cc, -a)
            if best is None or key < best[0]:
                best = (key, [a, b, cc])
    return p, best[1]


def tt_init_cores(p: Sequence[int], q: Sequence[int], ranks: Sequence[int], weight_dist: str = "normal",
                  sigma: float = 1.0, generator: Optional[torch.Generator] = None, device=None) -> List[torch.Tensor]:
    """Initial cores [p_k, r_{k-1}, q_k, r_k] (FBTT README, "Parameters": weight_dist).

    sigma is the standard deviation of the target distribution X: N(0, sigma^2)
    or U(-sqrt(3) sigma, sqrt(3) sigma).  Readings of the pages:
      "normal", "uniform"   cores i.i.d. from X;
      "approx-normal"       cores i.i.d. N(0, s^2), s^6 r1 r2 = sigma^2, so a full-table
                            entry (a sum of r1 r2 products of three core entries) has X's
                            mean and variance and is near-normal;
      "approx-uniform"      cores i.i.d. U(-c, c), (c^2 / 3)^3 r1 r2 = sigma^2 (X's mean
                            and variance for the full-table entries);
      "naive-uniform"       cores i.i.d. U(-b, b), b^3 = sqrt(3) sigma: X's bound split
                            evenly over the three cores, ignoring the r1 r2 summed terms.
    """
    dist = weight_dist.lower()
    if dist not in WEIGHT_DISTS:
        raise ValueError(f"weight_dist must be one of {WEIGHT_DISTS}")
    r = [1, int(ranks[0]), int(ranks[1]), 1]
    shapes = [(int(p[k]), r[k], int(q[k]), r[k + 1]) for k in range(3)]
    terms = r[1] * r[2]
    sigma = float(sigma)
    out = []
    for sh in shapes:
        if dist == "normal":
            t = torch.randn(sh, generator=generator) * sigma
        elif dist == "approx-normal":
            t = torch.randn(sh, generator=generator) * (sigma ** 2 / terms) ** (1.0 / 6.0)
        else:
            if dist == "uniform":
                bound = 3.0 ** 0.5 * sigma
            elif dist == "approx-uniform":
                bound = 3.0 ** 0.5 * (sigma ** 2 / terms) ** (1.0 / 6.0)
            else:
                bound = (3.0 ** 0.5 * sigma) ** (1.0 / 3.0)
            t = (torch.rand(sh, generator=generator) * 2.0 - 1.0) * bound
        out.append(t.to(device=device, dtype=torch.float32).contiguous())
    return out


def _csr_offsets(offsets: torch.Tensor, nnz: int, include_last_offset: bool) -> torch.Tensor:
    offsets = offsets.to(torch.int64).contiguous()
    if include_last_offset:
        return offsets
    tail = torch.full((1,), nnz, dtype=torch.int64, device=offsets.device)
    return torch.cat([offsets, tail])


class _TTBagFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, module, indices, offsets, weights, mode, *cores):
        D = module.embedding_dim
        out = torch.empty((offsets.numel() - 1, D), dtype=torch.float32, device=indices.device)
        tt_emb_forward(module._h, indices, offsets, weights, mode, out)
        ctx.module = module
        return out

    @staticmethod
    def backward(ctx, grad_out):
        m = ctx.module
        tt_emb_backward(m._h, grad_out.contiguous(), m.learning_rate)
        if m.sparse:  # fused update: no gradient leaves the module
            return (None,) * (5 + len(m._core_list()))
        return (None,) * 5 + tuple(m._grad_bufs)


class _TTBase(torch.nn.Module):
    _h = None
    sparse = True

    def _core_list(self) -> List[torch.Tensor]:
        raise NotImplementedError

    def _set_optimizer(self, sparse: bool, optimizer: str, eps: float):
        """FBTT README, "Parameters": sparse, optimizer, eps."""
        opt = optimizer.lower()
        if opt not in ("sgd", "adagrad"):
            raise ValueError("optimizer must be 'sgd' or 'adagrad'")
        self.sparse, self.optimizer, self.eps = bool(sparse), opt, float(eps)
        self._grad_bufs = []
        if not self.sparse:
            self._grad_bufs = [torch.zeros_like(c) for c in self._core_list()]
            tt_emb_set_optimizer(self._h, TT_OPT_GRAD, 0.0, self._grad_bufs)
        elif opt == "adagrad":
            for i, c in enumerate(self._core_list()):
                self.register_buffer(f"adagrad_state{i}", torch.zeros_like(c.detach()))
            tt_emb_set_optimizer(self._h, TT_OPT_ADAGRAD, self.eps, self.adagrad_states())
        else:
            tt_emb_set_optimizer(self._h, TT_OPT_SGD)

    def adagrad_states(self) -> List[torch.Tensor]:
        """The per-element Adagrad accumulators, one per core (sparse=True, optimizer='adagrad')."""
        return [getattr(self, f"adagrad_state{i}") for i in range(len(self._core_list()))]

    def _run(self, indices, offsets, per_sample_weights, mode, include_last_offset):
        if mode not in ("sum", "mean"):
            raise ValueError("mode must be 'sum' or 'mean'")
        indices = indices.to(torch.int64).contiguous()
        offsets = _csr_offsets(offsets, indices.numel(), include_last_offset)
        w = None if per_sample_weights is None else per_sample_weights.to(torch.float32).contiguous()
        return _TTBagFunction.apply(self, indices, offsets, w, TT_POOL_MEAN if mode == "mean" else TT_POOL_SUM,
                                    *self._core_list())

    def last_error(self) -> int:
        return tt_emb_get_last_error(self._h)

    def __del__(self):
        try:
            if self._h:
                tt_emb_destroy(self._h)
                self._h = None
        except Exception:
            pass


class TTEmbeddingBag(_TTBase):
    """TT-compressed EmbeddingBag (FBTT README, "Parameters" and "Fused Kernel").

    sparse=True fuses the update (optimizer 'sgd' or 'adagrad', learning_rate,
    eps) into the backward pass; sparse=False returns the cores' gradients.

    use_cache: a hot-row cache, filled by ``cache_populate()`` (with ``cache_size``
    rows by the LFU policy, or the given ``cache_rows``).  cache_trainable=True
    (FBTT's cache): cached rows are parameters of their own, initialised from the
    cores; their gradient updates them with the module's optimizer (sparse=True)
    or is read with ``cache_grad()`` (sparse=False).  False: cached rows are exact
    copies of TT rows and all gradients go to the cores.

    cores: optional initial cores ``[G1, G2, G3]`` with shapes
    ``[p_k, r_{k-1}, q_k, r_k]``; default i.i.d. N(0, sigma).
    """

    def __init__(self, num_embeddings: int, embedding_dim: int, tt_ranks: Sequence[int],
                 tt_p_shapes: Optional[Sequence[int]] = None, tt_q_shapes: Optional[Sequence[int]] = None,
                 learning_rate: float = 0.1, cores: Optional[Sequence[torch.Tensor]] = None, sigma: float = 0.1,
                 device=None, use_cache: bool = False, cache_rows: Optional[torch.Tensor] = None,
                 sparse: bool = True, optimizer: str = "sgd", eps: float = 1.0e-10, weight_dist: str = "normal",
                 generator: Optional[torch.Generator] = None, cache_size: int = 0, hashtbl_size: int = 0,
                 cache_trainable: bool = True):
        super().__init__()
        device = torch.device(device or "cuda")
        if tt_p_shapes is None or tt_q_shapes is None:
            ps, qs = suggested_tt_shapes(num_embeddings, embedding_dim)
            tt_p_shapes = ps if tt_p_shapes is None else tt_p_shapes
            tt_q_shapes = qs if tt_q_shapes is None else tt_q_shapes
        q = list(tt_q_shapes)
        if q[0] * q[1] * q[2] != embedding_dim:
            raise ValueError("prod(tt_q_shapes) must equal embedding_dim")
        self.num_embeddings, self.embedding_dim = int(num_embeddings), int(embedding_dim)
        self.p, self.q, self.ranks = list(tt_p_shapes), q, list(tt_ranks)
        self.learning_rate = float(learning_rate)
        r = [1, self.ranks[0], self.ranks[1], 1]
        shapes = [(self.p[k], r[k], q[k], r[k + 1]) for k in range(3)]
        if cores is None:
            cores = tt_init_cores(self.p, q, self.ranks, weight_dist, sigma, generator, device)
        self.G1, self.G2, self.G3 = (
            torch.nn.Parameter(c.to(device=device, dtype=torch.float32).contiguous().clone()) for c in cores
        )
        for k, c in enumerate(self._core_list()):
            if tuple(c.shape) != shapes[k]:
                raise ValueError(f"core {k} has shape {tuple(c.shape)}, expected {shapes[k]}")
        self._h = tt_emb_create(self.num_embeddings, self.p, self.q, self.ranks, self._core_list())
        self._set_optimizer(sparse, optimizer, eps)
        self.cache_trainable = bool(use_cache and cache_trainable)
        if self.cache_trainable:
            tt_emb_cache_set_trainable(self._h, True)
        if use_cache and cache_rows is not None:
            self.cache_populate(cache_rows)
        elif use_cache and cache_size > 0:
            # FBTT README, "Software Cache": count accesses, cache the most frequent rows on populate
            hsize = hashtbl_size if hashtbl_size > 0 else max(32, 4 * cache_size)
            hsize = 1 << max(5, (int(hsize) - 1).bit_length())
            tt_emb_lfu_enable(self._h, cache_size, hsize)

    def _core_list(self):
        return [self.G1, self.G2, self.G3]

    def full_weight(self, row0: int = 0, nrows: Optional[int] = None) -> torch.Tensor:
        """Rows [row0, row0 + nrows) of the E x D table, expanded from the cores (default: all rows)."""
        n = self.num_embeddings - row0 if nrows is None else int(nrows)
        out = torch.empty((n, self.embedding_dim), dtype=torch.float32, device=self.G1.device)
        tt_emb_full_weight(self._h, 0, row0, n, out)
        return out

    def cache_populate(self, rows: Optional[torch.Tensor] = None):
        """Fill the hot-row cache (FBTT README, "Software Cache"): with `rows`, exactly those
        rows; without, by the LFU policy from the access counts of the forward passes so far."""
        if rows is None:
            tt_emb_lfu_populate(self._h)
        else:
            tt_emb_cache_populate(self._h, rows.to(torch.int64).contiguous())

    def cache_rows(self):
        """Row per cache slot (set * 32 + way for the LFU policy; -1 = empty), numpy int64."""
        return tt_emb_lfu_cached_rows(self._h)

    def cache_values(self) -> torch.Tensor:
        """Copy of the cached values, [slots, embedding_dim]."""
        out = torch.empty((self.cache_rows().shape[0], self.embedding_dim), dtype=torch.float32, device=self.G1.device)
        tt_emb_cache_read(self._h, out)
        return out

    def cache_grad(self) -> torch.Tensor:
        """Gradient of the cached values from the last backward (sparse=False, trainable cache)."""
        out = torch.empty((self.cache_rows().shape[0], self.embedding_dim), dtype=torch.float32, device=self.G1.device)
        tt_emb_cache_read(self._h, None, out)
        return out

    def cache_write(self, vals: torch.Tensor):
        """Set the trainable cached values (an external optimizer's step, sparse=False)."""
        tt_emb_cache_write(self._h, vals.to(device=self.G1.device, dtype=torch.float32).contiguous())

    def forward(self, input, offsets, per_sample_weights=None, mode: str = "sum", include_last_offset=False):
        return self._run(input, offsets, per_sample_weights, mode, include_last_offset)


class TableBatchedTTEmbeddingBag(_TTBase):
    """Several TT tables in one call (FBTT README, "TableBatchedTTEmbeddingBag").

    tables: sequence of dicts with num_embeddings, ranks, optional p and q (None:
    suggested_tt_shapes, which then needs embedding_dim) and optional cores.
    Bags are ordered table-major: offsets cover num_tables * B bags, bag
    t * B + b is sample b of table t; the output is [num_tables * B, D].
    """

    def __init__(self, tables, learning_rate: float = 0.1, sigma: float = 0.1, device=None,
                 sparse: bool = True, optimizer: str = "sgd", eps: float = 1.0e-10, weight_dist: str = "normal",
                 generator: Optional[torch.Generator] = None):
        super().__init__()
        device = torch.device(device or "cuda")
        self.learning_rate = float(learning_rate)
        self.specs = []
        params = []
        for i, t in enumerate(tables):
            p, q, rk = t.get("p"), t.get("q"), list(t["ranks"])
            if p is None or q is None:
                ps, qs = suggested_tt_shapes(t["num_embeddings"], t["embedding_dim"])
                p, q = (ps if p is None else p), (qs if q is None else q)
            p, q = list(p), list(q)
            cores = t.get("cores") or tt_init_cores(p, q, rk, weight_dist, sigma, generator, device)
            cs = [torch.nn.Parameter(c.to(device=device, dtype=torch.float32).contiguous().clone()) for c in cores]
            for k in range(3):
                self.register_parameter(f"t{i}_G{k + 1}", cs[k])
            params.append(cs)
            self.specs.append((int(t["num_embeddings"]), p, q, rk))
        self.embedding_dim = int(self.specs[0][2][0] * self.specs[0][2][1] * self.specs[0][2][2])
        self._cores = params
        self._h = tt_emb_batch_create([(E, p, q, r, params[i]) for i, (E, p, q, r) in enumerate(self.specs)])
        self._set_optimizer(sparse, optimizer, eps)

    def _core_list(self):
        return [c for cs in self._cores for c in cs]

    def full_weight(self, table: int, row0: int = 0, nrows: Optional[int] = None) -> torch.Tensor:
        """Rows of table `table` expanded from its cores (default: all rows)."""
        E = self.specs[table][0]
        n = E - row0 if nrows is None else int(nrows)
        out = torch.empty((n, self.embedding_dim), dtype=torch.float32, device=self._cores[table][0].device)
        tt_emb_full_weight(self._h, table, row0, n, out)
        return out

    def forward(self, input, offsets, per_sample_weights=None, mode: str = "sum", include_last_offset=True):
        return self._run(input, offsets, per_sample_weights, mode, include_last_offset)
