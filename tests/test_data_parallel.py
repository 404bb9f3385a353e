"""The data-parallel step: bags split over ranks, one sum all-reduce of the core
gradients, the same update on every rank.

Bags are independent in the forward pass and each core gradient is a sum over
bags, so the ranks' summed gradients equal the whole batch's gradient and the
cores after the step equal one fused step over the whole batch.

* CPU (world size 2, gloo): the host sharding (table-major bags, contiguous
  ranges per table, rebased CSR offsets) with the float64 oracle standing in
  for each rank's device work; the all-reduced gradients and the updated cores
  equal the oracle's single whole-batch step.
* GPU (world size 2, both ranks on cuda:0, gloo all-reduce through host
  memory; the ranks' kernels never wait on one another): DataParallelStep
  through the C ABI against the oracle's whole-batch step, SGD and Adagrad.
"""
import os
import socket
import tempfile

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from tt_inputs import Workload, config


def _port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shard(wl, rank, world):
    import tensor_train_compressed_embeddingbag_gb300 as tt

    bags, look, off = tt.shard_bags(wl.offsets, wl.num_tables, rank, world)
    return Workload(**{**wl.__dict__, "indices": wl.indices[look], "offsets": off,
                       "weights": None if wl.weights is None else wl.weights[look],
                       "grad_out": wl.grad_out[bags], "batch": bags.shape[0] // wl.num_tables})


def _cpu_rank(rank, world, port, cid, batch, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = config(cid, batch=batch)
    sub = _shard(wl, rank, world)
    for t in range(wl.num_tables):
        for k in range(3):
            g = torch.from_numpy(oracle.workload_backward_core(sub, t, k))
            dist.all_reduce(g)
            new = oracle.sgd_update(wl.cores[t][k], g.numpy(), wl.lr)
            if rank == 0:
                np.save(os.path.join(outdir, f"g_{t}_{k}.npy"), g.numpy())
                np.save(os.path.join(outdir, f"c_{t}_{k}.npy"), new)
    dist.barrier()
    dist.destroy_process_group()


def test_shard_covers_every_bag_once():
    import tensor_train_compressed_embeddingbag_gb300 as tt

    wl = config(5, batch=37)
    seen = []
    for r in range(3):
        bags, look, off = tt.shard_bags(wl.offsets, wl.num_tables, r, 3)
        assert np.all(np.diff(off) == wl.offsets[bags + 1] - wl.offsets[bags])
        assert off[-1] == look.shape[0]
        # table-major: the same number of bags of every table, in table order
        t = bags // wl.batch
        assert np.all(np.diff(t) >= 0) and np.all(np.bincount(t, minlength=wl.num_tables) == bags.shape[0] // 26)
        seen.append(bags)
    allb = np.sort(np.concatenate(seen))
    np.testing.assert_array_equal(allb, np.arange(wl.num_bags))


@pytest.mark.parametrize("cid,batch", [(3, 48), (5, 12)])
def test_two_rank_gloo_step_equals_whole_batch_step(cid, batch):
    """World size 2 on CPU: the sharded gradients, all-reduced, equal the whole
    batch's gradient, and the updated cores equal the oracle's fused step
    (Zipf weighted mean: bag lengths stay whole under the split; 26 tables:
    table-major sharding)."""
    wl = config(cid, batch=batch)
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_cpu_rank, args=(2, _port(), cid, batch, d), nprocs=2, join=True)
        for t in range(wl.num_tables):
            for k in range(3):
                g = np.load(os.path.join(d, f"g_{t}_{k}.npy"))
                want = oracle.workload_backward_core(wl, t, k)
                np.testing.assert_allclose(g, want, rtol=1e-10, atol=1e-13 * max(np.abs(want).max(), 1e-300))
                c = np.load(os.path.join(d, f"c_{t}_{k}.npy"))
                np.testing.assert_allclose(c, oracle.workload_sgd_slices(wl, t, k), rtol=1e-12, atol=1e-15)


def _gpu_rank(rank, world, port, cid, batch, optim, outdir):
    import tensor_train_compressed_embeddingbag_gb300 as tt

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    wl = config(cid, batch=batch)
    sub = _shard(wl, rank, world)
    cores = [torch.from_numpy(c).cuda() for t in wl.cores for c in t]
    if wl.num_tables == 1:
        s = wl.tables[0]
        h = tt.tt_emb_create(s.num_embeddings, s.p, s.q, s.ranks, cores)
    else:
        h = tt.tt_emb_batch_create([(s.num_embeddings, s.p, s.q, s.ranks, cores[3 * t:3 * t + 3])
                                    for t, s in enumerate(wl.tables)])
    state = None
    if optim == tt.TT_OPT_ADAGRAD:
        rng = np.random.default_rng(21)
        state = [torch.from_numpy(rng.uniform(0.5, 1.5, size=c.shape).astype(np.float32)).cuda() for c in cores]
        if rank == 0:
            for i, st in enumerate(state):
                np.save(os.path.join(outdir, f"s0_{i}.npy"), st.cpu().numpy())
    step = tt.DataParallelStep(h, cores, optim=optim, eps=1e-10, state=state)
    out = torch.empty((sub.num_bags, wl.embedding_dim), dtype=torch.float32, device="cuda")
    mode = tt.TT_POOL_MEAN if wl.mode == "mean" else tt.TT_POOL_SUM
    step(torch.from_numpy(sub.indices).cuda(), torch.from_numpy(sub.offsets).cuda(),
         None if sub.weights is None else torch.from_numpy(sub.weights).cuda(), mode, out,
         torch.from_numpy(sub.grad_out).cuda(), wl.lr)
    torch.cuda.synchronize()
    assert tt.tt_emb_get_last_error(h) == tt.TT_OK
    if rank == 0:
        for i, c in enumerate(cores):
            np.save(os.path.join(outdir, f"c_{i}.npy"), c.cpu().numpy())
        if state is not None:
            for i, st in enumerate(state):
                np.save(os.path.join(outdir, f"s_{i}.npy"), st.cpu().numpy())
    tt.tt_emb_destroy(h)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.gpu
@pytest.mark.parametrize("cid,batch,optim", [(2, None, 0), (3, 512, 0), (5, 96, 1)])
def test_two_rank_step_on_one_gpu_matches_oracle(cid, batch, optim):
    """Two ranks on cuda:0 (gloo all-reduce): DataParallelStep's cores (and Adagrad
    accumulators) after one step against the oracle's whole-batch step, every slice;
    untouched slices keep their bits."""
    import tensor_train_compressed_embeddingbag_gb300 as tt
    from _gpu_harness import assert_rows_close, oracle_grad

    tt.build()
    wl = config(cid, batch=batch)
    with tempfile.TemporaryDirectory() as d:
        mp.spawn(_gpu_rank, args=(2, _port(), cid, batch, optim, d), nprocs=2, join=True)
        i = 0
        for t in range(wl.num_tables):
            for k in range(3):
                got = np.load(os.path.join(d, f"c_{i}.npy"))
                dG = oracle_grad(wl, t, k, np.arange(wl.tables[t].p[k]))
                touched = np.abs(dG).reshape(dG.shape[0], -1).max(axis=1) > 0
                np.testing.assert_array_equal(got[~touched], wl.cores[t][k][~touched])
                if optim == tt.TT_OPT_SGD:
                    want = oracle.sgd_update(wl.cores[t][k][touched], dG[touched], wl.lr)
                else:
                    s0 = np.load(os.path.join(d, f"s0_{i}.npy"))
                    want, want_s = oracle.adagrad_update(wl.cores[t][k][touched], s0[touched], dG[touched], wl.lr,
                                                         1e-10)
                    assert_rows_close(np.load(os.path.join(d, f"s_{i}.npy"))[touched], want_s, f"state t{t} G{k + 1}")
                assert_rows_close(got[touched], want, f"data-parallel step t{t} G{k + 1}")
                i += 1
