"""Host-side logic of bench.py on the CPU: the reference arm and the
max-over-ranks timing reduction with two gloo ranks."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank])
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res[0] == res[1] == [2.0, 10.0]


def test_max_over_ranks_without_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks([3.5, 1.0]) == [3.5, 1.0]


def run_bench(args, env_extra=None):
    env = dict(os.environ, **(env_extra or {}))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                       env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return r.stdout


def test_reference_arm_prints_one_json_line():
    out = run_bench(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    lines = [l for l in out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["unit"] == "lookups/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_stay_silent():
    out = run_bench(["--impl", "reference", "--steps", "1", "--warmup", "0"],
                    {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert out.strip() == ""


def test_flop_accounting_per_table():
    """The roofline's algorithmic FLOPs: per lookup A = q1 r1 q2 r2 and Bc = q1 q2 r2 q3 of
    its own table, summed over the lookups (checked by brute force over the bags)."""
    sys.path.insert(0, ROOT)
    import bench
    import tt_inputs

    wl = tt_inputs.config(5, batch=16)
    sa, sb = bench.lookup_flops(wl)
    want_a = want_b = 0
    for g in range(wl.num_bags):
        spec = wl.tables[g // wl.batch]
        n = int(wl.offsets[g + 1] - wl.offsets[g])
        q1, q2, q3 = spec.q
        r1, r2 = spec.ranks
        want_a += n * q1 * r1 * q2 * r2
        want_b += n * q1 * q2 * r2 * q3
    assert (sa, sb) == (want_a, want_b)
    spec = tt_inputs.config(2).tables[0]
    assert bench.flops_per_lookup(spec) == (16384, 2048)  # 11M x 64 rank-32: 4*32*4*32, 4*4*32*4


def test_workload_names():
    sys.path.insert(0, ROOT)
    import argparse

    import bench

    ns = argparse.Namespace
    assert bench.workload_name(ns(config=2, optimizer="sgd", cache="none")) == bench.WORKLOAD
    assert "fused Adagrad" in bench.workload_name(ns(config=2, optimizer="adagrad", cache="none"))
    assert bench.workload_name(ns(config=3, optimizer="sgd", cache="trainable")).endswith("trainable hot-row cache")
    assert "no cache" in bench.workload_name(ns(config=3, optimizer="sgd", cache="none"))


def test_dedup_flops_brute_force():
    """Pairs counted per table from the decoded (i1, i2) of every lookup."""
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    import tt_inputs

    wl = tt_inputs.config(5, batch=16)
    i1, i2, i3, bag = oracle.decode(wl.tables, wl.indices, wl.offsets, wl.batch)
    want = 0
    for t, spec in enumerate(wl.tables):
        m = (bag // wl.batch) == t
        pairs = len(set(zip(i1[m].tolist(), i2[m].tolist())))
        A, Bc = bench.flops_per_lookup(spec)
        want += 6 * A * pairs + 6 * Bc * int(m.sum())
    assert bench.dedup_step_flops(wl) == want


def test_kernel_parts_cover_the_step_flops():
    """The per-kernel split of the algorithmic FLOPs adds up to 6 (A + Bc) per lookup, and
    only the rank-16 / rank-32 q = [4, 4, 4] tables put T = G1 G2 on the tensor pipe."""
    sys.path.insert(0, ROOT)
    import bench
    from tt_inputs import config

    for cid, batch in ((2, None), (5, 64), (4, 64)):
        wl = config(cid, batch=batch)
        parts = bench.kernel_parts(wl)
        sa, sb = bench.lookup_flops(wl)
        assert sum(f for v in parts.values() for f, _ in v) == 6 * (sa + sb)
        tensor = sum(f for f, pp in parts["fwd_T"] if pp == "tensor")
        want = sum(2 * bench.flops_per_lookup(s)[0] * int(wl.offsets[(t + 1) * wl.batch] - wl.offsets[t * wl.batch])
                   for t, s in enumerate(wl.tables) if bench.tc_class(s))
        assert tensor == want


def test_traffic_record_voided_when_sources_change(tmp_path, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    rec = {"k_x": {"sources": ["tt_bwd.cu"], "source_sha": bench.source_sha(["tt_bwd.cu"]), "bytes_per_launch": 123.0}}
    f = tmp_path / "t.json"
    f.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.measured_traffic("k_x")[0] == 123.0
    rec["k_x"]["source_sha"] = "0" * 16
    f.write_text(json.dumps(rec))
    assert bench.measured_traffic("k_x")[0] is None
    assert bench.measured_traffic("k_missing")[0] is None


def test_pair_count_parts_match_dedup_flops():
    """With the touched pairs, the per-kernel split adds up to 6 A per pair + 6 Bc per
    lookup (the dedup count), and the pairs are counted from the decoded (i1, i2)."""
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from tt_inputs import config

    wl = config(4, batch=128)
    pairs = bench.touched_pairs(wl)
    i1, i2, i3, bag = oracle.decode(wl.tables, wl.indices, wl.offsets, wl.batch)
    assert pairs == [len(set(zip(i1.tolist(), i2.tolist())))]
    parts = bench.kernel_parts(wl, pairs)
    assert abs(sum(f for v in parts.values() for f, _ in v) - bench.dedup_step_flops(wl)) < 1e-6 * bench.dedup_step_flops(wl)
