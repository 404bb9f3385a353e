"""TT-EmbeddingBag forward + backward (fused SGD) throughput on GB300.

Workload: the FBTT README sample configuration, p = [200, 220, 250]
(E = 11,000,000), q = [4, 4, 4] (D = 64), ranks [32, 32], 512 bags of exactly
20 uniform lookups (nnz = 10,240), sum pooling, SGD lr = 0.1; seeded synthetic
data resident in HBM.  One step = forward + backward with the in-place core
update, through the C ABI.

Default arm prints one JSON line with the device-timed throughput (value,
lookups/s), the end-to-end number through the C ABI with host buffers (e2e),
the roofline of the dominant kernel from live CUDA events, clocks sampled
during the timed region and the float64 oracle timed on the host cores
(cpu_baseline).  ``--impl reference`` times that oracle alone on bounded
samples of the same workload.

Launch: ``python bench.py --gpus 1 --steps K --warmup W``; for N > 1 under
``torch.distributed.run`` every rank takes its own share of a batch of N times
the workload's bags (weak scaling), runs forward and backward with the core
gradients written out, the gradients are summed over the ranks (one NCCL
all-reduce) and every rank applies the same SGD update; rank 0 prints.
``--dp`` runs that data-parallel step at N = 1 too.

``--config N`` times another of the seeded workloads instead (1 tiny, 3 Zipf
weighted-mean with its 110,000 hot rows, 4 40M x 128 rank-64, 5 26 tables);
``--cache coherent|trainable`` adds the hot-row cache (single-table workloads
with hot rows: config 3) in its exact-copy or trainable-row mode.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TT-EmbeddingBag fwd+bwd ns/nnz (lookups/s) and % of roofline, 1×GB300"
WORKLOAD = "TT-EmbeddingBag 11M x 64 rank-32 (p=[200,220,250], q=[4,4,4]), B=512 x 20 uniform lookups, sum, fused SGD"
FP32_LANES_PER_SM = 128
SM_MAX_MHZ = 2070.0
# nominal dense tensor rates of the part (PFLOP/s): TF32 1.1, BF16 2.25
TF32_PER_BF16 = 1.1 / 2.25
L2_FLUSH_BYTES = 256 << 20
# FBTT README sample output for this exact workload: 0.416 us per lookup, fwd + bwd (GPU not stated)
PAGES_NS_PER_NNZ = 416.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
CSRC = os.path.join(ROOT, "tensor_train_compressed_embeddingbag_gb300", "csrc")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": SM_MAX_MHZ}, "fallback"


def fp32_peak_tflops(sms, sm_mhz):
    """FFMA peak: 128 FP32 lanes x 2 FLOP per SM per clock, SM count read from the device."""
    return sms * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12


def tf32x3_peak_tflops(pk):
    """Useful rate of a 3xTF32 contraction: the measured dense bf16 burst x the nominal
    TF32:BF16 ratio, / 3 (three TF32 products per useful product)."""
    return pk["bf16_tflops"] * TF32_PER_BF16 / 3.0


def source_sha(files):
    import hashlib

    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu record, or None when the
    record is missing or the kernel's sources changed since it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f).get(kernel)
    except (OSError, ValueError):
        return None, "no ncu record"
    if not rec:
        return None, "no ncu record"
    if rec.get("source_sha") != source_sha(rec.get("sources", [])):
        return None, "kernel changed since the ncu record"
    return float(rec["bytes_per_launch"]), rec.get("note", "")


def flops_per_lookup(spec):
    q1, q2, q3 = spec.q
    r1, r2 = spec.ranks
    A = q1 * r1 * q2 * r2
    Bc = q1 * q2 * r2 * q3
    return A, Bc


def touched_pairs(wl):
    """Distinct (i1, i2) pairs of every table's lookups (i1 p2 + i2 = row div p3)."""
    out = []
    for t, spec in enumerate(wl.tables):
        lo, hi = int(wl.offsets[t * wl.batch]), int(wl.offsets[(t + 1) * wl.batch])
        rows = np.asarray(wl.indices[lo:hi], dtype=np.int64)
        out.append(np.unique(rows // int(spec.p[2])).shape[0] if rows.size else 0)
    return out


def dedup_step_flops(wl):
    """Step FLOPs with the contractions shared per touched (table, i1, i2) pair, as the
    kernels do them: 6 A per pair (T = G1 G2 forward; Q and dG2 backward) plus 6 Bc
    per lookup (T G3 forward; dT and the dG3 partial backward)."""
    total = 0
    for spec, pairs, t in zip(wl.tables, touched_pairs(wl), range(len(wl.tables))):
        n = int(wl.offsets[(t + 1) * wl.batch] - wl.offsets[t * wl.batch])
        A, Bc = flops_per_lookup(spec)
        total += 6 * A * pairs + 6 * Bc * n
    return total


def lookup_flops(wl):
    """(sum over lookups of A, sum over lookups of Bc): per-table figures times the table's lookups."""
    sa = sb = 0
    for t, spec in enumerate(wl.tables):
        n = int(wl.offsets[(t + 1) * wl.batch] - wl.offsets[t * wl.batch])
        A, Bc = flops_per_lookup(spec)
        sa += A * n
        sb += Bc * n
    return sa, sb


# Which pipe runs each kernel's contractions (the rank-16 / rank-32 classes with
# q = [4, 4, 4] take the tensor-core paths: T = G1 G2 in the forward; in the backward
# the pair contractions dG1 = dT G2^T and dG2 = G1^T dT when every table of the
# handle is of one such class).
def tc_class(spec):
    return list(spec.q) == [4, 4, 4] and spec.ranks[0] == spec.ranks[1] and spec.ranks[0] in (16, 32)


def kernel_parts(wl, pairs=None):
    """Per kernel: [(algorithmic FLOPs per launch, pipe)] with the per-lookup counts of
    the path (A = q1 r1 q2 r2, Bc = q1 q2 r2 q3 per lookup): T = G1 G2 2A; row = T G3
    2Bc; backward dT and the dG3 partial 4Bc, the dG1 partial and dG2 4A.  With `pairs`
    (touched (i1, i2) pairs per table) the A terms count once per pair, as done."""
    out = {"fwd_T": [], "pool": [], "tile_bwd": []}
    acc = {}
    classes = {(tuple(s.q), tuple(s.ranks)) for s in wl.tables}
    bwd_tc = len(classes) == 1 and tc_class(wl.tables[0]) and os.environ.get("TTEMB_BWD_FFMA") != "1"
    for t, spec in enumerate(wl.tables):
        n = int(wl.offsets[(t + 1) * wl.batch] - wl.offsets[t * wl.batch])
        A, Bc = flops_per_lookup(spec)
        if pairs is not None:
            A = A * pairs[t] / max(n, 1)  # A per lookup, averaged over the shared pairs
        tc = tc_class(spec)
        for k, f, pp in (("fwd_T", 2 * A * n, "tensor" if tc else "fp32"), ("pool", 2 * Bc * n, "fp32"),
                         ("tile_bwd", 4 * A * n, "tensor" if bwd_tc else "fp32"), ("tile_bwd", 4 * Bc * n, "fp32")):
            acc[(k, pp)] = acc.get((k, pp), 0) + f
    for (k, pp), f in acc.items():
        out[k].append((f, pp))
    return out


def peak_source(parts, pipe_peak, sms, sm_mhz, kind):
    txt = []
    for f, pp in parts:
        if pp == "fp32":
            txt.append(f"{f:.3g} FLOP on FP32 FFMA at {pipe_peak['fp32']:.1f} TFLOP/s ({sms} SMs x 128 x 2 x {sm_mhz:.0f} MHz)")
        else:
            txt.append(f"{f:.3g} FLOP on tensor cores (three products per useful product: 3xTF32, or bf16 pieces "
                       f"at twice the TF32 rate) at {pipe_peak['tensor']:.1f} TFLOP/s (bf16 burst of {kind} peaks "
                       f"x 1.1/2.25 / 3)")
    return "; ".join(txt) + "; peak = FLOPs / sum(FLOPs_pipe / peak_pipe)"


def max_over_ranks(values, device=None):
    """Element-wise max of a list of floats over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi samples of the SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.seek(0)
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.file:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            n += 1
            for name, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        self.file.close()
        return {
            "sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "reasons": sorted(reasons),
            "samples": n,
        }


# ---------------------------------------------------------------- reference arm (oracle)


def sub_workload(wl, nbags):
    """The first `nbags` bags of every table (bags are table-major), as a workload."""
    from tt_inputs import Workload

    nbags = min(nbags, wl.batch)
    idx, lens, go, w = [], [], [], []
    for t in range(wl.num_tables):
        b0 = t * wl.batch
        lo, hi = int(wl.offsets[b0]), int(wl.offsets[b0 + nbags])
        idx.append(wl.indices[lo:hi])
        lens.append(np.diff(wl.offsets[b0:b0 + nbags + 1]))
        go.append(wl.grad_out[b0:b0 + nbags])
        if wl.weights is not None:
            w.append(wl.weights[lo:hi])
    offsets = np.concatenate([[0], np.cumsum(np.concatenate(lens))]).astype(np.int64)
    return Workload(**{**wl.__dict__, "indices": np.concatenate(idx), "offsets": offsets,
                       "weights": None if wl.weights is None else np.concatenate(w),
                       "grad_out": np.concatenate(go), "batch": nbags})


def oracle_step(sub):
    """Forward, then the SGD step of every core slice the lookups touch (the others keep
    their values), all in the float64 oracle."""
    import oracle

    oracle.workload_forward(sub)
    i1, i2, i3, bag = oracle.decode(sub.tables, sub.indices, sub.offsets, sub.batch)
    table = bag // sub.batch
    for t in range(sub.num_tables):
        m = table == t
        for k, ik in enumerate((i1, i2, i3)):
            sl = np.unique(ik[m])
            if sl.size:
                oracle.workload_sgd_slices(sub, t, k, sl)


def cpu_baseline(wl, nbags=None, budget_s=10.0):
    """Oracle fwd + bwd + SGD steps on the first `nbags` bags (default: as many as fit
    about `budget_s` seconds, at most all), repeated while a pass takes less than the
    budget so that about `budget_s` seconds of host work are timed."""
    import oracle

    oracle.build()
    if nbags is None:  # bags per table
        probe = sub_workload(wl, min(8, wl.batch))
        t0 = time.perf_counter()
        oracle_step(probe)
        per_bag = (time.perf_counter() - t0) / probe.num_bags
        nbags = int(max(1, min(wl.batch, budget_s / max(per_bag * wl.num_tables, 1e-9))))
    sub = sub_workload(wl, nbags)
    t0 = time.perf_counter()
    oracle_step(sub)
    one = time.perf_counter() - t0
    reps = int(max(1, min(1000, budget_s / max(one, 1e-9))))
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle_step(sub)
    dt = time.perf_counter() - t0
    return {
        "value": sub.nnz * reps / dt,
        "unit": "lookups/s",
        "cores": oracle.num_threads(),
        "kind": "oracle",
        "sample": (f"{nbags} of {wl.batch} bags" + (f" of each of {wl.num_tables} tables" if wl.num_tables > 1 else "")
                   + f" ({sub.nnz} lookups), {reps} forward + backward + SGD steps from the same cores, "
                   f"float64, {dt:.2f} s"),
    }


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    import tt_inputs

    wl = tt_inputs.config(2)
    oracle.build()
    # size each step's sample so that warmup + steps finish in about two minutes
    budget = max(0.05, min(2.0, 120.0 / max(1, args.steps + args.warmup)))
    probe = sub_workload(wl, 8)
    t0 = time.perf_counter()
    oracle_step(probe)
    per_bag = (time.perf_counter() - t0) / 8
    nbags = int(max(1, min(wl.num_bags, budget / max(per_bag, 1e-9))))
    sub = sub_workload(wl, nbags)
    for _ in range(args.warmup):
        oracle_step(sub)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(sub)
    dt = time.perf_counter() - t0
    value = sub.nnz * args.steps / dt
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "lookups/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3,
        "ns_per_nnz": 1e9 * dt / (sub.nnz * args.steps),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample_bags": nbags, "sample_nnz": sub.nnz},
        "cpu_baseline": {
            "value": value, "unit": "lookups/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"first {nbags} of 512 bags ({sub.nnz} lookups) per step, forward + backward + SGD, float64",
        },
        "e2e": {"value": value, "unit": "lookups/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------- GPU arm


def workload_name(args):
    import tt_inputs

    name = WORKLOAD if args.config == 2 else "TT-EmbeddingBag " + tt_inputs.CONFIG_NAMES[args.config]
    opt = {"sgd": "fused SGD", "adagrad": "fused Adagrad", "grad": "sparse=False gradients"}[args.optimizer]
    name = name.replace("fused SGD", opt) if args.config == 2 else f"{name}, {opt}"
    if args.cache != "none":
        name += f", {args.cache} hot-row cache"
    elif args.config == 3:
        name = name.replace(", hot-row cache", ", no cache")
    return name


def run_gpu(args):
    import torch
    import torch.distributed as dist

    import tensor_train_compressed_embeddingbag_gb300 as tt
    import tt_inputs

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tt.build()
    tt.load_library()

    # data-parallel step (N > 1, or --dp): every rank takes its own share of a batch of
    # N times the workload's bags, the core gradients are summed over the ranks (NCCL)
    # and every rank applies the same update; N = 1 without --dp runs the fused step
    dp = ws > 1 or args.dp
    wl = tt_inputs.config(args.config)
    if dp:
        if args.optimizer == "grad" or args.cache != "none":
            raise SystemExit("the data-parallel step takes --optimizer sgd|adagrad and no cache")
        if ws > 1:
            full = tt_inputs.config(args.config, batch=wl.batch * ws)
            bags, look, off_r = tt.shard_bags(full.offsets, full.num_tables, rank, ws)
            wl = tt_inputs.Workload(**{**full.__dict__, "indices": full.indices[look], "offsets": off_r,
                                       "weights": None if full.weights is None else full.weights[look],
                                       "grad_out": full.grad_out[bags], "batch": bags.shape[0] // full.num_tables})
    spec = wl.tables[0]
    D, nnz, B = spec.embedding_dim, wl.nnz, wl.num_bags
    cores = [torch.from_numpy(c).to(dev) for t in wl.cores for c in t]
    if wl.num_tables == 1:
        h = tt.tt_emb_create(spec.num_embeddings, spec.p, spec.q, spec.ranks, cores)
    else:
        h = tt.tt_emb_batch_create([(s.num_embeddings, s.p, s.q, s.ranks, cores[3 * t:3 * t + 3])
                                    for t, s in enumerate(wl.tables)])
    aux = None
    dpstep = None
    if dp:
        aux = [torch.zeros_like(c) for c in cores] if args.optimizer == "adagrad" else None
        dpstep = tt.DataParallelStep(h, cores, optim=tt.TT_OPT_ADAGRAD if aux else tt.TT_OPT_SGD, eps=1.0e-10,
                                     state=aux)
    elif args.optimizer == "adagrad":  # fused element-wise Adagrad, accumulators starting at 0
        aux = [torch.zeros_like(c) for c in cores]
        tt.tt_emb_set_optimizer(h, tt.TT_OPT_ADAGRAD, 1.0e-10, aux)
    elif args.optimizer == "grad":  # sparse=False: the gradients are written out, the cores stay
        aux = [torch.zeros_like(c) for c in cores]
        tt.tt_emb_set_optimizer(h, tt.TT_OPT_GRAD, 0.0, aux)
    if args.cache != "none":
        if wl.num_tables != 1 or wl.cache_rows is None:
            raise SystemExit("--cache needs a single-table workload with hot rows (--config 3)")
        if args.cache == "trainable":
            tt.tt_emb_cache_set_trainable(h, True)
        tt.tt_emb_cache_populate(h, torch.from_numpy(wl.cache_rows).to(dev))
    tt.tt_emb_reserve(h, nnz, B)
    # indices and offsets share one int64 buffer, so the end-to-end step copies them up at once
    io = torch.from_numpy(np.concatenate([wl.indices, wl.offsets])).to(dev)
    idx, off = io[:nnz], io[nnz:]
    go = torch.from_numpy(wl.grad_out).to(dev)
    wts = None if wl.weights is None else torch.from_numpy(wl.weights).to(dev)
    mode = tt.TT_POOL_MEAN if wl.mode == "mean" else tt.TT_POOL_SUM
    out = torch.empty((B, D), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    lr = wl.lr

    def step():
        if dpstep is not None:
            dpstep(idx, off, wts, mode, out, go, lr, stream)
            return
        tt.tt_emb_forward(h, idx, off, wts, mode, out, stream)
        tt.tt_emb_backward(h, go, lr, stream)

    def barrier():
        torch.cuda.synchronize(dev)
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    def timed(fn, steps):
        """Sum of per-step device times (ms), L2 flushed before every step outside the events."""
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        barrier()
        for s, e in ev:
            flush.fill_(1.0)
            s.record(stream)
            fn()
            e.record(stream)
        barrier()
        return sum(s.elapsed_time(e) for s, e in ev)

    for _ in range(max(3, args.warmup)):
        step()
    err = tt.tt_emb_get_last_error(h)
    if err != tt.TT_OK:
        raise RuntimeError(f"device error during warm-up: {tt.tt_emb_status_string(err)}")
    launches_per_step = tt.tt_emb_last_launch_count(h, 0) + tt.tt_emb_last_launch_count(h, 1)

    # the step as a CUDA graph: forward + backward captured once, replayed per step
    def capture(timing):
        tt.tt_emb_set_stage_timing(h, timing)
        step()  # creates the stage events outside the capture
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            cs = torch.cuda.current_stream(dev)
            tt.tt_emb_forward(h, idx, off, wts, mode, out, cs)
            tt.tt_emb_backward(h, go, lr, cs)
        tt.tt_emb_set_stage_timing(h, False)
        return g

    graph = capture(False) if not (args.eager or dp) else None
    run_step = graph.replay if graph is not None else step
    for _ in range(max(3, args.warmup)):
        run_step()

    vis = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    sampler = ClockSampler(vis[local] if local < len(vis) else str(local))
    sampler.start()
    time.sleep(0.2)
    ms_total = timed(run_step, args.steps)
    clocks = sampler.stop()
    ms_total = max_over_ranks([ms_total], dev)[0]
    if tt.tt_emb_get_last_error(h) != tt.TT_OK:
        raise RuntimeError("device error in the timed region")

    # eager launches (no graph), and the host time to enqueue them
    ms_eager = timed(step, args.steps)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(200):
        step()
    host_us = (time.perf_counter() - t0) / 200 * 1e6
    torch.cuda.synchronize(dev)

    # forward alone
    ms_fwd = timed(lambda: tt.tt_emb_forward(h, idx, off, wts, mode, out, stream), args.steps)

    # per-kernel durations: a graph of the same step with an event after every kernel
    gstage = capture(True) if not dp else None
    kstats = {}
    nstage = min(args.steps, 400)
    barrier()
    if dp:
        tt.tt_emb_set_stage_timing(h, True)
    for _ in range(nstage):
        flush.fill_(1.0)
        if gstage is not None:
            gstage.replay()
        else:
            step()
        for which in (0, 1):
            for name, ms in tt.tt_emb_stage_times(h, which):
                kstats.setdefault(name, []).append(ms)
    tt.tt_emb_set_stage_timing(h, False)
    kavg = {k: sum(v) / len(v) for k, v in kstats.items()}
    del gstage, graph

    # end to end through the C ABI with host buffers: inputs copied in, result copied out, every step
    io_h = torch.from_numpy(np.concatenate([wl.indices, wl.offsets])).pin_memory()
    go_h = torch.from_numpy(wl.grad_out).pin_memory()
    w_h = None if wts is None else torch.from_numpy(wl.weights).pin_memory()
    out_h = torch.empty((B, D), dtype=torch.float32).pin_memory()
    h2d = io_h.numel() * 8 + go_h.numel() * 4 + (0 if w_h is None else w_h.numel() * 4)
    d2h = out_h.numel() * 4

    # copies that the step does not wait for run on a side stream: grad_out goes up while
    # the forward runs, the output comes down while the backward runs
    side = torch.cuda.Stream(dev)
    ev_fwd, ev_go, ev_bwd = (torch.cuda.Event() for _ in range(3))
    ev_bwd.record(stream)

    def e2e_step():
        io.copy_(io_h, non_blocking=True)
        if w_h is not None:
            wts.copy_(w_h, non_blocking=True)
        side.wait_event(ev_bwd)  # the previous backward has read go
        with torch.cuda.stream(side):
            go.copy_(go_h, non_blocking=True)
            ev_go.record(side)
        tt.tt_emb_forward(h, idx, off, wts, mode, out, stream)
        ev_fwd.record(stream)
        side.wait_event(ev_fwd)
        with torch.cuda.stream(side):
            out_h.copy_(out, non_blocking=True)
        stream.wait_event(ev_go)
        tt.tt_emb_backward(h, go, lr, stream)
        if dpstep is not None:  # the rest of the data-parallel step: all-reduce, update
            if ws > 1:
                dist.all_reduce(dpstep.flat)
            tt.tt_emb_apply_gradients(h, dpstep.optim, lr, dpstep.grads, dpstep.state, dpstep.eps, stream)
        ev_bwd.record(stream)
        stream.wait_stream(side)  # the step ends when its output is on the host

    ms_e2e = timed(e2e_step, args.steps)
    ms_e2e, ms_fwd = max_over_ranks([ms_e2e, ms_fwd], dev)

    result = None
    if rank == 0:
        pk, pk_kind = peaks()
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        sA, sB = lookup_flops(wl)
        total_lookups = nnz * args.steps * ws
        value = total_lookups / (ms_total / 1e3)
        sm_mhz = float(pk.get("sm_max_mhz", SM_MAX_MHZ))
        pipe_peak = {"fp32": fp32_peak_tflops(sms, sm_mhz), "tensor": tf32x3_peak_tflops(pk)}
        pairs = touched_pairs(wl)
        parts_ns = kernel_parts(wl)
        parts_dd = kernel_parts(wl, pairs)
        # the roofline's FLOP count: per lookup (the metric's count), unless the lookups share
        # their (i1, i2) pairs so much that it counts more than twice the work done; then per
        # touched pair, with the per-lookup figure beside it
        dedup_primary = sum(f for v in parts_dd.values() for f, _ in v) < 0.5 * sum(f for v in parts_ns.values() for f, _ in v)
        parts = parts_dd if dedup_primary else parts_ns
        step_ms = ms_total / args.steps
        # ideal time of every kernel: its algorithmic FLOPs at the peak of the pipe that runs them
        ideal_ms = {k: sum(f / (pipe_peak[pp] * 1e12) for f, pp in v) * 1e3 for k, v in parts.items()}
        kflops = {k: sum(f for f, _ in v) for k, v in parts.items()}
        dom = max(kavg, key=kavg.get)
        if dom in parts:
            ach = kflops[dom] / (kavg[dom] * 1e-3) / 1e12
            eff_peak = kflops[dom] / (ideal_ms[dom] * 1e-3) / 1e12
            pipes = sorted({pp for _, pp in parts[dom]})
            traffic, tnote = measured_traffic(dom)
            other = parts_ns if dedup_primary else parts_dd
            other_ideal = sum(f / (pipe_peak[pp] * 1e12) for f, pp in other[dom]) * 1e3
            roof = {"bound": "tensor" if pipes == ["tensor"] else "alu", "achieved": ach, "peak": eff_peak,
                    "unit": "TFLOP/s", "frac": ach / eff_peak, "traffic": traffic, "traffic_note": tnote,
                    "kernel": dom, "avg_ms": kavg[dom], "pipes": {pp: f for f, pp in parts[dom]},
                    "peak_source": peak_source(parts[dom], pipe_peak, sms, sm_mhz, pk_kind),
                    "flop_count": ("per touched (i1, i2) pair for the pair contractions (the lookups share pairs: "
                                   "the per-lookup count is more than twice the work done)" if dedup_primary else
                                   "per lookup: 4 (q1 r1 q2 r2 + q1 q2 r2 q3) in the backward"),
                    ("frac_per_lookup_count" if dedup_primary else "frac_per_pair_count"): other_ideal / kavg[dom]}
        else:
            roof = {"bound": "hbm", "achieved": None, "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": None,
                    "traffic": None, "kernel": dom, "avg_ms": kavg[dom]}
        step_flops = 6 * (sA + sB)
        dedup_flops = dedup_step_flops(wl)
        step_tf = step_flops / (step_ms * 1e-3) / 1e12
        fwd_ms = ms_fwd / args.steps
        fwd_ideal = ideal_ms.get("fwd_T", 0.0) + ideal_ms.get("pool", 0.0)
        result = {
            "metric": METRIC,
            "value": value,
            "unit": "lookups/s",
            "n_gpus": ws,
            "steps": args.steps,
            "warmup": max(3, args.warmup),
            "ms_per_step": ms_total / args.steps,
            "ns_per_nnz": 1e6 * ms_total / (nnz * args.steps),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": value / (1e9 / PAGES_NS_PER_NNZ) if args.config == 2 else None,
            "vs_baseline_note": ("value / (1e9 / 416 ns), the FBTT README sample line for this workload (GPU not stated)"
                                 if args.config == 2 else "the pages give no figure for this workload"),
            "dtype": "f32",
            "data": "synthetic",
            "config": {
                "workload": workload_name(args),
                "nnz": nnz,
                "bags": B,
                "p": spec.p, "q": spec.q, "ranks": spec.ranks,
                "l2": f"flushed before every timed step ({L2_FLUSH_BYTES >> 20} MiB write, outside the events)",
                "optimizer": {"sgd": "fused SGD", "adagrad": "fused element-wise Adagrad",
                              "grad": "sparse=False (gradients written out)"}[args.optimizer],
                "parallelism": (f"data parallel over {ws} GPUs: bags split, NCCL sum all-reduce of the core "
                                f"gradients, same update on every rank" if dp and ws > 1 else
                                "data-parallel step on one GPU (gradients out, update), no all-reduce" if dp else
                                "one GPU, fused update"),
                "global_bags": B * ws,
                "cache": {"none": "none", "coherent": "110,000 hot rows, exact copies",
                          "trainable": "110,000 hot rows, trainable"}[args.cache],
            },
            "timing": ("CUDA graph of forward + backward replayed per step" if not (args.eager or dp) else
                       "eager launches"),
            "eager": {"ms_per_step": ms_eager / args.steps, "host_enqueue_us_per_step": host_us},
            "forward": {"ns_per_nnz": 1e6 * ms_fwd / (nnz * args.steps),
                        "lookups_per_s": nnz * args.steps * ws / (ms_fwd / 1e3),
                        "achieved_tflops": 2 * (sA + sB) / (fwd_ms * 1e-3) / 1e12,
                        "frac": fwd_ideal / fwd_ms,
                        "flop_formula": "2 (q1 r1 q2 r2 + q1 q2 r2 q3) per lookup; frac = sum over the forward "
                                        "kernels of FLOPs / peak of the pipe that runs them, over the forward time"},
            "step_roofline": {"flops_per_step": step_flops, "achieved_tflops": step_tf,
                              "ideal_ms": sum(ideal_ms.values()), "frac": sum(ideal_ms.values()) / step_ms,
                              "frac_formula": "sum over kernels of (algorithmic FLOPs / peak of the pipe that runs "
                                              "them), divided by ms_per_step",
                              "per_kernel": {k: {"flops": kflops[k], "ideal_ms": ideal_ms[k],
                                                 "avg_ms": kavg.get(k), "pipes": {pp: f for f, pp in parts[k]}}
                                             for k in parts},
                              "fp32_frac_of_step": step_tf / pipe_peak["fp32"],
                              "flop_formula": "6 (q1 r1 q2 r2 + q1 q2 r2 q3) per lookup (flops_per_step); frac with "
                                              + ("6 q1 r1 q2 r2 per touched pair + 6 q1 q2 r2 q3 per lookup"
                                                 if dedup_primary else "the per-lookup count"),
                              "dedup_flops_per_step": dedup_flops,
                              "dedup_frac": sum(sum(f / (pipe_peak[pp] * 1e12) for f, pp in v) * 1e3
                                                for v in parts_dd.values()) / step_ms,
                              "primary_count": "per touched pair" if dedup_primary else "per lookup",
                              "dedup_formula": "6 q1 r1 q2 r2 per touched (i1, i2) pair + 6 q1 q2 r2 q3 per lookup"},
            "peaks": {"sms": sms, "sm_mhz": sm_mhz, "fp32_tflops": pipe_peak["fp32"],
                      "tf32x3_tflops": pipe_peak["tensor"], "source": pk_kind,
                      "fp32_formula": f"{sms} SMs (device) x 128 lanes x 2 FLOP x {sm_mhz:.0f} MHz",
                      "tf32x3_formula": f"measured bf16 burst {pk['bf16_tflops']} x 1.1/2.25 (nominal TF32:BF16) / 3"},
            "roofline": roof,
            "kernels_ms": kavg,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "peaks_source": pk_kind,
            "e2e": {"value": total_lookups / (ms_e2e / 1e3), "unit": "lookups/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "copies": "pinned host buffers; indices and offsets (one buffer) before the forward, grad_out during "
                              "the forward and the output during the backward (side stream)"},
        }
    tt.tt_emb_destroy(h)
    if rank == 0 and not args.no_cpu_baseline and wl.num_tables > 1:
        # every oracle call promotes all tables' cores to float64, which dominates any
        # bounded sample of a 26-table step: no meaningful host rate
        result["cpu_baseline"] = {"value": None, "unit": "lookups/s", "kind": "oracle",
                                  "sample": "not sampled for table-batched workloads"}
    elif rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(wl)
        if args.cache != "none":
            result["cpu_baseline"]["sample"] += " (the oracle without the cache)"
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing")
    ap.add_argument("--eager", action="store_true", help="time eager launches instead of a CUDA graph replay")
    ap.add_argument("--dp", action="store_true",
                    help="run the data-parallel step (gradients out, all-reduce, update) also at N = 1")
    ap.add_argument("--optimizer", choices=["sgd", "adagrad", "grad"], default="sgd",
                    help="what the backward does with the core gradients (default: fused SGD)")
    ap.add_argument("--config", type=int, choices=[1, 2, 3, 4, 5], default=2,
                    help="seeded workload (default 2: the FBTT README sample configuration)")
    ap.add_argument("--cache", choices=["none", "coherent", "trainable"], default="none",
                    help="hot-row cache mode (config 3's hot rows)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
