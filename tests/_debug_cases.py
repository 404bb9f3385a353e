"""Run by test_debug_build_gpu.py in a fresh process with TTEMB_DEBUG=1: the
index-checking debug library takes small workloads and the edge cases through
the C ABI; every call must leave the error word clear (no index outside its
bound) and match the oracle."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import tensor_train_compressed_embeddingbag_gb300 as tt  # noqa: E402
from tt_inputs import config  # noqa: E402

from _gpu_harness import GpuRun, check_cores, check_decode, check_forward  # noqa: E402
from test_parity_gpu import synthetic  # noqa: E402


def run(wl):
    run = GpuRun(wl)
    out = run.forward().cpu().numpy()
    dec = check_decode(run, wl)
    run.backward()
    st = run.error()
    assert st == tt.TT_OK, tt.tt_emb_status_string(st)
    check_forward(out, wl)
    check_cores(run, wl, dec)
    run.close()


def main():
    assert tt.library_path().endswith("libttemb_debug.so"), tt.library_path()
    rng = np.random.default_rng(4)
    cases = [
        ("tiny", config(1)),
        ("11M x 64 rank 32, 64 bags", config(2, batch=64)),
        ("Zipf weighted mean, 96 bags", config(3, batch=96)),
        ("40M x 128 rank 64, 512 bags (large-path sort)", config(4, batch=512)),
        ("26 tables, 24 bags", config(5, batch=24)),
        ("empty and single bags", synthetic([4, 5, 6], [2, 2, 2], [4, 4], [0, 1, 0, 3, 1, 0, 0, 7, 1], weights=True,
                                            mode="mean")),
        ("groups over many tiles", synthetic([3, 2, 5], [2, 2, 2], [3, 5], rng.integers(0, 9, size=400), seed=1,
                                             weights=True)),
        ("repeated rows over tiles", synthetic([7, 3, 4], [2, 4, 1], [6, 2], rng.integers(1, 30, size=100), seed=2,
                                               dist="few")),
    ]
    for name, wl in cases:
        run(wl)
        print("ok", name, flush=True)


if __name__ == "__main__":
    main()
