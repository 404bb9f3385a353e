"""Write the oracle's expected values for the tiny seeded workload.

Calls only the float64 oracle (``oracle/``) and the seeded input generator;
no value here comes from the CUDA path.  Run from the repository root:

    python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from tt_inputs import config  # noqa: E402


def main():
    wl = config(1)
    out = oracle.workload_forward(wl)
    upd = [oracle.workload_sgd_slices(wl, 0, k) for k in range(3)]
    doc = {
        "source": "tiny TT-EmbeddingBag workload (p=[4,5,6], q=[2,2,2], r=[4,4], seed 0): "
                  "float64 oracle forward output and cores after one fused SGD step, lr=0.1",
        "indices": wl.indices.tolist(),
        "offsets": wl.offsets.tolist(),
        "out": out.tolist(),
        "updated_cores": [u.tolist() for u in upd],
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "config1_oracle.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")
    print("wrote", path)


if __name__ == "__main__":
    main()
