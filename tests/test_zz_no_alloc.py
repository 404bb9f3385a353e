"""The allocation-free forward entry point against the handle-based one.

tt_emb_forward_noalloc() serves callers that cannot allocate device memory
(a memory manager owns it all, or the call must not synchronize the device or
runs during stream capture); its scratch is a static device array.  Two calls
in a row must give the handle path's output within the parity tolerance:
the second call runs on the array as the first call left it.  This file is
collected last so that a failure here stops a -x run only after every other
test has run.
"""
import numpy as np
import pytest
import torch

import tensor_train_compressed_embeddingbag_gb300 as tt
from tt_inputs import config

from _gpu_harness import GpuRun, assert_rows_close, dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cid,batch", [(2, None), (3, 256)])
def test_noalloc_forward_matches_handle_forward(cid, batch):
    wl = config(cid, batch=batch)
    run = GpuRun(wl)
    ref = run.forward().cpu().numpy()
    assert run.error() == tt.TT_OK
    s = wl.tables[0]
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full((wl.num_bags, wl.embedding_dim), float("nan"), dtype=torch.float32, device="cuda")
        tt.tt_emb_forward_noalloc(s.num_embeddings, s.p, s.q, s.ranks, run.cores[0], run.idx, run.off, run.w,
                                  run.mode, out, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_rows_close(out.cpu().numpy(), ref.astype(np.float64), f"no-alloc forward, call {call}")
    run.close()
