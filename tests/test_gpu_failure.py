"""Failure detection on the GPU without a fault: a kernel waits, through the
pipeline's bounded mbarrier wait, on a barrier that nothing arrives at. The
wait must give up, the status word must say CRISP_ERR_TIMEOUT, and the
context must stay usable for the next layer."""
import time

import numpy as np
import pytest
import torch

import dynamic_sparse_prefill_crisp_gb300 as crisp
import synth
from gpu_helpers import empty, new_workspace, to_dev

pytestmark = pytest.mark.gpu

CRISP_ERR_TIMEOUT = 6


def test_bounded_wait_times_out_and_context_survives():
    w = synth.small("selftest", 4, 1, 1024, 101)
    q, k, v = w.generate()
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    out = empty((4, 1024, 128), torch.bfloat16)
    s = crisp.make_shape(4, 1, 1024, qd, kd, out)
    ws = new_workspace(s, layer=True)
    t0 = time.perf_counter()
    crisp.wait_selftest(ws, 200_000_000)  # 0.2 s
    assert crisp.read_status(ws) == CRISP_ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert 0.15 < elapsed < 5.0, elapsed
    # the context is usable: clear the status and run a layer
    crisp.workspace_init(ws)
    crisp.prefill_layer(s, crisp.params_default(), qd, kd, vd, out, ws)
    torch.cuda.synchronize()
    assert crisp.read_status(ws) == 0
    assert torch.isfinite(out.float()).all()
