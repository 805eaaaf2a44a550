"""The allocation-free proxy map entry point against the regular one.

crisp_proxy_map_noalloc serves callers that cannot allocate device memory
when the step runs (an engine that gave all free memory to its own pool, or
code that must not trigger the device-wide synchronisation of cudaMalloc).
It keeps its scratch in the library's static device memory, so two calls in
a row also check that a call does not depend on what the previous one left
there. The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import dynamic_sparse_prefill_crisp_gb300 as crisp
import synth

pytestmark = pytest.mark.gpu

MAP_ATOL, MAP_RTOL = 1e-6, 1e-3  # the proxy-map tolerance of the parity tests


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()


def _regular_and_noalloc(hq, hkv, n, seed):
    w = synth.small("noalloc", hq, hkv, n, seed)
    q, k, _ = w.generate()
    qd, kd = _dev(q), _dev(k)
    s = crisp.make_shape(hq, hkv, n, qd, kd)
    ws = torch.empty(crisp.workspace_size(s), dtype=torch.uint8, device="cuda")
    crisp.workspace_init(ws)
    ld = crisp.map_ld(n)  # 128 * ceil(n / 128): whole tiles, columns past n written as 0
    ref = torch.empty((hq, 128, ld), dtype=torch.float32, device="cuda")
    crisp.proxy_map(s, qd, kd, ref, ws)
    got = torch.full((hq, 128, ld), float("nan"), dtype=torch.float32, device="cuda")
    rc = crisp.lib().crisp_proxy_map_noalloc(ctypes.byref(s), ctypes.c_void_p(qd.data_ptr()),
                                             ctypes.c_void_p(kd.data_ptr()), ctypes.c_void_p(got.data_ptr()),
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, crisp.status_string(rc)
    torch.cuda.synchronize()
    assert crisp.read_status(ws) == 0
    # the static scratch's own status word: no bounded wait ran out
    assert crisp.noalloc_read_status() == 0
    return ref.cpu().numpy(), got.cpu().numpy()


def test_noalloc_matches_regular_entry_point_twice_in_a_row():
    # Calls in a row with different shapes: each reuses the static scratch
    # the one before filled; the last has a short final block (2300 tokens,
    # 128 does not divide n), the ragged instantiation of the proxy kernels.
    for hq, hkv, n, seed in ((8, 2, 4096, 71), (4, 1, 2304, 72), (4, 1, 2300, 73)):
        ref, got = _regular_and_noalloc(hq, hkv, n, seed)
        assert np.all(np.isfinite(got))
        assert np.all(np.abs(got - ref) <= MAP_ATOL + MAP_RTOL * np.abs(ref))


def test_noalloc_rejects_shapes_beyond_the_static_scratch():
    # 1M tokens x 64 heads needs 256 + 1024*64*(2*512+1) bytes > 32 MiB.
    s = crisp.make_shape(64, 8, 1 << 20)
    vp = ctypes.c_void_p
    rc = crisp.lib().crisp_proxy_map_noalloc(ctypes.byref(s), vp(256), vp(256), vp(256), None)
    assert rc == 4  # CRISP_ERR_WORKSPACE, nothing launched
