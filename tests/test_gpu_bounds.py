"""The bounds-checking build (libcrisp_debug.so, -DCRISP_DEBUG) on valid inputs.

Every global index and TMA coordinate of every kernel is checked against its
buffer there; a failed check would record CRISP_ERR_BOUNDS in the status word
and skip the access (nothing traps). Here the small parity shapes -- ragged
lengths, two and three blocks, GQA 7:1 and 16:1, token-major strided
layouts -- run through every step entry point and the whole layer with both
libraries. Every output buffer and workspace sits between canary regions.
Required: status OK, canaries untouched, and outputs bit-identical to the
release build. No invalid input is planted on the GPU.
"""
import numpy as np
import pytest
import torch

import dynamic_sparse_prefill_crisp_gb300 as crisp
import synth
from dynamic_sparse_prefill_crisp_gb300 import build as crisp_build
from gpu_helpers import B, to_dev

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes of canary on each side (keeps the guarded buffer 256-byte aligned)
CANARY = 0xA5


class Guarded:
    """Allocates device buffers between canary regions and checks them."""

    def __init__(self):
        self.bufs = []

    def __call__(self, shape, dtype, fill=0):
        nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        raw = torch.full((nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        mid = raw[GUARD:GUARD + nbytes]
        mid.fill_(fill)
        self.bufs.append(raw)
        return mid.view(dtype).view(shape)

    def intact(self):
        return all(bool((r[:GUARD] == CANARY).all()) and bool((r[-GUARD:] == CANARY).all()) for r in self.bufs)


def run_all(lib, q, k, v, params, layout):
    """Every step entry point and the whole layer through `lib`; returns the
    outputs (host copies), the final status words and whether the canaries
    held."""
    saved = crisp._lib
    crisp._lib = lib
    try:
        hq, n, _ = q.shape
        hkv = k.shape[0]
        nb = crisp.num_blocks(n)
        W = (nb + 31) // 32
        g = Guarded()
        if layout == "token-major":
            def dev(a, heads):
                t = g((n, heads, 128), torch.bfloat16)
                t.copy_(to_dev(np.ascontiguousarray(a.transpose(1, 0, 2))))
                return t.permute(1, 0, 2)
            out = g((n, hq, 128), torch.bfloat16).permute(1, 0, 2)
            out2 = g((n, hq, 128), torch.bfloat16).permute(1, 0, 2)
            out3 = g((n, hq, 128), torch.bfloat16).permute(1, 0, 2)
            out4 = g((n, hq, 128), torch.bfloat16).permute(1, 0, 2)
        else:
            def dev(a, heads):
                t = g((heads, n, 128), torch.bfloat16)
                t.copy_(to_dev(a))
                return t
            out, out2, out3, out4 = (g((hq, n, 128), torch.bfloat16) for _ in range(4))
        qd, kd, vd = dev(q, hq), dev(k, hkv), dev(v, hkv)
        s = crisp.make_shape(hq, hkv, n, qd, kd, out)
        ws = g((crisp.workspace_size(s),), torch.uint8)
        lws = g((crisp.layer_workspace_size(s),), torch.uint8)
        crisp.workspace_init(ws)
        crisp.workspace_init(lws)
        I64, I32, U8, F32 = torch.int64, torch.int32, torch.uint8, torch.float32
        r = {}
        r["pmap"] = g((hq, B, crisp.map_ld(n)), F32)
        for name in ("vmass", "smass", "vmass_f", "smass_f", "vmass_m", "smass_m"):
            r[name] = g((hq, nb), I64)
        for name in ("rmass", "rmass_f", "cstruct", "total", "cstruct_m", "total_m"):
            r[name] = g((hq,), I64)
        r["route"], r["route_m"] = g((hq,), U8), g((hq,), U8)
        for name in ("vbits", "sbits", "vbits_m", "sbits_m"):
            r[name] = g((hq, W), I32)
        r["pbar"] = g((hq, nb, nb), F32)
        r["pebits"], r["rowbits"] = g((hq, nb, W), I32), g((hq, nb, W), I32)
        r["counts"], r["order"] = g((hq, nb), I32), g((hq * nb,), I32)
        r["jsd"] = g((hq,), torch.float64)
        r["route_jsd"] = g((hq,), U8)
        crisp.proxy_masses(s, qd, kd, r["vmass_f"], r["smass_f"], r["rmass_f"], ws)
        crisp.proxy_map(s, qd, kd, r["pmap"], ws)
        crisp.block_masses(s, r["pmap"], r["vmass"], r["smass"], r["rmass"], ws)
        crisp.route_cstruct(s, params, r["pmap"], r["cstruct"], r["total"], r["route"], ws)
        crisp.route_cstruct_masses(s, params, r["vmass"], r["rmass"], r["cstruct_m"], r["total_m"], r["route_m"], ws)
        crisp.select_vs(s, params, r["pmap"], r["route"], r["vmass_m"], r["smass_m"], r["vbits"], r["sbits"], ws)
        crisp.select_vs_masses(s, params, r["vmass"], r["smass"], r["route"], r["vbits_m"], r["sbits_m"], ws)
        crisp.pe_pool(s, qd, kd, r["route"], r["pbar"], ws)
        crisp.select_pe(s, params, r["pbar"], r["route"], r["pebits"], ws)
        crisp.build_mask(s, r["route"], r["vbits"], r["sbits"], r["pebits"], r["rowbits"], r["counts"], r["order"], ws)
        crisp.sparse_prefill_mask(s, qd, kd, vd, r["rowbits"], r["order"], out, ws)
        crisp.sparse_prefill(s, qd, kd, vd, r["route"], r["vbits"], r["sbits"], r["pebits"], out2, ws)
        crisp.dense_prefill(s, qd, kd, vd, out3, ws)
        crisp.prefill_layer(s, params, qd, kd, vd, out4, lws)
        crisp.route_jsd(s, params, r["vmass"], r["pbar"], r["jsd"], r["route_jsd"], ws)
        torch.cuda.synchronize()
        status = (crisp.read_status(ws), crisp.read_status(lws))
        res = {k_: t.cpu().numpy() for k_, t in r.items()}
        for name, t in (("out", out), ("out_sets", out2), ("dense", out3), ("layer", out4)):
            res[name] = t.float().cpu().numpy()
        return res, status, g.intact()
    finally:
        crisp._lib = saved


@pytest.fixture(scope="module")
def debug_lib():
    return crisp.load_library(crisp_build.build(debug=True))


CASES = [
    # name, hq, hkv, n, seed, layout
    ("ragged-300", 2, 1, 300, 31, "contiguous"),
    ("ragged-1000", 4, 2, 1000, 32, "contiguous"),
    ("nb2-256", 2, 1, 256, 3, "contiguous"),
    ("nb3-384", 2, 2, 384, 4, "contiguous"),
    ("gqa7-1152", 7, 1, 1152, 6, "contiguous"),
    ("gqa16-640", 16, 1, 640, 13, "contiguous"),
    ("strided-1024", 4, 2, 1024, 41, "token-major"),
    ("strided-ragged-2175", 4, 2, 2175, 34, "token-major"),
]


@pytest.mark.parametrize("name,hq,hkv,n,seed,layout", CASES, ids=[c[0] for c in CASES])
def test_checking_build_matches_release_within_bounds(debug_lib, name, hq, hkv, n, seed, layout):
    w = synth.small(name, hq, hkv, n, seed)
    q, k, v = w.generate()
    params = crisp.params_default()
    rel, rel_status, rel_intact = run_all(crisp.lib(), q, k, v, params, layout)
    dbg, dbg_status, dbg_intact = run_all(debug_lib, q, k, v, params, layout)
    assert rel_status == (0, 0), [crisp.status_string(x) for x in rel_status]
    assert dbg_status == (0, 0), [crisp.status_string(x) for x in dbg_status]  # no CRISP_ERR_BOUNDS
    assert rel_intact and dbg_intact, "a canary word changed"
    for key in rel:
        assert np.array_equal(rel[key], dbg[key], equal_nan=True), key
    # the map, sets and layer forms agree with each other as in the release tests
    assert np.array_equal(dbg["out"], dbg["out_sets"]) and np.array_equal(dbg["out"], dbg["layer"])
    assert np.array_equal(dbg["route"], dbg["route_m"]) and np.array_equal(dbg["vbits"], dbg["vbits_m"])
