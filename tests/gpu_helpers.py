"""Shared plumbing for the GPU parity tests: move synthetic inputs to the
device, run the C-ABI steps one by one and bring every result back."""
import numpy as np
import torch

import dynamic_sparse_prefill_crisp_gb300 as crisp

B = 128


def to_dev(a_u16):
    return torch.from_numpy(np.ascontiguousarray(a_u16).view(np.int16)).view(torch.bfloat16).cuda()


def bf16_to_u16(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def empty(shape, dtype):
    return torch.empty(shape, dtype=dtype, device="cuda")


def new_workspace(shape, layer=False):
    n = crisp.layer_workspace_size(shape) if layer else crisp.workspace_size(shape)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    crisp.workspace_init(ws)
    return ws


def assert_status_ok(ws):
    st = crisp.read_status(ws)
    assert st == 0, crisp.status_string(st)


def run_steps(q, k, v, params, q_dev=None, k_dev=None, v_dev=None, pbar_rows_pe_only=True, out_dev=None, scale=0.0):
    """Runs A1..A8 through the step entry points; returns numpy copies. Also
    runs the fused A1+A3 pass (vmass_fused, smass_fused), whose outputs start
    as all-ones words so that an entry it fails to write shows."""
    hq, n, _ = q.shape
    hkv = k.shape[0]
    nb = crisp.num_blocks(n)
    W = (nb + 31) // 32
    qd = to_dev(q) if q_dev is None else q_dev
    kd = to_dev(k) if k_dev is None else k_dev
    vd = to_dev(v) if v_dev is None else v_dev
    out = empty((hq, n, 128), torch.bfloat16) if out_dev is None else out_dev
    s = crisp.make_shape(hq, hkv, n, qd, kd, out, scale=scale)
    ws = new_workspace(s)
    pmap = torch.full((hq, B, crisp.map_ld(n)), float("nan"), dtype=torch.float32, device="cuda")
    vmass = empty((hq, nb), torch.int64)
    smass = empty((hq, nb), torch.int64)
    rmass = empty((hq,), torch.int64)
    cstruct = empty((hq,), torch.int64)
    total = empty((hq,), torch.int64)
    route = empty((hq,), torch.uint8)
    vbits = empty((hq, W), torch.int32)
    sbits = empty((hq, W), torch.int32)
    pbar = torch.zeros((hq, nb, nb), dtype=torch.float32, device="cuda")
    pebits = empty((hq, nb, W), torch.int32)
    rowbits = empty((hq, nb, W), torch.int32)
    counts = empty((hq, nb), torch.int32)
    order = empty((hq * nb,), torch.int32)
    vmass_f = torch.full((hq, nb), -1, dtype=torch.int64, device="cuda")
    smass_f = torch.full((hq, nb), -1, dtype=torch.int64, device="cuda")
    rmass_f = torch.full((hq,), -1, dtype=torch.int64, device="cuda")
    crisp.proxy_masses(s, qd, kd, vmass_f, smass_f, rmass_f, ws)
    crisp.proxy_map(s, qd, kd, pmap, ws)
    crisp.block_masses(s, pmap, vmass, smass, rmass, ws)
    # Both forms of A2 and A4: from the map (the survey's calls) and from the
    # block masses (what the layer runs); they must agree bit for bit.
    crisp.route_cstruct(s, params, pmap, cstruct, total, route, ws)
    cstruct_m, total_m, route_m = empty((hq,), torch.int64), empty((hq,), torch.int64), empty((hq,), torch.uint8)
    crisp.route_cstruct_masses(s, params, vmass, rmass, cstruct_m, total_m, route_m, ws)
    vmass_s = torch.full((hq, nb), -1, dtype=torch.int64, device="cuda")
    smass_s = torch.full((hq, nb), -1, dtype=torch.int64, device="cuda")
    crisp.select_vs(s, params, pmap, route, vmass_s, smass_s, vbits, sbits, ws)
    vbits_m, sbits_m = empty((hq, W), torch.int32), empty((hq, W), torch.int32)
    crisp.select_vs_masses(s, params, vmass, smass, route, vbits_m, sbits_m, ws)
    crisp.pe_pool(s, qd, kd, route, pbar, ws)
    crisp.select_pe(s, params, pbar, route, pebits, ws)
    crisp.build_mask(s, route, vbits, sbits, pebits, rowbits, counts, order, ws)
    crisp.sparse_prefill_mask(s, qd, kd, vd, rowbits, order, out, ws)
    # A8 from the index sets: the mask is built in the workspace
    out_sets = torch.empty_strided(tuple(out.shape), out.stride(), dtype=torch.bfloat16, device="cuda")
    crisp.sparse_prefill(s, qd, kd, vd, route, vbits, sbits, pebits, out_sets, ws)
    torch.cuda.synchronize()
    assert_status_ok(ws)
    assert torch.equal(cstruct, cstruct_m) and torch.equal(total, total_m) and torch.equal(route, route_m)
    assert torch.equal(vmass_s, vmass) and torch.equal(smass_s, smass)
    assert torch.equal(vbits, vbits_m) and torch.equal(sbits, sbits_m)
    assert torch.equal(out_sets, out), "A8 from the index sets differs from A8 over the built mask"
    u64 = lambda t: t.cpu().numpy().view(np.uint64)
    u32 = lambda t: t.cpu().numpy().view(np.uint32)
    pm = pmap.cpu().numpy()
    # columns n..ld-1 of the map are written as zeros; the oracle's map has n columns
    assert np.all(pm[:, :, n:] == 0.0)
    return dict(pmap=np.ascontiguousarray(pm[:, :, :n]), vmass=u64(vmass), smass=u64(smass), rmass=u64(rmass),
                vmass_fused=u64(vmass_f), smass_fused=u64(smass_f), rmass_fused=u64(rmass_f),
                cstruct=u64(cstruct), total=u64(total),
                route=route.cpu().numpy(), vbits=u32(vbits), sbits=u32(sbits), pbar=pbar.cpu().numpy(),
                pebits=u32(pebits), rowbits=u32(rowbits), counts=counts.cpu().numpy(), order=order.cpu().numpy(),
                group=hq // hkv, out=out)


def attn_error(out_dev_or_np, ref):
    o = out_dev_or_np.float().cpu().numpy() if hasattr(out_dev_or_np, "cpu") else out_dev_or_np
    d = np.abs(o.astype(np.float64) - ref)
    return float(d.max()), float(d.mean())
