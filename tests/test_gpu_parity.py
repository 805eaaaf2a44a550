"""CUDA path vs the CPU oracle, step by step, through the C ABI.

Acceptance (stated once, used throughout):
  * index sets, masses, C_struct, routes, bitsets, counts: bit-exact, with the
    oracle run on the GPU's own fp32 proxy / pooled maps;
  * proxy and pooled maps: |gpu - oracle| <= 1e-6 + 1e-3 * oracle element-wise
    (fp32 accumulate and base-2 exponent vs fp64);
  * attention output (bf16): max |err| <= 2e-2 and mean |err| <= 2e-3 against
    fp64 attention over the same blocks.
"""
import numpy as np
import pytest
import torch

import dynamic_sparse_prefill_crisp_gb300 as crisp
import oracle
import synth
from gpu_helpers import (B, assert_status_ok, attn_error, bf16_to_u16, empty, new_workspace, run_steps, to_dev)

pytestmark = pytest.mark.gpu

MAP_ATOL, MAP_RTOL = 1e-6, 1e-3
ATT_MAX, ATT_MEAN = 2e-2, 2e-3


def check_map(gpu, ref):
    bad = np.abs(gpu.astype(np.float64) - ref) > MAP_ATOL + MAP_RTOL * np.abs(ref)
    assert not bad.any(), f"{bad.sum()} entries out of tolerance, max err {np.abs(gpu - ref).max()}"


def check_index_sets(r, params):
    """Oracle A2..A7 from the GPU's own fp32 maps; every integer result equal."""
    vm, sm = oracle.vs_masses(r["pmap"])
    assert np.array_equal(vm, r["vmass"])
    assert np.array_equal(sm, r["smass"])
    # the fused pass that never stores the map gives the same integers
    assert np.array_equal(vm, r["vmass_fused"])
    assert np.array_equal(sm, r["smass_fused"])
    assert np.array_equal(r["rmass"], r["rmass_fused"])
    S, T, route = oracle.route(r["pmap"], tau=(params.tau_num, params.tau_den))
    assert np.array_equal(S, r["cstruct"]) and np.array_equal(T, r["total"])
    # recency mass: the columns [n-128, n) (C_struct less the sink block)
    assert np.array_equal(r["rmass"], S - vm[:, 0])
    assert np.array_equal(route, r["route"])
    vb, sb = oracle.select_vs(vm, sm, route, alpha=(params.alpha_num, params.alpha_den), kmin=params.kmin_blocks)
    assert np.array_equal(vb, r["vbits"])
    assert np.array_equal(sb, r["sbits"])
    pbar = r["pbar"].copy()
    pbar[route == 1] = 0.0  # VS heads' pooled rows are not written
    pe = oracle.select_pe(pbar, route, pe_mode=params.pe_mode, gamma=(params.gamma_num, params.gamma_den),
                          alpha=(params.alpha_num, params.alpha_den), kmin=params.kmin_blocks)
    assert np.array_equal(pe, r["pebits"])
    rb = oracle.build_mask(route, vb, sb, pe)
    assert np.array_equal(rb, r["rowbits"])
    pop = np.unpackbits(rb.view(np.uint8), axis=-1).sum(-1).astype(np.int64)
    assert np.array_equal(pop, r["counts"])
    # schedule: kv group by kv group; within a group query blocks descending,
    # the group's heads ascending
    hq, nb = pop.shape
    G = r["group"]
    want = np.empty(hq * nb, np.int64)
    for h in range(hq):
        for qb in range(nb):
            want[((h // G) * nb + nb - 1 - qb) * G + h % G] = h * nb + qb
    assert np.array_equal(r["order"], want)
    return rb, route


def sample_rows(hq, n, count, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 127, 128, n - 129, n - 128, n - 1]
    heads, toks = [], []
    for h in range(hq):
        ts = sorted(set(fixed + rng.integers(0, n, count).tolist()))
        heads += [h] * len(ts)
        toks += ts
    return np.array(heads, np.int32), np.array(toks, np.int32)


def check_attention(q, k, v, out, rowbits, rows=None, scale=None):
    hq, n, _ = q.shape
    if rows is None:
        h, t = np.meshgrid(np.arange(hq), np.arange(n), indexing="ij")
        h, t = h.ravel().astype(np.int32), t.ravel().astype(np.int32)
    else:
        h, t = rows
    ref = oracle.attention_rows(q, k, v, h, t, rowbits=rowbits, scale=scale)
    got = out.float().cpu().numpy()[h, t]
    mx, mean = attn_error(got, ref)
    assert mx <= ATT_MAX and mean <= ATT_MEAN, (mx, mean)


CASES = [
    # name, hq, hkv, n, seed, vs_heads
    ("gqa4-1k", 4, 1, 1024, 1, None),
    ("mixed-2k", 8, 2, 2048, 2, None),
    ("nb2-256", 2, 1, 256, 3, None),
    ("nb3-384", 2, 2, 384, 4, None),
    ("nb5-640", 4, 2, 640, 5, [0]),
    ("gqa7-1152", 7, 1, 1152, 6, [0, 3, 6]),
    ("nb33-4224", 4, 2, 4224, 7, None),
    ("all-pe-2k", 4, 2, 2048, 8, []),
    ("single-head-512", 1, 1, 512, 12, None),
    ("gqa16-640", 16, 1, 640, 13, None),
    # 128 does not divide n: a short last block of t tokens (t = 44, 104, 1,
    # 127, 4); at 2049 the recency columns straddle two proxy CTAs
    ("ragged-300", 2, 1, 300, 31, None),
    ("ragged-1000", 4, 2, 1000, 32, None),
    ("ragged-2049", 4, 1, 2049, 33, [0]),
    ("ragged-2175", 4, 2, 2175, 34, None),
    ("ragged-4100", 8, 2, 4100, 35, None),
]


@pytest.mark.parametrize("name,hq,hkv,n,seed,vs", CASES, ids=[c[0] for c in CASES])
def test_pipeline_steps_match_oracle(name, hq, hkv, n, seed, vs):
    w = synth.small(name, hq, hkv, n, seed, vs_heads=vs)
    q, k, v = w.generate()
    params = crisp.params_default()
    r = run_steps(q, k, v, params)
    check_map(r["pmap"], oracle.proxy_map(q, k))
    rb, route = check_index_sets(r, params)
    if (route == 0).any():
        ref = oracle.pe_map(q, k)
        check_map(r["pbar"][route == 0], ref[route == 0])
    check_attention(q, k, v, r["out"], rb, rows=None if n <= 2048 else sample_rows(hq, n, 48, seed))


@pytest.mark.parametrize("overrides", [dict(alpha=(5, 4)), dict(alpha=(0, 1)), dict(alpha=(3, 1), kmin_blocks=0),
                                       dict(kmin_blocks=64), dict(pe_mode=crisp.PE_NOISE),
                                       dict(pe_mode=crisp.PE_NOISE, alpha=(5, 4), kmin_blocks=2),
                                       dict(gamma=(1, 1)), dict(gamma=(1, 2)), dict(tau=(1, 1)), dict(tau=(0, 1))],
                         ids=lambda d: "-".join(f"{k}{v}" for k, v in d.items()))
def test_parameter_variants(overrides):
    w = synth.small("params", 8, 2, 4096, 11)
    q, k, v = w.generate()
    params = crisp.params_default(**overrides)
    r = run_steps(q, k, v, params)
    rb, _ = check_index_sets(r, params)
    check_attention(q, k, v, r["out"], rb, rows=sample_rows(8, 4096, 24, 11))


def test_dense_prefill_matches_oracle():
    for hq, hkv, n, seed in ((4, 1, 1024, 21), (6, 2, 640, 22), (2, 2, 256, 23), (2, 1, 1, 24), (4, 2, 100, 25),
                             (2, 1, 129, 26), (4, 2, 777, 27)):
        w = synth.small("dense", hq, hkv, n, seed)
        q, k, v = w.generate()
        qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
        out = empty((hq, n, 128), torch.bfloat16)
        s = crisp.make_shape(hq, hkv, n, qd, kd, out)
        ws = new_workspace(s)
        crisp.dense_prefill(s, qd, kd, vd, out, ws)
        torch.cuda.synchronize()
        assert_status_ok(ws)
        check_attention(q, k, v, out, None)


def test_sparse_prefill_arbitrary_masks():
    # Masks not produced by the selection: rows without their diagonal block,
    # empty rows (zeros out), single far blocks, full rows.
    hq, hkv, n = 3, 1, 1536
    nb = n // B
    rng = np.random.default_rng(31)
    w = synth.small("masks", hq, hkv, n, 31)
    q, k, v = w.generate()
    rb = np.zeros((hq, nb, 1), np.uint32)
    for h in range(hq):
        for qb in range(nb):
            kind = rng.integers(0, 4)
            if kind == 0:
                bits = 0
            elif kind == 1:
                bits = (1 << (qb + 1)) - 1
            elif kind == 2:
                bits = 1 << int(rng.integers(0, qb + 1))
            else:
                bits = int(rng.integers(0, 1 << (qb + 1))) & ~(1 << qb)
            rb[h, qb, 0] = bits
    # stray bits above the diagonal must be ignored
    rb[0, 2, 0] |= np.uint32(1 << 9)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    out = empty((hq, n, 128), torch.bfloat16)
    s = crisp.make_shape(hq, hkv, n, qd, kd, out)
    ws = new_workspace(s)
    rbd = torch.from_numpy(rb.view(np.int32)).cuda()
    crisp.sparse_prefill_mask(s, qd, kd, vd, rbd, None, out, ws)  # default order: kv-group-major
    torch.cuda.synchronize()
    assert_status_ok(ws)
    rb_causal = rb.copy()
    for qb in range(nb):
        rb_causal[:, qb, 0] &= np.uint32((1 << (qb + 1)) - 1)
    check_attention(q, k, v, out, rb_causal)
    # empty rows are exactly zero
    o = out.float().cpu().numpy()
    for h in range(hq):
        for qb in range(nb):
            if rb_causal[h, qb, 0] == 0:
                assert np.all(o[h, qb * B:(qb + 1) * B] == 0.0)


def test_strided_token_major_layout():
    # [n][heads][128] storage (token-major), viewed as [heads][n][128]: head
    # stride 128, token stride heads*128. Results must equal the contiguous run.
    hq, hkv, n = 4, 2, 1024
    w = synth.small("strided", hq, hkv, n, 41)
    q, k, v = w.generate()
    params = crisp.params_default()
    ref = run_steps(q, k, v, params)
    qt = to_dev(np.ascontiguousarray(q.transpose(1, 0, 2))).permute(1, 0, 2)
    kt = to_dev(np.ascontiguousarray(k.transpose(1, 0, 2))).permute(1, 0, 2)
    vt = to_dev(np.ascontiguousarray(v.transpose(1, 0, 2))).permute(1, 0, 2)
    got = run_steps(q, k, v, params, q_dev=qt, k_dev=kt, v_dev=vt)
    assert np.array_equal(got["pmap"], ref["pmap"])
    assert np.array_equal(got["rowbits"], ref["rowbits"])
    assert torch.equal(got["out"], ref["out"])


def test_custom_scale_and_mixed_layouts():
    # A softmax scale other than 1/sqrt(128); q contiguous, k and v
    # token-major ([n][heads][128] storage) and the output token-major too.
    hq, hkv, n, scale = 4, 2, 1536, 0.05
    w = synth.small("scale", hq, hkv, n, 81)
    q, k, v = w.generate()
    params = crisp.params_default()
    kt = to_dev(np.ascontiguousarray(k.transpose(1, 0, 2))).permute(1, 0, 2)
    vt = to_dev(np.ascontiguousarray(v.transpose(1, 0, 2))).permute(1, 0, 2)
    ot = torch.empty((n, hq, 128), dtype=torch.bfloat16, device="cuda").permute(1, 0, 2)
    r = run_steps(q, k, v, params, k_dev=kt, v_dev=vt, out_dev=ot, scale=scale)
    check_map(r["pmap"], oracle.proxy_map(q, k, scale=scale))
    rb, route = check_index_sets(r, params)
    if (route == 0).any():
        check_map(r["pbar"][route == 0], oracle.pe_map(q, k, scale=scale)[route == 0])
    check_attention(q, k, v, r["out"], rb, scale=scale)


POOLED_CASES = [
    # hq, hkv, n, seed, scale (0: 1/sqrt(128))
    (4, 1, 256, 91, 0.0),      # the shortest layer the steps take: two blocks, one row tile
    (4, 2, 257, 92, 0.0),      # a one-token last block
    (8, 2, 131201, 93, 0.0),   # nb = 1026: nine row tiles, rows longer than the 1,024 kept in shared memory
    (4, 1, 4096, 94, 1.0),     # wide pooled logits
]


@pytest.mark.parametrize("hq,hkv,n,seed,scale", POOLED_CASES, ids=["n256", "n257", "nb1026", "scale1"])
def test_pooled_map_and_pe_selection_every_head(hq, hkv, n, seed, scale):
    # Every head routed to PE: the tensor-core pooled map against the fp64
    # estimate at the map tolerance (zeros above the diagonal exactly), and
    # both PE selection modes bit-exact against the oracle on the GPU's map.
    w = synth.small("pooled", hq, hkv, n, seed)
    q, k, _ = w.generate()
    nb = crisp.num_blocks(n)
    W = (nb + 31) // 32
    qd, kd = to_dev(q), to_dev(k)
    s = crisp.make_shape(hq, hkv, n, qd, kd, None, scale=scale)
    ws = new_workspace(s)
    route = torch.zeros((hq,), dtype=torch.uint8, device="cuda")
    pbar = torch.full((hq, nb, nb), float("nan"), dtype=torch.float32, device="cuda")
    crisp.pe_pool(s, qd, kd, route, pbar, ws)
    torch.cuda.synchronize()
    assert_status_ok(ws)
    got = pbar.cpu().numpy()
    assert np.isfinite(got).all()
    upper = np.triu(np.ones((nb, nb), dtype=bool), 1)
    assert (got[:, upper] == 0.0).all()
    check_map(got, oracle.pe_map(q, k, scale=scale if scale > 0 else None))
    route_h = route.cpu().numpy()
    for mode in (crisp.PE_GAMMA, crisp.PE_NOISE):
        params = crisp.params_default()
        params.pe_mode = mode
        pebits = empty((hq, nb, W), torch.int32)
        crisp.select_pe(s, params, pbar, route, pebits, ws)
        torch.cuda.synchronize()
        assert_status_ok(ws)
        ref = oracle.select_pe(got, route_h, pe_mode=mode, gamma=(params.gamma_num, params.gamma_den),
                               alpha=(params.alpha_num, params.alpha_den), kmin=params.kmin_blocks)
        assert np.array_equal(ref, pebits.cpu().numpy().view(np.uint32))


def test_attention_convenience_call_matches_the_layer():
    # crisp.attention allocates the output and workspace with torch and runs
    # the same layer call: identical bits, ragged length included.
    for hq, hkv, n, seed in ((8, 2, 2048, 54), (4, 1, 1000, 55)):
        w = synth.small("conv", hq, hkv, n, seed)
        q, k, v = w.generate()
        qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
        got = crisp.attention(qd, kd, vd)
        ref = empty((hq, n, 128), torch.bfloat16)
        s = crisp.make_shape(hq, hkv, n, qd, kd, ref)
        ws = new_workspace(s, layer=True)
        crisp.prefill_layer(s, crisp.params_default(), qd, kd, vd, ref, ws)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)


@pytest.mark.parametrize("scale", [1.0, 1e-3])
def test_extreme_softmax_scales(scale):
    # scale 1: logits with a spread of ~11 (rows ruled by single keys, whose
    # later blocks sit well above the first sub-block's max); scale 1e-3:
    # nearly uniform rows.
    hq, hkv, n = 4, 2, 1280
    w = synth.small("scales", hq, hkv, n, 82)
    q, k, v = w.generate()
    params = crisp.params_default()
    r = run_steps(q, k, v, params, scale=scale)
    check_map(r["pmap"], oracle.proxy_map(q, k, scale=scale))
    rb, route = check_index_sets(r, params)
    if (route == 0).any():
        check_map(r["pbar"][route == 0], oracle.pe_map(q, k, scale=scale)[route == 0])
    check_attention(q, k, v, r["out"], rb, scale=scale)


@pytest.mark.parametrize("window,n", [((100, 110), 2048), ((5, 15), 2048), ((60, 70), 2048), ((100, 110), 1999)],
                         ids=["second-sub-block", "first-sub-block", "both-sub-blocks", "ragged-1999"])
def test_attention_reference_rises_block_after_block(window, n):
    # The largest scores of each key block grow with the block and sit in one
    # window of columns, so a row's first sub-block sets a reference that
    # later blocks exceed by far more than 2^64 (the redo path: the row is run
    # again at its exact max) and, without it, by more than bf16 and fp32
    # can hold (p = 2^140 in the last block). Dense and full-mask sparse
    # launches against fp64 attention; n = 1999 ends in a short block of 79
    # tokens (zero-filled K/V rows in every pass of the redo).
    hq, hkv = 2, 1
    rng = np.random.default_rng(7)
    u = np.zeros(128)
    u[0] = 1.0
    q = 8.0 * u + 0.05 * rng.standard_normal((hq, n, 128))
    t = np.arange(n) % B
    kb = np.arange(n) // B
    # log2 units per raw unit here: 8 * 0.0884 * 1.4427 = 1.02, so each block's
    # window sits 9.2 above the last one's: 64 above the first block's from
    # block 7 on, 127 above from block 14 on
    amp = 9.0 * kb + np.where((t >= window[0]) & (t < window[1]), 6.0, 0.0)
    k = amp[None, :, None] * u + 0.05 * rng.standard_normal((hkv, n, 128))
    v = rng.standard_normal((hkv, n, 128))
    to_bits = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(torch.bfloat16).view(torch.int16) \
        .numpy().view(np.uint16)
    q, k, v = to_bits(q), to_bits(k), to_bits(v)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    nb = (n + B - 1) // B
    full = np.zeros((hq, nb, 1), np.uint32)
    for qb in range(nb):
        full[:, qb, 0] = (1 << (qb + 1)) - 1
    for dense in (True, False):
        out = empty((hq, n, 128), torch.bfloat16)
        s = crisp.make_shape(hq, hkv, n, qd, kd, out)
        ws = new_workspace(s)
        if dense:
            crisp.dense_prefill(s, qd, kd, vd, out, ws)
        else:
            crisp.sparse_prefill_mask(s, qd, kd, vd, torch.from_numpy(full.view(np.int32)).cuda(), None, out, ws)
        torch.cuda.synchronize()
        assert_status_ok(ws)
        check_attention(q, k, v, out, full)


def test_prefill_layer_matches_steps():
    for hq, hkv, n, seed in ((8, 2, 2048, 51), (4, 1, 640, 52), (4, 2, 1337, 53)):
        w = synth.small("layer", hq, hkv, n, seed)
        q, k, v = w.generate()
        params = crisp.params_default()
        steps = run_steps(q, k, v, params)
        qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
        out = empty((hq, n, 128), torch.bfloat16)
        s = crisp.make_shape(hq, hkv, n, qd, kd, out)
        ws = new_workspace(s, layer=True)
        crisp.prefill_layer(s, params, qd, kd, vd, out, ws)
        torch.cuda.synchronize()
        assert_status_ok(ws)
        views = crisp.layer_views(s, ws)
        nb = crisp.num_blocks(n)
        W = (nb + 31) // 32

        def grab(name, shape, dtype):
            t = torch.empty(shape, dtype=dtype, device="cuda")
            base = ws.data_ptr()
            off = views[name] - base
            nbytes = t.numel() * t.element_size()
            t.view(torch.uint8).view(-1).copy_(ws[off:off + nbytes])
            return t.cpu().numpy()

        assert np.array_equal(grab("vmass", (hq, nb), torch.int64).view(np.uint64), steps["vmass"])
        assert np.array_equal(grab("smass", (hq, nb), torch.int64).view(np.uint64), steps["smass"])
        assert np.array_equal(grab("rmass", (hq,), torch.int64).view(np.uint64), steps["rmass"])
        assert np.array_equal(grab("route", (hq,), torch.uint8), steps["route"])
        assert np.array_equal(grab("rowbits", (hq, nb, W), torch.int32).view(np.uint32), steps["rowbits"])
        assert torch.equal(out, steps["out"])


def test_prefill_layer_host_matches_device_layer():
    # Host buffers in, host buffer out, one kv group at a time with the copies
    # overlapped: bit-identical to the device-resident layer.
    pipe = crisp.HostPipeline()
    # 128k tokens: group size 4 (half-group chunks, the first and last groups
    # ramped 1, 2, 1) and group size 7 (whole groups, ramped 1, 2, 4 and
    # mirrored 4, 2, 1 in the last group)
    for hq, hkv, n, seed in ((8, 2, 2048, 71), (7, 1, 1152, 72), (4, 4, 640, 73), (8, 2, 131072, 74),
                             (14, 2, 131072, 77), (4, 2, 1001, 75), (2, 1, 200, 76)):
        w = synth.small("host", hq, hkv, n, seed)
        q, k, v = w.generate()
        params = crisp.params_default()
        qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
        ref = empty((hq, n, 128), torch.bfloat16)
        s = crisp.make_shape(hq, hkv, n, qd, kd, ref)
        ws = new_workspace(s, layer=True)
        crisp.prefill_layer(s, params, qd, kd, vd, ref, ws)
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).pin_memory()
        qh, kh, vh = pin(q), pin(k), pin(v)
        oh = torch.zeros((hq, n, 128), dtype=torch.int16).pin_memory()
        qs, ks, vs = (torch.empty_like(t) for t in (qd, kd, vd))
        os_ = empty((hq, n, 128), torch.bfloat16)
        ws2 = new_workspace(s, layer=True)
        crisp.prefill_layer_host(pipe, s, params, qh, kh, vh, oh, qs, ks, vs, os_, ws2)
        torch.cuda.synchronize()
        assert_status_ok(ws2)
        assert torch.equal(qs, qd) and torch.equal(ks, kd) and torch.equal(vs, vd)
        assert torch.equal(os_, ref)
        assert torch.equal(oh.view(torch.bfloat16).cuda(), ref)
    pipe.close()


def test_gqa4x1_2k_full_layer():
    w = synth.WORKLOADS["gqa4x1-2k"]
    q, k, v = w.generate()
    params = crisp.params_default()
    r = run_steps(q, k, v, params)
    check_map(r["pmap"], oracle.proxy_map(q, k))
    rb, route = check_index_sets(r, params)
    assert route.tolist() == [1, 1, 1, 1]
    check_attention(q, k, v, r["out"], rb)


def test_repeat_calls_are_deterministic():
    w = synth.small("repeat", 8, 2, 2048, 61)
    q, k, v = w.generate()
    params = crisp.params_default()
    a = run_steps(q, k, v, params)
    b = run_steps(q, k, v, params)
    for key in ("pmap", "vmass", "smass", "rowbits", "pbar"):
        assert np.array_equal(a[key], b[key]), key
    assert torch.equal(a["out"], b["out"])


# --------------------------------------------------------------------------
# FlexPrefill comparators (divergence routing, cumulative coverage on VS
# heads) and the length gate.

def run_comparator_steps(q, k, v, params):
    """A1+A3 fused, the pooled map of every head, divergence routing, then
    A4..A8 as in the layer; returns numpy copies and the output."""
    hq, n, _ = q.shape
    hkv = k.shape[0]
    nb = crisp.num_blocks(n)
    W = (nb + 31) // 32
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    out = empty((hq, n, 128), torch.bfloat16)
    s = crisp.make_shape(hq, hkv, n, qd, kd, out)
    ws = new_workspace(s)
    vmass, smass = empty((hq, nb), torch.int64), empty((hq, nb), torch.int64)
    rmass = empty((hq,), torch.int64)
    route = torch.zeros((hq,), dtype=torch.uint8, device="cuda")
    jsd = empty((hq,), torch.float64)
    vbits, sbits = empty((hq, W), torch.int32), empty((hq, W), torch.int32)
    pbar = torch.zeros((hq, nb, nb), dtype=torch.float32, device="cuda")
    pebits, rowbits = empty((hq, nb, W), torch.int32), empty((hq, nb, W), torch.int32)
    counts, order = empty((hq, nb), torch.int32), empty((hq * nb,), torch.int32)
    crisp.proxy_masses(s, qd, kd, vmass, smass, rmass, ws)
    crisp.pe_pool(s, qd, kd, route, pbar, ws)  # route all zeros: every head's pooled map
    crisp.route_jsd(s, params, vmass, pbar, jsd, route, ws)
    crisp.select_vs_masses(s, params, vmass, smass, route, vbits, sbits, ws)
    crisp.select_pe(s, params, pbar, route, pebits, ws)
    crisp.build_mask(s, route, vbits, sbits, pebits, rowbits, counts, order, ws)
    crisp.sparse_prefill_mask(s, qd, kd, vd, rowbits, order, out, ws)
    torch.cuda.synchronize()
    assert_status_ok(ws)
    u64 = lambda t: t.cpu().numpy().view(np.uint64)
    u32 = lambda t: t.cpu().numpy().view(np.uint32)
    return dict(vmass=u64(vmass), smass=u64(smass), route=route.cpu().numpy(), jsd=jsd.cpu().numpy(),
                vbits=u32(vbits), sbits=u32(sbits), pbar=pbar.cpu().numpy(), pebits=u32(pebits),
                rowbits=u32(rowbits), out=out)


COMPARATOR_CASES = [
    # name, hq, hkv, n, seed, jsd_tau, vs_gamma
    ("mixed-2k-t02", 8, 2, 2048, 2, 0.2, (95, 100)),
    ("gqa4-4k-t01", 4, 1, 4096, 9, 0.1, (95, 100)),
    ("gqa7-1152-t02", 7, 1, 1152, 6, 0.2, (97, 100)),
    ("nb33-4224-t03", 4, 2, 4224, 7, 0.3, (9, 10)),
    ("ragged-2100-t02", 4, 2, 2100, 36, 0.2, (95, 100)),
]


@pytest.mark.parametrize("name,hq,hkv,n,seed,tau,vg", COMPARATOR_CASES, ids=[c[0] for c in COMPARATOR_CASES])
def test_flexprefill_comparators_match_oracle(name, hq, hkv, n, seed, tau, vg):
    w = synth.small(name, hq, hkv, n, seed)
    q, k, v = w.generate()
    params = crisp.params_default(route_mode=crisp.ROUTE_JSD, vs_mode=crisp.VS_GAMMA, jsd_tau=tau, vs_gamma=vg)
    r = run_comparator_steps(q, k, v, params)
    nb = crisp.num_blocks(n)
    # masses as in the CRISP path (the fused pass is checked elsewhere)
    ref_map = run_steps(q, k, v, crisp.params_default())
    assert np.array_equal(r["vmass"], ref_map["vmass"]) and np.array_equal(r["smass"], ref_map["smass"])
    # divergence in fp64 on both sides, from the GPU's own masses and pooled rows
    D, route = oracle.route_jsd(r["vmass"], r["pbar"][:, nb - 1, :], tau=params.jsd_tau)
    assert np.allclose(r["jsd"], D, rtol=1e-12, atol=1e-15)
    near = np.abs(np.sqrt(np.maximum(D, 0)) - params.jsd_tau) < 1e-9  # either decision is correct there
    assert np.array_equal(r["route"][~near], route[~near])
    route = r["route"]
    vb, sb = oracle.select_vs_gamma(r["vmass"], r["smass"], route, gamma=vg, kmin=params.kmin_blocks)
    assert np.array_equal(vb, r["vbits"]) and np.array_equal(sb, r["sbits"])
    pbar = r["pbar"].copy()
    pe = oracle.select_pe(pbar, route, pe_mode=params.pe_mode, gamma=(params.gamma_num, params.gamma_den),
                          alpha=(params.alpha_num, params.alpha_den), kmin=params.kmin_blocks)
    assert np.array_equal(pe, r["pebits"])
    rb = oracle.build_mask(route, vb, sb, pe)
    assert np.array_equal(rb, r["rowbits"])
    check_attention(q, k, v, r["out"], rb, rows=sample_rows(hq, n, 24, seed))


def test_prefill_layer_comparator_mode_matches_steps():
    w = synth.small("layer-flex", 8, 2, 2048, 91)
    q, k, v = w.generate()
    params = crisp.params_default(route_mode=crisp.ROUTE_JSD, vs_mode=crisp.VS_GAMMA, jsd_tau=0.2)
    steps = run_comparator_steps(q, k, v, params)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    out = empty((8, 2048, 128), torch.bfloat16)
    s = crisp.make_shape(8, 2, 2048, qd, kd, out)
    ws = new_workspace(s, layer=True)
    crisp.prefill_layer(s, params, qd, kd, vd, out, ws)
    torch.cuda.synchronize()
    assert_status_ok(ws)
    assert torch.equal(out, steps["out"])
    assert 0 < steps["route"].sum() < 8  # both routes exercised


@pytest.mark.parametrize("n", [1024, 1000])
def test_route_cstruct_other_slice_widths(n):
    # crisp_route_cstruct reads the map itself, so any slice widths work; bit
    # for bit against the oracle on the GPU's own map, the overlap of the two
    # slices counted once.
    hq, hkv = 4, 2
    w = synth.small("slices", hq, hkv, n, 81, vs_heads=[0])
    q, k, _ = w.generate()
    qd, kd = to_dev(q), to_dev(k)
    s = crisp.make_shape(hq, hkv, n, qd, kd)
    ws = new_workspace(s)
    pmap = empty((hq, B, crisp.map_ld(n)), torch.float32)
    crisp.proxy_map(s, qd, kd, pmap, ws)
    pm = np.ascontiguousarray(pmap.cpu().numpy()[:, :, :n])
    for sink, recency, tau in ((64, 128, (1, 5)), (1, 300, (1, 10)), (0, 128, (1, 5)), (700, 500, (1, 2)),
                               (2000, 2000, (1, 1)), (128, 128, (1, 5))):
        params = crisp.params_default(sink_tokens=sink, recency_tokens=recency, tau=tau)
        cs, tot, route = empty((hq,), torch.int64), empty((hq,), torch.int64), empty((hq,), torch.uint8)
        crisp.route_cstruct(s, params, pmap, cs, tot, route, ws)
        torch.cuda.synchronize()
        assert_status_ok(ws)
        S, T, r = oracle.route(pm, tau=tau, sink=sink, recency=recency)
        assert np.array_equal(cs.cpu().numpy().view(np.uint64), S), (sink, recency)
        assert np.array_equal(tot.cpu().numpy().view(np.uint64), T), (sink, recency)
        assert np.array_equal(route.cpu().numpy(), r), (sink, recency)


# The pages' two ablations ("Main Findings"): routing alone (C_struct with
# FlexPrefill's coverage selection on VS heads) and sink-aware selection alone
# (FlexPrefill's divergence routing with CRISP's noise floor).
ABLATIONS = [("routing-only", crisp.ROUTE_CSTRUCT, crisp.VS_GAMMA), ("selection-only", crisp.ROUTE_JSD, crisp.VS_NOISE)]


@pytest.mark.parametrize("name,route_mode,vs_mode", ABLATIONS, ids=[a[0] for a in ABLATIONS])
def test_prefill_layer_ablation_modes(name, route_mode, vs_mode):
    hq, hkv, n, seed = 8, 2, 2048, 93
    w = synth.small("ablation", hq, hkv, n, seed)
    q, k, v = w.generate()
    params = crisp.params_default(route_mode=route_mode, vs_mode=vs_mode, jsd_tau=0.2)
    nb = crisp.num_blocks(n)
    if route_mode == crisp.ROUTE_JSD:
        steps = run_comparator_steps(q, k, v, params)
        D, route = oracle.route_jsd(steps["vmass"], steps["pbar"][:, nb - 1, :], tau=params.jsd_tau)
        near = np.abs(np.sqrt(np.maximum(D, 0)) - params.jsd_tau) < 1e-9
        assert np.array_equal(steps["route"][~near], route[~near])
        route = steps["route"]
        pbar = steps["pbar"]
    else:
        steps = run_steps(q, k, v, params)
        _, _, route = oracle.route(steps["pmap"])
        assert np.array_equal(route, steps["route"])
        pbar = steps["pbar"].copy()
        pbar[route == 1] = 0.0
    if vs_mode == crisp.VS_GAMMA:
        vb, sb = oracle.select_vs_gamma(steps["vmass"], steps["smass"], route, gamma=(95, 100), kmin=8)
    else:
        vb, sb = oracle.select_vs(steps["vmass"], steps["smass"], route, kmin=8)
    assert np.array_equal(vb, steps["vbits"]) and np.array_equal(sb, steps["sbits"])
    pe = oracle.select_pe(pbar, route)
    assert np.array_equal(pe, steps["pebits"])
    rb = oracle.build_mask(route, vb, sb, pe)
    assert np.array_equal(rb, steps["rowbits"])
    assert 0 < route.sum() < hq  # both routes exercised
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    out = empty((hq, n, 128), torch.bfloat16)
    s = crisp.make_shape(hq, hkv, n, qd, kd, out)
    ws = new_workspace(s, layer=True)
    crisp.prefill_layer(s, params, qd, kd, vd, out, ws)
    torch.cuda.synchronize()
    assert_status_ok(ws)
    assert torch.equal(out, steps["out"])
    check_attention(q, k, v, out, rb, rows=sample_rows(hq, n, 24, seed))


def test_length_gate_runs_dense():
    n = 4096  # 32 blocks: the sparse selection keeps fewer than all of them
    w = synth.small("gate", 4, 1, n, 92)
    q, k, v = w.generate()
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    out, ref = empty((4, n, 128), torch.bfloat16), empty((4, n, 128), torch.bfloat16)
    s = crisp.make_shape(4, 1, n, qd, kd, out)
    ws = new_workspace(s, layer=True)
    crisp.dense_prefill(s, qd, kd, vd, ref, ws)
    crisp.prefill_layer(s, crisp.params_default(dense_below=n + 1), qd, kd, vd, out, ws)
    torch.cuda.synchronize()
    assert_status_ok(ws)
    assert torch.equal(out, ref)
    crisp.prefill_layer(s, crisp.params_default(dense_below=n), qd, kd, vd, out, ws)  # not below: sparse
    torch.cuda.synchronize()
    assert not torch.equal(out, ref)


def test_short_and_empty_layers():
    # n = 0 launches nothing; below two blocks the layer is dense attention
    # (bit-identical to crisp_dense_prefill); a ragged short layer too.
    params = crisp.params_default()
    for hq, hkv, n, seed in ((4, 2, 0, 0), (4, 2, 1, 93), (2, 1, 100, 94), (4, 1, 200, 95)):
        qd = torch.randn((hq, n, 128), device="cuda").to(torch.bfloat16)
        kd = torch.randn((hkv, n, 128), device="cuda").to(torch.bfloat16)
        vd = torch.randn((hkv, n, 128), device="cuda").to(torch.bfloat16)
        out = torch.full((hq, n, 128), 7.0, dtype=torch.bfloat16, device="cuda")
        ref = empty((hq, n, 128), torch.bfloat16)
        s = crisp.make_shape(hq, hkv, n, qd, kd, out)
        ws = new_workspace(s, layer=True)
        crisp.prefill_layer(s, params, qd, kd, vd, out, ws)
        crisp.dense_prefill(s, qd, kd, vd, ref, ws)
        torch.cuda.synchronize()
        assert_status_ok(ws)
        assert torch.equal(out, ref)
        if n:
            q, k, v = (bf16_to_u16(t) for t in (qd, kd, vd))
            check_attention(q, k, v, out, None)


def test_attention_is_deterministic_under_load():
    # Many short rows (the first block of every row takes the exact path,
    # where the two warps of a lane quarter exchange maxima and re-read S):
    # repeated launches must give identical bits, and the shortest rows must
    # match the oracle.
    hq, hkv, n = 16, 4, 16384
    w = synth.small("stress", hq, hkv, n, 111)
    q, k, v = w.generate()
    params = crisp.params_default()
    r = run_steps(q, k, v, params)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    s = crisp.make_shape(hq, hkv, n, qd, kd, r["out"])
    ws = new_workspace(s)
    rb = torch.from_numpy(r["rowbits"].view(np.int32)).cuda()
    order = torch.from_numpy(r["order"]).cuda()
    for _ in range(4):
        out = empty((hq, n, 128), torch.bfloat16)
        crisp.sparse_prefill_mask(s, qd, kd, vd, rb, order, out, ws)
        torch.cuda.synchronize()
        assert_status_ok(ws)
        assert torch.equal(out, r["out"])
    heads = np.repeat(np.arange(hq), 3 * B).astype(np.int32)
    toks = np.tile(np.arange(3 * B), hq).astype(np.int32)  # query blocks 0..2 of every head
    ref = oracle.attention_rows(q, k, v, heads, toks, rowbits=r["rowbits"])
    got = r["out"].float().cpu().numpy()[heads, toks]
    mx, mean = attn_error(got, ref)
    assert mx <= ATT_MAX and mean <= ATT_MEAN, (mx, mean)


def test_prefill_layer_replays_from_a_cuda_graph():
    # Every call enqueues on the caller's stream and allocates nothing, so a
    # whole layer can be captured once and replayed (the short-sequence case
    # is launch-bound: 12 launches for a 2k-token layer).
    w = synth.small("graph", 8, 2, 2048, 121)
    q, k, v = w.generate()
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    out, ref = empty((8, 2048, 128), torch.bfloat16), empty((8, 2048, 128), torch.bfloat16)
    s = crisp.make_shape(8, 2, 2048, qd, kd, out)
    params = crisp.params_default()
    ws = new_workspace(s, layer=True)
    crisp.prefill_layer(s, params, qd, kd, vd, ref, ws)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up on a side stream before capture
        crisp.prefill_layer(s, params, qd, kd, vd, out, ws, stream=side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        crisp.prefill_layer(s, params, qd, kd, vd, out, ws, stream=torch.cuda.current_stream())
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert_status_ok(ws)
    assert torch.equal(out, ref)
