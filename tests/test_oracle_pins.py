"""Pins the CPU oracle to facts other than itself: closed forms, invariants,
library special cases (torch softmax / scaled_dot_product_attention in fp64),
hand-worked fixtures and brute force on tiny inputs. No GPU needed."""
import itertools
import os

import numpy as np
import pytest
import torch

import oracle
import synth

B = 128


def bf16_bits(x):
    """float array -> bf16 bit patterns (round to nearest even via torch)."""
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(b):
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).double()


def rand_qkv(hq, hkv, n, seed):
    rng = np.random.default_rng(seed)
    q = bf16_bits(rng.standard_normal((hq, n, 128)))
    k = bf16_bits(rng.standard_normal((hkv, n, 128)))
    v = bf16_bits(rng.standard_normal((hkv, n, 128)))
    return q, k, v


def sets_of(bits, nb):
    return oracle.bits_to_sets(bits, nb)


# ----------------------------------------------------------------- A1 proxy
def test_proxy_rows_sum_to_one_and_causal():
    q, k, _ = rand_qkv(3, 1, 384, 1)
    P = oracle.proxy_map(q, k)
    assert np.allclose(P.sum(-1), 1.0, atol=1e-12)
    n = 384
    for r in range(B):
        assert np.all(P[:, r, n - B + r + 1:] == 0.0)
        assert np.all(P[:, r, : n - B + r + 1] > 0.0)


def test_proxy_uniform_keys_closed_form():
    # Identical keys: every visible key gets the same logit, so P = 1/(i+1).
    rng = np.random.default_rng(2)
    n = 256
    q = bf16_bits(rng.standard_normal((2, n, 128)))
    row = bf16_bits(rng.standard_normal(128))
    k = np.broadcast_to(row, (1, n, 128)).copy()
    P = oracle.proxy_map(q, k)
    for r in range(B):
        i = n - B + r
        assert np.allclose(P[:, r, : i + 1], 1.0 / (i + 1), rtol=1e-12)


def test_proxy_matches_torch_softmax():
    # Library special case: softmax of masked logits computed by torch (fp64).
    q, k, _ = rand_qkv(4, 2, 512, 3)
    P = oracle.proxy_map(q, k)
    Q = bits_to_f64(q)[:, -B:, :]
    K = bits_to_f64(k).repeat_interleave(2, dim=0)
    S = torch.einsum("hrd,hjd->hrj", Q, K) / np.sqrt(128.0)
    n = 512
    i = torch.arange(n - B, n)[:, None]
    j = torch.arange(n)[None, :]
    S = S.masked_fill(j > i, float("-inf"))
    ref = torch.softmax(S, dim=-1).numpy()
    assert np.max(np.abs(ref - P)) < 1e-13


# ----------------------------------------------------------------- quanta
def test_quantize_round_half_even():
    p = np.array([0.0, 1.0, 0.5, 2.0 ** -33, 3 * 2.0 ** -33, 5 * 2.0 ** -33, 2.0 ** -40, 0.1], np.float32)
    got = oracle.quantize(p)
    want = np.rint(p.astype(np.float64) * 2.0 ** 32).astype(np.uint64)  # numpy rint: ties to even
    assert got.tolist() == want.tolist()
    assert got[1] == 2 ** 32 and got[2] == 2 ** 31
    assert got[3] == 0 and got[4] == 2 and got[5] == 2 and got[6] == 0


# ----------------------------------------------------------------- A2 route
def _small_map(seed=5):
    w = synth.small("pins", 4, 2, 1024, seed)
    q, k, _ = w.generate()
    return w, oracle.proxy_map(q, k).astype(np.float32)


def test_cstruct_equals_brute_force_slice_sum():
    w, P = _small_map()
    S, T, r = oracle.route(P)
    Q = np.rint(P.astype(np.float64) * 2.0 ** 32).astype(np.uint64)
    n = w.n
    S_bf = Q[:, :, :128].sum(axis=(1, 2)) + Q[:, :, n - 128:].sum(axis=(1, 2))
    assert S.tolist() == S_bf.tolist()
    assert T.tolist() == Q.sum(axis=(1, 2)).tolist()
    vm, _ = oracle.vs_masses(P)
    assert S.tolist() == (vm[:, 0] + vm[:, -1]).tolist()


@pytest.mark.parametrize("sink,recency", [(64, 128), (1, 300), (0, 128), (128, 0), (700, 500), (1024, 1024)])
def test_cstruct_other_slice_widths_brute_force(sink, recency):
    # The slice widths as parameters (the pages fix both at 128): brute-force
    # numpy sums over the union of the two column ranges, a column inside
    # both counted once (n = 1024: 700 + 500 overlap, 1024 + 1024 is all).
    w, P = _small_map()
    S, T, _ = oracle.route(P, sink=sink, recency=recency)
    Q = np.rint(P.astype(np.float64) * 2.0 ** 32).astype(np.uint64)
    n = w.n
    cols = np.zeros(n, bool)
    cols[:sink] = True
    if recency:
        cols[max(0, n - recency):] = True
    assert S.tolist() == Q[:, :, cols].sum(axis=(1, 2)).tolist()
    assert T.tolist() == Q.sum(axis=(1, 2)).tolist()
    if sink + recency >= n:
        assert S.tolist() == T.tolist()


def test_route_tau_tie_goes_to_vs():
    # n = 384: sink block 0, middle block 1, recency block 2. Every row puts
    # 1/8 at column 0, 3/4 at column 200 and 1/8 at column 300: C = 1/4.
    n = 384
    P = np.zeros((1, B, n), np.float32)
    P[0, :, 0] = 0.125
    P[0, :, 200] = 0.75
    P[0, :, 300] = 0.125
    _, _, r = oracle.route(P, tau=(1, 4))
    assert r[0] == 1  # tie: C_struct == tau -> VS
    _, _, r = oracle.route(P, tau=(3, 10))
    assert r[0] == 0
    _, _, r = oracle.route(P, tau=(1, 5))
    assert r[0] == 1


def test_route_planted_heads():
    # Diffuse heads attend to their query block's cluster (1/8 of the blocks);
    # at 16k that spreads the mass well below tau over sink + recency.
    w = synth.small("route", 4, 2, 16384, 11, vs_heads=[0, 3], d_sink=6.0)
    q, k, _ = w.generate()
    _, _, r = oracle.route(oracle.proxy_map(q, k).astype(np.float32))
    assert r.tolist() == [1, 0, 0, 1]


# ----------------------------------------------------------------- A3 masses
@pytest.mark.parametrize("r,j", [(0, 0), (5, 127), (5, 128), (127, 640), (10, 500), (127, 129), (0, 511)])
def test_vs_masses_single_entry_closed_form(r, j):
    n = 768
    i = n - B + r
    P = np.zeros((1, B, n), np.float32)
    P[0, r, j] = 1.0
    vm, sm = oracle.vs_masses(P)
    want_v = np.zeros(n // B, np.uint64)
    want_v[j // B] = 2 ** 32
    want_s = np.zeros(n // B, np.uint64)
    if 128 <= j <= i:
        want_s[(i - j) // B] = 2 ** 32
    assert vm[0].tolist() == want_v.tolist()
    assert sm[0].tolist() == want_s.tolist()


def test_vs_masses_sum_invariants():
    _, P = _small_map(7)
    vm, sm = oracle.vs_masses(P)
    _, T, _ = oracle.route(P)
    assert vm.sum(axis=1).tolist() == T.tolist()
    assert sm.sum(axis=1).tolist() == (T - vm[:, 0]).tolist()
    assert np.all(sm[:, -1] == 0)  # offsets >= (nb-1)*B cannot reach j >= 128


# ----------------------------------------------------------------- A4 select
def _read_vs_fixture(golden_dir):
    rows = []
    for line in open(os.path.join(golden_dir, "noise_floor_vs.txt")):
        if line.startswith("#") or not line.strip():
            continue
        a, ev, es = line.split("|")
        an, ad, km = (int(x) for x in a.split())
        rows.append((an, ad, km, [int(x) for x in ev.split()], [int(x) for x in es.split()]))
    return rows


def test_select_vs_hand_fixture(golden_dir):
    vmass = np.array([[1000, 10, 10, 50, 10, 10, 10, 30, 10, 10, 10, 500]], np.uint64)
    smass = np.array([[7, 0, 0, 40, 0, 0, 0, 0, 0, 0, 20, 0]], np.uint64)
    rows = _read_vs_fixture(golden_dir)
    assert len(rows) == 8
    for an, ad, km, ev, es in rows:
        vb, sb = oracle.select_vs(vmass, smass, np.ones(1, np.uint8), alpha=(an, ad), kmin=km)
        assert sets_of(vb, 12)[0] == ev, (an, ad, km)
        assert sets_of(sb, 12)[0] == es, (an, ad, km)


def test_select_vs_equal_masses_fill_lowest():
    nb = 40
    vm = np.full((1, nb), 1000, np.uint64)
    vb, sb = oracle.select_vs(vm, vm, np.ones(1, np.uint8), alpha=(1, 1), kmin=8)
    assert sets_of(vb, nb)[0] == [0, 1, 2, 3, 4, 5, 6, nb - 1]
    assert sets_of(sb, nb)[0] == [0, 1, 2, 3, 4, 5, 6, 7]


def test_select_vs_alpha_zero_keeps_nonzero():
    rng = np.random.default_rng(4)
    nb = 64
    vm = rng.integers(0, 5, (1, nb)).astype(np.uint64)
    vb, sb = oracle.select_vs(vm, vm, np.ones(1, np.uint8), alpha=(0, 1), kmin=0)
    nz = [c for c in range(1, nb - 1) if vm[0, c] > 0]
    assert sets_of(vb, nb)[0] == sorted(set([0, nb - 1] + nz))
    assert sets_of(sb, nb)[0] == sorted(set([0] + nz))


def test_select_vs_pe_heads_empty():
    vm = np.ones((2, 16), np.uint64)
    vb, sb = oracle.select_vs(vm, vm, np.array([0, 1], np.uint8))
    assert sets_of(vb, 16)[0] == [] and sets_of(sb, 16)[0] == []
    assert sets_of(vb, 16)[1] != []


def test_select_vs_small_nb_edges():
    for nb in (2, 3):
        vm = np.arange(1, nb + 1, dtype=np.uint64)[None, :]
        vb, sb = oracle.select_vs(vm, vm, np.ones(1, np.uint8), kmin=8)
        assert sets_of(vb, nb)[0] == list(range(nb))
        assert sets_of(sb, nb)[0] == list(range(nb - 1))  # slash candidates [1, nb-2]


def test_select_vs_recovers_planted_structure():
    w = synth.small("planted", 2, 1, 8192, 21, vs_heads=[0], d_sink=6.0, n_needles=4, d_needle=9.0, n_slash=1,
                    d_slash=9.0, slash_min=1024, slash_max=2048)
    q, k, _ = w.generate()
    P = oracle.proxy_map(q, k).astype(np.float32)
    _, _, r = oracle.route(P)
    assert r.tolist() == [1, 0]
    vm, sm = oracle.vs_masses(P)
    vb, sb = oracle.select_vs(vm, sm, r)
    nb = w.n // B
    V, S = sets_of(vb, nb)[0], sets_of(sb, nb)[0]
    for p in w.needle_positions(0):
        assert p // B in V
    # A slash at offset d crosses offset blocks floor(d/B) (and +1 for rows
    # past the block boundary) in the last query block.
    d = w.slash_offsets(0)[0]
    assert d // B in S or (d // B + 1) in S


def test_select_vs_count_flat_in_n():
    # The number of kept blocks is an output of the input, not of n.
    counts = []
    for n in (4096, 8192, 16384):
        w = synth.small("flat", 2, 1, n, 3, vs_heads=[0], d_sink=6.0, n_needles=4, d_needle=9.0, n_slash=0)
        q, k, _ = w.generate()
        P = oracle.proxy_map(q, k).astype(np.float32)
        vm, sm = oracle.vs_masses(P)
        vb, _ = oracle.select_vs(vm, sm, np.ones(2, np.uint8), kmin=0)
        counts.append(len(sets_of(vb[:1], n // B)[0]))
    assert max(counts) - min(counts) <= 3, counts


# ----------------------------------------------------------------- A5 PE map
def test_pe_map_matches_torch():
    q, k, _ = rand_qkv(4, 2, 1024, 8)
    got = oracle.pe_map(q, k)
    Q = bits_to_f64(q).reshape(4, 8, B, 128).mean(dim=2)
    K = bits_to_f64(k).reshape(2, 8, B, 128).mean(dim=2).repeat_interleave(2, dim=0)
    Z = torch.einsum("hbd,hcd->hbc", Q, K) / np.sqrt(128.0)
    mask = torch.triu(torch.ones(8, 8, dtype=torch.bool), diagonal=1)
    ref = torch.softmax(Z.masked_fill(mask, float("-inf")), dim=-1).numpy()
    assert np.max(np.abs(ref - got)) < 1e-13


# ----------------------------------------------------------------- A6 PE select
def _pe_row_fixture(golden_dir):
    rows = []
    for line in open(os.path.join(golden_dir, "pe_row.txt")):
        if line.startswith("#") or not line.strip():
            continue
        a, e = line.split("|")
        mode, num, den = a.split()
        rows.append((mode, int(num), int(den), [int(x) for x in e.split()]))
    return rows


def test_select_pe_hand_fixture(golden_dir):
    nb = 6
    pbar = np.zeros((1, nb, nb), np.float32)
    pbar[0, 5] = [0.5, 0.125, 0.25, 0.0625, 0.03125, 0.03125]
    rows = _pe_row_fixture(golden_dir)
    assert len(rows) == 8
    for mode, num, den, want in rows:
        if mode == "gamma":
            pe = oracle.select_pe(pbar, np.zeros(1, np.uint8), pe_mode=0, gamma=(num, den), kmin=1)
        else:
            pe = oracle.select_pe(pbar, np.zeros(1, np.uint8), pe_mode=1, alpha=(num, den), kmin=1)
        assert sets_of(pe[0, 5], nb)[0] == want, (mode, num, den)


def test_select_pe_gamma_one_keeps_all_nonzero():
    rng = np.random.default_rng(9)
    nb = 20
    pbar = rng.random((1, nb, nb)).astype(np.float32)
    pbar[0, :, 3] = 0.0
    pbar = np.tril(pbar[0])[None]
    pe = oracle.select_pe(pbar, np.zeros(1, np.uint8), gamma=(1, 1), kmin=0)
    for b in range(nb):
        want = sorted(set([c for c in range(b + 1) if pbar[0, b, c] > 0] + [0, b]))
        assert sets_of(pe[0, b], nb)[0] == want


def test_select_pe_gamma_tiny_keeps_top1():
    rng = np.random.default_rng(10)
    nb = 16
    pbar = np.tril(rng.random((nb, nb))).astype(np.float32)[None]
    pe = oracle.select_pe(pbar, np.zeros(1, np.uint8), gamma=(1, 10 ** 9), kmin=0)
    for b in range(nb):
        top = int(np.argmax(pbar[0, b, : b + 1]))
        assert sets_of(pe[0, b], nb)[0] == sorted({0, b, top})


def test_select_pe_gamma_brute_force():
    # Tiny rows with distinct masses: the kept prefix must be a minimum-size
    # subset reaching gamma of the row mass, and the heaviest such subset.
    rng = np.random.default_rng(12)
    nb = 8
    for trial in range(20):
        pbar = np.tril(rng.random((nb, nb)) + 1e-3).astype(np.float32)
        pbar /= pbar.sum(axis=1, keepdims=True)
        pbar = pbar.astype(np.float32)[None]
        gnum, gden = int(rng.integers(1, 20)), 20
        pe = oracle.select_pe(pbar, np.zeros(1, np.uint8), gamma=(gnum, gden), kmin=0)
        for b in range(nb):
            m = np.rint(pbar[0, b, : b + 1].astype(np.float64) * 2.0 ** 32).astype(np.int64)
            T = int(m.sum())
            best = None
            for size in range(0, b + 2):
                cands = [s for s in itertools.combinations(range(b + 1), size) if gden * int(m[list(s)].sum()) >= gnum * T]
                if cands:
                    best = max(cands, key=lambda s: int(m[list(s)].sum()))
                    break
            want = sorted(set(best) | {0, b})
            assert sets_of(pe[0, b], nb)[0] == want, (trial, b)


def test_select_pe_route_vs_gives_empty_rows():
    pbar = np.tril(np.ones((6, 6), np.float32))[None] / 6
    pe = oracle.select_pe(pbar, np.ones(1, np.uint8))
    assert all(s == [] for s in sets_of(pe[0], 6))


# ----------------------------------------------------------------- A7 mask
def test_build_mask_matches_token_level_definition():
    # Brute force over tokens (B = 128 per block): key block kb is in row qb iff
    # kb is a kept vertical block (kb <= qb) or some token pair (i, j), i in
    # block qb, j in block kb, j <= i, has floor((i - j)/B) in S.
    nb = 6
    vb = np.zeros((1, 1), np.uint32)
    sb = np.zeros((1, 1), np.uint32)
    vb[0, 0] = (1 << 0) | (1 << 4)
    sb[0, 0] = (1 << 0) | (1 << 2)
    pe = np.zeros((1, nb, 1), np.uint32)
    rb = oracle.build_mask(np.ones(1, np.uint8), vb, sb, pe)
    S = {0, 2}
    for qb in range(nb):
        want = set(kb for kb in (0, 4) if kb <= qb)
        ii = np.arange(qb * B, qb * B + B)[:, None]
        for kb in range(qb + 1):
            jj = np.arange(kb * B, kb * B + B)[None, :]
            off = (ii - jj) // B
            if np.any((jj <= ii) & np.isin(off, list(S))):
                want.add(kb)
        assert sets_of(rb[0, qb], nb)[0] == sorted(want), qb


def test_build_mask_pe_rows_copied():
    rng = np.random.default_rng(13)
    nb = 40
    pe = rng.integers(0, 2 ** 32, (1, nb, 2), dtype=np.uint64).astype(np.uint32)
    rb = oracle.build_mask(np.zeros(1, np.uint8), np.zeros((1, 2), np.uint32), np.zeros((1, 2), np.uint32), pe)
    for qb in range(nb):
        assert sets_of(rb[0, qb], nb)[0] == [c for c in sets_of(pe[0, qb], nb)[0] if c <= qb]


# ----------------------------------------------------------------- A8/A9 attention
def _all_tokens(hq, n):
    h, t = np.meshgrid(np.arange(hq), np.arange(n), indexing="ij")
    return h.ravel().astype(np.int32), t.ravel().astype(np.int32)


def test_dense_attention_matches_sdpa():
    hq, hkv, n = 4, 2, 384
    q, k, v = rand_qkv(hq, hkv, n, 14)
    h, t = _all_tokens(hq, n)
    got = oracle.attention_rows(q, k, v, h, t).reshape(hq, n, 128)
    Q, K, V = bits_to_f64(q), bits_to_f64(k), bits_to_f64(v)
    ref = torch.nn.functional.scaled_dot_product_attention(
        Q[None], K.repeat_interleave(2, 0)[None], V.repeat_interleave(2, 0)[None], is_causal=True)[0].numpy()
    assert np.max(np.abs(ref - got)) < 1e-12


def test_sparse_attention_matches_masked_sdpa():
    hq, hkv, n = 2, 1, 768
    nb = n // B
    q, k, v = rand_qkv(hq, hkv, n, 15)
    rng = np.random.default_rng(16)
    rb = np.zeros((hq, nb, 1), np.uint32)
    for hh in range(hq):
        for qb in range(nb):
            keep = [kb for kb in range(qb + 1) if rng.random() < 0.5] + [qb]
            for kb in keep:
                rb[hh, qb, 0] |= np.uint32(1 << kb)
    h, t = _all_tokens(hq, n)
    got = oracle.attention_rows(q, k, v, h, t, rowbits=rb).reshape(hq, n, 128)
    mask = torch.zeros(hq, n, n, dtype=torch.bool)
    for hh in range(hq):
        for qb in range(nb):
            for kb in range(nb):
                if (int(rb[hh, qb, 0]) >> kb) & 1:
                    mask[hh, qb * B:(qb + 1) * B, kb * B:(kb + 1) * B] = True
    mask &= torch.tril(torch.ones(n, n, dtype=torch.bool))
    Q, K, V = bits_to_f64(q), bits_to_f64(k), bits_to_f64(v)
    ref = torch.nn.functional.scaled_dot_product_attention(Q[None], K.repeat_interleave(2, 0)[None],
                                                           V.repeat_interleave(2, 0)[None], attn_mask=mask[None])
    assert np.max(np.abs(ref[0].numpy() - got)) < 1e-12


def test_attention_constant_v_returns_v():
    hq, n = 2, 256
    q, k, _ = rand_qkv(hq, 1, n, 17)
    vrow = bf16_bits(np.linspace(-2, 2, 128))
    v = np.broadcast_to(vrow, (1, n, 128)).copy()
    h, t = _all_tokens(hq, n)
    got = oracle.attention_rows(q, k, v, h, t)
    assert np.allclose(got, bits_to_f64(vrow).numpy()[None, :], atol=1e-12)


def test_attention_one_hot_v_gives_probabilities():
    # n = 128 and v_j = e_j: output row i is the softmax row of token i, which
    # is also the proxy map row (the last block is the only block).
    n = 128
    q, k, _ = rand_qkv(2, 1, n, 18)
    v = bf16_bits(np.eye(128))[None]
    h, t = _all_tokens(2, n)
    got = oracle.attention_rows(q, k, v, h, t).reshape(2, n, 128)
    P = oracle.proxy_map(q, k)
    assert np.max(np.abs(got - P)) < 1e-12


def test_select_all_equals_dense_and_pair_count():
    hq, n = 2, 512
    nb = n // B
    q, k, v = rand_qkv(hq, 1, n, 19)
    rb = np.zeros((hq, nb, 1), np.uint32)
    for qb in range(nb):
        rb[:, qb, 0] = (1 << (qb + 1)) - 1
    h, t = _all_tokens(hq, n)
    a = oracle.attention_rows(q, k, v, h, t, rowbits=rb)
    d = oracle.attention_rows(q, k, v, h, t)
    assert np.array_equal(a, d)
    assert oracle.selected_pairs(rb, n) == hq * n * (n + 1) // 2


def test_empty_row_mask_gives_zero_output():
    q, k, v = rand_qkv(1, 1, 256, 20)
    rb = np.zeros((1, 2, 1), np.uint32)
    out = oracle.attention_rows(q, k, v, np.zeros(3, np.int32), np.array([0, 130, 255], np.int32), rowbits=rb)
    assert np.all(out == 0.0)


# ----------------------------------------------------------------- ragged lengths
# n need not be a multiple of 128: blocks stay aligned at token 0 and only the
# last block is short; the proxy rows are the last 128 tokens (straddling two
# blocks); sink and recency are the token ranges [0, 128) and [n-128, n).
RAGGED = [257, 300, 383, 700]


@pytest.mark.parametrize("n", RAGGED)
def test_ragged_proxy_matches_torch_softmax(n):
    q, k, _ = rand_qkv(2, 1, n, 40 + n)
    P = oracle.proxy_map(q, k)
    Q = bits_to_f64(q)[:, -B:, :]
    K = bits_to_f64(k).repeat_interleave(2, dim=0)
    S = torch.einsum("hrd,hjd->hrj", Q, K) / np.sqrt(128.0)
    i = torch.arange(n - B, n)[:, None]
    S = S.masked_fill(torch.arange(n)[None, :] > i, float("-inf"))
    assert np.max(np.abs(torch.softmax(S, dim=-1).numpy() - P)) < 1e-13
    assert np.allclose(P.sum(-1), 1.0, atol=1e-12)


@pytest.mark.parametrize("n", RAGGED)
def test_ragged_cstruct_and_mass_invariants(n):
    w = synth.small("ragged", 2, 1, n, 50 + n)
    q, k, _ = w.generate()
    P = oracle.proxy_map(q, k).astype(np.float32)
    S, T, _ = oracle.route(P)
    Qm = np.rint(P.astype(np.float64) * 2.0 ** 32).astype(np.uint64)
    assert S.tolist() == (Qm[:, :, :128].sum(axis=(1, 2)) + Qm[:, :, n - 128:].sum(axis=(1, 2))).tolist()
    vm, sm = oracle.vs_masses(P)
    nb = -(-n // B)
    assert vm.shape == (2, nb)
    # vertical masses: plain column sums over each block's own columns
    for c in range(nb):
        assert vm[:, c].tolist() == Qm[:, :, c * B:min(n, c * B + B)].sum(axis=(1, 2)).tolist()
    assert vm.sum(axis=1).tolist() == T.tolist()
    assert sm.sum(axis=1).tolist() == (T - vm[:, 0]).tolist()
    assert np.all(sm[:, -1] == 0)


@pytest.mark.parametrize("n,r,j", [(300, 0, 172), (300, 1, 44), (300, 127, 299), (300, 50, 128),
                                   (700, 3, 575), (700, 127, 130), (700, 0, 200), (383, 127, 382)])
def test_ragged_vs_masses_single_entry_closed_form(n, r, j):
    i = n - B + r
    assert j <= i
    nb = -(-n // B)
    P = np.zeros((1, B, n), np.float32)
    P[0, r, j] = 1.0
    vm, sm = oracle.vs_masses(P)
    want_v = np.zeros(nb, np.uint64)
    want_v[j // B] = 2 ** 32
    want_s = np.zeros(nb, np.uint64)
    if j >= 128:
        want_s[(i - j) // B] = 2 ** 32
    assert vm[0].tolist() == want_v.tolist()
    assert sm[0].tolist() == want_s.tolist()


@pytest.mark.parametrize("n", [300, 700])
def test_ragged_pe_map_uses_block_means_over_own_tokens(n):
    # Independent statement: numpy block means over each block's tokens (the
    # short last block over its t tokens), torch softmax over c <= b.
    hq, hkv = 2, 1
    q, k, _ = rand_qkv(hq, hkv, n, 60 + n)
    got = oracle.pe_map(q, k)
    nb = -(-n // B)
    Q, K = bits_to_f64(q).numpy(), bits_to_f64(k).numpy()
    qb = np.stack([Q[:, b * B:min(n, b * B + B)].mean(axis=1) for b in range(nb)], axis=1)
    kb = np.stack([K[:, b * B:min(n, b * B + B)].mean(axis=1) for b in range(nb)], axis=1)
    Z = torch.from_numpy(np.einsum("hbd,hcd->hbc", qb, np.repeat(kb, hq // hkv, axis=0)) / np.sqrt(128.0))
    Z = Z.masked_fill(torch.arange(nb)[None, :] > torch.arange(nb)[:, None], float("-inf"))
    assert np.max(np.abs(torch.softmax(Z, dim=-1).numpy() - got)) < 1e-13
    # a short last block scaled to 128 tokens would differ: the means are not diluted
    t = n - (nb - 1) * B
    assert t < B and np.allclose(kb[:, -1], K[:, (nb - 1) * B:].sum(axis=1) / t)


@pytest.mark.parametrize("n", [130, 300, 383])
def test_ragged_dense_attention_matches_sdpa(n):
    hq, hkv = 2, 1
    q, k, v = rand_qkv(hq, hkv, n, 70 + n)
    h, t = _all_tokens(hq, n)
    got = oracle.attention_rows(q, k, v, h, t).reshape(hq, n, 128)
    Q, K, V = bits_to_f64(q), bits_to_f64(k), bits_to_f64(v)
    ref = torch.nn.functional.scaled_dot_product_attention(
        Q[None], K.repeat_interleave(2, 0)[None], V.repeat_interleave(2, 0)[None], is_causal=True)[0].numpy()
    assert np.max(np.abs(ref - got)) < 1e-12


def test_ragged_selected_pairs_closed_form():
    # Every block of every row: n(n+1)/2 causal pairs per head; one row of
    # just the short diagonal block: t(t+1)/2.
    n, hq = 300, 2
    nb = 3
    rb = np.zeros((hq, nb, 1), np.uint32)
    for qb in range(nb):
        rb[:, qb, 0] = (1 << (qb + 1)) - 1
    assert oracle.selected_pairs(rb, n) == hq * n * (n + 1) // 2
    rb[:] = 0
    rb[0, 2, 0] = 1 << 2
    assert oracle.selected_pairs(rb, n) == 44 * 45 // 2
    rb[0, 2, 0] = 1 << 0
    assert oracle.selected_pairs(rb, n) == 44 * 128


# ----------------------------------------------------------------- row samplers
def test_proxy_rows_match_torch_softmax_rows():
    q, k, _ = rand_qkv(4, 2, 640, 22)
    heads = np.array([0, 1, 3, 3], np.int32)
    rows = np.array([0, 127, 5, 64], np.int32)
    got = oracle.proxy_rows(q, k, heads, rows)
    Q = bits_to_f64(q)
    K = bits_to_f64(k).repeat_interleave(2, dim=0)
    n = 640
    for t, (h, r) in enumerate(zip(heads, rows)):
        i = n - B + r
        s = (K[h, : i + 1] @ Q[h, i]) / np.sqrt(128.0)
        ref = np.zeros(n)
        ref[: i + 1] = torch.softmax(s, dim=0).numpy()
        assert np.max(np.abs(got[t] - ref)) < 1e-13


def test_pe_rows_match_torch():
    q, k, _ = rand_qkv(4, 2, 1024, 23)
    heads = np.array([0, 2, 3], np.int32)
    blocks = np.array([7, 0, 4], np.int32)
    got = oracle.pe_rows(q, k, heads, blocks)
    Qb = bits_to_f64(q).reshape(4, 8, B, 128).mean(dim=2)
    Kb = bits_to_f64(k).reshape(2, 8, B, 128).mean(dim=2).repeat_interleave(2, dim=0)
    for t, (h, b) in enumerate(zip(heads, blocks)):
        z = (Kb[h, : b + 1] @ Qb[h, b]) / np.sqrt(128.0)
        ref = np.zeros(8)
        ref[: b + 1] = torch.softmax(z, dim=0).numpy()
        assert np.max(np.abs(got[t] - ref)) < 1e-13


# --------------------------------------------------------------------------
# FlexPrefill comparators: divergence routing and cumulative coverage on
# Vertical-Slash heads (the two rules CRISP replaces).

def _bits(row, nb):
    return {c for c in range(nb) if (int(row[c >> 5]) >> (c & 31)) & 1}


def test_route_jsd_matches_scipy_jensenshannon():
    scipy_distance = pytest.importorskip("scipy.spatial.distance")
    rng = np.random.default_rng(81)
    hq, nb = 6, 40
    vm = rng.integers(1, 2**36, size=(hq, nb)).astype(np.uint64)
    vm[1, 5:] = 0  # zero-mass blocks (0 log 0 = 0)
    e = rng.random((hq, nb)) ** 3
    e[2, :20] = 0.0
    e = (e / e.sum(1, keepdims=True)).astype(np.float32)
    D, _ = oracle.route_jsd(vm, e, tau=0.1)
    for h in range(hq):
        a = vm[h].astype(np.float64) / vm[h].astype(np.float64).sum()
        # scipy renormalises e in double; ours takes the fp32 row as given
        ref = scipy_distance.jensenshannon(a, e[h].astype(np.float64)) ** 2
        assert D[h] == pytest.approx(ref, rel=1e-5, abs=1e-12)


def test_route_jsd_closed_forms_and_threshold_direction():
    nb = 4
    # identical distributions: D = 0 -> the pooled estimate is faithful -> PE
    vm = np.array([[1, 1, 2, 4]], np.uint64)
    e = np.array([[0.125, 0.125, 0.25, 0.5]], np.float32)
    D, r = oracle.route_jsd(vm, e, tau=0.1)
    assert D[0] == 0.0 and r[0] == 0
    # disjoint supports: D = ln 2 -> VS for any tau <= sqrt(ln 2)
    vm = np.array([[5, 0, 0, 0]], np.uint64)
    e = np.array([[0.0, 0.5, 0.5, 0.0]], np.float32)
    D, r = oracle.route_jsd(vm, e, tau=0.8)
    assert D[0] == pytest.approx(np.log(2.0), rel=1e-15) and r[0] == 1
    # a = (1, 0), e = (1/2, 1/2): m = (3/4, 1/4),
    # D = [ln(4/3) + (1/2) ln(2/3) + (1/2) ln 2] / 2
    vm = np.array([[7, 0]], np.uint64)
    e = np.array([[0.5, 0.5]], np.float32)
    D, _ = oracle.route_jsd(vm, e, tau=0.1)
    want = 0.5 * (np.log(4.0 / 3.0) + 0.5 * np.log(2.0 / 3.0) + 0.5 * np.log(2.0))
    assert D[0] == pytest.approx(want, rel=1e-14)
    # threshold is inclusive: sqrt(D) == tau routes to VS
    _, r = oracle.route_jsd(vm, e, tau=float(np.sqrt(want)))
    assert r[0] == 1
    _, r = oracle.route_jsd(vm, e, tau=float(np.nextafter(np.sqrt(want), 1.0)))
    assert r[0] == 0
    del nb


def test_select_vs_gamma_sink_only_collapse():
    # The pages' failure mode: a sink block holding >= gamma of the vertical
    # mass ends the coverage inside the sink; only the always-retained blocks
    # and the k_min fill remain, however strong the other columns are.
    nb = 64
    vm = np.full((1, nb), 10, np.uint64)
    vm[0, 0] = 10**9          # sink block
    vm[0, [17, 33, 41]] = 10**6  # strong needles, far below the sink
    sm = np.full((1, nb), 3, np.uint64)
    vb, _ = oracle.select_vs_gamma(vm, sm, np.array([1], np.uint8), gamma=(95, 100), kmin=0)
    assert _bits(vb[0], nb) == {0, nb - 1}
    vb, _ = oracle.select_vs_gamma(vm, sm, np.array([1], np.uint8), gamma=(95, 100), kmin=5)
    assert _bits(vb[0], nb) == {0, nb - 1, 17, 33, 41}
    # the noise floor keeps the needles without any k_min help
    vb, _ = oracle.select_vs(vm, sm, np.array([1], np.uint8), alpha=(1, 1), kmin=0)
    assert {17, 33, 41} <= _bits(vb[0], nb)


def test_select_vs_gamma_one_keeps_all_nonzero_and_zero_keeps_forced():
    rng = np.random.default_rng(82)
    nb = 50
    vm = rng.integers(0, 1000, size=(2, nb)).astype(np.uint64)
    vm[:, ::7] = 0
    sm = rng.integers(0, 1000, size=(2, nb)).astype(np.uint64)
    route = np.array([1, 1], np.uint8)
    vb, sb = oracle.select_vs_gamma(vm, sm, route, gamma=(1, 1), kmin=0)
    for h in range(2):
        assert _bits(vb[h], nb) == set(np.nonzero(vm[h])[0].tolist()) | {0, nb - 1}
        assert _bits(sb[h], nb) == set(np.nonzero(sm[h])[0].tolist()) | {0}
    vb, sb = oracle.select_vs_gamma(vm, sm, route, gamma=(0, 1), kmin=0)
    assert _bits(vb[0], nb) == {0, nb - 1} and _bits(sb[0], nb) == {0}


def test_select_vs_gamma_prefix_properties():
    # Characterisation of the coverage prefix (kmin = 0, forced blocks given
    # the smallest masses so that they stay outside it): the chosen non-forced
    # blocks outrank every other block, cover gamma of the total, and stop
    # covering it once their lowest-ranked member is dropped.
    rng = np.random.default_rng(83)
    nb = 96
    for trial in range(20):
        g = (int(rng.integers(1, 100)), 100)
        m = rng.integers(10, 10**6, size=nb).astype(np.uint64)
        m[rng.integers(0, nb, 5)] = m[rng.integers(0, nb, 5)]  # some ties
        m[0], m[nb - 1] = 0, 0
        vb, _ = oracle.select_vs_gamma(m[None], m[None], np.array([1], np.uint8), gamma=g, kmin=0)
        chosen = _bits(vb[0], nb) - {0, nb - 1}
        key = lambda c: (int(m[c]), -c)
        rest = set(range(1, nb - 1)) - chosen
        assert chosen and all(key(a) > key(b) for a in chosen for b in rest)
        T = int(m.sum())
        mass = sum(int(m[c]) for c in chosen)
        assert g[1] * mass >= g[0] * T
        last = min(chosen, key=key)
        assert g[1] * (mass - int(m[last])) < g[0] * T


def test_select_vs_gamma_route_pe_gives_empty():
    vm = np.ones((2, 8), np.uint64)
    vb, sb = oracle.select_vs_gamma(vm, vm, np.array([0, 1], np.uint8), gamma=(95, 100), kmin=8)
    assert not vb[0].any() and not sb[0].any() and vb[1].any()
