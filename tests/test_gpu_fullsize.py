"""Full-size parity: the five workloads at their stated sizes, through the
same step entry points and launch configuration the benchmark times.

Index sets (masses, C_struct, routes, V/S/PE bitsets, row masks, counts,
schedule) are compared IN FULL, bit-exactly, with the oracle run on the GPU's
own fp32 maps. The proxy map, the pooled map and the attention output are
compared on seeded samples of rows the oracle computes one by one: per head
the proxy rows {0, 63, 127} plus 5 random rows; pooled rows {0, 1, nb-1} plus
5 random (PE heads); attention rows {0, 127, 128, n-129, n-128, n-1} plus 64
uniform ones (seed 0xC815 + workload index). Tolerances as in the parity
tests.
"""
import numpy as np
import pytest
import torch

import dynamic_sparse_prefill_crisp_gb300 as crisp
import oracle
import synth
from gpu_helpers import assert_status_ok, empty, new_workspace, run_steps, to_dev
from test_gpu_parity import ATT_MAX, ATT_MEAN, check_index_sets, check_map, sample_rows

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
B = 128


def _proxy_samples(hq, seed):
    rng = np.random.default_rng(seed)
    heads, rows = [], []
    for h in range(hq):
        rr = sorted(set([0, 63, 127] + rng.integers(0, B, 5).tolist()))
        heads += [h] * len(rr)
        rows += rr
    return np.array(heads, np.int32), np.array(rows, np.int32)


def _pe_samples(route, nb, seed):
    rng = np.random.default_rng(seed)
    heads, blocks = [], []
    for h in np.nonzero(route == 0)[0]:
        bb = sorted(set([0, 1, nb - 1] + rng.integers(0, nb, 5).tolist()))
        heads += [int(h)] * len(bb)
        blocks += bb
    return np.array(heads, np.int32), np.array(blocks, np.int32)


def _check_layer(w, index, params=None):
    params = params or crisp.params_default()
    q, k, v = w.generate()
    r = run_steps(q, k, v, params)
    seed = 0xC815 + index
    ph, pr = _proxy_samples(w.hq, seed)
    check_map(r["pmap"][ph, pr], oracle.proxy_rows(q, k, ph, pr))
    rb, route = check_index_sets(r, params)
    nb = crisp.num_blocks(w.n)
    if (route == 0).any():
        eh, eb = _pe_samples(route, nb, seed)
        check_map(r["pbar"][eh, eb], oracle.pe_rows(q, k, eh, eb))
    h, t = sample_rows(w.hq, w.n, 64, seed)
    ref = oracle.attention_rows(q, k, v, h, t, rowbits=rb)
    got = r["out"].float().cpu().numpy()[h, t]
    err = np.abs(got.astype(np.float64) - ref)
    assert err.max() <= ATT_MAX and err.mean() <= ATT_MEAN, (err.max(), err.mean())
    return route


def test_llama8b_32k():
    route = _check_layer(synth.WORKLOADS["llama8b-32k"], 2)
    assert route.tolist() == [1 - (h % 2) for h in range(32)]  # even heads sink-type, odd diffuse


def test_qwen7b_128k():
    route = _check_layer(synth.WORKLOADS["qwen7b-128k"], 3)
    assert route.tolist() == [1 - (h % 2) for h in range(28)]


@pytest.mark.parametrize("layer", [0, 1, 2, 3])
def test_llama8b_256k_stack_layer(layer):
    w = synth.WORKLOADS["llama8b-256k-stack"].layer(layer)
    route = _check_layer(w, 4 * 16 + layer)
    want = np.zeros(w.hq, np.uint8)
    want[w.vs_heads] = 1
    assert np.array_equal(route, want)


def test_llama8b_512k():
    route = _check_layer(synth.WORKLOADS["llama8b-512k"], 5)
    assert route.all()


def test_max_length_one_million_tokens():
    # The largest supported sequence, 2^20 tokens (8192 blocks; bitset rows
    # of 256 words), on 4 q / 1 kv heads so that the fp64 checks stay quick.
    w = synth.small("max-1m", 4, 1, 1 << 20, 77, d_sink=12.0)  # sink strong enough to dominate 1M keys
    route = _check_layer(w, 77)
    assert route.tolist() == [1, 0, 1, 0]


def test_ragged_long_sequence():
    # 128k + 77 tokens: a short last block of 77 keys, the proxy rows spread
    # over blocks 1024 and 1025, recency columns in two proxy CTAs' tiles.
    w = synth.small("ragged-128k", 8, 2, 131072 + 77, 78, d_sink=8.0)  # sink strong enough for 128k keys
    route = _check_layer(w, 78)
    assert route.any() and not route.all()  # both routes


def test_llama8b_512k_dense_sampled_rows():
    w = synth.WORKLOADS["llama8b-512k"]
    q, k, v = w.generate()
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    out = empty((w.hq, w.n, 128), torch.bfloat16)
    s = crisp.make_shape(w.hq, w.hkv, w.n, qd, kd, out)
    ws = new_workspace(s)
    crisp.dense_prefill(s, qd, kd, vd, out, ws)
    torch.cuda.synchronize()
    assert_status_ok(ws)
    rng = np.random.default_rng(0xC815 + 55)
    heads = np.repeat(np.arange(w.hq), 6).astype(np.int32)
    toks = np.concatenate([[0, 128, w.n - 1] + rng.integers(0, w.n, 3).tolist() for _ in range(w.hq)]).astype(np.int32)
    ref = oracle.attention_rows(q, k, v, heads, toks)
    got = out.float().cpu().numpy()[heads, toks]
    err = np.abs(got.astype(np.float64) - ref)
    assert err.max() <= ATT_MAX and err.mean() <= ATT_MEAN, (err.max(), err.mean())
