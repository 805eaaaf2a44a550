"""The C ABI library loads without a GPU, exports every declared symbol and
rejects bad arguments on the host (no kernel launch, no GPU needed)."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

import dynamic_sparse_prefill_crisp_gb300 as crisp
from dynamic_sparse_prefill_crisp_gb300 import build as crisp_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    crisp_build.build()
    return crisp.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "crisp.h")).read()
    return sorted(set(re.findall(r"CRISP_API\s+[\w\s\*]*?\b(crisp_\w+)\s*\(", text)))


def test_header_declares_the_steps():
    names = declared_functions()
    for want in ("crisp_proxy_map", "crisp_route_cstruct", "crisp_select_vs", "crisp_select_pe",
                 "crisp_sparse_prefill", "crisp_dense_prefill", "crisp_block_masses", "crisp_pe_pool",
                 "crisp_build_mask", "crisp_prefill_layer", "crisp_proxy_masses", "crisp_read_status",
                 "crisp_status_string", "crisp_route_cstruct_masses", "crisp_select_vs_masses",
                 "crisp_sparse_prefill_mask", "crisp_workspace_size", "crisp_params_default"):
        assert want in names


# The survey's boundary table, call by call: each row's name and its argument
# list as this header declares it (the survey's signature plus ws_bytes
# after every workspace; the workspace size takes the shape only).
SURVEY_BOUNDARY = {
    "crisp_proxy_map": ["shape", "q", "k", "pmap", "ws", "ws_bytes", "stream"],
    "crisp_route_cstruct": ["shape", "params", "pmap", "cstruct", "total", "route", "ws", "ws_bytes", "stream"],
    "crisp_select_vs": ["shape", "params", "pmap", "route", "vmass", "smass", "vbits", "sbits", "ws", "ws_bytes",
                        "stream"],
    "crisp_pe_pool": ["shape", "q", "k", "route", "pbar", "ws", "ws_bytes", "stream"],
    "crisp_select_pe": ["shape", "params", "pbar", "route", "pebits", "ws", "ws_bytes", "stream"],
    "crisp_sparse_prefill": ["shape", "q", "k", "v", "route", "vbits", "sbits", "pebits", "out", "ws", "ws_bytes",
                             "stream"],
    "crisp_dense_prefill": ["shape", "q", "k", "v", "out", "ws", "ws_bytes", "stream"],
    "crisp_prefill_layer": ["shape", "params", "q", "k", "v", "out", "ws", "ws_bytes", "stream"],
    "crisp_read_status": ["ws", "stream", "status"],
    "crisp_status_string": ["status"],
    "crisp_params_default": ["p"],
    "crisp_workspace_size": ["shape", "bytes"],
}


def declared_arguments(name):
    text = open(os.path.join(ROOT, "include", "crisp.h")).read()
    m = re.search(r"CRISP_API[\w\s\*]*?\b" + name + r"\s*\(([^)]*)\)", text)
    assert m, name
    args = []
    for a in m.group(1).split(","):
        a = re.sub(r"/\*.*?\*/", "", a).strip()
        args.append(re.findall(r"\w+", a)[-1])
    return args


@pytest.mark.parametrize("name", sorted(SURVEY_BOUNDARY))
def test_survey_boundary_calls_are_declared(name):
    assert declared_arguments(name) == SURVEY_BOUNDARY[name]


def test_survey_boundary_fields_and_codes():
    text = open(os.path.join(ROOT, "include", "crisp.h")).read()
    for field in ("tau_num", "tau_den", "alpha_num", "alpha_den", "gamma_num", "gamma_den", "kmin_blocks",
                  "sink_tokens", "recency_tokens", "pe_mode"):
        assert re.search(r"\b" + field + r"\b", text), field
    for code in ("CRISP_OK", "CRISP_ERR_INVALID_ARG", "CRISP_ERR_SHAPE", "CRISP_ERR_ALIGN", "CRISP_ERR_WORKSPACE",
                 "CRISP_ERR_CUDA", "CRISP_ERR_TIMEOUT", "CRISP_ERR_BOUNDS"):
        assert re.search(r"\b" + code + r"\s*=", text), code


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", crisp.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (crisp_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert getattr(L, n) is not None


def test_checking_build_exports_every_declared_symbol():
    # The bounds-checking build (-DCRISP_DEBUG) compiles and keeps the ABI.
    path = crisp_build.build(debug=True)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (crisp_\w+)", out))
    assert not [n for n in declared_functions() if n not in exported]
    assert crisp.load_library(path).crisp_status_string(8) == b"device index outside its buffer (bounds-checking build)"


def test_crisp_log_reports_calls_and_statuses(L):
    # CRISP_LOG=1: every entry point writes its name, shape and returned
    # status to stderr (here argument errors, no device needed).
    code = ("import ctypes, dynamic_sparse_prefill_crisp_gb300 as c; L = c.lib(); s = c.make_shape(8, 4, 1024); "
            "s.head_dim = 64; n = ctypes.c_size_t(); L.crisp_workspace_size(ctypes.byref(s), ctypes.byref(n)); "
            "L.crisp_read_status(None, None, None)")
    env = dict(os.environ, CRISP_LOG="1", PYTHONPATH=ROOT)
    err = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT).stderr
    assert "[crisp] crisp_workspace_size hq=8 hkv=4 n=1024 -> 2 (unsupported shape)" in err, err
    assert "[crisp] crisp_read_status -> 1 (invalid argument)" in err, err
    env.pop("CRISP_LOG")
    err = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, cwd=ROOT).stderr
    assert "[crisp]" not in err


def test_params_default_is_the_universal_configuration(L):
    p = crisp.params_default()
    assert (p.tau_num, p.tau_den) == (1, 5)
    assert (p.alpha_num, p.alpha_den) == (1, 1)
    assert (p.gamma_num, p.gamma_den) == (19, 20)
    assert p.kmin_blocks == 8 and p.pe_mode == crisp.PE_GAMMA
    # CRISP's own rules by default; the comparators' settings as we read FlexPrefill's
    assert p.route_mode == crisp.ROUTE_CSTRUCT and p.vs_mode == crisp.VS_NOISE
    assert (p.vs_gamma_num, p.vs_gamma_den) == (95, 100) and abs(p.jsd_tau - 0.1) < 1e-7
    assert p.dense_below == 0
    assert p.sink_tokens == 128 and p.recency_tokens == 128


def test_status_strings(L):
    for code in range(9):
        assert crisp.status_string(code)
    assert crisp.status_string(99) == "unknown status"


def test_workspace_sizes(L):
    s = crisp.make_shape(32, 8, 524288)
    small = crisp.workspace_size(s)
    layer = crisp.layer_workspace_size(s)
    assert 0 < small < layer
    # the layer workspace holds the fp32 pooled map (nb x nb per head) but not
    # the proxy map of the last block, which the fused mass pass never stores
    nb = 524288 // 128
    assert 4 * 32 * nb * nb < layer < 4 * 32 * 128 * 524288


@pytest.mark.parametrize("field,value,code", [
    ("hq", 6, 2), ("hkv", 0, 2), ("head_dim", 64, 2), ("block", 64, 2), ("seq_len", -1, 2),
    ("seq_len", (1 << 20) + 128, 2), ("q_tok_stride", 100, 3), ("kv_head_stride", 0, 3),
    ("scale", float("nan"), 1), ("scale", -1.0, 1)])
def test_shape_validation(L, field, value, code):
    s = crisp.make_shape(8, 4, 1024)
    setattr(s, field, value)
    n = ctypes.c_size_t()
    assert L.crisp_workspace_size(ctypes.byref(s), ctypes.byref(n)) == code
    # a step rejects the shape before touching any pointer or the device
    rc = L.crisp_proxy_map(ctypes.byref(s), ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                           ctypes.c_void_p(256), 1 << 30, None)
    assert rc == code


@pytest.mark.parametrize("field,value", [("tau_den", 0), ("tau_num", 6), ("alpha_den", 0), ("alpha_num", 70000),
                                         ("gamma_num", 21), ("kmin_blocks", -1), ("kmin_blocks", 9000),
                                         ("pe_mode", 2), ("route_mode", 2), ("vs_mode", -1), ("vs_gamma_den", 0),
                                         ("vs_gamma_num", 101), ("jsd_tau", -0.1), ("jsd_tau", 1.5),
                                         ("jsd_tau", float("nan")), ("dense_below", -1), ("sink_tokens", -1),
                                         ("recency_tokens", (1 << 20) + 1)])
def test_params_validation(L, field, value):
    s = crisp.make_shape(8, 4, 1024)
    p = crisp.params_default()
    setattr(p, field, value)
    vp = ctypes.c_void_p
    rc = L.crisp_route_cstruct(ctypes.byref(s), ctypes.byref(p), vp(256), vp(256), vp(256), vp(256), vp(256),
                               1 << 30, None)
    assert rc == 1


@pytest.mark.parametrize("sink,recency", [(64, 128), (128, 200), (0, 0)])
def test_mass_routing_needs_block_wide_slices(L, sink, recency):
    # Routing from block masses (and the layer, which does so) reads the sink
    # slice as block 0 and the recency slice as the recency mass: other widths
    # are refused on the host; the map-reading route accepts them.
    s = crisp.make_shape(8, 4, 1024)
    p = crisp.params_default(sink_tokens=sink, recency_tokens=recency)
    vp = ctypes.c_void_p
    assert L.crisp_route_cstruct_masses(ctypes.byref(s), ctypes.byref(p), vp(256), vp(256), vp(256), vp(256),
                                        vp(256), vp(256), 1 << 30, None) == 1
    assert L.crisp_prefill_layer(ctypes.byref(s), ctypes.byref(p), vp(16), vp(16), vp(16), vp(16), vp(256), 1 << 30,
                                 None) == 1
    assert L.crisp_prefill_layer_host(vp(256), ctypes.byref(s), ctypes.byref(p), *([vp(256)] * 9), 1 << 30,
                                      None) == 1
    # past the parameter check, the map-reading route stops at its first null pointer
    assert L.crisp_route_cstruct(ctypes.byref(s), ctypes.byref(p), None, vp(256), vp(256), vp(256), vp(256),
                                 1 << 30, None) == 1


def test_null_and_misaligned_pointers(L):
    s = crisp.make_shape(8, 4, 1024)
    vp = ctypes.c_void_p
    assert L.crisp_proxy_map(ctypes.byref(s), None, vp(16), vp(16), vp(256), 1 << 30, None) == 1
    assert L.crisp_proxy_map(ctypes.byref(s), vp(8), vp(16), vp(16), vp(256), 1 << 30, None) == 3
    assert L.crisp_sparse_prefill_mask(ctypes.byref(s), vp(16), vp(16), vp(16), None, vp(16), vp(16), vp(256),
                                       1 << 30, None) == 1
    assert L.crisp_sparse_prefill_mask(ctypes.byref(s), vp(16), vp(16), vp(16), vp(16), vp(18), vp(16), vp(256),
                                       1 << 30, None) == 3
    # the index-set form: route, vbits, sbits, pebits checked before any launch
    assert L.crisp_sparse_prefill(ctypes.byref(s), vp(16), vp(16), vp(16), None, vp(16), vp(16), vp(16), vp(16),
                                  vp(256), 1 << 30, None) == 1
    assert L.crisp_sparse_prefill(ctypes.byref(s), vp(16), vp(16), vp(16), vp(16), vp(18), vp(16), vp(16), vp(16),
                                  vp(256), 1 << 30, None) == 3
    assert L.crisp_sparse_prefill(ctypes.byref(s), vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), vp(16),
                                  vp(256), 64, None) == 4
    assert L.crisp_sparse_prefill(ctypes.byref(s), None, vp(16), vp(16), vp(16), vp(16), vp(16), vp(16), vp(16),
                                  vp(256), 1 << 30, None) == 1
    # A4 from the map
    pd0 = ctypes.byref(crisp.params_default())
    assert L.crisp_select_vs(ctypes.byref(s), pd0, None, vp(16), vp(16), vp(16), vp(16), vp(16), vp(256), 1 << 30,
                             None) == 1
    assert L.crisp_select_vs(ctypes.byref(s), pd0, vp(16), vp(16), vp(20), vp(16), vp(16), vp(16), vp(256), 1 << 30,
                             None) == 3
    assert L.crisp_select_vs_masses(ctypes.byref(s), pd0, vp(16), vp(16), None, vp(16), vp(16), vp(256), 1 << 30,
                                    None) == 1
    assert L.crisp_proxy_masses(ctypes.byref(s), vp(16), vp(16), None, vp(16), vp(16), vp(256), 1 << 30, None) == 1
    assert L.crisp_proxy_masses(ctypes.byref(s), vp(16), vp(16), vp(16), vp(16), None, vp(256), 1 << 30, None) == 1
    assert L.crisp_proxy_masses(ctypes.byref(s), vp(16), vp(16), vp(16), vp(20), vp(16), vp(256), 1 << 30,
                                None) == 3
    assert L.crisp_proxy_masses(ctypes.byref(s), vp(16), vp(16), vp(16), vp(16), vp(20), vp(256), 1 << 30,
                                None) == 3
    assert L.crisp_proxy_masses(ctypes.byref(s), vp(16), vp(16), vp(16), vp(16), vp(16), vp(256), 64, None) == 4
    assert L.crisp_block_masses(ctypes.byref(s), vp(16), vp(16), vp(16), None, vp(256), 1 << 30, None) == 1
    pd = ctypes.byref(crisp.params_default())
    assert L.crisp_route_cstruct_masses(ctypes.byref(s), pd, vp(256), None, vp(256), vp(256), vp(256), vp(256),
                                        1 << 30, None) == 1
    assert L.crisp_route_cstruct_masses(ctypes.byref(s), pd, vp(256), vp(260), vp(256), vp(256), vp(256), vp(256),
                                        1 << 30, None) == 3
    assert L.crisp_route_cstruct_masses(ctypes.byref(s), pd, vp(256), vp(256), vp(256), vp(256), vp(256), None,
                                        1 << 30, None) == 4
    assert L.crisp_route_cstruct(ctypes.byref(s), pd, vp(256), None, vp(256), vp(256), vp(256), 1 << 30, None) == 1
    assert L.crisp_route_cstruct(ctypes.byref(s), pd, vp(260), vp(256), vp(256), vp(256), vp(256), 1 << 30,
                                 None) == 3
    assert L.crisp_route_cstruct(ctypes.byref(s), pd, vp(256), vp(256), vp(256), vp(256), vp(256), 64, None) == 4
    # divergence routing and fused masses: argument errors before any CUDA call
    assert L.crisp_route_jsd(ctypes.byref(s), pd, None, vp(256), None, vp(256), vp(256), 1 << 30, None) == 1
    assert L.crisp_route_jsd(ctypes.byref(s), pd, vp(260), vp(256), None, vp(256), vp(256), 1 << 30, None) == 3
    assert L.crisp_route_jsd(ctypes.byref(s), pd, vp(256), vp(256), vp(260), vp(256), vp(256), 1 << 30, None) == 3
    bad = crisp.params_default(route_mode=7)
    assert L.crisp_route_jsd(ctypes.byref(s), ctypes.byref(bad), vp(256), vp(256), None, vp(256), vp(256), 1 << 30,
                             None) == 1
    # the allocation-free map's status reader needs a destination
    assert L.crisp_noalloc_read_status(None, None) == 1
    # failure-detection self-test: argument errors before any CUDA call
    assert L.crisp_wait_selftest(None, 1 << 20, 1000000, None) == 4
    assert L.crisp_wait_selftest(vp(256), 1 << 20, 0, None) == 1
    assert L.crisp_wait_selftest(vp(256), 1 << 20, 20 * 10**9, None) == 1
    # host-buffer path: argument errors before any CUDA call
    assert L.crisp_host_pipeline_create(None) == 1
    assert L.crisp_host_pipeline_destroy(None) == 0
    assert L.crisp_prefill_layer_host(None, ctypes.byref(s), ctypes.byref(crisp.params_default()),
                                      *([vp(256)] * 9), 1 << 30, None) == 1
    # workspace missing / misaligned / too small
    assert L.crisp_proxy_map(ctypes.byref(s), vp(16), vp(16), vp(16), None, 1 << 30, None) == 4
    assert L.crisp_proxy_map(ctypes.byref(s), vp(16), vp(16), vp(16), vp(272), 1 << 30, None) == 3
    assert L.crisp_proxy_map(ctypes.byref(s), vp(16), vp(16), vp(16), vp(256), 64, None) == 4
    assert L.crisp_prefill_layer(ctypes.byref(s), ctypes.byref(crisp.params_default()), vp(16), vp(16), vp(16),
                                 vp(16), vp(256), 1024, None) == 4


@pytest.mark.parametrize("n", [300, 1000, 2049, 524287])
def test_ragged_lengths_are_accepted(L, n):
    # 128 need not divide n: every step passes the shape check (and then
    # stops at its first pointer check, before any CUDA call)
    s = crisp.make_shape(8, 4, n)
    size = ctypes.c_size_t()
    assert L.crisp_workspace_size(ctypes.byref(s), ctypes.byref(size)) == 0
    nb = -(-n // 128)
    assert size.value >= 8 * nb * 8  # per-tile mass scratch of every head
    assert L.crisp_proxy_map(ctypes.byref(s), None, ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(256),
                             1 << 30, None) == 1
    assert L.crisp_proxy_masses(ctypes.byref(s), ctypes.c_void_p(16), ctypes.c_void_p(16), None, ctypes.c_void_p(16),
                                ctypes.c_void_p(16), ctypes.c_void_p(256), 1 << 30, None) == 1


@pytest.mark.parametrize("n", [0, 1, 100, 128, 255])
def test_short_and_empty_lengths(L, n):
    # The method's steps need two blocks; attention and the layer take any n,
    # and an empty input (n = 0) returns OK without launching anything.
    s = crisp.make_shape(8, 4, n)
    size = ctypes.c_size_t()
    assert L.crisp_workspace_size(ctypes.byref(s), ctypes.byref(size)) == 0
    assert L.crisp_layer_workspace_size(ctypes.byref(s), ctypes.byref(size)) == 0
    vp = ctypes.c_void_p
    assert L.crisp_proxy_map(ctypes.byref(s), vp(16), vp(16), vp(16), vp(256), 1 << 30, None) == 2
    assert L.crisp_proxy_masses(ctypes.byref(s), vp(16), vp(16), vp(16), vp(16), vp(16), vp(256), 1 << 30, None) == 2
    p = ctypes.byref(crisp.params_default())
    if n == 0:
        # nothing to compute: OK with null buffers and no device
        assert L.crisp_prefill_layer(ctypes.byref(s), p, None, None, None, None, None, 0, None) == 0
        assert L.crisp_dense_prefill(ctypes.byref(s), None, None, None, None, None, 0, None) == 0
        assert L.crisp_sparse_prefill_mask(ctypes.byref(s), None, None, None, None, None, None, None, 0, None) == 0
        # the index-set form needs the method's steps (n >= 256)
        assert L.crisp_sparse_prefill(ctypes.byref(s), *([None] * 9), 0, None) == 2
        assert L.crisp_prefill_layer_host(vp(256), ctypes.byref(s), p, *([None] * 9), 0, None) == 0
    else:
        # past the shape check: the first pointer check answers
        assert L.crisp_dense_prefill(ctypes.byref(s), None, vp(16), vp(16), vp(16), vp(256), 1 << 30, None) == 1
        assert L.crisp_prefill_layer(ctypes.byref(s), p, None, vp(16), vp(16), vp(16), vp(256), 1 << 30, None) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(crisp, "_lib", None)
    monkeypatch.setattr(crisp, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="missing"):
        crisp.lib()


def test_readme_names_exist_in_the_binding():
    # Every crisp.<name> the README shows is part of the binding.
    import re
    text = open(os.path.join(os.path.dirname(__file__), "..", "README.md")).read()
    names = set(re.findall(r"crisp\.([a-z_A-Z]+)\(", text))
    assert names, "README shows no calls"
    missing = sorted(n for n in names if not hasattr(crisp, n))
    assert not missing, missing
