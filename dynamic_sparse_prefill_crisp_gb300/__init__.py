"""Python binding of the CRISP sparse-prefill C ABI (``include/crisp.h``).

Argument marshalling only: every step runs in the CUDA kernels of
``libcrisp.so``. Tensors are passed by ``data_ptr()``; PyTorch provides the
device memory and the stream. Each wrapper raises :class:`CrispError` when the
library returns a non-OK status. Importing succeeds without a GPU; calling a
step without the built library raises immediately (there is no fallback).
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcrisp.so")
_lib = None

B = 128
D = 128


def num_blocks(n: int) -> int:
    """Blocks of an n-token layer: ceil(n / 128), the last one short when 128 does not divide n."""
    return (n + B - 1) // B


def map_ld(n: int) -> int:
    """Row stride (floats) of the proxy map: 128 * num_blocks(n)."""
    return num_blocks(n) * B

STATUS_NAMES = {0: "CRISP_OK", 1: "CRISP_ERR_INVALID_ARG", 2: "CRISP_ERR_SHAPE", 3: "CRISP_ERR_ALIGN",
                4: "CRISP_ERR_WORKSPACE", 5: "CRISP_ERR_CUDA", 6: "CRISP_ERR_TIMEOUT", 7: "CRISP_ERR_DEVICE",
                8: "CRISP_ERR_BOUNDS"}
PE_GAMMA, PE_NOISE = 0, 1
ROUTE_CSTRUCT, ROUTE_JSD = 0, 1
VS_NOISE, VS_GAMMA = 0, 1


class CrispError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({status_string(status)})")


class Shape(ctypes.Structure):
    _fields_ = [("hq", ctypes.c_int32), ("hkv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("seq_len", ctypes.c_int32), ("block", ctypes.c_int32),
                ("q_head_stride", ctypes.c_int64), ("q_tok_stride", ctypes.c_int64),
                ("kv_head_stride", ctypes.c_int64), ("kv_tok_stride", ctypes.c_int64),
                ("o_head_stride", ctypes.c_int64), ("o_tok_stride", ctypes.c_int64),
                ("scale", ctypes.c_float)]


class Params(ctypes.Structure):
    _fields_ = [("tau_num", ctypes.c_uint32), ("tau_den", ctypes.c_uint32),
                ("alpha_num", ctypes.c_uint32), ("alpha_den", ctypes.c_uint32),
                ("gamma_num", ctypes.c_uint32), ("gamma_den", ctypes.c_uint32),
                ("kmin_blocks", ctypes.c_int32), ("pe_mode", ctypes.c_int32),
                ("route_mode", ctypes.c_int32), ("vs_mode", ctypes.c_int32),
                ("vs_gamma_num", ctypes.c_uint32), ("vs_gamma_den", ctypes.c_uint32),
                ("jsd_tau", ctypes.c_float), ("dense_below", ctypes.c_int32),
                ("sink_tokens", ctypes.c_int32), ("recency_tokens", ctypes.c_int32)]


class LayerViews(ctypes.Structure):
    _fields_ = [(name, ctypes.c_void_p) for name in
                ("vmass", "smass", "rmass", "cstruct", "total", "route", "vbits", "sbits", "pbar", "pebits",
                 "rowbits", "counts", "order")]


def lib():
    """The loaded libcrisp.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with dynamic_sparse_prefill_crisp_gb300.build.build()")
        _lib = load_library(LIB_PATH)
    return _lib


def load_library(path):
    """Loads a build of the library (e.g. the bounds-checking one) with the
    argument types declared; the module's calls keep using lib()."""
    L = ctypes.CDLL(path)
    vp, sz, st = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p
    P = ctypes.POINTER
    L.crisp_params_default.argtypes = [P(Params)]
    L.crisp_params_default.restype = None
    L.crisp_workspace_size.argtypes = [P(Shape), P(sz)]
    L.crisp_layer_workspace_size.argtypes = [P(Shape), P(sz)]
    L.crisp_workspace_init.argtypes = [vp, sz, st]
    L.crisp_proxy_map.argtypes = [P(Shape), vp, vp, vp, vp, sz, st]
    L.crisp_proxy_map_noalloc.argtypes = [P(Shape), vp, vp, vp, st]
    L.crisp_noalloc_read_status.argtypes = [st, P(ctypes.c_int)]
    L.crisp_block_masses.argtypes = [P(Shape), vp, vp, vp, vp, vp, sz, st]
    L.crisp_proxy_masses.argtypes = [P(Shape), vp, vp, vp, vp, vp, vp, sz, st]
    L.crisp_host_pipeline_create.argtypes = [P(vp)]
    L.crisp_host_pipeline_destroy.argtypes = [vp]
    L.crisp_prefill_layer_host.argtypes = [vp, P(Shape), P(Params)] + [vp] * 9 + [sz, st]
    L.crisp_route_cstruct.argtypes = [P(Shape), P(Params), vp, vp, vp, vp, vp, sz, st]
    L.crisp_route_cstruct_masses.argtypes = [P(Shape), P(Params), vp, vp, vp, vp, vp, vp, sz, st]
    L.crisp_route_jsd.argtypes = [P(Shape), P(Params), vp, vp, vp, vp, vp, sz, st]
    L.crisp_wait_selftest.argtypes = [vp, sz, ctypes.c_int64, st]
    L.crisp_select_vs.argtypes = [P(Shape), P(Params), vp, vp, vp, vp, vp, vp, vp, sz, st]
    L.crisp_select_vs_masses.argtypes = [P(Shape), P(Params), vp, vp, vp, vp, vp, vp, sz, st]
    L.crisp_pe_pool.argtypes = [P(Shape), vp, vp, vp, vp, vp, sz, st]
    L.crisp_select_pe.argtypes = [P(Shape), P(Params), vp, vp, vp, vp, sz, st]
    L.crisp_build_mask.argtypes = [P(Shape), vp, vp, vp, vp, vp, vp, vp, vp, sz, st]
    L.crisp_sparse_prefill.argtypes = [P(Shape), vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, st]
    L.crisp_sparse_prefill_mask.argtypes = [P(Shape), vp, vp, vp, vp, vp, vp, vp, sz, st]
    L.crisp_dense_prefill.argtypes = [P(Shape), vp, vp, vp, vp, vp, sz, st]
    L.crisp_layer_views_get.argtypes = [P(Shape), vp, P(LayerViews)]
    L.crisp_prefill_layer.argtypes = [P(Shape), P(Params), vp, vp, vp, vp, vp, sz, st]
    L.crisp_read_status.argtypes = [vp, st, P(ctypes.c_int)]
    L.crisp_status_string.argtypes = [ctypes.c_int]
    L.crisp_status_string.restype = ctypes.c_char_p
    for name in ("crisp_workspace_size", "crisp_layer_workspace_size", "crisp_workspace_init", "crisp_proxy_map",
                 "crisp_proxy_map_noalloc", "crisp_noalloc_read_status", "crisp_block_masses",
                 "crisp_proxy_masses", "crisp_route_cstruct", "crisp_route_cstruct_masses", "crisp_route_jsd",
                 "crisp_select_vs", "crisp_select_vs_masses", "crisp_pe_pool", "crisp_select_pe",
                 "crisp_build_mask", "crisp_sparse_prefill", "crisp_sparse_prefill_mask", "crisp_dense_prefill",
                 "crisp_layer_views_get", "crisp_prefill_layer", "crisp_read_status",
                 "crisp_host_pipeline_create", "crisp_host_pipeline_destroy", "crisp_prefill_layer_host",
                 "crisp_wait_selftest"):
        getattr(L, name).restype = ctypes.c_int
    return L


def status_string(status: int) -> str:
    return lib().crisp_status_string(int(status)).decode()


def _check(rc: int, what: str):
    if rc != 0:
        raise CrispError(rc, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr() if hasattr(t, "data_ptr") else int(t))


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _nbytes(t):
    return t.numel() * t.element_size()


def make_shape(hq, hkv, n, q=None, k=None, out=None, scale=0.0) -> Shape:
    """Shape for [heads][tokens][128] tensors; strides are taken from the
    tensors when given (any layout with the 128 features contiguous)."""
    def strides(t, heads):
        if t is None:
            return n * D, D
        assert t.dim() == 3 and t.shape[0] == heads and t.shape[1] == n and t.shape[2] == D and t.stride(2) == 1
        return t.stride(0), t.stride(1)
    qs, ks, os_ = strides(q, hq), strides(k, hkv), strides(out, hq)
    return Shape(hq, hkv, D, n, B, qs[0], qs[1], ks[0], ks[1], os_[0], os_[1], scale)


def params_default(**overrides) -> Params:
    p = Params()
    lib().crisp_params_default(ctypes.byref(p))
    for key, val in overrides.items():
        if key in ("alpha", "tau", "gamma", "vs_gamma"):
            setattr(p, f"{key}_num", val[0])
            setattr(p, f"{key}_den", val[1])
        else:
            setattr(p, key, val)
    return p


def workspace_size(shape: Shape) -> int:
    n = ctypes.c_size_t()
    _check(lib().crisp_workspace_size(ctypes.byref(shape), ctypes.byref(n)), "crisp_workspace_size")
    return n.value


def layer_workspace_size(shape: Shape) -> int:
    n = ctypes.c_size_t()
    _check(lib().crisp_layer_workspace_size(ctypes.byref(shape), ctypes.byref(n)), "crisp_layer_workspace_size")
    return n.value


def workspace_init(ws, stream=None):
    _check(lib().crisp_workspace_init(_ptr(ws), _nbytes(ws), _stream(stream)), "crisp_workspace_init")


def proxy_map(shape, q, k, pmap, ws, stream=None):
    _check(lib().crisp_proxy_map(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(pmap), _ptr(ws), _nbytes(ws),
                                 _stream(stream)), "crisp_proxy_map")


def proxy_map_noalloc(shape, q, k, pmap, stream=None):
    """crisp_proxy_map with the library's static scratch instead of a workspace
    (for callers that cannot allocate device memory; see include/crisp.h)."""
    _check(lib().crisp_proxy_map_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(pmap), _stream(stream)),
           "crisp_proxy_map_noalloc")


def noalloc_read_status(stream=None) -> int:
    """The status word of proxy_map_noalloc's static scratch (syncs the stream)."""
    s = ctypes.c_int()
    _check(lib().crisp_noalloc_read_status(_stream(stream), ctypes.byref(s)), "crisp_noalloc_read_status")
    return s.value


def block_masses(shape, pmap, vmass, smass, rmass, ws, stream=None):
    _check(lib().crisp_block_masses(ctypes.byref(shape), _ptr(pmap), _ptr(vmass), _ptr(smass), _ptr(rmass), _ptr(ws),
                                    _nbytes(ws), _stream(stream)), "crisp_block_masses")


def proxy_masses(shape, q, k, vmass, smass, rmass, ws, stream=None):
    """Block masses of the proxy map straight from q and k (the map is not stored)."""
    _check(lib().crisp_proxy_masses(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(vmass), _ptr(smass), _ptr(rmass),
                                    _ptr(ws), _nbytes(ws), _stream(stream)), "crisp_proxy_masses")


def route_cstruct(shape, params, pmap, cstruct, total, route, ws, stream=None):
    """A2 from the proxy map (any sink / recency slice widths of params)."""
    _check(lib().crisp_route_cstruct(ctypes.byref(shape), ctypes.byref(params), _ptr(pmap), _ptr(cstruct),
                                     _ptr(total), _ptr(route), _ptr(ws), _nbytes(ws), _stream(stream)),
           "crisp_route_cstruct")


def route_cstruct_masses(shape, params, vmass, rmass, cstruct, total, route, ws, stream=None):
    """A2 from the block masses (both slices one block wide)."""
    _check(lib().crisp_route_cstruct_masses(ctypes.byref(shape), ctypes.byref(params), _ptr(vmass), _ptr(rmass),
                                            _ptr(cstruct), _ptr(total), _ptr(route), _ptr(ws), _nbytes(ws),
                                            _stream(stream)), "crisp_route_cstruct_masses")


def route_jsd(shape, params, vmass, pbar, jsd, route, ws, stream=None):
    """FlexPrefill's divergence routing (comparator); pbar must hold row nb-1 of every head."""
    _check(lib().crisp_route_jsd(ctypes.byref(shape), ctypes.byref(params), _ptr(vmass), _ptr(pbar), _ptr(jsd),
                                 _ptr(route), _ptr(ws), _nbytes(ws), _stream(stream)), "crisp_route_jsd")


def select_vs(shape, params, pmap, route, vmass, smass, vbits, sbits, ws, stream=None):
    """A4 from the proxy map (writes the block masses too)."""
    _check(lib().crisp_select_vs(ctypes.byref(shape), ctypes.byref(params), _ptr(pmap), _ptr(route), _ptr(vmass),
                                 _ptr(smass), _ptr(vbits), _ptr(sbits), _ptr(ws), _nbytes(ws), _stream(stream)),
           "crisp_select_vs")


def select_vs_masses(shape, params, vmass, smass, route, vbits, sbits, ws, stream=None):
    """A4 from the block masses."""
    _check(lib().crisp_select_vs_masses(ctypes.byref(shape), ctypes.byref(params), _ptr(vmass), _ptr(smass),
                                        _ptr(route), _ptr(vbits), _ptr(sbits), _ptr(ws), _nbytes(ws),
                                        _stream(stream)), "crisp_select_vs_masses")


def pe_pool(shape, q, k, route, pbar, ws, stream=None):
    """A5: the pooled estimate of the PE heads (route[h] == 0)."""
    _check(lib().crisp_pe_pool(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(route), _ptr(pbar), _ptr(ws), _nbytes(ws),
                               _stream(stream)), "crisp_pe_pool")


def select_pe(shape, params, pbar, route, pebits, ws, stream=None):
    _check(lib().crisp_select_pe(ctypes.byref(shape), ctypes.byref(params), _ptr(pbar), _ptr(route), _ptr(pebits),
                                 _ptr(ws), _nbytes(ws), _stream(stream)), "crisp_select_pe")


def build_mask(shape, route, vbits, sbits, pebits, rowbits, counts, order, ws, stream=None):
    _check(lib().crisp_build_mask(ctypes.byref(shape), _ptr(route), _ptr(vbits), _ptr(sbits), _ptr(pebits),
                                  _ptr(rowbits), _ptr(counts), _ptr(order), _ptr(ws), _nbytes(ws), _stream(stream)),
           "crisp_build_mask")


def sparse_prefill(shape, q, k, v, route, vbits, sbits, pebits, out, ws, stream=None):
    """A8 from the index sets (the mask and schedule are built in ws)."""
    _check(lib().crisp_sparse_prefill(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(route), _ptr(vbits),
                                      _ptr(sbits), _ptr(pebits), _ptr(out), _ptr(ws), _nbytes(ws), _stream(stream)),
           "crisp_sparse_prefill")


def sparse_prefill_mask(shape, q, k, v, rowbits, order, out, ws, stream=None):
    """A8 over a block mask; order: the schedule from build_mask, or None (the same kv-group-major order)."""
    _check(lib().crisp_sparse_prefill_mask(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(rowbits),
                                           _ptr(order), _ptr(out), _ptr(ws), _nbytes(ws), _stream(stream)),
           "crisp_sparse_prefill_mask")


def dense_prefill(shape, q, k, v, out, ws, stream=None):
    _check(lib().crisp_dense_prefill(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(ws),
                                     _nbytes(ws), _stream(stream)), "crisp_dense_prefill")


def layer_views(shape, ws) -> dict:
    v = LayerViews()
    _check(lib().crisp_layer_views_get(ctypes.byref(shape), _ptr(ws), ctypes.byref(v)), "crisp_layer_views_get")
    return {name: getattr(v, name) for name, _ in LayerViews._fields_}


def prefill_layer(shape, params, q, k, v, out, ws, stream=None):
    _check(lib().crisp_prefill_layer(ctypes.byref(shape), ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                     _ptr(ws), _nbytes(ws), _stream(stream)), "crisp_prefill_layer")


class HostPipeline:
    """Streams and events of crisp_prefill_layer_host (on the current device)."""

    def __init__(self):
        self._h = ctypes.c_void_p()
        _check(lib().crisp_host_pipeline_create(ctypes.byref(self._h)), "crisp_host_pipeline_create")

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h:
            _check(lib().crisp_host_pipeline_destroy(self._h), "crisp_host_pipeline_destroy")
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def prefill_layer_host(pipeline, shape, params, q_host, k_host, v_host, out_host, q, k, v, out, ws, stream=None):
    """crisp_prefill_layer from host buffers (pinned torch CPU tensors), copies
    overlapped with compute; q, k, v, out are the device staging buffers."""
    _check(lib().crisp_prefill_layer_host(pipeline.handle, ctypes.byref(shape), ctypes.byref(params), _ptr(q_host),
                                          _ptr(k_host), _ptr(v_host), _ptr(out_host), _ptr(q), _ptr(k), _ptr(v),
                                          _ptr(out), _ptr(ws), _nbytes(ws), _stream(stream)),
           "crisp_prefill_layer_host")


def wait_selftest(ws, limit_ns, stream=None):
    """Launches the bounded-wait self-test (a wait that nothing ends)."""
    _check(lib().crisp_wait_selftest(_ptr(ws), _nbytes(ws), int(limit_ns), _stream(stream)), "crisp_wait_selftest")


def read_status(ws, stream=None) -> int:
    s = ctypes.c_int()
    _check(lib().crisp_read_status(_ptr(ws), _stream(stream), ctypes.byref(s)), "crisp_read_status")
    return s.value


def attention(q, k, v, params=None, scale=0.0, stream=None, check=True):
    """One CRISP sparse-prefill layer on torch tensors: q [hq][n][128], k and v
    [hkv][n][128], bf16, on the current CUDA device, features contiguous (any
    head and token strides that are multiples of 8 elements). Allocates the
    output (contiguous [hq][n][128] bf16) and a layer workspace with torch,
    runs crisp_prefill_layer on `stream` and returns the output. params: a
    Params (default: the paper's universal configuration); scale 0 means
    1/sqrt(128). With check=True the stream is synchronised and a device-side
    error raises CrispError."""
    import torch
    if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape:
        raise ValueError("attention: q must be [hq][n][128], k and v [hkv][n][128]")
    hq, n, _ = q.shape
    hkv = k.shape[0]
    out = torch.empty((hq, n, D), dtype=torch.bfloat16, device=q.device)
    shape = make_shape(hq, hkv, n, q, k, out, scale=scale)
    if k.stride() != v.stride():
        raise ValueError("attention: k and v must share their strides")
    ws = torch.empty(max(layer_workspace_size(shape), 256), dtype=torch.uint8, device=q.device)
    workspace_init(ws, stream)
    prefill_layer(shape, params if params is not None else params_default(), q, k, v, out, ws, stream)
    if check:
        st = read_status(ws, stream)
        if st != 0:
            raise CrispError(st, "crisp_prefill_layer (device)")
    return out
