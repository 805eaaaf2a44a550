"""CPU oracle for CRISP sparse prefill (fp64, plain C++). TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package. The product library never calls
it and shares no code with it. See ``crisp_oracle.cpp`` for the definitions
and the readings of the pages they follow.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "crisp_oracle.cpp")
_LIB = os.path.join(_HERE, "libcrisp_oracle.so")
_lib = None
B = 128
D = 128


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def _p(a):
    return ctypes.c_void_p(a.ctypes.data)


def _configure(lib):
    """Declares the argument types of the oracle's C entry points on `lib`."""
    i, vp, d, u32, i64 = ctypes.c_int, ctypes.c_void_p, ctypes.c_double, ctypes.c_uint32, ctypes.c_int64
    lib.oracle_proxy_map.argtypes = [i, i, i, vp, vp, d, vp, i]
    lib.oracle_quantize.argtypes = [vp, i64, vp]
    lib.oracle_quantize.restype = None
    lib.oracle_proxy_rows.argtypes = [i, i, i, vp, vp, d, i64, vp, vp, vp, i]
    lib.oracle_route.argtypes = [i, i, vp, u32, u32, i, i, vp, vp, vp, i]
    lib.oracle_vs_masses.argtypes = [i, i, vp, vp, vp, i]
    lib.oracle_pe_rows.argtypes = [i, i, i, vp, vp, d, i64, vp, vp, vp, i]
    lib.oracle_select_vs.argtypes = [i, i, vp, vp, vp, u32, u32, i, vp, vp]
    lib.oracle_select_vs_gamma.argtypes = [i, i, vp, vp, vp, u32, u32, i, vp, vp]
    lib.oracle_route_jsd.argtypes = [i, i, vp, vp, d, vp, vp]
    lib.oracle_pe_map.argtypes = [i, i, i, vp, vp, d, vp, i]
    lib.oracle_select_pe.argtypes = [i, i, vp, vp, i, u32, u32, u32, u32, i, vp, i]
    lib.oracle_build_mask.argtypes = [i, i, vp, vp, vp, vp, vp]
    lib.oracle_attention_rows.argtypes = [i, i, i, vp, vp, vp, d, vp, i64, vp, vp, vp, i]
    lib.oracle_selected_pairs.argtypes = [i, i, vp]
    lib.oracle_selected_pairs.restype = ctypes.c_int64
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _configure(ctypes.CDLL(_LIB))
    return _lib


def _nt(nthreads):
    return nthreads or os.cpu_count() or 1


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"{what}: invalid arguments (rc={rc})")


def _u16(a):
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16
    return a


def num_blocks(n):
    """Blocks of n tokens: ceil(n / 128) (a short last block when 128 does not divide n)."""
    return (n + B - 1) // B


def default_scale():
    return 1.0 / np.sqrt(D)


def proxy_map(q, k, scale=None, nthreads=None):
    """A1: fp64 proxy map [hq][128][n] of the last query block."""
    q, k = _u16(q), _u16(k)
    hq, n, _ = q.shape
    hkv = k.shape[0]
    out = np.empty((hq, B, n), np.float64)
    _check(_load().oracle_proxy_map(hq, hkv, n, _p(q), _p(k), scale or default_scale(), _p(out), _nt(nthreads)),
           "proxy_map")
    return out


def proxy_rows(q, k, heads, rows, scale=None, nthreads=None):
    """A1 for selected (head, row of the last block) pairs: fp64 [count][n]."""
    q, k = _u16(q), _u16(k)
    hq, n, _ = q.shape
    heads = np.ascontiguousarray(heads, np.int32)
    rows = np.ascontiguousarray(rows, np.int32)
    out = np.empty((heads.size, n), np.float64)
    _check(_load().oracle_proxy_rows(hq, k.shape[0], n, _p(q), _p(k), scale or default_scale(), heads.size,
                                     _p(heads), _p(rows), _p(out), _nt(nthreads)), "proxy_rows")
    return out


def pe_rows(q, k, heads, blocks, scale=None, nthreads=None):
    """A5 for selected (head, query block) pairs: fp64 [count][nb]."""
    q, k = _u16(q), _u16(k)
    hq, n, _ = q.shape
    heads = np.ascontiguousarray(heads, np.int32)
    blocks = np.ascontiguousarray(blocks, np.int32)
    out = np.empty((heads.size, num_blocks(n)), np.float64)
    _check(_load().oracle_pe_rows(hq, k.shape[0], n, _p(q), _p(k), scale or default_scale(), heads.size,
                                  _p(heads), _p(blocks), _p(out), _nt(nthreads)), "pe_rows")
    return out


def quantize(p):
    p = np.ascontiguousarray(p, dtype=np.float32)
    out = np.empty(p.shape, np.uint64)
    _load().oracle_quantize(_p(p), p.size, _p(out))
    return out


def route(pmap32, tau=(1, 5), sink=128, recency=128, nthreads=None):
    """A2: (cstruct S, total T, route) from an fp32 map [hq][128][n]; the
    slices are key columns [0, sink) and [n - recency, n)."""
    pmap32 = np.ascontiguousarray(pmap32, dtype=np.float32)
    hq, _, n = pmap32.shape
    S, T, r = np.empty(hq, np.uint64), np.empty(hq, np.uint64), np.empty(hq, np.uint8)
    _check(_load().oracle_route(hq, n, _p(pmap32), tau[0], tau[1], int(sink), int(recency), _p(S), _p(T), _p(r),
                                _nt(nthreads)), "route")
    return S, T, r


def vs_masses(pmap32, nthreads=None):
    """A3: (vmass, smass) uint64 [hq][nb] from an fp32 map."""
    pmap32 = np.ascontiguousarray(pmap32, dtype=np.float32)
    hq, _, n = pmap32.shape
    nb = num_blocks(n)
    vm, sm = np.empty((hq, nb), np.uint64), np.empty((hq, nb), np.uint64)
    _check(_load().oracle_vs_masses(hq, n, _p(pmap32), _p(vm), _p(sm), _nt(nthreads)), "vs_masses")
    return vm, sm


def select_vs(vmass, smass, route_, alpha=(1, 1), kmin=8):
    """A4: (vbits, sbits) uint32 [hq][W]."""
    vmass = np.ascontiguousarray(vmass, np.uint64)
    smass = np.ascontiguousarray(smass, np.uint64)
    route_ = np.ascontiguousarray(route_, np.uint8)
    hq, nb = vmass.shape
    W = (nb + 31) // 32
    vb, sb = np.empty((hq, W), np.uint32), np.empty((hq, W), np.uint32)
    _check(_load().oracle_select_vs(hq, nb, _p(vmass), _p(smass), _p(route_), alpha[0], alpha[1], kmin, _p(vb),
                                    _p(sb)), "select_vs")
    return vb, sb


def select_vs_gamma(vmass, smass, route_, gamma=(95, 100), kmin=8):
    """A4 comparator (FlexPrefill's cumulative coverage): (vbits, sbits)."""
    vmass = np.ascontiguousarray(vmass, np.uint64)
    smass = np.ascontiguousarray(smass, np.uint64)
    route_ = np.ascontiguousarray(route_, np.uint8)
    hq, nb = vmass.shape
    W = (nb + 31) // 32
    vb, sb = np.empty((hq, W), np.uint32), np.empty((hq, W), np.uint32)
    _check(_load().oracle_select_vs_gamma(hq, nb, _p(vmass), _p(smass), _p(route_), gamma[0], gamma[1], kmin,
                                          _p(vb), _p(sb)), "select_vs_gamma")
    return vb, sb


def route_jsd(vmass, pbar_last32, tau=0.1):
    """A2 comparator (FlexPrefill's divergence routing): (jsd D, route) from
    the block masses [hq][nb] and the pooled map's last rows [hq][nb] (fp32)."""
    vmass = np.ascontiguousarray(vmass, np.uint64)
    pl = np.ascontiguousarray(pbar_last32, np.float32)
    hq, nb = vmass.shape
    D, r = np.empty(hq, np.float64), np.empty(hq, np.uint8)
    _check(_load().oracle_route_jsd(hq, nb, _p(vmass), _p(pl), float(tau), _p(D), _p(r)), "route_jsd")
    return D, r


def pe_map(q, k, scale=None, nthreads=None):
    """A5: fp64 pooled map [hq][nb][nb]."""
    q, k = _u16(q), _u16(k)
    hq, n, _ = q.shape
    nb = num_blocks(n)
    out = np.empty((hq, nb, nb), np.float64)
    _check(_load().oracle_pe_map(hq, k.shape[0], n, _p(q), _p(k), scale or default_scale(), _p(out),
                                 _nt(nthreads)), "pe_map")
    return out


def select_pe(pbar32, route_, pe_mode=0, gamma=(19, 20), alpha=(1, 1), kmin=8, nthreads=None):
    """A6: pebits uint32 [hq][nb][W] from an fp32 pooled map."""
    pbar32 = np.ascontiguousarray(pbar32, dtype=np.float32)
    route_ = np.ascontiguousarray(route_, np.uint8)
    hq, nb, _ = pbar32.shape
    W = (nb + 31) // 32
    out = np.empty((hq, nb, W), np.uint32)
    _check(_load().oracle_select_pe(hq, nb, _p(pbar32), _p(route_), pe_mode, gamma[0], gamma[1], alpha[0],
                                    alpha[1], kmin, _p(out), _nt(nthreads)), "select_pe")
    return out


def build_mask(route_, vbits, sbits, pebits):
    """A7: rowbits uint32 [hq][nb][W]."""
    route_ = np.ascontiguousarray(route_, np.uint8)
    vbits = np.ascontiguousarray(vbits, np.uint32)
    sbits = np.ascontiguousarray(sbits, np.uint32)
    pebits = np.ascontiguousarray(pebits, np.uint32)
    hq, nb, W = pebits.shape
    out = np.empty((hq, nb, W), np.uint32)
    _check(_load().oracle_build_mask(hq, nb, _p(route_), _p(vbits), _p(sbits), _p(pebits), _p(out)), "build_mask")
    return out


def attention_rows(q, k, v, heads, tokens, rowbits=None, scale=None, nthreads=None):
    """A8/A9: fp64 outputs [count][128] for (head, token) pairs; rowbits None = dense causal."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    hq, n, _ = q.shape
    heads = np.ascontiguousarray(heads, np.int32)
    tokens = np.ascontiguousarray(tokens, np.int32)
    out = np.empty((heads.size, D), np.float64)
    rb = None
    if rowbits is not None:
        rb = np.ascontiguousarray(rowbits, np.uint32)
    _check(_load().oracle_attention_rows(hq, k.shape[0], n, _p(q), _p(k), _p(v), scale or default_scale(),
                                         _p(rb) if rb is not None else None, heads.size, _p(heads), _p(tokens),
                                         _p(out), _nt(nthreads)), "attention_rows")
    return out


def selected_pairs(rowbits, n):
    """Causal (row, key) pairs over the selected blocks of an n-token layer."""
    rowbits = np.ascontiguousarray(rowbits, np.uint32)
    hq, nb, _ = rowbits.shape
    if nb != num_blocks(n):
        raise ValueError("selected_pairs: rowbits has the wrong block count for n")
    return int(_load().oracle_selected_pairs(hq, n, _p(rowbits)))


def bits_to_sets(bits, nb):
    """Decodes bitset rows (last axis = words) into sorted index lists."""
    bits = np.asarray(bits, np.uint32)
    flat = bits.reshape(-1, bits.shape[-1])
    out = []
    for row in flat:
        idx = np.nonzero(np.unpackbits(row.view(np.uint8), bitorder="little")[:nb])[0]
        out.append(idx.tolist())
    return out
