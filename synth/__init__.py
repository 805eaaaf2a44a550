"""Seeded synthetic Q/K/V with planted sink, slash, needle and cluster structure.

The single input source shared by the CUDA path's tests/benchmark and the CPU
oracle. It holds none of the sparse-attention method's arithmetic: it only
writes bf16 bit patterns. See ``synth.c`` for the recipe.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile libsynth.so next to its source (plain C, pthreads)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Config(ctypes.Structure):
    _fields_ = [
        ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32), ("n", ctypes.c_int32),
        ("seed", ctypes.c_uint64),
        ("sink_tokens", ctypes.c_int32), ("d_sink", ctypes.c_float),
        ("n_needles", ctypes.c_int32), ("d_needle", ctypes.c_float),
        ("n_slash", ctypes.c_int32), ("d_slash", ctypes.c_float),
        ("slash_min", ctypes.c_int32), ("slash_max", ctypes.c_int32),
        ("band_w", ctypes.c_int32), ("d_band", ctypes.c_float),
        ("d_cluster", ctypes.c_float),
        ("head_is_vs", ctypes.POINTER(ctypes.c_uint8)),
        ("nthreads", ctypes.c_int32),
    ]


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.synth_generate.argtypes = [ctypes.POINTER(_Config), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        lib.synth_generate.restype = ctypes.c_int
        lib.synth_needle_positions.argtypes = [ctypes.POINTER(_Config), ctypes.c_int, ctypes.POINTER(ctypes.c_int32)]
        lib.synth_needle_positions.restype = ctypes.c_int
        lib.synth_slash_offsets.argtypes = [ctypes.POINTER(_Config), ctypes.c_int, ctypes.POINTER(ctypes.c_int32)]
        lib.synth_slash_offsets.restype = None
        _lib = lib
    return _lib


@dataclass
class Workload:
    """One synthetic attention layer: shape plus planted structure."""

    name: str
    hq: int
    hkv: int
    n: int
    seed: int
    vs_heads: list  # q-heads with sink/slash/needle structure; the rest are diffuse
    sink_tokens: int = 128
    d_sink: float = 8.0
    n_needles: int = 8
    d_needle: float = 9.0
    n_slash: int = 2
    d_slash: float = 9.0
    slash_min: int = 256
    slash_max: int = 0  # 0 -> n // 2
    band_w: int = 128
    d_band: float = 0.0  # the low-frequency band only where a config asks for one
    d_cluster: float = 5.0
    layers: int = 1
    extra: dict = field(default_factory=dict)

    def _cfg(self, nthreads: int):
        vs = np.zeros(self.hq, dtype=np.uint8)
        vs[list(self.vs_heads)] = 1
        self._vs = vs  # keep alive for the C call
        c = _Config(self.hq, self.hkv, self.n, self.seed, self.sink_tokens, self.d_sink, self.n_needles,
                    self.d_needle, self.n_slash, self.d_slash, self.slash_min,
                    self.slash_max if self.slash_max > 0 else max(self.slash_min + 1, self.n // 2),
                    self.band_w, self.d_band, self.d_cluster,
                    vs.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), nthreads)
        return c

    def layer(self, layer: int) -> "Workload":
        """The workload of one layer of a stack (per-layer seed and head mix)."""
        if self.layers == 1:
            return self
        mix = self.extra["vs_fraction"][layer]
        seed = self.seed + layer
        rng = np.random.default_rng(seed)
        nvs = int(round(mix * self.hq))
        heads = sorted(rng.permutation(self.hq)[:nvs].tolist())
        return Workload(**{**self.__dict__, "name": f"{self.name}-L{layer}", "seed": seed, "vs_heads": heads,
                           "layers": 1, "extra": {}})

    def generate(self, q=None, k=None, v=None, nthreads: int | None = None):
        """Returns (q, k, v) as uint16 arrays holding bf16 bits, shapes
        [hq][n][128], [hkv][n][128], [hkv][n][128]. Buffers may be passed in
        (e.g. pinned host memory viewed as numpy)."""
        lib = _load()
        nthreads = nthreads or os.cpu_count() or 1
        q = np.empty((self.hq, self.n, 128), np.uint16) if q is None else q
        k = np.empty((self.hkv, self.n, 128), np.uint16) if k is None else k
        v = np.empty((self.hkv, self.n, 128), np.uint16) if v is None else v
        for a, shape in ((q, (self.hq, self.n, 128)), (k, (self.hkv, self.n, 128)), (v, (self.hkv, self.n, 128))):
            assert a.dtype == np.uint16 and a.shape == shape and a.flags.c_contiguous
        c = self._cfg(nthreads)
        rc = lib.synth_generate(ctypes.byref(c), q.ctypes.data, k.ctypes.data, v.ctypes.data)
        if rc != 0:
            raise RuntimeError(f"synth_generate failed: {rc}")
        return q, k, v

    def needle_positions(self, g: int):
        lib = _load()
        c = self._cfg(1)
        out = (ctypes.c_int32 * max(1, self.n_needles))()
        cnt = lib.synth_needle_positions(ctypes.byref(c), g, out)
        return sorted(out[i] for i in range(cnt))

    def slash_offsets(self, h: int):
        lib = _load()
        c = self._cfg(1)
        out = (ctypes.c_int32 * max(1, self.n_slash))()
        lib.synth_slash_offsets(ctypes.byref(c), h, out)
        return [out[i] for i in range(self.n_slash)]


def _alternating(hq):
    return [h for h in range(hq) if h % 2 == 0]


# The five workloads (1 layer unless stated): shapes of Llama-3.1-8B (32 q / 8
# kv heads) and Qwen2.5-7B (28 q / 4 kv heads), head_dim 128, block 128.
WORKLOADS = {
    # 4 q / 1 kv, 2k tokens, all heads sink-type: 64 sink keys at +4 logit,
    # a local band of width 64, 3 needle columns, no sharp slash.
    "gqa4x1-2k": Workload("gqa4x1-2k", 4, 1, 2048, 0, [0, 1, 2, 3], sink_tokens=64, d_sink=4.0, n_needles=3,
                     d_needle=7.0, n_slash=0, band_w=64, d_band=3.0),
    # Llama-shaped, 32k: even heads sink+2 slashes+8 needles, odd heads diffuse.
    "llama8b-32k": Workload("llama8b-32k", 32, 8, 32768, 1, _alternating(32), d_sink=7.0, n_needles=8,
                     d_needle=9.0, n_slash=2, d_slash=9.0),
    # Qwen-shaped, 128k: even heads sink/recency dominated (no sharp slash),
    # odd heads diffuse; 16 needles.
    "qwen7b-128k": Workload("qwen7b-128k", 28, 4, 131072, 2, _alternating(28), d_sink=8.0, n_needles=16,
                     d_needle=9.5, n_slash=0),
    # Llama-shaped 4-layer stack, 256k: 25/50/75/90% sink-type heads per layer.
    "llama8b-256k-stack": Workload("llama8b-256k-stack", 32, 8, 262144, 4000, list(range(32)), d_sink=8.5, n_needles=8,
                     d_needle=10.0, n_slash=2, d_slash=10.0, layers=4,
                     extra={"vs_fraction": [0.25, 0.50, 0.75, 0.90]}),
    # Llama-shaped, 512k, every head sink-type with 2 slashes and 32 needles.
    "llama8b-512k": Workload("llama8b-512k", 32, 8, 524288, 5, list(range(32)), d_sink=10.0, n_needles=32,
                     d_needle=10.0, n_slash=2, d_slash=10.0),
}


def small(name: str, hq: int, hkv: int, n: int, seed: int, vs_heads=None, **kw) -> Workload:
    """A small workload for parity tests (same recipe, chosen shape)."""
    vs = list(range(0, hq, 2)) if vs_heads is None else vs_heads
    base = dict(sink_tokens=64, d_sink=5.0, n_needles=3, d_needle=7.0, n_slash=1, d_slash=8.0, slash_min=256,
                band_w=64, d_band=0.0, d_cluster=5.0)
    base.update(kw)
    return Workload(name, hq, hkv, n, seed, vs, **base)
