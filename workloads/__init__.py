"""Synthetic workloads for the budgeted, importance-aware KV-cache decode step.

This module only *generates inputs*: the five workload shapes, seeded N(0,1)
query/key/value streams with heavy-hitter key scaling, and the per-head
budget tables.  It holds none of the method's arithmetic and imports neither
the CUDA library nor the oracle; both of those receive the arrays made here.

Every tensor is a counter-based stream keyed by (seed, tensor, layer, batch,
head) and indexed by token position, so any subset of units or positions can
be regenerated on its own (the oracle checks sampled layers of the big
workloads this way).

Five workload shapes: tiny fp32 (GQA group 2), a Llama-3-8B-shaped layer, a 32-layer 32K-context
stack evicting every 16 steps, HeadKV-style Dirichlet budgets, and a
Llama-3-70B-shaped 128K context.  Heavy-hitter keys stand in for the
observation (KV cache compression blog, sec. 2 "Heavy Hitter Tokens") that
5-20% of tokens hold most attention mass.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB = os.path.join(_HERE, "libsynth.so")

T_KEY, T_VALUE, T_QUERY, T_HEAVY = 1, 2, 3, 4


def build(verbose: bool = False) -> str:
    """Compile the generator (plain C, no method arithmetic) in place."""
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-o", _LIB, _SRC, "-lm"]
    if verbose:
        print(" ".join(cmd))
    subprocess.check_call(cmd)
    return _LIB


_lib = None
_lib_lock = threading.Lock()


def _load():
    global _lib
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
                build()
            lib = ctypes.CDLL(_LIB)
            lib.synth_fill.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                       ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int64,
                                       ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p,
                                       ctypes.c_int32, ctypes.c_void_p]
            lib.synth_fill.restype = None
            lib.synth_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                          ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int64,
                                          ctypes.c_int64, ctypes.c_void_p]
            lib.synth_uniform.restype = None
            _lib = lib
    return _lib


# ----------------------------------------------------------------------------
# workload definitions
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    layers: int
    batch: int
    hq: int
    hkv: int
    d: int
    dtype: str            # "f32" or "bf16": K/V, q and out
    prompt: int           # L_p, prompt tokens appended before decoding
    steps: int            # decode steps, one token appended per step
    budget: object        # int (uniform) or "dirichlet"
    sink: int
    window: int
    evict_every: int      # E: evict after every E decode steps
    heavy: Optional[str]  # heavy-hitter recipe
    nq: int = 16          # prefill observation window (queries scored)
    # a shard of a larger workload (see shard()): its first layer and batch
    # row there, and that workload's layer count (0: this one's).  Inputs
    # and budgets are those of the larger workload's units.
    layer0: int = 0
    batch0: int = 0
    layers_total: int = 0

    @property
    def group(self) -> int:
        return self.hq // self.hkv

    @property
    def units(self) -> int:
        return self.layers * self.batch * self.hkv

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    @property
    def total_positions(self) -> int:
        return self.prompt + self.steps

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def shard(w: Workload, l0: int, l1: int, b0: int, b1: int) -> Workload:
    """Layers [l0, l1) x batch rows [b0, b1) of w (every KV head) as a
    workload of its own, whose inputs and budgets are w's for those units."""
    assert 0 <= l0 < l1 <= w.layers and 0 <= b0 < b1 <= w.batch
    return w.with_(name=f"{w.name}[l{l0}:{l1},b{b0}:{b1}]", layers=l1 - l0, batch=b1 - b0,
                   layer0=w.layer0 + l0, batch0=w.batch0 + b0, layers_total=w.layers_total or w.layers)


WORKLOADS = [
    Workload(0, "tiny-fp32-gqa2", 1, 1, 4, 2, 64, "f32", 256, 64, 128, 4, 32, 1, "fixed8x4"),
    Workload(1, "llama3-8b-layer-b8-ctx8k", 1, 8, 32, 8, 128, "bf16", 8192, 256, 1024, 4, 64, 1,
             "bernoulli5x3"),
    Workload(2, "32layer-b4-ctx32k-evict16", 32, 4, 32, 8, 128, "bf16", 32768, 128, 2048, 4, 128, 16,
             "zipf1.1"),
    Workload(3, "headkv-dirichlet-32layer-b16-ctx16k", 32, 16, 32, 8, 128, "bf16", 16384, 128,
             "dirichlet", 4, 32, 1, None),
    Workload(4, "llama3-70b-b1-ctx128k", 80, 1, 64, 8, 128, "bf16", 131072, 64, 4096, 4, 256, 1,
             "zipf1.1"),
]


def kv_bytes(batch: int, length: int, layers: int, kv_heads: int, head_dim: int,
             elem_bytes: int) -> int:
    """Full KV-cache size M = 2 * B * L * N_L * N_KV * D * P (KV cache
    compression blog, sec. 1 "The KV Cache Memory and Bandwidth Wall")."""
    return 2 * batch * length * layers * kv_heads * head_dim * elem_bytes


def budgets(w: Workload, seed: Optional[int] = None) -> np.ndarray:
    """Per-(layer, KV head) budgets, int32 [layers * hkv], shared by all batch rows.

    Dirichlet case (HeadKV-style variable budgets): one Dirichlet(0.5) draw over
    all layers*hkv heads scaled to a mean of 256, rounded half up, clamped to
    [64, 2048] with no renormalisation after the clamp.
    """
    seed = w.index if seed is None else seed
    n = (w.layers_total or w.layers) * w.hkv
    rows = slice(w.layer0 * w.hkv, (w.layer0 + w.layers) * w.hkv)   # a shard's layers
    if w.budget == "dirichlet":
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0xB0D6E7])))
        frac = rng.dirichlet(np.full(n, 0.5))
        raw = frac * (256.0 * n)
        b = np.floor(raw + 0.5).astype(np.int64)
        b = np.clip(b, 64, 2048)
        return b.astype(np.int32)[rows].copy()
    return np.full(n, int(w.budget), dtype=np.int32)[rows].copy()


def retrieval_mask(w: Workload, frac: float, seed: Optional[int] = None) -> np.ndarray:
    """A seeded choice of DuoAttention retrieval heads: round(frac * heads) of
    the layers * hkv (layer, KV head) pairs, [layers][hkv] bool.  (The pages
    identify them by a trained gate; synthetic runs draw them.)"""
    seed = w.index if seed is None else seed
    n = w.layers * w.hkv
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0xD0A7])))
    m = np.zeros(n, dtype=bool)
    m[rng.permutation(n)[: int(round(frac * n))]] = True
    return m.reshape(w.layers, w.hkv)


def heavy_scale(w: Workload, seed: int, layer: int, batch: int, upto: int = 0) -> Optional[np.ndarray]:
    """Key scale per position [T] for one (layer, batch) sequence, where
    T = max(total_positions, upto): a run generating positions past the
    workload's own steps passes `upto` so every generated position has one.

    Applies to the keys of every KV head at that position.
      fixed8x4     : exactly 8 distinct prompt positions, x4
      bernoulli5x3 : each position heavy with probability 0.05, x3
      zipf1.1      : random rank r(p) in 1..T, x(1 + 3 r^-1.1)
    """
    if w.heavy is None:
        return None
    T = max(w.total_positions, int(upto))
    lib = _load()
    u = np.empty(T, dtype=np.float64)
    lib.synth_uniform(seed, T_HEAVY, layer, batch, 0, 0, T, u.ctypes.data)
    s = np.ones(T, dtype=np.float32)
    if w.heavy == "fixed8x4":
        idx = np.argsort(u[: w.prompt], kind="stable")[:8]
        s[idx] = 4.0
    elif w.heavy == "bernoulli5x3":
        s[u < 0.05] = 3.0
    elif w.heavy == "zipf1.1":
        rank = np.empty(T, dtype=np.int64)
        rank[np.argsort(u, kind="stable")] = np.arange(1, T + 1)
        s = (1.0 + 3.0 * rank.astype(np.float64) ** -1.1).astype(np.float32)
    else:
        raise ValueError(w.heavy)
    return s


_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max(1, os.cpu_count() or 1))
    return _POOL


def _fill_streams(jobs, dim, out_bf16):
    lib = _load()

    def run(job):
        (seed, tensor, layer, batch, head, pos0, npos, scale, dst) = job
        sp = scale.ctypes.data if scale is not None else None
        lib.synth_fill(seed, tensor, layer, batch, head, pos0, npos, dim, sp,
                       1 if out_bf16 else 0, dst.ctypes.data)

    list(_pool().map(run, jobs))


def gen_kv(w: Workload, layer0: int, nlayers: int, pos0: int, npos: int,
           seed: Optional[int] = None):
    """K and V for positions [pos0, pos0+npos) of layers [layer0, layer0+nlayers).

    Returns (k, v), each [nlayers][batch][hkv][npos][d]; float32 for f32
    workloads, uint16 bf16 bit patterns for bf16 workloads.  Heavy-hitter
    scaling applies to K only.
    """
    seed = w.index if seed is None else seed
    bf = w.dtype == "bf16"
    dt = np.uint16 if bf else np.float32
    k = np.empty((nlayers, w.batch, w.hkv, npos, w.d), dtype=dt)
    v = np.empty_like(k)
    jobs = []
    for li in range(nlayers):
        layer = w.layer0 + layer0 + li
        for b in range(w.batch):
            bg = w.batch0 + b
            hs = heavy_scale(w, seed, layer, bg, upto=pos0 + npos)
            sc = None if hs is None else np.ascontiguousarray(hs[pos0: pos0 + npos])
            assert sc is None or sc.size == npos
            for g in range(w.hkv):
                jobs.append((seed, T_KEY, layer, bg, g, pos0, npos, sc, k[li, b, g]))
                jobs.append((seed, T_VALUE, layer, bg, g, pos0, npos, None, v[li, b, g]))
    _fill_streams(jobs, w.d, bf)
    return k, v


def gen_kv_unit(w: Workload, layer: int, batch: int, g: int, pos0: int, npos: int,
                seed: Optional[int] = None):
    """K and V rows [npos][d] of one (layer, batch, KV head) stream."""
    seed = w.index if seed is None else seed
    bf = w.dtype == "bf16"
    dt = np.uint16 if bf else np.float32
    k = np.empty((npos, w.d), dtype=dt)
    v = np.empty_like(k)
    layer, batch = w.layer0 + layer, w.batch0 + batch
    hs = heavy_scale(w, seed, layer, batch, upto=pos0 + npos)
    sc = None if hs is None else np.ascontiguousarray(hs[pos0: pos0 + npos])
    assert sc is None or sc.size == npos
    _fill_streams([(seed, T_KEY, layer, batch, g, pos0, npos, sc, k),
                   (seed, T_VALUE, layer, batch, g, pos0, npos, None, v)], w.d, bf)
    return k, v


def gen_q(w: Workload, layer0: int, nlayers: int, pos0: int, npos: int,
          seed: Optional[int] = None):
    """Queries for positions [pos0, pos0+npos): [nlayers][batch][hq][npos][d]."""
    seed = w.index if seed is None else seed
    bf = w.dtype == "bf16"
    dt = np.uint16 if bf else np.float32
    q = np.empty((nlayers, w.batch, w.hq, npos, w.d), dtype=dt)
    jobs = []
    for li in range(nlayers):
        for b in range(w.batch):
            for h in range(w.hq):
                jobs.append((seed, T_QUERY, w.layer0 + layer0 + li, w.batch0 + b, h, pos0, npos, None,
                             q[li, b, h]))
    _fill_streams(jobs, w.d, bf)
    return q


def to_f32(a: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 exactly; float32 passes through."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32)
    return a.astype(np.float32, copy=False)


def to_torch(a: np.ndarray):
    """numpy array -> CPU torch tensor of the workload dtype (bf16 from uint16 bits)."""
    import torch
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(a)
