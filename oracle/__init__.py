"""ORACLE — test infrastructure only.

ctypes front end of the plain CPU model in ``hikv_oracle.cpp``.  Only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package; the CUDA library never does, and the two share no code.

Inputs are numpy float32 arrays (bf16 values widened exactly).  Layouts match
the library's: K/V ``[nl][batch][hkv][ntok][d]``, window queries
``[nl][batch][hq][nq][d]``, decode queries/outputs ``[nl][batch][hq][d]``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hikv_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")


def build(verbose: bool = False) -> str:
    """Compile the oracle (plain C++17, -O2, no fast-math, no FMA contraction)."""
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-o", _LIB, _SRC]
    if verbose:
        print(" ".join(cmd))
    subprocess.check_call(cmd)
    return _LIB


_lib = None
_lock = threading.Lock()

_P = ctypes.c_void_p
_I = ctypes.c_int


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
                build()
            lib = ctypes.CDLL(_LIB)
            sig = {
                "ora_create": ([_I] * 7 + [_P, ctypes.c_double, _I, _I], _P),
                "ora_destroy": ([_P], None),
                "ora_num_threads": ([_P, _I], _I),
                "ora_append": ([_P, _I, _I, _I, _P, _P], _I),
                "ora_score_window": ([_P, _I, _I, _I, _P], _I),
                "ora_score_band": ([_P, _I, _I, _I, _P], _I),
                "ora_stage2_alternatives": ([_P, _I, _I, _I, _P, _I], _I),
                "ora_pool_importance": ([_P, _I, _I, _I], _I),
                "ora_set_recent_only": ([_P, _I], _I),
                "ora_set_element_budget": ([_P, _I], _I),
                "ora_stage2_near_ties": ([_P, _I, _I, _P], _I),
                "ora_decode": ([_P, _I, _I, _P, _P], _I),
                "ora_evict": ([_P, _I, _I], _I),
                "ora_len": ([_P, _I], _I),
                "ora_next_pos": ([_P, _I], _I),
                "ora_num_evicted": ([_P, _I], _I),
                "ora_evicted_mass": ([_P, _I], ctypes.c_double),
                "ora_state": ([_P, _I, _P, _P, _P, _P], _I),
                "ora_evicted": ([_P, _I, _P, _P], _I),
                "ora_resync": ([_P, _I, _I, _P], _I),
            }
            for name, (args, res) in sig.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


class Oracle:
    """CPU oracle of one cache (all units of L layers x batch x KV heads)."""

    def __init__(self, layers, batch, hq, hkv, d, sink, window, budgets,
                 scale=0.0, out_bf16=False, threads=1):
        self.lib = _load()
        self.L, self.B, self.Hq, self.Hkv, self.d = layers, batch, hq, hkv, d
        self.G = hq // hkv
        self.S, self.W = sink, window
        self.budgets = np.ascontiguousarray(budgets, dtype=np.int32)
        assert self.budgets.size == layers * hkv
        self.h = self.lib.ora_create(layers, batch, hq, hkv, d, sink, window,
                                     _ptr(self.budgets), float(scale), int(out_bf16),
                                     int(threads))
        if not self.h:
            raise ValueError("oracle: invalid configuration")

    def __del__(self):
        h = getattr(self, "h", None)
        if h:
            self.lib.ora_destroy(h)
            self.h = None

    @property
    def units(self):
        return self.L * self.B * self.Hkv

    def unit(self, layer, batch, g):
        return (layer * self.B + batch) * self.Hkv + g

    def budget_of(self, u):
        return int(self.budgets[(u // (self.B * self.Hkv)) * self.Hkv + u % self.Hkv])

    def threads(self, n=0):
        return self.lib.ora_num_threads(self.h, n)

    def append(self, layer0, k, v):
        k, v = _f32(k), _f32(v)
        nl, ntok = k.shape[0], k.shape[3]
        assert self.lib.ora_append(self.h, layer0, nl, ntok, _ptr(k), _ptr(v)) == 0

    def score_window(self, layer0, q):
        q = _f32(q)
        nl, nq = q.shape[0], q.shape[3]
        assert self.lib.ora_score_window(self.h, layer0, nl, nq, _ptr(q)) == 0

    def score_band(self, layer0, q, band):
        """HiKV prefill initialisation: q [nl][B][Hq][n][d] holds the queries
        of every held position 0..n-1; each token's score grows by its causal
        attention column summed over the band of queries from its position."""
        q = _f32(q)
        nl = q.shape[0]
        rc = self.lib.ora_score_band(self.h, layer0, nl, int(band), _ptr(q))
        if rc:
            raise ValueError(f"oracle: score_band failed ({rc})")

    def set_recent_only(self, on=True):
        """HiKV Stage I: decode steps add mass only to the recent bank."""
        assert self.lib.ora_set_recent_only(self.h, 1 if on else 0) == 0

    def set_element_budget(self, b2):
        """HiKV Stage II: 0 < b2 < d dimensions of q and b2 entries of every
        d-entry chunk of P take part (0 or d: exact attention)."""
        if self.lib.ora_set_element_budget(self.h, int(b2)) != 0:
            raise ValueError(f"oracle: element budget {b2} outside [0, {self.d}]")

    def stage2_near_ties(self, layer0, nl):
        """[nl][B][Hq] uint8 for the latest Stage II step: 0 where every chunk
        selection is certain under float32 rounding of the logits, 1 where
        some is not (see stage2_alternatives), 2 where too many selections
        were admissible to list."""
        f = np.zeros((nl, self.B, self.Hq), np.uint8)
        assert self.lib.ora_stage2_near_ties(self.h, layer0, nl, _ptr(f)) == 0
        return f

    def stage2_alternatives(self, layer, b, head, max_alts=4096):
        """[count][d] float32: every output of query head `head` that a
        selection admissible under float32 rounding gives (the exact one
        included); None when there were too many."""
        out = np.empty((max_alts, self.d), np.float32)
        n = self.lib.ora_stage2_alternatives(self.h, layer, b, head, _ptr(out), max_alts)
        return None if n < 0 else out[:n].copy()

    def pool_importance(self, layer0, nl, kpool):
        """SnapKV: each score becomes the max over the next kpool positions."""
        assert self.lib.ora_pool_importance(self.h, layer0, nl, int(kpool)) == 0

    def decode(self, layer0, q):
        q = _f32(q)
        out = np.empty_like(q)
        rc = self.lib.ora_decode(self.h, layer0, q.shape[0], _ptr(q), _ptr(out))
        if rc:
            raise RuntimeError(f"oracle decode failed ({rc})")
        return out

    def evict(self, layer0, nl):
        assert self.lib.ora_evict(self.h, layer0, nl) == 0

    def length(self, u):
        return self.lib.ora_len(self.h, u)

    def next_pos(self, u):
        return self.lib.ora_next_pos(self.h, u)

    def evicted_mass(self, u):
        return self.lib.ora_evicted_mass(self.h, u)

    def state(self, u, with_kv=False):
        n = self.length(u)
        pos = np.empty(n, np.int32)
        imp = np.empty(n, np.float32)
        k = v = None
        if with_kv:
            k = np.empty((n, self.d), np.float32)
            v = np.empty((n, self.d), np.float32)
        self.lib.ora_state(self.h, u, _ptr(pos), _ptr(imp),
                           _ptr(k) if with_kv else None, _ptr(v) if with_kv else None)
        return (pos, imp, k, v) if with_kv else (pos, imp)

    def last_evicted(self, u):
        n = self.lib.ora_num_evicted(self.h, u)
        pos = np.empty(n, np.int32)
        imp = np.empty(n, np.float32)
        self.lib.ora_evicted(self.h, u, _ptr(pos), _ptr(imp))
        return pos, imp

    def resync(self, u, positions):
        p = np.ascontiguousarray(positions, dtype=np.int32)
        if self.lib.ora_resync(self.h, u, p.size, _ptr(p)) != 0:
            raise RuntimeError(f"oracle resync of unit {u} failed")
