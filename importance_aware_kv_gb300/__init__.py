"""Python binding of libhikv, the importance-aware budgeted KV-cache decode step.

Argument marshalling only: every function below takes torch CUDA tensors,
checks their dtype/shape/contiguity, and passes raw device pointers and the
current CUDA stream to the C ABI declared in ``include/hikv.h``.  All
arithmetic of the step runs in the library's CUDA kernels; there is no CPU
or PyTorch fallback, and importing this package fails loudly when
``libhikv.so`` has not been built (``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhikv.so")

HIKV_OK, HIKV_ERR_INVALID_ARG, HIKV_ERR_OUT_OF_MEMORY, HIKV_ERR_CAPACITY = 0, 1, 2, 3
HIKV_ERR_CUDA, HIKV_ERR_TIMEOUT, HIKV_ERR_STATE, HIKV_ERR_UNSUPPORTED = 4, 5, 6, 7
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "OUT_OF_MEMORY", 3: "CAPACITY", 4: "CUDA",
                5: "TIMEOUT", 6: "STATE", 7: "UNSUPPORTED"}
HIKV_F32, HIKV_BF16 = 0, 1

# every entry point of include/hikv.h
ABI_FUNCTIONS = ("hikv_create_cache", "hikv_destroy_cache", "hikv_append", "hikv_score_window",
                 "hikv_decode_step", "hikv_evict", "hikv_gather_retained", "hikv_get_lengths",
                 "hikv_device_status", "hikv_last_error", "hikv_score_window_noalloc",
                 "hikv_decode_step_fused", "hikv_kernel_launches", "hikv_budgets_pyramid",
                 "hikv_budgets_duo", "hikv_selftest_timeout", "hikv_element_rows",
                 "hikv_last_decode_config", "hikv_score_band", "hikv_read_floor",
                 "hikv_read_slot")


class HikvError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"hikv {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class hikv_config(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("num_sink", ctypes.c_int32), ("recent_window", ctypes.c_int32),
                ("budgets", ctypes.POINTER(ctypes.c_int32)), ("max_tokens", ctypes.c_int32),
                ("page_tokens", ctypes.c_int32), ("pool_pages", ctypes.c_int64),
                ("max_window_queries", ctypes.c_int32), ("scale", ctypes.c_float),
                ("pool_kernel", ctypes.c_int32), ("importance_mode", ctypes.c_int32),
                ("element_budget", ctypes.c_int32), ("band_scoring", ctypes.c_int32)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build the CUDA library first "
                          "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64, S = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int
    sig = {
        "hikv_create_cache": ([ctypes.POINTER(hikv_config), ctypes.POINTER(P)], S),
        "hikv_destroy_cache": ([P], S),
        "hikv_append": ([P, I32, I32, I32, P, P, P], S),
        "hikv_score_window": ([P, I32, I32, I32, P, P], S),
        "hikv_score_band": ([P, I32, I32, I32, P, P], S),
        "hikv_decode_step": ([P, I32, I32, P, P, P], S),
        "hikv_evict": ([P, I32, I32, P], S),
        "hikv_gather_retained": ([P, I32, I32, I32, P, P, P, P, P, P], S),
        "hikv_get_lengths": ([P, I32, I32, P], S),
        "hikv_device_status": ([P], S),
        "hikv_last_error": ([], ctypes.c_char_p),
        "hikv_score_window_noalloc": ([I32] * 8 + [ctypes.c_float, P, P, P, P], S),
        "hikv_decode_step_fused": ([P, I32, I32, P, P, P, P, I32, P], S),
        "hikv_kernel_launches": ([P], ctypes.c_int64),
        "hikv_element_rows": ([P, ctypes.POINTER(ctypes.c_int64)], ctypes.c_int),
        "hikv_last_decode_config": ([P, ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
        "hikv_budgets_pyramid": ([I32, I32, I32, I32, I32, P], S),
        "hikv_budgets_duo": ([I32, I32, P, I32, I32, I32, P], S),
        "hikv_selftest_timeout": ([P, I32, P], S),
        "hikv_read_floor": ([P, I64, I32, P, P], S),
        "hikv_read_slot": ([P, I32, I32, P, P, P, P], S),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


_lib = _load()


def _check(status: int):
    if status != HIKV_OK:
        raise HikvError(status, _lib.hikv_last_error().decode())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _raw_stream_fn():
    import torch
    return getattr(torch._C, "_cuda_getCurrentRawStream", None)


_RAW_STREAM = None


def _stream_of(t, stream):
    """The stream handle for a call: the given one, else the current stream of
    t's device (read without building a Stream object when torch allows)."""
    global _RAW_STREAM
    if stream is not None:
        return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    if _RAW_STREAM is None:
        _RAW_STREAM = _raw_stream_fn() or False
    if _RAW_STREAM:
        return _RAW_STREAM(t.device.index)
    return _stream(None).value


def _ptr_checked(t, name, dtype, shape):
    """One pass of the checks _dev makes, returning the device pointer as an int."""
    if not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if t.shape != shape:
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _dev(t, name, dtype=None, shape=None):
    import torch
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return ctypes.c_void_p(t.data_ptr())


@dataclass
class CacheConfig:
    num_layers: int
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    dtype: str                     # "f32" | "bf16"
    num_sink: int
    recent_window: int
    budgets: Sequence[int]         # [num_layers * num_kv_heads]
    max_tokens: int
    page_tokens: int = 64
    pool_pages: int = 0
    max_window_queries: int = 0
    scale: float = 0.0
    pool_kernel: int = 0           # SnapKV max-pool of the prompt scores (0/1: off)
    importance_mode: int = 0       # 0: H2O cumulative, 1: HiKV recent bank only
    element_budget: int = 0        # HiKV Stage II B2 (0 or head_dim: exact attention)
    band_scoring: int = 0          # 1: allow score_band (HiKV banded prefill scores)


def hikv_create_cache(cfg: CacheConfig) -> ctypes.c_void_p:
    b = np.ascontiguousarray(np.asarray(cfg.budgets, dtype=np.int32))
    c = hikv_config(cfg.num_layers, cfg.batch, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim,
                    HIKV_BF16 if cfg.dtype == "bf16" else HIKV_F32, cfg.num_sink,
                    cfg.recent_window, b.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                    cfg.max_tokens, cfg.page_tokens, cfg.pool_pages, cfg.max_window_queries,
                    cfg.scale, cfg.pool_kernel, cfg.importance_mode, cfg.element_budget,
                    cfg.band_scoring)
    h = ctypes.c_void_p()
    _check(_lib.hikv_create_cache(ctypes.byref(c), ctypes.byref(h)))
    return h


def hikv_destroy_cache(h) -> None:
    _check(_lib.hikv_destroy_cache(h))


def hikv_append(h, layer0: int, k, v, stream=None) -> None:
    nl, ntok = k.shape[0], k.shape[3]
    _check(_lib.hikv_append(h, layer0, nl, ntok, _dev(k, "k"), _dev(v, "v", k.dtype, k.shape),
                            _stream(stream)))


def hikv_score_window(h, layer0: int, q, stream=None) -> None:
    _check(_lib.hikv_score_window(h, layer0, q.shape[0], q.shape[3], _dev(q, "q"), _stream(stream)))


def hikv_decode_step(h, layer0: int, q, out, stream=None) -> None:
    _check(_lib.hikv_decode_step(h, layer0, q.shape[0], _dev(q, "q"),
                                 _dev(out, "out", q.dtype, q.shape), _stream(stream)))


def hikv_decode_step_fused(h, layer0: int, k, v, q, out, evict: bool = True, stream=None) -> None:
    _check(_lib.hikv_decode_step_fused(h, layer0, q.shape[0], _dev(k, "k"), _dev(v, "v", k.dtype, k.shape),
                                       _dev(q, "q", k.dtype), _dev(out, "out", q.dtype, q.shape),
                                       1 if evict else 0, _stream(stream)))


def budgets_pyramid(num_layers: int, num_kv_heads: int, avg: int, min_budget: int,
                    floor_budget: int = 1) -> np.ndarray:
    """PyramidKV per-layer budgets, [num_layers * num_kv_heads] int32 (C ABI)."""
    out = np.empty(num_layers * num_kv_heads, dtype=np.int32)
    _check(_lib.hikv_budgets_pyramid(num_layers, num_kv_heads, avg, min_budget, floor_budget, out.ctypes.data))
    return out


def budgets_duo(retrieval, full_budget: int, num_sink: int, recent_window: int) -> np.ndarray:
    """DuoAttention budgets from a [num_layers][num_kv_heads] retrieval-head mask (C ABI)."""
    m = np.ascontiguousarray(np.asarray(retrieval, dtype=bool), dtype=np.uint8)
    if m.ndim != 2:
        raise ValueError("retrieval must be [num_layers][num_kv_heads]")
    out = np.empty(m.size, dtype=np.int32)
    _check(_lib.hikv_budgets_duo(m.shape[0], m.shape[1], m.ctypes.data, full_budget, num_sink, recent_window,
                                 out.ctypes.data))
    return out


def hikv_evict(h, layer0: int, nlayers: int, stream=None) -> None:
    _check(_lib.hikv_evict(h, layer0, nlayers, _stream(stream)))


def hikv_gather_retained(h, layer0: int, nlayers: int, cap: int, lengths, positions, importance,
                         k_out=None, v_out=None, stream=None) -> None:
    import torch
    _check(_lib.hikv_gather_retained(
        h, layer0, nlayers, cap, _dev(lengths, "lengths", torch.int32),
        _dev(positions, "positions", torch.int32), _dev(importance, "importance", torch.float32),
        _dev(k_out, "k_out"), _dev(v_out, "v_out"), _stream(stream)))


def hikv_get_lengths(h, layer0: int, nlayers: int, units_per_layer: int) -> np.ndarray:
    out = np.empty(nlayers * units_per_layer, dtype=np.int32)
    _check(_lib.hikv_get_lengths(h, layer0, nlayers, out.ctypes.data))
    return out


def hikv_device_status(h) -> None:
    _check(_lib.hikv_device_status(h))


def hikv_score_window_noalloc(k, q, importance, num_q_heads: int, scale: float = 0.0,
                              stream=None) -> None:
    """Stateless prompt importance on caller-owned buffers (no allocation).

    k: [nl][B][Hkv][ntok][d], q: [nl][B][Hq][nq][d], importance: [nl][B][Hkv][ntok] fp32.
    """
    import torch
    nl, b, hkv, ntok, d = k.shape
    nq = q.shape[3]
    dt = HIKV_BF16 if k.dtype == torch.bfloat16 else HIKV_F32
    _check(_lib.hikv_score_window_noalloc(
        nl, b, num_q_heads, hkv, d, dt, ntok, nq, scale, _dev(k, "k"),
        _dev(q, "q", k.dtype, (nl, b, num_q_heads, nq, d)),
        _dev(importance, "importance", torch.float32, (nl, b, hkv, ntok)), _stream(stream)))


def read_floor(buf, ctas_per_sm: int = 2, sink=None, stream=None) -> None:
    """Measurement aid: one plain streaming read of a CUDA tensor's bytes
    (hikv_read_floor); `sink` a 4-byte CUDA tensor (allocated if None)."""
    import torch
    if sink is None:
        sink = torch.zeros(1, dtype=torch.int32, device=buf.device)
    _check(_lib.hikv_read_floor(_dev(buf, "buf"), buf.numel() * buf.element_size(), ctas_per_sm,
                                _dev(sink, "sink"), _stream(stream)))


def hikv_last_error() -> str:
    return _lib.hikv_last_error().decode()


class Cache:
    """Owning wrapper: one hikv cache on the current CUDA device."""

    def __init__(self, cfg: CacheConfig):
        self.cfg = cfg
        self._step_shapes = {}
        self.units_per_layer = cfg.batch * cfg.num_kv_heads
        self.units = cfg.num_layers * self.units_per_layer
        self.h = hikv_create_cache(cfg)

    def close(self):
        if getattr(self, "h", None) is not None and self.h.value:
            hikv_destroy_cache(self.h)
        self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # The C ABI takes raw pointers and cannot see buffer sizes: the binding
    # checks every tensor against the configuration before passing it on.
    def _dtype(self):
        import torch
        return torch.bfloat16 if self.cfg.dtype == "bf16" else torch.float32

    def _check_tensor(self, t, name, shape):
        if t.dtype != self._dtype():
            raise TypeError(f"{name} has dtype {t.dtype}, the cache holds {self._dtype()}")
        if tuple(t.shape) != tuple(shape):
            raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")

    def _layers(self, t, layer0):
        nl = t.shape[0] if t.dim() else 0
        if not (0 <= layer0 and nl >= 1 and layer0 + nl <= self.cfg.num_layers):
            raise ValueError(f"layers [{layer0}, {layer0 + nl}) outside [0, {self.cfg.num_layers})")
        return nl

    def append(self, k, v, layer0=0, stream=None):
        c = self.cfg
        nl = self._layers(k, layer0)
        ntok = k.shape[3] if k.dim() == 5 else -1
        self._check_tensor(k, "k", (nl, c.batch, c.num_kv_heads, ntok, c.head_dim))
        self._check_tensor(v, "v", tuple(k.shape))
        hikv_append(self.h, layer0, k, v, stream)

    def score_window(self, q, layer0=0, stream=None):
        c = self.cfg
        nl = self._layers(q, layer0)
        nq = q.shape[3] if q.dim() == 5 else -1
        self._check_tensor(q, "q", (nl, c.batch, c.num_q_heads, nq, c.head_dim))
        hikv_score_window(self.h, layer0, q, stream)

    def score_band(self, q, band, layer0=0, stream=None):
        """HiKV prefill initialisation: q [nl][B][Hq][n][d] holds the queries
        of every held position; each token's score grows by its attention
        column over the band of queries from its own position."""
        c = self.cfg
        nl = self._layers(q, layer0)
        n = q.shape[3] if q.dim() == 5 else -1
        self._check_tensor(q, "q", (nl, c.batch, c.num_q_heads, n, c.head_dim))
        lens = self.lengths(layer0, nl)
        if lens.size and int(lens[0]) != n:
            raise ValueError(f"q holds {n} positions, the units hold {int(lens[0])} tokens")
        _check(_lib.hikv_score_band(self.h, layer0, nl, int(band), _dev(q, "q"), _stream(stream)))

    def decode_step(self, q, out, layer0=0, stream=None):
        c = self.cfg
        nl = self._layers(q, layer0)
        self._check_tensor(q, "q", (nl, c.batch, c.num_q_heads, c.head_dim))
        self._check_tensor(out, "out", tuple(q.shape))
        hikv_decode_step(self.h, layer0, q, out, stream)

    def selftest_timeout(self, limit_us: int = 20000, stream=None):
        """Enqueue a kernel whose bounded wait runs out (see hikv.h)."""
        _check(_lib.hikv_selftest_timeout(self.h, limit_us, _stream(stream)))

    def kernel_launches(self) -> int:
        """Kernels this cache has launched so far (host counter)."""
        return int(_lib.hikv_kernel_launches(self.h))

    def last_decode_config(self) -> list:
        """The cluster-kernel launches of the latest decode call: units,
        cluster size, clusters and logits placement of each."""
        out = (ctypes.c_int32 * 8)()
        _check(_lib.hikv_last_decode_config(self.h, out))
        return [{"units": out[4 * i], "cluster_size": out[4 * i + 1], "clusters": out[4 * i + 2],
                 "smem_logits": bool(out[4 * i + 3])} for i in range(2) if out[4 * i + 1] > 0]

    def element_rows(self) -> int:
        """V rows the HiKV Stage II decode steps have read so far (synchronous)."""
        r = ctypes.c_int64()
        _check(_lib.hikv_element_rows(self.h, ctypes.byref(r)))
        return int(r.value)

    def step(self, k, v, q, out, evict=True, layer0=0, stream=None):
        """append + decode_step (+ evict) as one call (fused into the attention
        kernel in the steady state).
        The per-step call of a decode loop: each tensor is checked once."""
        import torch
        nl = self._layers(q, layer0)
        shapes = self._step_shapes.get(nl)
        if shapes is None:
            c = self.cfg
            shapes = (torch.Size((nl, c.batch, c.num_kv_heads, 1, c.head_dim)),
                      torch.Size((nl, c.batch, c.num_q_heads, c.head_dim)))
            self._step_shapes[nl] = shapes
        dt = self._dtype()
        kp = _ptr_checked(k, "k", dt, shapes[0])
        vp = _ptr_checked(v, "v", dt, shapes[0])
        qp = _ptr_checked(q, "q", dt, shapes[1])
        op = _ptr_checked(out, "out", dt, shapes[1])
        _check(_lib.hikv_decode_step_fused(self.h, layer0, nl, kp, vp, qp, op, 1 if evict else 0,
                                           _stream_of(q, stream)))

    def evict(self, layer0=0, nlayers=None, stream=None):
        hikv_evict(self.h, layer0, self.cfg.num_layers if nlayers is None else nlayers, stream)

    def lengths(self, layer0=0, nlayers=None) -> np.ndarray:
        nl = self.cfg.num_layers - layer0 if nlayers is None else nlayers
        return hikv_get_lengths(self.h, layer0, nl, self.units_per_layer)

    def gather(self, layer0=0, nlayers=None, cap=None, with_kv=False, stream=None):
        """Retained state of the layers as CUDA tensors (positions ascending)."""
        import torch
        nl = self.cfg.num_layers - layer0 if nlayers is None else nlayers
        nu = nl * self.units_per_layer
        if cap is None:
            cap = max(1, int(self.lengths(layer0, nl).max()))
        dev = torch.device("cuda", torch.cuda.current_device())
        lengths = torch.empty(nu, dtype=torch.int32, device=dev)
        positions = torch.empty(nu, cap, dtype=torch.int32, device=dev)
        importance = torch.empty(nu, cap, dtype=torch.float32, device=dev)
        k_out = v_out = None
        if with_kv:
            dt = torch.bfloat16 if self.cfg.dtype == "bf16" else torch.float32
            k_out = torch.empty(nu, cap, self.cfg.head_dim, dtype=dt, device=dev)
            v_out = torch.empty_like(k_out)
        hikv_gather_retained(self.h, layer0, nl, cap, lengths, positions, importance, k_out, v_out,
                             stream)
        return lengths, positions, importance, k_out, v_out

    def read_slot(self, unit: int, slot: int):
        """Raw contents of one slot (diagnostic, synchronous): K row, V row
        (numpy, bf16 as uint16 bit patterns), importance, position."""
        c = self.cfg
        dt = np.uint16 if c.dtype == "bf16" else np.float32
        k = np.empty(c.head_dim, dt)
        vv = np.empty(c.head_dim, dt)
        imp = ctypes.c_float()
        pos = ctypes.c_int32()
        _check(_lib.hikv_read_slot(self.h, unit, slot, k.ctypes.data, vv.ctypes.data, ctypes.byref(imp),
                                   ctypes.byref(pos)))
        return k, vv, imp.value, pos.value

    def device_status(self):
        hikv_device_status(self.h)
