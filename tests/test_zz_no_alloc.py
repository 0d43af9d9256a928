"""GPU tests of hikv_score_window_noalloc, the entry point for callers that
cannot allocate device memory (e.g. a plugin inside an inference engine that
owns all device allocations).

It is called through the C ABI on buffers the test owns and checked two
ways, each on two calls in a row with different inputs (the static scratch
keeps the previous call's contents):
  * against what the cache-based entry points (hikv_append +
    hikv_score_window) leave as importance, at the importance tolerance of
    the parity tests, with 32 to 256 query vectors per unit (one to four
    64-vector blocks of the kernels' query loop) and token counts that are
    multiples of neither its 32-token tiles nor its 1024-token chunks;
  * against the CPU oracle's append + window scoring directly, so that a
    misreading the two CUDA paths might share cannot pass.
This file is collected last so that, if it fails, a run stopping at the
first failure has already run every other test.
"""
import ctypes
from fractions import Fraction

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

IMP_REL, IMP_ABS_FRAC = 1e-4, 1e-6


@pytest.fixture(scope="module")
def hk():
    from tests.conftest import build_native
    build_native()
    import importance_aware_kv_gb300 as hk
    return hk


def _noalloc(hk, k, q, out, hq, scale=0.0):
    nl, b, hkv, ntok, d = k.shape
    nq = q.shape[3]
    return hk._lib.hikv_score_window_noalloc(nl, b, hq, hkv, d,
                                             hk.HIKV_BF16 if k.dtype == torch.bfloat16 else hk.HIKV_F32,
                                             ntok, nq, ctypes.c_float(scale), ctypes.c_void_p(k.data_ptr()),
                                             ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _reference_importance(hk, k, v, q, hq, scale):
    """Importance left by the cache entry points: append the prompt, score the window."""
    nl, b, hkv, ntok, d = k.shape
    cfg = hk.CacheConfig(nl, b, hq, hkv, d, "bf16" if k.dtype == torch.bfloat16 else "f32",
                         0, 0, [max(1, ntok)] * (nl * hkv), ntok, max_window_queries=q.shape[3],
                         scale=scale)
    c = hk.Cache(cfg)
    c.append(k, v)
    c.score_window(q)
    lengths, positions, importance, _, _ = c.gather()
    torch.cuda.synchronize()
    assert torch.all(lengths == ntok)
    assert torch.equal(positions, torch.arange(ntok, dtype=torch.int32, device=k.device).expand_as(positions))
    c.close()
    return importance.view(nl, b, hkv, ntok)


def _check_close(got, want):
    g = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    w = want.double().cpu().numpy() if isinstance(want, torch.Tensor) else np.asarray(want, np.float64)
    tol = IMP_REL * np.abs(w) + IMP_ABS_FRAC * np.abs(w).max()
    assert np.all(np.abs(g - w) <= tol), float(np.max(np.abs(g - w) - tol))


@pytest.mark.parametrize("dtype,d,hq,hkv,nq,ntok", [
    (torch.bfloat16, 128, 8, 2, 16, 2500),     # G = 4: 64 query vectors, one block
    (torch.float32, 64, 4, 2, 16, 2500),       # G = 2: 32 vectors
    (torch.bfloat16, 128, 32, 8, 32, 2500),    # G = 4: 128 vectors, two blocks
    (torch.bfloat16, 128, 64, 8, 32, 1111),    # G = 8: 256 vectors, four blocks
    (torch.float32, 128, 16, 2, 24, 1029),     # G = 8: 192 vectors, three blocks, fp32
], ids=["g4_64v", "f32_g2_32v", "g4_128v", "g8_256v", "f32_g8_192v"])
def test_noalloc_window_scoring_matches_cache_path(hk, dtype, d, hq, hkv, nq, ntok):
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev).manual_seed(1234)
    nl, b = 2, 2
    out = torch.empty(nl, b, hkv, ntok, dtype=torch.float32, device=dev)
    for call in range(2):   # two calls in a row, different inputs
        k = torch.randn(nl, b, hkv, ntok, d, generator=gen, device=dev).to(dtype)
        v = torch.randn(nl, b, hkv, ntok, d, generator=gen, device=dev).to(dtype)
        q = (torch.randn(nl, b, hq, nq, d, generator=gen, device=dev) * (1 + call)).to(dtype)
        out.fill_(float("nan"))
        st = _noalloc(hk, k, q, out, hq)
        assert st == hk.HIKV_OK, hk.hikv_last_error()
        want = _reference_importance(hk, k, v, q, hq, 0.0)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        _check_close(out, want)
        # every query adds G units of softmax mass
        assert abs(float(out.double().sum()) - nl * b * hkv * (hq // hkv) * nq) < 1e-3 * nl * b * hq * nq


@pytest.mark.parametrize("dtype,d,hq,hkv,nq,ntok", [
    (torch.bfloat16, 128, 8, 2, 16, 1500),     # 64 vectors
    (torch.bfloat16, 128, 32, 4, 32, 1100),    # G = 8: 256 vectors
    (torch.float32, 64, 4, 1, 20, 700),        # 80 vectors, two blocks, fp32
], ids=["bf16_64v", "bf16_256v", "f32_80v"])
def test_noalloc_window_scoring_matches_oracle(hk, dtype, d, hq, hkv, nq, ntok):
    import oracle
    dev = torch.device("cuda")
    rng = np.random.default_rng(77)
    nl, b = 1, 2
    out = torch.empty(nl, b, hkv, ntok, dtype=torch.float32, device=dev)
    for call in range(2):
        k = torch.from_numpy(rng.standard_normal((nl, b, hkv, ntok, d)).astype(np.float32) * (1 + call)).to(dev)
        q = torch.from_numpy(rng.standard_normal((nl, b, hq, nq, d)).astype(np.float32)).to(dev)
        k, q = k.to(dtype).contiguous(), q.to(dtype).contiguous()
        out.fill_(float("nan"))
        assert _noalloc(hk, k, q, out, hq) == hk.HIKV_OK, hk.hikv_last_error()
        torch.cuda.synchronize()
        ora = oracle.Oracle(nl, b, hq, hkv, d, 0, 0, np.full(nl * hkv, ntok), threads=8)
        kf, qf = k.float().cpu().numpy(), q.float().cpu().numpy()   # bf16 values widened exactly
        ora.append(0, kf, np.zeros_like(kf))
        ora.score_window(0, qf)
        got = out.cpu().numpy()
        for bb in range(b):
            for g in range(hkv):
                pos, imp = ora.state(ora.unit(0, bb, g))
                assert np.array_equal(pos, np.arange(ntok))
                _check_close(got[0, bb, g], imp)


def test_noalloc_rejects_oversized_scratch(hk):
    dev = torch.device("cuda")
    k = torch.zeros(1, 1, 8, 64, 64, device=dev)
    q = torch.zeros(1, 1, 64, 32, 64, device=dev)
    out = torch.empty(1, 1, 8, 64, device=dev)
    # 8 units x 1 chunk x (8 * 32) query vectors x 2 = 4096 floats: fits.
    # Zero keys: query at position p spreads 1/(p + 1) over tokens 0..p, so
    # token j gets G * sum over the 32 query positions p >= j of 1/(p + 1).
    hk.hikv_score_window_noalloc(k, q, out, num_q_heads=64)
    torch.cuda.synchronize()
    G, ntok, nq = 8, 64, 32
    want = [float(G * sum(Fraction(1, p + 1) for p in range(max(j, ntok - nq), ntok))) for j in range(ntok)]
    got = out.cpu().numpy()
    for g in range(8):
        _check_close(got[0, 0, g], want)
    # 64 layers x 8 KV heads x ceil(8192/1024) chunks x 256 query vectors x 2
    # = 2,097,152 floats > the 1,048,576 of the static scratch: rejected on the
    # host before anything runs (the small buffers are never touched)
    st = hk._lib.hikv_score_window_noalloc(64, 1, 64, 8, 64, hk.HIKV_F32, 8192, 32, ctypes.c_float(0.0),
                                           ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(q.data_ptr()),
                                           ctypes.c_void_p(out.data_ptr()),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == hk.HIKV_ERR_INVALID_ARG
    assert "static scratch" in hk.hikv_last_error()
