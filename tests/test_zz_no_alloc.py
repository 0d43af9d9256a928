"""GPU test of hikv_score_window_noalloc, the entry point for callers that
cannot allocate device memory (e.g. a plugin inside an inference engine that
owns all device allocations).

It is called through the C ABI on buffers the test owns and checked against
what the cache-based entry points (hikv_append + hikv_score_window) leave as
importance, within the importance tolerance used by the parity tests, on two
calls in a row with different inputs (the static scratch keeps the previous
call's contents).  This file is collected last so that, if it fails, a run
stopping at the first failure has already run every other test.
"""
import ctypes

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
    g = got.double().cpu().numpy()
    w = want.double().cpu().numpy()
    tol = IMP_REL * np.abs(w) + IMP_ABS_FRAC * np.abs(w).max()
    assert np.all(np.abs(g - w) <= tol), float(np.max(np.abs(g - w) - tol))


@pytest.mark.parametrize("dtype,d,hq,hkv", [(torch.bfloat16, 128, 8, 2), (torch.float32, 64, 4, 2)])
def test_noalloc_window_scoring_matches_cache_path(hk, dtype, d, hq, hkv):
    dev = torch.device("cuda")
    gen = torch.Generator(device=dev).manual_seed(1234)
    nl, b, ntok, nq = 2, 2, 2500, 16
    out = torch.empty(nl, b, hkv, ntok, dtype=torch.float32, device=dev)
    for call in range(2):   # two calls in a row, different inputs
        k = torch.randn(nl, b, hkv, ntok, d, generator=gen, device=dev).to(dtype)
        v = torch.randn(nl, b, hkv, ntok, d, generator=gen, device=dev).to(dtype)
        q = (torch.randn(nl, b, hq, nq, d, generator=gen, device=dev) * (1 + call)).to(dtype)
        out.fill_(float("nan"))
        lib = hk._lib
        st = lib.hikv_score_window_noalloc(nl, b, hq, hkv, d,
                                           hk.HIKV_BF16 if dtype == torch.bfloat16 else hk.HIKV_F32,
                                           ntok, nq, ctypes.c_float(0.0), ctypes.c_void_p(k.data_ptr()),
                                           ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == hk.HIKV_OK, hk.hikv_last_error()
        want = _reference_importance(hk, k, v, q, hq, 0.0)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        _check_close(out, want)
        # every query adds G units of softmax mass
        assert abs(float(out.double().sum()) - nl * b * hkv * (hq // hkv) * nq) < 1e-3 * nl * b * hq * nq


def test_noalloc_rejects_oversized_scratch(hk):
    dev = torch.device("cuda")
    k = torch.zeros(1, 1, 8, 64, 64, device=dev)
    q = torch.zeros(1, 1, 64, 32, 64, device=dev)
    out = torch.empty(1, 1, 8, 64, device=dev)
    # 8 units x 1 chunk x (8 * 32) query vectors x 2 = 4096 floats: fits
    hk.hikv_score_window_noalloc(k, q, out, num_q_heads=64)
    # 64 layers x 8 KV heads x ceil(8192/1024) chunks x 256 query vectors x 2
    # = 2,097,152 floats > the 1,048,576 of the static scratch: rejected on the
    # host before anything runs (the small buffers are never touched)
    st = hk._lib.hikv_score_window_noalloc(64, 1, 64, 8, 64, hk.HIKV_F32, 8192, 32, ctypes.c_float(0.0),
                                           ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(q.data_ptr()),
                                           ctypes.c_void_p(out.data_ptr()),
                                           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == hk.HIKV_ERR_INVALID_ARG
    assert "static scratch" in hk.hikv_last_error()
