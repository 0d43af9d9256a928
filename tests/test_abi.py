"""The C-ABI library loads here (no GPU) and exports every declared entry
point; host-side argument checks answer before any CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def hk():
    from tests.conftest import build_native
    build_native()
    import importance_aware_kv_gb300 as hk
    return hk


def header_functions():
    src = open(os.path.join(ROOT, "include", "hikv.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hikv_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(hk):
    names = header_functions()
    assert len(names) >= 10
    lib = ctypes.CDLL(hk.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/hikv.h but not exported"
    assert sorted(hk.ABI_FUNCTIONS) == names


def _cfg(hk, **kw):
    base = dict(num_layers=1, batch=1, num_q_heads=4, num_kv_heads=2, head_dim=64, dtype="f32",
                num_sink=4, recent_window=8, budgets=[32, 32], max_tokens=128)
    base.update(kw)
    return hk.CacheConfig(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(num_q_heads=6, num_kv_heads=4, budgets=[32] * 4), 1),   # Hq % Hkv
    (dict(num_q_heads=12, num_kv_heads=4, budgets=[32] * 4), 7),  # G = 3
    (dict(head_dim=96), 7),
    (dict(budgets=[8, 32]), 1),                                   # budget < S + W
    (dict(page_tokens=48), 1),
    (dict(max_tokens=0), 1),
    (dict(num_sink=-1), 1),
    (dict(pool_kernel=-1), 1),
    (dict(pool_kernel=65), 1),                                    # SnapKV kernel above 64
    (dict(importance_mode=2), 1),
    (dict(element_budget=-1), 1),
    (dict(element_budget=129), 1),                                # HiKV Stage II B2 above head_dim
])
def test_create_rejects_bad_config_on_host(hk, kw, status):
    with pytest.raises(hk.HikvError) as ei:
        hk.hikv_create_cache(_cfg(hk, **kw))
    assert ei.value.status == status


def test_null_and_range_errors_need_no_device(hk):
    lib = hk._lib
    assert lib.hikv_append(None, 0, 1, 1, None, None, None) == hk.HIKV_ERR_INVALID_ARG
    assert lib.hikv_decode_step(None, 0, 1, None, None, None) == hk.HIKV_ERR_INVALID_ARG
    assert lib.hikv_evict(None, 0, 1, None) == hk.HIKV_ERR_INVALID_ARG
    assert lib.hikv_destroy_cache(None) == hk.HIKV_OK
    assert "layer range" in hk.hikv_last_error() or hk.hikv_last_error() == ""


def test_create_without_device_reports_cuda(hk):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    with pytest.raises(hk.HikvError) as ei:
        hk.hikv_create_cache(_cfg(hk))
    assert ei.value.status == hk.HIKV_ERR_CUDA


def test_budget_schedules_match_the_oracle(hk):
    from oracle import budgets
    rng = np.random.default_rng(7)
    for L in (1, 2, 3, 5, 32, 80):
        for hkv in (1, 8):
            for avg, mn, fl in ((1024, 128, 68), (100, 20, 1), (10, 9, 1), (2048, 0, 260), (7, 7, 1)):
                np.testing.assert_array_equal(hk.budgets_pyramid(L, hkv, avg, mn, fl),
                                              budgets.pyramid(L, hkv, avg, mn, fl))
        mask = rng.random((L, 8)) < 0.3
        np.testing.assert_array_equal(hk.budgets_duo(mask, 4096, 4, 256), budgets.duo(mask, 4096, 4, 256))


def test_budget_schedules_reject_bad_arguments(hk):
    for args in ((0, 1, 10, 5, 1), (2, 1, 10, 11, 1), (2, 1, 0, 0, 1), (2, 1, 10, -1, 1), (2, 1, 10, 5, -1)):
        with pytest.raises(hk.HikvError) as ei:
            hk.budgets_pyramid(*args)
        assert ei.value.status == hk.HIKV_ERR_INVALID_ARG
    with pytest.raises(hk.HikvError):
        hk.budgets_duo(np.ones((2, 2), bool), 100, 64, 64)   # full budget below S + W
