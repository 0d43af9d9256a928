"""Failure detection on the GPU without a GPU fault.

* A device wait that runs out: hikv_selftest_timeout enqueues a kernel whose
  bounded wait on a barrier nothing arrives on gives up after 20 ms; the
  device error word reports TIMEOUT with its site, and the context stays
  usable (a decode step right after runs and matches the oracle).
* An allocation that fails inside create (injected on the host with
  HIKV_FAULT_ALLOC_AT): create reports OUT_OF_MEMORY and frees what it had.
* Misuse the binding catches before any launch: wrong dtype or shape, a
  closed cache.
No test traps, faults or hangs the GPU.
"""
import os

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hk():
    from tests.conftest import build_native
    build_native()
    import importance_aware_kv_gb300 as hk
    import oracle
    oracle._load()
    W._load()
    return hk


def test_bounded_wait_timeout_is_reported_and_the_context_stays_usable(hk):
    from tests.lockstep import Lockstep
    w = W.WORKLOADS[0].with_(steps=6)
    ls = Lockstep(w)
    ls.prefill()
    ls.cache.selftest_timeout(20000)                 # 20 ms, then the kernel returns
    with pytest.raises(hk.HikvError) as ei:
        ls.cache.device_status()
    assert ei.value.status == hk.HIKV_ERR_TIMEOUT
    assert "self-test" in str(ei.value)
    ls.cache.device_status()                         # reported once, then cleared
    rep = ls.decode(fused=True)                      # the context still computes correctly
    assert rep.outputs_checked > 0
    ls.cache.close()


def test_selftest_rejects_bad_limits(hk):
    c = hk.Cache(hk.CacheConfig(1, 1, 2, 1, 64, "f32", 0, 0, [8], 16))
    for bad in (0, -5, 2000001):
        with pytest.raises(hk.HikvError) as ei:
            c.selftest_timeout(bad)
        assert ei.value.status == hk.HIKV_ERR_INVALID_ARG
    c.close()


@pytest.mark.parametrize("at", [1, 2, 5, 12, 19])
def test_injected_allocation_failure_cleans_up(hk, at):
    cfg = hk.CacheConfig(2, 2, 4, 2, 64, "bf16", 2, 8, [32] * 4, 256)
    free0 = torch.cuda.mem_get_info()[0]
    os.environ["HIKV_FAULT_ALLOC_AT"] = str(at)
    try:
        with pytest.raises(hk.HikvError) as ei:
            hk.Cache(cfg)
        assert ei.value.status == hk.HIKV_ERR_OUT_OF_MEMORY
    finally:
        os.environ.pop("HIKV_FAULT_ALLOC_AT", None)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] >= free0 - (8 << 20)   # nothing of the failed create is kept
    c = hk.Cache(cfg)                                            # and a normal create still works
    c.close()


def test_binding_rejects_misuse_before_any_launch(hk):
    cfg = hk.CacheConfig(1, 2, 4, 2, 64, "bf16", 2, 8, [32, 32], 128)
    c = hk.Cache(cfg)
    dev = torch.device("cuda")
    n0 = c.kernel_launches()
    with pytest.raises(TypeError):
        c.append(torch.zeros(1, 2, 2, 4, 64, device=dev), torch.zeros(1, 2, 2, 4, 64, device=dev))  # fp32
    with pytest.raises(ValueError):
        k = torch.zeros(1, 2, 3, 4, 64, device=dev, dtype=torch.bfloat16)     # 3 KV heads, not 2
        c.append(k, k.clone())
    with pytest.raises(ValueError):
        q = torch.zeros(2, 2, 4, 64, device=dev, dtype=torch.bfloat16)       # 2 layers, cache has 1
        c.decode_step(q, q.clone())
    # the per-step call checks each tensor once, as thoroughly
    k1 = torch.zeros(1, 2, 2, 1, 64, device=dev, dtype=torch.bfloat16)
    q1 = torch.zeros(1, 2, 4, 64, device=dev, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        c.step(k1, k1.clone(), q1.float(), q1.clone())                          # fp32 q
    with pytest.raises(ValueError):
        c.step(k1[:, :, :1], k1.clone(), q1, q1.clone())                        # k has 1 KV head
    with pytest.raises(ValueError):
        c.step(k1, k1.clone(), q1, torch.zeros(1, 2, 64, 4, device=dev, dtype=torch.bfloat16).transpose(2, 3))
    with pytest.raises(TypeError):
        c.step(k1.cpu(), k1.clone(), q1, q1.clone())                            # host tensor
    assert c.kernel_launches() == n0
    c.close()
    with pytest.raises(hk.HikvError) as ei:                  # use after close
        c.evict()
    assert ei.value.status == hk.HIKV_ERR_INVALID_ARG
