"""Debug mode: parity with dead slots poisoned.

With HIKV_DEBUG=1 set when a cache is created, the pool starts as NaN, every
slot an eviction vacates (the fused move's source, a compaction's upper
slots) and every page returned to a shared pool is overwritten with NaN
rows, NaN importance and position -1, and slot indices taken from data are
range-checked and reported through the device error word.  The parity runs
below then fail if any kernel ever reads a dead slot: its NaN would reach an
output or an importance, which the comparisons reject, and a range error
makes device_status raise.  This stands in for a memory sanitizer, which is
closed on this pool.
"""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from tests.conftest import build_native
    build_native()
    import oracle
    oracle._load()
    W._load()


@pytest.fixture
def debug(monkeypatch):
    monkeypatch.setenv("HIKV_DEBUG", "1")


def _run(w, fused=False, **kw):
    from tests.lockstep import Lockstep
    ls = Lockstep(w, **kw)
    ls.prefill()
    rep = ls.decode(fused=fused)
    ls.cache.close()
    return rep


SMALL = W.Workload(100, "small", 2, 2, 8, 2, 128, "bf16", 300, 40, 96, 4, 16, 1, "bernoulli5x3")
FUSED = pytest.mark.parametrize("fused", [False, True], ids=["3calls", "fused"])


@FUSED
def test_debug_tiny_fp32_workload(debug, fused):
    rep = _run(W.WORKLOADS[0], fused=fused)
    assert rep.evictions_checked == 2 * (1 + 64)


@FUSED
def test_debug_llama3_8b_layer(debug, fused):
    rep = _run(W.WORKLOADS[1], fused=fused)
    assert rep.evictions_checked == 64 * (1 + 256)


@FUSED
@pytest.mark.parametrize("small_mode", [2, 0])
def test_debug_ragged_budgets(debug, fused, small_mode):
    b = np.array([40, 96, 33, 200], dtype=np.int32)
    _run(SMALL.with_(sink=1, window=16), budgets=b, fused=fused, small_mode=small_mode)


@FUSED
@pytest.mark.parametrize("cs", [None, 3])
def test_debug_group_of_eight_partial_tiles(debug, fused, cs):
    # G = 8 with partial tiles: their rows outside the CTA's slots (chunk
    # edges, the ragged tail) hold NaN in this mode, and must be skipped (or,
    # on the tensor-core path, zeroed before the mma) rather than weighted by 0
    _run(SMALL.with_(hq=16, hkv=2, prompt=700, budget=250, window=24), fused=fused, cs=cs)


def test_debug_batched_eviction_compaction(debug):
    _run(SMALL.with_(evict_every=16, steps=48, budget=120, window=20), fused=True)


@FUSED
def test_debug_shared_page_pool(debug, fused):
    # pages return to the free stack poisoned and are handed out again
    _run(SMALL, pool_pages=SMALL.units * 20, fused=fused, page_tokens=16)   # 19 pages of prompt, 22 for home pages


def test_debug_stage2_and_band_prefill(debug):
    _run(SMALL.with_(prompt=900, budget=300), element_budget=64, fused=True)
    _run(SMALL.with_(sink=0, window=48, budget=96), importance_mode=1, prefill_band=48, fused=True)


@pytest.mark.parametrize("debug_on", [True, False])
def test_vacated_slot_is_poisoned_only_in_debug_mode(monkeypatch, debug_on):
    import importance_aware_kv_gb300 as hk
    if debug_on:
        monkeypatch.setenv("HIKV_DEBUG", "1")
    else:
        monkeypatch.delenv("HIKV_DEBUG", raising=False)
    dev = torch.device("cuda")
    B, n0 = 16, 20
    c = hk.Cache(hk.CacheConfig(1, 1, 4, 1, 64, "f32", 1, 4, [B], 64))
    gen = torch.Generator(device=dev).manual_seed(3)
    k = torch.randn(1, 1, 1, n0, 64, generator=gen, device=dev)
    c.append(k, torch.randn(1, 1, 1, n0, 64, generator=gen, device=dev))
    q = torch.randn(1, 1, 4, 8, 64, generator=gen, device=dev)
    c.score_window(q)
    c.evict()                               # compaction: slots 16..19 vacated
    k1 = torch.randn(1, 1, 1, 1, 64, generator=gen, device=dev)
    qd = torch.randn(1, 1, 4, 64, generator=gen, device=dev)
    c.step(k1, k1.clone(), qd, torch.empty_like(qd))   # one launch: new token in slot 16, moved into the victim's
    torch.cuda.synchronize()
    kr, vr, imp, pos = c.read_slot(0, B)    # the new token's slot, vacated by the move
    kl, vl, impl, posl = c.read_slot(0, 3)  # a live slot
    assert np.all(np.isfinite(kl)) and np.isfinite(impl) and posl >= 0
    if debug_on:
        assert np.all(np.isnan(kr)) and np.all(np.isnan(vr)) and np.isnan(imp) and pos == -1
        for s in range(B + 1, n0):          # vacated by the compaction
            ks, _, imps, poss = c.read_slot(0, s)
            assert np.all(np.isnan(ks)) and np.isnan(imps) and poss == -1
        ke, _, impe, pose = c.read_slot(0, 40)   # never written: NaN from the start
        assert np.all(np.isnan(ke)) and np.isnan(impe) and pose == -1
    else:
        assert np.all(np.isfinite(kr)) and pos >= 0   # stale but untouched without the mode
    c.device_status()
    c.close()
