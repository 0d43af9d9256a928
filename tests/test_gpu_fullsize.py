"""GPU parity at the full sizes of the three large workloads.

The GPU runs every layer of each workload with all-layer calls (the launch
configuration of the benchmark); the CPU oracle checks sampled layers in
lockstep (the 70B workload through the fused single-launch step, the ragged
one through both paths): retained sets after every eviction (near-ties < 1e-6 relative
allowed, then resynced), importance, and the outputs of every step.
"""
import pytest

import workloads as W

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def built():
    from tests.conftest import build_native
    build_native()


def _run(w, fused=False, **kw):
    from tests.lockstep import Lockstep
    ls = Lockstep(w, **kw)
    ls.prefill()
    rep = ls.decode(fused=fused)
    print(f"{w.name}: evictions {rep.evictions_checked}, near-ties {rep.near_tie_swaps}, "
          f"max out err {rep.max_out_err:.4g}, max imp rel err {rep.max_imp_err_rel:.3g}")
    if ls.twin is not None:
        t = ls.twin.rep
        print(f"  full cache twin: outputs {t.outputs_checked}, max out err {t.max_out_err:.4g}, "
              f"max imp rel err {t.max_imp_err_rel:.3g}")
        ls.twin.cache.close()
    ls.cache.close()
    return rep


def test_32layer_ctx32k_evict_every_16():
    rep = _run(W.WORKLOADS[2], sample_layers=[0, 31])
    assert rep.evictions_checked == 2 * 32 * (1 + 128 // 16)


@pytest.mark.parametrize("fused", [False, True], ids=["3calls", "fused"])
def test_headkv_dirichlet_ragged_budgets(fused):
    rep = _run(W.WORKLOADS[3], fused=fused, sample_layers=[5])
    assert rep.evictions_checked == 128 * (1 + 128)


def test_llama3_70b_ctx128k_with_full_cache_twin():
    # every step is the single append+decode+evict launch
    rep = _run(W.WORKLOADS[4], fused=True, sample_layers=[0, 79], full_twin_layers=[40])
    assert rep.evictions_checked == 2 * 8 * (1 + 64)
