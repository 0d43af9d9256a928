"""GPU parity: the CUDA path against the CPU oracle, through the C ABI.

Small workloads run every unit and every step in lockstep with the oracle;
edge cases cover cluster splits, ragged tails, degenerate sink/window
settings, group sizes, dtypes, the long-chunk (global logits) path, the
exact tie rule, and host-detected errors.
"""
import os

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


def _ls(w, **kw):
    from tests.lockstep import Lockstep
    return Lockstep(w, **kw)


def _run(w, fused=False, **kw):
    ls = _ls(w, **kw)
    ls.prefill()
    rep = ls.decode(fused=fused)
    ls.cache.close()
    return rep


# fused: each decode step is the single append+decode+evict call
FUSED = pytest.mark.parametrize("fused", [False, True], ids=["3calls", "fused"])


@FUSED
def test_tiny_fp32_workload_full_lockstep(fused):
    rep = _run(W.WORKLOADS[0], fused=fused)
    assert rep.evictions_checked == 2 * (1 + 64)
    assert rep.max_out_err <= 1.0


@FUSED
def test_llama3_8b_layer_full_lockstep(fused):
    rep = _run(W.WORKLOADS[1], fused=fused)
    assert rep.evictions_checked == 64 * (1 + 256)
    assert rep.max_out_ulps <= 1.0
    print("near-tie swaps", rep.near_tie_swaps, "max bf16 err", rep.max_out_err, "max ulps", rep.max_out_ulps,
          "elements over 1 ulp (below the floor)", rep.bf16_over_1ulp, "max imp rel err", rep.max_imp_err_rel)


SMALL = W.Workload(100, "small", 2, 2, 8, 2, 128, "bf16", 300, 40, 96, 4, 16, 1, "bernoulli5x3")


@FUSED
@pytest.mark.parametrize("cs", [1, 2, 4, 8, 16])
def test_cluster_split_sizes(cs, fused):
    _run(SMALL, cs=cs, fused=fused)


@pytest.mark.parametrize("kw", [
    dict(sink=0, window=0, budget=40),
    dict(sink=0, window=12, budget=12),          # budget = S + W (StreamingLLM)
    dict(sink=3, window=0, budget=3),
    dict(sink=4, window=16, budget=20),
    dict(sink=1, window=5, budget=77),           # ragged tile tails
])
@FUSED
def test_degenerate_sink_window(kw, fused):
    _run(SMALL.with_(**kw), fused=fused)


@pytest.mark.parametrize("shape", [
    dict(hq=2, hkv=2, d=64, dtype="f32"),        # G = 1
    dict(hq=16, hkv=2, d=128, dtype="bf16"),     # G = 8
    dict(hq=8, hkv=2, d=128, dtype="f32"),
    dict(hq=8, hkv=2, d=64, dtype="bf16"),
])
@FUSED
def test_group_sizes_and_dtypes(shape, fused):
    _run(SMALL.with_(**shape), fused=fused)


@FUSED
def test_evict_every_16_batched_select(fused):
    # fused: 15 single-launch steps without eviction, then 16 over budget,
    # which the fused call hands to the three separate calls
    _run(SMALL.with_(evict_every=16, steps=48, budget=120, window=20), fused=fused)


@FUSED
@pytest.mark.parametrize("small_mode", [2, 0, 1], ids=["warp_per_unit", "clusters_only", "auto"])
def test_ragged_budgets(fused, small_mode):
    # ragged budgets may route units of at most 384 tokens (G = 4) to the
    # warp-per-unit kernel (2: always; 1: when they are many; 0: never)
    b = np.array([40, 96, 17 + 16, 200], dtype=np.int32)
    _run(SMALL.with_(sink=1, window=16), budgets=b, fused=fused, small_mode=small_mode)


@FUSED
def test_ragged_mix_of_small_and_large_units(fused):
    # budgets on both sides of the small-unit cap: both kernels in one call
    w = SMALL.with_(layers=4, prompt=1200, steps=24, sink=2, window=32)
    b = np.array([40, 1000, 380, 385, 64, 700, 120, 383], dtype=np.int32)
    _run(w, budgets=b, fused=fused, small_mode=2)


@pytest.mark.parametrize("shape", [
    dict(hq=2, hkv=2, d=64, dtype="f32"),        # G = 1
    dict(hq=4, hkv=2, d=128, dtype="bf16"),      # G = 2
    dict(hq=8, hkv=2, d=64, dtype="bf16"),
    dict(hq=8, hkv=2, d=128, dtype="f32"),
])
def test_warp_per_unit_group_sizes_and_dtypes(shape):
    b = np.array([40, 96, 33, 200], dtype=np.int32)
    _run(SMALL.with_(sink=1, window=16, **shape), budgets=b, fused=True, small_mode=2)
    _run(SMALL.with_(sink=1, window=16, **shape), budgets=b, importance_mode=1, small_mode=2)


@FUSED
def test_more_units_than_resident_clusters(fused):
    # 404 equal units: more than one round of clusters, so the host may launch
    # the full rounds and the remaining units separately
    _run(SMALL.with_(layers=1, batch=101, hq=8, hkv=4, steps=6), fused=fused)


def test_last_round_60_percent_busy_runs_as_two_launches():
    # 61 x 8 = 488 equal units of ~100 tokens: one round of 304 resident
    # clusters (2 CTAs per SM on 152 SMs) and a last round 60 % busy, which
    # the host launches separately at its own cluster size
    from tests.lockstep import Lockstep
    w = SMALL.with_(layers=1, batch=61, hq=32, hkv=8, prompt=120, steps=6)
    ls = Lockstep(w)
    ls.prefill()
    rep = ls.decode(fused=True)
    cfg = ls.cache.last_decode_config()
    ls.cache.close()
    assert rep.evictions_checked == w.units * (1 + w.steps)
    assert len(cfg) == 2, cfg
    first, rest = cfg
    assert first["units"] + rest["units"] == w.units
    assert first["units"] % first["clusters"] == 0          # full rounds only
    assert 0.5 < rest["units"] / first["clusters"] <= 0.7   # the remainder's share of a round


@FUSED
def test_page_size_variants(fused):
    # 16-token pages: the cache grows a page every 16 steps before the
    # budget is reached, steps the fused call runs as three calls
    _run(SMALL, page_tokens=16, fused=fused)
    _run(SMALL, page_tokens=256, fused=fused)


@FUSED
def test_shared_page_pool(fused):
    # a pool smaller than every unit's max_tokens (8 units x 5 pages of 64,
    # against 8 x 6 for home pages): pages come from the shared free stack,
    # the decode kernel reads page ids from the table, the cut returns pages
    w = SMALL
    _run(w, pool_pages=w.units * 5, fused=fused)


def test_long_chunk_global_logits_path():
    # 50k tokens in one unit at G = 8: even 16 CTAs leave chunks whose logits
    # exceed shared memory, so the kernel keeps them in the global buffer
    w = W.Workload(101, "long", 1, 1, 8, 1, 128, "bf16", 50000, 6, 60000, 4, 64, 1, "zipf1.1")
    _run(w)
    _run(w, fused=True)


@pytest.mark.parametrize("kpool", [3, 7, 64])
def test_snapkv_pooled_prefill_selection(kpool):
    # SnapKV: the prompt scores are max-pooled over the next k positions
    # before the cut; f32 (CUDA-core scoring) and bf16 (tensor-core scoring)
    _run(SMALL.with_(sink=1, window=16), pool_kernel=kpool)
    _run(SMALL.with_(sink=1, window=16, dtype="f32", d=64), pool_kernel=kpool, fused=True)


def test_snapkv_llama3_8b_layer():
    rep = _run(W.WORKLOADS[1], pool_kernel=7, fused=True)
    assert rep.evictions_checked == 64 * (1 + 256)


@FUSED
@pytest.mark.parametrize("kw", [
    dict(sink=0, window=48, budget=96),                     # HiKV's equal split, no sinks
    dict(sink=4, window=16, budget=96),
    dict(sink=0, window=48, budget=96, dtype="f32", d=64, hq=4, hkv=2),
])
def test_hikv_recent_bank_importance(kw, fused):
    _run(SMALL.with_(**kw), importance_mode=1, fused=fused)


def test_hikv_dual_bank_llama3_8b_layer():
    # budget 1024 split into a 512-token recent bank and a 512-token important bank
    w = W.WORKLOADS[1].with_(sink=0, window=512)
    rep = _run(w, importance_mode=1, fused=True)
    assert rep.evictions_checked == 64 * (1 + 256)


# HiKV prefill initialisation (HiKV sec. III-D): each prompt token's score is
# its attention column over its own band of W = B_I/2 queries; the cut keeps
# the last W prompt tokens (recent bank) and the W best-scored of the rest
# (important bank); decoding then runs the recent-bank rule.  Importance after
# the band pass, the retained sets and every decode output against the oracle.
@FUSED
@pytest.mark.parametrize("kw", [
    dict(sink=0, window=48, budget=96),                                   # bf16, G = 4
    dict(sink=0, window=48, budget=96, dtype="f32", d=64, hq=4, hkv=2),   # fp32, G = 2
    dict(sink=0, window=20, budget=40, hq=16, hkv=2),                     # G = 8
    dict(sink=0, window=33, budget=66, hq=2, hkv=2, prompt=301),          # G = 1, ragged tiles
], ids=["bf16_g4", "f32_g2", "g8", "g1_ragged"])
def test_hikv_band_prefill_and_dual_bank(kw, fused):
    rep = _run(SMALL.with_(**kw), importance_mode=1, prefill_band=kw["window"], fused=fused)
    assert rep.evictions_checked > 0


@pytest.mark.parametrize("band", [1, 64, 1000])
def test_hikv_band_prefill_band_widths(band):
    # a band of one query (the diagonal), one tile, and more than the prompt
    rep = _run(SMALL.with_(sink=2, window=16, prompt=200), prefill_band=band, fused=True)
    assert rep.evictions_checked > 0


def test_hikv_band_prefill_llama3_8b_shape():
    # the Llama-3-8B layer's head shape and 8192-token prompt, one batch row
    # (8 units: the oracle forms every prompt query's softmax), HiKV's equal
    # split of the 1024 budget: W = 512, no sinks, band 512
    w = W.WORKLOADS[1].with_(batch=1, sink=0, window=512)
    rep = _run(w, importance_mode=1, prefill_band=512, fused=True)
    assert rep.evictions_checked == 8 * (1 + 256)
    print("band prefill 8B shape: max bf16 err", rep.max_out_err, "ulps", rep.max_out_ulps,
          "over 1 ulp", rep.bf16_over_1ulp, "near-tie swaps", rep.near_tie_swaps)


def test_hikv_band_prefill_state_errors():
    import importance_aware_kv_gb300 as hk
    dev = torch.device("cuda")
    q = torch.randn(1, 1, 4, 40, 64, device=dev).to(torch.bfloat16)
    k = torch.randn(1, 1, 2, 40, 64, device=dev).to(torch.bfloat16)
    c = hk.Cache(hk.CacheConfig(1, 1, 4, 2, 64, "bf16", 1, 4, [16, 16], 64, page_tokens=16))
    c.append(k, k.clone())
    with pytest.raises(hk.HikvError) as ei:        # created without band_scoring
        c.score_band(q, 8)
    assert ei.value.status == hk.HIKV_ERR_STATE
    c.close()
    c = hk.Cache(hk.CacheConfig(1, 1, 4, 2, 64, "bf16", 1, 4, [16, 16], 64, page_tokens=16, band_scoring=1))
    c.append(k, k.clone())
    with pytest.raises(hk.HikvError) as ei:
        c.score_band(q, 0)
    assert ei.value.status == hk.HIKV_ERR_INVALID_ARG
    c.score_band(q, 8)
    c.evict()
    with pytest.raises(ValueError):                # the binding sees 16 held tokens, not 40
        c.score_band(q, 8)
    with pytest.raises(hk.HikvError) as ei:        # the library itself refuses a cut prompt
        hk._check(hk._lib.hikv_score_band(c.h, 0, 1, 8, hk._dev(q, "q"), hk._stream(None)))
    assert ei.value.status == hk.HIKV_ERR_STATE
    c.device_status()
    c.close()


# HiKV Stage II: element-level attention against the oracle's statement of it.
# Output rows whose chunk selection float32 rounding of the logits could
# change must equal one of the outputs the admissible selections give, at the
# dtype's normal bound; importance, which takes the whole P, and the retained
# sets are compared at the usual tolerances everywhere.
@FUSED
@pytest.mark.parametrize("kw,b2", [
    (dict(), 64),                                                   # one chunk of 97 entries
    (dict(prompt=1200, budget=700), 32),                            # two spans, six chunks, ragged tail
    (dict(prompt=1200, budget=700), 1),                             # extreme budgets
    (dict(prompt=1200, budget=700), 127),
    (dict(dtype="f32", d=64, hq=4, hkv=2, budget=300), 16),         # G = 2, d = 64, fp32
    (dict(hq=16, hkv=2, budget=600, prompt=900), 64),               # G = 8
    (dict(hq=2, hkv=2, budget=200), 48),                            # G = 1
    (dict(dtype="f32", d=128, hq=8, hkv=1, budget=1100, prompt=1500), 96),
    (dict(prompt=900, budget=300, evict_every=4), 64),              # fused steps without eviction, batched cuts
    (dict(budget=127), 64),                                         # n = 128: one full span, no tail
    (dict(budget=128), 64),                                         # n = 129: a second span of one rank
], ids=["b64_1chunk", "b32_2spans", "b1", "b127", "f32_d64_g2", "g8", "g1", "f32_g8_3spans", "evict_every4",
        "n128", "n129"])
def test_hikv_stage2_element_level(kw, b2, fused):
    rep = _run(SMALL.with_(**kw), element_budget=b2, fused=fused)
    assert rep.evictions_checked > 0
    print("stage2 near-tie rows:", rep.stage2_near_tie_rows, "matched another selection:", rep.stage2_alt_matches,
          "elements checked:", rep.outputs_checked)


def test_hikv_stage2_positions_spread_over_70k():
    # a 70,000-token prompt cut to 300: the retained positions span 0..70,011,
    # so the order kernel bins them 32 positions to a bucket and ranks inside
    # buckets; 16-token pages put a page boundary every 16 slots
    w = SMALL.with_(layers=1, batch=1, hq=8, hkv=2, prompt=70000, budget=300, steps=12)
    rep = _run(w, element_budget=64, fused=True, page_tokens=16)
    assert rep.evictions_checked == 2 * (1 + 12)


def test_hikv_stage2_with_recent_bank():
    rep = _run(SMALL.with_(sink=0, window=48, budget=96), element_budget=48, importance_mode=1, fused=True)
    assert rep.evictions_checked > 0


def test_hikv_stage2_llama3_8b_layer():
    # r_II = 2 on the Llama-3-8B layer: 1025 tokens = 9 chunks of 128 per head
    ls = _ls(W.WORKLOADS[1], element_budget=64)
    ls.prefill()
    rep = ls.decode(steps=24, fused=True)
    rows = ls.cache.element_rows()
    ls.cache.close()
    assert rep.evictions_checked == 64 * (1 + 24)
    # V rows read: at most every attended row (64 units x 1025 x 24 steps), and
    # at least the B2 of each full chunk that one head keeps (8 x 64 + 1 per unit)
    assert 64 * 24 * (8 * 64 + 1) <= rows <= 64 * 24 * 1025
    # rows whose selection rounding could change: a small share of the 8 x 32 x 24
    head_rows = 8 * 32 * 24
    assert rep.stage2_near_tie_rows <= 0.1 * head_rows, rep.stage2_near_tie_rows
    print("stage2 8B layer: near-tie rows", rep.stage2_near_tie_rows, "of", head_rows,
          "matched another selection", rep.stage2_alt_matches, "max bf16 err", rep.max_out_err)


def test_hikv_stage2_rejects_units_above_its_limit():
    import importance_aware_kv_gb300 as hk
    w = SMALL.with_(layers=1, batch=1, hkv=1, hq=4, prompt=16500, budget=17000, steps=1)
    cache = hk.Cache(hk.CacheConfig(w.layers, w.batch, w.hq, w.hkv, w.d, w.dtype, w.sink, w.window,
                                    [w.budget], w.total_positions, element_budget=64))
    k, v = W.gen_kv(w, 0, 1, 0, w.prompt, 1)
    cache.append(W.to_torch(k).cuda(), W.to_torch(v).cuda())
    q = torch.zeros((1, 1, w.hq, w.d), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(hk.HikvError) as ei:
        cache.decode_step(q, out)
    assert ei.value.status == hk.HIKV_ERR_CAPACITY
    cache.close()


@FUSED
def test_pyramidkv_layer_budgets(fused):
    import importance_aware_kv_gb300 as hk
    w = SMALL.with_(layers=4, sink=2, window=16)
    b = hk.budgets_pyramid(w.layers, w.hkv, 96, 40, w.sink + w.window)
    assert len(set(b.tolist())) == 4                 # a different budget per layer
    _run(w, budgets=b, fused=fused)


@FUSED
def test_duoattention_retrieval_and_streaming_heads(fused):
    import importance_aware_kv_gb300 as hk
    w = SMALL.with_(layers=4, sink=4, window=16)
    mask = W.retrieval_mask(w, 0.3, seed=5)
    b = hk.budgets_duo(mask, w.total_positions, w.sink, w.window)
    assert 0 < mask.sum() < mask.size
    rep = _run(w, budgets=b, fused=fused)
    assert rep.evictions_checked > 0


def test_snapkv_needs_the_uncut_prompt():
    import importance_aware_kv_gb300 as hk
    cfg = hk.CacheConfig(1, 1, 4, 2, 64, "bf16", 1, 4, [16, 16], 64, page_tokens=16, pool_kernel=5)
    c = hk.Cache(cfg)
    dev = torch.device("cuda")
    k = torch.randn(1, 1, 2, 40, 64, device=dev).to(torch.bfloat16)
    c.append(k, k.clone())
    q = torch.randn(1, 1, 4, 8, 64, device=dev).to(torch.bfloat16)
    c.score_window(q)
    c.evict()
    with pytest.raises(hk.HikvError) as ei:
        c.score_window(q)                           # slots no longer in position order
    assert ei.value.status == hk.HIKV_ERR_STATE
    c.device_status()
    c.close()


@FUSED
def test_zero_keys_tie_rule_exact(fused):
    """All-zero keys: uniform softmax, whole classes of tokens tie exactly; the
    GPU must keep the lowest positions, with no near-tie allowance."""
    from tests.lockstep import Lockstep
    w = W.Workload(102, "zero", 1, 1, 4, 1, 64, "f32", 200, 24, 60, 4, 16, 1, None)
    ls = Lockstep(w, check_kv=False)
    orig = W.gen_kv

    def zero_keys(*a, **k):
        kk, vv = orig(*a, **k)
        return np.zeros_like(kk), vv
    W.gen_kv = zero_keys
    try:
        ls.prefill()
        ls.decode(fused=fused)
    finally:
        W.gen_kv = orig
    assert ls.rep.near_tie_swaps == 0


def test_host_errors_leave_cache_usable():
    import importance_aware_kv_gb300 as hk
    cfg = hk.CacheConfig(1, 1, 4, 2, 64, "f32", 2, 4, [16, 16], 40, page_tokens=16, pool_pages=4)
    c = hk.Cache(cfg)
    dev = torch.device("cuda")
    q = torch.randn(1, 1, 4, 64, device=dev)
    out = torch.empty_like(q)
    with pytest.raises(hk.HikvError) as ei:
        c.decode_step(q, out)                       # empty units
    assert ei.value.status == hk.HIKV_ERR_STATE
    k = torch.randn(1, 1, 2, 33, 64, device=dev)
    with pytest.raises(hk.HikvError) as ei:
        c.append(k, k.clone())                      # 2 units x 3 pages > pool of 4
    assert ei.value.status == hk.HIKV_ERR_CAPACITY
    k = torch.randn(1, 1, 2, 20, 64, device=dev)
    c.append(k, k.clone())
    with pytest.raises(hk.HikvError) as ei:
        c.append(torch.randn(1, 1, 2, 21, 64, device=dev), torch.randn(1, 1, 2, 21, 64, device=dev))
    assert ei.value.status == hk.HIKV_ERR_CAPACITY  # 41 > max_tokens
    assert list(c.lengths()) == [20, 20]
    c.decode_step(q, out)
    c.evict()
    assert list(c.lengths()) == [16, 16]
    k1 = torch.randn(1, 1, 2, 1, 64, device=dev)
    with pytest.raises(hk.HikvError) as ei:
        c.step(k1, k1.clone(), q, q)                # out aliases q
    assert ei.value.status == hk.HIKV_ERR_INVALID_ARG
    c.step(k1, k1.clone(), q, out)                  # one launch: append, attend, evict
    assert list(c.lengths()) == [16, 16]
    c.step(k1, k1.clone(), q, out, evict=False)
    assert list(c.lengths()) == [17, 17]
    c.device_status()
    c.close()


# One fused call per layer, back to back on the stream: each launch may start
# while the previous one runs (programmatic dependent launch), loading its own
# layer's tiles (and, for small calls, prefetching them into L2) before the
# previous grid completes, and reading q and the new rows only after.
@pytest.mark.parametrize("kw", [
    dict(layers=6),                                          # G = 4, one eviction a step
    dict(layers=5, hq=16, hkv=2, budget=250, window=24),     # G = 8 (tensor cores)
    dict(layers=4, evict_every=4, steps=24),                 # batched evictions between the layer calls
], ids=["g4", "g8", "evict_every4"])
def test_per_layer_launches(kw):
    w = SMALL.with_(**kw)
    ls = _ls(w)
    ls.prefill()
    rep = ls.decode(fused=True, per_layer=True)
    ls.cache.close()
    assert rep.evictions_checked > 0
