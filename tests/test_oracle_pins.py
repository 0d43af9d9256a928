"""Pins of the CPU oracle to things other than itself.

Each test ties one part of the oracle to a library routine, a closed form, an
invariant or a brute force, chosen so that a plausible slip (a dropped scale,
a wrong head-to-group map, a transposed operand, a wrong tie order, a missing
increment) fails at least one of them.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(rng, *shape):
    return rng.standard_normal(shape).astype(np.float32)


def _sdpa_ref(q, k, v, G, scale=None):
    """Textbook attention via torch SDPA in float64; kv head of query head h is h // G."""
    qt = torch.from_numpy(q.astype(np.float64))            # [Hq, 1, d]
    kt = torch.from_numpy(k.astype(np.float64)).repeat_interleave(G, dim=0)  # [Hq, n, d]
    vt = torch.from_numpy(v.astype(np.float64)).repeat_interleave(G, dim=0)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return o.numpy()


# --------------------------------------------------------------------------
# attention: budget >= context means no eviction, so the decode output is
# plain full attention (library SDPA).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("out_bf16", [False, True])
def test_full_attention_equals_library_sdpa(out_bf16):
    rng = np.random.default_rng(11)
    L, B, Hq, Hkv, d = 2, 2, 8, 2, 32
    G = Hq // Hkv
    prompt, steps = 40, 5
    O = oracle.Oracle(L, B, Hq, Hkv, d, 4, 8, np.full(L * Hkv, 10_000), out_bf16=out_bf16)
    K = _rand(rng, L, B, Hkv, prompt + steps, d)
    V = _rand(rng, L, B, Hkv, prompt + steps, d)
    O.append(0, K[:, :, :, :prompt], V[:, :, :, :prompt])
    for s in range(steps):
        t = prompt + s
        O.append(0, K[:, :, :, t:t + 1], V[:, :, :, t:t + 1])
        q = _rand(rng, L, B, Hq, d)
        out = O.decode(0, q)
        O.evict(0, L)  # budget far above n: must be a no-op
        for l in range(L):
            for b in range(B):
                ref = _sdpa_ref(q[l, b][:, None, :], K[l, b, :, :t + 1], V[l, b, :, :t + 1], G)[:, 0]
                got = out[l, b]
                if not out_bf16:
                    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-6 * np.abs(ref).max())
                else:
                    # bf16: representable, and within half an ulp of the exact value
                    bits = got.view(np.uint32)
                    assert np.all(bits & 0xFFFF == 0)
                    e = np.floor(np.log2(np.abs(ref)))
                    half_ulp = 2.0 ** (e - 8)
                    assert np.all(np.abs(got - ref) <= half_ulp * (1 + 1e-9))
    for u in range(O.units):
        assert O.length(u) == prompt + steps


def test_scale_override_is_used():
    rng = np.random.default_rng(3)
    O = oracle.Oracle(1, 1, 2, 1, 16, 0, 0, [100], scale=0.5)
    K, V = _rand(rng, 1, 1, 1, 9, 16), _rand(rng, 1, 1, 1, 9, 16)
    O.append(0, K, V)
    q = _rand(rng, 1, 1, 2, 16)
    ref = _sdpa_ref(q[0, 0][:, None], K[0, 0], V[0, 0], 2, scale=0.5)[:, 0]
    np.testing.assert_allclose(O.decode(0, q)[0, 0], ref, rtol=0, atol=1e-6 * np.abs(ref).max())


# --------------------------------------------------------------------------
# importance: equals the attention columns summed over the group's heads,
# with the window queries causally masked (brute force on tiny inputs).
# --------------------------------------------------------------------------
def test_importance_equals_summed_attention_columns():
    rng = np.random.default_rng(5)
    L, B, Hq, Hkv, d = 1, 2, 4, 2, 8
    G = Hq // Hkv
    prompt, nq, steps = 12, 3, 4
    O = oracle.Oracle(L, B, Hq, Hkv, d, 1, 2, np.full(Hkv, 1000))
    K = _rand(rng, L, B, Hkv, prompt + steps, d) * 2
    V = _rand(rng, L, B, Hkv, prompt + steps, d)
    Qw = _rand(rng, L, B, Hq, nq, d) * 2
    O.append(0, K[:, :, :, :prompt], V[:, :, :, :prompt])
    O.score_window(0, Qw)
    expect = np.zeros((B, Hkv, prompt + steps))
    for b in range(B):
        for g in range(Hkv):
            for i in range(nq):
                qpos = prompt - nq + i
                for hh in range(G):
                    s = Qw[0, b, g * G + hh, i].astype(np.float64) @ K[0, b, g, :qpos + 1].T.astype(np.float64)
                    p = torch.softmax(torch.from_numpy(s / np.sqrt(d)), 0).numpy()
                    expect[b, g, :qpos + 1] += p
    for s_ in range(steps):
        t = prompt + s_
        O.append(0, K[:, :, :, t:t + 1], V[:, :, :, t:t + 1])
        q = _rand(rng, L, B, Hq, d)
        O.decode(0, q)
        for b in range(B):
            for g in range(Hkv):
                for hh in range(G):
                    s = q[0, b, g * G + hh].astype(np.float64) @ K[0, b, g, :t + 1].T.astype(np.float64)
                    expect[b, g, :t + 1] += torch.softmax(torch.from_numpy(s / np.sqrt(d)), 0).numpy()
    for b in range(B):
        for g in range(Hkv):
            pos, imp = O.state(O.unit(0, b, g))
            np.testing.assert_array_equal(pos, np.arange(prompt + steps))
            np.testing.assert_allclose(imp, expect[b, g], rtol=2e-6, atol=1e-7)


# --------------------------------------------------------------------------
# softmax sums to one, so every scored query adds exactly G to the unit's
# total importance: retained + evicted mass = G * (nq + steps).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("evict", [False, True])
def test_importance_mass_conservation(evict):
    rng = np.random.default_rng(7)
    L, B, Hq, Hkv, d = 2, 1, 6, 2, 16
    G = Hq // Hkv
    prompt, nq, steps, S, Wn = 64, 8, 20, 2, 6
    budget = np.array([24, 30, 20, 28]) if evict else np.full(L * Hkv, 500)
    O = oracle.Oracle(L, B, Hq, Hkv, d, S, Wn, budget)
    O.append(0, _rand(rng, L, B, Hkv, prompt, d), _rand(rng, L, B, Hkv, prompt, d))
    O.score_window(0, _rand(rng, L, B, Hq, nq, d))
    O.evict(0, L)
    for _ in range(steps):
        O.append(0, _rand(rng, L, B, Hkv, 1, d), _rand(rng, L, B, Hkv, 1, d))
        O.decode(0, _rand(rng, L, B, Hq, d))
        O.evict(0, L)
    for u in range(O.units):
        pos, imp = O.state(u)
        total = float(imp.astype(np.float64).sum()) + O.evicted_mass(u)
        assert abs(total - G * (nq + steps)) < 1e-5 * G * (nq + steps)
        if evict:
            assert len(pos) == min(prompt + steps, O.budget_of(u))


# --------------------------------------------------------------------------
# eviction rule
# --------------------------------------------------------------------------
def _h2o_keep(pos, imp, capacity, sink, window):
    """Keep set of the H2O eviction listing (KV cache compression blog, sec. 3
    "H2O"), restated: entries in position order; the first `sink` and the last
    `window` are protected; of the rest the `capacity - sink - window` with
    the largest scores (torch.topk) are kept."""
    order = np.argsort(pos)
    pos, imp = pos[order], imp[order]
    n = len(pos)
    if n <= capacity:
        return set(pos.tolist())
    cand = torch.ones(n, dtype=torch.bool)
    cand[:sink] = False
    if window:
        cand[n - window:] = False
    ci = torch.nonzero(cand).squeeze(1)
    _, top = torch.topk(torch.from_numpy(imp)[ci], k=capacity - sink - window, largest=True)
    kept = set(pos[:sink].tolist()) | set(pos[n - window:].tolist() if window else [])
    kept |= set(pos[ci[top].numpy()].tolist())
    return kept


def test_evict_matches_h2o_topk_on_distinct_scores():
    rng = np.random.default_rng(13)
    L, B, Hq, Hkv, d = 1, 2, 4, 2, 16
    S, Wn = 3, 5
    budget = np.array([20, 26])
    O = oracle.Oracle(L, B, Hq, Hkv, d, S, Wn, budget)
    O.append(0, _rand(rng, L, B, Hkv, 48, d) * 2, _rand(rng, L, B, Hkv, 48, d))
    O.score_window(0, _rand(rng, L, B, Hq, 6, d) * 2)
    checked = 0
    for step in range(30):
        if step:
            O.append(0, _rand(rng, L, B, Hkv, 1, d) * 2, _rand(rng, L, B, Hkv, 1, d))
            O.decode(0, _rand(rng, L, B, Hq, d) * 2)
        before = [O.state(u) for u in range(O.units)]
        O.evict(0, L)
        for u in range(O.units):
            pos, imp = before[u]
            t = O.next_pos(u) - 1
            mid = (pos >= S) & (pos <= t - Wn)
            assert len(np.unique(imp[mid])) == mid.sum(), "scores must be distinct here"
            want = _h2o_keep(pos, imp, O.budget_of(u), S, Wn)
            got, _ = O.state(u)
            assert set(got.tolist()) == want
            assert len(got) == min(len(pos), O.budget_of(u))
            assert len(np.unique(got)) == len(got)
            assert set(range(S)) <= set(got.tolist())
            assert set(range(t - Wn + 1, t + 1)) <= set(got.tolist())
            checked += 1
    assert checked == 30 * O.units


def test_budget_equal_sinks_plus_window_is_streaming_llm():
    """B = S + W leaves exactly {t_1..t_S} U {t_{i-W+1}..t_i} (StreamingLLM,
    KV cache compression blog sec. 3)."""
    rng = np.random.default_rng(17)
    S, Wn = 4, 12
    O = oracle.Oracle(1, 1, 2, 1, 8, S, Wn, [S + Wn])
    O.append(0, _rand(rng, 1, 1, 1, 40, 8), _rand(rng, 1, 1, 1, 40, 8))
    O.score_window(0, _rand(rng, 1, 1, 2, 4, 8))
    for step in range(25):
        if step:
            O.append(0, _rand(rng, 1, 1, 1, 1, 8), _rand(rng, 1, 1, 1, 1, 8))
            O.decode(0, _rand(rng, 1, 1, 2, 8))
        O.evict(0, 1)
        t = O.next_pos(0) - 1
        pos, _ = O.state(0)
        assert pos.tolist() == list(range(S)) + list(range(t - Wn + 1, t + 1))


def _exact_uniform_keep(history, S, Wn, B, G):
    """Brute force with exact rationals for all-zero keys (uniform softmax).

    history: list of ("window", nq) / ("decode",) / ("append", n) / ("evict",)
    Returns the retained position set after replaying it.
    """
    imp = {}
    nxt = 0
    for ev in history:
        if ev[0] == "append":
            for _ in range(ev[1]):
                imp[nxt] = Fraction(0)
                nxt += 1
        elif ev[0] == "window":
            nq = ev[1]
            t = nxt - 1
            for i in range(nq):
                qpos = t - nq + 1 + i
                vis = [p for p in imp if p <= qpos]
                for p in vis:
                    imp[p] += Fraction(G, len(vis))
        elif ev[0] == "decode":
            n = len(imp)
            for p in imp:
                imp[p] += Fraction(G, n)
        elif ev[0] == "evict":
            if len(imp) <= B:
                continue
            t = nxt - 1
            prot = [p for p in imp if p < S or p > t - Wn]
            cand = sorted((p for p in imp if not (p < S or p > t - Wn)),
                          key=lambda p: (-imp[p], p))
            keep = set(prot) | set(cand[:B - len(prot)])
            imp = {p: imp[p] for p in keep}
    return set(imp)


def test_zero_keys_uniform_softmax_tie_rule():
    """All-zero keys make every softmax uniform, so scores are closed forms
    and whole classes of tokens tie exactly; ties must keep the lowest
    positions."""
    S, Wn, Bu, G, d = 2, 5, 14, 2, 8
    prompt, nq = 40, 6
    rng = np.random.default_rng(19)
    O = oracle.Oracle(1, 1, G, 1, d, S, Wn, [Bu])
    zk = np.zeros((1, 1, 1, prompt, d), np.float32)
    O.append(0, zk, _rand(rng, 1, 1, 1, prompt, d))
    O.score_window(0, _rand(rng, 1, 1, G, nq, d))
    O.evict(0, 1)
    hist = [("append", prompt), ("window", nq), ("evict",)]
    assert set(O.state(0)[0].tolist()) == _exact_uniform_keep(hist, S, Wn, Bu, G)
    # the cut keeps the lowest candidate positions among the tied prompt class
    assert set(O.state(0)[0].tolist()) == set(range(Bu - Wn)) | set(range(prompt - Wn, prompt))
    for _ in range(12):
        O.append(0, np.zeros((1, 1, 1, 1, d), np.float32), _rand(rng, 1, 1, 1, 1, d))
        O.decode(0, _rand(rng, 1, 1, G, d))
        O.evict(0, 1)
        hist += [("append", 1), ("decode",), ("evict",)]
        assert set(O.state(0)[0].tolist()) == _exact_uniform_keep(hist, S, Wn, Bu, G)


def test_resync_moves_entries_and_mass():
    rng = np.random.default_rng(23)
    O = oracle.Oracle(1, 1, 2, 1, 8, 1, 2, [6])
    O.append(0, _rand(rng, 1, 1, 1, 10, 8), _rand(rng, 1, 1, 1, 10, 8))
    O.score_window(0, _rand(rng, 1, 1, 2, 3, 8))
    total_before = O.state(0)[1].astype(np.float64).sum()
    O.evict(0, 1)
    pos, _ = O.state(0)
    epos, _ = O.last_evicted(0)
    swapped = np.concatenate([pos[pos != pos[1]], epos[:1]])
    O.resync(0, swapped)
    assert set(O.state(0)[0].tolist()) == set(swapped.tolist())
    total = O.state(0)[1].astype(np.float64).sum() + O.evicted_mass(0)
    assert abs(total - total_before) < 1e-6
    with pytest.raises(RuntimeError):
        O.resync(0, np.array([99, 100]))


# --------------------------------------------------------------------------
# byte accounting used by the roofline: the page's worked KV-size example
# --------------------------------------------------------------------------
def test_kv_size_worked_example():
    vals = {}
    with open(os.path.join(GOLDEN, "kv_size_llama3_70b_128k.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, v = line.split()
            vals[k] = float(v)
    m = W.kv_bytes(int(vals["batch"]), int(vals["length"]), int(vals["layers"]),
                   int(vals["kv_heads"]), int(vals["head_dim"]), int(vals["elem_bytes"]))
    assert round(m / 1e9, 1) == vals["gigabytes"]


# --------------------------------------------------------------------------
# SnapKV pooling (blog sec. 3 "SnapKV"): S_pooled[i] = max_{0<=m<k} A_obs[i+m]
# --------------------------------------------------------------------------
def _window_scores_ref(K, Qw, G, prompt, nq, d):
    """Observation-window scores by brute force: each of the last nq prompt
    queries, causally masked, softmax in float64, summed over the group."""
    L, B, Hkv = K.shape[:3]
    out = np.zeros((B, Hkv, prompt))
    for b in range(B):
        for g in range(Hkv):
            for i in range(nq):
                qpos = prompt - nq + i
                for hh in range(G):
                    s = Qw[0, b, g * G + hh, i].astype(np.float64) @ K[0, b, g, :qpos + 1].T.astype(np.float64)
                    out[b, g, :qpos + 1] += torch.softmax(torch.from_numpy(s / np.sqrt(d)), 0).numpy()
    return out


def _forward_maxpool(pos, score, k):
    """max over the retained positions in [p, p + k), by explicit search."""
    out = np.empty_like(score)
    for j, p in enumerate(pos):
        out[j] = max(score[m] for m in range(len(pos)) if p <= pos[m] < p + k)
    return out


@pytest.mark.parametrize("kpool", [1, 3, 5, 7])
def test_pooled_window_score_equals_brute_force(kpool):
    rng = np.random.default_rng(11 + kpool)
    L, B, Hq, Hkv, d = 1, 2, 4, 2, 8
    G = Hq // Hkv
    prompt, nq = 20, 4
    O = oracle.Oracle(L, B, Hq, Hkv, d, 1, 2, np.full(Hkv, 1000))
    K = _rand(rng, L, B, Hkv, prompt, d) * 2
    Qw = _rand(rng, L, B, Hq, nq, d) * 2
    O.append(0, K, _rand(rng, L, B, Hkv, prompt, d))
    O.score_window(0, Qw)
    O.pool_importance(0, L, kpool)
    raw = _window_scores_ref(K, Qw, G, prompt, nq, d)
    for b in range(B):
        for g in range(Hkv):
            pos, imp = O.state(O.unit(0, b, g))
            want = _forward_maxpool(np.arange(prompt), raw[b, g], kpool)
            np.testing.assert_allclose(imp, want, rtol=2e-6, atol=1e-7)
            assert np.all(imp >= raw[b, g].astype(np.float32) - 1e-6)   # pooling never lowers a score


def test_pooled_spike_spreads_to_the_k_positions_before_it():
    # one key aligned with every window query takes almost all the mass: after
    # pooling with k, exactly positions p-k+1 .. p carry the spike
    L, B, Hq, Hkv, d = 1, 1, 2, 1, 4
    prompt, nq, k, p = 24, 2, 5, 10
    O = oracle.Oracle(L, B, Hq, Hkv, d, 0, 0, np.full(Hkv, 1000))
    K = np.zeros((L, B, Hkv, prompt, d), np.float32)
    K[0, 0, 0, p] = [40, 0, 0, 0]
    Qw = np.zeros((L, B, Hq, nq, d), np.float32)
    Qw[..., 0] = 40
    O.append(0, K, np.zeros_like(K))
    O.score_window(0, Qw)
    _, raw = O.state(0)
    assert raw[p] > 0.999 * Hq * nq and raw.sum() - raw[p] < 1e-3
    O.pool_importance(0, L, k)
    _, imp = O.state(0)
    spiked = np.nonzero(imp > 0.5 * Hq * nq)[0]
    np.testing.assert_array_equal(spiked, np.arange(p - k + 1, p + 1))


def test_pooling_after_an_eviction_uses_positions():
    # with gaps in the retained positions the window [p, p + k) is by position
    rng = np.random.default_rng(3)
    L, B, Hq, Hkv, d = 1, 1, 2, 1, 8
    prompt, nq, k = 40, 4, 4
    O = oracle.Oracle(L, B, Hq, Hkv, d, 2, 4, np.full(Hkv, 20))
    O.append(0, _rand(rng, L, B, Hkv, prompt, d) * 2, _rand(rng, L, B, Hkv, prompt, d))
    O.score_window(0, _rand(rng, L, B, Hq, nq, d) * 2)
    O.evict(0, L)
    pos, before = O.state(0)
    assert len(pos) == 20 and np.any(np.diff(pos) > 1)
    O.pool_importance(0, L, k)
    _, after = O.state(0)
    np.testing.assert_array_equal(after, _forward_maxpool(pos, before, k))


# --------------------------------------------------------------------------
# HiKV Stage I (HiKV sec. III-B, Algorithm 1): scores accumulate only in the
# recent bank; the token leaving it is promoted only if its score exceeds the
# important bank's minimum.
# --------------------------------------------------------------------------
def _softmax_row(q, keys, d):
    s = keys.astype(np.float64) @ q.astype(np.float64) / np.sqrt(d)
    return torch.softmax(torch.from_numpy(s), 0).numpy()


def test_recent_bank_accumulation_equals_brute_force():
    rng = np.random.default_rng(21)
    L, B, Hq, Hkv, d = 1, 1, 4, 2, 8
    G = Hq // Hkv
    prompt, nq, steps, W = 10, 3, 8, 4
    O = oracle.Oracle(L, B, Hq, Hkv, d, 0, W, np.full(Hkv, 1000))   # no eviction
    O.set_recent_only(True)
    K = _rand(rng, L, B, Hkv, prompt + steps, d) * 2
    V = _rand(rng, L, B, Hkv, prompt + steps, d)
    Qw = _rand(rng, L, B, Hq, nq, d) * 2
    O.append(0, K[:, :, :, :prompt], V[:, :, :, :prompt])
    O.score_window(0, Qw)
    expect = np.zeros((Hkv, prompt + steps))
    expect[:, :prompt] = _window_scores_ref(K, Qw, G, prompt, nq, d)[0]
    for s_ in range(steps):
        t = prompt + s_
        O.append(0, K[:, :, :, t:t + 1], V[:, :, :, t:t + 1])
        q = _rand(rng, L, B, Hq, d)
        before = [O.state(O.unit(0, 0, g))[1].copy() for g in range(Hkv)]
        O.decode(0, q)
        for g in range(Hkv):
            inc = sum(_softmax_row(q[0, 0, g * G + hh], K[0, 0, g, :t + 1], d) for hh in range(G))
            recent = np.arange(t + 1) >= t - W
            expect[g, :t + 1] += np.where(recent, inc, 0.0)
            _, now = O.state(O.unit(0, 0, g))
            old = np.arange(t) < t - W                       # frozen: bit-identical
            np.testing.assert_array_equal(now[:t][old], before[g][:t][old])
    for g in range(Hkv):
        _, imp = O.state(O.unit(0, 0, g))
        np.testing.assert_allclose(imp, expect[g], rtol=2e-6, atol=1e-7)


def test_recent_bank_with_a_window_covering_everything_is_h2o():
    rng = np.random.default_rng(22)
    L, B, Hq, Hkv, d = 1, 2, 2, 1, 8
    prompt, steps = 6, 5
    outs = []
    for recent in (False, True):
        r = np.random.default_rng(22)
        O = oracle.Oracle(L, B, Hq, Hkv, d, 0, 1000, np.full(Hkv, 2000))
        O.set_recent_only(recent)
        O.append(0, _rand(r, L, B, Hkv, prompt, d), _rand(r, L, B, Hkv, prompt, d))
        O.score_window(0, _rand(r, L, B, Hq, 2, d))
        for _ in range(steps):
            O.append(0, _rand(r, L, B, Hkv, 1, d), _rand(r, L, B, Hkv, 1, d))
            O.decode(0, _rand(r, L, B, Hq, d))
        outs.append([O.state(u)[1] for u in range(O.units)])
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)


def test_dual_bank_eviction_matches_hikv_fifo_and_min_heap():
    """Restate HiKV Stage I directly -- a FIFO recent bank of W tokens, an
    important bank of B - W tokens with frozen scores, the ejected token
    promoted only if its score exceeds the bank's minimum -- and compare the
    retained tokens and scores with the oracle's argmin formulation."""
    rng = np.random.default_rng(23)
    L, B_, Hq, Hkv, d = 1, 1, 2, 1, 8
    G = Hq // Hkv
    prompt, nq, steps, W, Bud = 24, 4, 30, 6, 12
    O = oracle.Oracle(L, B_, Hq, Hkv, d, 0, W, np.full(Hkv, Bud))
    O.set_recent_only(True)
    K = _rand(rng, L, B_, Hkv, prompt + steps, d) * 2
    V = _rand(rng, L, B_, Hkv, prompt + steps, d)
    Qw = _rand(rng, L, B_, Hq, nq, d) * 2
    O.append(0, K[:, :, :, :prompt], V[:, :, :, :prompt])
    O.score_window(0, Qw)
    O.evict(0, L)
    # the dual bank, initialised as HiKV sec. III-D describes: the last W
    # prompt tokens form the recent bank, the top B - W of the rest the
    # important bank
    score = dict(enumerate(_window_scores_ref(K, Qw, G, prompt, nq, d)[0, 0]))
    recent = list(range(prompt - W, prompt))
    rest = sorted(range(prompt - W), key=lambda p: (-score[p], p))
    important = set(rest[:Bud - W])
    for s_ in range(steps):
        t = prompt + s_
        O.append(0, K[:, :, :, t:t + 1], V[:, :, :, t:t + 1])
        q = _rand(rng, L, B_, Hq, d)
        O.decode(0, q)
        O.evict(0, L)
        recent.append(t)
        score[t] = 0.0
        kept = sorted(important) + recent
        inc = sum(_softmax_row(q[0, 0, hh], K[0, 0, 0, kept], d) for hh in range(G))
        for p, x in zip(kept, inc):
            if p in recent:
                score[p] += x
        evi = recent.pop(0)
        low = min(important, key=lambda p: (score[p], -p))
        if score[evi] > score[low]:
            important.remove(low)
            important.add(evi)
        pos, imp = O.state(0)
        assert sorted(important) + recent == list(pos), s_
        np.testing.assert_allclose(imp, [score[p] for p in pos], rtol=2e-6, atol=1e-7)


# --------------------------------------------------------------------------
# budget schedules (blog sec. 3 "PyramidKV", "DuoAttention")
# --------------------------------------------------------------------------
def test_pyramid_budgets_closed_forms():
    from oracle import budgets
    b = budgets.pyramid(5, 2, 100, 20, 1).reshape(5, 2)
    assert np.all(b[:, 0] == b[:, 1])                  # one budget per layer
    np.testing.assert_array_equal(b[:, 0], [180, 140, 100, 60, 20])   # C_max = 180 .. C_min, step 40
    assert b[:, 0].mean() == 100                       # mean = C_avg
    b = budgets.pyramid(4, 1, 10, 3, 1)                # 17, 12.33, 7.67, 3 -> nearest
    np.testing.assert_array_equal(b, [17, 12, 8, 3])
    b = budgets.pyramid(5, 1, 10, 9, 1)                # 11, 10.5, 10, 9.5, 9 -> halves go up
    np.testing.assert_array_equal(b, [11, 11, 10, 10, 9])
    assert np.all(np.diff(budgets.pyramid(32, 1, 2048, 256, 1)) <= 0)   # decaying
    np.testing.assert_array_equal(budgets.pyramid(1, 3, 77, 10, 1), [77, 77, 77])
    np.testing.assert_array_equal(budgets.pyramid(3, 1, 50, 10, 40), [90, 50, 40])   # raised to the floor
    b = budgets.pyramid(3, 1, 11, 10, 1)               # 12, 11, 10
    np.testing.assert_array_equal(b, [12, 11, 10])
    b = budgets.pyramid(4, 1, 11, 10, 1)               # 12, 11.33, 10.67, 10 -> 12, 11, 11, 10
    np.testing.assert_array_equal(b, [12, 11, 11, 10])


def test_duo_budgets():
    from oracle import budgets
    mask = np.array([[1, 0, 0], [0, 1, 0]], dtype=np.uint8)
    np.testing.assert_array_equal(budgets.duo(mask, 4096, 4, 256), [4096, 260, 260, 260, 4096, 260])


# --------------------------------------------------------------------------
# HiKV Stage II (sec. III-C, Algorithm 1): element-level selection.  Pinned
# by brute force over subsets (a top-k set is the k-subset with the largest
# sum), by the special case that reduces to exact attention, and by a
# construction whose selected entries are known in advance.
# --------------------------------------------------------------------------
def _best_subset(values, k):
    """Indices of the k-subset with the largest sum (values distinct)."""
    from itertools import combinations
    best, arg = -np.inf, None
    for c in combinations(range(len(values)), k):
        s = float(np.sum(np.asarray(values, np.float64)[list(c)]))
        if s > best:
            best, arg = s, c
    return list(arg)


def test_stage2_equals_brute_force_subsets():
    rng = np.random.default_rng(21)
    d, B2, G, n = 8, 3, 2, 21           # P chunks of 8, 8 and 5 entries
    O = oracle.Oracle(1, 1, G, 1, d, 0, 0, [1000])
    O.set_element_budget(B2)
    K, V = _rand(rng, 1, 1, 1, n, d), _rand(rng, 1, 1, 1, n, d)
    O.append(0, K, V)
    q = _rand(rng, 1, 1, G, d)
    out = O.decode(0, q)
    _, imp = O.state(0)
    scale = 1.0 / np.sqrt(d)
    colsum = np.zeros(n)
    for h in range(G):
        qh = q[0, 0, h].astype(np.float64)
        dims = _best_subset(np.abs(qh), B2)
        s = scale * (K[0, 0, 0][:, dims].astype(np.float64) @ qh[dims])
        p = np.exp(s - s.max())
        p /= p.sum()
        colsum += p
        keep = []
        for c0 in range(0, n, d):
            idx = list(range(c0, min(n, c0 + d)))
            keep += idx if len(idx) <= B2 else [idx[i] for i in _best_subset(p[idx], B2)]
        ref = p[keep] @ V[0, 0, 0][keep].astype(np.float64)
        np.testing.assert_allclose(out[0, 0, h], ref, rtol=0, atol=1e-12 * np.abs(ref).max() + 1e-7 * np.abs(ref).max())
        # a plain global top-3 of P would pick another set here
        assert sorted(keep) != sorted(np.argsort(-p)[:len(keep)].tolist())
    # the importance takes the whole P: its head-summed columns, and mass G
    np.testing.assert_allclose(imp, colsum.astype(np.float32), rtol=1e-7, atol=0)
    assert abs(float(np.sum(imp, dtype=np.float64)) - G) < 1e-5
    assert not O.stage2_near_ties(0, 1).any()


def test_stage2_with_sparse_query_and_short_context_is_exact_attention():
    # q has exactly B2 non-zero dimensions, some negative: the magnitude rule
    # keeps all of them, so the logits are the exact ones; n <= B2 leaves a
    # single chunk that keeps every entry.  Output = library SDPA.
    rng = np.random.default_rng(5)
    d, B2, G, n = 32, 16, 4, 16
    O = oracle.Oracle(1, 2, G, 1, d, 0, 0, [1000])
    O.set_element_budget(B2)
    K, V = _rand(rng, 1, 2, 1, n, d), _rand(rng, 1, 2, 1, n, d)
    O.append(0, K, V)
    q = np.zeros((1, 2, G, d), np.float32)
    for b in range(2):
        for h in range(G):
            dims = rng.choice(d, B2, replace=False)
            q[0, b, h, dims] = rng.uniform(0.2, 2.0, B2) * rng.choice([-1.0, 1.0], B2)
    out = O.decode(0, q)
    for b in range(2):
        ref = _sdpa_ref(q[0, b][:, None, :], K[0, b], V[0, b], G)[:, 0]
        np.testing.assert_allclose(out[0, b], ref, rtol=0, atol=1e-6 * np.abs(ref).max())


def test_stage2_chunks_are_retained_entries_in_position_order():
    # S = 2 sinks and a W = 10 window with budget S + W keep positions
    # {0, 1, 14..23} of a 24-token prompt; after position 24 is appended the
    # 13 entries form the chunks [0, 1, 14..19] and [20..24] (by rank, not by
    # position value).  Keys are a_p * ones, so the logits follow a_p and the
    # B2 = 3 entries kept in each chunk are known in advance.
    d, B2, S, Wn = 8, 3, 2, 10
    O = oracle.Oracle(1, 1, 1, 1, d, S, Wn, [S + Wn])
    O.set_element_budget(B2)
    a = np.zeros(25)
    a[[0, 1, 14, 15, 16, 17, 18, 19]] = [0.1, 0.9, 0.2, 0.8, 0.3, 0.7, 0.4, 0.6]
    a[[20, 21, 22, 23, 24]] = [0.5, 0.05, 0.95, 0.15, 0.85]
    a[2:14] = np.linspace(1.0, 2.0, 12)          # evicted before the decode step
    K = np.repeat(a[:, None], d, axis=1).astype(np.float32)[None, None, None]
    V = np.zeros((1, 1, 1, 25, d), np.float32)
    V[..., 0] = 1.0
    V[..., 1] = np.arange(25, dtype=np.float32)
    O.append(0, K[:, :, :, :24], V[:, :, :, :24])
    O.evict(0, 1)
    pos, _ = O.state(0)
    assert pos.tolist() == [0, 1] + list(range(14, 24))
    O.append(0, K[:, :, :, 24:], V[:, :, :, 24:])
    q = np.zeros((1, 1, 1, d), np.float32)
    q[0, 0, 0, [1, 4, 6]] = [3.0, 2.0, 1.0]       # the three largest |q|
    out = O.decode(0, q)[0, 0, 0]
    kept_pos = [0, 1] + list(range(14, 25))
    s = (1.0 / np.sqrt(d)) * 6.0 * a[kept_pos]    # <q, a_p * ones> = 6 a_p
    p = np.exp(s - s.max())
    p /= p.sum()
    chosen = {1, 15, 17, 20, 22, 24}              # top 3 of a in each chunk
    sel = np.array([x in chosen for x in kept_pos])
    assert abs(out[0] - p[sel].sum()) < 1e-6
    assert abs(out[1] - (p[sel] * np.array(kept_pos)[sel]).sum()) < 1e-5
    # the two plausible misreadings keep other sets: chunks by position value
    # (0-7, 8-15, 16-23, 24) and one global top 6
    for wrong in ({0, 1, 14, 15, 17, 19, 22, 24}, {1, 15, 17, 19, 22, 24}):
        assert abs(out[0] - p[np.array([x in wrong for x in kept_pos])].sum()) > 1e-3


# --------------------------------------------------------------------------
# HiKV prefill initialisation (HiKV sec. III-D with the IS definition of
# sec. III-B): IS(l) = sum over the band of queries l .. l + band - 1 of
# P_i[l], causal, summed over the group's heads.  Pinned by the full causal
# P matrix built with library softmax, a zero-key closed form in exact
# rationals, and the band's two extremes.
# --------------------------------------------------------------------------
def _causal_p(q, keys, d):
    """[n][n] causal softmax matrix of one head (row i = query at position i),
    library softmax in float64 with masked entries at -inf."""
    s = q.astype(np.float64) @ keys.astype(np.float64).T / np.sqrt(d)
    n = s.shape[0]
    s[np.triu_indices(n, 1)] = -np.inf
    return torch.softmax(torch.from_numpy(s), 1).numpy()


def _band_ref(Q, K, G, band, d):
    """IS per (b, g, token) from the full P matrices."""
    L, B, Hkv, n = K.shape[:4]
    out = np.zeros((B, Hkv, n))
    for b in range(B):
        for g in range(Hkv):
            for hh in range(G):
                P = _causal_p(Q[0, b, g * G + hh], K[0, b, g], d)
                for l in range(n):
                    out[b, g, l] += P[l:min(n, l + band), l].sum()
    return out


@pytest.mark.parametrize("band", [1, 3, 7, 20, 40])
def test_band_score_equals_full_attention_columns(band):
    rng = np.random.default_rng(31 + band)
    L, B, Hq, Hkv, d, n = 1, 2, 4, 2, 8, 20
    G = Hq // Hkv
    O = oracle.Oracle(L, B, Hq, Hkv, d, 0, 4, np.full(Hkv, 1000))
    K = _rand(rng, L, B, Hkv, n, d) * 2
    Q = _rand(rng, L, B, Hq, n, d) * 2
    O.append(0, K, _rand(rng, L, B, Hkv, n, d))
    O.score_band(0, Q, band)
    ref = _band_ref(Q, K, G, band, d)
    for b in range(B):
        for g in range(Hkv):
            pos, imp = O.state(O.unit(0, b, g))
            np.testing.assert_array_equal(pos, np.arange(n))
            np.testing.assert_allclose(imp, ref[b, g], rtol=2e-7, atol=1e-9)
    # the observation window of the last `band` queries is another score
    # unless the band covers the whole prompt, where the two coincide
    Ow = oracle.Oracle(L, B, Hq, Hkv, d, 0, 4, np.full(Hkv, 1000))
    Ow.append(0, K, np.zeros_like(K))
    Ow.score_window(0, Q[:, :, :, n - min(band, n):])
    same = np.allclose(Ow.state(0)[1], O.state(0)[1], rtol=1e-6, atol=1e-7)
    assert same == (band >= n)


def test_band_score_zero_keys_closed_form():
    # all-zero keys: query i spreads 1/(i+1) over tokens 0..i, so
    # IS(l) = G * sum_{i=l}^{min(l+band, n)-1} 1/(i+1), in exact rationals
    L, B, Hq, Hkv, d, n, band = 1, 1, 8, 1, 16, 37, 9
    G = Hq // Hkv
    rng = np.random.default_rng(4)
    O = oracle.Oracle(L, B, Hq, Hkv, d, 0, 0, [1000])
    O.append(0, np.zeros((L, B, Hkv, n, d), np.float32), _rand(rng, L, B, Hkv, n, d))
    O.score_band(0, _rand(rng, L, B, Hq, n, d), band)
    _, imp = O.state(0)
    for l in range(n):
        want = G * sum(Fraction(1, i + 1) for i in range(l, min(n, l + band)))
        assert abs(float(imp[l]) - float(want)) <= 2 ** -22 * float(want), l


def test_band_one_is_the_diagonal_and_a_full_band_holds_all_mass():
    rng = np.random.default_rng(5)
    L, B, Hq, Hkv, d, n = 1, 1, 2, 1, 8, 15
    G = Hq // Hkv
    K = _rand(rng, L, B, Hkv, n, d) * 2
    Q = _rand(rng, L, B, Hq, n, d) * 2
    O1 = oracle.Oracle(L, B, Hq, Hkv, d, 0, 0, [1000])
    O1.append(0, K, K)
    O1.score_band(0, Q, 1)
    _, imp = O1.state(0)
    diag = sum(np.diag(_causal_p(Q[0, 0, h], K[0, 0, 0], d)) for h in range(G))
    np.testing.assert_allclose(imp, diag, rtol=2e-7)
    assert imp[0] == G                             # query 0 sees only token 0
    On = oracle.Oracle(L, B, Hq, Hkv, d, 0, 0, [1000])
    On.append(0, K, K)
    On.score_band(0, Q, n)                         # every query's whole row
    assert abs(float(np.sum(On.state(0)[1], dtype=np.float64)) - G * n) < 1e-5


def test_band_score_needs_the_uncut_prompt():
    rng = np.random.default_rng(6)
    O = oracle.Oracle(1, 1, 2, 1, 8, 0, 2, [8])
    O.append(0, _rand(rng, 1, 1, 1, 12, 8), _rand(rng, 1, 1, 1, 12, 8))
    O.evict(0, 1)
    with pytest.raises(ValueError):
        O.score_band(0, _rand(rng, 1, 1, 2, 8, 8), 4)


def test_hikv_band_init_then_dual_bank_matches_fifo_and_min_heap():
    """HiKV from prefill to decode, restated directly: every prompt token's
    IS is its attention column over its own band of W = B_I/2 queries; the
    last W prompt tokens fill the recent bank and the top W of the rest the
    important bank (sec. III-D); decoding then runs the FIFO + frozen-score
    min-heap rule of sec. III-B.  The oracle (band scores, the cut, recent-
    bank accumulation, argmin eviction) must keep the same tokens with the
    same scores at every step."""
    rng = np.random.default_rng(41)
    L, B_, Hq, Hkv, d = 1, 1, 2, 1, 8
    G = Hq // Hkv
    prompt, steps, W = 30, 25, 5
    Bud = 2 * W
    O = oracle.Oracle(L, B_, Hq, Hkv, d, 0, W, np.full(Hkv, Bud))
    O.set_recent_only(True)
    K = _rand(rng, L, B_, Hkv, prompt + steps, d) * 2
    V = _rand(rng, L, B_, Hkv, prompt + steps, d)
    Q = _rand(rng, L, B_, Hq, prompt, d) * 2
    O.append(0, K[:, :, :, :prompt], V[:, :, :, :prompt])
    O.score_band(0, Q, W)
    O.evict(0, L)
    P = [_causal_p(Q[0, 0, h], K[0, 0, 0, :prompt], d) for h in range(G)]
    score = {l: sum(P[h][l:min(prompt, l + W), l].sum() for h in range(G)) for l in range(prompt)}
    recent = list(range(prompt - W, prompt))
    rest = sorted(range(prompt - W), key=lambda p: (-score[p], p))
    important = set(rest[:Bud - W])
    pos, imp = O.state(0)
    assert sorted(important) + recent == list(pos)
    np.testing.assert_allclose(imp, [score[p] for p in pos], rtol=2e-6, atol=1e-7)
    for s_ in range(steps):
        t = prompt + s_
        O.append(0, K[:, :, :, t:t + 1], V[:, :, :, t:t + 1])
        q = _rand(rng, L, B_, Hq, d)
        O.decode(0, q)
        O.evict(0, L)
        recent.append(t)
        score[t] = 0.0
        kept = sorted(important) + recent
        inc = sum(_softmax_row(q[0, 0, hh], K[0, 0, 0, kept], d) for hh in range(G))
        for p, x in zip(kept, inc):
            if p in recent:
                score[p] += x
        evi = recent.pop(0)
        low = min(important, key=lambda p: (score[p], -p))
        if score[evi] > score[low]:
            important.remove(low)
            important.add(evi)
        pos, imp = O.state(0)
        assert sorted(important) + recent == list(pos), s_
        np.testing.assert_allclose(imp, [score[p] for p in pos], rtol=2e-6, atol=1e-7)


# --------------------------------------------------------------------------
# HiKV Stage II near ties: when float32 rounding of the logits could change
# a chunk's selection, the oracle lists every admissible output.
# --------------------------------------------------------------------------
def test_stage2_exact_tie_lists_both_selections():
    # chunk of d = 8 entries, B2 = 3; entries 2 and 5 have identical keys, so
    # identical logits, and they are the 3rd and 4th largest: either may be
    # kept.  Their values differ, so the two admissible outputs differ.
    d, B2 = 8, 3
    O = oracle.Oracle(1, 1, 1, 1, d, 0, 0, [1000])
    O.set_element_budget(B2)
    a = np.array([0.9, 0.8, 0.5, 0.1, 0.2, 0.5, 0.0, 0.3])
    K = np.repeat(a[:, None], d, axis=1).astype(np.float32)[None, None, None]
    V = np.zeros((1, 1, 1, d, d), np.float32)
    V[0, 0, 0, np.arange(d), np.arange(d)] = 1.0          # one-hot values: out[j] = p_j if kept
    O.append(0, K, V)
    q = np.zeros((1, 1, 1, d), np.float32)
    q[0, 0, 0, :3] = [2.0, 1.5, 1.0]
    out = O.decode(0, q)[0, 0, 0]
    assert O.stage2_near_ties(0, 1)[0, 0, 0] == 1
    alts = O.stage2_alternatives(0, 0, 0)
    assert alts.shape == (2, d)
    kept_sets = sorted(tuple(np.nonzero(x)[0].tolist()) for x in alts)
    assert kept_sets == [(0, 1, 2), (0, 1, 5)]
    # the exact output keeps the lower position of the tie and is listed
    assert tuple(np.nonzero(out)[0].tolist()) == (0, 1, 2)
    assert any(np.array_equal(out, x) for x in alts)


def test_stage2_separated_logits_have_no_alternatives():
    d, B2 = 8, 3
    O = oracle.Oracle(1, 1, 1, 1, d, 0, 0, [1000])
    O.set_element_budget(B2)
    a = np.linspace(0.0, 1.0, d)
    K = np.repeat(a[:, None], d, axis=1).astype(np.float32)[None, None, None]
    O.append(0, K, K)
    q = np.ones((1, 1, 1, d), np.float32)
    O.decode(0, q)
    assert O.stage2_near_ties(0, 1)[0, 0, 0] == 0
    assert O.stage2_alternatives(0, 0, 0).shape == (0, d)
