"""The seeded input generator (shared by the oracle tests and the CUDA tests)."""
import numpy as np

import workloads as W


def test_positions_past_the_workload_get_their_own_heavy_scale():
    # the benchmark decodes more steps than the workload lists; every generated
    # position must have a heavy-hitter factor (none may be read past the end)
    w = W.WORKLOADS[1].with_(batch=1, hkv=2, hq=8, prompt=64, steps=8)
    k_long, v_long = W.gen_kv(w, 0, 1, w.prompt, 40)
    k_short, v_short = W.gen_kv(w, 0, 1, w.prompt, w.steps)
    assert k_long.shape[3] == 40
    # Bernoulli heavy hitters are drawn per position: the workload's own
    # positions are unchanged when more are generated
    assert np.array_equal(k_long[:, :, :, : w.steps], k_short)
    assert np.array_equal(v_long[:, :, :, : w.steps], v_short)
    kf = W.to_f32(k_long)
    assert np.isfinite(kf).all() and np.abs(kf).max() < 3 * 8   # N(0,1) x at most 3


def test_heavy_scale_length_follows_upto():
    w = W.WORKLOADS[4].with_(layers=1, prompt=128, steps=4)
    assert W.heavy_scale(w, 4, 0, 0).size == w.total_positions
    assert W.heavy_scale(w, 4, 0, 0, upto=500).size == 500
    s = W.heavy_scale(w, 4, 0, 0, upto=500)
    assert np.all((s >= 1.0) & (s <= 4.0))
