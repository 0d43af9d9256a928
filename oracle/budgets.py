"""ORACLE -- test infrastructure only: budget schedules restated in exact
rational arithmetic.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import it.

* PyramidKV (KV cache compression blog, sec. 3 "PyramidKV"): layer l of N_L
  (l = 1..N_L) gets C_l = C_max - (l - 1) (C_max - C_min) / (N_L - 1); the
  blog constrains the mean to C_avg, and for this linear profile the mean is
  (C_max + C_min) / 2, so C_max = 2 C_avg - C_min.  Each C_l is rounded half
  up and raised to at least `floor_budget` (a cache needs B >= max(1, S + W)).
  One layer gets C_avg.  Every KV head of a layer shares its budget.
* DuoAttention (blog sec. 3 "DuoAttention"): retrieval heads keep the full
  cache, streaming heads a sink + recent window of S + W tokens.
"""
from fractions import Fraction
import math

import numpy as np


def pyramid(num_layers, num_kv_heads, avg, min_budget, floor_budget):
    if num_layers == 1:
        per_layer = [max(avg, floor_budget)]
    else:
        cmax, cmin = 2 * avg - min_budget, min_budget
        per_layer = []
        for l in range(1, num_layers + 1):
            c = Fraction(cmax) - Fraction((l - 1) * (cmax - cmin), num_layers - 1)
            per_layer.append(max(math.floor(c + Fraction(1, 2)), floor_budget))
    return np.repeat(np.array(per_layer, dtype=np.int32), num_kv_heads)


def duo(retrieval, full_budget, num_sink, recent_window):
    retrieval = np.asarray(retrieval, dtype=bool).ravel()
    return np.where(retrieval, full_budget, num_sink + recent_window).astype(np.int32)
