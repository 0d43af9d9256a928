"""The N-rank path, on CPU with the gloo backend.

Units (layer, batch row, KV head) are independent: attention, importance and
eviction are all per unit, so N ranks share one workload's units out with no
data-path collective.  The benchmark gives each rank a rectangle of units --
batch rows when they divide evenly, else contiguous layer ranges balanced by
the sum of their units' budgets -- and takes the slowest rank's time.

Checked here: the split's balance on the ragged HeadKV budgets; and two gloo
ranks each running the CPU oracle on its own shard of a workload, whose
retained sets, importance and outputs, gathered on rank 0, must equal one
oracle run over the whole workload.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _spawn(target, world, *args):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=target, args=(r, world, port, q, *args)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    return sorted(got, key=lambda g: g[0])


def _init(rank, world, port):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://", rank=rank, world_size=world)
    return dist


def _timing_main(rank, world, port, q):
    dist = _init(rank, world, port)
    try:
        import bench
        r, wsz, local = bench.dist_env()
        t = bench.max_over_ranks(1.5 + rank, wsz, "cpu")
        q.put((r, wsz, local, t, bench.whole_job_rate(wsz, 100, t, "weak"),
               bench.whole_job_rate(wsz, 100, t, "strong")))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    got = _spawn(_timing_main, 2)
    assert [g[0] for g in got] == [0, 1] and all(g[1] == 2 for g in got)
    assert all(g[3] == 2.5 for g in got)                        # max over ranks
    assert all(abs(g[4] - 2 * 100 / 2.5) < 1e-12 for g in got)  # weak: a job step is 2 workload steps
    assert all(abs(g[5] - 100 / 2.5) < 1e-12 for g in got)      # strong: one workload, shared out


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.whole_job_rate(1, 10, 2.0) == 5.0


@pytest.mark.parametrize("world", [2, 3, 4, 8])
def test_layer_split_balances_ragged_budgets(world):
    import bench
    import workloads as W
    w = W.WORKLOADS[3].with_(batch=5)          # batch rows do not divide: split by layer
    b = W.budgets(w)
    loads = b.reshape(w.layers, w.hkv).sum(axis=1) * w.batch
    shares = [bench.rank_shard(w, world, r, b) for r in range(world)]
    # contiguous, non-empty, covering every layer once
    assert shares[0][0] == 0 and shares[-1][1] == w.layers
    assert all(s[0] < s[1] and s[2:] == (0, w.batch) for s in shares)
    assert all(shares[r][1] == shares[r + 1][0] for r in range(world - 1))
    per_rank = [int(loads[s[0]:s[1]].sum()) for s in shares]
    assert sum(per_rank) == int(loads.sum())
    # no rank exceeds the mean by more than the largest single layer
    assert max(per_rank) - loads.sum() / world <= loads.max()


def test_batch_split_is_exact():
    import bench
    import workloads as W
    w = W.WORKLOADS[1]
    b = W.budgets(w)
    assert [bench.rank_shard(w, 4, r, b) for r in range(4)] == [(0, 1, 2 * r, 2 * r + 2) for r in range(4)]
    gw = bench.global_workload(w, 4, "weak")
    assert gw.batch == 32 and [bench.rank_shard(gw, 4, r, b)[2:] for r in range(4)] == \
        [(8 * r, 8 * r + 8) for r in range(4)]


def test_shard_inputs_are_the_whole_workloads():
    import workloads as W
    w = W.WORKLOADS[0].with_(layers=3, batch=2, prompt=40, steps=4)
    k, v = W.gen_kv(w, 0, 3, 0, 44)
    q = W.gen_q(w, 0, 3, 0, 44)
    s = W.shard(w, 1, 3, 1, 2)
    ks, vs = W.gen_kv(s, 0, 2, 0, 44)
    np.testing.assert_array_equal(ks, k[1:3, 1:2])
    np.testing.assert_array_equal(vs, v[1:3, 1:2])
    np.testing.assert_array_equal(W.gen_q(s, 1, 1, 10, 5), q[2:3, 1:2, :, 10:15])
    ku, vu = W.gen_kv_unit(s, 1, 0, 1, 0, 44)
    np.testing.assert_array_equal(ku, k[2, 1, 1])
    d = W.WORKLOADS[3]
    np.testing.assert_array_equal(W.budgets(W.shard(d, 5, 9, 0, 16)), W.budgets(d)[5 * d.hkv:9 * d.hkv])


def _run_oracle(w, budgets):
    """The oracle over workload w: prompt, window scoring, cut, decode steps
    with eviction.  Returns ({(layer, b, g): (positions, importance)},
    [step][layer][b][Hq][d] outputs), indexed by w's global layers/rows."""
    import oracle
    import workloads as W
    O = oracle.Oracle(w.layers, w.batch, w.hq, w.hkv, w.d, w.sink, w.window, budgets, threads=2)
    k, v = W.gen_kv(w, 0, w.layers, 0, w.prompt)
    O.append(0, W.to_f32(k), W.to_f32(v))
    O.score_window(0, W.to_f32(W.gen_q(w, 0, w.layers, w.prompt - w.nq, w.nq)))
    O.evict(0, w.layers)
    ks, vs = W.gen_kv(w, 0, w.layers, w.prompt, w.steps)
    qs = W.gen_q(w, 0, w.layers, w.prompt, w.steps)
    outs = []
    for s in range(w.steps):
        O.append(0, W.to_f32(ks[:, :, :, s:s + 1]), W.to_f32(vs[:, :, :, s:s + 1]))
        outs.append(O.decode(0, W.to_f32(qs[:, :, :, s])))
        if (s + 1) % w.evict_every == 0:
            O.evict(0, w.layers)
    state = {}
    for l in range(w.layers):
        for b in range(w.batch):
            for g in range(w.hkv):
                pos, imp = O.state(O.unit(l, b, g))
                state[(w.layer0 + l, w.batch0 + b, g)] = (pos, imp)
    out = {(w.layer0 + l, w.batch0 + b): np.stack([o[l, b] for o in outs])
           for l in range(w.layers) for b in range(w.batch)}
    return state, out


def _shard_main(rank, world, port, q, wkw):
    dist = _init(rank, world, port)
    try:
        import bench
        import workloads as W
        w = W.WORKLOADS[0].with_(**wkw)
        b = W.budgets(w) if wkw.get("budget") != "ragged" else _ragged(w)
        l0, l1, b0, b1 = bench.rank_shard(w, world, rank, b)
        s = W.shard(w, l0, l1, b0, b1)
        state, out = _run_oracle(s, b[l0 * w.hkv:l1 * w.hkv])
        gathered = [None] * world
        dist.all_gather_object(gathered, (state, out, (l0, l1, b0, b1)))
        q.put((rank, gathered if rank == 0 else None))
    finally:
        dist.destroy_process_group()


def _ragged(w):
    rng = np.random.default_rng(9)
    return rng.integers(w.sink + w.window, 100, size=w.layers * w.hkv).astype(np.int32)


@pytest.mark.parametrize("wkw", [
    dict(layers=5, batch=1, prompt=120, steps=10, budget="ragged"),   # layer split by Sum B_u
    dict(layers=2, batch=4, prompt=120, steps=10),                    # batch split
], ids=["layers_ragged", "batch_rows"])
def test_two_gloo_ranks_decode_their_shards_as_one_workload(wkw):
    import workloads as W
    got = _spawn(_shard_main, 2, wkw)
    gathered = got[0][1]
    w = W.WORKLOADS[0].with_(**wkw)
    b = W.budgets(w) if wkw.get("budget") != "ragged" else _ragged(w)
    whole_state, whole_out = _run_oracle(w, b)
    state, out = {}, {}
    for st, o, _ in gathered:
        assert not set(st) & set(state), "a unit decoded by two ranks"
        state.update(st)
        out.update(o)
    assert set(state) == set(whole_state) and set(out) == set(whole_out)
    for u, (pos, imp) in whole_state.items():
        np.testing.assert_array_equal(state[u][0], pos)
        np.testing.assert_array_equal(state[u][1], imp)
    for key, o in whole_out.items():
        np.testing.assert_array_equal(out[key], o)
    shards = [g[2] for g in gathered]
    assert shards[0] != shards[1]
    if wkw.get("budget") == "ragged":
        loads = b.reshape(w.layers, w.hkv).sum(axis=1)
        per_rank = [int(loads[s[0]:s[1]].sum()) for s in shards]
        assert max(per_rank) - loads.sum() / 2 <= loads.max()
