"""Benchmark of the budgeted, importance-aware KV-cache decode step on GB300.

One step = the whole hot path for one decode token of every unit: append the
new k, v; attention with the importance update and victim argmin; evict back
to the budget -- timed through hikv_decode_step_fused, which runs it as one
kernel launch once every unit is at its budget (the three separate calls,
hikv_append -> hikv_decode_step -> hikv_evict, are timed after it and reported
as `three_call_path`).  Headline workload: the Llama-3-8B-shaped layer (batch
8, 32 query / 8 KV heads, d 128, bf16 K/V, 8192-token prompt, budget 1024, 4
sinks, 64-token window, eviction every step), seeded synthetic inputs resident
in HBM before timing.  The decode stream continues past the workload's 256
steps when more are timed; per-step work is fixed by the budget.  One step
reads 34.5 MB, which would fit in L2: the timed steps run in turn on copies
of the layer's cache holding together more than twice the L2, so each
step's K/V comes cold from HBM while code and small inputs stay warm, as in
a model's decode loop (the same steps after a 256 MB L2 flush are timed
too, `flushed_l2_steps`).  Larger workloads read more than twice the L2 per
step and need neither.

The same run then measures the other workloads (`other_workloads`): the
32-layer 32K-context stack evicting every 16 steps, the HeadKV Dirichlet
budgets, the Llama-3-70B 128K context, and the same 70B context with the
full cache (no eviction) as the uncompressed reference point -- each with its
step rate, HBM fraction, read floor, end-to-end rate and the CPU oracle's
rate.  Their prompt K/V are drawn on the device (torch's seeded generator,
N(0,1) with the workload's heavy-hitter key factors) so that 17-43 GB of
prompt need not be generated on the host; decode-step inputs come from the
workload generator as for the headline.

Prints one JSON line.  `--impl reference` times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "decode steps/s and achieved HBM GB/s (fraction of ~8 TB/s) at 1 GB300"
WORKLOAD_INDEX = 1
OTHER_WORKLOADS = (2, 3, 4, "4-full")
KERNEL_SOURCES = ["importance_aware_kv_gb300/csrc/k_decode.cuh",
                  "importance_aware_kv_gb300/csrc/hikv_internal.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "k_decode_llama3_8b_traffic.json")


def kernel_sha() -> str:
    """Hash of the decode kernel's code (comments and whitespace removed, so
    an edited comment keeps the traffic measured on the same code valid)."""
    import re
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of the ranks' values (the job ends with its slowest rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, steps: int, t_max: float, scaling: str = "weak") -> float:
    """Workload steps/s of the whole job, ended by its slowest rank.  A step
    decodes one token of every unit of the job's workload; under weak
    scaling that workload is `world` times the configured one, so a job
    step counts `world` configured-workload steps."""
    return (world if scaling == "weak" else 1) * steps / t_max


# --------------------------------------------------------------------------
# multi-GPU: the units of one workload shared out across ranks (no collective)
# --------------------------------------------------------------------------
def split_contiguous(loads, parts: int):
    """Contiguous, non-empty ranges [bounds[r], bounds[r + 1]) of `loads`:
    a sweep that closes range r once it holds its share of the load not yet
    assigned (an item joins while less than half of it overshoots that
    share), so no range exceeds its share by more than one item."""
    loads = [int(x) for x in loads]
    n = len(loads)
    if not 1 <= parts <= n:
        raise ValueError(f"cannot split {n} items into {parts} non-empty ranges")
    bounds = [0]
    for r in range(parts - 1):
        i0 = bounds[-1]
        share = sum(loads[i0:]) / (parts - r)
        last = n - (parts - r - 1)          # leave one item for each range still to come
        acc, i = 0, i0
        while i < last and (i == i0 or acc + loads[i] / 2 <= share):
            acc += loads[i]
            i += 1
        bounds.append(i)
    bounds.append(n)
    return bounds


def rank_shard(w, world: int, rank: int, budgets):
    """(l0, l1, b0, b1): the units of w that rank `rank` of `world` decodes.
    Batch rows when they divide evenly (every row has the same budgets, so
    the shares are equal); otherwise contiguous layer ranges balanced by the
    sum of their units' budgets B_u (a unit's decode work is proportional to
    its budget; per-head budgets make layers unequal).  The library's calls
    take whole layers, so a layer is the finest split."""
    if world == 1:
        return 0, w.layers, 0, w.batch
    if w.batch % world == 0:
        per = w.batch // world
        return 0, w.layers, rank * per, (rank + 1) * per
    loads = np.asarray(budgets, np.int64).reshape(w.layers, w.hkv).sum(axis=1) * w.batch
    bounds = split_contiguous(loads, world)
    return bounds[rank], bounds[rank + 1], 0, w.batch


def global_workload(w, world: int, scaling: str):
    """The workload all ranks decode together: `weak` scales the batch with
    the ranks (each rank then holds as many units as one GPU alone), `strong`
    shares out w itself."""
    return w.with_(batch=w.batch * world, name=f"{w.name}-x{world}batch") if scaling == "weak" and world > 1 else w


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 20 ms, from before
    the first timed step (the sampler's first sample is awaited) to after
    the last one."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        self.out = os.path.join("/tmp", f"hikv_clocks_{os.getpid()}.csv")
        try:
            self.f = open(self.out, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def wait_first(self, timeout_s: float = 3.0):
        """Block until the sampler has written a sample (or timeout)."""
        if self.proc is None:
            return
        t0 = time.time()
        while time.time() - t0 < timeout_s:
            try:
                if os.path.getsize(self.out) > 0:
                    return
            except OSError:
                pass
            time.sleep(0.01)

    def stop(self, linger_s: float = 0.05):
        if self.proc is None:
            return None
        time.sleep(linger_s)   # one more sample after the timed region
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.out) as f:
            for line in f:
                p = [x.strip() for x in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    mx.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.out)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "window": "20 ms samples from before the first timed step to after the last"}


def gpu_id_for(dev_index: int) -> str:
    import torch
    try:
        bus = torch.cuda.get_device_properties(dev_index).pci_bus_id
        if bus:
            return str(bus)
    except Exception:
        pass
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    if vis and "," not in vis and vis.strip().isdigit():
        return vis.strip()
    return str(dev_index)


# --------------------------------------------------------------------------
def step_bytes(w, n):
    """Algorithmic bytes of one decode step of units holding n tokens (array or
    scalar) during attention: K/V rows, importance read+write, positions, q in,
    out, plus the appended row (read once from the caller's buffer, written
    into the pool).  Returns the total over the units given."""
    n = np.asarray(n, dtype=np.int64)
    e = w.elem_bytes
    per_unit = 2 * n * w.d * e + 12 * n + 2 * w.group * w.d * e + 2 * w.d * e
    return int(per_unit.sum())


def layer_chunk(w, max_bytes=2e9):
    """Layers per prefill chunk: at most ~2 GB of prompt K/V at a time."""
    import workloads as W
    per_layer = W.kv_bytes(w.batch, w.prompt, 1, w.hkv, w.d, w.elem_bytes)
    return max(1, min(w.layers, int(max_bytes // max(1, per_layer))))


def schedule_budgets(w, seed, schedule):
    """Budget table of a run: the workload's own, or a schedule computed by
    the library -- "pyramid:AVG:MIN" (PyramidKV) or "duo:FRAC" (DuoAttention,
    a seeded FRAC of the heads retrieval heads with the full cache)."""
    import workloads as W
    if schedule in (None, "", "workload"):
        return W.budgets(w, seed)
    import importance_aware_kv_gb300 as hk
    kind, *args = schedule.split(":")
    if kind == "pyramid":
        avg, mn = int(args[0]), int(args[1])
        return hk.budgets_pyramid(w.layers, w.hkv, avg, mn, max(1, w.sink + w.window))
    if kind == "duo":
        mask = W.retrieval_mask(w, float(args[0]), seed)
        return hk.budgets_duo(mask, w.total_positions, w.sink, w.window)
    raise ValueError(f"unknown schedule {schedule!r}")


L2_ASSUMED = 160_000_000   # bytes; above a GB300's 129 MB L2, so NC copies are surely colder than L2


def cold_copies(w, budgets=None, full_cache=False):
    """(NC, bytes of one step): how many copies of the cache the timed steps
    rotate through so that each step's K/V is cold -- 1 when a step reads at
    least twice the L2 itself."""
    import workloads as W
    b = W.budgets(w) if budgets is None else np.asarray(budgets)
    n_est = np.minimum(np.repeat(b.astype(np.int64).reshape(w.layers, w.hkv), w.batch, axis=0).reshape(-1),
                       w.prompt) + 1
    if full_cache:
        n_est = np.full(w.units, w.prompt + 1, np.int64)
    est = step_bytes(w, n_est)
    nc = 1 if est >= 2 * L2_ASSUMED else int(-(-2 * L2_ASSUMED // max(1, est)))
    return (nc if nc <= 16 else 1), est   # more than 16 copies: flush L2 instead


def l2_policy(w, full_cache=False):
    nc, est = cold_copies(w, None, full_cache)
    if nc == 1 and est < 2 * L2_ASSUMED:
        return "flushed between timed steps (256 MB write, outside the timed events)"
    if nc == 1:
        return f"inputs larger than L2: one step reads {est / 1e6:.0f} MB, no flush"
    return (f"inputs larger than L2: {nc} copies of the cache ({nc * est / 1e6:.0f} MB of K/V) decoded in turn, "
            f"no flush")


def workload_config(w, schedule="workload", element_budget=0, full_cache=False, world=1, scaling="weak",
                    l2_mode="auto"):
    """The `config` of a bench line: the workload and the run's options only
    (no measured values), the same for the GPU arm and the reference arm."""
    return {"workload": w.name + ("-full-cache" if full_cache else ""), "layers": w.layers, "batch": w.batch,
            "q_heads": w.hq, "kv_heads": w.hkv, "head_dim": w.d, "kv_dtype": w.dtype, "prompt": w.prompt,
            "budget": "full cache" if full_cache else w.budget, "sink": w.sink, "window": w.window,
            "evict_every": w.evict_every, "budget_schedule": schedule or "workload",
            "element_budget": element_budget,
            "l2": (l2_policy(w, full_cache) if l2_mode != "flush"
                   else "flushed between timed steps (256 MB write, outside the timed events)"),
            "parallelism": (f"units of one workload ({'the configured one' if scaling == 'strong' else f'batch x{world}'})"
                            f" shared out across {world} ranks: batch rows, else layers balanced by Sum B_u;"
                            " no collective" if world > 1 else "one GPU")}


def run_cpu_oracle(w, seed, steps, warmup, budget_s=20.0, layers=None, budgets=None, element_budget=0,
                   steps_1thread=0, budget_1thread_s=10.0):
    """Time the oracle's decode loop (append -> decode -> evict when due) on the
    given layers (default all) and scale to whole-workload steps/s: a step of
    the workload needs every layer, so sampled rate x (sampled / all layers).
    With steps_1thread > 0 the loop then continues for up to that many steps
    (or budget_1thread_s seconds) on one thread.
    Returns (steps/s of the whole workload, threads, steps timed, sample text,
    (steps/s on one thread, steps timed on one thread) or None)."""
    import oracle
    import workloads as W
    threads = os.cpu_count() or 1
    layers = list(range(w.layers)) if layers is None else list(layers)
    b_all = W.budgets(w, seed) if budgets is None else np.asarray(budgets, np.int32)
    bs = np.concatenate([b_all[l * w.hkv:(l + 1) * w.hkv] for l in layers])
    O = oracle.Oracle(len(layers), w.batch, w.hq, w.hkv, w.d, w.sink, w.window, bs,
                      out_bf16=(w.dtype == "bf16"), threads=threads)
    O.set_element_budget(element_budget)
    for si, l in enumerate(layers):
        k, v = W.gen_kv(w, l, 1, 0, w.prompt, seed)
        O.append(si, W.to_f32(k), W.to_f32(v))
        del k, v
        O.score_window(si, W.to_f32(W.gen_q(w, l, 1, w.prompt - w.nq, w.nq, seed)))
    O.evict(0, len(layers))
    total = warmup + steps + steps_1thread
    ks = [W.gen_kv(w, l, 1, w.prompt, total, seed) for l in layers]
    qs = [W.gen_q(w, l, 1, w.prompt, total, seed) for l in layers]

    def one_step(s):
        t0 = time.perf_counter()
        for si in range(len(layers)):
            O.append(si, W.to_f32(ks[si][0][:, :, :, s:s + 1]), W.to_f32(ks[si][1][:, :, :, s:s + 1]))
            O.decode(si, W.to_f32(qs[si][:, :, :, s]))
        if (s + 1) % w.evict_every == 0:
            O.evict(0, len(layers))
        return time.perf_counter() - t0

    done, t_used, s = 0, 0.0, 0
    while s < warmup + steps:
        dt = one_step(s)
        s += 1
        if s > warmup:
            t_used += dt
            done += 1
            if t_used > budget_s:
                break
    frac = len(layers) / w.layers
    single = None
    if steps_1thread > 0:
        O.threads(1)
        done1, t1 = 0, 0.0
        for _ in range(steps_1thread):
            t1 += one_step(s)
            s += 1
            done1 += 1
            if t1 > budget_1thread_s:
                break
        single = (frac * done1 / t1, done1)
    sample = (f"{done} decode steps of all {w.units} units" if frac == 1 else
              f"{done} decode steps of layer(s) {layers} ({len(layers) * w.batch * w.hkv} of {w.units} "
              f"units), rate scaled by {len(layers)}/{w.layers} layers")
    return frac * done / t_used, threads, done, sample, single


def oracle_sample_layers(w):
    """Layers the CPU oracle times: all of a one-layer workload, else one."""
    return None if w.layers == 1 else [0]


def bench_reference(args):
    import workloads as W
    rank, world, _ = dist_env()
    if rank != 0:
        return
    w = W.WORKLOADS[args.workload]
    val, cores, done, sample, _ = run_cpu_oracle(w, w.index, args.steps, args.warmup, budget_s=120.0,
                                                 layers=oracle_sample_layers(w))
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "steps/s", "n_gpus": 0,
        "steps": done, "warmup": args.warmup, "ms_per_step": 1e3 / val, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": workload_config(w, args.schedule, 0, False, world, args.scaling),
        "cpu_baseline": {"value": val, "unit": "steps/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": val, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------
def device_prompt(w, l0, nl, seed, dev):
    """Prompt K, V of layers [l0, l0 + nl) drawn on the device: N(0,1) from
    torch's generator seeded by (seed, l0), keys times the workload's
    heavy-hitter factors of each (layer, batch) sequence."""
    import torch
    import workloads as W
    g = torch.Generator(device=dev)
    g.manual_seed(1_000_003 * (seed + 1) + l0)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    shape = (nl, w.batch, w.hkv, w.prompt, w.d)
    k = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
    if w.heavy is not None:
        f = np.stack([np.stack([W.heavy_scale(w, seed, w.layer0 + l0 + li, w.batch0 + b)[: w.prompt]
                                for b in range(w.batch)]) for li in range(nl)])
        k *= torch.from_numpy(f).to(dev)[:, :, None, :, None]
    k = k.to(dt)
    v = torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(dt)
    return k, v


def measure(w, seed, dev, opts, stage=lambda m: None):
    """Run one workload on the GPU: setup (untimed), then the timed fused
    steps, the three-call steps, per-layer launches, end-to-end steps and the
    read floor.  Returns the results as a dict."""
    import torch
    import importance_aware_kv_gb300 as hk
    import workloads as W

    K, Wu, K3, KL, Ke = opts["steps"], opts["warmup"], opts["three_call_steps"], opts["per_layer_steps"], \
        opts["e2e_steps"]
    L = w.layers
    total_steps = Wu + K + K3 + KL + Ke
    budgets = opts["budgets"]
    if opts["full_cache"]:   # no eviction: every unit keeps its whole context
        budgets = np.full_like(budgets, w.prompt + total_steps + 1)
    elem = opts["element_budget"] if 0 < opts["element_budget"] < w.d else 0
    # Cold data between timed steps.  A step whose bytes are at least twice
    # the L2 evicts its own data; a smaller one (one layer) runs on NC copies
    # of the cache in turn, NC x its bytes >= twice the L2, so each step's
    # K/V is cold while code and the next inputs stay warm as in a model's
    # decode loop; the same steps after an L2 flush (256 MB write) are timed
    # too and reported beside them.
    NC, est = cold_copies(w, budgets, opts["full_cache"])
    l2 = L2_ASSUMED
    if opts.get("l2_mode") == "flush":   # the earlier method: one cache, a 256 MB write before every step
        NC, l2 = 1, float("inf")
    cfg = hk.CacheConfig(w.layers, w.batch, w.hq, w.hkv, w.d, w.dtype, w.sink, w.window,
                         budgets, w.prompt + total_steps * NC + 1, element_budget=elem)
    caches = [hk.Cache(cfg) for _ in range(NC)]
    cache = caches[0]
    stage(f"{w.name}: {NC} cache(s) created")
    # ---- setup (untimed): prompt in layer chunks, window scoring, cut to budget ----
    stream = torch.cuda.current_stream()
    lc = layer_chunk(w)
    for l0 in range(0, L, lc):
        nl = min(lc, L - l0)
        if opts["prompt_source"] == "device":
            dk, dv = device_prompt(w, l0, nl, seed, dev)
        else:
            k, v = W.gen_kv(w, l0, nl, 0, w.prompt, seed)
            dk, dv = W.to_torch(k).to(dev), W.to_torch(v).to(dev)
            del k, v
        for c_ in caches:
            c_.append(dk, dv, layer0=l0)
        del dk, dv
    dq_win = W.to_torch(W.gen_q(w, 0, L, w.prompt - w.nq, w.nq, seed)).to(dev)
    se = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    torch.cuda.synchronize()
    se[0].record(stream)
    cache.score_window(dq_win)           # a0: prompt importance from the observation window
    se[1].record(stream)
    cache.evict()                        # a0: the cut to the budget
    se[2].record(stream)
    for c_ in caches[1:]:
        c_.score_window(dq_win)
        c_.evict()
    torch.cuda.synchronize()
    setup = {"prompt_tokens_per_unit": w.prompt, "window_queries": w.nq,
             "prompt_source": ("device (torch seeded N(0,1) x heavy-hitter factors)"
                               if opts["prompt_source"] == "device" else "workload generator (host)"),
             "window_scoring_ms": se[0].elapsed_time(se[1]), "prefill_cut_ms": se[1].elapsed_time(se[2]),
             "window_scoring_k_gbs": W.kv_bytes(w.batch, w.prompt, L, w.hkv, w.d, w.elem_bytes) / 2 /
             (se[0].elapsed_time(se[1]) / 1e3) / 1e9}
    del dq_win
    # decode inputs for R distinct steps, cycled when all steps' inputs would
    # exceed ~1 GB (the appended rows still take fresh positions every step)
    per_step_in = L * w.batch * (2 * w.hkv + w.hq) * w.d * w.elem_bytes
    R = int(min(total_steps, max(64, 1e9 // per_step_in)))
    ks, vs = W.gen_kv(w, 0, L, w.prompt, R, seed)
    qs = W.gen_q(w, 0, L, w.prompt, R, seed)
    ks = np.ascontiguousarray(np.moveaxis(ks, 3, 0)[:, :, :, :, None, :])
    vs = np.ascontiguousarray(np.moveaxis(vs, 3, 0)[:, :, :, :, None, :])
    qs = np.ascontiguousarray(np.moveaxis(qs, 3, 0))
    dks, dvs, dqs = (W.to_torch(x).to(dev) for x in (ks, vs, qs))
    out = torch.empty_like(dqs[0])
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    E = w.evict_every if not opts["full_cache"] else 1
    taken = [0] * NC                      # decode steps each cache has taken (its eviction cadence)
    turn = {"i": 0}

    def next_step():
        """The next cache in turn, its input index and whether it evicts."""
        ci = turn["i"] % NC
        turn["i"] += 1
        s = taken[ci]
        taken[ci] += 1
        return caches[ci], s % R, (s + 1) % E == 0

    def peek():
        return caches[turn["i"] % NC]

    def step_fused():
        c_, r, ev_ = next_step()
        c_.step(dks[r], dvs[r], dqs[r], out, evict=ev_)

    stage(f"{w.name}: setup done")
    for _ in range(max(Wu, NC)):
        step_fused()
    torch.cuda.synchronize()
    # A spin kernel before each timed step lets the host enqueue the whole
    # step before the GPU reaches it, so host launch overhead never shows up
    # inside the timed events (the spin is outside them).
    spin_cycles = int(opts["spin_us"] * 2.0e3)

    # ---- timed: the single-call step (append + decode + evict in one launch) ----
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = opts.get("sampler")
    if sampler is not None:
        sampler.wait_first()
    if opts["world"] > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    launches0 = sum(c_.kernel_launches() for c_ in caches)
    vrows0 = sum(c_.element_rows() for c_ in caches) if elem else 0
    alg_bytes = 0
    kv_bytes = 0
    for i in range(K):
        n_now = peek().lengths().astype(np.int64) + 1
        alg_bytes += step_bytes(w, n_now)
        kv_bytes += int((2 * n_now * w.d * w.elem_bytes).sum())
        if NC == 1 and est < 2 * l2:
            flush.fill_(float(i))
        torch.cuda._sleep(spin_cycles)
        e0, e1 = ev[i]
        e0.record(stream)
        step_fused()
        e1.record(stream)
    torch.cuda.synchronize()
    launches = sum(c_.kernel_launches() for c_ in caches) - launches0
    dec_cfg = cache.last_decode_config()
    vrows = sum(c_.element_rows() for c_ in caches) - vrows0 if elem else 0
    if elem:
        # HiKV Stage II reads whole K rows but only the V rows some head kept
        v_all = kv_bytes // 2
        alg_bytes = alg_bytes - v_all + vrows * w.d * w.elem_bytes
    if opts["world"] > 1:
        dist.barrier()
    clocks = sampler.stop() if sampler is not None else None
    step_ms = [e0.elapsed_time(e1) for (e0, e1) in ev]
    t_total = max_over_ranks(sum(step_ms) / 1e3, opts["world"], dev)
    stage(f"{w.name}: timed fused steps done")

    # ---- the same single-call steps, each after an L2 flush (cold code and
    # metadata as well as data) ----
    flushed = None
    if NC > 1 and opts.get("flushed_steps", 0) > 0:
        KF = opts["flushed_steps"]
        evf = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(KF)]
        for i in range(KF):
            flush.fill_(float(i))
            torch.cuda._sleep(spin_cycles)
            evf[i][0].record(stream)
            step_fused()
            evf[i][1].record(stream)
        torch.cuda.synchronize()
        msf = [a.elapsed_time(b) for a, b in evf]
        flushed = {"steps": KF, "ms_per_step": sum(msf) / KF, "steps_per_s": KF / (sum(msf) / 1e3),
                   "l2": "256 MB write before each step"}

    # ---- the same steps as three calls (append, decode_step, evict when due) ----
    ev3 = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(K3)]
    for i in range(K3):
        c_, r, ev_ = next_step()
        if NC == 1 and est < 2 * l2:
            flush.fill_(float(i))
        torch.cuda._sleep(spin_cycles)
        e0, e1, e2, e3 = ev3[i]
        e0.record(stream)
        c_.append(dks[r], dvs[r])
        e1.record(stream)
        c_.decode_step(dqs[r], out)
        e2.record(stream)
        if ev_:
            c_.evict()
        e3.record(stream)
    torch.cuda.synchronize()
    three = None
    if K3 > 0:
        ms3 = [e0.elapsed_time(e3) for (e0, e1, e2, e3) in ev3]
        dec3 = [e1.elapsed_time(e2) for (e0, e1, e2, e3) in ev3]
        three = {"steps": K3, "ms_per_step": sum(ms3) / K3, "steps_per_s": K3 / (sum(ms3) / 1e3),
                 "decode_kernel_us": 1e3 * sum(dec3) / K3}

    # ---- per-layer launches: one fused call per layer and step, as a model
    # whose layers run in turn would issue them ----
    per_layer = None
    if KL > 0 and L > 1:
        evl = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(KL)]
        pl_launch0 = sum(c_.kernel_launches() for c_ in caches)
        for i in range(KL):
            c_, r, ev_ = next_step()
            torch.cuda._sleep(spin_cycles + L * 40000)   # room to enqueue L calls
            e0, e1 = evl[i]
            e0.record(stream)
            for l in range(L):
                c_.step(dks[r][l:l + 1], dvs[r][l:l + 1], dqs[r][l:l + 1], out[l:l + 1], evict=ev_, layer0=l)
            e1.record(stream)
        torch.cuda.synchronize()
        msl = [e0.elapsed_time(e1) for (e0, e1) in evl]
        per_layer = {"steps": KL, "launches_per_step": (sum(c_.kernel_launches() for c_ in caches) - pl_launch0) / KL,
                     "ms_per_step": sum(msl) / KL, "steps_per_s": KL / (sum(msl) / 1e3)}

    # ---- e2e through the C ABI with pinned host buffers: every step copies
    # its k, v and q in (one packed copy) and the output back ----
    def flat(a):
        return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).reshape(a.shape[0], -1)
    packed = torch.cat([flat(ks), flat(vs), flat(qs)], dim=1).pin_memory()   # [R][k | v | q]
    nk, nq_ = flat(ks).shape[1], flat(qs).shape[1]
    in_dev = torch.empty(packed.shape[1], dtype=packed.dtype, device=dev)
    as_wdt = (lambda t: t.view(torch.bfloat16)) if w.dtype == "bf16" else (lambda t: t)
    k_dev = as_wdt(in_dev[:nk]).view(ks.shape[1:])
    v_dev = as_wdt(in_dev[nk:2 * nk]).view(vs.shape[1:])
    q_dev = as_wdt(in_dev[2 * nk:2 * nk + nq_]).view(qs.shape[1:])
    out_host = torch.empty(tuple(out.shape), dtype=out.dtype).pin_memory()
    torch.cuda.synchronize()
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e2e_ms = 0.0
    for i in range(Ke):
        c_, r, ev_ = next_step()
        if NC == 1 and est < 2 * l2:
            flush.fill_(float(i))
        e_start.record(stream)
        in_dev.copy_(packed[r], non_blocking=True)
        c_.step(k_dev, v_dev, q_dev, out, evict=ev_)
        out_host.copy_(out, non_blocking=True)
        e_end.record(stream)
        e_end.synchronize()
        e2e_ms += e_start.elapsed_time(e_end)
    h2d = packed[0].nbytes
    d2h = out_host.nbytes
    for c_ in caches:
        c_.device_status()
    lens = cache.lengths()
    for c_ in caches:
        c_.close()
    del dks, dvs, dqs, packed, in_dev, caches, cache
    stage(f"{w.name}: e2e steps done")

    # ---- read floor (context for the roofline fraction): a plain streaming
    # read, and a torch copy, of one step's algorithmic bytes from a flushed
    # L2, timed the same way as the steps ----
    def size_floor(nbytes, reps=20):
        """Plain reads (and a copy) of nbytes of cold data, cold the same way
        as the steps: NC buffers in turn, or one flushed buffer."""
        nb = max(16, nbytes // 16 * 16)
        bufs = [torch.empty(nb // 2, dtype=torch.bfloat16, device=dev).normal_() for _ in range(NC)]
        dst = torch.empty_like(bufs[0])
        sink = torch.zeros(1, dtype=torch.int32, device=dev)
        res = {}
        kernels = [(f"read_us_{c}cta", (lambda b, c=c: hk.read_floor(b, c, sink))) for c in (1, 2, 4)]
        kernels.append(("copy_us", lambda b: dst.copy_(b)))
        for name, fn in kernels:
            for b in bufs:
                fn(b)
            ts = []
            for i in range(reps):
                if NC == 1:
                    flush.fill_(float(i))
                torch.cuda._sleep(spin_cycles)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn(bufs[i % NC])
                b.record(stream)
                b.synchronize()
                ts.append(a.elapsed_time(b) * 1e3)
            res[name] = float(np.median(ts))
        res["read_us"] = min(v for k_, v in res.items() if k_.startswith("read_us_"))
        res["read_gbs"] = nb / res["read_us"] / 1e3
        del bufs, dst
        return res
    floor = size_floor(int(alg_bytes // K)) if K > 0 else None
    del flush
    torch.cuda.empty_cache()

    avg_s = t_total / K
    r = {"K": K, "Wu": Wu, "t_total": t_total, "avg_s": avg_s, "alg_bytes": alg_bytes, "kv_bytes": kv_bytes,
         "NC": NC, "flushed": flushed,
         "launches": launches, "dec_cfg": dec_cfg, "three": three, "per_layer": per_layer, "setup": setup,
         "clocks": clocks, "floor": floor, "lens": lens, "elem": elem, "vrows": vrows,
         "decode_inputs": f"{R} distinct steps" + (", cycled" if R < total_steps else ""),
         "e2e": ({"value": Ke / (e2e_ms / 1e3), "unit": "steps/s", "h2d_bytes_per_step": int(h2d),
                  "d2h_bytes_per_step": int(d2h), "steps": Ke} if Ke > 0 else None)}
    stage(f"{w.name}: read floor done")
    return r


def other_workloads(args, dev, peak, stage):
    """The other workloads and the 70B full-cache reference point, measured
    briefly in the same run."""
    import workloads as W
    out = []
    for key in OTHER_WORKLOADS:
        full = isinstance(key, str) and key.endswith("-full")
        w = W.WORKLOADS[int(str(key).split("-")[0])]
        seed = w.index
        K = 5 if full else args.other_steps
        opts = {"steps": K, "warmup": 3, "three_call_steps": 0, "per_layer_steps": 0 if full else 10,
                "e2e_steps": 3 if full else 10, "budgets": W.budgets(w, seed), "full_cache": full,
                "element_budget": 0, "prompt_source": "device", "spin_us": args.spin_us, "world": 1}
        t0 = time.time()
        r = measure(w, seed, dev, opts, stage)
        gpu_s = time.time() - t0
        achieved = r["alg_bytes"] / r["K"] / r["avg_s"] / 1e9
        e = {"config": workload_config(w, "workload", 0, full), "steps": r["K"],
             "steps_per_s": r["K"] / r["t_total"], "ms_per_step": r["avg_s"] * 1e3,
             "hbm_gbs": achieved, "frac": achieved / peak, "frac_nominal": achieved / 8000.0,
             "bytes_per_step": r["alg_bytes"] // r["K"],
             "retained_kv_gbs": r["kv_bytes"] / r["t_total"] / 1e9,
             "tokens_attended_per_unit_mean": float(r["lens"].mean()) + 1,
             "launches_per_step": r["launches"] / r["K"], "decode_launch": r["dec_cfg"],
             "read_floor": r["floor"], "step_over_read_floor": (r["avg_s"] * 1e6 / r["floor"]["read_us"])
             if r["floor"] else None,
             "per_layer_launches": r["per_layer"], "e2e": r["e2e"], "setup": r["setup"],
             "gpu_wall_s": gpu_s}
        if not args.no_cpu_baseline:
            t0 = time.time()
            val, cores, done, sample, _ = run_cpu_oracle(
                w, seed, 8, 1, budget_s=args.other_cpu_s, layers=[0],
                budgets=(np.full(w.layers * w.hkv, w.total_positions + 64, np.int32) if full else None))
            e["cpu_baseline"] = {"value": val, "unit": "steps/s", "cores": cores, "kind": "oracle", "sample": sample,
                                 "wall_s": time.time() - t0}
        out.append(e)
        stage(f"other workload {e['config']['workload']} done")
    return out


def bench_gpu(args):
    def stage(msg):
        if args.verbose:
            print(f"[bench {time.strftime('%H:%M:%S')}] {msg}", file=sys.stderr, flush=True)
    import torch
    import torch.distributed as dist
    import workloads as W

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.WORKLOADS[args.workload]
    if args.layers:   # the workload cut to its first L layers (small cases for profiling)
        w = w.with_(layers=min(args.layers, w.layers), name=f"{w.name}-first{min(args.layers, w.layers)}layers")
    if args.group:    # query heads per KV head: 1 runs the shape as multi-head attention
        w = w.with_(hq=w.hkv * args.group, name=f"{w.name}-group{args.group}")
    seed = w.index if args.seed is None else args.seed
    cfg_w = w
    gw = global_workload(w, world, args.scaling)
    g_budgets = schedule_budgets(gw, seed, args.schedule)
    l0, l1, b0, b1 = rank_shard(gw, world, rank, g_budgets)
    w = W.shard(gw, l0, l1, b0, b1) if world > 1 else gw
    budgets = g_budgets[l0 * gw.hkv:l1 * gw.hkv]
    L = w.layers
    opts = {"steps": args.steps, "warmup": args.warmup, "three_call_steps": args.three_call_steps,
            "per_layer_steps": args.per_layer_steps if args.per_layer_steps >= 0 else (0 if L == 1 else 100),
            "e2e_steps": args.e2e_steps, "budgets": budgets, "full_cache": args.full_cache,
            "element_budget": args.element_budget, "prompt_source": "host", "spin_us": args.spin_us,
            "world": world, "sampler": ClockSampler(gpu_id_for(local)), "flushed_steps": min(args.steps, 200),
            "l2_mode": args.l2}
    r = measure(w, seed, dev, opts, stage)
    K = r["K"]
    peaks, src = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    avg_s = r["avg_s"]
    achieved = r["alg_bytes"] / K / avg_s / 1e9
    elem = r["elem"]
    traffic = None
    try:
        with open(TRAFFIC_FILE) as f:
            tr = json.load(f)
        if tr.get("kernel_sha") == kernel_sha() and tr.get("workload") == w.name and not elem:
            traffic = tr.get("dram_bytes_per_launch")
    except (OSError, ValueError):
        pass
    value = whole_job_rate(world, K, r["t_total"], args.scaling)
    lens = r["lens"]
    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": K,
        "warmup": r["Wu"], "ms_per_step": r["t_total"] * 1e3 / K, "higher_is_better": True,
        "scaling": args.scaling, "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded)",
        "config": workload_config(cfg_w, args.schedule, elem if elem else 0, args.full_cache, world,
                                  args.scaling, args.l2),
        "workload_observed": {"tokens_attended_per_unit_max": int(lens.max()) + 1,
                              "tokens_attended_per_unit_mean": float(lens.mean()) + 1,
                              "decode_inputs": r["decode_inputs"], "units_rank0": int(lens.size),
                              "shard_rank0": {"layers": [l0, l1], "batch_rows": [b0, b1]}},
        "hbm_gbs_step": r["alg_bytes"] * world / r["t_total"] / 1e9,
        "retained_kv_gbs": r["kv_bytes"] * world / r["t_total"] / 1e9,
        "hbm_fraction_nominal": achieved / 8000.0,
        "roofline": {"kernel": ("k_decode (append + attention + importance + victim + evict, one launch)" if not elem
                                else "HiKV Stage II step (k_elem_order with the append, k_elem_span with the merge and the eviction in its last CTA per unit)"),
                     "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{src} hbm_gbs", "traffic": traffic,
                     "bytes_per_launch": r["alg_bytes"] // K, "avg_launch_us": avg_s * 1e6,
                     "launches_per_step": r["launches"] / K,
                     "frac_of_read_floor": (r["floor"]["read_us"] / (avg_s * 1e6)) if r["floor"] else None},
        "e2e": r["e2e"],
        "gpu_launches": r["launches"],
        "decode_launch": r["dec_cfg"],
        "three_call_path": r["three"],
        "flushed_l2_steps": r["flushed"],
        "stage2_v_rows_read_fraction": (r["vrows"] / max(1, r["kv_bytes"] // (2 * w.d * w.elem_bytes))) if elem
        else None,
        "per_layer_launches": r["per_layer"],
        "setup": r["setup"],
        "clocks": r["clocks"],
        "size_floor": ({"bytes": int(r["alg_bytes"] // K),
                        "kernels": "hikv_read_floor (plain 16-byte streaming loads, best of 1/2/4 CTAs per SM) "
                                   "and a torch copy of a buffer of one step's algorithmic bytes, cold the same "
                                   "way as the steps (as many buffers in turn as cache copies), median of 20",
                        **r["floor"], "step_us": avg_s * 1e6} if r["floor"] else None),
    }
    if rank == 0 and not args.no_cpu_baseline:
        val, cores, done, sample, single = run_cpu_oracle(w, seed, min(64, w.steps), 2, budget_s=20.0,
                                                          layers=oracle_sample_layers(w), budgets=budgets,
                                                          element_budget=elem, steps_1thread=16)
        line["cpu_baseline"] = {"value": val, "unit": "steps/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
        if single:
            line["cpu_baseline"]["value_1thread"] = single[0]
            line["cpu_baseline"]["sample_1thread"] = f"{single[1]} further steps of the same sample on one thread"
        stage("cpu baseline done")
    if rank == 0 and world == 1 and not args.no_other_workloads and args.workload == WORKLOAD_INDEX \
            and not args.layers and not args.group and not args.full_cache and not elem \
            and args.schedule in (None, "", "workload"):
        line["other_workloads"] = other_workloads(args, dev, peak, stage)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--scaling", default="weak", choices=["weak", "strong"],
                    help="N > 1: weak = the batch grows with the ranks (each rank as many units as one GPU "
                         "alone); strong = the configured workload's units shared out")
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--three-call-steps", type=int, default=500)
    ap.add_argument("--per-layer-steps", type=int, default=-1,
                    help="steps timed as one launch per layer (default 100 for multi-layer workloads)")
    ap.add_argument("--seed", type=int, default=None, help="input seed (default: the workload index)")
    ap.add_argument("--full-cache", action="store_true", help="budgets above the context: no eviction")
    ap.add_argument("--schedule", default="workload",
                    help='budgets: "workload", "pyramid:AVG:MIN" or "duo:FRAC"')
    ap.add_argument("--workload", type=int, default=WORKLOAD_INDEX,
                    help="workload index (default: the Llama-3-8B layer the metric is quoted on)")
    ap.add_argument("--layers", type=int, default=0,
                    help="cut the workload to its first L layers (profiling a smaller case; 0: all)")
    ap.add_argument("--group", type=int, default=0, choices=[0, 1, 2, 4, 8],
                    help="query heads per KV head (0: the workload's; 1: the shape as multi-head attention)")
    ap.add_argument("--spin-us", type=float, default=60.0)
    ap.add_argument("--impl", default="hikv", choices=["hikv", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="measure only the headline workload")
    ap.add_argument("--other-steps", type=int, default=20, help="timed steps of each other workload")
    ap.add_argument("--other-cpu-s", type=float, default=5.0, help="CPU-oracle seconds per other workload")
    ap.add_argument("--element-budget", type=int, default=0,
                    help="HiKV Stage II element budget B2 (0: exact attention)")
    ap.add_argument("--l2", default="auto", choices=["auto", "flush"],
                    help="cold data between timed steps: auto = inputs larger than L2 (cache copies in turn for "
                         "small steps), flush = a 256 MB write before every step")
    ap.add_argument("--verbose", action="store_true", help="stage markers on stderr")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_gpu(args)


if __name__ == "__main__":
    main()
