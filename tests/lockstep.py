"""Lockstep parity harness: CUDA library vs CPU oracle on the same seeded inputs.

The GPU cache runs the whole workload in the launch configuration the
benchmark uses (all layers per call).  The oracle runs a sample of layers
(all of them for small workloads) on the same inputs.  After every eviction
the retained position sets of the sampled units are compared: they must be
equal, except that a swap is accepted when the oracle's own scores of the
swapped tokens lie within 1e-6 relative of each other (near-ties); the oracle
is then resynced to the GPU's set so a near-tie cannot cascade.  Importance
and attention outputs are compared with the tolerances of the method's
statement: importance |d| <= 1e-4 |imp| + 1e-6 max|imp|; fp32 outputs per
(unit, head) row ||d||_inf <= 1e-5 max(||o||_inf, 1e-3); bf16 outputs
|d| <= 2e-2 elementwise (the statement's bound), and, tighter, within one
bf16 ulp of the larger of the two values (at least 2^-15): both sides sum in
at least fp32 and round once to bf16, so they can differ only where a
rounding boundary falls between their sums.  Elements more than one ulp of
the oracle's own value apart are counted.

HiKV Stage II rows whose chunk selection float32 rounding of the logits
could change (the oracle bounds each logit's rounding error) are compared
with every output an admissible selection gives: the GPU row must equal one
of them at the normal tolerance.
"""
from __future__ import annotations

import os
from dataclasses import dataclass, field

import numpy as np
import torch

import oracle
import workloads as W

TIE_REL = 1e-6
IMP_REL, IMP_ABS_FRAC = 1e-4, 1e-6
OUT_F32_REL, OUT_BF16_ABS = 1e-5, 2e-2
BF16_ULP_FLOOR = 2.0 ** -15


def bf16_ulp(x):
    """Spacing of bf16 values at |x| (8 significant bits): 2^(floor(log2|x|) - 7)."""
    _, e = np.frexp(np.abs(np.asarray(x, np.float64)))
    return np.ldexp(1.0, e - 8)


@dataclass
class Report:
    evictions_checked: int = 0
    near_tie_swaps: int = 0
    outputs_checked: int = 0
    importance_checked: int = 0
    max_out_err: float = 0.0
    max_imp_err_rel: float = 0.0
    bf16_over_1ulp: int = 0         # bf16 elements more than one ulp (of the oracle's value) apart
    max_out_ulps: float = 0.0       # largest bf16 difference in ulps of the larger value, where that ulp
                                    # is at least the 2^-15 floor
    stage2_near_tie_rows: int = 0   # HiKV Stage II rows matched against the admissible selections
    stage2_alt_matches: int = 0     # ... of which the GPU matched another selection than the exact one
    notes: list = field(default_factory=list)


def _to_dev(a: np.ndarray, dev):
    return W.to_torch(np.ascontiguousarray(a)).to(dev, non_blocking=False)


def _out_np(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy()


class Lockstep:
    def __init__(self, w: W.Workload, seed=None, sample_layers=None, cs=None, budgets=None,
                 device="cuda", layer_chunk=None, full_cache=False, page_tokens=64,
                 check_kv=True, full_twin_layers=None, pool_kernel=0, importance_mode=0, small_mode=None,
                 element_budget=0, prefill_band=0, pool_pages=0):
        import importance_aware_kv_gb300 as hk
        self.hk = hk
        self.w = w
        self.seed = w.index if seed is None else seed
        self.dev = torch.device(device)
        self.budgets = W.budgets(w, self.seed) if budgets is None else np.asarray(budgets, np.int32)
        if full_cache:
            self.budgets = np.full_like(self.budgets, w.total_positions)
        self.sample = list(range(w.layers)) if sample_layers is None else list(sample_layers)
        self.layer_chunk = layer_chunk or max(1, min(w.layers, int(2e9 // max(1, W.kv_bytes(
            w.batch, w.prompt, 1, w.hkv, w.d, w.elem_bytes)))))
        self.check_kv = check_kv
        self.pool = pool_kernel
        self.band = prefill_band   # > 0: HiKV banded prefill scores instead of the observation window
        if cs is not None:
            os.environ["HIKV_DECODE_CS"] = str(cs)
        if small_mode is not None:
            os.environ["HIKV_DECODE_SMALL"] = str(small_mode)
        try:
            self.cache = hk.Cache(hk.CacheConfig(
                w.layers, w.batch, w.hq, w.hkv, w.d, w.dtype, w.sink, w.window,
                self.budgets, w.total_positions, page_tokens=page_tokens,
                max_window_queries=max(32, w.nq), pool_kernel=pool_kernel,
                importance_mode=importance_mode, element_budget=element_budget,
                band_scoring=1 if prefill_band > 0 else 0, pool_pages=pool_pages))
        finally:
            if cs is not None:
                os.environ.pop("HIKV_DECODE_CS", None)
            os.environ.pop("HIKV_DECODE_SMALL", None)
        bs = np.concatenate([self.budgets[l * w.hkv:(l + 1) * w.hkv] for l in self.sample])
        self.ora = oracle.Oracle(len(self.sample), w.batch, w.hq, w.hkv, w.d, w.sink, w.window, bs,
                                 out_bf16=(w.dtype == "bf16"), threads=os.cpu_count() or 1)
        self.ora.set_recent_only(importance_mode == 1)
        self.ora.set_element_budget(element_budget)
        self.elem = 0 < element_budget < w.d
        self.rep = Report()
        self.upl = w.batch * w.hkv
        # optional twin: a no-eviction cache fed the same inputs, checked on
        # `full_twin_layers` against an oracle whose budget exceeds the context
        self.twin = None
        if full_twin_layers is not None:
            self.twin = Lockstep.__new__(Lockstep)
            self.twin.__dict__.update(dict(hk=hk, w=w, seed=self.seed, dev=self.dev,
                                           budgets=np.full_like(self.budgets, w.total_positions),
                                           sample=list(full_twin_layers), layer_chunk=self.layer_chunk,
                                           check_kv=False, rep=Report(), upl=self.upl, twin=None,
                                           pool=pool_kernel, elem=False, band=0))
            self.twin.cache = hk.Cache(hk.CacheConfig(
                w.layers, w.batch, w.hq, w.hkv, w.d, w.dtype, w.sink, w.window, self.twin.budgets,
                w.total_positions, page_tokens=page_tokens, max_window_queries=max(32, w.nq),
                pool_kernel=pool_kernel))
            self.twin.ora = oracle.Oracle(len(self.twin.sample), w.batch, w.hq, w.hkv, w.d, w.sink,
                                          w.window, np.full(len(self.twin.sample) * w.hkv, w.total_positions),
                                          out_bf16=(w.dtype == "bf16"), threads=os.cpu_count() or 1)

    # ------------------------------------------------------------------
    def prefill(self):
        w = self.w
        for l0 in range(0, w.layers, self.layer_chunk):
            nl = min(self.layer_chunk, w.layers - l0)
            k, v = W.gen_kv(w, l0, nl, 0, w.prompt, self.seed)
            dk, dv = _to_dev(k, self.dev), _to_dev(v, self.dev)
            for ls in self._all():
                ls.cache.append(dk, dv, layer0=l0)
                for si, l in enumerate(ls.sample):
                    if l0 <= l < l0 + nl:
                        ls.ora.append(si, W.to_f32(k[l - l0:l - l0 + 1]), W.to_f32(v[l - l0:l - l0 + 1]))
            del k, v, dk, dv
        torch.cuda.synchronize()
        for ls in self._all():
            if ls.band > 0:
                # HiKV: every prompt query, each token scored over its own band
                for l0 in range(0, w.layers, self.layer_chunk):
                    nl = min(self.layer_chunk, w.layers - l0)
                    q = W.gen_q(w, l0, nl, 0, w.prompt, self.seed)
                    ls.cache.score_band(_to_dev(q, self.dev), ls.band, layer0=l0)
                    for si, l in enumerate(ls.sample):
                        if l0 <= l < l0 + nl:
                            ls.ora.score_band(si, W.to_f32(q[l - l0:l - l0 + 1]), ls.band)
                    del q
            else:
                q = W.gen_q(w, 0, w.layers, w.prompt - w.nq, w.nq, self.seed)
                ls.cache.score_window(_to_dev(q, self.dev))
                for si, l in enumerate(ls.sample):
                    ls.ora.score_window(si, W.to_f32(q[l:l + 1]))
                    ls.ora.pool_importance(si, 1, getattr(ls, "pool", 0))
            ls.compare_state(after_evict=False)
            ls.cache.evict()
            for si in range(len(ls.sample)):
                ls.ora.evict(si, 1)
            ls.compare_state(after_evict=True, kv=True)

    def _all(self):
        return [self] + ([self.twin] if self.twin is not None else [])

    def _decode_inputs(self):
        w = self.w
        k, v = W.gen_kv(w, 0, w.layers, w.prompt, w.steps, self.seed)
        q = W.gen_q(w, 0, w.layers, w.prompt, w.steps, self.seed)
        # per-step contiguous slices: [steps][L][B][H][1][d] and [steps][L][B][Hq][d]
        ks = np.ascontiguousarray(np.moveaxis(k, 3, 0)[:, :, :, :, None, :])
        vs = np.ascontiguousarray(np.moveaxis(v, 3, 0)[:, :, :, :, None, :])
        qs = np.ascontiguousarray(np.moveaxis(q, 3, 0))
        return ks, vs, qs

    def decode(self, steps=None, compare_every=1, fused=False, per_layer=False):
        """Run the decode steps; fused=True drives each step through the
        single append+decode+evict call instead of the three calls;
        per_layer=True makes that one fused call per layer, back to back on
        the stream, as a model's layers issue them (consecutive launches on
        disjoint units may overlap by programmatic dependent launch)."""
        w = self.w
        steps = w.steps if steps is None else steps
        ks, vs, qs = self._decode_inputs()
        dks, dvs, dqs = _to_dev(ks, self.dev), _to_dev(vs, self.dev), _to_dev(qs, self.dev)
        out = torch.empty_like(dqs[0])
        for s in range(steps):
            evict_now = (s + 1) % w.evict_every == 0
            for ls in self._all():
                if fused and per_layer:
                    for l in range(w.layers):
                        ls.cache.step(dks[s][l:l + 1], dvs[s][l:l + 1], dqs[s][l:l + 1], out[l:l + 1],
                                      evict=evict_now, layer0=l)
                elif fused:
                    ls.cache.step(dks[s], dvs[s], dqs[s], out, evict=evict_now)
                else:
                    ls.cache.append(dks[s], dvs[s])
                    ls.cache.decode_step(dqs[s], out)
                    if evict_now:
                        ls.cache.evict()
                for si, l in enumerate(ls.sample):
                    ls.ora.append(si, W.to_f32(ks[s, l:l + 1]), W.to_f32(vs[s, l:l + 1]))
                ora_out = [ls.ora.decode(si, W.to_f32(qs[s, l:l + 1])) for si, l in enumerate(ls.sample)]
                ties = [ls.ora.stage2_near_ties(si, 1)[0] if ls.elem else None for si in range(len(ls.sample))]
                alts = [ls._stage2_alternatives(si, t) for si, t in enumerate(ties)]
                if evict_now:
                    for si in range(len(ls.sample)):
                        ls.ora.evict(si, 1)
                if (s % compare_every == 0) or s == steps - 1:
                    got = _out_np(out)
                    for si, l in enumerate(ls.sample):
                        ls.compare_out(got[l], ora_out[si][0], s, alternatives=alts[si])
                if evict_now:
                    ls.compare_state(after_evict=True)
        for ls in self._all():
            ls.compare_state(after_evict=False, kv=True)
            ls.cache.device_status()
        return self.rep

    # ------------------------------------------------------------------
    def _stage2_alternatives(self, si, ties):
        """{(b, head): [count][d] admissible outputs} for the near-tie heads
        of oracle layer si at the latest Stage II step (None: exact)."""
        if ties is None or not ties.any():
            return None
        out = {}
        for b, h in zip(*np.nonzero(ties)):
            if ties[b, h] == 2:
                raise AssertionError(f"Stage II head ({b}, {h}): too many admissible selections to list")
            out[(int(b), int(h))] = self.ora.stage2_alternatives(si, int(b), int(h))
        return out

    def _rows_ok(self, got, want):
        """Per-row check at the dtype's tolerance: (ok [rows], score [rows]),
        score = error / bound for fp32, largest |d| for bf16."""
        if self.w.dtype == "f32":
            err = np.abs(got - want).max(axis=1)
            bound = OUT_F32_REL * np.maximum(np.abs(want).max(axis=1), 1e-3)
            return err <= bound, err / bound
        d = np.abs(got.astype(np.float64) - want.astype(np.float64))
        tol = np.maximum(bf16_ulp(np.maximum(np.abs(got), np.abs(want))), BF16_ULP_FLOOR)
        ok = np.all((d <= tol) & (d <= OUT_BF16_ABS), axis=1)
        return ok, d.max(axis=1)

    def compare_out(self, got, want, step, alternatives=None):
        """got, want: [B][Hq][d].  alternatives: {(b, head): [count][d]} for
        Stage II heads whose selection float32 rounding could change; such a
        row must match one of its admissible outputs."""
        w = self.w
        rg = got.reshape(-1, w.d)
        rw = want.reshape(-1, w.d).copy()
        if alternatives:
            for (b, h), alts in alternatives.items():
                r = b * w.hq + h
                ok, _ = self._rows_ok(np.repeat(rg[r:r + 1], len(alts), axis=0), alts)
                if not ok.any():
                    raise AssertionError(f"step {step}: Stage II row (b={b}, head={h}) matches none of its "
                                         f"{len(alts)} admissible outputs")
                j = int(np.argmax(ok))
                self.rep.stage2_near_tie_rows += 1
                if not np.array_equal(alts[j], rw[r]):
                    self.rep.stage2_alt_matches += 1
                rw[r] = alts[j]   # checked: compare the rest against it
        ok, score = self._rows_ok(rg, rw)
        if not ok.all():
            i = int(np.argmin(ok))
            err = float(np.abs(rg[i].astype(np.float64) - rw[i]).max())
            raise AssertionError(f"step {step}: {w.dtype} output row {i} (b={i // w.hq}, head={i % w.hq}) "
                                 f"err {err:.3e} beyond tolerance")
        if w.dtype == "f32":
            self.rep.max_out_err = max(self.rep.max_out_err, float(score.max()))
        else:
            d = np.abs(rg.astype(np.float64) - rw.astype(np.float64))
            self.rep.max_out_err = max(self.rep.max_out_err, float(d.max()))
            ulp_big = bf16_ulp(np.maximum(np.abs(rg), np.abs(rw)))
            ruled = ulp_big >= BF16_ULP_FLOOR   # elements the one-ulp check governs (not the floor)
            if ruled.any():
                self.rep.max_out_ulps = max(self.rep.max_out_ulps, float((d[ruled] / ulp_big[ruled]).max()))
            self.rep.bf16_over_1ulp += int(np.count_nonzero(d > bf16_ulp(rw)))
        self.rep.outputs_checked += got.size

    def compare_state(self, after_evict: bool, kv: bool = False):
        w = self.w
        lens_host = self.cache.lengths()
        for si, l in enumerate(self.sample):
            lengths, positions, importance, kk, vv = self.cache.gather(
                l, 1, with_kv=kv and self.check_kv and si == 0)
            lengths = lengths.cpu().numpy()
            positions = positions.cpu().numpy()
            importance = importance.cpu().numpy()
            for j in range(self.upl):
                ou = si * self.upl + j
                gu = l * self.upl + j
                n = int(lengths[j])
                assert n == int(lens_host[gu]), f"unit {gu}: device length {n} != host mirror {lens_host[gu]}"
                gp = positions[j, :n]
                gi = importance[j, :n]
                assert np.all(np.diff(gp) > 0), f"unit {gu}: positions not strictly ascending"
                op, oi = self.ora.state(ou)
                if after_evict:
                    self._compare_sets(ou, gu, gp, op, oi)
                    op, oi = self.ora.state(ou)
                assert np.array_equal(gp, op), f"unit {gu}: retained positions differ"
                tol = IMP_REL * np.abs(oi) + IMP_ABS_FRAC * (np.abs(oi).max() if n else 0.0)
                err = np.abs(gi - oi)
                if np.any(err > tol):
                    i = int(np.argmax(err - tol))
                    raise AssertionError(f"unit {gu}: importance at pos {gp[i]}: gpu {gi[i]!r} oracle {oi[i]!r}")
                rel = err / np.maximum(np.abs(oi), 1e-30)
                self.rep.max_imp_err_rel = max(self.rep.max_imp_err_rel, float(rel.max()) if n else 0.0)
                self.rep.importance_checked += n
                if kk is not None and si == 0 and j in (0, self.upl - 1):
                    self._check_kv(l, j, gp, kk[j, :n], vv[j, :n])
            if after_evict:
                self.rep.evictions_checked += self.upl

    def _check_kv(self, layer, j, positions, kk, vv):
        """Retained K/V rows must be byte-identical to the generated inputs."""
        w = self.w
        b, g = j // w.hkv, j % w.hkv
        ka, va = W.gen_kv_unit(w, layer, b, g, 0, w.total_positions, self.seed)
        want_k = ka[positions]
        want_v = va[positions]
        got_k = kk.cpu()
        got_v = vv.cpu()
        if w.dtype == "bf16":
            got_k = got_k.view(torch.int16).numpy().view(np.uint16)
            got_v = got_v.view(torch.int16).numpy().view(np.uint16)
        else:
            got_k, got_v = got_k.numpy(), got_v.numpy()
        assert np.array_equal(got_k, want_k), f"layer {layer} unit {j}: K rows corrupted"
        assert np.array_equal(got_v, want_v), f"layer {layer} unit {j}: V rows corrupted"

    def _compare_sets(self, ou, gu, gp, op, oi):
        gs, os_ = set(gp.tolist()), set(op.tolist())
        if gs == os_:
            return
        gpu_only = np.array(sorted(gs - os_), dtype=np.int32)
        ora_only = np.array(sorted(os_ - gs), dtype=np.int32)
        assert len(gpu_only) == len(ora_only), f"unit {gu}: retained sizes differ"
        ep, ei = self.ora.last_evicted(ou)
        emap = dict(zip(ep.tolist(), ei.tolist()))
        rmap = dict(zip(op.tolist(), oi.tolist()))
        missing = [p for p in gpu_only.tolist() if p not in emap]
        assert not missing, f"unit {gu}: GPU kept positions {missing[:5]} the oracle never had"
        a = np.array([emap[p] for p in gpu_only.tolist()], dtype=np.float64)   # oracle evicted
        b = np.array([rmap[p] for p in ora_only.tolist()], dtype=np.float64)   # oracle kept
        hi = max(a.max(), b.max())
        spread = b.max() - a.min()
        if spread > TIE_REL * hi:
            raise AssertionError(
                f"unit {gu}: retained sets differ beyond near-ties: GPU kept {gpu_only[:4].tolist()} "
                f"(oracle imp {a[:4].tolist()}), oracle kept {ora_only[:4].tolist()} (imp {b[:4].tolist()})")
        self.rep.near_tie_swaps += len(gpu_only)
        self.ora.resync(ou, gp)
