"""GPU-vs-oracle parity harness (test infrastructure).

The CUDA path (through the C ABI, ``kv_cache_eviction_step_gb300``) runs every unit of a workload
in the real launch shape; the CPU oracle runs a chosen subset of units on the same seeded inputs,
step by step. Per step the harness compares the attention outputs (within the dtype's tolerance)
and the eviction decisions (exactly). Where the oracle's two lowest candidate scores differ by less
than ``TIE_REL`` (relative) the decision is a logged near-tie: the oracle follows the GPU's choice
if, and only if, that choice is one of the near-tied candidates, so that one benign tie does not
desynchronise every later step. Every near tie is logged with its step, unit and gap. Anything
else is a mismatch: there is no wider class of adopted decisions (the oracle's error-bound class is
given the same threshold, so it stays empty, and the report asserts that it does).
"""

from __future__ import annotations

import dataclasses

import numpy as np

import oracle
import synth

TIE_REL = 1e-6  # near-tie threshold on scores (relative): the only decisions the oracle may adopt
ERR_REL = TIE_REL  # no wider adoption class
OUT_TOL = {"bf16": 2e-2, "f32": 1e-5}


def score_rtol(steps: int) -> float:
    """Relative tolerance of a float32 accumulated score after ``steps`` additions: each addition
    rounds once on each side (2^-24 each) and the GPU's float32 p_j differs from the oracle's
    float64-rounded p_j by a few ulps; the bound grows linearly in the worst case."""
    return 1e-6 + 8.0 * (steps + 1) * 2.0 ** -24


@dataclasses.dataclass
class Report:
    workload: str
    units_checked: int
    steps: int
    decisions: int = 0
    near_ties: int = 0
    error_bound_ties: int = 0
    mismatches: int = 0
    prefill_near_ties: int = 0
    prefill_error_bound: int = 0
    prefill_mismatches: int = 0
    max_out_err: float = 0.0
    max_score_rel_err: float = 0.0
    max_prefill_out_err: float = 0.0
    topk: bool = False  # scores hold one step's weight, not a running sum
    notes: list = dataclasses.field(default_factory=list)
    near_tie_log: list = dataclasses.field(default_factory=list)  # (t or "prefill", unit, gap, adopted)
    min_decision_gap: float = float("inf")  # smallest oracle gap among decisions the GPU matched

    def ok(self) -> bool:
        return (self.mismatches == 0 and self.prefill_mismatches == 0 and self.error_bound_ties == 0
                and self.prefill_error_bound == 0 and not self.notes)

    def summary(self) -> str:
        ties = ", ".join(f"{t}/u{u}: gap {g:.2e}{' (adopted)' if a else ''}"
                         for t, u, g, a in self.near_tie_log[:20])
        return (f"{self.workload}: {self.mismatches} mismatches / {self.decisions} decisions, "
                f"near ties {self.near_ties} [{ties}], error-bound {self.error_bound_ties}, "
                f"prefill mismatches {self.prefill_mismatches}, prefill near ties "
                f"{self.prefill_near_ties}, prefill error-bound {self.prefill_error_bound}, "
                f"smallest matched gap {self.min_decision_gap:.2e}, max out err {self.max_out_err:.2e}, "
                f"max prefill out err {self.max_prefill_out_err:.2e}, max score rel err "
                f"{self.max_score_rel_err:.2e}, notes {self.notes}")


def check(rep: Report) -> None:
    """The parity bar: evictions and slot maps exact except at logged near ties (< TIE_REL),
    outputs within the dtype's tolerance, no adoption outside TIE_REL."""
    msg = rep.summary()
    print(msg)
    assert rep.ok(), msg


def dims_of(w: synth.Workload):
    import kv_cache_eviction_step_gb300 as h2o
    return h2o.Dims(units_b=w.units_b, heads=w.heads, head_dim=w.head_dim, budget=w.budget,
                    k_heavy=w.k_heavy, k_local=w.k_local,
                    dtype=h2o.F32 if w.dtype == "f32" else h2o.BF16)


def to_device(a: np.ndarray, dtype: str):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16) if a.dtype == np.uint16 else
                         np.ascontiguousarray(a))
    if a.dtype == np.uint16:
        t = t.view(torch.bfloat16)
    return t.cuda()


def to_host(t, dtype: str) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def widen(a: np.ndarray) -> np.ndarray:
    return synth.bf16_bits_to_f32(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


def run(w: synth.Workload, check_units=None, steps: int | None = None, seed: int = synth.DEFAULT_SEED,
        chunk_steps: int = 4096, state_every: int = 0, property_checks=None,
        policy: tuple[int, int, int] | None = None, prefill_out: bool = False,
        e4m3: bool = False) -> Report:
    """Run ``steps`` decode steps (default: all) of workload ``w`` on the GPU for every unit, and the
    oracle in lockstep on ``check_units`` (default: all units). ``policy`` = (kind, n_sink, stride)
    runs both sides under that eviction policy (None: H2O through the plain entry points).
    ``prefill_out`` builds the cache with h2o_prefill_forward and also compares the prompt's
    attention output with the oracle's on the checked units. ``e4m3`` runs both sides with the
    quantised (E4M3 codes + per-row scales) cache; codes and scales must then match bit for bit."""
    import torch

    import kv_cache_eviction_step_gb300 as h2o

    steps = w.decode_steps if steps is None else steps
    if state_every:
        chunk_steps = min(chunk_steps, state_every)  # the GPU state is read at chunk ends
    U, D, P, k = w.units, w.head_dim, w.prompt_len, w.budget
    check_units = np.arange(U) if check_units is None else np.asarray(check_units)
    rep = Report(w.name, len(check_units), steps)
    dims = dims_of(w)
    cache = h2o.H2OCache(dims, P, policy=None if policy is None else h2o.Policy(*policy), e4m3=e4m3)
    rep.topk = policy is not None and policy[0] == oracle.POLICY_TOPK

    # Prefill for every unit on the GPU.
    prompt = synth.generate(w, seed, steps=0)
    q, kk, v = (to_device(a, w.dtype) for a in (prompt.q_prompt, prompt.k_prompt, prompt.v_prompt))
    pout = torch.empty_like(q) if prefill_out else None
    cache.prefill(q, kk, v, out=pout)
    del q, kk, v
    torch.cuda.synchronize()
    assert h2o.h2o_get_device_error() == 0
    if prefill_out and len(check_units) > 0:
        got = widen(to_host(pout, w.dtype))[check_units]
        ref = oracle.prefill_attention(prompt.q_prompt[check_units], prompt.k_prompt[check_units],
                                       prompt.v_prompt[check_units])
        rep.max_prefill_out_err = float(np.max(np.abs(got - ref)))
        if rep.max_prefill_out_err > OUT_TOL[w.dtype]:
            rep.notes.append(f"prefill output error {rep.max_prefill_out_err:.3e}")
    del pout

    # Oracle prefill on the checked units, following the GPU's kept set only at near ties.
    follow = len(check_units) > 0
    orc = oracle.Oracle(k, w.k_heavy, w.k_local,
                        policy=None if policy is None else oracle.Policy(*policy))
    st = orc.new_state(len(check_units), D, synth.storage_dtype(w), e4m3=e4m3)
    if follow:
        gpu_pos = to_host(cache.slot_pos, "i32")[check_units]
        _, pinfo = orc.prefill_select(prompt.q_prompt[check_units], prompt.k_prompt[check_units],
                                      prompt.v_prompt[check_units], st, prefer_pos=gpu_pos,
                                      tie_rel=TIE_REL, err_rel=ERR_REL)
        compare_prefill(rep, pinfo, check_units)
        compare_state(rep, w, cache, st, check_units, 0)
    del prompt

    idx = torch.as_tensor(check_units, device="cuda", dtype=torch.long)
    s0 = 0
    while s0 < steps:
        ns = min(chunk_steps, steps - s0)
        chunk = synth.generate(w, seed, step0=s0, steps=ns, prompt=False)
        dq, dk, dv = (to_device(a, w.dtype) for a in (chunk.q_dec, chunk.k_dec, chunk.v_dec))
        outs = torch.empty((ns, len(check_units), D), dtype=cache.dtype, device="cuda")
        evs = torch.empty((ns, U), dtype=torch.int32, device="cuda")
        evp = torch.empty((ns, U), dtype=torch.int32, device="cuda")
        for s in range(ns):
            cache.step(dq[s], dk[s], dv[s], evicted_slot=evs[s], evicted_pos=evp[s])
            if follow:
                outs[s] = cache.out.index_select(0, idx)
        torch.cuda.synchronize()
        err = h2o.h2o_get_device_error()
        if err:
            rep.notes.append(f"device error word {err}")
            return rep
        outs_h = widen(to_host(outs, w.dtype))
        evs_h, evp_h = to_host(evs, "i32"), to_host(evp, "i32")
        for s in range(ns if follow else 0):
            t = P + s0 + s
            o_out, o_es, o_ep, _, infos = orc.decode_step(
                t, chunk.q_dec[s][check_units], chunk.k_dec[s][check_units],
                chunk.v_dec[s][check_units], st, prefer_victim=evs_h[s][check_units],
                tie_rel=TIE_REL, err_rel=ERR_REL)
            compare_step(rep, w.dtype, t, check_units, outs_h[s], evs_h[s][check_units],
                         evp_h[s][check_units], o_out, o_es, o_ep, infos)
        if follow and state_every:
            compare_state(rep, w, cache, st, check_units, s0 + ns)
        if property_checks is not None:
            property_checks(cache, P + s0 + ns - 1)
        s0 += ns
        del dq, dk, dv, outs, evs, evp
    if follow:
        compare_state(rep, w, cache, st, check_units, steps)
    return rep


def compare_prefill(rep: Report, pinfo, units) -> None:
    """The prefill's kept sets: exact, except at a logged near tie (< TIE_REL) at the boundary."""
    for j, i in enumerate(pinfo):
        rep.prefill_near_ties += i.kind == oracle.NEAR_TIE
        rep.prefill_error_bound += i.kind == oracle.ERROR_BOUND
        rep.prefill_mismatches += i.kind == oracle.REJECTED
        if i.kind == oracle.NEAR_TIE or (i.kind == oracle.RULE and 0 < i.gap_rel < TIE_REL):
            rep.near_tie_log.append(("prefill", int(units[j]), float(i.gap_rel),
                                     i.kind == oracle.NEAR_TIE))
        if i.kind == oracle.REJECTED and len(rep.notes) < 10:
            rep.notes.append(f"prefill unit {units[j]}: kept set differs (boundary gap {i.gap_rel:.2e})")


def run_segments(w: synth.Workload, check_units, seg_len: int, seed: int = synth.DEFAULT_SEED,
                 chunk_steps: int = 4096, property_checks=None, threads: int | None = None) -> Report:
    """Every decode step of a long run checked against the oracle, with the oracle's work spread over
    the host's cores. The GPU runs the whole workload (every unit, every step) in the launch shape of
    ``run``, recording the checked units' outputs and evictions at every step and their cache state
    every ``seg_len`` steps. The oracle then follows each checked unit through consecutive segments of
    ``seg_len`` steps, in parallel: the first starts from the oracle's own prefill; every later one
    from the GPU's state at its first step, which the previous segment's oracle state must match
    (slot map and K/V rows exactly, scores within the float32 tolerance of that segment's additions).
    Within a segment, evictions and outputs are compared at every step as in ``run``. The only
    difference from one unbroken oracle trajectory: at each segment boundary the oracle continues
    from the GPU's float32 scores rather than its own (after checking that the two agree)."""
    import concurrent.futures as cf
    import os

    import torch

    import kv_cache_eviction_step_gb300 as h2o

    steps = w.decode_steps
    assert seg_len % chunk_steps == 0 or chunk_steps % seg_len == 0
    chunk_steps = min(chunk_steps, seg_len)  # snapshots are taken at chunk ends
    U, D, P, k = w.units, w.head_dim, w.prompt_len, w.budget
    check_units = np.asarray(check_units)
    nc = len(check_units)
    dims = dims_of(w)
    cache = h2o.H2OCache(dims, P)
    gpu = Report(w.name, nc, steps)

    prompt = synth.generate(w, seed, steps=0)
    q, kk, v = (to_device(a, w.dtype) for a in (prompt.q_prompt, prompt.k_prompt, prompt.v_prompt))
    cache.prefill(q, kk, v)
    del q, kk, v
    torch.cuda.synchronize()
    assert h2o.h2o_get_device_error() == 0
    snaps = {0: snapshot(w, cache, check_units)}
    prompt_c = (prompt.q_prompt[check_units], prompt.k_prompt[check_units], prompt.v_prompt[check_units])
    del prompt
    out_h = np.empty((steps, nc, D), dtype=synth.storage_dtype(w))
    es_h = np.empty((steps, nc), dtype=np.int32)
    ep_h = np.empty((steps, nc), dtype=np.int32)
    idx = torch.as_tensor(check_units, device="cuda", dtype=torch.long)
    s0 = 0
    while s0 < steps:
        ns = min(chunk_steps, steps - s0)
        chunk = synth.generate(w, seed, step0=s0, steps=ns, prompt=False)
        dq, dk, dv = (to_device(a, w.dtype) for a in (chunk.q_dec, chunk.k_dec, chunk.v_dec))
        del chunk
        outs = torch.empty((ns, nc, D), dtype=cache.dtype, device="cuda")
        evs = torch.empty((ns, U), dtype=torch.int32, device="cuda")
        evp = torch.empty((ns, U), dtype=torch.int32, device="cuda")
        for s in range(ns):
            cache.step(dq[s], dk[s], dv[s], evicted_slot=evs[s], evicted_pos=evp[s])
            outs[s] = cache.out.index_select(0, idx)
        torch.cuda.synchronize()
        err = h2o.h2o_get_device_error()
        if err:
            gpu.notes.append(f"device error word {err}")
            return gpu
        out_h[s0:s0 + ns] = to_host(outs, w.dtype)
        es_h[s0:s0 + ns] = to_host(evs, "i32")[:, check_units]
        ep_h[s0:s0 + ns] = to_host(evp, "i32")[:, check_units]
        s0 += ns
        if s0 % seg_len == 0 or s0 == steps:
            snaps[s0] = snapshot(w, cache, check_units)
        if property_checks is not None:
            property_checks(cache, P + s0 - 1)
        del dq, dk, dv, outs, evs, evp

    orc = oracle.Oracle(k, w.k_heavy, w.k_local)
    bounds = sorted(snaps)

    def one(job):
        j, a, b = job
        u = check_units[j:j + 1]
        rep = Report(w.name, 1, b - a)
        st = orc.new_state(1, D, synth.storage_dtype(w))
        if a == 0:
            _, pinfo = orc.prefill_select(*(x[j:j + 1] for x in prompt_c), st,
                                          prefer_pos=snaps[0]["slot_pos"][j:j + 1],
                                          tie_rel=TIE_REL, err_rel=ERR_REL)
            compare_prefill(rep, pinfo, u)
            compare_snapshot(rep, {n: x[j:j + 1] for n, x in snaps[0].items()}, st, 0, 0)
        else:
            for n in ("slot_pos", "k_cache", "v_cache", "scores"):
                getattr(st, n)[...] = snaps[a][n][j:j + 1]
        x = synth.generate(w, seed, units=u, step0=a, steps=b - a, prompt=False, threads=1)
        for s in range(a, b):
            o_out, o_es, o_ep, _, infos = orc.decode_step(
                P + s, x.q_dec[s - a], x.k_dec[s - a], x.v_dec[s - a], st,
                prefer_victim=es_h[s, j:j + 1], tie_rel=TIE_REL, err_rel=ERR_REL)
            compare_step(rep, w.dtype, P + s, u, widen(out_h[s, j:j + 1]), es_h[s, j:j + 1],
                         ep_h[s, j:j + 1], o_out, o_es, o_ep, infos)
        compare_snapshot(rep, {n: x[j:j + 1] for n, x in snaps[b].items()}, st, b, b - a)
        return rep

    jobs = [(j, a, b) for j in range(nc) for a, b in zip(bounds[:-1], bounds[1:])]
    jobs.sort(key=lambda jb: -(jb[2] - jb[1]))
    with cf.ThreadPoolExecutor(threads or os.cpu_count() or 1) as ex:
        reports = list(ex.map(one, jobs))
    rep = merge([gpu] + reports, w.name, nc, steps)
    return rep


def compare_step(rep: Report, dtype: str, t: int, units, gpu_out, gpu_es, gpu_ep, o_out, o_es, o_ep,
                 infos) -> None:
    """One decode step of the checked units: outputs within the dtype's tolerance; eviction slot and
    position exact, except at a logged near tie (< TIE_REL) where the oracle took the GPU's choice.
    gpu_out: float64 [units, D]; gpu_es / gpu_ep: [units]."""
    e = float(np.max(np.abs(gpu_out - o_out)))
    rep.max_out_err = max(rep.max_out_err, e)
    if e > OUT_TOL[dtype] and len(rep.notes) < 10:
        rep.notes.append(f"t={t}: output error {e:.3e}")
    for j, inf in enumerate(infos):
        if inf.kind == oracle.NO_EVICTION:
            if gpu_es[j] != -1 or gpu_ep[j] != -1:
                rep.mismatches += 1
            continue
        rep.decisions += 1
        rep.near_ties += inf.kind == oracle.NEAR_TIE
        rep.error_bound_ties += inf.kind == oracle.ERROR_BOUND
        if inf.kind == oracle.NEAR_TIE or (inf.kind == oracle.RULE and 0 < inf.gap_rel < TIE_REL):
            rep.near_tie_log.append((t, int(units[j]), float(inf.gap_rel), inf.kind == oracle.NEAR_TIE))
        elif inf.kind == oracle.RULE and inf.gap_rel > 0:
            rep.min_decision_gap = min(rep.min_decision_gap, float(inf.gap_rel))
        if inf.kind == oracle.REJECTED or o_ep[j] != gpu_ep[j] or o_es[j] != gpu_es[j]:
            rep.mismatches += 1
            if len(rep.notes) < 10:
                rep.notes.append(f"t={t} unit {units[j]}: gpu victim {gpu_es[j]}, oracle {o_es[j]} "
                                 f"(kind {oracle.KIND_NAMES[inf.kind]}, gap {inf.gap_rel:.2e})")


def merge(reports: list, workload: str, units_checked: int, steps: int) -> Report:
    """One report from the reports of separate pieces of a run (counts added, extremes kept)."""
    rep = Report(workload, units_checked, steps)
    for r in reports:
        for f in ("decisions", "near_ties", "error_bound_ties", "mismatches", "prefill_near_ties",
                  "prefill_error_bound", "prefill_mismatches"):
            setattr(rep, f, getattr(rep, f) + getattr(r, f))
        for f in ("max_out_err", "max_score_rel_err", "max_prefill_out_err"):
            setattr(rep, f, max(getattr(rep, f), getattr(r, f)))
        rep.min_decision_gap = min(rep.min_decision_gap, r.min_decision_gap)
        rep.notes += r.notes
        rep.near_tie_log += r.near_tie_log
    return rep


def compare_state(rep: Report, w, cache, st: oracle.State, check_units, steps_done: int):
    """Slot map and K/V rows must be identical; scores within the accumulation tolerance."""
    snap = snapshot(w, cache, check_units)
    compare_snapshot(rep, snap, st, steps_done, 0 if rep.topk else steps_done)


def snapshot(w, cache, units) -> dict:
    """The GPU cache state of ``units`` on the host."""
    snap = {"slot_pos": to_host(cache.slot_pos, "i32")[units],
            "k_cache": to_host(cache.k_cache, w.dtype)[units],
            "v_cache": to_host(cache.v_cache, w.dtype)[units],
            "scores": to_host(cache.scores, "f32")[units]}
    if cache.e4m3:
        snap["k_scale"] = cache.k_scale.cpu().numpy()[units]
        snap["v_scale"] = cache.v_scale.cpu().numpy()[units]
    return snap


def compare_snapshot(rep: Report, snap: dict, st: oracle.State, steps_done: int, acc_steps: int):
    """GPU state ``snap`` against the oracle's ``st``: slot map, K/V rows (and E4M3 scales) exact;
    scores within the tolerance of ``acc_steps`` float32 additions since both sides last agreed."""
    sp = snap["slot_pos"]
    if not np.array_equal(sp, st.slot_pos):
        bad = np.argwhere(sp != st.slot_pos)
        rep.notes.append(f"after {steps_done} steps: slot map differs at {bad[:5].tolist()}")
        return
    kc, vc = snap["k_cache"], snap["v_cache"]
    if not (np.array_equal(kc, st.k_cache) and np.array_equal(vc, st.v_cache)):
        bad = np.argwhere((kc != st.k_cache).any(axis=-1) | (vc != st.v_cache).any(axis=-1))
        rep.notes.append(f"after {steps_done} steps: K/V cache rows differ at {bad[:4].tolist()}")
    if st.e4m3:
        if not (np.array_equal(snap["k_scale"], st.k_scale) and np.array_equal(snap["v_scale"], st.v_scale)):
            rep.notes.append(f"after {steps_done} steps: E4M3 row scales differ")
    sc = snap["scores"].astype(np.float64)
    ref = st.scores.astype(np.float64)
    rel = np.abs(sc - ref) / np.maximum(np.abs(ref), 1e-6)
    rep.max_score_rel_err = max(rep.max_score_rel_err, float(rel.max(initial=0.0)))
    tol = score_rtol(acc_steps) + 1e-5
    if float(rel.max(initial=0.0)) > tol:
        rep.notes.append(f"after {steps_done} steps: score rel err {rel.max():.3e} > {tol:.3e}")
