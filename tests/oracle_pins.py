"""Pins of the CPU oracle: checks against what the H2O pages and plain mathematics fix.

Each ``pin_*`` takes the path of an oracle shared library and raises ``AssertionError`` when the
oracle disagrees with an independent fact. They are run on the real oracle by
``test_oracle_pins.py`` and on deliberately broken copies of it by ``test_oracle_mutants.py``,
which shows that each plausible mistake is caught by at least one pin.

Sources of the facts (web pages on H2O):
  * ttsmallhot.github.io H2O post, §3.1.1 baselines: the Full KV cache (no eviction) and Local
    (sliding window) policies are the limits H2O must reduce to when the budget covers everything
    or when no heavy-hitter slots exist;
  * same post §2.1.2 / §2.2 and "H2O Heavy-Hitter Oracle 分析" §3.2: the score is the accumulated
    attention, the victim is its argmin outside the recent tokens, the new token is always kept;
  * "H2O Heavy-Hitter Oracle 分析" §3.1: heavy hitters are the top-k of the cumulative attention.
"""

from __future__ import annotations

import math

import numpy as np

import bruteforce as bf
import oracle
import synth
import trajectory as tj


def _close(a, b, rtol, atol, what):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    if not np.allclose(a, b, rtol=rtol, atol=atol):
        err = np.max(np.abs(a - b))
        raise AssertionError(f"{what}: max abs diff {err:.3e}\n{a}\n{b}")


def _cases(seed: int, count: int, max_p=10, max_s=10, max_budget=6, dims=(1, 4, 8)):
    rng = np.random.default_rng(seed)
    for _ in range(count):
        D = int(rng.choice(dims))
        P = int(rng.integers(1, max_p + 1))
        S = int(rng.integers(1, max_s + 1))
        budget = int(rng.integers(1, max_budget + 1))
        kl = int(rng.integers(0, budget + 1))
        dtype = "f32" if rng.random() < 0.5 else "bf16"
        yield rng, D, P, S, budget, budget - kl, kl, dtype


def pin_full_budget_is_dense(lib):
    """Budget >= every token: no eviction ever, and each output equals dense causal attention."""
    rng = np.random.default_rng(11)
    for _ in range(12):
        D = int(rng.choice([1, 4, 8]))
        P, S = int(rng.integers(1, 9)), int(rng.integers(1, 9))
        budget = P + S + int(rng.integers(0, 3))
        kl = int(rng.integers(0, budget + 1))
        dtype = "f32" if rng.random() < 0.5 else "bf16"
        q, k, v = tj.random_sequence(rng, P + S, D, dtype, hh=2)
        tr = tj.run(lib, q, k, v, P, S, budget, budget - kl, kl)
        Q, K, V = bf.widen(q), bf.widen(k), bf.widen(v)
        for rec in tr.steps:
            assert rec.evicted_slot == -1 and rec.evicted_pos == -1, "evicted under a full budget"
            _close(rec.out, bf.dense_causal_attention(Q, K, V, rec.t), 1e-12, 1e-13,
                   f"full-budget output at t={rec.t}")
            expect = np.full(budget, -1)
            expect[: rec.t + 1] = np.arange(rec.t + 1)
            assert np.array_equal(rec.slot_pos_after, expect), "slot map under a full budget"


def pin_no_heavy_is_sliding_window(lib):
    """k_heavy = 0: H2O is the Local baseline, a window over positions t-k .. t."""
    rng = np.random.default_rng(12)
    for _ in range(16):
        D = int(rng.choice([1, 4, 8]))
        budget = int(rng.integers(1, 7))
        P, S = int(rng.integers(1, 13)), int(rng.integers(1, 13))
        dtype = "f32" if rng.random() < 0.5 else "bf16"
        q, k, v = tj.random_sequence(rng, P + S, D, dtype, hh=3)
        tr = tj.run(lib, q, k, v, P, S, budget, 0, budget)
        Q, K, V = bf.widen(q), bf.widen(k), bf.widen(v)
        kept = sorted(p for p in tr.prefill_state.slot_pos[0] if p >= 0)
        assert kept == list(range(max(0, P - budget), P)), "prefill window"
        for rec in tr.steps:
            _close(rec.out, bf.window_attention(Q, K, V, rec.t, budget), 1e-12, 1e-13,
                   f"window output at t={rec.t}")
            pos = sorted(p for p in rec.slot_pos_after if p >= 0)
            assert pos == list(range(max(0, rec.t - budget + 1), rec.t + 1)), "window slot set"
            for j, p in enumerate(rec.slot_pos_after):
                if p >= 0:
                    assert np.array_equal(rec.k_after[j], k[p]) and np.array_equal(rec.v_after[j], v[p])


def pin_victim_is_argmin_of_recomputed_scores(lib):
    """Scores recomputed from scratch out of the attended-set history match the table, the prefill
    keeps the top column sums (full sort), and every victim is the argmin of the recomputed scores
    among positions <= t - k_local, equal scores evicting the lowest position."""
    checked = 0
    for rng, D, P, S, budget, kh, kl, dtype in _cases(13, 40, max_p=12, max_s=12):
        q, k, v = tj.random_sequence(rng, P + S, D, dtype, hh=2)
        tr = tj.run(lib, q, k, v, P, S, budget, kh, kl)
        Q, K = bf.widen(q), bf.widen(k)
        c = bf.causal_column_sums(Q[:P], K[:P])
        _close(tr.colsum, c, 1e-12, 1e-12, "prefill column sums")
        kept = bf.heavy_selection(c, budget, kh, kl)
        got = [int(p) for p in tr.prefill_state.slot_pos[0] if p >= 0]
        if P > budget and 0 < kh < P - kl:
            older = sorted(c[: P - kl], reverse=True)
            near = abs(older[kh - 1] - older[kh]) <= 1e-9 * max(abs(older[kh - 1]), 1e-300)
        else:
            near = False
        if not near:
            assert got == kept, f"prefill kept set {got} != {kept}"
        _close(tr.prefill_state.scores[0][: len(got)], c[got], 1e-6, 1e-7, "prefill scores")
        history = []
        for rec in tr.steps:
            attended = [int(p) for p in rec.slot_pos_before if p >= 0] + [rec.t]
            history.append((rec.t, attended))
            resident = [int(p) for p in rec.slot_pos_before if p >= 0]
            rs = bf.recomputed_scores(Q, K, P, history, resident + [rec.t])
            if rec.evicted_pos >= 0:
                cands = [p for p in resident if p <= rec.t - kl]
                order = sorted(cands, key=lambda p: (rs[p], p))
                if len(order) > 1:
                    a, b = rs[order[0]], rs[order[1]]
                    if abs(b - a) <= 1e-6 * max(abs(a), abs(b)):
                        continue  # fp32 table vs float64 recomputation may order a near tie
                assert rec.evicted_pos == order[0], (
                    f"t={rec.t}: evicted {rec.evicted_pos}, recomputed argmin {order[0]}")
                checked += 1
            for j, p in enumerate(rec.slot_pos_after):
                if p >= 0:
                    _close(rec.scores_after[j], rs[int(p)], 2e-6, 1e-7, f"score of position {p}")
    assert checked > 50, f"too few eviction decisions checked ({checked})"


def pin_uniform_attention_closed_form(lib):
    """All-zero queries: every weight is 1/(attended count), prefill column sums are the harmonic
    differences H_P - H_j, the oldest positions are the heavy hitters, outputs are plain means."""
    for P, budget, kh, S in [(9, 4, 2, 6), (5, 4, 2, 5), (12, 6, 3, 8), (7, 3, 0, 4)]:
        kl = budget - kh
        D = 4
        rng = np.random.default_rng(P * 100 + budget)
        q = np.zeros((P + S, D), dtype=np.float32)
        k = rng.standard_normal((P + S, D)).astype(np.float32)
        v = rng.standard_normal((P + S, D)).astype(np.float32)
        tr = tj.run(lib, q, k, v, P, S, budget, kh, kl)
        HP = bf.harmonic(P)
        _close(tr.colsum, [HP - bf.harmonic(j) for j in range(P)], 1e-13, 1e-14, "harmonic colsum")
        kept = [p for p in tr.prefill_state.slot_pos[0] if p >= 0]
        want = list(range(P)) if P <= budget else sorted(set(range(kh)) | set(range(P - kl, P)))
        assert kept == want, f"uniform prefill keeps {kept}, expected {want}"
        for rec in tr.steps:
            n = min(rec.t, budget)
            _close(rec.probs, np.full(n + 1, 1.0 / (n + 1)), 1e-14, 0, "uniform weights")
            rows = [v[p] for p in rec.slot_pos_before if p >= 0] + [v[rec.t]]
            _close(rec.out, np.mean(np.asarray(rows, dtype=np.float64), axis=0), 1e-13, 1e-14,
                   "uniform output")


def pin_mass_and_slot_invariants(lib):
    """Softmax mass 1 per step, prefill column sums add to P, the table gains 1 minus the evicted
    score each step, and the slot map stays a valid budgeted, windowed set of positions."""
    for rng, D, P, S, budget, kh, kl, dtype in _cases(14, 30, max_p=12, max_s=12):
        q, k, v = tj.random_sequence(rng, P + S, D, dtype, hh=2)
        tr = tj.run(lib, q, k, v, P, S, budget, kh, kl)
        assert math.isclose(float(tr.colsum.sum()), P, rel_tol=1e-12), "sum of column sums != P"
        for rec in tr.steps:
            t, n = rec.t, min(rec.t, budget)
            assert math.isclose(float(rec.probs.sum()), 1.0, rel_tol=1e-12), "softmax mass"
            before = float(np.sum(rec.scores_before, dtype=np.float64))
            after = float(np.sum(rec.scores_after, dtype=np.float64))
            lost = 0.0
            if rec.evicted_slot >= 0:
                j = rec.evicted_slot
                lost = float(np.float32(rec.scores_before[j]) + np.float32(rec.probs[j]))
            tol = (n + 3) * 2.0 ** -23 * max(1.0, before + 1.0)
            assert abs(after - (before + 1.0 - lost)) <= tol, (
                f"t={t}: mass {after} vs {before} + 1 - {lost}")
            pos = [int(p) for p in rec.slot_pos_after if p >= 0]
            assert len(pos) == len(set(pos)) == min(t + 1, budget), "slot count / duplicates"
            for p in range(max(0, t - kl + 1), t + 1):
                assert p in pos, f"t={t}: recent position {p} not resident"
            written = rec.evicted_slot if rec.evicted_slot >= 0 else n
            assert rec.slot_pos_after[written] == t, "new token not in the freed slot"
            if rec.evicted_slot >= 0:
                assert rec.evicted_pos == rec.slot_pos_before[rec.evicted_slot]
                assert rec.evicted_pos <= t - kl, "evicted a protected position"
            else:
                assert n < budget and rec.evicted_pos == -1
            changed = [j for j in range(budget) if rec.slot_pos_after[j] != rec.slot_pos_before[j]]
            assert changed == [written], "more than one slot rewritten (compaction?)"
            for j, p in enumerate(rec.slot_pos_after):
                if p >= 0:
                    assert np.array_equal(rec.k_after[j], k[p]) and np.array_equal(rec.v_after[j], v[p])
            assert np.float32(rec.scores_after[written]) == np.float32(rec.probs[n]), \
                "new token's score is not its own weight"


def pin_small_local_is_unprotected_argmin(lib):
    """k_local in {0, 1}: no cached slot is protected, so the victim is the plain argmin of the
    updated table over all slots (the rule as written in "H2O Heavy-Hitter Oracle 分析" §3.2)."""
    seen = 0
    for rng, D, P, S, budget, _, _, dtype in _cases(15, 30, max_p=12, max_s=12):
        for kl in (0, 1):
            if kl > budget:
                continue
            q, k, v = tj.random_sequence(rng, P + S, D, dtype, hh=2)
            tr = tj.run(lib, q, k, v, P, S, budget, budget - kl, kl)
            for rec in tr.steps:
                if rec.evicted_slot < 0:
                    continue
                upd = rec.scores_before + rec.probs[:-1].astype(np.float32)
                order = sorted(range(budget), key=lambda j: (upd[j], rec.slot_pos_before[j]))
                assert rec.evicted_slot == order[0], f"t={rec.t}: victim {rec.evicted_slot} != {order[0]}"
                seen += 1
    assert seen > 30


def _hand_state(lib, slot_pos, scores, t, kl, D=2):
    """One step from a hand-built full cache with all-zero keys and queries (uniform weights)."""
    budget = len(slot_pos)
    orc = oracle.Oracle(budget, budget - kl, kl, lib_path=lib)
    st = orc.new_state(1, D, np.float32)
    st.slot_pos[0] = slot_pos
    st.scores[0] = scores
    z = np.zeros((1, D), dtype=np.float32)
    out, es, ep, probs, infos = orc.decode_step(t, z, z, z + 1, st, want_probs=True)
    return int(es[0]), int(ep[0]), st


def pin_hand_built_ties_and_protection(lib):
    """Exact ties evict the lowest position; recent positions are never candidates."""
    # all scores equal -> uniform weights keep them equal -> lowest position among candidates
    assert _hand_state(lib, [7, 3, 9, 5], [0.0] * 4, 10, kl=1)[:2] == (1, 3)
    assert _hand_state(lib, [7, 3, 9, 5], [0.0] * 4, 10, kl=0)[:2] == (1, 3)
    # position 9 (score 0, the lowest) is protected with k_local = 2 (t = 10 keeps 9 and 10)
    assert _hand_state(lib, [7, 3, 9, 5], [0.1, 0.5, 0.0, 0.2], 10, kl=2)[:2] == (0, 7)
    # with k_local = 1 nothing is protected: position 9 goes
    assert _hand_state(lib, [7, 3, 9, 5], [0.1, 0.5, 0.0, 0.2], 10, kl=1)[:2] == (2, 9)
    # k_local = budget: only t - budget is a candidate (sliding window), whatever the scores
    assert _hand_state(lib, [7, 6, 9, 8], [0.0, 9.0, 0.0, 0.0], 10, kl=4)[:2] == (1, 6)
    # equal lowest scores at positions 5 and 2: position 2 goes
    assert _hand_state(lib, [5, 8, 2, 9], [0.25, 0.5, 0.25, 0.75], 10, kl=1)[:2] == (2, 2)
    _, _, st = _hand_state(lib, [5, 8, 2, 9], [0.25, 0.5, 0.25, 0.75], 10, kl=1)
    assert list(st.slot_pos[0]) == [5, 8, 10, 9]
    assert np.float32(st.scores[0][2]) == np.float32(0.2)  # the new token's own weight, 1/5
    assert np.allclose(st.scores[0][[0, 1, 3]], np.float32([0.25, 0.5, 0.75]) + np.float32(0.2))


def pin_prefill_equal_sums_keep_later(lib):
    """Equal column sums: the later position is kept (the decode order read backwards). Built with
    one key that takes all attention so every other column sum is exactly zero."""
    for P, budget, kh in [(8, 4, 3), (10, 5, 2), (6, 6, 0), (9, 3, 3)]:
        kl = budget - kh
        q = np.ones((P, 1), dtype=np.float32)
        k = np.full((P, 1), -1000.0, dtype=np.float32)
        k[0] = 30.0
        v = np.arange(P, dtype=np.float32)[:, None]
        orc = oracle.Oracle(budget, kh, kl, lib_path=lib)
        st = orc.new_state(1, 1, np.float32)
        c, _ = orc.prefill_select(q[None], k[None], v[None], st, want_colsum=True)
        assert c[0, 0] == P and not c[0, 1:].any()
        tail = list(range(P - kl, P))
        heavy = ([0] + list(range(P - kl - 1, P - kl - kh, -1)))[:kh] if kh else []
        want = sorted(set(heavy) | set(tail)) if P > budget else list(range(P))
        got = [int(p) for p in st.slot_pos[0] if p >= 0]
        assert got == want, f"P={P} k={budget} kh={kh}: kept {got}, expected {want}"


def pin_prompt_fits_budget(lib):
    """A prompt no longer than the budget is kept whole, in order; unused slots are empty."""
    rng = np.random.default_rng(16)
    for P, budget in [(1, 1), (3, 5), (5, 5), (4, 9)]:
        D = 4
        q, k, v = tj.random_sequence(rng, P + 1, D, "bf16")
        orc = oracle.Oracle(budget, budget // 2, budget - budget // 2, lib_path=lib)
        st = orc.new_state(1, D, np.uint16)
        st.k_cache[:] = 7
        orc.prefill_select(q[None, :P], k[None, :P], v[None, :P], st)
        assert list(st.slot_pos[0]) == list(range(P)) + [-1] * (budget - P)
        assert np.array_equal(st.k_cache[0, :P], k[:P]) and np.array_equal(st.v_cache[0, :P], v[:P])
        assert not st.k_cache[0, P:].any() and not st.scores[0, P:].any()


def pin_bf16_is_exact_widening(lib):
    """bf16 inputs give exactly the results of the same values passed as float32."""
    rng = np.random.default_rng(17)
    D, P, S, budget, kh, kl = 8, 10, 10, 5, 3, 2
    q, k, v = tj.random_sequence(rng, P + S, D, "bf16", hh=2)
    a = tj.run(lib, q, k, v, P, S, budget, kh, kl)
    w = lambda x: bf.widen(x).astype(np.float32)
    b = tj.run(lib, w(q), w(k), w(v), P, S, budget, kh, kl)
    assert np.array_equal(a.colsum, b.colsum)
    for ra, rb in zip(a.steps, b.steps):
        assert np.array_equal(ra.out, rb.out) and np.array_equal(ra.scores_after, rb.scores_after)
        assert np.array_equal(ra.slot_pos_after, rb.slot_pos_after)


def pin_near_tie_adoption(lib):
    """A preferred victim is adopted only when its score is within the tie tolerance."""
    base = dict(slot_pos=[5, 8, 2, 9], t=10, kl=1)
    budget = 4
    orc = oracle.Oracle(budget, 3, 1, lib_path=lib)
    for scores, prefer, tie, kind, victim in [
        ([0.25, 0.5, 0.2500001, 0.75], 2, 1e-6, oracle.NEAR_TIE, 2),
        ([0.25, 0.5, 0.2500001, 0.75], 2, 1e-8, oracle.REJECTED, 0),
        ([0.25, 0.5, 0.25, 0.75], 0, 1e-6, oracle.REJECTED, 2),  # exact tie: by position
        ([0.25, 0.5, 0.3, 0.75], 1, 1e-6, oracle.REJECTED, 0),
    ]:
        st = orc.new_state(1, 2, np.float32)
        st.slot_pos[0] = base["slot_pos"]
        st.scores[0] = scores
        z = np.zeros((1, 2), dtype=np.float32)
        _, es, _, _, infos = orc.decode_step(base["t"], z, z, z, st,
                                             prefer_victim=np.array([prefer]), tie_rel=tie,
                                             err_rel=tie)
        assert infos[0].kind == kind and es[0] == victim, (scores, prefer, infos[0].kind, es[0])


def _policy(kind, n_sink=0, stride=1):
    return oracle.Policy(kind, n_sink, stride)


def _resident(rec):
    return sorted(int(p) for p in rec.slot_pos_after if p >= 0)


def pin_local_policy_is_the_window(lib):
    """Local (the post's sliding-window baseline): whatever the k_heavy/k_local split, the cache is
    the last k positions and each output is the window attention over t-k .. t."""
    rng = np.random.default_rng(21)
    for _ in range(10):
        D, budget = int(rng.choice([1, 4, 8])), int(rng.integers(1, 7))
        P, S = int(rng.integers(1, 13)), int(rng.integers(1, 13))
        kl = int(rng.integers(0, budget + 1))
        q, k, v = tj.random_sequence(rng, P + S, D, "f32", hh=2)
        tr = tj.run(lib, q, k, v, P, S, budget, budget - kl, kl, policy=_policy(oracle.POLICY_LOCAL))
        Q, K, V = bf.widen(q), bf.widen(k), bf.widen(v)
        assert sorted(p for p in tr.prefill_state.slot_pos[0] if p >= 0) == list(range(max(0, P - budget), P))
        for rec in tr.steps:
            _close(rec.out, bf.window_attention(Q, K, V, rec.t, budget), 1e-12, 1e-13, "local output")
            assert _resident(rec) == list(range(max(0, rec.t - budget + 1), rec.t + 1)), "local set"


def pin_sink_window_keeps_sinks_and_recent(lib):
    """Sink + window (StreamingLLM's attention sinks, mentioned alongside H2O on the pages): the first
    n_sink positions stay, the rest is the most recent window; outputs attend exactly that set."""
    rng = np.random.default_rng(22)
    for _ in range(12):
        D, budget = int(rng.choice([1, 4, 8])), int(rng.integers(2, 8))
        n_sink = int(rng.integers(0, budget))
        P, S = int(rng.integers(1, 13)), int(rng.integers(1, 13))
        q, k, v = tj.random_sequence(rng, P + S, D, "f32", hh=2)
        tr = tj.run(lib, q, k, v, P, S, budget, budget // 2, budget - budget // 2,
                    policy=_policy(oracle.POLICY_SINK_WINDOW, n_sink=n_sink))
        Q, K, V = bf.widen(q), bf.widen(k), bf.widen(v)

        def want(last):  # resident positions once `last` is the newest token
            n = last + 1
            if n <= budget:
                return list(range(n))
            return sorted(set(range(n_sink)) | set(range(n - (budget - n_sink), n)))
        assert sorted(p for p in tr.prefill_state.slot_pos[0] if p >= 0) == want(P - 1)
        for rec in tr.steps:
            attended = want(rec.t - 1) + [rec.t]
            _close(rec.out, bf.attention(Q[rec.t], K[attended], V[attended])[0], 1e-12, 1e-13,
                   "sink+window output")
            assert _resident(rec) == want(rec.t), f"t={rec.t}: {_resident(rec)} != {want(rec.t)}"


def pin_strided_keeps_its_grid(lib):
    """Strided: beside the k_local recent positions (at least the new token), the older positions kept
    are the newest ones on the stride grid, then the newest off it -- the closed form of repeatedly
    evicting off-grid positions oldest first."""
    rng = np.random.default_rng(23)
    for _ in range(12):
        D, budget = int(rng.choice([1, 4])), int(rng.integers(2, 8))
        kl = int(rng.integers(0, budget + 1))
        kh = budget - kl
        stride = int(rng.integers(1, 5))
        P, S = int(rng.integers(1, 15)), int(rng.integers(1, 15))
        q, k, v = tj.random_sequence(rng, P + S, D, "f32")
        tr = tj.run(lib, q, k, v, P, S, budget, kh, kl, policy=_policy(oracle.POLICY_STRIDED, stride=stride))

        def want(last, recent):
            n = last + 1
            if n <= budget:
                return list(range(n))
            older = sorted(range(n - recent), key=lambda p: (p % stride == 0, p), reverse=True)
            return sorted(older[: budget - recent] + list(range(n - recent, n)))
        assert sorted(p for p in tr.prefill_state.slot_pos[0] if p >= 0) == want(P - 1, kl)
        for rec in tr.steps:
            # a decode step always admits the new token, even with k_local = 0
            w = want(rec.t, max(kl, 1))
            assert _resident(rec) == w, f"stride {stride}, kl {kl}, t={rec.t}: {_resident(rec)} != {w}"


def pin_topk_ranks_by_current_attention(lib):
    """Top-K (the post's baseline that keeps the K highest current scores): each step's scores are
    exactly that step's weights recomputed from raw Q/K, the victim is their argmin outside the
    recent tokens, and the prefill keeps the older positions the last prompt token attends to most."""
    checked = 0
    for rng, D, P, S, budget, kh, kl, dtype in _cases(24, 30, max_p=12, max_s=12):
        q, k, v = tj.random_sequence(rng, P + S, D, dtype, hh=2)
        tr = tj.run(lib, q, k, v, P, S, budget, kh, kl, policy=_policy(oracle.POLICY_TOPK))
        Q, K = bf.widen(q), bf.widen(k)
        last = bf.attention_weights(Q[P - 1], K[:P])
        kept = bf.heavy_selection(last, budget, kh, kl)
        got = [int(p) for p in tr.prefill_state.slot_pos[0] if p >= 0]
        older = sorted(last[: max(0, P - kl)], reverse=True)
        near = P > budget and 0 < kh < P - kl and abs(older[kh - 1] - older[kh]) <= 1e-9
        if not near:
            assert got == kept, f"Top-K prefill kept {got}, expected {kept}"
            _close(tr.prefill_state.scores[0][: len(got)], last[got], 1e-6, 1e-7, "Top-K prefill scores")
        for rec in tr.steps:
            resident = [int(p) for p in rec.slot_pos_before if p >= 0]
            w = bf.attention_weights(Q[rec.t], K[resident + [rec.t]])
            cur = dict(zip(resident, w[:-1]))
            if rec.evicted_pos >= 0:
                cands = sorted((p for p in resident if p <= rec.t - kl), key=lambda p: (cur[p], p))
                if len(cands) > 1 and abs(cur[cands[1]] - cur[cands[0]]) <= 1e-6 * cur[cands[1]]:
                    continue
                assert rec.evicted_pos == cands[0], f"t={rec.t}: Top-K evicted {rec.evicted_pos}, want {cands[0]}"
                checked += 1
            for j, p in enumerate(rec.slot_pos_after):
                if p >= 0:
                    _close(rec.scores_after[j], w[-1] if p == rec.t else cur[int(p)], 1e-6, 1e-8,
                           "Top-K score = current weight")
    assert checked > 30


def _as_storage(a, dtype):
    a = np.asarray(a, dtype=np.float32)
    return a if dtype == "f32" else synth.to_bf16_bits(a)


def pin_prefill_attention_closed_forms(lib):
    """Prompt-pass attention output (the step the column sums are taken from, post §2.1.1):
    all-zero queries give prefix means of the value rows; a key aligned with every query and
    thousands of logit units above the rest takes all the weight from its position on."""
    rng = np.random.default_rng(41)
    for dtype in ("f32", "bf16"):
        for P, D in [(1, 4), (7, 4), (19, 8), (33, 1)]:
            v = _as_storage(rng.standard_normal((P, D)), dtype)
            V = bf.widen(v)
            q = _as_storage(np.zeros((P, D)), dtype)
            k = _as_storage(rng.standard_normal((P, D)), dtype)
            out = oracle.prefill_attention(q[None], k[None], v[None], lib)[0]
            want = np.cumsum(V, axis=0) / np.arange(1, P + 1)[:, None]
            _close(out, want, 1e-13, 1e-14, f"zero-query prefix means P={P}")
            # one dominant key at position js: logits 64 * 64 / sqrt(D) against 0 for the others
            js = int(rng.integers(0, P))
            e0 = np.zeros(D)
            e0[0] = 64.0
            q = _as_storage(np.tile(e0, (P, 1)), dtype)
            kk = np.zeros((P, D))
            kk[js] = e0
            out = oracle.prefill_attention(q[None], _as_storage(kk, dtype)[None], v[None], lib)[0]
            want[js:] = V[js]
            _close(out, want, 1e-13, 1e-14, f"dominant key at {js}, P={P}")


def pin_prefill_attention_weights_are_the_column_sum_weights(lib):
    """With one-hot value rows (v_j = e_j, D = P) the output rows are the attention weight rows:
    each sums to 1 and, added over the rows, they give the prefill column sums computed by the
    selection path. The last row equals the decode step's output at t = P - 1 under a full budget."""
    rng = np.random.default_rng(42)
    for P in (1, 5, 12):
        for dtype in ("f32", "bf16"):
            D = P
            q, k, _ = tj.random_sequence(rng, P, D, dtype, hh=2)
            v = _as_storage(np.eye(P), dtype)
            out = oracle.prefill_attention(q[None], k[None], v[None], lib)[0]
            _close(out.sum(axis=1), np.ones(P), 1e-13, 1e-14, "one-hot output rows sum to 1")
            assert np.all(np.triu(out, 1) == 0.0), "weight on a later position"
            orc = oracle.Oracle(P + 1, 1, P, lib_path=lib)
            st = orc.new_state(1, D, q.dtype)
            c, _ = orc.prefill_select(q[None], k[None], v[None], st, want_colsum=True)
            _close(out.sum(axis=0), c[0], 1e-12, 1e-13, "column sums of the output rows")
    for dtype in ("f32", "bf16"):
        P, D = 9, 8
        q, k, v = tj.random_sequence(rng, P, D, dtype, hh=2)
        out = oracle.prefill_attention(q[None], k[None], v[None], lib)[0]
        orc = oracle.Oracle(P, 0, P, lib_path=lib)
        st = orc.new_state(1, D, q.dtype)
        orc.prefill_select(q[None, : P - 1], k[None, : P - 1], v[None, : P - 1], st)
        o, _, _, _, _ = orc.decode_step(P - 1, q[None, P - 1], k[None, P - 1], v[None, P - 1], st)
        _close(out[P - 1], o[0], 1e-12, 1e-13, "last prompt row vs decode step")


# ---- the E4M3 (FP8) cache --------------------------------------------------------------------

def _e4m3_table(lib):
    """Values of all 256 E4M3 codes as the oracle decodes them."""
    return np.array([oracle.e4m3_value(c, lib) for c in range(256)])


def _nearest_code(x: float, table) -> int:
    """Brute force: the finite code nearest to x, ties to the even mantissa, saturating at 448."""
    x = float(np.float32(x))
    x = max(-448.0, min(448.0, x))
    best = None
    for c in range(256):
        v = table[c]
        if np.isnan(v) or (v == 0.0 and c == 0x80):  # NaNs; -0 (x == 0 maps to the signed zero)
            continue
        d = abs(v - x)
        if best is None or d < best[0] or (d == best[0] and (c & 1) == 0 and (best[1] & 1) == 1):
            best = (d, c)
    c = best[1]
    if c == 0 and np.signbit(x):
        c = 0x80
    return c


def pin_e4m3_format(lib):
    """The E4M3 format (OCP 8-bit floating point): its stated limit values, NaN, and every
    conversion = the nearest finite code found by brute force, ties to the even mantissa,
    saturating at +-448."""
    t = _e4m3_table(lib)
    fixed = {0x7E: 448.0, 0x08: 2.0 ** -6, 0x07: 0.875 * 2.0 ** -6, 0x01: 2.0 ** -9, 0x38: 1.0,
             0x3F: 1.875, 0x40: 2.0, 0xB8: -1.0, 0xFE: -448.0, 0x00: 0.0}
    for c, v in fixed.items():
        assert t[c] == v, (hex(c), t[c], v)
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    finite = [c for c in range(256) if not np.isnan(t[c])]
    for c in finite:  # every finite code round-trips
        assert oracle.e4m3_code(float(t[c]), lib) == c or t[c] == 0.0, hex(c)
    pos = [t[c] for c in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:])), "codes 0..0x7E are increasing"
    # ties: 1.0625 lies between 1.0 (mantissa 0) and 1.125 (1): to 1.0; 1.1875 -> 1.25 (mantissa 2)
    assert oracle.e4m3_code(1.0625, lib) == 0x38 and oracle.e4m3_code(1.1875, lib) == 0x3A
    assert oracle.e4m3_code(464.0, lib) == 0x7E and oracle.e4m3_code(-1e9, lib) == 0xFE
    rng = np.random.default_rng(44)
    xs = np.concatenate([rng.standard_normal(300) * 10.0 ** rng.uniform(-4, 3, 300),
                         [t[c] + (t[c + 1] - t[c]) / 2 for c in range(0x7E)]])  # every midpoint
    for x in xs:
        want = _nearest_code(x, t)
        got = oracle.e4m3_code(float(x), lib)
        assert got == want or (t[got] == t[want]), (x, hex(got), hex(want))


def _quantise_row_bruteforce(x_bf16: np.ndarray, table):
    x = bf.widen(x_bf16).astype(np.float32)
    amax = np.float32(np.max(np.abs(x)))
    scale = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
    codes = np.array([_nearest_code(float(np.float32(xi / scale)), table) for xi in x], dtype=np.uint8)
    return codes, scale


def pin_e4m3_cache_rows(lib):
    """Every row the quantised cache holds after prefill and after each decode step is the row's
    bf16 values quantised by brute force (scale = amax / 448 in float32, nearest codes), and the
    outputs under a full budget are dense attention over the dequantised prompt rows plus the new
    token's bf16 values."""
    t = _e4m3_table(lib)
    rng = np.random.default_rng(45)
    for _ in range(6):
        D = int(rng.choice([4, 8, 16]))
        P, S = int(rng.integers(1, 7)), int(rng.integers(1, 6))
        budget = P + S + 1
        q, k, v = tj.random_sequence(rng, P + S, D, "bf16", hh=2)
        k[0] = 0  # an all-zero row: scale 1, zero codes
        tr = tj.run(lib, q, k, v, P, S, budget, budget // 2, budget - budget // 2, e4m3=True)
        Q, K, V = bf.widen(q), bf.widen(k), bf.widen(v)
        deq_k, deq_v = K.copy(), V.copy()
        for rec in tr.steps:
            for j, pos in enumerate(rec.slot_pos_after):
                if pos < 0:
                    continue
                ck, sk = _quantise_row_bruteforce(k[pos], t)
                cv, sv = _quantise_row_bruteforce(v[pos], t)
                assert np.array_equal(rec.k_after[j], ck) and rec.k_scale_after[j] == sk, (pos, j)
                assert np.array_equal(rec.v_after[j], cv) and rec.v_scale_after[j] == sv, (pos, j)
                deq_k[pos] = sk * t[ck]
                deq_v[pos] = sv * t[cv]
            # dense attention: cached (dequantised) rows 0..t-1, the new token's own bf16 row
            keys = np.concatenate([deq_k[: rec.t], K[rec.t: rec.t + 1]])
            vals = np.concatenate([deq_v[: rec.t], V[rec.t: rec.t + 1]])
            _close(rec.out, bf.attention(Q[rec.t], keys, vals)[0], 1e-12, 1e-13,
                   f"E4M3 full-budget output at t={rec.t}")


def pin_e4m3_exact_rows_reduce_to_bf16(lib):
    """K/V rows whose values are E4M3 values with magnitude maximum 448 are stored exactly (scale 1),
    so the quantised cache must then make every decision and output of the bf16 cache."""
    t = _e4m3_table(lib)
    finite = np.array([t[c] for c in range(256) if not np.isnan(t[c]) and abs(t[c]) <= 448.0])
    rng = np.random.default_rng(46)
    for _ in range(8):
        D = int(rng.choice([4, 8]))
        P, S = int(rng.integers(3, 12)), int(rng.integers(4, 12))
        budget = int(rng.integers(2, 6))
        kl = int(rng.integers(0, budget + 1))
        q, _, _ = tj.random_sequence(rng, P + S, D, "bf16", hh=2)
        rows = rng.choice(finite, size=(2, P + S, D))
        rows[:, :, 0] = 448.0 * rng.choice([-1.0, 1.0], size=(2, P + S))  # amax 448: scale 1
        k, v = (synth.to_bf16_bits(r.astype(np.float32)) for r in rows)
        assert np.array_equal(bf.widen(k), rows[0]), "E4M3 values are exact in bf16"
        plain = tj.run(lib, q, k, v, P, S, budget, budget - kl, kl)
        quant = tj.run(lib, q, k, v, P, S, budget, budget - kl, kl, e4m3=True)
        assert np.array_equal(plain.prefill_state.slot_pos, quant.prefill_state.slot_pos)
        for a, b in zip(plain.steps, quant.steps):
            assert (a.evicted_slot, a.evicted_pos) == (b.evicted_slot, b.evicted_pos)
            assert np.array_equal(a.scores_after, b.scores_after)
            _close(b.out, a.out, 1e-13, 1e-13, "E4M3 exact rows vs bf16")
            assert np.all(b.k_scale_after[b.slot_pos_after >= 0] == 1.0)


PINS = [pin_full_budget_is_dense, pin_no_heavy_is_sliding_window,
        pin_victim_is_argmin_of_recomputed_scores, pin_uniform_attention_closed_form,
        pin_mass_and_slot_invariants, pin_small_local_is_unprotected_argmin,
        pin_hand_built_ties_and_protection, pin_prefill_equal_sums_keep_later, pin_prompt_fits_budget, pin_bf16_is_exact_widening,
        pin_near_tie_adoption, pin_local_policy_is_the_window, pin_sink_window_keeps_sinks_and_recent,
        pin_strided_keeps_its_grid, pin_topk_ranks_by_current_attention,
        pin_prefill_attention_closed_forms, pin_prefill_attention_weights_are_the_column_sum_weights,
        pin_e4m3_format, pin_e4m3_cache_rows, pin_e4m3_exact_rows_reduce_to_bf16]
