"""Run the CPU oracle over one unit's prompt + decode steps and keep every step's record.

Test infrastructure: tiny random inputs and a step-by-step record for the oracle pins.
"""

from __future__ import annotations

import dataclasses

import numpy as np

import oracle
import synth


@dataclasses.dataclass
class StepRecord:
    t: int
    out: np.ndarray  # [D] float64
    probs: np.ndarray  # [n + 1] float64 (cached slots 0..n-1, then the new token)
    evicted_slot: int
    evicted_pos: int
    info: object
    slot_pos_before: np.ndarray
    scores_before: np.ndarray
    slot_pos_after: np.ndarray
    scores_after: np.ndarray
    k_after: np.ndarray
    v_after: np.ndarray


@dataclasses.dataclass
class Trajectory:
    colsum: np.ndarray
    prefill_info: object
    prefill_state: oracle.State
    steps: list[StepRecord]


def random_sequence(rng: np.random.Generator, length: int, D: int, dtype: str,
                    hh: int = 0, spread: float = 1.0) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Random Q/K/V rows [length, D] in storage dtype; ``hh`` keys get a common boost."""
    q = rng.standard_normal((length, D)) * spread
    k = rng.standard_normal((length, D)) * spread
    v = rng.standard_normal((length, D))
    if hh:
        u = rng.standard_normal(D)
        u /= np.linalg.norm(u)
        for p in rng.choice(length, size=min(hh, length), replace=False):
            k[p] += 3.0 * u
        q += 1.0 * u
    conv = (lambda a: a.astype(np.float32)) if dtype == "f32" else \
        (lambda a: synth.to_bf16_bits(a.astype(np.float32)))
    return conv(q), conv(k), conv(v)


def run(lib_path: str, q_seq, k_seq, v_seq, P: int, S: int, budget: int, k_heavy: int,
        k_local: int, prefer=None, policy=None, e4m3: bool = False) -> Trajectory:
    """One unit: prefill on positions 0..P-1, then decode positions P..P+S-1 (``e4m3``: with the
    quantised cache; the records then hold the codes, and the scales are in ``k_scale_after``)."""
    D = q_seq.shape[1]
    orc = oracle.Oracle(budget, k_heavy, k_local, lib_path=lib_path, policy=policy)
    st = orc.new_state(1, D, q_seq.dtype, e4m3=e4m3)
    colsum, pinfo = orc.prefill_select(q_seq[None, :P], k_seq[None, :P], v_seq[None, :P], st,
                                       want_colsum=True)
    pre = st.copy()
    steps = []
    for s in range(S):
        t = P + s
        sp0, sc0 = st.slot_pos[0].copy(), st.scores[0].copy()
        out, es, ep, probs, infos = orc.decode_step(
            t, q_seq[None, t], k_seq[None, t], v_seq[None, t], st, want_probs=True,
            prefer_victim=None if prefer is None else np.array([prefer(s)], dtype=np.int32))
        n = min(t, budget)
        rec = StepRecord(t, out[0], probs[0, : n + 1].copy(), int(es[0]), int(ep[0]),
                         infos[0], sp0, sc0, st.slot_pos[0].copy(), st.scores[0].copy(),
                         st.k_cache[0].copy(), st.v_cache[0].copy())
        if e4m3:
            rec.k_scale_after, rec.v_scale_after = st.k_scale[0].copy(), st.v_scale[0].copy()
        steps.append(rec)
    return Trajectory(colsum[0], pinfo[0], pre, steps)
