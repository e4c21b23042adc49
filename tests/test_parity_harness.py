"""The parity harness's acceptance rule, without a GPU: an eviction must equal the oracle's, except
at a near tie (the two lowest candidate scores within 1e-6 relative), where the oracle takes the
other implementation's choice and the step is logged with its gap. A disagreement at any larger gap
is a mismatch, including gaps below 2e-5, the float32 accumulation bound (no wider class of adopted
decisions). The real oracle decides; a hand-picked "GPU" choice plays the other implementation."""

import numpy as np
import pytest

import oracle
import parity

SLOT_POS = (5, 8, 2, 9)  # t = 10, k_local = 1: every slot is a candidate


def _step(scores, gpu_victim):
    orc = oracle.Oracle(4, 3, 1)
    st = orc.new_state(1, 2, np.float32)
    st.slot_pos[0] = SLOT_POS
    st.scores[0] = scores
    z = np.zeros((1, 2), dtype=np.float32)
    out, es, ep, _, infos = orc.decode_step(10, z, z, z, st, prefer_victim=np.array([gpu_victim], np.int32),
                                            tie_rel=parity.TIE_REL, err_rel=parity.ERR_REL)
    rep = parity.Report("hand-built", 1, 1)
    parity.compare_step(rep, "f32", 10, np.array([0]), out.copy(), np.array([gpu_victim], np.int32),
                        np.array([SLOT_POS[gpu_victim]], np.int32), out, es, ep, infos)
    return rep


def test_no_wider_adoption_class():
    assert parity.ERR_REL == parity.TIE_REL == 1e-6


def test_agreement_is_not_a_tie():
    # zero queries and keys: every weight is 1/5, so the scores become 0.45, 0.7, 0.5, 0.95 and the
    # gap is taken between the two lowest updated scores
    rep = _step([0.25, 0.5, 0.3, 0.75], 0)  # the rule's victim: slot 0
    assert rep.ok() and rep.decisions == 1 and rep.near_ties == 0
    assert rep.min_decision_gap == pytest.approx((0.5 - 0.45) / 0.5, rel=1e-5)


def test_near_tie_below_1e6_is_adopted_and_logged():
    rep = _step([0.25, 0.5, 0.2500001, 0.75], 2)  # updated gap 2e-7; the oracle's rule says slot 0
    assert rep.ok() and rep.near_ties == 1 and rep.mismatches == 0
    (t, unit, gap, adopted), = rep.near_tie_log
    assert t == 10 and unit == 0 and adopted and 0 < gap < 1e-6
    parity.check(rep)


@pytest.mark.parametrize("score2", [0.250001, 0.250004])  # updated gaps 2e-6 and 9e-6: below 2e-5
def test_disagreement_above_1e6_is_a_mismatch(score2):
    rep = _step([0.25, 0.5, score2, 0.75], 2)
    assert rep.mismatches == 1 and rep.near_ties == 0 and rep.error_bound_ties == 0
    assert not rep.ok() and "gap" in rep.notes[0]
    with pytest.raises(AssertionError):
        parity.check(rep)


def test_exact_tie_goes_by_position():
    rep = _step([0.25, 0.5, 0.25, 0.75], 0)  # equal scores: the lower position (slot 2, position 2) goes
    assert rep.mismatches == 1 and not rep.ok()


def test_prefill_kept_sets():
    rep = parity.Report("hand-built", 3, 0)
    infos = (oracle.PrefillInfo * 3)()
    for i, (kind, gap) in enumerate([(oracle.RULE, 3e-3), (oracle.NEAR_TIE, 4e-7), (oracle.REJECTED, 5e-6)]):
        infos[i].kind, infos[i].gap_rel = kind, gap
    parity.compare_prefill(rep, infos[:3], np.array([7, 8, 9]))
    assert rep.prefill_near_ties == 1 and rep.prefill_mismatches == 1 and not rep.ok()
    assert rep.near_tie_log == [("prefill", 8, 4e-7, True)]
    assert "unit 9" in rep.notes[0]


def test_merge_adds_counts_and_keeps_extremes():
    a, b = parity.Report("w", 1, 5), parity.Report("w", 1, 5)
    a.decisions, a.near_ties, a.max_out_err, a.min_decision_gap = 5, 1, 1e-3, 1e-4
    b.decisions, b.mismatches, b.max_out_err, b.min_decision_gap = 7, 1, 2e-3, 5e-5
    b.notes.append("x")
    m = parity.merge([a, b], "w", 2, 10)
    assert (m.decisions, m.near_ties, m.mismatches) == (12, 1, 1)
    assert m.max_out_err == 2e-3 and m.min_decision_gap == 5e-5 and m.notes == ["x"] and not m.ok()
