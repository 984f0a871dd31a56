"""The parity harness's own rules, on hand-made results (no GPU, no kernel)."""
from types import SimpleNamespace

import numpy as np

from tests.parity import MARGIN, PROB_EXCUSED_FRACTION, PROB_TOL, ParityReport, compare_probs


def _case(err, margin):
    """One sequence, gamma 1: target rows 0..1 and draft row 0 over V = 4; the
    first target row of the 'GPU' side is off by `err` and its oracle filter
    margin is `margin`."""
    G, V = 1, 4
    ref_p = np.full((1, G + 1, V), 0.25)
    ref_q = np.full((1, G, V), 0.25)
    p = ref_p.copy()
    p[0, 0, 0] += err
    p[0, 0, 1] -= err
    fm = np.full((1, 2 * G + 1), 1.0)
    fm[0, 0] = margin
    ora = SimpleNamespace(status=np.zeros(1, dtype=np.uint32), p_out=ref_p, q_out=ref_q, filter_margin=fm)
    return {"p_out": p, "q_out": ref_q.copy()}, ora, np.array([1])


def test_probabilities_within_tolerance_pass():
    gpu, ora, gam = _case(0.5 * PROB_TOL, 1.0)
    rep = compare_probs(gpu, ora, gam, ParityReport())
    assert rep.ok() and rep.prob_excused == 0 and 0 < rep.prob_err <= PROB_TOL and rep.prob_rows == 3


def test_probability_error_on_a_well_separated_row_fails():
    gpu, ora, gam = _case(3 * PROB_TOL, 10 * MARGIN)
    rep = compare_probs(gpu, ora, gam, ParityReport())
    assert not rep.ok() and rep.prob_excused == 0


def test_excused_row_without_inputs_to_check_it_fails():
    gpu, ora, gam = _case(3 * PROB_TOL, 0.1 * MARGIN)
    rep = compare_probs(gpu, ora, gam, ParityReport())
    assert not rep.ok() and rep.prob_excused == 1


def _nucleus_case(oracle_mod, gpu_keep: int, P: float, gpu_row=None):
    """A top-p row over V = 6 with probabilities (0.4, 0.3, 0.2, 0.1 - d, d/2, d/2) in a
    shuffled id order, and P placed so the oracle keeps 3 tokens with the mass
    of the third within rounding of P; the 'GPU' keeps `gpu_keep` tokens."""
    d = 1e-3
    probs = np.array([0.4, 0.3, 0.2, 0.1 - d, d / 2, d / 2])
    ids = np.array([3, 0, 5, 1, 2, 4])  # token ids of the ranks above
    lg = np.zeros(6, dtype=np.float32)
    lg[ids] = np.log(probs).astype(np.float32)
    pre = oracle_mod.normalise(lg, 1.0)
    order = np.lexsort((np.arange(6), -lg.astype(np.float64)))
    ref = oracle_mod.normalise(lg, 1.0, 0, np.float32(P))
    if gpu_row is None:
        keep = np.zeros(6, dtype=bool)
        keep[order[:gpu_keep]] = True
        gpu_row = np.where(keep, pre, 0.0) / pre[keep].sum()
    # one sequence, gamma 1: row 0 (target) is the case; the others agree exactly
    ref_p = np.stack([ref, ref])[None]
    ref_q = ref[None, None].copy()
    p = ref_p.copy()
    p[0, 0] = gpu_row
    fm = np.full((1, 3), 1.0)
    fm[0, 0] = 0.1 * MARGIN
    ora = SimpleNamespace(status=np.zeros(1, dtype=np.uint32), p_out=ref_p, q_out=ref_q, filter_margin=fm)
    inputs = {"target": np.stack([lg, lg])[None], "draft": lg[None, None], "temperature": np.ones(1, np.float32),
              "top_k": None, "top_p": np.array([P], np.float32)}
    return {"p_out": p, "q_out": ref_q.copy()}, ora, inputs, pre[order]


def test_excused_row_that_is_another_correct_nucleus_passes(oracle_mod):
    # P just below the mass of the top 3 (0.9): the oracle keeps 3, a kernel that saw the
    # running mass fall short by rounding keeps 4
    P = float(np.float32(0.9 - 2e-7))
    gpu, ora, inputs, srt = _nucleus_case(oracle_mod, 4, P)
    assert abs(np.cumsum(srt)[2] - P) < MARGIN
    rep = compare_probs(gpu, ora, np.array([1]), ParityReport(), inputs=inputs, oracle_mod=oracle_mod)
    assert rep.prob_excused == 1 and not rep.hard, str(rep)


def test_excused_row_with_a_wrong_kept_set_fails(oracle_mod):
    P = float(np.float32(0.9 - 2e-7))
    # five tokens kept: the longer set passes P well before its last token
    gpu, ora, inputs, _ = _nucleus_case(oracle_mod, 5, P)
    rep = compare_probs(gpu, ora, np.array([1]), ParityReport(), inputs=inputs, oracle_mod=oracle_mod)
    assert not rep.ok() and rep.hard[0][0] == "prob-excuse-invalid"
    # four tokens kept but not a prefix of the order: the 4th-ranked swapped for the 5th
    gpu, ora, inputs, _ = _nucleus_case(oracle_mod, 4, P)
    row = gpu["p_out"][0, 0]
    a, b = 1, 2  # token ids of ranks 4 and 5
    row[b], row[a] = row[a], 0.0
    rep = compare_probs(gpu, ora, np.array([1]), ParityReport(), inputs=inputs, oracle_mod=oracle_mod)
    assert not rep.ok() and "prefix" in rep.hard[0][3]
    # the right set with probabilities not renormalised over it
    gpu, ora, inputs, _ = _nucleus_case(oracle_mod, 4, P)
    gpu["p_out"][0, 0] *= 1.0 + 1e-3
    rep = compare_probs(gpu, ora, np.array([1]), ParityReport(), inputs=inputs, oracle_mod=oracle_mod)
    assert not rep.ok() and "renormalised" in rep.hard[0][3]


def test_excused_rows_count_against_a_budget():
    rep = ParityReport(prob_rows=100, prob_excused=int(PROB_EXCUSED_FRACTION * 100))
    assert rep.ok()
    rep.prob_excused += 1
    assert not rep.ok()
