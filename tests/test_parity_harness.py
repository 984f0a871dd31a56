"""The parity harness's own rules, on hand-made results (no GPU, no kernel)."""
from types import SimpleNamespace

import numpy as np

from tests.parity import MARGIN, PROB_TOL, ParityReport, compare_probs


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
    assert rep.ok() and rep.prob_excused == 0 and 0 < rep.prob_err <= PROB_TOL


def test_probability_error_on_a_well_separated_row_fails():
    gpu, ora, gam = _case(3 * PROB_TOL, 10 * MARGIN)
    rep = compare_probs(gpu, ora, gam, ParityReport())
    assert not rep.ok() and rep.prob_excused == 0


def test_probability_error_at_a_boundary_within_rounding_is_excused_and_counted():
    gpu, ora, gam = _case(3 * PROB_TOL, 0.1 * MARGIN)
    rep = compare_probs(gpu, ora, gam, ParityReport())
    assert rep.ok() and rep.prob_excused == 1 and rep.prob_err == 0.0
