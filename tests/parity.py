"""Parity checking between the CUDA path and the oracle (test infrastructure).

Rules (from the verification contract):
  * accepted_len / out_tokens and every per-position decision (acceptance at
    each position, residual/bonus token of each position) must agree exactly,
    except decisions whose oracle margin is below 1e-6 -- |u - p/q| for an
    acceptance, the distance of v/Z to the nearest CDF edge for a draw, or a
    filter (top-k / top-p) boundary margin of a row the decision reads.  Such
    excused mismatches are counted and must stay under 1e-4 of all decisions.
  * alpha within 1e-5 absolute; normalised probabilities within 1e-5 absolute,
    except rows whose oracle filter margin is below 1e-6: there the top-k / top-p
    boundary is within rounding of the mass threshold, so the fp32 kernel and
    the fp64 oracle may keep a different prefix (one more or one fewer tail
    token).  Such a row (prob_excused) must still be ANOTHER correct nucleus:
      - the kernel's kept set is a prefix of the row's (logit desc, id asc) order;
      - it differs from the oracle's only by boundary tokens: the shorter of the
        two sets already reaches P within 1e-6, and the longer one without its
        last token stays below P within 1e-6 (masses of the row after
        temperature and top-k, from the oracle);
      - the kernel's probabilities equal that row renormalised over the kernel's
        own kept set, within 1e-5.
    Excused rows count against a budget of PROB_EXCUSED_FRACTION of the rows.

Every report is recorded and printed in pytest's terminal summary.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

MARGIN = 1e-6
EXCUSED_FRACTION = 1e-4
ALPHA_TOL = 1e-5
PROB_TOL = 1e-5
PROB_EXCUSED_FRACTION = 0.05

# (test id, report text) of every report checked with assert_ok, for the terminal summary
REPORTS: list = []


@dataclass
class ParityReport:
    decisions: int = 0
    low_margin: int = 0
    excused: int = 0
    hard: list = field(default_factory=list)
    alpha_err: float = 0.0
    prob_err: float = 0.0
    prob_rows: int = 0
    prob_excused: int = 0

    def ok(self) -> bool:
        return not self.hard and self.excused <= EXCUSED_FRACTION * max(self.decisions, 1) and \
            self.alpha_err <= ALPHA_TOL and self.prob_err <= PROB_TOL and \
            self.prob_excused <= PROB_EXCUSED_FRACTION * max(self.prob_rows, 1)

    def __str__(self):
        return (f"decisions={self.decisions} low_margin={self.low_margin} excused={self.excused} "
                f"hard={self.hard[:5]} alpha_err={self.alpha_err:.3g} prob_err={self.prob_err:.3g} "
                f"prob_rows={self.prob_rows} prob_excused={self.prob_excused}")


def assert_ok(rep: ParityReport, name: str = ""):
    """Record the report for the terminal summary, then require it to pass."""
    if not name:
        import os
        name = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    REPORTS.append((name, str(rep)))
    assert rep.ok(), str(rep)


def to_np(t):
    return t.detach().cpu().numpy() if hasattr(t, "detach") else np.asarray(t)


def compare(gpu: dict, ora, gammas, G: int, report: ParityReport | None = None) -> ParityReport:
    """gpu: dict of tensors from spec_verify(..., positions=True); ora: OracleResult(all_positions=True)."""
    rep = report or ParityReport()
    acc, out = to_np(gpu["accepted_len"]), to_np(gpu["out_tokens"])
    alpha = to_np(gpu["alpha"])
    status = to_np(gpu["row_status"]).astype(np.uint32)
    pa, pt = to_np(gpu["pos_accept"]), to_np(gpu["pos_token"])
    B = acc.shape[0]
    for b in range(B):
        if status[b] != ora.status[b]:
            rep.hard.append(("status", b, int(status[b]), int(ora.status[b])))
            continue
        if ora.status[b]:
            if acc[b] != 0 or (out[b] != -1).any() or (alpha[b] != 0).any():
                rep.hard.append(("invalid-row-outputs", b))
            continue
        g = int(gammas[b])
        fm = ora.filter_margin[b]
        row_excuse_t = [fm[j] < MARGIN for j in range(G + 1)]
        row_excuse_d = [fm[G + 1 + j] < MARGIN for j in range(G)]
        first_diff_excused = True
        for i in range(g):
            rep.decisions += 1
            m = ora.accept_margin[b, i]
            low = (m < MARGIN) or row_excuse_t[i] or row_excuse_d[i]
            rep.low_margin += int(low)
            if pa[b, i] != ora.pos_accept[b, i]:
                if low:
                    rep.excused += 1
                else:
                    rep.hard.append(("accept", b, i, int(pa[b, i]), int(ora.pos_accept[b, i]), float(m)))
        for j in range(g + 1):
            rep.decisions += 1
            m = ora.resid_margin[b, j]
            low = (m < MARGIN) or row_excuse_t[j] or (j < g and row_excuse_d[j])
            rep.low_margin += int(low)
            if pt[b, j] != ora.pos_token[b, j]:
                if low:
                    rep.excused += 1
                else:
                    rep.hard.append(("token", b, j, int(pt[b, j]), int(ora.pos_token[b, j]), float(m)))
        # the emitted round follows from the per-position decisions
        if acc[b] != ora.accepted_len[b] or (out[b] != ora.out_tokens[b]).any():
            n = min(int(acc[b]), int(ora.accepted_len[b]))
            explained = any(pa[b, i] != ora.pos_accept[b, i] for i in range(n + 1) if i < g) or \
                any(pt[b, j] != ora.pos_token[b, j] for j in range(n + 2) if j <= g)
            if not explained:
                rep.hard.append(("round", b, int(acc[b]), int(ora.accepted_len[b])))
        err = np.abs(alpha[b, :g] - ora.alpha[b, :g]).max() if g else 0.0
        rep.alpha_err = max(rep.alpha_err, float(err))
        if (alpha[b, g:] != 0).any():
            rep.hard.append(("alpha-padding", b))
    return rep


def _logits_f32(a: np.ndarray) -> np.ndarray:
    """float32 logits, or bf16 bit patterns (uint16) widened exactly."""
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32)
    return np.asarray(a, dtype=np.float32)


def excused_row_problem(mine, ref, logits, T: float, k: int, P: float, oracle_mod) -> str:
    """Why the kernel's row `mine` is not another correct nucleus of the row (or "")."""
    lg = _logits_f32(logits).astype(np.float64)
    V = lg.size
    pre = oracle_mod.normalise(_logits_f32(logits), np.float32(T), int(k), 1.0)  # temperature and top-k only
    order = np.lexsort((np.arange(V), -lg))  # logit descending, id ascending
    kg, ko = mine > 0, ref > 0
    ng, no = int(kg.sum()), int(ko.sum())
    for name, mask, n in (("kernel", kg, ng), ("oracle", ko, no)):
        if n == 0 or not mask[order[:n]].all():
            return f"{name} kept set is not a prefix of the (logit desc, id asc) order"
    cum = np.cumsum(pre[order])
    m, M = min(ng, no), max(ng, no)
    if cum[m - 1] < P - MARGIN:
        return f"the shorter kept set's mass {cum[m - 1]:.9f} is short of P = {P:.9f}"
    if M >= 2 and cum[M - 2] > P + MARGIN:
        return f"the longer kept set passes P = {P:.9f} before its last token ({cum[M - 2]:.9f})"
    want = np.where(kg, pre, 0.0)
    want = want / want.sum()
    err = float(np.abs(mine - want).max())
    if err > PROB_TOL:
        return f"not the row renormalised over the kernel's own kept set (error {err:.3g})"
    return ""


def compare_probs(gpu: dict, ora, gammas, rep: ParityReport, inputs: dict | None = None,
                  oracle_mod=None) -> ParityReport:
    """Probability outputs, row by row.  `inputs` (the batch's numpy inputs, as
    given to the oracle) and `oracle_mod` let a boundary-excused row be checked
    for validity; without them an excused row is a failure."""
    p, q = to_np(gpu["p_out"]), to_np(gpu["q_out"])
    G = q.shape[1]
    fm_all = ora.filter_margin
    for b in range(p.shape[0]):
        if ora.status[b]:
            continue
        g = int(gammas[b])
        # (gpu row, oracle row, filter-margin index, logits): target rows 0..g, draft rows 0..g-1
        rows = [(p[b, j], ora.p_out[b, j], j, ("target", j)) for j in range(g + 1)] + \
               [(q[b, j], ora.q_out[b, j], G + 1 + j, ("draft", j)) for j in range(g)]
        for mine, ref, fi, (src, j) in rows:
            rep.prob_rows += 1
            err = float(np.abs(mine - ref).max())
            if err > PROB_TOL and fm_all is not None and fm_all[b, fi] < MARGIN:
                rep.prob_excused += 1  # a boundary within rounding of the threshold
                if inputs is None or oracle_mod is None:
                    rep.hard.append(("prob-excuse-unchecked", b, fi))
                    continue
                T = float(inputs["temperature"][b])
                k = 0 if inputs.get("top_k") is None else int(inputs["top_k"][b])
                P = 1.0 if inputs.get("top_p") is None else float(np.float32(inputs["top_p"][b]))
                why = excused_row_problem(mine, ref, inputs[src][b, j], T, k, P, oracle_mod)
                if why:
                    rep.hard.append(("prob-excuse-invalid", b, fi, why))
                continue
            rep.prob_err = max(rep.prob_err, err)
    return rep


# ---------------------------------------------------------------------------
# shared-noise (Gumbel-coupled) verification
# ---------------------------------------------------------------------------
# The kernel scores a kept token as l / T + g in fp32 (g = -ln(-ln u) from fast
# base-2 logarithms, an absolute error of a few 1e-6 at most at the largest g;
# l / T rounded once), against the oracle's fp64 log p + g: two scores can swap
# only when the oracle's gap between the best and the second best is within
# about 1e-5.  Positions whose oracle gap is below GUMBEL_MARGIN = 1e-4 are
# low-margin: a mismatch there is excused and counted against the same budget.
GUMBEL_MARGIN = 1e-4


def compare_gumbel(gpu: dict, ora, draft_tokens, gammas, rep: ParityReport | None = None) -> ParityReport:
    """gpu: spec_verify_gumbel(..., positions=True) outputs; ora: oracle.gumbel_verify result."""
    rep = rep or ParityReport()
    acc, out = to_np(gpu["accepted_len"]), to_np(gpu["out_tokens"])
    tt, st = to_np(gpu["target_tokens"]), to_np(gpu["row_status"]).astype(np.uint32)
    x = to_np(draft_tokens)
    G = x.shape[1]
    for b in range(acc.shape[0]):
        if st[b] != ora.status[b]:
            rep.hard.append(("status", b, int(st[b]), int(ora.status[b])))
            continue
        if ora.status[b]:
            if acc[b] != 0 or (out[b] != -1).any():
                rep.hard.append(("invalid-row-outputs", b))
            continue
        g = int(gammas[b])
        for k in range(g + 1):
            rep.decisions += 1
            low = ora.margin[b, k] < GUMBEL_MARGIN
            rep.low_margin += int(low)
            if tt[b, k] != ora.target_tokens[b, k]:
                if low:
                    rep.excused += 1
                else:
                    rep.hard.append(("token", b, k, int(tt[b, k]), int(ora.target_tokens[b, k]),
                                     float(ora.margin[b, k])))
        if (tt[b, g + 1:] != -1).any():
            rep.hard.append(("padding", b))
        # the round follows from the kernel's own tokens: the longest matching prefix, then t_{n+1}
        n = 0
        while n < g and x[b, n] == tt[b, n]:
            n += 1
        want = list(x[b, :n]) + [tt[b, n]] + [-1] * (G - n)
        if acc[b] != n or list(out[b]) != want:
            rep.hard.append(("round", b, int(acc[b]), n))
        if (acc[b] != ora.accepted_len[b] or (out[b] != ora.out_tokens[b]).any()) and \
                (tt[b, :g + 1] == ora.target_tokens[b, :g + 1]).all():
            rep.hard.append(("round-vs-oracle", b))
    return rep
