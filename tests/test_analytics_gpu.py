"""The expected round length on the GPU, against the kernel's own measured
accepted lengths (the ragged configuration's check).

For fixed rows, with each draft token x_i drawn afresh from the drafter's q_i,
the round emits n + 1 tokens with E[n + 1] = tau = 1 + sum_k prod_{i<=k} alpha_i
("Speculative decoding: the art of guessing well", the section on how many
tokens a round yields); with one alpha at every position this is the closed
form (1 - alpha^(gamma+1)) / (1 - alpha) ("Fast Inference from Transformers via
Speculative Decoding" review page, Analysis).  tau is computed from the alpha
the kernel returns, and compared with the mean of accepted_len + 1 over many
seeds, each with fresh draft tokens from the drafter, within 4 standard errors.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_20_gb300")
from speculative_decoding_verification_20_gb300 import analytics, workloads  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_20_gb300 import _build

    _build.build()


def _rounds(wl, seeds):
    """accepted_len + 1 of every sequence for each seed (fresh draft tokens each time) and
    the kernel's alpha (the same for every seed: it depends on the rows only)."""
    lengths, alpha = [], None
    for s in seeds:
        g = torch.Generator(device=wl.target.device).manual_seed(10_000 + s)
        x = workloads._propose(wl.draft, wl.temperature, wl.top_k, wl.top_p, g)
        r = sv.spec_verify(wl.target, wl.draft, x, wl.temperature, wl.num_draft, wl.top_k, wl.top_p, seed=s)
        lengths.append((r["accepted_len"] + 1).cpu().numpy())
        a = r["alpha"].cpu().numpy()
        assert (r["row_status"].cpu().numpy() == 0).all()
        if alpha is None:
            alpha = a
        else:
            np.testing.assert_array_equal(a, alpha)  # alpha does not depend on the draws
    return np.array(lengths, dtype=np.float64), alpha


def _check(lengths, tau, gam, S):
    mean = lengths.mean(axis=0)
    se = lengths.std(axis=0, ddof=1) / np.sqrt(S)
    bound = np.maximum(4 * se, 4 * (gam + 1) / 2 / np.sqrt(S) * 0.05)  # deterministic rows: se = 0
    assert (np.abs(mean - tau) <= bound + 1e-9).all(), (mean, tau, se)
    # the batch total, with its own standard error
    tot_se = lengths.sum(axis=1).std(ddof=1) / np.sqrt(S)
    assert abs(mean.sum() - tau.sum()) <= 4 * tot_se + 1e-9


def test_tau_of_the_kernels_alpha_matches_its_mean_round_length_ragged():
    wl = workloads.make("ragged", seed=12, device="cuda")
    S = 300
    lengths, alpha = _rounds(wl, range(S))
    gam = wl.gammas()
    tau = analytics.acceptance_length(alpha, gam)
    assert (tau >= 1).all() and (tau <= gam + 1).all()
    _check(lengths, tau, gam, S)


def test_closed_form_with_one_alpha_per_sequence():
    """Every position of a sequence holds the same (target, draft) rows, so alpha_i = alpha
    and E[#tokens] = (1 - alpha^(gamma+1)) / (1 - alpha)."""
    base = workloads.make("ragged", seed=13, device="cuda", V=40000)
    t = base.target[:, :1].expand(-1, base.G + 1, -1).contiguous()
    d = t[:, :1, :base.V] + (base.draft[:, :1] - base.target[:, :1])
    d = d.expand(-1, base.G, -1).contiguous()
    wl = workloads.Workload("ragged-iid", base.B, base.G, base.V, base.dtype, t, d, base.draft_tokens,
                            base.num_draft, base.temperature, base.top_k, base.top_p, base.seed)
    S = 300
    lengths, alpha = _rounds(wl, range(S))
    gam = wl.gammas()
    a = alpha[:, 0].astype(np.float64)
    for b in range(wl.B):  # one alpha at every position of the sequence
        np.testing.assert_allclose(alpha[b, :gam[b]], a[b], rtol=0, atol=1e-6)
    closed = analytics.expected_tokens(a, gam)
    _check(lengths, closed, gam, S)
    assert 0.2 < a[wl.temperature.cpu().numpy() > 0].mean() < 1.0
