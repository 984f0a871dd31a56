"""Shared-noise (Gumbel-coupled) verification on the GPU against the fp64 oracle
("Speculative decoding: the art of guessing well", section 共享噪声的采样).

Through the C ABI (spec_verify_gumbel): the target's token at every position
(the argmax of log p + g over the kept set, ties to the lower id) must equal
the oracle's, except at positions whose oracle gap between the best and second
best score is below 1e-4 (counted; the kernel's fp32 score error is about
1e-5 at most); the round must be the longest prefix of draft tokens equal to
those tokens, then the target's token.  Every path: the streaming top-k path
(top-k and greedy rows), the whole-row path (no filter, and top-p), and the
dense cluster path (forced).  The drafter shares the noise (oracle.gumbel_draft),
so rounds are long.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import ParityReport, assert_ok, compare_gumbel, to_np

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_20_gb300")
from speculative_decoding_verification_20_gb300 import workloads  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_20_gb300 import _build

    _build.build()
    oracle.build()


def run_gumbel(wl, seed, path="auto", tokens=None, rep=None):
    ni = wl.numpy_inputs()
    if tokens is None:  # the coupled drafter: its own noisy argmax with the same noise
        tokens = oracle.gumbel_draft(ni["draft"], ni["temperature"], ni["num_draft"], ni["top_k"], ni["top_p"],
                                     seed=seed)
    dev = torch.device("cuda")
    g = sv.spec_verify_gumbel(wl.target.to(dev), torch.as_tensor(tokens, device=dev), wl.temperature.to(dev),
                              None if wl.num_draft is None else wl.num_draft.to(dev),
                              None if wl.top_k is None else wl.top_k.to(dev),
                              None if wl.top_p is None else wl.top_p.to(dev), seed=seed, positions=True, path=path)
    torch.cuda.synchronize()
    ora = oracle.gumbel_verify(ni["target"], tokens, ni["temperature"], ni["num_draft"], ni["top_k"], ni["top_p"],
                               seed=seed)
    rep = compare_gumbel(g, ora, tokens, wl.gammas(), rep)
    return rep, g, ora, tokens


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("v32k", dict(B=32)), ("v128k", dict(B=8)),
                                     ("ragged", dict(B=12, V=30000)), ("b1024", dict(B=96))])
@pytest.mark.parametrize("path", ["auto", "dense"])
def test_gumbel_parity_each_workload(name, kw, path):
    wl = workloads.make(name, seed=3, **kw)
    rep = ParityReport()
    for seed in (11, 12):
        run_gumbel(wl, seed, path=path, rep=rep)
    assert_ok(rep)


def test_gumbel_full_size_v128k_leading_rounds():
    """The full 256-sequence batch in one call; the first 12 sequences (whose noise
    indices b = 0..11 the oracle reproduces on its own 12-sequence batch) compared."""
    wl = workloads.make("v128k", seed=4, device="cuda")
    n = 12
    ni = wl.subset(list(range(n))).numpy_inputs()
    x = np.zeros((wl.B, wl.G), np.int32)
    x[:n] = oracle.gumbel_draft(ni["draft"], ni["temperature"], None, ni["top_k"], ni["top_p"], seed=21)
    g = sv.spec_verify_gumbel(wl.target, torch.as_tensor(x, device="cuda"), wl.temperature, None, wl.top_k,
                              wl.top_p, seed=21, positions=True)
    torch.cuda.synchronize()
    ora = oracle.gumbel_verify(ni["target"], x[:n], ni["temperature"], None, ni["top_k"], ni["top_p"], seed=21)
    sel = {k: v[:n] for k, v in g.items()}
    rep = compare_gumbel(sel, ora, x[:n], np.full(n, wl.G))
    assert_ok(rep)
    assert (to_np(sel["accepted_len"]) > 0).mean() > 0.5  # the coupled drafter is often right
    assert (to_np(g["row_status"]) == 0).all()


def test_drafter_invariance_on_gpu():
    """The emitted tokens are the target's own t_1..t_{n+1} whatever the drafter proposes."""
    wl = workloads.make("v32k", seed=5, B=16)
    _, g1, _, x1 = run_gumbel(wl, 31)
    rng = np.random.default_rng(0)
    x2 = rng.integers(0, wl.V, size=x1.shape).astype(np.int32)
    x2[:, :2] = x1[:, :2]
    _, g2, _, _ = run_gumbel(wl, 31, tokens=x2)
    t1, t2 = to_np(g1["target_tokens"]), to_np(g2["target_tokens"])
    np.testing.assert_array_equal(t1, t2)  # the target's tokens do not depend on the drafter
    for g in (g1, g2):
        acc, out, tt = to_np(g["accepted_len"]), to_np(g["out_tokens"]), to_np(g["target_tokens"])
        for b in range(wl.B):
            n = acc[b]
            np.testing.assert_array_equal(out[b, :n + 1], tt[b, :n + 1])


def test_greedy_is_the_argmax_prefix():
    wl = workloads.make("v32k", seed=6, B=16, greedy=True)
    rep, g, _, x = run_gumbel(wl, 41)
    assert_ok(rep)
    am = wl.target.float().argmax(dim=2).numpy()
    np.testing.assert_array_equal(to_np(g["target_tokens"]), am)


def test_invalid_rows_and_nonfinite_logits():
    from tests.test_parity_gpu import _rand_batch
    B, G, V = 10, 3, 600
    wl = _rand_batch(B, G, V, "f32", seed=9, k=20, p=0.9)
    wl.temperature = torch.tensor([1.0, -1.0, float("nan")] + [1.0] * 7)
    wl.top_k = torch.tensor([20, 20, 20, -1] + [20] * 6, dtype=torch.int32)
    wl.top_p = torch.tensor([0.9] * 4 + [0.0] + [0.9, 0.9, 1.0, 1.0, 0.9], dtype=torch.float32)
    wl.num_draft = torch.tensor([3, 3, 3, 3, 3, 0, 3, 3, 3, 3], dtype=torch.int32)
    wl.target[6, 1, 5] = float("nan")
    wl.target[7, 3, :] = float("-inf")
    wl.top_k[7] = 0
    wl.top_k[8] = 0
    wl.target[8, 0, 3] = float("inf")
    x = np.random.default_rng(1).integers(0, V, (B, G)).astype(np.int32)
    for path in ("auto", "dense"):
        rep, g, ora, _ = run_gumbel(wl, 5, path=path, tokens=x)
        assert_ok(rep)
        assert list(to_np(g["row_status"])) == list(ora.status)
        assert (ora.status[1:9] != 0).all()


@pytest.mark.parametrize("k,p_top", [(None, None), (3, None), (None, 0.9)])
def test_target_token_follows_p_chisquare(k, p_top):
    """The Gumbel-max law on the GPU's noise: over 2 * 10^5 sequences with the same
    rows, the target's first token t_1 follows the (filtered) p."""
    stats = pytest.importorskip("scipy.stats")
    rng = np.random.default_rng(77 + (k or 0))
    V, B = 8, 200_000
    lp = np.log(rng.dirichlet(np.ones(V))).astype(np.float32)
    one = oracle.verify(np.stack([lp, lp])[None], lp[None, None], np.zeros((1, 1), np.int32), np.ones(1, np.float32),
                        None, None if k is None else np.array([k], np.int32),
                        None if p_top is None else np.array([p_top], np.float32), seed=0, probs=True)
    p_law = one.p_out[0, 0]
    dev = torch.device("cuda")
    tgt = torch.as_tensor(np.broadcast_to(np.stack([lp, lp])[None], (B, 2, V)).copy(), device=dev)
    g = sv.spec_verify_gumbel(tgt, torch.zeros(B, 1, dtype=torch.int32, device=dev), 1.0, None,
                              None if k is None else k, None if p_top is None else p_top, seed=123)
    torch.cuda.synchronize()
    t1 = to_np(g["target_tokens"])[:, 0]
    counts = np.bincount(t1, minlength=V)
    support = p_law > 0
    assert counts[~support].sum() == 0
    _, pval = stats.chisquare(counts[support], p_law[support] / p_law[support].sum() * B)
    assert pval > 1e-3, (counts / B, p_law, pval)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [3, 37, 1001, 4099, 40000])
def test_one_pass_rows_every_vocab_and_part_boundary(dtype, V):
    """Rows with no filter take the one-pass kernel, which cuts the batch's rows into
    equal parts that start and end inside rows: vocabularies that are not a multiple
    of the 16-byte vector (scalar loads), tiny rows (many rows per part) and wide ones
    (several parts per row), with ragged gamma."""
    from tests.test_parity_gpu import _rand_batch
    B, G = 40, 4
    nd = torch.tensor([1 + (b % G) for b in range(B)], dtype=torch.int32)
    wl = _rand_batch(B, G, V, dtype, seed=V + 1, T=np.linspace(0.5, 1.5, B), nd=nd)
    rep = ParityReport()
    for seed in (3, 4):
        run_gumbel(wl, seed, rep=rep)
    assert_ok(rep)


def test_one_pass_rows_mixed_with_every_other_path():
    """A batch mixing unfiltered rows (one-pass kernel) with greedy and top-k rows
    (streaming), top-p rows (whole-row kernel) and top-k > 256 rows (cluster kernel)."""
    from tests.test_parity_gpu import _rand_batch
    B, G, V = 30, 3, 5000
    wl = _rand_batch(B, G, V, "bf16", seed=21)
    wl.temperature = torch.tensor([1.0, 0.0, 0.8, 1.2, 1.0] * 6)
    wl.top_k = torch.tensor([0, 0, 40, 0, 600] * 6, dtype=torch.int32)
    wl.top_p = torch.tensor([1.0, 1.0, 1.0, 0.9, 1.0] * 6, dtype=torch.float32)
    rep = ParityReport()
    for seed in (8, 9):
        run_gumbel(wl, seed, rep=rep)
    assert_ok(rep)
