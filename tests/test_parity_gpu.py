"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, on the GPU.

Inputs come from the shared seeded workload generator; the oracle gets the
same inputs and, for row subsets, the uniforms of the original batch indices.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.parity import ParityReport, assert_ok, compare, compare_probs, to_np

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


def run(wl, seed=None, path="auto", probs=False, rows=None, report=None, lenience=None):
    seed = wl.seed if seed is None else seed
    dev = torch.device("cuda")
    w = wl.to(dev)
    gpu = sv.spec_verify(w.target, w.draft, w.draft_tokens, w.temperature, w.num_draft, w.top_k, w.top_p,
                         seed=seed, positions=True, probs=probs, path=path, lenience=lenience)
    torch.cuda.synchronize()
    rows = np.arange(wl.B) if rows is None else np.asarray(rows)
    sub = wl.subset(rows) if len(rows) != wl.B else wl
    ni = sub.numpy_inputs()
    ua, ur = oracle.philox_uniforms(seed, wl.B, wl.G)
    ora = oracle.verify(ni["target"], ni["draft"], ni["draft_tokens"], ni["temperature"], ni["num_draft"],
                        ni["top_k"], ni["top_p"], u_accept=ua[rows], u_resid=ur[rows], all_positions=True,
                        probs=probs, lenience=None if lenience is None else np.asarray(lenience)[rows])
    g = {k: v[torch.as_tensor(rows, device=v.device)] for k, v in gpu.items()}
    rep = compare(g, ora, sub.gammas(), wl.G, report)
    if probs:
        compare_probs(g, ora, sub.gammas(), rep, inputs=ni, oracle_mod=oracle)
    return rep, g, ora


# ---------------------------------------------------------------------------
# the five workload recipes
# ---------------------------------------------------------------------------

def test_tiny_2000_rounds():
    """B=1, gamma=4, V=1000 fp32, 2000 rounds with seed = base + round."""
    wl = workloads.make("tiny", seed=0)
    rep = ParityReport()
    for r in range(2000):
        w = workloads.make("tiny", seed=r)
        run(w, seed=r, report=rep)
    assert_ok(rep)
    assert rep.decisions >= 2000 * 9


@pytest.mark.parametrize("probs", [False, True])
def test_v32k_full(probs):
    wl = workloads.make("v32k", seed=1)
    rep, _, _ = run(wl, probs=probs)
    assert_ok(rep)


def test_v32k_greedy_is_argmax_prefix():
    wl = workloads.make("v32k", seed=2, greedy=True)
    rep, g, _ = run(wl)
    assert_ok(rep)
    am = wl.target.float().argmax(dim=2).numpy()
    x = wl.draft_tokens.numpy()
    acc, out = to_np(g["accepted_len"]), to_np(g["out_tokens"])
    for b in range(wl.B):
        n = 0
        while n < wl.G and x[b, n] == am[b, n]:
            n += 1
        assert acc[b] == n and out[b, n] == am[b, n]


def test_v128k_full_size_sampled_sequences():
    wl = workloads.make("v128k", seed=3, device="cuda")
    rep, _, _ = run(wl, rows=list(range(0, 256, 17)))
    assert_ok(rep)


def test_v128k_small_batch_all_sequences_both_paths():
    wl = workloads.make("v128k", seed=4, B=6)
    rep, g1, _ = run(wl, probs=True)
    assert_ok(rep)
    rep2, g2, _ = run(wl, path="dense", probs=True)
    assert_ok(rep2)


def test_ragged_full():
    wl = workloads.make("ragged", seed=5)
    rep, g, ora = run(wl)
    assert_ok(rep)


def test_b1024_full_size_sampled_and_back_to_back():
    wl = workloads.make("b1024", seed=6, device="cuda")
    rows = list(range(0, 1024, 97))
    rep, _, _ = run(wl, rows=rows)
    assert_ok(rep)
    # 100 back-to-back calls on one stream: each equals its own standalone call
    outs = []
    for k in range(100):
        r = sv.spec_verify(wl.target, wl.draft, wl.draft_tokens, wl.temperature, seed=1000 + k)
        outs.append(r["out_tokens"].clone())
    torch.cuda.synchronize()
    for k in (0, 37, 99):
        r = sv.spec_verify(wl.target, wl.draft, wl.draft_tokens, wl.temperature, seed=1000 + k)
        torch.cuda.synchronize()
        assert torch.equal(outs[k], r["out_tokens"])


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

def _rand_batch(B, G, V, dtype, seed, T=1.0, k=None, p=None, nd=None, ties=False):
    gen = torch.Generator().manual_seed(seed)
    if ties:
        t = torch.randint(-4, 4, (B, G + 1, V), generator=gen).float() * 0.5
    else:
        t = torch.randn(B, G + 1, V, generator=gen) * 2
    d = t[:, :G] + torch.randn(B, G, V, generator=gen) * 0.7
    if ties:
        d = torch.round(d * 2) / 2
    if dtype == "bf16":
        t, d = t.bfloat16(), d.bfloat16()
    x = torch.randint(0, V, (B, G), generator=gen, dtype=torch.int32)
    wl = workloads.Workload("edge", B, G, V, dtype, t.contiguous(), d.contiguous(), x, nd,
                            torch.full((B,), T) if np.isscalar(T) else torch.as_tensor(T, dtype=torch.float32),
                            None if k is None else torch.full((B,), k, dtype=torch.int32),
                            None if p is None else torch.full((B,), p, dtype=torch.float32), seed)
    return wl


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [2, 3, 5, 8, 37, 1000])
def test_small_and_ragged_vocab(dtype, V):
    for path in ("auto", "dense"):
        wl = _rand_batch(64, 3, V, dtype, seed=V, T=0.9, k=2 if V > 2 else None, p=0.8)
        rep, _, _ = run(wl, path=path, probs=True)
        assert_ok(rep)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_exact_ties(dtype):
    """Many equal logits: top-k / top-p / argmax ties must go to the lower token id."""
    # k = 100 and 200: every warp's share of a row holds more ties at the top than
    # the warps' lists can pass on together, so the piece's list is cut to exactly k
    for k, p in ((None, 0.7), (5, None), (5, 0.6), (100, None), (200, 0.9), (300, 0.9), (None, None)):
        for path in ("auto", "dense"):
            wl = _rand_batch(32, 4, 4096, dtype, seed=11, T=1.0, k=k, p=p, ties=True)
            rep, _, _ = run(wl, path=path, probs=True)
            assert_ok(rep)
    wl = _rand_batch(32, 4, 4096, dtype, seed=12, T=0.0, ties=True)
    for path in ("auto", "dense"):
        rep, _, _ = run(wl, path=path)
        assert_ok(rep)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_whole_row_top_p_both_variants(dtype):
    """Rows with top-p and no top-k take the whole-row kernel's nucleus cut.  A batch
    with at least two units per SM runs its 7-warp variant, a smaller one its 15-warp
    variant; both against the oracle, with the probability outputs (the kernel's
    generic per-element path) and without them (its packed full-tile path).  V spans
    one full segment and a ragged one in either variant."""
    from dataclasses import replace
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    G, V = 4, 9000
    for B in ((2 * sms) // (G + 1) + 8, 16):
        wl = _rand_batch(B, G, V, dtype, seed=40 + B, T=np.linspace(0.5, 1.5, B))
        wl = replace(wl, top_p=torch.as_tensor(np.linspace(0.5, 0.999, B), dtype=torch.float32),
                     num_draft=torch.as_tensor(1 + np.arange(B) % G, dtype=torch.int32))
        for probs in (False, True):
            rep, _, _ = run(wl, probs=probs)
            assert_ok(rep)


def test_mixed_parameters_per_row():
    B, G, V = 40, 5, 3000
    gen = torch.Generator().manual_seed(3)
    wl = _rand_batch(B, G, V, "f32", seed=3)
    wl.temperature = torch.tensor([0.0, 0.5, 1.0, 1.7] * 10)
    wl.top_k = torch.tensor([0, 1, 7, 50, 256, 257, 2999, 3000] * 5, dtype=torch.int32)
    wl.top_p = torch.tensor([1.0, 0.3, 0.95, 0.999, 0.5] * 8, dtype=torch.float32)
    wl.num_draft = torch.randint(1, G + 1, (B,), generator=gen, dtype=torch.int32)
    rep, _, _ = run(wl, probs=True)
    assert_ok(rep)


def test_invalid_rows_and_nonfinite_logits():
    B, G, V = 12, 3, 500
    wl = _rand_batch(B, G, V, "f32", seed=9, k=20, p=0.9)
    wl.temperature = torch.tensor([1.0, -1.0, float("nan"), float("inf")] + [1.0] * 8)
    wl.top_k = torch.tensor([20, 20, 20, 20, -1] + [20] * 7, dtype=torch.int32)
    wl.top_p = torch.tensor([0.9] * 5 + [0.0, 1.5, float("nan")] + [0.9] * 4, dtype=torch.float32)
    wl.num_draft = torch.tensor([3] * 8 + [0, 4, 3, 3], dtype=torch.int32)
    wl.draft_tokens[10, 1] = V
    wl.target[11, 2, 7] = float("nan")
    wl.target[0, 3, :] = float("-inf")  # bonus row of sequence 0 has no finite logit
    rep, g, ora = run(wl)
    assert_ok(rep)
    assert to_np(g["row_status"]).tolist() == ora.status.tolist()
    assert (ora.status[1:] != 0).sum() >= 10
    for path in ("dense",):
        rep, _, _ = run(wl, path=path)
        assert_ok(rep)


def test_masked_logits_and_zero_draft_probability():
    """-inf logits are masked tokens; a draft token outside q's support is accepted iff p(x) > 0."""
    B, G, V = 64, 4, 256
    wl = _rand_batch(B, G, V, "bf16", seed=21, k=30, p=0.8)
    wl.target[:, :, 200:] = float("-inf")
    wl.draft[:, :, :50] = float("-inf")
    wl.draft_tokens[:, :] = torch.randint(0, 60, (B, G), dtype=torch.int32)
    for path in ("auto", "dense"):
        rep, _, _ = run(wl, path=path, probs=True)
        assert_ok(rep)


def test_identical_rows_accept_everything():
    B, G, V = 16, 6, 2048
    wl = _rand_batch(B, G, V, "f32", seed=31)
    wl.draft = wl.target[:, :G].clone()
    gen = torch.Generator().manual_seed(1)
    probs = torch.softmax(wl.draft, dim=2)
    wl.draft_tokens = torch.multinomial(probs.view(-1, V), 1, generator=gen).view(B, G).to(torch.int32)
    for path in ("auto", "dense"):
        rep, g, _ = run(wl, path=path)
        assert_ok(rep)
        assert (to_np(g["accepted_len"]) == G).all()
        np.testing.assert_allclose(to_np(g["alpha"]), 1.0, atol=1e-5)


def test_empty_batch_and_host_entry_point():
    z = torch.empty(0, 4, 16, device="cuda")
    r = sv.spec_verify(z, torch.empty(0, 3, 16, device="cuda"), torch.empty(0, 3, dtype=torch.int32), [], seed=1)
    assert r["accepted_len"].numel() == 0
    wl = workloads.make("v32k", seed=8, B=8)
    dev = wl.to("cuda")
    ref = sv.spec_verify(dev.target, dev.draft, dev.draft_tokens, dev.temperature, seed=77)
    staging = torch.empty(sv.host_staging_size(8, 5, 32000, sv.SV_BF16, False, False, False), dtype=torch.uint8,
                          device="cuda")
    pin = lambda t: t.contiguous().pin_memory()
    h = sv.spec_verify_host(pin(wl.target), pin(wl.draft), pin(wl.draft_tokens), pin(wl.temperature), seed=77,
                            staging=staging)
    assert torch.equal(h["accepted_len"], ref["accepted_len"].cpu())
    assert torch.equal(h["out_tokens"], ref["out_tokens"].cpu())
    assert torch.equal(h["alpha"], ref["alpha"].cpu())


def test_determinism_and_seed_sensitivity():
    wl = workloads.make("v32k", seed=9, B=32).to("cuda")
    a = sv.spec_verify(wl.target, wl.draft, wl.draft_tokens, wl.temperature, seed=5)
    b = sv.spec_verify(wl.target, wl.draft, wl.draft_tokens, wl.temperature, seed=5)
    c = sv.spec_verify(wl.target, wl.draft, wl.draft_tokens, wl.temperature, seed=6)
    torch.cuda.synchronize()
    assert torch.equal(a["out_tokens"], b["out_tokens"]) and torch.equal(a["alpha"], b["alpha"])
    assert not torch.equal(a["out_tokens"], c["out_tokens"])
    assert torch.equal(a["alpha"], c["alpha"])  # alpha does not depend on the randomness


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_streaming_threshold_redo_and_overflow(dtype):
    """Rows that defeat the streaming kernel's speculative threshold: logits that
    fall along the row (the top-k all sit in the first tile, so fewer than k
    logits reach a threshold taken from that tile and the piece is redone
    conservatively), rows of equal logits (every logit passes, the warps'
    lists overflow and are cut exactly, ties to the lower id) and rows that
    rise along the row."""
    B, G, V = 6, 2, 128256 if dtype == "bf16" else 65536
    gen = torch.Generator().manual_seed(5)
    base = torch.linspace(4.0, -4.0, V)
    t = torch.empty(B, G + 1, V)
    t[0:2] = base + 0.01 * torch.randn(2, G + 1, V, generator=gen)   # falling
    t[2:4] = 1.5                                                       # all equal
    t[4:6] = base.flip(0) + 0.01 * torch.randn(2, G + 1, V, generator=gen)  # rising
    d = t[:, :G] + 0.05 * torch.randn(B, G, V, generator=gen)
    d[2:4] = 1.5
    if dtype == "bf16":
        t, d = t.bfloat16(), d.bfloat16()
    x = torch.randint(0, 64, (B, G), generator=gen, dtype=torch.int32)
    x[4:6] = V - 1 - x[4:6]
    for k in (1, 50, 200):
        wl = workloads.Workload("redo", B, G, V, dtype, t.contiguous(), d.contiguous(), x, None,
                                torch.full((B,), 0.9), torch.full((B,), k, dtype=torch.int32),
                                torch.full((B,), 0.95, dtype=torch.float32), 40 + k)
        rep, _, _ = run(wl, probs=True)
        assert_ok(rep)


# ---------------------------------------------------------------------------
# The output law on the GPU: the first emitted token follows the (filtered)
# target distribution p whatever the draft q ("Fast Inference from
# Transformers via Speculative Decoding" review page, Algorithm 1 and its
# correctness argument)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("k,p_top", [(None, None), (3, None), (None, 0.9)])
def test_chisquare_first_token_law_million_sequences(k, p_top):
    """10^6 sequences in one call (the select kernel's candidate lists are sized by
    the rows' length: 8 entries per row here), V = 8, gamma = 1, one (p, q) pair for
    all, x drawn from the filtered q: the first emitted token (the accepted draft or
    the residual draw) must follow the filtered p.  No filter runs the whole-row
    kernel, top-k 3 the select and combine kernels, top-p 0.9 the nucleus cut.
    The filtered laws come from the oracle (one row, probability outputs)."""
    stats = pytest.importorskip("scipy.stats")
    rng = np.random.default_rng(2024 + (k or 0) + int(100 * (p_top or 0)))
    V, B, calls = 8, 1_000_000, 1
    lp = np.log(rng.dirichlet(np.ones(V))).astype(np.float32)
    lq = np.log(rng.dirichlet(np.ones(V))).astype(np.float32)
    kk = None if k is None else np.array([k], dtype=np.int32)
    pp = None if p_top is None else np.array([p_top], dtype=np.float32)
    one = oracle.verify(np.stack([lp, lp])[None], lq[None, None], np.zeros((1, 1), dtype=np.int32),
                        np.ones(1, dtype=np.float32), None, kk, pp, seed=0, probs=True)
    p_law, q_law = one.p_out[0, 0], one.q_out[0, 0]
    dev = torch.device("cuda")
    tgt = torch.as_tensor(np.broadcast_to(np.stack([lp, lp])[None], (B, 2, V)).copy(), device=dev)
    drf = torch.as_tensor(np.broadcast_to(lq[None, None], (B, 1, V)).copy(), device=dev)
    counts = np.zeros(V, dtype=np.int64)
    for c in range(calls):
        x = rng.choice(V, size=(B, 1), p=q_law / q_law.sum()).astype(np.int32)
        res = sv.spec_verify(tgt, drf, torch.as_tensor(x, device=dev), 1.0, None,
                             None if k is None else k, None if p_top is None else p_top, seed=77 + c)
        torch.cuda.synchronize()
        assert (to_np(res["row_status"]) == 0).all()
        counts += np.bincount(to_np(res["out_tokens"])[:, 0], minlength=V)
    n = B * calls
    support = p_law > 0
    assert counts[~support].sum() == 0, (counts, p_law)
    _, pval = stats.chisquare(counts[support], p_law[support] / p_law[support].sum() * n)
    assert pval > 1e-3, (counts / n, p_law, pval)
