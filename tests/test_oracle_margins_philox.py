"""Pins of the oracle parts the parity rule leans on, against things other than
the oracle itself.

* Philox4x32-10 ("Parallel Random Numbers: As Easy as 1, 2, 3", Salmon et al.,
  SC'11): the oracle's block function against PyTorch's own header-only
  implementation of the same generator (``at::philox_engine``, written
  independently of this repository), on explicit counters and keys.  The
  engine's key is its seed (low word first), its counter words 2-3 are the
  subsequence and words 0-1 the offset; four calls return the four output words
  of one block.
* The decision margins that decide which GPU/oracle mismatches the parity rule
  excuses: each test builds a case whose margin is known by construction and
  checks the oracle reports exactly that margin.
    - acceptance ("Speculative decoding: the art of guessing well", section 投机采样,
      the `verify` listing: accept iff u < p/q): margin |u - p(x)/q(x)|;
    - residual draw ("Fast Inference from Transformers via Speculative Decoding"
      review page, Algorithm 1 steps 4-5): the distance of v = u Z to the nearest
      edge of the cumulative residual, relative to Z;
    - filters (same review page, section "Method: Speculative Decoding"): top-p's
      distance of the running mass to P at the cut, and the relative gap between
      the k-th and (k+1)-th probability for top-k.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

_PHILOX_PROBE = r"""
#include <ATen/core/PhiloxRNGEngine.h>
#include <cstdio>
int main() {
    unsigned c0, c1, c2, c3, k0, k1;
    while (std::scanf("%u %u %u %u %u %u", &c0, &c1, &c2, &c3, &k0, &k1) == 6) {
        at::philox_engine e(((uint64_t)k1 << 32) | k0, ((uint64_t)c3 << 32) | c2, ((uint64_t)c1 << 32) | c0);
        const unsigned w0 = e(), w1 = e(), w2 = e(), w3 = e();
        std::printf("%u %u %u %u\n", w0, w1, w2, w3);
    }
    return 0;
}
"""


@pytest.fixture(scope="module")
def torch_philox(tmp_path_factory):
    torch = pytest.importorskip("torch")
    inc = os.path.join(os.path.dirname(torch.__file__), "include")
    if not os.path.exists(os.path.join(inc, "ATen", "core", "PhiloxRNGEngine.h")) or not shutil.which("g++"):
        pytest.skip("PyTorch's Philox header or g++ is not available")
    d = tmp_path_factory.mktemp("philox")
    src, exe = d / "probe.cpp", d / "probe"
    src.write_text(_PHILOX_PROBE)
    subprocess.run(["g++", "-O1", "-std=c++17", "-I" + inc, str(src), "-o", str(exe)], check=True)

    def run(rows):
        inp = "".join(" ".join(str(int(v)) for v in r) + "\n" for r in rows)
        out = subprocess.run([str(exe)], input=inp, capture_output=True, text=True, check=True).stdout
        return np.array([[int(x) for x in line.split()] for line in out.strip().splitlines()], dtype=np.uint64)

    return run


def test_philox_block_matches_pytorch_engine(oracle_mod, torch_philox):
    rng = np.random.default_rng(7)
    rows = [(0, 0, 0, 0, 0, 0), (0xFFFFFFFF,) * 6, (1, 0, 0, 0, 0, 0), (0, 0, 0, 1, 0, 0), (0, 0, 0, 0, 0, 1),
            (3, 5, 1, 0, 0xDEADBEEF, 0x12345678)]
    rows += [tuple(int(x) for x in rng.integers(0, 2 ** 32, 6, dtype=np.uint64)) for _ in range(58)]
    ref = torch_philox(rows)
    assert ref.shape == (len(rows), 4)
    for r, want in zip(rows, ref):
        got = oracle_mod.philox4x32_10(r[:4], r[4:])
        assert [int(x) for x in got] == [int(x) for x in want], (r, got, want)


def test_uniforms_use_word0_of_the_documented_counter(oracle_mod, torch_philox):
    # U(seed, b, pos, draw) = ((w >> 8) + 1/2) 2^-24, w = word 0 of counter (b, pos, draw, 0), key (lo, hi) of seed
    seeds = [0, 1, 2 ** 32 + 7, 0xFEDCBA9876543210]
    cases = [(s, b, pos, draw) for s in seeds for (b, pos, draw) in ((0, 1, 0), (5, 3, 1), (1023, 8, 0), (7, 2, 2))]
    ref = torch_philox([(b, pos, draw, 0, s & 0xFFFFFFFF, s >> 32) for (s, b, pos, draw) in cases])
    for (s, b, pos, draw), w in zip(cases, ref):
        assert oracle_mod.uniform(s, b, pos, draw) == ((int(w[0]) >> 8) + 0.5) / 2 ** 24
    # the shared-noise draw of token i uses word i & 3 of counter (b, k, 2, i >> 2)
    for i in range(8):
        w = torch_philox([(3, 2, 2, i >> 2, 11, 0)])[0]
        assert oracle_mod.gumbel_uniform(11, 3, 2, i) == ((int(w[i & 3]) >> 8) + 0.5) / 2 ** 24


# ---------------------------------------------------------------------------
# decision margins
# ---------------------------------------------------------------------------

def _one(oracle_mod, tlog, dlog, x, ua, ur, T=1.0, k=None, p=None):
    """One sequence, gamma = len(x), explicit uniforms, every per-position output."""
    t = np.asarray(tlog, dtype=np.float32)[None]
    d = np.asarray(dlog, dtype=np.float32)[None]
    G = d.shape[1]
    return oracle_mod.verify(t, d, np.asarray(x, dtype=np.int32)[None], np.full(1, T, np.float32), None,
                             None if k is None else np.array([k], np.int32),
                             None if p is None else np.array([p], np.float32),
                             u_accept=np.asarray(ua, dtype=np.float64).reshape(1, G),
                             u_resid=np.asarray(ur, dtype=np.float64).reshape(1, G + 1), all_positions=True,
                             probs=True)


@pytest.mark.parametrize("delta", [3e-7, -2e-6, 0.25])
def test_acceptance_margin_is_distance_of_u_to_p_over_q(oracle_mod, delta):
    # target row 1 uniform over 2 tokens (p = 1/2 each); draft row 1 puts all its mass on token 1
    # (q(1) = 1): p(1)/q(1) = 1/2 exactly, so u = 1/2 + delta is delta away from the boundary
    neg = -np.inf
    r = _one(oracle_mod, [[0.0, 0.0], [0.0, 0.0]], [[neg, 0.0]], [1], [0.5 + delta], [0.5, 0.5])
    assert r.accept_margin[0, 0] == pytest.approx(abs(delta), rel=1e-12, abs=1e-16)
    assert r.pos_accept[0, 0] == int(0.5 + delta < 0.5)
    # the same row with q(1) = 1/4 (draft logits ln 3, 0): ratio 2 -> u is 2 - u away
    r = _one(oracle_mod, [[0.0, 0.0], [0.0, 0.0]], [[np.log(3.0), 0.0]], [1], [0.5], [0.5, 0.5])
    p1, q1 = r.p_out[0, 0, 1], r.q_out[0, 0, 1]
    assert r.accept_margin[0, 0] == pytest.approx(abs(0.5 - p1 / q1), rel=1e-12)
    assert abs(p1 / q1 - 2.0) < 1e-6


def test_acceptance_margin_infinite_when_draft_probability_is_zero(oracle_mod):
    neg = -np.inf
    r = _one(oracle_mod, [[0.0, 0.0], [0.0, 0.0]], [[neg, 0.0]], [0], [0.3], [0.5, 0.5])
    assert np.isinf(r.accept_margin[0, 0]) and r.pos_accept[0, 0] == 1


@pytest.mark.parametrize("delta", [1e-7, 0.013])
def test_residual_margin_is_relative_to_the_residual_mass(oracle_mod, delta):
    # p = (0.4, 0.4, 0.2), q = (0.2, 0.1, 0.7): r = (0.2, 0.3, 0), Z = 0.5 (not 1, so a margin
    # left unscaled by Z would be half the true one).  Edges of the running residual: 0.2, 0.5.
    # u chosen so v = u Z lies delta * Z above the edge 0.2.
    pt = np.log(np.array([0.4, 0.4, 0.2]))
    qd = np.log(np.array([0.2, 0.1, 0.7]))
    probe = _one(oracle_mod, [pt, pt], [qd], [2], [0.99], [0.5, 0.5])
    p, q = probe.p_out[0, 0], probe.q_out[0, 0]
    rr = np.maximum(p - q, 0.0)
    Z = rr.sum()
    assert abs(Z - 0.5) < 1e-6
    edge = rr[0]
    u = (edge + delta * Z) / Z
    r = _one(oracle_mod, [pt, pt], [qd], [2], [0.99], [u, 0.5])
    assert r.pos_token[0, 0] == 1
    assert r.resid_margin[0, 0] == pytest.approx(delta, rel=1e-9)
    # and from the upper edge of token 1's interval (the total Z)
    u = (Z - delta * Z) / Z
    r = _one(oracle_mod, [pt, pt], [qd], [2], [0.99], [u, 0.5])
    assert r.pos_token[0, 0] == 1 and r.resid_margin[0, 0] == pytest.approx(delta, rel=1e-9)


def test_bonus_margin_uses_target_mass(oracle_mod):
    # bonus row (q := 0): r = p, Z = 1; p = (0.25, 0.75) -> edges 0.25, 1.0
    pt = np.log(np.array([0.25, 0.75]))
    probe = _one(oracle_mod, [pt, pt], [pt], [0], [0.1], [0.5, 0.5])
    edge = probe.p_out[0, 1, 0]
    assert abs(edge - 0.25) < 1e-6 and abs(probe.p_out[0, 1].sum() - 1.0) < 1e-15
    r = _one(oracle_mod, [pt, pt], [pt], [0], [0.1], [0.5, edge + 0.0625])
    assert r.accepted_len[0] == 1
    assert r.pos_token[0, 1] == 1
    assert r.resid_margin[0, 1] == pytest.approx(0.0625, rel=1e-9)


@pytest.mark.parametrize("delta", [2e-7, 0.04])
def test_top_p_filter_margin_is_mass_distance_to_P(oracle_mod, delta):
    # sorted probabilities (0.5, 0.3, 0.2): with P = 0.8 - delta the running mass crosses at the
    # second token with 0.8 - P = delta to spare; with P = 0.5 + delta it needs the second token by
    # P - 0.5 = delta.  The other distances (0.3 - delta, the 1/3 ratio gap) are larger.
    row = np.log(np.array([0.3, 0.5, 0.2]))
    for P in (0.8 - delta, 0.5 + delta):
        probs, m = oracle_mod.normalise(row.astype(np.float32), 1.0, 0, np.float32(P), with_margin=True)
        Pf = float(np.float32(P))  # the kernels and the oracle take top-p as a float
        s = np.sort(oracle_mod.normalise(row.astype(np.float32), 1.0))[::-1]
        want = min(s[0] + s[1] - Pf, Pf - s[0])
        assert m == pytest.approx(want, rel=1e-9, abs=1e-15)
        assert abs(m - delta) < 1e-7
        assert (probs > 0).sum() == 2


@pytest.mark.parametrize("delta", [1e-7, 0.1])
def test_top_k_filter_margin_is_relative_gap_at_k(oracle_mod, delta):
    # k = 2 keeps (0.4, 0.3); the third probability is 0.3 (1 - delta): margin delta
    p = np.array([0.4, 0.3, 0.3 * (1 - delta), 0.1])
    row = np.log(p / p.sum()).astype(np.float64)
    probs, m = oracle_mod.normalise(row, 1.0, 2, 1.0, with_margin=True)
    s = np.sort(oracle_mod.normalise(row, 1.0))[::-1]
    assert m == pytest.approx((s[1] - s[2]) / s[1], rel=1e-9)
    assert m == pytest.approx(delta, rel=1e-6)
    # an exact tie at the cut is decided by token id on both sides: no margin from it
    tie = np.log(np.array([0.4, 0.3, 0.3, 0.1])).astype(np.float64)
    _, m2 = oracle_mod.normalise(tie, 1.0, 2, 1.0, with_margin=True)
    assert np.isinf(m2)


def test_filter_margins_reach_the_verify_outputs(oracle_mod):
    # the row margins verify reports are those of normalise, row by row (target rows 0..G, then draft)
    rng = np.random.default_rng(3)
    t = rng.normal(size=(3, 50)).astype(np.float32)
    d = rng.normal(size=(2, 50)).astype(np.float32)
    r = _one(oracle_mod, t, d, [1, 2], [0.5, 0.5], [0.5, 0.5, 0.5], T=0.9, k=10, p=0.7)
    for j in range(3):
        _, m = oracle_mod.normalise(t[j], np.float32(0.9), 10, np.float32(0.7), with_margin=True)
        assert r.filter_margin[0, j] == m
    for j in range(2):
        _, m = oracle_mod.normalise(d[j], np.float32(0.9), 10, np.float32(0.7), with_margin=True)
        assert r.filter_margin[0, 3 + j] == m
