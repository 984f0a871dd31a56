"""Pins of the oracle's SpecTr round ("SpecTr: Fast Speculative Decoding via Optimal
Transport" page, section SpecTr: K draft sequences, K-SEQ along their prefix tree),
CPU only.  A toy model over V = 3 tokens whose rows depend on the prefix:
target p1 = softmax(a0), p2(. | y1) = softmax(A[y1]), bonus p3(. | y1, y2) =
softmax(C[y1, y2]); draft q1 = softmax(d0), q2(. | x1) = softmax(D[x1])."""
import numpy as np
import pytest

stats = pytest.importorskip("scipy.stats")

V, L = 3, 2


def _model(seed):
    r = np.random.default_rng(seed)
    return dict(a0=r.normal(size=V), A=r.normal(size=(V, V)), C=r.normal(size=(V, V, V)),
                d0=r.normal(size=V), D=r.normal(size=(V, V)))


def _softmax(z):
    e = np.exp(z - z.max())
    return e / e.sum()


def _draw(m, K, rng):
    """K draft sequences of length 2 from the drafter, and their rows."""
    tok = np.zeros((K, L), dtype=np.int32)
    for j in range(K):
        x1 = rng.choice(V, p=_softmax(m["d0"]))
        tok[j] = (x1, rng.choice(V, p=_softmax(m["D"][x1])))
    tgt = np.stack([np.stack([m["a0"], m["A"][t[0]], m["C"][t[0], t[1]]]) for t in tok]).astype(np.float32)
    drf = np.stack([np.stack([m["d0"], m["D"][t[0]]]) for t in tok]).astype(np.float32)
    return tok, tgt, drf


def test_one_candidate_is_speculative_decoding(oracle_mod):
    """K = 1: the round is the sampling verification of one draft, with the same uniforms
    (acceptance U(seed, b, pos, 3), residual / bonus U(seed, b, pos, 1))."""
    m, rng, seed, n = _model(1), np.random.default_rng(2), 5, 300
    for b in range(n):
        tok, tgt, drf = _draw(m, 1, rng)
        got = oracle_mod.spectr_round(tgt, drf, tok, seed=seed, b=b)
        ua = np.array([[oracle_mod.uniform(seed, b, i + 1, 3) for i in range(L)]])
        ur = np.array([[oracle_mod.uniform(seed, b, j + 1, 1) for j in range(L + 1)]])
        r = oracle_mod.verify(tgt, drf, tok, np.ones(1, dtype=np.float32), u_accept=ua, u_resid=ur)
        n_acc = int(r.accepted_len[0])
        assert got.tolist() == r.out_tokens[0, : n_acc + 1].tolist()


def _rounds(oracle_mod, m, K, n, seed):
    rng = np.random.default_rng(100 + K)
    out = []
    for b in range(n):
        tok, tgt, drf = _draw(m, K, rng)
        out.append(oracle_mod.spectr_round(tgt, drf, tok, seed=seed, b=b))
    return out


def test_emitted_tokens_follow_the_target(oracle_mod):
    """The first emitted token follows p1; given the first token y1 and that the round
    went on, the second follows p2(. | y1) (the target's own autoregressive law)."""
    m = _model(3)
    outs = _rounds(oracle_mod, m, 3, 60_000, seed=11)
    first = np.array([o[0] for o in outs])
    _, pv = stats.chisquare(np.bincount(first, minlength=V), _softmax(m["a0"]) * len(outs))
    assert pv > 1e-3
    for y1 in range(V):
        sec = np.array([o[1] for o in outs if len(o) > 1 and o[0] == y1])
        if len(sec) < 2000:
            continue
        _, pv2 = stats.chisquare(np.bincount(sec, minlength=V), _softmax(m["A"][y1]) * len(sec))
        assert pv2 > 1e-3, (y1, len(sec))


def test_more_candidates_emit_more_tokens(oracle_mod):
    """Block efficiency: with K = 4 candidates a round emits more tokens on average than
    with one (the page's K-SEQ never accepts less mass than a single candidate)."""
    m = _model(4)
    n = 20_000
    one = np.mean([len(o) for o in _rounds(oracle_mod, m, 1, n, seed=21)])
    four = np.mean([len(o) for o in _rounds(oracle_mod, m, 4, n, seed=21)])
    assert four > one + 5 * np.sqrt(2 * 0.7 / n), (one, four)
    assert 1.0 <= one <= L + 1 and four <= L + 1
