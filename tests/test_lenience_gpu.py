"""Lenient acceptance on the GPU ("Fast Inference from Transformers via
Speculative Decoding" review page, section Lenience): a per-sequence l in
[0, 1] scales q(x) in the acceptance test, u * l * q(x) < p(x), and alpha
becomes sum_x min(q, p / l).  Every path of the library against the oracle on
the same inputs and uniforms: the streaming top-k path, the whole-row path
(with and without top-p) and the dense cluster path."""
import numpy as np
import pytest
import torch

from tests.parity import assert_ok
from tests.test_parity_gpu import _rand_batch, run

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_20_gb300")
from speculative_decoding_verification_20_gb300 import workloads  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import oracle
    from speculative_decoding_verification_20_gb300 import _build

    _build.build()
    oracle.build()


def _lenience(B, seed):
    rng = np.random.default_rng(seed)
    l = rng.uniform(0.05, 1.0, B).astype(np.float32)
    l[::5] = 1.0  # some sequences keep the exact rule
    return l


@pytest.mark.parametrize("name,kw", [("v128k", dict(B=6)), ("v32k", dict(B=24)), ("ragged", dict(B=12, V=20000)),
                                     ("b1024", dict(B=64))])
def test_lenient_parity_each_workload(name, kw):
    wl = workloads.make(name, seed=70, **kw)
    l = _lenience(wl.B, 1)
    rep, g, ora = run(wl, lenience=l, probs=True)
    assert_ok(rep)
    # lenience only raises alpha: compare with the exact rule on the same inputs
    rep1, g1, _ = run(wl)
    assert_ok(rep1)
    a_len, a_ex = g["alpha"].cpu().numpy(), g1["alpha"].cpu().numpy()
    assert (a_len >= a_ex - 1e-6).all()


@pytest.mark.parametrize("path", ["auto", "dense"])
def test_lenient_parity_mixed_rows(path):
    B, G, V = 40, 4, 3000
    wl = _rand_batch(B, G, V, "f32", seed=17)
    wl.temperature = torch.tensor([0.0, 0.5, 1.0, 1.7] * 10)
    wl.top_k = torch.tensor([0, 1, 7, 50, 256, 300, 0, 0] * 5, dtype=torch.int32)
    wl.top_p = torch.tensor([1.0, 0.3, 0.95, 0.999, 0.5] * 8, dtype=torch.float32)
    l = np.tile(np.array([1.0, 0.5, 0.2, 0.05, 0.9, 0.0, 0.33, 0.7], np.float32), 5)
    rep, _, _ = run(wl, lenience=l, path=path, probs=True)
    assert_ok(rep)


def test_bad_lenience_marks_the_sequence():
    wl = _rand_batch(6, 2, 500, "f32", seed=3, k=20)
    l = np.array([1.0, -0.5, 1.01, np.nan, 0.0, 0.25], np.float32)
    rep, g, ora = run(wl, lenience=l)
    assert_ok(rep)
    st = g["row_status"].cpu().numpy()
    assert list(st & sv.ROW_BAD_LENIENCE) == [0, sv.ROW_BAD_LENIENCE, sv.ROW_BAD_LENIENCE, sv.ROW_BAD_LENIENCE, 0, 0]
    assert list(st) == list(ora.status)
