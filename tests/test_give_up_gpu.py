"""The device side of failure detection, exercised without a GPU fault: every
wait of one kernel on another warp or on a copy is bounded, and the test
shortens the bound (sv_options.wait_limit_ns, the library's test hook) until
waits run out.  The call must still return, the sequences of a kernel that
gave up (and of the paths after it in the same call) must carry
SV_ROW_INTERNAL with the defaults of an invalid sequence, every other
sequence must be untouched, and the next call with the default limit on the
same workspace must be correct again."""
import numpy as np
import pytest
import torch

from tests.parity import assert_ok
from tests.test_parity_gpu import run

pytestmark = pytest.mark.gpu

sv = pytest.importorskip("speculative_decoding_verification_20_gb300")
from speculative_decoding_verification_20_gb300 import workloads  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from speculative_decoding_verification_20_gb300 import _build

    _build.build()


@pytest.mark.parametrize("name,kw", [("v128k", dict(B=16)), ("ragged", dict(B=16, V=60000)),
                                     ("b1024", dict(B=128))])
def test_waits_that_run_out_mark_sequences_and_leave_the_device_usable(name, kw):
    wl = workloads.make(name, seed=31, device="cuda", **kw)
    ws = torch.empty(sv.workspace_size(wl.B, wl.G, wl.V, sv.SV_BF16 if wl.dtype == "bf16" else sv.SV_F32),
                     dtype=torch.uint8, device="cuda")
    args = (wl.target, wl.draft, wl.draft_tokens, wl.temperature, wl.num_draft, wl.top_k, wl.top_p)
    ref = sv.spec_verify(*args, seed=5, workspace=ws)
    torch.cuda.synchronize()
    gave_up = 0
    for attempt in range(6):
        r = sv.spec_verify(*args, seed=5, workspace=ws, wait_limit_ns=1)
        torch.cuda.synchronize()  # the call returned and its kernels ended
        st = r["row_status"].cpu().numpy()
        bad = (st & sv.ROW_INTERNAL) != 0
        gave_up += int(bad.any())
        assert ((st == 0) | (st == sv.ROW_INTERNAL)).all(), st
        acc, out, alpha = (r[k].cpu().numpy() for k in ("accepted_len", "out_tokens", "alpha"))
        assert (acc[bad] == 0).all() and (out[bad] == -1).all() and (alpha[bad] == 0).all()
        ok = ~bad
        np.testing.assert_array_equal(acc[ok], ref["accepted_len"].cpu().numpy()[ok])
        np.testing.assert_array_equal(out[ok], ref["out_tokens"].cpu().numpy()[ok])
        np.testing.assert_array_equal(alpha[ok], ref["alpha"].cpu().numpy()[ok])
    assert gave_up >= 1, "no wait ran out at a 1 ns limit"
    # the default limit on the same workspace: correct again, against the oracle
    rep, g, _ = run(wl, seed=6, rows=list(range(0, wl.B, 3)))
    assert_ok(rep)
    assert (g["row_status"].cpu().numpy() & sv.ROW_INTERNAL == 0).all()
