"""spec_verify_static: the form that allocates nothing (the library's fixed
device scratch instead of a caller's workspace).

It must give what spec_verify gives on the same inputs, on consecutive calls
that reuse the one scratch buffer, and refuse shapes that need more scratch
than it has before touching the GPU.  This file is named to run last, so the
GPU test also runs after every other test has used the library.
"""
import ctypes

import numpy as np
import pytest
import torch

from tests.parity import ALPHA_TOL

sv = pytest.importorskip("speculative_decoding_verification_20_gb300")
from speculative_decoding_verification_20_gb300 import workloads  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_20_gb300 import _build

    _build.build()
    return sv.load_library()


def test_static_rejects_shapes_beyond_its_scratch(lib):
    # B = 4096 at gamma 7, V 128256 needs far more than the fixed scratch; the
    # call must say so before it looks at any pointer or the device
    B, G, V = 4096, 7, 128256
    assert sv.workspace_size(B, G, V, sv.SV_BF16) > sv.STATIC_SCRATCH_BYTES
    null = ctypes.c_void_p(0)
    rc = lib.spec_verify_static(null, null, sv.SV_BF16, null, null, null, null, null, ctypes.c_uint64(0), B, G, V,
                                null, null, null, null, null, null, null)
    assert rc == sv.SV_ESCRATCH
    assert "spec_verify_static" in sv.strerror(rc)
    # invalid shapes keep the errors of spec_verify
    assert lib.spec_verify_static(null, null, sv.SV_BF16, null, null, null, null, null, ctypes.c_uint64(0), 1, 0, V,
                                  null, null, null, null, null, null, null) == -1


def _fits(wl):
    es = sv.SV_BF16 if wl.dtype == "bf16" else sv.SV_F32
    return sv.workspace_size(wl.B, wl.G, wl.V, es) <= sv.STATIC_SCRATCH_BYTES


@pytest.mark.gpu
@pytest.mark.parametrize("name,B", [("v128k", 24), ("ragged", 6), ("v32k", 16)])
def test_static_matches_workspace_form_on_consecutive_calls(lib, name, B):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    wl = workloads.make(name, seed=5, device="cuda", B=B)
    assert _fits(wl)
    for seed in (101, 102):  # two calls in a row on the same scratch
        got = sv.spec_verify_static(wl.target, wl.draft, wl.draft_tokens, wl.temperature, wl.num_draft, wl.top_k,
                                    wl.top_p, seed=seed)
        ref = sv.spec_verify(wl.target, wl.draft, wl.draft_tokens, wl.temperature, wl.num_draft, wl.top_k, wl.top_p,
                             seed=seed)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(got["accepted_len"].cpu().numpy(), ref["accepted_len"].cpu().numpy())
        np.testing.assert_array_equal(got["out_tokens"].cpu().numpy(), ref["out_tokens"].cpu().numpy())
        np.testing.assert_array_equal(got["row_status"].cpu().numpy(), ref["row_status"].cpu().numpy())
        np.testing.assert_allclose(got["alpha"].cpu().numpy(), ref["alpha"].cpu().numpy(), rtol=0, atol=ALPHA_TOL)
