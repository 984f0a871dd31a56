"""The C ABI library: it loads without a GPU, exports every symbol include/*.h
declares, and rejects bad arguments on the host before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(spec_verify[a-z_0-9]*)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    import speculative_decoding_verification_20_gb300 as sv
    from speculative_decoding_verification_20_gb300 import _build

    _build.build()
    return sv.load_library()


def test_every_declared_symbol_is_exported(lib):
    import speculative_decoding_verification_20_gb300 as sv

    declared = _declared_functions()
    assert set(declared) == set(sv.EXPORTED), declared
    for name in declared:
        assert hasattr(lib, name), name


def test_workspace_size_is_a_host_function(lib):
    import speculative_decoding_verification_20_gb300 as sv

    a = sv.workspace_size(256, 7, 128256, sv.SV_BF16)
    b = sv.workspace_size(256, 7, 128256, sv.SV_F32)
    assert a > 0 and b > a  # fp32 pieces hold half the elements, so more pieces per row
    assert sv.workspace_size(0, 7, 128256, sv.SV_BF16) > 0
    assert sv.workspace_size(1, 0, 10, sv.SV_F32) == 0
    assert sv.workspace_size(1, 33, 10, sv.SV_F32) == 0
    assert sv.workspace_size(1, 4, 262145, sv.SV_F32) == 0
    assert sv.workspace_size(1, 4, 10, 7) == 0


def test_strerror(lib):
    import speculative_decoding_verification_20_gb300 as sv

    assert sv.strerror(0) == "success"
    for s in (-1, -2, -3, -4, -5):
        assert sv.strerror(s) and sv.strerror(s) != "unknown status"
    assert sv.strerror(-99) == "unknown status"


def test_bad_arguments_rejected_before_any_launch(lib):
    """These return before any CUDA call, so they run on a machine without a GPU."""
    P = ctypes.c_void_p
    good = P(0x10000)  # never dereferenced: validation fails first
    null = None

    def call(target=good, draft=good, dtype=0, tokens=good, temp=good, B=2, G=3, V=64, acc=good, out=good,
             alpha=good, ws=good, wsb=1 << 40):
        return lib.spec_verify(target, draft, dtype, tokens, null, temp, null, null, ctypes.c_uint64(1), B, G, V, acc,
                               out, alpha, null, null, null, ws, ctypes.c_size_t(wsb), null)

    assert call(B=0) == 0  # empty batch: nothing to do
    assert call(dtype=5) == -2
    assert call(G=0) == -1
    assert call(V=0) == -1
    assert call(B=-1) == -1
    assert call(G=33) == -4
    assert call(V=262145) == -4
    assert call(target=None) == -1
    assert call(tokens=None) == -1
    assert call(alpha=None) == -1
    assert call(target=P(0x10008)) == -1  # logits must be 16-byte aligned
    assert call(ws=None) == -5
    assert call(wsb=16) == -5
    assert call(ws=P(0x10010)) == -1  # workspace must be 256-byte aligned
