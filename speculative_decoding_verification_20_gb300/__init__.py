"""GB300-native batched speculative-sampling verification.

The computation lives in ``libspec_verify.so`` (hand-written sm_103a CUDA
behind the C ABI in ``include/spec_verify.h``).  This module is a thin ctypes
binding with the same names: it checks and marshals torch tensors (device
memory and streams) and nothing else.  There is no CPU fallback: if the
library is missing or no GPU is present, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import _build

SV_F32 = 0
SV_BF16 = 1
SV_PATH_AUTO = 0
SV_PATH_DENSE = 1
SV_STREAM_MAX_TOP_K = 256

ROW_BAD_TEMPERATURE = 0x01
ROW_BAD_TOP_K = 0x02
ROW_BAD_TOP_P = 0x04
ROW_BAD_NUM_DRAFT = 0x08
ROW_BAD_DRAFT_TOKEN = 0x10
ROW_NONFINITE = 0x20
ROW_INTERNAL = 0x40
ROW_BAD_LENIENCE = 0x80

# every symbol include/spec_verify.h declares
EXPORTED = ("spec_verify", "spec_verify_ex", "spec_verify_workspace_size", "spec_verify_host",
            "spec_verify_host_staging_size", "spec_verify_strerror", "spec_verify_static", "spec_verify_gumbel",
            "spec_verify_kseq", "spec_verify_kseq_workspace_size")
SV_MAX_KSEQ = 13

SV_ESCRATCH = -6
STATIC_SCRATCH_BYTES = 8 << 20  # SV_STATIC_SCRATCH_BYTES


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"spec_verify failed with status {status}: {msg}")
        self.status = status


class _Options(ctypes.Structure):
    _fields_ = [("struct_size", ctypes.c_uint32), ("pos_accept", ctypes.c_void_p), ("pos_token", ctypes.c_void_p),
                ("path", ctypes.c_int32), ("ev_stream", ctypes.c_void_p * 2), ("ev_dense", ctypes.c_void_p * 2),
                ("ev_free", ctypes.c_void_p * 2), ("lenience", ctypes.c_void_p), ("wait_limit_ns", ctypes.c_uint64),
                ("ev_gumbel", ctypes.c_void_p * 2)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load_library():
    """Load the in-tree CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise RuntimeError(f"{_build.LIB} is missing: build it with __graft_entry__.build() "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(_build.LIB)
    P, I, U64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t
    core = [P, P, I, P, P, P, P, P, U64, I, I, I, P, P, P, P, P, P, P, SZ, P]
    lib.spec_verify.argtypes = core
    lib.spec_verify.restype = I
    lib.spec_verify_ex.argtypes = core + [ctypes.POINTER(_Options)]
    lib.spec_verify_ex.restype = I
    lib.spec_verify_workspace_size.argtypes = [I, I, I, I]
    lib.spec_verify_workspace_size.restype = SZ
    lib.spec_verify_host_staging_size.argtypes = [I, I, I, I, I, I, I]
    lib.spec_verify_host_staging_size.restype = SZ
    lib.spec_verify_host.argtypes = [P, P, I, P, P, P, P, P, U64, I, I, I, P, P, P, P, SZ, P]
    lib.spec_verify_host.restype = I
    lib.spec_verify_static.argtypes = [P, P, I, P, P, P, P, P, U64, I, I, I, P, P, P, P, P, P, P]
    lib.spec_verify_static.restype = I
    lib.spec_verify_gumbel.argtypes = [P, I, P, P, P, P, P, U64, I, I, I, P, P, P, P, P, SZ, P,
                                       ctypes.POINTER(_Options)]
    lib.spec_verify_gumbel.restype = I
    lib.spec_verify_kseq_workspace_size.argtypes = [I, I, I, I]
    lib.spec_verify_kseq_workspace_size.restype = SZ
    lib.spec_verify_kseq.argtypes = [P, P, I, P, P, P, P, P, U64, I, I, I, P, P, P, P, SZ, P,
                                     ctypes.POINTER(_Options)]
    lib.spec_verify_kseq.restype = I
    lib.spec_verify_strerror.argtypes = [I]
    lib.spec_verify_strerror.restype = ctypes.c_char_p
    _lib = lib
    return lib


def strerror(status: int) -> str:
    return load_library().spec_verify_strerror(int(status)).decode()


def _check(status: int):
    if status != 0:
        raise SpecVerifyError(status, strerror(status))


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SV_F32
    if t.dtype == torch.bfloat16:
        return SV_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def workspace_size(B: int, G: int, V: int, dtype: int) -> int:
    return int(load_library().spec_verify_workspace_size(B, G, V, dtype))


def host_staging_size(B, G, V, dtype, has_num_draft, has_top_k, has_top_p) -> int:
    return int(load_library().spec_verify_host_staging_size(B, G, V, dtype, int(has_num_draft), int(has_top_k),
                                                            int(has_top_p)))


_ws_cache: dict = {}


def _workspace(nbytes: int, device: torch.device) -> torch.Tensor:
    key = (device.index,)
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = ws
    return ws


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev_vec(x, B: int, dtype: torch.dtype, device, name: str) -> Optional[torch.Tensor]:
    if x is None:
        return None
    if not torch.is_tensor(x):
        x = torch.as_tensor(x, dtype=dtype)
    if x.numel() == 1 and B != 1:
        x = x.reshape(1).expand(B)
    x = x.to(device=device, dtype=dtype).contiguous()
    if x.numel() != B:
        raise ValueError(f"{name} must have B={B} entries")
    return x


def spec_verify(target: torch.Tensor, draft: torch.Tensor, draft_tokens: torch.Tensor, temperature,
                num_draft=None, top_k=None, top_p=None, *, seed: int, probs: bool = False,
                positions: bool = False, path: str = "auto", events: Optional[dict] = None, stream=None,
                workspace: Optional[torch.Tensor] = None, lenience=None, wait_limit_ns: int = 0) -> dict:
    """Verify one batch of drafts on the GPU.

    target [B, G+1, V] and draft [B, G, V] (float32 or bfloat16, CUDA, contiguous),
    draft_tokens [B, G] int32; temperature / num_draft / top_k / top_p: per-sequence
    tensors, sequences or scalars (None = off / all G).  Returns a dict with
    accepted_len [B], out_tokens [B, G+1], alpha [B, G], row_status [B] and, on
    request, p_out / q_out (probs=True) and pos_accept / pos_token (positions=True).
    events: {"stream": (begin, end), "dense": (begin, end), "free": (begin, end)} torch.cuda.Event
    pairs that the library records on the launching stream around its streaming top-k, dense
    cluster and whole-row (no top-k) kernels.  lenience: per-sequence l in [0, 1] (None = 1, the
    exact rule): accept iff u * l * q(x) < p(x).  wait_limit_ns: limit of the kernels' waits on
    one another (0 = the default 2 s; a test hook for the give-up path).
    """
    lib = load_library()
    if not (target.is_cuda and draft.is_cuda):
        raise ValueError("target and draft must be CUDA tensors")
    dt = _dtype_code(target)
    if _dtype_code(draft) != dt:
        raise TypeError("target and draft dtypes differ")
    if target.dim() != 3 or draft.dim() != 3:
        raise ValueError("target must be [B, G+1, V] and draft [B, G, V]")
    B, G1, V = target.shape
    G = G1 - 1
    if tuple(draft.shape) != (B, G, V):
        raise ValueError(f"draft shape {tuple(draft.shape)} does not match target {tuple(target.shape)}")
    dev = target.device
    target = target.contiguous()
    draft = draft.contiguous()
    toks = draft_tokens.to(device=dev, dtype=torch.int32).contiguous()
    if tuple(toks.shape) != (B, G):
        raise ValueError("draft_tokens must be [B, G]")
    T = _dev_vec(temperature, B, torch.float32, dev, "temperature")
    nd = _dev_vec(num_draft, B, torch.int32, dev, "num_draft")
    tk = _dev_vec(top_k, B, torch.int32, dev, "top_k")
    tp = _dev_vec(top_p, B, torch.float32, dev, "top_p")
    ln = _dev_vec(lenience, B, torch.float32, dev, "lenience")

    acc = torch.empty(B, dtype=torch.int32, device=dev)
    out = torch.empty(B, G + 1, dtype=torch.int32, device=dev)
    alpha = torch.empty(B, G, dtype=torch.float32, device=dev)
    status = torch.empty(B, dtype=torch.int32, device=dev)
    p_out = torch.empty(B, G + 1, V, dtype=torch.float32, device=dev) if probs else None
    q_out = torch.empty(B, G, V, dtype=torch.float32, device=dev) if probs else None
    pa = torch.empty(B, G, dtype=torch.int32, device=dev) if positions else None
    pt = torch.empty(B, G + 1, dtype=torch.int32, device=dev) if positions else None

    need = workspace_size(B, G, V, dt)
    ws = workspace if workspace is not None else _workspace(need, dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    opts = _Options(ctypes.sizeof(_Options), _ptr(pa), _ptr(pt), SV_PATH_DENSE if path == "dense" else SV_PATH_AUTO)
    opts.lenience = None if ln is None else ln.data_ptr()
    opts.wait_limit_ns = int(wait_limit_ns)
    for key in ("stream", "dense", "free"):  # optional (begin, end) torch.cuda.Event pairs around each kernel
        if events and events.get(key):
            getattr(opts, "ev_" + key)[0] = events[key][0].cuda_event
            getattr(opts, "ev_" + key)[1] = events[key][1].cuda_event
    with torch.cuda.device(dev):
        rc = lib.spec_verify_ex(_ptr(target), _ptr(draft), dt, _ptr(toks), _ptr(nd), _ptr(T), _ptr(tk), _ptr(tp),
                                ctypes.c_uint64(int(seed) & 0xFFFFFFFFFFFFFFFF), B, G, V, _ptr(acc), _ptr(out),
                                _ptr(alpha), _ptr(p_out), _ptr(q_out), _ptr(status), _ptr(ws),
                                ws.numel(), ctypes.c_void_p(s.cuda_stream), ctypes.byref(opts))
    _check(rc)
    res = dict(accepted_len=acc, out_tokens=out, alpha=alpha, row_status=status)
    if probs:
        res.update(p_out=p_out, q_out=q_out)
    if positions:
        res.update(pos_accept=pa, pos_token=pt)
    return res


def spec_verify_gumbel(target: torch.Tensor, draft_tokens: torch.Tensor, temperature, num_draft=None, top_k=None,
                       top_p=None, *, seed: int, positions: bool = False, path: str = "auto",
                       events: Optional[dict] = None, stream=None, workspace: Optional[torch.Tensor] = None,
                       wait_limit_ns: int = 0) -> dict:
    """Shared-noise verification of one batch on the GPU: target [B, G+1, V] logits
    (float32 or bfloat16, CUDA), the drafter's tokens [B, G].  Returns accepted_len [B],
    out_tokens [B, G+1], target_tokens [B, G+1] (the target's noisy argmax at every
    position, -1 beyond gamma_b + 1), row_status [B] and, with positions=True,
    pos_accept [B, G] (draft k equals the target's token k).  events: as spec_verify,
    plus "gumbel": (begin, end) around the one-pass kernel of the unfiltered rows."""
    lib = load_library()
    if not target.is_cuda or target.dim() != 3:
        raise ValueError("target must be a CUDA tensor [B, G+1, V]")
    dt = _dtype_code(target)
    B, G1, V = target.shape
    G = G1 - 1
    dev = target.device
    target = target.contiguous()
    toks = draft_tokens.to(device=dev, dtype=torch.int32).contiguous()
    if tuple(toks.shape) != (B, G):
        raise ValueError("draft_tokens must be [B, G]")
    T = _dev_vec(temperature, B, torch.float32, dev, "temperature")
    nd = _dev_vec(num_draft, B, torch.int32, dev, "num_draft")
    tk = _dev_vec(top_k, B, torch.int32, dev, "top_k")
    tp = _dev_vec(top_p, B, torch.float32, dev, "top_p")
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    out = torch.empty(B, G + 1, dtype=torch.int32, device=dev)
    tt = torch.empty(B, G + 1, dtype=torch.int32, device=dev)
    status = torch.empty(B, dtype=torch.int32, device=dev)
    pa = torch.empty(B, G, dtype=torch.int32, device=dev) if positions else None
    need = workspace_size(B, G, V, dt)
    ws = workspace if workspace is not None else _workspace(need, dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    opts = _Options(ctypes.sizeof(_Options), _ptr(pa), None, SV_PATH_DENSE if path == "dense" else SV_PATH_AUTO)
    opts.wait_limit_ns = int(wait_limit_ns)
    for key in ("stream", "dense", "free", "gumbel"):
        if events and events.get(key):
            getattr(opts, "ev_" + key)[0] = events[key][0].cuda_event
            getattr(opts, "ev_" + key)[1] = events[key][1].cuda_event
    with torch.cuda.device(dev):
        rc = lib.spec_verify_gumbel(_ptr(target), dt, _ptr(toks), _ptr(nd), _ptr(T), _ptr(tk), _ptr(tp),
                                    ctypes.c_uint64(int(seed) & 0xFFFFFFFFFFFFFFFF), B, G, V, _ptr(acc), _ptr(out),
                                    _ptr(tt), _ptr(status), _ptr(ws), ws.numel(), ctypes.c_void_p(s.cuda_stream),
                                    ctypes.byref(opts))
    _check(rc)
    res = dict(accepted_len=acc, out_tokens=out, target_tokens=tt, row_status=status)
    if positions:
        res["pos_accept"] = pa
    return res


def spec_verify_kseq(target: torch.Tensor, draft: torch.Tensor, candidates: torch.Tensor, temperature,
                     num_candidates=None, top_k=None, top_p=None, *, seed: int, stream=None,
                     workspace: Optional[torch.Tensor] = None, events: Optional[dict] = None,
                     path: str = "auto") -> dict:
    """K-SEQ verification of one position per row on the GPU: target and draft logits
    [B, V] (float32 or bfloat16, CUDA), k candidates per row [B, K] (K <= 13).  Returns
    out_token [B], accepted [B] (the accepted candidate's index, -1: the residual draw)
    and row_status [B].  path="dense" sends every row to the cluster kernel; events:
    {"stream": (begin, end), "dense": (begin, end)} around those kernels."""
    lib = load_library()
    if not (target.is_cuda and draft.is_cuda) or target.dim() != 2 or tuple(draft.shape) != tuple(target.shape):
        raise ValueError("target and draft must be CUDA tensors [B, V] of one shape")
    dt = _dtype_code(target)
    if _dtype_code(draft) != dt:
        raise TypeError("target and draft dtypes differ")
    B, V = target.shape
    dev = target.device
    target, draft = target.contiguous(), draft.contiguous()
    cand = candidates.to(device=dev, dtype=torch.int32).contiguous()
    if cand.dim() != 2 or cand.shape[0] != B:
        raise ValueError("candidates must be [B, K]")
    K = cand.shape[1]
    T = _dev_vec(temperature, B, torch.float32, dev, "temperature")
    nc = _dev_vec(num_candidates, B, torch.int32, dev, "num_candidates")
    tk = _dev_vec(top_k, B, torch.int32, dev, "top_k")
    tp = _dev_vec(top_p, B, torch.float32, dev, "top_p")
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    acc = torch.empty(B, dtype=torch.int32, device=dev)
    status = torch.empty(B, dtype=torch.int32, device=dev)
    need = int(lib.spec_verify_kseq_workspace_size(B, K, V, dt))
    ws = workspace if workspace is not None else _workspace(max(need, 256), dev)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    opts = _Options(ctypes.sizeof(_Options), None, None, SV_PATH_DENSE if path == "dense" else SV_PATH_AUTO)
    for key in ("stream", "dense"):
        if events and events.get(key):
            getattr(opts, "ev_" + key)[0] = events[key][0].cuda_event
            getattr(opts, "ev_" + key)[1] = events[key][1].cuda_event
    with torch.cuda.device(dev):
        rc = lib.spec_verify_kseq(_ptr(target), _ptr(draft), dt, _ptr(cand), _ptr(nc), _ptr(T), _ptr(tk), _ptr(tp),
                                  ctypes.c_uint64(int(seed) & 0xFFFFFFFFFFFFFFFF), B, K, V, _ptr(tok), _ptr(acc),
                                  _ptr(status), _ptr(ws), ws.numel(), ctypes.c_void_p(s.cuda_stream),
                                  ctypes.byref(opts))
    _check(rc)
    return dict(out_token=tok, accepted=acc, row_status=status)


def spec_verify_host(target, draft, draft_tokens, temperature, num_draft=None, top_k=None, top_p=None, *,
                     seed: int, staging: torch.Tensor, outputs: Optional[dict] = None, stream=None) -> dict:
    """End-to-end form on host (ideally pinned) CPU tensors: copies in, verifies, copies out, synchronises."""
    lib = load_library()
    dt = _dtype_code(target)
    B, G1, V = target.shape
    G = G1 - 1
    host = lambda x, d: None if x is None else (x if torch.is_tensor(x) else torch.as_tensor(x)).to(d).contiguous()
    toks, T = host(draft_tokens, torch.int32), host(temperature, torch.float32)
    nd, tk, tp = host(num_draft, torch.int32), host(top_k, torch.int32), host(top_p, torch.float32)
    if outputs is None:
        outputs = dict(accepted_len=torch.empty(B, dtype=torch.int32).pin_memory(),
                       out_tokens=torch.empty(B, G + 1, dtype=torch.int32).pin_memory(),
                       alpha=torch.empty(B, G, dtype=torch.float32).pin_memory())
    s = stream if stream is not None else torch.cuda.current_stream(staging.device)
    with torch.cuda.device(staging.device):
        rc = lib.spec_verify_host(_ptr(target), _ptr(draft), dt, _ptr(toks), _ptr(nd), _ptr(T), _ptr(tk), _ptr(tp),
                                  ctypes.c_uint64(int(seed) & 0xFFFFFFFFFFFFFFFF), B, G, V,
                                  _ptr(outputs["accepted_len"]), _ptr(outputs["out_tokens"]), _ptr(outputs["alpha"]),
                                  _ptr(staging), staging.numel(), ctypes.c_void_p(s.cuda_stream))
    _check(rc)
    return outputs


def spec_verify_static(target: torch.Tensor, draft: torch.Tensor, draft_tokens: torch.Tensor, temperature,
                       num_draft=None, top_k=None, top_p=None, *, seed: int, stream=None,
                       outputs: Optional[dict] = None) -> dict:
    """The no-allocation form: the library's fixed device scratch instead of a workspace.

    For callers that must not allocate device memory between decode steps.  Pass
    ``outputs`` (accepted_len [B] int32, out_tokens [B, G+1] int32, alpha [B, G]
    float32, row_status [B] int32, all CUDA) to make the call allocate nothing
    here either; parameter vectors given as CUDA int32/float32 tensors of B
    entries are passed through as they are.  Raises SpecVerifyError with status
    SV_ESCRATCH when the shape needs more than STATIC_SCRATCH_BYTES of scratch.
    Calls that can overlap on the GPU share the scratch and race: keep them on
    one stream.
    """
    lib = load_library()
    if not (target.is_cuda and draft.is_cuda):
        raise ValueError("target and draft must be CUDA tensors")
    dt = _dtype_code(target)
    if _dtype_code(draft) != dt:
        raise TypeError("target and draft dtypes differ")
    B, G1, V = target.shape
    G = G1 - 1
    if tuple(draft.shape) != (B, G, V) or not (target.is_contiguous() and draft.is_contiguous()):
        raise ValueError("target [B, G+1, V] and draft [B, G, V] must be contiguous and match")
    dev = target.device
    toks = draft_tokens.to(device=dev, dtype=torch.int32).contiguous()
    T = _dev_vec(temperature, B, torch.float32, dev, "temperature")
    nd = _dev_vec(num_draft, B, torch.int32, dev, "num_draft")
    tk = _dev_vec(top_k, B, torch.int32, dev, "top_k")
    tp = _dev_vec(top_p, B, torch.float32, dev, "top_p")
    if outputs is None:
        outputs = dict(accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
                       out_tokens=torch.empty(B, G + 1, dtype=torch.int32, device=dev),
                       alpha=torch.empty(B, G, dtype=torch.float32, device=dev),
                       row_status=torch.empty(B, dtype=torch.int32, device=dev))
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    with torch.cuda.device(dev):
        rc = lib.spec_verify_static(_ptr(target), _ptr(draft), dt, _ptr(toks), _ptr(nd), _ptr(T), _ptr(tk), _ptr(tp),
                                    ctypes.c_uint64(int(seed) & 0xFFFFFFFFFFFFFFFF), B, G, V,
                                    _ptr(outputs["accepted_len"]), _ptr(outputs["out_tokens"]),
                                    _ptr(outputs["alpha"]), None, None, _ptr(outputs.get("row_status")),
                                    ctypes.c_void_p(s.cuda_stream))
    _check(rc)
    return outputs
