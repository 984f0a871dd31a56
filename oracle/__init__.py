"""CPU oracle for batched speculative-sampling verification (fp64, plain C).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (the CUDA library and its Python binding) never
imports, links or calls it, and it shares no code with them.

The arithmetic lives in ``spec_verify_ref.c`` (see its header for the passages
of the pages each function follows); this module only builds that file with
gcc and marshals numpy arrays through ctypes.

Parity status per function:
  * normalise / alpha / acceptance / residual -- pinned (tests/test_oracle_pins.py);
    decision margins pinned (tests/test_oracle_margins_philox.py)
  * lenience (verify with ``lenience``) -- pinned (tests/test_lenience_oracle.py)
  * gumbel_verify / gumbel_draft (shared-noise verification) -- pinned
    (tests/test_gumbel_oracle.py)
  * kseq_* / kseq_verify (K-SEQ multi-candidate verification: one position, and
    a batch of rows) -- pinned (tests/test_kseq_oracle.py)
  * spectr_round (one SpecTr round along the draft sequences' prefix tree) --
    pinned (tests/test_spectr_oracle.py)
  * philox4x32_10 -- pinned against PyTorch's independent header-only Philox
    engine on explicit counters and keys (tests/test_oracle_margins_philox.py).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "spec_verify_ref.c")
_LIB = os.path.join(_HERE, "libspec_verify_ref.so")

DTYPE_F32 = 0
DTYPE_BF16 = 1

ST_BAD_TEMPERATURE = 0x01
ST_BAD_TOP_K = 0x02
ST_BAD_TOP_P = 0x04
ST_BAD_NUM_DRAFT = 0x08
ST_BAD_DRAFT_TOKEN = 0x10
ST_NONFINITE = 0x20
ST_BAD_LENIENCE = 0x80


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libspec_verify_ref.so`` (gcc, -O2, fp64)."""
    hdr = os.path.join(_HERE, "spec_verify_ref.h")
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= max(os.path.getmtime(_SRC), os.path.getmtime(hdr))):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    # -ffp-contract=off: no fused multiply-adds, so every fp64 step rounds as written
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.svr_philox4x32_10.argtypes = [P, P, P]
        lib.svr_philox4x32_10.restype = None
        lib.svr_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
        lib.svr_uniform.restype = ctypes.c_double
        lib.svr_philox_uniforms.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int, P, P]
        lib.svr_philox_uniforms.restype = None
        lib.svr_normalise.argtypes = [P, ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_double, P, P]
        lib.svr_normalise.restype = ctypes.c_int
        common = [P, P, ctypes.c_int, P, P, P, P, P]
        outs = [P] * 11
        lib.svr_verify.argtypes = common + [P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int] + outs
        lib.svr_verify.restype = ctypes.c_int
        lib.svr_verify_seeded.argtypes = common + [ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_int] + outs
        lib.svr_verify_seeded.restype = ctypes.c_int
        lib.svr_verify_ex.argtypes = common + [P, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int] + outs
        lib.svr_verify_ex.restype = ctypes.c_int
        lib.svr_verify_ex_seeded.argtypes = common + [P, ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                                                      ctypes.c_int] + outs
        lib.svr_verify_ex_seeded.restype = ctypes.c_int
        lib.svr_gumbel_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]
        lib.svr_gumbel_uniform.restype = ctypes.c_double
        lib.svr_gumbel_verify.argtypes = [P, ctypes.c_int, P, P, P, P, P, ctypes.c_uint64, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, P, P, P, P, P]
        lib.svr_gumbel_verify.restype = ctypes.c_int
        lib.svr_gumbel_draft.argtypes = [P, ctypes.c_int, P, P, P, P, ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, P]
        lib.svr_gumbel_draft.restype = ctypes.c_int
        D, I = ctypes.c_double, ctypes.c_int
        lib.svr_kseq_beta.argtypes = [P, P, I, D]
        lib.svr_kseq_beta.restype = D
        lib.svr_kseq_rho.argtypes = [P, P, I, I]
        lib.svr_kseq_rho.restype = D
        lib.svr_kseq_direct.argtypes = [P, P, I, I, P, P]
        lib.svr_kseq_direct.restype = D
        lib.svr_kseq_step.argtypes = [P, P, I, I, P, P, D, P]
        lib.svr_kseq_step.restype = I
        lib.svr_kseq_verify.argtypes = [P, P, I, P, P, P, P, P, ctypes.c_uint64, I, I, I, P, P, P]
        lib.svr_kseq_verify.restype = I
        lib.svr_spectr_round.argtypes = [P, P, I, P, I, I, I, ctypes.c_float, I, ctypes.c_float, ctypes.c_uint64,
                                         ctypes.c_uint32, P]
        lib.svr_spectr_round.restype = I
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _load().svr_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, b: int, pos: int, draw: int) -> float:
    return _load().svr_uniform(seed, b, pos, draw)


def philox_uniforms(seed: int, B: int, G: int):
    ua = np.zeros((B, G), dtype=np.float64)
    ur = np.zeros((B, G + 1), dtype=np.float64)
    _load().svr_philox_uniforms(seed, B, G, _ptr(ua), _ptr(ur))
    return ua, ur


def normalise(logits, T: float, top_k: int = 0, top_p: float = 1.0, with_margin: bool = False):
    """One row of logits -> normalised probabilities (fp64)."""
    lg = np.ascontiguousarray(logits, dtype=np.float64)
    probs = np.zeros_like(lg)
    margin = np.zeros(1, dtype=np.float64)
    rc = _load().svr_normalise(_ptr(lg), lg.size, float(T), int(top_k), float(top_p), _ptr(probs), _ptr(margin))
    if rc != 0:
        raise ValueError("row has no finite maximum")
    return (probs, float(margin[0])) if with_margin else probs


@dataclass
class OracleResult:
    accepted_len: np.ndarray
    out_tokens: np.ndarray
    alpha: np.ndarray
    status: np.ndarray
    pos_accept: Optional[np.ndarray] = None
    pos_token: Optional[np.ndarray] = None
    accept_margin: Optional[np.ndarray] = None
    resid_margin: Optional[np.ndarray] = None
    filter_margin: Optional[np.ndarray] = None
    p_out: Optional[np.ndarray] = None
    q_out: Optional[np.ndarray] = None


def _as_logits(a: np.ndarray):
    """float32 -> (array, DTYPE_F32); bfloat16 carried as uint16 bit patterns -> DTYPE_BF16."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.float32:
        return a, DTYPE_F32
    if a.dtype == np.uint16:
        return a, DTYPE_BF16
    raise TypeError(f"logits must be float32 or bf16 bits in uint16, got {a.dtype}")


def verify(target, draft, draft_tokens, temperature, num_draft=None, top_k=None, top_p=None, *,
           seed: Optional[int] = None, u_accept=None, u_resid=None, all_positions: bool = False,
           probs: bool = False, lenience=None) -> OracleResult:
    """Run the oracle on one batch.

    ``target`` [B, G+1, V] and ``draft`` [B, G, V] are float32 arrays or bf16 bit
    patterns (uint16).  Either ``seed`` (Philox stream) or explicit ``u_accept``
    [B, G] / ``u_resid`` [B, G+1] uniforms must be given.  ``lenience`` [B]
    (None = 1 everywhere) scales q(x) in the acceptance test.
    """
    tgt, dt = _as_logits(target)
    drf, dt2 = _as_logits(draft)
    if dt != dt2:
        raise TypeError("target and draft dtypes differ")
    B, G1, V = tgt.shape
    G = G1 - 1
    if drf.shape != (B, G, V):
        raise ValueError("draft shape mismatch")
    xt = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, G)
    T = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    nd = None if num_draft is None else np.ascontiguousarray(num_draft, dtype=np.int32).reshape(B)
    tk = None if top_k is None else np.ascontiguousarray(top_k, dtype=np.int32).reshape(B)
    tpp = None if top_p is None else np.ascontiguousarray(top_p, dtype=np.float32).reshape(B)
    ln = None if lenience is None else np.ascontiguousarray(np.broadcast_to(lenience, (B,)), dtype=np.float32)

    acc = np.zeros(B, dtype=np.int32)
    out = np.zeros((B, G + 1), dtype=np.int32)
    alpha = np.zeros((B, G), dtype=np.float64)
    status = np.zeros(B, dtype=np.uint32)
    pa = pt = am = rm = fm = None
    if all_positions:
        pa = np.zeros((B, G), dtype=np.int32)
        pt = np.zeros((B, G + 1), dtype=np.int32)
        am = np.zeros((B, G), dtype=np.float64)
        rm = np.zeros((B, G + 1), dtype=np.float64)
        fm = np.zeros((B, 2 * G + 1), dtype=np.float64)
    po = qo = None
    if probs:
        po = np.zeros((B, G + 1, V), dtype=np.float64)
        qo = np.zeros((B, G, V), dtype=np.float64)
    outs = [_ptr(acc), _ptr(out), _ptr(alpha), _ptr(pa), _ptr(pt), _ptr(po), _ptr(qo), _ptr(status),
            _ptr(am), _ptr(rm), _ptr(fm)]
    lib = _load()
    if seed is not None:
        rc = lib.svr_verify_ex_seeded(_ptr(tgt), _ptr(drf), dt, _ptr(xt), _ptr(nd), _ptr(T), _ptr(tk), _ptr(tpp),
                                      _ptr(ln), int(seed), B, G, V, *outs)
    else:
        ua = np.ascontiguousarray(u_accept, dtype=np.float64).reshape(B, G)
        ur = np.ascontiguousarray(u_resid, dtype=np.float64).reshape(B, G + 1)
        rc = lib.svr_verify_ex(_ptr(tgt), _ptr(drf), dt, _ptr(xt), _ptr(nd), _ptr(T), _ptr(tk), _ptr(tpp),
                               _ptr(ln), _ptr(ua), _ptr(ur), B, G, V, *outs)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return OracleResult(acc, out, alpha, status, pa, pt, am, rm, fm, po, qo)


# ---------------------------------------------------------------------------
# Gumbel-coupled (shared-noise) verification
# ---------------------------------------------------------------------------

@dataclass
class GumbelResult:
    accepted_len: np.ndarray   # [B] int32
    out_tokens: np.ndarray     # [B, G+1] int32: draft_1..draft_n, t_{n+1}, then -1
    target_tokens: np.ndarray  # [B, G+1] int32: the target's own token t_k at every k <= gamma_b + 1
    margin: np.ndarray         # [B, G+1] float64: best minus second-best score at each position
    status: np.ndarray         # [B] uint32


def gumbel_uniform(seed: int, b: int, pos: int, token: int) -> float:
    return _load().svr_gumbel_uniform(seed, b, pos, token)


def _gumbel_params(B, temperature, num_draft, top_k, top_p):
    T = np.ascontiguousarray(temperature, dtype=np.float32).reshape(B)
    nd = None if num_draft is None else np.ascontiguousarray(num_draft, dtype=np.int32).reshape(B)
    tk = None if top_k is None else np.ascontiguousarray(top_k, dtype=np.int32).reshape(B)
    tpp = None if top_p is None else np.ascontiguousarray(top_p, dtype=np.float32).reshape(B)
    return T, nd, tk, tpp


def gumbel_verify(target, draft_tokens, temperature, num_draft=None, top_k=None, top_p=None, *,
                  seed: int) -> GumbelResult:
    """Shared-noise verification of one batch: target [B, G+1, V] logits (float32 or
    bf16 bit patterns), the drafter's tokens [B, G]."""
    tgt, dt = _as_logits(target)
    B, G1, V = tgt.shape
    G = G1 - 1
    xt = np.ascontiguousarray(draft_tokens, dtype=np.int32).reshape(B, G)
    T, nd, tk, tpp = _gumbel_params(B, temperature, num_draft, top_k, top_p)
    acc = np.zeros(B, dtype=np.int32)
    out = np.zeros((B, G + 1), dtype=np.int32)
    tt = np.zeros((B, G + 1), dtype=np.int32)
    mg = np.zeros((B, G + 1), dtype=np.float64)
    st = np.zeros(B, dtype=np.uint32)
    rc = _load().svr_gumbel_verify(_ptr(tgt), dt, _ptr(xt), _ptr(nd), _ptr(T), _ptr(tk), _ptr(tpp), int(seed), B,
                                   G, V, _ptr(acc), _ptr(out), _ptr(tt), _ptr(mg), _ptr(st))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return GumbelResult(acc, out, tt, mg, st)


def gumbel_draft(draft, temperature, num_draft=None, top_k=None, top_p=None, *, seed: int) -> np.ndarray:
    """The coupled drafter's tokens [B, G] for draft logits [B, G, V] and the same noise."""
    drf, dt = _as_logits(draft)
    B, G, V = drf.shape
    T, nd, tk, tpp = _gumbel_params(B, temperature, num_draft, top_k, top_p)
    x = np.zeros((B, G), dtype=np.int32)
    rc = _load().svr_gumbel_draft(_ptr(drf), dt, _ptr(nd), _ptr(T), _ptr(tk), _ptr(tpp), int(seed), B, G, V, _ptr(x))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return x


# ---------------------------------------------------------------------------
# K-SEQ multi-candidate verification (one position; p = target, q = draft)
# ---------------------------------------------------------------------------

def _prob_row(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def kseq_beta(p, q, rho: float) -> float:
    p, q = _prob_row(p), _prob_row(q)
    return _load().svr_kseq_beta(_ptr(p), _ptr(q), p.size, float(rho))


def kseq_rho(p, q, k: int) -> float:
    p, q = _prob_row(p), _prob_row(q)
    return _load().svr_kseq_rho(_ptr(p), _ptr(q), p.size, int(k))


def kseq_direct(p, q, k: int):
    """(A_rho*[V], P_A, rho*): the direct acceptance mass of each token."""
    p, q = _prob_row(p), _prob_row(q)
    A = np.zeros(p.size)
    rho = np.zeros(1)
    pa = _load().svr_kseq_direct(_ptr(p), _ptr(q), p.size, int(k), _ptr(A), _ptr(rho))
    return A, pa, float(rho[0])


def kseq_step(p, q, cand, u, u_res: float):
    """(emitted token, index of the accepted candidate or -1)."""
    p, q = _prob_row(p), _prob_row(q)
    c = np.ascontiguousarray(cand, dtype=np.int32)
    uu = np.ascontiguousarray(u, dtype=np.float64)
    idx = np.zeros(1, dtype=np.int32)
    tok = _load().svr_kseq_step(_ptr(p), _ptr(q), p.size, c.size, _ptr(c), _ptr(uu), float(u_res), _ptr(idx))
    return int(tok), int(idx[0])


def kseq_verify(target, draft, cand, temperature, num_cand=None, top_k=None, top_p=None, *, seed: int):
    """Batched K-SEQ at one position per row: target / draft logits [B, V] (float32 or
    bf16 bits), candidates [B, K].  Returns (out_token [B], accepted [B], status [B])."""
    tgt, dt = _as_logits(target)
    drf, dt2 = _as_logits(draft)
    if dt != dt2 or tgt.shape != drf.shape or tgt.ndim != 2:
        raise ValueError("target and draft must be [B, V] of one dtype")
    B, V = tgt.shape
    c = np.ascontiguousarray(cand, dtype=np.int32)
    K = c.shape[1]
    T, nc, tk, tpp = _gumbel_params(B, temperature, num_cand, top_k, top_p)
    tok = np.zeros(B, dtype=np.int32)
    acc = np.zeros(B, dtype=np.int32)
    st = np.zeros(B, dtype=np.uint32)
    rc = _load().svr_kseq_verify(_ptr(tgt), _ptr(drf), dt, _ptr(c), _ptr(nc), _ptr(T), _ptr(tk), _ptr(tpp),
                                 int(seed), B, K, V, _ptr(tok), _ptr(acc), _ptr(st))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (rc={rc})")
    return tok, acc, st


def spectr_round(target, draft, tok, temperature: float = 1.0, top_k: int = 0, top_p: float = 1.0, *, seed: int,
                 b: int = 0) -> np.ndarray:
    """One SpecTr round: target [K, L+1, V], draft [K, L, V] logits, draft sequences tok [K, L].
    Returns the emitted tokens (1..L+1 of them)."""
    tgt, dt = _as_logits(target)
    drf, dt2 = _as_logits(draft)
    K, L1, V = tgt.shape
    L = L1 - 1
    if dt != dt2 or drf.shape != (K, L, V):
        raise ValueError("target [K, L+1, V] and draft [K, L, V] of one dtype")
    t = np.ascontiguousarray(tok, dtype=np.int32).reshape(K, L)
    out = np.zeros(L + 1, dtype=np.int32)
    n = _load().svr_spectr_round(_ptr(tgt), _ptr(drf), dt, _ptr(t), K, L, V, float(temperature), int(top_k),
                                 float(top_p), int(seed), int(b), _ptr(out))
    if n < 0:
        raise ValueError("bad row")
    return out[:n]
