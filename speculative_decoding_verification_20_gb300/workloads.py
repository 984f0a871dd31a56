"""Seeded synthetic workloads shaped like the pages' decode rounds.

This module only *makes inputs*: logits for the target and the drafter, the
drafter's proposed tokens and the per-sequence sampling parameters.  It holds
none of the verification arithmetic (no normalisation, acceptance, residual
or alpha) and is the one module shared by the CUDA-path tests, the oracle-side
tests and the benchmark.

Recipes (sizes and distributions follow the workloads described for the
method: batches of decode rounds, gamma = 3..8, 1k..152k vocabularies, draft
logits = target logits + Gaussian noise):

  tiny      B=1,    G=4, V=1000,   fp32, T=1,   target N(0, 2^2), draft noise 0.5
  v32k      B=64,   G=5, V=32000,  bf16, T=0.8, target N(0, 3^2) + 8 on 20 random ids,
                                                 draft noise 1.0  (``greedy=True``: T=0)
  v128k     B=256,  G=7, V=128256, bf16, T=1,   top-k 50 then top-p 0.9,
                                                 target -1.1*log(rank) over a random
                                                 permutation + N(0, 0.3^2), draft noise 0.8
  ragged    B=32,   G=1..8 per row, V=151936, fp32, T in {0,.3,.7,1,1.2}, top-p U[.8,1],
                                                 draft noise sigma_b ~ U[0.2, 2.0];
                                                 target as v128k (Zipf-like)
  b1024     B=1024, G=3, V=32000,  bf16, T=1,   target as v32k, draft noise 1.5

The drafter's proposal x_i is sampled from the drafter's own filtered
distribution, the way the drafter would sample it: Gumbel-max over its
temperature-scaled logits (argmax at T=0), restricted to the kept set of the
row's top-k and then top-p (the smallest prefix of the drafter's tokens by
probability, ties to the lower id, whose mass reaches top-p).  This is input
generation only (it stands in for the draft model's sampler); the
verification arithmetic lives in the library and, independently, in the oracle.
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional

import numpy as np
import torch

CONFIGS = {
    "tiny": dict(B=1, G=4, V=1000, dtype="f32"),
    "v32k": dict(B=64, G=5, V=32000, dtype="bf16"),
    "v128k": dict(B=256, G=7, V=128256, dtype="bf16"),
    "ragged": dict(B=32, G=8, V=151936, dtype="f32"),
    "b1024": dict(B=1024, G=3, V=32000, dtype="bf16"),
}


@dataclass
class Workload:
    name: str
    B: int
    G: int
    V: int
    dtype: str  # "f32" | "bf16"
    target: torch.Tensor  # [B, G+1, V]
    draft: torch.Tensor  # [B, G, V]
    draft_tokens: torch.Tensor  # int32 [B, G]
    num_draft: Optional[torch.Tensor]  # int32 [B] or None (all G)
    temperature: torch.Tensor  # float32 [B]
    top_k: Optional[torch.Tensor]  # int32 [B] or None
    top_p: Optional[torch.Tensor]  # float32 [B] or None
    seed: int  # verification seed (Philox key)

    def to(self, device) -> "Workload":
        f = lambda t: None if t is None else t.to(device)
        return replace(self, target=f(self.target), draft=f(self.draft), draft_tokens=f(self.draft_tokens),
                       num_draft=f(self.num_draft), temperature=f(self.temperature), top_k=f(self.top_k),
                       top_p=f(self.top_p))

    def gammas(self) -> np.ndarray:
        if self.num_draft is None:
            return np.full(self.B, self.G, dtype=np.int64)
        return self.num_draft.cpu().numpy().astype(np.int64)

    def positions(self) -> int:
        """Verified draft positions in one call: sum_b gamma_b."""
        return int(self.gammas().sum())

    def logit_bytes(self) -> int:
        """Algorithmic bytes: every logit of every row in use read once, sum_b (2 gamma_b + 1) V size."""
        es = 2 if self.dtype == "bf16" else 4
        return int(((2 * self.gammas() + 1) * self.V * es).sum())

    def subset(self, rows) -> "Workload":
        idx = torch.as_tensor(np.asarray(rows), dtype=torch.long, device=self.target.device)
        f = lambda t: None if t is None else t.index_select(0, idx.to(t.device))
        return replace(self, B=len(idx), target=f(self.target), draft=f(self.draft),
                       draft_tokens=f(self.draft_tokens), num_draft=f(self.num_draft),
                       temperature=f(self.temperature), top_k=f(self.top_k), top_p=f(self.top_p))

    def numpy_inputs(self) -> dict:
        """CPU numpy copies: float32 logits, or bf16 bit patterns as uint16."""
        def logits(t):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16)
            return t.numpy()
        g = lambda t: None if t is None else t.detach().cpu().numpy()
        return dict(target=logits(self.target), draft=logits(self.draft), draft_tokens=g(self.draft_tokens),
                    num_draft=g(self.num_draft), temperature=g(self.temperature), top_k=g(self.top_k),
                    top_p=g(self.top_p))


def _gen(seed: int, salt: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + salt) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def _zipf_logits(rows: int, V: int, g: torch.Generator, device) -> torch.Tensor:
    # rank of each token id: a uniformly random permutation of 1..V per row
    ranks = torch.rand(rows, V, generator=g, device=device).argsort(dim=1).to(torch.float32) + 1.0
    noise = torch.randn(rows, V, generator=g, device=device) * 0.3
    return -1.1 * torch.log(ranks) + noise


def _boosted_normal(rows: int, V: int, g: torch.Generator, device) -> torch.Tensor:
    t = torch.randn(rows, V, generator=g, device=device) * 3.0
    boost_ids = torch.rand(rows, V, generator=g, device=device).topk(20, dim=1).indices
    t.scatter_add_(1, boost_ids, torch.full(boost_ids.shape, 8.0, device=device))
    return t


def _propose(draft: torch.Tensor, T: torch.Tensor, top_k: Optional[torch.Tensor], top_p: Optional[torch.Tensor],
             g: torch.Generator) -> torch.Tensor:
    """The drafter's own proposal per row: Gumbel-max on logits / T over the row's
    top-k-then-top-p kept set; argmax at T = 0."""
    B, G, V = draft.shape
    d = draft.to(torch.float32)
    u = torch.rand(d.shape, generator=g, device=d.device).clamp_(1e-12, 1.0 - 1e-7)
    gumbel = -torch.log(-torch.log(u))
    Tb = T.view(B, 1, 1).to(torch.float32)
    z = torch.where(Tb > 0, d / Tb.clamp_min(1e-30), d)
    if top_k is not None or top_p is not None:
        zs, order = torch.sort(z, dim=2, descending=True, stable=True)  # ties: lower id first
        rank = torch.arange(V, device=d.device).view(1, 1, V)
        keep = torch.ones_like(zs, dtype=torch.bool)
        if top_k is not None:
            k = top_k.view(B, 1, 1).to(torch.long)
            keep &= (k <= 0) | (k >= V) | (rank < k)
        if top_p is not None:
            w = torch.where(keep, torch.exp(zs - zs[:, :, :1]), torch.zeros_like(zs))
            w = w / w.sum(dim=2, keepdim=True)
            before = torch.cumsum(w.to(torch.float64), dim=2) - w.to(torch.float64)  # mass ahead of each token
            keep &= before < top_p.view(B, 1, 1).to(torch.float64)
        mask = torch.zeros_like(keep).scatter_(2, order, keep)
        z = torch.where(mask, z, torch.full_like(z, float("-inf")))
    score = torch.where(Tb > 0, z + gumbel, z)
    return score.argmax(dim=2).to(torch.int32)


def make(name: str, seed: int = 0, device="cpu", *, B: Optional[int] = None, G: Optional[int] = None,
         V: Optional[int] = None, greedy: bool = False, verify_seed: Optional[int] = None) -> Workload:
    """Build one workload.  ``B``/``G``/``V`` shrink a recipe for quick tests."""
    cfg = dict(CONFIGS[name])
    B = cfg["B"] if B is None else B
    G = cfg["G"] if G is None else G
    V = cfg["V"] if V is None else V
    dtype = cfg["dtype"]
    device = torch.device(device)
    g = _gen(seed, sum(map(ord, name)), device)

    num_draft = None
    top_k = top_p = None
    if name == "tiny":
        target = torch.randn(B, G + 1, V, generator=g, device=device) * 2.0
        sigma = torch.full((B,), 0.5, device=device)
        T = torch.ones(B, device=device)
    elif name in ("v32k", "b1024"):
        target = _boosted_normal(B * (G + 1), V, g, device).view(B, G + 1, V)
        sigma = torch.full((B,), 1.0 if name == "v32k" else 1.5, device=device)
        T = torch.full((B,), 0.8 if name == "v32k" else 1.0, device=device)
    elif name == "v128k":
        target = _zipf_logits(B * (G + 1), V, g, device).view(B, G + 1, V)
        sigma = torch.full((B,), 0.8, device=device)
        T = torch.ones(B, device=device)
        top_k = torch.full((B,), 50, dtype=torch.int32, device=device)
        top_p = torch.full((B,), 0.9, dtype=torch.float32, device=device)
    elif name == "ragged":
        target = _zipf_logits(B * (G + 1), V, g, device).view(B, G + 1, V)
        sigma = 0.2 + 1.8 * torch.rand(B, generator=g, device=device)
        choices = torch.tensor([0.0, 0.3, 0.7, 1.0, 1.2], device=device)
        T = choices[torch.randint(0, 5, (B,), generator=g, device=device)]
        top_p = (0.8 + 0.2 * torch.rand(B, generator=g, device=device)).to(torch.float32)
        num_draft = torch.randint(1, G + 1, (B,), generator=g, device=device).to(torch.int32)
    else:
        raise KeyError(name)
    if greedy:
        T = torch.zeros(B, device=device)

    draft = target[:, :G, :] + torch.randn(B, G, V, generator=g, device=device) * sigma.view(B, 1, 1)
    if dtype == "bf16":
        target = target.to(torch.bfloat16)
        draft = draft.to(torch.bfloat16)
    else:
        target = target.contiguous()
        draft = draft.contiguous()
    T = T.to(torch.float32)
    tokens = _propose(draft, T, top_k, top_p, g)
    if num_draft is not None:  # padding positions past gamma_b are never read; keep them valid anyway
        pos = torch.arange(G, device=device).view(1, G)
        tokens = torch.where(pos < num_draft.view(B, 1).to(torch.long), tokens, torch.zeros_like(tokens))
    return Workload(name=name + ("-greedy" if greedy else ""), B=B, G=G, V=V, dtype=dtype, target=target.contiguous(),
                    draft=draft.contiguous(), draft_tokens=tokens.contiguous(), num_draft=num_draft,
                    temperature=T.contiguous(), top_k=top_k, top_p=top_p,
                    seed=int(seed if verify_seed is None else verify_seed))


# ---------------------------------------------------------------------------
# K-SEQ (several candidates at one position per row)
# ---------------------------------------------------------------------------
KSEQ_CONFIGS = {
    # one decode position per row, k candidates drawn independently from the drafter
    "kseq32k": dict(B=256, K=4, V=32000, dtype="bf16"),   # v32k's rows, T = 0.8, no filter
    "kseq128k": dict(B=64, K=8, V=128256, dtype="bf16"),  # v128k's rows, T = 1, top-k 50, top-p 0.9
}


@dataclass
class KseqWorkload:
    name: str
    B: int
    K: int
    V: int
    dtype: str
    target: torch.Tensor        # [B, V]
    draft: torch.Tensor         # [B, V]
    candidates: torch.Tensor    # int32 [B, K]: i.i.d. draws from the drafter's filtered q
    num_candidates: Optional[torch.Tensor]  # int32 [B] or None (all K)
    temperature: torch.Tensor
    top_k: Optional[torch.Tensor]
    top_p: Optional[torch.Tensor]
    seed: int

    def numpy_inputs(self) -> dict:
        def logits(t):
            t = t.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                return t.view(torch.int16).numpy().view(np.uint16)
            return t.numpy()
        g = lambda t: None if t is None else t.detach().cpu().numpy()
        return dict(target=logits(self.target), draft=logits(self.draft), candidates=g(self.candidates),
                    num_candidates=g(self.num_candidates), temperature=g(self.temperature), top_k=g(self.top_k),
                    top_p=g(self.top_p))

    def positions(self) -> int:
        """Verified positions per call: one per row."""
        return self.B

    def logit_bytes(self) -> int:
        return 2 * self.B * self.V * (2 if self.dtype == "bf16" else 4)


def make_kseq(name: str, seed: int = 0, device="cpu", *, B: Optional[int] = None, K: Optional[int] = None,
              V: Optional[int] = None) -> KseqWorkload:
    """A K-SEQ batch: the target and draft rows of one position per row (the v32k or
    v128k recipe) and K candidates per row, each an independent draw of the drafter."""
    cfg = dict(KSEQ_CONFIGS[name])
    B = cfg["B"] if B is None else B
    K = cfg["K"] if K is None else K
    V = cfg["V"] if V is None else V
    device = torch.device(device)
    g = _gen(seed, sum(map(ord, name)), device)
    top_k = top_p = None
    if name == "kseq32k":
        target = _boosted_normal(B, V, g, device)
        sigma, T = 1.0, torch.full((B,), 0.8, device=device)
    else:
        target = _zipf_logits(B, V, g, device)
        sigma, T = 0.8, torch.ones(B, device=device)
        top_k = torch.full((B,), 50, dtype=torch.int32, device=device)
        top_p = torch.full((B,), 0.9, dtype=torch.float32, device=device)
    draft = target + torch.randn(B, V, generator=g, device=device) * sigma
    if cfg["dtype"] == "bf16":
        target, draft = target.to(torch.bfloat16), draft.to(torch.bfloat16)
    T = T.to(torch.float32)
    # K independent proposals of the drafter: its row repeated K times, fresh noise each
    cand = _propose(draft.unsqueeze(1).expand(B, K, V), T, top_k, top_p, g)
    return KseqWorkload(name, B, K, V, cfg["dtype"], target.contiguous(), draft.contiguous(), cand.contiguous(), None,
                        T.contiguous(), top_k, top_p, int(seed))
