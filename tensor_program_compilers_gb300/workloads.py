"""Seeded synthetic inputs for the attention forward.

This module holds only shapes and random-number recipes: no attention
arithmetic.  Both the CUDA path's tests/benchmark and the fp64 oracle are fed
from it, so the two sides always see the same bf16 bytes.

Recipe (all on the CPU, ``torch.Generator('cpu').manual_seed(seed)``):
  1. packed batches only: the sequence lengths, ``randint(lo, hi + 1)``;
  2. Q, K, V in that order, each ``randn`` in fp32, multiplied by its scale
     (1 unless stated), then rounded to bf16;
  3. row samples (for the oracle on the long case) come from a second
     generator seeded ``seed + 1``: per head, ``randperm(N)[:rows_per_head]``.

Layouts: fixed batch Q/O [B, N, Hq, d], K/V [B, N, Hkv, d]; packed
Q/O [T, Hq, d], K/V [T, Hkv, d] with ``cu_seqlens`` = [0, L0, L0+L1, ...].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int            # batch, or number of packed sequences
    Hq: int
    Hkv: int
    N: int            # sequence length (fixed batch); unused when packed
    d: int
    causal: bool
    q_scale: float = 1.0
    # packed variable-length batches: lengths ~ Uniform[len_lo, len_hi]
    varlen: bool = False
    len_lo: int = 0
    len_hi: int = 0
    # number of query rows per head the oracle checks (None = all rows)
    oracle_rows_per_head: Optional[int] = None
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# The five workloads the attention forward is measured and checked on.
TINY = Workload("tiny-mha B1 H2 N128 d64 noncausal", B=1, Hq=2, Hkv=2, N=128, d=64,
                causal=False, seed=1000)
BLOCK = Workload("block B4 H16 N512 d64 causal", B=4, Hq=16, Hkv=16, N=512, d=64,
                 causal=True, seed=1001)
GQA_PREFILL = Workload("gqa-prefill B2 Hq32 Hkv8 N4096 d128 causal", B=2, Hq=32, Hkv=8,
                       N=4096, d=128, causal=True, seed=1002)
LONG_D256 = Workload("long-d256 B1 Hq16 Hkv2 N16384 d256 causal", B=1, Hq=16, Hkv=2,
                     N=16384, d=256, causal=True, oracle_rows_per_head=512, seed=1003)
RAGGED = Workload("ragged 16 seqs L~U[256,8192] Hq32 Hkv8 d128 causal Qx4", B=16, Hq=32,
                  Hkv=8, N=0, d=128, causal=True, q_scale=4.0, varlen=True, len_lo=256,
                  len_hi=8192, seed=1004)

WORKLOADS = [TINY, BLOCK, GQA_PREFILL, LONG_D256, RAGGED]
BY_KEY = {"tiny": TINY, "block": BLOCK, "gqa": GQA_PREFILL, "d256": LONG_D256,
          "ragged": RAGGED}


@dataclass
class Inputs:
    wl: Workload
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    cu_seqlens: Optional[torch.Tensor]   # int32 [B+1] (CPU) or None
    lens: list = field(default_factory=list)

    @property
    def total_rows(self) -> int:
        return self.q.shape[0] if self.wl.varlen else self.wl.B * self.wl.N

    @property
    def n_arg(self) -> int:
        """The N argument of attn_fwd: tokens per sequence, or all tokens when packed."""
        return self.total_rows if self.wl.varlen else self.wl.N


def seq_lengths(wl: Workload, gen: torch.Generator) -> list:
    return torch.randint(wl.len_lo, wl.len_hi + 1, (wl.B,), generator=gen).tolist()


def make_inputs(wl: Workload, seed: Optional[int] = None) -> Inputs:
    seed = wl.seed if seed is None else seed
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    if wl.varlen:
        lens = seq_lengths(wl, g)
        T = sum(lens)
        cu = torch.zeros(wl.B + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
        qshape, kshape = (T, wl.Hq, wl.d), (T, wl.Hkv, wl.d)
    else:
        lens = [wl.N] * wl.B
        cu = None
        qshape, kshape = (wl.B, wl.N, wl.Hq, wl.d), (wl.B, wl.N, wl.Hkv, wl.d)
    q = _randn_bf16(qshape, g, wl.q_scale)
    k = _randn_bf16(kshape, g, 1.0)
    v = _randn_bf16(kshape, g, 1.0)
    return Inputs(wl, q, k, v, cu, lens)


def _randn_bf16(shape, g, mult):
    x = torch.randn(shape, generator=g, dtype=torch.float32)
    if mult != 1.0:
        x.mul_(mult)
    return x.to(torch.bfloat16)


def sample_rows(wl: Workload, lens: list, rows_per_head: int, seed: Optional[int] = None,
                heads=None):
    """(seq, h, i) triples for the oracle: rows_per_head distinct rows per head,
    spread over the sequences in proportion to their lengths."""
    seed = (wl.seed if seed is None else seed) + 1
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    total = sum(lens)
    starts = [0]
    for L in lens:
        starts.append(starts[-1] + L)
    out = []
    for h in (range(wl.Hq) if heads is None else heads):
        n = min(rows_per_head, total)
        flat = torch.randperm(total, generator=g)[:n].tolist()
        for r in flat:
            # the sequence holding flat row r
            s = 0
            while starts[s + 1] <= r:
                s += 1
            out.append((s, h, r - starts[s]))
    return out


def causal_flops(wl: Workload, lens: list) -> float:
    """Attention forward FLOPs under the convention 4*H*L^2*d per sequence,
    halved when causal."""
    f = sum(4.0 * wl.Hq * L * L * wl.d for L in lens)
    return f / 2 if wl.causal else f


def with_(wl: Workload, **kw) -> Workload:
    return replace(wl, **kw)
