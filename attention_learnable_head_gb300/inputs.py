"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws random numbers and packs them into the layouts the
library takes; it holds none of the attention arithmetic.  Every tensor is
created on the CPU with its own ``torch.Generator`` and cast to bf16 before it
is copied anywhere, so the CUDA path and the oracle read the same bytes.

Seeding: tensor t of workload c uses seed ``1000 * c + t`` with t = 0 (q),
1 (k), 2 (v), 3 (dout), 4 (sink), 5 (varlen lengths), 6 (sink permutation).

Workloads (GPT-OSS attention shapes; head_dim 64, H_q = 64, H_kv = 8 for the
large ones):
  1 tiny           B=1, H 2/2, N=128, causal
  2 gptoss_full    B=1, H 64/8, N=4096, causal
  3 swa            B=1, H 64/8, N=16384, causal, window 128
  4 varlen         packed lengths ~ U[512, 16384] up to 65536 tokens, causal,
                   sink[h] drawn from {-30, -2, 0, 2, 8}
  5 long_full      B=4, H 64/8, N=16384, causal, q scaled by 3, sink ~ N(0, 2^2)
  5 long_window    same inputs, window 128
  long_full_1seq / long_window_1seq: their first sequence alone (profiling)
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
import math

import torch

SINK_CHOICES = (-30.0, -2.0, 0.0, 2.0, 8.0)


@dataclass(frozen=True)
class Workload:
    name: str
    seed_index: int
    heads_q: int
    heads_kv: int
    head_dim: int = 64
    batch: int = 1
    seqlen: int = 0                 # dense N_q = N_k (ignored when lengths/varlen)
    lengths: tuple = ()             # explicit packed lengths (varlen)
    varlen_total: int = 0           # draw lengths until this many tokens
    varlen_range: tuple = (512, 16384)
    causal: bool = True
    window: int = 0
    q_mult: float = 1.0
    sink_kind: str = "normal"       # normal | choice | neginf | const
    sink_sigma: float = 1.0
    sink_const: float = 0.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def is_varlen(self) -> bool:
        return bool(self.lengths) or self.varlen_total > 0


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 2, batch=1, seqlen=128),
    "gptoss_full": Workload("gptoss_full", 2, 64, 8, batch=1, seqlen=4096),
    "swa": Workload("swa", 3, 64, 8, batch=1, seqlen=16384, window=128),
    "varlen": Workload("varlen", 4, 64, 8, varlen_total=65536, sink_kind="choice"),
    "long_full": Workload("long_full", 5, 64, 8, batch=4, seqlen=16384, q_mult=3.0,
                          sink_sigma=2.0),
    "long_window": Workload("long_window", 5, 64, 8, batch=4, seqlen=16384, window=128,
                            q_mult=3.0, sink_sigma=2.0),
    # the first sequence of long_full alone (the same seeds, so the same first
    # 16384 tokens): a profiler capture of one sequence stays a few GB
    "long_full_1seq": Workload("long_full_1seq", 5, 64, 8, batch=1, seqlen=16384, q_mult=3.0,
                               sink_sigma=2.0),
    "long_window_1seq": Workload("long_window_1seq", 5, 64, 8, batch=1, seqlen=16384,
                                 window=128, q_mult=3.0, sink_sigma=2.0),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def draw_lengths(w: Workload) -> list[int]:
    """Packed sequence lengths: explicit ones, dense B x N, or drawn uniformly."""
    if w.lengths:
        return [int(x) for x in w.lengths]
    if w.varlen_total <= 0:
        return [w.seqlen] * w.batch
    g = _gen(1000 * w.seed_index + 5)
    lo, hi = w.varlen_range
    lengths, total = [], 0
    while True:
        n = int(torch.randint(lo, hi + 1, (1,), generator=g))
        if total + n > w.varlen_total:
            break
        lengths.append(n)
        total += n
    return lengths


def cu_from_lengths(lengths) -> list[int]:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return cu


@dataclass
class Case:
    """One seeded problem: CPU tensors plus its shape parameters."""
    workload: Workload
    q: torch.Tensor           # [T, H_q, d] bf16
    k: torch.Tensor           # [T, H_kv, d] bf16
    v: torch.Tensor           # [T, H_kv, d] bf16
    dout: torch.Tensor        # [T, H_q, d] bf16
    sink: torch.Tensor        # [H_q] fp32
    lengths: list = field(default_factory=list)

    @property
    def cu_seqlens(self) -> list[int]:
        return cu_from_lengths(self.lengths)

    @property
    def total(self) -> int:
        return sum(self.lengths)


def make_case(w: Workload, with_dout: bool = True) -> Case:
    lengths = draw_lengths(w)
    t = sum(lengths)
    s = 1000 * w.seed_index
    q = torch.randn((t, w.heads_q, w.head_dim), generator=_gen(s + 0))
    if w.q_mult != 1.0:
        q = q * w.q_mult
    q = q.to(torch.bfloat16)
    k = torch.randn((t, w.heads_kv, w.head_dim), generator=_gen(s + 1)).to(torch.bfloat16)
    v = torch.randn((t, w.heads_kv, w.head_dim), generator=_gen(s + 2)).to(torch.bfloat16)
    if with_dout:
        dout = torch.randn((t, w.heads_q, w.head_dim), generator=_gen(s + 3)).to(torch.bfloat16)
    else:
        dout = torch.empty(0, dtype=torch.bfloat16)
    if w.sink_kind == "normal":
        sink = torch.randn((w.heads_q,), generator=_gen(s + 4)) * w.sink_sigma
    elif w.sink_kind == "choice":
        perm = torch.randperm(w.heads_q, generator=_gen(s + 6))
        sink = torch.tensor([SINK_CHOICES[int(perm[h]) % len(SINK_CHOICES)]
                             for h in range(w.heads_q)])
    elif w.sink_kind == "neginf":
        sink = torch.full((w.heads_q,), -math.inf)
    elif w.sink_kind == "const":
        sink = torch.full((w.heads_q,), float(w.sink_const))
    else:
        raise ValueError(w.sink_kind)
    return Case(w, q, k, v, dout, sink.to(torch.float32), lengths)


def small_workload(name: str, seed_index: int, heads_q: int, heads_kv: int,
                   lengths, head_dim: int = 64, causal: bool = True, window: int = 0,
                   **kw) -> Workload:
    """A small packed case for parity tests (ragged lengths, odd windows)."""
    return Workload(name, seed_index, heads_q, heads_kv, head_dim=head_dim,
                    lengths=tuple(int(x) for x in lengths), causal=causal,
                    window=window, **kw)


def with_(w: Workload, **kw) -> Workload:
    return replace(w, **kw)
