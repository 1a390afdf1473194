"""CPU float64 oracle of attention over key chunks and the sink-aware merge.

TEST INFRASTRUCTURE ONLY -- never imported by the product path.

Where this comes from
--------------------
Sequence parallelism that stays compatible with sinks is named on the pages but
not spelled out: page "Treinamento de RL Agêntico para modelos GPT-OSS"
(ai-engineering-academy-news), section "O QUE MUDA NA PRÁTICA PARA ENGENHEIROS
DE IA" (under "Custos"), credits sequence parallelism with training longer
contexts without running out of memory, and the keryc.com page on GPT-OSS
agentic RL fixes, section "Solutions implemented by the team", integrates
sequence parallelism compatible with attention sinks and FlashAttention v3 for
16k-token responses and 8k-token prompts.  The plainest reading, taken here:
keys are split into chunks; each
chunk yields the softmax-attention result and log-sum-exp of the queries over
that chunk alone, with no sink; the chunks are merged into the full result
with the sink entering the normaliser exactly once.  Over the widened row
[S_chunk_1 | ... | S_chunk_C | sink] of the concat listing "带汇聚的注意力（GPT-OSS）"
(euno.news page), with Z = sum_c exp(LSE_c) + exp(sink):

    P_ij = exp(S_ij) / Z      O_i = sum_c exp(LSE_c - log Z) O_c,i
    LSE_i = log Z

where O_c,i = sum_{j in c} exp(S_ij - LSE_c,i) v_j.  A chunk in which row i
sees no key has O_c,i = 0 and LSE_c,i = -inf and drops out.

Positions: query row i (local to its sequence) sees chunk key j (local to the
chunk) iff j <= i + q_pos0 (causal) and, with a window W > 0, also
j > i + q_pos0 - W.  For a full, unchunked key range q_pos0 = N_k - N_q (the
bottom-right alignment of the main oracle); the chunk starting at key k0 of
that range has q_pos0 = N_k - N_q - k0.
"""
from __future__ import annotations

import math
from typing import Sequence

import torch

from .attention_sink import F64, sequence_bounds, sink_softmax


def visible_mask_at(n_rows: int, n_cols: int, q_pos0: int, causal: bool,
                    window: int) -> torch.Tensor:
    """[n_rows, n_cols] bool: row i sees column j (positions as above)."""
    i = torch.arange(n_rows).unsqueeze(1)
    j = torch.arange(n_cols).unsqueeze(0)
    vis = torch.ones(n_rows, n_cols, dtype=torch.bool)
    if causal:
        diag = i + q_pos0
        vis &= j <= diag
        if window > 0:
            vis &= j > diag - window
    return vis


def oracle_fwd_chunk(q, k, v, *, scale: float, causal: bool, window: int, q_pos0: int,
                     cu_seqlens_q: Sequence[int], cu_seqlens_k: Sequence[int]):
    """Attention of every query over one key chunk, without the sink.

    q [T_q, H_q, d]; k, v [T_k, H_kv, d] hold the chunk's keys of every
    sequence (packed by cu_seqlens_k).  Returns out [T_q, H_q, d] and lse
    [H_q, T_q] in float64; rows that see no key of the chunk get out = 0 and
    lse = -inf (the softmax of the row with a sink of -inf).
    """
    if window > 0 and not causal:
        raise ValueError("a sliding window requires causal masking")
    qd, kd, vd = q.to(F64), k.to(F64), v.to(F64)
    t_q, h_q, d = qd.shape
    h_kv = kd.shape[1]
    group = h_q // h_kv
    out = torch.zeros((t_q, h_q, vd.shape[2]), dtype=F64)
    lse = torch.full((h_q, t_q), -math.inf, dtype=F64)
    for (qs, qe), (ks, ke) in zip(sequence_bounds(cu_seqlens_q), sequence_bounds(cu_seqlens_k)):
        n_q, n_k = qe - qs, ke - ks
        if n_q == 0 or n_k == 0:
            continue
        vis = visible_mask_at(n_q, n_k, q_pos0, causal, window)
        for h in range(h_q):
            g = h // group
            scores = scale * (qd[qs:qe, h] @ kd[ks:ke, g].T)
            scores = scores.masked_fill(~vis, -math.inf)
            p, _, lse_rows = sink_softmax(scores, -math.inf)   # no sink column mass
            out[qs:qe, h] = p @ vd[ks:ke, g]
            lse[h, qs:qe] = lse_rows
    return out, lse


def oracle_merge(o_parts: Sequence[torch.Tensor], lse_parts: Sequence[torch.Tensor],
                 sink: torch.Tensor):
    """Merge C chunk results (out [T_q, H_q, d], lse [H_q, T_q]) with the sink.

    Returns out [T_q, H_q, d] and lse [H_q, T_q] (float64), following the
    formula in the module docstring.
    """
    o = torch.stack([x.to(F64) for x in o_parts])          # [C, T, H, d]
    ls = torch.stack([x.to(F64) for x in lse_parts])       # [C, H, T]
    s = sink.to(F64).view(1, -1, 1).expand(1, ls.shape[1], ls.shape[2])
    allv = torch.cat([ls, s], dim=0)                       # [C + 1, H, T]
    m = allv.max(dim=0).values                             # [H, T]
    m_safe = torch.where(torch.isfinite(m), m, torch.zeros_like(m))
    w = torch.exp(allv - m_safe)                           # exp(-inf) = 0
    z = w.sum(dim=0)                                       # [H, T]
    z_safe = torch.where(z > 0, z, torch.ones_like(z))
    wc = (w[:-1] / z_safe).where(z > 0, torch.zeros_like(w[:-1]))   # [C, H, T]
    out = (wc.permute(0, 2, 1).unsqueeze(-1) * o).sum(dim=0)       # [T, H, d]
    lse = torch.where(z > 0, m_safe + torch.log(z_safe), torch.full_like(z, -math.inf))
    return out, lse
