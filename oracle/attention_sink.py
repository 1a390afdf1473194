"""Plain, slow CPU float64 oracle of attention with a learnable per-head sink.

TEST INFRASTRUCTURE ONLY -- never imported by the product path.

What it computes, and where the pages define it
------------------------------------------------
* Sink attention, concat form.  Page "解锁 GPT-OSS 的 Agentic RL 训练：实用回顾"
  (euno.news), section "FlashAttention V3 中的注意力汇聚支持", listing
  "带汇聚的注意力（GPT-OSS）"; the same listing appears on page "Treinamento de
  RL Agêntico para modelos GPT-OSS" (ai-engineering-academy-news), section
  "Desafio 3: Attention Sinks no FlashAttention".  Scores are scaled, the
  per-head sink logit is appended as one extra column, a softmax is taken over
  the widened row, the extra column is dropped and the rest multiplies V.
* Probabilities: euno.news page, section "数学公式", the P_ij and P_ih
  equations: P_ij = e^{S_ij} / (sum_j' e^{S_ij'} + e^{S_h}), P_ih likewise
  with e^{S_h} on top.
* Sink gradient: euno.news page, section "反向传播":
  dL/dS_h = - sum_i P_ih * (sum_j P_ij * dP_ij).  The printed inner factor
  reads dL/dS_ij; only dL/dP_ij makes the identity true (d P_ij / d S_h =
  -P_ij P_ih and the sink column has no value row), so that is the reading
  taken here.
* dQ, dK, dV are the ordinary softmax-attention backward written out
  explicitly (dP = dO V^T, dS = P o (dP - D), dQ = s dS K, dK = s dS^T Q,
  dV = P^T dO).  The pages state only that the backward was implemented.

Readings where the pages are silent (each is pinned by a test):
* one sink per *query* head; sink[h] is not multiplied by the softmax scale;
* grouped-query attention: query head h reads key/value head h // (H_q/H_kv);
* causal masking is bottom-right aligned: local query row i sees key j iff
  j <= i + (N_k - N_q);
* a sliding window W > 0 (causal only) keeps the W most recent keys including
  the diagonal: i + (N_k - N_q) - W < j;
* a row with no visible key keeps the sink alone: P_ih = 1, O = 0,
  LSE = sink[h].  With sink[h] = -inf as well, O = 0 and LSE = -inf.

Layouts (the same as the CUDA library's): q [T_q, H_q, d], k and v
[T_k, H_kv, d], dout like q, sink [H_q] float32, token-packed with the
sequence boundaries in cu_seqlens (a dense batch B x N is packed with
cu_seqlens = [0, N, 2N, ...]).  lse is [H_q, T_q].  All arithmetic is float64
on values upcast exactly from the inputs.

The only liberty taken with the definition: rows are processed in blocks of
``block`` queries and each block only looks at the key range its mask can
reach.  Hidden keys carry probability exactly zero, so this changes nothing
but the summation order of exact zeros.
"""
from __future__ import annotations

import math
from typing import Iterable, Sequence

import torch

F64 = torch.float64


def sequence_bounds(cu_seqlens: Sequence[int]) -> list[tuple[int, int]]:
    """[(start, end)] of each packed sequence from a cu_seqlens list."""
    cu = [int(x) for x in cu_seqlens]
    return [(cu[i], cu[i + 1]) for i in range(len(cu) - 1)]


def visible_mask(n_q: int, n_k: int, causal: bool, window: int,
                 row_lo: int = 0, row_hi: int | None = None,
                 col_lo: int = 0, col_hi: int | None = None) -> torch.Tensor:
    """Boolean [rows, cols] mask: True where query row i may attend key j.

    Bottom-right aligned causal mask; window W > 0 keeps W keys including the
    diagonal.  Rows/cols may be restricted to [row_lo,row_hi) x [col_lo,col_hi).
    """
    row_hi = n_q if row_hi is None else row_hi
    col_hi = n_k if col_hi is None else col_hi
    i = torch.arange(row_lo, row_hi).unsqueeze(1)
    j = torch.arange(col_lo, col_hi).unsqueeze(0)
    vis = torch.ones(row_hi - row_lo, col_hi - col_lo, dtype=torch.bool)
    if causal:
        diag = i + (n_k - n_q)
        vis &= j <= diag
        if window > 0:
            vis &= j > diag - window
    return vis


def sink_softmax(scores: torch.Tensor, sink_h: float):
    """Softmax over [scores | sink] with the sink column split off.

    ``scores`` is [rows, n_k] float64 with -inf at hidden keys.  Returns
    (P_content [rows, n_k], P_sink [rows], lse [rows]) following the concat
    listing and the P_ij / P_ih equations on the euno.news page ("数学公式").
    """
    rows = scores.shape[0]
    sink_col = torch.full((rows, 1), float(sink_h), dtype=F64)
    combined = torch.cat([scores, sink_col], dim=1)       # [rows, n_k + 1]
    m = combined.max(dim=1, keepdim=True).values
    m_safe = torch.where(torch.isfinite(m), m, torch.zeros_like(m))
    e = torch.exp(combined - m_safe)
    z = e.sum(dim=1, keepdim=True)
    p = torch.where(z > 0, e / torch.where(z > 0, z, torch.ones_like(z)),
                    torch.zeros_like(e))
    lse = torch.where(z > 0, m_safe + torch.log(torch.where(z > 0, z, torch.ones_like(z))),
                      torch.full_like(z, -math.inf))
    return p[:, :-1], p[:, -1], lse.squeeze(1)


def _key_range(n_q, n_k, causal, window, r0, r1):
    """Keys that rows [r0, r1) can see (a superset: the mask still applies)."""
    if not causal:
        return 0, n_k
    off = n_k - n_q
    hi = min(n_k, r1 - 1 + off + 1)
    lo = 0 if window <= 0 else max(0, r0 + off - window + 1)
    hi = max(hi, lo)
    return lo, hi


def _check(q, k, v, sink):
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k, v must be [tokens, heads, head_dim]")
    h_q, h_kv = q.shape[1], k.shape[1]
    if h_q % h_kv:
        raise ValueError("H_q must be a multiple of H_kv")
    if sink.shape != (h_q,):
        raise ValueError("sink must be [H_q]")
    return h_q // h_kv


def _as_list(x, n):
    return list(range(n)) if x is None else [int(i) for i in x]


def oracle_fwd(q, k, v, sink, *, scale: float, causal: bool, window: int,
               cu_seqlens_q: Sequence[int], cu_seqlens_k: Sequence[int],
               heads: Iterable[int] | None = None,
               seqs: Iterable[int] | None = None,
               rows: dict | None = None, block: int = 256):
    """Forward: out [T_q, H_q, d] and lse [H_q, T_q], both float64.

    ``heads`` / ``seqs`` restrict the work to some query heads / sequences;
    ``rows`` maps a sequence index to the local query rows to compute.
    Entries not computed are NaN.
    """
    out, lse, _ = _run(q, k, v, sink, None, scale=scale, causal=causal,
                       window=window, cu_q=cu_seqlens_q, cu_k=cu_seqlens_k,
                       heads=heads, seqs=seqs, rows=rows, block=block)
    return out, lse


def oracle_bwd(q, k, v, sink, dout, *, scale: float, causal: bool, window: int,
               cu_seqlens_q: Sequence[int], cu_seqlens_k: Sequence[int],
               heads: Iterable[int] | None = None,
               seqs: Iterable[int] | None = None, block: int = 256):
    """Forward and explicit backward.

    Returns a dict with out, lse, dq, dk, dv, dsink and D (= sum_j P_ij dP_ij,
    [H_q, T_q]).  dk/dv of a key/value head are complete only when every query
    head of its group is in ``heads``; dsink[h] sums over the sequences in
    ``seqs``.  Entries not computed are NaN (dsink: NaN for excluded heads).
    """
    out, lse, grads = _run(q, k, v, sink, dout, scale=scale, causal=causal,
                           window=window, cu_q=cu_seqlens_q, cu_k=cu_seqlens_k,
                           heads=heads, seqs=seqs, rows=None, block=block)
    grads.update(out=out, lse=lse)
    return grads


def _run(q, k, v, sink, dout, *, scale, causal, window, cu_q, cu_k,
         heads, seqs, rows, block):
    group = _check(q, k, v, sink)
    if window > 0 and not causal:
        raise ValueError("a sliding window requires causal masking")
    qd, kd, vd = q.to(F64), k.to(F64), v.to(F64)
    sd = sink.to(F64)
    t_q, h_q, d = qd.shape
    t_k, h_kv, d_v = vd.shape
    bq, bk = sequence_bounds(cu_q), sequence_bounds(cu_k)
    if len(bq) != len(bk):
        raise ValueError("cu_seqlens_q and cu_seqlens_k differ in length")
    heads = _as_list(heads, h_q)
    seqs = _as_list(seqs, len(bq))

    nan = float("nan")
    out = torch.full((t_q, h_q, d_v), nan, dtype=F64)
    lse = torch.full((h_q, t_q), nan, dtype=F64)
    grads = None
    if dout is not None:
        dod = dout.to(F64)
        grads = dict(
            dq=torch.full((t_q, h_q, d), nan, dtype=F64),
            dk=torch.full((t_k, h_kv, d), nan, dtype=F64),
            dv=torch.full((t_k, h_kv, d_v), nan, dtype=F64),
            dsink=torch.full((h_q,), nan, dtype=F64),
            D=torch.full((h_q, t_q), nan, dtype=F64),
        )
        for h in heads:
            grads["dsink"][h] = 0.0
            g = h // group
            for s in seqs:
                ks, ke = bk[s]
                grads["dk"][ks:ke, g] = 0.0
                grads["dv"][ks:ke, g] = 0.0

    for s in seqs:
        qs, qe = bq[s]
        ks, ke = bk[s]
        n_q, n_k = qe - qs, ke - ks
        if rows is not None and s in rows:
            row_list = torch.as_tensor(sorted(int(r) for r in rows[s]), dtype=torch.long)
        elif rows is not None:
            continue
        else:
            row_list = None
        for h in heads:
            g = h // group
            Q = qd[qs:qe, h]
            K = kd[ks:ke, g]
            V = vd[ks:ke, g]
            if row_list is not None:
                blocks = [(int(r), int(r) + 1) for r in row_list]
            else:
                blocks = [(r0, min(n_q, r0 + block)) for r0 in range(0, n_q, block)]
            for r0, r1 in blocks:
                c0, c1 = _key_range(n_q, n_k, causal, window, r0, r1)
                scores = scale * (Q[r0:r1] @ K[c0:c1].T)
                vis = visible_mask(n_q, n_k, causal, window, r0, r1, c0, c1)
                scores = scores.masked_fill(~vis, -math.inf)
                p, p_sink, lse_blk = sink_softmax(scores, float(sd[h]))
                o_blk = p @ V[c0:c1]                        # sink column dropped
                out[qs + r0:qs + r1, h] = o_blk
                lse[h, qs + r0:qs + r1] = lse_blk
                if grads is None:
                    continue
                dO = dod[qs + r0:qs + r1, h]
                dP = dO @ V[c0:c1].T                         # dL/dP_ij
                D = (p * dP).sum(dim=1)                      # sum_j P_ij dP_ij
                dS = p * (dP - D.unsqueeze(1))
                grads["dq"][qs + r0:qs + r1, h] = scale * (dS @ K[c0:c1])
                grads["dk"][ks + c0:ks + c1, g] += scale * (dS.T @ Q[r0:r1])
                grads["dv"][ks + c0:ks + c1, g] += p.T @ dO
                grads["dsink"][h] += -(p_sink * D).sum()      # - sum_i P_ih D_i
                grads["D"][h, qs + r0:qs + r1] = D
    return out, lse, grads


def dense_cu_seqlens(batch: int, seqlen: int) -> list[int]:
    """cu_seqlens of a dense batch packed token-major."""
    return [b * seqlen for b in range(batch + 1)]
