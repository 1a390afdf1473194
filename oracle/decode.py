"""CPU float64 oracle of the decode forward over a paged key/value cache.

TEST INFRASTRUCTURE ONLY -- never imported by the product path.

Where this comes from
--------------------
The rollout side of the pages serves GPT-OSS with attention sinks: page
"Treinamento de RL Agêntico para modelos GPT-OSS" (ai-engineering-academy-news),
section "Desafio 2: Inconsistência Treino-Inferência" (inference on vLLM/SGLang
with attention sinks) and section "Desafio 3: Attention Sinks no FlashAttention"
(the vLLM fork's forward pass adapted); the keryc.com page on GPT-OSS agentic
RL fixes, section "Problems that surfaced when trying agentic RL with GPT-OSS" (the
training-inference mismatch
between FSDP and the inference engines).  A decode step attends one
new query token per sequence to every cached key of that sequence, which is the
last row of the causal concat-sink attention (listing "带汇聚的注意力（GPT-OSS）"
of the euno.news page) with N_q = 1: under the bottom-right alignment the
single row sees all L cached keys, or the last W of them with a window.

The cache is paged the way serving engines lay it out: k_cache and v_cache
[num_pages, page_size, H_kv, d]; block_table[b, p] is the page that holds keys
[p * page_size, (p + 1) * page_size) of sequence b; seq_lens[b] = L_b.  The
oracle gathers each sequence's keys into a dense [L_b, H_kv, d] block and
calls the main oracle, so the decode oracle is the prefill definition applied
to the gathered keys.
"""
from __future__ import annotations

import torch

from .attention_sink import oracle_fwd


def gather_pages(cache: torch.Tensor, block_table: torch.Tensor, seq_len: int,
                 b: int) -> torch.Tensor:
    """Keys (or values) 0..seq_len-1 of sequence b from a paged cache."""
    page = cache.shape[1]
    n_pages = (seq_len + page - 1) // page
    if n_pages == 0:
        return cache.new_zeros((0,) + tuple(cache.shape[2:]))
    blocks = [cache[int(block_table[b, p])] for p in range(n_pages)]
    return torch.cat(blocks, dim=0)[:seq_len]


def oracle_decode(q, k_cache, v_cache, block_table, seq_lens, sink, *, scale: float,
                  window: int = 0):
    """out [B, H_q, d] and lse [H_q, B] (float64) of one decode step.

    q [B, H_q, d]: the new token of each sequence; the caches hold L_b keys of
    sequence b (the new token's own key included, as serving engines append it
    before attending).  L_b = 0 gives the sink alone: out = 0, lse = sink.
    """
    bsz = q.shape[0]
    outs, lses = [], []
    for b in range(bsz):
        L = int(seq_lens[b])
        k = gather_pages(k_cache, block_table, L, b)
        v = gather_pages(v_cache, block_table, L, b)
        out, lse = oracle_fwd(q[b:b + 1], k, v, sink, scale=scale, causal=True, window=window,
                              cu_seqlens_q=[0, 1], cu_seqlens_k=[0, L])
        outs.append(out[0])
        lses.append(lse[:, 0])
    return torch.stack(outs), torch.stack(lses, dim=1)
