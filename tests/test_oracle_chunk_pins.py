"""Pins of the chunked-attention oracle and its sink-aware merge (CPU only).

Splitting the keys into chunks, attending each without the sink and merging
with the sink must give exactly the attention of the concat definition
(`oracle_fwd`, itself pinned in test_oracle_pins.py) -- a check that does not
reuse the merge formula.  Plus a hand-worked closed form and the identities of
a single chunk and of an invisible chunk.
"""
import math

import pytest
import torch

from oracle import oracle_fwd
from oracle.attention_sink import dense_cu_seqlens
from oracle.chunk_merge import oracle_fwd_chunk, oracle_merge, visible_mask_at

F64 = torch.float64


def _case(seed, b, nq, nk, hq, hkv, d=16, sink_scale=1.0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(b * nq, hq, d, generator=g, dtype=F64)
    k = torch.randn(b * nk, hkv, d, generator=g, dtype=F64)
    v = torch.randn(b * nk, hkv, d, generator=g, dtype=F64)
    sink = sink_scale * torch.randn(hq, generator=g, dtype=F64)
    return q, k, v, sink


def _chunks_of(k, v, b, nk, bounds):
    """Per chunk [k0, k1): the chunk's keys of every sequence, packed."""
    out = []
    for k0, k1 in bounds:
        idx = torch.cat([torch.arange(s * nk + k0, s * nk + k1) for s in range(b)])
        out.append((k0, k1, k[idx], v[idx]))
    return out


@pytest.mark.parametrize("b,nq,nk,hq,hkv,causal,window,bounds", [
    (2, 48, 48, 2, 1, True, 0, [(0, 17), (17, 30), (30, 48)]),
    (1, 40, 64, 4, 2, True, 0, [(0, 24), (24, 64)]),
    (1, 64, 64, 2, 2, True, 9, [(0, 20), (20, 21), (21, 64)]),
    (2, 32, 50, 2, 1, False, 0, [(0, 7), (7, 50)]),
    (1, 16, 64, 2, 1, True, 8, [(0, 32), (32, 64)]),      # chunk 0 invisible to every row
])
def test_chunks_merged_equal_full_attention(b, nq, nk, hq, hkv, causal, window, bounds):
    q, k, v, sink = _case(7 + nq + nk, b, nq, nk, hq, hkv)
    scale = 0.3
    cu_q, cu_k = dense_cu_seqlens(b, nq), dense_cu_seqlens(b, nk)
    ref_out, ref_lse = oracle_fwd(q, k, v, sink, scale=scale, causal=causal, window=window,
                                  cu_seqlens_q=cu_q, cu_seqlens_k=cu_k)
    o_parts, l_parts = [], []
    for k0, k1, kc, vc in _chunks_of(k, v, b, nk, bounds):
        o, l = oracle_fwd_chunk(q, kc, vc, scale=scale, causal=causal, window=window,
                                q_pos0=(nk - nq) - k0, cu_seqlens_q=cu_q,
                                cu_seqlens_k=dense_cu_seqlens(b, k1 - k0))
        o_parts.append(o)
        l_parts.append(l)
    out, lse = oracle_merge(o_parts, l_parts, sink)
    torch.testing.assert_close(out, ref_out, rtol=1e-12, atol=1e-12)
    torch.testing.assert_close(lse, ref_lse, rtol=1e-12, atol=1e-12)


def test_invisible_chunk_is_zero_and_minus_inf():
    q, k, v, _ = _case(3, 1, 16, 64, 2, 1)
    o, l = oracle_fwd_chunk(q, k[:32], v[:32], scale=0.5, causal=True, window=8,
                            q_pos0=48, cu_seqlens_q=[0, 16], cu_seqlens_k=[0, 32])
    assert torch.all(o == 0)
    assert torch.all(torch.isneginf(l))


def test_single_chunk_without_sink_is_identity():
    q, k, v, _ = _case(5, 1, 24, 24, 2, 2)
    o, l = oracle_fwd_chunk(q, k, v, scale=0.4, causal=True, window=0, q_pos0=0,
                            cu_seqlens_q=[0, 24], cu_seqlens_k=[0, 24])
    out, lse = oracle_merge([o], [l], torch.full((2,), -math.inf, dtype=F64))
    torch.testing.assert_close(out, o, rtol=0, atol=1e-15)
    torch.testing.assert_close(lse, l, rtol=0, atol=1e-15)


def test_hand_worked_two_chunks_and_sink():
    # one query, d = 1, keys k = [1, 2] in separate chunks, v = [3, -1],
    # scale 1, q = 0.5, sink 0.25:  S = [0.5, 1.0]
    q = torch.tensor([[[0.5]]], dtype=F64)
    ks = [torch.tensor([[[1.0]]], dtype=F64), torch.tensor([[[2.0]]], dtype=F64)]
    vs = [torch.tensor([[[3.0]]], dtype=F64), torch.tensor([[[-1.0]]], dtype=F64)]
    sink = torch.tensor([0.25], dtype=F64)
    parts = [oracle_fwd_chunk(q, kk, vv, scale=1.0, causal=False, window=0, q_pos0=0,
                              cu_seqlens_q=[0, 1], cu_seqlens_k=[0, 1])
             for kk, vv in zip(ks, vs)]
    out, lse = oracle_merge([p[0] for p in parts], [p[1] for p in parts], sink)
    z = math.exp(0.5) + math.exp(1.0) + math.exp(0.25)
    assert abs(out.item() - (3 * math.exp(0.5) - math.exp(1.0)) / z) < 1e-14
    assert abs(lse.item() - math.log(z)) < 1e-14


def test_visible_mask_at_matches_main_alignment():
    # q_pos0 = N_k - N_q reproduces the bottom-right mask of the main oracle
    from oracle import visible_mask
    for nq, nk, w in ((8, 8, 0), (5, 12, 0), (12, 12, 3)):
        torch.testing.assert_close(visible_mask_at(nq, nk, nk - nq, True, w),
                                   visible_mask(nq, nk, True, w), rtol=0, atol=0)
