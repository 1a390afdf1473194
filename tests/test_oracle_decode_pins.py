"""Pins of the paged decode oracle (CPU only): a cache built from dense keys
through a random page layout must give exactly the attention of the last query
row over those dense keys (the main, separately pinned oracle), for full and
windowed attention, ragged lengths, a page-aligned length and an empty cache."""
import math

import pytest
import torch

from oracle import oracle_fwd
from oracle.decode import gather_pages, oracle_decode

F64 = torch.float64


def _paged(seed, lens, page, hkv, d=16, spare=3):
    """Random dense keys/values per sequence, scattered into shuffled pages."""
    g = torch.Generator().manual_seed(seed)
    n_pages = sum((L + page - 1) // page for L in lens) + spare
    perm = torch.randperm(n_pages, generator=g)
    kc = torch.randn(n_pages, page, hkv, d, generator=g, dtype=F64)
    vc = torch.randn(n_pages, page, hkv, d, generator=g, dtype=F64)
    max_p = max((L + page - 1) // page for L in lens) if lens else 1
    table = torch.full((len(lens), max(max_p, 1)), -1, dtype=torch.int32)
    dense_k, dense_v, nxt = [], [], 0
    for b, L in enumerate(lens):
        k = torch.randn(L, hkv, d, generator=g, dtype=F64)
        v = torch.randn(L, hkv, d, generator=g, dtype=F64)
        for p in range((L + page - 1) // page):
            pg = int(perm[nxt]); nxt += 1
            table[b, p] = pg
            n = min(page, L - p * page)
            kc[pg, :n] = k[p * page:p * page + n]
            vc[pg, :n] = v[p * page:p * page + n]
        dense_k.append(k)
        dense_v.append(v)
    return kc, vc, table, dense_k, dense_v


@pytest.mark.parametrize("lens,page,window", [
    ([37, 1, 64, 100], 16, 0),
    ([300, 5], 64, 0),
    ([129, 70], 32, 50),
    ([0, 16], 16, 0),
])
def test_paged_decode_equals_last_row_of_dense_attention(lens, page, window):
    hq, hkv = 8, 2
    kc, vc, table, dk, dv = _paged(sum(lens) + page, lens, page, hkv)
    g = torch.Generator().manual_seed(99)
    q = torch.randn(len(lens), hq, 16, generator=g, dtype=F64)
    sink = torch.randn(hq, generator=g, dtype=F64)
    out, lse = oracle_decode(q, kc, vc, table, torch.tensor(lens), sink, scale=0.3,
                             window=window)
    for b, L in enumerate(lens):
        ref_o, ref_l = oracle_fwd(q[b:b + 1], dk[b], dv[b], sink, scale=0.3, causal=True,
                                  window=window, cu_seqlens_q=[0, 1], cu_seqlens_k=[0, L])
        torch.testing.assert_close(out[b], ref_o[0], rtol=0, atol=1e-12)
        torch.testing.assert_close(lse[:, b], ref_l[:, 0], rtol=0, atol=1e-12)


def test_empty_cache_is_the_sink_alone():
    kc, vc, table, _, _ = _paged(1, [0, 3], 16, 1)
    q = torch.ones(2, 2, 16, dtype=F64)
    sink = torch.tensor([0.7, -1.5], dtype=F64)
    out, lse = oracle_decode(q, kc, vc, table, torch.tensor([0, 3]), sink, scale=0.25)
    assert torch.all(out[0] == 0)
    torch.testing.assert_close(lse[:, 0], sink, rtol=0, atol=0)


def test_gather_pages_follows_the_block_table():
    cache = torch.arange(4 * 4, dtype=F64).view(4, 4, 1, 1)     # page p holds 4p..4p+3
    table = torch.tensor([[2, 0, 3]], dtype=torch.int32)
    got = gather_pages(cache, table, 10, 0).flatten().tolist()
    assert got == [8, 9, 10, 11, 0, 1, 2, 3, 12, 13]


def test_single_key_closed_form():
    """L = 1: out = v * e^s / (e^s + e^sink), lse = log(e^s + e^sink)."""
    kc = torch.zeros(1, 16, 1, 4, dtype=F64)
    vc = torch.zeros(1, 16, 1, 4, dtype=F64)
    kc[0, 0, 0] = torch.tensor([1.0, 0.0, 2.0, -1.0], dtype=F64)
    vc[0, 0, 0] = torch.tensor([3.0, -2.0, 0.5, 1.0], dtype=F64)
    q = torch.tensor([[[0.5, 1.0, 0.25, 0.0]]], dtype=F64)
    sink = torch.tensor([0.1], dtype=F64)
    out, lse = oracle_decode(q, kc, vc, torch.tensor([[0]], dtype=torch.int32),
                             torch.tensor([1]), sink, scale=2.0)
    s = 2.0 * (0.5 * 1.0 + 0.25 * 2.0)
    z = math.exp(s) + math.exp(0.1)
    torch.testing.assert_close(out[0, 0], vc[0, 0, 0] * math.exp(s) / z, rtol=0, atol=1e-14)
    assert abs(lse[0, 0].item() - math.log(z)) < 1e-14
