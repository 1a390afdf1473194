"""Host logic of bench.py that needs no GPU: the seeded serving-shaped inputs of
the decode measurement, the stored DRAM-traffic lookup and its source hash."""
import torch

import bench


def test_decode_case_is_a_valid_paged_cache():
    q, kc, vc, table, lens, sink = bench.decode_case(batch=5, cached=100, heads_q=8,
                                                     heads_kv=2, page=16, seed=7)
    per_seq = (100 + 15) // 16
    assert q.shape == (5, 8, 64) and q.dtype == torch.bfloat16
    assert kc.shape == vc.shape == (5 * per_seq, 16, 2, 64)
    assert table.shape == (5, per_seq) and table.dtype == torch.int32
    # every page of the pool is handed to exactly one (sequence, slot)
    assert torch.equal(torch.sort(table.flatten()).values, torch.arange(5 * per_seq,
                                                                         dtype=torch.int32))
    assert torch.equal(lens, torch.full((5,), 100, dtype=torch.int32))
    assert sink.shape == (8,)


def test_decode_case_is_seeded():
    a = bench.decode_case(2, 40, 4, 1, 8, seed=11)
    b = bench.decode_case(2, 40, 4, 1, 8, seed=11)
    c = bench.decode_case(2, 40, 4, 1, 8, seed=12)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert not torch.equal(a[1], c[1])


def test_traffic_is_reported_only_for_unchanged_sources(monkeypatch):
    h = bench.kernel_sources_hash("attn_sink_fwd_kernel")
    assert len(h) == 16 and int(h, 16) >= 0
    # the committed table row for the current sources is found ...
    got = bench.dram_traffic("attn_sink_fwd_kernel", "gptoss_full")
    assert got is None or got > 0
    # ... and a kernel whose sources hash differently gets no traffic figure
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda kernel: "0" * 16)
    assert bench.dram_traffic("attn_sink_fwd_kernel", "gptoss_full") is None
