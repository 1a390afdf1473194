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
    # the committed entry for the current sources is found ...
    got = bench.dram_traffic("attn_sink_fwd_kernel", "gptoss_full")
    assert got is None or got > 0
    # ... and a kernel whose sources hash differently gets no traffic figure
    monkeypatch.setattr(bench, "kernel_sources_hash", lambda kernel: "0" * 16)
    assert bench.dram_traffic("attn_sink_fwd_kernel", "gptoss_full") is None


NCU_CSV = """==PROF== Connected to process 1
"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"
"0","1","python3","h","attn_sink::attn_sink_fwd_kernel(attn_sink::FwdParams)","1","7","(320, 1, 1)","(64, 1, 32)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Mbyte","40.00"
"0","1","python3","h","attn_sink::attn_sink_fwd_kernel(attn_sink::FwdParams)","1","7","(320, 1, 1)","(64, 1, 32)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","byte","1,000,000"
"1","1","python3","h","attn_sink::attn_sink_fwd_kernel(attn_sink::FwdParams)","1","7","(320, 1, 1)","(64, 1, 32)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Mbyte","44.00"
"1","1","python3","h","attn_sink::attn_sink_fwd_kernel(attn_sink::FwdParams)","1","7","(320, 1, 1)","(64, 1, 32)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","Mbyte","3.00"
"2","1","python3","h","void at::native::fill(int)","1","7","(128, 1, 1)","(64, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Mbyte","9.00"
"""


def test_record_traffic_parses_an_ncu_csv(tmp_path, monkeypatch):
    """--record-traffic: mean bytes per launch of each library kernel, scaled,
    stored with the kernel's current source hash, and read back by dram_traffic."""
    path = tmp_path / "dram.csv"
    path.write_text(NCU_CSV)
    monkeypatch.setattr(bench, "TRAFFIC_JSON", str(tmp_path / "traffic.json"))
    bench.record_traffic(str(path), "tinyish", 4.0, "ncu ...")
    got = bench.dram_traffic("attn_sink_fwd_kernel", "tinyish")
    assert got == 4.0 * ((40e6 + 44e6) / 2 + (1e6 + 3e6) / 2)
    assert bench.dram_traffic("attn_sink_bwd_main_kernel", "tinyish") is None
    # a second record of the same (kernel, workload) replaces the first
    bench.record_traffic(str(path), "tinyish", 1.0, "ncu ...")
    assert bench.dram_traffic("attn_sink_fwd_kernel", "tinyish") == got / 4.0


def test_both_arms_print_the_same_config():
    from attention_learnable_head_gb300.inputs import WORKLOADS, draw_lengths
    w = WORKLOADS["long_full"]
    a = bench.config_dict(w, draw_lengths(w), 1)
    assert a == bench.config_dict(w, draw_lengths(w), 1)
    assert a["workload"] == "long_full" and a["batch"] == 4 and a["seq_len"] == 16384
