"""Seeded input generators: determinism, shapes and the workload recipes."""
import math

import torch

from attention_learnable_head_gb300.inputs import (SINK_CHOICES, WORKLOADS, draw_lengths,
                                                   make_case, small_workload)


def test_deterministic_and_bf16():
    w = small_workload("x", 7, 4, 2, [10, 20])
    a, b = make_case(w), make_case(w)
    for name in ("q", "k", "v", "dout", "sink"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert a.q.dtype == torch.bfloat16 and a.sink.dtype == torch.float32
    assert a.q.shape == (30, 4, 64) and a.k.shape == (30, 2, 64)
    assert a.cu_seqlens == [0, 10, 30]


def test_varlen_lengths_recipe():
    w = WORKLOADS["varlen"]
    lengths = draw_lengths(w)
    assert all(512 <= n <= 16384 for n in lengths)
    assert sum(lengths) <= 65536
    assert lengths == draw_lengths(w)


def test_varlen_sinks_cover_all_choices():
    w = WORKLOADS["varlen"]
    g = torch.Generator().manual_seed(1000 * w.seed_index + 6)
    perm = torch.randperm(w.heads_q, generator=g)
    vals = {SINK_CHOICES[int(perm[h]) % 5] for h in range(w.heads_q)}
    assert vals == set(SINK_CHOICES)


def test_long_workloads_share_inputs():
    a, b = WORKLOADS["long_full"], WORKLOADS["long_window"]
    assert a.seed_index == b.seed_index and a.q_mult == 3.0 and b.window == 128
    assert math.isclose(a.scale, 0.125)
