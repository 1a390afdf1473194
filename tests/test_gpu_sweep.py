"""Seeded sweep of small shapes against the float64 oracle: sequence lengths
1..300 (mostly not multiples of the 128-row tile), packed 1-4 per call, GQA
groups G in {1, 2, 8}, windows in {none, 1, 127, 128, 129} and a few
non-causal cases, sinks from N(0, 1), -inf or +8.  The draws come from a
seeded torch.Generator, so every case is reproducible from its index."""
import pytest
import torch

from attention_learnable_head_gb300.inputs import make_case, small_workload
from oracle import oracle_bwd
from parity import check_against, run_gpu

pytestmark = pytest.mark.gpu

N_CASES = 24


def draw(idx: int):
    g = torch.Generator().manual_seed(7000 + idx)
    pick = lambda seq: seq[int(torch.randint(0, len(seq), (1,), generator=g))]  # noqa: E731
    group = pick([1, 2, 8])
    heads_kv = pick([1, 2])
    n_seqs = int(torch.randint(1, 5, (1,), generator=g))
    lengths = [int(x) for x in torch.randint(1, 301, (n_seqs,), generator=g)]
    window = pick([0, 0, 1, 127, 128, 129])
    causal = True if window > 0 else pick([True, True, False])
    sink_kind, sink_const = pick([("normal", 0.0), ("normal", 0.0), ("neginf", 0.0),
                                  ("const", 8.0)])
    return dict(group=group, heads_kv=heads_kv, lengths=lengths, window=window, causal=causal,
                sink_kind=sink_kind, sink_const=sink_const)


@pytest.mark.parametrize("idx", range(N_CASES))
def test_small_shape_sweep(idx):
    d = draw(idx)
    w = small_workload(f"sweep{idx}", 8000 + idx, d["group"] * d["heads_kv"], d["heads_kv"],
                       d["lengths"], causal=d["causal"], window=d["window"],
                       sink_kind=d["sink_kind"], sink_const=d["sink_const"])
    c = make_case(w)
    res = run_gpu(c)
    ref = oracle_bwd(c.q, c.k, c.v, c.sink, c.dout, scale=w.scale, causal=w.causal,
                     window=w.window, cu_seqlens_q=c.cu_seqlens, cu_seqlens_k=c.cu_seqlens)
    if d["sink_kind"] == "neginf":
        # standard attention: the sink has no gradient
        assert torch.equal(res["dsink"], torch.zeros_like(res["dsink"]))
        ref.pop("dsink")
    check_against(res, ref)
