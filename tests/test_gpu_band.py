"""GPU parity of the sliding-window forward (attn_sink_fwd_band_kernel: items of
128 / G tokens x the G query heads of a kv group, one window of up to 176 keys
each) through the C ABI against the float64 oracle, forward and backward.

Cases: every power-of-two GQA group from 1 to 32, windows from 1 key up to the
largest window an item holds, ragged tails (written directly, not through the
TMA-stored tiles) and
sequences shorter than one item, empty sequences, N_q != N_k in both
directions, a sink of -inf, a bf16 sink, and enough items that every CTA of
the persistent grid walks several of them."""
import pytest
import torch

from attention_learnable_head_gb300 import binding
from attention_learnable_head_gb300.inputs import make_case, small_workload
from oracle import oracle_bwd
from parity import check_against, run_gpu

pytestmark = pytest.mark.gpu


def _ref(case, cu_q=None, cu_k=None):
    w = case.workload
    cq = case.cu_seqlens if cu_q is None else cu_q
    ck = case.cu_seqlens if cu_k is None else cu_k
    return oracle_bwd(case.q, case.k, case.v, case.sink, case.dout, scale=w.scale,
                      causal=True, window=w.window, cu_seqlens_q=cq, cu_seqlens_k=ck)


def _window_cols(group, window):
    """Keys of an item's window, as the library computes it (multiple of 16)."""
    return -(-(128 // group + window - 1) // 16) * 16


CASES = [
    # name, heads_q, heads_kv, lengths, window
    ("g8_w128_ragged", 16, 2, [1000, 17, 16, 15, 1], 128),     # N = 144
    ("g8_w161_widest", 16, 2, [700, 33], 161),                 # N = 176, the widest window
    ("g8_w1", 8, 1, [300, 5], 1),                               # N = 16: half 1 has no keys
    ("g16_w128", 32, 2, [400, 9], 128),                         # 8 tokens per item
    ("g32_w100", 32, 1, [260, 3, 4], 100),                      # 4 tokens per item
    ("g4_w128", 8, 2, [500, 31, 32, 33], 128),                  # N = 160
    ("g2_w64", 4, 2, [450, 63, 64, 65], 64),
    ("g1_w49", 2, 2, [300, 129], 49),                           # 128 tokens, N = 176
    ("g8_empty_seq", 16, 2, [0, 200, 0, 130], 128),
]


@pytest.mark.parametrize("name,hq,hkv,lengths,window", CASES, ids=[c[0] for c in CASES])
def test_band_cases(name, hq, hkv, lengths, window):
    assert _window_cols(hq // hkv, window) <= 176
    w = small_workload(name, 700 + len(name), hq, hkv, lengths, causal=True, window=window)
    c = make_case(w)
    check_against(run_gpu(c), _ref(c))


def test_band_many_items():
    """20000 tokens x 2 kv groups of 8 heads, W = 128: 2500 items, several per
    CTA of the persistent grid (two per SM), both gradient dtypes."""
    w = small_workload("band_many", 777, 16, 2, [12000, 8000], causal=True, window=128)
    c = make_case(w)
    check_against(run_gpu(c), _ref(c))


@pytest.mark.parametrize("lq,lk", [([100, 64, 0, 130, 300], [150, 10, 40, 130, 200]),
                                   ([40, 300], [300, 40])])
def test_band_query_key_lengths_differ(lq, lk):
    """N_q != N_k per sequence with G = 8, W = 128 (bottom-right alignment):
    windows that start before the sequence's first key, rows that see no key,
    an empty query sequence."""
    cq, ck = [0], [0]
    for a, b in zip(lq, lk):
        cq.append(cq[-1] + a)
        ck.append(ck[-1] + b)
    w = small_workload("band_qk", 790 + len(lq), 16, 2, [sum(lq)], causal=True, window=128)
    c = make_case(w)
    g = torch.Generator().manual_seed(4343)
    c.k = torch.randn((sum(lk), 2, 64), generator=g).to(torch.bfloat16)
    c.v = torch.randn((sum(lk), 2, 64), generator=g).to(torch.bfloat16)
    res = run_gpu(c, cu_q=cq, cu_k=ck)
    check_against(res, _ref(c, cu_q=cq, cu_k=ck))


def test_band_sink_neginf_and_dense_layout():
    """Sink = -inf (the softmax over keys alone; W = 1 rows are exactly their
    one key's value) and the dense [B, N, H, d] layout."""
    w = small_workload("band_neginf", 795, 16, 2, [300, 300], causal=True, window=1,
                       sink_kind="neginf")
    c = make_case(w)
    check_against(run_gpu(c), _ref(c))
    w = small_workload("band_dense", 796, 16, 2, [257, 257, 257], causal=True, window=128)
    c = make_case(w)
    check_against(run_gpu(c, dense=True), _ref(c))


def test_band_repeatable():
    """The sliding-window forward has no atomics and no order-dependent sums:
    twelve runs on 6000 tokens x 2 kv groups of 8 heads (several items per
    persistent CTA, deferred epilogues, TMA-stored tiles) are bitwise equal."""
    w = small_workload("band_repeat", 781, 16, 2, [3000, 1500, 1500], causal=True, window=128)
    c = make_case(w)
    dev = torch.device("cuda:0")
    q, k, v, sink = (x.to(dev) for x in (c.q, c.k, c.v, c.sink))
    cu = torch.tensor(c.cu_seqlens, dtype=torch.int32, device=dev)
    kw = dict(causal=True, window=128, softmax_scale=w.scale, cu_seqlens_q=cu, cu_seqlens_k=cu,
              max_seqlen_q=max(c.lengths), max_seqlen_k=max(c.lengths))
    first = binding.forward(q, k, v, sink, **kw)
    for _ in range(11):
        again = binding.forward(q, k, v, sink, **kw)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    torch.cuda.synchronize()
    assert binding.attn_sink_device_error() == (0, 0)
