"""Parity on the full-size workloads (GPU runs the whole problem in the launch
configuration the bench uses; the oracle checks whole query heads, whole
GQA groups or sampled query rows, each computed exactly as defined).

  gptoss_full  B=1, H 64/8, N=4096, causal        (the bench workload, dense layout)
  swa          B=1, H 64/8, N=16384, causal, W=128
  varlen       packed lengths ~ U[512,16384] up to 65536 tokens, sinks {-30,-2,0,2,8}
  long_full    B=4, H 64/8, N=16384, causal, q x3, sink ~ N(0, 2^2)
  long_window  as long_full with W=128

Each backward runs with bf16 and with fp32 gradients; tests/parity.py says
which stored form each tolerance is applied to.
"""
import pytest
import torch

from attention_learnable_head_gb300.inputs import WORKLOADS, make_case
from oracle import oracle_bwd, oracle_fwd
from parity import check_against, check_tensor, err_stats, run_gpu, TOL_LSE

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _group_heads(kv_heads, group=8):
    return [g * group + i for g in kv_heads for i in range(group)]


def _oracle(case, **kw):
    w = case.workload
    return oracle_bwd(case.q, case.k, case.v, case.sink, case.dout, scale=w.scale,
                      causal=w.causal, window=w.window, cu_seqlens_q=case.cu_seqlens,
                      cu_seqlens_k=case.cu_seqlens, **kw)


def _sampled_rows(case, per_seq=24, seed=5):
    g = torch.Generator().manual_seed(seed)
    rows = {}
    for s, n in enumerate(case.lengths):
        pick = torch.randint(0, n, (per_seq,), generator=g).tolist()
        rows[s] = sorted(set(pick + [0, n - 1]))
    return rows


def _check_rows(res, case, rows):
    """Forward out / lse of every head on sampled query rows."""
    w = case.workload
    out, lse = oracle_fwd(case.q, case.k, case.v, case.sink, scale=w.scale, causal=w.causal,
                          window=w.window, cu_seqlens_q=case.cu_seqlens,
                          cu_seqlens_k=case.cu_seqlens, rows=rows)
    check_tensor(res, out, "out")
    a, _ = err_stats(res["lse"], lse)
    assert a <= TOL_LSE, f"lse(rows) max abs {a:.3e}"


def test_gptoss_full():
    c = make_case(WORKLOADS["gptoss_full"])
    res = run_gpu(c, dense=True)
    kv = [0, 7]
    ref = _oracle(c, heads=_group_heads(kv))
    check_against(res, ref, heads=_group_heads(kv), kv_heads=kv)


def test_swa():
    c = make_case(WORKLOADS["swa"])
    res = run_gpu(c, dense=True)
    kv = [0, 5]
    ref = _oracle(c, heads=_group_heads(kv))
    check_against(res, ref, heads=_group_heads(kv), kv_heads=kv)


def test_varlen():
    c = make_case(WORKLOADS["varlen"])
    res = run_gpu(c)
    _check_rows(res, c, _sampled_rows(c))
    # full backward of kv group 0 (dq, dk, dv) on the shortest and on the
    # longest packed sequence
    by_len = sorted(range(len(c.lengths)), key=lambda i: c.lengths[i])
    for s in (by_len[0], by_len[-1]):
        ref = _oracle(c, heads=_group_heads([0]), seqs=[s])
        q0, q1 = c.cu_seqlens[s], c.cu_seqlens[s + 1]
        rows = slice(q0, q1)
        for name in ("dq", "dk", "dv"):
            sel = (rows, slice(0, 8) if name == "dq" else slice(0, 1))
            check_tensor(res, ref[name][sel], name, sel)
    # dsink sums over every sequence: heads whose sinks span the five values
    heads = []
    seen = set()
    for h in range(64):
        v = float(c.sink[h])
        if v not in seen:
            seen.add(v)
            heads.append(h)
    ref = _oracle(c, heads=heads)
    check_against({"dsink": res["dsink"]}, ref, heads=heads)


def test_long_full():
    """Sampled rows of every head and sequence (forward), and the whole
    forward and backward of two kv groups: group 3 of sequence 1 and group 6
    of sequence 3 (the last one, whose tiles run last)."""
    c = make_case(WORKLOADS["long_full"])
    res = run_gpu(c, dense=True)
    _check_rows(res, c, _sampled_rows(c, per_seq=12))
    n = c.lengths[0]
    for kv, seq in ((3, 1), (6, 3)):
        ref = _oracle(c, heads=_group_heads([kv]), seqs=[seq])
        rows = slice(seq * n, (seq + 1) * n)
        for name in ("out", "dq"):
            sel = (rows, slice(8 * kv, 8 * kv + 8))
            check_tensor(res, ref[name][sel], name, sel)
        for name in ("dk", "dv"):
            sel = (rows, slice(kv, kv + 1))
            check_tensor(res, ref[name][sel], name, sel)
    ref = _oracle(c, heads=[5, 40])
    check_against({"dsink": res["dsink"]}, ref, heads=[5, 40])


def test_long_window():
    c = make_case(WORKLOADS["long_window"])
    res = run_gpu(c, dense=True)
    kv = [1, 6]
    ref = _oracle(c, heads=_group_heads(kv))
    check_against(res, ref, heads=_group_heads(kv), kv_heads=kv)
