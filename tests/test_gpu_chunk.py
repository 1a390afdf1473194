"""GPU parity of attention over key chunks (attn_sink_fwd_chunk) and of the
sink-aware merge (attn_sink_merge), through the C ABI, against the float64
oracle: each chunk against the chunk oracle, the merge alone against the merge
oracle, and chunk-then-merge against full attention with the sink.  Sizes span
several 128-row tiles, ragged tails, chunk boundaries off the tile grid, a
window, a chunk that no row sees and extreme sinks; the 4096-token layer is
checked on sampled rows."""
import math
import zlib

import pytest
import torch

from attention_learnable_head_gb300 import binding
from attention_learnable_head_gb300.inputs import WORKLOADS, make_case
from oracle import oracle_fwd
from oracle.attention_sink import dense_cu_seqlens
from oracle.chunk_merge import oracle_fwd_chunk, oracle_merge
from parity import TOL_LSE, assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _inputs(seed, b, nq, nk, hq, hkv, sink_vals=None):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(b * nq, hq, 64, generator=g).to(torch.bfloat16)
    k = torch.randn(b * nk, hkv, 64, generator=g).to(torch.bfloat16)
    v = torch.randn(b * nk, hkv, 64, generator=g).to(torch.bfloat16)
    sink = (torch.randn(hq, generator=g) if sink_vals is None
            else torch.tensor(sink_vals, dtype=torch.float32))
    return q, k, v, sink


def _chunk_keys(k, v, b, nk, k0, k1):
    idx = torch.cat([torch.arange(s * nk + k0, s * nk + k1) for s in range(b)])
    return k[idx], v[idx]


def _gpu_chunk(q, kc, vc, b, nq, nkc, q_pos0, causal, window, scale):
    q4 = q.to(DEV).view(b, nq, *q.shape[1:])
    k4 = kc.to(DEV).view(b, nkc, *kc.shape[1:])
    v4 = vc.to(DEV).view(b, nkc, *vc.shape[1:])
    out, lse, res = binding.forward_chunk(q4, k4, v4, q_pos0, causal=causal, window=window,
                                          softmax_scale=scale)
    return out.view(b * nq, *q.shape[1:]), lse, res.view(b * nq, *q.shape[1:])


def _check_lse(name, got, ref):
    got, ref = got.double().cpu(), ref.double()
    assert torch.equal(torch.isneginf(got), torch.isneginf(ref)), f"{name}: -inf pattern"
    fin = torch.isfinite(ref)
    err = (got[fin] - ref[fin]).abs().max().item() if fin.any() else 0.0
    assert err <= TOL_LSE, f"{name}: lse max abs {err:.3e}"


CASES = [
    # name, b, nq, nk, hq, hkv, causal, window, chunk bounds
    ("causal_3chunks", 2, 300, 300, 4, 2, True, 0, [(0, 100), (100, 131), (131, 300)]),
    ("nq_lt_nk", 1, 200, 333, 4, 1, True, 0, [(0, 256), (256, 333)]),
    ("window_100", 1, 385, 385, 2, 2, True, 100, [(0, 128), (128, 200), (200, 385)]),
    ("noncausal", 2, 129, 190, 2, 1, False, 0, [(0, 64), (64, 190)]),
    ("invisible_chunk", 1, 64, 400, 2, 1, True, 16, [(0, 256), (256, 400)]),
    # G = 8 with a window: the chunks take the sliding-window kernel
    ("window_g8", 2, 500, 500, 16, 2, True, 128, [(0, 200), (200, 263), (263, 500)]),
]


@pytest.mark.parametrize("name,b,nq,nk,hq,hkv,causal,window,bounds", CASES)
def test_chunks_and_merge(name, b, nq, nk, hq, hkv, causal, window, bounds):
    q, k, v, sink = _inputs(zlib.crc32(name.encode()) % 1000, b, nq, nk, hq, hkv)
    scale = 0.125
    cu_q = dense_cu_seqlens(b, nq)
    outs, lses, ress = [], [], []
    for k0, k1 in bounds:
        kc, vc = _chunk_keys(k, v, b, nk, k0, k1)
        q_pos0 = (nk - nq) - k0
        out, lse, res = _gpu_chunk(q, kc, vc, b, nq, k1 - k0, q_pos0, causal, window, scale)
        ref_o, ref_l = oracle_fwd_chunk(q, kc, vc, scale=scale, causal=causal, window=window,
                                        q_pos0=q_pos0, cu_seqlens_q=cu_q,
                                        cu_seqlens_k=dense_cu_seqlens(b, k1 - k0))
        assert_close(f"{name} chunk [{k0},{k1}) out", out, ref_o)
        _check_lse(f"{name} chunk [{k0},{k1})", lse, ref_l)
        outs.append(out)
        lses.append(lse)
        ress.append(res)
    out, lse, _ = binding.merge(outs, lses, sink.to(DEV), residuals=ress)
    ref_out, ref_lse = oracle_fwd(q, k, v, sink, scale=scale, causal=causal, window=window,
                                  cu_seqlens_q=cu_q, cu_seqlens_k=dense_cu_seqlens(b, nk))
    assert_close(f"{name} merged out", out, ref_out)
    _check_lse(f"{name} merged", lse, ref_lse)


def test_merge_alone_against_merge_oracle():
    """The merge kernel on oracle chunk results (bf16 + residual), with sinks
    of -inf, very large and ordinary values, and rows where every chunk is empty."""
    g = torch.Generator().manual_seed(11)
    c, t, h = 3, 257, 5
    o = [torch.randn(t, h, 64, generator=g, dtype=torch.float64) for _ in range(c)]
    ls = [4 * torch.randn(h, t, generator=g, dtype=torch.float64) for _ in range(c)]
    ls[1][:, :40] = -math.inf          # chunk 1 empty for the first rows
    for x in ls:
        x[2, 100:110] = -math.inf       # every chunk empty for some rows of head 2
    sink = torch.tensor([-math.inf, 30.0, -math.inf, 0.5, -3.0], dtype=torch.float64)
    ref_out, ref_lse = oracle_merge(o, ls, sink)
    hi = [x.to(torch.bfloat16) for x in o]
    lo = [(x - y.double()).to(torch.bfloat16) for x, y in zip(o, hi)]
    out, lse, res = binding.merge([x.to(DEV) for x in hi], [x.float().to(DEV) for x in ls],
                                  sink.float().to(DEV), residuals=[x.to(DEV) for x in lo])
    assert_close("merge out", out, ref_out)
    both = (out.double() + res.double()).cpu()
    assert_close("merge out + residual", both.float(), ref_out, max_abs=1e-3, rel_fro=1e-4)
    _check_lse("merge", lse, ref_lse)


def test_gptoss_layer_in_four_chunks_sampled_rows():
    """The 4096-token GPT-OSS-shaped layer (H 64/8, causal) split into four
    key chunks of 1024: chunk-then-merge against the oracle on sampled rows
    (ragged tail rows of the last tile included) of all heads."""
    w = WORKLOADS["gptoss_full"]
    c = make_case(w)
    n = c.lengths[0]
    outs, lses, ress = [], [], []
    for k0 in range(0, n, 1024):
        kc, vc = c.k[k0:k0 + 1024], c.v[k0:k0 + 1024]
        out, lse, res = _gpu_chunk(c.q, kc, vc, 1, n, 1024, -k0, True, 0, w.scale)
        outs.append(out)
        lses.append(lse)
        ress.append(res)
    out, lse, _ = binding.merge(outs, lses, c.sink.to(DEV), residuals=ress)
    rows = [0, 1, 127, 128, 1023, 1024, 2047, 2500, 3071, 3072, 4000, 4094, 4095]
    ref_out, ref_lse = oracle_fwd(c.q, c.k, c.v, c.sink, scale=w.scale, causal=True, window=0,
                                  cu_seqlens_q=c.cu_seqlens, cu_seqlens_k=c.cu_seqlens,
                                  rows={0: rows})
    idx = torch.tensor(rows)
    assert_close("gptoss 4 chunks out", out.cpu()[idx], ref_out[idx])
    _check_lse("gptoss 4 chunks", lse.cpu()[:, idx], ref_lse[:, idx])
