"""GPU tests of the flag entry points (attn_sink_fwd_ex / attn_sink_bwd_ex) for a
sink held as a bf16 training parameter and a dsink that accumulates over
micro-batches: a bf16 sink gives exactly the results of the same values in
fp32; the bf16 dsink is the fp32 one rounded; accumulation adds the gradient
onto the given dsink (fp32 and bf16); the deterministic flag composes; and the
result still meets the oracle."""
import torch
import pytest

from attention_learnable_head_gb300 import binding
from attention_learnable_head_gb300.inputs import make_case, small_workload
from oracle import oracle_bwd
from parity import check_against

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _case(window=0):
    w = small_workload("flags", 701, 8, 2, [300, 129], causal=True, window=window)
    c = make_case(w)
    cu = torch.tensor(c.cu_seqlens, dtype=torch.int32, device=DEV)
    kw = dict(causal=w.causal, window=w.window, softmax_scale=w.scale, cu_seqlens_q=cu,
              cu_seqlens_k=cu, max_seqlen_q=max(c.lengths), max_seqlen_k=max(c.lengths))
    t = [x.to(DEV) for x in (c.q, c.k, c.v, c.dout)]
    return c, w, kw, t


@pytest.mark.parametrize("window", [0, 128])
def test_bf16_sink_equals_its_fp32_value(window):
    """Full causal (the tile kernel) and W = 128 (the sliding-window kernel)."""
    c, w, kw, (q, k, v, do) = _case(window)
    sink16 = c.sink.to(torch.bfloat16).to(DEV)
    sink32 = sink16.float()
    o16, l16, r16 = binding.forward(q, k, v, sink16, **kw)
    o32, l32, r32 = binding.forward(q, k, v, sink32, **kw)
    assert torch.equal(o16, o32) and torch.equal(l16, l32) and torch.equal(r16, r32)
    g16 = binding.backward(q, k, v, sink16, o16, l16, do, out_residual=r16, deterministic=True,
                           **kw)
    g32 = binding.backward(q, k, v, sink32, o32, l32, do, out_residual=r32, deterministic=True,
                           **kw)
    for a, b in zip(g16[:3], g32[:3]):
        assert torch.equal(a, b)
    assert g16[3].dtype == torch.bfloat16
    assert torch.equal(g16[3], g32[3].to(torch.bfloat16))
    torch.cuda.synchronize()
    assert binding.attn_sink_device_error() == (0, 0)
    # and the oracle agrees with the bf16-sink run
    c.sink = sink32.cpu()
    ref = oracle_bwd(c.q, c.k, c.v, c.sink, c.dout, scale=w.scale, causal=w.causal,
                     window=w.window, cu_seqlens_q=c.cu_seqlens, cu_seqlens_k=c.cu_seqlens)
    check_against(dict(out=o16.cpu(), lse=l16.cpu(), dq=g16[0].cpu(), dk=g16[1].cpu(),
                       dv=g16[2].cpu(), dsink=g16[3].float().cpu()), ref)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_dsink_accumulates(dtype):
    c, w, kw, (q, k, v, do) = _case()
    sink = c.sink.to(dtype).to(DEV)
    out, lse, res = binding.forward(q, k, v, sink, **kw)
    fresh = binding.backward(q, k, v, sink, out, lse, do, out_residual=res, deterministic=True,
                             **kw)[3]
    start = torch.linspace(-1.0, 1.0, sink.numel(), device=DEV).to(dtype)
    acc = start.clone()
    binding.backward(q, k, v, sink, out, lse, do, out_residual=res, deterministic=True,
                     dsink=acc, accumulate_dsink=True, **kw)
    torch.cuda.synchronize()
    assert binding.attn_sink_device_error() == (0, 0)
    if dtype == torch.float32:
        assert torch.equal(acc, start + fresh)
    else:
        # fp32 gradient added to the bf16 value, rounded once
        assert (acc.float() - (start.float() + fresh.float())).abs().max().item() <= \
            2 ** -7 * (start.float().abs() + fresh.float().abs()).max().item() + 1e-6
