"""attn_sink_fwd_noalloc: the forward for callers that cannot allocate device
memory themselves (a host framework that owns all device memory through its
own pool, or a service that must not allocate once running).  Its scratch is
the library's static device array instead of a caller workspace; the results
must be identical to attn_sink_fwd's on the same inputs (the same kernels run
on the same bytes), on two calls in a row (the second call reuses the array
the first one left behind).

This file is collected last on purpose: a failure here leaves every other test
already run."""
import pytest
import torch

from attention_learnable_head_gb300 import binding
from attention_learnable_head_gb300.build import build
from attention_learnable_head_gb300.inputs import make_case, small_workload

pytestmark = pytest.mark.gpu


def _inputs(dev, window):
    w = small_workload("noalloc", 991, 8, 2, [300, 129, 511], window=window)
    c = make_case(w)
    cu = torch.tensor(c.cu_seqlens, dtype=torch.int32, device=dev)
    t = [x.to(dev) for x in (c.q, c.k, c.v, c.sink)]
    p = binding.make_params(c.q.shape, c.k.shape, causal=True, window=window,
                            softmax_scale=w.scale, num_seqs=len(c.lengths),
                            max_seqlen_q=max(c.lengths), max_seqlen_k=max(c.lengths))
    return p, cu, t


@pytest.mark.parametrize("window", [0, 128])
def test_noalloc_forward_matches_workspace_forward(window):
    """Full causal (the tile kernel, with the packed batch's tile order in the
    scratch) and W = 128 (the sliding-window kernel)."""
    build()
    dev = torch.device("cuda:0")
    p, cu, (q, k, v, sink) = _inputs(dev, window)
    ref_out, ref_res = torch.empty_like(q), torch.empty_like(q)
    ref_lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=dev)
    ws = torch.empty(binding.attn_sink_fwd_workspace_size(p), dtype=torch.uint8, device=dev)
    st = binding.attn_sink_fwd(p, q, k, v, sink, cu, cu, ref_out, ref_res, ref_lse, ws,
                               ws.numel())
    assert st == 0
    for call in range(2):
        out, res = torch.full_like(q, float("nan")), torch.full_like(q, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = binding.attn_sink_fwd_noalloc(p, q, k, v, sink, cu, cu, out, res, lse)
        assert st == 0, binding.attn_sink_status_string(st)
        torch.cuda.synchronize()
        e_st, code = binding.attn_sink_device_error()
        assert e_st == 0 and code == 0, f"device error word {code:#x}"
        # the same kernels on the same bytes: the results are identical
        assert torch.equal(out, ref_out), f"out differs (call {call})"
        assert torch.equal(res, ref_res), f"out residual differs (call {call})"
        assert torch.equal(lse, ref_lse), f"lse differs (call {call})"
