"""The bounded-wait path, exercised without a fault.

Every mbarrier wait in the kernels gives up after a time limit, records a code
in the device error word, lets the copies and products already in flight
finish, frees its tensor memory and returns.  The test build of the library
(the same sources with the limit lowered to 2 ms and a hook that withholds one
tile) makes such a wait run out: the forward's producer never issues one K
tile, or the backward's never loads one step's Q/dO tiles.  The call must come
back within a fraction of a second with ATTN_SINK_ERR_TIMEOUT from
attn_sink_device_error (0x1xx forward, 0x2xx backward), and calls made
afterwards, in the test build and in the product library, must be clean and
correct: the context stays usable."""
import ctypes
import time

import pytest
import torch

from attention_learnable_head_gb300 import binding
from attention_learnable_head_gb300.build import build
from attention_learnable_head_gb300.inputs import make_case, small_workload
from oracle import oracle_bwd
from parity import check_against, run_gpu

pytestmark = pytest.mark.gpu

TIMEOUT = 5


def _setup(dev):
    # 512 keys: query tiles 1-3 see 2-4 key tiles, so withholding K tile 1 or
    # the Q/dO of step 1 leaves waits that cannot complete
    w = small_workload("timeout", 953, 4, 2, [512, 300])
    c = make_case(w)
    t = {n: getattr(c, n).to(dev) for n in ("q", "k", "v", "dout", "sink")}
    cu = torch.tensor(c.cu_seqlens, dtype=torch.int32, device=dev)
    p = binding.make_params(c.q.shape, c.k.shape, causal=True, window=0, softmax_scale=w.scale,
                            num_seqs=len(c.lengths), max_seqlen_q=max(c.lengths),
                            max_seqlen_k=max(c.lengths))
    return c, t, cu, p


def _ptr(x):
    return None if x is None else x.data_ptr()


def _fwd(L, p, t, cu, out, res, lse, ws, stream):
    return L.attn_sink_fwd(ctypes.byref(p), _ptr(t["q"]), _ptr(t["k"]), _ptr(t["v"]),
                           _ptr(t["sink"]), _ptr(cu), _ptr(cu), _ptr(out), _ptr(res), _ptr(lse),
                           _ptr(ws), ws.numel(), stream)


def _bwd(L, p, t, cu, out, res, lse, grads, ws, stream):
    dq, dk, dv, dsink = grads
    return L.attn_sink_bwd(ctypes.byref(p), _ptr(t["q"]), _ptr(t["k"]), _ptr(t["v"]),
                           _ptr(t["sink"]), _ptr(cu), _ptr(cu), _ptr(out), _ptr(res), _ptr(lse),
                           _ptr(t["dout"]), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dsink), _ptr(ws),
                           ws.numel(), stream)


def _device_error(L, stream):
    code = ctypes.c_int(0)
    st = L.attn_sink_device_error(stream, ctypes.byref(code))
    return st, code.value


def test_wait_that_runs_out_returns_a_timeout_and_leaves_the_context_usable():
    Lt = binding.load_library(build(test=True))
    dev = torch.device("cuda:0")
    c, t, cu, p = _setup(dev)
    stream = torch.cuda.current_stream().cuda_stream
    out, res = torch.empty_like(t["q"]), torch.empty_like(t["q"])
    lse = torch.empty((t["q"].shape[1], t["q"].shape[0]), dtype=torch.float32, device=dev)
    grads = (torch.empty_like(t["q"]), torch.empty_like(t["k"]), torch.empty_like(t["v"]),
             torch.empty_like(t["sink"]))
    fws = torch.empty(max(Lt.attn_sink_fwd_workspace_size(ctypes.byref(p)), 1),
                      dtype=torch.uint8, device=dev)
    bws = torch.empty(max(Lt.attn_sink_bwd_workspace_size(ctypes.byref(p)), 1),
                      dtype=torch.uint8, device=dev)
    # the test build without a withheld tile: clean, and the product library's results
    assert Lt.attn_sink_test_withhold(-1, -1) == 0
    assert _fwd(Lt, p, t, cu, out, res, lse, fws, stream) == 0
    assert _bwd(Lt, p, t, cu, out, res, lse, grads, bws, stream) == 0
    assert _device_error(Lt, stream) == (0, 0)
    ref = run_gpu(c)
    assert torch.equal(out.cpu(), ref["out"]) and torch.equal(lse.cpu(), ref["lse"])
    assert torch.equal(grads[1].cpu(), ref["dk"]) and torch.equal(grads[2].cpu(), ref["dv"])

    # forward: K tile 1 is never issued
    assert Lt.attn_sink_test_withhold(1, -1) == 0
    t0 = time.perf_counter()
    assert _fwd(Lt, p, t, cu, out, res, lse, fws, stream) == 0
    st, code = _device_error(Lt, stream)
    elapsed = time.perf_counter() - t0
    assert st == TIMEOUT and code & 0xF00 == 0x100, (st, hex(code))
    assert elapsed < 1.0, f"the forward took {elapsed:.3f} s to give up"
    assert _device_error(Lt, stream) == (0, 0)          # the word was cleared

    # backward: the Q/dO tiles of step 1 are never loaded
    assert Lt.attn_sink_test_withhold(-1, 1) == 0
    assert _fwd(Lt, p, t, cu, out, res, lse, fws, stream) == 0
    assert _device_error(Lt, stream) == (0, 0)
    t0 = time.perf_counter()
    assert _bwd(Lt, p, t, cu, out, res, lse, grads, bws, stream) == 0
    st, code = _device_error(Lt, stream)
    elapsed = time.perf_counter() - t0
    assert st == TIMEOUT and code & 0xF00 == 0x200, (st, hex(code))
    assert elapsed < 1.0, f"the backward took {elapsed:.3f} s to give up"

    # afterwards: the test build and the product library both run clean and correct
    assert Lt.attn_sink_test_withhold(-1, -1) == 0
    assert _fwd(Lt, p, t, cu, out, res, lse, fws, stream) == 0
    assert _bwd(Lt, p, t, cu, out, res, lse, grads, bws, stream) == 0
    assert _device_error(Lt, stream) == (0, 0)
    assert torch.equal(grads[1].cpu(), ref["dk"])
    w = c.workload
    oref = oracle_bwd(c.q, c.k, c.v, c.sink, c.dout, scale=w.scale, causal=True, window=0,
                      cu_seqlens_q=c.cu_seqlens, cu_seqlens_k=c.cu_seqlens)
    check_against(run_gpu(c), oref)


def test_sliding_window_kernel_wait_runs_out():
    """The sliding-window forward (G = 2, W = 64: items of 64 tokens x 2 heads,
    one per CTA here): K of each CTA's first item is withheld, so every CTA's
    products wait for it; the call gives up with a 0x1xx timeout and the next
    call is clean and matches the oracle."""
    Lt = binding.load_library(build(test=True))
    dev = torch.device("cuda:0")
    w = small_workload("timeout_band", 954, 4, 2, [512, 300], causal=True, window=64)
    c = make_case(w)
    t = {n: getattr(c, n).to(dev) for n in ("q", "k", "v", "dout", "sink")}
    cu = torch.tensor(c.cu_seqlens, dtype=torch.int32, device=dev)
    p = binding.make_params(c.q.shape, c.k.shape, causal=True, window=64, softmax_scale=w.scale,
                            num_seqs=len(c.lengths), max_seqlen_q=max(c.lengths),
                            max_seqlen_k=max(c.lengths))
    stream = torch.cuda.current_stream().cuda_stream
    out, res = torch.empty_like(t["q"]), torch.empty_like(t["q"])
    lse = torch.empty((t["q"].shape[1], t["q"].shape[0]), dtype=torch.float32, device=dev)
    fws = torch.empty(max(Lt.attn_sink_fwd_workspace_size(ctypes.byref(p)), 1),
                      dtype=torch.uint8, device=dev)
    assert Lt.attn_sink_test_withhold(0, -1) == 0
    t0 = time.perf_counter()
    assert _fwd(Lt, p, t, cu, out, res, lse, fws, stream) == 0
    st, code = _device_error(Lt, stream)
    elapsed = time.perf_counter() - t0
    assert st == TIMEOUT and code & 0xF00 == 0x100, (st, hex(code))
    assert elapsed < 1.0, f"the forward took {elapsed:.3f} s to give up"
    assert Lt.attn_sink_test_withhold(-1, -1) == 0
    assert _fwd(Lt, p, t, cu, out, res, lse, fws, stream) == 0
    assert _device_error(Lt, stream) == (0, 0)
    ref = oracle_bwd(c.q, c.k, c.v, c.sink, c.dout, scale=w.scale, causal=True, window=64,
                     cu_seqlens_q=c.cu_seqlens, cu_seqlens_k=c.cu_seqlens)
    check_against({"out": out.cpu(), "out_res": res.cpu(), "lse": lse.cpu()}, ref)
