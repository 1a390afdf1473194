"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and compare with the float64 oracle element by element.

Tolerances (bf16 inputs, fp32 accumulation):
  out, dq, dk, dv : max |err| <= 2e-2 and ||err||_F / ||ref||_F <= 5e-3
                    (for bf16-stored results the max-abs bar is taken beyond
                    the half-ulp rounding of the bf16 store itself)
  dsink           : ||err||_2 / ||ref||_2 <= 1e-2 over the heads checked
  lse             : max |err| <= 1e-3 (natural log)
"""
from __future__ import annotations

import torch

from attention_learnable_head_gb300 import binding
from attention_learnable_head_gb300.inputs import Case

TOL_MAX_ABS = 2e-2
TOL_REL_FRO = 5e-3
TOL_DSINK = 1e-2
TOL_LSE = 1e-3


def err_stats(got: torch.Tensor, ref: torch.Tensor):
    got = got.double().cpu()
    ref = ref.double().cpu()
    mask = ~torch.isnan(ref)
    d = (got - ref)[mask]
    r = ref[mask]
    max_abs = d.abs().max().item() if d.numel() else 0.0
    rel = (d.norm() / r.norm()).item() if r.numel() and r.norm() > 0 else d.norm().item()
    return max_abs, rel


def bf16_half_ulp(ref: torch.Tensor) -> torch.Tensor:
    """Half a bf16 ulp at |ref|: the rounding any bf16-stored result carries."""
    a = ref.abs().clamp_min(2.0 ** -126)
    return torch.exp2(torch.floor(torch.log2(a)) - 8)


def assert_close(name, got, ref, max_abs=TOL_MAX_ABS, rel_fro=TOL_REL_FRO):
    """max |got - ref| <= max_abs and relative Frobenius error <= rel_fro.

    For a bf16-stored result the max-abs bar is taken on top of the storage
    rounding (half a bf16 ulp of the reference value); fp32-stored results
    meet the bar as it stands."""
    a, r = err_stats(got, ref)
    if got.dtype == torch.bfloat16:
        g, rr = got.double().cpu(), ref.double().cpu()
        m = ~torch.isnan(rr)
        excess = ((g - rr).abs() - bf16_half_ulp(rr))[m]
        a_eff = max(0.0, excess.max().item()) if excess.numel() else 0.0
    else:
        a_eff = a
    assert a_eff <= max_abs and r <= rel_fro, (
        f"{name}: max abs {a:.3e} (beyond storage rounding {a_eff:.3e}, <= {max_abs}), "
        f"rel fro {r:.3e} (<= {rel_fro})")
    return a, r


def run_gpu(case: Case, *, grad_dtype: int = 0, with_bwd: bool = True, dense: bool = False,
            cu_q=None, cu_k=None, q=None, k=None, v=None, dout=None, residual: bool = True,
            deterministic: bool = False):
    """Forward (+ backward) of a seeded case on cuda:0 through the C ABI."""
    dev = torch.device("cuda:0")
    w = case.workload
    q = (case.q if q is None else q).to(dev)
    k = (case.k if k is None else k).to(dev)
    v = (case.v if v is None else v).to(dev)
    do = (case.dout if dout is None else dout).to(dev)
    sink = case.sink.to(dev)
    cq = case.cu_seqlens if cu_q is None else cu_q
    ck = case.cu_seqlens if cu_k is None else cu_k
    if dense:
        b = len(cq) - 1
        n = cq[1]
        nk = ck[1]
        q4, do4 = q.view(b, n, *q.shape[1:]), do.view(b, n, *do.shape[1:])
        k4, v4 = k.view(b, nk, *k.shape[1:]), v.view(b, nk, *v.shape[1:])
        kw = dict(causal=w.causal, window=w.window, softmax_scale=w.scale)
        out, lse, ores = binding.forward(q4, k4, v4, sink, residual=residual, **kw)
        res = dict(out=out.view(q.shape), lse=lse)
        if with_bwd:
            dq, dk, dv, dsink = binding.backward(q4, k4, v4, sink, out, lse, do4,
                                                 out_residual=ores, grad_dtype=grad_dtype,
                                                 deterministic=deterministic, **kw)
            res.update(dq=dq.view(q.shape), dk=dk.view(k.shape), dv=dv.view(v.shape), dsink=dsink)
    else:
        tq = torch.tensor(cq, dtype=torch.int32, device=dev)
        tk = torch.tensor(ck, dtype=torch.int32, device=dev)
        lq = [cq[i + 1] - cq[i] for i in range(len(cq) - 1)]
        lk = [ck[i + 1] - ck[i] for i in range(len(ck) - 1)]
        kw = dict(causal=w.causal, window=w.window, softmax_scale=w.scale, cu_seqlens_q=tq,
                  cu_seqlens_k=tk, max_seqlen_q=max(lq + [0]), max_seqlen_k=max(lk + [0]))
        out, lse, ores = binding.forward(q, k, v, sink, residual=residual, **kw)
        res = dict(out=out, lse=lse)
        if with_bwd:
            dq, dk, dv, dsink = binding.backward(q, k, v, sink, out, lse, do,
                                                 out_residual=ores, grad_dtype=grad_dtype,
                                                 deterministic=deterministic, **kw)
            res.update(dq=dq, dk=dk, dv=dv, dsink=dsink)
    torch.cuda.synchronize()
    st, code = binding.attn_sink_device_error()
    assert st == 0 and code == 0, f"device error word {code:#x}"
    return {k2: v2.cpu() for k2, v2 in res.items()}


def check_against(res: dict, ref: dict, heads=None, kv_heads=None, rows=None, report=None):
    """Compare GPU results with oracle results (NaN in the oracle = not computed)."""
    out = {}
    hsel = slice(None) if heads is None else heads
    for name in ("out", "dq"):
        if name in res and name in ref:
            g, r = res[name][:, hsel], ref[name][:, hsel]
            out[name] = assert_close(name, g, r)
    for name in ("dk", "dv"):
        if name in res and name in ref:
            ksel = slice(None) if kv_heads is None else kv_heads
            out[name] = assert_close(name, res[name][:, ksel], ref[name][:, ksel])
    if "lse" in res:
        a, _ = err_stats(res["lse"][hsel], ref["lse"][hsel])
        assert a <= TOL_LSE, f"lse max abs {a:.3e}"
        out["lse"] = (a, None)
    if "dsink" in res and "dsink" in ref:
        g, r = res["dsink"].double()[hsel], ref["dsink"][hsel]
        m = ~torch.isnan(r)
        rel = ((g[m] - r[m]).norm() / r[m].norm().clamp_min(1e-30)).item()
        assert rel <= TOL_DSINK, f"dsink rel {rel:.3e}: got {g[m][:8]} ref {r[m][:8]}"
        out["dsink"] = (rel, None)
    if report is not None:
        report.update(out)
    return out
