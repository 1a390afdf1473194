"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and compare with the float64 oracle element by element.

Tolerances (bf16 inputs, fp32 accumulation), applied to the raw error:
  out, dq, dk, dv : max |err| <= 2e-2 and ||err||_F / ||ref||_F <= 5e-3
  dsink           : ||err||_2 / ||ref||_2 <= 1e-2 over the heads checked
  lse             : max |err| <= 1e-3 (natural log)

Which stored form each bar is applied to:
  * out: the near-fp32 value out + out_residual (the forward's bf16 result and
    its bf16 rounding residual), and the bf16 out by itself;
  * dq, dk, dv: the fp32 gradients (grad_dtype = 1) of every case, and the
    bf16 gradients (grad_dtype = 0) wherever the reference stays below 8 in
    magnitude.  At |x| >= 8 half a bf16 ulp is 0.031, above the 2e-2 bar, so a
    bf16 store cannot meet it whatever the kernel computes; there the fp32
    gradients carry the check and the bf16 store is only checked to lie
    within its own rounding of the bar (reported as such).
Every comparison is recorded (max |err|, rel-Frobenius, max |ref|) and printed
in the pytest terminal summary.
"""
from __future__ import annotations

import os

import torch

from attention_learnable_head_gb300 import binding
from attention_learnable_head_gb300.inputs import Case

TOL_MAX_ABS = 2e-2
TOL_REL_FRO = 5e-3
TOL_DSINK = 1e-2
TOL_LSE = 1e-3
BF16_RAW_LIMIT = 8.0     # |ref| at which half a bf16 ulp (2^-5) exceeds the max-abs bar

# (test id, tensor, form, max_abs, rel_fro, max_ref) of every comparison made
REPORT: list[tuple] = []


def _test_id() -> str:
    cur = os.environ.get("PYTEST_CURRENT_TEST", "")
    return cur.split(" ")[0].split("::")[-1] if cur else "?"


def err_stats(got: torch.Tensor, ref: torch.Tensor):
    """(max |got - ref|, ||got - ref||_F / ||ref||_F) over the entries the
    reference computed.  The relative error of an all-zero reference is
    undefined: it is returned as None and only the absolute bar applies (e.g.
    the gradients of a window of one key with the sink at -inf, where every
    row's single probability is exactly 1 and dS = 0)."""
    got = got.double().cpu()
    ref = ref.double().cpu()
    mask = ~torch.isnan(ref)
    d = (got - ref)[mask]
    r = ref[mask]
    max_abs = d.abs().max().item() if d.numel() else 0.0
    rel = (d.norm() / r.norm()).item() if r.numel() and r.norm() > 0 else None
    return max_abs, rel


def max_ref(ref: torch.Tensor) -> float:
    r = ref.double().cpu()
    r = r[~torch.isnan(r)]
    return r.abs().max().item() if r.numel() else 0.0


def bf16_half_ulp(ref: torch.Tensor) -> torch.Tensor:
    """Half a bf16 ulp at |ref|: the rounding any bf16-stored result carries."""
    a = ref.abs().clamp_min(2.0 ** -126)
    return torch.exp2(torch.floor(torch.log2(a)) - 8)


def assert_close(name, got, ref, max_abs=TOL_MAX_ABS, rel_fro=TOL_REL_FRO, form="raw"):
    """max |got - ref| <= max_abs and relative Frobenius error <= rel_fro, on the
    raw error (no allowance of any kind)."""
    a, r = err_stats(got, ref)
    REPORT.append((_test_id(), name, form, a, r, max_ref(ref)))
    assert a <= max_abs and (r is None or r <= rel_fro), (
        f"{name} ({form}): max abs {a:.3e} (<= {max_abs}), rel fro {r} (<= {rel_fro}), "
        f"max |ref| {max_ref(ref):.3g}")
    return a, r


def assert_close_bf16_store(name, got, ref):
    """A bf16-stored result whose reference reaches |x| >= 8: the 2e-2 bar is
    applied to the error beyond the storage rounding (half a bf16 ulp of the
    reference).  Only used next to the raw check of the fp32 form."""
    a, r = err_stats(got, ref)
    g, rr = got.double().cpu(), ref.double().cpu()
    m = ~torch.isnan(rr)
    excess = ((g - rr).abs() - bf16_half_ulp(rr))[m]
    a_eff = max(0.0, excess.max().item()) if excess.numel() else 0.0
    REPORT.append((_test_id(), name, "bf16 store beyond its rounding", a, r, max_ref(ref)))
    assert a_eff <= TOL_MAX_ABS and (r is None or r <= TOL_REL_FRO), (
        f"{name} (bf16 store): max abs {a:.3e} (beyond storage rounding {a_eff:.3e}), "
        f"rel fro {r}")
    return a, r


def run_gpu(case: Case, *, grad_dtype: int = 0, with_bwd: bool = True, dense: bool = False,
            cu_q=None, cu_k=None, q=None, k=None, v=None, dout=None, residual: bool = True,
            deterministic: bool = False):
    """Forward (+ backward) of a seeded case on cuda:0 through the C ABI.

    With grad_dtype = 0 the backward runs twice, once with bf16 and once with
    fp32 gradients (keys dq/dk/dv and dq_f32/dk_f32/dv_f32); with grad_dtype = 1
    only with fp32 gradients (dq/dk/dv).  out_res is the residual of out."""
    dev = torch.device("cuda:0")
    w = case.workload
    q = (case.q if q is None else q).to(dev)
    k = (case.k if k is None else k).to(dev)
    v = (case.v if v is None else v).to(dev)
    do = (case.dout if dout is None else dout).to(dev)
    sink = case.sink.to(dev)
    cq = case.cu_seqlens if cu_q is None else cu_q
    ck = case.cu_seqlens if cu_k is None else cu_k
    dtypes = [grad_dtype] if grad_dtype == 1 else [0, 1]
    if dense:
        b = len(cq) - 1
        n = cq[1]
        nk = ck[1]
        qa, doa = q.view(b, n, *q.shape[1:]), do.view(b, n, *do.shape[1:])
        ka, va = k.view(b, nk, *k.shape[1:]), v.view(b, nk, *v.shape[1:])
        kw = dict(causal=w.causal, window=w.window, softmax_scale=w.scale)
    else:
        tq = torch.tensor(cq, dtype=torch.int32, device=dev)
        tk = torch.tensor(ck, dtype=torch.int32, device=dev)
        lq = [cq[i + 1] - cq[i] for i in range(len(cq) - 1)]
        lk = [ck[i + 1] - ck[i] for i in range(len(ck) - 1)]
        qa, ka, va, doa = q, k, v, do
        kw = dict(causal=w.causal, window=w.window, softmax_scale=w.scale, cu_seqlens_q=tq,
                  cu_seqlens_k=tk, max_seqlen_q=max(lq + [0]), max_seqlen_k=max(lk + [0]))
    out, lse, ores = binding.forward(qa, ka, va, sink, residual=residual, **kw)
    res = dict(out=out.reshape(q.shape), lse=lse)
    if ores is not None:
        res["out_res"] = ores.reshape(q.shape)
    if with_bwd:
        for gd in dtypes:
            dq, dk, dv, dsink = binding.backward(qa, ka, va, sink, out, lse, doa,
                                                 out_residual=ores, grad_dtype=gd,
                                                 deterministic=deterministic, **kw)
            sfx = "_f32" if (gd == 1 and len(dtypes) == 2) else ""
            res.update({"dq" + sfx: dq.reshape(q.shape), "dk" + sfx: dk.reshape(k.shape),
                        "dv" + sfx: dv.reshape(v.shape)})
            if not sfx:
                res["dsink"] = dsink
    torch.cuda.synchronize()
    st, code = binding.attn_sink_device_error()
    assert st == 0 and code == 0, f"device error word {code:#x}"
    return {k2: v2.cpu() for k2, v2 in res.items()}


def check_tensor(res: dict, ref: torch.Tensor, name: str, sel=(slice(None),)):
    """The checks of one of out / dq / dk / dv (see the module docstring) on
    res[name][sel] against ref (already restricted to sel)."""
    got = res[name][sel]
    out = {}
    if name == "out" and "out_res" in res:
        hi = got.double() + res["out_res"][sel].double()
        out["out+res"] = assert_close("out+res", hi, ref)
    f32 = res.get(name + "_f32")
    if f32 is not None:
        out[name + "_f32"] = assert_close(name + "_f32", f32[sel], ref)
    if got.dtype == torch.float32 or max_ref(ref) < BF16_RAW_LIMIT:
        out[name] = assert_close(name, got, ref)
    else:
        if name != "out" and f32 is None:
            raise AssertionError(f"{name}: bf16 store with |ref| >= {BF16_RAW_LIMIT} and no "
                                 "fp32 gradients to check against the raw bar")
        out[name] = assert_close_bf16_store(name, got, ref)
    return out


def check_against(res: dict, ref: dict, heads=None, kv_heads=None, rows=None, report=None):
    """Compare GPU results with oracle results (NaN in the oracle = not computed)."""
    out = {}
    hsel = slice(None) if heads is None else heads
    ksel = slice(None) if kv_heads is None else kv_heads
    for name in ("out", "dq", "dk", "dv"):
        if name in res and name in ref:
            sel = (slice(None), hsel) if name in ("out", "dq") else (slice(None), ksel)
            out.update(check_tensor(res, ref[name][sel], name, sel))
    if "lse" in res:
        a, _ = err_stats(res["lse"][hsel], ref["lse"][hsel])
        REPORT.append((_test_id(), "lse", "raw", a, None, max_ref(ref["lse"][hsel])))
        assert a <= TOL_LSE, f"lse max abs {a:.3e}"
        out["lse"] = (a, None)
    if "dsink" in res and "dsink" in ref:
        g, r = res["dsink"].double()[hsel], ref["dsink"][hsel]
        m = ~torch.isnan(r)
        rel = ((g[m] - r[m]).norm() / r[m].norm().clamp_min(1e-30)).item()
        REPORT.append((_test_id(), "dsink", "rel L2", None, rel, max_ref(r)))
        assert rel <= TOL_DSINK, f"dsink rel {rel:.3e}: got {g[m][:8]} ref {r[m][:8]}"
        out["dsink"] = (rel, None)
    if report is not None:
        report.update(out)
    return out


def format_report(rows=REPORT) -> list[str]:
    """One line per comparison of the full-size workloads, then, per tensor and
    form, the worst case over every other test."""
    lines = []
    worst = {}
    for tid, name, form, a, r, mr in rows:
        if tid.startswith("test_") and any(w in tid for w in
                                           ("gptoss_full", "swa", "varlen", "long_")):
            lines.append(f"{tid:22s} {name:9s} {form:14s} max_abs={_f(a)} rel_fro={_f(r)} "
                         f"max|ref|={_f(mr)}")
        else:
            key = (name, form)
            cur = worst.get(key, (0.0, 0.0, 0.0, ""))
            worst[key] = (max(cur[0], a or 0.0), max(cur[1], r or 0.0), max(cur[2], mr or 0.0),
                          tid if (a or 0.0) >= cur[0] else cur[3])
    for (name, form), (a, r, mr, tid) in sorted(worst.items()):
        lines.append(f"{'(other tests, worst)':22s} {name:9s} {form:14s} max_abs={_f(a)} "
                     f"rel_fro={_f(r)} max|ref|={_f(mr)} [{tid}]")
    return lines


def _f(x):
    return "   -    " if x is None else f"{x:.2e}"
