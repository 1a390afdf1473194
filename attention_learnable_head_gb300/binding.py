"""ctypes binding of libattn_sink.so.

``attn_sink_fwd``, ``attn_sink_bwd``, ``attn_sink_fwd_workspace_size``,
``attn_sink_bwd_workspace_size``,
``attn_sink_status_string``, ``attn_sink_device_error``,
``attn_sink_launch_count``, ``attn_sink_last_cuda_error``,
``attn_sink_kernel_timing``, ``attn_sink_kernel_time``, ``attn_sink_fwd_chunk``,
``attn_sink_merge``, ``attn_sink_bwd_deterministic``, ``attn_sink_decode``,
``attn_sink_decode_workspace_size``, ``attn_sink_fwd_ex``, ``attn_sink_bwd_ex`` and
``attn_sink_fwd_noalloc`` mirror the C entry
points of ``include/attn_sink.h`` one to one: they only turn tensors into
device pointers and return the library's status.  ``forward``, ``backward``
and ``attn_sink`` (autograd) are conveniences on top that allocate outputs and
the workspace with torch and raise on a non-zero status.  Every step of the
computation runs in the library's CUDA kernels; there is no other code path,
and loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import math
import os
import re

import torch

from .build import LIB_PATH, INCLUDE

c_int, c_float, c_void_p, c_size_t = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t

ATTN_SINK_OK = 0
STATUS_NAMES = {0: "ATTN_SINK_OK", 1: "ATTN_SINK_ERR_INVALID_ARG", 2: "ATTN_SINK_ERR_UNSUPPORTED",
                3: "ATTN_SINK_ERR_WORKSPACE", 4: "ATTN_SINK_ERR_CUDA", 5: "ATTN_SINK_ERR_TIMEOUT"}


class AttnSinkParams(ctypes.Structure):
    """Mirror of ``attn_sink_params`` in include/attn_sink.h (field order matters)."""
    _fields_ = [
        ("batch", c_int), ("seqlen_q", c_int), ("seqlen_k", c_int),
        ("num_seqs", c_int), ("total_q", c_int), ("total_k", c_int),
        ("max_seqlen_q", c_int), ("max_seqlen_k", c_int),
        ("heads_q", c_int), ("heads_kv", c_int), ("head_dim", c_int),
        ("causal", c_int), ("window", c_int), ("softmax_scale", c_float),
        ("grad_dtype", c_int),
    ]


class AttnSinkDecodeParams(ctypes.Structure):
    """Mirror of ``attn_sink_decode_params`` in include/attn_sink.h."""
    _fields_ = [
        ("batch", c_int), ("heads_q", c_int), ("heads_kv", c_int), ("head_dim", c_int),
        ("page_size", c_int), ("num_pages", c_int), ("max_pages", c_int), ("window", c_int),
        ("softmax_scale", c_float),
    ]


class AttnSinkError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        extra = ""
        if status == 4:
            extra = f", last CUDA error {attn_sink_last_cuda_error()}"
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} "
                         f"({attn_sink_status_string(status)}{extra})")


_LIB = None


def header_functions() -> list[str]:
    """Names of the functions include/attn_sink.h declares."""
    text = open(os.path.join(INCLUDE, "attn_sink.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^(?:[A-Za-z_]\w*[\s*]+)+(attn_sink_\w+)\s*\(", text, flags=re.M)


def lib():
    """Load libattn_sink.so (built in-tree by ``build.build()``)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` (nvcc, sm_103a)")
    _LIB = load_library(LIB_PATH)
    return _LIB


def load_library(path: str):
    """A ctypes handle on a build of the library at `path` with the C
    signatures of include/attn_sink.h attached (the product library, or the
    test build that also exports attn_sink_test_withhold)."""
    L = ctypes.CDLL(path)
    P = ctypes.POINTER(AttnSinkParams)
    L.attn_sink_fwd.argtypes = [P, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                c_void_p, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]
    L.attn_sink_fwd_workspace_size.argtypes = [P]
    L.attn_sink_fwd_workspace_size.restype = c_size_t
    L.attn_sink_fwd_noalloc.argtypes = [P, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                        c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
    L.attn_sink_fwd_noalloc.restype = c_int
    L.attn_sink_fwd.restype = c_int
    L.attn_sink_fwd_chunk.argtypes = [P, c_int, c_void_p, c_void_p, c_void_p, c_void_p,
                                      c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                      c_void_p]
    L.attn_sink_fwd_chunk.restype = c_int
    L.attn_sink_merge.argtypes = [c_int, c_int, c_int, c_int, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_void_p, c_void_p, c_void_p, c_void_p]
    L.attn_sink_merge.restype = c_int
    PD = ctypes.POINTER(AttnSinkDecodeParams)
    L.attn_sink_decode_workspace_size.argtypes = [PD]
    L.attn_sink_decode_workspace_size.restype = c_size_t
    L.attn_sink_decode.argtypes = [PD, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                   c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_size_t,
                                   c_void_p]
    L.attn_sink_decode.restype = c_int
    L.attn_sink_bwd_workspace_size.argtypes = [P]
    L.attn_sink_bwd_workspace_size.restype = c_size_t
    L.attn_sink_bwd.argtypes = [P, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p,
                                c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]
    L.attn_sink_bwd.restype = c_int
    L.attn_sink_bwd_deterministic.argtypes = L.attn_sink_bwd.argtypes
    L.attn_sink_bwd_deterministic.restype = c_int
    L.attn_sink_fwd_ex.argtypes = [P, c_int] + L.attn_sink_fwd.argtypes[1:]
    L.attn_sink_fwd_ex.restype = c_int
    L.attn_sink_bwd_ex.argtypes = [P, c_int] + L.attn_sink_bwd.argtypes[1:]
    L.attn_sink_bwd_ex.restype = c_int
    L.attn_sink_status_string.argtypes = [c_int]
    L.attn_sink_status_string.restype = ctypes.c_char_p
    L.attn_sink_device_error.argtypes = [c_void_p, ctypes.POINTER(c_int)]
    L.attn_sink_device_error.restype = c_int
    L.attn_sink_last_cuda_error.argtypes = []
    L.attn_sink_last_cuda_error.restype = c_int
    L.attn_sink_launch_count.argtypes = []
    L.attn_sink_launch_count.restype = ctypes.c_ulonglong
    L.attn_sink_kernel_timing.argtypes = [c_int]
    L.attn_sink_kernel_timing.restype = c_int
    L.attn_sink_kernel_time.argtypes = [c_int, ctypes.POINTER(ctypes.c_double),
                                        ctypes.POINTER(ctypes.c_ulonglong)]
    L.attn_sink_kernel_time.restype = c_int
    if hasattr(L, "attn_sink_test_withhold"):
        L.attn_sink_test_withhold.argtypes = [c_int, c_int]
        L.attn_sink_test_withhold.restype = c_int
    return L


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _pref(params):
    return None if params is None else ctypes.byref(params)


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------------------------- C entry points
def attn_sink_fwd(params: AttnSinkParams, q, k, v, sink, cu_seqlens_q, cu_seqlens_k, out,
                  out_residual, lse, workspace, workspace_bytes: int, stream=None) -> int:
    return lib().attn_sink_fwd(_pref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(sink),
                               _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(out),
                               _ptr(out_residual), _ptr(lse), _ptr(workspace),
                               int(workspace_bytes), _stream(stream))


ATTN_SINK_FLAG_SINK_BF16 = 1
ATTN_SINK_FLAG_ACCUMULATE_DSINK = 2
ATTN_SINK_FLAG_DETERMINISTIC = 4


def attn_sink_fwd_ex(params: AttnSinkParams, flags: int, q, k, v, sink, cu_seqlens_q,
                     cu_seqlens_k, out, out_residual, lse, workspace, workspace_bytes: int,
                     stream=None) -> int:
    return lib().attn_sink_fwd_ex(_pref(params), int(flags), _ptr(q), _ptr(k), _ptr(v),
                                  _ptr(sink), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(out),
                                  _ptr(out_residual), _ptr(lse), _ptr(workspace),
                                  int(workspace_bytes), _stream(stream))


def attn_sink_bwd_ex(params: AttnSinkParams, flags: int, q, k, v, sink, cu_seqlens_q,
                     cu_seqlens_k, out, out_residual, lse, dout, dq, dk, dv, dsink, workspace,
                     workspace_bytes: int, stream=None) -> int:
    return lib().attn_sink_bwd_ex(_pref(params), int(flags), _ptr(q), _ptr(k), _ptr(v),
                                  _ptr(sink), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(out),
                                  _ptr(out_residual), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                  _ptr(dv), _ptr(dsink), _ptr(workspace), int(workspace_bytes),
                                  _stream(stream))


def attn_sink_fwd_chunk(params: AttnSinkParams, q_pos0: int, q, k, v, cu_seqlens_q,
                        cu_seqlens_k, out, out_residual, lse, workspace, workspace_bytes: int,
                        stream=None) -> int:
    return lib().attn_sink_fwd_chunk(_pref(params), int(q_pos0), _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(out),
                                     _ptr(out_residual), _ptr(lse), _ptr(workspace),
                                     int(workspace_bytes), _stream(stream))


def attn_sink_merge(num_chunks: int, total_q: int, heads_q: int, head_dim: int, o_parts,
                    o_residual_parts, lse_parts, sink, out, out_residual, lse,
                    stream=None) -> int:
    return lib().attn_sink_merge(int(num_chunks), int(total_q), int(heads_q), int(head_dim),
                                 _ptr(o_parts), _ptr(o_residual_parts), _ptr(lse_parts),
                                 _ptr(sink), _ptr(out), _ptr(out_residual), _ptr(lse),
                                 _stream(stream))


def attn_sink_decode_workspace_size(params: AttnSinkDecodeParams) -> int:
    return int(lib().attn_sink_decode_workspace_size(
        None if params is None else ctypes.byref(params)))


def attn_sink_decode(params: AttnSinkDecodeParams, q, k_cache, v_cache, block_table, seq_lens,
                     sink, out, out_residual, lse, workspace, workspace_bytes: int,
                     stream=None) -> int:
    return lib().attn_sink_decode(None if params is None else ctypes.byref(params), _ptr(q),
                                  _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
                                  _ptr(seq_lens), _ptr(sink), _ptr(out), _ptr(out_residual),
                                  _ptr(lse), _ptr(workspace), int(workspace_bytes),
                                  _stream(stream))


def make_decode_params(q_shape, cache_shape, max_pages: int, *, window: int = 0,
                       softmax_scale: float | None = None) -> AttnSinkDecodeParams:
    """Params from q [B, H_q, d] and a cache [num_pages, page_size, H_kv, d]."""
    p = AttnSinkDecodeParams()
    p.batch, p.heads_q, p.head_dim = int(q_shape[0]), int(q_shape[1]), int(q_shape[2])
    p.num_pages, p.page_size, p.heads_kv = (int(cache_shape[0]), int(cache_shape[1]),
                                            int(cache_shape[2]))
    p.max_pages = int(max_pages)
    p.window = int(window)
    p.softmax_scale = float(softmax_scale if softmax_scale is not None
                            else 1.0 / math.sqrt(p.head_dim))
    return p


def decode(q, k_cache, v_cache, block_table, seq_lens, sink, *, window: int = 0,
           softmax_scale: float | None = None, residual: bool = False, stream=None):
    """(out, lse, out_residual) of one decode step over a paged cache
    (attn_sink_decode): q [B, H_q, 64], caches [pages, page_size, H_kv, 64],
    block_table [B, max_pages] int32, seq_lens [B] int32."""
    p = make_decode_params(q.shape, k_cache.shape, block_table.shape[1], window=window,
                           softmax_scale=softmax_scale)
    out = torch.empty_like(q)
    res = torch.empty_like(q) if residual else None
    lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    nbytes = attn_sink_decode_workspace_size(p)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    _check(attn_sink_decode(p, q, k_cache, v_cache, block_table, seq_lens, sink, out, res, lse,
                            ws, ws.numel(), stream), "attn_sink_decode")
    return out, lse, res


# Bytes of the static scratch behind attn_sink_fwd_noalloc (the header's
# ATTN_SINK_NOALLOC_SCRATCH_BYTES).
ATTN_SINK_NOALLOC_SCRATCH_BYTES = 16 << 20


def attn_sink_fwd_noalloc(params: AttnSinkParams, q, k, v, sink, cu_seqlens_q, cu_seqlens_k, out,
                          out_residual, lse, stream=None) -> int:
    """Forward for callers that cannot allocate device memory: the library's
    own static scratch replaces the workspace (see include/attn_sink.h)."""
    return lib().attn_sink_fwd_noalloc(_pref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(sink),
                                       _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(out),
                                       _ptr(out_residual), _ptr(lse), _stream(stream))


def attn_sink_fwd_workspace_size(params: AttnSinkParams) -> int:
    return int(lib().attn_sink_fwd_workspace_size(_pref(params)))


def attn_sink_bwd_workspace_size(params: AttnSinkParams) -> int:
    return int(lib().attn_sink_bwd_workspace_size(_pref(params)))


def attn_sink_bwd(params: AttnSinkParams, q, k, v, sink, cu_seqlens_q, cu_seqlens_k, out,
                  out_residual, lse, dout, dq, dk, dv, dsink, workspace, workspace_bytes: int,
                  stream=None) -> int:
    return lib().attn_sink_bwd(_pref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(sink),
                               _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(out),
                               _ptr(out_residual), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                               _ptr(dv), _ptr(dsink), _ptr(workspace), int(workspace_bytes),
                               _stream(stream))


def attn_sink_bwd_deterministic(params: AttnSinkParams, q, k, v, sink, cu_seqlens_q, cu_seqlens_k, out,
                  out_residual, lse, dout, dq, dk, dv, dsink, workspace, workspace_bytes: int,
                  stream=None) -> int:
    return lib().attn_sink_bwd_deterministic(_pref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(sink),
                               _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), _ptr(out),
                               _ptr(out_residual), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                               _ptr(dv), _ptr(dsink), _ptr(workspace), int(workspace_bytes),
                               _stream(stream))


def attn_sink_status_string(status: int) -> str:
    return lib().attn_sink_status_string(int(status)).decode()


def attn_sink_last_cuda_error() -> int:
    return int(lib().attn_sink_last_cuda_error())


def attn_sink_launch_count() -> int:
    return int(lib().attn_sink_launch_count())


ATTN_SINK_KERNEL_FWD = 0
ATTN_SINK_KERNEL_BWD_MAIN = 1
ATTN_SINK_KERNEL_BWD_DQ = 2
ATTN_SINK_KERNEL_MERGE = 3


def attn_sink_kernel_timing(on: bool) -> int:
    return int(lib().attn_sink_kernel_timing(1 if on else 0))


def attn_sink_kernel_time(kernel: int) -> tuple[int, float, int]:
    """(status, summed milliseconds, launches) of `kernel` since its last read."""
    ms = ctypes.c_double(0.0)
    n = ctypes.c_ulonglong(0)
    st = lib().attn_sink_kernel_time(int(kernel), ctypes.byref(ms), ctypes.byref(n))
    return int(st), float(ms.value), int(n.value)


def attn_sink_device_error(stream=None) -> tuple[int, int]:
    code = c_int(0)
    st = lib().attn_sink_device_error(_stream(stream), ctypes.byref(code))
    return st, code.value


# ----------------------------------------------------------------------------- conveniences
def make_params(q_shape, k_shape, *, causal: bool, window: int, softmax_scale: float | None,
                num_seqs: int | None = None, max_seqlen_q: int | None = None,
                max_seqlen_k: int | None = None, grad_dtype: int = 0) -> AttnSinkParams:
    """Params from tensor shapes: q [B, N, H, d] (dense) or [T, H, d] (packed;
    then num_seqs and max_seqlen_* are required)."""
    p = AttnSinkParams()
    d = int(q_shape[-1])
    p.head_dim = d
    p.heads_q = int(q_shape[-2])
    p.heads_kv = int(k_shape[-2])
    p.causal = int(bool(causal))
    p.window = int(window)
    p.softmax_scale = float(softmax_scale if softmax_scale is not None else 1.0 / math.sqrt(d))
    p.grad_dtype = int(grad_dtype)
    if len(q_shape) == 4:
        p.batch, p.seqlen_q, p.seqlen_k = int(q_shape[0]), int(q_shape[1]), int(k_shape[1])
    else:
        if num_seqs is None or max_seqlen_q is None or max_seqlen_k is None:
            raise ValueError("packed inputs need num_seqs and max_seqlen_q / max_seqlen_k")
        p.num_seqs = int(num_seqs)
        p.total_q, p.total_k = int(q_shape[0]), int(k_shape[0])
        p.max_seqlen_q, p.max_seqlen_k = int(max_seqlen_q), int(max_seqlen_k)
    return p


def _check(status: int, where: str):
    if status != ATTN_SINK_OK:
        raise AttnSinkError(status, where)


def _lse_len(q) -> int:
    return q.shape[0] * q.shape[1] if q.dim() == 4 else q.shape[0]


def forward(q, k, v, sink, *, causal: bool = True, window: int = 0,
            softmax_scale: float | None = None, cu_seqlens_q=None, cu_seqlens_k=None,
            max_seqlen_q: int | None = None, max_seqlen_k: int | None = None,
            residual: bool = True, stream=None):
    """(out, lse, out_residual): out like q (bf16), lse [H_q, T_q] fp32, and the
    bf16 rounding residual of out (None when residual=False)."""
    num_seqs = None if cu_seqlens_q is None else cu_seqlens_q.numel() - 1
    p = make_params(q.shape, k.shape, causal=causal, window=window, softmax_scale=softmax_scale,
                    num_seqs=num_seqs, max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k)
    out = torch.empty_like(q)
    res = torch.empty_like(q) if residual else None
    lse = torch.empty((q.shape[-2], _lse_len(q)), dtype=torch.float32, device=q.device)
    nbytes = attn_sink_fwd_workspace_size(p)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    if sink.dtype == torch.bfloat16:      # a bf16 sink parameter, read exactly
        _check(attn_sink_fwd_ex(p, ATTN_SINK_FLAG_SINK_BF16, q, k, v, sink, cu_seqlens_q,
                                cu_seqlens_k, out, res, lse, ws, ws.numel(), stream),
               "attn_sink_fwd_ex")
    else:
        _check(attn_sink_fwd(p, q, k, v, sink, cu_seqlens_q, cu_seqlens_k, out, res, lse, ws,
                             ws.numel(), stream), "attn_sink_fwd")
    return out, lse, res


def forward_chunk(q, k, v, q_pos0: int, *, causal: bool = True, window: int = 0,
                  softmax_scale: float | None = None, cu_seqlens_q=None, cu_seqlens_k=None,
                  max_seqlen_q: int | None = None, max_seqlen_k: int | None = None,
                  residual: bool = True, stream=None):
    """(out, lse, out_residual) of the queries over one key chunk, without the
    sink (attn_sink_fwd_chunk); k, v hold the chunk's keys."""
    num_seqs = None if cu_seqlens_q is None else cu_seqlens_q.numel() - 1
    p = make_params(q.shape, k.shape, causal=causal, window=window, softmax_scale=softmax_scale,
                    num_seqs=num_seqs, max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k)
    out = torch.empty_like(q)
    res = torch.empty_like(q) if residual else None
    lse = torch.empty((q.shape[-2], _lse_len(q)), dtype=torch.float32, device=q.device)
    nbytes = attn_sink_fwd_workspace_size(p)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    _check(attn_sink_fwd_chunk(p, q_pos0, q, k, v, cu_seqlens_q, cu_seqlens_k, out, res, lse,
                               ws, ws.numel(), stream), "attn_sink_fwd_chunk")
    return out, lse, res


def merge(outs, lses, sink, *, residuals=None, stream=None):
    """(out, lse, out_residual) of the whole key sequence from the chunks'
    results (attn_sink_merge): outs like q, lses [H_q, T_q], residuals optional."""
    o = torch.stack(list(outs)).contiguous()
    ls = torch.stack(list(lses)).contiguous()
    r = None if residuals is None else torch.stack(list(residuals)).contiguous()
    out = torch.empty_like(o[0])
    res = torch.empty_like(o[0])
    lse = torch.empty_like(ls[0])
    heads, d = o.shape[-2], o.shape[-1]
    _check(attn_sink_merge(o.shape[0], ls.shape[-1], heads, d, o, r, ls, sink, out, res, lse,
                           stream), "attn_sink_merge")
    return out, lse, res


def backward(q, k, v, sink, out, lse, dout, *, out_residual=None, causal: bool = True,
             window: int = 0, softmax_scale: float | None = None, cu_seqlens_q=None,
             cu_seqlens_k=None, max_seqlen_q: int | None = None,
             max_seqlen_k: int | None = None, grad_dtype: int = 0, workspace=None,
             deterministic: bool = False, dsink=None, accumulate_dsink: bool = False,
             stream=None):
    """dq, dk, dv (bf16, or fp32 when grad_dtype = 1) and dsink ([H_q], the
    sink's dtype: fp32, or bf16 for a bf16 sink).
    deterministic=True: bitwise reproducible (attn_sink_bwd_deterministic);
    accumulate_dsink=True: the gradient is added into the given `dsink`."""
    num_seqs = None if cu_seqlens_q is None else cu_seqlens_q.numel() - 1
    p = make_params(q.shape, k.shape, causal=causal, window=window, softmax_scale=softmax_scale,
                    num_seqs=num_seqs, max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k,
                    grad_dtype=grad_dtype)
    gd = torch.float32 if grad_dtype == 1 else torch.bfloat16
    dq = torch.empty(q.shape, dtype=gd, device=q.device)
    dk = torch.empty(k.shape, dtype=gd, device=q.device)
    dv = torch.empty(v.shape, dtype=gd, device=q.device)
    if accumulate_dsink and dsink is None:
        raise ValueError("accumulate_dsink needs the dsink tensor to add into")
    if dsink is None:
        dsink = torch.empty_like(sink)
    nbytes = attn_sink_bwd_workspace_size(p)
    if workspace is None or workspace.numel() < nbytes:
        workspace = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=q.device)
    flags = ((ATTN_SINK_FLAG_SINK_BF16 if sink.dtype == torch.bfloat16 else 0)
             | (ATTN_SINK_FLAG_ACCUMULATE_DSINK if accumulate_dsink else 0)
             | (ATTN_SINK_FLAG_DETERMINISTIC if deterministic else 0))
    if flags & (ATTN_SINK_FLAG_SINK_BF16 | ATTN_SINK_FLAG_ACCUMULATE_DSINK):
        _check(attn_sink_bwd_ex(p, flags, q, k, v, sink, cu_seqlens_q, cu_seqlens_k, out,
                                out_residual, lse, dout, dq, dk, dv, dsink, workspace,
                                workspace.numel(), stream), "attn_sink_bwd_ex")
    else:
        fn = attn_sink_bwd_deterministic if deterministic else attn_sink_bwd
        _check(fn(p, q, k, v, sink, cu_seqlens_q, cu_seqlens_k, out, out_residual, lse,
                  dout, dq, dk, dv, dsink, workspace, workspace.numel(), stream), fn.__name__)
    return dq, dk, dv, dsink


class AttnSinkFunction(torch.autograd.Function):
    """Autograd wrapper: forward and backward both run in libattn_sink.so."""

    @staticmethod
    def forward(ctx, q, k, v, sink, causal, window, softmax_scale, cu_seqlens_q, cu_seqlens_k,
                max_seqlen_q, max_seqlen_k):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        sink32 = sink.detach().float().contiguous()
        out, lse, res = forward(q, k, v, sink32, causal=causal, window=window,
                                softmax_scale=softmax_scale, cu_seqlens_q=cu_seqlens_q,
                                cu_seqlens_k=cu_seqlens_k, max_seqlen_q=max_seqlen_q,
                                max_seqlen_k=max_seqlen_k)
        ctx.save_for_backward(q, k, v, sink32, out, res, lse, cu_seqlens_q, cu_seqlens_k)
        ctx.cfg = (causal, window, softmax_scale, max_seqlen_q, max_seqlen_k, sink.dtype)
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, sink32, out, res, lse, cu_q, cu_k = ctx.saved_tensors
        causal, window, scale, mq, mk, sink_dtype = ctx.cfg
        dq, dk, dv, dsink = backward(q, k, v, sink32, out, lse, dout.contiguous(),
                                     out_residual=res, causal=causal,
                                     window=window, softmax_scale=scale, cu_seqlens_q=cu_q,
                                     cu_seqlens_k=cu_k, max_seqlen_q=mq, max_seqlen_k=mk)
        return dq, dk, dv, dsink.to(sink_dtype), None, None, None, None, None, None, None


def attn_sink(q, k, v, sink, *, causal: bool = True, window: int = 0,
              softmax_scale: float | None = None, cu_seqlens_q=None, cu_seqlens_k=None,
              max_seqlen_q: int | None = None, max_seqlen_k: int | None = None):
    """Differentiable attention with a learnable per-head sink (bf16 q/k/v)."""
    return AttnSinkFunction.apply(q, k, v, sink, causal, window, softmax_scale, cu_seqlens_q,
                                  cu_seqlens_k, max_seqlen_q, max_seqlen_k)
