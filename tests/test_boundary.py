"""The C-ABI library without a GPU: it builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host (no launch, no device
call) with the documented status codes."""
import ctypes
import math

import pytest

from attention_learnable_head_gb300 import binding
from attention_learnable_head_gb300.build import build

OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build()
    return binding.lib()


def test_exports_every_declared_symbol():
    names = binding.header_functions()
    assert set(names) == {"attn_sink_fwd", "attn_sink_bwd", "attn_sink_bwd_workspace_size",
                          "attn_sink_fwd_workspace_size", "attn_sink_fwd_noalloc",
                          "attn_sink_last_cuda_error", "attn_sink_kernel_timing",
                          "attn_sink_kernel_time", "attn_sink_fwd_chunk", "attn_sink_merge",
                          "attn_sink_bwd_deterministic", "attn_sink_decode",
                          "attn_sink_decode_workspace_size", "attn_sink_fwd_ex",
                          "attn_sink_bwd_ex",
                          "attn_sink_status_string", "attn_sink_device_error",
                          "attn_sink_launch_count"}
    lib = binding.lib()
    for n in names:
        assert hasattr(lib, n), n
    # the tile-withholding hook exists only in the test build
    assert not hasattr(lib, "attn_sink_test_withhold")


def test_test_build_exports_the_withholding_hook():
    """The test build (waits lowered to 2 ms, one tile can be withheld) exports
    every declared entry point plus attn_sink_test_withhold."""
    from attention_learnable_head_gb300.build import build
    L = binding.load_library(build(test=True))
    for n in binding.header_functions():
        assert hasattr(L, n), n
    assert L.attn_sink_test_withhold(-1, -1) == 0


def test_params_struct_layout():
    # 14 ints + 1 float, no padding: must match attn_sink_params in the header.
    assert ctypes.sizeof(binding.AttnSinkParams) == 60


def test_status_strings():
    for code in range(6):
        s = binding.attn_sink_status_string(code)
        assert isinstance(s, str) and s
    assert binding.attn_sink_status_string(99) == "unknown status"


def _dense(**kw):
    p = binding.AttnSinkParams()
    p.batch, p.seqlen_q, p.seqlen_k = 1, 256, 256
    p.heads_q, p.heads_kv, p.head_dim = 8, 2, 64
    p.causal, p.window, p.softmax_scale, p.grad_dtype = 1, 0, 0.125, 0
    for k, v in kw.items():
        setattr(p, k, v)
    return p


FAKE = 0x7F0000000000       # never dereferenced: validation fails first
FAKE_ODD = FAKE + 8


def _fwd(p, q=FAKE, k=FAKE, v=FAKE, sink=FAKE, cu_q=None, cu_k=None, out=FAKE, res=None,
         lse=FAKE, ws=FAKE, ws_bytes=1 << 40):
    return binding.attn_sink_fwd(p, q, k, v, sink, cu_q, cu_k, out, res, lse, ws, ws_bytes,
                                 stream=0)


def _bwd(p, ws=FAKE, ws_bytes=1 << 40, fn=None, **kw):
    args = dict(q=FAKE, k=FAKE, v=FAKE, sink=FAKE, cu_q=None, cu_k=None, out=FAKE, res=None,
                lse=FAKE, dout=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, dsink=FAKE)
    args.update(kw)
    fn = binding.attn_sink_bwd if fn is None else fn
    return fn(p, args["q"], args["k"], args["v"], args["sink"], args["cu_q"], args["cu_k"],
              args["out"], args["res"], args["lse"], args["dout"], args["dq"], args["dk"],
              args["dv"], args["dsink"], ws, ws_bytes, stream=0)


def test_deterministic_backward_rejects_like_the_backward():
    det = binding.attn_sink_bwd_deterministic
    n0 = binding.attn_sink_launch_count()
    p = _dense()
    for kw in (dict(dsink=None), dict(dq=None), dict(dk=FAKE_ODD), dict(res=FAKE + 2),
               dict(sink=None)):
        assert _bwd(p, fn=det, **kw) == INVALID, kw
    assert _bwd(None, fn=det) == INVALID
    assert _bwd(_dense(head_dim=32), fn=det) == UNSUPPORTED
    assert _bwd(_dense(window=4, causal=0), fn=det) == INVALID
    assert binding.attn_sink_launch_count() == n0


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 128, UNSUPPORTED),
    ("head_dim", 32, UNSUPPORTED),
    ("heads_q", 7, INVALID),            # not a multiple of heads_kv
    ("heads_kv", 0, INVALID),
    ("causal", 2, INVALID),
    ("window", 16, None),               # window needs causal: tested with causal = 0 below
    ("softmax_scale", 0.0, INVALID),
    ("softmax_scale", -1.0, INVALID),
    ("softmax_scale", float("nan"), INVALID),
    ("softmax_scale", float("inf"), INVALID),
    ("grad_dtype", 2, INVALID),
    ("batch", -1, INVALID),
    ("num_seqs", 3, INVALID),           # packed field set without cu_seqlens
])
def test_invalid_params_rejected_on_host(field, value, status):
    p = _dense(**{field: value})
    if status is None:
        p.causal = 0
        status = INVALID
    assert _fwd(p) == status
    assert _bwd(p) == status
    if field not in ("num_seqs",):
        assert binding.attn_sink_bwd_workspace_size(p) == 0
        assert binding.attn_sink_fwd_workspace_size(p) == 0


def test_null_and_misaligned_pointers():
    p = _dense()
    assert binding.attn_sink_fwd(None, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, None, FAKE,
                                 FAKE, 1 << 40, 0) == INVALID
    assert _fwd(p, res=FAKE_ODD) == INVALID
    assert _bwd(p, res=FAKE + 2) == INVALID
    assert _fwd(p, q=None) == INVALID
    assert _fwd(p, sink=None) == INVALID
    assert _fwd(p, out=None) == INVALID
    assert _fwd(p, lse=None) == INVALID
    assert _fwd(p, q=FAKE_ODD) == INVALID
    assert _fwd(p, v=FAKE + 4) == INVALID
    assert _bwd(p, dsink=None) == INVALID
    assert _bwd(p, dq=None) == INVALID
    assert _bwd(p, dk=FAKE_ODD) == INVALID
    # one cu_seqlens without the other
    assert _fwd(p, cu_q=FAKE) == INVALID


def test_packed_mode_checks():
    p = _dense(batch=0, seqlen_q=0, seqlen_k=0, num_seqs=2, total_q=100, total_k=100,
               max_seqlen_q=60, max_seqlen_k=60)
    # dense batch field set together with cu_seqlens
    p2 = _dense(num_seqs=2, total_q=100, total_k=100, max_seqlen_q=60, max_seqlen_k=60)
    assert _fwd(p2, cu_q=FAKE, cu_k=FAKE) == INVALID
    # a max length above the total is inconsistent
    p3 = _dense(batch=0, num_seqs=2, total_q=100, total_k=100, max_seqlen_q=160,
                max_seqlen_k=60)
    assert _fwd(p3, cu_q=FAKE, cu_k=FAKE) == INVALID
    # too many sequences for the launch grid
    p4 = _dense(batch=0, num_seqs=70000, total_q=70000, total_k=70000, max_seqlen_q=1,
                max_seqlen_k=1)
    assert _fwd(p4, cu_q=FAKE, cu_k=FAKE) == UNSUPPORTED
    assert binding.attn_sink_bwd_workspace_size(p) > 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    # 16 MiB holds the fp16 copy of v for T_k * H_kv * 64 * 2 bytes; one more
    # token than fits returns ATTN_SINK_ERR_WORKSPACE before any device call.
    rows = binding.ATTN_SINK_NOALLOC_SCRATCH_BYTES // (64 * 2)
    p = _dense(batch=1, seqlen_q=16, seqlen_k=rows // 2 + 1, heads_q=2, heads_kv=2)
    n0 = binding.attn_sink_launch_count()
    assert binding.attn_sink_fwd_noalloc(p, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, None,
                                         FAKE, 0) == 3
    assert binding.attn_sink_fwd_noalloc(_dense(head_dim=32), FAKE, FAKE, FAKE, FAKE, None, None,
                                         FAKE, None, FAKE, 0) == UNSUPPORTED
    assert binding.attn_sink_fwd_noalloc(None, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, None,
                                         FAKE, 0) == INVALID
    assert binding.attn_sink_launch_count() == n0


def test_kernel_time_without_launches():
    # No timed launch has happened in this process: zero sums, OK status; a bad
    # id or a null pointer is an argument error.
    assert binding.attn_sink_kernel_timing(False) == OK
    for k in (binding.ATTN_SINK_KERNEL_FWD, binding.ATTN_SINK_KERNEL_BWD_MAIN,
              binding.ATTN_SINK_KERNEL_BWD_DQ, binding.ATTN_SINK_KERNEL_MERGE):
        assert binding.attn_sink_kernel_time(k) == (OK, 0.0, 0)
    assert binding.attn_sink_kernel_time(4)[0] == INVALID
    assert binding.attn_sink_kernel_time(-1)[0] == INVALID
    assert binding.lib().attn_sink_kernel_time(0, None, None) == INVALID


def _chunk(p, q_pos0=0, q=FAKE, k=FAKE, v=FAKE, out=FAKE, res=None, lse=FAKE, ws=FAKE,
           ws_bytes=1 << 40):
    return binding.attn_sink_fwd_chunk(p, q_pos0, q, k, v, None, None, out, res, lse, ws,
                                       ws_bytes, stream=0)


def _merge(c=2, t=16, h=4, d=64, o=FAKE, r=None, ls=FAKE, sink=FAKE, out=FAKE, res=None,
           lse=FAKE):
    return binding.attn_sink_merge(c, t, h, d, o, r, ls, sink, out, res, lse, stream=0)


def test_chunk_forward_rejects_bad_arguments_on_host():
    n0 = binding.attn_sink_launch_count()
    p = _dense()
    assert _chunk(p, q_pos0=(1 << 30) + 1) == INVALID
    assert _chunk(p, q_pos0=-(1 << 30) - 1) == INVALID
    assert _chunk(p, q=None) == INVALID
    assert _chunk(p, lse=None) == INVALID
    assert _chunk(p, out=FAKE_ODD) == INVALID
    assert _chunk(p, ws=None) == 3
    assert _chunk(_dense(head_dim=32)) == UNSUPPORTED
    assert binding.attn_sink_fwd_chunk(None, 0, FAKE, FAKE, FAKE, None, None, FAKE, None, FAKE,
                                       FAKE, 1 << 40, stream=0) == INVALID
    assert _chunk(_dense(batch=0)) == OK        # nothing to compute
    assert binding.attn_sink_launch_count() == n0


def test_merge_rejects_bad_arguments_on_host():
    n0 = binding.attn_sink_launch_count()
    assert _merge(c=0) == INVALID
    assert _merge(h=0) == INVALID
    assert _merge(t=-1) == INVALID
    assert _merge(d=32) == UNSUPPORTED
    assert _merge(t=0) == OK                    # no rows: a no-op
    for kw in (dict(o=None), dict(ls=None), dict(sink=None), dict(out=None), dict(lse=None),
               dict(o=FAKE_ODD), dict(r=FAKE_ODD), dict(out=FAKE_ODD), dict(res=FAKE_ODD)):
        assert _merge(**kw) == INVALID, kw
    assert binding.attn_sink_launch_count() == n0


def _dparams(**kw):
    p = binding.AttnSinkDecodeParams()
    p.batch, p.heads_q, p.heads_kv, p.head_dim = 4, 16, 2, 64
    p.page_size, p.num_pages, p.max_pages, p.window, p.softmax_scale = 16, 64, 8, 0, 0.125
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def _decode(p, q=FAKE, kc=FAKE, vc=FAKE, table=FAKE, lens=FAKE, sink=FAKE, out=FAKE, res=None,
            lse=FAKE, ws=FAKE, ws_bytes=1 << 40):
    return binding.attn_sink_decode(p, q, kc, vc, table, lens, sink, out, res, lse, ws,
                                    ws_bytes, stream=0)


def test_decode_params_struct_layout():
    assert ctypes.sizeof(binding.AttnSinkDecodeParams) == 36


def test_decode_rejects_bad_arguments_on_host():
    n0 = binding.attn_sink_launch_count()
    assert _decode(None) == INVALID
    assert _decode(_dparams(head_dim=32)) == UNSUPPORTED
    assert _decode(_dparams(heads_q=32, heads_kv=2)) == UNSUPPORTED     # 16 heads per kv head
    assert _decode(_dparams(heads_q=6)) == UNSUPPORTED                  # 3 heads per kv head
    assert _decode(_dparams(heads_q=15)) == INVALID                     # not a multiple
    assert _decode(_dparams(page_size=0)) == INVALID
    assert _decode(_dparams(softmax_scale=0.0)) == INVALID
    assert _decode(_dparams(softmax_scale=math.inf)) == INVALID
    assert _decode(_dparams(max_pages=1 << 20, page_size=1 << 12)) == INVALID   # > 2^30 keys
    assert _decode(_dparams(), q=None) == INVALID
    assert _decode(_dparams(), table=None) == INVALID
    assert _decode(_dparams(), lens=None) == INVALID
    assert _decode(_dparams(), out=FAKE_ODD) == INVALID
    assert _decode(_dparams(), ws=None) == 3
    assert _decode(_dparams(), ws_bytes=16) == 3
    assert _decode(_dparams(), ws=FAKE + 16) == 3
    assert _decode(_dparams(batch=0)) == OK
    # launch-grid limits (sequences in grid.z, kv heads in grid.y)
    assert _decode(_dparams(batch=65536)) == UNSUPPORTED
    assert _decode(_dparams(heads_q=65536, heads_kv=65536)) == UNSUPPORTED
    assert binding.attn_sink_decode_workspace_size(_dparams(batch=65536)) == 0
    assert binding.attn_sink_launch_count() == n0
    assert binding.attn_sink_decode_workspace_size(_dparams()) > 0
    assert binding.attn_sink_decode_workspace_size(_dparams(batch=0)) == 0
    assert binding.attn_sink_decode_workspace_size(_dparams(head_dim=32)) == 0
    assert binding.attn_sink_decode_workspace_size(None) == 0


def test_ex_entry_points_reject_unknown_flags_on_host():
    n0 = binding.attn_sink_launch_count()
    p = _dense()
    args = (FAKE, FAKE, FAKE, FAKE, None, None, FAKE, None, FAKE, FAKE, 1 << 40)
    for bad in (2, 4, 8, -1):                       # forward knows only SINK_BF16
        assert binding.attn_sink_fwd_ex(p, bad, *args, stream=0) == INVALID, bad
    bargs = (FAKE, FAKE, FAKE, FAKE, None, None, FAKE, None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
             FAKE, 1 << 40)
    for bad in (8, 16, -1):
        assert binding.attn_sink_bwd_ex(p, bad, *bargs, stream=0) == INVALID, bad
    assert binding.attn_sink_fwd_ex(None, 1, *args, stream=0) == INVALID
    assert binding.attn_sink_bwd_ex(None, 7, *bargs, stream=0) == INVALID
    assert binding.attn_sink_fwd_ex(_dense(head_dim=32), 1, *args, stream=0) == UNSUPPORTED
    assert binding.attn_sink_bwd_ex(_dense(head_dim=32), 3, *bargs, stream=0) == UNSUPPORTED
    assert binding.attn_sink_launch_count() == n0


def test_forward_workspace_checked_on_host():
    p = _dense()
    assert _fwd(p, ws=None) == 3
    assert _fwd(p, ws_bytes=16) == 3
    assert _fwd(p, ws=FAKE + 16) == 3     # not 256-byte aligned


def test_empty_problem_is_a_no_op():
    # Nothing to compute: returns OK without touching the device or launching.
    n0 = binding.attn_sink_launch_count()
    assert _fwd(_dense(batch=0)) == OK
    assert _fwd(_dense(seqlen_q=0)) == OK
    assert _fwd(_dense(head_dim=32)) == UNSUPPORTED
    assert binding.attn_sink_launch_count() == n0


def test_workspace_size():
    p = _dense(batch=2, seqlen_q=1000, seqlen_k=1000, heads_q=64, heads_kv=8)
    n_bf16 = binding.attn_sink_bwd_workspace_size(p)
    t, h = 2000, 64
    assert n_bf16 % 256 == 0
    # at least D, the partials, the fp32 dq accumulator and the fp16 copies
    assert n_bf16 >= t * h * 4 + t * h * 64 * 4 + 2 * t * h * 64 * 2 + 2 * t * 8 * 64 * 2
    p.grad_dtype = 1
    n_fp32 = binding.attn_sink_bwd_workspace_size(p)
    assert n_fp32 < n_bf16       # fp32 dq is accumulated in place
    assert binding.attn_sink_bwd_workspace_size(None) == 0
    # forward: the fp16 copy of v
    p.grad_dtype = 0
    assert binding.attn_sink_fwd_workspace_size(p) == 2000 * 8 * 64 * 2
    assert binding.attn_sink_fwd_workspace_size(None) == 0


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_LIB", None)
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        binding.lib()
