"""GPU parity of the paged decode forward (attn_sink_decode) through the C ABI
against the float64 oracle: shuffled page layouts, ragged lengths (empty, one
key, page-aligned, thousands of keys), windows, GQA groups of 1 to 8, page size
1; consistency with the prefill forward on the same keys (the training /
inference agreement the pages are about); the device-side bounds check of the
block table; and a GPT-OSS-shaped serving batch on sampled sequences."""
import pytest
import torch

from attention_learnable_head_gb300 import binding
from oracle.decode import oracle_decode
from parity import TOL_LSE, assert_close

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _paged_case(seed, lens, page, hq, hkv, spare=5):
    """bf16 q and a shuffled paged cache holding lens[b] random keys per sequence."""
    g = torch.Generator().manual_seed(seed)
    n_used = sum((L + page - 1) // page for L in lens)
    n_pages = n_used + spare
    perm = torch.randperm(n_pages, generator=g)
    kc = torch.randn(n_pages, page, hkv, 64, generator=g).to(torch.bfloat16)
    vc = torch.randn(n_pages, page, hkv, 64, generator=g).to(torch.bfloat16)
    max_p = max([(L + page - 1) // page for L in lens] + [1])
    table = torch.full((len(lens), max_p), -1, dtype=torch.int32)
    nxt = 0
    for b, L in enumerate(lens):
        for p in range((L + page - 1) // page):
            table[b, p] = int(perm[nxt])
            nxt += 1
    q = torch.randn(len(lens), hq, 64, generator=g).to(torch.bfloat16)
    sink = torch.randn(hq, generator=g)
    return q, kc, vc, table, torch.tensor(lens, dtype=torch.int32), sink


def _run(q, kc, vc, table, lens, sink, scale, window, residual=True):
    out, lse, res = binding.decode(q.to(DEV), kc.to(DEV), vc.to(DEV), table.to(DEV),
                                   lens.to(DEV), sink.to(DEV), window=window,
                                   softmax_scale=scale, residual=residual)
    torch.cuda.synchronize()
    st, code = binding.attn_sink_device_error()
    assert st == 0 and code == 0, f"device error word {code:#x}"
    return out.cpu(), lse.cpu(), None if res is None else res.cpu()


def _check_lse(got, ref):
    got, ref = got.double(), ref.double()
    assert torch.equal(torch.isneginf(got), torch.isneginf(ref))
    fin = torch.isfinite(ref)
    if fin.any():
        err = (got[fin] - ref[fin]).abs().max().item()
        assert err <= TOL_LSE, f"lse max abs {err:.3e}"


CASES = [
    # name, lens, page, hq, hkv, window
    ("ragged_g8", [0, 1, 16, 37, 300], 16, 16, 2, 0),
    ("window_g8", [129, 1000, 64], 64, 8, 1, 100),
    ("long_g8", [5000, 333], 128, 64, 8, 0),
    ("page1_g1", [50, 7], 1, 4, 4, 0),
    ("g4_window_short", [3, 40, 200], 32, 8, 2, 16),
    # page 8: the smallest page copied whole by TMA; page 48: not a power of
    # two, copied by the per-thread path
    ("page8_window", [9, 77, 513], 8, 16, 2, 70),
    ("page48_g2", [47, 48, 49, 700], 48, 4, 2, 0),
]


@pytest.mark.parametrize("name,lens,page,hq,hkv,window", CASES, ids=[c[0] for c in CASES])
def test_decode_matches_oracle(name, lens, page, hq, hkv, window):
    q, kc, vc, table, lens_t, sink = _paged_case(len(name) * 7 + page, lens, page, hq, hkv)
    scale = 0.125
    out, lse, res = _run(q, kc, vc, table, lens_t, sink, scale, window)
    ref_out, ref_lse = oracle_decode(q, kc, vc, table, lens_t, sink, scale=scale, window=window)
    assert_close(f"{name} out", out, ref_out)
    # out + residual carries ~16 significand bits of the fp32 result
    assert_close(f"{name} out+res", (out.double() + res.double()).float(), ref_out,
                 max_abs=2e-3, rel_fro=5e-4)
    _check_lse(lse, ref_lse)


def test_decode_agrees_with_prefill_forward():
    """The decode of each sequence's last token equals the last query row of
    the causal prefill forward over the same keys (training/inference
    consistency), both against the oracle and against each other."""
    hq, hkv, page = 16, 2, 16
    lens = [257, 64, 1]
    q_all, kc, vc, table, lens_t, sink = _paged_case(77, lens, page, hq, hkv, spare=0)
    g = torch.Generator().manual_seed(78)
    for b, L in enumerate(lens):
        # dense copies of this sequence's keys, and a full query block whose last
        # row is the decode token
        pages = [int(table[b, p]) for p in range((L + page - 1) // page)]
        k = torch.cat([kc[p] for p in pages])[:L]
        v = torch.cat([vc[p] for p in pages])[:L]
        qs = torch.randn(L, hq, 64, generator=g).to(torch.bfloat16)
        qs[-1] = q_all[b]
        out_f, lse_f, _ = binding.forward(qs.view(1, L, hq, 64).to(DEV), k.view(1, L, hkv, 64).to(DEV),
                                          v.view(1, L, hkv, 64).to(DEV), sink.to(DEV),
                                          causal=True, window=0, softmax_scale=0.125)
        out_d, lse_d, _ = _run(q_all[b:b + 1], kc, vc, table[b:b + 1], lens_t[b:b + 1], sink,
                               0.125, 0)
        last = out_f.view(L, hq, 64)[-1].cpu()
        assert_close(f"len {L} decode vs prefill", out_d[0], last.double())
        assert (lse_d[:, 0] - lse_f[:, -1].cpu()).abs().max().item() <= 2 * TOL_LSE


def test_decode_bad_block_table_entry_is_reported():
    """An out-of-range page index is skipped by the kernel's bounds check and
    reported as 0x800 in the device error word (nothing outside the cache is read)."""
    q, kc, vc, table, lens_t, sink = _paged_case(5, [40, 20], 16, 8, 1)
    table = table.clone()
    table[0, 1] = kc.shape[0] + 1000
    binding.decode(q.to(DEV), kc.to(DEV), vc.to(DEV), table.to(DEV), lens_t.to(DEV),
                   sink.to(DEV), softmax_scale=0.125)
    st, code = binding.attn_sink_device_error()
    assert st == 0 and code == 0x800, hex(code)
    # the next, valid call is clean again
    _run(q, kc, vc, table.clamp(max=kc.shape[0] - 1).clamp(min=0), lens_t, sink, 0.125, 0)


def test_decode_gptoss_serving_batch_sampled():
    """64 sequences with 1000..8192 cached keys each, H 64/8, page 16: every
    head of six sampled sequences against the oracle."""
    g = torch.Generator().manual_seed(91)
    lens = torch.randint(1000, 8193, (64,), generator=g).tolist()
    q, kc, vc, table, lens_t, sink = _paged_case(92, lens, 16, 64, 8)
    out, lse, _ = _run(q, kc, vc, table, lens_t, sink, 0.125, 0, residual=False)
    pick = [0, 5, 17, 31, 48, 63]
    idx = torch.tensor(pick)
    ref_out, ref_lse = oracle_decode(q[idx], kc, vc, table[idx], lens_t[idx], sink, scale=0.125)
    assert_close("serving batch out", out[idx], ref_out)
    _check_lse(lse[:, idx], ref_lse)


def test_decode_repeatable():
    """The split results are merged by whichever CTA of a (sequence, kv head)
    finishes last, in split order: ten runs of a batch with many splits per
    sequence are bitwise equal (a stale or early read of another split's
    partial would show up as a difference)."""
    q, kc, vc, table, lens, sink = _paged_case(77, [4000, 3000, 17, 2500] * 8, 16, 16, 2)
    first = _run(q, kc, vc, table, lens, sink, 0.125, 0)
    for _ in range(9):
        again = _run(q, kc, vc, table, lens, sink, 0.125, 0)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
