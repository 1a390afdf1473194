"""Pins of the CPU float64 oracle against things other than itself.

Each test ties the oracle to a library routine (torch's float64
scaled_dot_product_attention, logsumexp, autograd), a closed form, central
finite differences or a hand-worked example, so that a dropped term, a wrong
sign, a wrong index or a transposed operand anywhere in it fails a test.
"""
import math

import pytest
import torch
import torch.nn.functional as F
from torch.nn.attention.bias import causal_lower_right

from oracle import oracle_bwd, oracle_fwd, sink_softmax
from oracle.attention_sink import dense_cu_seqlens

F64 = torch.float64
pytestmark = pytest.mark.filterwarnings("ignore")


def _rand(shape, seed, dtype=F64):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=F64).to(dtype)


def _problem(lengths_q, lengths_k, hq, hkv, d, seed, sink_scale=1.0):
    tq, tk = sum(lengths_q), sum(lengths_k)
    q = _rand((tq, hq, d), seed)
    k = _rand((tk, hkv, d), seed + 1)
    v = _rand((tk, hkv, d), seed + 2)
    do = _rand((tq, hq, d), seed + 3)
    sink = _rand((hq,), seed + 4) * sink_scale
    cq = [0]
    for n in lengths_q:
        cq.append(cq[-1] + n)
    ck = [0]
    for n in lengths_k:
        ck.append(ck[-1] + n)
    return q, k, v, do, sink, cq, ck


def _library_mask(n_q, n_k, causal, window):
    """Boolean SDPA mask built from library pieces: torch's lower-right causal
    bias, intersected with a tril/triu band for the window."""
    if not causal:
        return None
    m = causal_lower_right(n_q, n_k)._materialize(torch.device("cpu"))
    if window > 0:
        off = n_k - n_q
        band = torch.ones(n_q, n_k, dtype=torch.bool).triu(diagonal=off - window + 1)
        m = m & band
    return m


def _sdpa_per_sequence(q, k, v, cq, ck, scale, causal, window):
    """Standard attention (no sink) from torch, plus its logsumexp."""
    hq, hkv = q.shape[1], k.shape[1]
    outs, lses = [], []
    for s in range(len(cq) - 1):
        qs, qe, ks, ke = cq[s], cq[s + 1], ck[s], ck[s + 1]
        Q = q[qs:qe].permute(1, 0, 2).unsqueeze(0)
        K = k[ks:ke].permute(1, 0, 2).unsqueeze(0)
        V = v[ks:ke].permute(1, 0, 2).unsqueeze(0)
        mask = _library_mask(qe - qs, ke - ks, causal, window)
        o = F.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale,
                                           enable_gqa=True)
        Kr = K.repeat_interleave(hq // hkv, dim=1)
        sc = (Q @ Kr.transpose(-1, -2)) * scale
        if mask is not None:
            sc = sc.masked_fill(~mask, -math.inf)
        outs.append(o[0].permute(1, 0, 2))
        lses.append(torch.logsumexp(sc[0], dim=-1))
    return torch.cat(outs, 0), torch.cat(lses, 1)


CASES = [
    # lengths_q, lengths_k, hq, hkv, d, causal, window
    ([37], [37], 4, 2, 16, True, 0),
    ([37], [37], 4, 4, 16, False, 0),
    ([5, 19, 1], [5, 19, 1], 8, 2, 8, True, 0),
    ([9, 17], [9, 17], 4, 1, 8, True, 3),
    ([12], [20], 2, 1, 8, True, 0),          # N_q < N_k: bottom-right causal
    ([12], [20], 2, 2, 8, True, 4),
    ([40], [40], 2, 1, 8, True, 1),
]


# Row blocks of the oracle: the default (one block per short sequence) and
# blocks of 3 rows, so that every block after the first takes its key range
# from the causal / window bounds of a later first row (r0 > 0).
BLOCKS = [256, 3]


@pytest.mark.parametrize("block", BLOCKS)
@pytest.mark.parametrize("lq,lk,hq,hkv,d,causal,window", CASES)
def test_neginf_sink_is_standard_attention(lq, lk, hq, hkv, d, causal, window, block):
    """sink = -inf removes the sink column: torch's SDPA (float64) must agree."""
    q, k, v, do, sink, cq, ck = _problem(lq, lk, hq, hkv, d, 11)
    sink = torch.full((hq,), -math.inf, dtype=F64)
    scale = 0.37
    out, lse = oracle_fwd(q, k, v, sink, scale=scale, causal=causal, window=window,
                          cu_seqlens_q=cq, cu_seqlens_k=ck, block=block)
    ref, ref_lse = _sdpa_per_sequence(q, k, v, cq, ck, scale, causal, window)
    torch.testing.assert_close(out, ref, rtol=1e-12, atol=1e-12)
    torch.testing.assert_close(lse, ref_lse, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("block", BLOCKS)
@pytest.mark.parametrize("lq,lk,hq,hkv,d,causal,window", CASES)
def test_finite_sink_gates_standard_attention(lq, lk, hq, hkv, d, causal, window, block):
    """With a finite sink, P_ih = sigmoid(sink - LSE_std), so the output is the
    standard output times (1 - P_ih) and LSE = logaddexp(LSE_std, sink).
    The scale is not 1, so a sink that were (wrongly) scaled would fail."""
    q, k, v, do, sink, cq, ck = _problem(lq, lk, hq, hkv, d, 23, sink_scale=2.0)
    scale = 0.29
    out, lse = oracle_fwd(q, k, v, sink, scale=scale, causal=causal, window=window,
                          cu_seqlens_q=cq, cu_seqlens_k=ck, block=block)
    ref, ref_lse = _sdpa_per_sequence(q, k, v, cq, ck, scale, causal, window)
    gate = torch.sigmoid(ref_lse - sink.unsqueeze(1))          # [H, T] = 1 - P_ih
    torch.testing.assert_close(out, ref * gate.T.unsqueeze(-1), rtol=1e-11, atol=1e-12)
    torch.testing.assert_close(lse, torch.logaddexp(ref_lse, sink.unsqueeze(1)),
                               rtol=1e-12, atol=1e-12)


def _gated_autograd(q, k, v, sink, do, cq, ck, scale, causal, window):
    """Backward of the gated standard-attention form via float64 autograd."""
    q = q.clone().requires_grad_()
    k = k.clone().requires_grad_()
    v = v.clone().requires_grad_()
    sink = sink.clone().requires_grad_()
    o_std, lse_std = _sdpa_per_sequence(q, k, v, cq, ck, scale, causal, window)
    gate = torch.sigmoid(lse_std - sink.unsqueeze(1))
    o = o_std * gate.T.unsqueeze(-1)
    (o * do).sum().backward()
    return q.grad, k.grad, v.grad, sink.grad


@pytest.mark.parametrize("block", BLOCKS)
@pytest.mark.parametrize("lq,lk,hq,hkv,d,causal,window", CASES)
def test_backward_matches_autograd_of_gated_form(lq, lk, hq, hkv, d, causal, window, block):
    q, k, v, do, sink, cq, ck = _problem(lq, lk, hq, hkv, d, 31, sink_scale=1.5)
    scale = 0.41
    g = oracle_bwd(q, k, v, sink, do, scale=scale, causal=causal, window=window,
                   cu_seqlens_q=cq, cu_seqlens_k=ck, block=block)
    dq, dk, dv, dsink = _gated_autograd(q, k, v, sink, do, cq, ck, scale, causal, window)
    torch.testing.assert_close(g["dq"], dq, rtol=1e-10, atol=1e-11)
    torch.testing.assert_close(g["dk"], dk, rtol=1e-10, atol=1e-11)
    torch.testing.assert_close(g["dv"], dv, rtol=1e-10, atol=1e-11)
    torch.testing.assert_close(g["dsink"], dsink, rtol=1e-10, atol=1e-11)


def test_probabilities_sum_to_one():
    """Sum_j P_ij + P_ih = 1 for every row, including rows with hidden keys."""
    s = _rand((50, 33), 5) * 4.0
    s[3, :] = -math.inf                     # a row with no visible key
    s[7, 10:] = -math.inf
    for sink_h in (-3.0, 0.0, 2.5, 40.0):
        p, p_sink, lse = sink_softmax(s, sink_h)
        total = p.sum(1) + p_sink
        torch.testing.assert_close(total, torch.ones_like(total), rtol=0, atol=1e-14)
        assert float(p_sink[3]) == 1.0 and float(lse[3]) == sink_h
        assert (p[7, 10:] == 0).all()
    p, p_sink, lse = sink_softmax(s, 1e4)   # huge sink takes all the mass
    assert torch.allclose(p_sink, torch.ones_like(p_sink))


def test_single_key_closed_form():
    """N_k = 1: O = sig(x) v, LSE = logaddexp(s q.k, sink), dv = sig(x) dO,
    dq = s sig(1-sig) u k, dk = s sig(1-sig) u q, dsink = -sig(1-sig) u,
    with x = s q.k - sink and u = dO.v."""
    d, scale = 8, 0.7
    q = _rand((1, 3, d), 41)
    k = _rand((1, 1, d), 42)
    v = _rand((1, 1, d), 43)
    do = _rand((1, 3, d), 44)
    sink = torch.tensor([0.3, -1.2, 2.0], dtype=F64)
    g = oracle_bwd(q, k, v, sink, do, scale=scale, causal=True, window=0,
                   cu_seqlens_q=[0, 1], cu_seqlens_k=[0, 1])
    dk = torch.zeros(d, dtype=F64)
    dv = torch.zeros(d, dtype=F64)
    for h in range(3):
        qk = scale * float(q[0, h] @ k[0, 0])
        x = qk - float(sink[h])
        sg = 1.0 / (1.0 + math.exp(-x))
        u = float(do[0, h] @ v[0, 0])
        torch.testing.assert_close(g["out"][0, h], sg * v[0, 0], rtol=1e-13, atol=1e-14)
        assert abs(float(g["lse"][h, 0]) - float(torch.logaddexp(
            torch.tensor(qk, dtype=F64), sink[h]))) < 1e-13
        torch.testing.assert_close(g["dq"][0, h], scale * sg * (1 - sg) * u * k[0, 0],
                                   rtol=1e-12, atol=1e-14)
        assert abs(float(g["dsink"][h]) + sg * (1 - sg) * u) < 1e-13
        dk += scale * sg * (1 - sg) * u * q[0, h]
        dv += sg * do[0, h]
    torch.testing.assert_close(g["dk"][0, 0], dk, rtol=1e-12, atol=1e-14)
    torch.testing.assert_close(g["dv"][0, 0], dv, rtol=1e-12, atol=1e-14)


def test_hand_worked_example():
    """One query, two keys, worked by hand from the P_ij / P_ih equations.

    s = 1, q = (1, 0), k1 = (0, 0), k2 = (ln 2, 0)  ->  S = (0, ln 2);
    sink = ln 3, so the denominator is 1 + 2 + 3 = 6: P = (1/6, 1/3), P_h = 1/2.
    v1 = (6, 0), v2 = (0, 3)  ->  O = (1, 1), LSE = ln 6.
    dO = (1, 0)  ->  dP = (6, 0), D = 1, dsink = -P_h D = -1/2,
    dS = P (dP - D) = (5/6, -1/3), dq = dS . K = (-ln2 / 3, 0),
    dk1 = (5/6, 0), dk2 = (-1/3, 0), dv1 = (1/6, 0), dv2 = (1/3, 0).
    """
    ln2, ln3 = math.log(2.0), math.log(3.0)
    q = torch.tensor([[[1.0, 0.0]]], dtype=F64)
    k = torch.tensor([[[0.0, 0.0]], [[ln2, 0.0]]], dtype=F64)
    v = torch.tensor([[[6.0, 0.0]], [[0.0, 3.0]]], dtype=F64)
    do = torch.tensor([[[1.0, 0.0]]], dtype=F64)
    sink = torch.tensor([ln3], dtype=F64)
    g = oracle_bwd(q, k, v, sink, do, scale=1.0, causal=False, window=0,
                   cu_seqlens_q=[0, 1], cu_seqlens_k=[0, 2])
    exact = dict(
        out=[[[1.0, 1.0]]], lse=[[math.log(6.0)]], dq=[[[-ln2 / 3, 0.0]]],
        dk=[[[5 / 6, 0.0]], [[-1 / 3, 0.0]]], dv=[[[1 / 6, 0.0]], [[1 / 3, 0.0]]],
        dsink=[-0.5], D=[[1.0]])
    for name, val in exact.items():
        torch.testing.assert_close(g[name], torch.tensor(val, dtype=F64),
                                   rtol=1e-14, atol=1e-14)


def _loss(q, k, v, sink, do, cq, ck, scale, causal, window, block=256):
    out, _ = oracle_fwd(q, k, v, sink, scale=scale, causal=causal, window=window,
                        cu_seqlens_q=cq, cu_seqlens_k=ck, block=block)
    return float((out * do).sum())


FD_CASES = [
    # lengths_q, lengths_k, causal, window, block
    ([3, 5], [3, 5], True, 0, 256),
    ([3, 5], [3, 5], True, 3, 256),
    ([3, 5], [3, 5], False, 0, 256),
    # blocks of 2 rows: windowed key ranges of later blocks, N_q != N_k
    ([3, 7], [3, 7], True, 3, 2),
    ([5, 4], [7, 9], True, 2, 2),
    ([6], [4], True, 0, 2),
]


@pytest.mark.parametrize("lq,lk,causal,window,block", FD_CASES)
def test_finite_differences(lq, lk, causal, window, block):
    """Central differences of L = <O, dO> for every element of q, k, v, sink:
    small packed sequences, H_q = 4, H_kv = 2, d = 8."""
    q, k, v, do, sink, cq, ck = _problem(lq, lk, 4, 2, 8, 57)
    scale, eps = 0.45, 1e-6
    g = oracle_bwd(q, k, v, sink, do, scale=scale, causal=causal, window=window,
                   cu_seqlens_q=cq, cu_seqlens_k=ck, block=block)
    args = dict(q=q, k=k, v=v, sink=sink)
    for name in ("q", "k", "v", "sink"):
        base = args[name]
        fd = torch.zeros_like(base)
        flat = base.view(-1)
        for idx in range(flat.numel()):
            old = float(flat[idx])
            flat[idx] = old + eps
            lp = _loss(q, k, v, sink, do, cq, ck, scale, causal, window, block)
            flat[idx] = old - eps
            lm = _loss(q, k, v, sink, do, cq, ck, scale, causal, window, block)
            flat[idx] = old
            fd.view(-1)[idx] = (lp - lm) / (2 * eps)
        an = g["d" + name]
        err = (fd - an).abs().max() / max(1.0, float(an.abs().max()))
        assert err < 1e-6, (name, float(err))


def test_dsink_is_minus_total_score_gradient():
    """Shift invariance: adding c to every score and to the sink leaves P
    unchanged, so dsink_h = -sum_ij dS_ij.  The sum is read off dq by giving
    every key an extra coordinate equal to 1 (then dq_i[extra] = s sum_j dS_ij)."""
    q, k, v, do, sink, cq, ck = _problem([6, 11], [6, 11], 4, 2, 8, 71)
    q = torch.cat([q, torch.zeros(q.shape[0], 4, 1, dtype=F64)], -1)
    k = torch.cat([k, torch.ones(k.shape[0], 2, 1, dtype=F64)], -1)
    v = torch.cat([v, torch.zeros(v.shape[0], 2, 1, dtype=F64)], -1)
    do = torch.cat([do, torch.zeros(do.shape[0], 4, 1, dtype=F64)], -1)
    scale = 0.6
    for causal, window in ((True, 0), (True, 2), (False, 0)):
        g = oracle_bwd(q, k, v, sink, do, scale=scale, causal=causal, window=window,
                       cu_seqlens_q=cq, cu_seqlens_k=ck)
        total_ds = g["dq"][:, :, -1].sum(0) / scale
        torch.testing.assert_close(g["dsink"], -total_ds, rtol=1e-12, atol=1e-13)


def test_delta_equals_rowsum_dout_out():
    """D_i = sum_j P_ij dP_ij equals <dO_i, O_i> because the sink has no value row."""
    q, k, v, do, sink, cq, ck = _problem([33, 70], [33, 70], 8, 2, 16, 81)
    g = oracle_bwd(q, k, v, sink, do, scale=0.25, causal=True, window=5,
                   cu_seqlens_q=cq, cu_seqlens_k=ck)
    torch.testing.assert_close(g["D"], (g["out"] * do).sum(-1).T, rtol=1e-12, atol=1e-13)


def test_window_limits():
    """W = 1: each query sees only its own key, so O_i = sig(s q_i.k_i - sink) v_i.
    W >= N: identical to plain causal."""
    q, k, v, do, sink, cq, ck = _problem([21], [21], 4, 2, 8, 91)
    scale = 0.5
    out1, _ = oracle_fwd(q, k, v, sink, scale=scale, causal=True, window=1,
                         cu_seqlens_q=cq, cu_seqlens_k=ck)
    for h in range(4):
        x = scale * (q[:, h] * k[:, h // 2]).sum(-1) - sink[h]
        torch.testing.assert_close(out1[:, h], torch.sigmoid(x).unsqueeze(1) * v[:, h // 2],
                                   rtol=1e-13, atol=1e-14)
    full, _ = oracle_fwd(q, k, v, sink, scale=scale, causal=True, window=0,
                         cu_seqlens_q=cq, cu_seqlens_k=ck)
    wide, _ = oracle_fwd(q, k, v, sink, scale=scale, causal=True, window=21,
                         cu_seqlens_q=cq, cu_seqlens_k=ck)
    assert torch.equal(full, wide)


def test_rows_without_keys_keep_the_sink():
    """N_q > N_k with bottom-right causal: the first N_q - N_k rows see no key,
    so P_ih = 1, O = 0, LSE = sink, and they add nothing to any gradient."""
    q, k, v, do, sink, cq, ck = _problem([9], [4], 2, 1, 8, 101)
    g = oracle_bwd(q, k, v, sink, do, scale=0.5, causal=True, window=0,
                   cu_seqlens_q=cq, cu_seqlens_k=ck)
    assert torch.equal(g["out"][:5], torch.zeros_like(g["out"][:5]))
    assert torch.equal(g["lse"][:, :5], sink.unsqueeze(1).expand(2, 5))
    assert torch.equal(g["dq"][:5], torch.zeros_like(g["dq"][:5]))
    ref, ref_lse = _sdpa_per_sequence(q[5:], k, v, [0, 4], ck, 0.5, True, 0)
    gate = torch.sigmoid(ref_lse - sink.unsqueeze(1))
    torch.testing.assert_close(g["out"][5:], ref * gate.T.unsqueeze(-1), rtol=1e-12, atol=1e-13)


def test_dense_batch_helper_and_subsets():
    """Head / sequence subsets reproduce the full computation exactly."""
    q, k, v, do, sink, cq, ck = _problem([20, 20], [20, 20], 4, 2, 8, 111)
    assert cq == dense_cu_seqlens(2, 20)
    full = oracle_bwd(q, k, v, sink, do, scale=0.3, causal=True, window=0,
                      cu_seqlens_q=cq, cu_seqlens_k=ck)
    part = oracle_bwd(q, k, v, sink, do, scale=0.3, causal=True, window=0,
                      cu_seqlens_q=cq, cu_seqlens_k=ck, heads=[2, 3], seqs=[1])
    assert torch.equal(part["out"][20:, 2:], full["out"][20:, 2:])
    assert torch.equal(part["dk"][20:, 1], full["dk"][20:, 1])
    assert torch.isnan(part["out"][:20]).all()
    rows_out, _ = oracle_fwd(q, k, v, sink, scale=0.3, causal=True, window=0,
                             cu_seqlens_q=cq, cu_seqlens_k=ck, rows={0: [3, 19]})
    torch.testing.assert_close(rows_out[[3, 19]], full["out"][[3, 19]], rtol=0, atol=1e-15)
