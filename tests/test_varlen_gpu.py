"""GPU parity for packed sequences of different lengths (page
"FlashAttention：快速且内存高效的准确注意力机制", sections "代码解读博客：FlashSelfAttention"
(cu_seqlens, max_seqlen) and "函数重命名" (flash_attn_varlen_func)).

The sequences mix one-row, empty, key-less, rectangular and ragged lengths, so
tiles straddle sequence ends. Tolerances as everywhere: bf16 max |err| <= 2e-2
and relative RMS <= 1e-2, fp32 L max |err| <= 1e-3 with -inf matched. dK and dV
sum over query rows, and a sequence of 129 query rows over one key sends all of
them to that key (|dV| ~ 10 to 35, where bf16's own rounding of the output is
up to 2^-8 |x|, 0.06 at 17), so dK and dV are checked for 2e-2 beyond that rounding.
"""
import numpy as np
import pytest

import oracle
from fa_inputs import alibi_slopes_geometric, bf16_bits_to_f64, normal_bf16_bits
from helpers import assert_bf16_close, assert_bf16_close_beyond_rounding, assert_lse_close, to_dev, to_f64

pytestmark = pytest.mark.gpu

LEN_Q = [1, 200, 0, 333, 128, 129, 40]
LEN_K = [50, 200, 10, 700, 128, 1, 0]  # the last sequence has query rows but no keys


def _cu(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def _run_fwd(H, Hk, D, causal=False, window=(-1, -1), alibi=None, seed=0, len_q=LEN_Q, len_k=LEN_K):
    import torch

    import exact_attention_56_gb300 as fa

    cq, ck = _cu(len_q), _cu(len_k)
    q_b = normal_bf16_bits((int(cq[-1]), H, D), seed * 8)
    k_b = normal_bf16_bits((int(ck[-1]), Hk, D), seed * 8 + 1)
    v_b = normal_bf16_bits((int(ck[-1]), Hk, D), seed * 8 + 2)
    q, k, v = to_dev(q_b), to_dev(k_b), to_dev(v_b)
    cu_q, cu_k = torch.from_numpy(cq).cuda(), torch.from_numpy(ck).cuda()
    al = None if alibi is None else torch.from_numpy(np.ascontiguousarray(alibi, dtype=np.float32)).cuda()
    out, lse = fa.fa_fwd_varlen(q, k, v, cu_q, cu_k, max(len_q), max(len_k), causal=causal, window_size=window,
                                alibi_slopes=al)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    o_ref, l_ref = oracle.attention_fwd_varlen(bf16_bits_to_f64(q_b), bf16_bits_to_f64(k_b), bf16_bits_to_f64(v_b),
                                               cq, ck, None, causal, window, alibi)
    assert_bf16_close(to_f64(out), o_ref, "O")
    assert_lse_close(lse.cpu().numpy().astype(np.float64), l_ref, "L")


def _run_bwd(H, Hk, D, causal=False, window=(-1, -1), alibi=None, seed=0, len_q=LEN_Q, len_k=LEN_K):
    import torch

    import exact_attention_56_gb300 as fa

    cq, ck = _cu(len_q), _cu(len_k)
    bits = {"q": normal_bf16_bits((int(cq[-1]), H, D), seed * 8), "k": normal_bf16_bits((int(ck[-1]), Hk, D), seed * 8 + 1),
            "v": normal_bf16_bits((int(ck[-1]), Hk, D), seed * 8 + 2),
            "do": normal_bf16_bits((int(cq[-1]), H, D), seed * 8 + 3)}
    q, k, v, do = (to_dev(bits[n]) for n in ("q", "k", "v", "do"))
    cu_q, cu_k = torch.from_numpy(cq).cuda(), torch.from_numpy(ck).cuda()
    al = None if alibi is None else torch.from_numpy(np.ascontiguousarray(alibi, dtype=np.float32)).cuda()
    kw = dict(causal=causal, window_size=window, alibi_slopes=al)
    out, lse = fa.fa_fwd_varlen(q, k, v, cu_q, cu_k, max(len_q), max(len_k), **kw)
    dq, dk, dv = fa.fa_bwd_varlen(do, q, k, v, out, lse, cu_q, cu_k, max(len_q), max(len_k), **kw)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    rq, rk, rv = oracle.attention_bwd_varlen(*(bf16_bits_to_f64(bits[n]) for n in ("do", "q", "k", "v")), cq, ck,
                                             None, causal, window, alibi)
    assert_bf16_close(to_f64(dq), rq, "dQ")
    assert_bf16_close_beyond_rounding(to_f64(dk), rk, "dK")
    assert_bf16_close_beyond_rounding(to_f64(dv), rv, "dV")


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_packed(D, causal):
    _run_fwd(2, 2, D, causal=causal, seed=500 + D + int(causal))


def test_forward_packed_groups_window_alibi():
    _run_fwd(4, 2, 128, causal=True, seed=510)
    _run_fwd(2, 1, 128, window=(64, 0), seed=511)
    _run_fwd(4, 4, 64, causal=True, alibi=alibi_slopes_geometric(4), seed=512)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_packed(D, causal):
    _run_bwd(2, 2, D, causal=causal, seed=520 + D + int(causal))


def test_backward_packed_groups_window_alibi():
    _run_bwd(4, 2, 128, causal=True, seed=530)
    _run_bwd(2, 2, 128, window=(100, 37), seed=531)
    _run_bwd(4, 4, 64, causal=True, alibi=alibi_slopes_geometric(4), seed=532)


def test_equal_lengths_match_the_padded_layout_bitwise():
    # Packed sequences of one length tile exactly like the padded layout, so the
    # results must be identical bit for bit (forward and backward).
    import torch

    import exact_attention_56_gb300 as fa

    B, S, H, D = 3, 300, 2, 128
    g = torch.Generator(device="cuda")
    g.manual_seed(540)
    q, k, v, do = (torch.randn((B, S, H, D), generator=g, device="cuda").to(torch.bfloat16) for _ in range(4))
    cu = torch.arange(0, (B + 1) * S, S, dtype=torch.int32, device="cuda")
    out, lse = fa.fa_fwd(q, k, v, causal=True)
    dq, dk, dv = fa.fa_bwd(do, q, k, v, out, lse, causal=True)
    flat = [t.reshape(B * S, H, D) for t in (q, k, v, do)]
    out_p, lse_p = fa.fa_fwd_varlen(flat[0], flat[1], flat[2], cu, cu, S, S, causal=True)
    dq_p, dk_p, dv_p = fa.fa_bwd_varlen(flat[3], flat[0], flat[1], flat[2], out_p, lse_p, cu, cu, S, S, causal=True)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    assert torch.equal(out.reshape(B * S, H, D).view(torch.int16), out_p.view(torch.int16))
    assert torch.equal(lse.permute(1, 0, 2).reshape(H, B * S), lse_p)
    for a, b in ((dq, dq_p), (dk, dk_p), (dv, dv_p)):
        assert torch.equal(a.reshape(B * S, H, D).view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("window", [(-1, 0), (1000, 0)])
def test_forward_packed_long_sequence_among_short_ones(window):
    # A 4500-row sequence gives the grid 18 query groups per head, enough for the
    # forward to order the groups across the whole grid; the short sequences'
    # CTAs past their own groups must leave without writing.
    _run_fwd(2, 1, 64, window=window, seed=31, len_q=[300, 4500, 129], len_k=[700, 4500, 1])
