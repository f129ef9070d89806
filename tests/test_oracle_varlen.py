"""Pins for the oracle's packed sequences (page "FlashAttention：快速且内存高效的准确注意力机制",
sections "代码解读博客：FlashSelfAttention" (cu_seqlens, max_seqlen) and "函数重命名"
(flash_attn_varlen_func)).

The independent routine is torch's scaled_dot_product_attention in float64 run
once over the whole packed tensor with a block-diagonal mask whose blocks carry
each sequence's own bottom-right causal / window band (built from numpy
tril/triu), forward and autograd. Invariants: empty sequences contribute no
rows, and a sequence's results do not depend on the other sequences.
"""
import numpy as np
import pytest
import torch

import oracle

CU_Q = [0, 3, 3, 40, 41]
CU_K = [0, 7, 12, 40, 41]   # sequence 1 has keys but no query rows


def _draw(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _band(Sq, Sk, wl, wr):
    N = max(Sq, Sk)
    full = np.ones((N, N), dtype=bool)
    m = full.copy()
    if wr >= 0:
        m &= np.tril(full, wr)
    if wl >= 0:
        m &= np.triu(full, -wl)
    return m[N - Sq:, N - Sk:]


def _block_mask(cu_q, cu_k, wl, wr):
    mask = np.zeros((cu_q[-1], cu_k[-1]), dtype=bool)
    for b in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if q1 > q0 and k1 > k0:
            mask[q0:q1, k0:k1] = _band(q1 - q0, k1 - k0, wl, wr)
    return mask


def _sdpa_packed(q, k, v, scale, mask, grad_out=None):
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x.transpose(1, 0, 2)))[None].requires_grad_(True)
                  for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(mask), scale=scale,
                                                         enable_gqa=True)
    if grad_out is None:
        return o.detach()[0].numpy().transpose(1, 0, 2)
    live = mask.any(axis=1)
    g = np.where(live[:, None, None], grad_out, 0.0)  # rows without keys are NaN in torch; the pages give 0
    o.backward(torch.from_numpy(np.ascontiguousarray(g.transpose(1, 0, 2)))[None])
    return tuple(np.nan_to_num(t.grad[0].numpy().transpose(1, 0, 2)) for t in (tq, tk, tv))


@pytest.mark.parametrize("causal,wl,wr", [(False, -1, -1), (True, -1, 0), (False, 3, 2)])
@pytest.mark.parametrize("H,Hk", [(2, 2), (4, 2)])
def test_forward_matches_block_diagonal_sdpa(causal, wl, wr, H, Hk):
    D, scale = 8, 0.4
    q, k, v = _draw((CU_Q[-1], H, D), 1), _draw((CU_K[-1], Hk, D), 2), _draw((CU_K[-1], Hk, D), 3)
    o, lse = oracle.attention_fwd_varlen(q, k, v, CU_Q, CU_K, scale, causal, (wl, wr))
    mask = _block_mask(CU_Q, CU_K, wl, 0 if causal else wr)
    live = mask.any(axis=1)
    ref = _sdpa_packed(q, k, v, scale, mask)
    np.testing.assert_allclose(o[live], ref[live], rtol=0, atol=1e-12)
    assert np.all(o[~live] == 0.0) and np.all(np.isneginf(lse[:, ~live]))
    assert o.shape == q.shape and lse.shape == (H, CU_Q[-1])


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_block_diagonal_sdpa(causal):
    H, Hk, D, scale = 4, 2, 8, 0.35
    q, k, v = _draw((CU_Q[-1], H, D), 4), _draw((CU_K[-1], Hk, D), 5), _draw((CU_K[-1], Hk, D), 6)
    do = _draw((CU_Q[-1], H, D), 7)
    dq, dk, dv = oracle.attention_bwd_varlen(do, q, k, v, CU_Q, CU_K, scale, causal)
    rq, rk, rv = _sdpa_packed(q, k, v, scale, _block_mask(CU_Q, CU_K, -1, 0 if causal else -1), grad_out=do)
    for name, a, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        np.testing.assert_allclose(a, r, rtol=0, atol=1e-11, err_msg=name)


def test_sequences_do_not_interact():
    H, D = 2, 8
    q, k, v = _draw((CU_Q[-1], H, D), 8), _draw((CU_K[-1], H, D), 9), _draw((CU_K[-1], H, D), 10)
    o, lse = oracle.attention_fwd_varlen(q, k, v, CU_Q, CU_K, None, True)
    k2, v2 = k.copy(), v.copy()
    k2[CU_K[2]:CU_K[3]] += 5.0  # change sequence 2 only
    v2[CU_K[2]:CU_K[3]] -= 3.0
    o2, lse2 = oracle.attention_fwd_varlen(q, k2, v2, CU_Q, CU_K, None, True)
    other = np.r_[0:CU_Q[2], CU_Q[3]:CU_Q[4]]
    np.testing.assert_array_equal(o[other], o2[other])
    np.testing.assert_array_equal(lse[:, other], lse2[:, other])
    assert not np.allclose(o[CU_Q[2]:CU_Q[3]], o2[CU_Q[2]:CU_Q[3]])


def test_equal_lengths_match_the_padded_layout():
    B, S, H, D = 3, 9, 2, 8
    q, k, v = _draw((B, S, H, D), 11), _draw((B, S, H, D), 12), _draw((B, S, H, D), 13)
    cu = [0, S, 2 * S, 3 * S]
    o, lse = oracle.attention_fwd_varlen(q.reshape(B * S, H, D), k.reshape(B * S, H, D), v.reshape(B * S, H, D),
                                         cu, cu, None, True)
    o_ref, l_ref = oracle.attention_fwd(q, k, v, None, True)
    np.testing.assert_array_equal(o, o_ref.reshape(B * S, H, D))
    np.testing.assert_array_equal(lse, l_ref.transpose(1, 0, 2).reshape(H, B * S))


def test_rejects_bad_cu_seqlens():
    q = np.zeros((4, 1, 8))
    with pytest.raises(ValueError):
        oracle.attention_fwd_varlen(q, q, q, [0, 3, 2, 4], [0, 1, 2, 4])
    with pytest.raises(ValueError):
        oracle.attention_fwd_varlen(q, q, q, [1, 4], [0, 4])
