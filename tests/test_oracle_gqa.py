"""Pins for the oracle's key/value head groups (k, v with Hk heads, H a multiple
of Hk; page "FlashAttention：快速且内存高效的准确注意力机制", section
"代码解读博客：FlashCrossAttention": kv of shape (B, Sk, 2, H_k, D)).

The independent routine is torch's scaled_dot_product_attention in float64 with
enable_gqa=True (forward, and autograd for the backward), plus closed forms: a
key/value head shared by identical query heads gets exactly the group size times
one head's gradient, and the split-KV merge stays exact.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def _draw(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _band(Sq, Sk, wl, wr):
    # bottom-right corner of an N x N band built from numpy's tril/triu
    N = max(Sq, Sk)
    full = np.ones((N, N), dtype=bool)
    m = full.copy()
    if wr >= 0:
        m &= np.tril(full, wr)
    if wl >= 0:
        m &= np.triu(full, -wl)
    return m[N - Sq:, N - Sk:]


def _sdpa_gqa(q, k, v, scale, mask=None, slopes=None, grad_out=None):
    """torch SDPA, float64, enable_gqa; q (B,Sq,H,D), k/v (B,Sk,Hk,D) in the oracle layout."""
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(x.transpose(0, 2, 1, 3))).requires_grad_(True)
                  for x in (q, k, v))
    B, Sq, H, _ = q.shape
    Sk = k.shape[1]
    attn = None
    if slopes is not None:
        N = max(Sq, Sk)
        dist = np.abs(np.subtract.outer(np.arange(N), np.arange(N)))[N - Sq:, N - Sk:].astype(np.float64)
        bias = -np.asarray(slopes, dtype=np.float64)[:, None, None] * dist[None]
        if mask is not None:
            bias = np.where(mask[None], bias, -np.inf)
        attn = torch.from_numpy(bias)[None].expand(B, H, Sq, Sk)
    elif mask is not None:
        attn = torch.from_numpy(mask)
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=attn, scale=scale, enable_gqa=True)
    if grad_out is None:
        return o.detach().numpy().transpose(0, 2, 1, 3)
    o.backward(torch.from_numpy(np.ascontiguousarray(grad_out.transpose(0, 2, 1, 3))))
    return tuple(t.grad.numpy().transpose(0, 2, 1, 3) for t in (tq, tk, tv))


def test_kv_head_mapping():
    assert [oracle.kv_head(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    assert [oracle.kv_head(h, 6, 1) for h in range(6)] == [0] * 6
    assert [oracle.kv_head(h, 4, 4) for h in range(4)] == [0, 1, 2, 3]
    for bad in ((4, 3), (4, 0), (4, 8)):
        with pytest.raises(ValueError):
            oracle.kv_head(0, *bad)


@pytest.mark.parametrize("H,Hk", [(6, 2), (4, 1), (3, 3)])
@pytest.mark.parametrize("Sq,Sk,causal,wl,wr", [(7, 11, False, -1, -1), (11, 7, True, -1, 0), (9, 9, False, 2, 1)])
def test_forward_matches_torch_sdpa_gqa(H, Hk, Sq, Sk, causal, wl, wr):
    B, D, scale = 2, 8, 0.37
    q, k, v = _draw((B, Sq, H, D), 1), _draw((B, Sk, Hk, D), 2), _draw((B, Sk, Hk, D), 3)
    o, _ = oracle.attention_fwd(q, k, v, scale, causal, (wl, wr))
    mask = _band(Sq, Sk, wl, 0 if causal else wr)
    if (~mask).all(axis=1).any():  # torch gives NaN for rows with no live key; the pages give 0
        live = mask.any(axis=1)
        ref = _sdpa_gqa(q, k, v, scale, mask)
        np.testing.assert_allclose(o[:, live], ref[:, live], rtol=0, atol=1e-12)
        assert np.all(o[:, ~live] == 0.0)
    else:
        np.testing.assert_allclose(o, _sdpa_gqa(q, k, v, scale, mask), rtol=0, atol=1e-12)


def test_forward_with_alibi_matches_torch_sdpa_gqa():
    B, Sq, Sk, H, Hk, D, scale = 1, 10, 10, 4, 2, 8, 0.5
    slopes = np.array([0.5, 0.25, 0.125, 0.0625])
    q, k, v = _draw((B, Sq, H, D), 4), _draw((B, Sk, Hk, D), 5), _draw((B, Sk, Hk, D), 6)
    o, _ = oracle.attention_fwd(q, k, v, scale, True, (-1, -1), slopes)
    ref = _sdpa_gqa(q, k, v, scale, _band(Sq, Sk, -1, 0), slopes)
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("H,Hk,causal", [(6, 2, False), (4, 1, True), (8, 4, True)])
def test_backward_matches_torch_autograd_gqa(H, Hk, causal):
    B, Sq, Sk, D, scale = 2, 9, 13, 8, 0.41
    q, k, v = _draw((B, Sq, H, D), 7), _draw((B, Sk, Hk, D), 8), _draw((B, Sk, Hk, D), 9)
    do = _draw((B, Sq, H, D), 10)
    dq, dk, dv = oracle.attention_bwd(do, q, k, v, scale, causal, (-1, -1))
    rq, rk, rv = _sdpa_gqa(q, k, v, scale, _band(Sq, Sk, -1, 0 if causal else -1), grad_out=do)
    for name, a, r in (("dQ", dq, rq), ("dK", dk, rk), ("dV", dv, rv)):
        np.testing.assert_allclose(a, r, rtol=0, atol=1e-11, err_msg=name)
    assert dk.shape == k.shape and dv.shape == v.shape


def test_identical_query_heads_give_group_times_one_head():
    # All G query heads identical (q and dO): every head's O equals the one-head
    # result, and the shared dK, dV are exactly G times the one-head gradients.
    G, B, Sq, Sk, D, scale = 4, 1, 6, 9, 8, 0.3
    q1, do1 = _draw((B, Sq, 1, D), 11), _draw((B, Sq, 1, D), 12)
    k, v = _draw((B, Sk, 1, D), 13), _draw((B, Sk, 1, D), 14)
    q, do = np.repeat(q1, G, axis=2), np.repeat(do1, G, axis=2)
    o, lse = oracle.attention_fwd(q, k, v, scale, True)
    o1, lse1 = oracle.attention_fwd(q1, k, v, scale, True)
    for h in range(G):
        np.testing.assert_array_equal(o[:, :, h], o1[:, :, 0])
        np.testing.assert_array_equal(lse[:, h], lse1[:, 0])
    dq, dk, dv = oracle.attention_bwd(do, q, k, v, scale, True)
    dq1, dk1, dv1 = oracle.attention_bwd(do1, q1, k, v, scale, True)
    np.testing.assert_allclose(dk, G * dk1, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dv, G * dv1, rtol=1e-13, atol=1e-14)
    for h in range(G):
        np.testing.assert_array_equal(dq[:, :, h], dq1[:, :, 0])


@pytest.mark.parametrize("n", [1, 3, 7])
def test_split_decode_with_shared_heads_equals_forward(n):
    B, Sq, Sk, H, Hk, D = 2, 2, 50, 6, 3, 8
    q, k, v = _draw((B, Sq, H, D), 15), _draw((B, Sk, Hk, D), 16), _draw((B, Sk, Hk, D), 17)
    o, lse = oracle.decode_splitkv(q, k, v, n, None, True)
    o_ref, lse_ref = oracle.attention_fwd(q, k, v, None, True)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)
