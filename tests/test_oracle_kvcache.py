"""Pins for the oracle's KV-cache decode step (page "FlashAttention：快速且内存高效的准确注意力机制",
section "2.2：针对推理进行优化": flash_attn_with_kvcache applies rotary embeddings and
updates the cache in place; the formula is the standard rotary embedding, a
reading stated in the oracle).

Rotary: closed forms for unit pairs, norm preservation, the relative-position
property of angle tables t * w_f, and the permutation relating the interleaved
and half-split pairings. Append: only rows [L, L + S_new) change, rows past the
capacity are dropped, and the attention equals the forward over the updated
cache with the rotated query.
"""
import numpy as np
import pytest
import torch

import oracle


def _bf16(x):
    # torch's round-to-nearest-even cast, an independent routine
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def test_round_bf16_matches_torch_cast():
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 0.0, -0.0, 65504.0])])
    np.testing.assert_array_equal(oracle.round_bf16(x), _bf16(x))


def _tables(n, r, base=10000.0):
    w = base ** (-np.arange(r // 2) * 2.0 / r)
    ang = np.arange(n)[:, None] * w[None, :]
    return np.cos(ang), np.sin(ang)


@pytest.mark.parametrize("interleaved", [False, True])
def test_unit_pairs_closed_form(interleaved):
    r, t = 8, 5
    cos, sin = _tables(10, r)
    for f in range(r // 2):
        i1, i2 = (2 * f, 2 * f + 1) if interleaved else (f, f + r // 2)
        e1 = np.zeros((1, r)); e1[0, i1] = 1.0
        e2 = np.zeros((1, r)); e2[0, i2] = 1.0
        y1 = oracle.rotary(e1, [t], cos, sin, interleaved)
        y2 = oracle.rotary(e2, [t], cos, sin, interleaved)
        assert y1[0, i1] == pytest.approx(cos[t, f], abs=1e-15) and y1[0, i2] == pytest.approx(sin[t, f], abs=1e-15)
        assert y2[0, i1] == pytest.approx(-sin[t, f], abs=1e-15) and y2[0, i2] == pytest.approx(cos[t, f], abs=1e-15)
        others = [d for d in range(r) if d not in (i1, i2)]
        assert np.all(y1[0, others] == 0.0) and np.all(y2[0, others] == 0.0)


def test_norms_preserved_and_tail_untouched():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((6, 3, 32))
    cos, sin = _tables(50, 16)
    for inter in (False, True):
        y = oracle.rotary(x, [0, 3, 7, 11, 49, 60], cos, sin, inter)
        np.testing.assert_allclose(np.linalg.norm(y[..., :16], axis=-1), np.linalg.norm(x[..., :16], axis=-1),
                                   rtol=1e-13)
        np.testing.assert_array_equal(y[..., 16:], x[..., 16:])
    np.testing.assert_array_equal(oracle.rotary(x[:1], [0], cos, sin), x[:1])  # angle 0 is the identity


@pytest.mark.parametrize("interleaved", [False, True])
def test_scores_depend_on_relative_position_only(interleaved):
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal((1, 32)), rng.standard_normal((1, 32))
    cos, sin = _tables(100, 32)
    a = oracle.rotary(q, [17], cos, sin, interleaved) @ oracle.rotary(k, [4], cos, sin, interleaved).T
    b = oracle.rotary(q, [57], cos, sin, interleaved) @ oracle.rotary(k, [44], cos, sin, interleaved).T
    assert a[0, 0] == pytest.approx(b[0, 0], rel=1e-12, abs=1e-12)


def test_interleaved_is_half_split_under_a_permutation():
    rng = np.random.default_rng(3)
    r = 16
    x = rng.standard_normal((4, r))
    cos, sin = _tables(20, r)
    perm = np.r_[np.arange(0, r, 2), np.arange(1, r, 2)]  # interleaved pair (2f, 2f+1) -> (f, f + r/2)
    inv = np.argsort(perm)
    y_inter = oracle.rotary(x, [1, 5, 9, 19], cos, sin, True)
    y_half = oracle.rotary(x[:, perm], [1, 5, 9, 19], cos, sin, False)[:, inv]
    np.testing.assert_allclose(y_inter, y_half, rtol=0, atol=1e-14)


def test_append_changes_only_new_rows_and_drops_overflow():
    rng = np.random.default_rng(4)
    B, cap, Hk, D, H, S_new = 2, 10, 2, 16, 4, 3
    kc, vc = rng.standard_normal((B, cap, Hk, D)), rng.standard_normal((B, cap, Hk, D))
    kn, vn = rng.standard_normal((B, S_new, Hk, D)), rng.standard_normal((B, S_new, Hk, D))
    q = rng.standard_normal((B, S_new, H, D))
    cos, sin = _tables(32, 16)
    seq = [4, 8]  # the second sequence has room for 2 of the 3 new rows
    o, lse, kc2, vc2 = oracle.decode_kvcache(q, kc, vc, seq, kn, vn, cos, sin, False, None, None, True)
    np.testing.assert_array_equal(kc2[0, :4], kc[0, :4])
    np.testing.assert_array_equal(kc2[0, 7:], kc[0, 7:])
    # a key written into the (bf16) cache is the rotated key rounded to bf16; values are copied
    np.testing.assert_array_equal(kc2[0, 4:7], _bf16(oracle.rotary(kn[0], [4, 5, 6], cos, sin)))
    np.testing.assert_array_equal(vc2[0, 4:7], vn[0])
    np.testing.assert_array_equal(kc2[1, 8:10], _bf16(oracle.rotary(kn[1, :2], [8, 9], cos, sin)))
    # attention: the forward over the updated cache with q rotated at i + Sk - Sq
    for b, n in ((0, 7), (1, 10)):
        qr = oracle.rotary(q[b], [i + n - S_new for i in range(S_new)], cos, sin)
        o_ref, l_ref = oracle.attention_fwd(qr[None], kc2[b:b + 1, :n], vc2[b:b + 1, :n], None, True)
        np.testing.assert_allclose(o[b], o_ref[0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[b], l_ref[0], rtol=0, atol=1e-13)


def test_paged_append_matches_dense_append():
    rng = np.random.default_rng(5)
    B, ps, P, Hk, D, H = 2, 4, 3, 1, 16, 2
    dense = rng.standard_normal((B, P * ps, Hk, D))
    vdense = rng.standard_normal((B, P * ps, Hk, D))
    kn, vn = rng.standard_normal((B, 2, Hk, D)), rng.standard_normal((B, 2, Hk, D))
    q = rng.standard_normal((B, 2, H, D))
    cos, sin = _tables(16, 16)
    table = np.array([[4, 0, 2], [1, 5, 3]])
    kp, vp = np.zeros((6, ps, Hk, D)), np.zeros((6, ps, Hk, D))
    for b in range(B):
        for p in range(P):
            kp[table[b, p]] = dense[b, p * ps:(p + 1) * ps]
            vp[table[b, p]] = vdense[b, p * ps:(p + 1) * ps]
    o_d, l_d, _, _ = oracle.decode_kvcache(q, dense, vdense, [5, 9], kn, vn, cos, sin, True, None, None, True)
    o_p, l_p, _, _ = oracle.decode_kvcache(q, kp, vp, [5, 9], kn, vn, cos, sin, True, table, None, True)
    np.testing.assert_array_equal(o_d, o_p)
    np.testing.assert_array_equal(l_d, l_p)
