"""Pins for the oracle's paged-cache decode (page "FlashAttention：快速且内存高效的准确注意力机制",
section "2.5：分页KV缓存", which names the feature; the page layout is the reading
stated in the oracle). Checks: an identity page table reproduces the dense
cache; permuting pages together with their table entries changes nothing; keys
past each sequence's length are never read; torch SDPA in float64 on a cache
gathered with torch.index_select agrees."""
import numpy as np
import pytest
import torch

import oracle


def _draw(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _dense_to_pages(k, page_size):
    B, Sk, Hk, D = k.shape
    P = Sk // page_size
    return k.reshape(B * P, page_size, Hk, D), np.arange(B * P).reshape(B, P)


def test_identity_table_equals_dense():
    B, Sq, Sk, H, Hk, D, ps = 2, 3, 12, 4, 2, 8, 4
    q, k, v = _draw((B, Sq, H, D), 1), _draw((B, Sk, Hk, D), 2), _draw((B, Sk, Hk, D), 3)
    kp, table = _dense_to_pages(k, ps)
    vp, _ = _dense_to_pages(v, ps)
    o, lse = oracle.decode_paged(q, kp, vp, table, [Sk] * B, None, True)
    o_ref, l_ref = oracle.attention_fwd(q, k, v, None, True)
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(lse, l_ref)


def test_permuted_pages_and_garbage_tails_change_nothing():
    B, Sq, H, D, ps, P = 3, 2, 2, 8, 4, 3
    lens = [5, 12, 1]
    q = _draw((B, Sq, H, D), 4)
    kp, vp = _draw((B * P, ps, H, D), 5), _draw((B * P, ps, H, D), 6)
    table = np.arange(B * P).reshape(B, P)
    o, lse = oracle.decode_paged(q, kp, vp, table, lens, None, True, (3, 0))
    perm = np.random.default_rng(7).permutation(B * P)
    inv = np.argsort(perm)
    o2, lse2 = oracle.decode_paged(q, kp[perm], vp[perm], inv[table], lens, None, True, (3, 0))
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)
    kg, vg = kp.copy(), vp.copy()
    for b, n in enumerate(lens):  # poison every key past the sequence's length
        for p in range(P):
            lo = max(0, n - p * ps)
            kg[table[b, p], lo:] = 1e6
            vg[table[b, p], lo:] = -1e6
    o3, lse3 = oracle.decode_paged(q, kg, vg, table, lens, None, True, (3, 0))
    np.testing.assert_array_equal(o, o3)
    np.testing.assert_array_equal(lse, lse3)


def test_empty_sequence_gives_zero_and_minus_inf():
    q = _draw((2, 1, 2, 8), 8)
    kp = _draw((2, 4, 2, 8), 9)
    o, lse = oracle.decode_paged(q, kp, kp, np.array([[0], [1]]), [0, 3])
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


@pytest.mark.parametrize("Hk", [4, 1])
def test_matches_torch_sdpa_on_index_select_gather(Hk):
    B, Sq, H, D, ps, P = 2, 1, 4, 8, 4, 4
    lens = [13, 7]
    q = _draw((B, Sq, H, D), 10)
    kp, vp = _draw((B * P + 2, ps, Hk, D), 11), _draw((B * P + 2, ps, Hk, D), 12)
    table = np.random.default_rng(13).permutation(B * P + 2)[:B * P].reshape(B, P)
    o, lse = oracle.decode_paged(q, kp, vp, table, lens, 0.3, True)
    tk, tv = torch.from_numpy(kp), torch.from_numpy(vp)
    for b, n in enumerate(lens):
        idx = torch.from_numpy(np.ascontiguousarray(table[b]))
        kb = torch.index_select(tk, 0, idx).reshape(-1, Hk, D)[:n]
        vb = torch.index_select(tv, 0, idx).reshape(-1, Hk, D)[:n]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[b]).permute(1, 0, 2)[None], kb.permute(1, 0, 2)[None], vb.permute(1, 0, 2)[None],
            scale=0.3, enable_gqa=True)[0].permute(1, 0, 2).numpy()
        np.testing.assert_allclose(o[b], ref, rtol=0, atol=1e-12)
