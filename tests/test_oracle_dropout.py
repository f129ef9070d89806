"""Pins for the oracle's dropout (page "FlashAttention：快速且内存高效的准确注意力机制",
section "参数说明": dropout_p) and its Philox4x32-10 generator (Salmon et al.,
"Parallel random numbers: as easy as 1, 2, 3", SC 2011), both readings stated in
the oracle since the pages give no generator.

Generator: the published known-answer vectors of Philox4x32-10 (Random123's
kat_vectors, tests/golden/philox4x32_10_kat.txt) fix the multipliers, the key
increments, the round count and the output word order; each round is also
inverted independently (modular inverses of the multipliers, Python integers),
so the round structure and key schedule are checked by recovering the counter;
output bits are balanced, the drop fraction matches p, and one flipped counter
bit changes about half the output bits.
Dropout: p = 0 gives the plain result; the forward and autograd backward of an
explicit torch float64 formula with the same mask agree; D = rowsum(dO o O)
still equals sum_j P o dP; averaged over many seeds the output is unbiased.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "philox4x32_10_kat.txt")

M0, M1, W0, W1 = oracle.attention.PHILOX_M0, oracle.attention.PHILOX_M1, oracle.attention.PHILOX_W0, \
    oracle.attention.PHILOX_W1


def _inverse_philox(y, k0, k1):
    inv0, inv1 = pow(M0, -1, 1 << 32), pow(M1, -1, 1 << 32)
    y0, y1, y2, y3 = (int(t) for t in y)
    for r in reversed(range(10)):
        kr0, kr1 = (k0 + r * W0) & 0xFFFFFFFF, (k1 + r * W1) & 0xFFFFFFFF
        x2 = (y1 * inv1) & 0xFFFFFFFF
        x0 = (y3 * inv0) & 0xFFFFFFFF
        x1 = y0 ^ ((M1 * x2) >> 32) ^ kr0
        x3 = y2 ^ ((M0 * x0) >> 32) ^ kr1
        y0, y1, y2, y3 = x0, x1, x2, x3
    return y0, y1, y2, y3


def _kat_rows():
    rows = []
    with open(GOLDEN) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                rows.append([int(t, 16) for t in ln.split()])
    return rows


def test_known_answer_vectors():
    rows = _kat_rows()
    assert len(rows) == 3
    for w in rows:
        y = [int(a[0]) for a in oracle.philox4x32_10(*([c] for c in w[:4]), w[4], w[5])]
        assert y == w[6:], [hex(t) for t in y]
    # the same vectors as one batch of counters (the array path the dropout mask uses)
    cols = np.array([w[:4] for w in rows], dtype=np.uint64).T
    for w, k in zip(rows, range(len(rows))):
        y = oracle.philox4x32_10(*(c[k:k + 1] for c in cols), w[4], w[5])
        assert [int(t[0]) for t in y] == w[6:]


def test_rounds_invert_to_the_counter():
    rng = np.random.default_rng(1)
    for _ in range(200):
        ctr = [int(t) for t in rng.integers(0, 1 << 32, 4, dtype=np.uint64)]
        k0, k1 = (int(t) for t in rng.integers(0, 1 << 32, 2, dtype=np.uint64))
        y = [int(w[0]) for w in oracle.philox4x32_10(*([c] for c in ctr), k0, k1)]
        assert list(_inverse_philox(y, k0, k1)) == ctr


def test_output_bits_balanced_and_drop_fraction():
    n = 1 << 18
    idx = np.arange(n)
    words = np.concatenate(oracle.philox4x32_10(idx, idx >> 7, np.zeros(n), np.full(n, 5), 12345, 678))
    bits = (words[:, None] >> np.arange(32, dtype=np.uint64)) & np.uint64(1)
    freq = bits.mean(axis=0)
    assert np.all(np.abs(freq - 0.5) < 0.004), freq
    for p in (0.1, 0.5, 0.9):
        frac = np.mean(words < np.uint64(oracle.dropout_threshold(p)))
        assert abs(frac - p) < 0.003, (p, frac)


def test_one_counter_bit_changes_half_the_output():
    rng = np.random.default_rng(2)
    base = rng.integers(0, 1 << 32, (4, 4000), dtype=np.uint64)
    a = np.stack(oracle.philox4x32_10(*base, 7, 9))
    for word, bit in ((0, 0), (1, 13), (2, 31), (3, 7)):
        flipped = base.copy()
        flipped[word] ^= np.uint64(1 << bit)
        b = np.stack(oracle.philox4x32_10(*flipped, 7, 9))
        changed = np.unpackbits((a ^ b).astype(">u4").view(np.uint8)).mean() * 32
        assert abs(changed - 16.0) < 0.5, changed


def test_zero_rate_is_the_plain_attention():
    rng = np.random.default_rng(3)
    q, k, v, do = (rng.standard_normal((1, 9, 2, 8)) for _ in range(4))
    o, lse = oracle.attention_fwd_dropout(q, k, v, 0.0, 99, 0, None, True)
    o_ref, l_ref = oracle.attention_fwd(q, k, v, None, True)
    np.testing.assert_array_equal(o, o_ref)
    np.testing.assert_array_equal(lse, l_ref)
    g = oracle.attention_bwd_dropout(do, q, k, v, 0.0, 99, 0, None, True)
    g_ref = oracle.attention_bwd(do, q, k, v, None, True)
    for a, b in zip(g, g_ref):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_explicit_torch_formula_with_the_same_mask(causal):
    rng = np.random.default_rng(4)
    B, Sq, Sk, H, Hk, D, p, seed, off = 2, 7, 11, 4, 2, 8, 0.3, 2 ** 40 + 17, 3
    q, do = rng.standard_normal((B, Sq, H, D)), rng.standard_normal((B, Sq, H, D))
    k, v = rng.standard_normal((B, Sk, Hk, D)), rng.standard_normal((B, Sk, Hk, D))
    o, lse = oracle.attention_fwd_dropout(q, k, v, p, seed, off, 0.4, causal)
    dq, dk, dv = oracle.attention_bwd_dropout(do, q, k, v, p, seed, off, 0.4, causal)
    tq, tk, tv = (torch.from_numpy(x).requires_grad_(True) for x in (q, k, v))
    G = H // Hk
    outs = []
    for b in range(B):
        for h in range(H):
            s = (tq[b, :, h] @ tk[b, :, h // G].T) * 0.4
            if causal:
                s = s.masked_fill(torch.ones(Sq, Sk, dtype=torch.bool).triu(Sk - Sq + 1), -math.inf)
            z = torch.from_numpy(oracle.dropout_scale_matrix(Sq, Sk, b * H + h, p, seed, off))
            outs.append((torch.softmax(s, dim=-1) * z) @ tv[b, :, h // G])
    ref = torch.stack(outs).reshape(B, H, Sq, D).permute(0, 2, 1, 3)
    np.testing.assert_allclose(o, ref.detach().numpy(), rtol=0, atol=1e-12)
    ref.backward(torch.from_numpy(do))
    for name, a, t in (("dQ", dq, tq), ("dK", dk, tk), ("dV", dv, tv)):
        np.testing.assert_allclose(a, t.grad.numpy(), rtol=0, atol=1e-11, err_msg=name)


def test_dropout_rate_and_scale_of_the_mask():
    z = oracle.dropout_scale_matrix(256, 256, 3, 0.25, 5, 0)
    assert set(np.unique(z)) <= {0.0, 1.0 / 0.75}
    assert abs(np.mean(z == 0.0) - 0.25) < 0.01


def test_output_is_unbiased_over_seeds():
    rng = np.random.default_rng(6)
    q, k, v = rng.standard_normal((1, 3, 1, 8)), rng.standard_normal((1, 16, 1, 8)), rng.standard_normal((1, 16, 1, 8))
    o_ref, _ = oracle.attention_fwd(q, k, v)
    samples = np.stack([oracle.attention_fwd_dropout(q, k, v, 0.5, s, 0)[0] for s in range(1500)])
    mean, sd = samples.mean(axis=0), samples.std(axis=0) / math.sqrt(len(samples))
    assert np.all(np.abs(mean - o_ref) <= 5 * sd + 1e-12)
