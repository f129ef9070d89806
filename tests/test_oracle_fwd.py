"""Pins for the oracle's forward (CPU only).

Checks against what the page and the mathematics fix, never against the
oracle's own formula retyped: softmax invariants, the fully-masked-row rule
(page "FlashAttention：快速且内存高效的准确注意力机制", section "2.1"),
closed forms (Sk = 1, constant V, Q = 0, the geometric ALiBi weights), and the
independent library routine torch.nn.functional.scaled_dot_product_attention
in float64 on the CPU.
"""
import math

import numpy as np
import pytest
import scipy.linalg
import scipy.special
import torch

from oracle import attention_fwd, head_fwd, live_mask


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("Sq,Sk,causal,wl,wr", [
    (16, 16, False, -1, -1), (16, 16, True, -1, -1), (9, 23, True, -1, -1),
    (23, 9, True, -1, -1), (20, 20, False, 3, 2), (12, 30, False, 4, 0)])
def test_rows_sum_to_one_and_lse(Sq, Sk, causal, wl, wr):
    q, k, v = _rand((Sq, 8), 1), _rand((Sk, 8), 2), _rand((Sk, 8), 3)
    o, lse, s, p = head_fwd(q, k, v, 0.3, causal, wl, wr, return_p=True)
    live = live_mask(Sq, Sk, causal, wl, wr)
    has = live.any(axis=1)
    assert np.allclose(p[has].sum(axis=1), 1.0, atol=1e-12, rtol=0)
    assert np.all(p[~live] == 0.0)
    # L is the natural-log logsumexp of the live scores (scipy as the independent routine)
    for i in np.nonzero(has)[0]:
        assert abs(lse[i] - scipy.special.logsumexp(s[i][live[i]])) < 1e-12
    assert np.all(np.isneginf(lse[~has]))
    assert np.all(o[~has] == 0.0)


def test_fully_masked_rows_give_zero():
    # Sq = 5, Sk = 2, causal: rows 0-2 see no key (section "2.1", last sentence)
    q, k, v = _rand((5, 4), 4), _rand((2, 4), 5), _rand((2, 4), 6)
    o, lse = head_fwd(q, k, v, 0.5, causal=True)
    assert np.all(o[:3] == 0.0) and np.all(np.isneginf(lse[:3]))
    assert np.allclose(o[3], v[0], atol=1e-15)  # row 3 sees only key 0
    assert np.all(np.isfinite(lse[3:]))


def test_single_key_returns_that_value():
    q, k, v = _rand((7, 16), 7), _rand((1, 16), 8), _rand((1, 16), 9)
    o, lse = head_fwd(q, k, v, 0.25)
    assert np.allclose(o, np.broadcast_to(v[0], o.shape), atol=1e-15)
    assert np.allclose(lse, 0.25 * (q @ k[0]), atol=1e-12)


def test_constant_value_rows():
    q, k = _rand((11, 8), 10), _rand((13, 8), 11)
    vec = _rand((8,), 12)
    v = np.tile(vec, (13, 1))
    o, _ = head_fwd(q, k, v, 0.7, causal=True)
    assert np.allclose(o, np.tile(vec, (11, 1)), atol=1e-13)


@pytest.mark.parametrize("causal,wl,wr", [(False, -1, -1), (True, -1, -1), (False, 2, 1)])
def test_zero_query_is_mean_of_live_values(causal, wl, wr):
    Sq, Sk = 6, 10
    q, k, v = np.zeros((Sq, 4)), _rand((Sk, 4), 13), _rand((Sk, 4), 14)
    o, lse = head_fwd(q, k, v, 1.0, causal, wl, wr)
    live = live_mask(Sq, Sk, causal, wl, wr)
    for i in range(Sq):
        n = live[i].sum()
        assert np.allclose(o[i], v[live[i]].mean(axis=0), atol=1e-14)
        assert abs(lse[i] - math.log(n)) < 1e-14


def _sdpa64(q, k, v, scale, mask_bool=None, bias=None):
    """torch's SDPA in float64 on the CPU, (Sq,D) per head."""
    tq = torch.from_numpy(q)[None, None]
    tk = torch.from_numpy(k)[None, None]
    tv = torch.from_numpy(v)[None, None]
    attn = None
    if mask_bool is not None and bias is not None:
        attn = torch.from_numpy(np.where(mask_bool, bias, -np.inf))
    elif mask_bool is not None:
        attn = torch.from_numpy(mask_bool)
    elif bias is not None:
        attn = torch.from_numpy(bias)
    return torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=attn, scale=scale)[0, 0].numpy()


def _band(Sq, Sk, wl, wr):
    # bottom-right corner of an N x N band (independent of the oracle's index formula)
    N = max(Sq, Sk)
    full = np.ones((N, N), dtype=bool)
    m = full.copy()
    if wr >= 0:
        m &= np.tril(full, wr)
    if wl >= 0:
        m &= np.triu(full, -wl)
    return m[N - Sq:, N - Sk:]


def _alibi_toeplitz(Sq, Sk, slope):
    # distance matrix from scipy's toeplitz, cut at the bottom-right corner
    N = max(Sq, Sk)
    dist = scipy.linalg.toeplitz(np.arange(N, dtype=np.float64))
    return -slope * dist[N - Sq:, N - Sk:]


@pytest.mark.parametrize("Sq,Sk,wl,wr,slope", [
    (32, 32, -1, -1, None), (32, 32, -1, 0, None), (17, 45, -1, 0, None), (40, 24, -1, 0, None),
    (33, 33, 5, 0, None), (29, 37, 3, 4, None), (32, 32, -1, -1, 0.25), (32, 32, -1, 0, 0.0625),
    (20, 52, -1, 0, 0.5), (24, 24, 6, 2, 0.125)])
def test_matches_torch_sdpa_float64(Sq, Sk, wl, wr, slope):
    D = 16
    q, k, v = _rand((Sq, D), 20), _rand((Sk, D), 21), _rand((Sk, D), 22)
    scale = 1.0 / math.sqrt(D)
    o, _ = head_fwd(q, k, v, scale, False, wl, wr, slope)
    m = _band(Sq, Sk, wl, wr)
    bias = None if slope is None else _alibi_toeplitz(Sq, Sk, slope)
    ref = _sdpa64(q, k, v, scale, m, bias)
    has = m.any(axis=1)
    assert np.allclose(o[has], ref[has], atol=1e-12, rtol=0)


@pytest.mark.parametrize("S,slope,causal", [(12, 0.5, False), (12, 0.5, True), (9, 0.125, False)])
def test_alibi_geometric_closed_form(S, slope, causal):
    # K = 0 makes every score equal to the bias; V = identity returns P itself.
    # Then row i of P is r^|i-j| / sum_j r^|i-j| with r = exp(-slope), whose
    # normaliser is a geometric series summed in closed form.
    q = _rand((S, S), 23)
    k = np.zeros((S, S))
    v = np.eye(S)
    o, lse = head_fwd(q, k, v, 1.0, causal, -1, -1, slope)
    r = math.exp(-slope)
    for i in range(S):
        left = (1 - r ** (i + 1)) / (1 - r)            # j = i, i-1, ..., 0
        right = 0.0 if causal else r * (1 - r ** (S - 1 - i)) / (1 - r)  # j = i+1..S-1
        z = left + right
        for j in range(S):
            want = 0.0 if (causal and j > i) else r ** abs(i - j) / z
            assert abs(o[i, j] - want) < 1e-14
        assert abs(lse[i] - math.log(z)) < 1e-12


def test_batched_layout_matches_heads():
    B, Sq, Sk, H, D = 2, 5, 7, 3, 4
    q, k, v = _rand((B, Sq, H, D), 30), _rand((B, Sk, H, D), 31), _rand((B, Sk, H, D), 32)
    slopes = np.array([[0.1, 0.2, 0.3], [0.4, 0.5, 0.6]])
    o, lse = attention_fwd(q, k, v, None, True, (-1, -1), slopes)
    for b in range(B):
        for h in range(H):
            oh, lh = head_fwd(q[b, :, h], k[b, :, h], v[b, :, h], 0.5, True, -1, -1, slopes[b, h])
            assert np.array_equal(o[b, :, h], oh) and np.array_equal(lse[b, h], lh)
