"""Pins for the oracle's backward (CPU only): central finite differences in fp64
and torch autograd through scaled_dot_product_attention in float64.

The gradient of f(Q,K,V) = <dO, O(Q,K,V)> with respect to each input is what
the backward returns; perturbing single entries and differencing f pins every
term (a dropped D_i, a wrong sign or a transposed product all fail).
"""
import math

import numpy as np
import pytest
import torch

from fa_inputs import bf16_bits_to_f64, f32_to_bf16_bits
from oracle import head_bwd, head_fwd


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _fd_check(S, D, causal, wl, wr, slope, n_entries, seed):
    q, k, v, do = (_rand((S, D), seed + i) for i in range(4))
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = head_bwd(do, q, k, v, scale, causal, wl, wr, slope)

    def f(qq, kk, vv):
        o, _ = head_fwd(qq, kk, vv, scale, causal, wl, wr, slope)
        return float(np.sum(do * o))

    rng = np.random.default_rng(seed + 99)
    h = 1e-5
    for which, grad in (("q", dq), ("k", dk), ("v", dv)):
        idx = rng.choice(S * D, size=min(n_entries, S * D), replace=False)
        fd = np.empty(len(idx))
        for n, flat in enumerate(idx):
            r, c = divmod(int(flat), D)
            args = {"q": q, "k": k, "v": v}
            plus = {kk: a.copy() for kk, a in args.items()}
            minus = {kk: a.copy() for kk, a in args.items()}
            plus[which][r, c] += h
            minus[which][r, c] -= h
            fd[n] = (f(plus["q"], plus["k"], plus["v"]) - f(minus["q"], minus["k"], minus["v"])) / (2 * h)
        g = grad.reshape(-1)[idx]
        rel = np.linalg.norm(fd - g) / max(np.linalg.norm(g), 1e-30)
        assert rel <= 1e-6, (which, rel)


@pytest.mark.parametrize("causal", [False, True])
def test_fd_tiny_config(causal):
    # B=1, H=2, S=128, D=64 per head; each head checked on 64 entries of Q, K, V
    for head_seed in (100, 200):
        _fd_check(128, 64, causal, -1, -1, None, 64, head_seed)


@pytest.mark.parametrize("wl,wr,slope,causal", [(3, 2, None, False), (4, 0, None, False),
                                                (-1, -1, 0.3, False), (-1, -1, 0.25, True),
                                                (2, 1, 0.5, False)])
def test_fd_window_and_alibi(wl, wr, slope, causal):
    _fd_check(16, 8, causal, wl, wr, slope, 64, 300)


def _band(Sq, Sk, wl, wr):
    N = max(Sq, Sk)
    full = np.ones((N, N), dtype=bool)
    m = full.copy()
    if wr >= 0:
        m &= np.tril(full, wr)
    if wl >= 0:
        m &= np.triu(full, -wl)
    return m[N - Sq:, N - Sk:]


@pytest.mark.parametrize("Sq,Sk,wl,wr", [(24, 24, -1, -1), (24, 24, -1, 0), (13, 29, -1, 0),
                                          (29, 13, -1, 0), (30, 30, 4, 3)])
def test_matches_torch_autograd_float64(Sq, Sk, wl, wr):
    D = 8
    q, k, v = _rand((Sq, D), 40), _rand((Sk, D), 41), _rand((Sk, D), 42)
    do = _rand((Sq, D), 43)
    m = _band(Sq, Sk, wl, wr)
    do[~m.any(axis=1)] = 0.0  # SDPA makes NaN on rows with no key; those rows carry no gradient here
    scale = 0.4
    dq, dk, dv = head_bwd(do, q, k, v, scale, False, wl, wr)
    tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], attn_mask=torch.from_numpy(m), scale=scale)[0, 0]
    out = torch.where(torch.from_numpy(m.any(axis=1))[:, None], out, torch.zeros_like(out))
    (out * torch.from_numpy(do)).sum().backward()
    assert np.allclose(dq, tq.grad.numpy(), atol=1e-12)
    assert np.allclose(dk, tk.grad.numpy(), atol=1e-12)
    assert np.allclose(dv, tv.grad.numpy(), atol=1e-12)


def test_row_blocked_backward_equals_whole():
    S, D = 70, 8
    q, k, v, do = (_rand((S, D), 50 + i) for i in range(4))
    a = head_bwd(do, q, k, v, 0.3, True, -1, -1, 0.1)
    b = head_bwd(do, q, k, v, 0.3, True, -1, -1, 0.1, row_block=16)
    for x, y in zip(a, b):
        assert np.allclose(x, y, atol=1e-13)


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(7).standard_normal(100000).astype(np.float32)
    x[:4] = [0.0, -0.0, 1.00390625, 1.01171875]  # ties: 1 + 2^-8 rounds to 1, 1 + 3*2^-8 rounds up
    mine = bf16_bits_to_f64(f32_to_bf16_bits(x))
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(mine, ref)
