"""Pins for the oracle's split-KV pieces (CPU only): the logsumexp merge is
exact, so any split of the key range merged back must give the unsplit
attention (page "FlashAttention：快速且内存高效的准确注意力机制", section
"2.2：针对推理进行优化": KV loading is split across blocks and a separate
kernel merges the results)."""
import numpy as np
import pytest

from oracle import attention_fwd, combine_partials, decode_splitkv, head_fwd, head_partial


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("n", [1, 2, 3, 7])
@pytest.mark.parametrize("Sq,Sk,causal,wl,wr,slope", [
    (1, 100, True, -1, -1, None), (4, 61, True, -1, -1, 0.2), (3, 50, False, 10, 0, None), (6, 6, True, -1, -1, None)])
def test_split_merge_equals_unsplit(n, Sq, Sk, causal, wl, wr, slope):
    q, k, v = _rand((Sq, 8), 1), _rand((Sk, 8), 2), _rand((Sk, 8), 3)
    o, lse = head_fwd(q, k, v, 0.35, causal, wl, wr, slope)
    bounds = [(Sk * s) // n for s in range(n + 1)]
    parts = [head_partial(q, k, v, bounds[s], bounds[s + 1], 0.35, causal, wl, wr, slope) for s in range(n)]
    om, lm = combine_partials([p[0] for p in parts], [p[1] for p in parts])
    assert np.allclose(om, o, atol=1e-12, rtol=0)
    fin = np.isfinite(lse)
    assert np.array_equal(np.isfinite(lm), fin)
    assert np.allclose(lm[fin], lse[fin], atol=1e-12, rtol=0)


def test_empty_split_weighs_nothing():
    # window (5, 0) at Sq=1, Sk=64 leaves keys 58..63 live: earlier splits are empty
    q, k, v = _rand((1, 8), 4), _rand((64, 8), 5), _rand((64, 8), 6)
    o_e, l_e = head_partial(q, k, v, 0, 32, 0.5, False, 5, 0)
    assert np.all(o_e == 0) and np.isneginf(l_e[0])
    o_l, l_l = head_partial(q, k, v, 32, 64, 0.5, False, 5, 0)
    om, lm = combine_partials([o_e, o_l], [l_e, l_l])
    assert np.allclose(om, o_l, atol=1e-15) and np.allclose(lm, l_l, atol=1e-15)
    oz, lz = combine_partials([o_e, o_e], [l_e, l_e])
    assert np.all(oz == 0) and np.isneginf(lz[0])


def test_equal_lse_is_plain_average():
    a, b = _rand((2, 8), 7), _rand((2, 8), 8)
    l = np.array([0.3, -1.2])
    om, lm = combine_partials([a, b], [l, l])
    assert np.allclose(om, 0.5 * (a + b), atol=1e-15)
    assert np.allclose(lm, l + np.log(2.0), atol=1e-15)


@pytest.mark.parametrize("n", [1, 4, 9])
def test_decode_equals_forward(n):
    B, Sq, Sk, H, D = 2, 1, 77, 3, 8
    q, k, v = _rand((B, Sq, H, D), 9), _rand((B, Sk, H, D), 10), _rand((B, Sk, H, D), 11)
    o1, l1 = decode_splitkv(q, k, v, n, None, True)
    o2, l2 = attention_fwd(q, k, v, None, True)
    assert np.allclose(o1, o2, atol=1e-12) and np.allclose(l1, l2, atol=1e-12)
