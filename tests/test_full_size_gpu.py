"""Parity at the workloads' full sizes, in the launch configuration the bench times.

Inputs are drawn on the device (seeded torch N(0,1) -> bf16); the oracle gets
the exact fp64 upcast of the sampled heads. Forward outputs are checked on a
seeded sample of query rows of the first, the last and two seeded random
(b, h); gradients on whole sampled heads (the oracle's backward runs per head
in row blocks). Tolerances as everywhere: bf16 max |err| <= 2e-2 and relative
RMS <= 1e-2, fp32 L max |err| <= 1e-3 with -inf matched.
"""
import math

import numpy as np
import pytest

import oracle
from fa_inputs import alibi_slopes_geometric, device_normal_bf16
from helpers import assert_bf16_close, assert_lse_close

pytestmark = pytest.mark.gpu


def _heads(B, H, seed, n_random=2):
    rng = np.random.default_rng(seed)
    hs = {(0, 0), (B - 1, H - 1)}
    while len(hs) < min(B * H, 2 + n_random):
        hs.add((int(rng.integers(B)), int(rng.integers(H))))
    return sorted(hs)


def _head64(t, b, h):
    return t[b, :, h, :].float().cpu().numpy().astype(np.float64)


def _check_fwd(q, k, v, out, lse, causal, window, alibi, heads, n_rows, seed):
    B, Sq, H, D = q.shape
    scale = 1.0 / math.sqrt(D)
    rng = np.random.default_rng(seed)
    for b, h in heads:
        rows = np.unique(np.concatenate([[0, Sq - 1], rng.integers(0, Sq, size=n_rows)]))
        slope = None if alibi is None else float(alibi[h])
        o_ref, l_ref = oracle.head_fwd(_head64(q, b, h), _head64(k, b, h), _head64(v, b, h), scale, causal,
                                       window[0], window[1], slope, rows=rows)
        o = out[b, rows, h, :].float().cpu().numpy().astype(np.float64)
        assert_bf16_close(o, o_ref, f"O (b={b}, h={h})")
        assert_lse_close(lse[b, h, rows].cpu().numpy().astype(np.float64), l_ref, f"L (b={b}, h={h})")


def _check_bwd(do, q, k, v, grads, causal, window, alibi, heads):
    D = q.shape[3]
    scale = 1.0 / math.sqrt(D)
    for b, h in heads[:2]:
        slope = None if alibi is None else float(alibi[h])
        refs = oracle.head_bwd(_head64(do, b, h), _head64(q, b, h), _head64(k, b, h), _head64(v, b, h), scale,
                               causal, window[0], window[1], slope, row_block=512)
        for name, g, r in zip(("dQ", "dK", "dV"), grads, refs):
            assert_bf16_close(_head64(g, b, h), r, f"{name} (b={b}, h={h})")


def _run(B, Sq, Sk, H, D, causal, window=(-1, -1), alibi=None, bwd=True, seed=0, n_rows=256):
    import torch

    import exact_attention_56_gb300 as fa

    dev = torch.device("cuda", 0)
    q = device_normal_bf16((B, Sq, H, D), seed * 8 + 0, dev)
    k = device_normal_bf16((B, Sk, H, D), seed * 8 + 1, dev)
    v = device_normal_bf16((B, Sk, H, D), seed * 8 + 2, dev)
    al = None if alibi is None else torch.from_numpy(alibi).to(dev)
    out, lse = fa.fa_fwd(q, k, v, causal=causal, window_size=window, alibi_slopes=al)
    grads = None
    if bwd:
        do = device_normal_bf16((B, Sq, H, D), seed * 8 + 3, dev)
        grads = fa.fa_bwd(do, q, k, v, out, lse, causal=causal, window_size=window, alibi_slopes=al)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    heads = _heads(B, H, seed)
    _check_fwd(q, k, v, out, lse, causal, window, alibi, heads, n_rows, seed)
    if bwd:
        _check_bwd(do, q, k, v, grads, causal, window, alibi, heads)


@pytest.mark.parametrize("D,H", [(64, 32), (128, 16)])
@pytest.mark.parametrize("causal", [False, True])
def test_training_sweep_16k(D, H, causal):
    _run(1, 16384, 16384, H, D, causal, seed=4100 + D + int(causal))


@pytest.mark.parametrize("S", [1024, 4096])
def test_training_sweep_mid(S):
    _run(16384 // S, S, S, 16, 128, True, seed=4200 + S)


def test_mask_variant_a_causal_rectangular():
    _run(2, 2048, 8192, 16, 128, True, seed=4301)


def test_mask_variant_b_sliding_window():
    _run(2, 16384, 16384, 16, 128, False, window=(4096, 0), seed=4302)


def test_mask_variant_c_causal_alibi():
    _run(2, 4096, 4096, 16, 128, True, alibi=alibi_slopes_geometric(16), seed=4303)


@pytest.mark.parametrize("causal", [False, True])
def test_long_head_dim_forward(causal):
    _run(1, 16384, 16384, 8, 256, causal, bwd=False, seed=4400 + int(causal))


@pytest.mark.parametrize("Sk", [4096, 32768, 131072])
def test_decode_full_size(Sk):
    import torch

    import exact_attention_56_gb300 as fa

    B, H, D = 16, 32, 128
    dev = torch.device("cuda", 0)
    q = device_normal_bf16((B, 1, H, D), 4500 + Sk, dev)
    k = device_normal_bf16((B, Sk, H, D), 4501 + Sk, dev)
    v = device_normal_bf16((B, Sk, H, D), 4502 + Sk, dev)
    out, lse = fa.fa_decode_splitkv(q, k, v, causal=True)  # split count chosen by the library, as in the bench
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    for b, h in _heads(B, H, Sk, n_random=4):
        o_ref, l_ref = oracle.head_fwd(_head64(q, b, h), _head64(k, b, h), _head64(v, b, h), 1.0 / math.sqrt(D),
                                       True)
        assert_bf16_close(out[b, :, h, :].float().cpu().numpy().astype(np.float64), o_ref, f"O (b={b}, h={h})")
        assert_lse_close(lse[b, h, :].cpu().numpy().astype(np.float64), l_ref, f"L (b={b}, h={h})")
    del k, v
    torch.cuda.empty_cache()
