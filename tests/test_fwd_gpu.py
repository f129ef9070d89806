"""GPU parity of fa_fwd against the fp64 oracle on the same seeded bf16 inputs.

Tolerances: bf16 O max |err| <= 2e-2 and relative RMS <= 1e-2; fp32 L max
|err| <= 1e-3 with -inf rows matched exactly.
"""
import math

import numpy as np
import pytest

import oracle
from fa_inputs import alibi_slopes_geometric, attention_inputs, bf16_bits_to_f64
from helpers import assert_bf16_close, assert_lse_close, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _run(B, Sq, Sk, H, D, causal=False, window=(-1, -1), alibi=None, seed=0, scale=None):
    import torch

    import exact_attention_56_gb300 as fa

    inp = attention_inputs(B, Sq, Sk, H, D, seed)
    q, k, v = (to_dev(inp[n]) for n in ("q", "k", "v"))
    al = None if alibi is None else torch.from_numpy(np.ascontiguousarray(alibi, dtype=np.float32)).cuda()
    out, lse = fa.fa_fwd(q, k, v, softmax_scale=scale, causal=causal, window_size=window, alibi_slopes=al)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    o_ref, l_ref = oracle.attention_fwd(*(bf16_bits_to_f64(inp[n]) for n in ("q", "k", "v")), scale, causal,
                                        window, alibi)
    assert_bf16_close(to_f64(out), o_ref, "O")
    assert_lse_close(lse.cpu().numpy().astype(np.float64), l_ref, "L")


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_config(causal):
    # B=1, H=2, Sq=Sk=128, D=64
    _run(1, 128, 128, 2, 64, causal=causal, seed=1)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_head_dims_ragged(D, causal):
    # several tiles plus a ragged tail in both Sq and Sk
    _run(2, 333, 333, 2, D, causal=causal, seed=10 + D)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Sq,Sk", [(77, 300), (300, 77), (1, 513), (257, 1), (130, 130), (200, 256)])
def test_bottom_right_causal_rectangular(Sq, Sk, D):
    _run(1, Sq, Sk, 3, D, causal=True, seed=Sq * 7 + Sk + D)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("window", [(64, 0), (100, 37), (0, 0), (-1, 50), (300, -1)])
def test_sliding_window(window, D):
    # the live key range of a tile starts past key tile 0 for most rows
    _run(1, 500, 640, 2, D, window=window, seed=sum(window) + 1000 + D)


@pytest.mark.parametrize("causal", [False, True])
def test_alibi_per_head_and_per_batch(causal):
    H = 4
    _run(1, 300, 300, H, 64, causal=causal, alibi=alibi_slopes_geometric(H), seed=5)
    slopes = np.stack([alibi_slopes_geometric(H), alibi_slopes_geometric(H)[::-1]]).astype(np.float32)
    _run(2, 200, 260, H, 128, causal=causal, alibi=slopes, seed=6)


def test_explicit_scale():
    _run(1, 256, 256, 2, 128, scale=0.5 / math.sqrt(128), seed=7)


@pytest.mark.parametrize("D,H", [(64, 32), (128, 16)])
@pytest.mark.parametrize("causal", [False, True])
def test_training_sweep_seqlen_512_all_heads(D, H, causal):
    # hidden 2048, seqlen 512, batch 16384/512 = 32: every head compared
    _run(32, 512, 512, H, D, causal=causal, seed=2000 + D + int(causal))


def test_fully_masked_rows_zero():
    # Sq > Sk with causal: the first Sq - Sk rows have no live key
    import torch

    import exact_attention_56_gb300 as fa

    inp = attention_inputs(1, 200, 50, 2, 64, 3)
    q, k, v = (to_dev(inp[n]) for n in ("q", "k", "v"))
    out, lse = fa.fa_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    o = to_f64(out)
    assert np.all(o[:, :150] == 0.0)
    assert np.all(np.isneginf(lse.cpu().numpy()[:, :, :150]))


@pytest.mark.parametrize("Sq,Sk,D", [(400, 512, 128), (300, 300, 64), (129, 700, 256)])
def test_one_key_window_returns_that_value_exactly(Sq, Sk, D):
    # With window (0, 0) each query row i sees only key c(i) = i + Sk - Sq, so
    # softmax weighs it 1 and O_i must equal V_c(i) bit for bit (bf16 V times
    # exactly 1), with L_i = scale * q_i . k_c(i).
    import torch

    import exact_attention_56_gb300 as fa

    inp = attention_inputs(1, Sq, Sk, 2, D, Sq + Sk)
    q, k, v = (to_dev(inp[n]) for n in ("q", "k", "v"))
    out, lse = fa.fa_fwd(q, k, v, window_size=(0, 0))
    torch.cuda.synchronize()
    c = np.arange(Sq) + Sk - Sq
    live = c >= 0
    vv = v.view(torch.int16).cpu().numpy()[0][c[live]]
    oo = out.view(torch.int16).cpu().numpy()[0][live]
    assert np.array_equal(oo, vv)
    q64, k64 = bf16_bits_to_f64(inp["q"])[0], bf16_bits_to_f64(inp["k"])[0]
    l_ref = np.einsum("ihd,ihd->hi", q64[live], k64[c[live]]) / math.sqrt(D)
    assert np.max(np.abs(lse.cpu().numpy()[0][:, live] - l_ref)) <= 1e-3


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal,window", [(False, (-1, -1)), (True, (-1, -1)), (False, (200, 100))])
@pytest.mark.parametrize("Sq,Sk", [(300, 700), (700, 300)])
def test_alibi_several_key_tiles_each_side(D, causal, window, Sq, Sk):
    # With ALiBi the key tiles of a query block run from the diagonal tile
    # leftward, then rightward. Several tiles on each side of the diagonal and a
    # steep slope (0.7, so the max moves by far more than the rescale threshold
    # across tiles in ascending order) exercise that order against the oracle.
    _run(1, Sq, Sk, 2, D, causal=causal, window=window, alibi=np.array([0.7, 0.05], dtype=np.float32), seed=11)
