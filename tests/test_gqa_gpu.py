"""GPU parity with key/value head groups: k, v (and the KV caches) with Hk < H
heads, query head h reading key/value head h // (H // Hk) (page
"FlashAttention：快速且内存高效的准确注意力机制", section
"代码解读博客：FlashCrossAttention"; the grouping is the reading in the oracle).

Same seeded bf16 inputs on both sides; tolerances as everywhere: bf16 max |err|
<= 2e-2 and relative RMS <= 1e-2, fp32 L max |err| <= 1e-3 with -inf matched.
For the backward, dK and dV of a shared head are the sums over its query heads;
they reach |x| ~ 15, where bf16's own rounding of the output (up to 2^-8 |x|)
exceeds 2e-2 by itself, so they are checked for 2e-2 beyond that rounding.
"""
import numpy as np
import pytest

import oracle
from fa_inputs import alibi_slopes_geometric, bf16_bits_to_f64, normal_bf16_bits
from helpers import assert_bf16_close, assert_bf16_close_beyond_rounding, assert_lse_close, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _inputs(B, Sq, Sk, H, Hk, D, seed, with_dout=False):
    out = {
        "q": normal_bf16_bits((B, Sq, H, D), seed * 8 + 0),
        "k": normal_bf16_bits((B, Sk, Hk, D), seed * 8 + 1),
        "v": normal_bf16_bits((B, Sk, Hk, D), seed * 8 + 2),
    }
    if with_dout:
        out["dout"] = normal_bf16_bits((B, Sq, H, D), seed * 8 + 3)
    return out


def _alibi(alibi, dev):
    import torch

    return None if alibi is None else torch.from_numpy(np.ascontiguousarray(alibi, dtype=np.float32)).to(dev)


def _fwd(B, Sq, Sk, H, Hk, D, causal=False, window=(-1, -1), alibi=None, seed=0):
    import torch

    import exact_attention_56_gb300 as fa

    inp = _inputs(B, Sq, Sk, H, Hk, D, seed)
    q, k, v = (to_dev(inp[n]) for n in ("q", "k", "v"))
    out, lse = fa.fa_fwd(q, k, v, causal=causal, window_size=window, alibi_slopes=_alibi(alibi, q.device))
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    o_ref, l_ref = oracle.attention_fwd(*(bf16_bits_to_f64(inp[n]) for n in ("q", "k", "v")), None, causal, window,
                                        alibi)
    assert_bf16_close(to_f64(out), o_ref, "O")
    assert_lse_close(lse.cpu().numpy().astype(np.float64), l_ref, "L")


def _bwd(B, Sq, Sk, H, Hk, D, causal=False, window=(-1, -1), alibi=None, seed=0, deterministic=False):
    import torch

    import exact_attention_56_gb300 as fa

    inp = _inputs(B, Sq, Sk, H, Hk, D, seed, with_dout=True)
    q, k, v, do = (to_dev(inp[n]) for n in ("q", "k", "v", "dout"))
    kw = dict(causal=causal, window_size=window, alibi_slopes=_alibi(alibi, q.device))
    out, lse = fa.fa_fwd(q, k, v, **kw)
    dq, dk, dv = fa.fa_bwd(do, q, k, v, out, lse, deterministic=deterministic, **kw)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    assert tuple(dk.shape) == (B, Sk, Hk, D) and tuple(dv.shape) == (B, Sk, Hk, D)
    f64 = [bf16_bits_to_f64(inp[n]) for n in ("dout", "q", "k", "v")]
    rq, rk, rv = oracle.attention_bwd(*f64, None, causal, window, alibi)
    assert_bf16_close(to_f64(dq), rq, "dQ")
    assert_bf16_close_beyond_rounding(to_f64(dk), rk, "dK")
    assert_bf16_close_beyond_rounding(to_f64(dv), rv, "dV")
    return dq, dk, dv


@pytest.mark.parametrize("Hk", [1, 2, 4])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_groups(Hk, D, causal):
    _fwd(2, 333, 333, 8, Hk, D, causal=causal, seed=100 + Hk + D + int(causal))


@pytest.mark.parametrize("Hk", [1, 2])
def test_forward_groups_long_head_dim(Hk):
    _fwd(1, 300, 300, 4, Hk, 256, causal=True, seed=130 + Hk)


def test_forward_groups_rectangular_window_alibi():
    _fwd(1, 200, 520, 6, 3, 128, causal=True, seed=140)
    _fwd(1, 400, 512, 4, 2, 128, window=(64, 0), seed=141)
    _fwd(2, 300, 300, 8, 2, 64, causal=True, alibi=alibi_slopes_geometric(8), seed=142)


@pytest.mark.parametrize("Hk", [1, 2])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_groups(Hk, D, causal):
    _bwd(2, 333, 333, 8, Hk, D, causal=causal, seed=200 + Hk + D + int(causal))


def test_backward_groups_rectangular_window_alibi():
    _bwd(1, 77, 300, 4, 2, 128, causal=True, seed=210)
    _bwd(1, 300, 77, 4, 1, 128, causal=True, seed=211)
    _bwd(1, 400, 512, 4, 2, 128, window=(100, 37), seed=212)
    _bwd(1, 300, 300, 8, 4, 64, causal=True, alibi=alibi_slopes_geometric(8), seed=213)


def test_backward_groups_training_shape():
    # hidden 4096 as 32 query heads over 8 key/value heads, seqlen 1024, causal
    _bwd(2, 1024, 1024, 32, 8, 128, causal=True, seed=220)


def test_backward_groups_bitwise_repeatable():
    import torch

    a = _bwd(2, 700, 700, 8, 2, 128, causal=True, seed=230, deterministic=True)
    b = _bwd(2, 700, 700, 8, 2, 128, causal=True, seed=230, deterministic=True)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("Hk", [1, 2])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("Sq", [1, 4])
def test_decode_groups(Hk, D, Sq):
    import torch

    import exact_attention_56_gb300 as fa

    B, Sk, H = 3, 1000, 8
    inp = _inputs(B, Sq, Sk, H, Hk, D, 300 + Hk + D + Sq)
    q, k, v = (to_dev(inp[n]) for n in ("q", "k", "v"))
    for n in (0, 3):
        out, lse = fa.fa_decode_splitkv(q, k, v, causal=True, num_splits=n)
        torch.cuda.synchronize()
        st, word = fa.fa_device_status()
        assert st == fa.FA_OK, hex(word)
        o_ref, l_ref = oracle.attention_fwd(*(bf16_bits_to_f64(inp[x]) for x in ("q", "k", "v")), None, True)
        assert_bf16_close(to_f64(out), o_ref, f"O (splits {n})")
        assert_lse_close(lse.cpu().numpy().astype(np.float64), l_ref, f"L (splits {n})")


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("H,Hk,Sq", [(6, 2, 1), (6, 2, 3), (4, 4, 3), (16, 1, 2), (12, 4, 2), (8, 2, 16),
                                     (64, 1, 3), (128, 1, 2)])
def test_decode_query_pairs_share_a_cta(H, Hk, Sq, D):
    # The (query row, query head) pairs of one key/value head share a split CTA:
    # up to four in the CUDA-core kernel, from four on as the rows of a tensor-core
    # tile. These shapes leave partial blocks (3 or 9 pairs), mix query rows with
    # different causal limits in one block, and put 32 pairs on one head (MQA).
    # G * Sq above 128 (64 x 3, 128 x 2) splits a head's pairs over several
    # tensor-core row blocks; Sq = 16 is the largest query length decode takes.
    import torch

    import exact_attention_56_gb300 as fa

    B, Sk = 2, 777
    inp = _inputs(B, Sq, Sk, H, Hk, D, 350 + H + Hk + Sq + D)
    q, k, v = (to_dev(inp[n]) for n in ("q", "k", "v"))
    f64 = [bf16_bits_to_f64(inp[x]) for x in ("q", "k", "v")]
    # the causal ALiBi case spans all 7 key tiles (run from the last tile down with ALiBi)
    cases = [dict(causal=True), dict(causal=False, window=(100, 0), alibi=alibi_slopes_geometric(H)),
             dict(causal=True, alibi=alibi_slopes_geometric(H))]
    for case in cases:
        window, alibi = case.get("window", (-1, -1)), case.get("alibi")
        for n in (0, 1, 5):
            out, lse = fa.fa_decode_splitkv(q, k, v, causal=case["causal"], window_size=window,
                                            alibi_slopes=_alibi(alibi, q.device), num_splits=n)
            torch.cuda.synchronize()
            st, word = fa.fa_device_status()
            assert st == fa.FA_OK, hex(word)
            o_ref, l_ref = oracle.attention_fwd(*f64, None, case["causal"], window, alibi)
            assert_bf16_close(to_f64(out), o_ref, f"O ({case}, splits {n})")
            assert_lse_close(lse.cpu().numpy().astype(np.float64), l_ref, f"L ({case}, splits {n})")


def test_binding_rejects_heads_that_do_not_divide():
    import torch

    import exact_attention_56_gb300 as fa

    q = torch.zeros((1, 8, 6, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 8, 4, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        fa.fa_fwd(q, k, k)
