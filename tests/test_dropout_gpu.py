"""GPU parity of attention with dropout (page "FlashAttention：快速且内存高效的准确注意力机制",
section "参数说明": dropout_p; the Philox4x32-10 mask rule is the reading stated in
include/fa.h and the oracle, each side implementing the generator from its
published definition).

The mask is checked entry for entry: with V the identity (Sk = D) the output
rows are P o Z themselves, so the GPU's dropped entries are exactly its zeros.
Values follow the tolerances used everywhere: bf16 max |err| <= 2e-2 and
relative RMS <= 1e-2, fp32 L max |err| <= 1e-3. Dropout scales kept entries by
1 / (1 - p), so dK, dV can reach the magnitudes where bf16's own rounding is
checked separately (2e-2 beyond 2^-8 |x|).
"""
import numpy as np
import pytest

import oracle
from fa_inputs import alibi_slopes_geometric, bf16_bits_to_f64, normal_bf16_bits
from helpers import assert_bf16_close, assert_bf16_close_beyond_rounding, assert_lse_close, to_dev, to_f64

pytestmark = pytest.mark.gpu

SEED = (1 << 40) + 12345


def _inputs(B, Sq, Sk, H, Hk, D, seed, with_dout=False):
    out = {"q": normal_bf16_bits((B, Sq, H, D), seed * 8), "k": normal_bf16_bits((B, Sk, Hk, D), seed * 8 + 1),
           "v": normal_bf16_bits((B, Sk, Hk, D), seed * 8 + 2)}
    if with_dout:
        out["do"] = normal_bf16_bits((B, Sq, H, D), seed * 8 + 3)
    return out


def test_mask_matches_entry_for_entry():
    import torch

    import exact_attention_56_gb300 as fa

    B, S, H, D = 2, 200, 2, 64
    inp = _inputs(B, S, D, H, H, D, 800)
    q, k = to_dev(inp["q"]), to_dev(inp["k"])
    eye = torch.eye(D, dtype=torch.bfloat16, device="cuda")
    v = eye[None, :, None, :].expand(B, D, H, D).contiguous()  # Sk = D keys, V row j = e_j
    for p in (0.1, 0.5):
        out, _ = fa.fa_fwd_dropout(q, k, v, p, SEED, 7)
        torch.cuda.synchronize()
        o = to_f64(out)
        for b in range(B):
            for h in range(H):
                z = oracle.dropout_scale_matrix(S, D, b * H + h, p, SEED, 7)
                assert np.array_equal(o[b, :, h, :] == 0.0, z == 0.0), (p, b, h)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_dropout(D, causal):
    import torch

    import exact_attention_56_gb300 as fa

    B, S, H, p = 2, 333, 2, 0.2
    inp = _inputs(B, S, S, H, H, D, 810 + D + int(causal))
    q, k, v = (to_dev(inp[n]) for n in ("q", "k", "v"))
    out, lse = fa.fa_fwd_dropout(q, k, v, p, SEED, 3, causal=causal)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    o_ref, l_ref = oracle.attention_fwd_dropout(*(bf16_bits_to_f64(inp[n]) for n in ("q", "k", "v")), p, SEED, 3,
                                                None, causal)
    assert_bf16_close(to_f64(out), o_ref, "O")
    assert_lse_close(lse.cpu().numpy().astype(np.float64), l_ref, "L")


def _bwd(B, S, H, Hk, D, p, causal, seed, window=(-1, -1), alibi=None):
    import torch

    import exact_attention_56_gb300 as fa

    inp = _inputs(B, S, S, H, Hk, D, seed, with_dout=True)
    q, k, v, do = (to_dev(inp[n]) for n in ("q", "k", "v", "do"))
    al = None if alibi is None else torch.from_numpy(np.ascontiguousarray(alibi, dtype=np.float32)).cuda()
    kw = dict(causal=causal, window_size=window, alibi_slopes=al)
    out, lse = fa.fa_fwd_dropout(q, k, v, p, SEED, 11, **kw)
    dq, dk, dv = fa.fa_bwd_dropout(do, q, k, v, out, lse, p, SEED, 11, **kw)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    f64 = [bf16_bits_to_f64(inp[n]) for n in ("do", "q", "k", "v")]
    rq, rk, rv = oracle.attention_bwd_dropout(*f64, p, SEED, 11, None, causal, window, alibi)
    assert_bf16_close(to_f64(dq), rq, "dQ")
    assert_bf16_close_beyond_rounding(to_f64(dk), rk, "dK")
    assert_bf16_close_beyond_rounding(to_f64(dv), rv, "dV")
    return dq, dk, dv


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_dropout(D, causal):
    _bwd(2, 333, 2, 2, D, 0.2, causal, 820 + D + int(causal))


def test_backward_dropout_groups_window_alibi():
    _bwd(1, 300, 4, 2, 128, 0.3, True, 830)
    _bwd(1, 400, 2, 2, 128, 0.1, False, 831, window=(64, 0))
    _bwd(1, 300, 4, 4, 64, 0.2, True, 832, alibi=alibi_slopes_geometric(4))


def test_same_seed_repeats_other_offset_differs():
    import torch

    import exact_attention_56_gb300 as fa

    inp = _inputs(1, 256, 256, 2, 2, 128, 840)
    q, k, v = (to_dev(inp[n]) for n in ("q", "k", "v"))
    a, _ = fa.fa_fwd_dropout(q, k, v, 0.3, SEED, 0)
    b, _ = fa.fa_fwd_dropout(q, k, v, 0.3, SEED, 0)
    c, _ = fa.fa_fwd_dropout(q, k, v, 0.3, SEED, 1)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert not torch.equal(a.view(torch.int16), c.view(torch.int16))
