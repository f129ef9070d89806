"""GPU parity of the backward for inputs far from unit size.

The backward's products run on fp16 copies of q, k, v and dout. fp16 covers
2^-14 .. 65504 in its normal range, while training gradients with respect to
the attention output are often 1e-5 .. 1e-8 (bf16, no loss scaling) and inputs
can exceed fp16's range. The library copies each (sequence, key/value head)
group with a power-of-two factor and takes it back out exactly, so the
gradients keep their precision at any magnitude (page
"FlashAttention：快速且内存高效的准确注意力机制", section "反向传播": the
backward is the plain derivative, with no range condition).

Each input is N(0, c^2) for a factor c per tensor, drawn from the seeded
generator and rounded to bf16, so the oracle sees the same bits. The exact
gradients scale with the inputs: dV with c_dO, dQ with c_dO c_V c_K and dK
with c_dO c_V c_Q (times a softmax-dependent factor of natural size). Each is
compared after dividing both sides by that product, with the bf16 bound
(max |err| <= 2e-2) and the scale-free relative RMS (<= 1e-2, no floor).
q and k are scaled in opposite directions (3e4 and 1/3e4), so that either
one leaves fp16's range while the scores q.k keep their natural size: scaling
q or k alone by 30 would sharpen the softmax 30-fold, a different problem in
which D = rowsum(dO o O), taken from the bf16-rounded output as the method
defines it, limits dQ and dK to about 3e-2 whatever the operand precision.
"""
import numpy as np
import pytest

import oracle
from fa_inputs import bf16_bits_to_f64, normal_bf16_bits
from helpers import assert_bf16_close_scaled, to_dev, to_f64

pytestmark = pytest.mark.gpu

# (c_q, c_k, c_v, c_dO)
SCALES = [
    (1, 1, 1, 1e-4), (1, 1, 1, 1e-6), (1, 1, 1, 1e-8),
    (1e-3, 1, 1, 1), (1, 1e-3, 1, 1), (1, 1, 1e-3, 1),
    (3e4, 1 / 3e4, 1, 1),       # |q| past fp16's 65504, scores of natural size
    (1 / 3e4, 3e4, 1, 1),       # |k| past it
    (1, 1, 30, 1), (1, 1, 3e4, 1),
    (1e-3, 1e-3, 1e-3, 1e-6),   # everything small at once
    (1, 1, 300, 300),           # dP = dO V^T alone would pass fp16's range
]


def _inputs(B, Sq, Sk, H, Hk, D, c, seed):
    cq, ck, cv, cdo = c
    return {"q": normal_bf16_bits((B, Sq, H, D), seed * 8, cq), "k": normal_bf16_bits((B, Sk, Hk, D), seed * 8 + 1, ck),
            "v": normal_bf16_bits((B, Sk, Hk, D), seed * 8 + 2, cv),
            "do": normal_bf16_bits((B, Sq, H, D), seed * 8 + 3, cdo)}


def _factors(c):
    cq, ck, cv, cdo = c
    return cdo * cv * ck, cdo * cv * cq, cdo


def _check(got, refs, c, tag):
    for name, g, r, f in zip(("dQ", "dK", "dV"), got, refs, _factors(c)):
        assert_bf16_close_scaled(to_f64(g), r, f, f"{name} {tag}")


def _run(B, Sq, Sk, H, Hk, D, c, causal, seed, ws=None):
    import torch

    import exact_attention_56_gb300 as fa

    bits = _inputs(B, Sq, Sk, H, Hk, D, c, seed)
    q, k, v, do = (to_dev(bits[n]) for n in ("q", "k", "v", "do"))
    out, lse = fa.fa_fwd(q, k, v, causal=causal)
    dq, dk, dv = fa.fa_bwd(do, q, k, v, out, lse, causal=causal, workspace=ws)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    refs = oracle.attention_bwd(*(bf16_bits_to_f64(bits[n]) for n in ("do", "q", "k", "v")), None, causal)
    _check((dq, dk, dv), refs, c, f"c={c} D={D} causal={causal}")


@pytest.mark.parametrize("c", SCALES, ids=[f"q{a:.3g}_k{b:.3g}_v{x:.3g}_do{d:.3g}" for a, b, x, d in SCALES])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_input_magnitudes(c, D, causal):
    _run(2, 300, 300, 2, 2, D, c, causal, seed=700 + D + int(causal))


@pytest.mark.parametrize("D", [64, 128])
def test_head_groups_small_gradient(D):
    # four query heads on two key/value heads: the factors are per group
    _run(2, 257, 257, 4, 2, D, (1, 1, 30, 1e-6), True, seed=710 + D)


def test_workspace_reused_across_magnitudes():
    # the group maxima are recomputed on every call, whatever the workspace held
    import torch

    import exact_attention_56_gb300 as fa

    B, S, H, D = 2, 300, 2, 128
    ws = torch.empty(fa.fa_bwd_workspace_size(B, S, S, H, D), dtype=torch.uint8, device="cuda")
    for i, c in enumerate(((1, 1, 1, 1e-6), (1, 1, 1, 1), (3e4, 1 / 3e4, 1, 1e-8), (1, 1, 1, 1))):
        _run(B, S, S, H, H, D, c, True, seed=720 + i, ws=ws)


def test_packed_sequences_of_different_magnitudes():
    # each sequence is its own group: one at dO ~ 1e-6, one at 1, one with large v
    import torch

    import exact_attention_56_gb300 as fa

    H, D = 2, 128
    lens = [300, 129, 200]
    cs = [(1, 1, 1, 1e-6), (1, 1, 1, 1), (1, 1, 30, 1e-3)]
    parts = [_inputs(1, n, n, H, H, D, c, 730 + i) for i, (n, c) in enumerate(zip(lens, cs))]
    bits = {x: np.concatenate([p_[x][0] for p_ in parts], axis=0) for x in ("q", "k", "v", "do")}
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q, k, v, do = (to_dev(bits[n]) for n in ("q", "k", "v", "do"))
    cu_d = torch.from_numpy(cu).cuda()
    out, lse = fa.fa_fwd_varlen(q, k, v, cu_d, cu_d, max(lens), max(lens), causal=True)
    dq, dk, dv = fa.fa_bwd_varlen(do, q, k, v, out, lse, cu_d, cu_d, max(lens), max(lens), causal=True)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    refs = oracle.attention_bwd_varlen(*(bf16_bits_to_f64(bits[n]) for n in ("do", "q", "k", "v")), cu, cu, None,
                                       True)
    for i, c in enumerate(cs):
        sl = slice(int(cu[i]), int(cu[i + 1]))
        _check((dq[sl], dk[sl], dv[sl]), [r[sl] for r in refs], c, f"sequence {i} c={c}")


def test_full_size_head_small_gradient():
    # a training-sweep point (S = 4096, D = 128, causal) at dO ~ 1e-6; two heads
    # checked in full against the oracle
    import torch

    import exact_attention_56_gb300 as fa

    B, S, H, D = 1, 4096, 16, 128
    c = (1, 1, 1, 1e-6)
    bits = _inputs(B, S, S, H, H, D, c, 740)
    q, k, v, do = (to_dev(bits[n]) for n in ("q", "k", "v", "do"))
    out, lse = fa.fa_fwd(q, k, v, causal=True)
    dq, dk, dv = fa.fa_bwd(do, q, k, v, out, lse, causal=True)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    scale = 1.0 / np.sqrt(D)
    for h in (0, H - 1):
        heads = [bf16_bits_to_f64(bits[n])[0, :, h, :] for n in ("do", "q", "k", "v")]
        refs = oracle.head_bwd(*heads, scale, True)
        _check((dq[0, :, h], dk[0, :, h], dv[0, :, h]), refs, c, f"head {h}")
