"""GPU parity of split-KV decode over a paged KV cache (page
"FlashAttention：快速且内存高效的准确注意力机制", section "2.5：分页KV缓存"; the page
layout is the reading stated in include/fa.h and the oracle).

Pages are shuffled through the block table, spare pages hold unrelated data,
and the sequences mix one key, empty, ragged and multi-page lengths. Tolerances
as everywhere: bf16 max |err| <= 2e-2 and relative RMS <= 1e-2, fp32 L max
|err| <= 1e-3 with -inf matched.
"""
import numpy as np
import pytest

import oracle
from fa_inputs import alibi_slopes_geometric, bf16_bits_to_f64, normal_bf16_bits
from helpers import assert_bf16_close, assert_lse_close, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _case(B, Sq, lens, H, Hk, D, ps, seed, spare=3):
    P = max(1, max((n + ps - 1) // ps for n in lens))
    num_pages = B * P + spare
    q_b = normal_bf16_bits((B, Sq, H, D), seed * 8)
    k_b = normal_bf16_bits((num_pages, ps, Hk, D), seed * 8 + 1)
    v_b = normal_bf16_bits((num_pages, ps, Hk, D), seed * 8 + 2)
    table = np.random.default_rng(seed).permutation(num_pages)[:B * P].reshape(B, P).astype(np.int32)
    return q_b, k_b, v_b, table, np.asarray(lens, dtype=np.int32)


def _run(B, Sq, lens, H, Hk, D, ps, seed, causal=True, window=(-1, -1), alibi=None, splits=(0, 3)):
    import torch

    import exact_attention_56_gb300 as fa

    q_b, k_b, v_b, table, sl = _case(B, Sq, lens, H, Hk, D, ps, seed)
    q, kp, vp = to_dev(q_b), to_dev(k_b), to_dev(v_b)
    bt, sk = torch.from_numpy(table).cuda(), torch.from_numpy(sl).cuda()
    al = None if alibi is None else torch.from_numpy(np.ascontiguousarray(alibi, dtype=np.float32)).cuda()
    o_ref, l_ref = oracle.decode_paged(bf16_bits_to_f64(q_b), bf16_bits_to_f64(k_b), bf16_bits_to_f64(v_b), table,
                                       sl, None, causal, window, alibi)
    for n in splits:
        out, lse = fa.fa_decode_paged(q, kp, vp, bt, sk, max(lens), causal=causal, window_size=window,
                                      alibi_slopes=al, num_splits=n)
        torch.cuda.synchronize()
        st, word = fa.fa_device_status()
        assert st == fa.FA_OK, hex(word)
        assert_bf16_close(to_f64(out), o_ref, f"O (splits {n})")
        assert_lse_close(lse.cpu().numpy().astype(np.float64), l_ref, f"L (splits {n})")


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("Hk", [8, 2])
@pytest.mark.parametrize("Sq", [1, 4])
def test_paged_decode(D, Hk, Sq):
    _run(4, Sq, [1, 700, 0, 300], 8, Hk, D, 128, seed=600 + D + Hk + Sq)


@pytest.mark.parametrize("ps", [128, 256])
def test_paged_decode_page_sizes_and_splits(ps):
    _run(3, 1, [257, 1000, 129], 4, 2, 128, ps, seed=620 + ps, splits=(0, 1, 7))


def test_paged_decode_window_and_alibi():
    _run(2, 2, [900, 333], 4, 4, 128, 256, seed=630, window=(100, 0))
    _run(2, 1, [900, 333], 8, 2, 64, 128, seed=631, alibi=alibi_slopes_geometric(8))


def test_paged_long_cache_grouped_heads():
    # 16 sequences over 8 key/value heads, up to 16k keys in 256-key pages
    lens = [16384 - 997 * i for i in range(16)]
    _run(16, 1, lens, 32, 8, 128, 256, seed=640, splits=(0,))


def test_identity_table_matches_dense_decode_bitwise():
    import torch

    import exact_attention_56_gb300 as fa

    B, Sk, H, Hk, D, ps = 3, 1024, 8, 2, 128, 256
    g = torch.Generator(device="cuda")
    g.manual_seed(650)
    q = torch.randn((B, 1, H, D), generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn((B, Sk, Hk, D), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((B, Sk, Hk, D), generator=g, device="cuda").to(torch.bfloat16)
    P = Sk // ps
    table = torch.arange(B * P, dtype=torch.int32, device="cuda").reshape(B, P)
    lens = torch.full((B,), Sk, dtype=torch.int32, device="cuda")
    for n in (1, 4):
        out_d, lse_d = fa.fa_decode_splitkv(q, k, v, causal=True, num_splits=n)
        out_p, lse_p = fa.fa_decode_paged(q, k.reshape(B * P, ps, Hk, D), v.reshape(B * P, ps, Hk, D), table, lens,
                                          Sk, causal=True, num_splits=n)
        torch.cuda.synchronize()
        assert torch.equal(out_d.view(torch.int16), out_p.view(torch.int16))
        assert torch.equal(lse_d, lse_p)
