"""GPU parity of fa_decode_splitkv (split kernel + merge kernel) against the fp64 oracle."""
import numpy as np
import pytest

import oracle
from fa_inputs import alibi_slopes_geometric, attention_inputs, bf16_bits_to_f64
from helpers import assert_bf16_close, assert_lse_close, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _run(B, Sq, Sk, H, D, n, causal=True, window=(-1, -1), alibi=None, seed=0):
    import torch

    import exact_attention_56_gb300 as fa

    inp = attention_inputs(B, Sq, Sk, H, D, seed)
    q, k, v = (to_dev(inp[n_]) for n_ in ("q", "k", "v"))
    al = None if alibi is None else torch.from_numpy(np.ascontiguousarray(alibi, dtype=np.float32)).cuda()
    out, lse = fa.fa_decode_splitkv(q, k, v, causal=causal, window_size=window, alibi_slopes=al, num_splits=n)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    o_ref, l_ref = oracle.attention_fwd(*(bf16_bits_to_f64(inp[n_]) for n_ in ("q", "k", "v")), None, causal,
                                        window, alibi)
    assert_bf16_close(to_f64(out), o_ref, "O")
    assert_lse_close(lse.cpu().numpy().astype(np.float64), l_ref, "L")


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("n", [1, 3, 0])
def test_decode_head_dims(D, n):
    _run(2, 1, 1000, 4, D, n, seed=D + n)


@pytest.mark.parametrize("Sk", [1, 63, 64, 65, 4096])
def test_decode_lengths(Sk):
    _run(3, 1, Sk, 2, 128, 0, seed=Sk)


def test_decode_more_splits_than_keys():
    _run(1, 1, 5, 2, 128, 16, seed=4)  # most splits are empty


@pytest.mark.parametrize("Sq", [2, 7, 16])
def test_decode_short_query_causal(Sq):
    _run(2, Sq, 777, 2, 128, 5, causal=True, seed=Sq)


def test_decode_window_and_alibi():
    _run(2, 1, 3000, 4, 128, 7, window=(512, 0), alibi=alibi_slopes_geometric(4), seed=9)


def test_decode_config_shape_small_cache():
    # the decode workload's head layout (B=16, H=32, D=128) on a 4096-key cache, every head compared
    _run(16, 1, 4096, 32, 128, 0, seed=5000)
