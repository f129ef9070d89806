"""fa_decode_splitkv_noalloc: the decode entry point for callers that cannot
allocate device memory (it keeps its split partials in a fixed array inside
the library instead of a caller workspace). Called through the C ABI and
checked against fa_decode_splitkv and against the fp64 oracle on the same
inputs, on calls in a row.

This file is collected last on purpose, so a failure here never hides the
other tests' results from a run that stops at the first failure."""
import ctypes

import numpy as np
import pytest

import oracle
from fa_inputs import alibi_slopes_geometric, attention_inputs, bf16_bits_to_f64, normal_bf16_bits
from helpers import assert_bf16_close, assert_lse_close, to_dev, to_f64

pytestmark = pytest.mark.gpu

FA_ERR_WORKSPACE = -5
SCRATCH_BYTES = 8 << 20


def _noalloc_fn():
    from exact_attention_56_gb300 import build

    build.build()
    import exact_attention_56_gb300 as fa

    fn = fa.library().fa_decode_splitkv_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.restype = I
    fn.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, I, I, P, I, I, P]
    return fa, fn


def _call(fn, q, k, v, out, lse, n, causal=1, window=(-1, -1), alibi=None):
    import torch

    B, Sq, H, D = q.shape
    Sk, Hk = k.shape[1], k.shape[2]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    al = None if alibi is None else ctypes.c_void_p(alibi.data_ptr())
    return fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, Sq, Sk, H, Hk, D, 0.0,
              causal, window[0], window[1], al, 0, n, stream)


def _inputs(B, Sq, Sk, H, Hk, D, seed):
    return {"q": normal_bf16_bits((B, Sq, H, D), seed * 8 + 0),
            "k": normal_bf16_bits((B, Sk, Hk, D), seed * 8 + 1),
            "v": normal_bf16_bits((B, Sk, Hk, D), seed * 8 + 2)}


def _partials_bytes(B, Sq, H, D, n):
    a256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    u = B * Sq * H * n
    return a256(u * D * 4) + a256(u * 4)


# (B, Sq, Sk, H, Hk, D, num_splits, window, alibi): multi-head on the CUDA-core split
# kernel, then grouped heads with ALiBi and a left window on the tensor-core kernel
CASES = [
    (4, 1, 3000, 8, 8, 128, 0, (-1, -1), False),
    (2, 3, 777, 4, 4, 64, 5, (-1, -1), False),
    (2, 4, 2500, 32, 4, 128, 3, (700, -1), True),
]


def test_noalloc_matches_workspace_entry_point_and_oracle():
    import torch

    fa, fn = _noalloc_fn()
    for call, (B, Sq, Sk, H, Hk, D, n, window, use_alibi) in enumerate(CASES):
        inp = _inputs(B, Sq, Sk, H, Hk, D, 900 + call)
        q, k, v = (to_dev(inp[x]) for x in ("q", "k", "v"))
        slopes = alibi_slopes_geometric(H) if use_alibi else None
        al = None if slopes is None else torch.from_numpy(np.ascontiguousarray(slopes, np.float32)).cuda()
        ref_out, ref_lse = fa.fa_decode_splitkv(q, k, v, causal=True, window_size=window, alibi_slopes=al,
                                                num_splits=n)
        out = torch.empty_like(q)
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
        assert _call(fn, q, k, v, out, lse, n, 1, window, al) == 0
        torch.cuda.synchronize()
        st, word = fa.fa_device_status()
        assert st == fa.FA_OK, hex(word)
        got_o, got_l = to_f64(out), lse.cpu().numpy().astype(np.float64)
        assert_bf16_close(got_o, to_f64(ref_out), f"O vs fa_decode_splitkv (call {call})")
        assert_lse_close(got_l, ref_lse.cpu().numpy().astype(np.float64), f"L vs fa_decode_splitkv (call {call})")
        o64, l64 = oracle.attention_fwd(*(bf16_bits_to_f64(inp[x]) for x in ("q", "k", "v")), None, True, window,
                                        slopes)
        assert_bf16_close(got_o, o64, f"O vs oracle (call {call})")
        assert_lse_close(got_l, l64, f"L vs oracle (call {call})")


def test_noalloc_automatic_splits_shrink_to_fit():
    """num_splits = 0 lowers the automatic count until the partials fit the array."""
    import torch

    fa, fn = _noalloc_fn()
    Sq, Sk, H, Hk, D = 16, 8192, 32, 32, 128
    # the automatic count depends on the SM count: take the first batch size whose
    # automatic count does not fit the array while one split does
    for B in (4, 6, 8, 12, 16):
        auto = fa.fa_decode_num_splits(B, Sq, Sk, H, D, Hk=Hk)
        if _partials_bytes(B, Sq, H, D, auto) > SCRATCH_BYTES >= _partials_bytes(B, Sq, H, D, 1):
            break
    else:
        pytest.fail("no batch size whose automatic split count overflows the array")
    inp = attention_inputs(B, Sq, Sk, H, D, 931)
    q, k, v = (to_dev(inp[x]) for x in ("q", "k", "v"))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    assert _call(fn, q, k, v, out, lse, 0) == 0
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    ref_out, ref_lse = fa.fa_decode_splitkv(q, k, v, causal=True, num_splits=0)
    assert_bf16_close(to_f64(out), to_f64(ref_out), "O vs fa_decode_splitkv")
    assert_lse_close(lse.cpu().numpy().astype(np.float64), ref_lse.cpu().numpy().astype(np.float64),
                     "L vs fa_decode_splitkv")
    # two sampled heads against the oracle
    for b, h in ((0, 0), (B - 1, H - 1)):
        o64, l64 = oracle.head_fwd(*(bf16_bits_to_f64(inp[x])[b, :, h, :] for x in ("q", "k", "v")),
                                   1.0 / np.sqrt(D), True)
        assert_bf16_close(to_f64(out)[b, :, h, :], o64, f"O head ({b},{h}) vs oracle")
        assert_lse_close(lse[b, h].cpu().numpy().astype(np.float64), l64, f"L head ({b},{h}) vs oracle")


def test_noalloc_rejects_requests_beyond_its_array():
    import torch

    fa, fn = _noalloc_fn()
    # caches sized to Sk, so nothing is out of range even if a launch happened
    for B, Sq, Sk, H, D, n in ((16, 16, 256, 32, 128, 64),   # explicit count: ~270 MB of partials
                               (64, 16, 128, 32, 128, 0)):   # one split alone: ~17 MB
        assert _partials_bytes(B, Sq, H, D, max(n, 1)) > SCRATCH_BYTES
        q = torch.zeros((B, Sq, H, D), dtype=torch.bfloat16, device="cuda")
        k = torch.zeros((B, Sk, H, D), dtype=torch.bfloat16, device="cuda")
        out = torch.full_like(q, 7.0)
        lse = torch.full((B, H, Sq), 7.0, dtype=torch.float32, device="cuda")
        assert _call(fn, q, k, k, out, lse, n) == FA_ERR_WORKSPACE
        torch.cuda.synchronize()
        assert bool((out == 7.0).all()) and bool((lse == 7.0).all())  # nothing was written
