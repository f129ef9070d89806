"""fa_decode_splitkv_noalloc: the decode entry point for callers that cannot
allocate device memory (it keeps its split partials in a fixed array inside
the library instead of a caller workspace). Called through the C ABI and
checked against fa_decode_splitkv on the same inputs, on two calls in a row.

This file is collected last on purpose, so a failure here never hides the
other tests' results from a run that stops at the first failure."""
import ctypes

import numpy as np
import pytest

from fa_inputs import attention_inputs
from helpers import assert_bf16_close, assert_lse_close, to_dev, to_f64

pytestmark = pytest.mark.gpu

FA_ERR_WORKSPACE = -5


def _noalloc_fn():
    from exact_attention_56_gb300 import build

    build.build()
    import exact_attention_56_gb300 as fa

    fn = fa.library().fa_decode_splitkv_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.restype = I
    fn.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, I, I, I, P, I, I, P]
    return fa, fn


def _call(fn, q, k, v, out, lse, n, causal=1):
    import torch

    B, Sq, H, D = q.shape
    Sk, Hk = k.shape[1], k.shape[2]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, Sq, Sk, H, Hk, D, 0.0,
              causal, -1, -1, None, 0, n, stream)


@pytest.mark.parametrize("first,second", [((4, 1, 3000, 8, 128, 0), (2, 3, 777, 4, 64, 5))])
def test_noalloc_matches_workspace_entry_point_twice(first, second):
    import torch

    fa, fn = _noalloc_fn()
    for call, (B, Sq, Sk, H, D, n) in enumerate((first, second)):
        inp = attention_inputs(B, Sq, Sk, H, D, 900 + call)
        q, k, v = (to_dev(inp[x]) for x in ("q", "k", "v"))
        ref_out, ref_lse = fa.fa_decode_splitkv(q, k, v, causal=True, num_splits=n)
        out = torch.empty_like(q)
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
        assert _call(fn, q, k, v, out, lse, n) == 0
        torch.cuda.synchronize()
        st, word = fa.fa_device_status()
        assert st == fa.FA_OK, hex(word)
        assert_bf16_close(to_f64(out), to_f64(ref_out), f"O (call {call})")
        assert_lse_close(lse.cpu().numpy().astype(np.float64), ref_lse.cpu().numpy().astype(np.float64),
                         f"L (call {call})")


def test_noalloc_rejects_requests_beyond_its_array():
    import torch

    fa, fn = _noalloc_fn()
    # B*Sq*H*splits*(D+1)*4 bytes of partials: 64*16*32*64*129*4 is ~1 GiB, far above 8 MiB
    B, Sq, Sk, H, D = 64, 16, 8192, 32, 128
    q = torch.zeros((B, Sq, H, D), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((B, 8, H, D), dtype=torch.bfloat16, device="cuda")  # never read: rejected before launch
    out = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = fn(q.data_ptr(), k.data_ptr(), k.data_ptr(), out.data_ptr(), lse.data_ptr(), B, Sq, Sk, H, H, D, 0.0, 1,
            -1, -1, None, 0, 64, stream)
    assert rc == FA_ERR_WORKSPACE
