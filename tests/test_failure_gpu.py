"""Failure detection on the GPU without a fault: a bounded wait that nothing
satisfies gives up after about a second, records the timeout and its site in
the device status word, and leaves the context usable for the next call."""
import time

import numpy as np
import pytest

import oracle
from fa_inputs import attention_inputs, bf16_bits_to_f64
from helpers import assert_bf16_close, to_dev, to_f64

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports():
    import torch

    import exact_attention_56_gb300 as fa

    st, _ = fa.fa_device_status()  # start from a clear status word
    assert st == fa.FA_OK
    t0 = time.perf_counter()
    fa.fa_selftest_wait_timeout()
    st, word = fa.fa_device_status()
    elapsed = time.perf_counter() - t0
    assert st == fa.FA_ERR_TIMEOUT
    assert word & 0x80000000
    assert (word & 0xFFFF) == fa.FA_SELFTEST_SITE
    assert 0.9 <= elapsed <= 10.0, elapsed
    # reading the status clears it, and the context still runs attention correctly
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK and word == 0
    inp = attention_inputs(1, 200, 200, 2, 64, 7)
    q, k, v = (to_dev(inp[n]) for n in ("q", "k", "v"))
    out, _ = fa.fa_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    o_ref, _ = oracle.attention_fwd(*(bf16_bits_to_f64(inp[n]) for n in ("q", "k", "v")), None, True)
    assert_bf16_close(to_f64(out), o_ref, "O after the timeout")
