"""Failure detection on the GPU without a fault: a bounded wait that nothing
satisfies gives up after about a second, records the timeout and its site in
the device status word, and leaves the context usable for the next call. The
same holds inside the attention kernels: with a diagnostic switch, the
forward's producer (or the dQ kernel's) leaves out one key tile, the wait for
it expires after a 10 ms limit, and the kernel returns through its abort path
(drains its copies and tensor-core work, frees its tensor memory)."""
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


def _injected(kind, run, site_nibble):
    """Run `run` with fault `kind` injected and a 10 ms wait limit; the kernel's own
    bounded wait must expire, the call must return quickly, and the status word must
    name a wait site of the expected kernel. Normal operation is restored after."""
    import exact_attention_56_gb300 as fa

    st, _ = fa.fa_device_status()
    assert st == fa.FA_OK
    fa.fa_debug_set_fault(kind, 10_000_000)
    try:
        t0 = time.perf_counter()
        run()
        st, word = fa.fa_device_status()
        elapsed = time.perf_counter() - t0
    finally:
        fa.fa_debug_set_fault(fa.FA_FAULT_NONE, 0)
    assert st == fa.FA_ERR_TIMEOUT, hex(word)
    assert word & 0x80000000
    assert (word & 0xF0) == site_nibble and (word & 0xFF00) == 0, hex(word)
    assert elapsed < 0.5, elapsed  # the 10 ms limit, not a hang nor the 1 s default
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK and word == 0


@pytest.mark.parametrize("D", [64, 128])
def test_forward_wait_expires_in_the_attention_kernel(D):
    import torch

    import exact_attention_56_gb300 as fa

    # two key tiles per head: the producer leaves out key tile 1
    inp = attention_inputs(1, 256, 256, 2, D, 17, with_dout=True)
    q, k, v, do = (to_dev(inp[n]) for n in ("q", "k", "v", "dout"))
    _injected(fa.FA_FAULT_FWD_SKIP_KEY_TILE, lambda: fa.fa_fwd(q, k, v, causal=False), 0x10)
    # the next normal calls are correct
    out, lse = fa.fa_fwd(q, k, v, causal=False)
    dq, dk, dv = fa.fa_bwd(do, q, k, v, out, lse, causal=False)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    f64 = [bf16_bits_to_f64(inp[n]) for n in ("q", "k", "v")]
    o_ref, _ = oracle.attention_fwd(*f64, None, False)
    assert_bf16_close(to_f64(out), o_ref, "O after the injected timeout")
    refs = oracle.attention_bwd(bf16_bits_to_f64(inp["dout"]), *f64, None, False)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), refs):
        assert_bf16_close(to_f64(g), r, f"{name} after the injected timeout")


@pytest.mark.parametrize("D", [64, 128])
def test_backward_wait_expires_in_the_dq_kernel(D):
    import torch

    import exact_attention_56_gb300 as fa

    inp = attention_inputs(1, 256, 256, 2, D, 18, with_dout=True)
    q, k, v, do = (to_dev(inp[n]) for n in ("q", "k", "v", "dout"))
    out, lse = fa.fa_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    # the two-kernel path (deterministic), whose dQ kernel's producer leaves out the key tile
    _injected(fa.FA_FAULT_BWD_SKIP_KEY_TILE,
              lambda: fa.fa_bwd(do, q, k, v, out, lse, causal=True, deterministic=True), 0x40)
    dq, dk, dv = fa.fa_bwd(do, q, k, v, out, lse, causal=True)
    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)
    refs = oracle.attention_bwd(*(bf16_bits_to_f64(inp[n]) for n in ("dout", "q", "k", "v")), None, True)
    for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), refs):
        assert_bf16_close(to_f64(g), r, f"{name} after the injected timeout")


def test_fault_setter_rejects_bad_arguments():
    import exact_attention_56_gb300 as fa

    lib = fa.library()
    assert lib.fa_debug_set_fault(7, 0) == fa.FA_ERR_INVALID
    assert lib.fa_debug_set_fault(0, 10) == fa.FA_ERR_INVALID          # below 1 ms
    assert lib.fa_debug_set_fault(0, 5_000_000_000) == fa.FA_ERR_INVALID  # above 1 s
    assert lib.fa_debug_set_fault(0, 0) == fa.FA_OK
