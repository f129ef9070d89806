"""Shared test helpers: device transfer of bf16 bits and the parity metrics."""
import numpy as np

# Tolerances for bf16 outputs and fp32 L against the fp64 oracle.
ATOL_BF16 = 2e-2
RELRMS_BF16 = 1e-2
ATOL_LSE = 1e-3


def to_dev(bits, device="cuda"):
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)


# Relative RMS needs a non-vanishing reference: where the exact result is ~0
# (e.g. a one-key window, where dS = P o (dP - D) cancels exactly) the
# denominator is floored at an RMS of 1e-3, about one bf16 step at unit scale.
REF_RMS_FLOOR = 1e-3


def rel_rms(x, ref):
    floor = REF_RMS_FLOOR * np.sqrt(max(ref.size, 1))
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), floor))


def assert_bf16_close(got, ref, what=""):
    err = np.max(np.abs(got - ref)) if got.size else 0.0
    rr = rel_rms(got, ref) if got.size else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert err <= ATOL_BF16, f"{what}: max |err| {err:.3e} > {ATOL_BF16}"
    assert rr <= RELRMS_BF16, f"{what}: rel RMS {rr:.3e} > {RELRMS_BF16}"


def assert_lse_close(got, ref, what=""):
    inf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf_ref), f"{what}: -inf pattern differs"
    fin = ~inf_ref
    if fin.any():
        err = np.max(np.abs(got[fin] - ref[fin]))
        assert err <= ATOL_LSE, f"{what}: L max |err| {err:.3e} > {ATOL_LSE}"


# bf16 keeps 8 significant bits, so rounding an output x alone moves it by up
# to half a unit in the last place: 2^(e-8) for x in [2^e, 2^(e+1)), that is up
# to 2^-8 |x| just above a power of two. Where outputs grow past |x| ~ 4 (sums
# over many query rows or over the query heads sharing a key/value head), that
# rounding approaches the 2e-2 bound by itself; such tests keep the 2e-2 budget
# for everything else.
BF16_HALF_ULP_REL = 2.0 ** -8


def assert_bf16_close_beyond_rounding(got, ref, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    excess = np.max(np.abs(got - ref) - BF16_HALF_ULP_REL * np.abs(ref)) if got.size else 0.0
    rr = rel_rms(got, ref) if got.size else 0.0
    assert excess <= ATOL_BF16, f"{what}: max (|err| - 2^-8 |ref|) {excess:.3e} > {ATOL_BF16}"
    assert rr <= RELRMS_BF16, f"{what}: rel RMS {rr:.3e} > {RELRMS_BF16}"


# A problem whose exact result is f times one of natural size (inputs scaled by
# known factors): the error divided by f must meet the bf16 bound, and the
# relative RMS (scale-free, no floor) the 1e-2 bound.
def assert_bf16_close_scaled(got, ref, f, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = float(np.max(np.abs(got / f - ref / f)))
    nref = np.linalg.norm(ref)
    assert nref > 0, f"{what}: reference is all zero"
    rr = float(np.linalg.norm(got - ref) / nref)
    assert err <= ATOL_BF16, f"{what}: max |err| / {f:g} = {err:.3e} > {ATOL_BF16}"
    assert rr <= RELRMS_BF16, f"{what}: rel RMS {rr:.3e} > {RELRMS_BF16}"


# Guard bands: an output (or workspace) is a view into a larger buffer whose
# bytes before and after it hold a canary pattern (a NaN bit pattern, also
# written into the view itself). After the call the bands must be bit-identical
# (no write outside the tensor) and, for outputs, every element must have been
# overwritten (no NaN pattern left). 4096 bytes of band keep every view's start
# 256-byte aligned, as the library asks of workspaces.
GUARD_BYTES = 4096
_CANARY = {2: 0x7FA5, 4: 0x7FA5A5A5, 1: 0xA5}


class Guarded:
    def __init__(self, shape, dtype, device="cuda"):
        import torch

        self.shape = tuple(shape)
        n = int(np.prod(self.shape)) if self.shape else 1
        esz = torch.empty((), dtype=dtype).element_size()
        self.pad = GUARD_BYTES // esz
        self.n = n
        self.buf = torch.empty(n + 2 * self.pad, dtype=dtype, device=device)
        ity = {1: torch.uint8, 2: torch.int16, 4: torch.int32}[esz]
        self.bits = self.buf.view(ity)
        pat = _CANARY[esz]
        if esz == 2 and pat > 0x7FFF:
            pat -= 1 << 16
        if esz == 4 and pat > 0x7FFFFFFF:
            pat -= 1 << 32
        self.pattern = pat
        self.bits.fill_(pat)
        self.view = self.buf[self.pad:self.pad + n].view(self.shape)

    def check(self, what, written=True):
        import torch

        lo, hi = self.bits[:self.pad], self.bits[self.pad + self.n:]
        assert bool((lo == self.pattern).all()), f"{what}: bytes before the tensor were overwritten"
        assert bool((hi == self.pattern).all()), f"{what}: bytes after the tensor were overwritten"
        if written:
            mid = self.bits[self.pad:self.pad + self.n]
            left = int((mid == self.pattern).sum())
            assert left == 0, f"{what}: {left} elements were never written"
        torch.cuda.synchronize()
