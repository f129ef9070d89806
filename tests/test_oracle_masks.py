"""Pins for the oracle's mask (CPU only).

Page "FlashAttention：快速且内存高效的准确注意力机制", section
"2.1：更改causal标志的行为" prints the Sq=2, Sk=5 causal mask; the rest of the
checks characterise the bottom-right alignment independently of the oracle's
formula: the mask is the bottom-right Sq x Sk block of the square banded
matrix built with numpy's tril/triu.
"""
import os

import numpy as np
import pytest

from oracle import live_mask

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(t) for t in line.split()])
    return np.array(rows, dtype=bool)


def test_page_example_sq2_sk5_bottom_right():
    want = _load("causal_mask_sq2_sk5_v2_1.txt")
    got = live_mask(2, 5, causal=True)
    assert got.shape == (2, 5)
    assert np.array_equal(got, want)


def test_page_example_sq2_sk5_not_top_left():
    old = _load("causal_mask_sq2_sk5_v2_0.txt")
    assert not np.array_equal(live_mask(2, 5, causal=True), old)


def test_sq5_sk2_rebuilt_case():
    # The page's Sq=5, Sk=2 matrices are missing from the extracted text; by the
    # section's rule (align bottom-right) rows 0-2 see no key, row 3 sees key 0, row 4 both.
    want = np.array([[0, 0], [0, 0], [0, 0], [1, 0], [1, 1]], dtype=bool)
    assert np.array_equal(live_mask(5, 2, causal=True), want)


def _bottom_right_block(Sq, Sk, wl, wr):
    """Independent characterisation: band of the N x N square matrix
    (N = max(Sq, Sk)) with lower width wl and upper width wr, cut to its
    bottom-right Sq x Sk corner."""
    N = max(Sq, Sk)
    full = np.ones((N, N), dtype=bool)
    band = full.copy()
    if wr >= 0:
        band &= np.tril(full, wr)
    if wl >= 0:
        band &= np.triu(full, -wl)
    return band[N - Sq:, N - Sk:]


@pytest.mark.parametrize("Sq", range(1, 9))
@pytest.mark.parametrize("Sk", range(1, 9))
@pytest.mark.parametrize("wl", [-1, 0, 1, 3])
@pytest.mark.parametrize("wr", [-1, 0, 1, 3])
def test_mask_equals_bottom_right_band(Sq, Sk, wl, wr):
    assert np.array_equal(live_mask(Sq, Sk, False, wl, wr), _bottom_right_block(Sq, Sk, wl, wr))


@pytest.mark.parametrize("Sq,Sk", [(1, 1), (4, 4), (3, 7), (7, 3), (16, 16)])
def test_causal_special_cases(Sq, Sk):
    # causal == window (-1, 0); causal keeps the left width of a window
    assert np.array_equal(live_mask(Sq, Sk, True), live_mask(Sq, Sk, False, -1, 0))
    assert np.array_equal(live_mask(Sq, Sk, True, 2, 5), live_mask(Sq, Sk, False, 2, 0))
    assert live_mask(Sq, Sk, False, -1, -1).all()
    if Sq == Sk:
        assert np.array_equal(live_mask(Sq, Sk, True), np.tril(np.ones((Sq, Sk), dtype=bool)))


def test_window_live_counts_long_mask_variants():
    # Exact live-pair counts of the mask-variant workloads (window (4096,0) at
    # 16k; causal 2048 x 8192), computed here by summing the band row by row.
    def count(Sq, Sk, causal, wl, wr):
        c = np.arange(Sq) + (Sk - Sq)
        lo = np.zeros(Sq, dtype=np.int64) if wl < 0 else np.maximum(c - wl, 0)
        hi = np.full(Sq, Sk - 1) if (wr < 0 and not causal) else np.minimum(c + (0 if causal else wr), Sk - 1)
        return int(np.maximum(hi - lo + 1, 0).sum())
    assert count(2048, 8192, True, -1, -1) == 14_681_088
    assert count(16384, 16384, False, 4096, 0) == 58_734_592
    # spot-check the counting rule against the oracle's mask on a small case
    assert count(48, 80, False, 10, 0) == int(live_mask(48, 80, False, 10, 0).sum())
