"""The C-ABI library builds, loads and exports every symbol include/fa.h declares;
host-side argument checks reject bad calls before any CUDA work (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_attention_56_gb300 import build as b

    b.build()
    import exact_attention_56_gb300 as fa

    return fa.library()


def _declared():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(fa_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = _declared()
    for required in ("fa_fwd", "fa_bwd", "fa_decode_splitkv", "fa_bwd_workspace_size",
                     "fa_decode_workspace_size", "fa_device_status", "fa_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_version_and_strings(lib):
    assert lib.fa_version() >= 10000
    assert lib.fa_status_string(0) == b"ok"
    assert b"workspace" in lib.fa_status_string(-5)


def _fwd(lib, **kw):
    a = dict(q=16, k=16, v=16, out=16, lse=16, B=1, Sq=8, Sk=8, H=1, Hk=None, D=64, scale=0.0, causal=0, wl=-1,
             wr=-1, alibi=None, ab=0)
    a.update(kw)
    Hk = a["H"] if a["Hk"] is None else a["Hk"]
    P = ctypes.c_void_p
    return lib.fa_fwd(P(a["q"]), P(a["k"]), P(a["v"]), P(a["out"]), P(a["lse"]), a["B"], a["Sq"], a["Sk"], a["H"],
                      Hk, a["D"], ctypes.c_float(a["scale"]), a["causal"], a["wl"], a["wr"], P(a["alibi"]), a["ab"],
                      P(None))


def test_argument_checks_without_gpu(lib):
    import exact_attention_56_gb300 as fa

    assert _fwd(lib, q=0) == fa.FA_ERR_INVALID          # NULL pointer
    assert _fwd(lib, q=8) == fa.FA_ERR_INVALID          # not 16-byte aligned
    assert _fwd(lib, Sq=0) == fa.FA_ERR_INVALID
    assert _fwd(lib, wl=-2) == fa.FA_ERR_INVALID
    assert _fwd(lib, alibi=16, ab=3, H=2) == fa.FA_ERR_INVALID
    assert _fwd(lib, D=96) == fa.FA_ERR_UNSUPPORTED
    # key/value heads: H must be a positive multiple of Hk
    assert _fwd(lib, H=4, Hk=0) == fa.FA_ERR_INVALID
    assert _fwd(lib, H=4, Hk=3) == fa.FA_ERR_INVALID
    assert _fwd(lib, H=4, Hk=8) == fa.FA_ERR_INVALID


def test_workspace_sizes(lib):
    lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fa_decode_workspace_size.restype = ctypes.c_size_t
    # two fp32 per-row vectors (L in log2 units and rowsum(dO*O)), rows padded to 128,
    # and fp16 copies of q, dout (B, Sq, H, D) and k, v (B, Sk, H, D)
    B, Sq, Sk, H, D = 1, 100, 128, 2, 64
    for Hk in (2, 1):  # the k/v copies have Hk heads
        assert lib.fa_bwd_workspace_size(B, Sq, Sk, H, Hk, D, 0) >= 2 * B * H * 128 * 4 + \
            2 * B * Sq * H * D * 2 + 2 * B * Sk * Hk * D * 2
    assert lib.fa_bwd_workspace_size(1, 128, 128, 2, 2, 96, 0) == 0
    assert lib.fa_bwd_workspace_size(1, 128, 128, 4, 3, 64, 0) == 0
    assert lib.fa_decode_workspace_size(2, 1, 1000, 4, 4, 128, 3) >= 2 * 4 * 3 * (128 + 1) * 4
    assert lib.fa_decode_workspace_size(2, 1, 1000, 4, 1, 128, 3) >= 2 * 4 * 3 * (128 + 1) * 4
    assert lib.fa_decode_workspace_size(2, 17, 1000, 4, 4, 128, 3) == 0


def test_grid_limits_without_gpu(lib):
    """Shapes whose grids exceed gridDim.y/z (65535) are refused before any launch."""
    import exact_attention_56_gb300 as fa

    assert _fwd(lib, B=65536) == fa.FA_ERR_UNSUPPORTED
    assert _fwd(lib, H=65536) == fa.FA_ERR_UNSUPPORTED
    # Decode with an append: Sq = 3 rows of one query head per key/value head
    # run on the CUDA-core kernel in blocks of 2 pairs, so 40000 key/value heads
    # need 80000 grid rows. The call must refuse before it appends to the cache.
    P = ctypes.c_void_p
    H = Hk = 40000
    st = lib.fa_decode_kvcache(P(16), P(16), P(16), P(16), P(16), P(16), 1, None, None, 0, 0, 0, None, 0, 0, 0,
                               P(16), P(16), P(256), ctypes.c_size_t(1 << 62), 1, 3, 1024, H, Hk, 64,
                               ctypes.c_float(0.0), 1, -1, -1, None, 0, 1, P(None))
    assert st == fa.FA_ERR_UNSUPPORTED
