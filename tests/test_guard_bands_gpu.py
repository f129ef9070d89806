"""Out-of-bounds writes, checked on the GPU without a sanitizer: every output
(and workspace) of these calls is a view into a larger buffer with canary
bands before and after it (tests/helpers.py Guarded). After the call each band
must be bit-identical, each output fully written, and the values must match
the fp64 oracle with the usual bounds (bf16 max |err| <= 2e-2, relative RMS
<= 1e-2; fp32 L max |err| <= 1e-3 with -inf matched).

The shapes are the ones where a wrong tile bound would write past a tensor:
ragged tails (S not a multiple of 128), packed sequences with empty and
key-less members, paged and appended KV caches, grouped heads, and dropout.
"""
import numpy as np
import pytest

import oracle
from fa_inputs import bf16_bits_to_f64, normal_bf16_bits
from helpers import Guarded, assert_bf16_close, assert_bf16_close_beyond_rounding, assert_lse_close, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _bits(shape, seed):
    return normal_bf16_bits(shape, seed)


def _ok(fa):
    import torch

    torch.cuda.synchronize()
    st, word = fa.fa_device_status()
    assert st == fa.FA_OK, hex(word)


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_forward_ragged(D, causal):
    import torch

    import exact_attention_56_gb300 as fa

    B, Sq, Sk, H, Hk = 2, 333, 461, 4, 2
    b = {"q": _bits((B, Sq, H, D), 901), "k": _bits((B, Sk, Hk, D), 902), "v": _bits((B, Sk, Hk, D), 903)}
    q, k, v = (to_dev(b[n]) for n in ("q", "k", "v"))
    go, gl = Guarded((B, Sq, H, D), torch.bfloat16), Guarded((B, H, Sq), torch.float32)
    fa.fa_fwd(q, k, v, causal=causal, out=go.view, lse=gl.view)
    _ok(fa)
    go.check("out")
    gl.check("lse")
    o_ref, l_ref = oracle.attention_fwd(*(bf16_bits_to_f64(b[n]) for n in ("q", "k", "v")), None, causal)
    assert_bf16_close(to_f64(go.view), o_ref, "O")
    assert_lse_close(gl.view.cpu().numpy().astype(np.float64), l_ref, "L")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_ragged(D, causal):
    import torch

    import exact_attention_56_gb300 as fa

    B, Sq, Sk, H, Hk = 2, 333, 461, 4, 2
    b = {"q": _bits((B, Sq, H, D), 911), "k": _bits((B, Sk, Hk, D), 912), "v": _bits((B, Sk, Hk, D), 913),
         "do": _bits((B, Sq, H, D), 914)}
    q, k, v, do = (to_dev(b[n]) for n in ("q", "k", "v", "do"))
    out, lse = fa.fa_fwd(q, k, v, causal=causal)
    gq = Guarded((B, Sq, H, D), torch.bfloat16)
    gk, gv = Guarded((B, Sk, Hk, D), torch.bfloat16), Guarded((B, Sk, Hk, D), torch.bfloat16)
    gw = Guarded((fa.fa_bwd_workspace_size(B, Sq, Sk, H, D, Hk=Hk),), torch.uint8)
    fa.fa_bwd(do, q, k, v, out, lse, causal=causal, dq=gq.view, dk=gk.view, dv=gv.view, workspace=gw.view)
    _ok(fa)
    for g, n in ((gq, "dq"), (gk, "dk"), (gv, "dv")):
        g.check(n)
    gw.check("workspace", written=False)
    rq, rk, rv = oracle.attention_bwd(*(bf16_bits_to_f64(b[n]) for n in ("do", "q", "k", "v")), None, causal)
    assert_bf16_close(to_f64(gq.view), rq, "dQ")
    assert_bf16_close_beyond_rounding(to_f64(gk.view), rk, "dK")  # sums over two query heads
    assert_bf16_close_beyond_rounding(to_f64(gv.view), rv, "dV")


def test_packed_sequences():
    import torch

    import exact_attention_56_gb300 as fa

    H, Hk, D = 4, 2, 128
    len_q, len_k = [1, 200, 0, 333, 129, 40], [50, 200, 10, 700, 1, 0]
    cq = np.concatenate([[0], np.cumsum(len_q)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(len_k)]).astype(np.int32)
    tq, tk = int(cq[-1]), int(ck[-1])
    b = {"q": _bits((tq, H, D), 921), "k": _bits((tk, Hk, D), 922), "v": _bits((tk, Hk, D), 923),
         "do": _bits((tq, H, D), 924)}
    q, k, v, do = (to_dev(b[n]) for n in ("q", "k", "v", "do"))
    cu_q, cu_k = torch.from_numpy(cq).cuda(), torch.from_numpy(ck).cuda()
    go, gl = Guarded((tq, H, D), torch.bfloat16), Guarded((H, tq), torch.float32)
    fa.fa_fwd_varlen(q, k, v, cu_q, cu_k, max(len_q), max(len_k), causal=True, out=go.view, lse=gl.view)
    _ok(fa)
    go.check("out")
    gl.check("lse")
    gq = Guarded((tq, H, D), torch.bfloat16)
    gk, gv = Guarded((tk, Hk, D), torch.bfloat16), Guarded((tk, Hk, D), torch.bfloat16)
    gw = Guarded((fa.fa_bwd_varlen_workspace_size(len(len_q), tq, tk, max(len_q), H, D, Hk=Hk),), torch.uint8)
    fa.fa_bwd_varlen(do, q, k, v, go.view, gl.view, cu_q, cu_k, max(len_q), max(len_k), causal=True, dq=gq.view,
                     dk=gk.view, dv=gv.view, workspace=gw.view)
    _ok(fa)
    for g, n in ((gq, "dq"), (gk, "dk"), (gv, "dv")):
        g.check(n)
    gw.check("workspace", written=False)
    f64 = [bf16_bits_to_f64(b[n]) for n in ("q", "k", "v")]
    o_ref, l_ref = oracle.attention_fwd_varlen(*f64, cq, ck, None, True)
    assert_bf16_close(to_f64(go.view), o_ref, "O")
    assert_lse_close(gl.view.cpu().numpy().astype(np.float64), l_ref, "L")
    rq, rk, rv = oracle.attention_bwd_varlen(bf16_bits_to_f64(b["do"]), *f64, cq, ck, None, True)
    assert_bf16_close(to_f64(gq.view), rq, "dQ")
    assert_bf16_close_beyond_rounding(to_f64(gk.view), rk, "dK")
    assert_bf16_close_beyond_rounding(to_f64(gv.view), rv, "dV")


@pytest.mark.parametrize("H,Hk,Sq", [(8, 8, 1), (32, 4, 3)])
@pytest.mark.parametrize("n", [0, 5])
def test_decode(H, Hk, Sq, n):
    import torch

    import exact_attention_56_gb300 as fa

    B, Sk, D = 3, 1777, 128
    b = {"q": _bits((B, Sq, H, D), 931), "k": _bits((B, Sk, Hk, D), 932), "v": _bits((B, Sk, Hk, D), 933)}
    q, k, v = (to_dev(b[x]) for x in ("q", "k", "v"))
    go, gl = Guarded((B, Sq, H, D), torch.bfloat16), Guarded((B, H, Sq), torch.float32)
    gw = Guarded((fa.fa_decode_workspace_size(B, Sq, Sk, H, D, n, Hk=Hk),), torch.uint8)
    fa.fa_decode_splitkv(q, k, v, causal=True, num_splits=n, workspace=gw.view, out=go.view, lse=gl.view)
    _ok(fa)
    go.check("out")
    gl.check("lse")
    gw.check("workspace", written=False)
    o_ref, l_ref = oracle.attention_fwd(*(bf16_bits_to_f64(b[x]) for x in ("q", "k", "v")), None, True)
    assert_bf16_close(to_f64(go.view), o_ref, "O")
    assert_lse_close(gl.view.cpu().numpy().astype(np.float64), l_ref, "L")


def test_paged_decode():
    import torch

    import exact_attention_56_gb300 as fa

    B, Sq, H, Hk, D, ps = 3, 2, 8, 2, 128, 128
    lens = [300, 1, 700]
    P = max((x + ps - 1) // ps for x in lens)
    num_pages = B * P + 2
    b = {"q": _bits((B, Sq, H, D), 941), "k": _bits((num_pages, ps, Hk, D), 942),
         "v": _bits((num_pages, ps, Hk, D), 943)}
    table = np.random.default_rng(944).permutation(num_pages)[:B * P].reshape(B, P).astype(np.int32)
    sl = np.asarray(lens, dtype=np.int32)
    q, kp, vp = (to_dev(b[x]) for x in ("q", "k", "v"))
    go, gl = Guarded((B, Sq, H, D), torch.bfloat16), Guarded((B, H, Sq), torch.float32)
    gw = Guarded((fa.fa_decode_workspace_size(B, Sq, max(lens), H, D, 3, Hk=Hk),), torch.uint8)
    fa.fa_decode_paged(q, kp, vp, torch.from_numpy(table).cuda(), torch.from_numpy(sl).cuda(), max(lens),
                       causal=True, num_splits=3, workspace=gw.view, out=go.view, lse=gl.view)
    _ok(fa)
    go.check("out")
    gl.check("lse")
    gw.check("workspace", written=False)
    o_ref, l_ref = oracle.decode_paged(*(bf16_bits_to_f64(b[x]) for x in ("q", "k", "v")), table, sl, None, True)
    assert_bf16_close(to_f64(go.view), o_ref, "O")
    assert_lse_close(gl.view.cpu().numpy().astype(np.float64), l_ref, "L")


@pytest.mark.parametrize("H,Hk", [(4, 4), (32, 8)])
def test_kvcache_append_stays_inside_the_cache(H, Hk):
    """The appended rows land inside the cache; rows past its capacity are dropped
    (sequence 2 fills the cache to its last row and beyond)."""
    import torch

    import exact_attention_56_gb300 as fa

    B, Sq, D, rows, S_new = 3, 1, 128, 640, 4
    seqlens = np.asarray([100, 0, rows - 2], dtype=np.int32)
    b = {"q": _bits((B, Sq, H, D), 951), "k": _bits((B, rows, Hk, D), 952), "v": _bits((B, rows, Hk, D), 953),
         "kn": _bits((B, S_new, Hk, D), 954), "vn": _bits((B, S_new, Hk, D), 955)}
    q, kn, vn = to_dev(b["q"]), to_dev(b["kn"]), to_dev(b["vn"])
    gkc, gvc = Guarded((B, rows, Hk, D), torch.bfloat16), Guarded((B, rows, Hk, D), torch.bfloat16)
    gkc.view.copy_(to_dev(b["k"]))
    gvc.view.copy_(to_dev(b["v"]))
    go, gl = Guarded((B, Sq, H, D), torch.bfloat16), Guarded((B, H, Sq), torch.float32)
    fa.fa_decode_kvcache(q, gkc.view, gvc.view, torch.from_numpy(seqlens).cuda(), kn, vn, causal=True,
                         out=go.view, lse=gl.view)
    _ok(fa)
    gkc.check("k_cache", written=False)
    gvc.check("v_cache", written=False)
    go.check("out")
    gl.check("lse")
    o_ref, l_ref, k_ref, v_ref = oracle.decode_kvcache(*(bf16_bits_to_f64(b[x]) for x in ("q", "k", "v")), seqlens,
                                                       bf16_bits_to_f64(b["kn"]), bf16_bits_to_f64(b["vn"]),
                                                       causal=True)
    assert np.array_equal(to_f64(gkc.view), k_ref) and np.array_equal(to_f64(gvc.view), v_ref)
    assert_bf16_close(to_f64(go.view), o_ref, "O")
    assert_lse_close(gl.view.cpu().numpy().astype(np.float64), l_ref, "L")


def test_dropout_forward_and_backward():
    import torch

    import exact_attention_56_gb300 as fa

    B, S, H, D, p, seed = 1, 300, 2, 64, 0.2, 12345
    b = {"q": _bits((B, S, H, D), 961), "k": _bits((B, S, H, D), 962), "v": _bits((B, S, H, D), 963),
         "do": _bits((B, S, H, D), 964)}
    q, k, v, do = (to_dev(b[x]) for x in ("q", "k", "v", "do"))
    go, gl = Guarded((B, S, H, D), torch.bfloat16), Guarded((B, H, S), torch.float32)
    fa.fa_fwd_dropout(q, k, v, p, seed, causal=True, out=go.view, lse=gl.view)
    _ok(fa)
    go.check("out")
    gl.check("lse")
    gq, gk, gv = (Guarded((B, S, H, D), torch.bfloat16) for _ in range(3))
    fa.fa_bwd_dropout(do, q, k, v, go.view, gl.view, p, seed, causal=True, dq=gq.view, dk=gk.view, dv=gv.view)
    _ok(fa)
    for g, n in ((gq, "dq"), (gk, "dk"), (gv, "dv")):
        g.check(n)
    f64 = [bf16_bits_to_f64(b[x]) for x in ("q", "k", "v")]
    o_ref, _ = oracle.attention_fwd_dropout(*f64, p, seed, causal=True)
    assert_bf16_close(to_f64(go.view), o_ref, "O")
    refs = oracle.attention_bwd_dropout(bf16_bits_to_f64(b["do"]), *f64, p, seed, causal=True)
    for name, g, r in zip(("dQ", "dK", "dV"), (gq, gk, gv), refs):
        assert_bf16_close_beyond_rounding(to_f64(g.view), r, name)
