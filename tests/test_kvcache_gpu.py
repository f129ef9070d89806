"""GPU parity of the KV-cache decode step: new keys/values appended in place,
rotary embedding on the new keys and the query (page
"FlashAttention：快速且内存高效的准确注意力机制", section "2.2：针对推理进行优化";
the rotary formula and the positions are the readings stated in include/fa.h).

Checked: the decode output and lse against the oracle, the appended cache rows
against the oracle's rotated rows, and every other cache row unchanged bit for
bit. Tolerances as everywhere: bf16 max |err| <= 2e-2 and relative RMS <= 1e-2,
fp32 L max |err| <= 1e-3 with -inf matched.
"""
import numpy as np
import pytest

import oracle
from fa_inputs import alibi_slopes_geometric, bf16_bits_to_f64, normal_bf16_bits
from helpers import assert_bf16_close, assert_lse_close, to_dev, to_f64

pytestmark = pytest.mark.gpu


def _tables(n, r, base=10000.0):
    w = base ** (-np.arange(r // 2) * 2.0 / r)
    ang = np.arange(n)[:, None] * w[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def _run(B, H, Hk, D, seq, S_new, Sq, rot_dim, interleaved, seed, paged=False, cap=1024, ps=256, causal=True,
         window=(-1, -1), alibi=None, splits=(0, 3)):
    import torch

    import exact_attention_56_gb300 as fa

    if paged:
        P = cap // ps
        num_pages = B * P + 2
        k_b = normal_bf16_bits((num_pages, ps, Hk, D), seed * 8)
        v_b = normal_bf16_bits((num_pages, ps, Hk, D), seed * 8 + 1)
        table = np.random.default_rng(seed).permutation(num_pages)[:B * P].reshape(B, P).astype(np.int32)
    else:
        k_b = normal_bf16_bits((B, cap, Hk, D), seed * 8)
        v_b = normal_bf16_bits((B, cap, Hk, D), seed * 8 + 1)
        table = None
    q_b = normal_bf16_bits((B, Sq, H, D), seed * 8 + 2)
    kn_b = normal_bf16_bits((B, S_new, Hk, D), seed * 8 + 3) if S_new else None
    vn_b = normal_bf16_bits((B, S_new, Hk, D), seed * 8 + 4) if S_new else None
    cos, sin = _tables(cap + 16, rot_dim) if rot_dim else (None, None)
    sl = np.asarray(seq, dtype=np.int32)
    o_ref, l_ref, kc_ref, vc_ref = oracle.decode_kvcache(
        bf16_bits_to_f64(q_b), bf16_bits_to_f64(k_b), bf16_bits_to_f64(v_b), sl,
        None if kn_b is None else bf16_bits_to_f64(kn_b), None if vn_b is None else bf16_bits_to_f64(vn_b),
        None if cos is None else cos.astype(np.float64), None if sin is None else sin.astype(np.float64), interleaved,
        table, None, causal, window, alibi)
    dev = torch.device("cuda")
    q = to_dev(q_b)
    kn = None if kn_b is None else to_dev(kn_b)
    vn = None if vn_b is None else to_dev(vn_b)
    tc = None if cos is None else torch.from_numpy(cos).to(dev)
    ts = None if sin is None else torch.from_numpy(sin).to(dev)
    bt = None if table is None else torch.from_numpy(table).to(dev)
    al = None if alibi is None else torch.from_numpy(np.ascontiguousarray(alibi, dtype=np.float32)).to(dev)
    changed = np.any(np.abs(kc_ref - bf16_bits_to_f64(k_b)) > 0, axis=(-1, -2)) | \
        np.any(np.abs(vc_ref - bf16_bits_to_f64(v_b)) > 0, axis=(-1, -2))
    for n in splits:
        kc, vc = to_dev(k_b), to_dev(v_b)  # fresh caches: the append is in place
        out, lse = fa.fa_decode_kvcache(q, kc, vc, torch.from_numpy(sl).to(dev), kn, vn, rotary_cos=tc,
                                        rotary_sin=ts, rotary_interleaved=interleaved, block_table=bt,
                                        causal=causal, window_size=window, alibi_slopes=al, num_splits=n)
        torch.cuda.synchronize()
        st, word = fa.fa_device_status()
        assert st == fa.FA_OK, hex(word)
        assert_bf16_close(to_f64(out), o_ref, f"O (splits {n})")
        assert_lse_close(lse.cpu().numpy().astype(np.float64), l_ref, f"L (splits {n})")
        kc_got, vc_got = to_f64(kc), to_f64(vc)
        assert_bf16_close(kc_got[changed], kc_ref[changed], "appended keys")
        assert np.array_equal(vc_got[changed], vc_ref[changed]), "appended values are copied exactly"
        kbits = kc.view(torch.int16).cpu().numpy()
        vbits = vc.view(torch.int16).cpu().numpy()
        assert np.array_equal(kbits[~changed], np.asarray(k_b).view(np.int16)[~changed]), "untouched key rows"
        assert np.array_equal(vbits[~changed], np.asarray(v_b).view(np.int16)[~changed]), "untouched value rows"


def test_dense_append_rotary_half_split_with_overflow():
    # the third sequence has room for 3 of its 4 new rows
    _run(3, 8, 2, 128, [0, 500, 1021], 4, 4, 128, False, seed=700)


def test_dense_one_token_interleaved_partial_rotary():
    _run(2, 8, 8, 64, [31, 900], 1, 1, 32, True, seed=701)


@pytest.mark.parametrize("interleaved", [False, True])
def test_paged_append_rotary(interleaved):
    _run(2, 8, 2, 128, [100, 700], 2, 2, 64, interleaved, seed=702 + int(interleaved), paged=True)


def test_append_only_and_rotary_only():
    _run(2, 4, 4, 128, [10, 300], 3, 3, 0, False, seed=704)           # append, no rotary
    _run(2, 4, 2, 128, [10, 300], 0, 2, 128, False, seed=705)         # rotary on the query only


def test_append_without_rotary_many_query_pairs():
    # no rotary and eight (query row, query head) pairs per key/value head: the
    # appended rows are read by the tensor-core decode (dense and paged caches,
    # one sequence filling its capacity)
    _run(2, 8, 2, 128, [100, 1021], 4, 2, 0, False, seed=709)
    _run(2, 8, 2, 64, [100, 700], 2, 2, 0, False, seed=710, paged=True)
    _run(3, 16, 2, 128, [0, 257, 900], 1, 1, 0, False, seed=711, window=(300, 0))


def test_rotary_many_query_pairs():
    # rotary with four or more (query row, query head) pairs per key/value head:
    # the query is rotated in fp32 and carried as a bf16 pair into the
    # tensor-core decode (D = 64, interleaved, partial rotary dims)
    _run(2, 8, 2, 64, [31, 900], 1, 2, 32, True, seed=712)
    _run(2, 16, 2, 128, [500, 1000], 3, 3, 128, False, seed=713, paged=True)


def test_long_head_dim_and_masks():
    _run(2, 4, 2, 256, [77, 600], 2, 2, 256, False, seed=706)
    _run(2, 8, 2, 128, [300, 900], 2, 2, 128, True, seed=707, window=(100, 0))
    _run(2, 8, 8, 64, [300, 900], 1, 1, 64, False, seed=708, alibi=alibi_slopes_geometric(8))
