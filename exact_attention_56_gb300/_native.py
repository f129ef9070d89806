"""ctypes marshalling for libfa_gb300.so (see include/fa.h for the contract)."""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libfa_gb300.so"

FA_OK = 0
FA_ERR_INVALID = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_CUDA = -3
FA_ERR_TIMEOUT = -4
FA_ERR_WORKSPACE = -5


class FAError(RuntimeError):
    """A libfa_gb300 call returned a non-zero status."""

    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: {msg} (status {status})")
        self.status = status


_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGS = {
    "fa_version": (_I, []),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P, _I, _P]),
    "fa_bwd_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "fa_fwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P, _I,
                           _P]),
    "fa_bwd_varlen_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "fa_bwd_varlen": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F,
                           _I, _I, _I, _P, _I, _I, _P]),
    "fa_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P,
                    _I, _I, _P]),
    "fa_decode_num_splits": (_I, [_I, _I, _I, _I, _I, _I]),
    "fa_decode_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "fa_decode_splitkv": (_I, [_P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P, _I,
                               _I, _P]),
    "fa_device_status": (_I, [_P, ctypes.POINTER(ctypes.c_uint)]),
    "fa_fwd_dropout": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P, _I, _F, ctypes.c_uint64,
                            ctypes.c_uint32, _P]),
    "fa_bwd_dropout": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P,
                            _I, _I, _F, ctypes.c_uint64, ctypes.c_uint32, _P]),
    "fa_decode_paged": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _SZ, _I, _I, _I, _I, _I, _I, _I, _I, _I, _F, _I, _I,
                             _I, _P, _I, _I, _P]),
    "fa_decode_kvcache": (_I, [_P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _P, _I, _I, _I, _P, _P, _P, _SZ,
                               _I, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P, _I, _I, _P]),
    "fa_selftest_wait_timeout": (_I, [_P]),
    "fa_debug_set_fault": (_I, [_I, ctypes.c_uint64]),
}


def library_path() -> str:
    return os.path.join(_PKG, _LIB_NAME)


def library() -> ctypes.CDLL:
    """Load libfa_gb300.so (built in-tree by ``build.py``); raise if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise FAError("load", FA_ERR_CUDA,
                              f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def fa_version() -> int:
    return int(library().fa_version())


def fa_status_string(status: int) -> str:
    return library().fa_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != FA_OK:
        raise FAError(fn, status, fa_status_string(status))


def _stream_ptr(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, name, dtype, shape=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _scale(softmax_scale, D):
    """The scale argument as the C ABI takes it: None passes 0, which the library
    folds to its default 1/sqrt(D) (as it does any value <= 0)."""
    return float(softmax_scale) if softmax_scale is not None else 0.0


def _alibi(alibi_slopes, B, H, device):
    if alibi_slopes is None:
        return None, 0
    _need(alibi_slopes, "alibi_slopes", torch.float32, device=device)
    if tuple(alibi_slopes.shape) == (H,):
        return alibi_slopes, 0
    if tuple(alibi_slopes.shape) == (B, H):
        return alibi_slopes, H
    raise ValueError(f"alibi_slopes must have shape ({H},) or ({B}, {H})")


def _kv_heads(k, H):
    """Key/value heads of a (B, Sk, Hk, D) tensor; H must be a multiple of Hk (query
    head h reads key/value head h // (H // Hk))."""
    if not isinstance(k, torch.Tensor) or k.dim() != 4:
        raise ValueError("k must be a 4-D (B, Sk, Hk, D) tensor")
    Hk = int(k.shape[2])
    if Hk < 1 or H % Hk != 0:
        raise ValueError(f"the query heads ({H}) must be a multiple of the key/value heads ({Hk})")
    return Hk


def fa_fwd(q, k, v, *, softmax_scale=None, causal=False, window_size=(-1, -1), alibi_slopes=None,
           out=None, lse=None, stream=None):
    """O, L = attention(q, k, v). q (B,Sq,H,D), k/v (B,Sk,Hk,D) bf16 -> out (B,Sq,H,D) bf16, lse (B,H,Sq) fp32."""
    _need(q, "q", torch.bfloat16)
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    Hk = _kv_heads(k, H)
    dev = q.device
    _need(k, "k", torch.bfloat16, (B, Sk, Hk, D), dev)
    _need(v, "v", torch.bfloat16, (B, Sk, Hk, D), dev)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, (B, Sq, H, D), dev)
    _need(lse, "lse", torch.float32, (B, H, Sq), dev)
    al, al_stride = _alibi(alibi_slopes, B, H, dev)
    st = library().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Sq, Sk, H, Hk, D,
                          _scale(softmax_scale, D), int(bool(causal)), int(window_size[0]), int(window_size[1]),
                          _ptr(al), al_stride, _stream_ptr(stream, dev))
    _check("fa_fwd", st)
    return out, lse


def fa_bwd_workspace_size(B, Sq, Sk, H, D, deterministic=False, Hk=None) -> int:
    Hk = H if Hk is None else Hk
    return int(library().fa_bwd_workspace_size(B, Sq, Sk, H, Hk, D, int(bool(deterministic))))


def fa_bwd(dout, q, k, v, out, lse, *, softmax_scale=None, causal=False, window_size=(-1, -1),
           alibi_slopes=None, deterministic=False, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """dQ, dK, dV of <dout, attention(q, k, v)>; out and lse are fa_fwd's outputs for the same arguments.
    With k/v of Hk < H heads, dk/dv (B,Sk,Hk,D) sum over the query heads sharing each key/value head."""
    _need(q, "q", torch.bfloat16)
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    Hk = _kv_heads(k, H)
    dev = q.device
    for name, t, shp in (("k", k, (B, Sk, Hk, D)), ("v", v, (B, Sk, Hk, D)), ("dout", dout, (B, Sq, H, D)),
                         ("out", out, (B, Sq, H, D))):
        _need(t, name, torch.bfloat16, shp, dev)
    _need(lse, "lse", torch.float32, (B, H, Sq), dev)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, shp in (("dq", dq, (B, Sq, H, D)), ("dk", dk, (B, Sk, Hk, D)), ("dv", dv, (B, Sk, Hk, D))):
        _need(t, name, torch.bfloat16, shp, dev)
    need = fa_bwd_workspace_size(B, Sq, Sk, H, D, deterministic, Hk=Hk)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, device=dev)
    al, al_stride = _alibi(alibi_slopes, B, H, dev)
    st = library().fa_bwd(_ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dq), _ptr(dk),
                          _ptr(dv), _ptr(workspace), workspace.numel(), B, Sq, Sk, H, Hk, D,
                          _scale(softmax_scale, D), int(bool(causal)), int(window_size[0]), int(window_size[1]),
                          _ptr(al), al_stride, int(bool(deterministic)), _stream_ptr(stream, dev))
    _check("fa_bwd", st)
    return dq, dk, dv


def _cu(t, name, B, total, dev):
    _need(t, name, torch.int32, (B + 1,), dev)
    return t


def fa_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, *, softmax_scale=None,
                  causal=False, window_size=(-1, -1), alibi_slopes=None, out=None, lse=None, stream=None):
    """Packed sequences: q (total_q,H,D), k/v (total_k,Hk,D) bf16, cu_seqlens int32 (B+1,) on the device;
    max_seqlen_* at least the longest sequence. -> out (total_q,H,D) bf16, lse (H,total_q) fp32."""
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3:
        raise ValueError("q must be (total_q, H, D)")
    total_q, H, D = q.shape
    total_k = k.shape[0]
    if k.dim() != 3:
        raise ValueError("k must be (total_k, Hk, D)")
    Hk = int(k.shape[1])
    if Hk < 1 or H % Hk != 0:
        raise ValueError(f"the query heads ({H}) must be a multiple of the key/value heads ({Hk})")
    dev = q.device
    B = int(cu_seqlens_q.numel()) - 1
    _cu(cu_seqlens_q, "cu_seqlens_q", B, total_q, dev)
    _cu(cu_seqlens_k, "cu_seqlens_k", B, total_k, dev)
    _need(k, "k", torch.bfloat16, (total_k, Hk, D), dev)
    _need(v, "v", torch.bfloat16, (total_k, Hk, D), dev)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((H, total_q), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, (total_q, H, D), dev)
    _need(lse, "lse", torch.float32, (H, total_q), dev)
    al, al_stride = _alibi(alibi_slopes, B, H, dev)
    st = library().fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q),
                                 _ptr(cu_seqlens_k), B, total_q, total_k, int(max_seqlen_q), int(max_seqlen_k), H,
                                 Hk, D, _scale(softmax_scale, D), int(bool(causal)), int(window_size[0]),
                                 int(window_size[1]), _ptr(al), al_stride, _stream_ptr(stream, dev))
    _check("fa_fwd_varlen", st)
    return out, lse


def fa_bwd_varlen_workspace_size(B, total_q, total_k, max_seqlen_q, H, D, Hk=None) -> int:
    Hk = H if Hk is None else Hk
    return int(library().fa_bwd_varlen_workspace_size(B, total_q, total_k, max_seqlen_q, H, Hk, D))


def fa_bwd_varlen(dout, q, k, v, out, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, *,
                  softmax_scale=None, causal=False, window_size=(-1, -1), alibi_slopes=None, deterministic=False,
                  dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward of fa_fwd_varlen: dq (total_q,H,D), dk/dv (total_k,Hk,D) bf16."""
    _need(q, "q", torch.bfloat16)
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("q must be (total_q, H, D) and k (total_k, Hk, D)")
    total_q, H, D = q.shape
    total_k, Hk = k.shape[0], int(k.shape[1])
    if Hk < 1 or H % Hk != 0:
        raise ValueError(f"the query heads ({H}) must be a multiple of the key/value heads ({Hk})")
    dev = q.device
    B = int(cu_seqlens_q.numel()) - 1
    _cu(cu_seqlens_q, "cu_seqlens_q", B, total_q, dev)
    _cu(cu_seqlens_k, "cu_seqlens_k", B, total_k, dev)
    for name, t, shp in (("k", k, (total_k, Hk, D)), ("v", v, (total_k, Hk, D)), ("dout", dout, (total_q, H, D)),
                         ("out", out, (total_q, H, D))):
        _need(t, name, torch.bfloat16, shp, dev)
    _need(lse, "lse", torch.float32, (H, total_q), dev)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, shp in (("dq", dq, (total_q, H, D)), ("dk", dk, (total_k, Hk, D)), ("dv", dv, (total_k, Hk, D))):
        _need(t, name, torch.bfloat16, shp, dev)
    need = fa_bwd_varlen_workspace_size(B, total_q, total_k, int(max_seqlen_q), H, D, Hk=Hk)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, device=dev)
    al, al_stride = _alibi(alibi_slopes, B, H, dev)
    st = library().fa_bwd_varlen(_ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dq), _ptr(dk),
                                 _ptr(dv), _ptr(workspace), workspace.numel(), _ptr(cu_seqlens_q),
                                 _ptr(cu_seqlens_k), B, total_q, total_k, int(max_seqlen_q), int(max_seqlen_k), H,
                                 Hk, D, _scale(softmax_scale, D), int(bool(causal)), int(window_size[0]),
                                 int(window_size[1]), _ptr(al), al_stride, int(bool(deterministic)),
                                 _stream_ptr(stream, dev))
    _check("fa_bwd_varlen", st)
    return dq, dk, dv


def fa_decode_num_splits(B, Sq, Sk, H, D, Hk=None) -> int:
    Hk = H if Hk is None else Hk
    return int(library().fa_decode_num_splits(B, Sq, Sk, H, Hk, D))


def fa_decode_workspace_size(B, Sq, Sk, H, D, num_splits=0, Hk=None) -> int:
    Hk = H if Hk is None else Hk
    return int(library().fa_decode_workspace_size(B, Sq, Sk, H, Hk, D, int(num_splits)))


def fa_decode_splitkv(q, k_cache, v_cache, *, softmax_scale=None, causal=False, window_size=(-1, -1),
                      alibi_slopes=None, num_splits=0, workspace=None, out=None, lse=None, stream=None):
    """Split-KV decode: q (B,Sq<=16,H,D), caches (B,Sk,Hk,D) bf16 -> out (B,Sq,H,D) bf16, lse (B,H,Sq) fp32."""
    _need(q, "q", torch.bfloat16)
    B, Sq, H, D = q.shape
    Sk = k_cache.shape[1]
    Hk = _kv_heads(k_cache, H)
    dev = q.device
    _need(k_cache, "k_cache", torch.bfloat16, (B, Sk, Hk, D), dev)
    _need(v_cache, "v_cache", torch.bfloat16, (B, Sk, Hk, D), dev)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, (B, Sq, H, D), dev)
    _need(lse, "lse", torch.float32, (B, H, Sq), dev)
    need = fa_decode_workspace_size(B, Sq, Sk, H, D, num_splits, Hk=Hk)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, device=dev)
    al, al_stride = _alibi(alibi_slopes, B, H, dev)
    st = library().fa_decode_splitkv(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse),
                                     _ptr(workspace), workspace.numel(), B, Sq, Sk, H, Hk, D,
                                     _scale(softmax_scale, D), int(bool(causal)), int(window_size[0]),
                                     int(window_size[1]), _ptr(al), al_stride, int(num_splits),
                                     _stream_ptr(stream, dev))
    _check("fa_decode_splitkv", st)
    return out, lse


def fa_decode_paged(q, k_pages, v_pages, block_table, seqlens_k, max_seqlen_k, *, softmax_scale=None,
                    causal=False, window_size=(-1, -1), alibi_slopes=None, num_splits=0, workspace=None, out=None,
                    lse=None, stream=None):
    """Split-KV decode over a paged cache: q (B,Sq<=16,H,D); k/v pages (num_pages,page_size,Hk,D) bf16;
    block_table (B,max_pages) and seqlens_k (B,) int32 on the device; max_seqlen_k >= every seqlens_k[b].
    -> out (B,Sq,H,D) bf16, lse (B,H,Sq) fp32."""
    _need(q, "q", torch.bfloat16)
    B, Sq, H, D = q.shape
    if k_pages.dim() != 4:
        raise ValueError("k_pages must be (num_pages, page_size, Hk, D)")
    num_pages, page_size, Hk = int(k_pages.shape[0]), int(k_pages.shape[1]), int(k_pages.shape[2])
    if Hk < 1 or H % Hk != 0:
        raise ValueError(f"the query heads ({H}) must be a multiple of the key/value heads ({Hk})")
    dev = q.device
    _need(k_pages, "k_pages", torch.bfloat16, (num_pages, page_size, Hk, D), dev)
    _need(v_pages, "v_pages", torch.bfloat16, (num_pages, page_size, Hk, D), dev)
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be (B, max_pages_per_seq)")
    max_pages = int(block_table.shape[1])
    _need(block_table, "block_table", torch.int32, (B, max_pages), dev)
    _need(seqlens_k, "seqlens_k", torch.int32, (B,), dev)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, (B, Sq, H, D), dev)
    _need(lse, "lse", torch.float32, (B, H, Sq), dev)
    need = fa_decode_workspace_size(B, Sq, int(max_seqlen_k), H, D, num_splits, Hk=Hk)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, device=dev)
    al, al_stride = _alibi(alibi_slopes, B, H, dev)
    st = library().fa_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), _ptr(seqlens_k),
                                   _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), B, Sq, int(max_seqlen_k),
                                   num_pages, page_size, max_pages, H, Hk, D, _scale(softmax_scale, D),
                                   int(bool(causal)), int(window_size[0]), int(window_size[1]), _ptr(al), al_stride,
                                   int(num_splits), _stream_ptr(stream, dev))
    _check("fa_decode_paged", st)
    return out, lse


def fa_decode_kvcache(q, k_cache, v_cache, cache_seqlens, k_new=None, v_new=None, *, rotary_cos=None,
                      rotary_sin=None, rotary_interleaved=False, block_table=None, softmax_scale=None, causal=False,
                      window_size=(-1, -1), alibi_slopes=None, num_splits=0, workspace=None, out=None, lse=None,
                      stream=None):
    """Decode step on a KV cache: appends k_new, v_new (B,S_new,Hk,D) behind cache_seqlens (B,) int32 in
    place (keys rotated), rotates q, and attends. Caches dense (B,rows,Hk,D) or, with block_table
    (B,max_pages) int32, pages (num_pages,page_size,Hk,D). rotary_cos/sin: (len, rotary_dim/2) fp32."""
    _need(q, "q", torch.bfloat16)
    B, Sq, H, D = q.shape
    dev = q.device
    if k_cache.dim() != 4:
        raise ValueError("k_cache must be 4-D")
    Hk = int(k_cache.shape[2])
    if Hk < 1 or H % Hk != 0:
        raise ValueError(f"the query heads ({H}) must be a multiple of the key/value heads ({Hk})")
    _need(k_cache, "k_cache", torch.bfloat16, tuple(k_cache.shape), dev)
    _need(v_cache, "v_cache", torch.bfloat16, tuple(k_cache.shape), dev)
    _need(cache_seqlens, "cache_seqlens", torch.int32, (B,), dev)
    if block_table is not None:
        num_pages, page_size = int(k_cache.shape[0]), int(k_cache.shape[1])
        max_pages = int(block_table.shape[1]) if block_table.dim() == 2 else -1
        _need(block_table, "block_table", torch.int32, (B, max_pages), dev)
        cache_rows = 0
        cap = max_pages * page_size
    else:
        if k_cache.shape[0] != B:
            raise ValueError("a dense cache must be (B, rows, Hk, D)")
        num_pages, page_size, max_pages = 0, 0, 0
        cache_rows = cap = int(k_cache.shape[1])
    S_new = 0
    if k_new is not None:
        S_new = int(k_new.shape[1])
        _need(k_new, "k_new", torch.bfloat16, (B, S_new, Hk, D), dev)
        _need(v_new, "v_new", torch.bfloat16, (B, S_new, Hk, D), dev)
    rot_dim = rot_len = 0
    if rotary_cos is not None:
        _need(rotary_cos, "rotary_cos", torch.float32, device=dev)
        rot_len, half = int(rotary_cos.shape[0]), int(rotary_cos.shape[1])
        _need(rotary_sin, "rotary_sin", torch.float32, (rot_len, half), dev)
        rot_dim = 2 * half
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, (B, Sq, H, D), dev)
    _need(lse, "lse", torch.float32, (B, H, Sq), dev)
    need = fa_decode_workspace_size(B, Sq, cap, H, D, num_splits, Hk=Hk)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, device=dev)
    al, al_stride = _alibi(alibi_slopes, B, H, dev)
    st = library().fa_decode_kvcache(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(cache_seqlens), _ptr(k_new), _ptr(v_new), S_new,
        _ptr(rotary_cos), _ptr(rotary_sin), rot_dim, rot_len, int(bool(rotary_interleaved)), _ptr(block_table),
        num_pages, page_size, max_pages, _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), B, Sq,
        cache_rows, H, Hk, D, _scale(softmax_scale, D), int(bool(causal)), int(window_size[0]), int(window_size[1]),
        _ptr(al), al_stride, int(num_splits), _stream_ptr(stream, dev))
    _check("fa_decode_kvcache", st)
    return out, lse


def fa_fwd_dropout(q, k, v, dropout_p, seed, offset=0, *, softmax_scale=None, causal=False, window_size=(-1, -1),
                   alibi_slopes=None, out=None, lse=None, stream=None):
    """fa_fwd with dropout on the probabilities (Philox4x32-10 mask from seed, offset; see include/fa.h)."""
    _need(q, "q", torch.bfloat16)
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    Hk = _kv_heads(k, H)
    dev = q.device
    _need(k, "k", torch.bfloat16, (B, Sk, Hk, D), dev)
    _need(v, "v", torch.bfloat16, (B, Sk, Hk, D), dev)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=dev)
    _need(out, "out", torch.bfloat16, (B, Sq, H, D), dev)
    _need(lse, "lse", torch.float32, (B, H, Sq), dev)
    al, al_stride = _alibi(alibi_slopes, B, H, dev)
    st = library().fa_fwd_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Sq, Sk, H, Hk, D,
                                  _scale(softmax_scale, D), int(bool(causal)), int(window_size[0]),
                                  int(window_size[1]), _ptr(al), al_stride, float(dropout_p), int(seed), int(offset),
                                  _stream_ptr(stream, dev))
    _check("fa_fwd_dropout", st)
    return out, lse


def fa_bwd_dropout(dout, q, k, v, out, lse, dropout_p, seed, offset=0, *, softmax_scale=None, causal=False,
                   window_size=(-1, -1), alibi_slopes=None, deterministic=False, dq=None, dk=None, dv=None,
                   workspace=None, stream=None):
    """Backward of fa_fwd_dropout with the same dropout_p, seed and offset."""
    _need(q, "q", torch.bfloat16)
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    Hk = _kv_heads(k, H)
    dev = q.device
    for name, t, shp in (("k", k, (B, Sk, Hk, D)), ("v", v, (B, Sk, Hk, D)), ("dout", dout, (B, Sq, H, D)),
                         ("out", out, (B, Sq, H, D))):
        _need(t, name, torch.bfloat16, shp, dev)
    _need(lse, "lse", torch.float32, (B, H, Sq), dev)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = fa_bwd_workspace_size(B, Sq, Sk, H, D, deterministic, Hk=Hk)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, device=dev)
    al, al_stride = _alibi(alibi_slopes, B, H, dev)
    st = library().fa_bwd_dropout(_ptr(dout), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dq), _ptr(dk),
                                  _ptr(dv), _ptr(workspace), workspace.numel(), B, Sq, Sk, H, Hk, D,
                                  _scale(softmax_scale, D), int(bool(causal)), int(window_size[0]),
                                  int(window_size[1]), _ptr(al), al_stride, int(bool(deterministic)),
                                  float(dropout_p), int(seed), int(offset), _stream_ptr(stream, dev))
    _check("fa_bwd_dropout", st)
    return dq, dk, dv


FA_SELFTEST_SITE = 0x7E


def fa_selftest_wait_timeout(stream=None):
    """Launch the diagnostic warp whose bounded wait runs out (about one second)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    _check("fa_selftest_wait_timeout", library().fa_selftest_wait_timeout(_stream_ptr(stream, dev)))


FA_FAULT_NONE = 0
FA_FAULT_FWD_SKIP_KEY_TILE = 1
FA_FAULT_BWD_SKIP_KEY_TILE = 2


def fa_debug_set_fault(fault=FA_FAULT_NONE, wait_limit_ns=0):
    """Diagnostic: set the kernels' bounded-wait limit (0 = default, one second) and a
    fault to inject in later launches (see include/fa.h)."""
    _check("fa_debug_set_fault", library().fa_debug_set_fault(int(fault), int(wait_limit_ns)))


def fa_device_status(stream=None):
    """Synchronise the stream and read/clear the device status word: (status, raw word)."""
    dev = torch.device("cuda", torch.cuda.current_device())
    word = ctypes.c_uint(0)
    st = library().fa_device_status(_stream_ptr(stream, dev), ctypes.byref(word))
    return int(st), int(word.value)
