"""Python binding of the C ABI in ``include/attn_b300.h`` (ctypes).

Argument marshalling only: every step of the computation runs in the CUDA
library.  Importing this module loads ``libattn_b300.so`` and raises
``ImportError`` when it has not been built; there is no fallback.

The preconditions of the forward call on "Beyond the memory wall"
(tiptinker), section "구현 가이드" -- CUDA tensors, bf16, contiguous, layout
``[batch, seq_len, num_heads, head_dim]`` -- are checked here, before the call,
because the C ABI sees only pointers.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libattn_b300.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is not built; run `python -m io_aware_attention_03_b300.build`")
_lib = ctypes.CDLL(_LIB_PATH)

_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_lib.attn_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]
_lib.attn_fwd.restype = _i
_lib.attn_fwd_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp]
_lib.attn_fwd_fp8.restype = _i
_lib.attn_bwd_workspace_size.argtypes = [_i, _i, _i, _i]
_lib.attn_bwd_workspace_size.restype = _sz
_lib.attn_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _vp, _sz,
                          _vp]
_lib.attn_bwd.restype = _i
_lib.attn_prefill_paged.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                                    _i, _f, _vp]
_lib.attn_prefill_paged.restype = _i
_lib.attn_decode_workspace_size.argtypes = [_i, _i, _i, _i]
_lib.attn_decode_workspace_size.restype = _sz
_lib.attn_decode.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _vp,
                             _sz, _vp]
_lib.attn_decode.restype = _i
_lib.attn_decode_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                                 _i, _i, _f, _vp, _sz, _vp]
_lib.attn_decode_fp8.restype = _i
_lib.attn_decode_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                                     _f, _vp]
_lib.attn_decode_noalloc.restype = _i
_lib.attn_last_device_status.argtypes = [_vp]
_lib.attn_last_device_status.restype = _i
_lib.attn_status_string.argtypes = [_i]
_lib.attn_status_string.restype = ctypes.c_char_p

LIBRARY_PATH = _LIB_PATH
EXPORTED = ("attn_fwd", "attn_fwd_fp8", "attn_bwd", "attn_bwd_workspace_size", "attn_prefill_paged", "attn_decode_workspace_size", "attn_decode",
            "attn_decode_fp8", "attn_decode_noalloc", "attn_last_device_status",
            "attn_status_string")
NOALLOC_SCRATCH_BYTES = 64 << 20  # ATTN_DECODE_NOALLOC_SCRATCH_BYTES


class AttnError(RuntimeError):
    """A non-zero attn_status from the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {attn_status_string(status)} ({status})")


def attn_status_string(status: int) -> str:
    return _lib.attn_status_string(int(status)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _require(t: torch.Tensor, name: str, dtype=torch.bfloat16, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
             scale: float | None = None, out: torch.Tensor | None = None,
             lse: torch.Tensor | None = None, return_lse: bool = True):
    """O = softmax(scale * Q K^T [+ causal mask]) V on the current CUDA stream.

    q, k, v: bf16 ``[B, N, H, d]`` contiguous CUDA tensors, d in {64, 128}.
    ``scale`` defaults to ``1/sqrt(d)``.  Returns ``(O, LSE)`` with O bf16
    ``[B, N, H, d]`` and LSE fp32 ``[B, H, N]`` (natural log), or O alone when
    ``return_lse`` is False.
    """
    for name, t in (("q", q), ("k", k), ("v", v)):
        _require(t, name, device=q.device)
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must all be [B, N, H, d] with the same shape")
    B, N, H, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    _require(out, "out", device=q.device)
    if out.shape != q.shape:
        raise ValueError("out must match q")
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if lse is not None:
        _require(lse, "lse", dtype=torch.float32, device=q.device)
        if lse.shape != (B, H, N):
            raise ValueError("lse must be [B, H, N]")
    rc = _lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d, int(bool(causal)),
                       float(scale), _vp(_stream_handle(q.device)))
    if rc != 0:
        raise AttnError(rc, "attn_fwd")
    return (out, lse) if return_lse else out


def attn_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(_lib.attn_bwd_workspace_size(B, H, N, d))


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
             dout: torch.Tensor, causal: bool = False, scale: float | None = None,
             dq: torch.Tensor | None = None, dk: torch.Tensor | None = None,
             dv: torch.Tensor | None = None, workspace: torch.Tensor | None = None):
    """Gradients of :func:`attn_fwd`: (dQ, dK, dV) for the upstream gradient ``dout``.

    q, k, v, o, dout: bf16 ``[B, N, H, d]``; lse: fp32 ``[B, H, N]`` -- o and lse as returned
    by :func:`attn_fwd` for the same q, k, v, causal and scale.  Returns bf16 tensors shaped
    like q.  ``workspace`` (uint8 CUDA tensor of ``attn_bwd_workspace_size`` bytes) is
    allocated when not given.
    """
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _require(t, name, device=dev)
        if t.shape != q.shape or q.dim() != 4:
            raise ValueError(f"{name} must be [B, N, H, d] like q")
    B, N, H, d = q.shape
    _require(lse, "lse", dtype=torch.float32, device=dev)
    if lse.shape != (B, H, N):
        raise ValueError("lse must be [B, H, N]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    grads = []
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        if t is None:
            t = torch.empty_like(q)
        _require(t, name, device=dev)
        if t.shape != q.shape:
            raise ValueError(f"{name} must match q")
        grads.append(t)
    if workspace is None:
        workspace = torch.empty(max(attn_bwd_workspace_size(B, H, N, d), 16), dtype=torch.uint8,
                                device=dev)
    _require(workspace, "workspace", dtype=torch.uint8, device=dev)
    rc = _lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(grads[0]),
                       _ptr(grads[1]), _ptr(grads[2]), B, H, N, d, int(bool(causal)), float(scale),
                       _ptr(workspace), workspace.numel(), _vp(_stream_handle(dev)))
    if rc != 0:
        raise AttnError(rc, "attn_bwd")
    return grads[0], grads[1], grads[2]


_E4M3_DTYPES = (torch.uint8, torch.float8_e4m3fn)


def _require_e4m3(t, name, device):
    if not isinstance(t, torch.Tensor) or t.dtype not in _E4M3_DTYPES:
        raise ValueError(f"{name} must be uint8 or float8_e4m3fn (e4m3 bytes)")
    _require(t, name, dtype=t.dtype, device=device)


def fp8_vt_stride(N: int) -> int:
    """Row stride (keys) of the transposed FP8 V operand: N rounded up to a multiple of 16."""
    return (int(N) + 15) // 16 * 16


def attn_fwd_fp8(q: torch.Tensor, k: torch.Tensor, vt: torch.Tensor, q_scale: torch.Tensor,
                 k_scale: torch.Tensor, v_scale: torch.Tensor, causal: bool = False,
                 scale: float | None = None, out: torch.Tensor | None = None,
                 lse: torch.Tensor | None = None, return_lse: bool = True):
    """FP8 (E4M3) forward attention with one fp32 scale per head for Q, K and V.

    q, k: e4m3 bytes (``torch.uint8`` or ``torch.float8_e4m3fn``) ``[B, N, H, d]``, d in {64, 128};
    vt: V transposed, ``[B, H, d, Np]`` with ``Np = fp8_vt_stride(N)`` (keys contiguous;
    entries at keys >= N are ignored); q_scale, k_scale, v_scale: fp32 ``[H]`` (value =
    scale[h] * e4m3).  Returns ``(O, LSE)``: O bf16 ``[B, N, H, d]``, LSE fp32 ``[B, H, N]``.
    """
    dev = q.device
    for name, t in (("q", q), ("k", k), ("vt", vt)):
        _require_e4m3(t, name, dev)
    for name, t in (("q_scale", q_scale), ("k_scale", k_scale), ("v_scale", v_scale)):
        _require(t, name, dtype=torch.float32, device=dev)
    if q.dim() != 4 or k.shape != q.shape:
        raise ValueError("q and k must be [B, N, H, d] with the same shape")
    B, N, H, d = q.shape
    if vt.shape != (B, H, d, fp8_vt_stride(N)):
        raise ValueError(f"vt must be [B, H, d, {fp8_vt_stride(N)}] (V transposed, keys padded to 16)")
    if q_scale.shape != (H,) or k_scale.shape != (H,) or v_scale.shape != (H,):
        raise ValueError("scales must be [H]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, N, H, d), dtype=torch.bfloat16, device=dev)
    _require(out, "out", device=dev)
    if out.shape != (B, N, H, d):
        raise ValueError("out must be [B, N, H, d]")
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    if lse is not None:
        _require(lse, "lse", dtype=torch.float32, device=dev)
        if lse.shape != (B, H, N):
            raise ValueError("lse must be [B, H, N]")
    rc = _lib.attn_fwd_fp8(_ptr(q), _ptr(k), _ptr(vt), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
                           _ptr(out), _ptr(lse), B, H, N, d, int(bool(causal)), float(scale),
                           _vp(_stream_handle(dev)))
    if rc != 0:
        raise AttnError(rc, "attn_fwd_fp8")
    return (out, lse) if return_lse else out


def attn_prefill_paged(q: torch.Tensor, kcache: torch.Tensor, vcache: torch.Tensor,
                       seqlens: torch.Tensor, page_table: torch.Tensor, causal: bool = True,
                       scale: float | None = None, out: torch.Tensor | None = None,
                       lse: torch.Tensor | None = None, return_lse: bool = True):
    """Prefill of a chunk of Nq new tokens per sequence against a 16-token paged K/V cache.

    q: bf16 ``[B, Nq, H, d]`` (row i of sequence b is cache position
    ``seqlens[b] - Nq + i``); kcache, vcache: pools ``[num_pages, 16, H, d]``
    holding every key of each sequence, the chunk's included; seqlens: int32
    ``[B]`` on the device (keys per sequence, >= Nq); page_table: int32
    ``[B, max_pages_per_seq]``.  Causal masking is aligned to the end of the
    cache.  Returns ``(O, LSE)``: O bf16 like q, LSE fp32 ``[B, H, Nq]``.
    """
    _require(q, "q")
    dev = q.device
    for name, t in (("kcache", kcache), ("vcache", vcache)):
        _require(t, name, device=dev)
    _require(seqlens, "seqlens", dtype=torch.int32, device=dev)
    _require(page_table, "page_table", dtype=torch.int32, device=dev)
    if q.dim() != 4 or kcache.dim() != 4 or kcache.shape != vcache.shape:
        raise ValueError("q must be [B, Nq, H, d] and the caches [num_pages, 16, H, d]")
    B, Nq, H, d = q.shape
    if kcache.shape[2:] != (H, d):
        raise ValueError("cache heads/head_dim must match q")
    if seqlens.shape != (B,) or page_table.dim() != 2 or page_table.shape[0] != B:
        raise ValueError("seqlens must be [B] and page_table [B, max_pages_per_seq]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    _require(out, "out", device=dev)
    if out.shape != q.shape:
        raise ValueError("out must match q")
    if lse is None and return_lse:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    if lse is not None:
        _require(lse, "lse", dtype=torch.float32, device=dev)
        if lse.shape != (B, H, Nq):
            raise ValueError("lse must be [B, H, Nq]")
    rc = _lib.attn_prefill_paged(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(seqlens), _ptr(page_table),
                                 _ptr(out), _ptr(lse), B, H, Nq, d, kcache.shape[1],
                                 page_table.shape[1], kcache.shape[0], int(bool(causal)),
                                 float(scale), _vp(_stream_handle(dev)))
    if rc != 0:
        raise AttnError(rc, "attn_prefill_paged")
    return (out, lse) if return_lse else out


def _decode_layout(q, kcache, vcache, seqlens, page_table, out, lse, max_seqlen):
    """Shape checks shared by the decode entry points; returns the C call's sizes.

    Checks q ``[S, 1, H, d]`` (or ``[S, H, d]``), caches 4-D of one shape whose
    heads and head_dim match q, seqlens ``[S]``, out like q and lse ``[S, H]``.
    Contiguous cache ``[S, L, H, d]``: the kernel addresses token t of sequence
    s at row ``s * max_seqlen + t``, so max_seqlen must be L.  Paged pools
    ``[num_pages, 16, H, d]`` with page_table ``[S, max_pages_per_seq]``:
    max_seqlen defaults to ``max_pages_per_seq * 16``.
    Returns ``(S, H, d, max_seqlen, page_size, max_pages, num_pages)``.
    """
    if kcache.dim() != 4 or kcache.shape != vcache.shape:
        raise ValueError("kcache and vcache must be 4-D with the same shape")
    S = q.shape[0]
    H, d = q.shape[-2], q.shape[-1]
    if q.dim() not in (3, 4) or q.numel() != S * H * d:
        raise ValueError("q must be [S, 1, H, d] or [S, H, d]")
    if seqlens.shape != (S,):
        raise ValueError("seqlens must be [S]")
    if kcache.shape[2:] != (H, d):
        raise ValueError("cache heads/head_dim must match q")
    if out is not None and out.shape != q.shape:
        raise ValueError("out must match q")
    if lse is not None and lse.shape != (S, H):
        raise ValueError("lse must be [S, H]")
    if page_table is None:
        if kcache.shape[0] != S:
            raise ValueError("contiguous cache must be [S, max_seqlen, H, d]")
        cache_len = kcache.shape[1]
        if max_seqlen is not None and int(max_seqlen) != cache_len:
            raise ValueError(f"contiguous cache: max_seqlen must be the cache's second dimension "
                             f"({cache_len}), the row stride of the cache")
        return S, H, d, cache_len, 16, 0, 0
    if page_table.dim() != 2 or page_table.shape[0] != S:
        raise ValueError("page_table must be [S, max_pages_per_seq]")
    page_size, max_pages, num_pages = kcache.shape[1], page_table.shape[1], kcache.shape[0]
    max_seqlen = max_pages * page_size if max_seqlen is None else int(max_seqlen)
    return S, H, d, max_seqlen, page_size, max_pages, num_pages


def attn_decode_workspace_size(num_seqs: int, H: int, d: int, max_seqlen: int) -> int:
    return int(_lib.attn_decode_workspace_size(num_seqs, H, d, max_seqlen))


def attn_decode(q: torch.Tensor, kcache: torch.Tensor, vcache: torch.Tensor, seqlens: torch.Tensor,
                page_table: torch.Tensor | None = None, scale: float | None = None,
                out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                workspace: torch.Tensor | None = None, max_seqlen: int | None = None,
                return_lse: bool = True):
    """One-token decode against a contiguous or 16-token paged K/V cache.

    q: bf16 ``[S, 1, H, d]`` (or ``[S, H, d]``).  Contiguous cache: kcache, vcache
    bf16 ``[S, max_seqlen, H, d]``.  Paged cache: pools ``[num_pages, 16, H, d]``
    and ``page_table`` int32 ``[S, max_pages_per_seq]``.  seqlens: int32 ``[S]``
    on the device.  Returns ``(O, LSE)``: O bf16 shaped like q, LSE fp32 ``[S, H]``.
    ``workspace`` (uint8 CUDA tensor) is allocated when not given.
    """
    _require(q, "q")
    dev = q.device
    _require(kcache, "kcache", device=dev)
    _require(vcache, "vcache", device=dev)
    _require(seqlens, "seqlens", dtype=torch.int32, device=dev)
    if page_table is not None:
        _require(page_table, "page_table", dtype=torch.int32, device=dev)
    if out is not None:
        _require(out, "out", device=dev)
    if lse is not None:
        _require(lse, "lse", dtype=torch.float32, device=dev)
    S, H, d, max_seqlen, page_size, max_pages, num_pages = _decode_layout(
        q, kcache, vcache, seqlens, page_table, out, lse, max_seqlen)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((S, H), dtype=torch.float32, device=dev)
    ws_bytes = attn_decode_workspace_size(S, H, d, max_seqlen)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    _require(workspace, "workspace", dtype=torch.uint8, device=dev)
    rc = _lib.attn_decode(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(seqlens), _ptr(page_table),
                          _ptr(out), _ptr(lse), S, H, d, max_seqlen, page_size, max_pages, num_pages,
                          float(scale), _ptr(workspace), workspace.numel(),
                          _vp(_stream_handle(dev)))
    if rc != 0:
        raise AttnError(rc, "attn_decode")
    return (out, lse) if return_lse else out


def attn_decode_fp8(q: torch.Tensor, kcache: torch.Tensor, vcache: torch.Tensor,
                    k_scale: torch.Tensor, v_scale: torch.Tensor, seqlens: torch.Tensor,
                    page_table: torch.Tensor | None = None, scale: float | None = None,
                    out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                    workspace: torch.Tensor | None = None, max_seqlen: int | None = None,
                    return_lse: bool = True):
    """attn_decode over an FP8 (E4M3) K/V cache with one fp32 scale per head.

    kcache, vcache: e4m3 bytes (``torch.uint8`` or ``torch.float8_e4m3fn``) in the
    layouts of :func:`attn_decode`; k_scale, v_scale: fp32 ``[H]`` on the device
    (key = k_scale[h] * e4m3 value, likewise for values).  Other arguments and the
    result as :func:`attn_decode`.
    """
    _require(q, "q")
    dev = q.device
    for name, t in (("kcache", kcache), ("vcache", vcache)):
        if not isinstance(t, torch.Tensor) or t.dtype not in (torch.uint8, torch.float8_e4m3fn):
            raise ValueError(f"{name} must be uint8 or float8_e4m3fn (e4m3 bytes)")
        _require(t, name, dtype=t.dtype, device=dev)
    _require(k_scale, "k_scale", dtype=torch.float32, device=dev)
    _require(v_scale, "v_scale", dtype=torch.float32, device=dev)
    _require(seqlens, "seqlens", dtype=torch.int32, device=dev)
    if page_table is not None:
        _require(page_table, "page_table", dtype=torch.int32, device=dev)
    if out is not None:
        _require(out, "out", device=dev)
    if lse is not None:
        _require(lse, "lse", dtype=torch.float32, device=dev)
    S, H, d, max_seqlen, page_size, max_pages, num_pages = _decode_layout(
        q, kcache, vcache, seqlens, page_table, out, lse, max_seqlen)
    if k_scale.shape != (H,) or v_scale.shape != (H,):
        raise ValueError("scales must be [H]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((S, H), dtype=torch.float32, device=dev)
    ws_bytes = attn_decode_workspace_size(S, H, d, max_seqlen)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    _require(workspace, "workspace", dtype=torch.uint8, device=dev)
    rc = _lib.attn_decode_fp8(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(k_scale), _ptr(v_scale),
                              _ptr(seqlens), _ptr(page_table), _ptr(out), _ptr(lse), S, H, d,
                              max_seqlen, page_size, max_pages, num_pages, float(scale),
                              _ptr(workspace), workspace.numel(), _vp(_stream_handle(dev)))
    if rc != 0:
        raise AttnError(rc, "attn_decode_fp8")
    return (out, lse) if return_lse else out


def attn_decode_noalloc(q: torch.Tensor, kcache: torch.Tensor, vcache: torch.Tensor,
                        seqlens: torch.Tensor, out: torch.Tensor, lse: torch.Tensor | None = None,
                        page_table: torch.Tensor | None = None, scale: float | None = None,
                        max_seqlen: int | None = None):
    """attn_decode without a workspace, for callers that cannot allocate device memory.

    The caller passes every tensor, outputs included (``out`` like q, ``lse``
    fp32 ``[S, H]`` or None); this function allocates nothing.  The split
    partials go to the library's fixed scratch array of ``NOALLOC_SCRATCH_BYTES``
    per device, so calls on one device must be ordered on one stream.
    """
    for name, t in (("q", q), ("kcache", kcache), ("vcache", vcache), ("out", out)):
        _require(t, name, device=q.device)
    _require(seqlens, "seqlens", dtype=torch.int32, device=q.device)
    if lse is not None:
        _require(lse, "lse", dtype=torch.float32, device=q.device)
    if page_table is not None:
        _require(page_table, "page_table", dtype=torch.int32, device=q.device)
    S, H, d, max_seqlen, page_size, max_pages, num_pages = _decode_layout(
        q, kcache, vcache, seqlens, page_table, out, lse, max_seqlen)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rc = _lib.attn_decode_noalloc(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(seqlens), _ptr(page_table),
                                  _ptr(out), _ptr(lse), S, H, d, max_seqlen, page_size, max_pages,
                                  num_pages, float(scale), _vp(_stream_handle(q.device)))
    if rc != 0:
        raise AttnError(rc, "attn_decode_noalloc")
    return out, lse


def attn_last_device_status(stream=None) -> int:
    """Synchronise the stream (default: current) and return/clear the device status word."""
    handle = _stream_handle(None) if stream is None else getattr(stream, "cuda_stream", stream)
    return int(_lib.attn_last_device_status(_vp(handle)))
