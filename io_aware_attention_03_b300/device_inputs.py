"""Move the seeded host inputs of :mod:`io_aware_attention_03_b300.inputs` to the GPU.

Layout plumbing only (uploads and index scatters with torch); no attention
arithmetic.  bf16 values travel as their raw bits, so the device sees exactly
the numbers the oracle sees.
"""

from __future__ import annotations

import numpy as np
import torch

from .inputs import DecodeInputs


def to_device_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bits (host) -> bf16 CUDA tensor with the same values."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def to_host_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bits on the host (exact)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def to_host_f64(t: torch.Tensor) -> np.ndarray:
    """bf16/fp32 tensor -> float64 numpy array (exact widening)."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def _token_rows(di: DecodeInputs, paged: bool, max_seqlen: int) -> np.ndarray:
    """Row index of every cached token (sequence-major order) in the target layout."""
    lens = di.seqlens.astype(np.int64)
    seq = np.repeat(np.arange(di.num_seqs, dtype=np.int64), lens)
    t = np.arange(int(lens.sum()), dtype=np.int64) - np.repeat(di.offsets[:-1], lens)
    if not paged:
        return seq * max_seqlen + t
    pages = di.pages_per_seq()
    page_start = np.zeros(di.num_seqs, np.int64)
    page_start[1:] = np.cumsum(pages)[:-1]
    gp = page_start[seq] + t // di.page_size
    return di.page_ids.astype(np.int64)[gp] * di.page_size + t % di.page_size


def decode_caches(di: DecodeInputs, paged: bool, device="cuda", max_seqlen: int | None = None):
    """Device K and V caches for a decode batch.

    Contiguous: ``[S, max_seqlen, H, d]``; paged: pools ``[num_pages, page_size, H, d]``.
    Slots that hold no token are zero.
    """
    H, d = di.q.shape[1], di.q.shape[2]
    L = di.max_seqlen if max_seqlen is None else int(max_seqlen)
    if paged:
        shape = (int(di.page_ids.shape[0]), di.page_size, H, d)
    else:
        shape = (di.num_seqs, L, H, d)
    rows = torch.from_numpy(_token_rows(di, paged, L)).to(device)
    out = []
    for tokens in (di.k_tokens, di.v_tokens):
        cache = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        flat = cache.view(-1, H, d)
        # upload in pieces to bound host->device staging
        step = 1 << 16
        for a in range(0, tokens.shape[0], step):
            flat[rows[a:a + step]] = to_device_bf16(tokens[a:a + step], device)
        out.append(cache)
    return out[0], out[1]


def fp8_caches(di: DecodeInputs, f8, paged: bool, device="cuda", max_seqlen: int | None = None):
    """Device FP8 K and V caches (raw e4m3 bytes as uint8) of an :class:`Fp8Cache`, in the
    contiguous or paged layout of :func:`decode_caches`, plus the per-head scales."""
    H, d = di.q.shape[1], di.q.shape[2]
    L = di.max_seqlen if max_seqlen is None else int(max_seqlen)
    shape = (int(di.page_ids.shape[0]), di.page_size, H, d) if paged else (di.num_seqs, L, H, d)
    rows = torch.from_numpy(_token_rows(di, paged, L)).to(device)
    out = []
    for tokens in (f8.k_tokens, f8.v_tokens):
        cache = torch.zeros(shape, dtype=torch.uint8, device=device)
        flat = cache.view(-1, H, d)
        step = 1 << 16
        for a in range(0, tokens.shape[0], step):
            flat[rows[a:a + step]] = torch.from_numpy(np.ascontiguousarray(tokens[a:a + step])).to(device)
        out.append(cache)
    ks = torch.from_numpy(f8.k_scale.astype(np.float32)).to(device)
    vs = torch.from_numpy(f8.v_scale.astype(np.float32)).to(device)
    return out[0], out[1], ks, vs


def decode_device_inputs(di: DecodeInputs, paged: bool, device="cuda"):
    """(q [S,1,H,d], kcache, vcache, seqlens int32, page_table int32 or None) on the device."""
    q = to_device_bf16(di.q, device).view(di.num_seqs, 1, di.q.shape[1], di.q.shape[2])
    kc, vc = decode_caches(di, paged, device)
    seqlens = torch.from_numpy(di.seqlens.astype(np.int32)).to(device)
    pt = torch.from_numpy(di.page_table()).to(device) if paged else None
    return q, kc, vc, seqlens, pt


def fp8_prefill_device(f8, device="cuda"):
    """Device tensors of :class:`~io_aware_attention_03_b300.inputs.Fp8Prefill`: q, k as e4m3
    bytes ``[B, N, H, d]`` (uint8), V transposed to ``[B, H, d, Np]`` with keys contiguous and
    zero padding up to ``Np`` (N rounded up to 16), and the three fp32 ``[H]`` scales."""
    B, N, H, d = f8.v.shape
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(device)
    q, k = up(f8.q), up(f8.k)
    Np = (N + 15) // 16 * 16
    vt = torch.zeros((B, H, d, Np), dtype=torch.uint8, device=device)
    vt[..., :N] = up(f8.v).permute(0, 2, 3, 1)
    scales = [up(s.astype(np.float32)) for s in (f8.q_scale, f8.k_scale, f8.v_scale)]
    return q, k, vt, scales[0], scales[1], scales[2]
