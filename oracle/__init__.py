"""fp64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs import this package.  The CUDA
library and its Python binding never import it, and it never imports them.

The arithmetic lives in ``oracle.c`` (plain fp64 C with OpenMP over rows); this
module builds it with gcc on first use and marshals numpy arrays into it.
Every function states the definition it computes; see ``oracle.c`` for the
passages of the pages it follows:

* "FlashAttention complete summary" (cell-devlog), section "Attention이 뭔가":
  ``softmax(Q K^T / sqrt(d_k)) V``.
* "Flash Attention ... complete guide" (holysheep), section "Online Softmax
  알고리즘": safe softmax, ``m = max``, ``l = sum exp(x - m)``, ``f / l``.

Inputs are bf16 values carried as their raw 16 bits in ``numpy.uint16`` arrays,
so the oracle sees exactly the numbers the GPU sees.  Outputs are fp64.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` with gcc (OpenMP) and return its path."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
        f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
        i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
        i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
        c_int, c_long, c_double = ctypes.c_int, ctypes.c_long, ctypes.c_double
        lib.oracle_attn_fwd.argtypes = [u16p, u16p, u16p, c_int, c_int, c_long, c_long, c_int,
                                        c_int, c_double, f64p, f64p, c_int]
        lib.oracle_attn_rows.argtypes = [u16p, u16p, u16p, c_int, c_int, c_long, c_long, c_int,
                                         c_int, c_double, i64p, c_long, f64p, f64p, c_int]
        lib.oracle_attn_probs.argtypes = [u16p, u16p, c_int, c_int, c_long, c_long, c_int, c_int,
                                          c_double, f64p]
        lib.oracle_decode.argtypes = [u16p, u16p, u16p, i32p, ctypes.c_void_p, c_int, c_int, c_int,
                                      c_long, c_int, c_long, c_long, c_double, f64p, f64p, c_int]
        lib.oracle_max_threads.argtypes = []
        for f in (lib.oracle_attn_fwd, lib.oracle_attn_rows, lib.oracle_attn_probs,
                  lib.oracle_decode, lib.oracle_max_threads):
            f.restype = c_int
        _lib = lib
        return lib


def max_threads() -> int:
    """OpenMP threads the oracle uses when ``nthreads=0`` (OMP_NUM_THREADS or all cores)."""
    return int(_load().oracle_max_threads())


def _u16(a: np.ndarray) -> np.ndarray:
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (numpy.uint16)")
    return np.ascontiguousarray(a)


def attn_fwd(q, k, v, causal: bool, scale: float, nthreads: int = 0):
    """O [B,Nq,H,d] and LSE [B,H,Nq] (fp64) of ``softmax(scale * Q K^T [+ causal mask]) V``.

    q: [B, Nq, H, d]; k, v: [B, Nk, H, d] (bf16 bits).  Causal keeps key j
    for query i when ``j <= i + (Nk - Nq)`` (``j <= i`` for square problems).
    """
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Nq, H, d = q.shape
    Nk = k.shape[1]
    if k.shape != (B, Nk, H, d) or v.shape != k.shape:
        raise ValueError("shape mismatch")
    o = np.empty((B, Nq, H, d), np.float64)
    lse = np.empty((B, H, Nq), np.float64)
    rc = _load().oracle_attn_fwd(q, k, v, B, H, Nq, Nk, d, int(bool(causal)), float(scale), o, lse,
                                 int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_attn_fwd failed")
    return o, lse


def attn_rows(q, k, v, causal: bool, scale: float, rows, nthreads: int = 0):
    """The same definition for selected rows only.

    rows: int array [R, 3] of (b, h, i).  Returns O rows [R, d] and LSE [R] (fp64).
    """
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Nq, H, d = q.shape
    Nk = k.shape[1]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    o = np.empty((rows.shape[0], d), np.float64)
    lse = np.empty((rows.shape[0],), np.float64)
    rc = _load().oracle_attn_rows(q, k, v, B, H, Nq, Nk, d, int(bool(causal)), float(scale), rows,
                                  rows.shape[0], o, lse, int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_attn_rows failed")
    return o, lse


def attn_probs(q, k, causal: bool, scale: float):
    """The softmax matrix P [B, H, Nq, Nk] (fp64), zero where a key is masked."""
    q, k = _u16(q), _u16(k)
    B, Nq, H, d = q.shape
    Nk = k.shape[1]
    P = np.empty((B, H, Nq, Nk), np.float64)
    rc = _load().oracle_attn_probs(q, k, B, H, Nq, Nk, d, int(bool(causal)), float(scale), P)
    if rc != 0:
        raise RuntimeError("oracle_attn_probs failed")
    return P


def decode(q, kcache, vcache, seqlens, scale: float, page_table=None, page_size: int = 16,
           nthreads: int = 0):
    """One-token decode: O [S, H, d] and LSE [S, H] (fp64).

    q: [S, H, d] (or [S, 1, H, d]).  Contiguous cache: kcache/vcache
    [S, max_seqlen, H, d].  Paged cache: pools [num_pages, page_size, H, d] with
    ``page_table`` int32 [S, max_pages_per_seq]; key t of sequence s is
    ``pool[page_table[s, t // page_size], t % page_size]``.
    """
    q = _u16(q)
    S = q.shape[0]
    H, d = q.shape[-2], q.shape[-1]
    q = q.reshape(S, H, d)
    kc, vc = _u16(kcache), _u16(vcache)
    seqlens = np.ascontiguousarray(np.asarray(seqlens, dtype=np.int32))
    if page_table is None:
        max_seqlen = kc.shape[1]
        pt, maxp, npages = None, 0, 0
    else:
        pt_arr = np.ascontiguousarray(np.asarray(page_table, dtype=np.int32))
        maxp = pt_arr.shape[1]
        npages = kc.shape[0]
        max_seqlen = maxp * page_size
        pt = pt_arr.ctypes.data_as(ctypes.c_void_p)
    o = np.empty((S, H, d), np.float64)
    lse = np.empty((S, H), np.float64)
    rc = _load().oracle_decode(q, kc, vc, seqlens, pt, S, H, d, max_seqlen, page_size, maxp, npages,
                               float(scale), o, lse, int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_decode failed")
    return o, lse


def prefill_paged(q, kpool, vpool, seqlens, page_table, causal: bool, scale: float,
                  page_size: int = 16, nthreads: int = 0):
    """Prefill of a chunk of Nq queries per sequence against a paged K/V cache (fp64).

    The definition of :func:`attn_fwd` per sequence, with its keys and values
    gathered from the pools: for sequence b the keys are t = 0 .. seqlens[b]-1,
    key t being ``pool[page_table[b, t // page_size], t % page_size]``; query
    row i is the token at position ``seqlens[b] - Nq + i``, so under the causal
    mask it sees keys ``j <= i + seqlens[b] - Nq`` (the bottom-right alignment
    of :func:`attn_fwd` for Nk = seqlens[b] keys).  q: [B, Nq, H, d]; pools
    [num_pages, page_size, H, d]; page_table int [B, max_pages_per_seq].
    Returns O [B, Nq, H, d] and LSE [B, H, Nq].
    """
    q, kpool, vpool = _u16(q), _u16(kpool), _u16(vpool)
    B, Nq, H, d = q.shape
    pt = np.asarray(page_table)
    o = np.empty((B, Nq, H, d), np.float64)
    lse = np.empty((B, H, Nq), np.float64)
    for b in range(B):
        L = int(seqlens[b])
        if L < Nq:
            raise ValueError("every sequence holds at least its Nq chunk tokens")
        t = np.arange(L)
        pages = pt[b, t // page_size]
        kb = np.ascontiguousarray(kpool[pages, t % page_size])[None]
        vb = np.ascontiguousarray(vpool[pages, t % page_size])[None]
        ob, lb = attn_fwd(q[b:b + 1], kb, vb, causal, scale, nthreads)
        o[b] = ob[0]
        lse[b] = lb[0]
    return o, lse


def e4m3_value(bits) -> np.ndarray:
    """FP8 E4M3 bits -> exact fp64 values, from the format's definition: sign bit,
    4 exponent bits e (bias 7), 3 mantissa bits m; e = 0 is subnormal
    (m/8 * 2^-6), otherwise (1 + m/8) * 2^(e-7); e = 15 with m = 7 is NaN (the
    format has no infinities)."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    s = (b >> 7) & 1
    e = (b >> 3) & 0xF
    m = b & 7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def decode_values(q, kvals, vvals, seqlens, scale: float, page_table=None, page_size: int = 16):
    """One-token decode over real-valued caches: O [S, H, d], LSE [S, H] (fp64).

    The definition of :func:`decode` with the keys and values given as fp64
    numbers instead of bf16 bits (q stays bf16 bits [S, H, d] or [S, 1, H, d]).
    Per sequence s and head h: s_t = scale * q . k_t over its L_s keys, m = max,
    l = sum exp(s_t - m), O = sum exp(s_t - m) / l * v_t, LSE = m + ln l;
    an empty sequence gives O = 0, LSE = -inf.
    """
    q = _u16(q)
    S = q.shape[0]
    H, d = q.shape[-2], q.shape[-1]
    qv = (q.reshape(S, H, d).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    kvals = np.asarray(kvals, np.float64)
    vvals = np.asarray(vvals, np.float64)
    o = np.zeros((S, H, d), np.float64)
    lse = np.full((S, H), -np.inf, np.float64)
    for s in range(S):
        L = int(seqlens[s])
        if L == 0:
            continue
        t = np.arange(L)
        if page_table is None:
            k, v = kvals[s, :L], vvals[s, :L]                        # [L, H, d]
        else:
            pages = np.asarray(page_table)[s, t // page_size]
            k, v = kvals[pages, t % page_size], vvals[pages, t % page_size]
        sc = scale * np.einsum("hd,lhd->hl", qv[s], k)               # [H, L]
        m = sc.max(axis=1, keepdims=True)
        w = np.exp(sc - m)
        l = w.sum(axis=1, keepdims=True)
        o[s] = np.einsum("hl,lhd->hd", w / l, v)
        lse[s] = m[:, 0] + np.log(l[:, 0])
    return o, lse


def decode_fp8(q, k8, v8, k_scale, v_scale, seqlens, scale: float, page_table=None,
               page_size: int = 16):
    """Decode over an FP8 (E4M3) cache with per-head scales: key t of head h is
    ``k_scale[h] * e4m3_value(k8[.., t, h, :])`` (likewise for values), then
    :func:`decode_values`, one sequence at a time (only its cached rows are
    dequantized).  The dequantization is exact in fp64."""
    q = _u16(q)
    S = q.shape[0]
    H, d = q.shape[-2], q.shape[-1]
    q = q.reshape(S, H, d)
    ks = np.asarray(k_scale, np.float32).astype(np.float64)[:, None]
    vs = np.asarray(v_scale, np.float32).astype(np.float64)[:, None]
    o = np.zeros((S, H, d), np.float64)
    lse = np.full((S, H), -np.inf, np.float64)
    for s in range(S):
        L = int(seqlens[s])
        if L == 0:
            continue
        t = np.arange(L)
        if page_table is None:
            kb, vb = k8[s, :L], v8[s, :L]
        else:
            pages = np.asarray(page_table)[s, t // page_size]
            kb, vb = k8[pages, t % page_size], v8[pages, t % page_size]
        o1, l1 = decode_values(q[s:s + 1], (e4m3_value(kb) * ks)[None], (e4m3_value(vb) * vs)[None],
                               [L], scale)
        o[s], lse[s] = o1[0], l1[0]
    return o, lse


def _visible(causal: bool, i, Nq: int, Nk: int):
    """Keys visible to query rows i: all Nk, or (causal) j <= i + (Nk - Nq), clipped to [0, Nk]."""
    i = np.asarray(i, dtype=np.int64)
    if not causal:
        return np.full(i.shape, Nk, np.int64)
    return np.clip(i + (Nk - Nq) + 1, 0, Nk)


def _rows_of_one_head(qrows, kh, vh, n_vis, scale: float):
    """The definition for some query rows of one (b, h): qrows [R, d], kh, vh [Nk, d] (fp64),
    n_vis [R] visible keys per row.  Score row s_j = scale * q . k_j, m = max, l = sum
    exp(s_j - m), P = exp(s - m) / l, o = P V, LSE = m + ln l (a row with no visible key gets
    O = 0, LSE = -inf, m = -inf).  Returns o [R, d], lse [R], m [R]."""
    s = scale * (qrows @ kh.T)                                     # materialised score rows
    visible = np.arange(kh.shape[0])[None, :] < n_vis[:, None]
    s = np.where(visible, s, -np.inf)
    m = s.max(axis=1, initial=-np.inf)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(s - m_safe[:, None])                                # pass 1: exponentials, sum
    l = e.sum(axis=1)
    p = e / np.where(empty, 1.0, l)[:, None]                       # pass 2: P, then P V
    o = p @ vh
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, m_safe + np.log(l))
    return o, lse, m


def attn_fwd_values(q, k, v, causal: bool, scale: float, return_max: bool = False,
                    rows_per_block: int = 1024):
    """:func:`attn_fwd` for real-valued (fp64) inputs instead of bf16 bits.

    q [B, Nq, H, d]; k, v [B, Nk, H, d].  The same definition ("FlashAttention complete
    summary", section "Attention이 뭔가"; holysheep, section "Online Softmax 알고리즘"):
    per query row the scaled score row is materialised, m = max, l = sum exp(s - m),
    O = sum_j exp(s_j - m) / l * v_j, LSE = m + ln l; causal keeps j <= i + (Nk - Nq).
    Rows are independent, so they are evaluated ``rows_per_block`` at a time (numpy
    matrix products on each block of score rows) to bound memory.  Returns O, LSE and,
    with ``return_max``, the row maxima m [B, H, Nq] of the scaled scores.
    """
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    B, Nq, H, d = q.shape
    Nk = k.shape[1]
    if k.shape != (B, Nk, H, d) or v.shape != k.shape:
        raise ValueError("shape mismatch")
    o = np.empty((B, Nq, H, d), np.float64)
    lse = np.empty((B, H, Nq), np.float64)
    mx = np.empty((B, H, Nq), np.float64)
    for b in range(B):
        for h in range(H):
            kh, vh = k[b, :, h, :], v[b, :, h, :]
            for i0 in range(0, Nq, rows_per_block):
                i = np.arange(i0, min(Nq, i0 + rows_per_block))
                ob, lb, mb = _rows_of_one_head(q[b, i, h, :], kh, vh, _visible(causal, i, Nq, Nk),
                                               scale)
                o[b, i, h, :] = ob
                lse[b, h, i] = lb
                mx[b, h, i] = mb
    return (o, lse, mx) if return_max else (o, lse)


def attn_rows_values(q, k, v, causal: bool, scale: float, rows, return_max: bool = False):
    """:func:`attn_fwd_values` for selected rows only: rows int [R, 3] of (b, h, i).
    Returns O rows [R, d], LSE [R] and, with ``return_max``, m [R]."""
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    B, Nq, H, d = q.shape
    Nk = k.shape[1]
    rows = np.asarray(rows, dtype=np.int64).reshape(-1, 3)
    o = np.empty((rows.shape[0], d), np.float64)
    lse = np.empty((rows.shape[0],), np.float64)
    mx = np.empty((rows.shape[0],), np.float64)
    heads = rows[:, 0] * H + rows[:, 1]
    for bh in np.unique(heads):
        sel = np.nonzero(heads == bh)[0]
        b, h = int(bh // H), int(bh % H)
        i = rows[sel, 2]
        ob, lb, mb = _rows_of_one_head(q[b, i, h, :], k[b, :, h, :], v[b, :, h, :],
                                       _visible(causal, i, Nq, Nk), scale)
        o[sel], lse[sel], mx[sel] = ob, lb, mb
    return (o, lse, mx) if return_max else (o, lse)


def dequantize_e4m3(bits, scale_per_head):
    """FP8 E4M3 bits [..., H, d] with one fp32 scale per head [H] -> exact fp64 values
    ``scale[h] * e4m3_value(bits)``."""
    s = np.asarray(scale_per_head, np.float32).astype(np.float64)
    return e4m3_value(bits) * s[:, None]


def attn_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal: bool, scale: float, rows=None,
                 return_max: bool = False):
    """Attention over FP8 (E4M3) Q, K, V with one fp32 scale per head each (FP8 forward,
    "FlashAttention complete summary", section "FlashAttention 3"; "Beyond the memory
    wall", section "FlashAttention-3가 다른 이유": FP8 support).

    q8, k8, v8: E4M3 bits [B, N, H, d] (V in the same token-major layout as Q and K).
    The inputs are the dequantized values ``scale[h] * e4m3`` (exact in fp64); the
    attention is :func:`attn_fwd_values` of them, or :func:`attn_rows_values` for
    ``rows`` [R, 3] of (b, h, i).
    """
    qv = dequantize_e4m3(q8, q_scale)
    kv = dequantize_e4m3(k8, k_scale)
    vv = dequantize_e4m3(v8, v_scale)
    if rows is None:
        return attn_fwd_values(qv, kv, vv, causal, scale, return_max=return_max)
    return attn_rows_values(qv, kv, vv, causal, scale, rows, return_max=return_max)


def attn_bwd_head(q, k, v, do, causal: bool, scale: float):
    """Gradients of one (b, h) of the attention definition, fp64, given the upstream gradient
    dO of the output.  q, do [Nq, d]; k, v [Nk, d] (real values); causal keeps j <= i + (Nk - Nq).

    Forward, as in :func:`attn_fwd_values`: S = scale * Q K^T on the visible keys, P = the
    row-wise safe softmax of S (m = max, exp(S - m) / sum), O = P V.  Backward, the chain rule
    of L = sum(O * dO) through it (the recomputation of S and P from Q, K is what the tiled
    method does instead of storing P; "Beyond the memory wall", section "FlashAttention: IO
    인식의 정점": tiling and recomputation):
        dV = P^T dO;   dP = dO V^T;   D_i = sum_j P_ij dP_ij;   dS = P * (dP - D);
        dQ = scale * dS K;   dK = scale * dS^T Q.
    Returns dict with dq, dk, dv and the intermediates p, dp, D, ds, o, lse (rows with no
    visible key get P = 0 and LSE = -inf).
    """
    q, k, v, do = (np.asarray(x, np.float64) for x in (q, k, v, do))
    Nq, Nk = q.shape[0], k.shape[0]
    s = scale * (q @ k.T)
    visible = np.arange(Nk)[None, :] < _visible(causal, np.arange(Nq), Nq, Nk)[:, None]
    s = np.where(visible, s, -np.inf)
    m = s.max(axis=1, initial=-np.inf)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(s - m_safe[:, None])
    l = e.sum(axis=1)
    p = e / np.where(empty, 1.0, l)[:, None]
    o = p @ v
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, m_safe + np.log(l))
    dv = p.T @ do
    dp = do @ v.T
    D = (p * dp).sum(axis=1)
    ds = p * (dp - D[:, None])
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dict(dq=dq, dk=dk, dv=dv, p=p, dp=dp, D=D, ds=ds, o=o, lse=lse)


def attn_bwd(q, k, v, do, causal: bool, scale: float, heads=None):
    """dQ, dK, dV [B, N, H, d] (fp64) of the attention definition for bf16-bit inputs
    q, k, v, do [B, N, H, d] (square: Nq = Nk = N), one (b, h) at a time through
    :func:`attn_bwd_head`.  With ``heads`` (a list of (b, h)) only those heads are computed
    and the others are left as NaN."""
    q, k, v, do = (_u16(x) for x in (q, k, v, do))
    B, N, H, d = q.shape
    f = lambda x: (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    out = [np.full((B, N, H, d), np.nan) for _ in range(3)]
    todo = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    for b, h in todo:
        g = attn_bwd_head(f(q[b, :, h]), f(k[b, :, h]), f(v[b, :, h]), f(do[b, :, h]), causal, scale)
        out[0][b, :, h], out[1][b, :, h], out[2][b, :, h] = g["dq"], g["dk"], g["dv"]
    return out[0], out[1], out[2]
