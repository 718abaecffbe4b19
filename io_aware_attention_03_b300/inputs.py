"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module draws numbers and lays them out; it holds none of the attention
arithmetic.  Both the CUDA path and the CPU oracle receive exactly the arrays
built here.

Recipe (the workloads are bf16 Q/K/V drawn from N(0, 1) from a seed):
* one ``numpy.random.Generator(PCG64(seed))`` per workload;
* ``standard_normal(dtype=float32)`` draws, optionally multiplied by a
  power-of-two factor (exact in bf16; the "peaky softmax" variant scales Q by 4);
* fp32 -> bf16 by round-to-nearest-even on the bit pattern (``bf16_bits``);
* prefill: Q, then K, then V, each ``[B, N, H, d]``, drawn in that order;
* decode: sequence lengths first (``integers(lo, hi, endpoint=True)``), then Q
  ``[S, H, d]``, then K for every sequence in order (``[L_s, H, d]`` each), then
  V likewise, then ``permutation(num_pages)`` for the page ids.
"""

from __future__ import annotations

import dataclasses

import numpy as np


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 round-to-nearest-even, returned as raw ``uint16`` bits.

    Finite inputs only (normal draws never produce inf/NaN).
    """
    x = np.asarray(x, dtype=np.float32)
    u = np.ascontiguousarray(x.reshape(-1)).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16).reshape(x.shape)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact bf16 -> fp32 widening of raw ``uint16`` bits."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(g: np.random.Generator, shape, factor: float = 1.0) -> np.ndarray:
    x = g.standard_normal(size=shape, dtype=np.float32)
    if factor != 1.0:
        x *= np.float32(factor)
    return bf16_bits(x)


def prefill_inputs(seed: int, B: int, H: int, N: int, d: int, q_factor: float = 1.0):
    """(q, k, v) bf16 bits, each ``[B, N, H, d]``, drawn Q then K then V."""
    g = np.random.Generator(np.random.PCG64(seed))
    q = _normal_bf16(g, (B, N, H, d), q_factor)
    k = _normal_bf16(g, (B, N, H, d))
    v = _normal_bf16(g, (B, N, H, d))
    return q, k, v


def sample_rows(seed: int, B: int, H: int, N: int, count: int, include_edges: bool = True):
    """Distinct (b, h, i) query rows, ``int64 [R, 3]``, for checks on large problems.

    Drawn with its own generator (seed) so that the input draw is untouched.
    With ``include_edges`` the first and last row of every 128-row tile boundary
    near the start and end of the sequence are added for batch 0, head 0.
    """
    g = np.random.Generator(np.random.PCG64(seed))
    total = B * H * N
    count = min(count, total)
    flat = g.choice(total, size=count, replace=False)
    b = flat // (H * N)
    h = (flat // N) % H
    i = flat % N
    rows = np.stack([b, h, i], axis=1).astype(np.int64)
    if include_edges:
        edge_i = sorted({x for x in (0, 1, 126, 127, 128, 129, 255, 256, N - 129, N - 128, N - 2, N - 1)
                         if 0 <= x < N})
        edges = np.array([[B - 1, H - 1, x] for x in edge_i] + [[0, 0, x] for x in edge_i], np.int64)
        rows = np.unique(np.concatenate([rows, edges]), axis=0)
    return rows


@dataclasses.dataclass
class DecodeInputs:
    """One decode batch.  All arrays are host numpy arrays.

    q:          bf16 bits [S, H, d]
    k_tokens:   bf16 bits [sum(L), H, d]  (sequence s occupies rows offsets[s]:offsets[s+1])
    v_tokens:   bf16 bits [sum(L), H, d]
    seqlens:    int32 [S]
    offsets:    int64 [S + 1]
    page_ids:   int32 [num_pages]  (page ids in the order pages are assigned)
    page_size:  tokens per page
    """

    q: np.ndarray
    k_tokens: np.ndarray
    v_tokens: np.ndarray
    seqlens: np.ndarray
    offsets: np.ndarray
    page_ids: np.ndarray
    page_size: int

    @property
    def num_seqs(self) -> int:
        return int(self.seqlens.shape[0])

    @property
    def max_seqlen(self) -> int:
        return int(self.seqlens.max()) if self.seqlens.size else 0

    def pages_per_seq(self) -> np.ndarray:
        return (self.seqlens.astype(np.int64) + self.page_size - 1) // self.page_size

    def page_table(self, max_pages_per_seq: int | None = None) -> np.ndarray:
        """int32 [S, max_pages_per_seq]: page ids assigned to sequences in order; unused slots -1."""
        per = self.pages_per_seq()
        width = int(per.max()) if max_pages_per_seq is None else int(max_pages_per_seq)
        pt = np.full((self.num_seqs, max(width, 1)), -1, np.int32)
        pos = 0
        for s, n in enumerate(per):
            pt[s, :n] = self.page_ids[pos:pos + n]
            pos += n
        return pt

    def contiguous_cache(self, tokens: np.ndarray, max_seqlen: int | None = None) -> np.ndarray:
        """[S, max_seqlen, H, d] with sequence s in rows [0, L_s); the rest zero."""
        L = self.max_seqlen if max_seqlen is None else int(max_seqlen)
        out = np.zeros((self.num_seqs, L) + tokens.shape[1:], tokens.dtype)
        for s in range(self.num_seqs):
            a, b = self.offsets[s], self.offsets[s + 1]
            out[s, :b - a] = tokens[a:b]
        return out

    def paged_pool(self, tokens: np.ndarray) -> np.ndarray:
        """[num_pages, page_size, H, d]; the tail slots of each last page are zero."""
        num_pages = int(self.page_ids.shape[0])
        pool = np.zeros((num_pages, self.page_size) + tokens.shape[1:], tokens.dtype)
        pt = self.page_table()
        for s in range(self.num_seqs):
            a, b = int(self.offsets[s]), int(self.offsets[s + 1])
            for p in range(int(self.pages_per_seq()[s])):
                t0 = p * self.page_size
                t1 = min(t0 + self.page_size, b - a)
                pool[pt[s, p], :t1 - t0] = tokens[a + t0:a + t1]
        return pool


def decode_inputs(seed: int, num_seqs: int, H: int, d: int, len_lo: int, len_hi: int,
                  page_size: int = 16, seqlens=None) -> DecodeInputs:
    """A decode batch: lengths ~ U[len_lo, len_hi] (inclusive) unless ``seqlens`` is given."""
    g = np.random.Generator(np.random.PCG64(seed))
    if seqlens is None:
        lens = g.integers(len_lo, len_hi, endpoint=True, size=num_seqs).astype(np.int32)
    else:
        lens = np.asarray(seqlens, dtype=np.int32).copy()
    offsets = np.zeros(num_seqs + 1, np.int64)
    offsets[1:] = np.cumsum(lens.astype(np.int64))
    q = _normal_bf16(g, (num_seqs, H, d))
    total = int(offsets[-1])
    k = np.empty((total, H, d), np.uint16)
    v = np.empty((total, H, d), np.uint16)
    for s in range(num_seqs):
        k[offsets[s]:offsets[s + 1]] = _normal_bf16(g, (int(lens[s]), H, d))
    for s in range(num_seqs):
        v[offsets[s]:offsets[s + 1]] = _normal_bf16(g, (int(lens[s]), H, d))
    pages = int(((lens.astype(np.int64) + page_size - 1) // page_size).sum())
    page_ids = g.permutation(pages).astype(np.int32)
    return DecodeInputs(q, k, v, lens, offsets, page_ids, page_size)


def e4m3_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
    infinities) by round-to-nearest-even, saturating at +-448; raw ``uint8`` bits.

    From 2^-6 up the rounding keeps 3 of fp32's 23 mantissa bits (add half an
    E4M3 quantum, plus one when the kept last bit is odd, then truncate; a carry
    moves into the exponent as it should); below 2^-6 the quantum is 2^-9
    (subnormals), rounded half to even with ``rint``.  Finite inputs only.
    """
    x = np.asarray(x, dtype=np.float32)
    sign = np.signbit(x)
    a = np.minimum(np.abs(x), np.float32(448.0))
    u = a.view(np.uint32)
    r = (u + np.uint32(0x7FFFF) + ((u >> np.uint32(20)) & np.uint32(1))) & np.uint32(0xFFF00000)
    exp_field = (r >> np.uint32(23)).astype(np.int64) - 127 + 7
    normal = ((exp_field << 3) | ((r >> np.uint32(20)) & np.uint32(7)).astype(np.int64))
    sub = np.rint(a * np.float32(512.0)).astype(np.int64)      # multiples of 2^-9
    bits = np.where(a >= np.float32(2.0 ** -6), normal, sub)
    bits = np.where(sign, bits | 0x80, bits)
    return bits.astype(np.uint8)


@dataclasses.dataclass
class Fp8Cache:
    """FP8 (E4M3) copies of a decode batch's K and V tokens with one fp32 scale per head:
    token value = scale[h] * e4m3(bits)."""

    k_tokens: np.ndarray   # uint8 [sum(L), H, d]
    v_tokens: np.ndarray
    k_scale: np.ndarray    # float32 [H]
    v_scale: np.ndarray


def e4m3_per_head(tokens: np.ndarray, pow2_scales: bool = True):
    """Quantize bf16 bits ``[..., H, d]`` to E4M3 with one fp32 scale per head.

    The scale of head h makes its largest |value| land at or below 448 (the largest
    E4M3 number): amax / 448, rounded up to a power of two when ``pow2_scales``.
    With a power-of-two scale, value / scale is exact in bf16, so every head is
    quantized through a 65536-entry table over bf16 bit patterns (fast for
    multi-GB tensors); otherwise each value is divided in fp32 and encoded.
    Returns (bits uint8 like ``tokens``, scale float32 [H]); value = scale[h] * e4m3.
    """
    H = tokens.shape[-2]
    if tokens.size:
        amax_bits = (tokens & np.uint16(0x7FFF)).reshape(-1, H, tokens.shape[-1]).max(axis=(0, 2))
        amax = bf16_to_f32(amax_bits)   # finite bf16: the bit order is the magnitude order
    else:
        amax = np.ones(H, np.float32)
    scale = np.maximum(amax, np.float32(1e-30)) / np.float32(448.0)
    if pow2_scales:
        scale = np.exp2(np.ceil(np.log2(scale.astype(np.float64)))).astype(np.float32)
        bits = np.empty(tokens.shape, np.uint8)
        every_bf16 = bf16_to_f32(np.arange(65536, dtype=np.uint32).astype(np.uint16))
        finite = np.isfinite(every_bf16)
        for h in range(H):
            table = np.zeros(65536, np.uint8)
            with np.errstate(over="ignore"):   # entries beyond 448 saturate
                table[finite] = e4m3_bits(every_bf16[finite] / scale[h])
            bits[..., h, :] = table[tokens[..., h, :]]
    else:
        scale = scale.astype(np.float32)
        bits = e4m3_bits(bf16_to_f32(tokens) / scale[:, None])
    return bits, scale.astype(np.float32)


def fp8_cache(di: DecodeInputs, pow2_scales: bool = True) -> Fp8Cache:
    """Quantize a decode batch's bf16 K and V tokens to E4M3 with per-head scales
    (:func:`e4m3_per_head`)."""
    kb, ks = e4m3_per_head(di.k_tokens, pow2_scales)
    vb, vs = e4m3_per_head(di.v_tokens, pow2_scales)
    return Fp8Cache(kb, vb, ks, vs)


@dataclasses.dataclass
class Fp8Prefill:
    """FP8 (E4M3) prefill inputs: Q, K, V bits ``[B, N, H, d]`` (token-major, like the
    bf16 inputs) and one fp32 scale per head for each; value = scale[h] * e4m3(bits)."""

    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    q_scale: np.ndarray
    k_scale: np.ndarray
    v_scale: np.ndarray


def fp8_prefill_inputs(seed: int, B: int, H: int, N: int, d: int, q_factor: float = 1.0,
                       pow2_scales: bool = True) -> Fp8Prefill:
    """The bf16 prefill draw of :func:`prefill_inputs` (Q, then K, then V, N(0, 1)),
    each quantized to E4M3 per head by :func:`e4m3_per_head`."""
    q, k, v = prefill_inputs(seed, B, H, N, d, q_factor)
    (q8, qs), (k8, ks), (v8, vs) = (e4m3_per_head(x, pow2_scales) for x in (q, k, v))
    return Fp8Prefill(q8, k8, v8, qs, ks, vs)


def chunk_queries(seed: int, num_seqs: int, Nq: int, H: int, d: int) -> np.ndarray:
    """Queries of a prefill chunk: bf16 bits ``[num_seqs, Nq, H, d]``, N(0, 1), from
    their own generator (the cache of the same sequences comes from ``decode_inputs``)."""
    g = np.random.Generator(np.random.PCG64(seed))
    return _normal_bf16(g, (num_seqs, Nq, H, d))


# The workloads, by what they are.  Seeds: tiny 1, prefill 2, sweep 100+i, chunked 400 and 401,
# long context 200+i, decode 300.
TINY = dict(seed=1, B=1, H=2, N=128, d=64)
PREFILL = dict(seed=2, B=4, H=16, N=2048, d=128, causal=True)
SWEEP_TOKENS = 16384
SWEEP_N = (512, 1024, 2048, 4096, 8192, 16384)
SWEEP_SHAPES = ((16, 128), (32, 64))
LONG = (dict(seed=200, B=1, H=32, N=32768, d=128, causal=True),
        dict(seed=201, B=1, H=32, N=131072, d=128, causal=True))
DECODE = dict(seed=300, num_seqs=64, H=32, d=128, len_lo=512, len_hi=8192, page_size=16)
# chunked prefill: a 512-token chunk per sequence against a cached prefix, the
# whole sequence (prefix + chunk) ~ U[1024, 8192] tokens in 16-token pages
CHUNKED = dict(seed=400, q_seed=401, num_seqs=16, Nq=512, H=32, d=128, len_lo=1024, len_hi=8192,
               page_size=16)


def sweep_configs():
    """The sequence-length sweep at B*N = 16384 tokens: list of dicts with a seed each."""
    out = []
    idx = 0
    for H, d in SWEEP_SHAPES:
        for N in SWEEP_N:
            for causal in (False, True):
                for q_factor in (1.0, 4.0):
                    out.append(dict(seed=100 + idx, B=SWEEP_TOKENS // N, H=H, N=N, d=d,
                                    causal=causal, q_factor=q_factor))
                    idx += 1
    return out


def backward_inputs(seed: int, B: int, H: int, N: int, d: int, q_factor: float = 1.0):
    """(q, k, v, do) bf16 bits, each ``[B, N, H, d]``, N(0, 1): the prefill draw of
    :func:`prefill_inputs` (Q, then K, then V) followed by the upstream gradient dO of the
    output from the same generator."""
    g = np.random.Generator(np.random.PCG64(seed))
    q = _normal_bf16(g, (B, N, H, d), q_factor)
    k = _normal_bf16(g, (B, N, H, d))
    v = _normal_bf16(g, (B, N, H, d))
    do = _normal_bf16(g, (B, N, H, d))
    return q, k, v, do
