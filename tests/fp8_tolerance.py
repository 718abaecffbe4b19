"""Error bounds for FP8 (E4M3) prefill against the fp64 oracle, derived from the arithmetic.

The oracle computes attention exactly on the dequantized inputs scale[h] * e4m3.  The
GPU path differs from it only by rounding:

* S = Q K^T: products of two E4M3 numbers are exact in fp32 and 128 of them are summed
  in fp32; the per-head scales fold into one fp32 factor.  Relative error ~1e-6.
* P is kept relative to a reference max mu that never exceeds the true row max m minus
  4 ln 2 (the kernel holds 2^4 of headroom) and that lags m by at most 2^8, so every
  P'_j = exp(s_j - mu) lies in [0, 2^8], inside the E4M3 range (448).  The row sum l'
  is accumulated in fp32 from the unrounded P', and O' = sum_j e4m3(P'_j) v_j / l'.
* E4M3 keeps 3 mantissa bits: for P'_j >= 2^-6 the rounding error is at most 2^-4 P'_j
  (half a unit in the last place); below 2^-6 (subnormals, quantum 2^-9) it is at most
  2^-10.  Since l' = exp(LSE - mu) >= 16 exp(LSE - m):

      |O' - O|_c <= 2^-4 * sum_j p_j |v_jc|  +  2^-14 * exp(m - LSE) * sum_j |v_jc|

  over the visible keys j, with p_j the exact softmax weights.  O' is then rounded to
  bf16 (8 significant bits: at most 2^-8 of the value).  This is the element-wise bound
  below.
* Rounding errors that are uniform within half a unit have RMS at most 1/sqrt(3) of
  their bound, so with independent errors per key the RMS of the output error is at
  most sigma_c = sqrt((2^-8/3) sum_j p_j^2 v_jc^2 + (2^-28/3) exp(2(m - LSE)) sum_j v_jc^2).
  The mean absolute error over many elements is then about sqrt(2/pi) sigma; the test
  asks for mean |err| <= mean sigma + the bf16 rounding's RMS, 2^-8/sqrt(3) |O|.
* LSE = ln l' + mu uses the unrounded P', so it keeps the bf16 path's 1e-3.

sum_j p_j |v_jc| is attention of |V|; sum_j p_j^2 v_jc^2 follows from attention at twice
the scale: p_j^2 = exp(2 s_j - 2 LSE) = p2_j exp(LSE2 - 2 LSE), where p2, LSE2 are the
softmax weights and log-sum-exp of the doubled scores, so the sum is
attn(2 scale; V^2)_c * exp(LSE2 - 2 LSE).
"""

from __future__ import annotations

import numpy as np

import oracle

LSE_MAX = 1e-3


def _visible_sums(vv, rows, causal):
    """sum_j |v_jc| and sum_j v_jc^2 over the keys visible to each row (b, h, i); vv fp64
    [B, N, H, d] (square problems: query i sees keys j <= i when causal)."""
    a1 = np.cumsum(np.abs(vv), axis=1)
    a2 = np.cumsum(vv * vv, axis=1)
    N = vv.shape[1]
    b, h, i = rows[:, 0], rows[:, 1], rows[:, 2]
    last = i if causal else np.full_like(i, N - 1)
    return a1[b, last, h, :], a2[b, last, h, :]


def oracle_and_bounds(f8, causal: bool, scale: float, rows=None):
    """Oracle O [R, d], LSE [R] for the rows (all rows when None) of an FP8 prefill problem,
    with the element-wise bound [R, d] and the RMS estimate sigma [R, d] described above.
    Rows are (b, h, i) triples; the returned arrays follow their order."""
    B, N, H, d = f8.q.shape
    if rows is None:
        b, h, i = np.meshgrid(np.arange(B), np.arange(H), np.arange(N), indexing="ij")
        rows = np.stack([b.ravel(), h.ravel(), i.ravel()], axis=1)
    rows = np.asarray(rows, np.int64)
    qv = oracle.dequantize_e4m3(f8.q, f8.q_scale)
    kv = oracle.dequantize_e4m3(f8.k, f8.k_scale)
    vv = oracle.dequantize_e4m3(f8.v, f8.v_scale)
    o, lse, m = oracle.attn_rows_values(qv, kv, vv, causal, scale, rows, return_max=True)
    a_abs, _ = oracle.attn_rows_values(qv, kv, np.abs(vv), causal, scale, rows)
    o2, lse2 = oracle.attn_rows_values(qv, kv, vv * vv, causal, scale * 2.0, rows)
    v1, v2 = _visible_sums(vv, rows, causal)
    inv_l = np.exp(m - lse)[:, None]                           # 1 / sum_j exp(s_j - m)
    p2v2 = o2 * np.exp(lse2 - 2.0 * lse)[:, None]              # sum_j p_j^2 v_jc^2
    bound = (2.0 ** -4 * a_abs + 2.0 ** -14 * inv_l * v1 + 2.0 ** -8 * np.abs(o)
             + 1e-4 * a_abs + 1e-6)
    sigma = np.sqrt(2.0 ** -8 / 3.0 * p2v2 + 2.0 ** -28 / 3.0 * inv_l ** 2 * v2)
    return o, lse, bound, sigma


def check(o_gpu, lse_gpu, o, lse, bound, sigma, what=""):
    """The FP8 tolerance: every element within `bound`, the mean error within the mean of
    sigma plus bf16 output rounding, LSE within 1e-3."""
    err = np.abs(o_gpu - o)
    assert np.all(np.isfinite(o_gpu)), what
    worst = np.max(err - bound)
    assert worst <= 0.0, f"{what} O exceeds its element bound by {worst:.3e}"
    mean_bound = sigma.mean() + 2.0 ** -8 / np.sqrt(3.0) * np.abs(o).mean() + 1e-6
    assert err.mean() <= mean_bound, f"{what} O mean-abs {err.mean():.3e} > {mean_bound:.3e}"
    lerr = np.abs(lse_gpu - lse)
    assert lerr.max() <= LSE_MAX, f"{what} LSE max-abs {lerr.max():.3e}"
