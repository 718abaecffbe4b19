"""Error bounds for the backward kernels against the fp64 oracle, derived from the arithmetic.

The oracle (``oracle.attn_bwd_head``) computes the exact gradients of the attention
definition.  The GPU path recomputes P from the forward's fp32 log-sum-exp and differs from
the oracle only by rounding:

* P'_ij = exp(s_ij - LSE'_i) with LSE' the GPU forward's LSE: relative error
  rho_ij <= |LSE' - LSE|_i + (fp32 rounding of the exponent and ex2.approx, ~1e-6 (1 + |s| + |LSE|)).
* bf16 keeps 8 significant bits: rounding to it changes a value by at most 2^-8 of itself.
* dV = bf16(P')^T dO, fp32 accumulation: per term |err| <= (rho + 2^-8) P_ij |dO_ic|.
* dP_ij = dO_i . V_j in fp32 (products of bf16 numbers are exact; the sum rounds, <= 1e-5 |dO||V|).
* D_i = dO_i . O'_i with O' the GPU forward's bf16 output: |D' - D|_i <= sum_c |dO_ic| |O' - O|_ic.
* dS = bf16(P' (dP - D')): per element |err| <= A_ij = (rho P |dP - D| + P (|D' - D| + 1e-5 |dO||V|))
  (1 + 2^-8) + 2^-8 |dS_ij|.
* dQ = scale dS K and dK = scale dS^T Q, fp32 accumulation of bf16 products, then every
  output is rounded to bf16 (relative 2^-8).

Summing the per-term bounds gives the element-wise worst case (`max` check).  Rounding errors
that are uniform within their bounds and independent have RMS sqrt(sum t^2 / 3), which the
mean error must respect (`mean` check, with the output rounding's 2^-8/sqrt(3) |ref| added).
"""

from __future__ import annotations

import numpy as np

import oracle

R = 2.0 ** -8   # bf16 unit roundoff


def head_bounds(q, k, v, do, causal: bool, scale: float, o_gpu, lse_gpu):
    """Oracle gradients and bounds for one head.  q, k, v, do [N, d] fp64 values; o_gpu
    [N, d], lse_gpu [N] the GPU forward's output and LSE of the same head.  Returns dict name ->
    (ref, max_bound, rms_bound) for dq, dk, dv."""
    r = oracle.attn_bwd_head(q, k, v, do, causal, scale)
    P, dP, D, dS = r["p"], r["dp"], r["D"], r["ds"]
    lse = r["lse"]
    s = np.abs(scale * (q @ k.T))
    eps_l = np.abs(lse_gpu - lse)
    rho = 1.01 * (eps_l[:, None] + 1e-6 * (1.0 + s + np.abs(lse)[:, None]))
    ado, av, ak, aq = np.abs(do), np.abs(v), np.abs(k), np.abs(q)
    # dV: terms (rho + 2^-8) P_ij |dO_ic| over i
    w = (rho + R) * P
    dv_max = w.T @ ado + 1e-5 * (P.T @ ado)
    dv_rms = np.sqrt((w * w).T @ (do * do) / 3.0)
    # dS
    eps_d = (ado * np.abs(o_gpu - r["o"])).sum(axis=1) + 1e-6 * (ado * np.abs(r["o"])).sum(axis=1)
    dp_err = 1e-5 * (ado @ av.T)
    A = (rho * P * np.abs(dP - D[:, None]) + P * (eps_d[:, None] + dp_err)) * (1.0 + R) + R * np.abs(dS)
    dq_max = scale * (A @ ak) + 1e-5 * scale * (np.abs(dS) @ ak)
    dq_rms = scale * np.sqrt((A * A) @ (k * k) / 3.0)
    dk_max = scale * (A.T @ aq) + 1e-5 * scale * (np.abs(dS).T @ aq)
    dk_rms = scale * np.sqrt((A * A).T @ (q * q) / 3.0)
    out = {}
    for name, mx, rms in (("dq", dq_max, dq_rms), ("dk", dk_max, dk_rms), ("dv", dv_max, dv_rms)):
        ref = r[name]
        out[name] = (ref, mx + R * np.abs(ref) + 1e-7, rms + R / np.sqrt(3.0) * np.abs(ref) + 1e-8)
    return out


def check_head(grads_gpu, bounds, what=""):
    """grads_gpu: dict name -> [N, d] fp64 of one head.  Every element within its max bound and
    the mean error within the mean RMS bound, for dq, dk and dv."""
    for name in ("dq", "dk", "dv"):
        ref, mx, rms = bounds[name]
        got = grads_gpu[name]
        assert np.all(np.isfinite(got)), f"{what} {name} not finite"
        err = np.abs(got - ref)
        worst = np.max(err - mx)
        assert worst <= 0.0, f"{what} {name} exceeds its element bound by {worst:.3e}"
        assert err.mean() <= rms.mean(), f"{what} {name} mean-abs {err.mean():.3e} > {rms.mean():.3e}"
