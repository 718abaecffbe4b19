"""The derived FP8-prefill and backward tolerances have teeth: a numpy model of each kernel's
rounding steps stays inside them, and a model with a plausible mistake planted in it does not.

The models are test-side only (neither the oracle nor the CUDA path): they replay, in float32
with the kernels' roundings, what tests/fp8_tolerance.py and tests/bwd_tolerance.py assume:
* FP8 prefill: scores of the dequantized E4M3 inputs; per 128-key block a running maximum that
  moves only when the block maximum exceeds it by more than 8 (log2 units) and is then set 4
  below it; P = 2^(s - m) rounded to E4M3 (nearest even); l summed from the unrounded P; O
  rounded to bf16.
* backward: P from the fp32 log-sum-exp, rounded to bf16 for dV; D from the bf16 forward
  output; dS = P (dP - D) rounded to bf16; every gradient rounded to bf16.
"""

import math

import numpy as np
import pytest

import bwd_tolerance
import fp8_tolerance
import oracle
from io_aware_attention_03_b300.inputs import (backward_inputs, bf16_bits, bf16_to_f32, e4m3_bits,
                                               fp8_prefill_inputs)

LOG2E = 1.4426950408889634


def bf(x):
    return bf16_to_f32(bf16_bits(np.asarray(x, np.float32))).astype(np.float64)


def fp8_model(f8, causal, scale, shift_keys=False):
    """O [B, N, H, d], LSE [B, H, N] of the FP8 kernel's arithmetic (see module docstring)."""
    q = oracle.dequantize_e4m3(f8.q, f8.q_scale)
    k = oracle.dequantize_e4m3(f8.k, f8.k_scale)
    v = oracle.dequantize_e4m3(f8.v, f8.v_scale)
    B, N, H, d = q.shape
    sl2 = np.float32(scale * LOG2E)
    O = np.zeros((B, N, H, d))
    L = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            s_all = (q[b, :, h] @ k[b, :, h].T).astype(np.float32) * sl2     # [N, N], log2 units
            vis = (np.arange(N)[None, :] <= np.arange(N)[:, None]) if causal else np.ones((N, N), bool)
            s_all = np.where(vis, s_all, -np.inf)
            m = np.full(N, -np.inf)
            l = np.zeros(N)
            acc = np.zeros((N, d))
            for j0 in range(0, N, 128):
                s = s_all[:, j0:j0 + 128].astype(np.float64)
                cand = s.max(axis=1)
                m_new = np.where(cand > m + 8, cand - 4, m)
                with np.errstate(invalid="ignore"):
                    alpha = np.where(np.isfinite(m), np.exp2(m - m_new), 0.0)
                p = np.exp2(s - m_new[:, None])
                p8 = oracle.e4m3_value(e4m3_bits(p.astype(np.float32)))
                vv = v[b, j0:j0 + s.shape[1], h]
                if shift_keys:
                    vv = np.roll(vv, 1, axis=0)
                l = l * alpha + p.sum(axis=1)
                acc = acc * alpha[:, None] + p8 @ vv
                m = m_new
            O[b, :, h] = bf(acc / l[:, None])
            L[b, h] = (m + np.log2(l)) * math.log(2)
    return O, L


@pytest.mark.parametrize("case", [(False, 1.0), (True, 1.0), (True, 4.0)], ids=["full", "causal", "peaky"])
def test_fp8_tolerance_accepts_the_kernel_arithmetic(case):
    causal, qf = case
    f8 = fp8_prefill_inputs(5, 1, 2, 300, 128, q_factor=qf)
    scale = float(np.float32(1 / math.sqrt(128)))
    o_m, l_m = fp8_model(f8, causal, scale)
    o, lse, bound, sigma = fp8_tolerance.oracle_and_bounds(f8, causal, scale)
    b, h, i = (x.ravel() for x in np.meshgrid(np.arange(1), np.arange(2), np.arange(300), indexing="ij"))
    fp8_tolerance.check(o_m[b, i, h], l_m[b, h, i], o, lse, bound, sigma, "model")


def test_fp8_tolerance_rejects_a_shifted_key():
    f8 = fp8_prefill_inputs(5, 1, 2, 300, 128)
    scale = float(np.float32(1 / math.sqrt(128)))
    o_m, l_m = fp8_model(f8, True, scale, shift_keys=True)
    o, lse, bound, sigma = fp8_tolerance.oracle_and_bounds(f8, True, scale)
    b, h, i = (x.ravel() for x in np.meshgrid(np.arange(1), np.arange(2), np.arange(300), indexing="ij"))
    with pytest.raises(AssertionError):
        fp8_tolerance.check(o_m[b, i, h], l_m[b, h, i], o, lse, bound, sigma, "shifted")


def bwd_model(q, k, v, do, causal, scale, o_gpu, lse_gpu, mistake=None):
    """dQ, dK, dV of one head with the backward kernels' roundings (see module docstring)."""
    N = q.shape[0]
    sl2 = np.float32(scale * LOG2E)
    s = (q @ k.T).astype(np.float32)
    lse2 = lse_gpu.astype(np.float32) * np.float32(LOG2E)
    p = np.exp2((s * sl2 - lse2[:, None]).astype(np.float32)).astype(np.float64)
    if causal:
        off = 1 if mistake == "mask" else 0
        p = np.where(np.arange(N)[None, :] <= np.arange(N)[:, None] + off, p, 0.0)
    dp = (do @ v.T).astype(np.float32).astype(np.float64)
    D = (do * o_gpu).sum(axis=1).astype(np.float32).astype(np.float64)
    if mistake == "D":
        D = -D
    ds = bf(p * (dp - D[:, None]))
    return dict(dq=bf(scale * (ds @ k)), dk=bf(scale * (ds.T @ q)), dv=bf(bf(p).T @ do))


def _bwd_case(causal, qf=1.0):
    q, k, v, do = backward_inputs(7, 1, 1, 300, 128, q_factor=qf)
    f = lambda x: bf16_to_f32(x[0, :, 0]).astype(np.float64)
    qh, kh, vh, doh = f(q), f(k), f(v), f(do)
    scale = float(np.float32(1 / math.sqrt(128)))
    fw = oracle.attn_bwd_head(qh, kh, vh, doh, causal, scale)
    o_gpu, lse_gpu = bf(fw["o"]), fw["lse"].astype(np.float32).astype(np.float64)
    bounds = bwd_tolerance.head_bounds(qh, kh, vh, doh, causal, scale, o_gpu, lse_gpu)
    return (qh, kh, vh, doh, scale, o_gpu, lse_gpu), bounds


@pytest.mark.parametrize("case", [(False, 1.0), (True, 1.0), (True, 4.0)], ids=["full", "causal", "peaky"])
def test_backward_tolerance_accepts_the_kernel_arithmetic(case):
    causal, qf = case
    (qh, kh, vh, doh, scale, o_gpu, lse_gpu), bounds = _bwd_case(causal, qf)
    bwd_tolerance.check_head(bwd_model(qh, kh, vh, doh, causal, scale, o_gpu, lse_gpu), bounds, "model")


@pytest.mark.parametrize("mistake,causal", [("mask", True), ("D", False)])
def test_backward_tolerance_rejects_planted_mistakes(mistake, causal):
    (qh, kh, vh, doh, scale, o_gpu, lse_gpu), bounds = _bwd_case(causal)
    grads = bwd_model(qh, kh, vh, doh, causal, scale, o_gpu, lse_gpu, mistake=mistake)
    with pytest.raises(AssertionError):
        bwd_tolerance.check_head(grads, bounds, mistake)
