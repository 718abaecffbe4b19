"""Bounded device waits: a pipeline wait that runs out gives up, records
ATTN_ERR_TIMEOUT in the device status word and winds down, and the context
stays usable for the next call.

The failure is made without a fault: ATTN_TEST_DROP_LOAD=1 (read by the
library at every call) makes the kernel's producer leave one load unissued, so
the wait for it can only run out, here after ATTN_WAIT_TIMEOUT_MS=20.  The
kernels' wind-down waits for the copies and MMAs already issued before tensor
memory is released, so nothing faults and nothing hangs; an ordinary call
afterwards must be correct.  Tiny problems only.
"""

import math

import numpy as np
import pytest

import oracle
from io_aware_attention_03_b300.inputs import chunk_queries, decode_inputs, prefill_inputs

pytestmark = pytest.mark.gpu

ATTN_ERR_TIMEOUT = 6
O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from io_aware_attention_03_b300 import attn, device_inputs

    return torch, attn, device_inputs


def drop_one_load(monkeypatch):
    monkeypatch.setenv("ATTN_WAIT_TIMEOUT_MS", "20")
    monkeypatch.setenv("ATTN_TEST_DROP_LOAD", "1")


def restore(monkeypatch):
    monkeypatch.delenv("ATTN_TEST_DROP_LOAD")
    monkeypatch.delenv("ATTN_WAIT_TIMEOUT_MS")


@pytest.mark.parametrize("d", [64, 128])
def test_forward_wait_runs_out_then_context_is_usable(dev, monkeypatch, d):
    torch, attn, dvi = dev
    q, k, v = prefill_inputs(11, 1, 2, 256, d)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    tq, tk, tv = (dvi.to_device_bf16(x) for x in (q, k, v))
    assert attn.attn_last_device_status() == 0

    drop_one_load(monkeypatch)
    attn.attn_fwd(tq, tk, tv, causal=True, scale=scale)
    assert attn.attn_last_device_status() == ATTN_ERR_TIMEOUT
    restore(monkeypatch)

    o, lse = attn.attn_fwd(tq, tk, tv, causal=True, scale=scale)
    assert attn.attn_last_device_status() == 0
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, scale)
    err = np.abs(dvi.to_host_f64(o) - o_ref)
    assert err.max() <= O_MAX and err.mean() <= O_MEAN
    assert np.abs(dvi.to_host_f64(lse) - lse_ref).max() <= LSE_MAX


def test_backward_wait_runs_out_then_context_is_usable(dev, monkeypatch):
    torch, attn, dvi = dev
    q, k, v = prefill_inputs(12, 1, 2, 256, 128)
    scale = float(np.float32(1.0 / math.sqrt(128)))
    tq, tk, tv = (dvi.to_device_bf16(x) for x in (q, k, v))
    o, lse = attn.attn_fwd(tq, tk, tv, causal=False, scale=scale)
    do = torch.randn(tq.shape, device=tq.device, dtype=torch.float32).to(torch.bfloat16)
    ref = attn.attn_bwd(tq, tk, tv, o, lse, do, causal=False, scale=scale)
    assert attn.attn_last_device_status() == 0

    drop_one_load(monkeypatch)
    attn.attn_bwd(tq, tk, tv, o, lse, do, causal=False, scale=scale)
    assert attn.attn_last_device_status() == ATTN_ERR_TIMEOUT
    restore(monkeypatch)

    again = attn.attn_bwd(tq, tk, tv, o, lse, do, causal=False, scale=scale)
    assert attn.attn_last_device_status() == 0
    for a, b in zip(ref, again):  # the backward is deterministic
        assert torch.equal(a, b)


def test_dynamic_deal_wait_runs_out_then_context_is_usable(dev, monkeypatch):
    """The paged prefill takes its units from a device counter and hands them to the MMA and
    softmax warps through a ring in shared memory; with a load dropped, every wait of that
    ring and of the pipeline must still give up and wind down.  Three sequences, H=2."""
    torch, attn, dvi = dev
    lens, Nq, H, d = (256, 300, 520), 128, 2, 128
    di = decode_inputs(13, len(lens), H, d, 0, 0, seqlens=lens)
    qc = chunk_queries(14, len(lens), Nq, H, d)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    _, kp, vp, seqlens, pt = dvi.decode_device_inputs(di, paged=True)
    q = dvi.to_device_bf16(qc)
    ref = attn.attn_prefill_paged(q, kp, vp, seqlens, pt, causal=True, scale=scale)
    assert attn.attn_last_device_status() == 0

    drop_one_load(monkeypatch)
    attn.attn_prefill_paged(q, kp, vp, seqlens, pt, causal=True, scale=scale)
    assert attn.attn_last_device_status() == ATTN_ERR_TIMEOUT
    restore(monkeypatch)

    again = attn.attn_prefill_paged(q, kp, vp, seqlens, pt, causal=True, scale=scale)
    assert attn.attn_last_device_status() == 0
    for a, b in zip(ref, again):  # the order of the units does not change the results
        assert torch.equal(a, b)
