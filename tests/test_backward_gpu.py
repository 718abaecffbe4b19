"""Backward parity: attn_bwd (through the C ABI) against the fp64 oracle's gradients.

The forward runs on the GPU first (attn_fwd), and its bf16 output and fp32 LSE feed the
backward, as in training.  The oracle differentiates the attention definition exactly
("Beyond the memory wall", section "FlashAttention: IO 인식의 정점": tiling and
recomputation).  The tolerance is derived in tests/bwd_tolerance.py from the kernels'
rounding steps: every gradient element within its worst-case bound, and the mean error
within the RMS those roundings predict.  Whole heads are compared (all heads for small
problems, a seeded subset for the large ones).
"""

import math

import numpy as np
import pytest

import bwd_tolerance
from io_aware_attention_03_b300.inputs import PREFILL, backward_inputs, bf16_to_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from io_aware_attention_03_b300 import attn, device_inputs

    return torch, attn, device_inputs


def run_bwd(dev, q, k, v, do, causal, scale):
    torch, attn, dvi = dev
    tq, tk, tv, tdo = (dvi.to_device_bf16(x) for x in (q, k, v, do))
    o, lse = attn.attn_fwd(tq, tk, tv, causal=causal, scale=scale)
    dq, dk, dv = attn.attn_bwd(tq, tk, tv, o, lse, tdo, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_last_device_status() == 0
    host = [dvi.to_host_f64(x) for x in (dq, dk, dv, o, lse)]
    return dict(dq=host[0], dk=host[1], dv=host[2], o=host[3], lse=host[4])


def check(dev, seed, B, H, N, d, causal, heads=None, q_factor=1.0):
    q, k, v, do = backward_inputs(seed, B, H, N, d, q_factor)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    g = run_bwd(dev, q, k, v, do, causal, scale)
    f = lambda x: bf16_to_f32(x).astype(np.float64)
    heads = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    for b, h in heads:
        bounds = bwd_tolerance.head_bounds(f(q[b, :, h]), f(k[b, :, h]), f(v[b, :, h]),
                                           f(do[b, :, h]), causal, scale, g["o"][b, :, h],
                                           g["lse"][b, h])
        got = {name: g[name][b, :, h] for name in ("dq", "dk", "dv")}
        bwd_tolerance.check_head(got, bounds, f"B={B} H={H} N={N} d={d} causal={causal} head={b, h}")


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_backward(dev, causal):
    check(dev, 1, 1, 2, 128, 64, causal)


RAGGED = [(1, 1, 1, 64), (1, 2, 100, 128), (2, 1, 129, 64), (1, 2, 257, 128), (1, 1, 300, 64),
          (1, 2, 640, 128), (1, 1, 1000, 64)]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", RAGGED, ids=lambda s: "x".join(map(str, s)))
def test_ragged_backward(dev, shape, causal):
    B, H, N, d = shape
    check(dev, 1100 + N, B, H, N, d, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_peaky_backward(dev, causal):
    """Q scaled x4: sharp softmax rows."""
    check(dev, 1200, 1, 2, 300, 128, causal, q_factor=4.0)


def test_prefill_workload_backward_sampled_heads(dev):
    """The prefill workload's shape (B=4, H=16, N=2048, d=128, causal): every head is
    computed on the GPU, four seeded heads are checked in full."""
    P = PREFILL
    pick = np.random.Generator(np.random.PCG64(1300)).choice(P["B"] * P["H"], 4, replace=False)
    heads = [(int(x) // P["H"], int(x) % P["H"]) for x in pick]
    check(dev, 1301, P["B"], P["H"], P["N"], P["d"], True, heads)


@pytest.mark.parametrize("cfg", [(1, 4, 4096, 128, True), (2, 8, 2048, 64, False)],
                         ids=["N4096-d128-causal", "N2048-d64"])
def test_longer_backward_sampled_heads(dev, cfg):
    B, H, N, d, causal = cfg
    pick = np.random.Generator(np.random.PCG64(1400 + N)).choice(B * H, 2, replace=False)
    check(dev, 1401 + N, B, H, N, d, causal, [(int(x) // H, int(x) % H) for x in pick])


def test_backward_is_deterministic(dev):
    torch, attn, dvi = dev
    q, k, v, do = (dvi.to_device_bf16(x) for x in backward_inputs(1500, 2, 3, 700, 128))
    o, lse = attn.attn_fwd(q, k, v, causal=True)
    a = attn.attn_bwd(q, k, v, o, lse, do, causal=True)
    b = attn.attn_bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_backward_binding_checks(dev):
    torch, attn, dvi = dev
    q, k, v, do = (dvi.to_device_bf16(x) for x in backward_inputs(1501, 1, 2, 100, 64))
    o, lse = attn.attn_fwd(q, k, v)
    with pytest.raises(ValueError):
        attn.attn_bwd(q, k, v, o, lse[:, :1], do)
    small = torch.empty(16, dtype=torch.uint8, device=q.device)
    with pytest.raises(attn.AttnError) as e:
        attn.attn_bwd(q, k, v, o, lse, do, workspace=small)
    assert e.value.status == 4
