"""Prefill parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Tolerances for bf16 inputs drawn from N(0, 1): output max-abs error <= 2e-2,
mean-abs error <= 2e-3; LSE within 1e-3 absolute.
"""

import math
import os

import numpy as np
import pytest

import oracle
from io_aware_attention_03_b300.inputs import (LONG, PREFILL, TINY, bf16_to_f32, prefill_inputs,
                                               sample_rows, sweep_configs)

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3
IMPLS = ("tmem2", "tmem1", "smem1")


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from io_aware_attention_03_b300 import attn, device_inputs

    return torch, attn, device_inputs


@pytest.fixture
def impl_env():
    old = os.environ.get("ATTN_PREFILL_IMPL")

    def set_impl(name):
        os.environ["ATTN_PREFILL_IMPL"] = name

    yield set_impl
    if old is None:
        os.environ.pop("ATTN_PREFILL_IMPL", None)
    else:
        os.environ["ATTN_PREFILL_IMPL"] = old


def run_gpu(dev, q, k, v, causal, scale):
    torch, attn, di = dev
    tq, tk, tv = (di.to_device_bf16(x) for x in (q, k, v))
    o, lse = attn.attn_fwd(tq, tk, tv, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_last_device_status() == 0
    return di.to_host_f64(o), di.to_host_f64(lse)


def check(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    err = np.abs(o_gpu - o_ref)
    assert np.all(np.isfinite(o_gpu)), what
    assert err.max() <= O_MAX, f"{what} O max-abs {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"{what} O mean-abs {err.mean():.3e}"
    lerr = np.abs(lse_gpu - lse_ref)
    assert lerr.max() <= LSE_MAX, f"{what} LSE max-abs {lerr.max():.3e}"


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("impl", IMPLS)
def test_tiny_config(dev, impl_env, impl, causal):
    impl_env(impl)
    q, k, v = prefill_inputs(TINY["seed"], TINY["B"], TINY["H"], TINY["N"], TINY["d"])
    scale = float(np.float32(1.0 / math.sqrt(TINY["d"])))
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    o, lse = run_gpu(dev, q, k, v, causal, scale)
    check(o, lse, o_ref, lse_ref, f"tiny {impl} causal={causal}")


SMALL = [(1, 1, 1, 64), (1, 2, 100, 128), (2, 3, 129, 64), (1, 2, 257, 128), (2, 2, 300, 64),
         (1, 1, 640, 128), (1, 4, 1000, 128), (3, 1, 383, 64)]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("impl", IMPLS)
def test_ragged_shapes_full_output(dev, impl_env, shape, causal, impl):
    impl_env(impl)
    B, H, N, d = shape
    q, k, v = prefill_inputs(40 + N + d, B, H, N, d)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    o, lse = run_gpu(dev, q, k, v, causal, scale)
    check(o, lse, o_ref, lse_ref, f"{shape} {impl} causal={causal}")


def test_peaky_scores(dev):
    q, k, v = prefill_inputs(77, 2, 2, 384, 128, q_factor=4.0)
    scale = float(np.float32(1.0 / math.sqrt(128)))
    for causal in (False, True):
        o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
        o, lse = run_gpu(dev, q, k, v, causal, scale)
        check(o, lse, o_ref, lse_ref, f"peaky causal={causal}")


def sampled_check(dev, cfg, nrows, what):
    B, H, N, d = cfg["B"], cfg["H"], cfg["N"], cfg["d"]
    causal = cfg.get("causal", False)
    q, k, v = prefill_inputs(cfg["seed"], B, H, N, d, cfg.get("q_factor", 1.0))
    scale = float(np.float32(1.0 / math.sqrt(d)))
    o, lse = run_gpu(dev, q, k, v, causal, scale)
    rows = sample_rows(cfg["seed"] + 1000, B, H, N, nrows)
    o_ref, lse_ref = oracle.attn_rows(q, k, v, causal, scale, rows)
    b, h, i = rows[:, 0], rows[:, 1], rows[:, 2]
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    check(o[b, i, h], lse[b, h, i], o_ref, lse_ref, what)


def test_prefill_config_sampled(dev):
    sampled_check(dev, PREFILL, 512, "prefill B=4 H=16 N=2048 d=128 causal")


@pytest.mark.parametrize("cfg", sweep_configs(),
                         ids=lambda c: f"N{c['N']}-H{c['H']}-d{c['d']}-c{int(c['causal'])}-q{c['q_factor']:g}")
def test_seqlen_sweep_sampled(dev, cfg):
    sampled_check(dev, cfg, 256, f"sweep {cfg}")


@pytest.mark.parametrize("cfg", LONG, ids=lambda c: f"N{c['N']}")
def test_long_context_sampled(dev, cfg):
    """Long context: the oracle checks a seeded subset of 256 query rows."""
    torch, attn, di = dev
    B, H, N, d = cfg["B"], cfg["H"], cfg["N"], cfg["d"]
    q, k, v = prefill_inputs(cfg["seed"], B, H, N, d)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    tq, tk, tv = (di.to_device_bf16(x) for x in (q, k, v))
    o, lse = attn.attn_fwd(tq, tk, tv, causal=True, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_last_device_status() == 0
    g = np.random.Generator(np.random.PCG64(cfg["seed"] + 5000))
    flat = g.choice(H * N, size=256, replace=False)
    rows = np.stack([np.zeros_like(flat), flat // N, flat % N], axis=1).astype(np.int64)
    o_ref, lse_ref = oracle.attn_rows(q, k, v, True, scale, rows)
    b, h, i = (torch.from_numpy(rows[:, c]).cuda() for c in range(3))
    o_rows = di.to_host_f64(o[b, i, h])
    lse_rows = di.to_host_f64(lse[b, h, i])
    check(o_rows, lse_rows, o_ref, lse_ref, f"long N={N}")
    assert bool(torch.isfinite(o.float()).all())


@pytest.mark.parametrize("causal", [False, True])
def test_banded_deal_matches_single_head_calls(dev, causal):
    """B=1, H=16, N=16384, d=128: the K/V of all heads (128 MB) is more than L2 holds, so the
    kernel deals its units band by band from a device counter.  Each unit's arithmetic does
    not depend on the order, so every head must equal, bit for bit, a call on that head alone
    (8 MB of K/V: the static deal)."""
    torch, attn, di = dev
    B, H, N, d = 1, 16, 16384, 128
    g = torch.Generator(device="cuda")
    g.manual_seed(31 + int(causal))
    q, k, v = (torch.randn((B, N, H, d), generator=g, device="cuda").to(torch.bfloat16)
               for _ in range(3))
    o, lse = attn.attn_fwd(q, k, v, causal=causal)
    for h in (0, 7, 15):
        qh, kh, vh = (x[:, :, h:h + 1, :].contiguous() for x in (q, k, v))
        oh, lseh = attn.attn_fwd(qh, kh, vh, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(o[:, :, h:h + 1, :], oh), f"head {h}"
        assert torch.equal(lse[:, h:h + 1, :], lseh), f"head {h}"
    assert attn.attn_last_device_status() == 0


def test_banded_calls_on_two_streams(dev):
    """Two banded calls (B=1, H=32, N=8192: 128 MB of K/V each) in flight at once on two
    streams: each takes its own unit counter, so both must equal their one-at-a-time results
    bit for bit."""
    torch, attn, di = dev
    B, H, N, d = 1, 32, 8192, 128
    g = torch.Generator(device="cuda")
    g.manual_seed(41)
    x1, x2 = ([torch.randn((B, N, H, d), generator=g, device="cuda").to(torch.bfloat16)
               for _ in range(3)] for _ in range(2))
    ref1 = attn.attn_fwd(*x1, causal=True)
    ref2 = attn.attn_fwd(*x2, causal=True)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s1):
        out1 = attn.attn_fwd(*x1, causal=True)
    with torch.cuda.stream(s2):
        out2 = attn.attn_fwd(*x2, causal=True)
    torch.cuda.synchronize()
    assert attn.attn_last_device_status() == 0
    for a, b in zip(out1 + out2, ref1 + ref2):
        assert torch.equal(a, b)


def test_deterministic(dev):
    torch, attn, di = dev
    q, k, v = prefill_inputs(91, 2, 4, 1000, 128)
    tq, tk, tv = (di.to_device_bf16(x) for x in (q, k, v))
    o1, l1 = attn.attn_fwd(tq, tk, tv, causal=True)
    o2, l2 = attn.attn_fwd(tq, tk, tv, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_lse_optional_and_scale_default(dev):
    torch, attn, di = dev
    q, k, v = prefill_inputs(92, 1, 2, 200, 64)
    tq, tk, tv = (di.to_device_bf16(x) for x in (q, k, v))
    o_a = attn.attn_fwd(tq, tk, tv, causal=False, return_lse=False)
    o_b, _ = attn.attn_fwd(tq, tk, tv, causal=False, scale=1.0 / math.sqrt(64))
    torch.cuda.synchronize()
    assert torch.equal(o_a, o_b)


def test_empty_problem(dev):
    torch, attn, di = dev
    z = torch.empty((2, 0, 4, 64), dtype=torch.bfloat16, device="cuda")
    o, lse = attn.attn_fwd(z, z, z, causal=True)
    assert o.shape == z.shape and lse.shape == (2, 4, 0)


def test_python_preconditions(dev):
    torch, attn, di = dev
    x = torch.zeros((1, 16, 2, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):
        attn.attn_fwd(x, x, x)
    y = torch.zeros((1, 16, 2, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn.attn_fwd(y, y, y)
    z = torch.zeros((1, 2, 16, 64), dtype=torch.bfloat16, device="cuda").transpose(1, 2)
    with pytest.raises(ValueError):
        attn.attn_fwd(z, z, z)
    w = torch.zeros((1, 16, 2, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(attn.AttnError):
        attn.attn_fwd(w, w, w)
