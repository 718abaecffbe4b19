"""FP8 (E4M3) prefill parity: attn_fwd_fp8 (through the C ABI) against the fp64 oracle on
the dequantized inputs.

Q, K, V are E4M3 with one fp32 scale per head ("FlashAttention complete summary", section
"FlashAttention 3"; "Beyond the memory wall", section "FlashAttention-3가 다른 이유").  The
tolerance is derived from the arithmetic in tests/fp8_tolerance.py: every output element
within 2^-4 * sum_j p_j |v_j| (E4M3 rounding of P) plus smaller terms, the mean error within
the RMS that rounding predicts, and LSE within 1e-3 as for bf16.
"""

import math

import numpy as np
import pytest

import fp8_tolerance
from io_aware_attention_03_b300.inputs import PREFILL, fp8_prefill_inputs, sample_rows

pytestmark = pytest.mark.gpu

D = 128
SCALE = float(np.float32(1.0 / math.sqrt(D)))
DIMS = (64, 128)


def scale_for(d):
    return float(np.float32(1.0 / math.sqrt(d)))


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from io_aware_attention_03_b300 import attn, device_inputs

    return torch, attn, device_inputs


def run_fp8(dev, f8, causal, scale=SCALE):
    torch, attn, dvi = dev
    q, k, vt, qs, ks, vs = dvi.fp8_prefill_device(f8)
    o, lse = attn.attn_fwd_fp8(q, k, vt, qs, ks, vs, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert attn.attn_last_device_status() == 0
    return dvi.to_host_f64(o), dvi.to_host_f64(lse)


def compare(dev, f8, causal, rows=None, what=""):
    scale = scale_for(f8.q.shape[3])
    o_gpu, lse_gpu = run_fp8(dev, f8, causal, scale)
    o, lse, bound, sigma = fp8_tolerance.oracle_and_bounds(f8, causal, scale, rows)
    if rows is None:
        B, N, H, _ = f8.q.shape
        b, h, i = (x.ravel() for x in np.meshgrid(np.arange(B), np.arange(H), np.arange(N),
                                                   indexing="ij"))
    else:
        b, h, i = np.asarray(rows).T
    fp8_tolerance.check(o_gpu[b, i, h], lse_gpu[b, h, i], o, lse, bound, sigma, what)


@pytest.mark.parametrize("d", DIMS)
@pytest.mark.parametrize("pow2", [True, False], ids=["pow2-scales", "float-scales"])
@pytest.mark.parametrize("causal", [False, True])
def test_tiny_fp8(dev, causal, pow2, d):
    f8 = fp8_prefill_inputs(1, 1, 2, 128, d, pow2_scales=pow2)
    compare(dev, f8, causal, what=f"tiny d={d} causal={causal} pow2={pow2}")


RAGGED = [(1, 1, 1), (1, 2, 100), (2, 3, 129), (1, 2, 257), (2, 2, 300), (1, 1, 640), (1, 4, 1000)]


@pytest.mark.parametrize("d", DIMS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("shape", RAGGED, ids=lambda s: "x".join(map(str, s)))
def test_ragged_fp8(dev, shape, causal, d):
    B, H, N = shape
    f8 = fp8_prefill_inputs(900 + N + d, B, H, N, d, pow2_scales=(N % 2 == 0))
    compare(dev, f8, causal, what=f"{shape} d={d} causal={causal}")


@pytest.mark.parametrize("d", DIMS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [300, 1000])
def test_peaky_fp8(dev, N, causal, d):
    """Q scaled x4 before quantization: sharp softmax rows, where P's rounding matters most."""
    f8 = fp8_prefill_inputs(950 + N + d, 1, 2, N, d, q_factor=4.0)
    compare(dev, f8, causal, what=f"peaky N={N} d={d} causal={causal}")


def test_prefill_workload_fp8_sampled(dev):
    """The prefill workload (B=4, H=16, N=2048, d=128, causal) in FP8; 512 seeded rows plus
    tile-edge rows checked."""
    P = PREFILL
    f8 = fp8_prefill_inputs(P["seed"], P["B"], P["H"], P["N"], P["d"])
    rows = sample_rows(960, P["B"], P["H"], P["N"], 512)
    compare(dev, f8, True, rows, "prefill workload fp8")


@pytest.mark.parametrize("causal", [False, True])
def test_long_sequence_fp8_sampled(dev, causal):
    """B=1, H=16, N=16384 (the sweep's longest d=128 shape) in FP8; 256 seeded rows."""
    f8 = fp8_prefill_inputs(970 + int(causal), 1, 16, 16384, D)
    rows = sample_rows(971, 1, 16, 16384, 256)
    compare(dev, f8, causal, rows, f"N=16384 fp8 causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_long_sequence_fp8_d64_sampled(dev, causal):
    """B=1, H=32, N=16384, d=64 (the sweep's longest d=64 shape) in FP8; 256 seeded rows."""
    f8 = fp8_prefill_inputs(972 + int(causal), 1, 32, 16384, 64)
    rows = sample_rows(973, 1, 32, 16384, 256)
    compare(dev, f8, causal, rows, f"N=16384 d=64 fp8 causal={causal}")


def test_long_sequence_fp8_banded_sampled(dev):
    """B=1, H=32, N=16384, d=128 causal in FP8: the K/V of all heads (128 MB) is more than L2
    holds, so the kernel takes its units band by band with the dynamic deal; 256 seeded rows."""
    f8 = fp8_prefill_inputs(974, 1, 32, 16384, D)
    rows = sample_rows(975, 1, 32, 16384, 256)
    compare(dev, f8, True, rows, "N=16384 H=32 fp8 banded")


def test_fp8_scales_are_applied_per_head(dev):
    """Doubling head 1's v_scale doubles exactly its output; moving a factor 2 from k_scale
    to q_scale changes nothing (the product q_scale * k_scale is the same number)."""
    torch, attn, dvi = dev
    f8 = fp8_prefill_inputs(980, 2, 3, 200, D)
    q, k, vt, qs, ks, vs = dvi.fp8_prefill_device(f8)
    o1, l1 = attn.attn_fwd_fp8(q, k, vt, qs, ks, vs, causal=True)
    vs2 = vs.clone()
    vs2[1] *= 2
    o2, l2 = attn.attn_fwd_fp8(q, k, vt, qs, ks, vs2, causal=True)
    o3, l3 = attn.attn_fwd_fp8(q, k, vt, qs * 2, ks / 2, vs, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(l1, l2) and torch.equal(o1[:, :, [0, 2]], o2[:, :, [0, 2]])
    assert torch.equal(o2[:, :, 1].float(), 2 * o1[:, :, 1].float())
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


def test_fp8_output_is_deterministic(dev):
    torch, attn, dvi = dev
    f8 = fp8_prefill_inputs(981, 2, 4, 700, D)
    q, k, vt, qs, ks, vs = dvi.fp8_prefill_device(f8)
    a = attn.attn_fwd_fp8(q, k, vt, qs, ks, vs, causal=False)
    b = attn.attn_fwd_fp8(q, k, vt, qs, ks, vs, causal=False)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_fp8_binding_checks(dev):
    torch, attn, dvi = dev
    f8 = fp8_prefill_inputs(982, 1, 2, 100, D)
    q, k, vt, qs, ks, vs = dvi.fp8_prefill_device(f8)
    with pytest.raises(ValueError):
        attn.attn_fwd_fp8(q, k, vt[..., :100].contiguous(), qs, ks, vs)   # keys not padded to 16
    with pytest.raises(ValueError):
        attn.attn_fwd_fp8(q, k, vt, qs[:1], ks, vs)
    q96 = torch.zeros((1, 100, 2, 96), dtype=torch.uint8, device=q.device)
    vt96 = torch.zeros((1, 2, 96, 112), dtype=torch.uint8, device=q.device)
    with pytest.raises(attn.AttnError) as e:  # head_dim 64 or 128 only
        attn.attn_fwd_fp8(q96, q96, vt96, qs, ks, vs)
    assert e.value.status == 2
    assert attn.fp8_vt_stride(100) == 112 and attn.fp8_vt_stride(128) == 128
