"""Split-KV decode over an FP8 (E4M3) K/V cache with per-head scales: the CUDA
path (through the C ABI) against the fp64 oracle on the dequantized cache.

The cache holds e4m3 bytes and one fp32 scale per head for K and for V; the
attention is that of attn_decode over the values scale[h] * e4m3 ("Beyond the
memory wall", section "FlashInfer").  Tolerances as for bf16 decode: O max-abs
<= 2e-2, mean-abs <= 2e-3, LSE within 1e-3.  Contiguous and paged caches must
give bit-identical results.
"""

import math

import numpy as np
import pytest

import oracle
from io_aware_attention_03_b300.inputs import DECODE, decode_inputs, fp8_cache

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from io_aware_attention_03_b300 import attn, device_inputs

    return torch, attn, device_inputs


def run_fp8(dev, di, f8, paged, scale):
    torch, attn, dvi = dev
    q, _, _, seqlens, pt = dvi.decode_device_inputs(di, paged)
    kc, vc, ks, vs = dvi.fp8_caches(di, f8, paged)
    o, lse = attn.attn_decode_fp8(q, kc, vc, ks, vs, seqlens, page_table=pt, scale=scale)
    torch.cuda.synchronize()
    return o, lse, attn.attn_last_device_status()


def oracle_fp8(di, f8, scale):
    # paged pools of the fp8 bytes, built like the bf16 ones
    kp = di.paged_pool(f8.k_tokens)
    vp = di.paged_pool(f8.v_tokens)
    return oracle.decode_fp8(di.q, kp, vp, f8.k_scale, f8.v_scale, di.seqlens, scale,
                             page_table=di.page_table(), page_size=di.page_size)


def check(o, lse, o_ref, lse_ref, what):
    o = o.reshape(o_ref.shape)
    finite = np.isfinite(lse_ref)
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX, f"{what} O max-abs {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"{what} O mean-abs {err.mean():.3e}"
    assert np.array_equal(np.isfinite(lse), finite), what
    assert np.abs(lse[finite] - lse_ref[finite]).max(initial=0.0) <= LSE_MAX, what


@pytest.mark.parametrize("pow2", [False, True], ids=["float-scales", "pow2-scales"])
@pytest.mark.parametrize("d", [64, 128])
def test_small_lengths_contiguous_and_paged(dev, d, pow2):
    torch, attn, dvi = dev
    lens = (1, 15, 16, 17, 255, 256, 257, 1000, 513, 0)
    di = decode_inputs(710 + d, len(lens), 6, d, 0, 0, seqlens=lens)
    f8 = fp8_cache(di, pow2_scales=pow2)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    o_ref, lse_ref = oracle_fp8(di, f8, scale)
    outs = []
    for paged in (False, True):
        o, lse, status = run_fp8(dev, di, f8, paged, scale)
        assert status == 0
        check(dvi.to_host_f64(o), dvi.to_host_f64(lse), o_ref, lse_ref, f"d={d} paged={paged}")
        outs.append((o, lse))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_decode_workload_fp8_sampled(dev):
    """64 sequences, H=32, d=128, lengths ~ U[512, 8192], paged e4m3 cache; the kernel runs
    the whole batch, the oracle checks every head of a seeded subset of 12 sequences."""
    torch, attn, dvi = dev
    di = decode_inputs(DECODE["seed"], DECODE["num_seqs"], DECODE["H"], DECODE["d"],
                       DECODE["len_lo"], DECODE["len_hi"], page_size=DECODE["page_size"])
    f8 = fp8_cache(di)
    scale = float(np.float32(1.0 / math.sqrt(DECODE["d"])))
    o, lse, status = run_fp8(dev, di, f8, True, scale)
    assert status == 0
    o, lse = dvi.to_host_f64(o).reshape(di.num_seqs, DECODE["H"], DECODE["d"]), dvi.to_host_f64(lse)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    pick = np.sort(np.random.Generator(np.random.PCG64(722)).choice(di.num_seqs, 12, replace=False))
    pick = np.unique(np.concatenate([pick, [int(np.argmax(di.seqlens))]]))  # the longest too
    kp, vp, pt = di.paged_pool(f8.k_tokens), di.paged_pool(f8.v_tokens), di.page_table()
    o_ref, lse_ref = oracle.decode_fp8(di.q[pick], kp, vp, f8.k_scale, f8.v_scale,
                                       di.seqlens[pick], scale, page_table=pt[pick])
    check(o[pick], lse[pick], o_ref, lse_ref, "fp8 decode workload")


def test_scales_are_applied_per_head(dev):
    """Doubling one head's value scale doubles that head's output and nothing else."""
    torch, attn, dvi = dev
    di = decode_inputs(720, 3, 4, 128, 0, 0, seqlens=(50, 300, 17))
    f8 = fp8_cache(di)
    q, _, _, seqlens, pt = dvi.decode_device_inputs(di, True)
    kc, vc, ks, vs = dvi.fp8_caches(di, f8, True)
    o1, l1 = attn.attn_decode_fp8(q, kc, vc, ks, vs, seqlens, page_table=pt)
    vs2 = vs.clone()
    vs2[2] *= 2
    o2, l2 = attn.attn_decode_fp8(q, kc, vc, ks, vs2, seqlens, page_table=pt)
    torch.cuda.synchronize()
    assert torch.equal(l1, l2)
    assert torch.equal(o2[:, :, 2].float(), 2 * o1[:, :, 2].float())
    keep = [0, 1, 3]
    assert torch.equal(o1[:, :, keep], o2[:, :, keep])


def test_fp8_rejects_missing_scales(dev):
    torch, attn, dvi = dev
    di = decode_inputs(721, 2, 2, 64, 0, 0, seqlens=(10, 20))
    f8 = fp8_cache(di)
    q, _, _, seqlens, _ = dvi.decode_device_inputs(di, False)
    kc, vc, ks, vs = dvi.fp8_caches(di, f8, False)
    with pytest.raises(ValueError):
        attn.attn_decode_fp8(q, kc, vc, ks[:1], vs, seqlens)
