"""Split-KV decode parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances: output max-abs <= 2e-2, mean-abs <= 2e-3, LSE within 1e-3.
Contiguous and paged caches must give bit-identical results.
"""

import math

import numpy as np
import pytest

import oracle
from io_aware_attention_03_b300.inputs import DECODE, decode_inputs

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from io_aware_attention_03_b300 import attn, device_inputs

    return torch, attn, device_inputs


def run_decode(dev, di, paged, scale):
    torch, attn, dvi = dev
    q, kc, vc, seqlens, pt = dvi.decode_device_inputs(di, paged)
    o, lse = attn.attn_decode(q, kc, vc, seqlens, page_table=pt, scale=scale)
    torch.cuda.synchronize()
    status = attn.attn_last_device_status()
    return o, lse, status


def check(o, lse, o_ref, lse_ref, what):
    o = o.reshape(o_ref.shape)
    finite = np.isfinite(lse_ref)
    err = np.abs(o - o_ref)
    assert err.max() <= O_MAX, f"{what} O max-abs {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"{what} O mean-abs {err.mean():.3e}"
    assert np.array_equal(np.isfinite(lse), finite), what
    assert np.abs(lse[finite] - lse_ref[finite]).max(initial=0.0) <= LSE_MAX, what


def oracle_for(di, scale):
    kp, vp = di.paged_pool(di.k_tokens), di.paged_pool(di.v_tokens)
    return oracle.decode(di.q, kp, vp, di.seqlens, scale, page_table=di.page_table(),
                         page_size=di.page_size)


@pytest.mark.parametrize("d", [64, 128])
def test_small_lengths_contiguous_and_paged(dev, d):
    torch, attn, dvi = dev
    lens = (1, 15, 16, 17, 255, 256, 257, 1000, 513)
    di = decode_inputs(310 + d, len(lens), 6, d, 0, 0, seqlens=lens)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    o_ref, lse_ref = oracle_for(di, scale)
    outs = []
    for paged in (False, True):
        o, lse, status = run_decode(dev, di, paged, scale)
        assert status == 0
        check(dvi.to_host_f64(o), dvi.to_host_f64(lse), o_ref, lse_ref, f"d={d} paged={paged}")
        outs.append((o, lse))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_decode_config_full(dev):
    """64 sequences, H=32, d=128, lengths ~ U[512, 8192], contiguous and paged, every output row."""
    torch, attn, dvi = dev
    di = decode_inputs(DECODE["seed"], DECODE["num_seqs"], DECODE["H"], DECODE["d"],
                       DECODE["len_lo"], DECODE["len_hi"], page_size=DECODE["page_size"])
    scale = float(np.float32(1.0 / math.sqrt(DECODE["d"])))
    o_ref, lse_ref = oracle_for(di, scale)
    res = []
    for paged in (False, True):
        o, lse, status = run_decode(dev, di, paged, scale)
        assert status == 0
        check(dvi.to_host_f64(o), dvi.to_host_f64(lse), o_ref, lse_ref, f"decode paged={paged}")
        res.append((o, lse))
        del o, lse
        torch.cuda.empty_cache()
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])


def test_zero_length_sequence(dev):
    torch, attn, dvi = dev
    lens = (0, 40, 0, 300)
    di = decode_inputs(320, len(lens), 4, 128, 0, 0, seqlens=lens)
    scale = 0.1
    o_ref, lse_ref = oracle_for(di, scale)
    for paged in (False, True):
        q, kc, vc, seqlens, pt = dvi.decode_device_inputs(di, paged)
        o, lse = attn.attn_decode(q, kc, vc, seqlens, page_table=pt, scale=scale)
        torch.cuda.synchronize()
        assert attn.attn_last_device_status() == 0
        o_h, lse_h = dvi.to_host_f64(o), dvi.to_host_f64(lse)
        check(o_h, lse_h, o_ref, lse_ref, f"zero-length paged={paged}")
        assert np.all(o_h[0] == 0) and np.all(np.isneginf(lse_h[0]))


def test_out_of_range_inputs_are_recorded_not_faulted(dev):
    """A length beyond max_seqlen is clamped and an invalid page id skipped; both are reported."""
    torch, attn, dvi = dev
    lens = (20, 40)
    di = decode_inputs(321, 2, 4, 64, 0, 0, seqlens=lens)
    q, kc, vc, seqlens, pt = dvi.decode_device_inputs(di, paged=True)
    bad_pt = pt.clone()
    bad_pt[1, 1] = 10_000  # beyond the pool
    attn.attn_decode(q, kc, vc, seqlens, page_table=bad_pt, scale=0.1)
    assert attn.attn_last_device_status() == 1
    assert attn.attn_last_device_status() == 0  # reading clears it
    q2, kc2, vc2, seqlens2, _ = dvi.decode_device_inputs(di, paged=False)
    seqlens2[0] = 10_000  # beyond the cache
    o, _ = attn.attn_decode(q2, kc2, vc2, seqlens2, scale=0.1)
    assert attn.attn_last_device_status() == 1
    assert bool(torch.isfinite(o.float()).all())


def test_split_invariance(dev):
    """One sequence spanning many splits equals the oracle at every split boundary length."""
    torch, attn, dvi = dev
    lens = (256 * 3, 256 * 3 + 1, 256 * 7 - 1, 4096)
    di = decode_inputs(330, len(lens), 2, 128, 0, 0, seqlens=lens)
    scale = float(np.float32(1.0 / math.sqrt(128)))
    o_ref, lse_ref = oracle_for(di, scale)
    o, lse, status = run_decode(dev, di, True, scale)
    assert status == 0
    check(dvi.to_host_f64(o), dvi.to_host_f64(lse), o_ref, lse_ref, "splits")


def test_workspace_too_small_is_rejected(dev):
    torch, attn, dvi = dev
    di = decode_inputs(340, 2, 4, 64, 0, 0, seqlens=(100, 300))
    q, kc, vc, seqlens, _ = dvi.decode_device_inputs(di, paged=False)
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(attn.AttnError):
        attn.attn_decode(q, kc, vc, seqlens, scale=0.1, workspace=ws)


def test_binding_shape_checks(dev):
    """The decode wrappers refuse mismatched shapes before the call (the C ABI sees only pointers)."""
    torch, attn, dvi = dev
    di = decode_inputs(330, 3, 4, 64, 20, 40)
    q, kc, vc, seqlens, _ = dvi.decode_device_inputs(di, paged=False)
    L = kc.shape[1]
    # contiguous: max_seqlen is the cache's row stride, so it must equal the second dimension
    with pytest.raises(ValueError, match="max_seqlen"):
        attn.attn_decode(q, kc, vc, seqlens, max_seqlen=L - 1)
    o_ref, _ = attn.attn_decode(q, kc, vc, seqlens, max_seqlen=L)
    out = torch.empty_like(q)
    lse = torch.empty((3, 4), dtype=torch.float32, device=q.device)
    for fn in (attn.attn_decode_noalloc,):
        with pytest.raises(ValueError, match="lse"):
            fn(q, kc, vc, seqlens, out, torch.empty((3, 3), dtype=torch.float32, device=q.device))
        with pytest.raises(ValueError, match="heads"):
            fn(q, kc[:, :, :3].contiguous(), vc[:, :, :3].contiguous(), seqlens, out, lse)
        with pytest.raises(ValueError, match="same shape"):
            fn(q, kc, vc[:, :-1].contiguous(), seqlens, out, lse)
        with pytest.raises(ValueError, match="contiguous cache"):
            fn(q, kc[:2].contiguous(), vc[:2].contiguous(), seqlens, out, lse)
        with pytest.raises(ValueError, match="seqlens"):
            fn(q, kc, vc, seqlens[:2].contiguous(), out, lse)
        with pytest.raises(ValueError, match="max_seqlen"):
            fn(q, kc, vc, seqlens, out, lse, max_seqlen=L - 1)
    with pytest.raises(ValueError, match="lse"):
        attn.attn_decode(q, kc, vc, seqlens, lse=torch.empty((4, 3), dtype=torch.float32, device=q.device))
    torch.cuda.synchronize()
    assert attn.attn_last_device_status() == 0
    assert o_ref.shape == q.shape
