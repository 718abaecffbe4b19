"""The layout plumbing that carries the seeded host inputs to the device, checked with
torch CPU tensors: every GPU parity test relies on it placing each value where the C ABI's
layout says it is."""

import numpy as np
import pytest

from io_aware_attention_03_b300 import device_inputs as dvi
from io_aware_attention_03_b300.inputs import decode_inputs, fp8_cache, fp8_prefill_inputs, prefill_inputs

torch = pytest.importorskip("torch")


def test_bf16_round_trip_is_exact():
    q, _, _ = prefill_inputs(60, 1, 2, 37, 64)
    t = dvi.to_device_bf16(q, "cpu")
    assert t.dtype == torch.bfloat16 and tuple(t.shape) == q.shape
    assert np.array_equal(dvi.to_host_bits(t), q)


@pytest.mark.parametrize("N", [1, 100, 128, 130])
def test_fp8_prefill_vt_layout(N):
    """vt[b, h, c, n] = v[b, n, h, c] for n < N, zero padding up to the next multiple of 16."""
    f8 = fp8_prefill_inputs(61, 2, 3, N, 128)
    q, k, vt, qs, ks, vs = dvi.fp8_prefill_device(f8, "cpu")
    Np = (N + 15) // 16 * 16
    assert tuple(vt.shape) == (2, 3, 128, Np) and vt.dtype == torch.uint8
    vt = vt.numpy()
    assert np.array_equal(vt[..., :N], np.transpose(f8.v, (0, 2, 3, 1)))
    assert not vt[..., N:].any()
    assert np.array_equal(q.numpy(), f8.q) and np.array_equal(k.numpy(), f8.k)
    assert np.array_equal(vs.numpy(), f8.v_scale)


@pytest.mark.parametrize("paged", [False, True])
def test_decode_caches_place_every_token(paged):
    """Token t of sequence s sits at [s, t] (contiguous) or at slot t % 16 of page
    page_table[s, t // 16] (paged); everything else is zero."""
    di = decode_inputs(62, 3, 2, 64, 0, 0, seqlens=(5, 40, 17))
    kc, vc = dvi.decode_caches(di, paged, "cpu")
    kb = dvi.to_host_bits(kc)
    pt = di.page_table()
    filled = np.zeros(kb.shape[:2], bool)
    for s in range(di.num_seqs):
        for t in range(int(di.seqlens[s])):
            row = di.k_tokens[di.offsets[s] + t]
            if paged:
                assert np.array_equal(kb[pt[s, t // 16], t % 16], row)
                filled[pt[s, t // 16], t % 16] = True
            else:
                assert np.array_equal(kb[s, t], row)
                filled[s, t] = True
    assert not kb[~filled].any()
    f8 = fp8_cache(di)
    k8, v8, ks, vs = dvi.fp8_caches(di, f8, paged, "cpu")
    k8 = k8.numpy()
    s, t = 1, 33
    where = (pt[s, t // 16], t % 16) if paged else (s, t)
    assert np.array_equal(k8[where], f8.k_tokens[di.offsets[s] + t])
