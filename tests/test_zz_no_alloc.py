"""attn_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers may not call cudaMalloc on their call path -- a plugin inside
another runtime that owns all device memory and gives it no allocator, or a
serving loop that forbids allocation (and the synchronisation it can bring)
once running.  attn_decode_noalloc takes the caller's inputs and outputs but no
workspace; the split partials go to a fixed scratch array in the library.

Its results must match the allocating entry point attn_decode within the
parity tolerance, on two calls in a row (the second call sees whatever the
first left in the shared scratch array).  This file is collected last.
"""

import ctypes
import math

import numpy as np
import pytest

from io_aware_attention_03_b300.inputs import decode_inputs

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3
SCRATCH_BYTES = 64 << 20


def test_noalloc_rejects_sizes_beyond_its_scratch_without_cuda():
    """Host-side: a problem whose workspace exceeds the fixed scratch is refused (no GPU needed)."""
    from io_aware_attention_03_b300 import build as b

    lib = ctypes.CDLL(b.build())
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    lib.attn_decode_noalloc.restype = i
    lib.attn_decode_workspace_size.argtypes = [i, i, i, i]
    lib.attn_decode_workspace_size.restype = ctypes.c_size_t
    A = 0x10000000
    # 1024 sequences x 64 heads x 8192 tokens needs far more than the scratch
    assert lib.attn_decode_workspace_size(1024, 64, 128, 8192) > SCRATCH_BYTES
    rc = lib.attn_decode_noalloc(A, A, A, A, None, A + 0x100000, None, 1024, 64, 128, 8192, 16, 0, 0,
                                 0.1, None)
    assert rc == 4  # ATTN_ERR_WORKSPACE
    assert lib.attn_decode_noalloc(None, A, A, A, None, A, None, 4, 8, 128, 512, 16, 0, 0, 0.1,
                                   None) == 1
    assert lib.attn_decode_noalloc(A, A, A, A, None, A, None, 0, 8, 128, 512, 16, 0, 0, 0.1, None) == 0


def test_noalloc_validates_everything_before_its_first_cuda_call():
    """Misaligned pointers and oversized grids are refused on the host, before the scratch
    address is looked up: these calls must return without touching CUDA (no GPU here)."""
    from io_aware_attention_03_b300 import build as b

    lib = ctypes.CDLL(b.build())
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    lib.attn_decode_noalloc.restype = i
    A = 0x10000000

    def call(q=A, kc=A + 0x1000000, vc=A + 0x2000000, seqlens=A + 0x3000000, pt=None,
             o=A + 0x4000000, lse=None, S=4, H=8, d=128, max_seqlen=512, page_size=16,
             max_pages=0, num_pages=0):
        return lib.attn_decode_noalloc(q, kc, vc, seqlens, pt, o, lse, S, H, d, max_seqlen,
                                       page_size, max_pages, num_pages, 0.1, None)

    assert call(q=A + 8) == 3
    assert call(kc=A + 0x1000004) == 3
    assert call(o=A + 0x4000002) == 3
    assert call(seqlens=A + 0x3000002) == 3
    assert call(lse=A + 0x5000001) == 3
    assert call(pt=A + 0x6000002, max_pages=32, num_pages=64) == 3
    assert call(pt=A + 0x6000000, page_size=32, max_pages=32, num_pages=64) == 2
    assert call(pt=A + 0x6000000, max_pages=8, num_pages=64) == 1  # 8 * 16 < 512
    assert call(S=70000, H=1, max_seqlen=16) == 2  # grid y limit
    assert call(d=96) == 2


@pytest.mark.gpu
def test_noalloc_matches_allocating_decode_on_two_calls():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from io_aware_attention_03_b300 import attn
    from io_aware_attention_03_b300 import device_inputs as dvi

    batches = [
        (decode_inputs(400, 16, 8, 128, 1, 3000), True),     # paged cache, d=128
        (decode_inputs(401, 24, 6, 64, 200, 2000), False),   # contiguous cache, d=64
    ]
    for di, paged in batches:
        q, kc, vc, seqlens, pt = dvi.decode_device_inputs(di, paged)
        d = di.q.shape[2]
        scale = 1.0 / math.sqrt(d)
        o_ref, lse_ref = attn.attn_decode(q, kc, vc, seqlens, page_table=pt, scale=scale)
        o = torch.empty_like(q)
        lse = torch.empty_like(lse_ref)
        attn.attn_decode_noalloc(q, kc, vc, seqlens, o, lse, page_table=pt, scale=scale)
        torch.cuda.synchronize()
        assert attn.attn_last_device_status() == 0
        err = (o.float() - o_ref.float()).abs()
        assert float(err.max()) <= O_MAX and float(err.mean()) <= O_MEAN
        assert float((lse - lse_ref).abs().max()) <= LSE_MAX
