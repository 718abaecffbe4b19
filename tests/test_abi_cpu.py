"""The C-ABI library on a machine without a GPU: it loads, exports every symbol
the header declares, and rejects bad arguments before touching CUDA.

Validation runs on the host before any CUDA call, so these calls use fake
(never dereferenced) addresses and need no device.
"""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_b300.h")


@pytest.fixture(scope="module")
def lib():
    from io_aware_attention_03_b300 import build as b

    path = b.build()
    lib = ctypes.CDLL(path)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.attn_fwd.restype = i
    lib.attn_decode_workspace_size.argtypes = [i, i, i, i]
    lib.attn_decode_workspace_size.restype = sz
    lib.attn_decode.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp, sz, vp]
    lib.attn_decode.restype = i
    lib.attn_status_string.argtypes = [i]
    lib.attn_status_string.restype = ctypes.c_char_p
    lib.attn_prefill_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, vp]
    lib.attn_prefill_paged.restype = i
    lib.attn_decode_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp, sz,
                                    vp]
    lib.attn_decode_fp8.restype = i
    lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
    lib.attn_fwd_fp8.restype = i
    lib.attn_bwd_workspace_size.argtypes = [i, i, i, i]
    lib.attn_bwd_workspace_size.restype = sz
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
    lib.attn_bwd.restype = i
    return lib


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)


def test_header_declares_the_abi():
    names = declared_symbols()
    assert set(names) >= {"attn_fwd", "attn_fwd_fp8", "attn_bwd", "attn_bwd_workspace_size",
                          "attn_prefill_paged", "attn_decode", "attn_decode_fp8",
                          "attn_decode_workspace_size", "attn_last_device_status",
                          "attn_status_string"}


def test_library_exports_every_declared_symbol(lib):
    from io_aware_attention_03_b300 import build as b

    out = subprocess.run(["nm", "-D", "--defined-only", b.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_symbols():
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings(lib):
    names = {0: b"ATTN_OK", 1: b"ATTN_ERR_INVALID_ARG", 2: b"ATTN_ERR_UNSUPPORTED",
             3: b"ATTN_ERR_MISALIGNED", 4: b"ATTN_ERR_WORKSPACE", 5: b"ATTN_ERR_CUDA",
             6: b"ATTN_ERR_TIMEOUT"}
    for code, name in names.items():
        assert lib.attn_status_string(code) == name
    assert lib.attn_status_string(99) == b"ATTN_ERR_UNKNOWN"


A = 0x10000000  # a 16-byte aligned fake device address (never dereferenced)


def fwd(lib, q=A, k=A + 0x1000000, v=A + 0x2000000, o=A + 0x3000000, lse=None, B=1, H=2, N=128,
        d=64, causal=0, scale=0.125):
    return lib.attn_fwd(q, k, v, o, lse, B, H, N, d, causal, scale, None)


def test_fwd_rejects_bad_arguments_before_cuda(lib):
    assert fwd(lib, q=None) == 1
    assert fwd(lib, o=None) == 1
    assert fwd(lib, B=-1) == 1
    assert fwd(lib, N=-5) == 1
    assert fwd(lib, scale=0.0) == 1
    assert fwd(lib, scale=-1.0) == 1
    assert fwd(lib, scale=float("nan")) == 1
    assert fwd(lib, scale=float("inf")) == 1
    assert fwd(lib, d=96) == 2
    assert fwd(lib, d=256) == 2
    assert fwd(lib, q=A + 8) == 3
    assert fwd(lib, o=A + 0x3000002) == 3
    assert fwd(lib, lse=A + 0x4000001) == 3
    # output aliasing an input
    assert fwd(lib, o=A) == 1


def test_fwd_empty_problem_is_a_no_op(lib):
    assert fwd(lib, B=0) == 0
    assert fwd(lib, H=0) == 0
    assert fwd(lib, N=0) == 0


def fwd8(lib, q=A, k=A + 0x1000000, vt=A + 0x2000000, qs=A + 0x2F00000, ks=A + 0x2F00100,
         vs=A + 0x2F00200, o=A + 0x3000000, lse=None, B=1, H=2, N=100, d=128, causal=1, scale=0.1):
    return lib.attn_fwd_fp8(q, k, vt, qs, ks, vs, o, lse, B, H, N, d, causal, scale, None)


def test_fwd_fp8_rejects_bad_arguments_before_cuda(lib):
    for name in ("q", "k", "vt", "qs", "ks", "vs", "o"):
        assert fwd8(lib, **{name: None}) == 1, name
    assert fwd8(lib, B=-1) == 1
    assert fwd8(lib, scale=float("nan")) == 1 and fwd8(lib, scale=0.0) == 1
    assert fwd8(lib, d=96) == 2            # FP8 prefill is d = 64 or 128
    assert fwd8(lib, vt=A + 0x2000008) == 3
    assert fwd8(lib, qs=A + 0x2F00002) == 3
    assert fwd8(lib, o=A + 0x1000000) == 1  # output aliasing k
    assert fwd8(lib, B=0) == 0 and fwd8(lib, H=0) == 0 and fwd8(lib, N=0) == 0


def bwd(lib, q=A, k=A + 0x1000000, v=A + 0x2000000, o=A + 0x3000000, lse=A + 0x4000000,
        dout=A + 0x5000000, dq=A + 0x6000000, dk=A + 0x7000000, dv=A + 0x8000000, B=1, H=2, N=200,
        d=128, causal=1, scale=0.1, ws=A + 0x9000000, ws_bytes=1 << 20):
    return lib.attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, causal, scale, ws, ws_bytes, None)


def test_bwd_workspace_size(lib):
    # LSE*log2(e) and D, fp32 [B*H, N rounded up to 128], each padded to 256 bytes
    assert lib.attn_bwd_workspace_size(1, 2, 200, 128) == 2 * 2 * 256 * 4
    assert lib.attn_bwd_workspace_size(4, 16, 2048, 128) == 2 * 4 * 16 * 2048 * 4
    assert lib.attn_bwd_workspace_size(1, 1, 1, 64) == 2 * 512
    assert lib.attn_bwd_workspace_size(1, 1, 100, 96) == 0
    assert lib.attn_bwd_workspace_size(0, 1, 100, 64) == 0


def test_bwd_rejects_bad_arguments_before_cuda(lib):
    for name in ("q", "k", "v", "o", "lse", "dout", "dq", "dk", "dv"):
        assert bwd(lib, **{name: None}) == 1, name
    assert bwd(lib, B=-1) == 1 and bwd(lib, scale=float("inf")) == 1
    assert bwd(lib, d=96) == 2
    assert bwd(lib, dq=A + 0x6000008) == 3 and bwd(lib, lse=A + 0x4000002) == 3
    assert bwd(lib, ws=None) == 4 and bwd(lib, ws_bytes=100) == 4
    assert bwd(lib, ws=A + 0x9000004) == 3
    assert bwd(lib, dq=A) == 1                    # dq aliases q
    assert bwd(lib, dk=A + 0x6000000) == 1        # dk aliases dq
    assert bwd(lib, dv=A + 0x9000000) == 1        # dv aliases the workspace
    assert bwd(lib, B=0) == 0 and bwd(lib, N=0) == 0 and bwd(lib, H=0) == 0


def pp(lib, q=A, kc=A + 0x1000000, vc=A + 0x2000000, seqlens=A + 0x3000000, pt=A + 0x3100000,
       o=A + 0x4000000, lse=None, B=2, H=2, Nq=64, d=128, page_size=16, max_pages=16, num_pages=32,
       causal=1, scale=0.1):
    return lib.attn_prefill_paged(q, kc, vc, seqlens, pt, o, lse, B, H, Nq, d, page_size, max_pages,
                                  num_pages, causal, scale, None)


def test_prefill_paged_rejects_bad_arguments_before_cuda(lib):
    assert pp(lib, q=None) == 1
    assert pp(lib, pt=None) == 1
    assert pp(lib, seqlens=None) == 1
    assert pp(lib, B=-1) == 1
    assert pp(lib, scale=float("nan")) == 1
    assert pp(lib, d=96) == 2
    assert pp(lib, page_size=32) == 2
    assert pp(lib, max_pages=0) == 1
    assert pp(lib, num_pages=0) == 1
    assert pp(lib, Nq=300, max_pages=16) == 1  # the chunk cannot fit in 16 pages
    assert pp(lib, num_pages=(1 << 26) + 1) == 2
    assert pp(lib, kc=A + 0x1000008) == 3
    assert pp(lib, pt=A + 0x3100002) == 3
    assert pp(lib, o=A) == 1  # output aliasing q
    assert pp(lib, B=0) == 0 and pp(lib, Nq=0) == 0 and pp(lib, H=0) == 0


def dec(lib, q=A, kc=A + 0x1000000, vc=A + 0x2000000, seqlens=A + 0x3000000, pt=None,
        o=A + 0x4000000, lse=None, S=4, H=2, d=128, max_seqlen=1024, page_size=16, max_pages=64,
        num_pages=256, scale=0.1, ws=A + 0x5000000, ws_bytes=1 << 30):
    return lib.attn_decode(q, kc, vc, seqlens, pt, o, lse, S, H, d, max_seqlen, page_size, max_pages,
                           num_pages, scale, ws, ws_bytes, None)


def test_decode_workspace_size(lib):
    # splits of 256 tokens: per (sequence, split, head) d+1 floats, each part padded to 256 bytes
    size = lib.attn_decode_workspace_size(64, 32, 128, 8192)
    slots = 64 * 32 * 32
    assert size == ((slots * 128 * 4 + 255) // 256) * 256 + ((slots * 4 + 255) // 256) * 256
    assert lib.attn_decode_workspace_size(0, 32, 128, 8192) == 0
    assert lib.attn_decode_workspace_size(4, 32, 96, 8192) == 0
    assert lib.attn_decode_workspace_size(4, 32, 64, 1) > 0


def test_decode_rejects_bad_arguments_before_cuda(lib):
    assert dec(lib, q=None) == 1
    assert dec(lib, seqlens=None) == 1
    assert dec(lib, S=-1) == 1
    assert dec(lib, scale=0.0) == 1
    assert dec(lib, d=80) == 2
    assert dec(lib, pt=A + 0x6000000, page_size=32) == 2
    assert dec(lib, pt=A + 0x6000000, max_pages=0) == 1
    assert dec(lib, pt=A + 0x6000000, num_pages=0) == 1
    assert dec(lib, pt=A + 0x6000000, max_pages=8, max_seqlen=1024) == 1  # 8*16 < 1024
    assert dec(lib, kc=A + 0x1000004) == 3
    assert dec(lib, seqlens=A + 0x3000002) == 3
    assert dec(lib, ws=None) == 4
    assert dec(lib, ws_bytes=16) == 4
    assert dec(lib, ws=A + 0x5000008) == 3


def test_decode_fp8_rejects_bad_arguments_before_cuda(lib):
    def call(ks=A + 0x7000000, vs=A + 0x7100000, **kw):
        a = dict(q=A, kc=A + 0x1000000, vc=A + 0x2000000, seqlens=A + 0x3000000, pt=None,
                 o=A + 0x4000000, lse=None, S=4, H=2, d=128, max_seqlen=1024, page_size=16,
                 max_pages=64, num_pages=256, scale=0.1, ws=A + 0x5000000, ws_bytes=1 << 30)
        a.update(kw)
        return lib.attn_decode_fp8(a["q"], a["kc"], a["vc"], ks, vs, a["seqlens"], a["pt"], a["o"],
                                   a["lse"], a["S"], a["H"], a["d"], a["max_seqlen"], a["page_size"],
                                   a["max_pages"], a["num_pages"], a["scale"], a["ws"],
                                   a["ws_bytes"], None)
    assert call(ks=None) == 1
    assert call(vs=None) == 1
    assert call(ks=A + 0x7000002) == 3
    assert call(d=96) == 2
    assert call(ws=None) == 4
    assert call(S=0) == 0


def test_decode_empty_batch_is_a_no_op(lib):
    assert dec(lib, S=0) == 0
    assert dec(lib, H=0) == 0


def test_binding_refuses_to_import_without_library(tmp_path):
    """The Python binding raises instead of falling back when the library is missing."""
    import shutil
    import sys

    pkg_src = os.path.join(ROOT, "io_aware_attention_03_b300")
    pkg_dst = tmp_path / "io_aware_attention_03_b300"
    shutil.copytree(pkg_src, pkg_dst, ignore=shutil.ignore_patterns("*.so", "__pycache__"))
    code = ("import sys; sys.path.insert(0, %r)\n"
            "try:\n    import io_aware_attention_03_b300.attn\nexcept ImportError as e:\n"
            "    print('IMPORT_ERROR', e)\n" % str(tmp_path))
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert "IMPORT_ERROR" in out.stdout, out.stdout + out.stderr
