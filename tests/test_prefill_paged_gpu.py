"""Chunked prefill against a 16-token paged K/V cache: the CUDA path (through the
C ABI) against the fp64 CPU oracle.

A chunk of Nq query tokens per sequence attends to every cached key of its
sequence, the chunk's own included, with the causal mask aligned to the end of
the cache ("Beyond the memory wall", section "FlashInfer": prefill and decode
kernels over a paged cache).  Tolerances as for attn_fwd: O max-abs <= 2e-2,
mean-abs <= 2e-3, LSE within 1e-3.
"""

import math

import numpy as np
import pytest

import oracle
from io_aware_attention_03_b300.inputs import (CHUNKED, chunk_queries, decode_inputs,
                                               prefill_inputs, sample_rows)

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module")
def dev():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from io_aware_attention_03_b300 import attn, device_inputs

    return torch, attn, device_inputs


def run_paged(dev, di, qc, causal, scale):
    torch, attn, dvi = dev
    _, kp, vp, seqlens, pt = dvi.decode_device_inputs(di, paged=True)
    q = dvi.to_device_bf16(qc)
    o, lse = attn.attn_prefill_paged(q, kp, vp, seqlens, pt, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o, lse, attn.attn_last_device_status()


def check(o, lse, o_ref, lse_ref, what):
    err = np.abs(o - o_ref)
    assert np.all(np.isfinite(o)), what
    assert err.max() <= O_MAX, f"{what} O max-abs {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"{what} O mean-abs {err.mean():.3e}"
    assert np.abs(lse - lse_ref).max() <= LSE_MAX, f"{what} LSE"


CASES = [  # (Nq, cache lengths incl. the chunk, d)
    (1, (1, 2, 17, 300), 128),
    (37, (37, 38, 100, 200, 1000), 64),
    (128, (128, 129, 256, 640), 128),
    (200, (200, 255, 256, 1111), 64),
    (256, (256, 300, 2048), 128),
    (300, (300, 301, 777, 1500), 128),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"Nq{c[0]}-d{c[2]}")
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_prefix_lengths_full_output(dev, case, causal):
    torch, attn, dvi = dev
    Nq, lens, d = case
    H = 3
    di = decode_inputs(500 + Nq + d, len(lens), H, d, 0, 0, seqlens=lens)
    qc = chunk_queries(600 + Nq + d, len(lens), Nq, H, d)
    scale = float(np.float32(1.0 / math.sqrt(d)))
    o, lse, status = run_paged(dev, di, qc, causal, scale)
    assert status == 0
    kp, vp = di.paged_pool(di.k_tokens), di.paged_pool(di.v_tokens)
    o_ref, lse_ref = oracle.prefill_paged(qc, kp, vp, di.seqlens, di.page_table(), causal, scale)
    check(dvi.to_host_f64(o), dvi.to_host_f64(lse), o_ref, lse_ref, f"Nq={Nq} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_no_prefix_in_page_order_equals_attn_fwd_bitwise(dev, causal):
    """With the whole sequence in the chunk and pages in order, the paged kernel
    reads the same tiles as attn_fwd and must give the same bits."""
    torch, attn, dvi = dev
    B, H, N, d = 2, 4, 640, 128
    q, k, v = prefill_inputs(71, B, H, N, d)
    tq, tk, tv = (dvi.to_device_bf16(x) for x in (q, k, v))
    o_ref, l_ref = attn.attn_fwd(tq, tk, tv, causal=causal)
    pages = N // 16
    kp = tk.view(B * pages, 16, H, d)
    vp = tv.view(B * pages, 16, H, d)
    pt = torch.arange(B * pages, dtype=torch.int32, device="cuda").view(B, pages)
    seqlens = torch.full((B,), N, dtype=torch.int32, device="cuda")
    o, l = attn.attn_prefill_paged(tq, kp, vp, seqlens, pt, causal=causal)
    torch.cuda.synchronize()
    assert attn.attn_last_device_status() == 0
    assert torch.equal(o, o_ref) and torch.equal(l, l_ref)


def test_chunked_workload_sampled(dev):
    """16 sequences ~ U[1024, 8192] tokens, a 512-token chunk each, H=32, d=128, causal."""
    torch, attn, dvi = dev
    c = CHUNKED
    di = decode_inputs(c["seed"], c["num_seqs"], c["H"], c["d"], c["len_lo"], c["len_hi"],
                       page_size=c["page_size"])
    qc = chunk_queries(c["q_seed"], c["num_seqs"], c["Nq"], c["H"], c["d"])
    scale = float(np.float32(1.0 / math.sqrt(c["d"])))
    o, lse, status = run_paged(dev, di, qc, True, scale)
    assert status == 0
    o, lse = dvi.to_host_f64(o), dvi.to_host_f64(lse)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    rows = sample_rows(c["seed"] + 7, c["num_seqs"], c["H"], c["Nq"], 256)
    kp, vp = di.paged_pool(di.k_tokens), di.paged_pool(di.v_tokens)
    pt = di.page_table()
    for b in np.unique(rows[:, 0]):
        sel = rows[rows[:, 0] == b]
        o_ref, lse_ref = oracle.prefill_paged(qc[b:b + 1], kp, vp, di.seqlens[b:b + 1], pt[b:b + 1],
                                              True, scale)
        h, i = sel[:, 1], sel[:, 2]
        check(o[b, i, h], lse[b, h, i], o_ref[0, i, h], lse_ref[0, h, i], f"seq {b}")


def test_bad_page_ids_and_lengths_are_recorded_not_faulted(dev):
    torch, attn, dvi = dev
    di = decode_inputs(77, 3, 2, 64, 0, 0, seqlens=(40, 100, 64))
    _, kp, vp, seqlens, pt = dvi.decode_device_inputs(di, paged=True)
    q = dvi.to_device_bf16(chunk_queries(78, 3, 32, 2, 64))
    bad = pt.clone()
    bad[1, 2] = 10_000_000
    attn.attn_prefill_paged(q, kp, vp, seqlens, bad, causal=True)
    torch.cuda.synchronize()
    assert attn.attn_last_device_status() == 1  # ATTN_ERR_INVALID_ARG
    short = seqlens.clone()
    short[0] = 5  # fewer keys than the 32-token chunk
    attn.attn_prefill_paged(q, kp, vp, short, pt, causal=True)
    torch.cuda.synchronize()
    assert attn.attn_last_device_status() == 1
    o, _ = attn.attn_prefill_paged(q, kp, vp, seqlens, pt, causal=True)
    torch.cuda.synchronize()
    assert attn.attn_last_device_status() == 0
    assert bool(torch.isfinite(o.float()).all())


def test_empty_chunk(dev):
    torch, attn, dvi = dev
    z = torch.empty((2, 0, 4, 64), dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros((4, 16, 4, 64), dtype=torch.bfloat16, device="cuda")
    sl = torch.zeros(2, dtype=torch.int32, device="cuda")
    pt = torch.zeros((2, 2), dtype=torch.int32, device="cuda")
    o, lse = attn.attn_prefill_paged(z, pool, pool, sl, pt)
    assert o.shape == z.shape and lse.shape == (2, 4, 0)
