"""Pins for the fp64 CPU oracle, checked against what the pages and mathematics fix.

None of these re-types the oracle's formula: each compares it with an
independent algorithm (the online recurrence), a closed form, an invariant, a
special case with a known answer, a library routine, or the pages' own counts.

Sources:
* "FlashAttention complete summary" (cell-devlog), section "Attention이 뭔가":
  the formula softmax(QK^T/sqrt(d_k))V.
* same page, section "FlashAttention의 핵심 아이디어 — Tiling": blockwise
  processing with online softmax gives the exact result; section
  "FlashAttention 1": accuracy identical to standard attention (not approximate).
* "Flash Attention ... complete guide" (holysheep), section "Online Softmax
  알고리즘": m = max, f = exp(x - m), l = sum f, softmax = f / l; section
  "왜 Flash Attention이 필요한가?": N^2 attention weights.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
from io_aware_attention_03_b300.inputs import (bf16_bits, bf16_to_f32, decode_inputs,
                                               prefill_inputs, sample_rows)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f64(bits):
    return bf16_to_f32(bits).astype(np.float64)


def online_softmax_tiled(q, k, v, causal, scale, tile):
    """The online-softmax recurrence, keys visited in tiles of ``tile``.

    Independent of the oracle: it never materialises a score row and never
    runs a second pass.  Per tile: new max m', alpha = exp(m - m'),
    l <- alpha*l + sum exp(s - m'), acc <- alpha*acc + exp(s - m') V;
    finally O = acc / l and LSE = m + ln l.
    """
    Q, K, V = f64(q), f64(k), f64(v)
    B, N, H, d = Q.shape
    O = np.zeros_like(Q)
    LSE = np.zeros((B, H, N))
    for b in range(B):
        for h in range(H):
            for i in range(N):
                visible = i + 1 if causal else N
                m, l, acc = -math.inf, 0.0, np.zeros(d)
                for j0 in range(0, visible, tile):
                    j1 = min(j0 + tile, visible)
                    s = scale * (K[b, j0:j1, h, :] @ Q[b, i, h, :])
                    m_new = max(m, float(s.max()))
                    alpha = 0.0 if m == -math.inf else math.exp(m - m_new)
                    p = np.exp(s - m_new)
                    l = alpha * l + float(p.sum())
                    acc = alpha * acc + p @ V[b, j0:j1, h, :]
                    m = m_new
                O[b, i, h] = acc / l
                LSE[b, h, i] = m + math.log(l)
    return O, LSE


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("tile", [1, 3, 16, 128])
def test_online_tiled_recurrence_equals_oracle(causal, tile):
    q, k, v = prefill_inputs(11, 1, 2, 100, 64)
    scale = 1.0 / math.sqrt(64)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, scale)
    o_t, lse_t = online_softmax_tiled(q, k, v, causal, scale, tile)
    assert np.max(np.abs(o_t - o_ref)) <= 1e-12 * max(1.0, np.max(np.abs(o_ref)))
    assert np.max(np.abs(lse_t - lse_ref)) <= 1e-12 * max(1.0, np.max(np.abs(lse_ref)))


@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(causal):
    q, k, v = prefill_inputs(12, 2, 3, 70, 32)
    scale = 0.3
    P = oracle.attn_probs(q, k, causal, scale)
    assert P.shape == (2, 3, 70, 70)
    assert np.all(P >= 0.0)
    assert np.max(np.abs(P.sum(axis=-1) - 1.0)) <= 1e-12
    if causal:
        upper = np.triu(np.ones((70, 70), bool), k=1)
        assert np.all(P[..., upper] == 0.0)
        assert np.all(P[..., ~upper] > 0.0)
    # the forward's output is P applied to V (the aggregation step)
    o, _ = oracle.attn_fwd(q, k, v, causal, scale)
    o_from_p = np.einsum("bhij,bjhc->bihc", P, f64(v))
    assert np.max(np.abs(o - o_from_p)) <= 1e-12


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_values(causal):
    B, N, H, d = 1, 50, 2, 16
    q, _, v = prefill_inputs(13, B, H, N, d)
    k_row = prefill_inputs(14, 1, H, 1, d)[1]
    k = np.repeat(k_row, N, axis=1)  # every key identical (per head)
    scale = 0.25
    o, lse = oracle.attn_fwd(q, k, v, causal, scale)
    V = f64(v)
    for h in range(H):
        for i in range(N):
            n = i + 1 if causal else N
            assert np.max(np.abs(o[0, i, h] - V[0, :n, h].mean(axis=0))) <= 1e-12
            s = scale * float(f64(q)[0, i, h] @ f64(k_row)[0, 0, h])
            assert abs(lse[0, h, i] - (s + math.log(n))) <= 1e-12 * max(1.0, abs(s))


def test_single_key_returns_its_value():
    q, k, v = prefill_inputs(15, 2, 3, 1, 64)
    scale = 0.125
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal, scale)
        assert np.array_equal(o, f64(v))
        s = scale * np.einsum("bnhc,bnhc->bhn", f64(q), f64(k))
        assert np.max(np.abs(lse - s)) <= 1e-14 * max(1.0, np.max(np.abs(s)))


def test_causal_first_row_sees_only_first_key():
    q, k, v = prefill_inputs(16, 1, 2, 300, 64)
    o, _ = oracle.attn_fwd(q, k, v, True, 0.125)
    assert np.array_equal(o[:, 0], f64(v)[:, 0])
    # the last causal row sees every key, like the non-causal last row
    o_nc, _ = oracle.attn_fwd(q, k, v, False, 0.125)
    assert np.max(np.abs(o[:, -1] - o_nc[:, -1])) <= 1e-13


def test_dominant_key_returns_its_value():
    B, N, H, d = 1, 64, 1, 64
    q, k, v = prefill_inputs(17, B, H, N, d)
    q = q.copy()
    k = k.copy()
    i, jstar = 10, 37
    big = bf16_bits(np.float32(16.0))
    q[0, i, 0, :] = 0
    q[0, i, 0, 0] = big
    k[0, :, 0, 0] = 0  # no other key scores on component 0
    k[0, jstar, 0, 0] = big
    scale = 1.0 / 8.0
    # score of j*: 16*16/8 = 32; others: 0.  gap 32 -> weight e^-32 ~ 1.3e-14 each
    o, lse = oracle.attn_fwd(q, k, v, False, scale)
    assert np.max(np.abs(o[0, i, 0] - f64(v)[0, jstar, 0])) <= 64 * math.exp(-32) * 8
    assert abs(lse[0, 0, i] - 32.0) <= 1e-12


def test_permutation_invariance_non_causal():
    q, k, v = prefill_inputs(18, 2, 2, 90, 32)
    perm = np.random.Generator(np.random.PCG64(5)).permutation(90)
    o1, l1 = oracle.attn_fwd(q, k, v, False, 0.2)
    o2, l2 = oracle.attn_fwd(q, k[:, perm], v[:, perm], False, 0.2)
    assert np.max(np.abs(o1 - o2)) <= 1e-13
    assert np.max(np.abs(l1 - l2)) <= 1e-13


def test_common_score_shift_moves_only_lse():
    """Adding the same constant to every score of a row leaves O and shifts LSE.

    Built with an extra component: q_extra = 1 for every query and k_extra = c
    for every key, so each score gains scale*c.
    """
    q, k, v = prefill_inputs(19, 1, 2, 40, 16)
    q2, k2 = q.copy(), k.copy()
    c = 8.0
    q2[..., -1] = bf16_bits(np.float32(1.0))
    k2[..., -1] = bf16_bits(np.float32(c))
    q3, k3 = q2.copy(), k2.copy()
    k3[..., -1] = 0  # same problem without the shift
    scale = 0.5
    for causal in (False, True):
        o_a, l_a = oracle.attn_fwd(q2, k2, v, causal, scale)
        o_b, l_b = oracle.attn_fwd(q3, k3, v, causal, scale)
        assert np.max(np.abs(o_a - o_b)) <= 1e-12
        assert np.max(np.abs(l_a - (l_b + scale * c))) <= 1e-12


def test_two_key_closed_form():
    """d=2, scale 1: q=(1,0), keys (1,0),(0,1), values (1,2),(3,4).

    Scores (1, 0): P = (e/(e+1), 1/(e+1)), O = P0*(1,2) + P1*(3,4), LSE = ln(e+1).
    """
    one = bf16_bits(np.float32(1.0))
    q = np.zeros((1, 1, 1, 2), np.uint16)
    q[0, 0, 0, 0] = one
    k = np.zeros((1, 2, 1, 2), np.uint16)
    k[0, 0, 0, 0] = one
    k[0, 1, 0, 1] = one
    v = bf16_bits(np.array([1.0, 2.0, 3.0, 4.0], np.float32)).reshape(1, 2, 1, 2)
    o, lse = oracle.attn_fwd(q, k, v, False, 1.0)
    e = math.e
    p0, p1 = e / (e + 1.0), 1.0 / (e + 1.0)
    assert abs(o[0, 0, 0, 0] - (p0 * 1 + p1 * 3)) <= 1e-15
    assert abs(o[0, 0, 0, 1] - (p0 * 2 + p1 * 4)) <= 1e-15
    assert abs(lse[0, 0, 0] - math.log(e + 1.0)) <= 1e-15


def test_quadratic_weight_count_from_the_pages():
    with open(os.path.join(GOLDEN, "quadratic_weight_counts.json")) as f:
        golden = json.load(f)
    for case in golden["cases"]:
        n = case["tokens"]
        if n <= 4096:
            q, k, _ = prefill_inputs(20, 1, 1, n, 8)
            P = oracle.attn_probs(q, k, False, 0.3)
            count = P[0, 0].size
            assert count == n * n
            assert np.count_nonzero(P[0, 0]) == n * n
            Pc = oracle.attn_probs(q, k, True, 0.3)
            assert np.count_nonzero(Pc[0, 0]) == n * (n + 1) // 2
        else:
            count = n * n
        assert abs(count - case["page_value"]) <= case["rel_tol"] * count


@pytest.mark.parametrize("causal", [False, True])
def test_matches_library_sdpa_float64(causal):
    torch = pytest.importorskip("torch")
    q, k, v = prefill_inputs(21, 2, 3, 77, 64)
    scale = 1.0 / 8.0
    o, lse = oracle.attn_fwd(q, k, v, causal, scale)
    tq, tk, tv = (torch.from_numpy(f64(x)).permute(0, 2, 1, 3) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    ref = ref.permute(0, 2, 1, 3).numpy()
    assert np.max(np.abs(o - ref)) <= 1e-10
    # LSE against torch.logsumexp over the masked score matrix
    s = torch.einsum("bhic,bhjc->bhij", tq, tk) * scale
    if causal:
        s = s.masked_fill(torch.ones(77, 77, dtype=torch.bool).triu(1), float("-inf"))
    assert np.max(np.abs(lse - torch.logsumexp(s, dim=-1).numpy())) <= 1e-10


def test_bottom_right_causal_reading_for_rectangular():
    """Nq < Nk with causal keeps key j for query i iff j <= i + (Nk - Nq).

    The last Nq rows of a square causal problem equal the rectangular problem
    whose queries are those rows.
    """
    q, k, v = prefill_inputs(22, 1, 2, 64, 32)
    o_sq, l_sq = oracle.attn_fwd(q, k, v, True, 0.2)
    o_r, l_r = oracle.attn_fwd(np.ascontiguousarray(q[:, 40:]), k, v, True, 0.2)
    assert np.array_equal(o_r, o_sq[:, 40:])
    assert np.array_equal(l_r, l_sq[:, :, 40:])


def _small_decode(seed=30, num_seqs=5, H=3, d=32, lens=(1, 15, 16, 17, 70)):
    return decode_inputs(seed, num_seqs, H, d, 0, 0, page_size=16, seqlens=lens)


def test_decode_equals_single_query_prefill_row():
    di = _small_decode()
    kc, vc = di.contiguous_cache(di.k_tokens), di.contiguous_cache(di.v_tokens)
    o, lse = oracle.decode(di.q, kc, vc, di.seqlens, 0.17)
    for s in range(di.num_seqs):
        a, b = di.offsets[s], di.offsets[s + 1]
        kk = di.k_tokens[a:b][None]
        vv = di.v_tokens[a:b][None]
        o1, l1 = oracle.attn_fwd(di.q[s][None, None], kk, vv, False, 0.17)
        assert np.array_equal(o[s], o1[0, 0])
        assert np.array_equal(lse[s], l1[0, :, 0])


def test_decode_last_token_equals_causal_last_row():
    """Decoding the newest token over a cache of L keys equals row L-1 of causal prefill."""
    q, k, v = prefill_inputs(31, 1, 2, 48, 32)
    o_p, l_p = oracle.attn_fwd(q, k, v, True, 0.2)
    o_d, l_d = oracle.decode(np.ascontiguousarray(q[:, -1]), k, v, np.array([48], np.int32), 0.2)
    assert np.max(np.abs(o_d[0] - o_p[0, -1])) <= 1e-14
    assert np.max(np.abs(l_d[0] - l_p[0, :, -1])) <= 1e-14


def test_decode_paged_equals_contiguous_exactly():
    di = _small_decode()
    kc, vc = di.contiguous_cache(di.k_tokens), di.contiguous_cache(di.v_tokens)
    kp, vp = di.paged_pool(di.k_tokens), di.paged_pool(di.v_tokens)
    pt = di.page_table()
    # the page table is a permutation spread over the sequences
    used = np.sort(pt[pt >= 0])
    assert np.array_equal(used, np.arange(kp.shape[0]))
    o_c, l_c = oracle.decode(di.q, kc, vc, di.seqlens, 0.3)
    o_p, l_p = oracle.decode(di.q, kp, vp, di.seqlens, 0.3, page_table=pt, page_size=16)
    assert np.array_equal(o_c, o_p)
    assert np.array_equal(l_c, l_p)


def test_split_merge_identity():
    """Attention over keys [0, L) equals the LSE-weighted merge of [0, a) and [a, L):

    lse = ln(e^lse1 + e^lse2),  O = e^(lse1 - lse) O1 + e^(lse2 - lse) O2.
    """
    q, k, v = prefill_inputs(32, 1, 2, 1, 32)
    _, k, v = prefill_inputs(33, 1, 2, 200, 32)
    scale = 0.2
    o, lse = oracle.attn_fwd(q, k, v, False, scale)
    parts = []
    for a, b in ((0, 37), (37, 128), (128, 200)):
        parts.append(oracle.attn_fwd(q, np.ascontiguousarray(k[:, a:b]), np.ascontiguousarray(v[:, a:b]),
                                     False, scale))
    lses = np.stack([p[1] for p in parts])
    m = lses.max(axis=0)
    merged_lse = m + np.log(np.exp(lses - m).sum(axis=0))
    merged_o = sum(np.exp(p[1] - merged_lse)[:, :, :, None].transpose(0, 2, 1, 3) * p[0] for p in parts)
    assert np.max(np.abs(merged_lse - lse)) <= 1e-12
    assert np.max(np.abs(merged_o - o)) <= 1e-12


def test_rows_entry_matches_full():
    q, k, v = prefill_inputs(34, 2, 3, 130, 64)
    rows = np.array([[0, 0, 0], [1, 2, 129], [0, 1, 64], [1, 0, 127], [1, 1, 128]], np.int64)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal, 0.125)
        o_r, l_r = oracle.attn_rows(q, k, v, causal, 0.125, rows)
        for r, (b, h, i) in enumerate(rows):
            assert np.array_equal(o_r[r], o[b, i, h])
            assert l_r[r] == lse[b, h, i]


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, 1.0 + 2**-9, -2.5, 3.0e38], np.float32)
    bits = bf16_bits(x)
    back = bf16_to_f32(bits)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even (1); 1 + 3*2^-8 ties up to 1 + 2^-6
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == np.float32(1.0 + 2**-6)
    assert back[3] == 1.0 and back[4] == -2.5
    # every bf16 value round-trips
    allbits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = bf16_to_f32(allbits)
    finite = np.isfinite(vals)
    assert np.array_equal(bf16_bits(vals[finite]), allbits[finite])


# ---- chunked prefill against a paged cache ("Beyond the memory wall", section
# "FlashInfer": prefill and decode kernels over a paged K/V cache)

def _chunk_case(Nq=24, lens=(24, 25, 40, 70, 33), H=3, d=32, seed=40):
    from io_aware_attention_03_b300.inputs import chunk_queries

    di = decode_inputs(seed, len(lens), H, d, 0, 0, page_size=16, seqlens=lens)
    q = chunk_queries(seed + 1, len(lens), Nq, H, d)
    return di, q


@pytest.mark.parametrize("causal", [False, True])
def test_prefill_paged_gathers_the_right_keys(causal):
    """Through a shuffled page table, the paged prefill equals attn_fwd on each
    sequence's keys taken straight from its token arrays (no page table)."""
    di, q = _chunk_case()
    kp, vp = di.paged_pool(di.k_tokens), di.paged_pool(di.v_tokens)
    pt = di.page_table()
    assert not np.array_equal(np.sort(pt[pt >= 0]), pt[pt >= 0])  # the table really is shuffled
    o, lse = oracle.prefill_paged(q, kp, vp, di.seqlens, pt, causal, 0.21)
    for s in range(di.num_seqs):
        a, b = di.offsets[s], di.offsets[s + 1]
        o1, l1 = oracle.attn_fwd(q[s:s + 1], di.k_tokens[a:b][None], di.v_tokens[a:b][None],
                                 causal, 0.21)
        assert np.array_equal(o[s], o1[0])
        assert np.array_equal(lse[s], l1[0])


def test_prefill_paged_chunk_equals_last_rows_of_square_causal():
    """A chunk of the last Nq tokens over a cache of L keys gives the last Nq rows of
    the square causal problem over all L tokens (queries of the prefix drawn freely)."""
    Nq, L, H, d = 20, 57, 2, 32
    di, qc = _chunk_case(Nq=Nq, lens=(L,), H=H, d=d, seed=41)
    full_q, _, _ = prefill_inputs(42, 1, H, L, d)
    full_q = full_q.copy()
    full_q[0, L - Nq:] = qc[0]
    k, v = di.k_tokens[None], di.v_tokens[None]
    o_sq, l_sq = oracle.attn_fwd(full_q, k, v, True, 0.19)
    o_c, l_c = oracle.prefill_paged(qc, di.paged_pool(di.k_tokens), di.paged_pool(di.v_tokens),
                                    di.seqlens, di.page_table(), True, 0.19)
    assert np.array_equal(o_c[0], o_sq[0, L - Nq:])
    assert np.array_equal(l_c[0], l_sq[0, :, L - Nq:])


def test_prefill_paged_single_query_equals_decode():
    di, q = _chunk_case(Nq=1, lens=(1, 16, 17, 70), H=2, d=32, seed=43)
    kp, vp = di.paged_pool(di.k_tokens), di.paged_pool(di.v_tokens)
    pt = di.page_table()
    for causal in (False, True):
        o, lse = oracle.prefill_paged(q, kp, vp, di.seqlens, pt, causal, 0.23)
        o_d, l_d = oracle.decode(q[:, 0], kp, vp, di.seqlens, 0.23, page_table=pt, page_size=16)
        assert np.max(np.abs(o[:, 0] - o_d)) <= 1e-14
        assert np.max(np.abs(lse[:, :, 0] - l_d)) <= 1e-14


# ---- FP8 (E4M3) K/V cache for decode ("Beyond the memory wall", section
# "FlashInfer": quantized K/V among the cache options)

def test_e4m3_decoding_of_known_codes():
    """Values fixed by the E4M3 format: bias 7, 3 mantissa bits, subnormals below
    2^-6, largest finite 448, S.1111.111 is NaN, no infinities."""
    v = oracle.e4m3_value(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x39, 0x7E, 0xFE, 0xB8, 0x80],
                                   np.uint8))
    assert v.tolist() == [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.125, 448.0, -448.0,
                          -1.0, 0.0]
    assert np.isnan(oracle.e4m3_value(np.array([0x7F, 0xFF], np.uint8))).all()
    pos = oracle.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)                         # codes 0..126 strictly increasing
    assert len(set(oracle.e4m3_value(np.arange(256, dtype=np.uint8)).tolist()) - {np.nan}) >= 253


def test_e4m3_encoder_round_trip_and_rounding():
    from io_aware_attention_03_b300.inputs import e4m3_bits

    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_value(codes)
    assert np.array_equal(e4m3_bits(vals.astype(np.float32)), codes)
    # nearest-even rounding: within half a quantum, ties to an even mantissa
    g = np.random.Generator(np.random.PCG64(5))
    x = (g.standard_normal(20000) * 30).astype(np.float32)
    y = oracle.e4m3_value(e4m3_bits(x))
    a = np.minimum(np.abs(x.astype(np.float64)), 448.0)
    quantum = 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -6))) - 3)
    assert np.all(np.abs(np.abs(y) - a) <= quantum / 2)
    ties = oracle.e4m3_value(e4m3_bits(np.array([1.0625, 1.1875, 2.0 ** -10], np.float32)))
    assert ties.tolist() == [1.0, 1.25, 0.0]


@pytest.mark.parametrize("paged", [False, True])
def test_decode_over_values_equals_bf16_decode(paged):
    """decode_values fed the bf16 caches' exact values equals the C decode."""
    di = _small_decode()
    if paged:
        kb, vb = di.paged_pool(di.k_tokens), di.paged_pool(di.v_tokens)
        pt = di.page_table()
    else:
        kb, vb = di.contiguous_cache(di.k_tokens), di.contiguous_cache(di.v_tokens)
        pt = None
    o_c, l_c = oracle.decode(di.q, kb, vb, di.seqlens, 0.3, page_table=pt, page_size=16)
    o_v, l_v = oracle.decode_values(di.q, f64(kb), f64(vb), di.seqlens, 0.3, page_table=pt)
    assert np.max(np.abs(o_c - o_v)) <= 1e-12
    assert np.max(np.abs(l_c - l_v)) <= 1e-12


def test_fp8_decode_single_key_closed_form():
    """One cached token: O = v_scale[h] * e4m3(v), LSE = scale * q . (k_scale[h] * e4m3(k))."""
    H, d = 3, 16
    g = np.random.Generator(np.random.PCG64(9))
    q = bf16_bits(g.standard_normal((1, H, d)).astype(np.float32))
    k8 = g.integers(0, 0x7F, size=(1, 1, H, d)).astype(np.uint8)
    v8 = g.integers(0x80, 0xFF, size=(1, 1, H, d)).astype(np.uint8)
    ks = np.array([0.5, 0.03125, 2.0], np.float32)
    vs = np.array([0.25, 4.0, 0.0078125], np.float32)
    o, lse = oracle.decode_fp8(q, k8, v8, ks, vs, np.array([1], np.int32), 0.7)
    kv = oracle.e4m3_value(k8[0, 0]) * ks[:, None]
    vv = oracle.e4m3_value(v8[0, 0]) * vs[:, None]
    assert np.array_equal(o[0], vv)
    assert np.max(np.abs(lse[0] - 0.7 * (f64(q[0]) * kv).sum(axis=1))) <= 1e-12


def _e4m3_tokens(g, shape):
    """Random E4M3 codes without the two NaN codes (0x7F, 0xFF)."""
    b = g.integers(0, 256, size=shape).astype(np.uint8)
    return np.where((b & 0x7F) == 0x7F, b ^ 0x01, b).astype(np.uint8)


def test_fp8_decode_paged_equals_contiguous_exactly():
    """The paged gather of decode_fp8 reads the same tokens as the contiguous layout: a cache
    scattered into 16-token pages in shuffled order (scattered here, token by token) gives
    bit-identical O and LSE, ragged lengths included ("Beyond the memory wall", section
    "FlashInfer": decode against a paged K/V cache)."""
    g = np.random.Generator(np.random.PCG64(31))
    S, H, d, Lmax, P = 3, 2, 16, 50, 16
    lens = np.array([50, 17, 1], np.int32)
    kt, vt = _e4m3_tokens(g, (S, Lmax, H, d)), _e4m3_tokens(g, (S, Lmax, H, d))
    q = bf16_bits(g.standard_normal((S, H, d)).astype(np.float32))
    ks = np.array([0.5, 0.0625], np.float32)
    vs = np.array([2.0, 0.125], np.float32)
    npages = [(int(L) + P - 1) // P for L in lens]
    perm = g.permutation(sum(npages))
    table = np.zeros((S, max(npages)), np.int32)
    kpool = np.zeros((sum(npages), P, H, d), np.uint8)
    vpool = np.zeros_like(kpool)
    nxt = 0
    for s in range(S):
        for j in range(npages[s]):
            table[s, j] = perm[nxt]
            nxt += 1
        for t in range(int(lens[s])):
            kpool[table[s, t // P], t % P] = kt[s, t]
            vpool[table[s, t // P], t % P] = vt[s, t]
    o_c, l_c = oracle.decode_fp8(q, kt, vt, ks, vs, lens, 0.4)
    o_p, l_p = oracle.decode_fp8(q, kpool, vpool, ks, vs, lens, 0.4, page_table=table, page_size=P)
    assert np.array_equal(o_c, o_p) and np.array_equal(l_c, l_p)


def test_fp8_decode_identical_keys_give_mean_of_values():
    """Every cached key of a sequence equal: P is uniform over its L tokens, so O is the mean
    of the dequantized values and LSE = scale * q . k + ln L ("Flash Attention ... complete
    guide", section "Online Softmax 알고리즘": softmax = f / l)."""
    g = np.random.Generator(np.random.PCG64(32))
    S, H, d, Lmax = 2, 2, 8, 40
    lens = np.array([40, 7], np.int32)
    k1 = _e4m3_tokens(g, (S, 1, H, d))
    kt = np.repeat(k1, Lmax, axis=1)
    vt = _e4m3_tokens(g, (S, Lmax, H, d))
    q = bf16_bits(g.standard_normal((S, H, d)).astype(np.float32))
    ks = np.array([0.25, 1.5], np.float32)
    vs = np.array([0.5, 3.0], np.float32)
    o, lse = oracle.decode_fp8(q, kt, vt, ks, vs, lens, 0.6)
    for s in range(S):
        L = int(lens[s])
        vv = oracle.e4m3_value(vt[s, :L]) * vs.astype(np.float64)[None, :, None]   # [L, H, d]
        assert np.max(np.abs(o[s] - vv.mean(axis=0))) <= 1e-12
        kv = oracle.e4m3_value(k1[s, 0]) * ks.astype(np.float64)[:, None]          # [H, d]
        expect = 0.6 * (f64(q[s]) * kv).sum(axis=1) + math.log(L)
        assert np.max(np.abs(lse[s] - expect)) <= 1e-12


def test_fp8_decode_key_scale_acts_as_softmax_scale():
    """k_scale multiplies every score of its head: scaling it by c equals scaling the softmax
    scale by c, and v_scale scales O linearly while leaving LSE unchanged."""
    g = np.random.Generator(np.random.PCG64(33))
    S, H, d, Lmax = 2, 2, 8, 30
    lens = np.array([30, 11], np.int32)
    kt, vt = _e4m3_tokens(g, (S, Lmax, H, d)), _e4m3_tokens(g, (S, Lmax, H, d))
    q = bf16_bits(g.standard_normal((S, H, d)).astype(np.float32))
    ks = np.array([0.125, 0.125], np.float32)
    vs = np.array([1.0, 1.0], np.float32)
    o1, l1 = oracle.decode_fp8(q, kt, vt, ks * 4, vs, lens, 0.3)
    o2, l2 = oracle.decode_fp8(q, kt, vt, ks, vs, lens, 1.2)
    assert np.max(np.abs(o1 - o2)) <= 1e-12 and np.max(np.abs(l1 - l2)) <= 1e-12
    o3, l3 = oracle.decode_fp8(q, kt, vt, ks, vs * np.array([2.0, 0.5], np.float32), lens, 1.2)
    assert np.max(np.abs(o3 - o2 * np.array([2.0, 0.5])[None, :, None])) <= 1e-12
    assert np.array_equal(l3, l2)


# ---- Real-valued oracle and FP8 (E4M3) prefill ("FlashAttention complete summary",
# section "FlashAttention 3"; "Beyond the memory wall", section "FlashAttention-3가 다른
# 이유": FP8 forward)

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("nq_nk", [(70, 70), (33, 90), (1, 5)])
def test_values_oracle_equals_bf16_oracle(causal, nq_nk):
    """attn_fwd_values (numpy, row blocks of 7) fed the exact values of bf16 inputs equals
    the C oracle; rectangular shapes use the bottom-right causal alignment of both."""
    Nq, Nk = nq_nk
    q, _, _ = prefill_inputs(31, 2, 3, Nq, 64)
    _, k, v = prefill_inputs(32, 2, 3, Nk, 64)
    o_c, l_c = oracle.attn_fwd(q, k, v, causal, 0.17)
    o_v, l_v = oracle.attn_fwd_values(f64(q), f64(k), f64(v), causal, 0.17, rows_per_block=7)
    assert np.max(np.abs(o_c - o_v)) <= 1e-12
    assert np.max(np.abs(l_c - l_v)) <= 1e-12


def test_values_oracle_row_max_brackets_lse():
    """LSE - m = ln sum_j exp(s_j - m) lies in [0, ln n]: the max term alone gives 1, n
    terms give at most n; identical keys reach ln n exactly."""
    q, k, v = prefill_inputs(33, 1, 2, 96, 64)
    for causal in (False, True):
        _, lse, m = oracle.attn_fwd_values(f64(q), f64(k), f64(v), causal, 0.2, return_max=True)
        n = (np.arange(96) + 1.0) if causal else np.full(96, 96.0)
        assert np.all(lse - m >= -1e-14) and np.all(lse - m <= np.log(n)[None, None, :] + 1e-12)
    kk = np.repeat(f64(k)[:, :1], 96, axis=1)
    _, lse, m = oracle.attn_fwd_values(f64(q), kk, f64(v), True, 0.2, return_max=True)
    assert np.max(np.abs((lse - m) - np.log(np.arange(96) + 1.0)[None, None, :])) <= 1e-12


def test_values_rows_match_full():
    q, k, v = prefill_inputs(34, 2, 2, 150, 64)
    rows = sample_rows(3, 2, 2, 150, 40)
    for causal in (False, True):
        o, lse = oracle.attn_fwd_values(f64(q), f64(k), f64(v), causal, 0.3)
        o_r, l_r = oracle.attn_rows_values(f64(q), f64(k), f64(v), causal, 0.3, rows)
        b, h, i = rows.T
        assert np.array_equal(o_r, o[b, i, h]) and np.array_equal(l_r, lse[b, h, i])


@pytest.mark.parametrize("causal", [False, True])
def test_values_oracle_matches_library_sdpa_float64(causal):
    """Generic fp64 inputs (not bf16-representable): torch SDPA in float64 agrees."""
    torch = pytest.importorskip("torch")
    g = np.random.Generator(np.random.PCG64(35))
    q, k, v = (g.standard_normal((2, 40, 3, 32)) for _ in range(3))
    o, lse = oracle.attn_fwd_values(q, k, v, causal, 0.4)
    tq, tk, tv = (torch.from_numpy(x).permute(0, 2, 1, 3) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=0.4)
    assert np.max(np.abs(o - ref.permute(0, 2, 1, 3).numpy())) <= 1e-12
    s = 0.4 * torch.einsum("bhid,bhjd->bhij", tq, tk)
    if causal:
        s = s.masked_fill(torch.ones(40, 40, dtype=torch.bool).triu(1), -math.inf)
    assert np.max(np.abs(lse - torch.logsumexp(s, dim=-1).numpy())) <= 1e-12


def test_fp8_prefill_equals_bf16_oracle_on_dequantized_values():
    """With power-of-two scales every dequantized value scale[h] * e4m3 is a bf16 number, so
    the FP8 oracle must equal the C oracle fed those bf16 numbers."""
    from io_aware_attention_03_b300.inputs import fp8_prefill_inputs

    f8 = fp8_prefill_inputs(36, 1, 3, 77, 128, q_factor=4.0)
    deq = [oracle.dequantize_e4m3(x, s) for x, s in
           ((f8.q, f8.q_scale), (f8.k, f8.k_scale), (f8.v, f8.v_scale))]
    as_bf16 = [bf16_bits(x.astype(np.float32)) for x in deq]
    for x, b in zip(deq, as_bf16):
        assert np.array_equal(f64(b), x)                       # exactly representable
    for causal in (False, True):
        o8, l8 = oracle.attn_fwd_fp8(f8.q, f8.k, f8.v, f8.q_scale, f8.k_scale, f8.v_scale, causal,
                                     0.09)
        o, lse = oracle.attn_fwd(*as_bf16, causal, 0.09)
        assert np.max(np.abs(o8 - o)) <= 1e-12 and np.max(np.abs(l8 - lse)) <= 1e-12


def test_fp8_prefill_single_key_closed_form():
    """N = 1: O = v_scale[h] * e4m3(v), LSE = scale * (q_scale[h] e4m3(q)) . (k_scale[h] e4m3(k))."""
    g = np.random.Generator(np.random.PCG64(37))
    q8, k8, v8 = (g.integers(0, 0xFF, size=(1, 1, 2, 128)).astype(np.uint8) for _ in range(3))
    for x in (q8, k8, v8):
        x[(x & 0x7F) == 0x7F] = 0x3C                           # no NaN codes
    qs, ks, vs = (np.array(s, np.float32) for s in ([0.5, 0.01], [2.0, 0.3], [0.125, 7.0]))
    o, lse = oracle.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, True, 0.05)
    qv = oracle.e4m3_value(q8[0, 0]) * qs.astype(np.float64)[:, None]
    kv = oracle.e4m3_value(k8[0, 0]) * ks.astype(np.float64)[:, None]
    vv = oracle.e4m3_value(v8[0, 0]) * vs.astype(np.float64)[:, None]
    assert np.array_equal(o[0, 0], vv)
    assert np.max(np.abs(lse[0, :, 0] - 0.05 * (qv * kv).sum(axis=1))) <= 1e-12


def test_fp8_tolerance_second_moment_identity():
    """The FP8 tolerance's sum_j p_j^2 v_j^2, taken from attention at twice the scale, equals
    the same sum formed from the C oracle's probability matrix."""
    import fp8_tolerance

    q, k, v = prefill_inputs(38, 1, 2, 50, 64)
    for causal in (False, True):
        P = oracle.attn_probs(q, k, causal, 0.25)[0]            # [H, N, N]
        vv = f64(v)[0]                                           # [N, H, d]
        direct = np.einsum("hij,jhc->ihc", P * P, vv * vv)
        o, lse = oracle.attn_fwd_values(f64(q), f64(k), f64(v), causal, 0.25)
        o2, lse2 = oracle.attn_fwd_values(f64(q), f64(k), f64(v) ** 2, causal, 0.5)
        via = o2[0] * np.exp(lse2[0] - 2.0 * lse[0]).T[:, :, None]
        assert np.max(np.abs(direct - via)) <= 1e-12
        assert fp8_tolerance.LSE_MAX == 1e-3


# ---- Backward with recomputation ("Beyond the memory wall", section "FlashAttention:
# IO 인식의 정점": tiling and recomputation; FlashAttention as the training standard)

def _loss(q, k, v, do, causal, scale):
    """L = sum(O * dO) with O from the (separately pinned) forward oracle."""
    o, _ = oracle.attn_fwd_values(q[None, :, None], k[None, :, None], v[None, :, None], causal, scale)
    return float((o[0, :, 0] * do).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences_of_the_forward(causal):
    """Central differences of L = sum(O * dO) through the forward oracle (step 1e-5, error
    O(h^2)) agree with the analytic gradients to 1e-7."""
    g = np.random.Generator(np.random.PCG64(40))
    N, d, scale = 6, 5, 0.7
    q, k, v, do = (g.standard_normal((N, d)) for _ in range(4))
    grads = oracle.attn_bwd_head(q, k, v, do, causal, scale)
    h = 1e-5
    for name, x in (("dq", q), ("dk", k), ("dv", v)):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = [xp if y is x else y for y in (q, k, v)]
            args_m = [xm if y is x else y for y in (q, k, v)]
            num[idx] = (_loss(*args_p, do, causal, scale) - _loss(*args_m, do, causal, scale)) / (2 * h)
        assert np.max(np.abs(num - grads[name])) <= 1e-7, name


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd_float64(causal):
    torch = pytest.importorskip("torch")
    g = np.random.Generator(np.random.PCG64(41))
    N, d, scale = 33, 16, 0.3
    q, k, v, do = (g.standard_normal((N, d)) for _ in range(4))
    grads = oracle.attn_bwd_head(q, k, v, do, causal, scale)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq[None], tk[None], tv[None],
                                                         is_causal=causal, scale=scale)[0]
    o.backward(torch.tensor(do))
    for name, t in (("dq", tq), ("dk", tk), ("dv", tv)):
        assert np.max(np.abs(t.grad.numpy() - grads[name])) <= 1e-12, name


def test_backward_invariants():
    """Rows of dS sum to zero (softmax is shift-invariant), so sum_j dK_j = 0; rows of P sum
    to one, so sum_j dV_j = sum_i dO_i; D_i = dO_i . O_i."""
    g = np.random.Generator(np.random.PCG64(42))
    q, k, v, do = (g.standard_normal((40, 8)) for _ in range(4))
    for causal in (False, True):
        r = oracle.attn_bwd_head(q, k, v, do, causal, 0.5)
        assert np.max(np.abs(r["ds"].sum(axis=1))) <= 1e-12
        assert np.max(np.abs(r["dk"].sum(axis=0))) <= 1e-12
        assert np.max(np.abs(r["dv"].sum(axis=0) - do.sum(axis=0))) <= 1e-12
        assert np.max(np.abs(r["D"] - (do * r["o"]).sum(axis=1))) <= 1e-12


def test_backward_special_cases():
    """N = 1: the softmax is constant, so dQ = dK = 0 and dV = dO.  Identical keys: P is
    uniform whatever Q is, so dQ = 0 (and causal row 0 always has dQ = 0)."""
    g = np.random.Generator(np.random.PCG64(43))
    q, k, v, do = (g.standard_normal((1, 8)) for _ in range(4))
    r = oracle.attn_bwd_head(q, k, v, do, False, 0.4)
    assert np.array_equal(r["dq"], np.zeros_like(q)) and np.array_equal(r["dk"], np.zeros_like(k))
    assert np.array_equal(r["dv"], do)
    q, v, do = (g.standard_normal((20, 8)) for _ in range(3))
    k = np.repeat(g.standard_normal((1, 8)), 20, axis=0)
    for causal in (False, True):
        r = oracle.attn_bwd_head(q, k, v, do, causal, 0.4)
        assert np.max(np.abs(r["dq"])) <= 1e-12
    r = oracle.attn_bwd_head(g.standard_normal((20, 8)), g.standard_normal((20, 8)), v, do, True, 0.4)
    assert np.max(np.abs(r["dq"][0])) <= 1e-15


def test_backward_on_bf16_inputs_uses_the_head_definition():
    """attn_bwd (bf16 bits, all heads or a subset) equals attn_bwd_head per head."""
    from io_aware_attention_03_b300.inputs import backward_inputs

    q, k, v, do = backward_inputs(44, 2, 3, 50, 16)
    dq, dk, dv = oracle.attn_bwd(q, k, v, do, True, 0.25)
    r = oracle.attn_bwd_head(f64(q[1, :, 2]), f64(k[1, :, 2]), f64(v[1, :, 2]), f64(do[1, :, 2]),
                             True, 0.25)
    assert np.array_equal(dq[1, :, 2], r["dq"]) and np.array_equal(dk[1, :, 2], r["dk"])
    assert np.array_equal(dv[1, :, 2], r["dv"])
    dq1, _, _ = oracle.attn_bwd(q, k, v, do, True, 0.25, heads=[(0, 1)])
    assert np.array_equal(dq1[0, :, 1], dq[0, :, 1]) and np.isnan(dq1[1]).all()
