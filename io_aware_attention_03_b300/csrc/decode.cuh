// Split-KV decode attention for sm_103a: one query token per sequence against
// a contiguous or 16-token paged K/V cache.
//
// What it computes: the attention row of the newest token over the whole cache
// ("Beyond the memory wall" (tiptinker), section "FlashInfer": in decode a
// single query meets an ever-growing K/V cache, optionally paged).  The cache
// of each sequence is cut into splits of kSplitTokens tokens; each split is
// reduced with its own exact softmax (max, sum of exp, weighted sum of V) into
// a partial output O_s and its log-sum-exp lse_s, and a second kernel merges
// the splits exactly:  lse = ln sum_s e^{lse_s},  O = sum_s e^{lse_s - lse} O_s
// (the same rescaling the online softmax applies between key blocks).
//
// How it maps onto the B300: decode reads every cached byte once and does ~1
// FLOP per byte, so it is bound by HBM bandwidth.  A warp owns one (sequence,
// split, head); lanes split the head dimension into 16-byte pieces (8 bf16) so
// each token-head row (d*2 bytes, contiguous) is fetched with coalesced 128-bit
// loads, several tokens in flight per lane.  Contiguous and paged caches share
// the same arithmetic in the same order, so their results are bit-identical.
// An FP8 (e4m3) cache with per-head scales halves the bytes per token: e4m3
// values convert exactly to f16 and enter mixed-precision FMAs (fp32
// accumulation); for the scores two lanes cover a token's row, half each.  The
// key scale multiplies the scores and the value scale the partial output.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace attn {

constexpr int kSplitTokens = 256;   // tokens per split (a multiple of the 16-token page)
constexpr int kDecodeHeadsPerCta = 4;
constexpr int kPageSize = 16;

struct DecodeParams {
    const __nv_bfloat16* q;
    const void* kc;          // bf16, or fp8 e4m3 with a per-head scale
    const void* vc;
    const float* k_scale;    // fp8 caches: key j of head h is k_scale[h] * kc[..]
    const float* v_scale;
    const int* seqlens;
    const int* page_table;   // nullptr: contiguous cache
    __nv_bfloat16* o;
    float* lse;
    float* ws_o;     // [S, max_splits, H, D]
    float* ws_lse;   // [S, max_splits, H]
    int S, H, max_seqlen, max_pages, num_pages, max_splits;
    float scale_log2;
};

// Number of valid tokens of sequence s, clamped to [0, max_seqlen]; an
// out-of-range length is recorded in the device status word.
__device__ __forceinline__ int decode_seqlen(const DecodeParams& p, int s) {
    int L = __ldg(p.seqlens + s);
    if (L < 0 || L > p.max_seqlen) {
        record_status(ATTN_ERR_INVALID_ARG);
        L = min(max(L, 0), p.max_seqlen);
    }
    return L;
}

// Row index (into [rows, H, D]) of token t of sequence s, or -1 for an invalid page id.
template <bool PAGED>
__device__ __forceinline__ long long token_row(const DecodeParams& p, int s, int t) {
    if constexpr (PAGED) {
        const int pg = __ldg(p.page_table + (size_t)s * p.max_pages + t / kPageSize);
        if (pg < 0 || pg >= p.num_pages) {
            record_status(ATTN_ERR_INVALID_ARG);
            return -1;
        }
        return (long long)pg * kPageSize + (t % kPageSize);
    } else {
        return (long long)s * p.max_seqlen + t;
    }
}

// Two e4m3 values (low byte first) -> fp32; e4m3 -> fp16 is exact.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two_bytes) {
    uint32_t h2;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
        : "=r"(h2)
        : "r"(two_bytes));
    return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}

// 16 e4m3 values (one 16-byte load) -> fp32, in memory order.
__device__ __forceinline__ void e4m3x16_to_f32(const uint4& u, float (&f)[16]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 a = e4m3x2_to_f32x2(w[i] & 0xFFFFu);
        const float2 b = e4m3x2_to_f32x2(w[i] >> 16);
        f[4 * i] = a.x;
        f[4 * i + 1] = a.y;
        f[4 * i + 2] = b.x;
        f[4 * i + 3] = b.y;
    }
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// FP8 path, arithmetic on half-precision operands with fp32 accumulation (one
// mixed-precision FMA per element, no conversion to fp32): e4m3 -> f16 is exact,
// and so is a product of an f16 and an e4m3 value in fp32.
//
// acc + sum_e q[e] * k[e] over the 16 e4m3 values of one 16-byte load, q as eight
// f16x2 words in the same order (two interleaved chains).
__device__ __forceinline__ float dot16_e4m3_f16(const uint4& u, const uint32_t (&q2)[8], float acc) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    float a0 = acc, a1 = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        asm("{\n\t.reg .b16 lo, hi, k0, k1, k2, k3, q0, q1, q2, q3;\n\t.reg .b32 kk01, kk23;\n\t"
            "mov.b32 {lo, hi}, %2;\n\t"
            "cvt.rn.f16x2.e4m3x2 kk01, lo;\n\tcvt.rn.f16x2.e4m3x2 kk23, hi;\n\t"
            "mov.b32 {k0, k1}, kk01;\n\tmov.b32 {k2, k3}, kk23;\n\t"
            "mov.b32 {q0, q1}, %3;\n\tmov.b32 {q2, q3}, %4;\n\t"
            "fma.rn.f32.f16 %0, q0, k0, %0;\n\tfma.rn.f32.f16 %1, q1, k1, %1;\n\t"
            "fma.rn.f32.f16 %0, q2, k2, %0;\n\tfma.rn.f32.f16 %1, q3, k3, %1;\n\t}"
            : "+f"(a0), "+f"(a1)
            : "r"(w[i]), "r"(q2[2 * i]), "r"(q2[2 * i + 1]));
    }
    return a0 + a1;
}

// acc[e] += p * v[e] for the 16 e4m3 values of one 16-byte load, p in f16.
__device__ __forceinline__ void axpy16_e4m3_f16(uint16_t p16, const uint4& u, float (&acc)[16]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        asm("{\n\t.reg .b16 lo, hi, v0, v1, v2, v3;\n\t.reg .b32 vv01, vv23;\n\t"
            "mov.b32 {lo, hi}, %4;\n\t"
            "cvt.rn.f16x2.e4m3x2 vv01, lo;\n\tcvt.rn.f16x2.e4m3x2 vv23, hi;\n\t"
            "mov.b32 {v0, v1}, vv01;\n\tmov.b32 {v2, v3}, vv23;\n\t"
            "fma.rn.f32.f16 %0, %5, v0, %0;\n\tfma.rn.f32.f16 %1, %5, v1, %1;\n\t"
            "fma.rn.f32.f16 %2, %5, v2, %2;\n\tfma.rn.f32.f16 %3, %5, v3, %3;\n\t}"
            : "+f"(acc[4 * i]), "+f"(acc[4 * i + 1]), "+f"(acc[4 * i + 2]), "+f"(acc[4 * i + 3])
            : "r"(w[i]), "h"(p16));
    }
}

// EPL elements of a cached row piece (one 16-byte load) -> fp32.
template <bool FP8>
__device__ __forceinline__ void kv_piece_to_f32(const uint4& u, float (&f)[FP8 ? 16 : 8]) {
    if constexpr (FP8) e4m3x16_to_f32(u, f);
    else bf16x8_to_f32(u, f);
}

// Grid: (max_splits, S, ceil(H / kDecodeHeadsPerCta)); block: 32 * kDecodeHeadsPerCta.
// FP8: K/V rows are e4m3 (d bytes per token-head, half the bf16 traffic); the
// per-head key scale is folded into q and the value scale into the partial O.
template <int D, bool PAGED, bool FP8>
__global__ void __launch_bounds__(32 * kDecodeHeadsPerCta)
    decode_split_kernel(const DecodeParams p) {
    constexpr int EPL = FP8 ? 16 : 8;          // elements per 16-byte lane load
    constexpr int ROW_BYTES = FP8 ? D : 2 * D; // one token-head row of the cache
    constexpr int LPT = D / EPL;               // lanes per token row
    constexpr int TPW = 32 / LPT;              // tokens per warp step
    constexpr int UNROLL = 8;                  // warp steps in flight
    __shared__ float scores[kDecodeHeadsPerCta][kSplitTokens];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x, s = blockIdx.y;
    const int h = blockIdx.z * kDecodeHeadsPerCta + warp;
    if (h >= p.H) return;
    const int L = decode_seqlen(p, s);
    const int t0 = split * kSplitTokens;
    if (t0 >= L) return;
    const int n = min(kSplitTokens, L - t0);
    const int sub = lane % LPT;       // which EPL-element piece of the row
    const int tok = lane / LPT;       // which token of the warp step
    const uint8_t* kbytes = static_cast<const uint8_t*>(p.kc);
    const uint8_t* vbytes = static_cast<const uint8_t*>(p.vc);

    // q piece: bf16, pre-scaled by scale*log2(e); FP8: converted exactly to f16 pairs
    // (bf16 values of f16 range are f16 numbers), the scale and the key scale applied
    // to the dot product instead
    float qf[FP8 ? 1 : EPL];
    const float qs = FP8 ? p.scale_log2 * __ldg(p.k_scale + h) : p.scale_log2;
    if constexpr (!FP8) {
        const uint4* qrow = reinterpret_cast<const uint4*>(p.q + ((size_t)s * p.H + h) * D);
#pragma unroll
        for (int c = 0; c < EPL / 8; ++c) {
            float f8[8];
            bf16x8_to_f32(__ldg(qrow + sub * (EPL / 8) + c), f8);
#pragma unroll
            for (int i = 0; i < 8; ++i) qf[c * 8 + i] = f8[i] * qs;
        }
    }
    float* sc = scores[warp];

    // ---- pass 1: scores of the split's tokens (K read once)
    float mx = -INFINITY;
    if constexpr (FP8) {
        // Two lanes per token, each the dot product over half the row (D/32 pieces of 16
        // e4m3 values), then one shuffle: the half-row sums replace the eight-lane
        // reduction of a 16-byte-per-lane layout (measured +4.6 % on a 64-sequence batch;
        // the kernel is held by its per-warp instruction latency).  q as f16 pairs (exact
        // conversions of its bf16 values of f16 range) in shared memory, read back per piece
        // (held in registers instead, it cost a CTA per SM and measured slower); the scale
        // and the key scale apply to the sum.
        constexpr int PL = D / 32;          // 16-byte pieces per lane
        constexpr int TPW1 = 16;            // tokens per warp step
        constexpr int U1 = 2;               // warp steps in flight
        const int hsel = lane & 1, tok1 = lane >> 1;
        __shared__ __align__(16) uint32_t qbuf[kDecodeHeadsPerCta][D / 2];
        {
            // word w of the row holds elements 2w, 2w+1; lane l writes words (D/64) l ..
            constexpr int WPL = D / 64;
            const uint32_t* qw = reinterpret_cast<const uint32_t*>(p.q + ((size_t)s * p.H + h) * D);
#pragma unroll
            for (int x = 0; x < WPL; ++x) {
                const uint32_t bw = __ldg(qw + lane * WPL + x);
                const __half2 hq = __floats2half2_rn(__uint_as_float(bw << 16), __uint_as_float(bw & 0xffff0000u));
                qbuf[warp][lane * WPL + x] = *reinterpret_cast<const uint32_t*>(&hq);
            }
            __syncwarp();
        }
        for (int base = 0; base < n; base += TPW1 * U1) {
            uint4 kv[U1][PL];
            bool valid[U1];
#pragma unroll
            for (int u = 0; u < U1; ++u) {
                const int i = base + u * TPW1 + tok1;
                valid[u] = false;
#pragma unroll
                for (int c = 0; c < PL; ++c) kv[u][c] = make_uint4(0, 0, 0, 0);
                if (i < n) {
                    const long long row = token_row<PAGED>(p, s, t0 + i);
                    if (row >= 0) {
                        valid[u] = true;
                        const uint4* src = reinterpret_cast<const uint4*>(
                                               kbytes + ((size_t)row * p.H + h) * ROW_BYTES) + hsel * PL;
#pragma unroll
                        for (int c = 0; c < PL; ++c) kv[u][c] = __ldg(src + c);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U1; ++u) {
                float a = 0.f;
#pragma unroll
                for (int c = 0; c < PL; ++c) {
                    // q words of this piece (elements 16 c .. 16 c + 15 of the lane's half)
                    const uint4 qa = *reinterpret_cast<const uint4*>(&qbuf[warp][hsel * (D / 4) + 8 * c]);
                    const uint4 qb = *reinterpret_cast<const uint4*>(&qbuf[warp][hsel * (D / 4) + 8 * c + 4]);
                    const uint32_t q8[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
                    a = dot16_e4m3_f16(kv[u][c], q8, a);
                }
                a += __shfl_xor_sync(0xffffffffu, a, 1);
                a *= qs;
                const int i = base + u * TPW1 + tok1;
                if (i < n) {
                    const float v = valid[u] ? a : -INFINITY;
                    if (hsel == 0) sc[i] = v;
                    mx = fmaxf(mx, v);
                }
            }
        }
    } else {
    for (int base = 0; base < n; base += TPW * UNROLL) {
        uint4 kv[UNROLL];
        bool valid[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int i = base + u * TPW + tok;
            valid[u] = false;
            kv[u] = make_uint4(0, 0, 0, 0);
            if (i < n) {
                const long long row = token_row<PAGED>(p, s, t0 + i);
                if (row >= 0) {
                    valid[u] = true;
                    kv[u] = __ldg(reinterpret_cast<const uint4*>(
                                      kbytes + ((size_t)row * p.H + h) * ROW_BYTES) + sub);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            float acc = 0.f;
            {
                float kf[EPL];
                kv_piece_to_f32<FP8>(kv[u], kf);
#pragma unroll
                for (int e = 0; e < EPL; ++e) acc = fmaf(qf[e], kf[e], acc);
            }
#pragma unroll
            for (int off = LPT / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            const int i = base + u * TPW + tok;
            if (i < n) {
                const float v = valid[u] ? acc : -INFINITY;
                if (sub == 0) sc[i] = v;
                mx = fmaxf(mx, v);
            }
        }
    }
    }  // pass 1 layouts
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0 && mx == -INFINITY) record_status(ATTN_ERR_INVALID_ARG);  // every page invalid
    const float m_use = (mx == -INFINITY) ? 0.f : mx;
    __syncwarp();

    // ---- pass 2: P = 2^(score - m), l = sum P, O = sum P V (V read once)
    float acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    float lsum = 0.f;
    for (int base = 0; base < n; base += TPW * UNROLL) {
        uint4 vv[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int i = base + u * TPW + tok;
            vv[u] = make_uint4(0, 0, 0, 0);
            if (i < n) {
                const long long row = token_row<PAGED>(p, s, t0 + i);
                if (row >= 0)
                    vv[u] = __ldg(reinterpret_cast<const uint4*>(
                                      vbytes + ((size_t)row * p.H + h) * ROW_BYTES) + sub);
            }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int i = base + u * TPW + tok;
            if (i < n) {
                const float pw = ex2_approx(sc[i] - m_use);
                lsum += pw;
                if constexpr (FP8) {
                    // P in f16 (relative rounding 2^-11) for the mixed-precision FMAs
                    const __half ph = __float2half_rn(pw);
                    axpy16_e4m3_f16(*reinterpret_cast<const uint16_t*>(&ph), vv[u], acc);
                } else {
                    float vf[EPL];
                    kv_piece_to_f32<FP8>(vv[u], vf);
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc[e] = fmaf(pw, vf[e], acc[e]);
                }
            }
        }
    }
    // combine the token groups of the warp (lanes with equal `sub`)
#pragma unroll
    for (int off = LPT; off < 32; off <<= 1) {
        lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], off);
    }
    const size_t slot = ((size_t)s * p.max_splits + split) * p.H + h;
    if (tok == 0) {
        float inv = (lsum > 0.f) ? 1.f / lsum : 0.f;
        if constexpr (FP8) inv *= __ldg(p.v_scale + h);
        float4* dst = reinterpret_cast<float4*>(p.ws_o + slot * D + sub * EPL);
#pragma unroll
        for (int c = 0; c < EPL / 4; ++c)
            dst[c] = make_float4(acc[4 * c] * inv, acc[4 * c + 1] * inv, acc[4 * c + 2] * inv,
                                 acc[4 * c + 3] * inv);
    }
    if (lane == 0)
        p.ws_lse[slot] = (lsum > 0.f) ? (m_use + __log2f(lsum)) * kLn2 : -INFINITY;
}

// Grid: ceil(S * H / 4); block: 128 (one warp per (sequence, head)).
template <int D>
__global__ void __launch_bounds__(128) decode_merge_kernel(const DecodeParams p) {
    constexpr int EPL = D / 32;  // output elements per lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int idx = blockIdx.x * 4 + warp;
    if (idx >= p.S * p.H) return;
    const int s = idx / p.H, h = idx % p.H;
    int L = __ldg(p.seqlens + s);
    L = min(max(L, 0), p.max_seqlen);
    const int nsplit = (L + kSplitTokens - 1) / kSplitTokens;
    const size_t slot0 = (size_t)s * p.max_splits * p.H + h;  // split x at slot0 + x * H

    float mx = -INFINITY;
    for (int x = lane; x < nsplit; x += 32) mx = fmaxf(mx, p.ws_lse[slot0 + (size_t)x * p.H]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));

    float out[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) out[e] = 0.f;
    float wsum = 0.f;
    if (mx != -INFINITY) {
        for (int x = 0; x < nsplit; ++x) {
            const size_t slot = slot0 + (size_t)x * p.H;
            const float w = ex2_approx((p.ws_lse[slot] - mx) * kLog2e);
            wsum += w;
            const float* src = p.ws_o + slot * D + lane * EPL;
#pragma unroll
            for (int e = 0; e < EPL; ++e) out[e] = fmaf(w, src[e], out[e]);
        }
    }
    const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
    __nv_bfloat16* dst = p.o + ((size_t)s * p.H + h) * D + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; e += 2) {
        const uint32_t pk = pack_bf16x2(out[e] * inv, out[e + 1] * inv);
        *reinterpret_cast<uint32_t*>(dst + e) = pk;
    }
    if (lane == 0 && p.lse != nullptr)
        p.lse[(size_t)s * p.H + h] = (wsum > 0.f) ? mx + __logf(wsum) : -INFINITY;
}

}  // namespace attn
