// Prefill (forward) attention kernel for sm_103a.
//
// What it computes: "FlashAttention complete summary" (cell-devlog), section
// "FlashAttention의 핵심 아이디어 — Tiling": Q is cut into row blocks (outer loop),
// K and V into key blocks (inner loop); per block S = Q_i K_j^T, the online
// softmax of the section that follows and of "Flash Attention ... complete
// guide" (holysheep), section "Online Softmax 알고리즘" (running max m, running
// sum l of exp(x - m), earlier partial results rescaled when m grows), and
// O_i += P_ij V_j.  Device memory sees only the reads of Q, K, V and the writes
// of O and the row log-sum-exp.
//
// How it maps onto the B300:
//   * a persistent grid (one CTA per SM) deals out work units -- QT query
//     tiles of 128 rows of one (batch, head) -- in snake order, heaviest
//     causal units first; for long sequences whose K/V would not stay in L2
//     (DYN), the units are numbered band by band of a few heads and taken from
//     a device counter by whichever CTA's producer is near the end of its
//     current unit, so the K/V of the heads at work is read from DRAM once;
//     paged K/V (chunked prefill) takes its longest-cache-first units the same
//     dynamic way, since their costs differ with the cache lengths;
//   * warp 0 is the TMA producer: Q tiles per unit, then K_j and V_j tiles of
//     128 keys into shared-memory rings (128-byte swizzle, completion counted on
//     mbarriers; lane 0 posts each barrier's bytes, the boxes are spread over the
//     lanes); the next unit's loads start while the current one finishes;
//   * warp 1 issues tcgen05.mma as a converged warp (elect.sync picks the
//     issuing lane): S_t = Q_t K_j^T into tensor memory (M=128, N=128, fp32),
//     and O_t += P_t V_j with P_t read from tensor memory (or shared memory)
//     and O_t accumulated in tensor memory; where P has a place of its own
//     (P_SEP) warp 3 issues for the second tile;
//   * warps 4.. form one 128-thread softmax group per query tile: thread r owns
//     row r (TMEM lane r), reads its S row, applies the causal / tail mask,
//     updates m and l, rescales its O row when m grew, writes P (bf16) back and
//     signals the MMA warp; at the end of a unit it divides O by l and stores
//     O and LSE while the tensor core already works on the next unit;
//   * the MMA order per key block j is PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), so
//     the tensor core works on one tile while the other tile's softmax runs
//     (P_t aliases S_t, so S_t(j+1) must follow P_t(j) V_j);
//   * P_SEP (bf16 d=64, FP8): P_t has its own tensor-memory columns (FP8
//     d=128: its own shared-memory tile), the softmax hands S_t back as soon as
//     it is in registers, and each tile's MMA warp issues S_t(j+1) before
//     P_t(j) V_j;
//   * causal: key blocks wholly above the diagonal are never loaded; only the
//     diagonal block is masked.
// FP8 mode (FlashAttention-3's FP8 forward, cell-devlog "FlashAttention 3",
// tiptinker "FlashAttention-3가 다른 이유"): Q, K and V are E4M3 with one scale per
// head; both products run as tcgen05 kind::f8f6f4 with every operand K-major (V
// arrives transposed, keys contiguous; d=64 Q/K rows use the 64-byte swizzle),
// P is rounded to E4M3, the q*k scale folds into the exponent and the v scale
// into the epilogue.
// Every wait is bounded in time; on expiry the kernel records ATTN_ERR_TIMEOUT
// in the device status word and winds down instead of hanging.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace attn {

// The running max is moved only when it grows by more than this (log2 units).
constexpr float kMaxSlack = 8.f;
// FP8: a moved reference max is set this far (log2 units) below the new row
// max, so small P keep 4 more bits above the E4M3 subnormals.  The largest P
// is still bounded by the slack: the reference moves only when a block's max
// exceeds m + kMaxSlack, so P = 2^(s - m) <= 2^kMaxSlack = 256 < 448 (the
// largest finite E4M3 value).
constexpr float kFp8Headroom = 4.f;
static_assert(kFp8Headroom <= kMaxSlack, "a moved reference stays at or below the row max");
static_assert((1 << (int)kMaxSlack) <= 448, "P = 2^(s - m) <= 2^kMaxSlack must fit E4M3");

struct PrefillParams {
    __nv_bfloat16* o;
    float* lse;
    int B, H, N;       // N: query rows per sequence (and keys, when K/V are contiguous)
    float scale_log2;  // scale * log2(e)
    unsigned long long timeout_ns;
    int num_units;     // query-tile groups x B x H
    // Test hook (0 in normal use): the producer leaves its first K load unissued,
    // so the MMA warp's wait for it can only run out -- a fault-free way to make a
    // bounded wait expire and exercise the wind-down.
    int test_drop_load;
    // K/V in a 16-token paged cache (chunked prefill): sequence b has seqlens[b]
    // keys, the last N of which belong to this chunk's queries; token t of it is
    // slot t % 16 of pool page page_table[b * max_pages + t / 16]
    const int* seqlens;
    const int* page_table;
    int max_pages, num_pages;
    // FP8 mode: per-head scales of Q, K, V (value = scale[h] * e4m3)
    const float* q_scale;
    const float* k_scale;
    const float* v_scale;
    // Contiguous K/V too large to stay in L2 all at once: units are numbered
    // band by band, band_heads (batch, head) pairs per band (heaviest causal
    // query groups first within a band), and dealt dynamically -- each CTA takes
    // the next unit index from *unit_counter (zero at launch) when it is ready
    // for one -- so the CTAs at work at any moment share a few heads' K/V in L2.
    // band_heads = 0: the static snake-order deal over all heads.
    int band_heads;
    unsigned int* unit_counter;
};

// Keys of sequence b, and the offset of its first query row among them
// (query row i sees keys j <= i + offset under the causal mask).  An
// out-of-range cache length is recorded and clamped.
template <bool KV_PAGED>
__device__ __forceinline__ int prefill_kv_len(const PrefillParams& p, int b) {
    if constexpr (KV_PAGED) {
        int L = __ldg(p.seqlens + b);
        const int hi = p.max_pages * 16;
        if (L < p.N || L > hi) {
            record_status(ATTN_ERR_INVALID_ARG);
            L = min(max(L, p.N), hi);
        }
        return L;
    } else {
        return p.N;
    }
}

// Paged (chunked) prefill orders its units by the sequences' cache lengths,
// longest first, from a rank table in shared memory; batches of more
// sequences than this keep the sequences' own order.
constexpr int kMaxRankedSeqs = 256;

template <int D, int QT, bool P_TMEM, bool FP8 = false, bool KV_PAGED = false>
struct PrefillLayout {
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    static_assert(QT == 1 || QT == 2, "one or two query tiles per CTA");
    static_assert(P_TMEM || QT == 1, "P in shared memory only with one query tile");
    static_assert(!FP8 || (QT == 2 && P_TMEM), "FP8: two tiles");
    static constexpr int BM = 128;                 // query rows per tile = TMEM lanes
    static constexpr int BN = 128;                 // keys per block
    static constexpr int ROW_BYTES = D * (FP8 ? 1 : 2);
    // Q and K rows of FP8 d=64 are 64 bytes: one 64-byte box per row, 64-byte swizzle
    static constexpr bool QK_SW64 = FP8 && D == 64;
    static constexpr int KB = QK_SW64 ? 1 : ROW_BYTES / 128;  // column boxes per Q/K row
    static constexpr int BOX_COLS = FP8 ? (QK_SW64 ? 64 : 128) : 64;  // elements per box row
    static constexpr int BOX_BYTES = 128 * (QK_SW64 ? 64 : 128);      // one TMA box of 128 rows
    static constexpr int TILE_BYTES = 128 * ROW_BYTES;  // Q, K or V tile (FP8 V: V^T tile)
    // P in shared memory: the one-tile bf16 variant (128 x 128 bf16), and FP8
    // d=128 (one 128 x 128 E4M3 tile per query tile: tensor memory has no room for
    // P next to two S and two d=128 O accumulators, so P lives here instead)
    static constexpr bool P_SMEM8 = FP8 && D == 128;
    static constexpr int P_BYTES = P_SMEM8 ? QT * 128 * 128 : (P_TMEM ? 0 : 128 * 128 * 2);
    // Two query tiles of 16 KB (bf16 d=64, FP8 d=128): each softmax warp owns a
    // 4 KB staging area (32 rows x 128 bytes) through which its O rows are
    // transposed for coalesced stores.  (With 32 KB tiles the 32 KB of staging
    // would cost the third K stage, which measured slower than direct stores.)
    static constexpr bool STG = (QT == 2) && (TILE_BYTES <= 16384);
    static constexpr int STG_BYTES = STG ? QT * 4 * 4096 : 0;
    // K and V rings, as deep as shared memory allows: a 32 KB tile (bf16 d=128)
    // leaves room for 3 K + 2 V stages next to two Q tiles (or one Q tile and
    // P); a 16 KB tile gets 5 + 5 next to the staging (bf16 d=64), 4 + 4 next
    // to the staging and P (FP8 d=128)
    static constexpr int KSTAGES = (TILE_BYTES == 32768) ? 3 : (TILE_BYTES == 8192 ? 6 : (P_SMEM8 ? 4 : 5));
    static constexpr int VSTAGES =
        (TILE_BYTES == 32768) ? ((QT == 1 && P_TMEM) ? 3 : 2) : (TILE_BYTES == 8192 ? 6 : (P_SMEM8 ? 4 : 5));
    // keys (columns of S) per MMA k-step: 32 bytes of a row
    static constexpr int K_STEP = FP8 ? 32 : 16;
    static constexpr int THREADS = 128 + 128 * QT;
    // shared memory (offsets from a 1024-byte aligned base)
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + QT * TILE_BYTES;
    static constexpr int V_OFF = K_OFF + KSTAGES * TILE_BYTES;
    static constexpr int P_OFF = V_OFF + VSTAGES * TILE_BYTES;
    static constexpr int STG_OFF = P_OFF + P_BYTES;
    static constexpr int BAR_OFF = STG_OFF + STG_BYTES;
    // bf16 d=64 with two tiles keeps P in its own tensor-memory columns (S 2x128,
    // O 2x64, P 2x64 = 512), so S(j+1) need not wait for P(j)V(j): see P_SEP below
    // (FP8 keeps P in shared memory, with the same effect)
    static constexpr bool P_SEP = P_TMEM && QT == 2 && (D == 64 || FP8);
    // MMA-issuing warps: one per query tile with P_SEP, else one for both
    static constexpr int MMA_WARPS = P_SEP ? 2 : 1;
    static constexpr int NUM_BARS = 8 * QT + 2 * KSTAGES + 2 * VSTAGES;
    // after the barriers: the TMEM base address (16 bytes), then (paged) the rank table
    static constexpr int RANK_OFF = BAR_OFF + NUM_BARS * 8 + 16;
    static constexpr int RANK_BYTES = KV_PAGED ? kMaxRankedSeqs * 4 : 0;
    // dynamic deal: a ring of units from warp 0 to the other warps (full and
    // empty barriers per slot, then per slot the unit index, first query row,
    // batch and head)
    static constexpr int UNIT_SLOTS = 2;
    static constexpr int UNIT_BAR_OFF = RANK_OFF + RANK_BYTES;
    static constexpr int UNIT_IDX_OFF = UNIT_BAR_OFF + 2 * UNIT_SLOTS * 8;
    // warps that read the ring: the MMA warps and the softmax warps
    static constexpr int UNIT_READERS = MMA_WARPS + 4 * QT;
    static constexpr int SMEM_BYTES = UNIT_IDX_OFF + UNIT_SLOTS * 16 + 1024;  // + alignment slack
    // tensor memory columns
    static constexpr int S_COL0 = 0;          // S_t at t*128 (P_t aliases its first 64 columns)
    static constexpr int O_COL0 = QT * 128;   // O_t at O_COL0 + t*D
    // P_SEP with P in tensor memory: P_t at P_COL0 + t * P_COLS (bf16: 64 columns,
    // E4M3: 32, four values per column)
    static constexpr int P_COL0 = QT * (128 + D);
    static constexpr int P_COLS = FP8 ? 32 : 64;
    static constexpr int TMEM_COLS = (QT * (128 + D) <= 256) ? 256 : 512;
    // register split for two query tiles (launch: 384 threads x 168 registers):
    // producer/MMA warpgroup 72, each softmax warpgroup 216; 128*72 + 256*216 = 384*168
    static constexpr int LAUNCH_REGS = 168;
    static constexpr int REGS_CTRL = 72;
    static constexpr int REGS_SOFTMAX = 216;
    static_assert(QT != 2 || 128 * REGS_CTRL + 256 * REGS_SOFTMAX <= 384 * LAUNCH_REGS,
                  "register split exceeds the launch allocation");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// One work unit = QT query tiles of 128 rows of one (batch, head).  Units are
// numbered heaviest first for causal (query groups from the last one down),
// so that a snake-order deal over the persistent CTAs balances the causal work.
// Paged (chunked) prefill, where a unit's cost grows with its sequence's cache
// length: units are numbered sequence by sequence, longest cache first (`rank`:
// the sequence of each rank, or null to keep the batch order), each head's query
// groups heaviest first.
struct PrefillUnit {
    int q0, b, h;
};

template <int QT, bool CAUSAL, bool KV_PAGED = false, bool BANDED = false>
__device__ __forceinline__ PrefillUnit prefill_unit(const PrefillParams& p, int k,
                                                    const int* rank = nullptr) {
    const int BH = p.B * p.H;
    const int n_groups = (p.N + 128 * QT - 1) / (128 * QT);
    if constexpr (BANDED) {
        // band-major: band b holds heads [b*band_heads, ...) (the last band may be
        // narrower); within a band, query groups heaviest first, heads inner
        const int per_band = p.band_heads * n_groups;
        const int band = k / per_band;
        const int r = k - band * per_band;
        const int heads = min(p.band_heads, BH - band * p.band_heads);
        int grp = r / heads;
        const int bh = band * p.band_heads + (r - grp * heads);
        if (CAUSAL) grp = n_groups - 1 - grp;
        return PrefillUnit{grp * 128 * QT, bh / p.H, bh % p.H};
    }
    if constexpr (KV_PAGED) {
        const int bhr = k / n_groups;
        int grp = k % n_groups;
        if (CAUSAL) grp = n_groups - 1 - grp;
        const int r = bhr / p.H;
        return PrefillUnit{grp * 128 * QT, rank != nullptr ? rank[r] : r, bhr % p.H};
    }
    int grp = k / BH;
    if (CAUSAL) grp = n_groups - 1 - grp;
    const int bh = k % BH;
    return PrefillUnit{grp * 128 * QT, bh / p.H, bh % p.H};
}

// Key blocks query tile t of a unit needs (0 when the tile lies past N), for
// kv_len keys whose first query row sits at key kv_len - N.
template <bool CAUSAL>
__device__ __forceinline__ int prefill_nkv(const PrefillParams& p, int q0, int t, int kv_len) {
    const int r0 = q0 + 128 * t;
    if (r0 >= p.N) return 0;
    const int keys = CAUSAL ? min(kv_len, r0 + 128 + (kv_len - p.N)) : kv_len;
    return (keys + 127) / 128;
}

// Unit index of this CTA's `round`-th unit: rounds alternate direction.
__device__ __forceinline__ int prefill_unit_index(int round) {
    const int G = gridDim.x, c = blockIdx.x;
    return round * G + ((round & 1) ? (G - 1 - c) : c);
}

// This thread's S row: 128 fp32 columns of its TMEM lane, with keys at
// column >= limit (causal diagonal, or past N) set to -inf.
__device__ __forceinline__ void load_s_row(uint32_t s_addr, int limit, float (&s)[128]) {
    uint32_t raw[128];
    tmem_ld128(s_addr, raw);
#pragma unroll
    for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(raw[i]);
    if (limit < 128) {
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = (c < limit) ? s[c] : -INFINITY;
    }
}

// Maximum of 128 values: eight independent chains of 3-input max.
__device__ __forceinline__ float row_max128(const float (&s)[128]) {
    float mx8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(s[i], s[i + 8]);
#pragma unroll
    for (int c = 16; c < 128; c += 16) {
#pragma unroll
        for (int i = 0; i < 8; ++i) mx8[i] = max3(mx8[i], s[c + i], s[c + 8 + i]);
    }
    return fmaxf(max3(mx8[0], mx8[1], mx8[2]),
                 max3(fmaxf(mx8[3], mx8[4]), max3(mx8[5], mx8[6], mx8[7]), -INFINITY));
}

// One exponent sweep over a row, in place: s <- 2^(s * sl2 - mu); returns the
// row sum.  With TRACK_MAX it also returns the maximum of the incoming s in mx,
// taken chunk by chunk just before each chunk is overwritten, so the max and
// the exponentials are independent work the scheduler can interleave.
template <bool TRACK_MAX>
__device__ __forceinline__ float exp_pass(float (&s)[128], float sl2, float mu, float& mx) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float mx8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mx8[i] = -INFINITY;
#pragma unroll
    for (int c = 0; c < 128; c += 16) {
        if constexpr (TRACK_MAX) {
#pragma unroll
            for (int i = 0; i < 8; ++i) mx8[i] = max3(mx8[i], s[c + i], s[c + 8 + i]);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int e = c + 2 * q;
            fma2(s[e], s[e + 1], s[e], s[e + 1], sl2, sl2, -mu, -mu);
            s[e] = ex2_approx(s[e]);
            s[e + 1] = ex2_approx(s[e + 1]);
            add2(acc[2 * (q & 3)], acc[2 * (q & 3) + 1], s[e], s[e + 1]);
        }
    }
    if constexpr (TRACK_MAX)
        mx = fmaxf(max3(mx8[0], mx8[1], mx8[2]),
                   max3(fmaxf(mx8[3], mx8[4]), max3(mx8[5], mx8[6], mx8[7]), -INFINITY));
    return ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
}

template <int D, bool CAUSAL, int QT, bool P_TMEM, bool KV_PAGED, bool FP8, bool DYN>
__global__ void __launch_bounds__(128 + 128 * QT, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
    static_assert(!(FP8 && KV_PAGED), "FP8 reads contiguous Q, K, V^T");
    using L = PrefillLayout<D, QT, P_TMEM, FP8, KV_PAGED>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::BAR_OFF;
    // barrier addresses
    auto q_full = [&](int t) { return bar0 + 8u * t; };
    auto q_empty = [&](int t) { return bar0 + 8u * (QT + t); };
    auto k_full = [&](int s) { return bar0 + 8u * (2 * QT + s); };
    constexpr int KST = L::KSTAGES, VST = L::VSTAGES;
    auto k_empty = [&](int s) { return bar0 + 8u * (2 * QT + KST + s); };
    auto v_full = [&](int s) { return bar0 + 8u * (2 * QT + 2 * KST + s); };
    auto v_empty = [&](int s) { return bar0 + 8u * (2 * QT + 2 * KST + VST + s); };
    auto s_full = [&](int t) { return bar0 + 8u * (2 * QT + 2 * KST + 2 * VST + t); };
    auto p_full = [&](int t) { return bar0 + 8u * (3 * QT + 2 * KST + 2 * VST + t); };
    auto o_final = [&](int t) { return bar0 + 8u * (4 * QT + 2 * KST + 2 * VST + t); };
    auto drain_bar = [&](int t) { return bar0 + 8u * (5 * QT + 2 * KST + 2 * VST + t); };
    // P_SEP only: S_t has been loaded into registers (its columns may be overwritten), and
    // P_t V_j has completed (P_t may be overwritten, O_t holds it)
    auto s_free = [&](int t) { return bar0 + 8u * (6 * QT + 2 * KST + 2 * VST + t); };
    auto pv_done = [&](int t) { return bar0 + 8u * (7 * QT + 2 * KST + 2 * VST + t); };
    constexpr bool P_SEP = L::P_SEP;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::BAR_OFF + L::NUM_BARS * 8);
    // dynamic deal (unit_counter set): the ring of unit indices
    auto unit_full = [&](int s) { return sbase + L::UNIT_BAR_OFF + 8u * s; };
    auto unit_empty = [&](int s) { return sbase + L::UNIT_BAR_OFF + 8u * (L::UNIT_SLOTS + s); };
    volatile int* unit_idx = reinterpret_cast<volatile int*>(smem + L::UNIT_IDX_OFF);
    // dynamic deal (p.unit_counter): contiguous K/V in bands of heads; paged K/V in
    // the longest-cache-first order of the static deal
    constexpr bool dyn = DYN;
    constexpr bool banded = DYN && !KV_PAGED;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_units = p.num_units;

    // ---- setup: barriers (thread 0), tensor memory (warp 2)
    if (threadIdx.x == 0) {
        for (int t = 0; t < QT; ++t) {
            mbar_init(q_full(t), 1);
            mbar_init(q_empty(t), 1);
            mbar_init(s_full(t), 1);
            mbar_init(p_full(t), 128);
            mbar_init(o_final(t), 1);
            mbar_init(s_free(t), 128);
            mbar_init(pv_done(t), 1);
            mbar_init(drain_bar(t), 1);
        }
        // K and V slots are released once by each MMA warp
        for (int s = 0; s < KST; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), L::MMA_WARPS);
        }
        for (int s = 0; s < VST; ++s) {
            mbar_init(v_full(s), 1);
            mbar_init(v_empty(s), L::MMA_WARPS);
        }
        for (int s = 0; s < L::UNIT_SLOTS; ++s) {
            mbar_init(unit_full(s), 1);
            mbar_init(unit_empty(s), L::UNIT_READERS);
        }
        fence_mbar_init();
    }
    if (warp == 2) {
        tmem_alloc(smem_u32(tmem_slot), L::TMEM_COLS);
        tmem_relinquish();
    }
    // paged: rank table of the sequences by cache length, longest first (ties in batch
    // order), so that the heaviest units are dealt first
    const int* rank = nullptr;
    if constexpr (KV_PAGED) {
        if (p.B <= kMaxRankedSeqs) {
            int* table = reinterpret_cast<int*>(smem + L::RANK_OFF);
            for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
                const int li = __ldg(p.seqlens + i);
                int r = 0;
                for (int j = 0; j < p.B; ++j) {
                    const int lj = __ldg(p.seqlens + j);
                    r += (lj > li || (lj == li && j < i)) ? 1 : 0;
                }
                table[r] = i;
            }
            rank = table;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint64_t tmo = p.timeout_ns;
    const uint64_t tdrain = tmo > kDrainTimeoutNs ? tmo : kDrainTimeoutNs;  // wind-down waits
    // The unit index of this CTA's `round`-th unit, for the warps other than the
    // producer (whole warp; the dynamic deal reads it from the ring, and a wait that
    // runs out ends the sequence with ok = false).
    // (The dynamic deal passes the unit decoded -- index, first query row, batch,
    // head -- so that these warps do no index arithmetic of their own.)
    auto unit_of_round = [&](int round, bool& ok, PrefillUnit& u) -> bool {
        if constexpr (!dyn) {
            const int k = prefill_unit_index(round);
            if (k >= num_units) return false;
            u = prefill_unit<QT, CAUSAL, KV_PAGED>(p, k, rank);
            return true;
        } else {
            const int sl = round % L::UNIT_SLOTS;
            if (!mbar_wait_warp(unit_full(sl), (round / L::UNIT_SLOTS) & 1, p.timeout_ns)) {
                ok = false;
                return false;
            }
            const int k = unit_idx[4 * sl];
            u.q0 = unit_idx[4 * sl + 1];
            u.b = unit_idx[4 * sl + 2];
            u.h = unit_idx[4 * sl + 3];
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_arrive(unit_empty(sl));
            return k < num_units;
        }
    };

    if (warp < 4) {
        if constexpr (QT == 2) regs_decrease<L::REGS_CTRL>();
        if (warp == 0) {
            // =========================== TMA producer ===========================
            // The whole warp runs this branch: lane 0 posts each barrier's expected
            // bytes, then the copies of a tile are spread over the lanes (one box
            // per lane), and every wait has one warp-wide verdict.
            if (lane == 0) {
                prefetch_tensormap(&tm_q);
                prefetch_tensormap(&tm_k);
                prefetch_tensormap(&tm_v);
            }
            int kn = 0, vn = 0;    // K and V tiles issued so far (ring positions)
            int uq[QT] = {};       // Q loads issued per tile
            bool ok = true;
            // Paged K/V: this lane's page id for key block j of unit u (lane = page
            // i of the block x column box), read from the page table and checked.
            // Pages past the sequence's last one read as its first page (finite
            // values the causal/length mask zeroes); an out-of-range id is recorded
            // and replaced by page 0, so no copy leaves the pool.
            auto page_id = [&](const PrefillUnit& u, int j, int kv_len) -> int {
                if constexpr (KV_PAGED) {
                    if (lane >= 8 * L::KB) return 0;
                    const int slot = j * 8 + lane / L::KB;
                    int id = __ldg(p.page_table + (size_t)u.b * p.max_pages +
                                   (slot * 16 < kv_len ? slot : 0));
                    if (id < 0 || id >= p.num_pages) {
                        record_status(ATTN_ERR_INVALID_ARG);
                        id = 0;
                    }
                    return id;
                } else {
                    return 0;
                }
            };
            // One 128-key tile (K or V) of unit u into shared memory at dst.
            // Contiguous K/V: one 64-column box per lane (lanes < KB).  Paged K/V:
            // eight 16-token pages x KB column boxes, one per lane (lanes < 8 KB),
            // each at page `id` (this lane's, from page_id) and landing at its row
            // offset (16 rows = two 1024-byte swizzle atoms, so the layout is that of
            // one 128-row box).
            auto load_tile = [&](const CUtensorMap* map, uint32_t dst, uint32_t bar,
                                 const PrefillUnit& u, int j, int id, bool is_v) {
                if constexpr (FP8) {
                    // one 128 x 128-byte box: 128 keys x d of K, or d x 128 keys of V^T
                    // (keys past N read as zero)
                    if (lane == 0) {
                        if (is_v)
                            tma_load_4d(dst, map, bar, j * 128, 0, u.h, u.b);
                        else
                            tma_load_4d(dst, map, bar, 0, u.h, j * 128, u.b);
                    }
                } else if constexpr (KV_PAGED) {
                    if (lane < 8 * L::KB) {
                        const int i = lane / L::KB, kb = lane % L::KB;
                        tma_load_3d(dst + kb * L::BOX_BYTES + i * 2048, map, bar, kb * 64, u.h,
                                    id * 16);
                    }
                } else {
                    if (lane < L::KB)
                        tma_load_4d(dst + lane * L::BOX_BYTES, map, bar, lane * L::BOX_COLS, u.h,
                                    j * 128, u.b);
                }
            };
            // K tile `j` of unit `u` into the next K slot, once the S MMAs that read
            // that slot's previous tile have completed (likewise for V)
            auto load_k = [&](const PrefillUnit& u, int j, int id) {
                const int st = kn % KST;
                if (!mbar_wait_warp(k_empty(st), ((kn / KST) & 1) ^ 1, tmo)) return false;
                if (p.test_drop_load && kn == 0) {  // test hook: the slot's full phase never completes
                    ++kn;
                    return true;
                }
                if (lane == 0) mbar_arrive_expect_tx(k_full(st), L::TILE_BYTES);
                __syncwarp();
                load_tile(&tm_k, sbase + L::K_OFF + st * L::TILE_BYTES, k_full(st), u, j, id, false);
                ++kn;
                return true;
            };
            auto load_v = [&](const PrefillUnit& u, int j, int id) {
                const int st = vn % VST;
                if (!mbar_wait_warp(v_empty(st), ((vn / VST) & 1) ^ 1, tmo)) return false;
                if (lane == 0) mbar_arrive_expect_tx(v_full(st), L::TILE_BYTES);
                __syncwarp();
                load_tile(&tm_v, sbase + L::V_OFF + st * L::TILE_BYTES, v_full(st), u, j, id, true);
                ++vn;
                return true;
            };
            // dynamic deal: lane 0 takes the next unit index from the device counter
            // a few key blocks before the current unit's loads end (the take's latency
            // is hidden, and the unit is claimed close to when this CTA needs it)
            unsigned int taken = 0;
            if (dyn && lane == 0) taken = atomicAdd(p.unit_counter, 1u);
            for (int round = 0; ok; ++round) {
                PrefillUnit u{0, 0, 0};
                if constexpr (dyn) {
                    const int k = (int)min(__shfl_sync(0xffffffffu, taken, 0), (unsigned int)num_units);
                    // publish it decoded (num_units: the end) once its ring slot is free
                    const int sl = round % L::UNIT_SLOTS;
                    if (!mbar_wait_warp(unit_empty(sl), ((round / L::UNIT_SLOTS) & 1) ^ 1, tmo)) {
                        ok = false;
                        break;
                    }
                    if (k < num_units) u = prefill_unit<QT, CAUSAL, KV_PAGED, banded>(p, k, rank);
                    if (lane == 0) {
                        unit_idx[4 * sl] = k;
                        unit_idx[4 * sl + 1] = u.q0;
                        unit_idx[4 * sl + 2] = u.b;
                        unit_idx[4 * sl + 3] = u.h;
                        mbar_arrive(unit_full(sl));
                    }
                    __syncwarp();
                    if (k >= num_units) break;
                } else {
                    const int k = prefill_unit_index(round);
                    if (k >= num_units) break;
                    u = prefill_unit<QT, CAUSAL, KV_PAGED>(p, k, rank);
                }
                const int kv_len = prefill_kv_len<KV_PAGED>(p, u.b);
                int nkv_max = 0;
                for (int t = 0; t < QT; ++t) {
                    const int n = prefill_nkv<CAUSAL>(p, u.q0, t, kv_len);
                    if (n == 0) continue;
                    nkv_max = max(nkv_max, n);
                    // Q tile t of this unit, once the previous unit's S MMAs no longer read it
                    if (!mbar_wait_warp(q_empty(t), (uq[t] & 1) ^ 1, tmo)) { ok = false; break; }
                    if (lane == 0) mbar_arrive_expect_tx(q_full(t), L::TILE_BYTES);
                    __syncwarp();
                    if (lane < L::KB)
                        tma_load_4d(sbase + L::Q_OFF + t * L::TILE_BYTES + lane * L::BOX_BYTES, &tm_q,
                                    q_full(t), lane * L::BOX_COLS, u.h, u.q0 + 128 * t, u.b);
                    ++uq[t];
                }
                // the order the MMAs consume them: K_0, then V_j followed by K_{j+1}.
                // Paged: K_j and V_j use the page ids of block j; those of block j + 1 are
                // read while block j's copies wait for their slots, so no page-table load
                // sits between a free slot and its copy.
                int id_cur = page_id(u, 0, kv_len);
                int id_next = nkv_max > 1 ? page_id(u, 1, kv_len) : 0;
                if (ok) ok = load_k(u, 0, id_cur);
                for (int j = 0; ok && j < nkv_max; ++j) {
                    if (dyn && lane == 0 && j == max(0, nkv_max - 3)) taken = atomicAdd(p.unit_counter, 1u);
                    ok = load_v(u, j, id_cur);
                    if (ok && j + 1 < nkv_max) {
                        id_cur = id_next;
                        id_next = j + 2 < nkv_max ? page_id(u, j + 2, kv_len) : 0;
                        ok = load_k(u, j + 1, id_cur);
                    }
                }
            }
            if (!ok && lane == 0) record_status(ATTN_ERR_TIMEOUT);
            // Let copies still in flight land before the CTA can exit.  (After a normal
            // run the consumers have waited for every one of them and these waits
            // return at once; after a consumer gave up they are what keeps the
            // CTA's shared memory alive until the copies are done.)
            for (int t = 0; t < QT; ++t)
                if (uq[t] > 0) mbar_wait(q_full(t), (uq[t] - 1) & 1, tdrain);
            for (int x = max(0, kn - KST); x < kn; ++x)
                if (!(p.test_drop_load && x == 0)) mbar_wait(k_full(x % KST), (x / KST) & 1, tdrain);
            for (int x = max(0, vn - VST); x < vn; ++x) mbar_wait(v_full(x % VST), (x / VST) & 1, tdrain);
        } else if (warp == 1 || (L::MMA_WARPS == 2 && warp == 3)) {
            // ============================ MMA issuers ===========================
            // The whole warp runs this branch; each tcgen05 instruction is issued by
            // one elected lane (see umma_ss), and every wait is warp-uniform.
            //
            // P in its own tensor-memory columns (bf16 d=64): one warp per query
            // tile (warp 1: tile 0, warp 3: tile 1), each issuing S(j+1) as soon
            // as its softmax holds S(j) and P(j) V_j as soon as P(j) is written --
            // neither tile waits for the issuer to come back from the other tile
            // (a single issuing warp was measured taking ~0.3 us to get back).
            // Both warps walk every K and V tile of a unit: a tile this warp's
            // query tile does not use (a causal tile's last block, or an inactive
            // tile) is released with a plain arrive once it has landed, so the
            // rings' empty barriers count one release per MMA warp.
            //
            // P aliasing S: one warp issues for both tiles in the fixed order
            // PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), which keeps one tile's softmax
            // under the other tile's MMAs.  (Two warps there, even taking turns,
            // measured slower: the two tiles' MMA batches then took longer to
            // complete.)
            const int tm = (warp == 1) ? 0 : 1;  // this warp's query tile (P_SEP)
            constexpr uint32_t kIdescS =
                FP8 ? idesc_e4m3_f32(128, 128) : idesc_bf16_f32(128, 128, false, false);
            constexpr uint32_t kIdescPV =
                FP8 ? idesc_e4m3_f32(128, D) : idesc_bf16_f32(128, D, false, true);
            // Descriptors: a base per operand tile, then the k-step's byte offset
            // (>> 4) added to the low word (start-address field); shared memory is
            // below 256 KB, so the 14-bit field never carries.
            const uint64_t dq0 = L::QK_SW64 ? sdesc_sw64(sbase + L::Q_OFF, 16, 512)
                                            : sdesc_sw128(sbase + L::Q_OFF, 16, 1024);
            const uint64_t dk0 = L::QK_SW64 ? sdesc_sw64(sbase + L::K_OFF, 16, 512)
                                            : sdesc_sw128(sbase + L::K_OFF, 16, 1024);
            // bf16 V is MN-major (d contiguous, 64-wide blocks BOX_BYTES apart); the
            // FP8 V^T tile is K-major like K
            const uint64_t dv0 = sdesc_sw128(sbase + L::V_OFF, FP8 ? 16 : L::BOX_BYTES, 1024);
            const uint32_t q_lo = (uint32_t)dq0, q_hi = (uint32_t)(dq0 >> 32);
            const uint32_t k_lo = (uint32_t)dk0, k_hi = (uint32_t)(dk0 >> 32);
            const uint32_t v_lo = (uint32_t)dv0, v_hi = (uint32_t)(dv0 >> 32);
            auto issue_s = [&](int t, int st) {
                // A = Q_t, B = K_j, both K-major: 32 bytes (16 bf16 or 32 e4m3) per
                // k-step inside a 128-byte swizzle block, blocks BOX_BYTES apart
                const uint32_t a = q_lo + ((t * L::TILE_BYTES) >> 4);
                const uint32_t b = k_lo + ((st * L::TILE_BYTES) >> 4);
                const uint32_t d_tmem = tmem + L::S_COL0 + t * 128;
#pragma unroll
                for (int k = 0; k < D / L::K_STEP; ++k) {
                    const uint32_t off = ((k >> 2) * L::BOX_BYTES + (k & 3) * 32) >> 4;
                    if constexpr (FP8)
                        umma_ss_f8(d_tmem, a + off, q_hi, b + off, k_hi, kIdescS, k > 0 ? 1u : 0u);
                    else
                        umma_ss(d_tmem, a + off, q_hi, b + off, k_hi, kIdescS, k > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int t, int st, bool acc) {
                // bf16: B = V_j, MN-major: 16 keys x 128 B per k-step; 64-wide d blocks
                // at BOX_BYTES.  FP8: B = V_j^T, K-major: 32 keys (bytes) per k-step.
                // A = P_t from tensor memory: 8 columns per k-step either way.
                const uint32_t b = v_lo + ((st * L::TILE_BYTES) >> 4);
                const uint32_t d_tmem = tmem + L::O_COL0 + t * D;
#pragma unroll
                for (int k = 0; k < 128 / L::K_STEP; ++k) {
                    const uint32_t accf = (acc || k > 0) ? 1u : 0u;
                    const uint32_t boff = FP8 ? ((k * 32) >> 4) : ((k * 16 * 128) >> 4);
                    if constexpr (FP8 && L::P_SMEM8) {
                        // A = P_t, E4M3 in shared memory (K-major, 32 keys per k-step)
                        const uint64_t dp = sdesc_sw128(sbase + L::P_OFF + t * 128 * 128, 16, 1024);
                        umma_ss_f8(d_tmem, (uint32_t)dp + ((k * 32) >> 4), (uint32_t)(dp >> 32), b + boff,
                                   v_hi, kIdescPV, accf);
                    } else if constexpr (FP8) {
                        // A = P_t, E4M3 in its own tensor-memory columns (8 columns per k-step)
                        umma_ts_f8(d_tmem, tmem + L::P_COL0 + t * L::P_COLS + k * 8, b + boff, v_hi,
                                   kIdescPV, accf);
                    } else if constexpr (P_TMEM) {
                        const uint32_t pa = P_SEP ? (L::P_COL0 + t * L::P_COLS) : (L::S_COL0 + t * 128);
                        umma_ts(d_tmem, tmem + pa + k * 8, b + boff, v_hi, kIdescPV, accf);
                    } else {
                        const uint64_t dp = sdesc_sw128(sbase + L::P_OFF, 16, 1024);
                        const uint32_t off = ((k >> 2) * L::BOX_BYTES + (k & 3) * 32) >> 4;
                        umma_ss(d_tmem, (uint32_t)dp + off, (uint32_t)(dp >> 32), b + boff, v_hi,
                                kIdescPV, accf);
                    }
                }
            };
            if constexpr (L::MMA_WARPS == 2) {
                // release a K or V slot: after this warp's MMAs that read it (commit), or
                // at once when it read nothing from it (the slot's full phase was waited)
                auto release = [&](uint32_t bar, bool used) {
                    if (used)
                        umma_commit(bar);
                    else if (lane == 0)
                        mbar_arrive(bar);
                    __syncwarp();
                };
                int it = 0;   // K/V tiles consumed (ring position)
                int uq = 0;   // units started by this tile (q_full phase)
                int pf = 0;   // P blocks consumed (p_full phase)
                int sf = 0;   // S blocks issued (s_free phase)
                bool ok = true;
                for (int round = 0; ok; ++round) {
                    PrefillUnit u;
                    if (!unit_of_round(round, ok, u)) break;
                    const int kv_len = prefill_kv_len<KV_PAGED>(p, u.b);
                    int nkv_max = 0;
#pragma unroll
                    for (int t = 0; t < QT; ++t) nkv_max = max(nkv_max, prefill_nkv<CAUSAL>(p, u.q0, t, kv_len));
                    const int n = prefill_nkv<CAUSAL>(p, u.q0, tm, kv_len);  // this tile's key blocks
                    // S_tm of key block jb from K slot stk, once the softmax has loaded
                    // the previous S into registers
                    auto issue_s_block = [&](int stk, int jb) -> bool {
                        if (sf > 0 && !mbar_wait_warp(s_free(tm), (sf - 1) & 1, tmo)) return false;
                        tc_fence_after();
                        issue_s(tm, stk);
                        ++sf;
                        umma_commit(s_full(tm));
                        if (jb + 1 == n) umma_commit(q_empty(tm));
                        return true;
                    };
                    // prologue: S_tm(0)
                    {
                        const int st = it % KST;
                        if (!mbar_wait_warp(k_full(st), (it / KST) & 1, tmo)) { ok = false; break; }
                        if (n > 0 && !mbar_wait_warp(q_full(tm), uq & 1, tmo)) { ok = false; break; }
                        if (n > 0 && !issue_s_block(st, 0)) { ok = false; break; }
                        release(k_empty(st), n > 0);
                    }
                    for (int j = 0; ok && j < nkv_max; ++j) {
                        const int i = it + j;
                        const int st = i % VST;                  // V_j
                        const int stn = (i + 1) % KST;           // K_{j+1}
                        const bool more = j + 1 < nkv_max;       // K_{j+1} exists in this unit
                        // S_tm(j+1) as soon as the softmax holds S_tm(j), then P_tm(j) V_j
                        if (more) {
                            if (!mbar_wait_warp(k_full(stn), ((i + 1) / KST) & 1, tmo)) { ok = false; break; }
                            if (j + 1 < n && !issue_s_block(stn, j + 1)) { ok = false; break; }
                            release(k_empty(stn), j + 1 < n);
                        }
                        if (!mbar_wait_warp(v_full(st), (i / VST) & 1, tmo)) { ok = false; break; }
                        if (j < n) {
                            if (!mbar_wait_warp(p_full(tm), pf & 1, tmo)) { ok = false; break; }
                            ++pf;
                            tc_fence_after();
                            issue_pv(tm, st, j > 0);
                            umma_commit(j + 1 == n ? o_final(tm) : pv_done(tm));
                        }
                        release(v_empty(st), j < n);
                    }
                    it += nkv_max;
                    if (n > 0) ++uq;
                }
                if (!ok && lane == 0) record_status(ATTN_ERR_TIMEOUT);
                umma_commit(drain_bar(tm));
                mbar_wait(drain_bar(tm), 0, tdrain);
            } else {
                int it = 0;        // K/V tiles consumed (ring position)
                int uq[QT] = {};   // units started per tile (q_full phase)
                int pf[QT] = {};   // P blocks consumed per tile (p_full phase)
                bool ok = true;
                for (int round = 0; ok; ++round) {
                    PrefillUnit u;
                    if (!unit_of_round(round, ok, u)) break;
                    const int kv_len = prefill_kv_len<KV_PAGED>(p, u.b);
                    int nkv[QT];
                    int n_active = 0, nkv_max = 0;
#pragma unroll
                    for (int t = 0; t < QT; ++t) {
                        nkv[t] = prefill_nkv<CAUSAL>(p, u.q0, t, kv_len);
                        if (nkv[t] > 0) n_active = t + 1;
                        nkv_max = max(nkv_max, nkv[t]);
                    }
                    // prologue: S_t(0) for every active tile
                    {
                        const int st = it % KST;
                        if (!mbar_wait_warp(k_full(st), (it / KST) & 1, tmo)) { ok = false; break; }
                        for (int t = 0; t < n_active; ++t) {
                            if (!mbar_wait_warp(q_full(t), uq[t] & 1, tmo)) { ok = false; break; }
                            tc_fence_after();
                            issue_s(t, st);
                            umma_commit(s_full(t));
                            if (nkv[t] == 1) umma_commit(q_empty(t));
                        }
                        if (!ok) break;
                        umma_commit(k_empty(st));
                    }
                    for (int j = 0; ok && j < nkv_max; ++j) {
                        const int i = it + j;
                        const int st = i % VST;                  // V_j
                        const uint32_t ph = (i / VST) & 1;
                        const int stn = (i + 1) % KST;           // K_{j+1}
                        const uint32_t phn = ((i + 1) / KST) & 1;
                        bool v_ready = false, k_next_ready = false;
                        for (int t = 0; t < n_active; ++t) {
                            if (j >= nkv[t]) continue;
                            if (!mbar_wait_warp(p_full(t), pf[t] & 1, tmo)) { ok = false; break; }
                            ++pf[t];
                            if (!v_ready) {
                                if (!mbar_wait_warp(v_full(st), ph, tmo)) { ok = false; break; }
                                v_ready = true;
                            }
                            tc_fence_after();
                            issue_pv(t, st, j > 0);
                            if (j + 1 == nkv[t]) {
                                umma_commit(o_final(t));
                            } else {
                                if (!k_next_ready) {
                                    if (!mbar_wait_warp(k_full(stn), phn, tmo)) { ok = false; break; }
                                    tc_fence_after();
                                    k_next_ready = true;
                                }
                                issue_s(t, stn);
                                umma_commit(s_full(t));
                                if (j + 2 == nkv[t]) umma_commit(q_empty(t));
                            }
                        }
                        if (v_ready) umma_commit(v_empty(st));
                        if (k_next_ready) umma_commit(k_empty(stn));
                    }
                    it += nkv_max;
                    for (int t = 0; t < n_active; ++t) ++uq[t];
                }
                if (!ok && lane == 0) record_status(ATTN_ERR_TIMEOUT);
                umma_commit(drain_bar(0));
                mbar_wait(drain_bar(0), 0, tdrain);
            }
        }
    } else {
        // ========================= softmax / epilogue ========================
        if constexpr (QT == 2) regs_increase<L::REGS_SOFTMAX>();
        const int t = (warp - 4) >> 2;
        const int wq = warp & 3;                 // TMEM lane quarter of this warp
        const int r = wq * 32 + lane;            // row within the tile
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t s_addr = tmem + lane_off + L::S_COL0 + t * 128;
        const uint32_t o_addr = tmem + lane_off + L::O_COL0 + t * D;
        const uint32_t p_addr = (P_SEP && !L::P_SMEM8) ? (tmem + lane_off + L::P_COL0 + t * L::P_COLS) : s_addr;
        int pvw = 0;  // P_SEP: pv_done phases waited
        int js = 0;   // S blocks consumed (s_full phase)
        int uo = 0;   // units finished (o_final phase)
        bool ok = true;
        for (int round = 0; ok; ++round) {
            PrefillUnit u;
            if (!unit_of_round(round, ok, u)) break;
            const int kv_len = prefill_kv_len<KV_PAGED>(p, u.b);
            const int nkv = prefill_nkv<CAUSAL>(p, u.q0, t, kv_len);
            if (nkv == 0) continue;
            const int row = u.q0 + 128 * t + r;  // query index
            // scale*log2(e), times the head's q and k scales for FP8 (S holds the
            // products of the E4M3 codes)
            const float sl2 = FP8 ? p.scale_log2 * (__ldg(p.q_scale + u.h) * __ldg(p.k_scale + u.h))
                                  : p.scale_log2;
            constexpr float head = FP8 ? kFp8Headroom : 0.f;
            float m = -INFINITY;  // running max of scale*log2(e)*s
            float l = 0.f;        // running sum of 2^(scale*log2(e)*s - m)
            for (int j = 0; j < nkv; ++j) {
                if (!mbar_wait(s_full(t), js & 1, tmo)) { ok = false; break; }
                ++js;
                tc_fence_after();
                // keys [kv0, kv0 + limit) are visible to this row
                const int limit = (CAUSAL ? min(kv_len, row + 1 + (kv_len - p.N)) : kv_len) - j * 128;
                float s[128];
                load_s_row(s_addr, limit, s);
                // The running max moves only when it would grow by more than 8
                // (a factor 2^8): until then P stays <= 256 and O, l keep the
                // same reference, so the final O / l and LSE are unchanged.
                float m_new, sum;
                if constexpr (P_SEP) {
                    // S is in registers: its columns go back to the MMA warp for S(j+1)
                    // right away; the row max comes first, so no redo is ever needed
                    tc_fence_before();
                    mbar_arrive(s_free(t));
                    const float cand = row_max128(s) * sl2;
                    m_new = (cand > m + kMaxSlack) ? cand - head : m;
                    float unused;
                    sum = exp_pass<false>(s, sl2, (m_new == -INFINITY) ? 0.f : m_new, unused);
                } else if (__all_sync(0xffffffffu, m != -INFINITY)) {
                    // Every row has a reference max already: exponentiate against it
                    // right away and take the block max in the same sweep.
                    float mx;
                    sum = exp_pass<true>(s, sl2, m, mx);
                    const float cand = mx * sl2;
                    m_new = (cand > m + kMaxSlack) ? cand - head : m;
                    if (__any_sync(0xffffffffu, m_new != m)) {
                        // rare: a row's max grew past the slack -- redo from S, which
                        // is still in tensor memory, against the raised max
                        load_s_row(s_addr, limit, s);
                        sum = exp_pass<false>(s, sl2, m_new, mx);
                    }
                } else {
                    // first key block of this unit: the max comes first
                    const float cand = row_max128(s) * sl2;
                    m_new = (cand > m + kMaxSlack) ? cand - head : m;
                    float unused;
                    sum = exp_pass<false>(s, sl2, (m_new == -INFINITY) ? 0.f : m_new,
                                                   unused);
                }
                const float alpha = ex2_approx(m - m_new);  // 1 if unchanged, 0 on the first block
                l = l * alpha + sum;
                m = m_new;
                // P (bf16, or E4M3 in FP8 mode) for the PV product
                if constexpr (FP8 && !L::P_SMEM8) {
                    // E4M3 P row into its own 32 tensor-memory columns (the lowest key
                    // of each group of four in the low byte)
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        pk[i] = pack_e4m3x4(s[4 * i], s[4 * i + 1], s[4 * i + 2], s[4 * i + 3]);
                    if (j > 0) {
                        // P_t(j-1) V_{j-1} must have finished reading P_t and writing O_t
                        if (!mbar_wait_warp(pv_done(t), pvw & 1, tmo)) { ok = false; break; }
                        ++pvw;
                        tc_fence_after();
                    }
                    tmem_st32(p_addr, pk);
                    tmem_st_wait();
                } else if constexpr (FP8) {
                    // E4M3 P row into shared memory: 128 bytes, 16-byte chunks
                    // swizzled by row (the 128-byte swizzle the MMA descriptor reads)
                    if (j > 0) {
                        // P_t(j-1) V_{j-1} must have finished reading P_t and writing O_t
                        if (!mbar_wait_warp(pv_done(t), pvw & 1, tmo)) { ok = false; break; }
                        ++pvw;
                        tc_fence_after();
                    }
                    uint8_t* prow = smem + L::P_OFF + t * 128 * 128 + r * 128;
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint4 v;
                        v.x = pack_e4m3x4(s[16 * c + 0], s[16 * c + 1], s[16 * c + 2], s[16 * c + 3]);
                        v.y = pack_e4m3x4(s[16 * c + 4], s[16 * c + 5], s[16 * c + 6], s[16 * c + 7]);
                        v.z = pack_e4m3x4(s[16 * c + 8], s[16 * c + 9], s[16 * c + 10], s[16 * c + 11]);
                        v.w = pack_e4m3x4(s[16 * c + 12], s[16 * c + 13], s[16 * c + 14], s[16 * c + 15]);
                        *reinterpret_cast<uint4*>(prow + ((c ^ (r & 7)) << 4)) = v;
                    }
                    fence_proxy_async_smem();
                } else if constexpr (P_TMEM) {
                    uint32_t pk[64];
#pragma unroll
                    for (int i = 0; i < 64; ++i) pk[i] = pack_bf16x2(s[2 * i], s[2 * i + 1]);
                    if (P_SEP && j > 0) {
                        // P_t(j-1) V_{j-1} must have finished reading P_t and writing O_t
                        if (!mbar_wait_warp(pv_done(t), pvw & 1, tmo)) { ok = false; break; }
                        ++pvw;
                        tc_fence_after();
                    }
                    tmem_st64(p_addr, pk);
                    tmem_st_wait();
                } else {
                    tmem_st_wait();
                    uint8_t* prow = smem + L::P_OFF + r * 128;
#pragma unroll
                    for (int c8 = 0; c8 < 16; ++c8) {
                        const int blk = c8 >> 3, chunk = c8 & 7;
                        uint4 v;
                        v.x = pack_bf16x2(s[c8 * 8 + 0], s[c8 * 8 + 1]);
                        v.y = pack_bf16x2(s[c8 * 8 + 2], s[c8 * 8 + 3]);
                        v.z = pack_bf16x2(s[c8 * 8 + 4], s[c8 * 8 + 5]);
                        v.w = pack_bf16x2(s[c8 * 8 + 6], s[c8 * 8 + 7]);
                        *reinterpret_cast<uint4*>(prow + blk * L::BOX_BYTES +
                                                  ((chunk ^ (r & 7)) << 4)) = v;
                    }
                    fence_proxy_async_smem();
                }
                // rescale the running O row -- after the P store, when the S row's
                // registers are free.  Its last PV has completed: S_t(j) was issued
                // after it and s_full(t) covers it (P_SEP: the pv_done wait above).
                if (j > 0 && __any_sync(0xffffffffu, alpha < 1.f)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t raw[32];
                        tmem_ld32(o_addr + c * 32, raw);
#pragma unroll
                        for (int i = 0; i < 32; i += 2) {
                            float a0 = __uint_as_float(raw[i]), a1 = __uint_as_float(raw[i + 1]);
                            mul2(a0, a1, alpha);
                            raw[i] = __float_as_uint(a0);
                            raw[i + 1] = __float_as_uint(a1);
                        }
                        tmem_st32(o_addr + c * 32, raw);
                    }
                    tmem_st_wait();
                }
                tc_fence_before();
                mbar_arrive(p_full(t));
            }
            if (!ok) break;
            // epilogue: O / l -> bf16, LSE.  The MMA warp may already be
            // computing the next unit's S_t into this tile's S columns.
            if (!mbar_wait(o_final(t), uo & 1, tmo)) { ok = false; break; }
            ++uo;
            tc_fence_after();
            const float inv_l = (FP8 ? __ldg(p.v_scale + u.h) : 1.f) / l;
            const bool store = row < p.N;
            if constexpr (L::STG) {
                // Per 64-column half of the row: bf16 into this warp's staging area
                // (lane = row, 16-byte chunks XOR-swizzled by row, so both sweeps are
                // free of bank conflicts), then read back transposed -- eight lanes per
                // row, four rows per instruction -- so that every store writes whole
                // 128-byte row segments instead of 32 scattered 16-byte pieces.
                uint8_t* stg = smem + L::STG_OFF + (warp - 4) * 4096;
                // this lane's store target: row 4k + lane/8 of the warp's 32, columns
                // 8 (lane % 8) .. + 8 of the current 64-column half
                const int rr0 = lane >> 3, ch = lane & 7;
                const int row0 = u.q0 + 128 * t + 32 * wq + rr0;  // query row of k = 0
                const size_t row_stride = (size_t)p.H * D;        // elements between query rows
                __nv_bfloat16* obase = p.o + ((size_t)u.b * p.N + row0) * row_stride + (size_t)u.h * D + ch * 8;
#pragma unroll
                for (int c = 0; c < D / 64; ++c) {
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        uint32_t raw[32];
                        tmem_ld32(o_addr + c * 64 + c2 * 32, raw);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint4 v;
                            v.x = pack_bf16x2(__uint_as_float(raw[8 * q + 0]) * inv_l,
                                              __uint_as_float(raw[8 * q + 1]) * inv_l);
                            v.y = pack_bf16x2(__uint_as_float(raw[8 * q + 2]) * inv_l,
                                              __uint_as_float(raw[8 * q + 3]) * inv_l);
                            v.z = pack_bf16x2(__uint_as_float(raw[8 * q + 4]) * inv_l,
                                              __uint_as_float(raw[8 * q + 5]) * inv_l);
                            v.w = pack_bf16x2(__uint_as_float(raw[8 * q + 6]) * inv_l,
                                              __uint_as_float(raw[8 * q + 7]) * inv_l);
                            const int chw = 4 * c2 + q;  // 16-byte chunk of the 128-byte row
                            *reinterpret_cast<uint4*>(stg + lane * 128 + ((chw ^ (lane & 7)) << 4)) = v;
                        }
                    }
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int rr = 4 * k + rr0;
                        const uint4 v =
                            *reinterpret_cast<const uint4*>(stg + rr * 128 + ((ch ^ (rr & 7)) << 4));
                        if (row0 + 4 * k < p.N)
                            *reinterpret_cast<uint4*>(obase + (size_t)(4 * k) * row_stride + c * 64) = v;
                    }
                    __syncwarp();
                }
            } else {
                __nv_bfloat16* orow = p.o + (((size_t)u.b * p.N + (store ? row : 0)) * p.H + u.h) * D;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t raw[32];
                    tmem_ld32(o_addr + c * 32, raw);
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack_bf16x2(__uint_as_float(raw[2 * i]) * inv_l,
                                            __uint_as_float(raw[2 * i + 1]) * inv_l);
                    if (store) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    }
                }
            }
            if (store && p.lse != nullptr)
                p.lse[((size_t)u.b * p.H + u.h) * p.N + row] = (m + __log2f(l)) * kLn2;
        }
        if (!ok) record_status(ATTN_ERR_TIMEOUT);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

}  // namespace attn
