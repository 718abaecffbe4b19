// Backward (gradient) attention kernels for sm_103a.
//
// What they compute: the gradients of O = softmax(scale * Q K^T [+ causal mask]) V
// ("FlashAttention complete summary", section "Attention이 뭔가") for an upstream
// gradient dO, by recomputation: the N x N matrices S and P are rebuilt tile by tile
// from Q, K and the forward's row log-sum-exp instead of being stored ("Beyond the
// memory wall", section "FlashAttention: IO 인식의 정점": tiling and recomputation).
// With P = exp(scale * S - LSE):
//     dV = P^T dO,   dP = dO V^T,   D_i = dO_i . O_i,   dS = P * (dP - D),
//     dQ = scale * dS K,   dK = scale * dS^T Q.
//
// Three kernels, in stream order:
//   * bwd_prep_kernel: -D = -rowsum(dO * O) and -LSE * log2(e) into a workspace laid out
//     [B*H, Npad] (Npad = N rounded up to 128; 0 / -inf past N), one pass over O and dO
//     (negated, so that the compute warps form P and dS with packed adds and FMAs);
//   * bwd_kernel<.., KEY_TILES = true> (dK, dV): a persistent CTA per (b, h, 128-key tile).  K_j and V_j stay in
//     shared memory while (Q_i, dO_i, LSE_i, D_i) stream through a TMA ring.  Each query
//     tile is taken in two halves of 64 queries: S^T = K_j Q_i^T and dP^T = V_j dO_i^T of a
//     half (tcgen05, fp32 in tensor memory); eight warps turn them into P^T and dS^T (bf16,
//     written back into tensor memory); then dV += P^T dO_i and dK += dS^T Q_i accumulate
//     in tensor memory.  With the two halves in separate columns the tensor core works on
//     one half while the warps work on the other: the MMA order per query tile i is
//     grad(a, i), S/dP(a, i+1), grad(b, i), S/dP(b, i+1);
//   * bwd_kernel<.., KEY_TILES = false> (dQ): a persistent CTA per (b, h, 128-query tile) with Q_i, dO_i resident
//     and (K_j, V_j) streaming, in halves of 64 keys: S, dP, then dQ += dS K_j.
// No atomics: every output row is owned by one CTA, so results are deterministic.  The
// extra cost is recomputing S and dP in both kernels (7 products instead of 5).
//
// Causal: key tiles wholly above the diagonal are skipped in both kernels; the diagonal
// tile is masked.  Every wait is bounded in time (ATTN_ERR_TIMEOUT in the status word).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "prefill.cuh"  // prefill_unit_index: the snake-order deal of units to CTAs
#include "ptx.cuh"

namespace attn {

struct BwdParams {
    const __nv_bfloat16* o;     // forward output [B, N, H, d]   (prep)
    const __nv_bfloat16* dout;  // upstream gradient [B, N, H, d] (prep)
    const float* lse;           // forward LSE [B, H, N]          (prep)
    __nv_bfloat16* dq;
    __nv_bfloat16* dk;
    __nv_bfloat16* dv;
    float* ws_lse2;  // [B*H, Npad]: -LSE * log2(e), -inf for rows >= N
    float* ws_d;     // [B*H, Npad]: -rowsum(dO * O), 0 for rows >= N
    int B, H, N, Npad;
    float scale;       // softmax scale (dQ and dK carry one factor of it)
    float scale_log2;  // scale * log2(e)
    unsigned long long timeout_ns;
    int num_units;
    // Test hook (0 in normal use): the producer leaves its first resident-tile load
    // unissued, so the MMA warp's wait for it can only run out.
    int test_drop_load;
    // Long sequences (the DYN kernels): units numbered band by band of band_heads
    // (batch, head) pairs whose streamed tiles fit in L2, heaviest first within a
    // band, each CTA taking its next unit from *unit_counter (zero at launch).
    int band_heads;
    unsigned int* unit_counter;
};

template <int D>
struct BwdLayout {
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    static constexpr int KB = D / 64;               // 128-byte column blocks per row
    static constexpr int BOX_BYTES = 128 * 128;     // one TMA box: 128 rows x 64 bf16
    static constexpr int TILE_BYTES = 128 * D * 2;  // a 128-row tile of Q, K, V or dO
    static constexpr int VEC_BYTES = 2 * 128 * 4;   // LSE*log2(e) and D of one query tile
    static constexpr int NST = (D == 128) ? 2 : 4;  // ring stages, two tiles (+ vectors) each
    static constexpr int RES_OFF = 0;               // the two resident tiles
    static constexpr int ST_OFF = 2 * TILE_BYTES;
    static constexpr int ST_BYTES = 2 * TILE_BYTES + VEC_BYTES;  // keeps 1024-byte alignment
    static constexpr int BAR_OFF = ST_OFF + NST * ST_BYTES;
    static constexpr int NUM_BARS = 2 * NST + 8;
    // dynamic deal: a two-slot ring of units from the producer to the MMA warp and
    // the compute warps (full and empty barriers per slot, then per slot the unit
    // index, tile, batch and head), after the TMEM address
    static constexpr int UNIT_SLOTS = 2;
    static constexpr int UNIT_BAR_OFF = BAR_OFF + NUM_BARS * 8 + 16;
    static constexpr int UNIT_IDX_OFF = UNIT_BAR_OFF + 2 * UNIT_SLOTS * 8;
    static constexpr int UNIT_READERS = 1 + 8;
    static constexpr int SMEM_BYTES = UNIT_IDX_OFF + UNIT_SLOTS * 16 + 1024;
    static constexpr int THREADS = 384;             // 4 control warps + 8 compute warps
    static constexpr int COMPUTE_THREADS = 256;
    // tensor memory columns: per half h of the streamed tile (64 streamed rows) S (or
    // S^T) at 128 h and dP (or dP^T) at 128 h + 64, then the accumulators
    static constexpr int DP_OFF = 64;
    static constexpr int ACC0_COL = 256;            // dV (dK/dV kernel) or dQ (dQ kernel)
    static constexpr int ACC1_COL = 256 + D;        // dK
    static constexpr int TMEM_COLS = 512;
    // Where tensor memory has room after the accumulators (the dQ kernel; the dK/dV
    // kernel at d=64), the two resident tiles are copied into it once per unit and the
    // S-type products read their A operand from there: an M=128, N=64 product with
    // both operands in shared memory needs 6 KB per k-step, more than shared memory
    // delivers in the step's 32 tensor cycles (measured at 2/3 of the tensor rate),
    // while with A in tensor memory it reads 2 KB and runs at the full rate.
    template <bool KEY_TILES>
    __host__ __device__ static constexpr bool res_in_tmem() { return !KEY_TILES || D == 64; }
    template <bool KEY_TILES>
    __host__ __device__ static constexpr int res_col() { return KEY_TILES ? ACC1_COL + D : ACC0_COL + D; }
    static_assert(ST_BYTES % 1024 == 0, "stage alignment");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// Tensor-memory column, relative to the S (or dP) columns of half h, of the bf16 A operand
// (P^T, dS^T or dS) for k-step k = 0..3 of that half (16 streamed rows each): the compute
// warps of column group g own 32 streamed rows and pack them, two per column, into the
// first 16 of their own 32 columns.
__device__ __forceinline__ uint32_t bwd_a_col(int h, int k) {
    return 128u * h + 32u * (k >> 1) + 8u * (k & 1);
}

// Unit k of the persistent grid: the tile index (keys for dK/dV, queries for dQ) and the
// (b, h) pair.  Causal units are numbered heaviest first: key tile 0 meets every query
// tile; query tile nt-1 meets every key tile.
// BANDED: numbered band by band of p.band_heads (batch, head) pairs (the last band
// may be narrower), tiles heaviest first within a band, heads inner.
template <bool CAUSAL, bool KEY_TILES, bool BANDED = false>
__device__ __forceinline__ void bwd_unit(const BwdParams& p, int k, int& tile, int& b, int& h) {
    const int BH = p.B * p.H;
    const int nt = (p.N + 127) / 128;
    int t, bh;
    if constexpr (BANDED) {
        const int per_band = p.band_heads * nt;
        const int band = k / per_band;
        const int r = k - band * per_band;
        const int heads = min(p.band_heads, BH - band * p.band_heads);
        t = r / heads;
        bh = band * p.band_heads + (r - t * heads);
    } else {
        t = k / BH;
        bh = k % BH;
    }
    if (CAUSAL && !KEY_TILES) t = nt - 1 - t;
    tile = t;
    b = bh / p.H;
    h = bh % p.H;
}

// ---------------------------------------------------------------------------- prep --
// One row (b, h, n) of -D and -LSE*log2(e) per D/8 lanes (16-byte loads of O and dO).
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const BwdParams p) {
    constexpr int LPR = D / 8;       // lanes per row
    constexpr int RPW = 32 / LPR;    // rows per warp
    const long long warp_id = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long long total = (long long)p.B * p.H * p.Npad;
    const long long row = warp_id * RPW + lane / LPR;
    const int sub = lane % LPR;
    float acc = 0.f;
    bool valid = false;
    long long bh = 0, n = 0;
    if (row < total) {
        bh = row / p.Npad;
        n = row % p.Npad;
        if (n < p.N) {
            valid = true;
            const long long b = bh / p.H, h = bh % p.H;
            const size_t base = (((size_t)b * p.N + n) * p.H + h) * D + sub * 8;
            const uint4 o4 = *reinterpret_cast<const uint4*>(p.o + base);
            const uint4 g4 = *reinterpret_cast<const uint4*>(p.dout + base);
            const uint32_t ow[4] = {o4.x, o4.y, o4.z, o4.w}, gw[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc = fmaf(__uint_as_float(ow[i] << 16), __uint_as_float(gw[i] << 16), acc);
                acc = fmaf(__uint_as_float(ow[i] & 0xffff0000u), __uint_as_float(gw[i] & 0xffff0000u), acc);
            }
        }
    }
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row < total && sub == 0) {
        p.ws_d[row] = valid ? -acc : 0.f;
        p.ws_lse2[row] = valid ? -(p.lse[bh * p.N + n] * kLog2e) : -INFINITY;
    }
}

// Shared memory -> tensor memory copy of a 128-row x 32-byte slice of a K-major
// tile (the slice one MMA k-step reads), described by a shared-memory matrix
// descriptor as for tcgen05.mma: row r lands in lane r, 8 consecutive 32-bit
// columns, two bf16 per column (the A-operand layout the .ts MMA reads).
// Asynchronous, in order with the issuing thread's later MMAs.
__device__ __forceinline__ void tmem_cp_128x256b(uint32_t taddr, uint32_t d_lo, uint32_t d_hi) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .b64 d;\n\t"
        "mov.b64 d, {%1, %2};\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.cp.cta_group::1.128x256b [%0], d;\n\t}" ::"r"(taddr),
        "r"(d_lo), "r"(d_hi)
        : "memory");
}

// bf16 pack of 32 fp32 values (optionally times `mul`) and a 64-byte row store.
__device__ __forceinline__ void bwd_store32(__nv_bfloat16* dst, const uint32_t (&raw)[32], float mul,
                                            bool store) {
    uint32_t pk[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        pk[i] = pack_bf16x2(__uint_as_float(raw[2 * i]) * mul, __uint_as_float(raw[2 * i + 1]) * mul);
    if (store) {
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int i = 0; i < 4; ++i) d4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
    }
}

// ------------------------------------------------------------------- dK/dV and dQ --
// KEY_TILES = true: the dK/dV kernel (resident K_j, V_j; streaming Q_i, dO_i, vectors).
// KEY_TILES = false: the dQ kernel (resident Q_i, dO_i; streaming K_j, V_j).
template <int D, bool CAUSAL, bool KEY_TILES, bool DYN>
__global__ void __launch_bounds__(384, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
               const BwdParams p) {
    using L = BwdLayout<D>;
    // resident tiles in tensor memory: A at RA_COL, B at RB_COL (D / 2 columns each)
    constexpr bool RES_TMEM = L::template res_in_tmem<KEY_TILES>();
    constexpr int RA_COL = L::template res_col<KEY_TILES>();
    constexpr int RB_COL = RA_COL + D / 2;
    static_assert(!RES_TMEM || RB_COL + D / 2 <= L::TMEM_COLS, "resident tiles fit in tensor memory");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::BAR_OFF;
    constexpr int NST = L::NST;
    const uint32_t res_full = bar0, res_empty = bar0 + 8;
    auto st_full = [&](int s) { return bar0 + 8u * (2 + s); };
    auto st_empty = [&](int s) { return bar0 + 8u * (2 + NST + s); };
    // per half h: its S and dP are in tensor memory / its P and dS are written back
    auto sdp_full = [&](int h) { return bar0 + 8u * (2 + 2 * NST + h); };
    auto p_ready = [&](int h) { return bar0 + 8u * (4 + 2 * NST + h); };
    const uint32_t acc_full = bar0 + 8u * (6 + 2 * NST);
    const uint32_t drain_bar = bar0 + 8u * (7 + 2 * NST);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::BAR_OFF + L::NUM_BARS * 8);
    // DYN: the ring of units (see BwdLayout)
    auto unit_full = [&](int s) { return sbase + L::UNIT_BAR_OFF + 8u * s; };
    auto unit_empty = [&](int s) { return sbase + L::UNIT_BAR_OFF + 8u * (L::UNIT_SLOTS + s); };
    volatile int* unit_idx = reinterpret_cast<volatile int*>(smem + L::UNIT_IDX_OFF);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nt = (p.N + 127) / 128;
    // other-operand tiles a unit visits: [lo, hi)
    auto range = [&](int tile, int& lo, int& hi) {
        if (KEY_TILES) {
            lo = CAUSAL ? tile : 0;
            hi = nt;
        } else {
            lo = 0;
            hi = CAUSAL ? tile + 1 : nt;
        }
    };

    if (threadIdx.x == 0) {
        mbar_init(res_full, 1);
        mbar_init(res_empty, 1);
        for (int s = 0; s < NST; ++s) {
            mbar_init(st_full(s), 1);
            mbar_init(st_empty(s), 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(sdp_full(h), 1);
            mbar_init(p_ready(h), L::COMPUTE_THREADS);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain_bar, 1);
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint64_t tmo = p.timeout_ns;
    const uint64_t tdrain = tmo > kDrainTimeoutNs ? tmo : kDrainTimeoutNs;  // wind-down waits
    // The unit of this CTA's `round`-th step for the MMA and compute warps (whole warp):
    // the static snake deal, or (DYN) the ring the producer fills; false ends the loop
    // (ok = false if a wait ran out).
    auto unit_of_round = [&](int round, bool& ok, int& tile, int& b, int& h) -> bool {
        if constexpr (!DYN) {
            const int k = prefill_unit_index(round);
            if (k >= p.num_units) return false;
            bwd_unit<CAUSAL, KEY_TILES>(p, k, tile, b, h);
            return true;
        } else {
            const int sl = round % L::UNIT_SLOTS;
            if (!mbar_wait_warp(unit_full(sl), (round / L::UNIT_SLOTS) & 1, tmo)) {
                ok = false;
                return false;
            }
            const int k = unit_idx[4 * sl];
            tile = unit_idx[4 * sl + 1];
            b = unit_idx[4 * sl + 2];
            h = unit_idx[4 * sl + 3];
            __syncwarp();
            if ((threadIdx.x & 31) == 0) mbar_arrive(unit_empty(sl));
            return k < p.num_units;
        }
    };

    if (warp == 0) {
        // ============================== TMA producer ===============================
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            prefetch_tensormap(&tm_do);
        }
        // resident: K_j, V_j (dK/dV) or Q_i, dO_i (dQ); streaming: the other pair
        const CUtensorMap* res_a = KEY_TILES ? &tm_k : &tm_q;
        const CUtensorMap* res_b = KEY_TILES ? &tm_v : &tm_do;
        const CUtensorMap* st_a = KEY_TILES ? &tm_q : &tm_k;
        const CUtensorMap* st_b = KEY_TILES ? &tm_do : &tm_v;
        int nres = 0, ns = 0;
        bool ok = true;
        // DYN: lane 0 takes the next unit index from the device counter three streamed
        // tiles before the current unit's loads end (its latency hidden, the unit
        // claimed close to when this CTA needs it) and publishes it decoded
        unsigned int taken = 0;
        if (DYN && lane == 0) taken = atomicAdd(p.unit_counter, 1u);
        for (int round = 0; ok; ++round) {
            int tile = 0, b = 0, h = 0, lo, hi;
            if constexpr (DYN) {
                const int k = (int)min(__shfl_sync(0xffffffffu, taken, 0), (unsigned int)p.num_units);
                const int sl = round % L::UNIT_SLOTS;
                if (!mbar_wait_warp(unit_empty(sl), ((round / L::UNIT_SLOTS) & 1) ^ 1, tmo)) {
                    ok = false;
                    break;
                }
                if (k < p.num_units) bwd_unit<CAUSAL, KEY_TILES, true>(p, k, tile, b, h);
                if (lane == 0) {
                    unit_idx[4 * sl] = k;
                    unit_idx[4 * sl + 1] = tile;
                    unit_idx[4 * sl + 2] = b;
                    unit_idx[4 * sl + 3] = h;
                    mbar_arrive(unit_full(sl));
                }
                __syncwarp();
                if (k >= p.num_units) break;
            } else {
                const int k = prefill_unit_index(round);
                if (k >= p.num_units) break;
                bwd_unit<CAUSAL, KEY_TILES>(p, k, tile, b, h);
            }
            range(tile, lo, hi);
            if (!mbar_wait_warp(res_empty, (nres & 1) ^ 1, tmo)) { ok = false; break; }
            const bool drop = p.test_drop_load && nres == 0;  // test hook: res_full never completes
            if (lane == 0 && !drop) mbar_arrive_expect_tx(res_full, 2 * L::TILE_BYTES);
            __syncwarp();
            if (lane < L::KB && !drop) {
                tma_load_4d(sbase + L::RES_OFF + lane * L::BOX_BYTES, res_a, res_full, lane * 64, h,
                            tile * 128, b);
                tma_load_4d(sbase + L::RES_OFF + L::TILE_BYTES + lane * L::BOX_BYTES, res_b, res_full,
                            lane * 64, h, tile * 128, b);
            }
            ++nres;
            for (int t = lo; t < hi; ++t) {
                if (DYN && lane == 0 && t == max(lo, hi - 3)) taken = atomicAdd(p.unit_counter, 1u);
                const int st = ns % NST;
                if (!mbar_wait_warp(st_empty(st), ((ns / NST) & 1) ^ 1, tmo)) { ok = false; break; }
                const uint32_t dst = sbase + L::ST_OFF + st * L::ST_BYTES;
                if (lane == 0)
                    mbar_arrive_expect_tx(st_full(st),
                                          2 * L::TILE_BYTES + (KEY_TILES ? L::VEC_BYTES : 0));
                __syncwarp();
                if (lane < L::KB) {
                    tma_load_4d(dst + lane * L::BOX_BYTES, st_a, st_full(st), lane * 64, h, t * 128, b);
                    tma_load_4d(dst + L::TILE_BYTES + lane * L::BOX_BYTES, st_b, st_full(st), lane * 64,
                                h, t * 128, b);
                }
                if (KEY_TILES && lane == 31) {
                    const size_t v0 = ((size_t)b * p.H + h) * p.Npad + (size_t)t * 128;
                    bulk_load(dst + 2 * L::TILE_BYTES, p.ws_lse2 + v0, 512, st_full(st));
                    bulk_load(dst + 2 * L::TILE_BYTES + 512, p.ws_d + v0, 512, st_full(st));
                }
                ++ns;
            }
        }
        if (!ok && lane == 0) record_status(ATTN_ERR_TIMEOUT);
        // copies still in flight land before the CTA can exit (immediate after a normal run)
        if (nres > 0 && !(p.test_drop_load && nres == 1)) mbar_wait(res_full, (nres - 1) & 1, tdrain);
        for (int x = max(0, ns - NST); x < ns; ++x) mbar_wait(st_full(x % NST), (x / NST) & 1, tdrain);
    } else if (warp == 1) {
        // =============================== MMA issuer ================================
        // S-type products (M = 128 rows of the resident tile, N = 64 rows of one half of
        // the streamed tile, K = d): both operands K-major.  Gradient products (M = 128,
        // N = d, K = the 64 rows of a half): A = bf16 from tensor memory, B MN-major (d
        // contiguous, 64-wide blocks BOX_BYTES apart).
        constexpr uint32_t kIdescS = idesc_bf16_f32(128, 64, false, false);
        constexpr uint32_t kIdescG = idesc_bf16_f32(128, D, false, true);
        const uint64_t d_ra = sdesc_sw128(sbase + L::RES_OFF, 16, 1024);
        const uint64_t d_rb = sdesc_sw128(sbase + L::RES_OFF + L::TILE_BYTES, 16, 1024);
        const uint64_t d_sa = sdesc_sw128(sbase + L::ST_OFF, 16, 1024);
        const uint64_t d_sa_mn = sdesc_sw128(sbase + L::ST_OFF, L::BOX_BYTES, 1024);
        const uint32_t hi_k = (uint32_t)(d_ra >> 32), hi_mn = (uint32_t)(d_sa_mn >> 32);
        const uint32_t ra_lo = (uint32_t)d_ra, rb_lo = (uint32_t)d_rb;
        const uint32_t sa_lo = (uint32_t)d_sa, sa_mn_lo = (uint32_t)d_sa_mn;
        // S and dP of half h of the streamed tiles in stage st (dK/dV: S^T = K_j Q_h^T,
        // dP^T = V_j dO_h^T; dQ: S = Q_i K_h^T, dP = dO_i V_h^T).  Rows 64 h.. of a
        // streamed tile start 64 * 128 bytes into each 64-column box.
        // (RES_TMEM: the resident operand from its tensor-memory copy, 8 columns per k-step.)
        auto issue_sd = [&](int h, int st) {
            const uint32_t a_off = (st * L::ST_BYTES + h * 64 * 128) >> 4;
            const uint32_t b_off = (st * L::ST_BYTES + L::TILE_BYTES + h * 64 * 128) >> 4;
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t off = ((k >> 2) * L::BOX_BYTES + (k & 3) * 32) >> 4;
                if constexpr (RES_TMEM)
                    umma_ts(tmem + 128 * h, tmem + RA_COL + 8 * k, sa_lo + a_off + off, hi_k, kIdescS,
                            k > 0 ? 1u : 0u);
                else
                    umma_ss(tmem + 128 * h, ra_lo + off, hi_k, sa_lo + a_off + off, hi_k, kIdescS,
                            k > 0 ? 1u : 0u);
            }
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t off = ((k >> 2) * L::BOX_BYTES + (k & 3) * 32) >> 4;
                if constexpr (RES_TMEM)
                    umma_ts(tmem + 128 * h + L::DP_OFF, tmem + RB_COL + 8 * k, sa_lo + b_off + off, hi_k,
                            kIdescS, k > 0 ? 1u : 0u);
                else
                    umma_ss(tmem + 128 * h + L::DP_OFF, rb_lo + off, hi_k, sa_lo + b_off + off, hi_k,
                            kIdescS, k > 0 ? 1u : 0u);
            }
        };
        // RES_TMEM: copy both resident tiles into tensor memory, k-step by k-step.  The
        // previous unit's S-type products, the only readers of these columns, have
        // completed: the compute warps consumed every S/dP they wrote (the last p_ready
        // waits of that unit) before this warp gets here.
        auto copy_res = [&]() {
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const uint32_t off = ((k >> 2) * L::BOX_BYTES + (k & 3) * 32) >> 4;
                tmem_cp_128x256b(tmem + RA_COL + 8 * k, ra_lo + off, hi_k);
                tmem_cp_128x256b(tmem + RB_COL + 8 * k, rb_lo + off, hi_k);
            }
        };
        // acc[col] (+)= A[half h's bf16 operand at column part a_part] * B[MN-major tile
        // b_lo, rows 64 h .. 64 h + 63]
        auto issue_g = [&](uint32_t col, uint32_t a_part, uint32_t b_lo, int h, bool acc) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t boff = ((64 * h + 16 * k) * 128) >> 4;
                umma_ts(tmem + col, tmem + a_part + bwd_a_col(h, k), b_lo + boff, hi_mn, kIdescG,
                        (acc || k > 0) ? 1u : 0u);
            }
        };
        int nres = 0, ns = 0;
        int np[2] = {0, 0};
        bool ok = true;
        for (int round = 0; ok; ++round) {
            int tile, b, h, lo, hi;
            if (!unit_of_round(round, ok, tile, b, h)) break;
            range(tile, lo, hi);
            if (!mbar_wait_warp(res_full, nres & 1, tmo)) { ok = false; break; }
            ++nres;
            if constexpr (RES_TMEM) {
                // the shared-memory copies are read only by the tensor-memory copy: release
                // them as soon as it completes, so the next unit's tiles can load early
                tc_fence_after();
                copy_res();
                umma_commit(res_empty);
            }
            // prologue: both halves of the first streamed tile
            {
                const int st = ns % NST;
                if (!mbar_wait_warp(st_full(st), (ns / NST) & 1, tmo)) { ok = false; break; }
                tc_fence_after();
                issue_sd(0, st);
                umma_commit(sdp_full(0));
                issue_sd(1, st);
                umma_commit(sdp_full(1));
            }
            for (int t = lo; t < hi; ++t) {
                const int st = ns % NST, stn = (ns + 1) % NST;
                const bool more = t + 1 < hi;
                const uint32_t s_off = (st * L::ST_BYTES) >> 4;
                const uint32_t t_off = (st * L::ST_BYTES + L::TILE_BYTES) >> 4;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    if (!mbar_wait_warp(p_ready(hh), np[hh] & 1, tmo)) { ok = false; break; }
                    ++np[hh];
                    tc_fence_after();
                    const bool acc = t > lo || hh > 0;
                    if (KEY_TILES) {
                        issue_g(L::ACC0_COL, 0, sa_mn_lo + t_off, hh, acc);          // dV += P^T dO_h
                        issue_g(L::ACC1_COL, L::DP_OFF, sa_mn_lo + s_off, hh, acc);  // dK += dS^T Q_h
                    } else {
                        issue_g(L::ACC0_COL, 0, sa_mn_lo + s_off, hh, acc);          // dQ += dS K_h
                    }
                    if (hh == 1) umma_commit(st_empty(st));
                    if (more) {
                        // half hh of the next streamed tile into the columns just read
                        if (hh == 0) {
                            if (!mbar_wait_warp(st_full(stn), ((ns + 1) / NST) & 1, tmo)) { ok = false; break; }
                            tc_fence_after();
                        }
                        issue_sd(hh, stn);
                        umma_commit(sdp_full(hh));
                    }
                }
                if (!ok) break;
                ++ns;
            }
            if (!ok) break;
            umma_commit(acc_full);
            if constexpr (!RES_TMEM) umma_commit(res_empty);
        }
        if (!ok && lane == 0) record_status(ATTN_ERR_TIMEOUT);
        umma_commit(drain_bar);
        mbar_wait(drain_bar, 0, tdrain);
    } else if (warp >= 4) {
        // ============================ compute warps ================================
        // Thread (quarter wq, group hf) owns TMEM lane r = 32 wq + lane (a row of the
        // resident tile) and, in each half of the streamed tile, the 32 streamed rows
        // [32 hf, 32 hf + 32) of that half: 32 columns of its S and of its dP.
        const int wq = warp & 3;
        const int hf = (warp - 4) >> 2;
        const int r = wq * 32 + lane;
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const float sl2 = p.scale_log2;
        int ns = 0, nacc = 0;
        int nsd[2] = {0, 0};
        bool ok = true;
        for (int round = 0; ok; ++round) {
            int tile, b, h, lo, hi;
            if (!unit_of_round(round, ok, tile, b, h)) break;
            range(tile, lo, hi);
            const size_t vrow = ((size_t)b * p.H + h) * p.Npad + (size_t)tile * 128 + r;
            // dQ kernel: this row's -LSE*log2(e) and -D (-inf / 0 past N)
            const float nlse2_r = KEY_TILES ? 0.f : __ldg(p.ws_lse2 + vrow);
            const float nd_r = KEY_TILES ? 0.f : __ldg(p.ws_d + vrow);
            for (int t = lo; t < hi; ++t) {
                const int st = ns % NST;
                const uint32_t st_phase = (ns / NST) & 1;
                ++ns;
                const float* vec = reinterpret_cast<const float*>(smem + L::ST_OFF + st * L::ST_BYTES +
                                                                  2 * L::TILE_BYTES);
                const bool diag = CAUSAL && t == tile;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    if (!mbar_wait(sdp_full(hh), nsd[hh] & 1, tmo)) { ok = false; break; }
                    ++nsd[hh];
                    // the stage's LSE/D vectors were written by TMA: observe its completion
                    // here too (the stage cannot be refilled before this thread arrives on
                    // p_ready of both halves, so the phase is still the one of this tile)
                    if (KEY_TILES && hh == 0 && !mbar_wait(st_full(st), st_phase, tmo)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t s_addr = tmem + lane_off + 128 * hh + 32 * hf;
                    const uint32_t dp_addr = s_addr + L::DP_OFF;
                    const int col0 = 64 * hh + 32 * hf;   // streamed row within the 128-row tile
                    uint32_t sr[32], dr[32];
                    tmem_ld32x2(s_addr, sr, dp_addr, dr);
                    // P = 2^(S * scale * log2(e) - LSE * log2(e)) and dS = P * (dP - D), two
                    // columns per packed f32x2 step.  dK/dV: row r = key, column = query, the
                    // subtrahends per column from the stage's vectors; dQ: row r = query,
                    // column = key, the subtrahends this row's.
                    float pv[32], dsv[32];
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        float4 nl, nd;
                        if (KEY_TILES) {
                            nl = *reinterpret_cast<const float4*>(vec + col0 + e);
                            nd = *reinterpret_cast<const float4*>(vec + 128 + col0 + e);
                        } else {
                            nl = make_float4(nlse2_r, nlse2_r, nlse2_r, nlse2_r);
                            nd = make_float4(nd_r, nd_r, nd_r, nd_r);
                        }
                        fma2(pv[e], pv[e + 1], __uint_as_float(sr[e]), __uint_as_float(sr[e + 1]), sl2, sl2,
                             nl.x, nl.y);
                        fma2(pv[e + 2], pv[e + 3], __uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3]), sl2,
                             sl2, nl.z, nl.w);
#pragma unroll
                        for (int x = 0; x < 4; ++x) pv[e + x] = ex2_approx(pv[e + x]);
                        add2v(dsv[e], dsv[e + 1], __uint_as_float(dr[e]), __uint_as_float(dr[e + 1]), nd.x, nd.y);
                        add2v(dsv[e + 2], dsv[e + 3], __uint_as_float(dr[e + 2]), __uint_as_float(dr[e + 3]),
                              nd.z, nd.w);
                    }
                    // causal diagonal tile (dK/dV: query < key; dQ: key > query) and, in the dQ
                    // kernel, keys past N: P = 0
                    const bool tail = !KEY_TILES && (t + 1) * 128 > p.N;
                    if (diag || tail) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int col = col0 + e;
                            const bool drop = KEY_TILES ? (diag && col < r)
                                                        : ((diag && col > r) || t * 128 + col >= p.N);
                            if (drop) pv[e] = 0.f;
                        }
                    }
                    uint32_t pp[16], pd[16];
#pragma unroll
                    for (int e = 0; e < 32; e += 2) {
                        mul2v(dsv[e], dsv[e + 1], pv[e], pv[e + 1], dsv[e], dsv[e + 1]);
                        pp[e / 2] = pack_bf16x2(pv[e], pv[e + 1]);
                        pd[e / 2] = pack_bf16x2(dsv[e], dsv[e + 1]);
                    }
                    // packed entries go to the first 16 of this thread's 32 columns, which
                    // it has already read
                    if (KEY_TILES) {
                        tmem_st16(s_addr, pp);    // P^T
                        tmem_st16(dp_addr, pd);   // dS^T
                    } else {
                        tmem_st16(s_addr, pd);    // dS
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    mbar_arrive(p_ready(hh));
                }
                if (!ok) break;
            }
            if (!ok) break;
            // epilogue: this thread's row, columns [hf d/2, (hf+1) d/2) of each accumulator
            if (!mbar_wait(acc_full, nacc & 1, tmo)) { ok = false; break; }
            ++nacc;
            tc_fence_after();
            const int row = tile * 128 + r;
            const bool store = row < p.N;
            const size_t obase = (((size_t)b * p.N + (store ? row : 0)) * p.H + h) * D + hf * (D / 2);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t raw[32];
                tmem_ld32(tmem + lane_off + L::ACC0_COL + hf * (D / 2) + 32 * c, raw);
                if (KEY_TILES)
                    bwd_store32(p.dv + obase + 32 * c, raw, 1.f, store);
                else
                    bwd_store32(p.dq + obase + 32 * c, raw, p.scale, store);
                if (KEY_TILES) {
                    tmem_ld32(tmem + lane_off + L::ACC1_COL + hf * (D / 2) + 32 * c, raw);
                    bwd_store32(p.dk + obase + 32 * c, raw, p.scale, store);
                }
            }
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
