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
//   * one CTA owns QT query tiles of 128 rows of one (batch, head);
//   * warp 0 (one lane) is the TMA producer: Q tiles once, then K_j and V_j
//     tiles of 128 keys into a STAGES-deep shared-memory ring (128-byte
//     swizzle, completion counted on mbarriers);
//   * warp 1 (one lane) issues tcgen05.mma: S_t = Q_t K_j^T into tensor memory
//     (M=128, N=128, fp32), and O_t += P_t V_j with P_t read from tensor memory
//     (or shared memory) and O_t accumulated in tensor memory;
//   * warps 4.. form one 128-thread softmax group per query tile: thread r owns
//     row r (TMEM lane r), reads its S row, applies the causal / tail mask,
//     updates m and l, rescales its O row when m grew, writes P (bf16) back and
//     signals the MMA warp; at the end it divides O by l and stores O and LSE;
//   * the MMA order per key block j is PV_0(j), S_0(j+1), PV_1(j), S_1(j+1), so
//     the tensor core works on one tile while the other tile's softmax runs;
//   * causal: key blocks wholly above the diagonal are never loaded; only the
//     diagonal block is masked.  CTAs are numbered heaviest-first.
// Every wait is bounded in time; on expiry the kernel records ATTN_ERR_TIMEOUT
// in the device status word and winds down instead of hanging.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace attn {

struct PrefillParams {
    __nv_bfloat16* o;
    float* lse;
    int B, H, N;
    float scale_log2;  // scale * log2(e)
    unsigned long long timeout_ns;
};

template <int D, int QT, bool P_TMEM>
struct PrefillLayout {
    static_assert(D == 64 || D == 128, "head_dim 64 or 128");
    static_assert(QT == 1 || QT == 2, "one or two query tiles per CTA");
    static_assert(P_TMEM || QT == 1, "P in shared memory only with one query tile");
    static constexpr int BM = 128;                 // query rows per tile = TMEM lanes
    static constexpr int BN = 128;                 // keys per block
    static constexpr int KB = D / 64;              // 128-byte column blocks per row
    static constexpr int BOX_BYTES = 128 * 128;    // one TMA box: 128 rows x 64 bf16
    static constexpr int TILE_BYTES = 128 * D * 2; // Q, K or V tile
    static constexpr int P_BYTES = P_TMEM ? 0 : 128 * 128 * 2;
    static constexpr int STAGES = (D == 128) ? 2 : 3;
    static constexpr int THREADS = 128 + 128 * QT;
    // shared memory (offsets from a 1024-byte aligned base)
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + QT * TILE_BYTES;
    static constexpr int V_OFF = K_OFF + STAGES * TILE_BYTES;
    static constexpr int P_OFF = V_OFF + STAGES * TILE_BYTES;
    static constexpr int BAR_OFF = P_OFF + P_BYTES;
    static constexpr int NUM_BARS = 1 + 4 * STAGES + 3 * QT + 1;
    static constexpr int SMEM_BYTES = BAR_OFF + NUM_BARS * 8 + 16 + 1024;  // + alignment slack
    // tensor memory columns
    static constexpr int S_COL0 = 0;          // S_t at t*128 (P_t aliases its first 64 columns)
    static constexpr int O_COL0 = QT * 128;   // O_t at O_COL0 + t*D
    static constexpr int TMEM_COLS = (QT * (128 + D) <= 256) ? 256 : 512;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <int D, bool CAUSAL, int QT, bool P_TMEM>
__global__ void __launch_bounds__(128 + 128 * QT, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
    using L = PrefillLayout<D, QT, P_TMEM>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::BAR_OFF;
    // barrier addresses
    const uint32_t q_full = bar0;
    auto k_full = [&](int s) { return bar0 + 8u * (1 + s); };
    auto k_empty = [&](int s) { return bar0 + 8u * (1 + L::STAGES + s); };
    auto v_full = [&](int s) { return bar0 + 8u * (1 + 2 * L::STAGES + s); };
    auto v_empty = [&](int s) { return bar0 + 8u * (1 + 3 * L::STAGES + s); };
    auto s_full = [&](int t) { return bar0 + 8u * (1 + 4 * L::STAGES + t); };
    auto p_full = [&](int t) { return bar0 + 8u * (1 + 4 * L::STAGES + QT + t); };
    auto o_final = [&](int t) { return bar0 + 8u * (1 + 4 * L::STAGES + 2 * QT + t); };
    const uint32_t drain_bar = bar0 + 8u * (1 + 4 * L::STAGES + 3 * QT);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::BAR_OFF + L::NUM_BARS * 8);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work unit: (query-tile group, batch, head), heaviest group first for causal
    const int BH = p.B * p.H;
    const int n_groups = (p.N + 128 * QT - 1) / (128 * QT);
    int grp = blockIdx.x / BH;
    if (CAUSAL) grp = n_groups - 1 - grp;
    const int bh = blockIdx.x % BH;
    const int b = bh / p.H;
    const int h = bh % p.H;
    const int q0 = grp * 128 * QT;
    const int n_kv_all = (p.N + 127) / 128;
    int nkv[QT];
    int n_active = 0, nkv_max = 0;
#pragma unroll
    for (int t = 0; t < QT; ++t) {
        const int r0 = q0 + 128 * t;
        nkv[t] = (r0 >= p.N) ? 0 : (CAUSAL ? min(n_kv_all, r0 / 128 + 1) : n_kv_all);
        if (nkv[t] > 0) n_active = t + 1;
        nkv_max = max(nkv_max, nkv[t]);
    }

    // ---- setup: barriers (thread 0), tensor memory (warp 2)
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < L::STAGES; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), 1);
            mbar_init(v_full(s), 1);
            mbar_init(v_empty(s), 1);
        }
        for (int t = 0; t < QT; ++t) {
            mbar_init(s_full(t), 1);
            mbar_init(p_full(t), 128);
            mbar_init(o_final(t), 1);
        }
        mbar_init(drain_bar, 1);
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

    if (warp == 0) {
        // =========================== TMA producer ===========================
        if (lane == 0) {
            prefetch_tensormap(&tm_q);
            prefetch_tensormap(&tm_k);
            prefetch_tensormap(&tm_v);
            mbar_arrive_expect_tx(q_full, n_active * L::TILE_BYTES);
            for (int t = 0; t < n_active; ++t)
                for (int kb = 0; kb < L::KB; ++kb)
                    tma_load_4d(sbase + L::Q_OFF + t * L::TILE_BYTES + kb * L::BOX_BYTES, &tm_q,
                                q_full, kb * 64, h, q0 + 128 * t, b);
            int issued = 0;
            bool ok = true;
            for (int j = 0; j < nkv_max; ++j) {
                const int st = j % L::STAGES;
                const uint32_t ph = (j / L::STAGES) & 1;
                if (!mbar_wait(k_empty(st), ph ^ 1, tmo)) { ok = false; break; }
                mbar_arrive_expect_tx(k_full(st), L::TILE_BYTES);
                for (int kb = 0; kb < L::KB; ++kb)
                    tma_load_4d(sbase + L::K_OFF + st * L::TILE_BYTES + kb * L::BOX_BYTES, &tm_k,
                                k_full(st), kb * 64, h, j * 128, b);
                if (!mbar_wait(v_empty(st), ph ^ 1, tmo)) { ok = false; issued = j * 2 + 1; break; }
                mbar_arrive_expect_tx(v_full(st), L::TILE_BYTES);
                for (int kb = 0; kb < L::KB; ++kb)
                    tma_load_4d(sbase + L::V_OFF + st * L::TILE_BYTES + kb * L::BOX_BYTES, &tm_v,
                                v_full(st), kb * 64, h, j * 128, b);
                issued = j * 2 + 2;
            }
            if (!ok) {
                record_status(ATTN_ERR_TIMEOUT);
                // let copies already in flight land before the CTA can exit
                mbar_wait(q_full, 0, tmo);
                for (int x = max(0, issued - 2 * L::STAGES); x < issued; ++x) {
                    const int j = x / 2, st = j % L::STAGES;
                    const uint32_t ph = (j / L::STAGES) & 1;
                    mbar_wait((x & 1) ? v_full(st) : k_full(st), ph, tmo);
                }
            }
        }
    } else if (warp == 1) {
        // ============================ MMA issuer ============================
        if (lane == 0) {
            constexpr uint32_t kIdescS = idesc_bf16_f32(128, 128, false, false);
            constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);
            bool ok = mbar_wait(q_full, 0, tmo) && mbar_wait(k_full(0), 0, tmo);
            tc_fence_after();
            auto issue_s = [&](int t, int st) {
                const uint32_t a0 = sbase + L::Q_OFF + t * L::TILE_BYTES;
                const uint32_t b0 = sbase + L::K_OFF + st * L::TILE_BYTES;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k >> 2) * L::BOX_BYTES + (k & 3) * 32;
                    umma_ss(tmem + L::S_COL0 + t * 128, sdesc_sw128(a0 + off, 16, 1024),
                            sdesc_sw128(b0 + off, 16, 1024), kIdescS, k > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int t, int st, bool acc) {
                const uint32_t v0 = sbase + L::V_OFF + st * L::TILE_BYTES;
#pragma unroll
                for (int k = 0; k < 128 / 16; ++k) {
                    // B = V_j, MN-major: 16 keys x 128 B per k-step; 64-wide d blocks at BOX_BYTES
                    const uint64_t bdesc = sdesc_sw128(v0 + k * 16 * 128, L::BOX_BYTES, 1024);
                    const uint32_t accf = (acc || k > 0) ? 1u : 0u;
                    if constexpr (P_TMEM) {
                        umma_ts(tmem + L::O_COL0 + t * D, tmem + L::S_COL0 + t * 128 + k * 8, bdesc,
                                kIdescPV, accf);
                    } else {
                        const uint32_t a = sbase + L::P_OFF + (k >> 2) * L::BOX_BYTES + (k & 3) * 32;
                        umma_ss(tmem + L::O_COL0 + t * D, sdesc_sw128(a, 16, 1024), bdesc, kIdescPV,
                                accf);
                    }
                }
            };
            if (ok) {
                for (int t = 0; t < n_active; ++t) {
                    issue_s(t, 0);
                    umma_commit(s_full(t));
                }
                umma_commit(k_empty(0));
            }
            for (int j = 0; ok && j < nkv_max; ++j) {
                const int st = j % L::STAGES;
                const uint32_t ph = (j / L::STAGES) & 1;
                const int jn = j + 1;
                bool v_ready = false, k_next_ready = false;
                for (int t = 0; t < n_active && ok; ++t) {
                    if (j >= nkv[t]) continue;
                    if (!mbar_wait(p_full(t), j & 1, tmo)) { ok = false; break; }
                    if (!v_ready) {
                        if (!mbar_wait(v_full(st), ph, tmo)) { ok = false; break; }
                        v_ready = true;
                    }
                    tc_fence_after();
                    issue_pv(t, st, j > 0);
                    if (jn == nkv[t]) {
                        umma_commit(o_final(t));
                    } else {
                        if (!k_next_ready) {
                            if (!mbar_wait(k_full(jn % L::STAGES), (jn / L::STAGES) & 1, tmo)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                            k_next_ready = true;
                        }
                        issue_s(t, jn % L::STAGES);
                        umma_commit(s_full(t));
                    }
                }
                if (v_ready) umma_commit(v_empty(st));
                if (k_next_ready) umma_commit(k_empty(jn % L::STAGES));
            }
            if (!ok) record_status(ATTN_ERR_TIMEOUT);
            // every MMA this thread issued has finished before TMEM is released
            umma_commit(drain_bar);
            mbar_wait(drain_bar, 0, tmo);
        }
    } else if (warp >= 4) {
        // ========================= softmax / epilogue ========================
        const int t = (warp - 4) >> 2;
        const int wq = warp & 3;                 // TMEM lane quarter of this warp
        const int r = wq * 32 + lane;            // row within the tile
        if (t < n_active) {
            const int row = q0 + 128 * t + r;    // query index
            const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
            const uint32_t s_addr = tmem + lane_off + L::S_COL0 + t * 128;
            const uint32_t o_addr = tmem + lane_off + L::O_COL0 + t * D;
            const float sl2 = p.scale_log2;
            float m = -INFINITY;  // running max of scale*log2(e)*s
            float l = 0.f;        // running sum of 2^(scale*log2(e)*s - m)
            bool ok = true;
            for (int j = 0; j < nkv[t]; ++j) {
                if (!mbar_wait(s_full(t), j & 1, tmo)) { ok = false; break; }
                tc_fence_after();
                float s[128];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t raw[32];
                    tmem_ld32(s_addr + c * 32, raw);
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(raw[i]);
                }
                // keys [kv0, kv0 + limit) are visible to this row
                const int kv0 = j * 128;
                const int limit = (CAUSAL ? min(p.N, row + 1) : p.N) - kv0;
                if (limit < 128) {
#pragma unroll
                    for (int c = 0; c < 128; ++c) s[c] = (c < limit) ? s[c] : -INFINITY;
                }
                float mx = s[0];
#pragma unroll
                for (int c = 1; c < 128; ++c) mx = fmaxf(mx, s[c]);
                const float m_new = fmaxf(m, mx * sl2);
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
                const float alpha = ex2_approx(m - m_use);
                float sum = 0.f;
#pragma unroll
                for (int c = 0; c < 128; ++c) {
                    s[c] = ex2_approx(fmaf(s[c], sl2, -m_use));
                    sum += s[c];
                }
                l = l * alpha + sum;
                m = m_new;
                // rescale the running O row (its last PV has completed: S_t(j)
                // was issued after it and s_full(t) covers it)
                if (j > 0 && __any_sync(0xffffffffu, alpha < 1.f)) {
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t raw[32];
                        tmem_ld32(o_addr + c * 32, raw);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            raw[i] = __float_as_uint(__uint_as_float(raw[i]) * alpha);
                        tmem_st32(o_addr + c * 32, raw);
                    }
                }
                // P (bf16) for the PV product
                if constexpr (P_TMEM) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t pk[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            pk[i] = pack_bf16x2(s[c * 32 + 2 * i], s[c * 32 + 2 * i + 1]);
                        tmem_st16(s_addr + c * 16, pk);
                    }
                    tmem_st_wait();
                } else {
                    if (D / 32 > 0) tmem_st_wait();
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
                tc_fence_before();
                mbar_arrive(p_full(t));
            }
            // epilogue: O / l -> bf16, LSE
            if (ok && mbar_wait(o_final(t), 0, tmo)) {
                tc_fence_after();
                const float inv_l = 1.f / l;
                const bool store = row < p.N;
                __nv_bfloat16* orow = p.o + (((size_t)b * p.N + (store ? row : 0)) * p.H + h) * D;
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
                if (store && p.lse != nullptr)
                    p.lse[((size_t)b * p.H + h) * p.N + row] = (m + __log2f(l)) * kLn2;
            } else {
                record_status(ATTN_ERR_TIMEOUT);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, L::TMEM_COLS);
    }
}

}  // namespace attn
