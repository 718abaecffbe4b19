// C ABI of the B300 attention library: argument validation, kernel selection
// over head_dim {64, 128} x causal (prefill) or contiguous / paged (decode),
// TMA tensor-map encoding, and launches.  The kernels live in prefill.cuh and
// decode.cuh; this file is the only translation unit.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>

#include "../../include/attn_b300.h"
#include "backward.cuh"
#include "common.cuh"
#include "decode.cuh"
#include "prefill.cuh"

namespace attn {
namespace {

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s per pipeline wait

// Per-wait limit of the pipelined kernels, read at every call: ATTN_WAIT_TIMEOUT_MS
// (milliseconds) overrides the default.
unsigned long long wait_timeout_ns() {
    const char* env = std::getenv("ATTN_WAIT_TIMEOUT_MS");
    if (env != nullptr) {
        const long long ms = std::atoll(env);
        if (ms > 0) return (unsigned long long)ms * 1000000ull;
    }
    return kDefaultTimeoutNs;
}

// Test hook, read at every call: ATTN_TEST_DROP_LOAD=1 makes the next prefill or
// backward launch leave one load unissued, so that a wait for it runs out (see
// PrefillParams::test_drop_load).  Unset in normal use.
int test_drop_load() {
    const char* env = std::getenv("ATTN_TEST_DROP_LOAD");
    return (env != nullptr && std::atoi(env) != 0) ? 1 : 0;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }
bool aligned4(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 3u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// ---- cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda)
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// [B, N, H, d] bf16 viewed as a 4-D tensor (d, H, N, B); box = 64 x 1 x 128 x 1
// (one 128-row x 128-byte tile of one head), 128-byte swizzle, zero fill past N.
bool encode_bnhd(CUtensorMap* map, const void* base, int B, int N, int H, int d) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2,
                                   (cuuint64_t)N * H * d * 2};
    const cuuint32_t box[4] = {64, 1, 128, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A 16-token paged pool [num_pages, 16, H, d] bf16 viewed as a 3-D tensor
// (d, H, num_pages * 16); box = 64 x 1 x 16 (one page of one head, 128-byte
// rows), 128-byte swizzle.
bool encode_pool(CUtensorMap* map, const void* base, int num_pages, int H, int d) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)num_pages * 16};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    const cuuint32_t box[3] = {64, 1, 16};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// FP8 (E4M3) [B, N, H, d] bytes viewed as (d, H, N, B); box = d x 1 x 128 x 1
// (128 rows of one head), 128-byte swizzle for d = 128, 64-byte for d = 64,
// zero fill past N.
bool encode_bnhd_e4m3(CUtensorMap* map, const void* base, int B, int N, int H, int d) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)N, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)d, (cuuint64_t)H * d, (cuuint64_t)N * H * d};
    const cuuint32_t box[4] = {(cuuint32_t)d, 1, 128, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              d == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// FP8 V^T [B, H, d, Np] bytes (keys contiguous, rows Np = N rounded up to 16
// bytes apart) viewed as (N, d, H, B); box = 128 x d x 1 x 1 (d rows x 128
// keys), 128-byte swizzle, zero fill for keys >= N (the padding is never read).
bool encode_vt_e4m3(CUtensorMap* map, const void* base, int B, int H, int d, int N, int Np) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)N, (cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)Np, (cuuint64_t)d * Np, (cuuint64_t)H * d * Np};
    const cuuint32_t box[4] = {128, (cuuint32_t)d, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Streaming multiprocessors of the current device (cached per device).
int sm_count(int* out) {
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && cache[dev] > 0) {
        *out = cache[dev];
        return ATTN_OK;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return ATTN_ERR_CUDA;
    if (dev >= 0 && dev < 64) cache[dev] = n;
    *out = n;
    return ATTN_OK;
}

// Contiguous prefill with long sequences (K and V of one (batch, head) at least
// kPrefillBandMinHead bytes) whose static deal would keep more K/V live than
// kPrefillBandAbove -- the CTAs at work at once span min(B*H, CTAs) heads -- is
// worked through in bands of heads whose K/V fits in kPrefillBandBytes, with a
// dynamic deal (see PrefillParams::band_heads).  L2 holds 126 MB; a band uses a
// quarter of it, so that the band being finished and the next one fit together
// with room to spare (32, 48 and 64 MB bands measured the same speed; 32 MB
// re-reads the least).  Shorter sequences, where a unit takes a few
// microseconds, keep the static deal at d=128 (the dynamic one measured 2-9 %
// slower at N=512-4096); bf16 d=64 takes the dynamic deal in bands of 32 heads
// there too, measured 4-8 % faster than the static deal at N=512-4096, causal
// and not (the cause of the difference between the head dims was not isolated).
constexpr size_t kPrefillBandMinHead = 4ull << 20;
constexpr size_t kPrefillShortBandHeads64 = 32;
constexpr size_t kPrefillBandAbove = 64ull << 20;
constexpr size_t kPrefillBandBytes = 32ull << 20;

int prefill_band_heads(int B, int H, int N, int d, int elem_bytes) {
    const size_t per_head = (size_t)N * d * elem_bytes * 2;  // K and V of one (batch, head)
    const size_t bh = (size_t)B * H;
    int sms = 0;
    if (sm_count(&sms) != ATTN_OK || sms <= 0) return 0;
    const size_t live = bh < (size_t)sms ? bh : (size_t)sms;
    if (per_head < kPrefillBandMinHead || live * per_head <= kPrefillBandAbove)
        return (d == 64 && elem_bytes == 2) ? (int)(bh < kPrefillShortBandHeads64 ? bh : kPrefillShortBandHeads64) : 0;
    const size_t band = kPrefillBandBytes / per_head;
    return (int)(band < 1 ? 1 : (band > bh ? bh : band));
}

// Backward: each gradient kernel streams one pair of [B, N, H, d] tensors (Q and
// dO, or K and V) per unit, all of its (batch, head)'s rows; a unit takes a few
// to a few hundred microseconds.  d=128 works band by band (16 MB of streamed
// pairs per band, dynamic deal) once the static deal would keep more than 32 MB
// of them live and a (batch, head)'s pair is at least 1 MB: measured +3 % on
// B=4 H=16 N=2048 causal, +10 % at N=16384 non-causal, level at N=16384 causal.
// d=64 keeps the static deal (its kernels are bound by the compute warps'
// elementwise work; the banded deal measured 2-3 % slower at N=16384).
constexpr size_t kBwdBandMinHead = 1ull << 20;
constexpr size_t kBwdBandAbove = 32ull << 20;
constexpr size_t kBwdBandBytes = 16ull << 20;

int bwd_band_heads(int B, int H, int N, int d) {
    if (d != 128) return 0;
    const size_t per_head = (size_t)N * d * 2 * 2;
    const size_t bh = (size_t)B * H;
    int sms = 0;
    if (sm_count(&sms) != ATTN_OK || sms <= 0) return 0;
    const size_t live = bh < (size_t)sms ? bh : (size_t)sms;
    if (per_head < kBwdBandMinHead || live * per_head <= kBwdBandAbove) return 0;
    const size_t band = kBwdBandBytes / per_head;
    return (int)(band < 1 ? 1 : (band > bh ? bh : band));
}

// Unit counters of the dynamic deal: each launch that uses one takes the next
// slot in turn and zeroes it on its stream first, so launches in flight at the
// same time use different counters unless kUnitCounters of them overlap.
constexpr int kUnitCounters = 4096;
static __device__ unsigned int g_unit_counters[kUnitCounters];
std::atomic<unsigned int> g_unit_counter_next{0};

int unit_counter_for_launch(cudaStream_t stream, unsigned int** out) {
    static std::mutex mu;
    static void* base[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    void* b = nullptr;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev >= 0 && dev < 64) b = base[dev];
        if (b == nullptr) {
            if (cudaGetSymbolAddress(&b, g_unit_counters) != cudaSuccess) return ATTN_ERR_CUDA;
            if (dev >= 0 && dev < 64) base[dev] = b;
        }
    }
    unsigned int* c = static_cast<unsigned int*>(b) + (g_unit_counter_next.fetch_add(1) % kUnitCounters);
    if (cudaMemsetAsync(c, 0, sizeof(unsigned int), stream) != cudaSuccess) return ATTN_ERR_CUDA;
    *out = c;
    return ATTN_OK;
}

// Prefill variants: "tmem2" (default: two query tiles per CTA, P in tensor
// memory), "tmem1" (one tile, P in tensor memory), "smem1" (one tile, P in
// shared memory).  ATTN_PREFILL_IMPL selects one; used by the tests.
enum class PrefillImpl { kTmem2, kTmem1, kSmem1 };

PrefillImpl prefill_impl() {
    const char* env = std::getenv("ATTN_PREFILL_IMPL");
    if (env != nullptr) {
        if (std::strcmp(env, "tmem1") == 0) return PrefillImpl::kTmem1;
        if (std::strcmp(env, "smem1") == 0) return PrefillImpl::kSmem1;
    }
    return PrefillImpl::kTmem2;
}

template <int D, bool CAUSAL, int QT, bool P_TMEM, bool KV_PAGED = false, bool FP8 = false,
          bool DYN = false>
int launch_prefill_instance(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const PrefillParams& prm, cudaStream_t stream) {
    using L = PrefillLayout<D, QT, P_TMEM, FP8, KV_PAGED>;
    auto kern = prefill_kernel<D, CAUSAL, QT, P_TMEM, KV_PAGED, FP8, DYN>;
    // Once per device and kernel instance: the shared-memory opt-in, and (two
    // query tiles) a check that the kernel is launched with the per-thread
    // register count its setmaxnreg split between warpgroups assumes.
    static std::mutex mu;
    static uint64_t configured = 0;  // bit per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (bit == 0 || (configured & bit) == 0) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     L::SMEM_BYTES) != cudaSuccess)
                return ATTN_ERR_CUDA;
            if constexpr (QT == 2) {
                cudaFuncAttributes fa;
                if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return ATTN_ERR_CUDA;
                if (fa.numRegs < L::LAUNCH_REGS) return ATTN_ERR_UNSUPPORTED;
            }
            configured |= bit;
        }
    }
    const long long groups = (prm.N + 128 * QT - 1) / (128 * QT);
    const long long units = groups * prm.B * prm.H;
    if (units > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    int sms = 0;
    if (sm_count(&sms) != ATTN_OK) return ATTN_ERR_CUDA;
    // persistent: one CTA per SM (shared memory and TMEM admit one), each
    // working through its share of the units
    PrefillParams run = prm;
    run.num_units = (int)units;
    if constexpr (DYN) {
        const int rc = unit_counter_for_launch(stream, &run.unit_counter);
        if (rc != ATTN_OK) return rc;
    } else {
        run.band_heads = 0;
        run.unit_counter = nullptr;
    }
    const unsigned grid = (unsigned)(units < sms ? units : sms);
    kern<<<grid, L::THREADS, L::SMEM_BYTES, stream>>>(tq, tk, tv, run);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int D>
int launch_prefill_fp8_d(bool causal, const CUtensorMap& tq, const CUtensorMap& tk,
                         const CUtensorMap& tv, const PrefillParams& prm, cudaStream_t stream) {
    if (prm.band_heads > 0)
        return causal ? launch_prefill_instance<D, true, 2, true, false, true, true>(tq, tk, tv, prm, stream)
                      : launch_prefill_instance<D, false, 2, true, false, true, true>(tq, tk, tv, prm, stream);
    return causal ? launch_prefill_instance<D, true, 2, true, false, true>(tq, tk, tv, prm, stream)
                  : launch_prefill_instance<D, false, 2, true, false, true>(tq, tk, tv, prm, stream);
}

template <int D, bool CAUSAL>
int launch_prefill_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                     const PrefillParams& prm, cudaStream_t stream) {
    switch (prefill_impl()) {
        case PrefillImpl::kTmem1:
            return launch_prefill_instance<D, CAUSAL, 1, true>(tq, tk, tv, prm, stream);
        case PrefillImpl::kSmem1:
            return launch_prefill_instance<D, CAUSAL, 1, false>(tq, tk, tv, prm, stream);
        default:
            return prm.band_heads > 0
                       ? launch_prefill_instance<D, CAUSAL, 2, true, false, false, true>(tq, tk, tv, prm, stream)
                       : launch_prefill_instance<D, CAUSAL, 2, true>(tq, tk, tv, prm, stream);
    }
}

template <int D, bool PAGED, bool FP8>
int launch_decode_instance(const DecodeParams& prm, cudaStream_t stream) {
    const dim3 grid_split((unsigned)prm.max_splits, (unsigned)prm.S,
                          (unsigned)((prm.H + kDecodeHeadsPerCta - 1) / kDecodeHeadsPerCta));
    decode_split_kernel<D, PAGED, FP8><<<grid_split, 32 * kDecodeHeadsPerCta, 0, stream>>>(prm);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    const long long rows = (long long)prm.S * prm.H;
    decode_merge_kernel<D><<<(unsigned)((rows + 3) / 4), 128, 0, stream>>>(prm);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Backward: the prep kernel, then the dK/dV and dQ kernels (persistent grids).
template <int D, bool CAUSAL, bool KEY_TILES, bool DYN>
int launch_bwd_instance(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& tdo, const BwdParams& prm, cudaStream_t stream) {
    using L = BwdLayout<D>;
    auto kern = bwd_kernel<D, CAUSAL, KEY_TILES, DYN>;
    static std::mutex mu;
    static uint64_t configured = 0;  // bit per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (bit == 0 || (configured & bit) == 0) {
            if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     L::SMEM_BYTES) != cudaSuccess)
                return ATTN_ERR_CUDA;
            configured |= bit;
        }
    }
    int sms = 0;
    if (sm_count(&sms) != ATTN_OK) return ATTN_ERR_CUDA;
    BwdParams run = prm;
    if constexpr (DYN) {
        const int rc = unit_counter_for_launch(stream, &run.unit_counter);
        if (rc != ATTN_OK) return rc;
    } else {
        run.band_heads = 0;
        run.unit_counter = nullptr;
    }
    const unsigned grid = (unsigned)(prm.num_units < sms ? prm.num_units : sms);
    kern<<<grid, L::THREADS, L::SMEM_BYTES, stream>>>(tq, tk, tv, tdo, run);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

template <int D, bool CAUSAL>
int launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const CUtensorMap& tdo, const BwdParams& prm, cudaStream_t stream) {
    const long long rows = (long long)prm.B * prm.H * prm.Npad;
    constexpr int rows_per_block = 8 * (32 / (D / 8));  // 8 warps of 256 threads
    bwd_prep_kernel<D><<<(unsigned)((rows + rows_per_block - 1) / rows_per_block), 256, 0, stream>>>(prm);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
    if (prm.band_heads > 0) {
        const int rc = launch_bwd_instance<D, CAUSAL, true, true>(tq, tk, tv, tdo, prm, stream);
        if (rc != ATTN_OK) return rc;
        return launch_bwd_instance<D, CAUSAL, false, true>(tq, tk, tv, tdo, prm, stream);
    }
    const int rc = launch_bwd_instance<D, CAUSAL, true, false>(tq, tk, tv, tdo, prm, stream);
    if (rc != ATTN_OK) return rc;
    return launch_bwd_instance<D, CAUSAL, false, false>(tq, tk, tv, tdo, prm, stream);
}

// Backward workspace: LSE * log2(e) and D, each fp32 [B*H, Npad], 256-byte aligned.
size_t bwd_vec_bytes(int B, int H, int N) {
    const size_t npad = ((size_t)N + 127) / 128 * 128;
    return ((size_t)B * H * npad * sizeof(float) + 255) & ~size_t(255);
}

struct DecodeWorkspace {
    size_t o_bytes, lse_bytes, total;
    int max_splits;
};

bool decode_workspace_layout(int num_seqs, int H, int d, int max_seqlen, DecodeWorkspace* w) {
    if (num_seqs < 0 || H < 0 || (d != 64 && d != 128) || max_seqlen < 0) return false;
    w->max_splits = (max_seqlen + kSplitTokens - 1) / kSplitTokens;
    const size_t slots = (size_t)num_seqs * (size_t)w->max_splits * (size_t)H;
    w->o_bytes = (slots * (size_t)d * sizeof(float) + 255) & ~size_t(255);
    w->lse_bytes = (slots * sizeof(float) + 255) & ~size_t(255);
    w->total = w->o_bytes + w->lse_bytes;
    return true;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                        int H, int N, int d, int causal, float scale, void* stream) {
    if (B < 0 || H < 0 || N < 0) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || N == 0) return ATTN_OK;  // empty tensors may carry NULL pointers
    if (q == nullptr || k == nullptr || v == nullptr || o == nullptr) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
        (lse != nullptr && !aligned4(lse)))
        return ATTN_ERR_MISALIGNED;
    const size_t elems = (size_t)B * N * H * d;
    if ((size_t)B * H * N > (size_t)0x7fffffff) return ATTN_ERR_UNSUPPORTED;
    const size_t bytes = elems * 2;
    if (overlaps(o, bytes, q, bytes) || overlaps(o, bytes, k, bytes) || overlaps(o, bytes, v, bytes))
        return ATTN_ERR_INVALID_ARG;
    if (lse != nullptr && overlaps(lse, (size_t)B * H * N * 4, o, bytes)) return ATTN_ERR_INVALID_ARG;

    CUtensorMap tq, tk, tv;
    if (!encode_bnhd(&tq, q, B, N, H, d) || !encode_bnhd(&tk, k, B, N, H, d) ||
        !encode_bnhd(&tv, v, B, N, H, d))
        return ATTN_ERR_CUDA;
    PrefillParams prm;
    prm.o = static_cast<__nv_bfloat16*>(o);
    prm.lse = lse;
    prm.B = B;
    prm.H = H;
    prm.N = N;
    prm.scale_log2 = scale * kLog2e;
    prm.timeout_ns = wait_timeout_ns();
    prm.test_drop_load = test_drop_load();
    prm.seqlens = nullptr;
    prm.page_table = nullptr;
    prm.max_pages = 0;
    prm.num_pages = 0;
    prm.q_scale = prm.k_scale = prm.v_scale = nullptr;
    prm.band_heads = prefill_band_heads(B, H, N, d, 2);
    prm.unit_counter = nullptr;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (d == 64)
        return causal ? launch_prefill_d<64, true>(tq, tk, tv, prm, st)
                      : launch_prefill_d<64, false>(tq, tk, tv, prm, st);
    return causal ? launch_prefill_d<128, true>(tq, tk, tv, prm, st)
                  : launch_prefill_d<128, false>(tq, tk, tv, prm, st);
}

extern "C" int attn_fwd_fp8(const void* q, const void* k, const void* vt, const float* q_scale,
                            const float* k_scale, const float* v_scale, void* o, float* lse, int B,
                            int H, int N, int d, int causal, float scale, void* stream) {
    if (B < 0 || H < 0 || N < 0) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || N == 0) return ATTN_OK;  // empty tensors may carry NULL pointers
    if (q == nullptr || k == nullptr || vt == nullptr || o == nullptr || q_scale == nullptr ||
        k_scale == nullptr || v_scale == nullptr)
        return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(vt) || !aligned16(o) || !aligned4(q_scale) ||
        !aligned4(k_scale) || !aligned4(v_scale) || (lse != nullptr && !aligned4(lse)))
        return ATTN_ERR_MISALIGNED;
    if ((size_t)B * H * N > (size_t)0x7fffffff || N > 0x7fffffff - 15) return ATTN_ERR_UNSUPPORTED;
    const int Np = (N + 15) & ~15;
    const size_t elems = (size_t)B * N * H * d;
    const size_t obytes = elems * 2, vtbytes = (size_t)B * H * d * Np;
    if (overlaps(o, obytes, q, elems) || overlaps(o, obytes, k, elems) || overlaps(o, obytes, vt, vtbytes))
        return ATTN_ERR_INVALID_ARG;
    if (lse != nullptr && overlaps(lse, (size_t)B * H * N * 4, o, obytes)) return ATTN_ERR_INVALID_ARG;

    CUtensorMap tq, tk, tv;
    if (!encode_bnhd_e4m3(&tq, q, B, N, H, d) || !encode_bnhd_e4m3(&tk, k, B, N, H, d) ||
        !encode_vt_e4m3(&tv, vt, B, H, d, N, Np))
        return ATTN_ERR_CUDA;
    PrefillParams prm;
    prm.o = static_cast<__nv_bfloat16*>(o);
    prm.lse = lse;
    prm.B = B;
    prm.H = H;
    prm.N = N;
    prm.scale_log2 = scale * kLog2e;
    prm.timeout_ns = wait_timeout_ns();
    prm.test_drop_load = test_drop_load();
    prm.seqlens = nullptr;
    prm.page_table = nullptr;
    prm.max_pages = 0;
    prm.num_pages = 0;
    prm.q_scale = q_scale;
    prm.k_scale = k_scale;
    prm.v_scale = v_scale;
    prm.band_heads = prefill_band_heads(B, H, N, d, 1);
    prm.unit_counter = nullptr;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (d == 64)
        return launch_prefill_fp8_d<64>(causal != 0, tq, tk, tv, prm, st);
    return launch_prefill_fp8_d<128>(causal != 0, tq, tk, tv, prm, st);
}

extern "C" int attn_prefill_paged(const void* q, const void* kcache, const void* vcache,
                                  const int* seqlens, const int* page_table, void* o, float* lse,
                                  int B, int H, int Nq, int d, int page_size, int max_pages_per_seq,
                                  int num_pages, int causal, float scale, void* stream) {
    if (B < 0 || H < 0 || Nq < 0) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (page_size != kPageSize) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || Nq == 0) return ATTN_OK;  // empty tensors may carry NULL pointers
    if (q == nullptr || kcache == nullptr || vcache == nullptr || seqlens == nullptr ||
        page_table == nullptr || o == nullptr)
        return ATTN_ERR_INVALID_ARG;
    if (max_pages_per_seq <= 0 || num_pages <= 0) return ATTN_ERR_INVALID_ARG;
    if ((long long)Nq > (long long)max_pages_per_seq * kPageSize) return ATTN_ERR_INVALID_ARG;
    if (num_pages > (1 << 26)) return ATTN_ERR_UNSUPPORTED;  // page row coordinates stay int32
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) ||
        !aligned4(seqlens) || !aligned4(page_table) || (lse != nullptr && !aligned4(lse)))
        return ATTN_ERR_MISALIGNED;
    if ((size_t)B * H * Nq > (size_t)0x7fffffff) return ATTN_ERR_UNSUPPORTED;
    const size_t qbytes = (size_t)B * Nq * H * d * 2;
    const size_t pool_bytes = (size_t)num_pages * kPageSize * H * d * 2;
    if (overlaps(o, qbytes, q, qbytes) || overlaps(o, qbytes, kcache, pool_bytes) ||
        overlaps(o, qbytes, vcache, pool_bytes))
        return ATTN_ERR_INVALID_ARG;
    if (lse != nullptr && overlaps(lse, (size_t)B * H * Nq * 4, o, qbytes)) return ATTN_ERR_INVALID_ARG;

    CUtensorMap tq, tk, tv;
    if (!encode_bnhd(&tq, q, B, Nq, H, d) || !encode_pool(&tk, kcache, num_pages, H, d) ||
        !encode_pool(&tv, vcache, num_pages, H, d))
        return ATTN_ERR_CUDA;
    PrefillParams prm;
    prm.o = static_cast<__nv_bfloat16*>(o);
    prm.lse = lse;
    prm.B = B;
    prm.H = H;
    prm.N = Nq;
    prm.scale_log2 = scale * kLog2e;
    prm.timeout_ns = wait_timeout_ns();
    prm.test_drop_load = test_drop_load();
    prm.seqlens = seqlens;
    prm.page_table = page_table;
    prm.max_pages = max_pages_per_seq;
    prm.num_pages = num_pages;
    prm.q_scale = prm.k_scale = prm.v_scale = nullptr;
    // paged: the longest-cache-first order, dealt dynamically (unit costs differ
    // with the cache lengths)
    prm.band_heads = 0;
    prm.unit_counter = nullptr;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (d == 64)
        return causal ? launch_prefill_instance<64, true, 2, true, true, false, true>(tq, tk, tv, prm, st)
                      : launch_prefill_instance<64, false, 2, true, true, false, true>(tq, tk, tv, prm, st);
    return causal ? launch_prefill_instance<128, true, 2, true, true, false, true>(tq, tk, tv, prm, st)
                  : launch_prefill_instance<128, false, 2, true, true, false, true>(tq, tk, tv, prm, st);
}

extern "C" size_t attn_bwd_workspace_size(int B, int H, int N, int d) {
    if (B <= 0 || H <= 0 || N <= 0 || (d != 64 && d != 128)) return 0;
    return 2 * bwd_vec_bytes(B, H, N);
}

extern "C" int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                        int causal, float scale, void* workspace, size_t workspace_bytes,
                        void* stream) {
    if (B < 0 || H < 0 || N < 0) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (B == 0 || H == 0 || N == 0) return ATTN_OK;  // empty tensors may carry NULL pointers
    const void* ins[6] = {q, k, v, o, lse, dout};
    void* outs[3] = {dq, dk, dv};
    for (const void* x : ins)
        if (x == nullptr) return ATTN_ERR_INVALID_ARG;
    for (void* x : outs)
        if (x == nullptr) return ATTN_ERR_INVALID_ARG;
    for (const void* x : {q, k, v, o, dout, (const void*)dq, (const void*)dk, (const void*)dv})
        if (!aligned16(x)) return ATTN_ERR_MISALIGNED;
    if (!aligned4(lse)) return ATTN_ERR_MISALIGNED;
    if ((size_t)B * H * N > (size_t)0x7fffffff || N > 0x7fffffff - 127) return ATTN_ERR_UNSUPPORTED;
    const size_t vec = bwd_vec_bytes(B, H, N);
    if (workspace == nullptr || workspace_bytes < 2 * vec) return ATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return ATTN_ERR_MISALIGNED;
    const size_t bytes = (size_t)B * N * H * d * 2, lse_bytes = (size_t)B * H * N * 4;
    // outputs alias neither an input, the workspace nor each other
    for (int i = 0; i < 3; ++i) {
        for (int j = 0; j < 6; ++j)
            if (overlaps(outs[i], bytes, ins[j], j == 4 ? lse_bytes : bytes)) return ATTN_ERR_INVALID_ARG;
        for (int j = i + 1; j < 3; ++j)
            if (overlaps(outs[i], bytes, outs[j], bytes)) return ATTN_ERR_INVALID_ARG;
        if (overlaps(outs[i], bytes, workspace, 2 * vec)) return ATTN_ERR_INVALID_ARG;
    }
    for (int j = 0; j < 6; ++j)
        if (overlaps(workspace, 2 * vec, ins[j], j == 4 ? lse_bytes : bytes)) return ATTN_ERR_INVALID_ARG;

    CUtensorMap tq, tk, tv, tdo;
    if (!encode_bnhd(&tq, q, B, N, H, d) || !encode_bnhd(&tk, k, B, N, H, d) ||
        !encode_bnhd(&tv, v, B, N, H, d) || !encode_bnhd(&tdo, dout, B, N, H, d))
        return ATTN_ERR_CUDA;
    BwdParams prm;
    prm.o = static_cast<const __nv_bfloat16*>(o);
    prm.dout = static_cast<const __nv_bfloat16*>(dout);
    prm.lse = lse;
    prm.dq = static_cast<__nv_bfloat16*>(dq);
    prm.dk = static_cast<__nv_bfloat16*>(dk);
    prm.dv = static_cast<__nv_bfloat16*>(dv);
    prm.ws_lse2 = static_cast<float*>(workspace);
    prm.ws_d = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + vec);
    prm.B = B;
    prm.H = H;
    prm.N = N;
    prm.Npad = (N + 127) / 128 * 128;
    prm.scale = scale;
    prm.scale_log2 = scale * kLog2e;
    prm.timeout_ns = wait_timeout_ns();
    prm.test_drop_load = test_drop_load();
    const long long units = (long long)(prm.Npad / 128) * B * H;
    if (units > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
    prm.num_units = (int)units;
    prm.band_heads = bwd_band_heads(B, H, N, d);
    prm.unit_counter = nullptr;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (d == 64)
        return causal ? launch_bwd<64, true>(tq, tk, tv, tdo, prm, st)
                      : launch_bwd<64, false>(tq, tk, tv, tdo, prm, st);
    return causal ? launch_bwd<128, true>(tq, tk, tv, tdo, prm, st)
                  : launch_bwd<128, false>(tq, tk, tv, tdo, prm, st);
}

extern "C" size_t attn_decode_workspace_size(int num_seqs, int H, int d, int max_seqlen) {
    DecodeWorkspace w;
    if (!decode_workspace_layout(num_seqs, H, d, max_seqlen, &w)) return 0;
    if (num_seqs == 0 || H == 0 || max_seqlen == 0) return 0;
    return w.total;
}

namespace attn {
namespace {

// Host-side checks shared by attn_decode, attn_decode_fp8 and
// attn_decode_noalloc.  Makes no CUDA call.  Returns the status to report, or
// ATTN_OK with the workspace layout in *w; *empty is set when the call has
// nothing to do (an empty dimension).
int decode_validate(const void* q, const void* kcache, const void* vcache, const float* k_scale,
                    const float* v_scale, bool fp8, const int* seqlens, const int* page_table,
                    const void* o, const float* lse, int num_seqs, int H, int d, int max_seqlen,
                    int page_size, int max_pages_per_seq, int num_pages, float scale,
                    DecodeWorkspace* w, bool* empty) {
    *empty = false;
    if (num_seqs < 0 || H < 0 || max_seqlen < 0) return ATTN_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
    if (num_seqs == 0 || H == 0) {  // empty tensors may carry NULL pointers
        *empty = true;
        return ATTN_OK;
    }
    if (q == nullptr || kcache == nullptr || vcache == nullptr || seqlens == nullptr || o == nullptr)
        return ATTN_ERR_INVALID_ARG;
    if (fp8 && (k_scale == nullptr || v_scale == nullptr)) return ATTN_ERR_INVALID_ARG;
    const bool paged = page_table != nullptr;
    if (paged) {
        if (page_size != kPageSize) return ATTN_ERR_UNSUPPORTED;
        if (max_pages_per_seq <= 0 || num_pages <= 0) return ATTN_ERR_INVALID_ARG;
        if ((long long)max_seqlen > (long long)max_pages_per_seq * kPageSize)
            return ATTN_ERR_INVALID_ARG;
    }
    if (!aligned16(q) || !aligned16(kcache) || !aligned16(vcache) || !aligned16(o) ||
        !aligned4(seqlens) || (paged && !aligned4(page_table)) || (lse != nullptr && !aligned4(lse)) ||
        (fp8 && (!aligned4(k_scale) || !aligned4(v_scale))))
        return ATTN_ERR_MISALIGNED;
    if (!decode_workspace_layout(num_seqs, H, d, max_seqlen, w)) return ATTN_ERR_INVALID_ARG;
    if (num_seqs > 65535 || (H + kDecodeHeadsPerCta - 1) / kDecodeHeadsPerCta > 65535)
        return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

// Launch of a validated decode call; `workspace` holds at least w.total bytes
// (unused when max_seqlen == 0).
int decode_launch(const void* q, const void* kcache, const void* vcache, const float* k_scale,
                  const float* v_scale, bool fp8, const int* seqlens, const int* page_table, void* o,
                  float* lse, int num_seqs, int H, int d, int max_seqlen, int max_pages_per_seq,
                  int num_pages, float scale, const DecodeWorkspace& w, void* workspace,
                  void* stream) {
    const bool paged = page_table != nullptr;
    DecodeParams prm;
    prm.q = static_cast<const __nv_bfloat16*>(q);
    prm.kc = kcache;
    prm.vc = vcache;
    prm.k_scale = fp8 ? k_scale : nullptr;
    prm.v_scale = fp8 ? v_scale : nullptr;
    prm.seqlens = seqlens;
    prm.page_table = page_table;
    prm.o = static_cast<__nv_bfloat16*>(o);
    prm.lse = lse;
    prm.ws_o = static_cast<float*>(workspace);
    prm.ws_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + w.o_bytes);
    prm.S = num_seqs;
    prm.H = H;
    prm.max_seqlen = max_seqlen;
    prm.max_pages = paged ? max_pages_per_seq : 0;
    prm.num_pages = paged ? num_pages : 0;
    prm.max_splits = w.max_splits > 0 ? w.max_splits : 1;
    prm.scale_log2 = scale * kLog2e;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (max_seqlen == 0) {
        // no cache at all: only the merge runs (every sequence has length 0)
        prm.max_splits = 1;
        const long long rows = (long long)num_seqs * H;
        if (d == 64)
            decode_merge_kernel<64><<<(unsigned)((rows + 3) / 4), 128, 0, st>>>(prm);
        else
            decode_merge_kernel<128><<<(unsigned)((rows + 3) / 4), 128, 0, st>>>(prm);
        return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
    }
    if (fp8) {
        if (d == 64)
            return paged ? launch_decode_instance<64, true, true>(prm, st)
                         : launch_decode_instance<64, false, true>(prm, st);
        return paged ? launch_decode_instance<128, true, true>(prm, st)
                     : launch_decode_instance<128, false, true>(prm, st);
    }
    if (d == 64)
        return paged ? launch_decode_instance<64, true, false>(prm, st)
                     : launch_decode_instance<64, false, false>(prm, st);
    return paged ? launch_decode_instance<128, true, false>(prm, st)
                 : launch_decode_instance<128, false, false>(prm, st);
}

// attn_decode and attn_decode_fp8: validation, the caller's workspace, launch.
// fp8: e4m3 caches (one byte per element) with fp32 per-head scales.
int decode_impl(const void* q, const void* kcache, const void* vcache, const float* k_scale,
                const float* v_scale, bool fp8, const int* seqlens, const int* page_table, void* o,
                float* lse, int num_seqs, int H, int d, int max_seqlen, int page_size,
                int max_pages_per_seq, int num_pages, float scale, void* workspace,
                size_t workspace_bytes, void* stream) {
    DecodeWorkspace w;
    bool empty = false;
    const int rc = decode_validate(q, kcache, vcache, k_scale, v_scale, fp8, seqlens, page_table, o,
                                   lse, num_seqs, H, d, max_seqlen, page_size, max_pages_per_seq,
                                   num_pages, scale, &w, &empty);
    if (rc != ATTN_OK || empty) return rc;
    if (max_seqlen > 0) {
        if (workspace == nullptr || workspace_bytes < w.total) return ATTN_ERR_WORKSPACE;
        if (!aligned16(workspace)) return ATTN_ERR_MISALIGNED;
    }
    return decode_launch(q, kcache, vcache, k_scale, v_scale, fp8, seqlens, page_table, o, lse,
                         num_seqs, H, d, max_seqlen, max_pages_per_seq, num_pages, scale, w,
                         workspace, stream);
}

}  // namespace
}  // namespace attn

extern "C" int attn_decode(const void* q, const void* kcache, const void* vcache, const int* seqlens,
                           const int* page_table, void* o, float* lse, int num_seqs, int H, int d,
                           int max_seqlen, int page_size, int max_pages_per_seq, int num_pages,
                           float scale, void* workspace, size_t workspace_bytes, void* stream) {
    return decode_impl(q, kcache, vcache, nullptr, nullptr, false, seqlens, page_table, o, lse,
                       num_seqs, H, d, max_seqlen, page_size, max_pages_per_seq, num_pages, scale,
                       workspace, workspace_bytes, stream);
}

extern "C" int attn_decode_fp8(const void* q, const void* kcache, const void* vcache,
                               const float* k_scale, const float* v_scale, const int* seqlens,
                               const int* page_table, void* o, float* lse, int num_seqs, int H,
                               int d, int max_seqlen, int page_size, int max_pages_per_seq,
                               int num_pages, float scale, void* workspace, size_t workspace_bytes,
                               void* stream) {
    return decode_impl(q, kcache, vcache, k_scale, v_scale, true, seqlens, page_table, o, lse,
                       num_seqs, H, d, max_seqlen, page_size, max_pages_per_seq, num_pages, scale,
                       workspace, workspace_bytes, stream);
}

extern "C" int attn_last_device_status(void* stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
    int value = 0;
    if (cudaMemcpyFromSymbol(&value, g_status, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
    return value;
}

extern "C" const char* attn_status_string(int status) {
    switch (status) {
        case ATTN_OK: return "ATTN_OK";
        case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
        case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
        case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED";
        case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
        case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
        case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT";
        default: return "ATTN_ERR_UNKNOWN";
    }
}

// ---- attn_decode_noalloc: attn_decode with the split partials in a fixed
// device array instead of a caller-provided workspace, for callers that cannot
// allocate device memory.  The array lives as long as the library is loaded.
namespace attn {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_address[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device, looked up once
// per device.  In host code the symbol itself is only a host-side handle, so
// kernels must be given this address.
int noalloc_scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_noalloc_address[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return ATTN_ERR_CUDA;
        g_noalloc_address[dev] = ptr;
    }
    *out = g_noalloc_address[dev];
    return ATTN_OK;
}

}  // namespace
}  // namespace attn

extern "C" int attn_decode_noalloc(const void* q, const void* kcache, const void* vcache,
                                   const int* seqlens, const int* page_table, void* o, float* lse,
                                   int num_seqs, int H, int d, int max_seqlen, int page_size,
                                   int max_pages_per_seq, int num_pages, float scale, void* stream) {
    // Every host-side check of attn_decode runs first, so that a bad call is
    // rejected before any CUDA call (the address lookup below).
    DecodeWorkspace w;
    bool empty = false;
    const int rc = decode_validate(q, kcache, vcache, nullptr, nullptr, false, seqlens, page_table, o,
                                   lse, num_seqs, H, d, max_seqlen, page_size, max_pages_per_seq,
                                   num_pages, scale, &w, &empty);
    if (rc != ATTN_OK || empty) return rc;
    if (max_seqlen > 0 && w.total > ATTN_DECODE_NOALLOC_SCRATCH_BYTES) return ATTN_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (max_seqlen > 0) {
        const int rs = noalloc_scratch_address(&scratch);
        if (rs != ATTN_OK) return rs;
    }
    return decode_launch(q, kcache, vcache, nullptr, nullptr, false, seqlens, page_table, o, lse,
                         num_seqs, H, d, max_seqlen, max_pages_per_seq, num_pages, scale, w, scratch,
                         stream);
}
