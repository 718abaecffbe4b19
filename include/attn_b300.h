/*
 * attn_b300.h -- C ABI of the B300 (sm_103a) exact-attention library.
 *
 * The library computes exact scaled-dot-product attention,
 *     O = softmax(scale * Q K^T [+ causal mask]) V,
 * tile by tile with the online-softmax recurrence, so that the N x N score
 * matrix never reaches device memory:
 *   - "FlashAttention complete summary" (cell-devlog.tistory.com/81), section
 *     "Attention이 뭔가": the formula softmax(QK^T / sqrt(d_k)) V;
 *   - same page, section "FlashAttention의 핵심 아이디어 — Tiling": Q blocks outer,
 *     K/V blocks inner, device-memory traffic limited to reading Q, K, V and
 *     writing O; online softmax keeps the result exact;
 *   - "Flash Attention ... complete guide" (holysheep.ai), section "Online
 *     Softmax 알고리즘": running maximum m, running sum l of exp(x - m);
 *   - "Beyond the memory wall" (tiptinker.com), section "구현 가이드": tensors
 *     are [batch, seq_len, num_heads, head_dim], bf16, contiguous, on the GPU;
 *     section "FlashInfer": decode processes one query per sequence against a
 *     growing K/V cache, optionally paged.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or retains them, and allocates no device memory
 *     of its own -- except two fixed arrays in the library's own device
 *     memory: the scratch array that attn_decode_noalloc uses (see its
 *     "Scratch" note), and 4096 work-unit counters of 4 bytes that
 *     attn_prefill_paged, and attn_fwd and attn_fwd_fp8 for long sequences,
 *     use (see attn_fwd).  bf16 means IEEE bfloat16 (raw
 *     16-bit storage), fp32 means IEEE binary32.  Every tensor is dense and
 *     row-major in the layout stated; every pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Work is enqueued on it and the call returns without waiting.
 *   - The return value is an attn_status.  Arguments are validated on the host
 *     before any CUDA call; a call that returns non-zero enqueued nothing,
 *     except ATTN_ERR_CUDA, which reports a failed launch.
 *   - Problems with an empty dimension (B, H, N or num_seqs == 0) return
 *     ATTN_OK and enqueue nothing.
 *   - Device-side failures (a pipeline wait that exceeded its time limit, a
 *     sequence length or page id out of range) are recorded in a device status
 *     word instead of faulting; read it with attn_last_device_status().
 *   - Thread safety: calls may be made from several host threads; the library
 *     keeps no per-call state.  The exception is attn_decode_noalloc, whose
 *     calls on one device share its scratch array (see its "Sharing" note).
 */
#ifndef ATTN_B300_H
#define ATTN_B300_H

#include <stddef.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,  /* NULL pointer, negative size, non-finite or non-positive scale,
                                  out-of-range device value (device status) */
    ATTN_ERR_UNSUPPORTED = 2,  /* head_dim not in {64, 128}, page_size != 16,
                                  sizes beyond int32 */
    ATTN_ERR_MISALIGNED = 3,   /* a pointer is not 16-byte aligned */
    ATTN_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than attn_decode_workspace_size() */
    ATTN_ERR_CUDA = 5,         /* a CUDA call (launch, attribute, tensor-map encode) failed */
    ATTN_ERR_TIMEOUT = 6       /* device status: a pipeline wait gave up after its time limit */
} attn_status;

/*
 * attn_fwd -- prefill / forward attention.
 *   "FlashAttention complete summary", sections "Attention이 뭔가" and
 *   "FlashAttention의 핵심 아이디어 — Tiling"; "Beyond the memory wall",
 *   section "구현 가이드" (the [batch, seq_len, num_heads, head_dim] layout and the
 *   softmax_scale and causal arguments of the forward call).
 *
 *   q, k, v : bf16 [B, N, H, d]   (element (b, n, h, c) at ((b*N + n)*H + h)*d + c)
 *   o       : bf16 [B, N, H, d]   output, rounded to nearest even from fp32
 *   lse     : fp32 [B, H, N] or NULL; lse[b,h,i] = ln sum_j exp(scale * q_i . k_j)
 *             over the visible keys j (natural log of the scaled scores)
 *   d       : head dimension, 64 or 128
 *   causal  : non-zero keeps key j for query i only when j <= i
 *   scale   : finite, > 0 (pass 1/sqrt(d) for the usual softmax scale)
 *   Accumulation is fp32; P is rounded to bf16 before the P V product.
 *   o must not alias q, k or v.
 *   Long sequences (K and V of one (batch, head) >= 4 MB, and more K/V than L2
 *   keeps at once for the heads the GPU's SMs would work on together): the
 *   work is taken band by band of heads whose K/V fits in L2, each SM taking
 *   its next unit from a counter in device memory.  The call zeroes one of
 *   4096 such counters on `stream` first, taking them in turn; calls in flight
 *   at the same time (on unordered streams, or replays of one captured call)
 *   must number fewer than 4096.  Results do not depend on the order.
 */
ATTN_API int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
             int B, int H, int N, int d, int causal, float scale, void* stream);

/*
 * attn_fwd_fp8 -- attn_fwd with Q, K and V in FP8 (E4M3), one fp32 scale per
 * head for each: the value of an element of head h is scale[h] * e4m3(byte).
 * Both products run on the FP8 tensor cores; P is rounded to E4M3 before the
 * P V product (relative error at most 2^-4 per weight), everything else
 * accumulates in fp32.  The output and LSE are those of attn_fwd on the
 * dequantized values, up to that rounding.
 *   "FlashAttention complete summary", section "FlashAttention 3" and "Beyond
 *   the memory wall", section "FlashAttention-3가 다른 이유" (FP8 support of the
 *   forward pass); the computation is attn_fwd's.
 *
 *   q, k    : E4M3 bytes [B, N, H, d]   (element (b, n, h, c) at ((b*N + n)*H + h)*d + c)
 *   vt      : E4M3 bytes [B, H, d, Np], V transposed so that keys are contiguous:
 *             element (b, h, c, n) at ((b*H + h)*d + c)*Np + n = V[b, n, h, c], with
 *             Np = N rounded up to a multiple of 16; bytes at n >= N are never read.
 *             (Every tensor-core operand is then K-major.)
 *   q_scale, k_scale, v_scale: fp32 [H], DEVICE memory
 *   o       : bf16 [B, N, H, d];  lse: fp32 [B, H, N] or NULL (natural log of the
 *             scaled scores of the dequantized values)
 *   d       : 64 or 128 (other head dimensions return ATTN_ERR_UNSUPPORTED)
 *   causal, scale: as attn_fwd.  o must not alias q, k or vt.
 *   Long sequences use attn_fwd's banded order and unit counters (K/V of one
 *   (batch, head) counted at one byte per element).
 */
ATTN_API int attn_fwd_fp8(const void* q, const void* k, const void* vt, const float* q_scale,
             const float* k_scale, const float* v_scale, void* o, float* lse, int B, int H, int N,
             int d, int causal, float scale, void* stream);

/*
 * attn_prefill_paged -- prefill of a new chunk of Nq query tokens per sequence
 * against its K/V cache in 16-token pages (chunked prefill, or prefill after a
 * cached prefix).  The same computation as attn_fwd, with the keys and values
 * of sequence b taken from the paged cache and the causal mask aligned to the
 * end of the cache.
 *   "Beyond the memory wall", section "FlashInfer" (prefill and decode
 *   kernels over a paged K/V cache); "FlashAttention complete summary",
 *   section "FlashAttention의 핵심 아이디어 — Tiling" (the tiled computation).
 *
 *   q        : bf16 [B, Nq, H, d]; row i of sequence b is the token at cache
 *              position seqlens[b] - Nq + i
 *   kcache, vcache: bf16 pools [num_pages, page_size, H, d]; key t of sequence b
 *              is slot t % page_size of page page_table[b*max_pages_per_seq + t/page_size].
 *              The chunk's own K/V are already in the cache.  Whole pages are
 *              read: slots of a sequence's last page beyond its length must hold
 *              finite values (e.g. zeros).
 *   seqlens  : int32 [B], DEVICE memory, Nq <= seqlens[b] <= max_pages_per_seq*page_size
 *              (keys of sequence b, chunk included).  A value outside is clamped
 *              and recorded as ATTN_ERR_INVALID_ARG in the device status.
 *   page_table: int32 [B, max_pages_per_seq], DEVICE memory.  An id outside
 *              [0, num_pages) is replaced by page 0 and recorded as
 *              ATTN_ERR_INVALID_ARG in the device status.
 *   o        : bf16 [B, Nq, H, d]
 *   lse      : fp32 [B, H, Nq] or NULL (natural log of the scaled scores)
 *   d        : 64 or 128;  page_size: 16;  num_pages <= 2^26
 *   causal   : non-zero keeps key j for query row i only when j <= seqlens[b] - Nq + i
 *   scale    : finite, > 0
 *   Accumulation is fp32; P is rounded to bf16 before the P V product.
 *   o must not alias q or the caches.
 *   The work (longest cache first) is dealt to the SMs through one of
 *   attn_fwd's 4096 unit counters, with the same rule on calls in flight.
 */
ATTN_API int attn_prefill_paged(const void* q, const void* kcache, const void* vcache,
                const int* seqlens, const int* page_table, void* o, float* lse, int B, int H,
                int Nq, int d, int page_size, int max_pages_per_seq, int num_pages, int causal,
                float scale, void* stream);

/*
 * attn_bwd -- gradients of attn_fwd (the backward pass, for training): given the
 * forward's inputs, its output O and row log-sum-exp LSE, and the upstream gradient
 * dO = dL/dO, writes dQ, dK, dV.  S and P are recomputed tile by tile from Q, K and
 * LSE instead of being stored (P = exp(scale * Q K^T - LSE)):
 *     dV = P^T dO,  dP = dO V^T,  D_i = dO_i . O_i,  dS = P * (dP - D),
 *     dQ = scale * dS K,  dK = scale * dS^T Q.
 *   "Beyond the memory wall", section "FlashAttention: IO 인식의 정점" (tiling and
 *   recomputation); "FlashAttention complete summary", section "Attention이 뭔가"
 *   (the function being differentiated).
 *
 *   q, k, v, o, dout: bf16 [B, N, H, d] (o and lse as written by attn_fwd with the
 *             same q, k, v, causal and scale)
 *   lse     : fp32 [B, H, N]
 *   dq, dk, dv: bf16 [B, N, H, d] outputs; fp32 accumulation, P and dS rounded to bf16
 *             before their products.  No atomics: the result is deterministic.
 *   d       : 64 or 128;  causal, scale: as attn_fwd
 *   workspace: device buffer of at least attn_bwd_workspace_size(B, H, N, d) bytes,
 *             16-byte aligned, no initialisation needed; calls that share it must be
 *             ordered on one stream.  Outputs alias neither inputs, workspace nor
 *             each other.
 */
ATTN_API size_t attn_bwd_workspace_size(int B, int H, int N, int d);

ATTN_API int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, int B, int H, int N, int d,
             int causal, float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_decode_workspace_size -- bytes of device workspace attn_decode needs
 * for these sizes (the per-split partial outputs and log-sum-exps of the
 * split-KV scheme).  Returns 0 for invalid or empty sizes.
 */
ATTN_API size_t attn_decode_workspace_size(int num_seqs, int H, int d, int max_seqlen);

/*
 * attn_decode -- one query token per sequence against its K/V cache
 * (split-KV: each split of 256 cache tokens is reduced with its own softmax,
 * then the splits are merged by their log-sum-exps).
 *   "Beyond the memory wall", section "FlashInfer" (decode against the K/V
 *   cache; PagedAttention); "Transformers local LLM slow? apply
 *   FlashAttention2" (beautifulsoup.dev), section on prefill and decode.
 *
 *   q        : bf16 [num_seqs, 1, H, d]
 *   kcache, vcache:
 *     page_table == NULL : bf16 [num_seqs, max_seqlen, H, d]; token t of
 *                          sequence s at row (s, t)
 *     page_table != NULL : bf16 pools [num_pages, page_size, H, d]; token t of
 *                          sequence s in page page_table[s*max_pages_per_seq + t/page_size],
 *                          slot t % page_size
 *   seqlens  : int32 [num_seqs], DEVICE memory, 0 <= seqlens[s] <= max_seqlen;
 *              the cache already holds the current token's K/V.  A sequence of
 *              length 0 gets O = 0 and LSE = -inf.  A length outside the range
 *              is clamped and recorded as ATTN_ERR_INVALID_ARG in the device status.
 *   page_table: int32 [num_seqs, max_pages_per_seq], DEVICE memory, or NULL.
 *              An id outside [0, num_pages) is skipped (its tokens ignored) and
 *              recorded as ATTN_ERR_INVALID_ARG in the device status.
 *   o        : bf16 [num_seqs, 1, H, d]
 *   lse      : fp32 [num_seqs, H] or NULL
 *   d        : 64 or 128
 *   max_seqlen: contiguous: the cache's second dimension; paged: at most
 *              max_pages_per_seq * page_size
 *   page_size: 16 (paged); ignored when page_table == NULL
 *   max_pages_per_seq, num_pages: paged layout sizes; ignored when page_table == NULL
 *   scale    : finite, > 0
 *   workspace: device buffer of at least attn_decode_workspace_size(num_seqs,
 *              H, d, max_seqlen) bytes, 16-byte aligned, owned by the caller;
 *              its contents need no initialisation.  Calls that share a
 *              workspace must be ordered on one stream.
 */
ATTN_API int attn_decode(const void* q, const void* kcache, const void* vcache, const int* seqlens,
                const int* page_table, void* o, float* lse, int num_seqs, int H, int d,
                int max_seqlen, int page_size, int max_pages_per_seq, int num_pages,
                float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_decode_fp8 -- attn_decode over a K/V cache quantized to FP8 (e4m3), one
 * fp32 scale per head for keys and one for values: the key of token t, head h
 * is k_scale[h] * e4m3(kcache[..]), likewise for values.  The attention itself
 * is attn_decode's; the cache is half the bytes, so the bandwidth-bound decode
 * reads half as much per token.
 *   "Beyond the memory wall", section "FlashInfer" (decode against a paged
 *   K/V cache, quantized K/V among its options).
 *
 *   kcache, vcache: e4m3 bytes, layouts as attn_decode (contiguous
 *              [num_seqs, max_seqlen, H, d] or pools [num_pages, page_size, H, d])
 *   k_scale, v_scale: fp32 [H], DEVICE memory
 *   Every other argument, layout and rule as attn_decode; the workspace size is
 *   attn_decode_workspace_size() of the same sizes.
 */
ATTN_API int attn_decode_fp8(const void* q, const void* kcache, const void* vcache,
                const float* k_scale, const float* v_scale, const int* seqlens,
                const int* page_table, void* o, float* lse, int num_seqs, int H, int d,
                int max_seqlen, int page_size, int max_pages_per_seq, int num_pages,
                float scale, void* workspace, size_t workspace_bytes, void* stream);

/*
 * attn_decode_noalloc -- attn_decode for callers that cannot allocate device
 * memory: a plugin hosted inside another runtime that owns all device memory
 * and hands it no allocator, or a serving loop that forbids cudaMalloc (and
 * the device-wide synchronisation it can bring) once it is running.  Such a
 * caller still passes q, the caches, seqlens, page_table, o and lse, but no
 * workspace: the split partials go to a scratch array inside the library.
 * (The pages have no counterpart to this entry point; it is an interface
 * convenience, the arithmetic is attn_decode's.)
 *
 *   Arguments and layouts: as attn_decode, without workspace/workspace_bytes.
 *   Scratch: a fixed array of ATTN_DECODE_NOALLOC_SCRATCH_BYTES in device
 *            memory, reserved on every GPU that loads the library until the
 *            process exits.  Sizes whose attn_decode_workspace_size() exceeds
 *            it are rejected with ATTN_ERR_WORKSPACE before anything runs.
 *   Set-up:  the first call on a device (with that device current) looks up
 *            the array's device address; make that first call before any
 *            stream capture.  No call allocates or frees memory.
 *   Sharing: every call on a device uses the same array and leaves its
 *            contents behind; nothing in it needs to start at zero.  Calls
 *            that can overlap on the GPU (different streams without ordering
 *            between them) race on the array: order them on one stream.
 */
#define ATTN_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

ATTN_API int attn_decode_noalloc(const void* q, const void* kcache, const void* vcache,
                const int* seqlens, const int* page_table, void* o, float* lse, int num_seqs,
                int H, int d, int max_seqlen, int page_size, int max_pages_per_seq,
                int num_pages, float scale, void* stream);

/*
 * attn_last_device_status -- synchronises `stream`, then returns and clears
 * the device status word of the current device (ATTN_OK when no kernel
 * recorded a failure since the last call), or ATTN_ERR_CUDA if the
 * synchronisation itself failed.
 */
ATTN_API int attn_last_device_status(void* stream);

/* attn_status_string -- a static, human-readable name for a status code. */
ATTN_API const char* attn_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_B300_H */
