/*
 * gbattn.h -- C ABI of the GB300 (sm_103a) fused attention library.
 *
 * Two operations, both from the-ai.news, "Kernels de atencao rapida e fusao de
 * operadores", section "Atencao do tipo FlashAttention e atencao paginada":
 *
 *   attn_fwd           softmax attention computed block by block (scores for a
 *                      block, softmax statistics updated, output accumulated on
 *                      chip) so the T x T score matrix is never stored; i.e. the
 *                      result of the naive matmul / scale / causal mask / softmax /
 *                      matmul sequence (aiexpert.news, "Hugging Face Reduz
 *                      Sobrecarga de Atencao na Inferencia em 20-40% com Nucleos
 *                      Fundidos", second paragraph) in one kernel.
 *   paged_attn_decode  one new query token per request against a KV cache kept in
 *                      fixed-size blocks, every logical position translated
 *                      through a block table (block_size = 16, the value of the
 *                      page's vLLM example).
 *
 * Conventions for every entry point:
 *   - Tensor arguments are DEVICE pointers owned by the caller (any CUDA
 *     allocator).  The library never allocates, frees or keeps them, never
 *     synchronises the host, and enqueues work only on `stream` (a cudaStream_t
 *     passed as void*; NULL = the legacy default stream).
 *   - Tensors are contiguous, row-major, in the layouts stated below.  bf16 data
 *     pointers must be 16-byte aligned, fp32/int32 pointers 4-byte aligned.
 *   - Arguments are validated before anything is launched.  A non-OK status
 *     means nothing was enqueued (except ATTN_ERR_CUDA, see below).  There is no
 *     fallback path: unsupported inputs are an error, never a slower kernel.
 *   - Numerics: bf16 inputs, fp32 accumulation and fp32 softmax statistics; the
 *     probabilities are rounded to bf16 before they multiply V; O is rounded to
 *     bf16 (round-to-nearest-even).  LSE is the natural log of the sum of
 *     exp(scale * q.k) over the visible keys.
 *   - Thread-safe.  The first call on a device performs one-time set-up
 *     (kernel attributes, device checks).
 */
#ifndef GBATTN_H
#define GBATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, Hq % Hkv != 0, bad scale, small workspace */
    ATTN_ERR_UNSUPPORTED = 2, /* head dim not 64/128, block_size != 16, group > 16, not an sm_103 device, size limits */
    ATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call or a launch failed; work may be partially enqueued */
    ATTN_ERR_DEVICE = 4       /* reported only by attn_device_status(): a kernel flagged bad data or a timeout */
} attn_status_t;

/* Human-readable name of a status code (static string, never NULL). */
const char *attn_status_string(int status);

/*
 * attn_fwd -- fused attention forward (prefill / full attention).
 *
 *   q   [B, Hq,  T, D] bf16      k, v [B, Hkv, T, D] bf16
 *   o   [B, Hq,  T, D] bf16 (written)
 *   lse [B, Hq,  T]    fp32 (written; may be NULL to skip)
 *
 * Query head h reads KV head h / (Hq / Hkv) (grouped-query attention; Hkv = Hq
 * is multi-head attention).  With causal != 0 query i sees keys 0..i;
 * otherwise all T keys.  scale multiplies q.k (typically 1/sqrt(D)); it must be
 * finite and > 0.  D must be 64 or 128.  B = 0 or T = 0 is a no-op.
 * Returns ATTN_OK once the kernel is enqueued.
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
             int Hkv, int T, int D, int causal, float scale, void *stream);

/*
 * Bytes of scratch workspace paged_attn_decode needs for these sizes (partial
 * outputs of the split-KV pass).  Depends only on the arguments.
 */
size_t paged_attn_decode_workspace_size(int num_seqs, int Hq, int D, int max_seq_len);

/*
 * paged_attn_decode -- one query token per request against a paged KV cache.
 *
 *   q            [num_seqs, Hq, D] bf16  (the newest token of each request)
 *   k_pool/v_pool [num_pool_blocks, Hkv, block_size, D] bf16
 *   block_table  [num_seqs, max_blocks_per_seq] int32: logical block b of
 *                request r lives in physical block block_table[r][b]; entries
 *                past ceil(seq_lens[r] / block_size) are never read
 *   seq_lens     [num_seqs] int32 (device memory): tokens in each request's
 *                cache, the new token's own K/V included
 *   o            [num_seqs, Hq, D] bf16 (written)
 *   lse          [num_seqs, Hq] fp32 (written; may be NULL)
 *   workspace    >= paged_attn_decode_workspace_size(...) bytes of device
 *                memory, 256-byte aligned; its contents need no initialisation
 *                and are scratch after the call
 *
 * The query of request r attends to all seq_lens[r] cached tokens.  A request
 * with seq_lens[r] == 0 gets O = 0 and LSE = -inf.  max_seq_len bounds every
 * seq_lens[r] (it sizes the split-KV grid).  block_size must be 16, D 64 or 128,
 * Hq / Hkv <= 16.  Per-request data is checked on the device: a length outside
 * [0, min(max_seq_len, max_blocks_per_seq * block_size)] or a block id outside
 * [0, num_pool_blocks) makes that request's O and LSE NaN and sets a flag that
 * attn_device_status() reports; the kernel never traps.
 */
int paged_attn_decode(const void *q, const void *k_pool, const void *v_pool,
                      const int32_t *block_table, const int32_t *seq_lens, int block_size,
                      int num_seqs, int Hq, int Hkv, int D, int max_blocks_per_seq,
                      int num_pool_blocks, int max_seq_len, float scale, void *o, float *lse,
                      void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of device scratch paged_attn_decode_noalloc reserves on each device. */
#define GBATTN_DECODE_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * paged_attn_decode_noalloc -- paged_attn_decode without a caller workspace.
 *
 * The pages have no counterpart of this entry point; it exists for callers that
 * cannot allocate device memory at the point where they decode: code running
 * inside an allocator's own hooks, a host application that owns every device
 * allocation and hands out none, or a latency-critical loop that must never
 * enter the allocator.  Such a caller still owns and passes every input and
 * output (same arguments, layouts and checks as paged_attn_decode); only the
 * split-KV scratch comes from the library, from one fixed array of
 * GBATTN_DECODE_NOALLOC_SCRATCH_BYTES (16 MiB) in the library's device image.
 * Every GPU on which the library's kernels are loaded holds that array until
 * the process exits.  The call itself allocates nothing: no cudaMalloc, no
 * cudaFree, no allocating library routine.
 *
 *   - Sizes whose scratch, paged_attn_decode_workspace_size(num_seqs, Hq, D,
 *     max_seq_len), exceeds the array return ATTN_ERR_UNSUPPORTED before any
 *     work is enqueued (at D = 128 that is about 32,000 (request, query head,
 *     512-token chunk) partial results; 64 requests x 12 heads x 8192 tokens
 *     need 6.3 MB).
 *   - The first call on a device looks up the array's device address (once,
 *     with that device current); make that first call before any stream
 *     capture begins.
 *   - All calls on a device share the one array and it keeps whatever the last
 *     call wrote.  Nothing in it needs to start at zero: each call writes every
 *     scratch element it later reads.  Calls whose executions overlap on the GPU
 *     (different streams with no ordering between them) race on the array and
 *     give wrong results: order them on one stream or with events.
 */
int paged_attn_decode_noalloc(const void *q, const void *k_pool, const void *v_pool,
                              const int32_t *block_table, const int32_t *seq_lens, int block_size,
                              int num_seqs, int Hq, int Hkv, int D, int max_blocks_per_seq,
                              int num_pool_blocks, int max_seq_len, float scale, void *o,
                              float *lse, void *stream);

/*
 * Synchronises the current device, then reads and clears the library's device
 * flag word.  *flags (if not NULL) receives the raw bits: 1 = a bounded wait in
 * a kernel timed out, 2 = a decode request had an invalid length, 4 = a decode
 * block id was out of range.  Returns ATTN_ERR_DEVICE if any bit was set,
 * ATTN_ERR_CUDA if the synchronisation failed, else ATTN_OK.
 */
int attn_device_status(unsigned int *flags);

/* Library version as MAJOR * 10000 + MINOR * 100 + PATCH. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GBATTN_H */
