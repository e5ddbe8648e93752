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
 * paged_attn_prefill -- attention of a chunk of new tokens against a paged KV
 * cache (chunked prefill).  The blockwise computation of attn_fwd, with every key
 * and value position translated through the block table (same the-ai.news
 * section; block_size = 16 as in its vLLM example).
 *
 *   q             [B, Hq, Tq, D] bf16: the Tq newest tokens of each batch item
 *   k_pool/v_pool [num_pool_blocks, Hkv, block_size, D] bf16
 *   block_table   [B, max_blocks_per_seq] int32: logical block t / block_size of
 *                 item b lives in physical block block_table[b][t / block_size];
 *                 entries past ceil(kv_lens[b] / block_size) are never read
 *   kv_lens       [B] int32 (device memory): tokens in each item's cache, the Tq
 *                 new tokens' own keys and values included
 *   o             [B, Hq, Tq, D] bf16 (written)
 *   lse           [B, Hq, Tq] fp32 (written; may be NULL)
 *
 * Query i of item b is the token at logical position kv_lens[b] - Tq + i.  With
 * causal != 0 it sees keys 0 .. kv_lens[b] - Tq + i (the mask is aligned with the
 * last key); otherwise all kv_lens[b] keys.  A query that sees no key (causal
 * with kv_lens[b] < Tq) gets O = 0 and LSE = -inf.  max_kv_len bounds every
 * kv_lens[b].  block_size must be 16 and D 64 or 128.  Per-item data is checked
 * on the device: a kv_lens[b] outside [0, min(max_kv_len, max_blocks_per_seq *
 * block_size)] makes that item's O and LSE NaN and sets flag bit 2; a block id
 * outside [0, num_pool_blocks) is read as block 0 and sets flag bit 4 (that
 * item's output is then unspecified).  Pool slots past kv_lens[b] may hold any
 * bits, NaN included: they never reach the output.
 */
int paged_attn_prefill(const void *q, const void *k_pool, const void *v_pool,
                       const int32_t *block_table, const int32_t *kv_lens, int block_size, int B,
                       int Hq, int Hkv, int Tq, int D, int max_blocks_per_seq,
                       int num_pool_blocks, int max_kv_len, int causal, float scale, void *o,
                       float *lse, void *stream);

/*
 * Bytes of scratch workspace paged_attn_decode needs for these sizes.  The
 * decode cuts the batch's (request, KV head, 16-token block) sequence into equal
 * ranges of at least 256 tokens; each range that meets a request's cache yields
 * one partial output (D fp32) and LSE per query head, at most
 * ceil(max_seq_len / 256) + 1 per (request, query head).  Depends only on the
 * arguments; the block size is not one of them (it is fixed at 16 and checked by
 * paged_attn_decode).
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
 * seq_lens[r] (it sizes the workspace).  The split of the work depends on the
 * lengths of the whole batch, never on where the blocks sit in the pool: the
 * same inputs give the same bits, whatever the placement.  block_size must be 16, D 64 or 128,
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
 *     range) partial results; 64 requests x 12 heads x 8192 tokens need
 *     13.1 MB).
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
 * Synchronises the current device (every stream), then reads and clears the
 * library's device flag word.  The word is one per device, shared by every
 * stream and every caller of the library in the process: a flag raised by any
 * kernel of this library on that device stays set until the next call of this
 * function, which reports and clears it for everyone.  *flags (if not NULL) receives the raw bits: 1 = a bounded wait in
 * a kernel timed out, 2 = a decode request had an invalid length, 4 = a decode
 * block id was out of range.  Returns ATTN_ERR_DEVICE if any bit was set,
 * ATTN_ERR_CUDA if the synchronisation failed, else ATTN_OK.
 */
int attn_device_status(unsigned int *flags);

/*
 * paged_kv_append -- writes Tn new tokens per request into the paged KV cache (the
 * cache "grows one token at a time", same the-ai.news section).
 *
 *   k_new, v_new  [num_seqs, Hkv, Tn, D] bf16: the new tokens' keys and values
 *   k_pool/v_pool [num_pool_blocks, Hkv, block_size, D] bf16 (written in place)
 *   block_table   [num_seqs, max_blocks_per_seq] int32; the blocks that the new
 *                 positions fall into must already be assigned
 *   seq_lens      [num_seqs] int32 (device): tokens already cached, L_r
 *   new_seq_lens  [num_seqs] int32 (device, may be NULL): receives L_r + Tn; it
 *                 must not overlap seq_lens
 *
 * Token t of request r goes to logical position L_r + t, i.e. physical block
 * block_table[r][(L_r + t) / 16], slot (L_r + t) % 16.  The copy is exact (bits
 * in = bits out).  Device-side checks: L_r < 0 or L_r + Tn > max_blocks_per_seq *
 * block_size skips the request, sets flag bit 2 and writes L_r unchanged to
 * new_seq_lens; a block id outside the pool skips that token and sets flag bit 4.
 * block_size must be 16, D 64 or 128.
 */
int paged_kv_append(const void *k_new, const void *v_new, void *k_pool, void *v_pool,
                    const int32_t *block_table, const int32_t *seq_lens, int32_t *new_seq_lens,
                    int block_size, int num_seqs, int Hkv, int Tn, int D, int max_blocks_per_seq,
                    int num_pool_blocks, void *stream);

/*
 * paged_kv_gather -- copies each request's cached keys (or values) out of the
 * paged pool in logical order, with the same block-table translation and the
 * same TMA box copies that the attention kernels use.
 *
 *   pool          [num_pool_blocks, Hkv, block_size, D] bf16
 *   block_table   [num_seqs, max_blocks_per_seq] int32
 *   seq_lens      [num_seqs] int32 (device)
 *   out           [num_seqs, Hkv, max_seq_len, D] bf16: out[r][h][t] = the row of
 *                 token t < seq_lens[r]; rows t >= seq_lens[r] are not written
 *
 * Device-side checks: a length outside [0, min(max_seq_len, max_blocks_per_seq
 * * block_size)] skips the request and sets flag bit 2; a block id outside the
 * pool writes NaN rows for that block and sets flag bit 4.
 */
int paged_kv_gather(const void *pool, const int32_t *block_table, const int32_t *seq_lens,
                    int block_size, int num_seqs, int Hkv, int D, int max_blocks_per_seq,
                    int num_pool_blocks, int max_seq_len, void *out, void *stream);

/*
 * Test hook for the kernels' failure detection (not for production use).
 * Kernels launched after this call use wait_limit_ns as the limit, in
 * nanoseconds, of every pipeline wait (0 restores the default of 2 s).  With
 * withhold_copy = 1 the copy warp of every CTA of the next kernels skips its
 * first data copy, so a consumer's wait for it is certain to run out: the
 * waiting role raises flag bit 1, tells the CTA's other roles to stop, lets the
 * copies and MMAs already in flight finish, and the kernel returns with
 * unspecified outputs; attn_device_status() then reports ATTN_ERR_DEVICE.  No
 * fault, trap or hang is involved.  Call attn_test_set_failure(0, 0) to restore
 * normal operation.  Process-wide; not meant for use while other threads launch
 * kernels of this library.  Returns ATTN_OK, or ATTN_ERR_INVALID_ARG if
 * withhold_copy is not 0 or 1.
 */
int attn_test_set_failure(unsigned long long wait_limit_ns, int withhold_copy);

/* Library version as MAJOR * 10000 + MINOR * 100 + PATCH. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GBATTN_H */
