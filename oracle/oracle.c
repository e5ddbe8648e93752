/*
 * oracle.c -- plain fp64 CPU reference for softmax attention and paged-KV decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU
 * baseline load this file's library.  It shares no code, header, table or helper
 * with the CUDA path, and it is deliberately slow: for every query row it
 * materialises that row's full score vector, takes a two-pass softmax (max, then
 * exp and sum) and contracts the probabilities with V.  No tiling, no online
 * softmax, no blocking.
 *
 * What it computes: the plain definition that FlashAttention reaches without
 * storing the score matrix (the-ai.news, "Kernels de atencao rapida e fusao de
 * operadores", section "Atencao do tipo FlashAttention e atencao paginada"),
 * i.e. the naive matmul / scale / causal mask / softmax / matmul sequence of
 * aiexpert.news, "Hugging Face Reduz Sobrecarga de Atencao na Inferencia em
 * 20-40% com Nucleos Fundidos", second paragraph:
 *
 *   for batch b, query head h, query row i, with kv = h / (Hq / Hkv) and the
 *   visible key set V_i = { j : 0 <= j < Tk, and j <= i + (Tk - Tq) if causal }:
 *     s_ij  = scale * sum_d q[b,h,i,d] * k[b,kv,j,d]
 *     m_i   = max_{j in V_i} s_ij
 *     l_i   = sum_{j in V_i} exp(s_ij - m_i)
 *     P_ij  = exp(s_ij - m_i) / l_i                 (0 for j not in V_i)
 *     O_i   = sum_j P_ij * v[b,kv,j,:]
 *     LSE_i = m_i + ln(l_i)                          (natural log, scale included)
 *
 * Paged decode (same the-ai.news section: the cache is cut into fixed-size
 * blocks, a block table maps logical positions to physical blocks, and the
 * attention kernel translates every position through it; its vLLM example uses
 * block_size = 16): request r with length L gathers K_r[t] = k_pool[block_table[r][t/bs],
 * kv, t % bs, :] for t < L (likewise V), and its one query (the newest token,
 * position L-1) sees all L keys.  L = 0 gives O = 0 and LSE = -inf.
 *
 * Inputs are bf16 bit patterns (uint16); they are widened to double exactly.
 * Layouts: q [B,Hq,Tq,D], k/v [B,Hkv,Tk,D], o [B,Hq,Tq,D], lse [B,Hq,Tq] (all
 * contiguous, row-major).  Paged: q [S,Hq,D], pools [NB,Hkv,bs,D], block_table
 * [S,max_blocks] int32, seq_lens [S] int32, o [S,Hq,D], lse [S,Hq].
 *
 * Return codes: 0 ok, -1 invalid argument / index, -2 out of memory.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * One query row against a key/value set given as arrays of row pointers.
 * kr[j], vr[j] point at the D bf16 values of key/value j (j < nk).  visible(j)
 * is j < n_vis (the caller orders keys so the visible ones come first).
 * p is scratch of nk doubles; on return p[j] holds P_ij for j < n_vis.
 */
static void attend_row(const uint16_t *qrow, const uint16_t *const *kr, const uint16_t *const *vr,
                       int n_vis, int D, double scale, double *p, double *orow, double *lse)
{
    if (n_vis <= 0) {
        for (int d = 0; d < D; ++d) orow[d] = 0.0;
        *lse = -INFINITY;
        return;
    }
    /* scores: s_j = scale * q . k_j */
    for (int j = 0; j < n_vis; ++j) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += bf16_to_double(qrow[d]) * bf16_to_double(kr[j][d]);
        p[j] = scale * acc;
    }
    /* pass 1: row max */
    double m = p[0];
    for (int j = 1; j < n_vis; ++j)
        if (p[j] > m) m = p[j];
    /* pass 2: exponentials and their sum */
    double l = 0.0;
    for (int j = 0; j < n_vis; ++j) {
        p[j] = exp(p[j] - m);
        l += p[j];
    }
    /* normalised probabilities, then O = P V */
    for (int j = 0; j < n_vis; ++j) p[j] /= l;
    for (int d = 0; d < D; ++d) orow[d] = 0.0;
    for (int j = 0; j < n_vis; ++j) {
        const double pj = p[j];
        for (int d = 0; d < D; ++d) orow[d] += pj * bf16_to_double(vr[j][d]);
    }
    *lse = m + log(l);
}

static int check_dims(int B, int Hq, int Hkv, int Tq, int Tk, int D)
{
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Tq < 0 || Tk < 0 || D <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    return 0;
}

/* Number of keys visible to query row i (keys 0 .. n-1). */
static int visible_keys(int i, int Tq, int Tk, int causal)
{
    if (!causal) return Tk;
    long long n = (long long)i + (Tk - Tq) + 1; /* bottom-right alignment; Tq == Tk is top-left too */
    if (n < 0) n = 0;
    if (n > Tk) n = Tk;
    return (int)n;
}

/*
 * Attention for an explicit list of rows.  rows[n] = ((b * Hq) + h) * Tq + i.
 * o_rows [n_rows, D], lse_rows [n_rows].  p_rows (nullable) [n_rows, Tk]
 * receives the probability row (zeros past the visible keys).
 */
int oracle_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, int B, int Hq,
                     int Hkv, int Tq, int Tk, int D, int causal, double scale, long long n_rows,
                     const long long *rows, double *o_rows, double *lse_rows, double *p_rows)
{
    if (check_dims(B, Hq, Hkv, Tq, Tk, D)) return -1;
    if (n_rows < 0 || (n_rows > 0 && (!q || !k || !v || !rows || !o_rows || !lse_rows))) return -1;
    const long long total = (long long)B * Hq * Tq;
    for (long long n = 0; n < n_rows; ++n)
        if (rows[n] < 0 || rows[n] >= total) return -1;
    const int group = Hq / Hkv;
    int status = 0;

#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)(Tk > 0 ? Tk : 1));
        const uint16_t **kr = (const uint16_t **)malloc(sizeof(void *) * (size_t)(Tk > 0 ? Tk : 1));
        const uint16_t **vr = (const uint16_t **)malloc(sizeof(void *) * (size_t)(Tk > 0 ? Tk : 1));
        const int ok = p && kr && vr;
        if (!ok) {
#pragma omp atomic write
            status = -2;
        }
#pragma omp for schedule(dynamic, 16)
        for (long long n = 0; n < n_rows; ++n) {
            if (ok) {
                const long long r = rows[n];
                const int i = (int)(r % Tq);
                const long long bh = r / Tq;
                const int h = (int)(bh % Hq);
                const int b = (int)(bh / Hq);
                const int kvh = h / group;
                const uint16_t *qrow = q + r * D;
                const long long kv_base = ((long long)b * Hkv + kvh) * Tk;
                for (int j = 0; j < Tk; ++j) {
                    kr[j] = k + (kv_base + j) * D;
                    vr[j] = v + (kv_base + j) * D;
                }
                const int nv = visible_keys(i, Tq, Tk, causal);
                attend_row(qrow, kr, vr, nv, D, scale, p, o_rows + n * D, lse_rows + n);
                if (p_rows) {
                    double *pr = p_rows + n * (long long)Tk;
                    for (int j = 0; j < Tk; ++j) pr[j] = j < nv ? p[j] : 0.0;
                }
            }
        }
        free(p);
        free(kr);
        free(vr);
    }
    return status;
}

/* Full attention: every row of every (b, h). o [B,Hq,Tq,D], lse [B,Hq,Tq]. */
int oracle_attn_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, double *o,
                    double *lse, int B, int Hq, int Hkv, int Tq, int Tk, int D, int causal,
                    double scale)
{
    if (check_dims(B, Hq, Hkv, Tq, Tk, D)) return -1;
    const long long total = (long long)B * Hq * Tq;
    long long *rows = (long long *)malloc(sizeof(long long) * (size_t)(total > 0 ? total : 1));
    if (!rows) return -2;
    for (long long r = 0; r < total; ++r) rows[r] = r;
    int st = oracle_attn_rows(q, k, v, B, Hq, Hkv, Tq, Tk, D, causal, scale, total, rows, o, lse,
                              NULL);
    free(rows);
    return st;
}

/*
 * Translate logical token t of request r through the block table:
 * element offset of pool[block_table[r][t / bs], kvh, t % bs, 0].
 * Returns -1 when the table entry is outside [0, num_pool_blocks).
 */
static long long paged_offset(const int32_t *block_table, int max_blocks, int r, int t, int kvh,
                              int Hkv, int bs, int D, int num_pool_blocks)
{
    const int32_t phys = block_table[(long long)r * max_blocks + t / bs];
    if (phys < 0 || phys >= num_pool_blocks) return -1;
    return (((long long)phys * Hkv + kvh) * bs + (t % bs)) * (long long)D;
}

/*
 * Gather the contiguous K (or V) history of request r, kv head kvh: out [L, D].
 * Exposed so tests can check the paged and contiguous forms against each other.
 */
int oracle_paged_gather(const uint16_t *pool, const int32_t *block_table, const int32_t *seq_lens,
                        int r, int kvh, int Hkv, int block_size, int D, int max_blocks,
                        int num_pool_blocks, uint16_t *out)
{
    const int L = seq_lens[r];
    if (L < 0 || L > max_blocks * block_size || kvh < 0 || kvh >= Hkv) return -1;
    for (int t = 0; t < L; ++t) {
        long long off = paged_offset(block_table, max_blocks, r, t, kvh, Hkv, block_size, D,
                                     num_pool_blocks);
        if (off < 0) return -1;
        memcpy(out + (long long)t * D, pool + off, sizeof(uint16_t) * (size_t)D);
    }
    return 0;
}

/* Single-token decode per request against the paged cache. */
int oracle_paged_decode(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                        const int32_t *block_table, const int32_t *seq_lens, int num_seqs, int Hq,
                        int Hkv, int D, int block_size, int max_blocks, int num_pool_blocks,
                        double scale, double *o, double *lse)
{
    if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || block_size <= 0 || Hq % Hkv) return -1;
    for (int r = 0; r < num_seqs; ++r) {
        const int L = seq_lens[r];
        if (L < 0 || L > max_blocks * block_size) return -1;
        for (int lb = 0; lb < (L + block_size - 1) / block_size; ++lb) {
            const int32_t phys = block_table[(long long)r * max_blocks + lb];
            if (phys < 0 || phys >= num_pool_blocks) return -1;
        }
    }
    const int group = Hq / Hkv;
    int status = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long long rh = 0; rh < (long long)num_seqs * Hq; ++rh) {
        const int r = (int)(rh / Hq);
        const int h = (int)(rh % Hq);
        const int kvh = h / group;
        const int L = seq_lens[r];
        double *p = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        const uint16_t **kr = (const uint16_t **)malloc(sizeof(void *) * (size_t)(L > 0 ? L : 1));
        const uint16_t **vr = (const uint16_t **)malloc(sizeof(void *) * (size_t)(L > 0 ? L : 1));
        if (!p || !kr || !vr) {
#pragma omp atomic write
            status = -2;
        } else {
            for (int t = 0; t < L; ++t) {
                const long long off = paged_offset(block_table, max_blocks, r, t, kvh, Hkv,
                                                   block_size, D, num_pool_blocks);
                kr[t] = k_pool + off;
                vr[t] = v_pool + off;
            }
            /* the query is token L-1 and sees keys 0 .. L-1 */
            attend_row(q + rh * D, kr, vr, L, D, scale, p, o + rh * D, lse + rh);
        }
        free(p);
        free(kr);
        free(vr);
    }
    return status;
}

/* Threads the OpenMP runtime will use (for reporting the CPU baseline). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
