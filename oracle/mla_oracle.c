/*
 * Float64 CPU oracle for MLA decode attention.
 *
 * TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference arm of bench.py may load or call this file.  It
 * shares no code, header, table or helper with the CUDA library in
 * mla_decode_attention_05_gb300/, and the library never calls it.
 *
 * What it computes, for one query row (batch b, query token t, head h):
 *
 *   K_n   = the 576 values of the latent KV row of logical token n of sequence
 *           b, reached through block_table[b][n / page_size] and slot
 *           n % page_size (vLLM MlaQuery.insert: page, offset = slot //
 *           page_size, slot % page_size);  V_n = K_n[0:512]
 *           (STAGE_D2.md "DSV4 is MQA": all query heads share one K/V;
 *           FlashMLA issue #169 "dual gemm": the 64 RoPE values are just one
 *           more block of the QK reduction, so no rotation happens here, and
 *           vLLM MlaQuery.insert stores k_pe unrotated at columns 512..575).
 *   N     = the valid keys: n < s_k (dense), n < s_k - T + t + 1 (causal,
 *           query token t of T sees the keys up to its own position), or the
 *           top-k indices of (b, t) other than -1 (sparse; FlashMLA issue #169
 *           is the sparse decode kernel, whose mask step drops invalid slots).
 *           The indices of one list are distinct positions (a list that
 *           repeats one is refused: see oracle_valid_keys).
 *   s_n   = softmax_scale * sum_d q_d K_{n,d}           (d over all 576)
 *   LSE   = m + ln(sum_{n in N} exp(s_n - m)),  m = max_n s_n
 *   O     = sum_{n in N} exp(s_n - LSE) V_n
 *   empty N: O = 0, LSE = -inf (the natural log of an empty sum).
 *
 * Element decoders follow the public formats: bf16 is the upper half of an
 * IEEE binary32; OCP FP8 E4M3 has 1 sign, 4 exponent (bias 7) and 3 mantissa
 * bits, subnormals at exponent 0, no infinities, and S.1111.111 = NaN.
 * FP8 rows: 512 e4m3 bytes then 64 bf16 RoPE values (640 bytes), with one
 * fp32 scale per 128-wide tile of the 512; the dequantised value is the exact
 * product e4m3(byte) * scale.  Per-tensor FP8 rows (the layout vLLM's
 * MlaQuery.insert writes): 576 e4m3 bytes, RoPE included, all dequantised
 * with one fp32 scale (the reciprocal of the writer's k_scale_inv).
 *
 * Everything is plain double arithmetic; the only library calls are exp, log
 * and ldexp.  Row-level OpenMP parallelism does not change any result.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_D_QK 576
#define ORACLE_D_V 512
#define ORACLE_FP8_ROW 640
#define ORACLE_FP8T_ROW 576

double oracle_bf16_to_f64(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double oracle_e4m3_to_f64(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* The KV cache as the oracle sees it. */
typedef struct {
    const void *kv;           /* bf16 bits [P][page][576], bytes [P][page][640] or [P][page][576] */
    int kv_format;            /* 0 = bf16, 1 = fp8 e4m3 + bf16 rope, 2 = per-tensor fp8 (576 e4m3) */
    int num_pages;
    int page_size;
    const float *kv_scales;   /* format 1: [P][page][4]; format 2: one scale */
    const int32_t *block_table;
    int max_pages;
} oracle_cache;

/* Dequantise the row of logical token n of sequence b into row[576].
 * Returns 0, or -1 if the token's page is outside the pool. */
static int load_key_row(const oracle_cache *c, int b, int n, double *row)
{
    int page = c->block_table[(int64_t)b * c->max_pages + n / c->page_size];
    int slot = n % c->page_size;
    if (page < 0 || page >= c->num_pages)
        return -1;
    int64_t r = (int64_t)page * c->page_size + slot;
    if (c->kv_format == 0) {
        const uint16_t *p = (const uint16_t *)c->kv + r * ORACLE_D_QK;
        for (int d = 0; d < ORACLE_D_QK; d++)
            row[d] = oracle_bf16_to_f64(p[d]);
    } else if (c->kv_format == 2) {
        const uint8_t *p = (const uint8_t *)c->kv + r * ORACLE_FP8T_ROW;
        for (int d = 0; d < ORACLE_D_QK; d++)
            row[d] = oracle_e4m3_to_f64(p[d]) * (double)c->kv_scales[0];
    } else {
        const uint8_t *p = (const uint8_t *)c->kv + r * ORACLE_FP8_ROW;
        const float *sc = c->kv_scales + r * 4;
        for (int d = 0; d < ORACLE_D_V; d++)
            row[d] = oracle_e4m3_to_f64(p[d]) * (double)sc[d / 128];
        const uint8_t *rope = p + ORACLE_D_V;
        for (int d = 0; d < ORACLE_D_QK - ORACLE_D_V; d++) {
            uint16_t bits = (uint16_t)(rope[2 * d] | (rope[2 * d + 1] << 8));
            row[ORACLE_D_V + d] = oracle_bf16_to_f64(bits);
        }
    }
    return 0;
}

/* The valid key set of query token t of sequence b, sorted ascending.
 * Writes at most cap entries; returns the set's size, or -2 when a top-k
 * list names one position twice: the indices of one query token are a
 * selection of distinct cache positions (top-k of a score over the tokens,
 * FlashMLA issue #169's sparse decode), so a repeated position is outside
 * the definition and the oracle refuses it rather than pick a meaning. */
int oracle_valid_keys(int b, int t, int T, const int32_t *cache_seqlens,
                      const int32_t *topk, int topk_len, int causal,
                      int32_t *out, int cap)
{
    int sk = cache_seqlens[b];
    int count = 0;
    if (topk != NULL && topk_len > 0) {
        const int32_t *ids = topk + ((int64_t)b * T + t) * topk_len;
        /* membership by scanning the key positions in order (sorted) */
        char *seen = (char *)calloc((size_t)(sk > 0 ? sk : 1), 1);
        for (int k = 0; k < topk_len; k++)
            if (ids[k] >= 0 && ids[k] < sk) {
                if (seen[ids[k]]) {
                    free(seen);
                    return -2;
                }
                seen[ids[k]] = 1;
            }
        for (int n = 0; n < sk; n++)
            if (seen[n]) {
                if (count < cap)
                    out[count] = n;
                count++;
            }
        free(seen);
        return count;
    }
    int limit = causal ? sk - T + t + 1 : sk;
    if (limit > sk)
        limit = sk;
    for (int n = 0; n < limit; n++) {
        if (count < cap)
            out[count] = n;
        count++;
    }
    return count;
}

/* Attention of one query row q[576] (double) over an explicit key list.
 * out[512], *lse.  Returns 0, or -1 on a bad page. */
int oracle_attend_keys(const double *q, const oracle_cache *c, int b,
                       const int32_t *keys, int n_keys, double scale,
                       double *out, double *lse)
{
    for (int j = 0; j < ORACLE_D_V; j++)
        out[j] = 0.0;
    if (n_keys == 0) {
        *lse = -INFINITY;
        return 0;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)n_keys);
    double row[ORACLE_D_QK];
    double m = -INFINITY;
    for (int i = 0; i < n_keys; i++) {
        if (load_key_row(c, b, keys[i], row) != 0) {
            free(s);
            return -1;
        }
        double dot = 0.0;
        for (int d = 0; d < ORACLE_D_QK; d++)
            dot += q[d] * row[d];
        s[i] = scale * dot;
        if (s[i] > m)
            m = s[i];
    }
    double sum = 0.0;
    for (int i = 0; i < n_keys; i++)
        sum += exp(s[i] - m);
    double L = m + log(sum);
    for (int i = 0; i < n_keys; i++) {
        load_key_row(c, b, keys[i], row);
        double p = exp(s[i] - L);
        for (int j = 0; j < ORACLE_D_V; j++)
            out[j] += p * row[j];
    }
    *lse = L;
    free(s);
    return 0;
}

/*
 * Decode for a list of query rows.
 *   q            bf16 bits [B][T][H][576]
 *   rows         n_rows triples (b, t, h)
 *   out          [n_rows][512] doubles, lse [n_rows] doubles
 * Returns 0, -1 on a bad argument or page index, or -2 when a row's top-k
 * list repeats a position.
 */
int oracle_mla_decode_rows(const uint16_t *q, int B, int T, int H,
                           const void *kv, int kv_format, int num_pages,
                           int page_size, const float *kv_scales,
                           const int32_t *block_table, int max_pages,
                           const int32_t *cache_seqlens,
                           const int32_t *topk, int topk_len,
                           double softmax_scale, int causal,
                           const int32_t *rows, int n_rows,
                           double *out, double *lse)
{
    oracle_cache c = {kv, kv_format, num_pages, page_size, kv_scales,
                      block_table, max_pages};
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int r = 0; r < n_rows; r++) {
        int b = rows[3 * r], t = rows[3 * r + 1], h = rows[3 * r + 2];
        if (b < 0 || b >= B || t < 0 || t >= T || h < 0 || h >= H) {
            bad |= 1;
            continue;
        }
        int sk = cache_seqlens[b];
        int cap = topk_len > sk ? topk_len : sk;
        int32_t *keys = (int32_t *)malloc(sizeof(int32_t) * (size_t)(cap > 0 ? cap : 1));
        int nk = oracle_valid_keys(b, t, T, cache_seqlens, topk, topk_len,
                                   causal, keys, cap);
        if (nk < 0) {
            bad |= 2;
            free(keys);
            continue;
        }
        double qd[ORACLE_D_QK];
        const uint16_t *qr = q + (((int64_t)b * T + t) * H + h) * ORACLE_D_QK;
        for (int d = 0; d < ORACLE_D_QK; d++)
            qd[d] = oracle_bf16_to_f64(qr[d]);
        if (oracle_attend_keys(qd, &c, b, keys, nk, softmax_scale,
                               out + (int64_t)r * ORACLE_D_V, lse + r) != 0)
            bad |= 1;
        free(keys);
    }
    return (bad & 2) ? -2 : (bad ? -1 : 0);
}

/* Same, with an explicit key list instead of the mask rule (used to check
 * that splitting the key set and merging by LSE gives the unsplit result). */
int oracle_attend_key_list(const uint16_t *q_row,
                           const void *kv, int kv_format, int num_pages,
                           int page_size, const float *kv_scales,
                           const int32_t *block_table, int max_pages, int b,
                           const int32_t *keys, int n_keys,
                           double softmax_scale, double *out, double *lse)
{
    oracle_cache c = {kv, kv_format, num_pages, page_size, kv_scales,
                      block_table, max_pages};
    double qd[ORACLE_D_QK];
    for (int d = 0; d < ORACLE_D_QK; d++)
        qd[d] = oracle_bf16_to_f64(q_row[d]);
    return oracle_attend_keys(qd, &c, b, keys, n_keys, softmax_scale, out, lse);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
