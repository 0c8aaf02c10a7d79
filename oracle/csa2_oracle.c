/*
 * csa2_oracle.c -- float64 CPU oracle for the CSA2 global-attention step.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library.  It shares no code, header, table or
 * constant with the CUDA library; the two only see the same seeded inputs.
 *
 * Every function is written from its definition, in plain loops, with no
 * blocking or reordering beyond what the definition states.  Sources:
 *   [Notes]     "DeepSeek-V4.1-Flash KV-Cache Compression" reading notes
 *               (jianyuh.github.io), sections 1-5.
 *   [Summary]   picx.dev summary of the technical report, "Methodology".
 *   [Deep read] "DeepSeek-V4.1-Flash: reading a model through its three memory
 *               costs", section 03 (CSA2 mode table).
 *   [Thread]    threadnavigator notes thread, items 4-6.
 *
 * Readings of points the pages leave open (same reading as the CUDA path):
 *   - indexer score s_j = sum_h w_h * ReLU(q_h . k_j), one key per entry shared
 *     by all indexer heads (DSA lineage named in [Notes] section 2);
 *   - FP8 = E4M3 (bias 7, max 448, no inf), round to nearest even, power-of-two
 *     scale per vector = smallest 2^e with 448 * 2^e >= amax (1 when amax = 0);
 *     a zero result is always the byte 0x00;
 *   - FP4 scale = smallest E4M3 value s with 6 s >= amax, codes by round to
 *     nearest even on the E2M1 grid, magnitude 0 always the code 0x0, amax over
 *     6 * 448 saturates to scale 448 and codes +-6;
 *   - top-k ties go to the lower position; the result is listed by ascending
 *     position;
 *   - attention uses the dequantised latent as both key and value, logits
 *     sm_scale * q . v, fp64 softmax, no sink.
 *
 * Parity pins (what checks this file against something other than itself)
 * live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_D 512          /* latent width [Notes] section 4: "512-channel KV latent" */
#define OR_GROUP 16       /* channels per E4M3 scale [Notes] section 4 */
#define OR_NGROUP (OR_D / OR_GROUP)

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

/* E2M1: sign bit, 2 exponent bits (bias 1), 1 mantissa bit; exponent 0 is
 * subnormal.  [Notes] section 4 (main-KV elements are E2M1). */
double or_e2m1_value(int nib)
{
    int s = (nib >> 3) & 1, e = (nib >> 1) & 3, mt = nib & 1;
    double mag = (e == 0) ? 0.5 * mt : ldexp(1.0 + 0.5 * mt, e - 1);
    return s ? -mag : mag;
}

/* E4M3 (OCP "FN" variant): sign, 4 exponent bits (bias 7), 3 mantissa bits,
 * exponent 0 subnormal, S.1111.111 is NaN, no infinities, max 448.
 * [Notes] section 4: range "448 x 6 = 2688". */
double or_e4m3_value(int b)
{
    int s = (b >> 7) & 1, e = (b >> 3) & 15, mt = b & 7;
    if (e == 15 && mt == 7) return NAN;
    double mag = (e == 0) ? ldexp(mt / 8.0, -6) : ldexp(1.0 + mt / 8.0, e - 7);
    return s ? -mag : mag;
}

/* bf16 bit pattern -> value (exact). */
double or_bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* Nearest E4M3 byte to y, ties to the even byte, |y| >= 448 saturates to 448,
 * a zero result is 0x00.  Positive bytes 0x00..0x7E increase with value, so
 * the largest byte not above |y| is found by bisection and compared with its
 * upper neighbour. */
int or_e4m3_nearest(double y)
{
    double a = fabs(y);
    int c;
    if (a >= 448.0) {
        c = 0x7E;
    } else {
        int lo = 0, hi = 0x7E;                  /* value(lo) <= a < value(hi) */
        while (hi - lo > 1) {
            int mid = (lo + hi) / 2;
            if (or_e4m3_value(mid) <= a) lo = mid; else hi = mid;
        }
        double dlo = a - or_e4m3_value(lo), dhi = or_e4m3_value(hi) - a;
        if (dlo < dhi) c = lo;
        else if (dhi < dlo) c = hi;
        else c = (lo % 2 == 0) ? lo : hi;       /* tie: even mantissa */
    }
    if (c == 0) return 0;
    return (y < 0) ? (c | 0x80) : c;
}

/* ------------------------------------------------------------------------ */
/* FP8 indexer vectors                                                       */
/* ------------------------------------------------------------------------ */

/* Power-of-two scale for one vector: smallest 2^e with 448 * 2^e >= amax. */
double or_fp8_pow2_scale(double amax)
{
    if (amax == 0.0) return 1.0;
    int e = ilogb(amax) - 10;           /* 448 * 2^e < amax here */
    while (ldexp(448.0, e) < amax) ++e;
    return ldexp(1.0, e);
}

/* Encode one vector of d values: bytes out[d], returns the scale. */
double or_fp8_encode_vec(const double *x, int d, uint8_t *out)
{
    double amax = 0.0;
    for (int c = 0; c < d; ++c) amax = fmax(amax, fabs(x[c]));
    double s = or_fp8_pow2_scale(amax);
    for (int c = 0; c < d; ++c) out[c] = (uint8_t)or_e4m3_nearest(x[c] / s);
    return s;
}

/* Batch form over fp32 input rows, for the tests. */
void or_fp8_encode_rows(const float *x, int64_t rows, int d, uint8_t *out, float *scale)
{
#pragma omp parallel
    {
        double *tmp = (double *)malloc(sizeof(double) * d);
#pragma omp for schedule(static)
        for (int64_t r = 0; r < rows; ++r) {
            for (int c = 0; c < d; ++c) tmp[c] = x[r * d + c];
            scale[r] = (float)or_fp8_encode_vec(tmp, d, out + r * d);
        }
        free(tmp);
    }
}

/* ------------------------------------------------------------------------ */
/* FP4 main-KV entries: E2M1 codes, one E4M3 scale per 16 channels           */
/* [Notes] section 4, [Summary] Methodology item 5, [Thread] item 6.          */
/* ------------------------------------------------------------------------ */

/* Scale byte for a 16-channel group: smallest positive E4M3 s with 6 s >= amax.
 * amax = 0 gives the byte 0x00; amax above 6 * 448 gives 0x7E and *sat = 1. */
int or_fp4_scale_byte(double amax, int *sat)
{
    if (amax == 0.0) return 0;
    for (int b = 1; b <= 0x7E; ++b)
        if (6.0 * or_e4m3_value(b) >= amax) return b;
    *sat = 1;
    return 0x7E;
}

/* E2M1 code of x under scale s: the magnitude index 0..7 whose value v * s is
 * nearest to |x|, ties to the even index; sign from x unless the index is 0. */
int or_fp4_code(double x, double s)
{
    double ax = fabs(x);
    int best = 0;
    double bd = ax;
    for (int i = 1; i < 8; ++i) {
        double d = fabs(ax - or_e2m1_value(i) * s);
        if (d < bd || (d == bd && i % 2 == 0)) { best = i; bd = d; }
    }
    if (best == 0) return 0;
    return (x < 0) ? (8 | best) : best;
}

/* Encode one 512-channel entry.  codes[256]: channel 2i in the low nibble of
 * byte i; scales[32]: byte g covers channels 16g..16g+15.  Returns the number
 * of saturated groups. */
int or_fp4_encode_entry(const double *x, uint8_t *codes, uint8_t *scales)
{
    int nsat = 0;
    int nib[OR_D];
    for (int g = 0; g < OR_NGROUP; ++g) {
        double amax = 0.0;
        for (int c = 0; c < OR_GROUP; ++c) amax = fmax(amax, fabs(x[g * OR_GROUP + c]));
        int sat = 0;
        int sb = or_fp4_scale_byte(amax, &sat);
        nsat += sat;
        scales[g] = (uint8_t)sb;
        double s = or_e4m3_value(sb);
        for (int c = 0; c < OR_GROUP; ++c)
            nib[g * OR_GROUP + c] = (sb == 0) ? 0 : or_fp4_code(x[g * OR_GROUP + c], s);
    }
    for (int i = 0; i < OR_D / 2; ++i)
        codes[i] = (uint8_t)(nib[2 * i] | (nib[2 * i + 1] << 4));
    return nsat;
}

/* Dequantise one entry: value = e2m1(code) * e4m3(scale). */
void or_fp4_decode_entry(const uint8_t *codes, const uint8_t *scales, double *out)
{
    for (int c = 0; c < OR_D; ++c) {
        int nib = (codes[c / 2] >> (4 * (c % 2))) & 15;
        out[c] = or_e2m1_value(nib) * or_e4m3_value(scales[c / OR_GROUP]);
    }
}

/* ------------------------------------------------------------------------ */
/* Sequence-block compression by m, weighted by softmax(Z) per channel       */
/* [Notes] section 1 (C_l, Z_l projected from H_{L/2}) and section 2 (block   */
/* compression by m; no overlapping blocks, no absolute positions).           */
/* ------------------------------------------------------------------------ */

/* C, Z: m rows of 512 fp32 values (one block of m tokens). out: 512 values. */
void or_compress_block(const float *C, const float *Z, int m, double *out)
{
    for (int c = 0; c < OR_D; ++c) {
        if (m == 1) { out[c] = C[c]; continue; }
        double zmax = -INFINITY;
        for (int i = 0; i < m; ++i) zmax = fmax(zmax, (double)Z[i * OR_D + c]);
        double den = 0.0, num = 0.0;
        for (int i = 0; i < m; ++i) {
            double e = exp((double)Z[i * OR_D + c] - zmax);
            den += e;
            num += e * (double)C[i * OR_D + c];
        }
        out[c] = num / den;
    }
}

/* Append for a batch: B sequences, n_tok tokens each (n_tok a multiple of m).
 * C, Z: [B][n_tok][512] (Z unused when m == 1); key: [B][n_tok/m][d_idx].
 * Entry e of sequence b goes to output row b * (n_tok/m) + e.
 * Also returns the compressed fp64 latent in xout (nullable) for the tests. */
int64_t or_append(int B, int n_tok, int m, int d_idx, const float *C, const float *Z,
                  const float *key, uint8_t *codes, uint8_t *scales, uint8_t *kidx,
                  float *kscale, double *xout)
{
    int ne = n_tok / m;
    int64_t nsat = 0;
#pragma omp parallel for reduction(+ : nsat) schedule(static)
    for (int64_t r = 0; r < (int64_t)B * ne; ++r) {
        int64_t b = r / ne, e = r % ne;
        double x[OR_D];
        const float *cb = C + (b * n_tok + e * m) * OR_D;
        const float *zb = (m > 1) ? Z + (b * n_tok + e * m) * OR_D : NULL;
        or_compress_block(cb, zb, m, x);
        if (xout) memcpy(xout + r * OR_D, x, sizeof(x));
        nsat += or_fp4_encode_entry(x, codes + r * (OR_D / 2), scales + r * OR_NGROUP);
        double kv[1024];
        for (int c = 0; c < d_idx; ++c) kv[c] = key[r * d_idx + c];
        kscale[r] = (float)or_fp8_encode_vec(kv, d_idx, kidx + r * d_idx);
    }
    return nsat;
}

/* Append with the indexer key projected from the stored entry: the key of an
 * entry is the dequantised FP4 latent times W_IK ([Notes] section 1: the
 * indexer key is a linear projection of the main KV; this library's reading:
 * of the dequantised FP4 entry, so that the key can be rebuilt from the
 * persisted cache alone), then FP8-encoded like a caller-given key.
 * w_ik: bf16 bit patterns [512][d_idx], row c = latent channel c.  Other
 * arguments and outputs as in or_append (no key input). */
int64_t or_append_project(int B, int n_tok, int m, int d_idx, const float *C, const float *Z,
                          const uint16_t *w_ik, uint8_t *codes, uint8_t *scales, uint8_t *kidx,
                          float *kscale, double *kout)
{
    int ne = n_tok / m;
    int64_t nsat = 0;
#pragma omp parallel for reduction(+ : nsat) schedule(static)
    for (int64_t r = 0; r < (int64_t)B * ne; ++r) {
        int64_t b = r / ne, e = r % ne;
        double x[OR_D], v[OR_D], k[1024];
        const float *cb = C + (b * n_tok + e * m) * OR_D;
        const float *zb = (m > 1) ? Z + (b * n_tok + e * m) * OR_D : NULL;
        or_compress_block(cb, zb, m, x);
        uint8_t *cr = codes + r * (OR_D / 2), *sr = scales + r * OR_NGROUP;
        nsat += or_fp4_encode_entry(x, cr, sr);
        or_fp4_decode_entry(cr, sr, v);
        for (int d = 0; d < d_idx; ++d) {
            double acc = 0.0;
            for (int c = 0; c < OR_D; ++c) acc += v[c] * or_bf16_value(w_ik[c * d_idx + d]);
            k[d] = acc;
        }
        if (kout) memcpy(kout + r * d_idx, k, sizeof(double) * d_idx);
        kscale[r] = (float)or_fp8_encode_vec(k, d_idx, kidx + r * d_idx);
    }
    return nsat;
}

/* ------------------------------------------------------------------------ */
/* Indexer scores  [Notes] sections 2-3, [Deep read] section 03               */
/* ------------------------------------------------------------------------ */

/* Quantise one query's indexer heads: q [h_idx][d_idx] fp32 -> q8, sq. */
static void or_quant_query(const float *q, int h_idx, int d_idx, uint8_t *q8, double *sq)
{
    double v[1024];
    for (int h = 0; h < h_idx; ++h) {
        for (int c = 0; c < d_idx; ++c) v[c] = q[h * d_idx + c];
        sq[h] = or_fp8_encode_vec(v, d_idx, q8 + h * d_idx);
    }
}

/* score(q, j) = sum_h w_h * ReLU(q_h . k_j) on the dequantised FP8 vectors. */
static double or_score_one(const uint8_t *q8, const double *sq, const float *w, int h_idx,
                           int d_idx, const uint8_t *k8, double sk, const double *lut)
{
    double s = 0.0;
    for (int h = 0; h < h_idx; ++h) {
        double dot = 0.0;
        for (int c = 0; c < d_idx; ++c)
            dot += (sq[h] * lut[q8[h * d_idx + c]]) * (sk * lut[k8[c]]);
        s += (double)w[h] * (dot > 0.0 ? dot : 0.0);
    }
    return s;
}

static void or_e4m3_lut(double *lut)
{
    for (int b = 0; b < 256; ++b) lut[b] = or_e4m3_value(b);
}

/* Scores of one query at n cache rows rows[0..n) (absolute row numbers).
 * kidx: [*][d_idx], kscale: [*]; q: [h_idx][d_idx]; w: [h_idx]. */
void or_scores_at(const uint8_t *kidx, const float *kscale, int d_idx, int h_idx,
                  const float *q, const float *w, const int64_t *rows, int64_t n,
                  double *out)
{
    double lut[256], sq[64];
    uint8_t q8[64 * 1024];
    or_e4m3_lut(lut);
    or_quant_query(q, h_idx, d_idx, q8, sq);
    for (int64_t i = 0; i < n; ++i)
        out[i] = or_score_one(q8, sq, w, h_idx, d_idx, kidx + rows[i] * d_idx,
                              (double)kscale[rows[i]], lut);
}

/* Full mode: scores of one query over the n contiguous rows base..base+n-1. */
void or_scores_full(const uint8_t *kidx, const float *kscale, int d_idx, int h_idx,
                    const float *q, const float *w, int64_t base, int64_t n, double *out)
{
    double lut[256], sq[64];
    uint8_t q8[64 * 1024];
    or_e4m3_lut(lut);
    or_quant_query(q, h_idx, d_idx, q8, sq);
    for (int64_t j = 0; j < n; ++j)
        out[j] = or_score_one(q8, sq, w, h_idx, d_idx, kidx + (base + j) * d_idx,
                              (double)kscale[base + j], lut);
}

/* ------------------------------------------------------------------------ */
/* Top-k  (ties to the lower position, output by ascending position)         */
/* ------------------------------------------------------------------------ */

typedef struct { double s; int64_t p; } or_sp;

static int or_cmp_score_desc(const void *a, const void *b)
{
    const or_sp *x = (const or_sp *)a, *y = (const or_sp *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->p < y->p) ? -1 : (x->p > y->p);
}

static int or_cmp_i32(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x < y) ? -1 : (x > y);
}

/* scores[0..n); pos[i] is candidate i's position (NULL: pos = i).  Writes the
 * min(k, n) positions with the largest scores, ascending; returns the count. */
int or_topk(const double *scores, const int32_t *pos, int64_t n, int k, int32_t *out)
{
    or_sp *v = (or_sp *)malloc(sizeof(or_sp) * (n > 0 ? n : 1));
    for (int64_t i = 0; i < n; ++i) {
        v[i].s = scores[i];
        v[i].p = pos ? pos[i] : i;
    }
    qsort(v, n, sizeof(or_sp), or_cmp_score_desc);
    int cnt = (n < k) ? (int)n : k;
    for (int i = 0; i < cnt; ++i) out[i] = (int32_t)v[i].p;
    qsort(out, cnt, sizeof(int32_t), or_cmp_i32);
    free(v);
    return cnt;
}

/* Same from fp32 scores (the bit-exact top-k check feeds identical arrays). */
int or_topk_f32(const float *scores, const int32_t *pos, int64_t n, int k, int32_t *out)
{
    double *d = (double *)malloc(sizeof(double) * (n > 0 ? n : 1));
    for (int64_t i = 0; i < n; ++i) d[i] = scores[i];
    int c = or_topk(d, pos, n, k, out);
    free(d);
    return c;
}

/* ------------------------------------------------------------------------ */
/* Hierarchical candidate pool  [Notes] section 3, [Summary] item 3           */
/* ------------------------------------------------------------------------ */

/* Block maxima: max score over the visible entries of each aligned 8-entry block. */
void or_blockmax(const double *scores, int64_t n, double *out)
{
    for (int64_t b = 0; b < (n + 7) / 8; ++b) {
        double m = -INFINITY;
        for (int64_t j = 8 * b; j < 8 * b + 8 && j < n; ++j) m = fmax(m, scores[j]);
        out[b] = m;
    }
}

/* Block score = max token score over the visible entries of each aligned
 * 8-entry block; the top nblk_max blocks (ties to the lower block) form the
 * pool.  blk_out gets the chosen block ids ascending; returns the number of
 * visible positions in the pool.  *nblk gets the number of blocks. */
int or_pool(const double *scores, int64_t n, int nblk_max, int32_t *blk_out, int *nblk)
{
    int64_t nb = (n + 7) / 8;
    double *bm = (double *)malloc(sizeof(double) * (nb > 0 ? nb : 1));
    or_blockmax(scores, n, bm);
    int c = or_topk(bm, NULL, nb, nblk_max, blk_out);
    free(bm);
    *nblk = c;
    int pool_n = 0;
    for (int i = 0; i < c; ++i) {
        int64_t lo = 8 * (int64_t)blk_out[i], hi = lo + 8 < n ? lo + 8 : n;
        pool_n += (int)(hi - lo);
    }
    return pool_n;
}

/* ------------------------------------------------------------------------ */
/* Sparse attention over selected main-KV entries + window KV                 */
/* [Thread] item 4: select main KV, concatenate with the windowed KV, then    */
/* attend; [Deep read] section 03: every mode computes its own main Q and SWA */
/* KV; [Notes] section 5: window [max(s, i - n_win + 1), i].                  */
/* ------------------------------------------------------------------------ */

/* Rows of the concatenated set for one query: the dequantised entries
 * seq_base + idx[0..cnt) followed by the window rows of positions
 * max(s, t - n_win + 1, 0)..t, held at win[(p mod wcap)].  win: [wcap][512]
 * bf16 of this query's sequence.  Returns the number of rows written. */
int or_gather_rows(const uint8_t *codes, const uint8_t *scales, int64_t seq_base,
                   const int32_t *idx, int cnt, const uint16_t *win, int wcap,
                   int64_t t, int64_t s, int n_win, double *rows)
{
    int r = 0;
    for (int i = 0; i < cnt; ++i, ++r) {
        int64_t row = seq_base + idx[i];
        or_fp4_decode_entry(codes + row * (OR_D / 2), scales + row * OR_NGROUP, rows + (int64_t)r * OR_D);
    }
    if (win && n_win > 0) {
        int64_t lo = t - n_win + 1;
        if (lo < s) lo = s;
        if (lo < 0) lo = 0;
        for (int64_t p = lo; p <= t; ++p, ++r)
            for (int c = 0; c < OR_D; ++c)
                rows[(int64_t)r * OR_D + c] = or_bf16_value(win[(p % wcap) * OR_D + c]);
    }
    return r;
}

/* Multi-head softmax attention of H query heads (bf16 [H][512]) over n rows
 * used as both keys and values.  out [H][512], lse [H] (natural log). */
void or_attention(int H, const uint16_t *q, int64_t n, const double *rows, double sm_scale,
                  double *out, double *lse)
{
    double *logit = (double *)malloc(sizeof(double) * (n > 0 ? n : 1));
    for (int h = 0; h < H; ++h) {
        double qd[OR_D];
        for (int c = 0; c < OR_D; ++c) qd[c] = or_bf16_value(q[h * OR_D + c]);
        double mx = -INFINITY;
        for (int64_t j = 0; j < n; ++j) {
            double d = 0.0;
            for (int c = 0; c < OR_D; ++c) d += qd[c] * rows[j * OR_D + c];
            logit[j] = sm_scale * d;
            mx = fmax(mx, logit[j]);
        }
        double l = 0.0;
        for (int c = 0; c < OR_D; ++c) out[h * OR_D + c] = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            double p = exp(logit[j] - mx);
            l += p;
            for (int c = 0; c < OR_D; ++c) out[h * OR_D + c] += p * rows[j * OR_D + c];
        }
        for (int c = 0; c < OR_D; ++c) out[h * OR_D + c] /= l;
        if (lse) lse[h] = mx + log(l);
    }
    free(logit);
}

/* ------------------------------------------------------------------------ */
/* One CSA2 layer for a batch of queries  [Notes] section 2 (modes),          */
/* [Deep read] section 03 (what each mode computes and reuses).               */
/* ------------------------------------------------------------------------ */

enum { OR_FULL = 0, OR_REINDEX = 1, OR_REUSE = 2 };

typedef struct {
    /* cache */
    const uint8_t *codes, *scales, *kidx;
    const float *kscale;
    const int64_t *seq_base;
    int d_idx, m;
    /* queries */
    int nq;
    const int32_t *q_seq, *q_pos;
    /* indexer (Full, Reindex) */
    int h_idx;
    const float *q_idx, *w;   /* [nq][h_idx][d_idx], [nq][h_idx] */
    int k;
    int pool_blocks;          /* blocks in the candidate pool (Full layer that builds it) */
    /* attention */
    int H;
    const uint16_t *q_attn;   /* [nq][H][512] bf16 */
    const uint16_t *win;      /* [B][wcap][512] bf16 */
    int wcap, n_win;
    const int32_t *win_start; /* [B], nullable */
    double sm_scale;
} or_layer_args;

/* mode FULL: scores all visible entries, top-k, optionally the pool.
 * mode REINDEX: scores the pool given in pool_blk/pool_n, top-k over it.
 * mode REUSE: takes idx_io/cnt_io as input.
 * idx_io [nq][k], cnt_io [nq]; pool_blk [nq][pool_blocks], pool_n [nq];
 * out [nq][H][512], lse [nq][H] (nullable). */
void or_layer(int mode, const or_layer_args *a, int32_t *idx_io, int32_t *cnt_io,
              int build_pool, int32_t *pool_blk, int32_t *pool_n, double *out, double *lse)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int qi = 0; qi < a->nq; ++qi) {
        int b = a->q_seq[qi];
        int64_t t = a->q_pos[qi];
        int64_t nt = (t + 1) / a->m;                 /* visible entries */
        int64_t base = a->seq_base[b];
        int32_t *idx = idx_io + (int64_t)qi * a->k;
        const float *qv = a->q_idx ? a->q_idx + (int64_t)qi * a->h_idx * a->d_idx : NULL;
        const float *wv = a->w ? a->w + (int64_t)qi * a->h_idx : NULL;
        if (mode == OR_FULL) {
            double *sc = (double *)malloc(sizeof(double) * (nt > 0 ? nt : 1));
            or_scores_full(a->kidx, a->kscale, a->d_idx, a->h_idx, qv, wv, base, nt, sc);
            cnt_io[qi] = or_topk(sc, NULL, nt, a->k, idx);
            if (build_pool) {
                int nb;
                pool_n[qi] = or_pool(sc, nt, a->pool_blocks,
                                     pool_blk + (int64_t)qi * a->pool_blocks, &nb);
            }
            free(sc);
        } else if (mode == OR_REINDEX) {
            const int32_t *pb = pool_blk + (int64_t)qi * a->pool_blocks;
            int pn = pool_n[qi];
            int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (pn > 0 ? pn : 1));
            int32_t *pos = (int32_t *)malloc(sizeof(int32_t) * (pn > 0 ? pn : 1));
            for (int i = 0; i < pn; ++i) {
                pos[i] = 8 * pb[i / 8] + i % 8;
                rows[i] = base + pos[i];
            }
            double *sc = (double *)malloc(sizeof(double) * (pn > 0 ? pn : 1));
            or_scores_at(a->kidx, a->kscale, a->d_idx, a->h_idx, qv, wv, rows, pn, sc);
            cnt_io[qi] = or_topk(sc, pos, pn, a->k, idx);
            free(sc);
            free(pos);
            free(rows);
        }
        int cnt = cnt_io[qi];
        int64_t s = a->win_start ? a->win_start[b] : 0;
        double *rows = (double *)malloc(sizeof(double) * OR_D * (size_t)(cnt + a->n_win + 1));
        int n = or_gather_rows(a->codes, a->scales, base, idx, cnt,
                               a->win ? a->win + (int64_t)b * a->wcap * OR_D : NULL, a->wcap,
                               t, s, a->n_win, rows);
        or_attention(a->H, a->q_attn + (int64_t)qi * a->H * OR_D, n, rows, a->sm_scale,
                     out + (int64_t)qi * a->H * OR_D, lse ? lse + (int64_t)qi * a->H : NULL);
        free(rows);
    }
}

int or_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void or_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
