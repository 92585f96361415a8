/*
 * Oracle for the fused grouped-query scaled-dot-product attention forward.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously correct CPU
 * definition that the CUDA path is checked against. Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it. It shares
 * no code, header, table or constant with the CUDA library and includes none
 * of its files.
 *
 * What it computes (plain definition, fp64 throughout). For batch b, query
 * head h and query row i:
 *
 *   g        = h / (Hq / Hkv)            grouped-query head mapping: each KV head
 *                                        serves Hq/Hkv consecutive query heads
 *                                        ("xe2-sdp-hd256" page, header: 32 Q heads
 *                                        over 2 KV heads; "SyclKittens" summary,
 *                                        section E.1: the grouped baseline repeats
 *                                        each KV head)
 *   s_j      = scale * sum_d Q[b,h,i,d] * K[b,g,j,d]          for 0 <= j < Skv
 *   M        = max_j s_j
 *   L        = sum_j exp(s_j - M)
 *   O[b,h,i] = sum_j exp(s_j - M) * V[b,g,j,:] / L
 *   LSE      = M + ln L                  natural log, one value per (b,h,i)
 *
 * Causal variant (causal != 0): row i sees keys j <= i only (top-left
 * alignment, the convention of PyTorch's is_causal; the "SyclKittens" summary,
 * sections E.4 and E.6, measures causal attention without fixing one). The
 * maximum, sum and weighted sum then run over those keys; every row keeps
 * at least key 0.
 *
 * This is the result the single-pass online-softmax kernel of the
 * "xe2-sdp-hd256" page (section "HD=256 Architecture Differences") and the
 * "xe2-sdp-bf16" page (section "Data flow diagram") reaches up to rounding
 * order. The oracle does not block, fuse or reorder: it forms each score
 * row in full, then its maximum, then the exponentials, then the weighted
 * sum of V rows.
 *
 * Inputs are the exact 16-bit patterns the GPU receives (fp16 or bf16),
 * decoded here to double ("xe2-sdp-bf16" page, section "CPU reference must
 * match input type": the reference consumes the type-quantised values).
 *
 * Layout: Q [B, Hq, Sq, D], K and V [B, Hkv, Skv, D], all contiguous
 * row-major 16-bit patterns. Outputs are double and unrounded.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_FP16 0
#define ORACLE_BF16 1

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_fp16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double x;
    if (e == 0)
        x = ldexp((double)m, -24); /* subnormal: m * 2^-14 * 2^-10 */
    else if (e == 31)
        x = m ? NAN : INFINITY;
    else
        x = ldexp((double)(m | 0x400), e - 25); /* (1024 + m) * 2^(e-15-10) */
    return sign ? -x : x;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_double(uint16_t b)
{
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int m = b & 0x7f;
    double x;
    if (e == 0)
        x = ldexp((double)m, -133); /* subnormal: m * 2^-126 * 2^-7 */
    else if (e == 255)
        x = m ? NAN : INFINITY;
    else
        x = ldexp((double)(m | 0x80), e - 134); /* (128 + m) * 2^(e-127-7) */
    return sign ? -x : x;
}

static double decode(uint16_t bits, int dtype)
{
    return dtype == ORACLE_BF16 ? oracle_bf16_to_double(bits) : oracle_fp16_to_double(bits);
}

/*
 * One query row against one KV head, straight from the definition above.
 * p receives the Skv softmax weights exp(s_j - M) / L.
 */
static void attend_row(const double *q, const double *Kg, const double *Vg, int Skv, int D,
                       double scale, double *s, double *p, double *o, double *lse)
{
    /* Skv here is the number of keys this row sees (all keys, or i+1 when causal) */
    /* scores */
    for (int j = 0; j < Skv; ++j) {
        double acc = 0.0;
        const double *kj = Kg + (size_t)j * D;
        for (int d = 0; d < D; ++d)
            acc += q[d] * kj[d];
        s[j] = scale * acc;
    }
    /* row maximum */
    double M = -INFINITY;
    for (int j = 0; j < Skv; ++j)
        if (s[j] > M)
            M = s[j];
    /* exponentials and their sum */
    double L = 0.0;
    for (int j = 0; j < Skv; ++j) {
        p[j] = exp(s[j] - M);
        L += p[j];
    }
    /* weighted sum of value rows, then normalise */
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    for (int j = 0; j < Skv; ++j) {
        const double *vj = Vg + (size_t)j * D;
        for (int d = 0; d < D; ++d)
            o[d] += p[j] * vj[d];
    }
    for (int d = 0; d < D; ++d)
        o[d] /= L;
    for (int j = 0; j < Skv; ++j)
        p[j] /= L;
    *lse = M + log(L);
}

static int check_shape(int B, int Hq, int Hkv, int Sq, int Skv, int D, int dtype)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || D <= 0)
        return -1;
    if (Hq % Hkv != 0)
        return -1;
    if (dtype != ORACLE_FP16 && dtype != ORACLE_BF16)
        return -1;
    return 0;
}

/*
 * Attention forward on a chosen set of query rows.
 *
 * rows:   int32 [B*Hq*nrows], the query-row indices evaluated for each (b, h),
 *         in (b, h) order; every index must lie in [0, Sq).
 * o_out:  double [B*Hq*nrows*D], O for those rows in the same order.
 * lse_out: double [B*Hq*nrows] (may be NULL).
 * causal: 0 for full attention, nonzero for row i seeing keys 0..i.
 * Returns 0, or -1 on a bad shape or row index.
 */
int oracle_sdp_fwd_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, int dtype,
                        int B, int Hq, int Hkv, int Sq, int Skv, int D, double scale, int causal,
                        const int32_t *rows, int nrows, double *o_out, double *lse_out)
{
    if (check_shape(B, Hq, Hkv, Sq, Skv, D, dtype) || nrows < 0)
        return -1;
    for (long t = 0; t < (long)B * Hq * nrows; ++t)
        if (rows[t] < 0 || rows[t] >= Sq)
            return -1;
    const int G = Hq / Hkv;
    double *Kg = (double *)malloc(sizeof(double) * (size_t)Skv * D);
    double *Vg = (double *)malloc(sizeof(double) * (size_t)Skv * D);
    if (!Kg || !Vg) {
        free(Kg);
        free(Vg);
        return -1;
    }
    int status = 0;
    for (int b = 0; b < B && !status; ++b) {
        for (int g = 0; g < Hkv && !status; ++g) {
            const size_t kv_off = ((size_t)b * Hkv + g) * (size_t)Skv * D;
            const long nkv = (long)Skv * D;
#pragma omp parallel for schedule(static)
            for (long t = 0; t < nkv; ++t) {
                Kg[t] = decode(k[kv_off + t], dtype);
                Vg[t] = decode(v[kv_off + t], dtype);
            }
            /* every (query head of this group, sampled row) pair */
            const long npairs = (long)G * nrows;
#pragma omp parallel
            {
                double *qrow = (double *)malloc(sizeof(double) * D);
                double *s = (double *)malloc(sizeof(double) * Skv);
                double *p = (double *)malloc(sizeof(double) * Skv);
                int ok = qrow && s && p;
                if (!ok) {
#pragma omp atomic write
                    status = -1;
                }
#pragma omp for schedule(dynamic, 1)
                for (long t = 0; t < npairs; ++t) {
                    if (!ok)
                        continue;
                    const int h = g * G + (int)(t / nrows);
                    const long slot = ((long)b * Hq + h) * nrows + (t % nrows);
                    const int i = rows[slot];
                    const size_t q_off = (((size_t)b * Hq + h) * (size_t)Sq + i) * D;
                    for (int d = 0; d < D; ++d)
                        qrow[d] = decode(q[q_off + d], dtype);
                    double lse;
                    const int seen = (causal && i + 1 < Skv) ? i + 1 : Skv;
                    attend_row(qrow, Kg, Vg, seen, D, scale, s, p, o_out + (size_t)slot * D, &lse);
                    if (lse_out)
                        lse_out[slot] = lse;
                }
                free(qrow);
                free(s);
                free(p);
            }
        }
    }
    free(Kg);
    free(Vg);
    return status;
}

/*
 * The softmax weights of one query row (b, h, i): p_out double [Skv] (keys a
 * causal row does not see get weight 0).
 * Exposed so that properties of the weights themselves can be checked.
 */
int oracle_sdp_row_probs(const uint16_t *q, const uint16_t *k, const uint16_t *v, int dtype,
                         int B, int Hq, int Hkv, int Sq, int Skv, int D, double scale, int causal,
                         int b, int h, int i, double *p_out, double *o_out, double *lse_out)
{
    if (check_shape(B, Hq, Hkv, Sq, Skv, D, dtype))
        return -1;
    if (b < 0 || b >= B || h < 0 || h >= Hq || i < 0 || i >= Sq)
        return -1;
    const int g = h / (Hq / Hkv);
    const size_t kv_off = ((size_t)b * Hkv + g) * (size_t)Skv * D;
    const size_t q_off = (((size_t)b * Hq + h) * (size_t)Sq + i) * D;
    double *Kg = (double *)malloc(sizeof(double) * (size_t)Skv * D);
    double *Vg = (double *)malloc(sizeof(double) * (size_t)Skv * D);
    double *qrow = (double *)malloc(sizeof(double) * D);
    double *s = (double *)malloc(sizeof(double) * Skv);
    int status = -1;
    if (Kg && Vg && qrow && s) {
        for (size_t t = 0; t < (size_t)Skv * D; ++t) {
            Kg[t] = decode(k[kv_off + t], dtype);
            Vg[t] = decode(v[kv_off + t], dtype);
        }
        for (int d = 0; d < D; ++d)
            qrow[d] = decode(q[q_off + d], dtype);
        const int seen = (causal && i + 1 < Skv) ? i + 1 : Skv;
        for (int j = seen; j < Skv; ++j)
            p_out[j] = 0.0;
        attend_row(qrow, Kg, Vg, seen, D, scale, s, p_out, o_out, lse_out);
        status = 0;
    }
    free(Kg);
    free(Vg);
    free(qrow);
    free(s);
    return status;
}

/*
 * Variable-length batch: sequences of different lengths packed back to back
 * (no counterpart on the pages; the plain generalisation of the ragged last
 * tile of one sequence to a batch of ragged sequences). Sequence b owns query
 * rows [cu_q[b], cu_q[b+1]) and key rows [cu_k[b], cu_k[b+1]); each of its
 * query rows attends to that sequence's keys only, by the definition at the
 * top of this file with Sq = len_q(b) and Skv = len_k(b) (causal: row i of the
 * sequence sees the sequence's keys 0..i). A row that sees no key (a
 * sequence with no keys) has O = 0 and LSE = -inf.
 *
 * Layout (token, head, dim), contiguous 16-bit patterns:
 *   Q [total_q, Hq, D], K and V [total_k, Hkv, D];
 *   o_out double [total_q, Hq, D]; lse_out double [Hq, total_q] (may be NULL).
 * cu_q, cu_k: int32 [nseq + 1], cu[0] = 0, non-decreasing, cu[nseq] = total.
 * Returns 0, or -1 on bad sizes or offsets.
 */
int oracle_sdp_fwd_varlen(const uint16_t *q, const uint16_t *k, const uint16_t *v, int dtype, int nseq,
                          int Hq, int Hkv, int D, double scale, int causal, const int32_t *cu_q,
                          const int32_t *cu_k, long total_q, long total_k, double *o_out, double *lse_out)
{
    if (nseq <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0 || total_q < 0 || total_k < 0)
        return -1;
    if (dtype != ORACLE_FP16 && dtype != ORACLE_BF16)
        return -1;
    if (cu_q[0] != 0 || cu_k[0] != 0 || cu_q[nseq] != total_q || cu_k[nseq] != total_k)
        return -1;
    int max_k = 0;
    for (int b = 0; b < nseq; ++b) {
        if (cu_q[b + 1] < cu_q[b] || cu_k[b + 1] < cu_k[b])
            return -1;
        if (cu_k[b + 1] - cu_k[b] > max_k)
            max_k = cu_k[b + 1] - cu_k[b];
    }
    const int G = Hq / Hkv;
    const size_t kv_elems = (size_t)(max_k > 0 ? max_k : 1) * D;
    double *Kg = (double *)malloc(sizeof(double) * kv_elems);
    double *Vg = (double *)malloc(sizeof(double) * kv_elems);
    if (!Kg || !Vg) {
        free(Kg);
        free(Vg);
        return -1;
    }
    int status = 0;
    for (int b = 0; b < nseq && !status; ++b) {
        const int row_q = cu_q[b], len_q = cu_q[b + 1] - cu_q[b];
        const int row_k = cu_k[b], len_k = cu_k[b + 1] - cu_k[b];
        for (int g = 0; g < Hkv && !status; ++g) {
            /* this sequence's keys and values of KV head g, row j at Kg + j*D */
#pragma omp parallel for schedule(static)
            for (long t = 0; t < (long)len_k * D; ++t) {
                const size_t src = ((size_t)(row_k + t / D) * Hkv + g) * D + t % D;
                Kg[t] = decode(k[src], dtype);
                Vg[t] = decode(v[src], dtype);
            }
            const long npairs = (long)G * len_q;
#pragma omp parallel
            {
                double *qrow = (double *)malloc(sizeof(double) * D);
                double *s = (double *)malloc(sizeof(double) * (len_k > 0 ? len_k : 1));
                double *p = (double *)malloc(sizeof(double) * (len_k > 0 ? len_k : 1));
                int ok = qrow && s && p;
                if (!ok) {
#pragma omp atomic write
                    status = -1;
                }
#pragma omp for schedule(dynamic, 4)
                for (long t = 0; t < npairs; ++t) {
                    if (!ok)
                        continue;
                    const int h = g * G + (int)(t / len_q);
                    const int i = (int)(t % len_q);
                    const size_t at = ((size_t)(row_q + i) * Hq + h) * D;
                    double *o = o_out + at;
                    const int seen = (causal && i + 1 < len_k) ? i + 1 : len_k;
                    double lse;
                    if (seen == 0) {
                        for (int d = 0; d < D; ++d)
                            o[d] = 0.0;
                        lse = -INFINITY;
                    } else {
                        for (int d = 0; d < D; ++d)
                            qrow[d] = decode(q[at + d], dtype);
                        attend_row(qrow, Kg, Vg, seen, D, scale, s, p, o, &lse);
                    }
                    if (lse_out)
                        lse_out[(size_t)h * total_q + row_q + i] = lse;
                }
                free(qrow);
                free(s);
                free(p);
            }
        }
    }
    free(Kg);
    free(Vg);
    return status;
}

/*
 * Merge of partial attention results over disjoint key sets — the state
 * exchange of ring / context-parallel attention ("SyclKittens" summary,
 * section I.2: each step merges the online-softmax state of the next key
 * shard). For each row r, with parts p = 0..P-1 each holding a normalised
 * output O_p[r,:] over its keys and the log-sum-exp LSE_p[r] of its scores:
 *
 *   LSE[r] = ln sum_p exp(LSE_p[r])          (taken relative to M = max_p LSE_p)
 *   O[r,:] = sum_p exp(LSE_p[r] - LSE[r]) * O_p[r,:]
 *
 * which is attention over the union of the parts' keys. A part with
 * LSE_p = -inf (no keys) gets weight 0; at least one part must be finite.
 * o_parts double [P, rows, D], lse_parts double [P, rows]; o_out double
 * [rows, D], lse_out double [rows]. Returns 0, or -1 on bad sizes.
 */
int oracle_sdp_merge(const double *o_parts, const double *lse_parts, int P, long rows, int D,
                     double *o_out, double *lse_out)
{
    if (P <= 0 || rows < 0 || D <= 0)
        return -1;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int p = 0; p < P; ++p)
            if (lse_parts[(size_t)p * rows + r] > M)
                M = lse_parts[(size_t)p * rows + r];
        double sum = 0.0;
        for (int p = 0; p < P; ++p)
            sum += exp(lse_parts[(size_t)p * rows + r] - M);
        const double lse = M + log(sum);
        for (int d = 0; d < D; ++d)
            o_out[(size_t)r * D + d] = 0.0;
        for (int p = 0; p < P; ++p) {
            const double w = exp(lse_parts[(size_t)p * rows + r] - lse);
            const double *op = o_parts + ((size_t)p * rows + r) * D;
            for (int d = 0; d < D; ++d)
                o_out[(size_t)r * D + d] += w * op[d];
        }
        lse_out[r] = lse;
    }
    return 0;
}

/* Threads an OpenMP parallel region of the oracle uses (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
