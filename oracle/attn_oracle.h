/*
 * attn_oracle.h -- fp64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this library: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg use it. It shares no code, header, table or helper with the
 * CUDA library.
 *
 * Sources (page title, then section):
 *   [Streaming] "FlashAttention: Exact Attention as an IO-Aware Streaming Computation"
 *   [Lesson]    "IO-aware exact attention"
 *   [Glossary]  "FlashAttention" (glossary entry)
 *
 * Layouts (all contiguous, row-major, last index fastest):
 *   q    [B][H][Nq][d]      k, v [B][H][Nk][d]
 *   mask [B][Nq][Nk] or NULL (additive, shared by every head; finite or -inf)
 *   out  [B][H][Nq][d]      lse  [B][H][Nq] (natural log)
 * causal != 0 allows key j for query i iff j <= i + (Nk - Nq); with Nq == Nk this
 * is "at or before each query position" ([Lesson], "Tile order and on-chip capacity").
 * A row whose every score is -inf gets out = 0 and lse = -inf.
 */
#ifndef ATTN_ORACLE_H
#define ATTN_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Materialised definition, every row. Returns 0, or -1 on a bad argument. */
int oracle_attn_f64(const double *q, const double *k, const double *v, const double *mask,
                    double *out, double *lse, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                    int64_t d, double scale, int causal);

/* Same definition for a chosen list of rows. rows[r] = (b*H + h)*Nq + i;
 * out is [nrows][d], lse is [nrows]. */
int oracle_attn_rows_f64(const double *q, const double *k, const double *v, const double *mask,
                         double *out, double *lse, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                         int64_t d, double scale, int causal, const int64_t *rows, int64_t nrows);

/* Block summary of one row's block of n scores s (already scaled and masked) and
 * values vals[n][dv]: m = max s, l = sum exp(s - m), u = sum exp(s - m) v.
 * An all -inf block gives (m, l, u) = (-inf, 0, 0). */
void oracle_block_summary_f64(const double *s, const double *vals, int64_t n, int64_t dv,
                              double *m, double *l, double *u);

/* Merge of two block summaries onto their common maximum ([Glossary], "Why a
 * tile can be discarded"). Output may alias either input. */
void oracle_merge_f64(double mA, double lA, const double *uA, double mB, double lB,
                      const double *uB, int64_t dv, double *m, double *l, double *u);

/* Blockwise evaluation: keys in blocks of `block`, each summarised and merged
 * into the running triple; o = u / l at the end. Must agree with the
 * materialised routine to rounding. */
int oracle_attn_blockwise_f64(const double *q, const double *k, const double *v, const double *mask,
                              double *out, double *lse, int64_t B, int64_t H, int64_t Nq, int64_t Nk,
                              int64_t d, double scale, int causal, int64_t block);

/* Gradients of sum(dout * out) with respect to q, k, v, from the materialised
 * softmax ([Lesson], "Backward recomputation" states what backward produces). */
int oracle_attn_bwd_f64(const double *q, const double *k, const double *v, const double *mask,
                        const double *dout, double *dq, double *dk, double *dv, int64_t B, int64_t H,
                        int64_t Nq, int64_t Nk, int64_t d, double scale, int causal);

/* Number of OpenMP threads the routines above use. */
int oracle_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
