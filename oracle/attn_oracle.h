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

/* ---- dropout ---------------------------------------------------------------
 * [Lesson] "Why implementations form a family" names dropout as one of the
 * variants that modify the calculation and defines nothing further. Reading
 * used (the usual one for attention): the normalised probabilities P_ij are
 * multiplied by keep_ij / q before the weighted sum over V; lse stays that of
 * the undropped scores. The keep probability is q = threshold / 256
 * (1 <= threshold <= 256) and keep_ij = [u_ij < threshold] for a byte u_ij of a
 * counter-based stream:
 *   u_ij = byte (j mod 32) of Philox4x64-10(counter = {i, j div 32, b*H + h, offset},
 *                                            key = {seed, 0}),
 * bytes numbered from the least significant byte of output word 0 upward
 * (word j mod 32 div 8, bits 8 * (j mod 8) ...).
 * Philox4x64-10 is the generator of Salmon, Moraes, Dror and Shaw, "Parallel
 * random numbers: as easy as 1, 2, 3" (SC 2011). */

/* One Philox4x64-10 block: out = the 256-bit image of the counter under the key. */
void oracle_philox4x64_10(const uint64_t ctr[4], const uint64_t key[2], uint64_t out[4]);

/* keep[B][H][Nq][Nk] (0 or 1) as defined above. Returns 0, or -1 on a bad argument. */
int oracle_dropout_keep(uint8_t *keep, int64_t B, int64_t H, int64_t Nq, int64_t Nk, int threshold,
                        uint64_t seed, uint64_t offset);

/* Attention with dropout (no mask; causal as above). Returns 0, or -1 on a bad argument. */
int oracle_attn_dropout_f64(const double *q, const double *k, const double *v, double *out, double *lse,
                            int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t d, double scale,
                            int causal, int threshold, uint64_t seed, uint64_t offset);

#ifdef __cplusplus
}
#endif
#endif
