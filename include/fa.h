/*
 * fa.h -- C ABI of the exact tiled attention forward for GB300 (sm_103a).
 *
 * Operation ("FlashAttention: Exact Attention as an IO-Aware Streaming
 * Computation", sections "Problem setting" and "Mathematical structure";
 * "FlashAttention" glossary, section "Move less data" for the additive mask M):
 *
 *     O = softmax(scale * Q K^T + M) V,   lse_i = ln sum_j exp(s_ij)
 *
 * computed exactly (up to floating-point rounding) by streaming key/value
 * tiles past an on-chip query tile that keeps its running row maximum m,
 * denominator l and unnormalised accumulator a ("IO-aware exact attention",
 * section "One tiled forward-pass iteration"). Only O and lse are written to
 * device memory; no N x N score or probability tensor is ever stored.
 *
 * Layouts (all contiguous, row-major, last index fastest; all DEVICE pointers):
 *   q, k, v, out : [B][H][N][d], element type per entry point (bf16, fp16, fp32);
 *                  out has the same element type as q.
 *   lse          : float [B][H][N], natural log of the softmax normaliser of the
 *                  scaled, masked scores; -inf for a fully masked row.
 *   mask_or_null : NULL, or float [B][N][N], additive, shared by all H heads;
 *                  entries finite or -inf (+inf and NaN are not supported).
 *   causal       : nonzero allows key j for query i iff j <= i ("IO-aware exact
 *                  attention", section "Tile order and on-chip capacity").
 *                  Causal and mask combine additively when both are given.
 *   scale        : multiplies Q K^T (typically 1/sqrt(d)).
 * A query row whose every key is excluded gets out = 0 and lse = -inf.
 *
 * Ownership: every pointer is caller-owned device memory. The library allocates
 * no device memory, keeps no per-call state and may be called from several
 * host threads. Calls are stream-ordered and asynchronous: they enqueue work on
 * `stream` (a cudaStream_t; NULL = legacy default stream) and return.
 *
 * Errors: arguments are checked on the host before anything is launched; a
 * failed check returns the negative status below and launches nothing. A
 * launch failure returns FA_ERR_LAUNCH. Device-side pipeline waits are bounded:
 * if one gives up, the kernel records FA_ERR_TIMEOUT in a device status word
 * (read it with fa_get_device_status) and the outputs are undefined.
 */
#ifndef FA_H
#define FA_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_NULL = -1,        /* a required pointer is NULL */
    FA_ERR_ALIGN = -2,       /* a pointer is not 16-byte aligned */
    FA_ERR_SHAPE = -3,       /* B, H or N < 1, or a size overflows its limit */
    FA_ERR_UNSUPPORTED = -4, /* d not supported for this element type */
    FA_ERR_LAUNCH = -5,      /* the CUDA launch (or tensor-map encoding) failed */
    FA_ERR_TIMEOUT = -6,     /* a device-side wait gave up (device status word) */
    FA_ERR_WORKSPACE = -7,   /* workspace missing or smaller than the problem needs */
    FA_ERR_SEQLENS = -8,     /* packed batch: cu_seqlens inconsistent (device status word) */
    FA_ERR_ARG = -9          /* an argument is outside its range (dropout probability) */
} fa_status;

/* bf16 Q/K/V/out, fp32 accumulation. d in {64, 128}. */
int fa_fwd(const void *q, const void *k, const void *v, const float *mask_or_null, void *out,
           float *lse, int B, int H, int N, int d, float scale, int causal, void *stream);

/* fp16 Q/K/V/out, fp32 accumulation. d in {64, 128}. */
int fa_fwd_fp16(const void *q, const void *k, const void *v, const float *mask_or_null, void *out,
                float *lse, int B, int H, int N, int d, float scale, int causal, void *stream);

/* fp32 Q/K/V/out, computed in fp32 on the CUDA cores (no tensor cores, no
 * rounding of the inputs). d in {64, 128}; B*H must not exceed 65535. */
int fa_fwd_fp32(const void *q, const void *k, const void *v, const float *mask_or_null, void *out,
                float *lse, int B, int H, int N, int d, float scale, int causal, void *stream);

/* ---- forward from host memory ---------------------------------------------
 * The same forward (bf16 / fp16, no mask, Hkv = H) for inputs and outputs in
 * HOST memory: q_host, k_host, v_host, out_host : [B][H][N][d], lse_host : float
 * [B][H][N], and caller-owned DEVICE buffers of the same shapes (q_dev .. lse_dev)
 * that the call uses as staging. The B*H head slabs are cut into n_chunks
 * (1 .. min(B*H, 64)) contiguous chunks, shrinking toward the end in the ratio
 * n_chunks : n_chunks-1 : ... : 1 (rounded to whole heads; a chunk that rounds
 * to none is skipped) so that the last forward and copy-out, which no copy
 * overlaps, are short. Each chunk's host->device copies, forward and
 * device->host copies are pipelined on two internal copy streams (created on
 * the first call per device) and `stream`; everything is ordered after earlier
 * work on `stream` and complete when later work on `stream` starts, so
 * cudaStreamSynchronize(stream) waits for the results in host memory. Host
 * buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for the
 * copies to overlap; the results equal fa_fwd's bit for bit. Errors as for
 * fa_fwd (host pointers must be non-NULL). */
int fa_fwd_host(const void *q_host, const void *k_host, const void *v_host, void *out_host, float *lse_host,
                void *q_dev, void *k_dev, void *v_dev, void *out_dev, float *lse_dev, int B, int H, int N, int d,
                float scale, int causal, int n_chunks, void *stream);
int fa_fwd_host_fp16(const void *q_host, const void *k_host, const void *v_host, void *out_host, float *lse_host,
                     void *q_dev, void *k_dev, void *v_dev, void *out_dev, float *lse_dev, int B, int H, int N,
                     int d, float scale, int causal, int n_chunks, void *stream);

/* ---- grouped-query attention ------------------------------------------------
 * Same operation and layouts as fa_fwd / fa_fwd_fp16, except that k and v hold
 * Hkv heads, [B][Hkv][N][d], each shared by H / Hkv consecutive query heads:
 * query head h reads key/value head h / (H / Hkv). Hkv must divide H; Hkv = H
 * is plain multi-head attention. (The variant is named by "IO-aware exact
 * attention", section "Why implementations form a family".) */
int fa_fwd_gqa(const void *q, const void *k, const void *v, const float *mask_or_null, void *out, float *lse,
               int B, int H, int Hkv, int N, int d, float scale, int causal, void *stream);
int fa_fwd_gqa_fp16(const void *q, const void *k, const void *v, const float *mask_or_null, void *out,
                    float *lse, int B, int H, int Hkv, int N, int d, float scale, int causal, void *stream);

/* ---- per-head additive bias -------------------------------------------------
 * Same operation as fa_fwd / fa_fwd_fp16 with the additive term M given per head:
 * bias is float [B][H][N][N] (DEVICE, 16-byte aligned, required), and score
 * (b, h, i, j) = scale q_i k_j^T + bias[b][h][i][j] (+ the causal term). Entries
 * are finite or -inf; a row whose every key is -inf gets out = 0 and lse = -inf.
 * ("IO-aware exact attention", section "Why implementations form a family":
 * bias is one of the variants that modify the calculation; "FlashAttention"
 * glossary, section "Move less data", for the additive M.) Errors as for fa_fwd;
 * FA_ERR_NULL if bias is NULL. */
int fa_fwd_bias(const void *q, const void *k, const void *v, const float *bias, void *out, float *lse, int B, int H,
                int N, int d, float scale, int causal, void *stream);
int fa_fwd_bias_fp16(const void *q, const void *k, const void *v, const float *bias, void *out, float *lse, int B,
                     int H, int N, int d, float scale, int causal, void *stream);

/* ---- additive mask, packed -------------------------------------------------
 * The forward of fa_fwd_gqa / fa_fwd_gqa_fp16 with a shared mask (required,
 * float [B][N][N], 16-byte aligned) and a caller-owned DEVICE workspace
 * (256-byte aligned, at least fa_fwd_masked_workspace_bytes(B, N) bytes; the
 * call owns it until later work on `stream` starts). Hkv = H is multi-head
 * attention.
 * Most masks hold only 0 and -inf (padding, causal variants, sparsity
 * patterns, fully masked rows), and for those the mask term of the glossary
 * "FlashAttention", section "Move less data", is one bit per entry. Every call
 * first reads the mask once and writes its one-bit form into the workspace
 * (about B*N*N/8 bytes), with a verdict word. Then two kernels are queued:
 * the 128-key-block kernel, which applies the bits, and the fp32-mask kernel
 * of fa_fwd. Only the one that matches the verdict does any work. With a
 * 0/-inf mask every head reads 16 bytes of bits per 128 keys instead of
 * 512 bytes of fp32 mask. The results are those of the 128-key kernel
 * without a mask, with masked keys excluded. A mask with any other value is
 * applied as given, with the same results as fa_fwd. Errors as for fa_fwd;
 * FA_ERR_NULL if mask is NULL, FA_ERR_WORKSPACE if the workspace is missing,
 * misaligned or too small. fa_fwd_masked_workspace_bytes returns the size, or
 * FA_ERR_SHAPE for B or N < 1. */
long long fa_fwd_masked_workspace_bytes(int B, int N);
int fa_fwd_masked(const void *q, const void *k, const void *v, const float *mask, void *out, float *lse, int B, int H,
                  int Hkv, int N, int d, float scale, int causal, void *workspace, unsigned long long workspace_bytes,
                  void *stream);
int fa_fwd_masked_fp16(const void *q, const void *k, const void *v, const float *mask, void *out, float *lse, int B,
                       int H, int Hkv, int N, int d, float scale, int causal, void *workspace,
                       unsigned long long workspace_bytes, void *stream);

/* ---- dropout --------------------------------------------------------------
 * The forward of fa_fwd_gqa / fa_fwd_gqa_fp16 (no mask) with dropout on the
 * attention probabilities ("IO-aware exact attention", section "Why
 * implementations form a family", names dropout as a variant of the
 * calculation): out_i = sum_j P_ij keep_ij / q v_j, with P the softmax of the
 * undropped scores; lse is unchanged. keep_ij is 1 with probability
 * q = t / 256, t = floor((1 - p_drop) * 256 + 0.5), as follows:
 *   keep_ij = [byte (j mod 32) of Philox4x64-10(counter = {i, j / 32, b*H + h,
 *              offset}, key = {seed, 0}) < t],
 * bytes numbered from the least significant byte of output word 0 upward.
 * Philox4x64-10 is the counter-based generator of Salmon, Moraes, Dror and
 * Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC 2011). The same
 * (seed, offset) gives the same keep pattern on every call; callers advance
 * `offset` (or change `seed`) between steps. p_drop = 0 gives fa_fwd_gqa's
 * results bit for bit. Errors as for fa_fwd_gqa; FA_ERR_ARG if t < 1 (p_drop
 * keeps nothing) or p_drop < 0 or NaN. */
int fa_fwd_dropout(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H, int Hkv, int N,
                   int d, float scale, int causal, float p_drop, unsigned long long seed, unsigned long long offset,
                   void *stream);
int fa_fwd_dropout_fp16(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H, int Hkv,
                        int N, int d, float scale, int causal, float p_drop, unsigned long long seed,
                        unsigned long long offset, void *stream);

/* ---- split-KV forward for decoding ------------------------------------------
 * Same operation for Nq query rows (1 <= Nq <= 16) against Nk >= 1 keys:
 *   q, out : [B][H][Nq][d]      k, v : [B][H][Nk][d]      lse : float [B][H][Nq]
 * causal != 0 aligns the last query with the last key: query i sees keys
 * j <= i + (Nk - Nq); otherwise every query sees every key. No mask argument.
 * The key range is cut into n_splits contiguous blocks; each block's summary
 * (its partial output and log-sum-exp) is written to `workspace`, and a second
 * kernel merges the summaries onto their common maximum ("FlashAttention"
 * glossary, sections "Why a tile can be discarded" and "Practice: can you
 * average block outputs?"). The result equals the unsplit attention.
 * workspace: caller-owned device memory, 256-byte aligned, of at least
 * fa_splitkv_workspace_bytes(B, H, Nq, d, n_splits) bytes; its contents on
 * entry do not matter and are overwritten. Calls that share a workspace must
 * not overlap on the GPU. B*H <= 65535, 1 <= n_splits <= Nk. */

/* A split count that gives the GPU enough independent blocks (>= 1). */
int fa_splitkv_num_splits(int B, int H, int Nq, int Nk, int d);

/* Workspace bytes fa_fwd_splitkv needs, or a negative status. */
long long fa_splitkv_workspace_bytes(int B, int H, int Nq, int d, int n_splits);

/* bf16 q/k/v/out, fp32 accumulation. d in {64, 128}. */
int fa_fwd_splitkv(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H, int Nq,
                   int Nk, int d, float scale, int causal, int n_splits, void *workspace,
                   unsigned long long workspace_bytes, void *stream);

/* fp16 q/k/v/out, fp32 accumulation. d in {64, 128}. */
int fa_fwd_splitkv_fp16(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
                        int Nq, int Nk, int d, float scale, int causal, int n_splits, void *workspace,
                        unsigned long long workspace_bytes, void *stream);

/* bf16 split-KV forward that allocates nothing and takes no workspace (the
 * method's pages have no counterpart of this entry point; it exists for
 * callers that cannot allocate device memory where they call attention: a
 * host framework that owns every device allocation through its own pool, a
 * serving loop in which cudaMalloc's implicit device-wide synchronisation
 * would stall other work, or an embedded host with a fixed memory budget).
 * Same arguments and results as fa_fwd_splitkv minus the workspace: the
 * per-split scratch lives in one 16 MiB device array inside the library, which
 * every GPU that loads the library holds until exit. Problems whose scratch,
 * fa_splitkv_workspace_bytes(B, H, Nq, d, n_splits), exceeds 16 MiB are
 * rejected with FA_ERR_WORKSPACE. The first call on a device looks up the
 * array's device address (with that device current); make that first call
 * before any stream capture. All calls share the array: calls that overlap
 * on the GPU race and must be serialised by the caller. */
int fa_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
                           int Nq, int Nk, int d, float scale, int causal, int n_splits, void *stream);

/* ---- packed variable-length batch ------------------------------------------
 * The same attention for nseq independent sequences packed back to back
 * ("IO-aware exact attention", section "Tile order and on-chip capacity":
 * packed sequences add bounds and indexing). Sequence s holds tokens
 * [cu_seqlens[s], cu_seqlens[s+1]) and attends only within itself; causal
 * allows key j for query i of the same sequence iff j <= i.
 * Layouts (DEVICE pointers, token-major, last index fastest):
 *   q, out : [total][H][d]      k, v : [total][Hkv][d]      lse : float [H][total]
 *   cu_seqlens : int32 [nseq + 1], cu_seqlens[0] = 0, non-decreasing,
 *                cu_seqlens[nseq] <= total (tokens past it are left untouched).
 * max_seqlen is a host-side upper bound on every sequence length; work is
 * sized by nseq * H * ceil(max_seqlen / 256). The bounds are read on the
 * device: a sequence with cu_seqlens[s+1] < cu_seqlens[s], a negative start,
 * an end past total or a length above max_seqlen is skipped (its rows are not
 * written) and FA_ERR_SEQLENS is recorded in the device status word. A
 * zero-length sequence is allowed. Hkv must divide H (grouped-query attention
 * as in fa_fwd_gqa). No mask argument. d in {64, 128}. */
int fa_fwd_varlen(const void *q, const void *k, const void *v, void *out, float *lse, const int *cu_seqlens,
                  int nseq, int total, int max_seqlen, int H, int Hkv, int d, float scale, int causal,
                  void *stream);
int fa_fwd_varlen_fp16(const void *q, const void *k, const void *v, void *out, float *lse, const int *cu_seqlens,
                       int nseq, int total, int max_seqlen, int H, int Hkv, int d, float scale, int causal,
                       void *stream);

/* ---- backward by recomputation ---------------------------------------------
 * Gradients of L = sum(dout o out) for out = softmax(scale Q K^T) V ("IO-aware
 * exact attention", section "Backward recomputation"): from q, k, v, the
 * forward's out and lse, and dout, every score and probability tile is
 * rebuilt on chip (P = exp(scale Q K^T - lse)), so no N x N tensor is stored:
 *   dV = P^T dout,  dS = P o (dout V^T - D),  D_i = sum_t dout_it out_it,
 *   dQ = scale dS K,  dK = scale dS^T Q.
 * Layouts: q, k, v, out, dout, dq, dk, dv : [B][H][N][d], one element type per
 * entry point (bf16 / fp16); lse : float [B][H][N] as written by fa_fwd.
 * All are DEVICE pointers, caller-owned, 16-byte aligned (lse 4). No mask
 * argument; causal as in fa_fwd. Every query row must see at least one key
 * (true without a mask), so that lse is finite.
 * workspace: caller-owned device memory, 256-byte aligned, of at least
 * fa_bwd_workspace_bytes(B, H, N, d) bytes (an fp32 dQ accumulator of
 * B*H*N*d floats plus two per-row fp32 arrays); contents on entry do not
 * matter. Calls sharing a workspace must not overlap on the GPU. Three kernels
 * are enqueued on `stream`: row statistics, the tiled backward, and the
 * conversion of the dQ accumulator. d in {64, 128}.
 * Errors as for fa_fwd; FA_ERR_WORKSPACE if the workspace is missing, too
 * small or misaligned. */
long long fa_bwd_workspace_bytes(int B, int H, int N, int d);
int fa_bwd(const void *q, const void *k, const void *v, const void *out, const void *dout, const float *lse,
           void *dq, void *dk, void *dv, int B, int H, int N, int d, float scale, int causal, void *workspace,
           unsigned long long workspace_bytes, void *stream);
int fa_bwd_fp16(const void *q, const void *k, const void *v, const void *out, const void *dout, const float *lse,
                void *dq, void *dk, void *dv, int B, int H, int N, int d, float scale, int causal,
                void *workspace, unsigned long long workspace_bytes, void *stream);

/* Static text for a status code (never NULL). */
const char *fa_status_string(int status);

/* Synchronises `stream`, returns the device status word of the current device
 * (FA_OK, FA_ERR_TIMEOUT or FA_ERR_SEQLENS) and clears it. Returns FA_ERR_LAUNCH if the
 * synchronisation itself fails. */
int fa_get_device_status(void *stream);

/* Failure-detection self-test (the pages have no counterpart; it checks this
 * library's own error path). Enqueues one warp that waits on an mbarrier that
 * nothing ever completes, through the same bounded wait that every pipeline
 * role of every kernel uses. After timeout_ns (1 ns .. 1 s) the wait gives up,
 * FA_ERR_TIMEOUT is recorded in the device status word and the kernel exits;
 * the CUDA context stays usable. Returns FA_OK once enqueued, FA_ERR_SHAPE for
 * a timeout outside that range. */
int fa_selftest_wait_timeout(unsigned long long timeout_ns, void *stream);

/* Number of streaming multiprocessors the persistent grid is sized for on the
 * current device, or a negative status. */
int fa_num_sms(void);

#ifdef __cplusplus
}
#endif
#endif /* FA_H */
