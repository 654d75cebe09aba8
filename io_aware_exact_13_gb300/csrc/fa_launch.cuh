// fa_launch.cuh -- host-side launch of the forward kernel for one element type.
// Included by one translation unit per element type; the C ABI in fa_api.cu
// validates arguments first and then calls launch_fwd<T>().
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_fwd_bk128.cuh"
#include "fa_fwd_kernel.cuh"

namespace fa {

struct LaunchArgs {
    const void *q, *k, *v;
    const float *mask;
    void *out;
    float *lse;
    int B, H, N, d;
    int Hkv;          // key/value heads (H for plain multi-head attention)
    float scale;
    int causal;
    cudaStream_t stream;
    int *status;      // device status word
    int num_sms;
    uint64_t timeout_ns;
    // packed variable-length batch (B = number of sequences, N = max_seqlen)
    const int *cu_seqlens = nullptr;
    int total = 0;
    int mask_per_head = 0;  // the mask is a per-head bias [B][H][N][N]
    // the shared mask packed to one bit per entry, and the packing pass's verdict (fa_mask_pack.cu);
    // nullptr: the fp32 mask is applied as given
    const void *mask_bits = nullptr;
    const int *mask_kind = nullptr;
    // dropout: keep threshold 1..256 (0 = no dropout), Philox key and counter offset
    int drop_threshold = 0;
    uint64_t drop_seed = 0, drop_offset = 0;
};

// Defined in fa_mask_pack.cu: bytes of the packed form of a [rows][nk] mask, and the packing pass
// (zeroes *kind, then sets it to 1 if some entry is neither 0 nor -inf). Returns 0 or -5.
size_t mask_bits_bytes(long long rows, int nk);
int launch_mask_pack(const float *mask, void *bits, int *kind, long long rows, int nk, int num_sms,
                     cudaStream_t stream);

// Defined in fa_api.cu: encodes a [B*H][N][d] tensor map with box_rows-row x
// 128-byte boxes and 128-byte swizzle. Returns false on failure.
bool encode_rows_map(CUtensorMap *map, CUtensorMapDataType dtype, int elem_bytes, const void *base, int d, int N,
                     int BH, int box_rows);
// Defined in fa_api.cu: encodes a token-major [total][heads][d] tensor as the
// 3-D map (d, heads, total) with 128-byte x 1 head x box_rows-token boxes and
// 128-byte swizzle. Returns false on failure.
bool encode_tokens_map(CUtensorMap *map, CUtensorMapDataType dtype, int elem_bytes, const void *base, int d,
                       int heads, int total, int box_rows);

// Work units of the dense schedule. n2 two-tile items over G persistent CTAs leave a last wave of
// rem = n2 % G items (all n2 when n2 < G). When those rem items, cut into their 2 rem single query tiles, fit
// in one wave, they are cut: the last wave then takes about the time of one tile instead of two. Equal
// (non-causal) items gain whenever that holds; causal items are sorted longest first, so only a grid with
// at most G / 2 items (one wave with idle CTAs) gains.
inline void split_tail(FwdParams &p, int n2, int G, bool causal) {
    const int rem = n2 % G;
    const bool split = rem > 0 && 2 * rem <= G && (!causal || n2 <= G / 2);
    p.n_pair = split ? n2 - rem : n2;
    p.n_items = split ? n2 + rem : n2;
}

template <typename T, int D, bool CAUSAL, bool MASK>
int launch_variant(const LaunchArgs &a) {
    using C = Cfg<T, D, MASK>;
    auto kern = fa_fwd_kernel<T, D, CAUSAL, MASK>;
    // The register split between warpgroups assumes 128 registers per thread at
    // launch (512 x 128 = 256 x 200 + 256 x 56). Refuse to launch otherwise.
    cudaFuncAttributes attr;
    if (cudaFuncGetAttributes(&attr, kern) != cudaSuccess) return -5;
    if (attr.numRegs * kThreads < 256 * 200 + 256 * 56) return -5;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
        return -5;
    CUtensorMap tq, tk, tv;
    const int BH = a.B * a.H;
    if (!encode_rows_map(&tq, Elem<T>::tma, sizeof(T), a.q, D, a.N, BH, kBQ)) return -5;
    const int BHkv = a.B * a.Hkv;
    if (!encode_rows_map(&tk, Elem<T>::tma, sizeof(T), a.k, D, a.N, BHkv, kBK)) return -5;
    if (!encode_rows_map(&tv, Elem<T>::tma, sizeof(T), a.v, D, a.N, BHkv, kBK)) return -5;
    // the mask [B][N][N] fp32 as (key, query row, b) with 32-key x 32-row boxes; its row stride must be a
    // multiple of 16 bytes (N % 4 == 0), otherwise the softmax warps read it directly
    CUtensorMap tm = tq;
    const bool mask_tma = MASK && a.mask && (a.N % 4) == 0;
    if (mask_tma && !encode_rows_map(&tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.mask, a.N, a.N,
                                     a.mask_per_head ? BH : a.B, 32))
        return -5;
    FwdParams p;
    p.out = a.out;
    p.lse = a.lse;
    p.mask = a.mask;
    p.status = a.status;
    p.B = a.B;
    p.kv_group = a.H / a.Hkv;
    p.H = a.H;
    p.N = a.N;
    p.rows_per_item = kRowsPerItem;
    p.n_qblk = (a.N + kRowsPerItem - 1) / kRowsPerItem;
    p.n_kv = (a.N + kBK - 1) / kBK;
    split_tail(p, BH * p.n_qblk, a.num_sms, CAUSAL);
    p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
    p.timeout_ns = a.timeout_ns;
    p.cu_seqlens = nullptr;
    p.total = 0;
    p.Hkv = a.Hkv;
    p.mask_tma = mask_tma ? 1 : 0;
    p.mask_per_head = a.mask_per_head;
    p.mask_bits = nullptr;
    p.mask_bits_blk = 0;
    p.mask_kind = MASK ? a.mask_kind : nullptr;
    p.drop_seed = p.drop_offset = 0;
    p.drop_threshold = 256;
    p.drop_scale = 1.0f;
    const int grid = p.n_items < a.num_sms ? p.n_items : a.num_sms;
    if (MASK && a.mask_kind != nullptr)  // behind the 128-key kernel on the packed mask (see launch_mask_fwd_d)
        return launch_dependent(kern, dim3(grid), dim3(kThreads), C::SMEM_BYTES, a.stream, tq, tk, tv, tm, p) ==
                       cudaSuccess
                   ? 0
                   : -5;
    kern<<<grid, kThreads, C::SMEM_BYTES, a.stream>>>(tq, tk, tv, tm, p);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

// The 128-key-block kernel: dense [B][H][N][d] tensors, or a packed batch; MASK: a shared
// [B][N][N] mask in its packed one-bit form; DROP: dropout (dense, no mask).
template <typename T, int D, bool CAUSAL, bool VARLEN, bool MASK = false, bool DROP = false>
int launch_bk128(const LaunchArgs &a) {
    static_assert(!(VARLEN && MASK), "no mask in a packed batch");
    using C = Cfg128<T, D>;
    auto kern = fa_fwd_bk128_kernel<T, D, CAUSAL, VARLEN, MASK, DROP>;
    if (MASK && (a.mask_bits == nullptr || a.mask_kind == nullptr)) return -5;
    if (DROP && (a.drop_threshold < 1 || a.drop_threshold > 256)) return -5;
    // The register split between warpgroups assumes 128 registers per thread at
    // launch (512 x 128 = 256 x 184 + 256 x 72). Refuse to launch otherwise.
    cudaFuncAttributes attr;
    if (cudaFuncGetAttributes(&attr, kern) != cudaSuccess) return -5;
    if (attr.numRegs * kThreads < 256 * 184 + 256 * 72) return -5;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
        return -5;
    CUtensorMap tq, tk, tv;
    if (VARLEN) {
        if (!encode_tokens_map(&tq, Elem<T>::tma, sizeof(T), a.q, D, a.H, a.total, kBQ)) return -5;
        if (!encode_tokens_map(&tk, Elem<T>::tma, sizeof(T), a.k, D, a.Hkv, a.total, kBK128)) return -5;
        if (!encode_tokens_map(&tv, Elem<T>::tma, sizeof(T), a.v, D, a.Hkv, a.total, kBK128)) return -5;
    } else {
        if (!encode_rows_map(&tq, Elem<T>::tma, sizeof(T), a.q, D, a.N, a.B * a.H, kBQ)) return -5;
        if (!encode_rows_map(&tk, Elem<T>::tma, sizeof(T), a.k, D, a.N, a.B * a.Hkv, kBK128)) return -5;
        if (!encode_rows_map(&tv, Elem<T>::tma, sizeof(T), a.v, D, a.N, a.B * a.Hkv, kBK128)) return -5;
    }
    FwdParams p;
    p.out = a.out;
    p.lse = a.lse;
    p.mask = nullptr;
    p.status = a.status;
    p.B = a.B;
    p.H = a.H;
    p.kv_group = a.H / a.Hkv;
    p.N = a.N;  // max_seqlen for a packed batch
    p.rows_per_item = kRowsPerItem;
    p.n_qblk = (a.N + kRowsPerItem - 1) / kRowsPerItem;
    p.n_kv = (a.N + kBK128 - 1) / kBK128;
    if (VARLEN) {
        p.n_items = a.B * a.H * p.n_qblk;
        p.n_pair = p.n_items;  // the packed-batch list has its own order
    } else {
        split_tail(p, a.B * a.H * p.n_qblk, a.num_sms, CAUSAL);
    }
    p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
    p.timeout_ns = a.timeout_ns;
    p.cu_seqlens = VARLEN ? a.cu_seqlens : nullptr;
    p.total = VARLEN ? a.total : 0;
    p.Hkv = a.Hkv;
    p.mask_tma = 0;
    p.mask_per_head = 0;
    p.mask_bits = MASK ? static_cast<const uint4 *>(a.mask_bits) : nullptr;
    p.mask_bits_blk = MASK ? (a.N + kBK128 - 1) / kBK128 : 0;
    p.mask_kind = MASK ? a.mask_kind : nullptr;
    p.drop_seed = DROP ? a.drop_seed : 0;
    p.drop_offset = DROP ? a.drop_offset : 0;
    p.drop_threshold = DROP ? a.drop_threshold : 256;
    p.drop_scale = DROP ? static_cast<float>(256.0 / a.drop_threshold) : 1.0f;
    const int grid = p.n_items < a.num_sms ? p.n_items : a.num_sms;
    // a programmatic dependent of the work ahead (MASK: the packing pass, whose verdict and bits it waits
    // for; otherwise whatever ran before, waited for before any global access)
    return launch_dependent(kern, dim3(grid), dim3(kThreads), C::SMEM_BYTES, a.stream, tq, tk, tv, p) == cudaSuccess
               ? 0
               : -5;
}

template <typename T, int D, bool VARLEN>
int launch_bk128_d(const LaunchArgs &a) {
    return a.causal ? launch_bk128<T, D, true, VARLEN>(a) : launch_bk128<T, D, false, VARLEN>(a);
}

// The 64-key-block kernel with an additive mask.
template <typename T, int D>
int launch_masked_d(const LaunchArgs &a) {
    return a.causal ? launch_variant<T, D, true, true>(a) : launch_variant<T, D, false, true>(a);
}

// A forward with an additive mask. With the packed form of a shared mask, both kernels are queued:
// the 128-key kernel applies the bits when every entry was 0 or -inf, the 64-key kernel the fp32
// mask otherwise, and each returns at once when the verdict is the other one's. The 64-key kernel
// is the 128-key kernel's programmatic dependent: when it only has to return, its CTAs do so on the
// SMs the 128-key grid's last wave leaves idle, after waiting for that grid to finish.
template <typename T, int D>
int launch_mask_fwd_d(const LaunchArgs &a) {
    if (a.mask_bits != nullptr && a.mask_kind != nullptr && !a.mask_per_head) {
        const int rc = a.causal ? launch_bk128<T, D, true, false, true>(a) : launch_bk128<T, D, false, false, true>(a);
        if (rc != 0) return rc;
    }
    return launch_masked_d<T, D>(a);
}

int launch_fwd_mask_bf16(const LaunchArgs &a);  // fa_fwd_mask_bf16.cu
int launch_fwd_mask_fp16(const LaunchArgs &a);  // fa_fwd_mask_fp16.cu
int launch_fwd_drop_bf16(const LaunchArgs &a);  // fa_fwd_drop_bf16.cu
int launch_fwd_drop_fp16(const LaunchArgs &a);  // fa_fwd_drop_fp16.cu

// A forward with dropout (dense, no mask).
template <typename T, int D>
int launch_drop_fwd_d(const LaunchArgs &a) {
    return a.causal ? launch_bk128<T, D, true, false, false, true>(a) : launch_bk128<T, D, false, false, false, true>(a);
}

}  // namespace fa
