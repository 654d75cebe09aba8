// fa_splitkv.cu -- split-KV attention forward for decoding (few query rows, long
// key/value sequence), and the exact merge of the per-split results.
//
// Each split s of the key range is one block of keys in the sense of the
// glossary page "FlashAttention", section "Why a tile can be discarded": a CTA
// streams its keys once, keeps the running maximum m, normaliser l and
// unnormalised accumulator a of every query row on chip ("FlashAttention:
// Exact Attention as an IO-Aware Streaming Computation", section "Mathematical
// structure"), and writes the block's summary as (o_s = a / l, lse_s = m + ln l)
// to a workspace. The combine kernel re-expresses every summary relative to the
// common maximum lse = ln sum_s exp(lse_s) and adds them:
//     o = sum_s exp(lse_s - lse) o_s
// which is the glossary's merge rule (its worked "Practice" example: block
// outputs 5 and 10 with masses 4 and 2 merge to 20/3). A split with no visible
// key has lse_s = -inf and weight 0; if every split is empty, o = 0, lse = -inf.
//
// Decoding reads every key and value once and does ~4d flop per 4d bytes, so the
// kernel is bound by HBM bandwidth: a warp reads one 128- or 256-byte K row per
// load instruction (each lane d/32 elements), several rows in flight per lane.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fa_splitkv.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

constexpr int kWarpsSK = 4;
constexpr int kUnroll = 4;  // key rows in flight per lane

template <typename T>
struct Vec;  // D/32 elements of one row owned by a lane
template <>
struct Vec<__nv_bfloat16> {
    __device__ static float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
    __device__ static __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
};
template <>
struct Vec<__half> {
    __device__ static float to_f(__half x) { return __half2float(x); }
    __device__ static __half from_f(float x) { return __float2half_rn(x); }
};

template <typename T, int E>
__device__ __forceinline__ void load_row(const T *row, int lane, float (&f)[E]) {
    // E consecutive elements at lane * E: 8 bytes (E = 4) or 4 bytes (E = 2)
    if constexpr (E == 4) {
        const uint2 u = __ldg(reinterpret_cast<const uint2 *>(row) + lane);
        const T *h = reinterpret_cast<const T *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) f[e] = Vec<T>::to_f(h[e]);
    } else {
        const uint32_t u = __ldg(reinterpret_cast<const uint32_t *>(row) + lane);
        const T *h = reinterpret_cast<const T *>(&u);
#pragma unroll
        for (int e = 0; e < 2; ++e) f[e] = Vec<T>::to_f(h[e]);
    }
}

// One CTA = one (split, b*h). Warps take keys w, w+4, w+8, ... of the split.
template <typename T, int D, int NQ, bool CAUSAL>
__global__ void __launch_bounds__(kWarpsSK * 32) fa_splitkv_partial(const T *__restrict__ q, const T *__restrict__ k,
                                                                    const T *__restrict__ v, float *__restrict__ o_part,
                                                                    float *__restrict__ lse_part, int BH, int Nq,
                                                                    int Nk, int split_len, float scale_log2) {
    constexpr int E = D / 32;
    const int split = blockIdx.x, bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k0 = split * split_len, k1 = min(Nk, k0 + split_len);
    const T *qb = q + (size_t)bh * Nq * D;
    const T *kb = k + (size_t)bh * Nk * D;
    const T *vb = v + (size_t)bh * Nk * D;

    float qf[NQ][E], acc[NQ][E], m[NQ], l[NQ];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        if (i < Nq) {
            load_row<T, E>(qb + (size_t)i * D, lane, qf[i]);
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) qf[i][e] = 0.f;
        }
#pragma unroll
        for (int e = 0; e < E; ++e) acc[i][e] = 0.f;
        m[i] = -INFINITY;
        l[i] = 0.f;
    }
    const int shift = Nk - Nq;  // causal: query i sees keys j <= i + shift
    for (int j0 = k0 + warp; j0 < k1; j0 += kWarpsSK * kUnroll) {
        float kf[kUnroll][E], vf[kUnroll][E];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int j = j0 + u * kWarpsSK;
            if (j < k1) {
                load_row<T, E>(kb + (size_t)j * D, lane, kf[u]);
                load_row<T, E>(vb + (size_t)j * D, lane, vf[u]);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) kf[u][e] = vf[u][e] = 0.f;
            }
        }
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            if (i >= Nq) break;
            float s[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                float part = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) part = fmaf(qf[i][e], kf[u][e], part);
                s[u] = part;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) s[u] += __shfl_xor_sync(0xffffffffu, s[u], off);
            float mb = -INFINITY;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int j = j0 + u * kWarpsSK;
                const bool ok = j < k1 && (!CAUSAL || j <= i + shift);
                s[u] = ok ? s[u] * scale_log2 : -INFINITY;
                mb = fmaxf(mb, s[u]);
            }
            const float m_new = fmaxf(m[i], mb);
            if (m_new == -INFINITY) continue;  // nothing visible yet for this row
            const float corr = ex2_approx(m[i] - m_new);  // 0 when m was -inf
            m[i] = m_new;
            l[i] *= corr;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[i][e] *= corr;
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const float pu = ex2_approx(s[u] - m_new);
                l[i] += pu;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[i][e] = fmaf(pu, vf[u][e], acc[i][e]);
            }
        }
    }
    // merge the four warps' summaries of this split (same rule as the combine)
    __shared__ float sm_m[kWarpsSK][NQ], sm_l[kWarpsSK][NQ];
    __shared__ float sm_a[kWarpsSK][NQ][D];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        if (lane == 0) {
            sm_m[warp][i] = m[i];
            sm_l[warp][i] = l[i];
        }
#pragma unroll
        for (int e = 0; e < E; ++e) sm_a[warp][i][lane * E + e] = acc[i][e];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < Nq * D; idx += kWarpsSK * 32) {
        const int i = idx / D, e = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarpsSK; ++w) M = fmaxf(M, sm_m[w][i]);
        float L = 0.f, A = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarpsSK; ++w) {
                const float f = ex2_approx(sm_m[w][i] - M);  // 0 for an empty warp
                L += f * sm_l[w][i];
                A += f * sm_a[w][i][e];
            }
        }
        const size_t row = ((size_t)split * BH + bh) * Nq + i;
        o_part[row * D + e] = L > 0.f ? A / L : 0.f;
        if (e == 0) lse_part[row] = L > 0.f ? (M + lg2_approx(L)) * 0.6931471805599453f : -INFINITY;
    }
}

// One CTA of D threads per (b*h, query row): merge the n_splits summaries.
template <typename T, int D>
__global__ void __launch_bounds__(D) fa_splitkv_combine(const float *__restrict__ o_part,
                                                       const float *__restrict__ lse_part, T *__restrict__ out,
                                                       float *__restrict__ lse, int rows, int n_splits) {
    const int row = blockIdx.x;  // (b*h)*Nq + i
    const int e = threadIdx.x;
    float M = -INFINITY;
    for (int s = 0; s < n_splits; ++s) M = fmaxf(M, lse_part[(size_t)s * rows + row]);
    float W = 0.f, A = 0.f;
    if (M != -INFINITY) {
        for (int s = 0; s < n_splits; ++s) {
            const float ls = lse_part[(size_t)s * rows + row];
            const float w = __expf(ls - M);  // 0 for an empty split
            W += w;
            A = fmaf(w, o_part[((size_t)s * rows + row) * D + e], A);
        }
    }
    out[(size_t)row * D + e] = Vec<T>::from_f(W > 0.f ? A / W : 0.f);
    if (e == 0) lse[row] = W > 0.f ? M + __logf(W) : -INFINITY;
}

template <typename T, int D, int NQ, bool CAUSAL>
int launch_sk(const SplitKVArgs &a) {
    const int BH = a.B * a.H;
    const int split_len = (a.Nk + a.n_splits - 1) / a.n_splits;
    const float sl2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
    dim3 grid(a.n_splits, BH);
    fa_splitkv_partial<T, D, NQ, CAUSAL><<<grid, kWarpsSK * 32, 0, a.stream>>>(
        static_cast<const T *>(a.q), static_cast<const T *>(a.k), static_cast<const T *>(a.v), a.o_part, a.lse_part,
        BH, a.Nq, a.Nk, split_len, sl2);
    if (cudaGetLastError() != cudaSuccess) return -5;
    fa_splitkv_combine<T, D><<<BH * a.Nq, D, 0, a.stream>>>(a.o_part, a.lse_part, static_cast<T *>(a.out), a.lse,
                                                            BH * a.Nq, a.n_splits);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

template <typename T, int D, bool CAUSAL>
int launch_sk_nq(const SplitKVArgs &a) {
    if (a.Nq <= 1) return launch_sk<T, D, 1, CAUSAL>(a);
    if (a.Nq <= 2) return launch_sk<T, D, 2, CAUSAL>(a);
    if (a.Nq <= 4) return launch_sk<T, D, 4, CAUSAL>(a);
    if (a.Nq <= 8) return launch_sk<T, D, 8, CAUSAL>(a);
    return launch_sk<T, D, 16, CAUSAL>(a);
}

template <typename T>
int launch_sk_t(const SplitKVArgs &a) {
    if (a.d == 128) return a.causal ? launch_sk_nq<T, 128, true>(a) : launch_sk_nq<T, 128, false>(a);
    if (a.d == 64) return a.causal ? launch_sk_nq<T, 64, true>(a) : launch_sk_nq<T, 64, false>(a);
    return -4;
}

}  // namespace

int launch_splitkv(const SplitKVArgs &a, bool fp16) {
    return fp16 ? launch_sk_t<__half>(a) : launch_sk_t<__nv_bfloat16>(a);
}

}  // namespace fa
