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

// Several query rows per head (2 <= Nq <= 16). With one key row per warp every
// key costs log2(32) shuffle steps per query row, which makes the kernel
// issue-bound long before HBM is busy. Here a group of L lanes owns one key row
// (each lane D/L consecutive elements), so a warp handles 32/L keys per step and
// a dot product needs only log2(L) shuffle steps. Each lane group keeps its own
// running (m, l, acc) per query row, with the lazy rescaling of the forward
// (the reference maximum moves only when a score exceeds it by more than
// kTauSK, in log2 units); the groups and then the warps are merged with the
// same block-summary rule as the combine kernel.
constexpr float kTauSK = 8.0f;

template <typename T, int E>
__device__ __forceinline__ void load_vec(const T *src, float (&f)[E]) {
    // E consecutive 16-bit elements, E in {4, 8, 16}: 8- or 16-byte loads
    if constexpr (E == 4) {
        const uint2 u = __ldg(reinterpret_cast<const uint2 *>(src));
        const T *h = reinterpret_cast<const T *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) f[e] = Vec<T>::to_f(h[e]);
    } else {
#pragma unroll
        for (int c = 0; c < E / 8; ++c) {
            const uint4 u = __ldg(reinterpret_cast<const uint4 *>(src) + c);
            const T *h = reinterpret_cast<const T *>(&u);
#pragma unroll
            for (int e = 0; e < 8; ++e) f[8 * c + e] = Vec<T>::to_f(h[e]);
        }
    }
}

template <typename T, int D, int NQ, int L, bool CAUSAL>
__global__ void __launch_bounds__(kWarpsSK * 32) fa_splitkv_partial_lg(
    const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v, float *__restrict__ o_part,
    float *__restrict__ lse_part, int BH, int Nq, int Nk, int split_len, float scale_log2) {
    constexpr int G = 32 / L;  // key rows per warp step
    constexpr int E = D / L;   // elements of a row per lane
    constexpr int STEP = kWarpsSK * G;
    const int split = blockIdx.x, bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gi = lane / L, li = lane % L;
    const int k0 = split * split_len, k1 = min(Nk, k0 + split_len);
    const T *qb = q + (size_t)bh * Nq * D + li * E;
    const T *kb = k + (size_t)bh * Nk * D + li * E;
    const T *vb = v + (size_t)bh * Nk * D + li * E;

    float qf[NQ][E], acc[NQ][E], m[NQ], l[NQ];
#pragma unroll
    for (int i = 0; i < NQ; ++i) {
        if (i < Nq) {
            load_vec<T, E>(qb + (size_t)i * D, qf[i]);
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
    for (int j0 = k0 + warp * G + gi; j0 < k1 + gi; j0 += 2 * STEP) {
        float kf[2][E], vf[2][E];
        bool ok[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {  // two key rows in flight per lane
            const int j = j0 + u * STEP;
            ok[u] = j < k1;
            if (ok[u]) {
                load_vec<T, E>(kb + (size_t)j * D, kf[u]);
                load_vec<T, E>(vb + (size_t)j * D, vf[u]);
            } else {
#pragma unroll
                for (int e = 0; e < E; ++e) kf[u][e] = vf[u][e] = 0.f;
            }
        }
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            if (i >= Nq) break;
            float sc[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                float part = 0.f;
#pragma unroll
                for (int e = 0; e < E; ++e) part = fmaf(qf[i][e], kf[u][e], part);
                sc[u] = part;
            }
#pragma unroll
            for (int off = L / 2; off > 0; off >>= 1)
#pragma unroll
                for (int u = 0; u < 2; ++u) sc[u] += __shfl_xor_sync(0xffffffffu, sc[u], off);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int j = j0 + u * STEP;
                const bool vis = ok[u] && (!CAUSAL || j <= i + shift);
                const float x = vis ? sc[u] * scale_log2 : -INFINITY;
                if (x > m[i] + kTauSK) {  // (also true for the first visible key, m = -inf)
                    const float corr = ex2_approx(m[i] - x);  // 0 when m was -inf
                    l[i] *= corr;
#pragma unroll
                    for (int e = 0; e < E; ++e) acc[i][e] *= corr;
                    m[i] = x;
                }
                const float pu = vis ? ex2_approx(x - m[i]) : 0.f;
                l[i] += pu;
#pragma unroll
                for (int e = 0; e < E; ++e) acc[i][e] = fmaf(pu, vf[u][e], acc[i][e]);
            }
        }
    }
    // merge the G lane groups of the warp (lanes li, li + L, li + 2L, ... hold the same elements)
#pragma unroll
    for (int off = L; off < 32; off <<= 1) {
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            const float mo = __shfl_xor_sync(0xffffffffu, m[i], off);
            const float lo = __shfl_xor_sync(0xffffffffu, l[i], off);
            const float mn = fmaxf(m[i], mo);
            const float fa = mn == -INFINITY ? 0.f : ex2_approx(m[i] - mn);
            const float fb = mn == -INFINITY ? 0.f : ex2_approx(mo - mn);
            l[i] = l[i] * fa + lo * fb;
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float ao = __shfl_xor_sync(0xffffffffu, acc[i][e], off);
                acc[i][e] = acc[i][e] * fa + ao * fb;
            }
            m[i] = mn;
        }
    }
    // merge the four warps' summaries of this split
    __shared__ float sm_m[kWarpsSK][NQ], sm_l[kWarpsSK][NQ];
    __shared__ float sm_a[kWarpsSK][NQ][D];
    if (gi == 0) {
#pragma unroll
        for (int i = 0; i < NQ; ++i) {
            if (li == 0) {
                sm_m[warp][i] = m[i];
                sm_l[warp][i] = l[i];
            }
#pragma unroll
            for (int e = 0; e < E; ++e) sm_a[warp][i][li * E + e] = acc[i][e];
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < Nq * D; idx += kWarpsSK * 32) {
        const int i = idx / D, e = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarpsSK; ++w) M = fmaxf(M, sm_m[w][i]);
        float Lsum = 0.f, A = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarpsSK; ++w) {
                const float f = ex2_approx(sm_m[w][i] - M);  // 0 for an empty warp
                Lsum += f * sm_l[w][i];
                A += f * sm_a[w][i][e];
            }
        }
        const size_t row = ((size_t)split * BH + bh) * Nq + i;
        o_part[row * D + e] = Lsum > 0.f ? A / Lsum : 0.f;
        if (e == 0) lse_part[row] = Lsum > 0.f ? (M + lg2_approx(Lsum)) * 0.6931471805599453f : -INFINITY;
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

// Lanes per key row for the several-row kernel: as few as possible (fewer
// shuffle steps per dot product) while q, acc and two key rows in flight stay
// near 128 registers, so that four CTAs fit on an SM.
constexpr int lanes_per_key(int D, int NQ) { return D == 128 ? (NQ <= 4 ? 16 : 32) : (NQ <= 4 ? 8 : 16); }

template <typename T, int D, int NQ>
int occupancy_d_nq() {
    int nb = 0;
    cudaError_t e;
    if constexpr (NQ == 1)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fa_splitkv_partial<T, D, NQ, false>, kWarpsSK * 32,
                                                          0);
    else
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &nb, fa_splitkv_partial_lg<T, D, NQ, lanes_per_key(D, NQ), false>, kWarpsSK * 32, 0);
    return e == cudaSuccess && nb > 0 ? nb : 1;
}

template <int D>
int occupancy_d(int Nq) {
    using T = __nv_bfloat16;
    if (Nq <= 1) return occupancy_d_nq<T, D, 1>();
    if (Nq <= 2) return occupancy_d_nq<T, D, 2>();
    if (Nq <= 4) return occupancy_d_nq<T, D, 4>();
    if (Nq <= 8) return occupancy_d_nq<T, D, 8>();
    return occupancy_d_nq<T, D, 16>();
}

template <typename T, int D, int NQ, bool CAUSAL>
int launch_sk(const SplitKVArgs &a) {
    const int BH = a.B * a.H;
    const int split_len = (a.Nk + a.n_splits - 1) / a.n_splits;
    const float sl2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
    dim3 grid(a.n_splits, BH);
    if constexpr (NQ == 1) {  // one query row: a warp per key row needs no lane groups
        fa_splitkv_partial<T, D, NQ, CAUSAL><<<grid, kWarpsSK * 32, 0, a.stream>>>(
            static_cast<const T *>(a.q), static_cast<const T *>(a.k), static_cast<const T *>(a.v), a.o_part,
            a.lse_part, BH, a.Nq, a.Nk, split_len, sl2);
    } else {
        fa_splitkv_partial_lg<T, D, NQ, lanes_per_key(D, NQ), CAUSAL><<<grid, kWarpsSK * 32, 0, a.stream>>>(
            static_cast<const T *>(a.q), static_cast<const T *>(a.k), static_cast<const T *>(a.v), a.o_part,
            a.lse_part, BH, a.Nq, a.Nk, split_len, sl2);
    }
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

int splitkv_blocks_per_sm(int d, int Nq) { return d == 64 ? occupancy_d<64>(Nq) : occupancy_d<128>(Nq); }

int launch_splitkv(const SplitKVArgs &a, bool fp16) {
    return fp16 ? launch_sk_t<__half>(a) : launch_sk_t<__nv_bfloat16>(a);
}

}  // namespace fa
