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
// Decoding reads every key and value once and does about Nq flop per byte, so
// the kernels are bound by HBM bandwidth. With one query row a warp reads one
// 128- or 256-byte K row per load instruction (each lane d/32 elements), several
// rows in flight per lane, on the CUDA cores; with 2..16 rows the dot products
// and P V run on 16-row warp-level MMA tiles (fa_splitkv_partial_mma below).
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "fa_splitkv.cuh"
#include "pdl.cuh"
#include "ptx.cuh"
#include "warp_mma.cuh"

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

template <typename T>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
    if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
}

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
    grid_launch_dependents();
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

// Several query rows per head (2 <= Nq <= 16), on the tensor cores with 16-row
// warp-level MMA tiles (the rows padded to 16). A warp streams its 16-key chunks
// of K and V into shared memory with asynchronous copies (two stages, 16-byte
// units swizzled by the row so that ldmatrix reads are conflict-free), forms
// S = Q K^T from K fragments (ldmatrix) and O += P V from V fragments
// (ldmatrix.trans), keeping P in registers: the S accumulator fragment is the A
// fragment of the P V product. Per row it keeps (m, l) with the forward's lazy
// rescaling (the reference maximum moves only when a score exceeds it by more
// than kTauSK, log2 units); the four warps merge by the block-summary rule.
constexpr float kTauSK = 8.0f;
constexpr int kChunkSK = 16;  // keys per warp step

template <int D>
constexpr int splitkv_mma_smem_bytes() {
    return kWarpsSK * 2 * 2 * kChunkSK * D * 2;  // warps x stages x (K, V) x 16 keys x D x 2 bytes
}

template <typename T, int D, bool CAUSAL>
__global__ void __launch_bounds__(kWarpsSK * 32) fa_splitkv_partial_mma(
    const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v, float *__restrict__ o_part,
    float *__restrict__ lse_part, int BH, int Nq, int Nk, int split_len, float scale_log2) {
    constexpr bool BF16 = std::is_same<T, __nv_bfloat16>::value;
    constexpr int NCH = D / 8;               // 16-byte units per row
    constexpr int ROWB = D * 2;              // bytes per row
    constexpr int TILE = kChunkSK * ROWB;    // one 16-key K or V tile
    constexpr int KS = D / 16;               // k-steps of S over the head dimension
    constexpr int NT = D / 8;                // n-tiles of O over the head dimension
    extern __shared__ __align__(128) uint8_t sm_raw[];
    grid_launch_dependents();
    const int split = blockIdx.x, bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int mi = lane >> 3, ri = lane & 7;  // ldmatrix: matrix and row this lane addresses
    const int k0 = split * split_len, k1 = min(Nk, k0 + split_len);
    const T *qb = q + (size_t)bh * Nq * D;
    const T *kb = k + (size_t)bh * Nk * D;
    const T *vb = v + (size_t)bh * Nk * D;
    const uint32_t wbase = smem_u32(sm_raw) + warp * 4 * TILE;  // [stage][K, V]

    uint32_t qa[KS][4];  // Q as A fragments; rows >= Nq are zero
#pragma unroll
    for (int st = 0; st < KS; ++st)
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const int row = g + (h & 1) * 8, col = st * 16 + 2 * c + (h >> 1) * 8;
            qa[st][h] = row < Nq ? __ldg(reinterpret_cast<const uint32_t *>(qb + (size_t)row * D + col)) : 0u;
        }
    float o[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};  // rows g and g + 8
    const int shift = Nk - Nq;                                 // causal: row i sees keys j <= i + shift
    const int n_chunks = (k1 - k0 + kChunkSK - 1) / kChunkSK;

    auto issue = [&](int chunk, int stage) {  // copy a 16-key chunk of K and V, zero past k1
        const int key0 = k0 + chunk * kChunkSK;
        const uint32_t kt = wbase + stage * 2 * TILE, vt = kt + TILE;
#pragma unroll
        for (int idx = lane; idx < kChunkSK * NCH; idx += 32) {
            const int r = idx / NCH, u = idx % NCH;
            const int key = key0 + r;
            const bool ok = key < k1;
            const size_t off = (size_t)(ok ? key : k0) * D + u * 8;
            const uint32_t so = r * ROWB + ((u ^ (r & 7)) * 16);
            cp_async16(kt + so, kb + off, ok ? 16u : 0u);
            cp_async16(vt + so, vb + off, ok ? 16u : 0u);
        }
    };

    int chunk = warp;
    if (chunk < n_chunks) issue(chunk, 0);
    cp_async_commit();
    for (int it = 0; chunk < n_chunks; ++it, chunk += kWarpsSK) {
        const int stage = it & 1;
        if (chunk + kWarpsSK < n_chunks) issue(chunk + kWarpsSK, stage ^ 1);
        cp_async_commit();
        cp_async_wait<1>();  // this chunk has landed
        __syncwarp();
        const uint32_t kt = wbase + stage * 2 * TILE, vt = kt + TILE;
        // S (16 rows x 16 keys) = Q K^T: B fragments of both 8-key tiles per k-step
        float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int st = 0; st < KS; ++st) {
            const int key = (mi >> 1) * 8 + ri, u = 2 * st + (mi & 1);
            uint32_t b00, b01, b10, b11;
            ldsm_x4(kt + key * ROWB + ((u ^ (key & 7)) * 16), b00, b01, b10, b11);
            mma16816<BF16>(sacc[0], qa[st], b00, b01);
            mma16816<BF16>(sacc[1], qa[st], b10, b11);
        }
        // base-2 scores with the key-range and causal masks
        const int key0 = k0 + chunk * kChunkSK;
        float x[2][4];
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = key0 + t * 8 + 2 * c + (e & 1);
                const int row = g + (e >> 1) * 8;
                const bool vis = key < k1 && (!CAUSAL || key <= row + shift);
                x[t][e] = vis ? sacc[t][e] * scale_log2 : -INFINITY;
            }
        // row maxima (a row's 16 scores sit in the 4 lanes of a quad), lazy rescale
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            float mb = fmaxf(fmaxf(x[0][2 * hr], x[0][2 * hr + 1]), fmaxf(x[1][2 * hr], x[1][2 * hr + 1]));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
            mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
            if (mb > m[hr] + kTauSK) {
                const float corr = ex2_approx(m[hr] - mb);  // 0 when m was -inf
                l[hr] *= corr;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    o[nt][2 * hr] *= corr;
                    o[nt][2 * hr + 1] *= corr;
                }
                m[hr] = mb;
            }
        }
        float pv[2][4];
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float mr = m[e >> 1];
                pv[t][e] = mr == -INFINITY ? 0.f : ex2_approx(x[t][e] - mr);
            }
        l[0] += (pv[0][0] + pv[0][1]) + (pv[1][0] + pv[1][1]);
        l[1] += (pv[0][2] + pv[0][3]) + (pv[1][2] + pv[1][3]);
        const uint32_t pa[4] = {pack16<T>(pv[0][0], pv[0][1]), pack16<T>(pv[0][2], pv[0][3]),
                                pack16<T>(pv[1][0], pv[1][1]), pack16<T>(pv[1][2], pv[1][3])};
        // O += P V: V fragments (keys x head columns) by transposing loads, two n-tiles per load
#pragma unroll
        for (int nt = 0; nt < NT; nt += 2) {
            const int key = (mi & 1) * 8 + ri, u = nt + (mi >> 1);
            uint32_t b0a, b1a, b0b, b1b;
            ldsm_x4_trans(vt + key * ROWB + ((u ^ (key & 7)) * 16), b0a, b1a, b0b, b1b);
            mma16816<BF16>(o[nt], pa, b0a, b1a);
            mma16816<BF16>(o[nt + 1], pa, b0b, b1b);
        }
        __syncwarp();  // the stage is refilled two chunks later
    }
    cp_async_wait<0>();
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 1);
        l[hr] += __shfl_xor_sync(0xffffffffu, l[hr], 2);
    }
    // merge the four warps' summaries (the staging buffers are free once every warp is here)
    __syncthreads();
    float *sm_m = reinterpret_cast<float *>(sm_raw);  // [warp][16]
    float *sm_l = sm_m + kWarpsSK * 16;                // [warp][16]
    float *sm_o = sm_l + kWarpsSK * 16;                // [warp][16][D]
    if (c == 0) {
        sm_m[warp * 16 + g] = m[0];
        sm_m[warp * 16 + g + 8] = m[1];
        sm_l[warp * 16 + g] = l[0];
        sm_l[warp * 16 + g + 8] = l[1];
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        float *r0 = sm_o + ((size_t)warp * 16 + g) * D + nt * 8 + 2 * c;
        r0[0] = o[nt][0];
        r0[1] = o[nt][1];
        r0[8 * D] = o[nt][2];
        r0[8 * D + 1] = o[nt][3];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < Nq * D; idx += kWarpsSK * 32) {
        const int i = idx / D, e = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarpsSK; ++w) M = fmaxf(M, sm_m[w * 16 + i]);
        float Lsum = 0.f, A = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarpsSK; ++w) {
                const float f = ex2_approx(sm_m[w * 16 + i] - M);  // 0 for a warp that saw nothing
                Lsum += f * sm_l[w * 16 + i];
                A += f * sm_o[((size_t)w * 16 + i) * D + e];
            }
        }
        const size_t row = ((size_t)split * BH + bh) * Nq + i;
        o_part[row * D + e] = Lsum > 0.f ? A / Lsum : 0.f;
        if (e == 0) lse_part[row] = Lsum > 0.f ? (M + lg2_approx(Lsum)) * 0.6931471805599453f : -INFINITY;
    }
}

// One CTA of D threads per (b*h, query row): merge the n_splits summaries.
// Launched as a programmatic dependent of the partial kernel: its CTAs may be
// scheduled while the partial kernel drains and wait here for all its results.
template <typename T, int D>
__global__ void __launch_bounds__(D) fa_splitkv_combine(const float *__restrict__ o_part,
                                                       const float *__restrict__ lse_part, T *__restrict__ out,
                                                       float *__restrict__ lse, int rows, int n_splits) {
    grid_dependency_wait();
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

template <typename T, int D, int NQ>
int occupancy_d_nq() {
    int nb = 0;
    cudaError_t e;
    if constexpr (NQ == 1) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, fa_splitkv_partial<T, D, NQ, false>, kWarpsSK * 32,
                                                          0);
    } else {
        auto kern = fa_splitkv_partial_mma<T, D, false>;
        constexpr int smem = splitkv_mma_smem_bytes<D>();
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, kWarpsSK * 32, smem);
    }
    return e == cudaSuccess && nb > 0 ? nb : 1;
}

template <int D>
int occupancy_d(int Nq) {
    using T = __nv_bfloat16;
    return Nq <= 1 ? occupancy_d_nq<T, D, 1>() : occupancy_d_nq<T, D, 16>();
}

template <typename T, int D, int NQ, bool CAUSAL>
int launch_sk(const SplitKVArgs &a) {
    const int BH = a.B * a.H;
    const int split_len = (a.Nk + a.n_splits - 1) / a.n_splits;
    const float sl2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
    dim3 grid(a.n_splits, BH);
    if constexpr (NQ == 1) {  // one query row: a warp per key row, CUDA cores
        fa_splitkv_partial<T, D, NQ, CAUSAL><<<grid, kWarpsSK * 32, 0, a.stream>>>(
            static_cast<const T *>(a.q), static_cast<const T *>(a.k), static_cast<const T *>(a.v), a.o_part,
            a.lse_part, BH, a.Nq, a.Nk, split_len, sl2);
    } else {  // 2..16 rows: 16-row tensor-core tiles
        auto kern = fa_splitkv_partial_mma<T, D, CAUSAL>;
        constexpr int smem = splitkv_mma_smem_bytes<D>();
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return -5;
        kern<<<grid, kWarpsSK * 32, smem, a.stream>>>(static_cast<const T *>(a.q), static_cast<const T *>(a.k),
                                                      static_cast<const T *>(a.v), a.o_part, a.lse_part, BH, a.Nq,
                                                      a.Nk, split_len, sl2);
    }
    if (cudaGetLastError() != cudaSuccess) return -5;
    // programmatic dependent launch: the combine's launch overlaps the partial kernel's tail
    if (launch_dependent(fa_splitkv_combine<T, D>, dim3(BH * a.Nq), dim3(D), 0, a.stream,
                         static_cast<const float *>(a.o_part), static_cast<const float *>(a.lse_part),
                         static_cast<T *>(a.out), a.lse, BH * a.Nq, a.n_splits) != cudaSuccess)
        return -5;
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

template <typename T, int D, bool CAUSAL>
int launch_sk_nq(const SplitKVArgs &a) {
    if (a.Nq <= 1) return launch_sk<T, D, 1, CAUSAL>(a);
    return launch_sk<T, D, 16, CAUSAL>(a);  // the tensor-core kernel pads the rows to 16
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
