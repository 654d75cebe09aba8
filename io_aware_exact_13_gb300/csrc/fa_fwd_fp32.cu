// fa_fwd_fp32.cu -- exact tiled attention forward for fp32 inputs, in fp32 on the
// CUDA cores.
//
// Same method as the tensor-core kernel ("FlashAttention: Exact Attention as an
// IO-Aware Streaming Computation", sections "Core idea" and "Mathematical
// structure"): a block keeps 32 query rows and their running (m, l, a) on chip
// while 32-key K/V tiles stream through shared memory; each score tile is
// folded into the running state and dropped. Arithmetic is plain fp32 FFMA:
// tcgen05 kind::tf32 would round Q, K, P and V to TF32, and it does not accept
// the value tile in its stored (N-major) order, so fp32 inputs take this kernel.
//
// Layout of the work: 128 threads = 32 rows x 4 threads. The 4 threads of a row
// split the head dimension in interleaved float4 chunks (chunk 4c + quad), so a
// warp reads a K or V row from shared memory without bank conflicts; the partial
// dot products are summed with two shuffles. The next 32-key K/V tile is loaded
// into registers while the current one is used.
#include <cuda_runtime.h>
#include <stdint.h>

#include "fa_launch.cuh"

namespace fa {
namespace {

constexpr int kRows = 32;  // query rows per block
constexpr int kKeys = 32;  // keys per K/V tile
constexpr int kThreadsF32 = 128;

template <int D, bool CAUSAL, bool MASK>
__global__ void __launch_bounds__(kThreadsF32) fa_fwd_fp32_kernel(const float *__restrict__ q,
                                                                  const float *__restrict__ k,
                                                                  const float *__restrict__ v,
                                                                  const float *__restrict__ mask,
                                                                  float *__restrict__ out, float *__restrict__ lse,
                                                                  int H, int N, float scale_log2) {
    constexpr int C4 = D / 16;  // float4 chunks per thread
    __shared__ float4 sk[kKeys][D / 4];
    __shared__ float4 sv[kKeys][D / 4];
    // launched as a programmatic dependent of the work ahead: nothing in global memory is touched before it is
    // complete; the next forward may be scheduled as this grid's blocks finish
    grid_launch_dependents();
    grid_dependency_wait();
    const int bh = blockIdx.y;
    const int b = bh / H;
    const int r0 = blockIdx.x * kRows;
    const int tid = threadIdx.x;
    const int quad = tid & 3;
    const int row = r0 + (tid >> 2);
    const bool row_ok = row < N;
    const size_t head = (size_t)bh * N * D;

    float4 qr[C4], o[C4];
#pragma unroll
    for (int c = 0; c < C4; ++c) {
        qr[c] = row_ok ? reinterpret_cast<const float4 *>(q + head + (size_t)row * D)[4 * c + quad]
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        o[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float m_run = -INFINITY, l = 0.0f;
    const int key_end = CAUSAL ? min(N, r0 + kRows) : N;
    // the next K/V tile is loaded into registers while this one is used (PF float4 of each per thread)
    constexpr int PF = kKeys * D / 4 / kThreadsF32;
    float4 pk[PF], pv[PF];
    auto fetch = [&](int j0) {
#pragma unroll
        for (int u = 0; u < PF; ++u) {
            const int i = tid + u * kThreadsF32;
            const int kr = i / (D / 4), kc = i % (D / 4);
            const bool in = j0 + kr < N;
            pk[u] = in ? reinterpret_cast<const float4 *>(k + head + (size_t)(j0 + kr) * D)[kc]
                       : make_float4(0.f, 0.f, 0.f, 0.f);
            pv[u] = in ? reinterpret_cast<const float4 *>(v + head + (size_t)(j0 + kr) * D)[kc]
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    fetch(0);
    for (int j0 = 0; j0 < key_end; j0 += kKeys) {
        __syncthreads();  // the last tile's readers are done
#pragma unroll
        for (int u = 0; u < PF; ++u) {
            const int i = tid + u * kThreadsF32;
            sk[i / (D / 4)][i % (D / 4)] = pk[u];
            sv[i / (D / 4)][i % (D / 4)] = pv[u];
        }
        __syncthreads();
        if (j0 + kKeys < key_end) fetch(j0 + kKeys);
        float x[kKeys];
#pragma unroll
        for (int j = 0; j < kKeys; ++j) {
            float part = 0.f;
#pragma unroll
            for (int c = 0; c < C4; ++c) {
                const float4 kk = sk[j][4 * c + quad];
                part = fmaf(qr[c].x, kk.x, part);
                part = fmaf(qr[c].y, kk.y, part);
                part = fmaf(qr[c].z, kk.z, part);
                part = fmaf(qr[c].w, kk.w, part);
            }
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            const int key = j0 + j;
            float xv = part * scale_log2;
            if (MASK && row_ok && key < N) xv = fmaf(mask[((size_t)b * N + row) * N + key], 1.4426950408889634f, xv);
            const bool allowed = key < N && (!CAUSAL || key <= row);
            x[j] = allowed ? xv : -INFINITY;
        }
        float mb = x[0];
#pragma unroll
        for (int j = 1; j < kKeys; ++j) mb = fmaxf(mb, x[j]);
        const float m_new = fmaxf(m_run, mb);
        if (m_new == -INFINITY) continue;  // nothing visible yet for this row
        const float alpha = ex2_approx(m_run - m_new);  // 0 when m_run = -inf
        m_run = m_new;
        l *= alpha;
#pragma unroll
        for (int c = 0; c < C4; ++c) {
            o[c].x *= alpha;
            o[c].y *= alpha;
            o[c].z *= alpha;
            o[c].w *= alpha;
        }
#pragma unroll
        for (int j = 0; j < kKeys; ++j) {
            const float pj = ex2_approx(x[j] - m_new);
            l += pj;
#pragma unroll
            for (int c = 0; c < C4; ++c) {
                const float4 vv = sv[j][4 * c + quad];
                o[c].x = fmaf(pj, vv.x, o[c].x);
                o[c].y = fmaf(pj, vv.y, o[c].y);
                o[c].z = fmaf(pj, vv.z, o[c].z);
                o[c].w = fmaf(pj, vv.w, o[c].w);
            }
        }
    }
    if (!row_ok) return;
    const float inv = l > 0.f ? 1.0f / l : 0.f;
    float4 *orow = reinterpret_cast<float4 *>(out + head + (size_t)row * D);
#pragma unroll
    for (int c = 0; c < C4; ++c)
        orow[4 * c + quad] = make_float4(o[c].x * inv, o[c].y * inv, o[c].z * inv, o[c].w * inv);
    if (quad == 0) lse[(size_t)bh * N + row] = l > 0.f ? (m_run + lg2_approx(l)) * 0.6931471805599453f : -INFINITY;
}

template <int D, bool CAUSAL, bool MASK>
int launch_fp32(const LaunchArgs &a) {
    dim3 grid((a.N + kRows - 1) / kRows, a.B * a.H);
    const float sl2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
    return launch_dependent(fa_fwd_fp32_kernel<D, CAUSAL, MASK>, grid, dim3(kThreadsF32), 0, a.stream,
                            static_cast<const float *>(a.q), static_cast<const float *>(a.k),
                            static_cast<const float *>(a.v), a.mask, static_cast<float *>(a.out), a.lse, a.H, a.N,
                            sl2) == cudaSuccess
               ? 0
               : -5;
}

template <int D>
int launch_fp32_d(const LaunchArgs &a) {
    if (a.causal) return a.mask ? launch_fp32<D, true, true>(a) : launch_fp32<D, true, false>(a);
    return a.mask ? launch_fp32<D, false, true>(a) : launch_fp32<D, false, false>(a);
}

}  // namespace

int launch_fwd_fp32(const LaunchArgs &a) {
    if ((int64_t)a.B * a.H > 65535) return -3;  // grid.y limit
    if (a.d == 128) return launch_fp32_d<128>(a);
    if (a.d == 64) return launch_fp32_d<64>(a);
    return -4;
}

}  // namespace fa
