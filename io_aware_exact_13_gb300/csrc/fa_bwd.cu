// fa_bwd.cu -- backward of the exact attention forward, by recomputation.
//
// "IO-aware exact attention", section "Backward recomputation": the forward
// keeps only O and the per-row log-sum-exp; the backward rebuilds each score
// and probability tile from Q, K and lse and accumulates dQ, dK, dV without an
// N x N tensor in device memory. With S = Q K^T and P = exp(scale S - lse),
//     dV = P^T dO,   dP = dO V^T,   dS = P o (dP - D),   D_i = sum_t dO_it O_it,
//     dQ = scale dS K,   dK = scale dS^T Q,
// the gradient of sum(dO o O) (D_i = sum_j P_ij dP_ij because the rows of P
// sum to one).
//
// One CTA owns a 128-key block j of one (b, h) and loops over the 128-row query
// blocks i that can see it (all of them, or i >= j when causal):
//   warp 0      TMA: K_j and V_j once, then Q_i and dO_i through a ring
//   warp 1      MMA issue (warp-uniform loop, lane 0 issues), tcgen05 kind::f16
//   warps 4-7   one thread per key (TMEM lane): P^T and dS^T from S^T, dP^T,
//               lse and D; then one thread per query row: dQ read-out
// Tensor memory (512 columns) per iteration:
//   [0,128)     S^T = K_j Q_i^T  (fp32; then P^T in 16 bit in [0,64), and the
//               dQ columns 0..63 of this block in [64,128))
//   [128,256)   dP^T = V_j dO_i^T (fp32; then dS^T in 16 bit in [128,192), and
//               dQ columns 64..127 in [192,256) when d = 128)
//   [256,256+d) dV_j accumulator,  [256+d,256+2d) dK_j accumulator
// dV_j += P^T dO_i and dK_j += dS^T Q_i take A from tensor memory; dQ_i = dS K_j
// takes A = dS from shared memory, written by the key threads with the query
// index contiguous (an M-major operand). The dQ block partials of all key
// blocks are added with fp32 vector reductions into a workspace and converted
// to the output type by a last kernel.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fa_bwd.cuh"
#include "fa_launch.cuh"

namespace fa {
namespace {

constexpr int kBwdThreads = 256;
constexpr int kBlk = kBwdRows;  // keys per CTA block and query rows per iteration

template <typename T, int D>
struct BwdCfg {
    static constexpr int NCH = D * 2 / 128;          // 128-byte swizzle chunks per row
    static constexpr int CHUNK = 128 * 128;          // 128 rows x 128 bytes
    static constexpr int TILE = NCH * CHUNK;         // one 128-row tile of Q, K, V or dO
    static constexpr int KSTEPS_D = D * 2 / 32;      // K-steps of 16 over the head dimension
    static constexpr int KSTEPS_R = kBlk / 16;       // K-steps of 16 over 128 rows or keys
    static constexpr int STAGES = (TILE == 32768) ? 2 : 3;
    static constexpr int SMEM_K = 0;
    static constexpr int SMEM_V = TILE;
    static constexpr int SMEM_QD = 2 * TILE;                     // STAGES x (Q_i, dO_i)
    static constexpr int SMEM_DS = SMEM_QD + STAGES * 2 * TILE;  // dS: 2 chunks (queries 0-63, 64-127) x 128 keys
    static constexpr int SMEM_BAR = SMEM_DS + 2 * CHUNK;
    static constexpr int NUM_BARS = 1 + 2 * STAGES + 5;
    static constexpr int SMEM_BYTES = SMEM_BAR + NUM_BARS * 8 + 16 + 1024;
    static constexpr uint32_t FMT = Elem<T>::fmt;
    static constexpr uint32_t ID_ST = make_idesc_ab(FMT, 128, 128, 0, 0);  // S^T, dP^T: A, B K-major
    static constexpr uint32_t ID_ACC = make_idesc_ab(FMT, 128, D, 0, 1);   // dV, dK: A in TMEM, B N-major
    static constexpr uint32_t ID_DQ = make_idesc_ab(FMT, 128, 64, 1, 1);   // dQ: A M-major, B N-major
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(256 + 2 * D <= 512, "tensor memory budget");
};

struct BwdParams {
    const float *lse2;  // [BH][Npad]
    const float *dsum;  // [BH][Npad]
    float *dq_acc;      // [BH][N][d]
    void *dk, *dv;      // [BH][N][d]
    int *status;
    int BH, N, Npad;
    float scale, scale_log2;
    uint64_t timeout_ns;
};

__device__ __forceinline__ bool bwd_wait(uint32_t bar, uint32_t parity, const BwdParams &p) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_suspend(bar, parity, 100000u)) return true;
        if (global_timer_ns() - t0 > p.timeout_ns) {
            atomicExch(p.status, kStatusTimeout);
            return false;
        }
    }
}
__device__ __forceinline__ bool bwd_wait_warp(uint32_t bar, uint32_t parity, const BwdParams &p) {
    return __all_sync(0xffffffffu, bwd_wait(bar, parity, p));
}

template <typename T>
__device__ __forceinline__ uint32_t pk2(float lo, float hi) {
    if constexpr (Elem<T>::fmt == 1) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
}

template <typename T, int D, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const BwdParams p) {
    using C = BwdCfg<T, D>;
    constexpr int ST = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::SMEM_BAR);
    const uint32_t bar_kv = smem_u32(bars);
    auto bar_qd_full = [&](int s) { return smem_u32(bars + 1 + s); };
    auto bar_qd_empty = [&](int s) { return smem_u32(bars + 1 + ST + s); };
    const uint32_t bar_sp_full = smem_u32(bars + 1 + 2 * ST);  // S^T, dP^T in TMEM
    const uint32_t bar_p_full = smem_u32(bars + 2 + 2 * ST);   // P^T, dS^T, dS written (128 arrivals)
    const uint32_t bar_dq_full = smem_u32(bars + 3 + 2 * ST);  // every product of the iteration done
    const uint32_t bar_dq_free = smem_u32(bars + 4 + 2 * ST);  // dQ read out (128 arrivals)
    const uint32_t bar_drain = smem_u32(bars + 5 + 2 * ST);    // all issued MMAs done (exit)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::SMEM_BAR + C::NUM_BARS * 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Block b -> (key block j, head bh); low j first, which in the causal case
    // are the blocks with the most query blocks to visit.
    const int bh = blockIdx.x % p.BH;
    const int j = blockIdx.x / p.BH;
    const int n_qblk = p.Npad / kBlk;
    const int i0 = CAUSAL ? j : 0;  // first query block that sees key block j
    const int n_it = n_qblk - i0;   // >= 1

    if (threadIdx.x == 0) {
        mbar_init(bar_kv, 1);
        for (int s = 0; s < ST; ++s) {
            mbar_init(bar_qd_full(s), 1);
            mbar_init(bar_qd_empty(s), 1);
        }
        mbar_init(bar_sp_full, 1);
        mbar_init(bar_p_full, 128);
        mbar_init(bar_dq_full, 1);
        mbar_init(bar_dq_free, 128);
        mbar_init(bar_drain, 1);
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_last();
            mbar_arrive_expect_tx(bar_kv, 2 * C::TILE);
            for (int c = 0; c < C::NCH; ++c) {
                tma_load_3d(smem_u32(smem + C::SMEM_K + c * C::CHUNK), &tm_k, bar_kv, c * 64, j * kBlk, bh, pol);
                tma_load_3d(smem_u32(smem + C::SMEM_V + c * C::CHUNK), &tm_v, bar_kv, c * 64, j * kBlk, bh, pol);
            }
            int issued = 0;
            for (int it = 0; it < n_it; ++it) {
                const int s = it % ST;
                if (!bwd_wait(bar_qd_empty(s), ((it / ST) & 1u) ^ 1u, p)) break;
                const uint32_t dst = smem_u32(smem + C::SMEM_QD + s * 2 * C::TILE);
                mbar_arrive_expect_tx(bar_qd_full(s), 2 * C::TILE);
                const int row0 = (i0 + it) * kBlk;
                for (int c = 0; c < C::NCH; ++c) {
                    tma_load_3d(dst + c * C::CHUNK, &tm_q, bar_qd_full(s), c * 64, row0, bh, pol);
                    tma_load_3d(dst + C::TILE + c * C::CHUNK, &tm_do, bar_qd_full(s), c * 64, row0, bh, pol);
                }
                issued = it + 1;
            }
            // Before the CTA may exit, every copy into its shared memory must have
            // landed (they all have on the normal path; this matters after a timeout).
            bwd_wait(bar_kv, 0, p);
            for (int it = issued - ST > 0 ? issued - ST : 0; it < issued; ++it)
                bwd_wait(bar_qd_full(it % ST), (it / ST) & 1u, p);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        const uint32_t issue = lane == 0 ? 1u : 0u;
        const uint64_t k_km = smem_desc_sw128(smem_u32(smem + C::SMEM_K), 16, 1024);         // K_j as A, K-major
        const uint64_t v_km = smem_desc_sw128(smem_u32(smem + C::SMEM_V), 16, 1024);         // V_j as A, K-major
        const uint64_t k_mn = smem_desc_sw128(smem_u32(smem + C::SMEM_K), C::CHUNK, 1024);   // K_j as B, N-major
        const uint64_t ds_mn = smem_desc_sw128(smem_u32(smem + C::SMEM_DS), C::CHUNK, 1024); // dS as A, M-major
        bool ok = bwd_wait_warp(bar_kv, 0, p);
        for (int it = 0; ok && it < n_it; ++it) {
            const int s = it % ST;
            ok = bwd_wait_warp(bar_qd_full(s), (it / ST) & 1u, p);
            if (ok && it > 0) ok = bwd_wait_warp(bar_dq_free, (it - 1) & 1u, p);
            if (!ok) break;
            tc_fence_after();
            const uint32_t q_s = smem_u32(smem + C::SMEM_QD + s * 2 * C::TILE);
            const uint64_t q_km = smem_desc_sw128(q_s, 16, 1024);
            const uint64_t do_km = smem_desc_sw128(q_s + C::TILE, 16, 1024);
            const uint64_t q_mn = smem_desc_sw128(q_s, C::CHUNK, 1024);
            const uint64_t do_mn = smem_desc_sw128(q_s + C::TILE, C::CHUNK, 1024);
            // S^T = K_j Q_i^T and dP^T = V_j dO_i^T, contracted over the head dimension
#pragma unroll
            for (int k = 0; k < C::KSTEPS_D; ++k) {
                const uint64_t off = (uint64_t)(((k / 4) * C::CHUNK + (k % 4) * 32) >> 4);
                mma_ss(tmem + 0, k_km + off, q_km + off, C::ID_ST, k > 0 ? 1u : 0u, issue);
                mma_ss(tmem + 128, v_km + off, do_km + off, C::ID_ST, k > 0 ? 1u : 0u, issue);
            }
            tc_commit(bar_sp_full, issue);
            ok = bwd_wait_warp(bar_p_full, it & 1u, p);
            if (!ok) break;
            tc_fence_after();
            // dV_j += P^T dO_i and dK_j += dS^T Q_i, contracted over the 128 query rows
#pragma unroll
            for (int k = 0; k < C::KSTEPS_R; ++k) {
                const uint64_t off = (uint64_t)((k * 2048) >> 4);
                const uint32_t acc = (it > 0 || k > 0) ? 1u : 0u;
                mma_ts(tmem + 256, tmem + 0 + k * 8, do_mn + off, C::ID_ACC, acc, issue);
                mma_ts(tmem + 256 + D, tmem + 128 + k * 8, q_mn + off, C::ID_ACC, acc, issue);
            }
            // dQ_i = dS K_j, contracted over the 128 keys, 64 head columns at a time
#pragma unroll
            for (int h = 0; h < D / 64; ++h)
#pragma unroll
                for (int k = 0; k < C::KSTEPS_R; ++k) {
                    const uint64_t off = (uint64_t)((k * 2048) >> 4);
                    mma_ss(tmem + (h == 0 ? 64 : 192), ds_mn + off, k_mn + (uint64_t)((h * C::CHUNK) >> 4) + off,
                           C::ID_DQ, k > 0 ? 1u : 0u, issue);
                }
            tc_commit(bar_dq_full, issue);
            tc_commit(bar_qd_empty(s), issue);
        }
        // Every MMA this warp issued is complete before tensor memory is freed.
        tc_commit(bar_drain, issue);
        bwd_wait_warp(bar_drain, 0, p);
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- gradient warps
        const int r = threadIdx.x - 128;  // TMEM lane: key r of block j, later query row r of block i
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int key = j * kBlk + r;
        const bool key_ok = key < p.N;
        const uint32_t ds_row = smem_u32(smem + C::SMEM_DS) + r * 128;
        const float *lse2_bh = p.lse2 + (size_t)bh * p.Npad;
        const float *dsum_bh = p.dsum + (size_t)bh * p.Npad;
        bool ok = true;
        for (int it = 0; ok && it < n_it; ++it) {
            const int row0 = (i0 + it) * kBlk;
            ok = bwd_wait_warp(bar_sp_full, it & 1u, p);
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 32) {  // 32 query rows (TMEM columns) at a time
                float4 l4[8], d4[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {  // same address across the warp: broadcast loads
                    l4[u] = ld_global_nc_v4(lse2_bh + row0 + c0 + 4 * u);
                    d4[u] = ld_global_nc_v4(dsum_bh + row0 + c0 + 4 * u);
                }
                uint32_t sv[32], dpv[32];
                tmem_ld32x2_wait(tmem + lane_base + c0, sv, tmem + lane_base + 128 + c0, dpv);
                const float *lf = reinterpret_cast<const float *>(l4);
                const float *df = reinterpret_cast<const float *>(d4);
                uint32_t pp[16], dsp[16];
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    float pr[2], dsr[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        bool vis = key_ok;
                        if (CAUSAL) vis = vis && (key <= row0 + c0 + c + u);
                        const float x = fmaf(__uint_as_float(sv[c + u]), p.scale_log2, -lf[c + u]);
                        const float pe = vis ? ex2_approx(x) : 0.0f;
                        pr[u] = pe;
                        dsr[u] = pe * (__uint_as_float(dpv[c + u]) - df[c + u]);
                    }
                    pp[c / 2] = pk2<T>(pr[0], pr[1]);
                    dsp[c / 2] = pk2<T>(dsr[0], dsr[1]);
                }
                // P^T and dS^T overwrite columns this thread has already read.
                tmem_st16(tmem + lane_base + 0 + c0 / 2, pp);
                tmem_st16(tmem + lane_base + 128 + c0 / 2, dsp);
                // dS row of key r: queries c0..c0+31 = 64 bytes of chunk c0/64, 128-byte swizzle
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t unit = (uint32_t)(((c0 % 64) / 8 + u) ^ (r & 7));
                    st_shared_v4(ds_row + (c0 / 64) * C::CHUNK + unit * 16, dsp[4 * u], dsp[4 * u + 1],
                                 dsp[4 * u + 2], dsp[4 * u + 3]);
                }
            }
            tmem_wait_st();
            fence_proxy_async_smem();  // dS is read by the tensor core (async proxy)
            tc_fence_before();
            mbar_arrive(bar_p_full);
            // dQ_i rows (TMEM lane = query row r): scale and add into the fp32 accumulator
            ok = bwd_wait_warp(bar_dq_full, it & 1u, p);
            if (!ok) break;
            tc_fence_after();
            const int row = row0 + r;
            float *dq_row = p.dq_acc + ((size_t)bh * p.N + (size_t)(row < p.N ? row : 0)) * D;
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                uint32_t qa[32], qb[32];
                const uint32_t col = h == 0 ? 64u : 192u;
                tmem_ld32x2_wait(tmem + lane_base + col, qa, tmem + lane_base + col + 32, qb);
                if (row < p.N) {
#pragma unroll
                    for (int c = 0; c < 32; c += 4) {
                        red_add_v4(dq_row + h * 64 + c, __uint_as_float(qa[c]) * p.scale,
                                   __uint_as_float(qa[c + 1]) * p.scale, __uint_as_float(qa[c + 2]) * p.scale,
                                   __uint_as_float(qa[c + 3]) * p.scale);
                        red_add_v4(dq_row + h * 64 + 32 + c, __uint_as_float(qb[c]) * p.scale,
                                   __uint_as_float(qb[c + 1]) * p.scale, __uint_as_float(qb[c + 2]) * p.scale,
                                   __uint_as_float(qb[c + 3]) * p.scale);
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(bar_dq_free);
        }
        // ---------------------------------------------------------------- dK_j, dV_j
        // The last dq_full completion covers every dV and dK product (a commit
        // tracks all earlier MMAs of the issuing thread).
        if (ok) {
            tc_fence_after();
            T *dv_row = reinterpret_cast<T *>(p.dv) + ((size_t)bh * p.N + (size_t)(key_ok ? key : 0)) * D;
            T *dk_row = reinterpret_cast<T *>(p.dk) + ((size_t)bh * p.N + (size_t)(key_ok ? key : 0)) * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t a[32], b[32];
                tmem_ld32x2_wait(tmem + lane_base + 256 + c0, a, tmem + lane_base + 256 + D + c0, b);
                if (key_ok) {
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        st_global_v4(dv_row + c0 + c, pk2<T>(__uint_as_float(a[c]), __uint_as_float(a[c + 1])),
                                     pk2<T>(__uint_as_float(a[c + 2]), __uint_as_float(a[c + 3])),
                                     pk2<T>(__uint_as_float(a[c + 4]), __uint_as_float(a[c + 5])),
                                     pk2<T>(__uint_as_float(a[c + 6]), __uint_as_float(a[c + 7])));
                        st_global_v4(dk_row + c0 + c,
                                     pk2<T>(__uint_as_float(b[c]) * p.scale, __uint_as_float(b[c + 1]) * p.scale),
                                     pk2<T>(__uint_as_float(b[c + 2]) * p.scale, __uint_as_float(b[c + 3]) * p.scale),
                                     pk2<T>(__uint_as_float(b[c + 4]) * p.scale, __uint_as_float(b[c + 5]) * p.scale),
                                     pk2<T>(__uint_as_float(b[c + 6]) * p.scale, __uint_as_float(b[c + 7]) * p.scale));
                    }
                }
            }
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Row statistics for the backward, one warp per padded row:
//   dsum = sum_t dO_t O_t (0 past N), lse2 = lse * log2(e) (+inf past N),
// and the row's dQ accumulator is zeroed.
template <typename T, int D>
__global__ void __launch_bounds__(256) fa_bwd_pre(const T *__restrict__ out, const T *__restrict__ dout,
                                                  const float *__restrict__ lse, float *__restrict__ lse2,
                                                  float *__restrict__ dsum, float *__restrict__ dq_acc, int BH,
                                                  int N, int Npad) {
    const int64_t prow = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (prow >= (int64_t)BH * Npad) return;
    const int64_t bh = prow / Npad;
    const int i = (int)(prow - bh * Npad);
    if (i >= N) {
        if (lane == 0) {
            lse2[prow] = INFINITY;
            dsum[prow] = 0.0f;
        }
        return;
    }
    const int64_t row = bh * N + i;
    float acc = 0.f;
#pragma unroll
    for (int e = lane; e < D; e += 32) {
        float o, g;
        if constexpr (Elem<T>::fmt == 1) {
            o = __bfloat162float(out[row * D + e]);
            g = __bfloat162float(dout[row * D + e]);
        } else {
            o = __half2float(out[row * D + e]);
            g = __half2float(dout[row * D + e]);
        }
        acc = fmaf(o, g, acc);
        dq_acc[row * D + e] = 0.f;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) {
        dsum[prow] = acc;
        lse2[prow] = lse[row] * 1.4426950408889634f;
    }
}

template <typename T>
__global__ void __launch_bounds__(256) fa_bwd_post(const float *__restrict__ dq_acc, T *__restrict__ dq, size_t n4) {
    const size_t i = (size_t)blockIdx.x * 256 + threadIdx.x;
    if (i >= n4) return;
    const float4 v = reinterpret_cast<const float4 *>(dq_acc)[i];
    uint2 o;
    o.x = pk2<T>(v.x, v.y);
    o.y = pk2<T>(v.z, v.w);
    reinterpret_cast<uint2 *>(dq)[i] = o;
}

template <typename T, int D, bool CAUSAL>
int launch_bwd_variant(const BwdArgs &a) {
    using C = BwdCfg<T, D>;
    auto kern = fa_bwd_kernel<T, D, CAUSAL>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) != cudaSuccess)
        return -5;
    const int BH = a.B * a.H;
    const int Npad = static_cast<int>(bwd_padded_rows(a.N));
    const int64_t prows = static_cast<int64_t>(BH) * Npad;
    fa_bwd_pre<T, D><<<static_cast<unsigned>((prows + 7) / 8), 256, 0, a.stream>>>(
        static_cast<const T *>(a.out), static_cast<const T *>(a.dout), a.lse, a.lse2, a.dsum, a.dq_acc, BH, a.N,
        Npad);
    if (cudaGetLastError() != cudaSuccess) return -5;
    CUtensorMap tq, tk, tv, tdo;
    if (!encode_rows_map(&tq, Elem<T>::tma, 2, a.q, D, a.N, BH, kBlk)) return -5;
    if (!encode_rows_map(&tk, Elem<T>::tma, 2, a.k, D, a.N, BH, kBlk)) return -5;
    if (!encode_rows_map(&tv, Elem<T>::tma, 2, a.v, D, a.N, BH, kBlk)) return -5;
    if (!encode_rows_map(&tdo, Elem<T>::tma, 2, a.dout, D, a.N, BH, kBlk)) return -5;
    BwdParams p;
    p.lse2 = a.lse2;
    p.dsum = a.dsum;
    p.dq_acc = a.dq_acc;
    p.dk = a.dk;
    p.dv = a.dv;
    p.status = a.status;
    p.BH = BH;
    p.N = a.N;
    p.Npad = Npad;
    p.scale = a.scale;
    p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
    p.timeout_ns = a.timeout_ns;
    const int64_t grid = static_cast<int64_t>(BH) * (Npad / kBlk);
    kern<<<static_cast<unsigned>(grid), kBwdThreads, C::SMEM_BYTES, a.stream>>>(tq, tk, tv, tdo, p);
    if (cudaGetLastError() != cudaSuccess) return -5;
    const size_t n4 = static_cast<size_t>(BH) * a.N * D / 4;
    fa_bwd_post<T><<<static_cast<unsigned>((n4 + 255) / 256), 256, 0, a.stream>>>(a.dq_acc, static_cast<T *>(a.dq),
                                                                                   n4);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

template <typename T>
int launch_bwd_t(const BwdArgs &a) {
    if (a.d == 128) return a.causal ? launch_bwd_variant<T, 128, true>(a) : launch_bwd_variant<T, 128, false>(a);
    if (a.d == 64) return a.causal ? launch_bwd_variant<T, 64, true>(a) : launch_bwd_variant<T, 64, false>(a);
    return -4;
}

}  // namespace

int launch_bwd(const BwdArgs &a, bool fp16) { return fp16 ? launch_bwd_t<__half>(a) : launch_bwd_t<__nv_bfloat16>(a); }

}  // namespace fa
