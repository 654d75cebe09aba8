// fa_fwd_kernel.cuh -- exact tiled attention forward for sm_103a.
//
// What it computes ("FlashAttention: Exact Attention as an IO-Aware Streaming
// Computation", sections "Problem setting", "Core idea" and "Mathematical
// structure"; "IO-aware exact attention", section "One tiled forward-pass
// iteration"): for every query row i,
//     o_i = sum_j exp(s_ij) v_j / sum_j exp(s_ij),  s_ij = scale <q_i, k_j> + M_ij,
// by keeping a query tile on chip with its running maximum m, denominator l and
// unnormalised accumulator a, streaming key/value tiles past it, and discarding
// each score tile once it has been folded into (m, l, a). Only O and the
// per-row log-sum-exp reach global memory.
//
// GB300 mapping (one persistent CTA per SM, 12 warps):
//   warps 0-3   softmax + epilogue for query tile 0 (thread r owns row r = TMEM lane r)
//   warps 4-7   softmax + epilogue for query tile 1
//   warp  8     TMA producer: Q tiles once per work item, then a K/V ring
//   warp  9     MMA issuer: S = Q K^T and O += P V on tcgen05, fp32
//               accumulators in tensor memory (TMEM); the warp runs the loop,
//               lane 0 issues
//   warps 10-11 idle
// TMEM (512 columns x 128 lanes x 32 bit):
//   S_t  columns [128 t, 128 t + 128)       P_t aliases the start of S_t
//   O_t  columns [256 + 128 t, 256 + 128 t + D)
// A work item is (batch*head, 256 query rows) = two 128-row query tiles that
// share every K/V tile; items are visited longest-first (causal rows near the
// end of the sequence see the most keys).
//
// Scores are handled in the base-2 domain: x = s * scale * log2(e) (+ M * log2(e)),
// p = 2^(x - m_ref). The reference maximum m_ref is only moved when the block
// maximum exceeds it by more than TAU (= 8, a factor 256), in which case l and
// the accumulator O are rescaled by 2^(m_ref_old - m_ref_new) before the next
// P V product; otherwise p <= 2^TAU and the sums stay exact relative to the
// same m_ref (the merge rule of the glossary page "FlashAttention", section
// "Why a tile can be discarded"). A row with no visible key so far keeps
// m_ref = -inf and subtracts 0 instead, which avoids (-inf) - (-inf).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "ptx.cuh"

namespace fa {

constexpr int kBQ = 128;           // rows per query tile (= TMEM lanes)
constexpr int kBK = 128;           // keys per K/V tile
constexpr int kRowsPerItem = 256;  // two query tiles per work item
constexpr int kThreads = 384;
constexpr float kTau = 8.0f;       // lazy-rescale threshold, log2 units
constexpr int kStatusTimeout = -6; // value written to the device status word

template <typename T>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
    static constexpr uint32_t fmt = 1;
    static constexpr CUtensorMapDataType tma = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
};
template <>
struct Elem<__half> {
    static constexpr uint32_t fmt = 0;
    static constexpr CUtensorMapDataType tma = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
};

template <typename T, int D>
struct Cfg {
    static constexpr int EB = sizeof(T);
    static constexpr int ROW_BYTES = D * EB;               // one row of Q/K/V
    static constexpr int CHUNK_ELEMS = 128 / EB;           // elements per 128-byte swizzle row
    static constexpr int NCH = ROW_BYTES / 128;            // swizzle chunks per row
    static constexpr int CHUNK_BYTES = 128 * 128;          // 128 rows x 128 bytes
    static constexpr int TILE_BYTES = NCH * CHUNK_BYTES;   // one 128-row tile
    static constexpr int STAGES = (TILE_BYTES <= 16384) ? 8 : 5;
    static constexpr int KSTEPS_S = ROW_BYTES / 32;        // 32 bytes of K per MMA instruction
    static constexpr int P_COLS = 64;                      // TMEM columns holding P (two 16-bit values each)
    static constexpr int KSTEPS_PV = P_COLS / 8;           // 8 TMEM columns of P per MMA instruction
    static constexpr int V_KSTEP_BYTES = (32 / EB) * 128;  // keys per instruction x 128 bytes per key row
    static constexpr uint32_t IDESC_S = make_idesc(Elem<T>::fmt, 128, kBK, 0);
    static constexpr uint32_t IDESC_PV = make_idesc(Elem<T>::fmt, 128, D, 1);
    // shared memory: Q0 Q1 | K/V ring | barriers
    static constexpr int SMEM_Q = 0;
    static constexpr int SMEM_KV = 2 * TILE_BYTES;
    static constexpr int SMEM_BAR = SMEM_KV + STAGES * TILE_BYTES;
    static constexpr int NUM_BARS = 2 + 2 + 2 * STAGES + 2 + 2 + 2 + 1;
    static constexpr int SMEM_BYTES = SMEM_BAR + NUM_BARS * 8 + 16 + 1024;  // + alignment slack
    static_assert(NCH >= 1 && ROW_BYTES % 128 == 0, "row must be a whole number of 128-byte swizzle rows");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct FwdParams {
    void *out;
    float *lse;
    const float *mask;  // [B][N][N] or nullptr
    int *status;        // device status word
    int B, H, N;
    int n_items;        // B * H * ceil(N / 256)
    int n_qblk;         // ceil(N / 256)
    int n_kv;           // ceil(N / 128)
    float scale_log2;   // scale * log2(e)
    uint64_t timeout_ns;
};

// Static schedule: CTA c takes item w*G + c in even waves w and w*G + (G-1-c)
// in odd waves ("snake" order). With items sorted longest-first this balances
// the causal triangle to within a few percent of greedy longest-first
// assignment (98% vs 87% for plain round robin on 32 heads x 32 blocks over
// 152 CTAs), without a global work counter. Returns -1 past the last item.
__device__ __forceinline__ int item_at(const FwdParams &p, int w) {
    const int G = gridDim.x;
    const int c = (w & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x;
    const long long item = (long long)w * G + c;
    return item < p.n_items ? (int)item : -1;
}

// Work item -> (bh, first query row). Longest items first for causal.
__device__ __forceinline__ void item_coords(const FwdParams &p, int item, int &bh, int &q0) {
    const int BH = p.B * p.H;
    const int qb = p.n_qblk - 1 - item / BH;
    bh = item % BH;
    q0 = qb * kRowsPerItem;
}

// Number of K/V tiles query tile t of an item at q0 must visit.
template <bool CAUSAL>
__device__ __forceinline__ int tile_nkv(const FwdParams &p, int q0, int t) {
    const int r0 = q0 + t * kBQ;
    if (r0 >= p.N) return 0;
    if (!CAUSAL) return p.n_kv;
    const int last_row = min(p.N, r0 + kBQ) - 1;
    return last_row / kBK + 1;
}

struct Sync {
    uint64_t *bars;
    __device__ __forceinline__ uint32_t q_full(int t) const { return smem_u32(bars + t); }
    __device__ __forceinline__ uint32_t q_empty(int t) const { return smem_u32(bars + 2 + t); }
    __device__ __forceinline__ uint32_t kv_full(int s) const { return smem_u32(bars + 4 + s); }
    __device__ __forceinline__ uint32_t kv_empty(int s, int stages) const { return smem_u32(bars + 4 + stages + s); }
    __device__ __forceinline__ uint32_t s_full(int t, int stages) const { return smem_u32(bars + 4 + 2 * stages + t); }
    __device__ __forceinline__ uint32_t p_full(int t, int stages) const { return smem_u32(bars + 6 + 2 * stages + t); }
    __device__ __forceinline__ uint32_t o_full(int t, int stages) const { return smem_u32(bars + 8 + 2 * stages + t); }
    __device__ __forceinline__ uint32_t drain(int stages) const { return smem_u32(bars + 10 + 2 * stages); }
};

// Bounded wait: returns false (after recording a timeout and raising the CTA's
// abort flag) if the phase does not complete within timeout_ns, or returns
// false at once if another role of this CTA has already aborted.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             const FwdParams &p) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > p.timeout_ns) {
                *abort_flag = 1;
                atomicExch(p.status, kStatusTimeout);
                return false;
            }
        }
    }
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

template <typename T, int D, bool CAUSAL, bool HAS_MASK>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    using C = Cfg<T, D>;
    constexpr int ST = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Sync sy{reinterpret_cast<uint64_t *>(smem + C::SMEM_BAR)};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::SMEM_BAR + C::NUM_BARS * 8);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(sy.q_full(t), 1);
            mbar_init(sy.q_empty(t), 1);
            mbar_init(sy.s_full(t, ST), 1);
            mbar_init(sy.p_full(t, ST), kBQ);
            mbar_init(sy.o_full(t, ST), 1);
        }
        for (int s = 0; s < ST; ++s) {
            mbar_init(sy.kv_full(s), 1);
            mbar_init(sy.kv_empty(s, ST), 1);
        }
        mbar_init(sy.drain(ST), 1);
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 9) {  // TMEM: all 512 columns (one CTA per SM)
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == 8 && lane == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);

    if (warp >= 8) {
        setmaxnreg_dec<88>();
        if (warp == 8) {
            // ---------------------------------------------------------- TMA producer
            // The whole warp runs the (uniform) loop; lane 0 issues the copies.
            const bool leader = lane == 0;
            const uint64_t pol_kv = policy_evict_last();
            const uint64_t pol_q = policy_evict_first();
            uint32_t qcount[2] = {0, 0};
            uint32_t kvpos = 0;
            bool ok = true;
            for (int w = 0, item; ok && (item = item_at(p, w)) >= 0; ++w) {
                int bh, q0;
                item_coords(p, item, bh, q0);
                const int n0 = tile_nkv<CAUSAL>(p, q0, 0), n1 = tile_nkv<CAUSAL>(p, q0, 1);
                const int nmax = max(n0, n1);
                for (int t = 0; t < 2 && ok; ++t) {
                    if ((t == 0 ? n0 : n1) == 0) continue;
                    ok = __all_sync(0xffffffffu, wait_bounded(sy.q_empty(t), (qcount[t] & 1u) ^ 1u, abort_flag, p));
                    if (!ok) break;
                    if (leader) {
                        const uint32_t dst = smem_u32(smem + C::SMEM_Q + t * C::TILE_BYTES);
                        mbar_arrive_expect_tx(sy.q_full(t), C::TILE_BYTES);
#pragma unroll
                        for (int c = 0; c < C::NCH; ++c)
                            tma_load_3d(dst + c * C::CHUNK_BYTES, &tm_q, sy.q_full(t), c * C::CHUNK_ELEMS,
                                        q0 + t * kBQ, bh, pol_q);
                    }
                    __syncwarp();
                    ++qcount[t];
                }
                for (int j = 0; ok && j < nmax; ++j) {
                    for (int kv = 0; kv < 2; ++kv) {  // K_j then V_j
                        const int s = kvpos % ST;
                        const uint32_t ph = (kvpos / ST) & 1u;
                        ok = __all_sync(0xffffffffu, wait_bounded(sy.kv_empty(s, ST), ph ^ 1u, abort_flag, p));
                        if (!ok) break;
                        if (leader) {
                            const uint32_t dst = smem_u32(smem + C::SMEM_KV + s * C::TILE_BYTES);
                            mbar_arrive_expect_tx(sy.kv_full(s), C::TILE_BYTES);
                            const CUtensorMap *m = kv == 0 ? &tm_k : &tm_v;
#pragma unroll
                            for (int c = 0; c < C::NCH; ++c)
                                tma_load_3d(dst + c * C::CHUNK_BYTES, m, sy.kv_full(s), c * C::CHUNK_ELEMS, j * kBK,
                                            bh, pol_kv);
                        }
                        __syncwarp();
                        ++kvpos;
                    }
                }
            }
            if (!ok && leader) {  // let every copy in flight land before the CTA can exit
                const uint64_t t0 = global_timer_ns();
                for (int t = 0; t < 2; ++t)
                    if (qcount[t] > 0)
                        while (!mbar_try_wait(sy.q_full(t), (qcount[t] - 1) & 1u) &&
                               global_timer_ns() - t0 < p.timeout_ns) {
                        }
                // the most recent load of each ring slot is positions kvpos-ST .. kvpos-1
                for (uint32_t pos = kvpos > (uint32_t)ST ? kvpos - ST : 0; pos < kvpos; ++pos)
                    while (!mbar_try_wait(sy.kv_full(pos % ST), (pos / ST) & 1u) &&
                           global_timer_ns() - t0 < p.timeout_ns) {
                    }
            }
        } else if (warp == 9) {
            // ---------------------------------------------------------- MMA issuer
            // Whole warp, uniform control flow; lane 0 issues every MMA and every
            // commit. Descriptors are built once and advanced by constant
            // offsets (in 16-byte units).
            const uint32_t issue = lane == 0 ? 1u : 0u;
            uint32_t qcount[2] = {0, 0}, pcount[2] = {0, 0};
            uint32_t kvpos = 0;
            const uint32_t q_base = smem_u32(smem + C::SMEM_Q);
            const uint32_t kv_base = smem_u32(smem + C::SMEM_KV);
            const uint64_t dq = smem_desc_sw128(q_base, 16, 1024);               // Q tile 0, K-major
            const uint64_t dk = smem_desc_sw128(kv_base, 16, 1024);              // ring slot 0 as K (K-major)
            const uint64_t dv = smem_desc_sw128(kv_base, C::CHUNK_BYTES, 1024);  // ring slot 0 as V (N-major)
            constexpr uint64_t TILE16 = C::TILE_BYTES >> 4;
            bool ok = true;
            auto s_mma = [&](int t, int slot) {  // S_t = Q_t K^T
                const uint64_t a0 = dq + t * TILE16, b0 = dk + slot * TILE16;
#pragma unroll
                for (int k = 0; k < C::KSTEPS_S; ++k) {
                    const uint64_t off = (uint64_t)(((k / 4) * C::CHUNK_BYTES + (k % 4) * 32) >> 4);
                    mma_ss(tmem + t * 128, a0 + off, b0 + off, C::IDESC_S, k > 0 ? 1u : 0u, issue);
                }
            };
            auto pv_mma = [&](int t, int slot, uint32_t acc) {  // O_t (+)= P_t V
                const uint64_t b0 = dv + slot * TILE16;
#pragma unroll
                for (int k = 0; k < C::KSTEPS_PV; ++k)
                    mma_ts(tmem + 256 + t * 128, tmem + t * 128 + k * 8,
                           b0 + (uint64_t)((k * C::V_KSTEP_BYTES) >> 4), C::IDESC_PV, k > 0 ? 1u : acc, issue);
            };
            for (int w = 0, item; ok && (item = item_at(p, w)) >= 0; ++w) {
                int bh, q0;
                item_coords(p, item, bh, q0);
                const int n[2] = {tile_nkv<CAUSAL>(p, q0, 0), tile_nkv<CAUSAL>(p, q0, 1)};
                const int nmax = max(n[0], n[1]);
                for (int t = 0; t < 2 && ok; ++t) {
                    if (n[t] == 0) continue;
                    ok = __all_sync(0xffffffffu, wait_bounded(sy.q_full(t), qcount[t] & 1u, abort_flag, p));
                    ++qcount[t];
                }
                if (!ok) break;
                int slot_v = 0;  // slot of V_{j-1}
                for (int j = 0; j <= nmax && ok; ++j) {
                    int slot_k = 0;
                    if (j > 0) {  // V_{j-1}
                        slot_v = kvpos % ST;
                        ok = __all_sync(0xffffffffu,
                                        wait_bounded(sy.kv_full(slot_v), (kvpos / ST) & 1u, abort_flag, p));
                        ++kvpos;
                        if (!ok) break;
                    }
                    if (j < nmax) {  // K_j
                        slot_k = kvpos % ST;
                        ok = __all_sync(0xffffffffu,
                                        wait_bounded(sy.kv_full(slot_k), (kvpos / ST) & 1u, abort_flag, p));
                        ++kvpos;
                        if (!ok) break;
                    }
                    tc_fence_after();
                    for (int t = 0; t < 2; ++t) {
                        if (j > 0 && j - 1 < n[t]) {
                            ok = __all_sync(0xffffffffu,
                                            wait_bounded(sy.p_full(t, ST), pcount[t] & 1u, abort_flag, p));
                            ++pcount[t];
                            if (!ok) break;
                            tc_fence_after();
                            pv_mma(t, slot_v, j - 1 > 0 ? 1u : 0u);
                            tc_commit(sy.o_full(t, ST), issue);
                        }
                        if (j < n[t]) {
                            s_mma(t, slot_k);
                            tc_commit(sy.s_full(t, ST), issue);
                            if (j == n[t] - 1) tc_commit(sy.q_empty(t), issue);
                        }
                    }
                    if (!ok) break;
                    if (j > 0) tc_commit(sy.kv_empty(slot_v, ST), issue);
                    if (j < nmax) tc_commit(sy.kv_empty(slot_k, ST), issue);
                }
            }
            // every MMA lane 0 issued must be complete before TMEM is released
            __syncwarp();
            tc_commit(sy.drain(ST), issue);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(sy.drain(ST), 0) && global_timer_ns() - t0 < p.timeout_ns) {
            }
        }
    } else {
        setmaxnreg_inc<208>();
        // -------------------------------------------------------------- softmax + epilogue
        const int t = warp >> 2;                   // query tile of this warpgroup
        const int r = threadIdx.x & 127;           // row within the tile = TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_addr = tmem + lane_base + t * 128;
        const uint32_t o_addr = tmem + lane_base + 256 + t * 128;
        const float scale_log2 = p.scale_log2;
        uint32_t scount = 0, ocount = 0;
        bool ok = true;
        for (int w = 0, item; ok && (item = item_at(p, w)) >= 0; ++w) {
            int bh, q0;
            item_coords(p, item, bh, q0);
            const int nt = tile_nkv<CAUSAL>(p, q0, t);
            if (nt == 0) continue;
            const int row = q0 + t * kBQ + r;  // global query row (may be >= N in a ragged tail)
            const int b = bh / p.H;
            float m_ref = -INFINITY, l = 0.0f;
            for (int j = 0; j < nt; ++j) {
                ok = __all_sync(0xffffffffu, wait_bounded(sy.s_full(t, ST), scount & 1u, abort_flag, p));
                ++scount;
                if (!ok) break;
                tc_fence_after();
                float x[128];
                const int kbase = j * kBK;
                // sl2 multiplies x inside the exponent: raw scores with sl2 = scale*log2(e)
                // on the fast path (no mask, positive scale), pre-scaled scores with sl2 = 1
                // otherwise (a -inf raw score times a non-positive scale is not -inf).
                float sl2 = 1.0f;
                if constexpr (HAS_MASK) {
                    // 32 columns at a time so that S and mask values are not all live at once
                    const bool row_ok = row < p.N;
                    const float *mrow = p.mask + ((size_t)b * p.N + (size_t)(row_ok ? row : 0)) * p.N + kbase;
                    const bool vec = row_ok && ((p.N & 3) == 0) && (kbase + kBK <= p.N);
#pragma unroll
                    for (int c0 = 0; c0 < 128; c0 += 32) {
                        uint32_t sr[32];
                        tmem_ld32_wait(s_addr + c0, sr);
                        if (vec) {
#pragma unroll
                            for (int c = 0; c < 32; c += 4) {
                                const float4 mv = ld_global_nc_v4(mrow + c0 + c);
                                x[c0 + c + 0] = fmaf(__uint_as_float(sr[c + 0]), scale_log2, mv.x * 1.4426950408889634f);
                                x[c0 + c + 1] = fmaf(__uint_as_float(sr[c + 1]), scale_log2, mv.y * 1.4426950408889634f);
                                x[c0 + c + 2] = fmaf(__uint_as_float(sr[c + 2]), scale_log2, mv.z * 1.4426950408889634f);
                                x[c0 + c + 3] = fmaf(__uint_as_float(sr[c + 3]), scale_log2, mv.w * 1.4426950408889634f);
                            }
                        } else {
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                const float mv = (row_ok && kbase + c0 + c < p.N) ? __ldg(mrow + c0 + c) : 0.0f;
                                x[c0 + c] = fmaf(__uint_as_float(sr[c]), scale_log2, mv * 1.4426950408889634f);
                            }
                        }
                    }
                } else {
                    // two 64-column halves: the second load is in flight while the first is converted
                    uint32_t sa[64], sb[64];
                    tmem_ld64_nowait(s_addr, sa);
                    tmem_wait_ld_dep64(sa);
                    tmem_ld64_nowait(s_addr + 64, sb);
                    const bool fast = scale_log2 > 0.0f;
                    sl2 = fast ? scale_log2 : 1.0f;
                    const float pre = fast ? 1.0f : scale_log2;
#pragma unroll
                    for (int c = 0; c < 64; ++c) x[c] = __uint_as_float(sa[c]) * pre;
                    tmem_wait_ld_dep64(sb);
#pragma unroll
                    for (int c = 0; c < 64; ++c) x[64 + c] = __uint_as_float(sb[c]) * pre;
                }
                // keys past the end of the sequence, and (causal) keys after the query
                const int tile_row0 = q0 + t * kBQ;
                const bool ragged = kbase + kBK > p.N;
                const bool diag = CAUSAL && (kbase + kBK - 1 > tile_row0);
                if (ragged || diag) {
                    int lim = p.N - 1 - kbase;
                    if (CAUSAL) lim = min(lim, row - kbase);
#pragma unroll
                    for (int c = 0; c < 128; ++c) x[c] = (c > lim) ? -INFINITY : x[c];
                }
                // row maximum: eight independent three-input chains, then a short tree
                float m8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) m8[i] = x[i];
#pragma unroll
                for (int c = 8; c < 120; c += 16)
#pragma unroll
                    for (int i = 0; i < 8; ++i) m8[i] = fmax3(m8[i], x[c + i], x[c + 8 + i]);
#pragma unroll
                for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], x[120 + i]);
                const float mraw =
                    fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                const float mb = mraw * sl2;  // sl2 > 0, so scaling commutes with the maximum
                const float m_new = fmaxf(m_ref, mb);
                // lazy rescale: move the reference only when the maximum grew by more than TAU
                const bool need = (m_new > m_ref + kTau) || (m_ref == -INFINITY && m_new != -INFINITY);
                const float alpha = need ? ex2_approx(m_ref - m_new) : 1.0f;  // 2^-inf = 0
                if (__any_sync(0xffffffffu, need) && j > 0) {
                    // O holds P V for blocks < j: wait for the product of block j-1, then scale rows in place
                    ok = __all_sync(0xffffffffu,
                                    wait_bounded(sy.o_full(t, ST), (ocount + j - 1) & 1u, abort_flag, p));
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t ov[32];
                        tmem_ld32_wait(o_addr + c0, ov);
#pragma unroll
                        for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
                        tmem_st32(o_addr + c0, ov);
                    }
                }
                if (need) {
                    l *= alpha;
                    m_ref = m_new;
                }
                const float neg = (m_ref == -INFINITY) ? 0.0f : -m_ref;
                float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int c0 = 0; c0 < 128; c0 += 64) {
                    uint32_t pv[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float e0 = ex2_approx(fmaf(x[c0 + 2 * c], sl2, neg));
                        const float e1 = ex2_approx(fmaf(x[c0 + 2 * c + 1], sl2, neg));
                        ls[c & 3] += e0 + e1;
                        pv[c] = pack2<T>(e0, e1);
                    }
                    tmem_st32(s_addr + c0 / 2, pv);
                }
                l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(sy.p_full(t, ST));
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue
            ok = __all_sync(0xffffffffu, wait_bounded(sy.o_full(t, ST), (ocount + nt - 1) & 1u, abort_flag, p));
            ocount += nt;
            if (!ok) break;
            tc_fence_after();
            const float inv = (l > 0.0f) ? 1.0f / l : 0.0f;
            T *orow = reinterpret_cast<T *>(p.out) + ((size_t)bh * p.N + (size_t)row) * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t ov[32];
                tmem_ld32_wait(o_addr + c0, ov);
                if (row < p.N) {
#pragma unroll
                    for (int c = 0; c < 32; c += 8)
                        st_global_v4(orow + c0 + c,
                                     pack2<T>(__uint_as_float(ov[c]) * inv, __uint_as_float(ov[c + 1]) * inv),
                                     pack2<T>(__uint_as_float(ov[c + 2]) * inv, __uint_as_float(ov[c + 3]) * inv),
                                     pack2<T>(__uint_as_float(ov[c + 4]) * inv, __uint_as_float(ov[c + 5]) * inv),
                                     pack2<T>(__uint_as_float(ov[c + 6]) * inv, __uint_as_float(ov[c + 7]) * inv));
                }
            }
            if (row < p.N)
                p.lse[(size_t)bh * p.N + row] =
                    (l > 0.0f) ? (m_ref + lg2_approx(l)) * 0.6931471805599453f : -INFINITY;
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace fa
