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
// Two kernels share that plan: fa_bwd_kernel_h64 (d = 64, further below), which
// overlaps the tensor core with the gradient warps over half blocks, and
// fa_bwd_kernel (used for d = 128, where the dV and dK accumulators leave no
// tensor memory for that overlap), described here.
//
// One CTA owns a 128-key block j of one (b, h) and loops over the 128-row query
// blocks i that can see it (all of them, or i >= j when causal):
//   warp 0      TMA: K_j and V_j once, then Q_i and dO_i through a ring
//   warps 1, 2  MMA issue (warp-uniform loops, lane 0 issues), tcgen05 kind::f16: warp 1 S^T, dV
//               and dQ's head columns 0..63, warp 2 dP^T, dK and dQ's columns 64..127
//   warps 4-11  two warpgroups; thread r of a group owns TMEM lane r. Group g
//               first turns query columns [64 g, 64 g + 64) of S^T, dP^T into
//               P^T and dS^T for key r, then reads out dQ for query row r,
//               head columns of half g, and at the end stores dV (g = 0) or
//               dK (g = 1) of key r.
// Tensor memory (512 columns) per iteration. Query chunk x (32 queries) has
// its scores in S^T columns [32x, 32x+32); group 0 handles chunks 0, 1 in that
// order, group 1 chunks 3, 2. Each group packs P^T (16 bit, two queries per
// column) only into columns it has already read itself: chunk x goes to
// columns 16x (x < 2) or 64 + 16x (x >= 2). So the two groups never touch each
// other's unread scores, and columns [32,96) are free afterwards.
//   [0,128)     S^T = K_j Q_i^T (fp32), then P^T in [0,32) and [96,128), and
//               dQ head columns 0..63 in [32,96)
//   [128,256)   dP^T = V_j dO_i^T (fp32), then dS^T in [128,160) and
//               [224,256), and dQ head columns 64..127 in [160,224) (d = 128)
//   [256,256+d) dV_j accumulator,  [256+d,256+2d) dK_j accumulator
// dV_j += P^T dO_i and dK_j += dS^T Q_i take A from tensor memory; dQ_i = dS K_j
// takes A = dS from shared memory, written by the gradient warps with the
// query index contiguous (an M-major operand). Each warp then stages its two
// 32 x 32 fp32 tiles of dQ_i, one in its own part of that dS buffer and one
// in the dO half of block i's stage (dead once every product of the block is
// done), and adds them into an fp32 workspace with bulk tensor reductions
// (reduce-add in L2); a last kernel converts the workspace to the output type.
// So a stage's Q and dO halves have their own barriers: Q goes back to the
// producer by the issuing warps' commits, dO by the gradient warps once their
// reductions have read the tiles, which they wait for before the next pass
// writes dS. The row statistics of block i (lse * log2 e and D, padded past N)
// are loaded one iteration ahead and handed over in shared memory.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fa_bwd.cuh"
#include "fa_launch.cuh"
#include "pdl.cuh"

namespace fa {
namespace {

constexpr int kBwdThreads = 384;
constexpr int kGradThreads = 256;  // warps 4-11
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
    static constexpr int SMEM_STATS = SMEM_DS + 2 * CHUNK;       // -lse2[128], -D[128] of the current block
    static constexpr int SMEM_BAR = SMEM_STATS + 256 * 4;
    static constexpr int NUM_BARS = 1 + 4 * STAGES + 6;
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
    float *dq_acc;      // [BH][N][d], reduced into through tm_dq
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

// Two packed 16-bit values -> (low, high) as floats.
template <typename T>
__device__ __forceinline__ float2 up2(uint32_t v) {
    if constexpr (Elem<T>::fmt == 1) {
        return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&v));
    } else {
        return __half22float2(*reinterpret_cast<__half2 *>(&v));
    }
}

// P and dS for 32 query columns of one key (this thread's TMEM lane), packed in
// pairs to the 16-bit input type: P = 2^(S * scale * log2 e - lse * log2 e) and
// dS = P (dP - D). neg_l and neg_d are shared-memory addresses of -lse*log2e and
// -D for the 32 columns (the same for every lane: broadcast loads). Keys past
// the end, and (causal) keys after the query, get P = dS = 0 when need_mask is
// set. MASKING = false compiles a copy without that code, for the blocks that
// need none: in the causal kernels the masking code kept in the common path
// cost 30-40 registers and about a fifth of the time per block.
template <typename T, bool CAUSAL, bool MASKING>
__device__ __forceinline__ void p_ds_chunk(const uint32_t (&sv)[32], const uint32_t (&dpv)[32], uint32_t neg_l,
                                           uint32_t neg_d, float scale_log2, bool need_mask, bool key_ok, int key,
                                           int q_first, uint32_t (&pp)[16], uint32_t (&dsp)[16]) {
#pragma unroll
    for (int c = 0; c < 32; c += 4) {
        const float4 nl = ld_shared_v4f(neg_l + c * 4);
        const float4 nd = ld_shared_v4f(neg_d + c * 4);
#pragma unroll
        for (int h = 0; h < 4; h += 2) {
            const float2 x = ffma2(make_float2(__uint_as_float(sv[c + h]), __uint_as_float(sv[c + h + 1])),
                                   make_float2(scale_log2, scale_log2),
                                   h == 0 ? make_float2(nl.x, nl.y) : make_float2(nl.z, nl.w));
            float2 pe = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            if (MASKING && need_mask) {
                const int q0 = q_first + c + h;
                const bool v0 = key_ok && (!CAUSAL || key <= q0);
                const bool v1 = key_ok && (!CAUSAL || key <= q0 + 1);
                pe.x = v0 ? pe.x : 0.0f;
                pe.y = v1 ? pe.y : 0.0f;
            }
            const float2 t = fadd2(make_float2(__uint_as_float(dpv[c + h]), __uint_as_float(dpv[c + h + 1])),
                                   h == 0 ? make_float2(nd.x, nd.y) : make_float2(nd.z, nd.w));
            const float2 ds = fmul2(pe, t);
            pp[(c + h) / 2] = pk2<T>(pe.x, pe.y);
            dsp[(c + h) / 2] = pk2<T>(ds.x, ds.y);
        }
    }
}

// Stage one 32 x 32 fp32 tile (this warp's 32 rows x 32 head columns, already
// scaled) in shared memory with the 128-byte swizzle of tm_dq, and reduce-add it
// into the dQ accumulator. Lane 0 first waits until its previous reduction from
// the same staging area has been read.
__device__ __forceinline__ void stage_and_reduce_dq(const CUtensorMap *tm_dq, uint32_t box, const uint32_t (&qv)[32],
                                                    float mul, int lane, int x, int y, int z) {
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
#pragma unroll
    for (int u = 0; u < 8; ++u)
        st_shared_v4(box + lane * 128 + ((u ^ (lane & 7)) * 16), __float_as_uint(__uint_as_float(qv[4 * u]) * mul),
                     __float_as_uint(__uint_as_float(qv[4 * u + 1]) * mul),
                     __float_as_uint(__uint_as_float(qv[4 * u + 2]) * mul),
                     __float_as_uint(__uint_as_float(qv[4 * u + 3]) * mul));
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_reduce_add_3d(tm_dq, box, x, y, z);
        bulk_commit_group();
    }
}

template <typename T, int D, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
    using C = BwdCfg<T, D>;
    static_assert(D == 128, "the two issuing warps take one 64-column half of dQ each");
    constexpr int ST = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::SMEM_BAR);
    const uint32_t bar_kv = smem_u32(bars);
    auto bar_q_full = [&](int s) { return smem_u32(bars + 1 + s); };
    auto bar_q_empty = [&](int s) { return smem_u32(bars + 1 + ST + s); };       // both warps' last Q reader
    auto bar_do_full = [&](int s) { return smem_u32(bars + 1 + 2 * ST + s); };
    auto bar_do_empty = [&](int s) { return smem_u32(bars + 1 + 3 * ST + s); };  // dQ tiles staged there read
    const uint32_t bar_sp_full = smem_u32(bars + 1 + 4 * ST);  // S^T, dP^T in TMEM
    const uint32_t bar_p_full = smem_u32(bars + 2 + 4 * ST);   // P^T, dS^T, dS written (256 arrivals)
    const uint32_t bar_dq_full = smem_u32(bars + 3 + 4 * ST);  // every product of the iteration done
    const uint32_t bar_dq_free = smem_u32(bars + 4 + 4 * ST);  // dQ loaded from TMEM (256 arrivals)
    const uint32_t bar_drain = smem_u32(bars + 5 + 4 * ST);    // all issued MMAs done (exit)
    const uint32_t bar_stats = smem_u32(bars + 6 + 4 * ST);    // row statistics of the block stored (256 arrivals)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::SMEM_BAR + C::NUM_BARS * 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Block b -> (key block j, head bh); low j first, which in the causal case
    // are the blocks with the most query blocks to visit.
    const int bh = blockIdx.x % p.BH;
    const int j = blockIdx.x / p.BH;
    const int n_qblk = p.Npad / kBlk;
    const int i0 = CAUSAL ? j : 0;  // first query block that sees key block j
    const int n_it = n_qblk - i0;   // >= 1
    grid_launch_dependents();       // fa_bwd_post may be scheduled once every CTA has started

    if (threadIdx.x == 0) {
        mbar_init(bar_kv, 1);
        // the completion barriers of the products take one commit from each issuing warp
        for (int s = 0; s < ST; ++s) {
            mbar_init(bar_q_full(s), 1);
            mbar_init(bar_q_empty(s), 2);
            mbar_init(bar_do_full(s), 1);
            mbar_init(bar_do_empty(s), kGradThreads / 32);  // one arrival per gradient warp
        }
        mbar_init(bar_sp_full, 2);
        mbar_init(bar_p_full, kGradThreads);
        mbar_init(bar_dq_full, 2);
        mbar_init(bar_dq_free, kGradThreads);
        mbar_init(bar_drain, 2);
        mbar_init(bar_stats, kGradThreads);
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
            int issued_q = 0, issued_do = 0;
            for (int it = 0; it < n_it; ++it) {
                const int s = it % ST;
                const uint32_t dst = smem_u32(smem + C::SMEM_QD + s * 2 * C::TILE);
                const int row0 = (i0 + it) * kBlk;
                if (!bwd_wait(bar_q_empty(s), ((it / ST) & 1u) ^ 1u, p)) break;
                mbar_arrive_expect_tx(bar_q_full(s), C::TILE);
                for (int c = 0; c < C::NCH; ++c) tma_load_3d(dst + c * C::CHUNK, &tm_q, bar_q_full(s), c * 64, row0, bh, pol);
                issued_q = it + 1;
                // dO's half also held the dQ tiles of the stage's last block until they were read
                if (!bwd_wait(bar_do_empty(s), ((it / ST) & 1u) ^ 1u, p)) break;
                mbar_arrive_expect_tx(bar_do_full(s), C::TILE);
                for (int c = 0; c < C::NCH; ++c)
                    tma_load_3d(dst + C::TILE + c * C::CHUNK, &tm_do, bar_do_full(s), c * 64, row0, bh, pol);
                issued_do = it + 1;
            }
            // Before the CTA may exit, every copy into its shared memory must have
            // landed (they all have on the normal path; this matters after a timeout).
            bwd_wait(bar_kv, 0, p);
            for (int it = issued_q - ST > 0 ? issued_q - ST : 0; it < issued_q; ++it)
                bwd_wait(bar_q_full(it % ST), (it / ST) & 1u, p);
            for (int it = issued_do - ST > 0 ? issued_do - ST : 0; it < issued_do; ++it)
                bwd_wait(bar_do_full(it % ST), (it / ST) & 1u, p);
        }
    } else if (warp == 1 || warp == 2) {
        // ---------------------------------------------------------------- MMA issuers
        // One warp issues only about one product every 77 cycles, so the products are split over two
        // warps: warp 1 issues S^T, dV and dQ's head columns 0..63, warp 2 dP^T, dK and dQ's columns
        // 64..127. Each product's columns are its own warp's (S^T, packed P^T, dQ half 0 in [0, 128);
        // dP^T, dS^T, dQ half 1 in [128, 256)); sp_full, dq_full, q_empty and drain take a commit from
        // each warp, and each warp waits dq_free (every product of the last block done and dQ read
        // out) before its next S^T or dP^T overwrites its columns.
        const int h = warp - 1;  // 0: S^T, dV, dQ half 0; 1: dP^T, dK, dQ half 1
        const uint32_t issue = lane == 0 ? 1u : 0u;
        const uint64_t a_km = smem_desc_sw128(smem_u32(smem + (h == 0 ? C::SMEM_K : C::SMEM_V)), 16, 1024);
        const uint64_t k_mn = smem_desc_sw128(smem_u32(smem + C::SMEM_K), C::CHUNK, 1024);   // K_j as B, N-major
        const uint64_t ds_mn = smem_desc_sw128(smem_u32(smem + C::SMEM_DS), C::CHUNK, 1024); // dS as A, M-major
        bool ok = bwd_wait_warp(bar_kv, 0, p);
        for (int it = 0; ok && it < n_it; ++it) {
            const int s = it % ST;
            ok = bwd_wait_warp(bar_q_full(s), (it / ST) & 1u, p) && bwd_wait_warp(bar_do_full(s), (it / ST) & 1u, p);
            if (ok && it > 0) ok = bwd_wait_warp(bar_dq_free, (it - 1) & 1u, p);
            if (!ok) break;
            tc_fence_after();
            const uint32_t q_s = smem_u32(smem + C::SMEM_QD + s * 2 * C::TILE);
            // B of S^T is Q_i, of dP^T dO_i (K-major); B of dV is dO_i, of dK Q_i (N-major)
            const uint64_t b_km = smem_desc_sw128(q_s + (h == 0 ? 0 : C::TILE), 16, 1024);
            const uint64_t b_mn = smem_desc_sw128(q_s + (h == 0 ? C::TILE : 0), C::CHUNK, 1024);
            // S^T = K_j Q_i^T (h = 0) or dP^T = V_j dO_i^T (h = 1), contracted over the head dimension
#pragma unroll
            for (int k = 0; k < C::KSTEPS_D; ++k) {
                const uint64_t off = (uint64_t)(((k / 4) * C::CHUNK + (k % 4) * 32) >> 4);
                mma_ss(tmem + 128 * h, a_km + off, b_km + off, C::ID_ST, k > 0 ? 1u : 0u, issue);
            }
            tc_commit(bar_sp_full, issue);
            ok = bwd_wait_warp(bar_p_full, it & 1u, p);
            if (!ok) break;
            tc_fence_after();
            // dV_j += P^T dO_i (h = 0) or dK_j += dS^T Q_i (h = 1), contracted over the 128 query rows
#pragma unroll
            for (int k = 0; k < C::KSTEPS_R; ++k) {
                const uint64_t off = (uint64_t)((k * 2048) >> 4);
                const uint32_t acc = (it > 0 || k > 0) ? 1u : 0u;
                const uint32_t pcol = (uint32_t)(k < 4 ? 8 * k : 64 + 8 * k);  // packed P^T / dS^T of queries 16k..
                mma_ts(tmem + 256 + D * h, tmem + 128 * h + pcol, b_mn + off, C::ID_ACC, acc, issue);
            }
            // dQ_i = dS K_j, contracted over the 128 keys, head columns 64h..64h+63
#pragma unroll
            for (int k = 0; k < C::KSTEPS_R; ++k) {
                const uint64_t off = (uint64_t)((k * 2048) >> 4);
                mma_ss(tmem + (h == 0 ? 32 : 160), ds_mn + off, k_mn + (uint64_t)((h * C::CHUNK) >> 4) + off,
                       C::ID_DQ, k > 0 ? 1u : 0u, issue);
            }
            tc_commit(bar_dq_full, issue);
            tc_commit(bar_q_empty(s), issue);  // dO's half is released by the gradient warps
        }
        // Every MMA of both warps is complete before tensor memory is freed.
        tc_commit(bar_drain, issue);
        if (warp == 1) bwd_wait_warp(bar_drain, 0, p);
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- gradient warps
        const int g = (warp - 4) >> 2;             // warpgroup: query columns / head columns half g
        const int w = warp & 3;                    // TMEM lane group
        const int r = w * 32 + lane;               // TMEM lane: key r of block j, later query row r of block i
        const uint32_t lane_base = (uint32_t)(w * 32) << 16;
        const int key = j * kBlk + r;
        const bool key_ok = key < p.N;
        const uint32_t ds_base = smem_u32(smem + C::SMEM_DS);
        const uint32_t stats = smem_u32(smem + C::SMEM_STATS);
        // this warp's 4 KB of the dS buffer (its 32 key rows of chunk g), reused to stage dQ tiles
        const uint32_t stage = ds_base + g * C::CHUNK + w * 4096;
        // one statistic per thread: -lse2 (group 0) or -D (group 1) of query row r of the block
        const float *stat_src = (g == 0 ? p.lse2 : p.dsum) + (size_t)bh * p.Npad + r;
        grid_dependency_wait();  // statistics and the zeroed dQ accumulator are written by fa_bwd_pre
        float stat_next = -__ldg(stat_src + i0 * kBlk);
        const bool ragged_keys = (j + 1) * kBlk > p.N;
        bool ok = true;
        for (int it = 0; ok && it < n_it; ++it) {
            const int i = i0 + it;
            const int row0 = i * kBlk;
            // hand over the block's statistics (their last readers passed p_full of the previous block)
            st_shared_f32(stats + (g * 128 + r) * 4, stat_next);
            mbar_arrive(bar_stats);
            ok = bwd_wait_warp(bar_stats, it & 1u, p) && bwd_wait_warp(bar_sp_full, it & 1u, p);
            if (!ok) break;
            tc_fence_after();
            const bool need_mask = ragged_keys || (CAUSAL && i == j);
#pragma unroll 1
            for (int step = 0; step < 2; ++step) {  // 32 query rows (TMEM columns) at a time
                const int c0 = g == 0 ? 32 * step : 96 - 32 * step;
                const uint32_t pcol = (uint32_t)(c0 < 64 ? c0 / 2 : 64 + c0 / 2);  // packed P^T / dS^T column
                uint32_t sv[32], dpv[32];
                tmem_ld32x2_wait(tmem + lane_base + c0, sv, tmem + lane_base + 128 + c0, dpv);
                uint32_t pp[16], dsp[16];
                if (CAUSAL && !need_mask)  // (a separate copy gained nothing without causal masking)
                    p_ds_chunk<T, CAUSAL, false>(sv, dpv, stats + c0 * 4, stats + (128 + c0) * 4, p.scale_log2, false,
                                                 key_ok, key, row0 + c0, pp, dsp);
                else
                    p_ds_chunk<T, CAUSAL, true>(sv, dpv, stats + c0 * 4, stats + (128 + c0) * 4, p.scale_log2,
                                                need_mask, key_ok, key, row0 + c0, pp, dsp);
                // P^T and dS^T overwrite columns this warpgroup has already read.
                tmem_st16(tmem + lane_base + 0 + pcol, pp);
                tmem_st16(tmem + lane_base + 128 + pcol, dsp);
                // dS row of key r: queries c0..c0+31 = 64 bytes of chunk g, 128-byte swizzle
                const uint32_t ds_row = ds_base + g * C::CHUNK + r * 128;
                if (step == 0) {  // the previous block's dQ reductions (staged in these rows and in the dO half
                                  // of its stage) must have read them; that dO half goes back to the producer
                    if (lane == 0) {
                        bulk_wait_read_all();
                        if (it > 0) mbar_arrive(bar_do_empty((it - 1) % ST));
                    }
                    __syncwarp();
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t unit = (uint32_t)(((c0 % 64) / 8 + u) ^ (r & 7));
                    st_shared_v4(ds_row + unit * 16, dsp[4 * u], dsp[4 * u + 1], dsp[4 * u + 2], dsp[4 * u + 3]);
                }
            }
            tmem_wait_st();
            fence_proxy_async_smem();  // dS is read by the tensor core (async proxy)
            tc_fence_before();
            mbar_arrive(bar_p_full);
            if (it + 1 < n_it) stat_next = -__ldg(stat_src + (i + 1) * kBlk);  // in flight during the read-out
            // dQ_i rows 32w..32w+31, head columns of half g: load them, release the
            // tensor memory at once (the next block's S^T, dP^T may then be computed),
            // then stage 32 x 32 fp32 tiles and reduce-add them into the workspace.
            ok = bwd_wait_warp(bar_dq_full, it & 1u, p);
            if (!ok) break;
            tc_fence_after();
            constexpr int COLS = D / 2;  // head columns per warpgroup (32 or 64)
            const uint32_t qcol = (D == 64) ? (32u + 32u * g) : (g == 0 ? 32u : 160u);
            uint32_t qv[COLS];
            if constexpr (COLS == 32) {
                tmem_ld32_wait(tmem + lane_base + qcol, *reinterpret_cast<uint32_t(*)[32]>(qv));
            } else {
                tmem_ld32x2_wait(tmem + lane_base + qcol, *reinterpret_cast<uint32_t(*)[32]>(qv),
                                 tmem + lane_base + qcol + 32, *reinterpret_cast<uint32_t(*)[32]>(qv + 32));
            }
            tc_fence_before();
            mbar_arrive(bar_dq_free);
            // tile 0 in this warp's dS rows, tile 1 in the dO half of the block's stage (every product of the
            // block is done: dq_full)
            const uint32_t stage1 = smem_u32(smem + C::SMEM_QD + (it % ST) * 2 * C::TILE + C::TILE) + (g * 4 + w) * 4096;
#pragma unroll
            for (int t = 0; t < COLS / 32; ++t) {
                const uint32_t box = t == 0 ? stage : stage1;
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    st_shared_v4(box + lane * 128 + ((u ^ (lane & 7)) * 16),
                                 __float_as_uint(__uint_as_float(qv[32 * t + 4 * u]) * p.scale),
                                 __float_as_uint(__uint_as_float(qv[32 * t + 4 * u + 1]) * p.scale),
                                 __float_as_uint(__uint_as_float(qv[32 * t + 4 * u + 2]) * p.scale),
                                 __float_as_uint(__uint_as_float(qv[32 * t + 4 * u + 3]) * p.scale));
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_reduce_add_3d(&tm_dq, box, g * COLS + 32 * t, row0 + w * 32, bh);
                    bulk_commit_group();
                }
            }
        }
        // ---------------------------------------------------------------- dV_j (group 0), dK_j (group 1)
        // The last dq_full completion covers every dV and dK product (a commit
        // tracks all earlier MMAs of the issuing thread).
        if (ok) {
            tc_fence_after();
            const float mul = g == 0 ? 1.0f : p.scale;
            T *dst = reinterpret_cast<T *>(g == 0 ? p.dv : p.dk) + ((size_t)bh * p.N + (size_t)(key_ok ? key : 0)) * D;
            const uint32_t src_col = 256u + (uint32_t)(g * D);
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 64) {
                uint32_t a[32], b[32];
                tmem_ld32x2_wait(tmem + lane_base + src_col + c0, a, tmem + lane_base + src_col + c0 + 32, b);
                if (key_ok) {
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        st_global_v4(dst + c0 + c, pk2<T>(__uint_as_float(a[c]) * mul, __uint_as_float(a[c + 1]) * mul),
                                     pk2<T>(__uint_as_float(a[c + 2]) * mul, __uint_as_float(a[c + 3]) * mul),
                                     pk2<T>(__uint_as_float(a[c + 4]) * mul, __uint_as_float(a[c + 5]) * mul),
                                     pk2<T>(__uint_as_float(a[c + 6]) * mul, __uint_as_float(a[c + 7]) * mul));
                        st_global_v4(dst + c0 + 32 + c,
                                     pk2<T>(__uint_as_float(b[c]) * mul, __uint_as_float(b[c + 1]) * mul),
                                     pk2<T>(__uint_as_float(b[c + 2]) * mul, __uint_as_float(b[c + 3]) * mul),
                                     pk2<T>(__uint_as_float(b[c + 4]) * mul, __uint_as_float(b[c + 5]) * mul),
                                     pk2<T>(__uint_as_float(b[c + 6]) * mul, __uint_as_float(b[c + 7]) * mul));
                    }
                }
            }
        }
        if (lane == 0) bulk_wait_all();  // the dQ reductions, behind the dV / dK stores
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// d = 64: the same products with the tensor core and the gradient warps
// overlapped. Each 128-row query block is handled as two 64-row halves h (A =
// rows 0-63, B = rows 64-127), gradient warpgroup h owning half h, with their
// own barriers. The tensor core runs, per block i,
//   dV,dK(A, i)   S,dP(A, i+1)   dV,dK(B, i)   S,dP(B, i+1)   dQ(i)
// so that each warpgroup's P/dS pass of one block overlaps the other half's
// products (the two warpgroups alternate like a ping-pong). Nothing the dV
// and dK products read lives where the next block's S and dP are written:
// P^T (16 bit) is packed into its own tensor-memory columns, and dK takes
// dS^T straight from shared memory, where the pass writes dS for dQ anyway
// (keys as rows, queries contiguous: K-major for dS^T, M-major for dS). So the
// issuing warp never waits for its own products to finish; a warpgroup's wait
// for its next S covers every earlier product (a commit tracks all earlier
// MMAs of the issuing thread), which is when it may overwrite its packed P and
// its dS buffer. dS is kept in two shared-memory buffers (block parity),
// because the pass of half A of block i+1 runs before dQ(i) has read dS(i).
// dQ of block i is read out by the gradient warps after their pass of block
// i+1 (it has its own tensor-memory columns; its staging tiles reuse block
// i's dS buffer, which dK(i) and dQ(i) have finished reading by then);
// dQ(i+1) waits for that read-out.
// Tensor memory: S_A [0,64), dP_A [64,128), S_B [128,192), dP_B [192,256),
// P^T_A [256,288), P^T_B [288,320), dV [320,384), dK [384,448), dQ [448,512).
template <typename T>
struct BwdCfgH64 {
    static constexpr int D = 64;
    static constexpr int CHUNK = 128 * 128;          // 128 rows x 128 bytes (one tile at d = 64)
    static constexpr int STAGES = 3;
    static constexpr int SMEM_K = 0;
    static constexpr int SMEM_V = CHUNK;
    static constexpr int SMEM_QD = 2 * CHUNK;                      // STAGES x (Q_i, dO_i)
    static constexpr int SMEM_DS = SMEM_QD + STAGES * 2 * CHUNK;   // dS[2]: queries 0-63 | 64-127, 128 keys each
    static constexpr int SMEM_STATS = SMEM_DS + 4 * CHUNK;         // [half][buffer][-lse2 x64, -D x64]
    static constexpr int SMEM_BAR = SMEM_STATS + 2 * 2 * 128 * 4;
    // kv, qd_full[ST], qd_empty[ST], sp_full[2], p_full[2], dq_full, dq_free, stats[2], drain, acc_done[2]
    static constexpr int NUM_BARS = 1 + 2 * STAGES + 2 + 2 + 2 + 2 + 1 + 2;
    static constexpr int SMEM_BYTES = SMEM_BAR + NUM_BARS * 8 + 16 + 1024;
    static constexpr uint32_t FMT = Elem<T>::fmt;
    static constexpr uint32_t ID_S = make_idesc_ab(FMT, 128, 64, 0, 0);   // S_h^T, dP_h^T: 128 keys x 64 queries
    static constexpr uint32_t ID_ACC = make_idesc_ab(FMT, 128, 64, 0, 1); // dV (A in TMEM), dK (A K-major): B N-major
    static constexpr uint32_t ID_DQ = make_idesc_ab(FMT, 128, 64, 1, 1);  // dQ: A M-major, B N-major
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <typename T, bool CAUSAL>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_kernel_h64(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                      const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
    using C = BwdCfgH64<T>;
    constexpr int ST = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::SMEM_BAR);
    const uint32_t bar_kv = smem_u32(bars);
    auto bar_qd_full = [&](int s) { return smem_u32(bars + 1 + s); };
    auto bar_qd_empty = [&](int s) { return smem_u32(bars + 1 + ST + s); };
    auto bar_sp_full = [&](int h) { return smem_u32(bars + 1 + 2 * ST + h); };  // S_h, dP_h computed
    auto bar_p_full = [&](int h) { return smem_u32(bars + 3 + 2 * ST + h); };   // half h packed (128 arrivals)
    const uint32_t bar_dq_full = smem_u32(bars + 5 + 2 * ST);                  // dQ of the block computed
    const uint32_t bar_dq_free = smem_u32(bars + 6 + 2 * ST);                  // dQ loaded by all (256 arrivals)
    auto bar_stats = [&](int h) { return smem_u32(bars + 7 + 2 * ST + h); };   // half h statistics (128 arrivals)
    const uint32_t bar_drain = smem_u32(bars + 9 + 2 * ST);                    // both issuing warps' products done
    auto bar_acc_done = [&](int h) { return smem_u32(bars + 10 + 2 * ST + h); }; // dV, dK of half h done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::SMEM_BAR + C::NUM_BARS * 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x % p.BH;
    const int j = blockIdx.x / p.BH;
    const int n_qblk = p.Npad / kBlk;
    const int i0 = CAUSAL ? j : 0;
    const int n_it = n_qblk - i0;  // >= 1
    grid_launch_dependents();      // fa_bwd_post may be scheduled once every CTA has started

    if (threadIdx.x == 0) {
        mbar_init(bar_kv, 1);
        for (int s = 0; s < ST; ++s) {
            mbar_init(bar_qd_full(s), 1);
            mbar_init(bar_qd_empty(s), 2);  // the last S/dP product and the last dV/dK product of the stage
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(bar_sp_full(h), 1);
            mbar_init(bar_p_full(h), 128);
            mbar_init(bar_stats(h), 128);
            mbar_init(bar_acc_done(h), 1);
        }
        mbar_init(bar_dq_full, 1);
        mbar_init(bar_dq_free, kGradThreads);
        mbar_init(bar_drain, 2);  // one commit per issuing warp
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
            mbar_arrive_expect_tx(bar_kv, 2 * C::CHUNK);
            tma_load_3d(smem_u32(smem + C::SMEM_K), &tm_k, bar_kv, 0, j * kBlk, bh, pol);
            tma_load_3d(smem_u32(smem + C::SMEM_V), &tm_v, bar_kv, 0, j * kBlk, bh, pol);
            int issued = 0;
            for (int it = 0; it < n_it; ++it) {
                const int s = it % ST;
                if (!bwd_wait(bar_qd_empty(s), ((it / ST) & 1u) ^ 1u, p)) break;
                const uint32_t dst = smem_u32(smem + C::SMEM_QD + s * 2 * C::CHUNK);
                mbar_arrive_expect_tx(bar_qd_full(s), 2 * C::CHUNK);
                const int row0 = (i0 + it) * kBlk;
                tma_load_3d(dst, &tm_q, bar_qd_full(s), 0, row0, bh, pol);
                tma_load_3d(dst + C::CHUNK, &tm_do, bar_qd_full(s), 0, row0, bh, pol);
                issued = it + 1;
            }
            bwd_wait(bar_kv, 0, p);  // every copy into this CTA's shared memory lands before exit
            for (int it = issued - ST > 0 ? issued - ST : 0; it < issued; ++it)
                bwd_wait(bar_qd_full(it % ST), (it / ST) & 1u, p);
        }
    } else if (warp == 1 || warp == 2) {
        // ---------------------------------------------------------------- MMA issuers
        // One warp issues about one product every 77 cycles, so the products are split over two
        // warps: warp 1 issues every S/dP product, warp 2 the dV/dK products of each half and dQ of
        // the block (the tensor core runs both streams). What one thread's order used to guarantee is
        // explicit: a stage is released by a commit from each warp (qd_empty counts two), a half's
        // packed P^T is overwritten by the next pass only after acc_done(h), and dQ(i) and dK(i, h)
        // have read a half's dS rows by dq_full(i), which the warpgroup waits for before it stages dQ
        // there or, a block later, writes dS there again.
        const uint32_t issue = lane == 0 ? 1u : 0u;
        const uint64_t k_km = smem_desc_sw128(smem_u32(smem + C::SMEM_K), 16, 1024);
        const uint64_t v_km = smem_desc_sw128(smem_u32(smem + C::SMEM_V), 16, 1024);
        const uint64_t k_mn = smem_desc_sw128(smem_u32(smem + C::SMEM_K), C::CHUNK, 1024);
        bool ok = bwd_wait_warp(bar_kv, 0, p);
        if (warp == 1) {
            // S_h^T = K_j Q_h^T, dP_h^T = V_j dO_h^T of block it (query rows 64h.. of the stage = +8 KB)
            auto issue_s = [&](int it, int h) {
                const uint32_t q_s = smem_u32(smem + C::SMEM_QD + (it % ST) * 2 * C::CHUNK);
                const uint64_t q_km = smem_desc_sw128(q_s, 16, 1024);
                const uint64_t do_km = smem_desc_sw128(q_s + C::CHUNK, 16, 1024);
                const uint64_t hoff = (uint64_t)((h * 64 * 128) >> 4);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint64_t off = (uint64_t)((k * 32) >> 4);
                    mma_ss(tmem + 128 * h, k_km + off, q_km + hoff + off, C::ID_S, k > 0 ? 1u : 0u, issue);
                    mma_ss(tmem + 128 * h + 64, v_km + off, do_km + hoff + off, C::ID_S, k > 0 ? 1u : 0u, issue);
                }
                tc_commit(bar_sp_full(h), issue);
            };
            ok = ok && bwd_wait_warp(bar_qd_full(0), 0, p);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                issue_s(0, 1);
                tc_commit(bar_qd_empty(0), issue);  // this warp's last reader of stage 0
            }
            for (int it = 0; ok && it < n_it; ++it) {
                const bool next = it + 1 < n_it;
                ok = bwd_wait_warp(bar_p_full(0), it & 1u, p);  // half A's S/dP columns were read
                if (ok && next) {
                    ok = bwd_wait_warp(bar_qd_full((it + 1) % ST), ((it + 1) / ST) & 1u, p);
                    if (ok) {
                        tc_fence_after();
                        issue_s(it + 1, 0);
                    }
                }
                if (ok) ok = bwd_wait_warp(bar_p_full(1), it & 1u, p);
                if (ok && next) {
                    tc_fence_after();
                    issue_s(it + 1, 1);
                    tc_commit(bar_qd_empty((it + 1) % ST), issue);
                }
            }
        } else {
            // dV_j += P_h^T dO_h (A = packed P^T in TMEM), dK_j += dS_h^T Q_h (A = dS^T, K-major, from the
            // block's dS buffer), contracted over the 64 rows of half h of block it
            auto issue_acc = [&](int it, int h) {
                const uint32_t q_s = smem_u32(smem + C::SMEM_QD + (it % ST) * 2 * C::CHUNK);
                const uint64_t q_mn = smem_desc_sw128(q_s, C::CHUNK, 1024);
                const uint64_t do_mn = smem_desc_sw128(q_s + C::CHUNK, C::CHUNK, 1024);
                const uint64_t dst_km =
                    smem_desc_sw128(smem_u32(smem + C::SMEM_DS + (it & 1) * 2 * C::CHUNK + h * C::CHUNK), 16, 1024);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint64_t off = (uint64_t)(((h * 64 + k * 16) * 128) >> 4);
                    const uint32_t acc = (it > 0 || h > 0 || k > 0) ? 1u : 0u;
                    mma_ts(tmem + 320, tmem + 256 + 32 * h + 8 * k, do_mn + off, C::ID_ACC, acc, issue);
                    mma_ss(tmem + 384, dst_km + (uint64_t)((k * 32) >> 4), q_mn + off, C::ID_ACC, acc, issue);
                }
                tc_commit(bar_acc_done(h), issue);
            };
            for (int it = 0; ok && it < n_it; ++it) {
                const int s = it % ST;
                ok = bwd_wait_warp(bar_p_full(0), it & 1u, p) && bwd_wait_warp(bar_qd_full(s), (it / ST) & 1u, p);
                if (!ok) break;
                tc_fence_after();
                issue_acc(it, 0);
                ok = bwd_wait_warp(bar_p_full(1), it & 1u, p);
                if (!ok) break;
                tc_fence_after();
                issue_acc(it, 1);
                tc_commit(bar_qd_empty(s), issue);  // this warp's last reader of the stage
                if (it > 0) ok = bwd_wait_warp(bar_dq_free, (it - 1) & 1u, p);  // dQ of the last block read out
                if (!ok) break;
                tc_fence_after();
                // dQ_i = dS_i K_j, contracted over the 128 keys (dS buffer it & 1)
                const uint64_t ds_mn =
                    smem_desc_sw128(smem_u32(smem + C::SMEM_DS + (it & 1) * 2 * C::CHUNK), C::CHUNK, 1024);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint64_t off = (uint64_t)((k * 2048) >> 4);
                    mma_ss(tmem + 448, ds_mn + off, k_mn + off, C::ID_DQ, k > 0 ? 1u : 0u, issue);
                }
                tc_commit(bar_dq_full, issue);
            }
        }
        tc_commit(bar_drain, issue);
        if (warp == 1) bwd_wait_warp(bar_drain, 0, p);  // both warps' products, before TMEM is freed
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- gradient warps
        const int g = (warp - 4) >> 2;  // half of the query block
        const int w = warp & 3;
        const int r = w * 32 + lane;    // TMEM lane: key r, later query row r
        const uint32_t lane_base = (uint32_t)(w * 32) << 16;
        const uint32_t s_col = tmem + lane_base + 128u * g;  // S_g; dP_g at +64
        const int key = j * kBlk + r;
        const bool key_ok = key < p.N;
        const bool ragged_keys = (j + 1) * kBlk > p.N;
        const uint32_t ds_row0 = smem_u32(smem + C::SMEM_DS) + g * C::CHUNK + r * 128;  // + (block & 1) * 32 KB
        // dQ of block b is staged in this warp's own 32 rows of b's dS buffer: dK(b) and dQ(b) have read it by
        // the time dQ(b) is read out, and this warp writes those rows again only in the pass of block b + 2
        const uint32_t box0 = smem_u32(smem + C::SMEM_DS) + g * C::CHUNK + w * 4096;  // + (block & 1) * 32 KB
        const uint32_t stats0 = smem_u32(smem + C::SMEM_STATS) + g * 1024;  // + buffer * 512
        // thread r hands over -lse2 (r < 64) or -D (r >= 64) of query row 64g + (r & 63)
        const float *stat_src = (r < 64 ? p.lse2 : p.dsum) + (size_t)bh * p.Npad + 64 * g + (r & 63);
        grid_dependency_wait();  // statistics and the zeroed dQ accumulator are written by fa_bwd_pre
        float stat_next = -__ldg(stat_src + i0 * kBlk);
        bool ok = true;
        auto readout = [&](int blk) -> bool {  // dQ rows of query block blk, head columns 32g..32g+31
            if (!bwd_wait_warp(bar_dq_full, (uint32_t)(blk - i0) & 1u, p)) return false;
            tc_fence_after();
            uint32_t qv[32];
            tmem_ld32_wait(tmem + lane_base + 448 + 32 * g, qv);
            tc_fence_before();
            mbar_arrive(bar_dq_free);
            const uint32_t box = box0 + ((blk - i0) & 1) * 2 * C::CHUNK;
            stage_and_reduce_dq(&tm_dq, box, qv, p.scale, lane, 32 * g, blk * kBlk + w * 32, bh);
            return true;
        };
        for (int it = 0; ok && it < n_it; ++it) {
            const int i = i0 + it;
            const uint32_t stats = stats0 + (it & 1) * 512;
            st_shared_f32(stats + r * 4, stat_next);
            mbar_arrive(bar_stats(g));
            ok = bwd_wait_warp(bar_stats(g), it & 1u, p) && bwd_wait_warp(bar_sp_full(g), it & 1u, p);
            if (!ok) break;
            tc_fence_after();
            const bool need_mask = ragged_keys || (CAUSAL && i == j);
            const uint32_t ds_row = ds_row0 + (it & 1) * 2 * C::CHUNK;
            // the reduction of dQ(i - 2), staged in these rows, must have read them
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            // dV(i - 1, g) read this half's packed P^T before it is overwritten below
            if (it > 0 && !bwd_wait_warp(bar_acc_done(g), (it - 1) & 1u, p)) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < 64; c0 += 32) {
                uint32_t sv[32], dpv[32];
                tmem_ld32x2_wait(s_col + c0, sv, s_col + 64 + c0, dpv);
                uint32_t pp[16], dsp[16];
                if (need_mask)
                    p_ds_chunk<T, CAUSAL, true>(sv, dpv, stats + c0 * 4, stats + (64 + c0) * 4, p.scale_log2, true,
                                                key_ok, key, i * kBlk + 64 * g + c0, pp, dsp);
                else
                    p_ds_chunk<T, CAUSAL, false>(sv, dpv, stats + c0 * 4, stats + (64 + c0) * 4, p.scale_log2, false,
                                                 key_ok, key, i * kBlk + 64 * g + c0, pp, dsp);
                tmem_st16(tmem + lane_base + 256u + 32u * g + c0 / 2, pp);  // packed P^T of half g
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t unit = (uint32_t)((c0 / 8 + u) ^ (r & 7));
                    st_shared_v4(ds_row + unit * 16, dsp[4 * u], dsp[4 * u + 1], dsp[4 * u + 2], dsp[4 * u + 3]);
                }
            }
            tmem_wait_st();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar_p_full(g));
            if (it + 1 < n_it) stat_next = -__ldg(stat_src + (i + 1) * kBlk);
            if (it > 0) ok = readout(i - 1);
        }
        if (ok) ok = readout(i0 + n_it - 1);
        // ---------------------------------------------------------------- dV_j (half A's group), dK_j (B's)
        if (ok) {  // the last dq_full covers every dV and dK product
            tc_fence_after();
            const float mul = g == 0 ? 1.0f : p.scale;
            T *dst = reinterpret_cast<T *>(g == 0 ? p.dv : p.dk) + ((size_t)bh * p.N + (size_t)(key_ok ? key : 0)) * 64;
            uint32_t a[32], b[32];
            tmem_ld32x2_wait(tmem + lane_base + 320 + 64 * g, a, tmem + lane_base + 320 + 64 * g + 32, b);
            if (key_ok) {
#pragma unroll
                for (int c = 0; c < 32; c += 8) {
                    st_global_v4(dst + c, pk2<T>(__uint_as_float(a[c]) * mul, __uint_as_float(a[c + 1]) * mul),
                                 pk2<T>(__uint_as_float(a[c + 2]) * mul, __uint_as_float(a[c + 3]) * mul),
                                 pk2<T>(__uint_as_float(a[c + 4]) * mul, __uint_as_float(a[c + 5]) * mul),
                                 pk2<T>(__uint_as_float(a[c + 6]) * mul, __uint_as_float(a[c + 7]) * mul));
                    st_global_v4(dst + 32 + c, pk2<T>(__uint_as_float(b[c]) * mul, __uint_as_float(b[c + 1]) * mul),
                                 pk2<T>(__uint_as_float(b[c + 2]) * mul, __uint_as_float(b[c + 3]) * mul),
                                 pk2<T>(__uint_as_float(b[c + 4]) * mul, __uint_as_float(b[c + 5]) * mul),
                                 pk2<T>(__uint_as_float(b[c + 6]) * mul, __uint_as_float(b[c + 7]) * mul));
                }
            }
        }
        if (lane == 0) bulk_wait_all();  // the dQ reductions, behind the dV / dK stores
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Row statistics for the backward:
//   dsum = sum_t dO_t O_t (0 past N), lse2 = lse * log2(e) (+inf past N),
// and the row's dQ accumulator is zeroed. D / 8 consecutive threads share a
// padded row, each with 8 elements (one 16-byte load of O and of dO, two
// 16-byte stores of zeros); the row sum is a shuffle tree within the group.
template <typename T, int D>
__global__ void __launch_bounds__(256) fa_bwd_pre(const T *__restrict__ out, const T *__restrict__ dout,
                                                  const float *__restrict__ lse, float *__restrict__ lse2,
                                                  float *__restrict__ dsum, float *__restrict__ dq_acc, int BH,
                                                  int N, int Npad) {
    constexpr int TPR = D / 8;          // threads per row (8 or 16: a power of two dividing 32)
    constexpr int RPB = 256 / TPR;      // rows per CTA
    grid_launch_dependents();
    const int64_t prow = (int64_t)blockIdx.x * RPB + threadIdx.x / TPR;
    const int t = threadIdx.x % TPR;
    const bool in = prow < (int64_t)BH * Npad;
    const int64_t bh = in ? prow / Npad : 0;
    const int i = in ? (int)(prow - bh * Npad) : 0;
    const bool real = in && i < N;
    const int64_t row = bh * N + i;
    float acc = 0.f;
    if (real) {
        const uint4 o = *reinterpret_cast<const uint4 *>(out + row * D + t * 8);
        const uint4 g = *reinterpret_cast<const uint4 *>(dout + row * D + t * 8);
        const uint32_t ov[4] = {o.x, o.y, o.z, o.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float2 of = up2<T>(ov[u]), gf = up2<T>(gv[u]);
            acc = fmaf(of.x, gf.x, acc);
            acc = fmaf(of.y, gf.y, acc);
        }
        float4 *z = reinterpret_cast<float4 *>(dq_acc + row * D + t * 8);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // every lane takes part (rows past the end contribute 0); xor < TPR stays within the row's group
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (in && t == 0) {
        dsum[prow] = real ? acc : 0.0f;
        lse2[prow] = real ? lse[row] * 1.4426950408889634f : INFINITY;
    }
}

// dQ accumulator -> output type; launched as a programmatic dependent of the
// backward kernel, whose reductions into the accumulator it waits for.
template <typename T>
__global__ void __launch_bounds__(256) fa_bwd_post(const float *__restrict__ dq_acc, T *__restrict__ dq, size_t n4) {
    grid_dependency_wait();
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
    // d = 64 runs the overlapped half-block kernel; d = 128 (tensor memory full) the serial one
    auto kern = [] {
        if constexpr (D == 64) return fa_bwd_kernel_h64<T, CAUSAL>;
        else return fa_bwd_kernel<T, D, CAUSAL>;
    }();
    constexpr int smem_bytes = D == 64 ? BwdCfgH64<T>::SMEM_BYTES : BwdCfg<T, D>::SMEM_BYTES;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) != cudaSuccess)
        return -5;
    const int BH = a.B * a.H;
    const int Npad = static_cast<int>(bwd_padded_rows(a.N));
    const int64_t prows = static_cast<int64_t>(BH) * Npad;
    constexpr int kPreRows = 256 / (D / 8);  // padded rows per CTA of fa_bwd_pre
    fa_bwd_pre<T, D><<<static_cast<unsigned>((prows + kPreRows - 1) / kPreRows), 256, 0, a.stream>>>(
        static_cast<const T *>(a.out), static_cast<const T *>(a.dout), a.lse, a.lse2, a.dsum, a.dq_acc, BH, a.N,
        Npad);
    if (cudaGetLastError() != cudaSuccess) return -5;
    CUtensorMap tq, tk, tv, tdo;
    if (!encode_rows_map(&tq, Elem<T>::tma, 2, a.q, D, a.N, BH, kBlk)) return -5;
    if (!encode_rows_map(&tk, Elem<T>::tma, 2, a.k, D, a.N, BH, kBlk)) return -5;
    if (!encode_rows_map(&tv, Elem<T>::tma, 2, a.v, D, a.N, BH, kBlk)) return -5;
    if (!encode_rows_map(&tdo, Elem<T>::tma, 2, a.dout, D, a.N, BH, kBlk)) return -5;
    CUtensorMap tdq;  // fp32 dQ accumulator, 32 x 32 boxes (128-byte rows), reduced into
    if (!encode_rows_map(&tdq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, a.dq_acc, D, a.N, BH, 32)) return -5;
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
    // programmatic dependents: the backward's copies of K, V, Q, dO start while fa_bwd_pre drains (its
    // gradient warps wait for the statistics), and fa_bwd_post's launch overlaps the backward's tail
    if (launch_dependent(kern, dim3(static_cast<unsigned>(grid)), dim3(kBwdThreads), smem_bytes, a.stream, tq, tk,
                         tv, tdo, tdq, p) != cudaSuccess)
        return -5;
    const size_t n4 = static_cast<size_t>(BH) * a.N * D / 4;
    if (launch_dependent(fa_bwd_post<T>, dim3(static_cast<unsigned>((n4 + 255) / 256)), dim3(256), 0, a.stream,
                         static_cast<const float *>(a.dq_acc), static_cast<T *>(a.dq), n4) != cudaSuccess)
        return -5;
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
