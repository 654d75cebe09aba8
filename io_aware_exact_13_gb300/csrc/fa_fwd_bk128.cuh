// fa_fwd_bk128.cuh -- the exact tiled attention forward with 128-key K/V blocks,
// for sm_103a (no mask, or a mask of 0 and -inf entries in its one-bit form).
//
// Same computation as fa_fwd_kernel.cuh ("FlashAttention: Exact Attention as an
// IO-Aware Streaming Computation", sections "Core idea" and "Mathematical
// structure"; "IO-aware exact attention", section "One tiled forward-pass
// iteration"): a 256-row work item keeps two 128-row query tiles on chip with
// their running (m, l, a); K/V blocks stream past them; S, P and O live in
// tensor memory; only O and lse are written.
//
// Why 128-key blocks: one warp issues about one tcgen05.mma every 77-84 cycles
// whatever its size, even alternating between several accumulators, and the
// tensor core keeps up with two or more issuing warps: an M=128 K=16 product
// with N = 128 takes 64 cycles at the full rate, one with N = 64 takes 48 (its
// shared-memory operands are the limit, 67 % of the rate). So S = Q K^T
// products over 128 keys cost half the tensor time per flop of 64-key ones.
//
// Tensor memory (512 columns) holds ONE S buffer that the two tiles use in turn
// (S_0(j), S_1(j), S_0(j+1), ...), P_0 and P_1 (16-bit, 64 columns each) and
// O_0, O_1 (D columns each):
//   S [0, 128) | P_0 [128, 192) | P_1 [192, 256) | O_0 [256, 256 + D) | O_1 [256 + D, 256 + 2D)
// The softmax copies S to registers and releases the buffer at once, so the
// next S product never waits for a P V product; P_t(j+1) is stored after
// P V_t(j) has read P_t(j). (Keeping an S buffer per tile leaves no room for P
// at D = 128; P written over S makes the next S wait until the same warp has
// issued the P V product, which put about 1200 cycles of issue into every
// block's dependency chain.)
//
// Softmax: warpgroup t works on tile t; thread r owns query row r (TMEM lane r)
// and all 128 keys of a block, so no two threads share a row. The two tiles'
// S products alternate in the S buffer, so the two warpgroups' softmax passes
// overlap in time: while one runs its exponent loop, the other loads, reduces
// or stores. (Both warpgroups on one tile at a time, 64 keys each with the row
// maximum exchanged through shared memory, ran the passes back to back: about
// 1650 cycles per tile and block, nearly twice the tensor time.)
//
// Roles (16 warps, one persistent CTA per SM):
//   warps 0-3   softmax + epilogue of query tile 0
//   warps 4-7   softmax + epilogue of query tile 1
//   warp  8     TMA producer: Q tiles per item, then K and V rings
//   warp  9     S issuer: S_t(j) = Q_t K_j^T for t = 0, 1 in turn, into the S buffer
//   warps 10-11 P V issuer of tile t = warp - 10: O_t += P_t(j) V_j, issued after S_t(j+1)
//   warp  12    packed batch only: publishes the CTA's work items (ItemRing)
//   warps 13-15 idle (they complete the last warpgroup)
// Shared memory holds no static variables: the abort word and the item ring
// live after the barriers in the dynamic region.
#pragma once
#include "fa_fwd_kernel.cuh"

namespace fa {

constexpr int kBK128 = 128;           // keys per K/V block
constexpr int kItemConsumers128 = 12; // producer, three issuers, eight softmax warps
constexpr int kStatusSmemAlign = -5;  // device status: the dynamic shared memory base was misaligned

template <typename T, int D>
struct Cfg128 {
    static constexpr int EB = sizeof(T);
    static constexpr int ROW_BYTES = D * EB;
    static constexpr int CHUNK_ELEMS = 128 / EB;       // elements per 128-byte swizzle row
    static constexpr int NCH = ROW_BYTES / 128;        // swizzle chunks per row
    static constexpr int Q_CHUNK = kBQ * 128;          // 128 rows x 128 bytes
    static constexpr int KV_CHUNK = kBK128 * 128;      // 128 keys x 128 bytes
    static constexpr int Q_TILE = NCH * Q_CHUNK;
    static constexpr int KV_TILE = NCH * KV_CHUNK;
    static constexpr int KSTEPS_S = ROW_BYTES / 32;    // 32 bytes of the head dim per MMA
    static constexpr int KSTEPS_PV = kBK128 / 16;      // 16 keys per MMA
    static constexpr int V_KSTEP_BYTES = 16 * 128;     // 16 key rows x 128 bytes
    static constexpr uint32_t IDESC_S = make_idesc(Elem<T>::fmt, 128, kBK128, 0);
    static constexpr uint32_t IDESC_PV = make_idesc(Elem<T>::fmt, 128, D, 1);
    // tensor memory columns: S | P_0 P_1 | O_0 O_1
    static constexpr int TM_S = 0;
    static constexpr int TM_P = 128;                   // P_t at TM_P + 64 t
    static constexpr int TM_O = 256;                   // O_t at TM_O + D t
    // shared memory: Q0 Q1 | K ring | V ring | barriers
    static constexpr int SMEM_Q = 0;
    static constexpr int SMEM_K = 2 * Q_TILE;
    static constexpr int FREE = 232448 - 1024 - 512 - SMEM_K;
    static constexpr int SLOTS = FREE / KV_TILE > 12 ? 12 : FREE / KV_TILE;
    static constexpr int RK = (SLOTS + 1) / 2;         // K slots (the S products run ahead of the P V ones)
    static constexpr int RV = SLOTS - RK;              // V slots
    static constexpr int SMEM_V = SMEM_K + RK * KV_TILE;
    static constexpr int SMEM_BAR = SMEM_V + RV * KV_TILE;
    // q_full[2] q_empty[2] k_full[RK] k_empty[RK] v_full[RV] v_empty[RV] s_full[2] s_free p_full[2]
    // pv_done[2][2] drain s_issued[2][2]
    static constexpr int NUM_BARS = 4 + 2 * RK + 2 * RV + 9 + 1 + 4;
    static constexpr int SMEM_TMEM_SLOT = SMEM_BAR + ((NUM_BARS * 8 + 15) / 16) * 16;
    static constexpr int SMEM_RING = SMEM_TMEM_SLOT + 16;         // ItemRing (packed batches)
    static constexpr int SMEM_ABORT = SMEM_RING + 128;
    static constexpr int SMEM_USED = SMEM_ABORT + 16;
    // up to 1024 bytes to align the base (SW128 tiles need 1024-byte alignment), within the 227 KB limit
    static constexpr int SMEM_BYTES = SMEM_USED + 1024 <= 232448 ? SMEM_USED + 1024 : 232448;
    static constexpr int SLACK = SMEM_BYTES - SMEM_USED;
    static_assert(NCH >= 1 && ROW_BYTES % 128 == 0, "row must be a whole number of 128-byte swizzle rows");
    static_assert(RK >= 2 && RV >= 2, "K/V rings too small");
    static_assert(SLACK >= 256, "shared memory budget");
    static_assert(TM_O + 2 * D <= 512, "tensor memory budget");
};

template <int RK, int RV>
struct Sync128 {
    uint64_t *bars;
    static constexpr int B0 = 4 + 2 * RK + 2 * RV;
    __device__ __forceinline__ uint32_t at(int i) const { return smem_u32(bars + i); }
    __device__ __forceinline__ uint32_t q_full(int t) const { return at(t); }
    __device__ __forceinline__ uint32_t q_empty(int t) const { return at(2 + t); }
    __device__ __forceinline__ uint32_t k_full(int s) const { return at(4 + s); }
    __device__ __forceinline__ uint32_t k_empty(int s) const { return at(4 + RK + s); }
    __device__ __forceinline__ uint32_t v_full(int s) const { return at(4 + 2 * RK + s); }
    __device__ __forceinline__ uint32_t v_empty(int s) const { return at(4 + 2 * RK + RV + s); }
    // S ready for tile t (MMA commit), the S buffer copied out (the 128 threads of the
    // tile's warpgroup), P ready for tile t (the same 128), P V_t(g) done (MMA commit to
    // pv_done(t, g & 1)). No barrier can get two phases ahead of a waiter (see the
    // roles below), so parity waits are exact.
    __device__ __forceinline__ uint32_t s_full(int t) const { return at(B0 + t); }
    __device__ __forceinline__ uint32_t s_free() const { return at(B0 + 2); }
    __device__ __forceinline__ uint32_t p_full(int t) const { return at(B0 + 3 + t); }
    __device__ __forceinline__ uint32_t pv_done(int t, int b) const { return at(B0 + 5 + 2 * t + b); }
    __device__ __forceinline__ uint32_t drain() const { return at(B0 + 9); }
    // S_t(g) issued (the S issuer's lane 0 arrives once its products are in the queue)
    __device__ __forceinline__ uint32_t s_issued(int t, int b) const { return at(B0 + 10 + 2 * t + b); }
};

// Row maximum of 128 values: eight independent three-input chains, then a short tree.
__device__ __forceinline__ float row_max128(const float (&x)[128]) {
    float m8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m8[i] = fmax3(x[i], x[8 + i], x[16 + i]);
#pragma unroll
    for (int c = 24; c < 120; c += 16) {
#pragma unroll
        for (int i = 0; i < 8; ++i) m8[i] = fmax3(m8[i], x[c + i], x[c + 8 + i]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], x[120 + i]);
    return fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
}

// Philox4x64-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as
// 1, 2, 3", SC 2011): ten rounds on a 256-bit counter; each multiplies counter words 0 and 2
// by the two multipliers and mixes the halves of the products with words 1 and 3 and the round
// key, which the two Weyl constants bump between rounds. The 256-bit result is returned as
// eight 32-bit words, least significant first.
__device__ __forceinline__ void philox4x64_10(uint64_t c0, uint64_t c1, uint64_t c2, uint64_t c3, uint64_t k0,
                                              uint64_t k1, uint32_t (&w)[8]) {
    constexpr uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
    constexpr uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint64_t lo0 = M0 * c0, hi0 = __umul64hi(M0, c0);
        const uint64_t lo1 = M1 * c2, hi1 = __umul64hi(M1, c2);
        c0 = hi1 ^ c1 ^ k0;
        c1 = lo1;
        c2 = hi0 ^ c3 ^ k1;
        c3 = lo0;
        k0 += W0;
        k1 += W1;
    }
    w[0] = (uint32_t)c0, w[1] = (uint32_t)(c0 >> 32), w[2] = (uint32_t)c1, w[3] = (uint32_t)(c1 >> 32);
    w[4] = (uint32_t)c2, w[5] = (uint32_t)(c2 >> 32), w[6] = (uint32_t)c3, w[7] = (uint32_t)(c3 >> 32);
}

// MASK: an additive [B][N][N] mask whose entries are all 0 or -inf, in its packed form
// (p.mask_bits, one bit per entry, set = -inf; see fa_mask_pack.cu). Thread r reads the 16
// bytes of its row and key block from global memory (L2: the packed mask of a batch index is
// shared by its heads), one block ahead of its use.
// DROP: dropout ("IO-aware exact attention", section "Why implementations form a family",
// names the variant). The softmax keeps the row maximum and sum of the undropped scores (lse
// is unchanged); P is stored with dropped keys set to 0, and the epilogue multiplies O by
// 1 / q. The keep bytes of a 32-key group come from one Philox block (see FwdParams).
template <typename T, int D, bool CAUSAL, bool VARLEN, bool MASK = false, bool DROP = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_bk128_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    static_assert(!(VARLEN && MASK), "no mask in a packed batch");
    static_assert(!(DROP && (VARLEN || MASK)), "dropout with dense unmasked inputs only");
    using C = Cfg128<T, D>;
    constexpr int RK = C::RK, RV = C::RV;
    if constexpr (MASK) {
        grid_dependency_wait();  // launched behind the packing pass: its verdict and bits
        if (*p.mask_kind != 0) return;  // the mask had other values: the 64-key kernel applies it as given
        grid_launch_dependents();  // that kernel (queued next) may take the SMs this grid leaves idle
    }
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (uint32_t)((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    if (pad > (uint32_t)C::SLACK) {  // cannot happen with no static shared memory; never overflow
        if (threadIdx.x == 0) atomicExch(p.status, kStatusSmemAlign);
        return;
    }
    uint8_t *smem = smem_raw + pad;
    Sync128<RK, RV> sy{reinterpret_cast<uint64_t *>(smem + C::SMEM_BAR)};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::SMEM_TMEM_SLOT);
    ItemRing *ring = reinterpret_cast<ItemRing *>(smem + C::SMEM_RING);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::SMEM_ABORT);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(sy.q_full(t), 1);
            mbar_init(sy.q_empty(t), 1);
            mbar_init(sy.s_full(t), 1);
            mbar_init(sy.p_full(t), kBQ);  // the tile's softmax warpgroup
            mbar_init(sy.pv_done(t, 0), 1);
            mbar_init(sy.pv_done(t, 1), 1);
        }
        mbar_init(sy.s_free(), kBQ);  // the warpgroup of the tile whose S the buffer holds
        for (int t = 0; t < 2; ++t) {
            mbar_init(sy.s_issued(t, 0), 1);
            mbar_init(sy.s_issued(t, 1), 1);
        }
        for (int s = 0; s < RK; ++s) {  // a K slot is released by the S issuer
            mbar_init(sy.k_full(s), 1);
            mbar_init(sy.k_empty(s), 1);
        }
        for (int s = 0; s < RV; ++s) {  // a V slot by both P V issuers
            mbar_init(sy.v_full(s), 1);
            mbar_init(sy.v_empty(s), 2);
        }
        mbar_init(sy.drain(), 3);  // one commit per issuing warp
        if constexpr (VARLEN) {
            for (int i = 0; i < kItemRing; ++i) {
                mbar_init(smem_u32(&ring->full[i]), 1);
                mbar_init(smem_u32(&ring->empty[i]), kItemConsumers128);
            }
        }
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
    if constexpr (!MASK) {
        // Launched as a programmatic dependent of the work ahead on the stream: the set-up above overlaps
        // its tail, and nothing in global memory is read or written before it is complete. The next
        // forward may likewise be scheduled onto the SMs this grid frees.
        grid_launch_dependents();
        grid_dependency_wait();
    }

    if (warp >= 8) {
        setmaxnreg_dec<72>();
        if (warp == 8) {
            // ---------------------------------------------------------- TMA producer
            // Load order per item: Q tiles, K_0, then K_{j+1}, V_j for j = 0 .. nmax-1
            // (the order in which the issuers consume them).
            const bool leader = lane == 0;
            const uint64_t pol_kv = policy_evict_last();
            const uint64_t pol_q = policy_evict_first();
            uint32_t qcount[2] = {0, 0};
            uint32_t kpos = 0, vpos = 0;
            int kv_y = 0, kv_z = 0, tok0 = 0;
            bool ok = true;
            auto load_kv = [&](bool is_v, int blk) -> bool {
                uint32_t &pos = is_v ? vpos : kpos;
                const int R = is_v ? RV : RK;
                const int s = pos % R;
                const uint32_t full = is_v ? sy.v_full(s) : sy.k_full(s);
                const uint32_t empty = is_v ? sy.v_empty(s) : sy.k_empty(s);
                if (!wait_warp(empty, ((pos / R) & 1u) ^ 1u, abort_flag, p)) return false;
                if (leader) {
                    const uint32_t dst = smem_u32(smem + (is_v ? C::SMEM_V : C::SMEM_K) + s * C::KV_TILE);
                    mbar_arrive_expect_tx(full, C::KV_TILE);
#pragma unroll
                    for (int c = 0; c < C::NCH; ++c)
                        tma_load_3d(dst + c * C::KV_CHUNK, is_v ? &tm_v : &tm_k, full, c * C::CHUNK_ELEMS,
                                    VARLEN ? kv_y : blk * kBK128, VARLEN ? tok0 + blk * kBK128 : kv_z, pol_kv);
                }
                __syncwarp();
                ++pos;
                return true;
            };
            ItemIter<VARLEN> iter(p, abort_flag, ring);
            for (Item itm; ok && iter.next(p, itm, ok);) {
                const int q0 = itm.q0, cur_bh = itm.bh;
                const int kv_h = (cur_bh % p.H) / p.kv_group;  // grouped-query: kv_group query heads per K/V head
                if (VARLEN) {
                    kv_y = kv_h;
                    tok0 = itm.tok0;
                } else {
                    kv_z = (cur_bh / p.H) * (p.H / p.kv_group) + kv_h;
                }
                const int n0 = tile_nkv<CAUSAL, kBK128>(itm, 0), n1 = tile_nkv<CAUSAL, kBK128>(itm, 1);
                const int nmax = max(n0, n1);
                for (int t = 0; t < 2 && ok; ++t) {
                    if ((t == 0 ? n0 : n1) == 0) continue;
                    ok = wait_warp(sy.q_empty(t), (qcount[t] & 1u) ^ 1u, abort_flag, p);
                    if (!ok) break;
                    if (leader) {
                        const uint32_t dst = smem_u32(smem + C::SMEM_Q + t * C::Q_TILE);
                        mbar_arrive_expect_tx(sy.q_full(t), C::Q_TILE);
#pragma unroll
                        for (int c = 0; c < C::NCH; ++c)
                            tma_load_3d(dst + c * C::Q_CHUNK, &tm_q, sy.q_full(t), c * C::CHUNK_ELEMS,
                                        VARLEN ? cur_bh % p.H : q0 + t * kBQ,
                                        VARLEN ? tok0 + q0 + t * kBQ : cur_bh, pol_q);
                    }
                    __syncwarp();
                    ++qcount[t];
                }
                // an item with no rows loads nothing: every slot filled here is consumed by the issuers
                if (ok && nmax > 0) ok = load_kv(false, 0);
                for (int j = 0; ok && j < nmax; ++j) {
                    if (j + 1 < nmax) ok = load_kv(false, j + 1);
                    if (ok) ok = load_kv(true, j);
                }
            }
            if (!ok && leader) {  // let every copy in flight land before the CTA can exit
                const uint64_t t0 = global_timer_ns();
                for (int t = 0; t < 2; ++t)
                    if (qcount[t] > 0)
                        while (!mbar_try_wait(sy.q_full(t), (qcount[t] - 1) & 1u) &&
                               global_timer_ns() - t0 < p.timeout_ns) {
                        }
                for (uint32_t q = kpos > (uint32_t)RK ? kpos - RK : 0; q < kpos; ++q)
                    while (!mbar_try_wait(sy.k_full(q % RK), (q / RK) & 1u) && global_timer_ns() - t0 < p.timeout_ns) {
                    }
                for (uint32_t q = vpos > (uint32_t)RV ? vpos - RV : 0; q < vpos; ++q)
                    while (!mbar_try_wait(sy.v_full(q % RV), (q / RV) & 1u) && global_timer_ns() - t0 < p.timeout_ns) {
                    }
            }
        } else if (warp == 9) {
            // ---------------------------------------------------------- S issuer
            // S_t(j) = Q_t K_j^T for t = 0, 1 in turn (blocks a tile does not need are
            // skipped), each into the S buffer once the softmax has copied the previous S
            // out. The whole warp runs the loop (warp-uniform), lane 0 issues.
            const uint32_t issue = lane == 0 ? 1u : 0u;
            const uint64_t qd0 = smem_desc_sw128(smem_u32(smem + C::SMEM_Q), 16, 1024);
            const uint64_t kd0 = smem_desc_sw128(smem_u32(smem + C::SMEM_K), 16, 1024);
            const uint32_t d_s = tmem + C::TM_S;
            constexpr uint64_t KVT16 = C::KV_TILE >> 4;
            constexpr uint64_t QT16 = C::Q_TILE >> 4;
            uint32_t qcount[2] = {0, 0}, kpos = 0, s_issued = 0;
            uint32_t sg[2] = {0, 0};  // S products of each tile so far
            bool ok = true;
            ItemIter<VARLEN> iter(p, abort_flag, ring);
            for (Item itm; ok && iter.next(p, itm, ok);) {
                const int nt[2] = {tile_nkv<CAUSAL, kBK128>(itm, 0), tile_nkv<CAUSAL, kBK128>(itm, 1)};
                const int nmax = max(nt[0], nt[1]);
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (ok && nt[t] > 0) {
                        ok = wait_warp(sy.q_full(t), qcount[t] & 1u, abort_flag, p);
                        ++qcount[t];
                    }
                }
                for (int j = 0; ok && j < nmax; ++j) {
                    const int slot = kpos % RK;
                    ok = wait_warp(sy.k_full(slot), (kpos / RK) & 1u, abort_flag, p);
                    ++kpos;
                    if (!ok) break;
#pragma unroll
                    for (int t = 0; t < 2; ++t) {
                        if (!ok || j >= nt[t]) continue;
                        if (s_issued > 0) ok = wait_warp(sy.s_free(), (s_issued - 1) & 1u, abort_flag, p);
                        if (!ok) break;
                        ++s_issued;
                        tc_fence_after();
                        const uint64_t a0 = qd0 + t * QT16;
                        const uint64_t b0 = kd0 + slot * KVT16;
#pragma unroll
                        for (int k = 0; k < C::KSTEPS_S; ++k) {
                            const uint64_t aoff = (uint64_t)(((k / 4) * C::Q_CHUNK + (k % 4) * 32) >> 4);
                            const uint64_t boff = (uint64_t)(((k / 4) * C::KV_CHUNK + (k % 4) * 32) >> 4);
                            mma_ss(d_s, a0 + aoff, b0 + boff, C::IDESC_S, k > 0 ? 1u : 0u, issue);
                        }
                        tc_commit(sy.s_full(t), issue);
                        if (j == nt[t] - 1) tc_commit(sy.q_empty(t), issue);
                        if (lane == 0) mbar_arrive(sy.s_issued(t, sg[t] & 1u));
                        ++sg[t];
                    }
                    tc_commit(sy.k_empty(slot), issue);  // after the last product that reads K_j
                }
            }
            __syncwarp();
            tc_commit(sy.drain(), issue);
        } else if (warp == 10 || warp == 11) {
            // ---------------------------------------------------------- P V issuer of tile t
            // O_t (+)= P_t(j) V_j once the softmax has written P_t(j); the g-th product of the
            // tile is committed to pv_done(t, g & 1). V slots of blocks this tile does not
            // need are released at once.
            const int t = warp - 10;
            const uint32_t issue = lane == 0 ? 1u : 0u;
            const uint64_t vd0 = smem_desc_sw128(smem_u32(smem + C::SMEM_V), C::KV_CHUNK, 1024);
            const uint32_t d_o = tmem + C::TM_O + D * t;
            const uint32_t a_p = tmem + C::TM_P + 64 * t;
            constexpr uint64_t KVT16 = C::KV_TILE >> 4;
            uint32_t vpos = 0, pcount = 0;
            bool ok = true;
            ItemIter<VARLEN> iter(p, abort_flag, ring);
            for (Item itm; ok && iter.next(p, itm, ok);) {
                const int nt = tile_nkv<CAUSAL, kBK128>(itm, t);
                const int nmax = max(tile_nkv<CAUSAL, kBK128>(itm, 0), tile_nkv<CAUSAL, kBK128>(itm, 1));
                for (int j = 0; ok && j < nmax; ++j) {
                    const int slot = vpos % RV;
                    ok = wait_warp(sy.v_full(slot), (vpos / RV) & 1u, abort_flag, p);
                    ++vpos;
                    if (!ok) break;
                    if (j >= nt) {
                        if (lane == 0) mbar_arrive(sy.v_empty(slot));
                        continue;
                    }
                    ok = wait_warp(sy.p_full(t), pcount & 1u, abort_flag, p);
                    // The tile's next S product goes into the tensor core's queue first: this product
                    // is not on the critical path, S(j+1) is (the softmax waits for it).
                    if (ok && j + 1 < nt)
                        ok = wait_warp(sy.s_issued(t, (pcount + 1) & 1u), ((pcount + 1) >> 1) & 1u, abort_flag, p);
                    ++pcount;
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t b0 = vd0 + slot * KVT16;
#pragma unroll
                    for (int k = 0; k < C::KSTEPS_PV; ++k)
                        mma_ts(d_o, a_p + k * 8, b0 + (uint64_t)((k * C::V_KSTEP_BYTES) >> 4), C::IDESC_PV,
                               (k > 0 || j > 0) ? 1u : 0u, issue);
                    tc_commit(sy.pv_done(t, (pcount - 1) & 1u), issue);
                    tc_commit(sy.v_empty(slot), issue);
                }
            }
            __syncwarp();
            tc_commit(sy.drain(), issue);
        } else if (VARLEN && warp == 12) {
            // ---------------------------------------------------------- packed-batch item list
            VarlenCursor cur(p);
            bool more = true;
            for (uint32_t i = 0; more; ++i) {
                Item it;
                more = cur.next(p, it);
                const uint32_t slot = i % kItemRing;
                if (!wait_warp(smem_u32(&ring->empty[slot]), ((i / kItemRing) & 1u) ^ 1u, abort_flag, p)) break;
                if (lane == 0) {
                    ring->desc[slot] = more ? make_int4(it.bh, it.q0, it.n, it.tok0) : make_int4(-1, 0, 0, 0);
                    mbar_arrive(smem_u32(&ring->full[slot]));
                }
                __syncwarp();
            }
        }
    } else {
        setmaxnreg_inc<184>();
        // -------------------------------------------------------------- softmax + epilogue
        const int t = warp >> 2;  // query tile of this warpgroup
        const int r = threadIdx.x & 127;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_addr = tmem + lane_base + C::TM_S;
        const uint32_t p_addr = tmem + lane_base + C::TM_P + 64 * t;
        const uint32_t o_addr = tmem + lane_base + C::TM_O + D * t;
        const float scale_log2 = p.scale_log2;
        // raw scores scaled inside the exponent when the scale is positive (the maximum
        // commutes with it); otherwise pre-scaled scores (a -inf raw score times a
        // non-positive scale is not -inf)
        const bool fast = scale_log2 > 0.0f;
        const float sl2 = fast ? scale_log2 : 1.0f;
        uint32_t scount = 0;  // S products of this tile consumed (all items)
        uint32_t g = 0;       // P blocks produced (all items) = P V products of this tile
        bool ok = true;
        ItemIter<VARLEN> iter(p, abort_flag, ring);
        for (Item itm; ok && iter.next(p, itm, ok);) {
            const int bh = itm.bh, q0 = itm.q0, n = itm.n;
            const int nt = tile_nkv<CAUSAL, kBK128>(itm, t);
            if (nt == 0) continue;
            const int row = q0 + t * kBQ + r;  // query row within the sequence (may be >= n in a ragged tail)
            const int tile_row0 = q0 + t * kBQ;
            float m_ref = -INFINITY, l = 0.0f;
            // packed mask: this row's 16-byte units (a row past the end reads row 0; its output is not stored)
            const uint4 *bits_row = nullptr;
            uint4 bits = make_uint4(0u, 0u, 0u, 0u);
            if constexpr (MASK) {
                bits_row = p.mask_bits +
                           ((size_t)(bh / p.H) * p.N + (size_t)(row < n ? row : 0)) * (size_t)p.mask_bits_blk;
                bits = __ldg(bits_row);
            }
            for (int j = 0; j < nt; ++j, ++g) {
                ok = wait_warp(sy.s_full(t), scount & 1u, abort_flag, p);
                ++scount;
                if (!ok) break;
                tc_fence_after();
                float x[128];
                {
                    uint32_t sr[128];
                    tmem_ld128_wait(s_addr, sr);
                    if (fast) {  // warp-uniform
#pragma unroll
                        for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(sr[c]);
                    } else {
#pragma unroll
                        for (int c = 0; c < 128; ++c) x[c] = __uint_as_float(sr[c]) * scale_log2;
                    }
                }
                tc_fence_before();
                mbar_arrive(sy.s_free());  // the S buffer may now take the next product
                if constexpr (MASK) {
                    // bit e of word c is key 4 e + c of the block; the next block's bits are loaded now. A block
                    // in which no row of the warp has a masked key is skipped (padding and block-structured masks).
                    const uint4 nb = (j + 1 < nt) ? __ldg(bits_row + j + 1) : make_uint4(0u, 0u, 0u, 0u);
                    if (__any_sync(0xffffffffu, (bits.x | bits.y | bits.z | bits.w) != 0u)) {
                        const uint32_t w[4] = {bits.x, bits.y, bits.z, bits.w};
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                x[4 * e + c] = ((w[c] >> e) & 1u) ? -INFINITY : x[4 * e + c];
                        }
                    }
                    bits = nb;
                }
                // keys past the end of the sequence, and (causal) keys after the query
                const int kbase = j * kBK128;
                const bool ragged = kbase + kBK128 > n;
                const bool diag = CAUSAL && (kbase + kBK128 - 1 > tile_row0);
                if (ragged || diag) {
                    int lim = n - 1 - kbase;
                    if (CAUSAL) lim = min(lim, row - kbase);
#pragma unroll
                    for (int c = 0; c < 128; ++c) x[c] = (c > lim) ? -INFINITY : x[c];
                }
                const float mb = row_max128(x) * sl2;  // sl2 > 0
                const float m_new = fmaxf(m_ref, mb);
                // lazy rescale: move the reference only when the maximum grew by more than TAU
                const bool need = (m_new > m_ref + kTau) || (m_ref == -INFINITY && m_new != -INFINITY);
                const float alpha = need ? ex2_approx(m_ref - m_new) : 1.0f;  // 2^-inf = 0
                const bool rescale = __any_sync(0xffffffffu, need) && j > 0;
                if (need) {
                    l *= alpha;
                    m_ref = m_new;
                }
                const float neg = (m_ref == -INFINITY) ? 0.0f : -m_ref;
                const float2 sl2v = make_float2(sl2, sl2), negv = make_float2(neg, neg);
                float2 ls[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                                make_float2(0.0f, 0.0f)};
                // P in chunks of 2 PC keys (PC packed columns), each stored as soon as it is ready: halves, or
                // quarters in the masked variants, whose mask registers would not fit beside a half
                constexpr int PC = MASK ? 16 : 32;
#pragma unroll
                for (int qq = 0; qq < 64 / PC; ++qq) {
                    uint32_t pv[PC];
                    if constexpr (DROP) {
#pragma unroll
                        for (int gq = 0; gq < PC / 16; ++gq) {  // 32-key groups: one Philox block each
                            uint32_t kw[8];
                            philox4x64_10((uint64_t)row, (uint64_t)(4 * j + (PC / 16) * qq + gq), (uint64_t)bh,
                                          p.drop_offset, p.drop_seed, 0ull, kw);
#pragma unroll
                            for (int c2 = 0; c2 < 16; ++c2) {
                                const int c = 16 * gq + c2;
                                const int i = 2 * PC * qq + 2 * c;
                                const float2 a = ffma2(make_float2(x[i], x[i + 1]), sl2v, negv);
                                const float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
                                ls[c & 3] = fadd2(ls[c & 3], e);  // the row sum is of the undropped scores
                                const uint32_t w = kw[c2 / 2];    // keys 2 c2, 2 c2 + 1 of the group: bytes of w
                                const uint32_t b0 = (w >> (16 * (c2 & 1))) & 0xFFu, b1 = (w >> (16 * (c2 & 1) + 8)) & 0xFFu;
                                pv[c] = pack2<T>(b0 < (uint32_t)p.drop_threshold ? e.x : 0.0f,
                                                 b1 < (uint32_t)p.drop_threshold ? e.y : 0.0f);
                            }
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < PC; ++c) {
                            const int i = 2 * PC * qq + 2 * c;
                            const float2 a = ffma2(make_float2(x[i], x[i + 1]), sl2v, negv);
                            const float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
                            ls[c & 3] = fadd2(ls[c & 3], e);
                            pv[c] = pack2<T>(e.x, e.y);
                        }
                    }
                    // P V(g-1), the tile's previous product, read P_t and accumulated into O_t:
                    // wait for its commit before overwriting P_t (and before rescaling O_t below).
                    if (qq == 0 && g > 0) {
                        ok = wait_warp(sy.pv_done(t, (g - 1) & 1u), ((g - 1) >> 1) & 1u, abort_flag, p);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    if constexpr (PC == 16)
                        tmem_st16(p_addr + 16 * qq, pv);
                    else
                        tmem_st32(p_addr + 32 * qq, pv);
                }
                if (!ok) break;
                l += ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) + ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
                if (rescale) {
                    // O holds P V for blocks < j relative to the old reference: scale its rows
                    // (alpha = 1 for rows whose reference did not move) before P V(j) adds to it
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        uint32_t ov[32];
                        tmem_ld32_wait(o_addr + c0, ov);
#pragma unroll
                        for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
                        tmem_st32(o_addr + c0, ov);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(sy.p_full(t));
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue
            ok = wait_warp(sy.pv_done(t, (g - 1) & 1u), ((g - 1) >> 1) & 1u, abort_flag, p);
            if (!ok) break;
            tc_fence_after();
            float inv = (l > 0.0f) ? 1.0f / l : 0.0f;
            if constexpr (DROP) inv *= p.drop_scale;  // kept probabilities are scaled by 1 / q
            const size_t orow_idx = VARLEN ? ((size_t)(itm.tok0 + row) * p.H + (size_t)(bh % p.H))
                                           : ((size_t)bh * p.N + (size_t)row);
            T *orow = reinterpret_cast<T *>(p.out) + orow_idx * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t ov[32];
                tmem_ld32_wait(o_addr + c0, ov);
                if (row < n) {
#pragma unroll
                    for (int c = 0; c < 32; c += 8)
                        st_global_v4(orow + c0 + c,
                                     pack2<T>(__uint_as_float(ov[c]) * inv, __uint_as_float(ov[c + 1]) * inv),
                                     pack2<T>(__uint_as_float(ov[c + 2]) * inv, __uint_as_float(ov[c + 3]) * inv),
                                     pack2<T>(__uint_as_float(ov[c + 4]) * inv, __uint_as_float(ov[c + 5]) * inv),
                                     pack2<T>(__uint_as_float(ov[c + 6]) * inv, __uint_as_float(ov[c + 7]) * inv));
                }
            }
            tc_fence_before();  // the O reads above come before the next item's first P V (after p_full)
            if (row < n)  // lse: [B][H][N], or [H][total] for a packed batch
                p.lse[VARLEN ? (size_t)(bh % p.H) * p.total + itm.tok0 + row : (size_t)bh * p.N + row] =
                    (l > 0.0f) ? (m_ref + lg2_approx(l)) * 0.6931471805599453f : -INFINITY;
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        // every MMA of both issuing warps must be complete before TMEM is released
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(sy.drain(), 0) && global_timer_ns() - t0 < p.timeout_ns) {
        }
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace fa
