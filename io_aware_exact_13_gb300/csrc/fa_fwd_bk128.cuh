// fa_fwd_bk128.cuh -- the exact tiled attention forward with 128-key K/V blocks
// (no additive mask), for sm_103a.
//
// Same computation as fa_fwd_kernel.cuh ("FlashAttention: Exact Attention as an
// IO-Aware Streaming Computation", sections "Core idea" and "Mathematical
// structure"; "IO-aware exact attention", section "One tiled forward-pass
// iteration"): a 256-row work item keeps two 128-row query tiles on chip with
// their running (m, l, a); K/V blocks stream past them; S, P and O live in
// tensor memory; only O and lse are written.
//
// What changes against the 64-key kernel is the shape of the products. An
// S = Q K^T product with N = 64 keys reads its Q operand from shared memory as
// often as one with N = 128 but does half the work, and the tensor core issues
// both at about the same rate, so 128-key blocks halve the tensor time of the
// S products. Tensor memory (512 columns) then holds S_0, S_1 (128 columns
// each) and O_0, O_1 (D columns each):
//   D = 128: P_t (16-bit, 64 columns) is written over S_t's columns. The
//            issuing warp of tile t issues O_t += P_t V_j and then
//            S_t = Q_t K_{j+1}^T; the tensor core runs the products of one
//            issuing thread in issue order, so the next S never overwrites a
//            P that the product before it still reads. The softmax of tile t
//            for block j+1 therefore starts after O_t += P_t V_j: the two
//            tiles take turns (while one tile's softmax runs, the tensor core
//            runs the other tile's P V and next S).
//   D = 64:  P_t has its own 64 columns [384 + 64 t, ...); S_t(j+1) is issued
//            as soon as the softmax has copied S_t(j) to registers, so the
//            softmax of block j+1 can start while P_t V_j runs.
//
// Softmax: four warpgroups work on one tile at a time. Warpgroup h takes keys
// [32 h, 32 h + 32) of each 128-key block; thread r of each owns query row r
// (TMEM lane r). The four parts of a row agree on the row maximum through
// shared memory (warps q, q + 4, q + 8, q + 12 own the same 32 lanes and meet at
// an mbarrier), so all keep the same reference maximum; each keeps its own
// partial denominator, and the four are added at the epilogue. The warpgroups
// take the two tiles in turn: while they compute one tile's P, the tensor core
// runs the other tile's P V and next S. Measured on the way here: one warpgroup
// per tile doing all 128 keys of a row ran the two tiles' softmax side by side
// (about 2200 cycles per block); two warpgroups per tile (64 keys each) spent
// about 800 cycles in the exponent loop, which runs at 6.1 cycles per ex2
// instruction with two warps per scheduler and 4.9 with four (the pipe's limit
// is 4).
//
// Roles (20 warps, 640 threads, 96 registers each, one persistent CTA per SM):
//   warps 0-15  softmax + epilogue: warpgroup h = warp / 4 takes key quarter h
//   warp  16    TMA producer: Q tiles per item, then K and V rings
//   warps 17-18 issuer of tile t = warp - 17: S_t products and P_t V products
//   warp  19    packed batch only: publishes the CTA's work items (ItemRing)
// Shared memory holds no static variables: the abort word, the item ring and
// the row-maximum exchange live after the barriers in the dynamic region.
#pragma once
#include "fa_fwd_kernel.cuh"

namespace fa {

constexpr int kBK128 = 128;           // keys per K/V block
constexpr int kThreads128 = 640;       // 20 warps
constexpr int kSoftmaxWarps = 16;
constexpr int kProducerWarp = 16;
constexpr int kItemConsumers128 = 19;  // producer, two issuers, sixteen softmax warps
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
    // tensor memory columns
    static constexpr bool ALIAS = D > 64;              // P_t over S_t (no free columns at D = 128)
    static constexpr int TM_O = 256;                   // O_t at TM_O + D t
    static constexpr int TM_P = ALIAS ? 0 : 256 + 2 * D;
    static constexpr int TM_P_STRIDE = ALIAS ? 128 : 64;
    // shared memory: Q0 Q1 | K ring | V ring | barriers
    static constexpr int SMEM_Q = 0;
    static constexpr int SMEM_K = 2 * Q_TILE;
    static constexpr int FREE = 232448 - 1024 - 512 - SMEM_K;
    static constexpr int SLOTS = FREE / KV_TILE > 12 ? 12 : FREE / KV_TILE;
    static constexpr int RK = (SLOTS + 1) / 2;         // K slots (K_{j+1} is loaded before V_j)
    static constexpr int RV = SLOTS - RK;              // V slots
    static constexpr int SMEM_V = SMEM_K + RK * KV_TILE;
    static constexpr int SMEM_BAR = SMEM_V + RV * KV_TILE;
    // q_full[2] q_empty[2] k_full[RK] k_empty[RK] v_full[RV] v_empty[RV] s_full[2] s_free[2] p_full[2]
    // pv_done[2][2] drain
    static constexpr int NUM_BARS = 4 + 2 * RK + 2 * RV + 10 + 1;
    static constexpr int SMEM_TMEM_SLOT = SMEM_BAR + ((NUM_BARS * 8 + 15) / 16) * 16;
    static constexpr int SMEM_XBAR = SMEM_TMEM_SLOT + 16;         // 4 exchange barriers (one per lane quadrant)
    static constexpr int SMEM_XCH = SMEM_XBAR + 32;               // float [4 quarters][128 rows]
    static constexpr int SMEM_RING = SMEM_XCH + 4 * 128 * 4;      // ItemRing (packed batches)
    static constexpr int SMEM_ABORT = SMEM_RING + 128;
    static constexpr int SMEM_USED = SMEM_ABORT + 16;
    // up to 1024 bytes to align the base (SW128 tiles need 1024-byte alignment), within the 227 KB limit
    static constexpr int SMEM_BYTES = SMEM_USED + 1024 <= 232448 ? SMEM_USED + 1024 : 232448;
    static constexpr int SLACK = SMEM_BYTES - SMEM_USED;
    static_assert(NCH >= 1 && ROW_BYTES % 128 == 0, "row must be a whole number of 128-byte swizzle rows");
    static_assert(RK >= 2 && RV >= 2, "K/V rings too small");
    static_assert(SLACK >= 256, "shared memory budget");
    static_assert(TM_O + 2 * D <= 512 && TM_P + 2 * TM_P_STRIDE <= (ALIAS ? 256 : 512), "tensor memory budget");
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
    // Per tile: S ready (MMA commit), S copied out (D = 64 only), P ready (256 softmax
    // threads), P V(g) done (MMA commit to pv_done(t, g & 1)). No barrier can get two
    // phases ahead of a waiter (see the roles below), so parity waits are exact.
    __device__ __forceinline__ uint32_t s_full(int t) const { return at(B0 + t); }
    __device__ __forceinline__ uint32_t s_free(int t) const { return at(B0 + 2 + t); }
    __device__ __forceinline__ uint32_t p_full(int t) const { return at(B0 + 4 + t); }
    __device__ __forceinline__ uint32_t pv_done(int t, int b) const { return at(B0 + 6 + 2 * t + b); }
    __device__ __forceinline__ uint32_t drain() const { return at(B0 + 10); }
};

template <typename T, int D, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kThreads128, 1)
    fa_fwd_bk128_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
    using C = Cfg128<T, D>;
    constexpr int RK = C::RK, RV = C::RV;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (uint32_t)((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    if (pad > (uint32_t)C::SLACK) {  // cannot happen with no static shared memory; never overflow
        if (threadIdx.x == 0) atomicExch(p.status, kStatusSmemAlign);
        return;
    }
    uint8_t *smem = smem_raw + pad;
    Sync128<RK, RV> sy{reinterpret_cast<uint64_t *>(smem + C::SMEM_BAR)};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::SMEM_TMEM_SLOT);
    float *xch = reinterpret_cast<float *>(smem + C::SMEM_XCH);
    uint64_t *xbar = reinterpret_cast<uint64_t *>(smem + C::SMEM_XBAR);
    ItemRing *ring = reinterpret_cast<ItemRing *>(smem + C::SMEM_RING);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::SMEM_ABORT);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(sy.q_full(t), 1);
            mbar_init(sy.q_empty(t), 1);
            mbar_init(sy.s_full(t), 1);
            mbar_init(sy.s_free(t), 4 * kBQ);  // all four softmax warpgroups
            mbar_init(sy.p_full(t), 4 * kBQ);
            mbar_init(sy.pv_done(t, 0), 1);
            mbar_init(sy.pv_done(t, 1), 1);
        }
        for (int s = 0; s < RK; ++s) {  // a slot is released by both tiles' issuers
            mbar_init(sy.k_full(s), 1);
            mbar_init(sy.k_empty(s), 2);
        }
        for (int s = 0; s < RV; ++s) {
            mbar_init(sy.v_full(s), 1);
            mbar_init(sy.v_empty(s), 2);
        }
        mbar_init(sy.drain(), 2);  // one commit per issuing warp
        for (int q = 0; q < 4; ++q) mbar_init(smem_u32(xbar + q), 128);  // warps q, q + 4, q + 8, q + 12
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
    if (warp == kProducerWarp + 1) {  // TMEM: all 512 columns (one CTA per SM)
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tensormap(&tm_q);
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = __shfl_sync(0xffffffffu, *tmem_slot, 0);

    if (warp >= kSoftmaxWarps) {
        if (warp == kProducerWarp) {
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
        } else if (warp == kProducerWarp + 1 || warp == kProducerWarp + 2) {
            // ---------------------------------------------------------- issuer of tile t
            // The whole warp runs the loop (warp-uniform), lane 0 issues.
            //   S_t(j)  = Q_t K_j^T     into S_t's columns, committed to s_full(t)
            //   O_t    (+)= P_t(j) V_j  once the softmax has written P_t(j); the g-th product of the
            //                            tile is committed to pv_done(t, g & 1)
            // D = 128: P V(j) then S(j+1) (P_t lives in S_t's columns, in-order products).
            // D = 64:  S(j+1) as soon as the softmax has copied S(j) out, then P V(j).
            // K and V slots of blocks this tile does not need are released at once.
            const int t = warp - (kProducerWarp + 1);
            const uint32_t issue = lane == 0 ? 1u : 0u;
            const uint64_t a0 = smem_desc_sw128(smem_u32(smem + C::SMEM_Q + t * C::Q_TILE), 16, 1024);
            const uint64_t kd0 = smem_desc_sw128(smem_u32(smem + C::SMEM_K), 16, 1024);
            const uint64_t vd0 = smem_desc_sw128(smem_u32(smem + C::SMEM_V), C::KV_CHUNK, 1024);
            const uint32_t d_s = tmem + 128 * t;
            const uint32_t d_o = tmem + C::TM_O + D * t;
            const uint32_t a_p = tmem + C::TM_P + C::TM_P_STRIDE * t;
            constexpr uint64_t KVT16 = C::KV_TILE >> 4;
            uint32_t qcount = 0, kpos = 0, vpos = 0, pcount = 0, s_issued = 0;
            bool ok = true;
            auto issue_s = [&](int j, int nt) -> bool {
                const int slot = kpos % RK;
                if (!wait_warp(sy.k_full(slot), (kpos / RK) & 1u, abort_flag, p)) return false;
                ++kpos;
                if (j >= nt) {
                    if (lane == 0) mbar_arrive(sy.k_empty(slot));
                    return true;
                }
                if (!C::ALIAS && s_issued > 0 && !wait_warp(sy.s_free(t), (s_issued - 1) & 1u, abort_flag, p))
                    return false;
                ++s_issued;
                tc_fence_after();
                const uint64_t b0 = kd0 + slot * KVT16;
#pragma unroll
                for (int k = 0; k < C::KSTEPS_S; ++k) {
                    const uint64_t aoff = (uint64_t)(((k / 4) * C::Q_CHUNK + (k % 4) * 32) >> 4);
                    const uint64_t boff = (uint64_t)(((k / 4) * C::KV_CHUNK + (k % 4) * 32) >> 4);
                    mma_ss(d_s, a0 + aoff, b0 + boff, C::IDESC_S, k > 0 ? 1u : 0u, issue);
                }
                tc_commit(sy.s_full(t), issue);
                if (j == nt - 1) tc_commit(sy.q_empty(t), issue);
                tc_commit(sy.k_empty(slot), issue);
                return true;
            };
            auto issue_pv = [&](int j, int nt) -> bool {
                const int slot = vpos % RV;
                if (!wait_warp(sy.v_full(slot), (vpos / RV) & 1u, abort_flag, p)) return false;
                ++vpos;
                if (j >= nt) {
                    if (lane == 0) mbar_arrive(sy.v_empty(slot));
                    return true;
                }
                if (!wait_warp(sy.p_full(t), pcount & 1u, abort_flag, p)) return false;
                ++pcount;
                tc_fence_after();
                const uint64_t b0 = vd0 + slot * KVT16;
#pragma unroll
                for (int k = 0; k < C::KSTEPS_PV; ++k)
                    mma_ts(d_o, a_p + k * 8, b0 + (uint64_t)((k * C::V_KSTEP_BYTES) >> 4), C::IDESC_PV,
                           (k > 0 || j > 0) ? 1u : 0u, issue);
                tc_commit(sy.pv_done(t, (pcount - 1) & 1u), issue);
                tc_commit(sy.v_empty(slot), issue);
                return true;
            };
            ItemIter<VARLEN> iter(p, abort_flag, ring);
            for (Item itm; ok && iter.next(p, itm, ok);) {
                const int nt = tile_nkv<CAUSAL, kBK128>(itm, t);
                const int nmax = max(tile_nkv<CAUSAL, kBK128>(itm, 0), tile_nkv<CAUSAL, kBK128>(itm, 1));
                if (nmax == 0) continue;
                if (nt > 0) {
                    ok = wait_warp(sy.q_full(t), qcount & 1u, abort_flag, p);
                    ++qcount;
                }
                if (ok) ok = issue_s(0, nt);
                for (int j = 0; ok && j < nmax; ++j) {
                    if constexpr (C::ALIAS) {
                        ok = issue_pv(j, nt);
                        if (ok && j + 1 < nmax) ok = issue_s(j + 1, nt);
                    } else {
                        if (j + 1 < nmax) ok = issue_s(j + 1, nt);
                        if (ok) ok = issue_pv(j, nt);
                    }
                }
            }
            __syncwarp();
            tc_commit(sy.drain(), issue);
        } else if (VARLEN && warp == kProducerWarp + 3) {
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
        // -------------------------------------------------------------- softmax + epilogue
        constexpr int HK = kBK128 / 4;  // keys per quarter
        constexpr int HD = D / 4;       // O columns per quarter
        const int h = warp >> 2;        // key quarter of this warpgroup
        const int qd = warp & 3;        // TMEM lane quadrant (warps qd, qd + 4, qd + 8, qd + 12 share it)
        const int r = threadIdx.x & 127;
        const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
        const float scale_log2 = p.scale_log2;
        // raw scores scaled inside the exponent when the scale is positive (the maximum
        // commutes with it); otherwise pre-scaled scores (a -inf raw score times a
        // non-positive scale is not -inf)
        const bool fast = scale_log2 > 0.0f;
        const float sl2 = fast ? scale_log2 : 1.0f;
        // The four parts of a row (same row, other key quarters) exchange one value each at the
        // quadrant's mbarrier, with the same bounded wait as every pipeline wait (a warp that gives
        // up does not leave the others waiting forever). Each exchange takes two phases: all four
        // write and arrive (even phase), read the other three, and arrive again (odd phase); the
        // next exchange writes only after the odd phase, so one buffer suffices.
        uint32_t xk = 0;
        const uint32_t quad_bar = smem_u32(xbar + qd);
        auto exchange = [&](float v, bool &okx, float &o1, float &o2, float &o3) {
            if (xk > 0) {
                okx = wait_warp(quad_bar, 1u, abort_flag, p);  // the previous values have been read
                if (!okx) return;
            }
            xch[h * 128 + r] = v;
            tc_fence_before();  // this thread's tensor-memory reads come before the others' writes
            mbar_arrive(quad_bar);
            okx = wait_warp(quad_bar, 0u, abort_flag, p);
            if (!okx) return;
            tc_fence_after();
            o1 = xch[((h + 1) & 3) * 128 + r];
            o2 = xch[((h + 2) & 3) * 128 + r];
            o3 = xch[((h + 3) & 3) * 128 + r];
            mbar_arrive(quad_bar);
            ++xk;
        };
        uint32_t scount[2] = {0, 0};  // S blocks consumed per tile (all items)
        uint32_t g[2] = {0, 0};       // P blocks produced per tile = its P V products
        bool ok = true;
        ItemIter<VARLEN> iter(p, abort_flag, ring);
        for (Item itm; ok && iter.next(p, itm, ok);) {
            const int bh = itm.bh, q0 = itm.q0, n = itm.n;
            const int nt[2] = {tile_nkv<CAUSAL, kBK128>(itm, 0), tile_nkv<CAUSAL, kBK128>(itm, 1)};
            const int nmax = max(nt[0], nt[1]);
            float m_ref[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};
            for (int j = 0; ok && j < nmax; ++j) {
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (!ok || j >= nt[t]) continue;
                    const uint32_t s_addr = tmem + lane_base + 128 * t + HK * h;  // fp32 S columns of this quarter
                    const uint32_t p_addr = tmem + lane_base + C::TM_P + C::TM_P_STRIDE * t + HK / 2 * h;
                    const uint32_t o_addr = tmem + lane_base + C::TM_O + D * t + HD * h;
                    ok = wait_warp(sy.s_full(t), scount[t] & 1u, abort_flag, p);
                    ++scount[t];
                    if (!ok) break;
                    tc_fence_after();
                    float x[HK];
                    {
                        uint32_t sr[HK];
                        tmem_ld32_wait(s_addr, sr);
#pragma unroll
                        for (int c = 0; c < HK; ++c)
                            x[c] = fast ? __uint_as_float(sr[c]) : __uint_as_float(sr[c]) * scale_log2;
                    }
                    if constexpr (!C::ALIAS) {
                        tc_fence_before();
                        mbar_arrive(sy.s_free(t));  // S_t may now be overwritten by the next block
                    }
                    // keys past the end of the sequence, and (causal) keys after the query
                    const int row = q0 + t * kBQ + r;  // query row within the sequence (may be >= n)
                    const int kbase = j * kBK128 + HK * h;
                    const bool ragged = kbase + HK > n;
                    const bool diag = CAUSAL && (kbase + HK - 1 > q0 + t * kBQ);
                    if (ragged || diag) {
                        int lim = n - 1 - kbase;
                        if (CAUSAL) lim = min(lim, row - kbase);
#pragma unroll
                        for (int c = 0; c < HK; ++c) x[c] = (c > lim) ? -INFINITY : x[c];
                    }
                    float m8[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) m8[i] = fmax3(x[i], x[8 + i], x[16 + i]);
#pragma unroll
                    for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], x[24 + i]);
                    const float mq =
                        fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                    float mo1, mo2, mo3;
                    exchange(mq, ok, mo1, mo2, mo3);
                    if (!ok) break;
                    const float mb = fmaxf(mq, fmax3(mo1, mo2, mo3)) * sl2;  // sl2 > 0
                    const float m_new = fmaxf(m_ref[t], mb);
                    // lazy rescale: move the reference only when the maximum grew by more than TAU
                    const bool need = (m_new > m_ref[t] + kTau) || (m_ref[t] == -INFINITY && m_new != -INFINITY);
                    const float alpha = need ? ex2_approx(m_ref[t] - m_new) : 1.0f;  // 2^-inf = 0
                    const bool rescale = __any_sync(0xffffffffu, need) && j > 0;
                    if (need) {
                        l[t] *= alpha;
                        m_ref[t] = m_new;
                    }
                    const float neg = (m_ref[t] == -INFINITY) ? 0.0f : -m_ref[t];
                    const float2 sl2v = make_float2(sl2, sl2), negv = make_float2(neg, neg);
                    float2 ls[4] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f),
                                    make_float2(0.0f, 0.0f)};
                    uint32_t pv[HK / 2];
#pragma unroll
                    for (int c = 0; c < HK / 2; ++c) {
                        const float2 a = ffma2(make_float2(x[2 * c], x[2 * c + 1]), sl2v, negv);
                        const float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
                        ls[c & 3] = fadd2(ls[c & 3], e);
                        pv[c] = pack2<T>(e.x, e.y);
                    }
                    l[t] += ((ls[0].x + ls[0].y) + (ls[1].x + ls[1].y)) + ((ls[2].x + ls[2].y) + (ls[3].x + ls[3].y));
                    // P V(g-1), the tile's previous product, read P_t and accumulated into O_t. Its
                    // commit can reach pv_done several hundred cycles after the commit of S(g), which
                    // was issued after it, so the softmax waits for it only where it must:
                    //  D = 64:  before storing P, which reuses P_t's buffer;
                    //  D = 128: before rescaling O. P(g) goes over S(g)'s columns, which the tensor
                    //           core wrote after P V(g-1) had read P(g-1) there (it runs one issuing
                    //           thread's products in order), and the softmax stores only after it
                    //           has seen S(g) complete. (The P of key quarter h lands on S columns
                    //           [16 h, 16 h + 16), which quarters 0 and 1 copied out before the
                    //           exchange.)
                    // Besides, P V(g-2) (long complete) is waited for before P(g) is released, so
                    // that neither pv_done barrier can get two phases ahead of these waits.
                    auto wait_pv = [&](uint32_t gg) -> bool {
                        return wait_warp(sy.pv_done(t, gg & 1u), (gg >> 1) & 1u, abort_flag, p);
                    };
                    if (!C::ALIAS && g[t] > 0) {
                        ok = wait_pv(g[t] - 1);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    tmem_st16(p_addr, pv);
                    if (rescale) {
                        if (C::ALIAS) {
                            ok = wait_pv(g[t] - 1);
                            if (!ok) break;
                            tc_fence_after();
                        }
                        // O holds P V for blocks < j relative to the old reference: scale this half's
                        // columns of the row (alpha = 1 where the reference did not move)
#pragma unroll
                        for (int c0 = 0; c0 < HD; c0 += 16) {
                            uint32_t ov[16];
                            tmem_ld16_wait(o_addr + c0, ov);
#pragma unroll
                            for (int c = 0; c < 16; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
                            tmem_st16(o_addr + c0, ov);
                        }
                    }
                    if (C::ALIAS && g[t] >= 2) {
                        ok = wait_pv(g[t] - 2);
                        if (!ok) break;
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(sy.p_full(t));
                    ++g[t];
                }
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue, tile by tile
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (!ok || nt[t] == 0) continue;
                float lo1, lo2, lo3;
                exchange(l[t], ok, lo1, lo2, lo3);  // the other quarters' partial denominators
                if (!ok) break;
                const float l_row = (l[t] + lo1) + (lo2 + lo3);
                ok = wait_warp(sy.pv_done(t, (g[t] - 1) & 1u), ((g[t] - 1) >> 1) & 1u, abort_flag, p);
                if (!ok) break;
                tc_fence_after();
                const int row = q0 + t * kBQ + r;
                const uint32_t o_addr = tmem + lane_base + C::TM_O + D * t + HD * h;
                const float inv = (l_row > 0.0f) ? 1.0f / l_row : 0.0f;
                const size_t orow_idx = VARLEN ? ((size_t)(itm.tok0 + row) * p.H + (size_t)(bh % p.H))
                                               : ((size_t)bh * p.N + (size_t)row);
                T *orow = reinterpret_cast<T *>(p.out) + orow_idx * D + HD * h;
#pragma unroll
                for (int c0 = 0; c0 < HD; c0 += 16) {
                    uint32_t ov[16];
                    tmem_ld16_wait(o_addr + c0, ov);
                    if (row < n) {
#pragma unroll
                        for (int c = 0; c < 16; c += 8)
                            st_global_v4(orow + c0 + c,
                                         pack2<T>(__uint_as_float(ov[c]) * inv, __uint_as_float(ov[c + 1]) * inv),
                                         pack2<T>(__uint_as_float(ov[c + 2]) * inv, __uint_as_float(ov[c + 3]) * inv),
                                         pack2<T>(__uint_as_float(ov[c + 4]) * inv, __uint_as_float(ov[c + 5]) * inv),
                                         pack2<T>(__uint_as_float(ov[c + 6]) * inv, __uint_as_float(ov[c + 7]) * inv));
                    }
                }
                tc_fence_before();  // the O reads come before the next item's first P V (after p_full)
                if (h == 0 && row < n)
                    p.lse[VARLEN ? (size_t)(bh % p.H) * p.total + itm.tok0 + row : (size_t)bh * p.N + row] =
                        (l_row > 0.0f) ? (m_ref[t] + lg2_approx(l_row)) * 0.6931471805599453f : -INFINITY;
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kProducerWarp + 1) {
        // every MMA of both issuing warps must be complete before TMEM is released
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(sy.drain(), 0) && global_timer_ns() - t0 < p.timeout_ns) {
        }
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace fa
