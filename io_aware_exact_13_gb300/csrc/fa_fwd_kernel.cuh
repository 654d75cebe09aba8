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
// GB300 mapping (one persistent CTA per SM, 16 warps):
//   warps 0-3   softmax + epilogue for query tile 0 (thread r owns row r = TMEM lane r)
//   warps 4-7   softmax + epilogue for query tile 1
//   warp  8     TMA producer: Q tiles once per work item, then K and V rings
//   warps 9-10  S issuers: S_t = Q_t K^T on tcgen05 for tile t = 0, 1
//   warps 11-12 PV issuers: O_t += P_t V for tile t = 0, 1
//   warp  13    packed batch only: publishes the CTA's work items (see ItemRing)
//   warps 14-15 idle (they complete the last warpgroup)
// Each issuing warp runs its loop warp-uniformly and lane 0 issues. Four
// independent issue streams keep the per-wait and per-instruction issue cost
// (barrier operations compete with MMA operand reads for shared memory) off
// the tensor core's critical path; accumulators are fp32 in tensor memory.
// A work item is (batch*head, 256 query rows) = two 128-row query tiles that
// share every K/V tile; items are visited longest-first (causal rows near the
// end of the sequence see the most keys).
//
// K/V blocks are 64 keys, so that tensor memory (512 columns x 128 lanes x 32
// bit) holds, without aliasing,
//   S_t      columns [64 t, 64 t + 64)                 (fp32 scores, one block)
//   P_t,b    columns [128 + 64 t + 32 b, ... + 32)     (16-bit P, two buffers)
//   O_t      columns [256 + 128 t, 256 + 128 t + D)    (fp32 accumulator)
// The softmax warps copy S_t(j) to registers and release it at once, so the MMA
// for S_t(j+1) runs while they compute P_t(j); with P double-buffered the only
// ordering left between the softmax and the tensor core is the data itself.
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

#include "pdl.cuh"
#include "ptx.cuh"

namespace fa {

constexpr int kBQ = 128;           // rows per query tile (= TMEM lanes)
constexpr int kBK = 64;            // keys per K/V block
constexpr int kRowsPerItem = 256;  // two query tiles per work item
constexpr int kThreads = 512;
constexpr float kTau = 8.0f;       // lazy-rescale threshold, log2 units
constexpr int kStatusTimeout = -6; // value written to the device status word
constexpr int kStatusSeqlens = -8; // packed batch: cu_seqlens inconsistent with total / max_seqlen

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

// MASK: each softmax warp stages the next key block's mask values for its 32
// rows in shared memory (8 KB per warp, 32 KB per query tile), taken from the
// K/V rings' share.
template <typename T, int D, bool MASK = false>
struct Cfg {
    static constexpr int EB = sizeof(T);
    static constexpr int ROW_BYTES = D * EB;                // one row of Q/K/V
    static constexpr int CHUNK_ELEMS = 128 / EB;            // elements per 128-byte swizzle row
    static constexpr int NCH = ROW_BYTES / 128;             // swizzle chunks per row
    static constexpr int Q_CHUNK = kBQ * 128;               // 128 rows x 128 bytes
    static constexpr int KV_CHUNK = kBK * 128;              // 64 rows x 128 bytes
    static constexpr int Q_TILE = NCH * Q_CHUNK;            // one 128-row query tile
    static constexpr int KV_TILE = NCH * KV_CHUNK;          // one 64-key K or V block
    static constexpr int KSTEPS_S = ROW_BYTES / 32;         // 32 bytes of the head dim per MMA
    static constexpr int KSTEPS_PV = kBK / 16;              // 16 keys per MMA
    static constexpr int V_KSTEP_BYTES = 16 * 128;          // 16 key rows x 128 bytes
    static constexpr uint32_t IDESC_S = make_idesc(Elem<T>::fmt, 128, kBK, 0);
    static constexpr uint32_t IDESC_PV = make_idesc(Elem<T>::fmt, 128, D, 1);
    // shared memory: Q0 Q1 | K ring | V ring | barriers
    static constexpr int SMEM_Q = 0;
    static constexpr int SMEM_KV = 2 * Q_TILE;
    static constexpr int MASK_TILE = kBQ * kBK * 4;           // 128 rows x 64 fp32 mask values
    static constexpr int MASK_BYTES = MASK ? 2 * MASK_TILE : 0;
    static constexpr int RING_FREE = 232448 - 1024 - 512 - SMEM_KV - MASK_BYTES;
    static constexpr int RING = (RING_FREE / KV_TILE / 2) > 6 ? 6 : (RING_FREE / KV_TILE / 2);  // slots per ring
    static constexpr int STAGES = 2 * RING;
    static constexpr int SMEM_V = SMEM_KV + RING * KV_TILE;
    static constexpr int SMEM_MASK = SMEM_KV + STAGES * KV_TILE;
    static constexpr int SMEM_BAR = SMEM_MASK + MASK_BYTES;
    // q_full[2] q_empty[2] k_full[R] k_empty[R] v_full[R] v_empty[R] s_full[2] s_free[2] p_full[2][2]
    // pv_done[2][2] drain
    static constexpr int NUM_BARS = 2 + 2 + 4 * RING + 2 + 2 + 4 + 4 + 1;
    static constexpr int SMEM_BYTES = SMEM_BAR + NUM_BARS * 8 + 16 + 1024;  // + alignment slack
    static_assert(NCH >= 1 && ROW_BYTES % 128 == 0, "row must be a whole number of 128-byte swizzle rows");
    static_assert(RING >= 2, "K/V rings too small");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct FwdParams {
    void *out;
    float *lse;
    const float *mask;  // [B][N][N] or nullptr
    int *status;        // device status word
    int B, H, N;
    int kv_group;       // query heads per key/value head (1 unless grouped-query attention)
    int n_items;        // work units: n_pair two-tile items, then single query tiles
    int n_pair;         // two-tile items (B * H * ceil(N / 256) unless the tail is split, see split_tail)
    int n_qblk;         // ceil(N / 256)
    int n_kv;           // ceil(N / 64)
    float scale_log2;   // scale * log2(e)
    uint64_t timeout_ns;
    // packed variable-length batch (B = number of sequences, N = max_seqlen):
    const int *cu_seqlens;  // [B + 1] token offsets of the sequences
    int total;              // tokens in the batch
    int Hkv;                // key/value heads
    int rows_per_item;      // query rows per work item: 256 (two 128-row tiles) or 128 (one tile)
    int mask_tma;           // 1: the mask tensor map is valid (N % 4 == 0) and mask blocks arrive by TMA
    int mask_per_head;      // 1: the mask is a per-head bias [B][H][N][N]; 0: [B][N][N] shared by the heads
    // A [B][N][N] mask packed to one bit per entry (fa_mask_pack.cu): [B][N][mask_bits_blk] 16-byte units,
    // or nullptr. mask_kind is the packing pass's verdict, read at kernel start: 0 = every entry was 0 or
    // -inf (the 128-key kernel applies the bits), 1 = some other value (the 64-key kernel applies the fp32
    // mask). Each of the two kernels returns at once when the verdict is the other one's.
    const uint4 *mask_bits;
    int mask_bits_blk;
    const int *mask_kind;
    // Dropout (128-key kernel): key j of query row i of head bh is kept when byte j mod 32 of
    // Philox4x64-10(counter {i, j / 32, bh, drop_offset}, key {drop_seed, 0}) is below drop_threshold
    // (1..256); kept probabilities are scaled by drop_scale = 256 / drop_threshold.
    uint64_t drop_seed, drop_offset;
    int drop_threshold;
    float drop_scale;
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
    q0 = qb * p.rows_per_item;
}

// One work item as every role sees it: head row bh (= b*H + h), first query row
// q0 within its sequence, the sequence length n and, in a packed batch, the
// token index of the sequence's first row.
struct Item {
    int bh, q0, n, tok0;
    int nrow;  // rows of the sequence this unit covers end before nrow (q0 + 128 for a single-tile unit)
};

__device__ __forceinline__ Item get_item(const FwdParams &p, int item) {
    Item it;
    // units past n_pair are the two query tiles of the remaining items, one at a time
    const int split = item - p.n_pair;
    if (split >= 0) item = p.n_pair + (split >> 1);
    item_coords(p, item, it.bh, it.q0);
    it.n = p.N;
    it.tok0 = 0;
    it.nrow = p.N;
    if (split >= 0) {
        it.q0 += (split & 1) * kBQ;
        it.nrow = min(p.N, it.q0 + kBQ);
    }
    return it;
}

// Length of packed sequence s, or 0 when its bounds do not fit the batch
// (such a sequence is skipped and reported once).
__device__ __forceinline__ int seq_len(const FwdParams &p, int s, int &a, bool &bad) {
    a = __ldg(p.cu_seqlens + s);
    const int b = __ldg(p.cu_seqlens + s + 1);
    bad = a < 0 || b < a || b > p.total || b - a > p.N;
    return bad ? 0 : b - a;
}

// Packed batch work list. A grid over nseq x H x ceil(max_seqlen / R) slots (R =
// rows per item) is mostly empty for short sequences, and empty slots unbalance
// the static schedule. Instead the non-empty items form one compact list, longest
// first: level l (query rows [R l, R l + R)) from the top level down, and within
// a level every sequence longer than R l in index order, each with its H
// heads. A CTA takes list positions in the snake order of item_at. Positions
// grow monotonically, so a cursor suffices: the current level, its first
// position and sequence count, and a scan point (rank sequences of the level
// lie below sequence pos). Counting a level and finding the j-th sequence of a
// level are warp ballots over 32 sequences at a time; all 32 lanes call.
struct VarlenCursor {
    int w = 0, lvl, cnt, start = 0, pos = 0, rank = 0;

    __device__ __forceinline__ static int count_level(const FwdParams &p, int l) {
        const int thr = l * p.rows_per_item;
        int c = 0;
        for (int s0 = 0; s0 < p.B; s0 += 32) {
            const int s = s0 + (int)(threadIdx.x & 31);
            int a;
            bool bad;
            const bool q = s < p.B && seq_len(p, s, a, bad) > thr;
            c += __popc(__ballot_sync(0xffffffffu, q));
        }
        return c;
    }

    __device__ __forceinline__ explicit VarlenCursor(const FwdParams &p) {
        int mx = 0;
        bool any_bad = false;
        for (int s0 = 0; s0 < p.B; s0 += 32) {
            const int s = s0 + (int)(threadIdx.x & 31);
            int a;
            bool bad = false;
            if (s < p.B) mx = max(mx, seq_len(p, s, a, bad));
            any_bad |= bad;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (__any_sync(0xffffffffu, any_bad) && blockIdx.x == 0 && (threadIdx.x & 31) == 0)
            atomicExch(p.status, kStatusSeqlens);
        lvl = mx > 0 ? (mx - 1) / p.rows_per_item : -1;
        cnt = lvl >= 0 ? count_level(p, lvl) : 0;
    }

    __device__ __forceinline__ bool next(const FwdParams &p, Item &it) {
        if (lvl < 0) return false;
        const int G = gridDim.x;
        const int c = (w & 1) ? (G - 1 - (int)blockIdx.x) : (int)blockIdx.x;
        const int k = w * G + c;  // list positions < B*H*levels, an int
        ++w;
        while (k >= start + cnt * p.H) {
            start += cnt * p.H;
            if (--lvl < 0) return false;
            cnt = count_level(p, lvl);
            pos = 0;
            rank = 0;
        }
        const int r = k - start;
        const int j = r / p.H, h = r - j * p.H;
        const int thr = lvl * p.rows_per_item;
        // the j-th sequence (0-based, index order) with rows at this level
        for (; pos < p.B; pos += 32) {
            const int s = pos + (int)(threadIdx.x & 31);
            int a = 0, n = 0;
            bool bad;
            if (s < p.B) n = seq_len(p, s, a, bad);
            uint32_t bal = __ballot_sync(0xffffffffu, n > thr);
            const int nb = __popc(bal);
            if (rank + nb > j) {
                for (int i = rank; i < j; ++i) bal &= bal - 1u;  // drop the lower set bits
                const int src = __ffs(bal) - 1;
                it.bh = (pos + src) * p.H + h;
                it.q0 = thr;
                it.n = __shfl_sync(0xffffffffu, n, src);
                it.tok0 = __shfl_sync(0xffffffffu, a, src);
                it.nrow = it.n;
                return true;
            }
            rank += nb;
        }
        lvl = -1;  // not reached while cu_seqlens is unchanged during the launch
        return false;
    }
};

// Number of BK-key blocks query tile t of an item must visit.
template <bool CAUSAL, int BK = kBK>
__device__ __forceinline__ int tile_nkv(const Item &it, int t) {
    const int r0 = it.q0 + t * kBQ;
    if (r0 >= it.nrow) return 0;
    if (!CAUSAL) return (it.n + BK - 1) / BK;
    const int last_row = min(it.n, r0 + kBQ) - 1;
    return last_row / BK + 1;
}

template <int R>
struct Sync {
    uint64_t *bars;
    __device__ __forceinline__ uint32_t at(int i) const { return smem_u32(bars + i); }
    __device__ __forceinline__ uint32_t q_full(int t) const { return at(t); }
    __device__ __forceinline__ uint32_t q_empty(int t) const { return at(2 + t); }
    __device__ __forceinline__ uint32_t k_full(int s) const { return at(4 + s); }
    __device__ __forceinline__ uint32_t k_empty(int s) const { return at(4 + R + s); }
    __device__ __forceinline__ uint32_t v_full(int s) const { return at(4 + 2 * R + s); }
    __device__ __forceinline__ uint32_t v_empty(int s) const { return at(4 + 3 * R + s); }
    __device__ __forceinline__ uint32_t s_full(int t) const { return at(4 + 4 * R + t); }
    __device__ __forceinline__ uint32_t s_free(int t) const { return at(6 + 4 * R + t); }
    // One P-ready and one P-consumed barrier per (tile, P buffer): each can then
    // run at most one phase ahead of its waiter, which the parity waits need.
    __device__ __forceinline__ uint32_t p_full(int t, int b) const { return at(8 + 4 * R + 2 * t + b); }
    __device__ __forceinline__ uint32_t pv_done(int t, int b) const { return at(12 + 4 * R + 2 * t + b); }
    __device__ __forceinline__ uint32_t drain() const { return at(16 + 4 * R); }
};

// Bounded wait: returns false (after recording a timeout and raising the CTA's
// abort flag) if the phase does not complete within timeout_ns, or returns
// false at once if another role of this CTA has already aborted.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             const FwdParams &p) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        // sleep until the phase completes (or 100 us pass) rather than polling, so that
        // waiting warps leave the issue slots to the warps that are computing
        if (mbar_try_wait_suspend(bar, parity, 100000u)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > p.timeout_ns) {
            *abort_flag = 1;
            atomicExch(p.status, kStatusTimeout);
            return false;
        }
    }
}

// Warp-uniform bounded wait (every lane waits; all lanes agree on the result).
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          const FwdParams &p) {
    return __all_sync(0xffffffffu, wait_bounded(bar, parity, abort_flag, p));
}

// The items of one CTA, in the order every role visits them. All 32 lanes of
// a warp call next() together; every warp of the CTA sees the same sequence.
template <bool VARLEN>
struct ItemIter;

struct ItemRing;

template <>
struct ItemIter<false> {
    int w = 0;
    __device__ __forceinline__ ItemIter(const FwdParams &, volatile int *, ItemRing * = nullptr) {}
    __device__ __forceinline__ bool next(const FwdParams &p, Item &it, bool &) {
        const int item = item_at(p, w++);
        if (item < 0) return false;
        it = get_item(p, item);
        return true;
    }
};

// Packed batch: one otherwise idle warp walks the cursor and publishes each
// item in a 4-slot ring in shared memory (a descriptor plus a full and an
// empty barrier per slot); the other roles read it from there, so the issuing
// warps keep no cursor state and do no scans. A descriptor with bh < 0 ends
// the list. The 13 consumers are the producer, the four issuing warps and the
// eight softmax warps (lane 0 of each arrives on the empty barrier).
constexpr int kItemRing = 4;
constexpr int kItemConsumers = 13;

struct ItemRing {
    uint64_t full[kItemRing];
    uint64_t empty[kItemRing];
    int4 desc[kItemRing];
};

// Masked variant: one mbarrier per softmax warp for its mask copies.
__device__ __forceinline__ uint64_t *mask_bars() {
    __shared__ uint64_t bars[8];
    return bars;
}

__device__ __forceinline__ ItemRing &item_ring() {
    __shared__ __align__(16) ItemRing ring;
    return ring;
}

template <>
struct ItemIter<true> {
    uint32_t i = 0;
    volatile int *abort_flag;
    ItemRing *ring_ptr;  // the CTA's ring (static shared memory, or a slot of the dynamic region)
    __device__ __forceinline__ ItemIter(const FwdParams &, volatile int *abort, ItemRing *ring)
        : abort_flag(abort), ring_ptr(ring) {}
    // false at the end of the list; a wait that gives up also clears ok
    __device__ __forceinline__ bool next(const FwdParams &p, Item &it, bool &ok) {
        ItemRing &ring = *ring_ptr;
        const uint32_t slot = i % kItemRing;
        if (!wait_warp(smem_u32(&ring.full[slot]), (i / kItemRing) & 1u, abort_flag, p)) {
            ok = false;
            return false;
        }
        const int4 d = ring.desc[slot];
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(smem_u32(&ring.empty[slot]));
        ++i;
        if (d.x < 0) return false;
        it.bh = d.x;
        it.q0 = d.y;
        it.n = d.z;
        it.tok0 = d.w;
        it.nrow = d.z;
        return true;
    }
};

// The item ring of the 64-key kernel (static shared memory; packed batches only).
template <bool VARLEN>
__device__ __forceinline__ ItemRing *static_item_ring() {
    if constexpr (VARLEN) return &item_ring();
    else return nullptr;
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

// VARLEN: q, out are [total][H][d] and k, v [total][Hkv][d] (token-major, packed
// sequences); their tensor maps are (d, heads, total) with 1 x 128 / 1 x 64 boxes,
// so a tile lands in shared memory exactly as in the [B][H][N][d] case.
template <typename T, int D, bool CAUSAL, bool HAS_MASK, bool VARLEN = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_m,
                  const FwdParams p) {
    static_assert(!(VARLEN && HAS_MASK), "no mask in a packed batch");
    using C = Cfg<T, D, HAS_MASK>;
    constexpr int R = C::RING;
    if constexpr (HAS_MASK) {
        if (p.mask_kind != nullptr) {
            // queued behind the 128-key kernel as its programmatic dependent: let that grid finish
            // (so that later work on the stream is ordered after it), then return if it applied the mask
            grid_dependency_wait();
            if (*p.mask_kind == 0) return;
        }
    }
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Sync<R> sy{reinterpret_cast<uint64_t *>(smem + C::SMEM_BAR)};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::SMEM_BAR + C::NUM_BARS * 8);
    // a static shared word: its address is a constant, so no register holds it
    __shared__ int abort_word;
    volatile int *abort_flag = &abort_word;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(sy.q_full(t), 1);
            mbar_init(sy.q_empty(t), 1);
            mbar_init(sy.s_full(t), 1);
            mbar_init(sy.s_free(t), kBQ);
            mbar_init(sy.p_full(t, 0), kBQ);
            mbar_init(sy.p_full(t, 1), kBQ);
            mbar_init(sy.pv_done(t, 0), 1);
            mbar_init(sy.pv_done(t, 1), 1);
        }
        for (int s = 0; s < R; ++s) {  // a K or V slot is released by both tiles' issuers
            mbar_init(sy.k_full(s), 1);
            mbar_init(sy.k_empty(s), 2);
            mbar_init(sy.v_full(s), 1);
            mbar_init(sy.v_empty(s), 2);
        }
        mbar_init(sy.drain(), 4);  // one commit per issuing warp
        if constexpr (HAS_MASK) {
            for (int w = 0; w < 8; ++w) mbar_init(smem_u32(mask_bars() + w), 1);
        }
        if constexpr (VARLEN) {
            ItemRing &ring = item_ring();
            for (int i = 0; i < kItemRing; ++i) {
                mbar_init(smem_u32(&ring.full[i]), 1);
                mbar_init(smem_u32(&ring.empty[i]), kItemConsumers);
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

    if (warp >= 8) {
        setmaxnreg_dec<56>();
        if (warp == 8) {
            // ---------------------------------------------------------- TMA producer
            // The whole warp runs the (uniform) loop; lane 0 issues the copies.
            // Load order per item: K_0, then K_{j+1}, V_j for j = 0 .. nmax-1.
            const bool leader = lane == 0;
            const uint64_t pol_kv = policy_evict_last();
            const uint64_t pol_q = policy_evict_first();
            uint32_t qcount[2] = {0, 0};
            uint32_t kpos = 0, vpos = 0;
            int kv_y = 0, kv_z = 0, tok0 = 0;  // K/V tensor-map coordinates of the item
            bool ok = true;
            auto load_kv = [&](bool is_v, int blk) -> bool {
                uint32_t &pos = is_v ? vpos : kpos;
                const int s = pos % R;
                const uint32_t full = is_v ? sy.v_full(s) : sy.k_full(s);
                const uint32_t empty = is_v ? sy.v_empty(s) : sy.k_empty(s);
                if (!wait_warp(empty, ((pos / R) & 1u) ^ 1u, abort_flag, p)) return false;
                if (leader) {
                    const uint32_t dst = smem_u32(smem + (is_v ? C::SMEM_V : C::SMEM_KV) + s * C::KV_TILE);
                    mbar_arrive_expect_tx(full, C::KV_TILE);
#pragma unroll
                    for (int c = 0; c < C::NCH; ++c)
                        tma_load_3d(dst + c * C::KV_CHUNK, is_v ? &tm_v : &tm_k, full, c * C::CHUNK_ELEMS,
                                    VARLEN ? kv_y : blk * kBK, VARLEN ? tok0 + blk * kBK : kv_z, pol_kv);
                }
                __syncwarp();
                ++pos;
                return true;
            };
            ItemIter<VARLEN> iter(p, abort_flag, static_item_ring<VARLEN>());
            for (Item itm; ok && iter.next(p, itm, ok);) {
                const int q0 = itm.q0, cur_bh = itm.bh;
                // grouped-query attention: kv_group consecutive query heads share one K/V head
                const int kv_h = (cur_bh % p.H) / p.kv_group;
                if (VARLEN) {
                    kv_y = kv_h;
                    tok0 = itm.tok0;
                } else {
                    kv_z = (cur_bh / p.H) * (p.H / p.kv_group) + kv_h;
                }
                const int n0 = tile_nkv<CAUSAL>(itm, 0), n1 = tile_nkv<CAUSAL>(itm, 1);
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
                // an item with no rows (a packed sequence shorter than q0) loads nothing:
                // every K/V slot filled here must be consumed by the issuers
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
                // the most recent load of each slot is positions pos-R .. pos-1
                for (uint32_t q = kpos > (uint32_t)R ? kpos - R : 0; q < kpos; ++q)
                    while (!mbar_try_wait(sy.k_full(q % R), (q / R) & 1u) && global_timer_ns() - t0 < p.timeout_ns) {
                    }
                for (uint32_t q = vpos > (uint32_t)R ? vpos - R : 0; q < vpos; ++q)
                    while (!mbar_try_wait(sy.v_full(q % R), (q / R) & 1u) && global_timer_ns() - t0 < p.timeout_ns) {
                    }
            }
        } else if (warp == 9 || warp == 10) {
            // ---------------------------------------------------------- S issuer for tile t
            // S_t(j) = Q_t K_j^T into S_t's columns, after the softmax has copied the
            // previous S_t out. K slots this tile does not need are released at once.
            const int t = warp - 9;
            const uint32_t issue = lane == 0 ? 1u : 0u;
            const uint64_t a0 = smem_desc_sw128(smem_u32(smem + C::SMEM_Q + t * C::Q_TILE), 16, 1024);
            const uint64_t kd0 = smem_desc_sw128(smem_u32(smem + C::SMEM_KV), 16, 1024);
            const uint32_t d_s = tmem + t * 64;
            constexpr uint64_t KVT16 = C::KV_TILE >> 4;
            uint32_t qcount = 0, s_issued = 0, kpos = 0;
            bool ok = true;
            ItemIter<VARLEN> iter(p, abort_flag, static_item_ring<VARLEN>());
            for (Item itm; ok && iter.next(p, itm, ok);) {
                const int nt = tile_nkv<CAUSAL>(itm, t);
                const int nmax = max(tile_nkv<CAUSAL>(itm, 0), tile_nkv<CAUSAL>(itm, 1));
                if (nt > 0) {
                    ok = wait_warp(sy.q_full(t), qcount & 1u, abort_flag, p);
                    ++qcount;
                }
                for (int j = 0; ok && j < nmax; ++j, ++kpos) {
                    const int slot = kpos % R;
                    ok = wait_warp(sy.k_full(slot), (kpos / R) & 1u, abort_flag, p);
                    if (!ok) break;
                    if (j >= nt) {
                        if (lane == 0) mbar_arrive(sy.k_empty(slot));
                        continue;
                    }
                    if (s_issued > 0) ok = wait_warp(sy.s_free(t), (s_issued - 1) & 1u, abort_flag, p);
                    if (!ok) break;
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
                }
            }
            __syncwarp();
            tc_commit(sy.drain(), issue);
        } else if (warp == 11 || warp == 12) {
            // ---------------------------------------------------------- PV issuer for tile t
            // O_t (+)= P_t(j) V_j once the softmax has written P_t(j) into buffer g & 1.
            const int t = warp - 11;
            const uint32_t issue = lane == 0 ? 1u : 0u;
            const uint64_t vd0 = smem_desc_sw128(smem_u32(smem + C::SMEM_V), C::KV_CHUNK, 1024);
            const uint32_t d_o = tmem + 256 + t * 128;
            const uint32_t a_p = tmem + 128 + t * 64;
            constexpr uint64_t KVT16 = C::KV_TILE >> 4;
            uint32_t g = 0, vpos = 0;
            bool ok = true;
            ItemIter<VARLEN> iter(p, abort_flag, static_item_ring<VARLEN>());
            for (Item itm; ok && iter.next(p, itm, ok);) {
                const int nt = tile_nkv<CAUSAL>(itm, t);
                const int nmax = max(tile_nkv<CAUSAL>(itm, 0), tile_nkv<CAUSAL>(itm, 1));
                for (int j = 0; ok && j < nmax; ++j, ++vpos) {
                    const int slot = vpos % R;
                    ok = wait_warp(sy.v_full(slot), (vpos / R) & 1u, abort_flag, p);
                    if (!ok) break;
                    if (j >= nt) {
                        if (lane == 0) mbar_arrive(sy.v_empty(slot));
                        continue;
                    }
                    const uint32_t b = g & 1u;
                    ok = wait_warp(sy.p_full(t, b), (g >> 1) & 1u, abort_flag, p);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t b0 = vd0 + slot * KVT16;
#pragma unroll
                    for (int k = 0; k < C::KSTEPS_PV; ++k)
                        mma_ts(d_o, a_p + b * 32 + k * 8, b0 + (uint64_t)((k * C::V_KSTEP_BYTES) >> 4), C::IDESC_PV,
                               (k > 0 || j > 0) ? 1u : 0u, issue);
                    tc_commit(sy.pv_done(t, b), issue);
                    tc_commit(sy.v_empty(slot), issue);
                    ++g;
                }
            }
            __syncwarp();
            tc_commit(sy.drain(), issue);
        } else if (VARLEN && warp == 13) {
            // ---------------------------------------------------------- packed-batch item list
            // Walks the compact list and publishes one descriptor per item, then an
            // end marker, each into the next ring slot once all consumers have read
            // the slot's previous descriptor.
            ItemRing &ring = item_ring();
            VarlenCursor cur(p);
            bool more = true;
            for (uint32_t i = 0; more; ++i) {
                Item it;
                more = cur.next(p, it);
                const uint32_t slot = i % kItemRing;
                if (!wait_warp(smem_u32(&ring.empty[slot]), ((i / kItemRing) & 1u) ^ 1u, abort_flag, p)) break;
                if (lane == 0) {
                    ring.desc[slot] = more ? make_int4(it.bh, it.q0, it.n, it.tok0) : make_int4(-1, 0, 0, 0);
                    mbar_arrive(smem_u32(&ring.full[slot]));  // release: the descriptor is visible to waiters
                }
                __syncwarp();
            }
        }
    } else {
        setmaxnreg_inc<200>();
        // -------------------------------------------------------------- softmax + epilogue
        const int t = warp >> 2;                   // query tile of this warpgroup
        const int r = threadIdx.x & 127;           // row within the tile = TMEM lane
        // mask staging area of this warp (masked variant only): two 32-row x 128-byte TMA boxes
        const uint32_t mwarp = smem_u32(smem + C::SMEM_MASK + t * C::MASK_TILE + (warp & 3) * 8192);
        const uint64_t mpol = policy_evict_last();  // the mask is shared by every head of a batch index
        uint32_t mcount = 0;    // mask blocks consumed by this warp (parity of its barrier)
        bool mpending = false;  // a mask copy is in flight
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_addr = tmem + lane_base + t * 64;
        const uint32_t p_addr = tmem + lane_base + 128 + t * 64;
        const uint32_t o_addr = tmem + lane_base + 256 + t * 128;
        const float scale_log2 = p.scale_log2;
        const bool fast = !HAS_MASK && scale_log2 > 0.0f;
        // x holds raw scores, scaled by sl2 inside the exponent, on the fast path
        // (no mask, positive scale); otherwise pre-scaled scores with sl2 = 1 (a
        // -inf raw score times a non-positive scale is not -inf).
        const float sl2 = fast ? scale_log2 : 1.0f;
        uint32_t scount = 0;  // S blocks consumed (all items)
        uint32_t g = 0;       // P blocks produced (all items) = P V products of this tile
        bool ok = true;
        ItemIter<VARLEN> iter(p, abort_flag, static_item_ring<VARLEN>());
        for (Item itm; ok && iter.next(p, itm, ok);) {
            const int bh = itm.bh, q0 = itm.q0, n = itm.n;
            const int nt = tile_nkv<CAUSAL>(itm, t);
            if (nt == 0) continue;
            const int row = q0 + t * kBQ + r;  // global query row (may be >= N in a ragged tail)
            const int b = bh / p.H;
            const int mz = p.mask_per_head ? bh : b;  // the mask's [B] or [B][H] slab of this item
            // HAS_MASK (mask_tma): the warp's 32 rows x 64 mask values of a key block arrive by two TMA
            // boxes (32 rows x 32 fp32, 128-byte swizzle; rows past N and keys past N read as 0) into the
            // warp's 8 KB staging area, issued while the block before it is processed
            const int mrow0 = q0 + t * kBQ + (warp & 3) * 32;
            auto stage_mask = [&](int jj) {  // all 32 lanes
                fence_proxy_async_smem();  // this lane's reads of the area come before the copy's writes
                __syncwarp();
                if (lane == 0) {
                    const uint32_t bar = smem_u32(mask_bars() + warp);
                    mbar_arrive_expect_tx(bar, 2 * 32 * 128);
                    tma_load_3d(mwarp, &tm_m, bar, jj * kBK, mrow0, mz, mpol);
                    tma_load_3d(mwarp + 4096, &tm_m, bar, jj * kBK + 32, mrow0, mz, mpol);
                }
                __syncwarp();
                mpending = true;
            };
            if constexpr (HAS_MASK) {
                if (p.mask_tma && nt > 0) stage_mask(0);
            }
            float m_ref = -INFINITY, l = 0.0f;
            for (int j = 0; j < nt; ++j, ++g) {
                ok = wait_warp(sy.s_full(t), scount & 1u, abort_flag, p);
                ++scount;
                if (!ok) break;
                tc_fence_after();
                uint32_t sr[64];
                tmem_ld64_nowait(s_addr, sr);
                tmem_wait_ld_dep64(sr);
                tc_fence_before();
                mbar_arrive(sy.s_free(t));  // S_t may now be overwritten by the next block
                float x[64];
                const int kbase = j * kBK;
                if constexpr (HAS_MASK) {
                    const bool row_ok = row < p.N;
                    const float *mrow = p.mask + ((size_t)mz * p.N + (size_t)(row_ok ? row : 0)) * p.N + kbase;
                    if (p.mask_tma) {  // warp-uniform
                        ok = wait_warp(smem_u32(mask_bars() + warp), mcount & 1u, abort_flag, p);
                        if (!ok) break;
                        ++mcount;
                        mpending = false;
#pragma unroll
                        for (int c = 0; c < 64; c += 4) {
                            // float c of this row: box c / 32, 16-byte chunk (c % 32) / 4 swizzled by row
                            const uint32_t chunk = (uint32_t)((c & 31) >> 2) ^ (uint32_t)(lane & 7);
                            const float4 mv =
                                ld_shared_v4f(mwarp + (uint32_t)((c >> 5) * 4096 + lane * 128) + (chunk << 4));
                            x[c + 0] = fmaf(__uint_as_float(sr[c + 0]), scale_log2, mv.x * 1.4426950408889634f);
                            x[c + 1] = fmaf(__uint_as_float(sr[c + 1]), scale_log2, mv.y * 1.4426950408889634f);
                            x[c + 2] = fmaf(__uint_as_float(sr[c + 2]), scale_log2, mv.z * 1.4426950408889634f);
                            x[c + 3] = fmaf(__uint_as_float(sr[c + 3]), scale_log2, mv.w * 1.4426950408889634f);
                        }
                        if (j + 1 < nt) stage_mask(j + 1);
                    } else {
#pragma unroll
                        for (int c = 0; c < 64; ++c) {
                            const float mv = (row_ok && kbase + c < p.N) ? __ldg(mrow + c) : 0.0f;
                            x[c] = fmaf(__uint_as_float(sr[c]), scale_log2, mv * 1.4426950408889634f);
                        }
                    }
                } else if (fast) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) x[c] = __uint_as_float(sr[c]);
                } else {
#pragma unroll
                    for (int c = 0; c < 64; ++c) x[c] = __uint_as_float(sr[c]) * scale_log2;
                }
                // keys past the end of the sequence, and (causal) keys after the query
                const int tile_row0 = q0 + t * kBQ;
                const bool ragged = kbase + kBK > n;
                const bool diag = CAUSAL && (kbase + kBK - 1 > tile_row0);
                if (ragged || diag) {
                    int lim = n - 1 - kbase;
                    if (CAUSAL) lim = min(lim, row - kbase);
#pragma unroll
                    for (int c = 0; c < 64; ++c) x[c] = (c > lim) ? -INFINITY : x[c];
                }
                // row maximum: eight independent three-input chains, then a short tree
                float m8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) m8[i] = fmax3(x[i], x[8 + i], x[16 + i]);
#pragma unroll
                for (int i = 0; i < 8; ++i) m8[i] = fmax3(m8[i], x[24 + i], x[32 + i]);
#pragma unroll
                for (int i = 0; i < 8; ++i) m8[i] = fmax3(m8[i], x[40 + i], x[48 + i]);
#pragma unroll
                for (int i = 0; i < 8; ++i) m8[i] = fmaxf(m8[i], x[56 + i]);
                const float mraw =
                    fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                const float mb = mraw * sl2;  // sl2 > 0, so scaling commutes with the maximum
                const float m_new = fmaxf(m_ref, mb);
                // lazy rescale: move the reference only when the maximum grew by more than TAU
                const bool need = (m_new > m_ref + kTau) || (m_ref == -INFINITY && m_new != -INFINITY);
                const float alpha = need ? ex2_approx(m_ref - m_new) : 1.0f;  // 2^-inf = 0
                if (__any_sync(0xffffffffu, need) && j > 0) {
                    // O holds P V for blocks < j: wait for the product of block j-1, then scale rows in place
                    const uint32_t gp = g - 1;
                    ok = wait_warp(sy.pv_done(t, gp & 1u), (gp >> 1) & 1u, abort_flag, p);
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
                // exponent arguments and partial sums in packed pairs (one instruction per two keys)
                const float2 sl2v = make_float2(sl2, sl2), negv = make_float2(neg, neg);
                float2 ls[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
                uint32_t pv[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float2 a = ffma2(make_float2(x[2 * c], x[2 * c + 1]), sl2v, negv);
                    const float2 e = make_float2(ex2_approx(a.x), ex2_approx(a.y));
                    ls[c & 1] = fadd2(ls[c & 1], e);
                    pv[c] = pack2<T>(e.x, e.y);
                }
                l += (ls[0].x + ls[0].y) + (ls[1].x + ls[1].y);
                // P buffer (g & 1) was last read by the product of block g - 2
                if (g >= 2) {
                    ok = wait_warp(sy.pv_done(t, g & 1u), ((g - 2) >> 1) & 1u, abort_flag, p);
                    if (!ok) break;
                    tc_fence_after();
                }
                tmem_st32(p_addr + (g & 1u) * 32, pv);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(sy.p_full(t, g & 1u));
            }
            if (!ok) break;
            // ---------------------------------------------------------- epilogue
            const uint32_t gl = g - 1;  // the last product of this item
            ok = wait_warp(sy.pv_done(t, gl & 1u), (gl >> 1) & 1u, abort_flag, p);
            if (!ok) break;
            tc_fence_after();
            const float inv = (l > 0.0f) ? 1.0f / l : 0.0f;
            // [B][H][N][d] rows, or token-major [total][H][d] rows of a packed batch
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
            if (row < n)  // lse: [B][H][N], or [H][total] for a packed batch
                p.lse[VARLEN ? (size_t)(bh % p.H) * p.total + itm.tok0 + row : (size_t)bh * p.N + row] =
                    (l > 0.0f) ? (m_ref + lg2_approx(l)) * 0.6931471805599453f : -INFINITY;
        }
        if constexpr (HAS_MASK) {  // a mask copy still in flight (after a timeout) lands before the CTA exits
            if (mpending) {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(smem_u32(mask_bars() + warp), mcount & 1u) &&
                       global_timer_ns() - t0 < p.timeout_ns) {
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        // every MMA of the four issuing warps must be complete before TMEM is released
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(sy.drain(), 0) && global_timer_ns() - t0 < p.timeout_ns) {
        }
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace fa
