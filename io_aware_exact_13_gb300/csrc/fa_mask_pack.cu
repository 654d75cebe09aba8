// fa_mask_pack.cu -- one bit per entry for an additive mask whose entries are
// all 0 or -inf.
//
// The glossary "FlashAttention", section "Move less data", adds a mask M to the
// scaled scores inside the tile loop. Most masks in practice (padding, causal
// variants, block or random sparsity, fully masked rows) hold only 0 and -inf,
// and for those s + M is either s or -inf: one bit per entry carries all of M.
// Each head of a batch index reads the same [N][Nk] mask, so packing it once per
// call replaces H reads of 4 bytes per (row, key) on chip with H reads of one
// bit. Any other value (finite nonzero, +inf, NaN) sets the kind word, and the
// fp32 mask is then used as given.
//
// Layout of the bits: [rows][ceil(Nk / 128)] 16-byte units; unit (r, j) covers
// keys 128 j .. 128 j + 127 of row r as four 32-bit words, and bit l of word c
// is key 128 j + 4 l + c (set = -inf). Keys past Nk are 0. The interleave is
// what one warp produces when lane l reads keys 4 l .. 4 l + 3 with one 16-byte
// load and the four words are ballots over the lanes.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "fa_launch.cuh"
#include "pdl.cuh"

namespace fa {

namespace {

constexpr int kPackThreads = 256;
constexpr int kPackUnroll = 8;  // units in flight per warp

// streaming load: the mask is read once per call
__device__ __forceinline__ float4 ld_stream_v4(const float *ptr) {
    float4 v;
    asm volatile("ld.global.cs.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(ptr));
    return v;
}

__device__ __forceinline__ float ld_stream(const float *ptr) {
    float v;
    asm volatile("ld.global.cs.f32 %0, [%1];" : "=f"(v) : "l"(ptr));
    return v;
}

// Each warp packs a contiguous range of (row, 128-key block) units, kPackUnroll at a time
// with all their loads issued before any is reduced; (row, block) advance without division.
// VEC: rows start on 16-byte boundaries (Nk % 4 == 0 and an aligned base), so lane l reads
// its four keys with one load.
template <bool VEC>
__global__ void __launch_bounds__(kPackThreads) fa_mask_pack_kernel(const float *__restrict__ mask,
                                                                    uint4 *__restrict__ bits, int *__restrict__ kind,
                                                                    long long rows, int nk, int nblk) {
    grid_launch_dependents();  // the 128-key kernel may be scheduled; it waits for this grid to finish
    const int lane = threadIdx.x & 31;
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const long long units = rows * nblk;
    const long long per_warp = (units + nwarps - 1) / nwarps;
    long long u = warp * per_warp;
    const long long u_end = u + per_warp < units ? u + per_warp : units;
    long long row = u / nblk;
    int blk = (int)(u - row * nblk);
    bool other = false;  // a value that is neither 0 nor -inf
    for (; u < u_end; u += kPackUnroll) {
        float v[kPackUnroll][4];
        long long r = row;
        int b = blk;
#pragma unroll
        for (int i = 0; i < kPackUnroll; ++i) {
            const bool in = u + i < u_end;
            const int key = b * 128 + 4 * lane;
            const float *src = mask + r * (long long)nk + key;
            if (in && VEC && key + 4 <= nk) {
                const float4 f = ld_stream_v4(src);
                v[i][0] = f.x, v[i][1] = f.y, v[i][2] = f.z, v[i][3] = f.w;
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) v[i][c] = (in && key + c < nk) ? ld_stream(src + c) : 0.0f;
            }
            if (++b == nblk) b = 0, ++r;
        }
#pragma unroll
        for (int i = 0; i < kPackUnroll; ++i) {
            if (u + i >= u_end) break;  // warp-uniform
            uint32_t w[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const bool neg_inf = v[i][c] == -INFINITY;
                other |= !(neg_inf || v[i][c] == 0.0f);
                w[c] = __ballot_sync(0xffffffffu, neg_inf);
            }
            if (lane == 0) bits[u + i] = make_uint4(w[0], w[1], w[2], w[3]);
        }
        row = r;
        blk = b;
    }
    if (__any_sync(0xffffffffu, other) && lane == 0) *kind = 1;
}

}  // namespace

size_t mask_bits_bytes(long long rows, int nk) {
    return static_cast<size_t>(rows) * static_cast<size_t>((nk + 127) / 128) * 16u;
}

int launch_mask_pack(const float *mask, void *bits, int *kind, long long rows, int nk, int num_sms,
                     cudaStream_t stream) {
    if (cudaMemsetAsync(kind, 0, sizeof(int), stream) != cudaSuccess) return -5;
    const int nblk = (nk + 127) / 128;
    const long long units = rows * nblk;
    const long long per_block = kPackThreads / 32;
    long long grid = (units + per_block - 1) / per_block;
    const long long cap = static_cast<long long>(num_sms) * (2048 / kPackThreads);  // one full wave
    if (grid > cap) grid = cap;
    const bool vec = (nk % 4) == 0 && (reinterpret_cast<uintptr_t>(mask) & 15u) == 0;
    if (vec)
        fa_mask_pack_kernel<true><<<(unsigned)grid, kPackThreads, 0, stream>>>(mask, static_cast<uint4 *>(bits), kind,
                                                                               rows, nk, nblk);
    else
        fa_mask_pack_kernel<false><<<(unsigned)grid, kPackThreads, 0, stream>>>(mask, static_cast<uint4 *>(bits),
                                                                                kind, rows, nk, nblk);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

}  // namespace fa
