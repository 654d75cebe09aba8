// fa_bwd.cuh -- host-side arguments of the attention backward (recomputation).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

constexpr int kBwdRows = 128;  // query rows per recomputed tile and keys per CTA

struct BwdArgs {
    const void *q, *k, *v, *out, *dout;  // [B][H][N][d]
    const float *lse;                    // [B][H][N], natural log
    void *dq, *dk, *dv;                  // [B][H][N][d]
    int B, H, N, d;
    float scale;
    int causal;
    float *dq_acc;   // workspace: fp32 [B*H][N][d]
    float *lse2;     // workspace: fp32 [B*H][Npad], lse * log2(e), +inf past N
    float *dsum;     // workspace: fp32 [B*H][Npad], rowsum(dO o O), 0 past N
    cudaStream_t stream;
    int *status;
    uint64_t timeout_ns;
};

inline int64_t bwd_padded_rows(int N) { return ((static_cast<int64_t>(N) + kBwdRows - 1) / kBwdRows) * kBwdRows; }

// Workspace bytes for B*H heads of N rows and head dimension d, each part
// 256-byte aligned: dQ accumulator, then lse2, then dsum.
inline size_t bwd_workspace_bytes(int64_t BH, int N, int d) {
    const size_t acc = static_cast<size_t>(BH) * static_cast<size_t>(N) * static_cast<size_t>(d) * sizeof(float);
    const size_t row = static_cast<size_t>(BH) * static_cast<size_t>(bwd_padded_rows(N)) * sizeof(float);
    return ((acc + 255) / 256) * 256 + 2 * (((row + 255) / 256) * 256);
}

int launch_bwd(const BwdArgs &a, bool fp16);

}  // namespace fa
