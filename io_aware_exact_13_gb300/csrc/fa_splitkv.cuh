// fa_splitkv.cuh -- host-side arguments of the split-KV decoding forward.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

constexpr int kSplitKVMaxNq = 16;

struct SplitKVArgs {
    const void *q, *k, *v;
    void *out;
    float *lse;
    int B, H, Nq, Nk, d;
    float scale;
    int causal;
    int n_splits;
    float *o_part;    // workspace: [n_splits][B*H*Nq][d]
    float *lse_part;  // workspace: [n_splits][B*H*Nq]
    cudaStream_t stream;
};

// Workspace bytes for (rows = B*H*Nq, d, n_splits), each part 256-byte aligned.
inline size_t splitkv_workspace_bytes(int64_t rows, int d, int n_splits) {
    const size_t o = (size_t)n_splits * (size_t)rows * (size_t)d * sizeof(float);
    const size_t l = (size_t)n_splits * (size_t)rows * sizeof(float);
    return ((o + 255) / 256) * 256 + ((l + 255) / 256) * 256;
}

int launch_splitkv(const SplitKVArgs &a, bool fp16);

// Resident CTAs per SM of the partial kernel used for (d, Nq) (bf16 variant).
int splitkv_blocks_per_sm(int d, int Nq);
// FA_LOG=1: one line per call to stderr (defined in fa_api.cu).
void log_call(const char *fmt, ...);

}  // namespace fa
