// fa_splitkv_noalloc.cu -- split-KV decoding forward that needs no workspace
// from the caller.
//
// Some callers cannot allocate device memory at the point where they call
// attention: a host framework that owns every device allocation through its
// own pool, a serving loop in which cudaMalloc's implicit device-wide
// synchronisation would stall other work, or an embedded host with a fixed
// memory budget. For them this entry point keeps its scratch (the per-split
// partial outputs and log-sum-exps) in one fixed array compiled into the
// library, so a call allocates nothing.
//
// The array is kNoAllocScratchBytes (16 MiB) of device memory that every GPU
// which loads the library holds until the process exits. All calls share it,
// so calls that overlap on the GPU (different streams, or different host
// threads) race on it and must be serialised by the caller. It keeps the last
// call's contents; nothing in it needs to start at zero, because every entry
// the merge kernel reads is written earlier in the same call.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/fa.h"
#include "fa_splitkv.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

// The scratch itself. In host code this name is only a stand-in for the device
// symbol, never a device address: the address is looked up per device below.
static __device__ __align__(256) unsigned char g_splitkv_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevicesNA = 64;
std::mutex g_scratch_mutex;
std::atomic<void *> g_scratch[kMaxDevicesNA];  // device address of g_splitkv_scratch per device, or null

// Set-up per device, with that device current (it is the caller's current
// device when a call is made on it). Only a successful lookup is kept: if the
// lookup fails (for instance because the first call was made while a stream
// capture was in progress), the next call tries again.
void *scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesNA) return nullptr;
    void *ptr = g_scratch[dev].load(std::memory_order_acquire);
    if (ptr) return ptr;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    ptr = g_scratch[dev].load(std::memory_order_relaxed);
    if (ptr) return ptr;
    if (cudaGetSymbolAddress(&ptr, g_splitkv_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();  // leave no sticky error from the failed lookup behind
        return nullptr;
    }
    g_scratch[dev].store(ptr, std::memory_order_release);
    return ptr;
}

bool aligned_na(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" int fa_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *out, float *lse, int B,
                                      int H, int Nq, int Nk, int d, float scale, int causal, int n_splits,
                                      void *stream) {
    if (!q || !k || !v || !out || !lse) return FA_ERR_NULL;
    if (!aligned_na(q, 16) || !aligned_na(k, 16) || !aligned_na(v, 16) || !aligned_na(out, 16) ||
        !aligned_na(lse, 4))
        return FA_ERR_ALIGN;
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || Nq > fa::kSplitKVMaxNq) return FA_ERR_SHAPE;
    if (static_cast<int64_t>(B) * H > 65535) return FA_ERR_SHAPE;
    if (n_splits < 1 || n_splits > Nk || n_splits > 65535) return FA_ERR_SHAPE;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    const int64_t rows = static_cast<int64_t>(B) * H * Nq;
    if (fa::splitkv_workspace_bytes(rows, d, n_splits) > kNoAllocScratchBytes) return FA_ERR_WORKSPACE;
    fa::log_call("split-KV noalloc bf16 d=%d causal=%d B=%d H=%d Nq=%d Nk=%d splits=%d", d, causal ? 1 : 0, B, H,
                 Nq, Nk, n_splits);
    void *scratch = scratch_address();
    if (!scratch) return FA_ERR_LAUNCH;
    fa::SplitKVArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.lse = lse;
    a.B = B;
    a.H = H;
    a.Nq = Nq;
    a.Nk = Nk;
    a.d = d;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.n_splits = n_splits;
    const size_t o_bytes = ((static_cast<size_t>(n_splits) * rows * d * sizeof(float) + 255) / 256) * 256;
    a.o_part = static_cast<float *>(scratch);
    a.lse_part = reinterpret_cast<float *>(static_cast<char *>(scratch) + o_bytes);
    a.stream = static_cast<cudaStream_t>(stream);
    return fa::launch_splitkv(a, false);
}
