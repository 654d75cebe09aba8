// fa_api.cu -- the C ABI declared in include/fa.h: argument checks, the device
// status word, tensor-map encoding, and dispatch to the per-type launchers.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "../../include/fa.h"
#include "fa_launch.cuh"
#include "fa_bwd.cuh"
#include "fa_splitkv.cuh"

namespace fa {
int launch_fwd_bf16(const LaunchArgs &a);
int launch_fwd_fp16(const LaunchArgs &a);
int launch_fwd_fp32(const LaunchArgs &a);
int launch_fwd_varlen_bf16(const LaunchArgs &a);
int launch_fwd_varlen_fp16(const LaunchArgs &a);
}  // namespace fa

namespace fa {
// FA_LOG=1 in the environment prints one line per call to stderr: the entry
// point, the kernel variant it dispatches to and the problem size.
static bool log_enabled() {
    static const bool on = [] {
        const char *v = std::getenv("FA_LOG");
        return v != nullptr && v[0] != '\0' && v[0] != '0';
    }();
    return on;
}
void log_call(const char *fmt, ...) {
    if (!log_enabled()) return;
    va_list ap;
    va_start(ap, fmt);
    std::fputs("[fa] ", stderr);
    std::vfprintf(stderr, fmt, ap);
    std::fputc('\n', stderr);
    va_end(ap);
}
}  // namespace fa
using fa::log_call;

// Device status word: FA_OK, or FA_ERR_TIMEOUT once any bounded wait gave up.
__device__ int g_fa_status = 0;

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 4000000000ull;  // 4 s per pipeline wait

struct DeviceInfo {
    std::once_flag once;
    int num_sms = -1;
    int *status = nullptr;
    bool ok = false;
    // copy streams of the host-buffer entry points (created on first use)
    std::once_flag streams_once;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    bool streams_ok = false;
};
DeviceInfo g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

// Per-device set-up, once: SM count and the device address of the status word.
DeviceInfo *device_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    DeviceInfo &di = g_dev[dev];
    std::call_once(di.once, [&di, dev] {
        int sms = 0;
        void *addr = nullptr;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return;
        if (cudaGetSymbolAddress(&addr, g_fa_status) != cudaSuccess || addr == nullptr) return;
        di.num_sms = sms;
        di.status = static_cast<int *>(addr);
        di.ok = true;
    });
    return di.ok ? &di : nullptr;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }


enum class Type { BF16, FP16, FP32 };

int check_args(Type ty, const void *q, const void *k, const void *v, const float *mask, const void *out,
               const float *lse, int B, int H, int N, int d) {
    if (!q || !k || !v || !out || !lse) return FA_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
        (mask && !aligned(mask, 16)))
        return FA_ERR_ALIGN;
    if (B < 1 || H < 1 || N < 1) return FA_ERR_SHAPE;
    const int64_t bh = static_cast<int64_t>(B) * H;
    if (bh > INT32_MAX) return FA_ERR_SHAPE;
    const int64_t items = bh * ((static_cast<int64_t>(N) + 255) / 256);
    if (items > INT32_MAX) return FA_ERR_SHAPE;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    if (ty == Type::FP32 && bh > 65535) return FA_ERR_SHAPE;
    return FA_OK;
}

int fwd_common(Type ty, const void *q, const void *k, const void *v, const float *mask, void *out, float *lse,
               int B, int H, int N, int d, float scale, int causal, void *stream, int Hkv = -1,
               int mask_per_head = 0, void *workspace = nullptr) {
    int rc = check_args(ty, q, k, v, mask, out, lse, B, H, N, d);
    if (rc != FA_OK) return rc;
    if (Hkv == -1) Hkv = H;
    if (Hkv < 1 || H % Hkv != 0) return FA_ERR_SHAPE;
    log_call("forward %s d=%d causal=%d mask=%s B=%d H=%d Hkv=%d N=%d scale=%g",
             ty == Type::BF16 ? "bf16 tcgen05" : ty == Type::FP16 ? "fp16 tcgen05" : "fp32 cuda-core", d,
             causal ? 1 : 0, mask == nullptr ? "none" : mask_per_head ? "per-head bias" : "shared", B, H, Hkv, N,
             static_cast<double>(scale));
    DeviceInfo *di = device_info();
    if (!di || !encoder()) return FA_ERR_LAUNCH;
    fa::LaunchArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.mask = mask;
    a.out = out;
    a.lse = lse;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.Hkv = Hkv;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.stream = static_cast<cudaStream_t>(stream);
    a.status = di->status;
    a.num_sms = di->num_sms;
    a.timeout_ns = kDefaultTimeoutNs;
    a.mask_per_head = mask_per_head;
    // With a workspace, a shared mask is first packed to one bit per entry (on every call: the mask
    // may change between calls); without one the fp32 mask is applied as given.
    if (workspace && mask && !mask_per_head && ty != Type::FP32) {
        const long long rows = static_cast<long long>(B) * N;
        int *kind = reinterpret_cast<int *>(static_cast<char *>(workspace) + fa::mask_bits_bytes(rows, N));
        if (fa::launch_mask_pack(mask, workspace, kind, rows, N, di->num_sms, a.stream) != 0) return FA_ERR_LAUNCH;
        a.mask_bits = workspace;
        a.mask_kind = kind;
    }
    switch (ty) {
        case Type::BF16: rc = fa::launch_fwd_bf16(a); break;
        case Type::FP16: rc = fa::launch_fwd_fp16(a); break;
        case Type::FP32: rc = fa::launch_fwd_fp32(a); break;
    }
    return rc;
}

// Keep threshold of drop probability p: (1 - p) rounded to a multiple of 1/256 (halves up), as
// the count of byte values that keep; 0 when nothing would be kept (or p < 0, or p is NaN).
int dropout_threshold(float p_drop) {
    const double x = std::floor((1.0 - static_cast<double>(p_drop)) * 256.0 + 0.5);
    if (!(x >= 1.0 && x <= 256.0)) return 0;
    return static_cast<int>(x);
}

int dropout_common(Type ty, const void *q, const void *k, const void *v, void *out, float *lse, int B, int H, int Hkv,
                   int N, int d, float scale, int causal, float p_drop, unsigned long long seed,
                   unsigned long long offset, void *stream) {
    int rc = check_args(ty, q, k, v, nullptr, out, lse, B, H, N, d);
    if (rc != FA_OK) return rc;
    if (Hkv < 1 || H % Hkv != 0) return FA_ERR_SHAPE;
    const int t = dropout_threshold(p_drop);
    if (!(p_drop >= 0.0f) || t == 0) return FA_ERR_ARG;
    log_call("forward with dropout %s d=%d causal=%d B=%d H=%d Hkv=%d N=%d p=%g (keep %d/256) seed=%llu offset=%llu",
             ty == Type::BF16 ? "bf16" : "fp16", d, causal ? 1 : 0, B, H, Hkv, N, static_cast<double>(p_drop), t, seed,
             offset);
    DeviceInfo *di = device_info();
    if (!di || !encoder()) return FA_ERR_LAUNCH;
    fa::LaunchArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.mask = nullptr;
    a.out = out;
    a.lse = lse;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.Hkv = Hkv;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.stream = static_cast<cudaStream_t>(stream);
    a.status = di->status;
    a.num_sms = di->num_sms;
    a.timeout_ns = kDefaultTimeoutNs;
    a.drop_threshold = t;
    a.drop_seed = seed;
    a.drop_offset = offset;
    return ty == Type::BF16 ? fa::launch_fwd_drop_bf16(a) : fa::launch_fwd_drop_fp16(a);
}

// bytes of the masked forward's workspace: the packed mask, then the packing pass's verdict word
size_t masked_workspace_bytes(int B, int N) {
    return fa::mask_bits_bytes(static_cast<long long>(B) * N, N) + 256;
}

int masked_common(Type ty, const void *q, const void *k, const void *v, const float *mask, void *out, float *lse,
                  int B, int H, int Hkv, int N, int d, float scale, int causal, void *workspace,
                  unsigned long long workspace_bytes, void *stream) {
    if (!mask) return FA_ERR_NULL;
    int rc = check_args(ty, q, k, v, mask, out, lse, B, H, N, d);
    if (rc != FA_OK) return rc;
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < masked_workspace_bytes(B, N))
        return FA_ERR_WORKSPACE;
    return fwd_common(ty, q, k, v, mask, out, lse, B, H, N, d, scale, causal, stream, Hkv, 0, workspace);
}

// Forward from host buffers: the B*H head slabs are cut into n_chunks contiguous
// chunks; chunk c's Q, K, V copies (h2d stream), its forward (the caller's
// stream) and its O, lse copies (d2h stream) are chained by events, so the
// copies of one chunk overlap the forward of another.
int host_common(Type ty, const void *qh, const void *kh, const void *vh, void *oh, float *lh, void *qd, void *kd,
                void *vd, void *od, float *ld, int B, int H, int N, int d, float scale, int causal, int n_chunks,
                void *stream) {
    if (!qh || !kh || !vh || !oh || !lh) return FA_ERR_NULL;
    int rc = check_args(ty, qd, kd, vd, nullptr, od, ld, B, H, N, d);
    if (rc != FA_OK) return rc;
    const int64_t bh = static_cast<int64_t>(B) * H;
    if (n_chunks < 1 || n_chunks > bh || n_chunks > 64) return FA_ERR_SHAPE;
    DeviceInfo *di = device_info();
    if (!di || !encoder()) return FA_ERR_LAUNCH;
    std::call_once(di->streams_once, [di] {
        di->streams_ok = cudaStreamCreateWithFlags(&di->h2d, cudaStreamNonBlocking) == cudaSuccess &&
                         cudaStreamCreateWithFlags(&di->d2h, cudaStreamNonBlocking) == cudaSuccess;
    });
    if (!di->streams_ok) return FA_ERR_LAUNCH;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const size_t eb = ty == Type::FP32 ? 4 : 2;
    const size_t slab = static_cast<size_t>(N) * d * eb;  // bytes of one (b, h) slab of Q, K, V or O
    const size_t lslab = static_cast<size_t>(N) * sizeof(float);
    cudaEvent_t ev[2 * 64 + 2];
    int n_ev = 0;
    auto new_event = [&]() -> cudaEvent_t {
        cudaEvent_t e = nullptr;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
        ev[n_ev++] = e;
        return e;
    };
    rc = FA_OK;
    cudaEvent_t start = new_event();
    if (!start || cudaEventRecord(start, cs) != cudaSuccess || cudaStreamWaitEvent(di->h2d, start, 0) != cudaSuccess)
        rc = FA_ERR_LAUNCH;
    auto cpy = [](void *dst, const void *src, size_t n, cudaMemcpyKind kind, cudaStream_t st) {
        return cudaMemcpyAsync(dst, src, n, kind, st) == cudaSuccess;
    };
    // Chunk sizes shrink linearly (n_chunks : n_chunks-1 : ... : 1): the link is
    // the bound, and the last chunk's forward and copy-out, which no copy in
    // overlaps, should be short. cum(c) = sum of the first c weights.
    const int64_t wsum = static_cast<int64_t>(n_chunks) * (n_chunks + 1) / 2;
    auto cum = [n_chunks](int64_t c) { return c * n_chunks - c * (c - 1) / 2; };
    for (int c = 0; c < n_chunks && rc == FA_OK; ++c) {
        const int64_t h0 = bh * cum(c) / wsum, h1 = bh * cum(c + 1) / wsum;
        const int64_t nh = h1 - h0;
        if (nh == 0) continue;  // a chunk that rounds to no head
        const size_t off = static_cast<size_t>(h0) * slab, n = static_cast<size_t>(nh) * slab;
        const size_t loff = static_cast<size_t>(h0) * lslab, ln = static_cast<size_t>(nh) * lslab;
        char *qdc = static_cast<char *>(qd) + off, *kdc = static_cast<char *>(kd) + off;
        char *vdc = static_cast<char *>(vd) + off, *odc = static_cast<char *>(od) + off;
        float *ldc = reinterpret_cast<float *>(reinterpret_cast<char *>(ld) + loff);
        cudaEvent_t in_done = new_event(), fwd_done = new_event();
        if (!in_done || !fwd_done || !cpy(qdc, static_cast<const char *>(qh) + off, n, cudaMemcpyHostToDevice, di->h2d) ||
            !cpy(kdc, static_cast<const char *>(kh) + off, n, cudaMemcpyHostToDevice, di->h2d) ||
            !cpy(vdc, static_cast<const char *>(vh) + off, n, cudaMemcpyHostToDevice, di->h2d) ||
            cudaEventRecord(in_done, di->h2d) != cudaSuccess || cudaStreamWaitEvent(cs, in_done, 0) != cudaSuccess) {
            rc = FA_ERR_LAUNCH;
            break;
        }
        fa::LaunchArgs a;
        a.q = qdc;
        a.k = kdc;
        a.v = vdc;
        a.mask = nullptr;
        a.out = odc;
        a.lse = ldc;
        a.B = 1;
        a.H = static_cast<int>(nh);
        a.N = N;
        a.d = d;
        a.Hkv = static_cast<int>(nh);
        a.scale = scale;
        a.causal = causal ? 1 : 0;
        a.stream = cs;
        a.status = di->status;
        a.num_sms = di->num_sms;
        a.timeout_ns = kDefaultTimeoutNs;
        int lr = ty == Type::BF16 ? fa::launch_fwd_bf16(a) : fa::launch_fwd_fp16(a);
        if (lr != 0) {
            rc = lr;
            break;
        }
        if (cudaEventRecord(fwd_done, cs) != cudaSuccess || cudaStreamWaitEvent(di->d2h, fwd_done, 0) != cudaSuccess ||
            !cpy(static_cast<char *>(oh) + off, odc, n, cudaMemcpyDeviceToHost, di->d2h) ||
            !cpy(reinterpret_cast<char *>(lh) + loff, ldc, ln, cudaMemcpyDeviceToHost, di->d2h)) {
            rc = FA_ERR_LAUNCH;
            break;
        }
    }
    // the call is complete, on the caller's stream, when the last copy out is
    cudaEvent_t end = new_event();
    if (!end || cudaEventRecord(end, di->d2h) != cudaSuccess || cudaStreamWaitEvent(cs, end, 0) != cudaSuccess)
        rc = rc == FA_OK ? FA_ERR_LAUNCH : rc;
    for (int i = 0; i < n_ev; ++i) cudaEventDestroy(ev[i]);  // released once they have completed
    if (rc == FA_OK)
        log_call("forward from host %s d=%d causal=%d B=%d H=%d N=%d chunks=%d", ty == Type::BF16 ? "bf16" : "fp16",
                 d, causal ? 1 : 0, B, H, N, n_chunks);
    return rc;
}

int check_splitkv(const void *q, const void *k, const void *v, const void *out, const float *lse, int B, int H,
                  int Nq, int Nk, int d, int n_splits) {
    if (!q || !k || !v || !out || !lse) return FA_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(lse, 4))
        return FA_ERR_ALIGN;
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || Nq > fa::kSplitKVMaxNq) return FA_ERR_SHAPE;
    if (static_cast<int64_t>(B) * H > 65535) return FA_ERR_SHAPE;
    if (n_splits < 1 || n_splits > Nk || n_splits > 65535) return FA_ERR_SHAPE;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

int splitkv_common(bool fp16, const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
                   int Nq, int Nk, int d, float scale, int causal, int n_splits, void *workspace,
                   unsigned long long workspace_bytes, void *stream) {
    int rc = check_splitkv(q, k, v, out, lse, B, H, Nq, Nk, d, n_splits);
    if (rc != FA_OK) return rc;
    const int64_t rows = static_cast<int64_t>(B) * H * Nq;
    const size_t need = fa::splitkv_workspace_bytes(rows, d, n_splits);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return FA_ERR_WORKSPACE;
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
    a.o_part = static_cast<float *>(workspace);
    a.lse_part = reinterpret_cast<float *>(static_cast<char *>(workspace) + o_bytes);
    a.stream = static_cast<cudaStream_t>(stream);
    log_call("split-KV %s d=%d causal=%d B=%d H=%d Nq=%d Nk=%d splits=%d", fp16 ? "fp16" : "bf16", d, a.causal, B,
             H, Nq, Nk, n_splits);
    return fa::launch_splitkv(a, fp16);
}

int varlen_common(bool fp16, const void *q, const void *k, const void *v, void *out, float *lse,
                  const int *cu_seqlens, int nseq, int total, int max_seqlen, int H, int Hkv, int d, float scale,
                  int causal, void *stream) {
    if (!q || !k || !v || !out || !lse || !cu_seqlens) return FA_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
        !aligned(cu_seqlens, 4))
        return FA_ERR_ALIGN;
    if (nseq < 1 || total < 1 || max_seqlen < 1 || H < 1 || Hkv < 1 || H % Hkv != 0) return FA_ERR_SHAPE;
    const int64_t items = static_cast<int64_t>(nseq) * H * ((static_cast<int64_t>(max_seqlen) + 255) / 256);
    if (items > INT32_MAX) return FA_ERR_SHAPE;
    if (static_cast<int64_t>(H) * total > INT32_MAX) return FA_ERR_SHAPE;  // lse index
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    DeviceInfo *di = device_info();
    if (!di || !encoder()) return FA_ERR_LAUNCH;
    fa::LaunchArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.mask = nullptr;
    a.out = out;
    a.lse = lse;
    a.B = nseq;
    a.H = H;
    a.N = max_seqlen;
    a.d = d;
    a.Hkv = Hkv;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    a.stream = static_cast<cudaStream_t>(stream);
    a.status = di->status;
    a.num_sms = di->num_sms;
    a.timeout_ns = kDefaultTimeoutNs;
    a.cu_seqlens = cu_seqlens;
    a.total = total;
    log_call("packed forward %s d=%d causal=%d nseq=%d total=%d max_seqlen=%d H=%d Hkv=%d", fp16 ? "fp16" : "bf16",
             d, a.causal, nseq, total, max_seqlen, H, Hkv);
    return fp16 ? fa::launch_fwd_varlen_fp16(a) : fa::launch_fwd_varlen_bf16(a);
}

int bwd_common(bool fp16, const void *q, const void *k, const void *v, const void *out, const void *dout,
               const float *lse, void *dq, void *dk, void *dv, int B, int H, int N, int d, float scale, int causal,
               void *workspace, unsigned long long workspace_bytes, void *stream) {
    if (!q || !k || !v || !out || !dout || !lse || !dq || !dk || !dv) return FA_ERR_NULL;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(dout, 16) ||
        !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) || !aligned(lse, 4))
        return FA_ERR_ALIGN;
    if (B < 1 || H < 1 || N < 1) return FA_ERR_SHAPE;
    const int64_t bh = static_cast<int64_t>(B) * H;
    if (bh > INT32_MAX) return FA_ERR_SHAPE;
    const int64_t npad = fa::bwd_padded_rows(N);
    if (bh * (npad / fa::kBwdRows) > INT32_MAX) return FA_ERR_SHAPE;  // one CTA per (head, 128-key block)
    if (bh * npad > (int64_t(1) << 36)) return FA_ERR_SHAPE;           // row-statistics grid
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    const size_t need = fa::bwd_workspace_bytes(bh, N, d);
    if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return FA_ERR_WORKSPACE;
    DeviceInfo *di = device_info();
    if (!di || !encoder()) return FA_ERR_LAUNCH;
    fa::BwdArgs a;
    a.q = q;
    a.k = k;
    a.v = v;
    a.out = out;
    a.dout = dout;
    a.lse = lse;
    a.dq = dq;
    a.dk = dk;
    a.dv = dv;
    a.B = B;
    a.H = H;
    a.N = N;
    a.d = d;
    a.scale = scale;
    a.causal = causal ? 1 : 0;
    const size_t acc = static_cast<size_t>(bh) * static_cast<size_t>(N) * static_cast<size_t>(d) * sizeof(float);
    const size_t row = static_cast<size_t>(bh) * static_cast<size_t>(npad) * sizeof(float);
    char *ws = static_cast<char *>(workspace);
    a.dq_acc = reinterpret_cast<float *>(ws);
    a.lse2 = reinterpret_cast<float *>(ws + ((acc + 255) / 256) * 256);
    a.dsum = reinterpret_cast<float *>(ws + ((acc + 255) / 256) * 256 + ((row + 255) / 256) * 256);
    a.stream = static_cast<cudaStream_t>(stream);
    a.status = di->status;
    a.timeout_ns = kDefaultTimeoutNs;
    log_call("backward %s d=%d (%s kernel) causal=%d B=%d H=%d N=%d", fp16 ? "fp16" : "bf16", d,
             d == 64 ? "half-block" : "serial", a.causal, B, H, N);
    return fa::launch_bwd(a, fp16);
}

}  // namespace

namespace fa {
bool encode_rows_map(CUtensorMap *map, CUtensorMapDataType dtype, int elem_bytes, const void *base, int d, int N,
                     int BH, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * elem_bytes,
                             static_cast<cuuint64_t>(d) * elem_bytes * static_cast<cuuint64_t>(N)};
    // box: one 128-byte swizzle row of elements x box_rows rows x 1 head
    cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elem_bytes), static_cast<cuuint32_t>(box_rows), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, dtype, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Self-test of the bounded waits: one warp waits on an mbarrier that nothing
// ever completes, through the same wait routine every pipeline role uses. The
// wait gives up after p.timeout_ns, records FA_ERR_TIMEOUT in the device status
// word and returns; the kernel then exits normally.
__global__ void fa_selftest_wait_kernel(FwdParams p) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    wait_warp(smem_u32(&bar), 0, &abort_flag, p);
}

bool encode_tokens_map(CUtensorMap *map, CUtensorMapDataType dtype, int elem_bytes, const void *base, int d,
                       int heads, int total, int box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                          static_cast<cuuint64_t>(total)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * elem_bytes,
                             static_cast<cuuint64_t>(d) * elem_bytes * static_cast<cuuint64_t>(heads)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elem_bytes), 1, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, dtype, 3, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}
}  // namespace fa

extern "C" {

int fa_fwd(const void *q, const void *k, const void *v, const float *mask_or_null, void *out, float *lse, int B,
           int H, int N, int d, float scale, int causal, void *stream) {
    return fwd_common(Type::BF16, q, k, v, mask_or_null, out, lse, B, H, N, d, scale, causal, stream);
}

int fa_fwd_fp16(const void *q, const void *k, const void *v, const float *mask_or_null, void *out, float *lse,
                int B, int H, int N, int d, float scale, int causal, void *stream) {
    return fwd_common(Type::FP16, q, k, v, mask_or_null, out, lse, B, H, N, d, scale, causal, stream);
}

long long fa_fwd_masked_workspace_bytes(int B, int N) {
    if (B < 1 || N < 1) return FA_ERR_SHAPE;
    return static_cast<long long>(masked_workspace_bytes(B, N));
}

int fa_fwd_masked(const void *q, const void *k, const void *v, const float *mask, void *out, float *lse, int B, int H,
                  int Hkv, int N, int d, float scale, int causal, void *workspace, unsigned long long workspace_bytes,
                  void *stream) {
    return masked_common(Type::BF16, q, k, v, mask, out, lse, B, H, Hkv, N, d, scale, causal, workspace,
                         workspace_bytes, stream);
}

int fa_fwd_masked_fp16(const void *q, const void *k, const void *v, const float *mask, void *out, float *lse, int B,
                       int H, int Hkv, int N, int d, float scale, int causal, void *workspace,
                       unsigned long long workspace_bytes, void *stream) {
    return masked_common(Type::FP16, q, k, v, mask, out, lse, B, H, Hkv, N, d, scale, causal, workspace,
                         workspace_bytes, stream);
}

int fa_fwd_dropout(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H, int Hkv, int N,
                   int d, float scale, int causal, float p_drop, unsigned long long seed, unsigned long long offset,
                   void *stream) {
    return dropout_common(Type::BF16, q, k, v, out, lse, B, H, Hkv, N, d, scale, causal, p_drop, seed, offset,
                          stream);
}

int fa_fwd_dropout_fp16(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H, int Hkv,
                        int N, int d, float scale, int causal, float p_drop, unsigned long long seed,
                        unsigned long long offset, void *stream) {
    return dropout_common(Type::FP16, q, k, v, out, lse, B, H, Hkv, N, d, scale, causal, p_drop, seed, offset,
                          stream);
}

int fa_fwd_fp32(const void *q, const void *k, const void *v, const float *mask_or_null, void *out, float *lse,
                int B, int H, int N, int d, float scale, int causal, void *stream) {
    return fwd_common(Type::FP32, q, k, v, mask_or_null, out, lse, B, H, N, d, scale, causal, stream);
}

int fa_fwd_host(const void *q_host, const void *k_host, const void *v_host, void *out_host, float *lse_host,
                void *q_dev, void *k_dev, void *v_dev, void *out_dev, float *lse_dev, int B, int H, int N, int d,
                float scale, int causal, int n_chunks, void *stream) {
    return host_common(Type::BF16, q_host, k_host, v_host, out_host, lse_host, q_dev, k_dev, v_dev, out_dev, lse_dev,
                       B, H, N, d, scale, causal, n_chunks, stream);
}

int fa_fwd_host_fp16(const void *q_host, const void *k_host, const void *v_host, void *out_host, float *lse_host,
                     void *q_dev, void *k_dev, void *v_dev, void *out_dev, float *lse_dev, int B, int H, int N, int d,
                     float scale, int causal, int n_chunks, void *stream) {
    return host_common(Type::FP16, q_host, k_host, v_host, out_host, lse_host, q_dev, k_dev, v_dev, out_dev, lse_dev,
                       B, H, N, d, scale, causal, n_chunks, stream);
}

int fa_splitkv_num_splits(int B, int H, int Nq, int Nk, int d) {
    if (B < 1 || H < 1 || Nk < 1 || Nq < 1) return FA_ERR_SHAPE;
    DeviceInfo *di = device_info();
    const int64_t sms = di ? di->num_sms : 148;
    const int64_t bh = static_cast<int64_t>(B) * H;
    // Fill the GPU in exactly one wave: as many splits per head as there are
    // resident CTA slots per head (a partly filled second wave would cost
    // almost a whole extra wave of time).
    const int64_t slots = sms * fa::splitkv_blocks_per_sm(d == 64 ? 64 : 128, Nq);
    int64_t n = slots / bh;
    const int64_t max_by_len = (static_cast<int64_t>(Nk) + 63) / 64;  // at least ~64 keys per split
    if (n > max_by_len) n = max_by_len;
    if (n > 1024) n = 1024;
    return n < 1 ? 1 : static_cast<int>(n);
}

long long fa_splitkv_workspace_bytes(int B, int H, int Nq, int d, int n_splits) {
    if (B < 1 || H < 1 || Nq < 1 || n_splits < 1) return FA_ERR_SHAPE;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    return static_cast<long long>(
        fa::splitkv_workspace_bytes(static_cast<int64_t>(B) * H * Nq, d, n_splits));
}

int fa_fwd_splitkv(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H, int Nq,
                   int Nk, int d, float scale, int causal, int n_splits, void *workspace,
                   unsigned long long workspace_bytes, void *stream) {
    return splitkv_common(false, q, k, v, out, lse, B, H, Nq, Nk, d, scale, causal, n_splits, workspace,
                          workspace_bytes, stream);
}

int fa_fwd_splitkv_fp16(const void *q, const void *k, const void *v, void *out, float *lse, int B, int H,
                        int Nq, int Nk, int d, float scale, int causal, int n_splits, void *workspace,
                        unsigned long long workspace_bytes, void *stream) {
    return splitkv_common(true, q, k, v, out, lse, B, H, Nq, Nk, d, scale, causal, n_splits, workspace,
                          workspace_bytes, stream);
}

int fa_fwd_bias(const void *q, const void *k, const void *v, const float *bias, void *out, float *lse, int B, int H,
                int N, int d, float scale, int causal, void *stream) {
    if (!bias) return FA_ERR_NULL;
    return fwd_common(Type::BF16, q, k, v, bias, out, lse, B, H, N, d, scale, causal, stream, -1, 1);
}

int fa_fwd_bias_fp16(const void *q, const void *k, const void *v, const float *bias, void *out, float *lse, int B,
                     int H, int N, int d, float scale, int causal, void *stream) {
    if (!bias) return FA_ERR_NULL;
    return fwd_common(Type::FP16, q, k, v, bias, out, lse, B, H, N, d, scale, causal, stream, -1, 1);
}

int fa_fwd_gqa(const void *q, const void *k, const void *v, const float *mask_or_null, void *out, float *lse,
               int B, int H, int Hkv, int N, int d, float scale, int causal, void *stream) {
    if (Hkv < 1) return FA_ERR_SHAPE;
    return fwd_common(Type::BF16, q, k, v, mask_or_null, out, lse, B, H, N, d, scale, causal, stream, Hkv);
}

int fa_fwd_gqa_fp16(const void *q, const void *k, const void *v, const float *mask_or_null, void *out, float *lse,
                    int B, int H, int Hkv, int N, int d, float scale, int causal, void *stream) {
    if (Hkv < 1) return FA_ERR_SHAPE;
    return fwd_common(Type::FP16, q, k, v, mask_or_null, out, lse, B, H, N, d, scale, causal, stream, Hkv);
}

int fa_fwd_varlen(const void *q, const void *k, const void *v, void *out, float *lse, const int *cu_seqlens,
                  int nseq, int total, int max_seqlen, int H, int Hkv, int d, float scale, int causal, void *stream) {
    return varlen_common(false, q, k, v, out, lse, cu_seqlens, nseq, total, max_seqlen, H, Hkv, d, scale, causal,
                         stream);
}

int fa_fwd_varlen_fp16(const void *q, const void *k, const void *v, void *out, float *lse, const int *cu_seqlens,
                       int nseq, int total, int max_seqlen, int H, int Hkv, int d, float scale, int causal,
                       void *stream) {
    return varlen_common(true, q, k, v, out, lse, cu_seqlens, nseq, total, max_seqlen, H, Hkv, d, scale, causal,
                         stream);
}

long long fa_bwd_workspace_bytes(int B, int H, int N, int d) {
    if (B < 1 || H < 1 || N < 1) return FA_ERR_SHAPE;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
    return static_cast<long long>(fa::bwd_workspace_bytes(static_cast<int64_t>(B) * H, N, d));
}

int fa_bwd(const void *q, const void *k, const void *v, const void *out, const void *dout, const float *lse,
           void *dq, void *dk, void *dv, int B, int H, int N, int d, float scale, int causal, void *workspace,
           unsigned long long workspace_bytes, void *stream) {
    return bwd_common(false, q, k, v, out, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, workspace,
                      workspace_bytes, stream);
}

int fa_bwd_fp16(const void *q, const void *k, const void *v, const void *out, const void *dout, const float *lse,
                void *dq, void *dk, void *dv, int B, int H, int N, int d, float scale, int causal, void *workspace,
                unsigned long long workspace_bytes, void *stream) {
    return bwd_common(true, q, k, v, out, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, workspace,
                      workspace_bytes, stream);
}

int fa_selftest_wait_timeout(unsigned long long timeout_ns, void *stream) {
    if (timeout_ns == 0 || timeout_ns > 1000000000ull) return FA_ERR_SHAPE;
    DeviceInfo *di = device_info();
    if (!di) return FA_ERR_LAUNCH;
    fa::FwdParams p = {};
    p.status = di->status;
    p.timeout_ns = timeout_ns;
    fa::fa_selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(p);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

const char *fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "ok";
        case FA_ERR_NULL: return "a required pointer is NULL";
        case FA_ERR_ALIGN: return "a pointer is not aligned (16 bytes; 4 for lse)";
        case FA_ERR_SHAPE: return "bad shape: B, H, N must be >= 1 and B*H*ceil(N/256) must fit in int32";
        case FA_ERR_UNSUPPORTED: return "unsupported head dimension for this element type";
        case FA_ERR_LAUNCH: return "CUDA launch or tensor-map encoding failed";
        case FA_ERR_TIMEOUT: return "a device-side pipeline wait timed out";
        case FA_ERR_WORKSPACE: return "workspace missing or smaller than the problem needs";
        case FA_ERR_SEQLENS: return "cu_seqlens inconsistent with total or max_seqlen (device status)";
        case FA_ERR_ARG: return "an argument is outside its range (dropout: the drop probability keeps nothing)";
        default: return "unknown status";
    }
}

int fa_get_device_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_LAUNCH;
    int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_fa_status, sizeof(int)) != cudaSuccess) return FA_ERR_LAUNCH;
    if (cudaMemcpyToSymbol(g_fa_status, &zero, sizeof(int)) != cudaSuccess) return FA_ERR_LAUNCH;
    return v;
}

int fa_num_sms(void) {
    DeviceInfo *di = device_info();
    return di ? di->num_sms : FA_ERR_LAUNCH;
}

}  // extern "C"
