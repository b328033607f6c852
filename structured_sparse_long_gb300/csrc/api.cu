// api.cu -- the extern "C" boundary declared in include/pi_attn.h.
//
// Every entry point validates its arguments on the host before anything is
// launched, picks the kernel for the dtype and head size, and launches it on the
// caller's stream.  No entry point allocates device memory: the status word is
// a static __device__ variable, one per device.
#include <atomic>
#include <cstdint>
#include <cstring>

#include "pi_attn.h"
#include "pi_launch.h"

namespace {

__device__ int g_status_word;

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // bound on every device-side wait
constexpr int kMaxDevices = 64;
constexpr int kDebugMaxN = 2048;

// Device address of g_status_word for the current device, looked up once per device (two
// threads may both look it up the first time; they store the same address).
int *status_word() {
    static std::atomic<int *> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    int *p = cache[dev].load(std::memory_order_acquire);
    if (!p) {
        void *a = nullptr;
        if (cudaGetSymbolAddress(&a, g_status_word) != cudaSuccess) return nullptr;
        p = static_cast<int *>(a);
        cache[dev].store(p, std::memory_order_release);
    }
    return p;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int validate_shape(int B, int H, int Hkv, int N, int d, int k_local, int period, int S, int mode) {
    if (mode != PI_MODE_PI && mode != PI_MODE_ECP && mode != PI_MODE_PI_BIDIR) return PI_ERR_UNSUPPORTED;
    if (B <= 0 || H <= 0 || Hkv <= 0 || N <= 0) return PI_ERR_SHAPE;
    if (H % Hkv != 0) return PI_ERR_SHAPE;
    if (k_local < 0 || S < 0) return PI_ERR_SHAPE;
    if (mode != PI_MODE_ECP && S > 0 && period <= 0) return PI_ERR_SHAPE;
    if (mode == PI_MODE_ECP && (k_local <= 0 || S != 0)) return PI_ERR_SHAPE;
    if (d != 32 && d != 64 && d != 128) return PI_ERR_UNSUPPORTED;
    const long long rows = (long long)B * H * N;
    if (rows > 0x7fffffffLL) return PI_ERR_UNSUPPORTED;
    return PI_OK;
}

int validate_fwd(const void *q, const void *k, const void *v, const float *alpha, int B, int H,
                 int Hkv, int N, int d, int k_local, int period, int S, int mode, const void *out,
                 const float *lse) {
    if (!q || !k || !v || !out || !lse) return PI_ERR_NULL;
    if (mode != PI_MODE_ECP && !alpha) return PI_ERR_NULL;
    const int rc = validate_shape(B, H, Hkv, N, d, k_local, period, S, mode);
    if (rc != PI_OK) return rc;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16)) return PI_ERR_ALIGN;
    if (!aligned(lse, 4) || (alpha && !aligned(alpha, 4))) return PI_ERR_ALIGN;
    return PI_OK;
}

// Query rows of a sequence shard's call: nq rows whose first is the query at key position
// qoff.  A whole-sequence call has none (shard = false: the queries are the N key rows).
struct Window {
    bool shard;
    int nq, qoff;
};

// A sequence shard's window: inside the key rows, starting on a 128-row boundary, so that the
// kernels see the same query blocks as in a whole-sequence run over the key rows.
int validate_window(int N, Window w) {
    if (w.nq <= 0 || w.qoff < 0 || (long long)w.qoff + w.nq > (long long)N) return PI_ERR_SHAPE;
    if (w.qoff % 128 != 0) return PI_ERR_SHAPE;
    return PI_OK;
}

pi::Shape make_shape(int B, int H, int Hkv, int N, int d, int k_local, int period, int S, int mode,
                     Window w = Window{false, 0, 0}) {
    pi::Shape s;
    s.B = B; s.H = H; s.Hkv = Hkv; s.N = N; s.d = d;
    s.k_local = k_local; s.period = period; s.S = (mode != PI_MODE_ECP) ? S : 0; s.mode = mode;
    s.scale_log2 = (float)(1.4426950408889634 / __builtin_sqrt((double)d));
    s.nq = w.shard ? w.nq : N;
    s.qoff = w.shard ? w.qoff : 0;
    return s;
}

int map_cuda(cudaError_t e) { return e == cudaSuccess ? PI_OK : PI_ERR_CUDA; }

int run_fwd(const void *q, const void *k, const void *v, const float *alpha, int B, int H, int Hkv,
            int N, int d, int k_local, int period, int S, int mode, void *out, float *lse, void *stream,
            bool fp32, int dbg, int *cnt, long long *isum, const float *lse_in, float *P,
            Window w = Window{false, 0, 0}) {
    int rc = validate_fwd(q, k, v, alpha, B, H, Hkv, N, d, k_local, period, S, mode, out, lse);
    if (rc != PI_OK) return rc;
    if (w.shard && (rc = validate_window(N, w)) != PI_OK) return rc;
    int *status = status_word();
    if (!status) return PI_ERR_CUDA;
    pi::LaunchFwd L;
    L.q = q; L.k = k; L.v = v; L.alpha = (mode != PI_MODE_ECP) ? alpha : nullptr;
    L.out = out; L.lse = lse;
    L.s = make_shape(B, H, Hkv, N, d, k_local, period, S, mode, w);
    L.fp32 = fp32; L.dbg = dbg; L.cnt = cnt; L.isum = isum; L.lse_in = lse_in; L.P = P;
    L.trace = nullptr; L.n_trace = 0;
    L.status = status; L.timeout_ns = kWaitTimeoutNs;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!fp32 && d != 32) return map_cuda(pi::launch_fwd_tc(L, st));
    return map_cuda(pi::launch_fwd_simt(L, st));
}

int run_bwd(const void *q, const void *k, const void *v, const float *alpha, const void *out,
            const float *lse, const void *dout, int B, int H, int Hkv, int N, int d, int k_local,
            int period, int S, int mode, void *dq, void *dk, void *dv, float *dalpha, void *workspace,
            size_t workspace_bytes, void *stream, bool fp32, Window w = Window{false, 0, 0}) {
    if (!q || !k || !v || !out || !lse || !dout || !dq || !dk || !dv) return PI_ERR_NULL;
    if (mode != PI_MODE_ECP && !alpha) return PI_ERR_NULL;
    int rc = validate_shape(B, H, Hkv, N, d, k_local, period, S, mode);
    if (rc != PI_OK) return rc;
    if (w.shard && (rc = validate_window(N, w)) != PI_OK) return rc;
    const void *p16[] = {q, k, v, out, dout, dq, dk, dv};
    for (const void *p : p16)
        if (!aligned(p, 16)) return PI_ERR_ALIGN;
    if (!aligned(lse, 4) || (alpha && !aligned(alpha, 4)) || (dalpha && !aligned(dalpha, 4)))
        return PI_ERR_ALIGN;
    const size_t need = pi_attn_bwd_workspace_size(B, H, Hkv, w.shard ? w.nq : N, d);
    if (!workspace || workspace_bytes < need) return PI_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return PI_ERR_ALIGN;
    pi::LaunchBwd L;
    L.q = q; L.k = k; L.v = v; L.alpha = (mode != PI_MODE_ECP) ? alpha : nullptr;
    L.out = out; L.lse = lse; L.dout = dout; L.dq = dq; L.dk = dk; L.dv = dv; L.dalpha = dalpha;
    L.Dws = static_cast<float *>(workspace);
    L.s = make_shape(B, H, Hkv, N, d, k_local, period, S, mode, w);
    L.fp32 = fp32;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!fp32 && d != 32) {
        int *status = status_word();
        if (!status) return PI_ERR_CUDA;
        const cudaError_t e = pi::launch_bwd_dq_tc(L, status, kWaitTimeoutNs, st);
        if (e != cudaSuccess) return PI_ERR_CUDA;
        return map_cuda(pi::launch_bwd_dkdv_tc(L, status, kWaitTimeoutNs, st));
    }
    return map_cuda(pi::launch_bwd_simt(L, st));
}

}  // namespace

// Scratch of pi_attn_bwd_noalloc: one fp32 per query row, fixed size, shared by every call
// on a device.  In host code the name is only a host-side stand-in; kernels get the
// device address from noalloc_scratch().
static __device__ __align__(256) float g_noalloc_scratch[PI_ATTN_NOALLOC_MAX_ROWS];

namespace {

// Device address of g_noalloc_scratch for the current device, looked up once per device (two
// threads may both look it up the first time; they store the same address).
float *noalloc_scratch() {
    static std::atomic<float *> cache[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    float *p = cache[dev].load(std::memory_order_acquire);
    if (!p) {
        if (cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_noalloc_scratch) != cudaSuccess)
            return nullptr;
        cache[dev].store(p, std::memory_order_release);
    }
    return p;
}

}  // namespace

extern "C" {

int pi_attn_fwd(const void *q, const void *k, const void *v, const float *alpha, int B, int H, int Hkv,
                int N, int d, int k_local, int period, int S, int mode, void *out, float *lse,
                void *stream) {
    return run_fwd(q, k, v, alpha, B, H, Hkv, N, d, k_local, period, S, mode, out, lse, stream, false,
                   0, nullptr, nullptr, nullptr, nullptr);
}

int pi_attn_fwd_f32(const void *q, const void *k, const void *v, const float *alpha, int B, int H,
                    int Hkv, int N, int d, int k_local, int period, int S, int mode, void *out,
                    float *lse, void *stream) {
    return run_fwd(q, k, v, alpha, B, H, Hkv, N, d, k_local, period, S, mode, out, lse, stream, true,
                   0, nullptr, nullptr, nullptr, nullptr);
}

int pi_attn_fwd_gated(const void *q, const void *k, const void *v, const void *gate_w1,
                      const float *gate_b1, const float *gate_w2, const float *gate_b2, int B, int H,
                      int Hkv, int N, int d, int k_local, int period, int S, int mode, void *out,
                      float *lse, float *alpha_out, void *stream) {
    if (!gate_w1 || !gate_b1 || !gate_w2 || !gate_b2) return PI_ERR_NULL;
    // the gate is the pi mode's (causal or bidirectional); ECP has no prior to weight
    if (mode != PI_MODE_PI && mode != PI_MODE_PI_BIDIR) return PI_ERR_UNSUPPORTED;
    const int rc = validate_fwd(q, k, v, gate_b2, B, H, Hkv, N, d, k_local, period, S, mode, out, lse);
    if (rc != PI_OK) return rc;
    if (d != 64 && d != 128) return PI_ERR_UNSUPPORTED;  // the tensor-core forward only
    if (!aligned(gate_w1, 16) || !aligned(gate_b1, 4) || !aligned(gate_w2, 4) || !aligned(gate_b2, 4) ||
        (alpha_out && !aligned(alpha_out, 4)))
        return PI_ERR_ALIGN;
    int *status = status_word();
    if (!status) return PI_ERR_CUDA;
    pi::LaunchFwd L;
    L.q = q; L.k = k; L.v = v; L.alpha = nullptr;
    L.out = out; L.lse = lse;
    L.s = make_shape(B, H, Hkv, N, d, k_local, period, S, mode);
    L.fp32 = false; L.dbg = 0; L.cnt = nullptr; L.isum = nullptr; L.lse_in = nullptr; L.P = nullptr;
    L.trace = nullptr; L.n_trace = 0;
    L.status = status; L.timeout_ns = kWaitTimeoutNs;
    L.gate_w1 = gate_w1; L.gate_b1 = gate_b1; L.gate_w2 = gate_w2; L.gate_b2 = gate_b2; L.alpha_out = alpha_out;
    return map_cuda(pi::launch_fwd_tc(L, static_cast<cudaStream_t>(stream)));
}

size_t pi_attn_bwd_workspace_size(int B, int H, int Hkv, int N, int d) {
    (void)Hkv;
    (void)d;
    if (B <= 0 || H <= 0 || N <= 0) return 0;
    const size_t rows = (size_t)B * H * N;
    return ((rows * sizeof(float) + 255) / 256) * 256;
}

int pi_attn_bwd(const void *q, const void *k, const void *v, const float *alpha, const void *out,
                const float *lse, const void *dout, int B, int H, int Hkv, int N, int d, int k_local,
                int period, int S, int mode, void *dq, void *dk, void *dv, float *dalpha,
                void *workspace, size_t workspace_bytes, void *stream) {
    return run_bwd(q, k, v, alpha, out, lse, dout, B, H, Hkv, N, d, k_local, period, S, mode, dq, dk,
                   dv, dalpha, workspace, workspace_bytes, stream, false);
}

int pi_attn_bwd_f32(const void *q, const void *k, const void *v, const float *alpha, const void *out,
                    const float *lse, const void *dout, int B, int H, int Hkv, int N, int d,
                    int k_local, int period, int S, int mode, void *dq, void *dk, void *dv,
                    float *dalpha, void *workspace, size_t workspace_bytes, void *stream) {
    return run_bwd(q, k, v, alpha, out, lse, dout, B, H, Hkv, N, d, k_local, period, S, mode, dq, dk,
                   dv, dalpha, workspace, workspace_bytes, stream, true);
}

int pi_attn_fwd_shard(const void *q, const void *k, const void *v, const float *alpha, int B, int H,
                      int Hkv, int Nq, int Nkv, int q_offset, int d, int k_local, int period, int S,
                      int mode, void *out, float *lse, void *stream) {
    return run_fwd(q, k, v, alpha, B, H, Hkv, Nkv, d, k_local, period, S, mode, out, lse, stream, false,
                   0, nullptr, nullptr, nullptr, nullptr, Window{true, Nq, q_offset});
}

int pi_attn_bwd_shard(const void *q, const void *k, const void *v, const float *alpha, const void *out,
                      const float *lse, const void *dout, int B, int H, int Hkv, int Nq, int Nkv,
                      int q_offset, int d, int k_local, int period, int S, int mode, void *dq, void *dk,
                      void *dv, float *dalpha, void *workspace, size_t workspace_bytes, void *stream) {
    return run_bwd(q, k, v, alpha, out, lse, dout, B, H, Hkv, Nkv, d, k_local, period, S, mode, dq, dk,
                   dv, dalpha, workspace, workspace_bytes, stream, false, Window{true, Nq, q_offset});
}

int pi_attn_bwd_noalloc(const void *q, const void *k, const void *v, const float *alpha,
                        const void *out, const float *lse, const void *dout, int B, int H, int Hkv,
                        int N, int d, int k_local, int period, int S, int mode, void *dq, void *dk,
                        void *dv, float *dalpha, void *stream) {
    const int rc = validate_shape(B, H, Hkv, N, d, k_local, period, S, mode);
    if (rc != PI_OK) return rc;
    if ((long long)B * H * N > (long long)PI_ATTN_NOALLOC_MAX_ROWS) return PI_ERR_WORKSPACE;
    float *scratch = noalloc_scratch();
    if (!scratch) return PI_ERR_CUDA;
    return run_bwd(q, k, v, alpha, out, lse, dout, B, H, Hkv, N, d, k_local, period, S, mode, dq, dk,
                   dv, dalpha, scratch, sizeof(float) * (size_t)PI_ATTN_NOALLOC_MAX_ROWS, stream,
                   false);
}

int pi_attn_decode(const void *q, const void *k_cache, const void *v_cache, const float *alpha, int B,
                   int H, int Hkv, int N, int d, int k_local, int period, int S, int mode, void *out,
                   float *lse, void *stream) {
    if (!q || !k_cache || !v_cache || !out || !lse) return PI_ERR_NULL;
    if (mode != PI_MODE_ECP && !alpha) return PI_ERR_NULL;
    const int rc = validate_shape(B, H, Hkv, N, d, k_local, period, S, mode);
    if (rc != PI_OK) return rc;
    if (mode == PI_MODE_PI_BIDIR || (d != 64 && d != 128) || H / Hkv > 16) return PI_ERR_UNSUPPORTED;
    if ((long long)B * Hkv * N * d > (1LL << 62)) return PI_ERR_UNSUPPORTED;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
        return PI_ERR_ALIGN;
    if (!aligned(lse, 4) || (alpha && !aligned(alpha, 4))) return PI_ERR_ALIGN;
    int *status = status_word();
    if (!status) return PI_ERR_CUDA;
    pi::LaunchDecode L;
    L.q = q; L.k = k_cache; L.v = v_cache; L.alpha = (mode != PI_MODE_ECP) ? alpha : nullptr;
    L.out = out; L.lse = lse;
    L.s = make_shape(B, H, Hkv, N, d, k_local, period, S, mode);
    L.status = status; L.timeout_ns = kWaitTimeoutNs;
    return map_cuda(pi::launch_decode(L, static_cast<cudaStream_t>(stream)));
}

int pi_attn_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PI_ERR_CUDA;
    int *status = status_word();
    if (!status) return PI_ERR_CUDA;
    int value = 0;
    if (cudaMemcpy(&value, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return PI_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpy(status, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return PI_ERR_CUDA;
    return value;
}

const char *pi_attn_strerror(int code) {
    switch (code) {
        case PI_OK: return "PI_OK";
        case PI_ERR_NULL: return "PI_ERR_NULL: a required pointer is NULL";
        case PI_ERR_SHAPE: return "PI_ERR_SHAPE: inconsistent sizes or parameters";
        case PI_ERR_UNSUPPORTED: return "PI_ERR_UNSUPPORTED: unsupported head size, mode or size";
        case PI_ERR_ALIGN: return "PI_ERR_ALIGN: misaligned pointer";
        case PI_ERR_WORKSPACE: return "PI_ERR_WORKSPACE: workspace missing or too small";
        case PI_ERR_CUDA: return "PI_ERR_CUDA: CUDA runtime error";
        case PI_ERR_DEVICE_TIMEOUT: return "PI_ERR_DEVICE_TIMEOUT: a device-side wait gave up";
        default: return "unknown pi_attn status";
    }
}

int pi_attn_debug_counts(const void *q, const void *k, const void *v, const float *alpha, int B, int H,
                         int Hkv, int N, int d, int k_local, int period, int S, int mode, int dtype,
                         void *out, float *lse, int *count, long long *idx_sum, void *stream) {
    if (!count || !idx_sum) return PI_ERR_NULL;
    if (dtype != 0 && dtype != 1) return PI_ERR_UNSUPPORTED;
    if (!aligned(count, 4) || !aligned(idx_sum, 8)) return PI_ERR_ALIGN;
    return run_fwd(q, k, v, alpha, B, H, Hkv, N, d, k_local, period, S, mode, out, lse, stream,
                   dtype == 1, 1, count, idx_sum, nullptr, nullptr);
}

int pi_attn_debug_probs(const void *q, const void *k, const void *v, const float *alpha,
                        const float *lse_in, int B, int H, int Hkv, int N, int d, int k_local,
                        int period, int S, int mode, int dtype, void *out, float *lse, float *P,
                        void *stream) {
    if (!P || !lse_in) return PI_ERR_NULL;
    if (dtype != 0 && dtype != 1) return PI_ERR_UNSUPPORTED;
    if (N > kDebugMaxN) return PI_ERR_UNSUPPORTED;
    if (!aligned(P, 4) || !aligned(lse_in, 4)) return PI_ERR_ALIGN;
    return run_fwd(q, k, v, alpha, B, H, Hkv, N, d, k_local, period, S, mode, out, lse, stream,
                   dtype == 1, 2, nullptr, nullptr, lse_in, P);
}

int pi_attn_debug_trace(const void *q, const void *k, const void *v, const float *alpha, int B, int H,
                        int Hkv, int N, int d, int k_local, int period, int S, int mode, void *out,
                        float *lse, long long *trace, int n_trace_ctas, void *stream) {
    const int rc = validate_fwd(q, k, v, alpha, B, H, Hkv, N, d, k_local, period, S, mode, out, lse);
    if (rc != PI_OK) return rc;
    if (!trace) return PI_ERR_NULL;
    if (d != 64 && d != 128) return PI_ERR_UNSUPPORTED;
    if (n_trace_ctas < 0) return PI_ERR_SHAPE;
    if (!aligned(trace, 8)) return PI_ERR_ALIGN;
    int *status = status_word();
    if (!status) return PI_ERR_CUDA;
    pi::LaunchFwd L;
    L.q = q; L.k = k; L.v = v; L.alpha = (mode != PI_MODE_ECP) ? alpha : nullptr;
    L.out = out; L.lse = lse;
    L.s = make_shape(B, H, Hkv, N, d, k_local, period, S, mode);
    L.fp32 = false; L.dbg = 3; L.cnt = nullptr; L.isum = nullptr; L.lse_in = nullptr; L.P = nullptr;
    L.trace = trace; L.n_trace = n_trace_ctas;
    L.status = status; L.timeout_ns = kWaitTimeoutNs;
    return map_cuda(pi::launch_fwd_tc(L, static_cast<cudaStream_t>(stream)));
}

int pi_attn_debug_wait_timeout(int timeout_us, void *stream) {
    if (timeout_us <= 0) return PI_ERR_SHAPE;
    int *status = status_word();
    if (!status) return PI_ERR_CUDA;
    return map_cuda(pi::launch_wait_timeout_probe(status, (uint64_t)timeout_us * 1000ull,
                                                  static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
