// pi_launch.h -- host-side launch descriptors shared by the C ABI and the kernel files.
#pragma once

#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>

#include "pi_common.cuh"

namespace pi {

constexpr int kGateHidden = 8;  // hidden units per head of the fused gate

// A host-side set-up done once per device (devices 0-63; others redo it on every call).
// Thread-safe: two threads may both do the set-up the first time, which is harmless.
struct PerDeviceOnce {
    std::atomic<unsigned long long> done{0};
    bool needed(int dev) const {
        return dev < 0 || dev >= 64 || !((done.load(std::memory_order_acquire) >> dev) & 1ull);
    }
    void mark(int dev) {
        if (dev >= 0 && dev < 64) done.fetch_or(1ull << dev, std::memory_order_acq_rel);
    }
};

struct LaunchFwd {
    const void *q, *k, *v;
    const float *alpha;
    void *out;
    float *lse;
    Shape s;
    bool fp32;
    int dbg;               // 0 forward, 1 + counts, 2 + probability dump, 3 + timeline trace
    int *cnt;              // dbg 1
    long long *isum;       // dbg 1
    const float *lse_in;   // dbg 2
    float *P;              // dbg 2
    long long *trace;      // dbg 3: per-CTA clock64() stamps (tcgen05 kernel)
    int n_trace;           // dbg 3: number of traced CTAs
    int *status;           // device status word
    uint64_t timeout_ns;   // bound on every device-side wait
    // fused gate (tensor-core path): alpha from the per-head MLP of one hidden layer,
    // hid = max(0, W1_h q_i + b1_h), alpha = 1 / (1 + exp(-(w2_h . hid + b2_h))), computed in
    // the kernel instead of read from alpha; alpha_out (may be null) receives it
    const void *gate_w1 = nullptr;   // [H, kGateHidden, d] bf16
    const float *gate_b1 = nullptr;  // [H, kGateHidden]
    const float *gate_w2 = nullptr;  // [H, kGateHidden]
    const float *gate_b2 = nullptr;  // [H]
    float *alpha_out = nullptr;      // [B, H, N]
};

struct LaunchBwd {
    const void *q, *k, *v;
    const float *alpha;
    const void *out;
    const float *lse;
    const void *dout;
    void *dq, *dk, *dv;
    float *dalpha;
    float *Dws;
    Shape s;
    bool fp32;
};

struct LaunchDecode {
    const void *q, *k, *v;  // q [B,H,d]; k, v the cache [B,Hkv,N,d]
    const float *alpha;     // [B,H] or null (ECP)
    void *out;              // [B,H,d]
    float *lse;             // [B,H]
    Shape s;
    int *status;
    uint64_t timeout_ns;
};

// CUDA-core kernels (pi_simt.cu)
cudaError_t launch_fwd_simt(const LaunchFwd &L, cudaStream_t st);
cudaError_t launch_bwd_simt(const LaunchBwd &L, cudaStream_t st);
// key-major dk/dv pass alone; reads D_i from L.Dws (pi_simt.cu)
cudaError_t launch_bwd_dkdv_simt(const LaunchBwd &L, cudaStream_t st);

// tcgen05 backward, bf16, d in {64, 128} (pi_bwd_tc.cu): query-major pass writing dq,
// D_i (into L.Dws) and dalpha
cudaError_t launch_bwd_dq_tc(const LaunchBwd &L, int *status, uint64_t timeout_ns, cudaStream_t st);
// key-major pass writing dk and dv from D_i in L.Dws (pi_bwd_tc.cu)
cudaError_t launch_bwd_dkdv_tc(const LaunchBwd &L, int *status, uint64_t timeout_ns, cudaStream_t st);

// tcgen05 / TMEM / TMA forward, bf16, d in {64, 128} (pi_fwd_tc.cu).
// Returns cudaErrorNotSupported when the tensor-map encoder is unavailable.
cudaError_t launch_fwd_tc(const LaunchFwd &L, cudaStream_t st);

// decode step against a KV cache, bf16, d in {64, 128} (pi_decode.cu)
cudaError_t launch_decode(const LaunchDecode &L, cudaStream_t st);

// bounded-wait self test (pi_fwd_tc.cu)
cudaError_t launch_wait_timeout_probe(int *status, uint64_t timeout_ns, cudaStream_t st);

}  // namespace pi
