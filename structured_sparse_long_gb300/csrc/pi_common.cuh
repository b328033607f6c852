// pi_common.cuh -- definitions shared by every kernel of the library.
//
// The neighbour set of a query row (the only place the kernels decide which
// keys a row attends to):
//   pi mode  ("pi-Attention: Periodic Sparse Transformers for Efficient
//            Long-Context Modeling", section 2.1 and 2.2):
//            band  [max(0, i - k_local), i]
//            skip  i - m*period for m = 1..S when m*period > k_local and >= 0
//   bidirectional pi mode (same page, 2.1 and 2.2 in their general form):
//            band  [max(0, i - k_local), min(N - 1, i + k_local)]
//            skip  i -/+ m*period for m = 1..S when m*period > k_local, inside [0, N)
//   ECP mode ("Efficient Context Propagating Perceiver Architectures...",
//            section 2, PAR block): [max(0, (floor(i/c) - 1) * c), i], c = k_local
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace pi {

constexpr int kStatusOk = 0;
constexpr int kStatusTimeout = -7;

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Problem description passed by value to every kernel.
struct Shape {
    int B, H, Hkv, N, d;
    int k_local;       // band width k (pi) or half-segment length c (ECP)
    int period;        // skip stride (pi mode)
    int S;             // skip multiples (pi mode)
    int mode;          // 0 = pi (causal), 1 = ECP, 2 = pi (bidirectional)
    float scale_log2;  // log2(e) / sqrt(d): raw score -> log2-domain logit
    // Query rows.  Row r of a (b, h) plane of q, out, lse, alpha (and of their gradients) is
    // the query at key position qoff + r, for r < nq; N counts the key/value rows.  A whole
    // sequence has nq = N and qoff = 0; a sequence shard has its queries [t0, t1) against a
    // local key window that starts qoff = t0 - (window start) rows before them.
    int nq, qoff;
};

constexpr int kModeEcp = 1;
constexpr int kModeBidir = 2;

// First band key of query i.
__host__ __device__ __forceinline__ int band_lo(int i, int mode, int k_local) {
    int lo;
    if (mode != kModeEcp) {
        lo = i - k_local;
    } else {
        lo = (i / k_local - 1) * k_local;
    }
    return lo < 0 ? 0 : lo;
}

// Last band key of query i.
__host__ __device__ __forceinline__ int band_hi(int i, int N, int mode, int k_local) {
    if (mode != kModeBidir) return i;
    const long long hi = (long long)i + k_local;
    return hi > N - 1 ? N - 1 : (int)hi;
}

// First query position whose band contains key j (for key-major passes): the band of i reaches
// back to i - k, or (ECP) to the previous half-segment's start, which is never after j for i >= j.
__host__ __device__ __forceinline__ int band_first_query(int j, int mode, int k_local) {
    if (mode != kModeBidir) return j;
    return j - k_local < 0 ? 0 : j - k_local;
}

// Last query position whose band contains key j (for key-major passes).
__host__ __device__ __forceinline__ int band_last_query(int j, int N, int mode, int k_local) {
    long long hi;
    if (mode != kModeEcp) {
        hi = (long long)j + k_local;
    } else {
        hi = ((long long)(j / k_local) + 2) * k_local - 1;
    }
    return hi > N - 1 ? N - 1 : (int)hi;
}

// Smallest skip multiple m with m*period > k_local, at most S + 1 (no skip key at all then);
// computed in 64 bits, as k_local may be as large as INT_MAX.
__host__ __device__ __forceinline__ int first_skip_multiple(const Shape &s) {
    if (s.period <= 0) return 1;
    const long long m = (long long)s.k_local / s.period + 1;
    return (int)(m < (long long)s.S + 1 ? m : (long long)s.S + 1);
}

// Skip multiple m contributes a key distinct from the band iff m*period > k_local.
__host__ __device__ __forceinline__ bool skip_in_use(int m, int period, int k_local) {
    return (long long)m * period > (long long)k_local;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// First failure wins; later ones do not overwrite it.
__device__ __forceinline__ void record_status(int *status, int code) {
    if (status) atomicCAS(status, kStatusOk, code);
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Load 8 consecutive elements (16 B for bf16, 32 B for fp32) as fp32.
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float *o) {
    uint4 u = *reinterpret_cast<const uint4 *>(p);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        o[2 * t] = __uint_as_float(w[t] << 16);
        o[2 * t + 1] = __uint_as_float(w[t] & 0xffff0000u);
    }
}
__device__ __forceinline__ void load8(const float *p, float *o) {
    float4 a = *reinterpret_cast<const float4 *>(p);
    float4 b = *reinterpret_cast<const float4 *>(p + 4);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

}  // namespace pi
