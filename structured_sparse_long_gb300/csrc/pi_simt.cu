// pi_simt.cu -- CUDA-core kernels: the fp32 forward, the d = 32 forward, and
// the backward (all dtypes).
//
// Forward (pi-Attention section 2.1-2.3; ECP section 2): one warp per query
// row.  Lane j of a 32-key chunk scores key j (full-length dot product against
// the query row staged in shared memory), the warp keeps one online-softmax
// state (running max via warp-shuffle max, running sum via shuffle sum), and
// every lane accumulates d/32 output columns.  Skip keys i - m*period form one
// more chunk with lane m-1 holding multiple m; their logits carry
// log2(1 - alpha) instead of log2(alpha).
//
// Backward (chain rule through the same definition):
//   D_i = sum_j p_ij (dout_i . v_j)   (= dout_i . out_i in exact arithmetic)
//   dz_ij = p_ij (dout_i . v_j - D_i),  p_ij = exp(z_ij - lse_i)
//   dq_i = sum_j dz_ij k_j / sqrt(d)            (query-major kernel)
//   dk_j = sum_{h in group} sum_i dz_ij q_i / sqrt(d),  dv_j = sum p_ij dout_i
//                                               (key-major kernel)
//   dalpha_i = -(sum_{j in P(i)} dz_ij) / (alpha_i (1 - alpha_i))
// Both kernels are deterministic (no atomics).
#include "pi_common.cuh"
#include "pi_launch.h"

namespace pi {
namespace simt {

constexpr int kWarps = 4;
constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, o));
    return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}
__device__ __forceinline__ long long warp_sum_ll(long long x) {
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
    return x;
}

// dot(row staged in shared memory as fp32, row in global memory of type T)
template <typename T, int D>
__device__ __forceinline__ float dot_row(const float *__restrict__ xs, const T *__restrict__ y) {
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < D; c += 8) {
        float t[8];
        load8(y + c, t);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(xs[c + e], t[e], acc);
    }
    return acc;
}

struct FwdArgs {
    const void *q, *k, *v;
    const float *alpha;
    void *out;
    float *lse;
    int *cnt;
    long long *isum;
    const float *lse_in;
    float *P;
};

// DBG: 0 = forward, 1 = forward + per-row counts, 2 = forward + dense P dump
template <typename T, int D, int DBG>
__global__ void __launch_bounds__(kWarps * 32) fwd_kernel(FwdArgs a, Shape s) {
    __shared__ __align__(16) float qs[kWarps][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long rows = (long long)s.B * s.H * s.nq;
    const long long row = (long long)blockIdx.x * kWarps + warp;
    if (row >= rows) return;  // uniform per warp
    const int i = s.qoff + (int)(row % s.nq);  // key position of the query
    const long long bh = row / s.nq;
    const int h = (int)(bh % s.H), b = (int)(bh / s.H);
    const int g = h / (s.H / s.Hkv);
    const T *qrow = static_cast<const T *>(a.q) + row * D;
    const long long kvoff = ((long long)b * s.Hkv + g) * s.N * D;
    const T *kb = static_cast<const T *>(a.k) + kvoff;
    const T *vb = static_cast<const T *>(a.v) + kvoff;
    for (int c = lane; c < D; c += 32) qs[warp][c] = to_f32(qrow[c]);
    __syncwarp();

    const float al = a.alpha ? a.alpha[row] : 1.f;
    const float off_b = (s.mode != kModeEcp) ? log2f(al) : 0.f;
    const float off_s = log2f(1.f - al);
    constexpr int RC = D / 32;
    float o[RC];
#pragma unroll
    for (int r = 0; r < RC; ++r) o[r] = 0.f;
    float m = -INFINITY, l = 0.f;
    long long cnt = 0, isum = 0;
    float lse2_in = 0.f;
    if (DBG == 2) lse2_in = a.lse_in[row] * kLog2e;

    auto chunk = [&](int j, bool valid, float off) {
        float z = -INFINITY;
        if (valid) z = fmaf(dot_row<T, D>(qs[warp], kb + (long long)j * D), s.scale_log2, off);
        if (DBG == 1 && valid) { cnt += 1; isum += j; }
        if (DBG == 2 && valid)
            a.P[row * s.N + j] = (lse2_in == -INFINITY) ? 0.f : exp2f(z - lse2_in);
        const float mn = fmaxf(m, warp_max(z));
        if (mn == -INFINITY) return;  // nothing finite yet (uniform)
        const float corr = exp2f(m - mn);
        const float p = exp2f(z - mn);
        l = l * corr + warp_sum(p);
#pragma unroll
        for (int r = 0; r < RC; ++r) o[r] *= corr;
        for (int c = 0; c < 32; ++c) {
            const float pc = __shfl_sync(kFull, p, c);
            const int jc = __shfl_sync(kFull, j, c);
            if (pc != 0.f) {  // same value in every lane
                const T *vr = vb + (long long)jc * D;
#pragma unroll
                for (int r = 0; r < RC; ++r) o[r] = fmaf(pc, to_f32(vr[lane + 32 * r]), o[r]);
            }
        }
        m = mn;
    };

    const int lo = band_lo(i, s.mode, s.k_local), hi = band_hi(i, s.N, s.mode, s.k_local);
    for (int j0 = lo; j0 <= hi; j0 += 32) {
        const int j = j0 + lane;
        chunk(j, j <= hi, off_b);
    }
    if (s.mode != kModeEcp) {
        for (int dir = -1; dir <= ((s.mode == kModeBidir) ? 1 : -1); dir += 2) {  // i - m pi, i + m pi
            for (int m0 = 1; m0 <= s.S; m0 += 32) {
                const int mm = m0 + lane;
                const long long off = (long long)mm * s.period;
                const long long jj = (long long)i + dir * off;
                const bool valid = mm <= s.S && off > s.k_local && jj >= 0 && jj < s.N;
                chunk(valid ? (int)jj : 0, valid, off_s);
            }
        }
    }

    T *orow = static_cast<T *>(a.out) + row * D;
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int r = 0; r < RC; ++r) orow[lane + 32 * r] = from_f32<T>(o[r] * inv);
    if (lane == 0) a.lse[row] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    if (DBG == 1) {
        cnt = warp_sum_ll(cnt);
        isum = warp_sum_ll(isum);
        if (lane == 0) {
            a.cnt[row] = (int)cnt;
            a.isum[row] = isum;
        }
    }
}

// ------------------------------------------------------------------ backward

struct BwdArgs {
    const void *q, *k, *v;
    const float *alpha;
    const void *out;
    const float *lse;
    const void *dout;
    void *dq, *dk, *dv;
    float *dalpha;
    float *Dws;  // [B*H*N]
};

// One warp per query row: D_i, dq and dalpha in one pass over the row's keys.
// D_i = sum_j p_ij dp_ij (equal to dout_i . out_i in exact arithmetic, but free of
// the rounding of the stored bf16 out, which 1/(alpha(1-alpha)) would amplify in
// dalpha); dq_i = tau (sum_j p dp k_j - D_i sum_j p k_j) = tau sum_j dz_ij k_j.
// D_i is written to the workspace for the key-major pass.
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_dq_kernel(BwdArgs a, Shape s) {
    __shared__ __align__(16) float qs[kWarps][D];
    __shared__ __align__(16) float gs[kWarps][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long rows = (long long)s.B * s.H * s.nq;
    const long long row = (long long)blockIdx.x * kWarps + warp;
    if (row >= rows) return;
    const int i = s.qoff + (int)(row % s.nq);  // key position of the query
    const long long bh = row / s.nq;
    const int h = (int)(bh % s.H), b = (int)(bh / s.H);
    const int g = h / (s.H / s.Hkv);
    const T *qrow = static_cast<const T *>(a.q) + row * D;
    const T *grow = static_cast<const T *>(a.dout) + row * D;
    const long long kvoff = ((long long)b * s.Hkv + g) * s.N * D;
    const T *kb = static_cast<const T *>(a.k) + kvoff;
    const T *vb = static_cast<const T *>(a.v) + kvoff;
    for (int c = lane; c < D; c += 32) {
        qs[warp][c] = to_f32(qrow[c]);
        gs[warp][c] = to_f32(grow[c]);
    }
    __syncwarp();
    const float al = a.alpha ? a.alpha[row] : 1.f;
    const float off_b = (s.mode != kModeEcp) ? log2f(al) : 0.f;
    const float off_s = log2f(1.f - al);
    const float lse2 = a.lse[row] * kLog2e;
    constexpr int RC = D / 32;
    float acc_pdk[RC], acc_pk[RC];
#pragma unroll
    for (int r = 0; r < RC; ++r) { acc_pdk[r] = 0.f; acc_pk[r] = 0.f; }
    float d_part = 0.f, skip_p = 0.f, skip_pdp = 0.f;
    bool any_skip = false;

    auto chunk = [&](int j, bool valid, float off, bool is_skip) {
        float p = 0.f, dp = 0.f;
        if (valid && lse2 != -INFINITY) {
            const float z = fmaf(dot_row<T, D>(qs[warp], kb + (long long)j * D), s.scale_log2, off);
            p = exp2f(z - lse2);
            dp = dot_row<T, D>(gs[warp], vb + (long long)j * D);
        }
        const float pdp = p * dp;
        d_part += pdp;
        if (is_skip) { skip_p += p; skip_pdp += pdp; }
        for (int c = 0; c < 32; ++c) {
            const float pc = __shfl_sync(kFull, p, c);
            const float pdc = __shfl_sync(kFull, pdp, c);
            const int jc = __shfl_sync(kFull, j, c);
            if (pc != 0.f) {
                const T *kr = kb + (long long)jc * D;
#pragma unroll
                for (int r = 0; r < RC; ++r) {
                    const float kv = to_f32(kr[lane + 32 * r]);
                    acc_pk[r] = fmaf(pc, kv, acc_pk[r]);
                    acc_pdk[r] = fmaf(pdc, kv, acc_pdk[r]);
                }
            }
        }
    };

    const int lo = band_lo(i, s.mode, s.k_local), hi = band_hi(i, s.N, s.mode, s.k_local);
    for (int j0 = lo; j0 <= hi; j0 += 32) {
        const int j = j0 + lane;
        chunk(j, j <= hi, off_b, false);
    }
    if (s.mode != kModeEcp) {
        for (int dir = -1; dir <= ((s.mode == kModeBidir) ? 1 : -1); dir += 2) {  // i - m pi, i + m pi
            for (int m0 = 1; m0 <= s.S; m0 += 32) {
                const int mm = m0 + lane;
                const long long back = (long long)mm * s.period;
                const long long jj = (long long)i + dir * back;
                const bool valid = mm <= s.S && back > s.k_local && jj >= 0 && jj < s.N;
                any_skip |= valid;
                chunk(valid ? (int)jj : 0, valid, off_s, true);
            }
        }
    }
    const float Drow = warp_sum(d_part);
    const float scale = s.scale_log2 / kLog2e;  // 1/sqrt(d)
    T *dqrow = static_cast<T *>(a.dq) + row * D;
#pragma unroll
    for (int r = 0; r < RC; ++r)
        dqrow[lane + 32 * r] = from_f32<T>((acc_pdk[r] - Drow * acc_pk[r]) * scale);
    const float sdz = warp_sum(skip_pdp) - Drow * warp_sum(skip_p);  // sum over P(i) of dz
    any_skip = __any_sync(kFull, any_skip);
    if (lane == 0) {
        a.Dws[row] = Drow;
        if (a.dalpha)
            a.dalpha[row] = (s.mode != kModeEcp && any_skip && al > 0.f && al < 1.f)
                                ? -sdz / (al * (1.f - al)) : 0.f;  // saturated gate: 0
    }
}

// one warp per key row (b, g, j): dk and dv, summed over the query heads of group g
template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32) bwd_dkdv_kernel(BwdArgs a, Shape s) {
    __shared__ __align__(16) float ks[kWarps][D];
    __shared__ __align__(16) float vs[kWarps][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long krows = (long long)s.B * s.Hkv * s.N;
    const long long krow = (long long)blockIdx.x * kWarps + warp;
    if (krow >= krows) return;
    const int j = (int)(krow % s.N);
    const long long bg = krow / s.N;
    const int g = (int)(bg % s.Hkv), b = (int)(bg / s.Hkv);
    const int G = s.H / s.Hkv;
    const T *krp = static_cast<const T *>(a.k) + krow * D;
    const T *vrp = static_cast<const T *>(a.v) + krow * D;
    for (int c = lane; c < D; c += 32) {
        ks[warp][c] = to_f32(krp[c]);
        vs[warp][c] = to_f32(vrp[c]);
    }
    __syncwarp();
    constexpr int RC = D / 32;
    float dk[RC], dv[RC];
#pragma unroll
    for (int r = 0; r < RC; ++r) { dk[r] = 0.f; dv[r] = 0.f; }

    for (int hh = 0; hh < G; ++hh) {
        const int h = g * G + hh;
        // the query at key position i is row i - qoff of the plane; only positions inside the
        // query window [wlo, whi] are visited
        const long long rbase = ((long long)b * s.H + h) * s.nq;
        const T *qb = static_cast<const T *>(a.q) + rbase * D;
        const T *gb = static_cast<const T *>(a.dout) + rbase * D;
        const int wlo = s.qoff, whi = s.qoff + s.nq - 1;

        auto chunk = [&](int i, bool valid, bool is_skip) {
            float p = 0.f, dz = 0.f;
            if (valid) {
                const long long row = rbase + (i - s.qoff);
                const float lse2 = a.lse[row] * kLog2e;
                if (lse2 != -INFINITY) {
                    const float al = a.alpha ? a.alpha[row] : 1.f;
                    const float off = (s.mode != kModeEcp) ? (is_skip ? log2f(1.f - al) : log2f(al)) : 0.f;
                    const float z = fmaf(dot_row<T, D>(ks[warp], qb + (long long)(i - s.qoff) * D), s.scale_log2, off);
                    p = exp2f(z - lse2);
                    const float dp = dot_row<T, D>(vs[warp], gb + (long long)(i - s.qoff) * D);
                    dz = p * (dp - a.Dws[row]);
                }
            }
            for (int c = 0; c < 32; ++c) {
                const float pc = __shfl_sync(kFull, p, c);
                const float dzc = __shfl_sync(kFull, dz, c);
                const int ic = __shfl_sync(kFull, i, c);
                if (pc != 0.f || dzc != 0.f) {
                    const T *qr = qb + (long long)(ic - s.qoff) * D;
                    const T *gr = gb + (long long)(ic - s.qoff) * D;
#pragma unroll
                    for (int r = 0; r < RC; ++r) {
                        dv[r] = fmaf(pc, to_f32(gr[lane + 32 * r]), dv[r]);
                        dk[r] = fmaf(dzc, to_f32(qr[lane + 32 * r]), dk[r]);
                    }
                }
            }
        };

        const int ifirst = max(band_first_query(j, s.mode, s.k_local), wlo);
        const int ilast = min(band_last_query(j, s.N, s.mode, s.k_local), whi);
        for (int i0 = ifirst; i0 <= ilast; i0 += 32) {
            const int i = i0 + lane;
            chunk(i, i <= ilast, false);
        }
        if (s.mode != kModeEcp) {
            // queries j + m pi (whose skip key i - m pi is j) and, bidirectionally, j - m pi
            for (int dir = 1; dir >= ((s.mode == kModeBidir) ? -1 : 1); dir -= 2) {
                for (int m0 = 1; m0 <= s.S; m0 += 32) {
                    const int mm = m0 + lane;
                    const long long back = (long long)mm * s.period;
                    const long long ii = (long long)j + dir * back;
                    const bool valid = mm <= s.S && back > s.k_local && ii >= wlo && ii <= whi;
                    chunk(valid ? (int)ii : wlo, valid, true);
                }
            }
        }
    }
    const float scale = s.scale_log2 / kLog2e;
    T *dkr = static_cast<T *>(a.dk) + krow * D;
    T *dvr = static_cast<T *>(a.dv) + krow * D;
#pragma unroll
    for (int r = 0; r < RC; ++r) {
        dkr[lane + 32 * r] = from_f32<T>(dk[r] * scale);
        dvr[lane + 32 * r] = from_f32<T>(dv[r]);
    }
}

// ------------------------------------------------------------------ launchers

template <typename T, int D>
static cudaError_t fwd_dispatch_dbg(const FwdArgs &a, const Shape &s, int dbg, cudaStream_t st) {
    const long long rows = (long long)s.B * s.H * s.nq;
    const dim3 grid((unsigned)((rows + kWarps - 1) / kWarps));
    if (dbg == 0) fwd_kernel<T, D, 0><<<grid, kWarps * 32, 0, st>>>(a, s);
    else if (dbg == 1) fwd_kernel<T, D, 1><<<grid, kWarps * 32, 0, st>>>(a, s);
    else fwd_kernel<T, D, 2><<<grid, kWarps * 32, 0, st>>>(a, s);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t fwd_dispatch(const FwdArgs &a, const Shape &s, int dbg, cudaStream_t st) {
    switch (s.d) {
        case 32: return fwd_dispatch_dbg<T, 32>(a, s, dbg, st);
        case 64: return fwd_dispatch_dbg<T, 64>(a, s, dbg, st);
        case 128: return fwd_dispatch_dbg<T, 128>(a, s, dbg, st);
        default: return cudaErrorInvalidValue;
    }
}

template <typename T, int D>
static cudaError_t bwd_run(const BwdArgs &a, const Shape &s, cudaStream_t st) {
    const long long rows = (long long)s.B * s.H * s.nq;
    const long long krows = (long long)s.B * s.Hkv * s.N;
    const dim3 g1((unsigned)((rows + kWarps - 1) / kWarps));
    const dim3 g2((unsigned)((krows + kWarps - 1) / kWarps));
    bwd_dq_kernel<T, D><<<g1, kWarps * 32, 0, st>>>(a, s);
    bwd_dkdv_kernel<T, D><<<g2, kWarps * 32, 0, st>>>(a, s);
    return cudaGetLastError();
}

template <typename T, int D>
static cudaError_t dkdv_run(const BwdArgs &a, const Shape &s, cudaStream_t st) {
    const long long krows = (long long)s.B * s.Hkv * s.N;
    const dim3 g2((unsigned)((krows + kWarps - 1) / kWarps));
    bwd_dkdv_kernel<T, D><<<g2, kWarps * 32, 0, st>>>(a, s);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t bwd_dispatch(const BwdArgs &a, const Shape &s, cudaStream_t st) {
    switch (s.d) {
        case 32: return bwd_run<T, 32>(a, s, st);
        case 64: return bwd_run<T, 64>(a, s, st);
        case 128: return bwd_run<T, 128>(a, s, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace simt

cudaError_t launch_fwd_simt(const LaunchFwd &L, cudaStream_t st) {
    simt::FwdArgs a{L.q, L.k, L.v, L.alpha, L.out, L.lse, L.cnt, L.isum, L.lse_in, L.P};
    if (L.fp32) return simt::fwd_dispatch<float>(a, L.s, L.dbg, st);
    return simt::fwd_dispatch<__nv_bfloat16>(a, L.s, L.dbg, st);
}

cudaError_t launch_bwd_dkdv_simt(const LaunchBwd &L, cudaStream_t st) {
    simt::BwdArgs a{L.q, L.k, L.v, L.alpha, L.out, L.lse, L.dout, L.dq, L.dk, L.dv, L.dalpha,
                    L.Dws};
    if (L.fp32) return cudaErrorInvalidValue;
    switch (L.s.d) {
        case 32: return simt::dkdv_run<__nv_bfloat16, 32>(a, L.s, st);
        case 64: return simt::dkdv_run<__nv_bfloat16, 64>(a, L.s, st);
        case 128: return simt::dkdv_run<__nv_bfloat16, 128>(a, L.s, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_bwd_simt(const LaunchBwd &L, cudaStream_t st) {
    simt::BwdArgs a{L.q, L.k, L.v, L.alpha, L.out, L.lse, L.dout, L.dq, L.dk, L.dv, L.dalpha,
                    L.Dws};
    if (L.fp32) return simt::bwd_dispatch<float>(a, L.s, st);
    return simt::bwd_dispatch<__nv_bfloat16>(a, L.s, st);
}

}  // namespace pi
