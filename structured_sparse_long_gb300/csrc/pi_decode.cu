// pi_decode.cu -- one decode step of pi-Attention / ECP attention against a KV cache.
//
// What it computes: row i = N-1 of the forward ("pi-Attention: Periodic Sparse Transformers for
// Efficient Long-Context Modeling", section 2.1-2.3, causal form; ECP page, section 2), for a
// new query per (batch entry, head) whose key/value rows 0 .. N-1 -- its own included -- are in
// the cache: one softmax over the band rows lo .. N-1 and the skip rows N-1 - m*period, with
// log2(alpha) on band logits and log2(1 - alpha) on skip logits.
//
// How (HBM-bound gather, no dense contraction):
//   * The key list of row N-1 is the band (one contiguous run of cache rows) followed by the
//     skip rows; it is cut into 32-key chunks.  A cluster of P CTAs serves one (batch entry,
//     KV head); CTA r takes chunks r, r+P, ...  so that small batches still fill the GPU.
//   * Thread 0 stages each chunk's K and V rows in shared memory with bulk copies
//     (cp.async.bulk, one per contiguous band run and one per skip row) into a two-stage ring
//     completed by an mbarrier.
//   * Groups of at most 4 query heads (KSG > 0): warp w takes keys 8w .. 8w+7 of each chunk for
//     every head of the group, so that each K and V row is unpacked once for all of them.
//     Lanes split d for the dot products (conflict-free 256-byte row reads); one butterfly
//     reduce-scatter of the 8 x KSG partial scores leaves lane t with key t & 7 of head
//     (t & (8 KSG - 1)) >> 3; each lane keeps its head's online softmax state and every lane
//     the output slice of every head.  The four warps' states are merged in the CTA first.
//   * Larger groups: warp w handles the query heads w, w+4, ... for all 32 keys of a chunk,
//     with one reduce-scatter per head (lane t: key t).
//   * The P partial states (m, l, o) of head hh are merged by CTA hh % P of the cluster through
//     distributed shared memory (vector loads, all issued before use), which writes out (bf16)
//     and lse.
//   * Every mbarrier wait is bounded; a CTA that gives up still takes part in both cluster
//     barriers, so its cluster never waits forever.
#include <cuda.h>

#include "pi_common.cuh"
#include "pi_launch.h"
#include "pi_tc_ptx.cuh"

namespace pi {
namespace dec {

using tc::mbar_init;
using tc::mbar_expect_tx;
using tc::wait_bar;
using tc::WaitCtx;

constexpr int WARPS = 4;
constexpr int THREADS = WARPS * 32;
constexpr int KEYS = 32;     // keys per chunk: one lane per key
constexpr int NST = 2;       // chunk stages in the shared-memory ring (3 or 4 ran 32 and 33 us at D4)
constexpr int MAX_P = 8;     // CTAs per cluster (portable limit)
constexpr int MAX_G = 16;    // query heads per KV head
constexpr unsigned kFull = 0xffffffffu;

struct DecArgs {
    const __nv_bfloat16 *q, *k, *v;  // q [B,H,d]; k, v [B,Hkv,N,d]
    const float *alpha;              // [B,H] or null (ECP)
    __nv_bfloat16 *out;              // [B,H,d]
    float *lse;                      // [B,H]
    Shape s;                         // N is the cache length; the query sits at position N-1
    int lo, n_band, n_keys, m_first, n_chunks;
    int *status;
    uint64_t timeout_ns;
};

template <int D>
struct Lay {
    static constexpr int ROW = D * 2;                       // bytes of one bf16 row
    static constexpr int STAGE = 2 * KEYS * ROW;            // K then V rows of one chunk
    static constexpr int PART_OFF = NST * STAGE;            // partial states after the ring
    static constexpr int PART = (D + 4) * 4;                // o[D], m, l of one head (fp32), 16-B rows
    static constexpr int BAR_OFF = PART_OFF + MAX_G * PART; // full[NST], abort flag
    static constexpr int BYTES = BAR_OFF + 8 * NST + 16;
};

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t local_addr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
    return remote;
}
// Loads from another CTA's shared memory.  Volatile, so they stay after the cluster barrier and
// in program order, but without a memory clobber, so a run of them is issued back to back.
__device__ __forceinline__ void ld_dsmem2(uint32_t remote, float &x, float &y) {
    asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(x), "=f"(y) : "r"(remote));
}
template <int E>
__device__ __forceinline__ void ld_dsmem_vec(uint32_t remote, float *f) {
    if (E == 4)
        asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(f[0]), "=f"(f[1]), "=f"(f[2]), "=f"(f[3]) : "r"(remote));
    else
        ld_dsmem2(remote, f[0], f[1]);
}

// E consecutive bf16 of a shared-memory row (E = 2 or 4: one 4- or 8-byte load) as fp32.
template <int E>
__device__ __forceinline__ void lds_bf16(const uint8_t *p, float *f) {
    if (E == 4) {
        const uint2 u = *reinterpret_cast<const uint2 *>(p);
        f[0] = __uint_as_float(u.x << 16);
        f[1] = __uint_as_float(u.x & 0xffff0000u);
        f[2] = __uint_as_float(u.y << 16);
        f[3] = __uint_as_float(u.y & 0xffff0000u);
    } else {
        const uint32_t u = *reinterpret_cast<const uint32_t *>(p);
        f[0] = __uint_as_float(u << 16);
        f[1] = __uint_as_float(u & 0xffff0000u);
    }
}

// KSG > 0: every warp takes all heads (KSG, a power of two, at least G) for 8 keys of each chunk.
// KSG = 0: HPW query heads per warp, ceil(G / 4) rounded up to 1, 2 or 4, for all 32 keys.
// (Registers scale with the heads a warp holds.)
template <int D, int HPW, int KSG>
__global__ void __launch_bounds__(THREADS) decode_kernel(const DecArgs a) {
    using L = Lay<D>;
    constexpr int E = D / 32;  // columns per lane
    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t sbase = tc::smem_u32(smem);
    const uint32_t bar0 = sbase + L::BAR_OFF;
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + L::BAR_OFF + 8 * NST);
    float *part = reinterpret_cast<float *>(smem + L::PART_OFF);

    const Shape &s = a.s;
    const int P = gridDim.x;
    const int r = (int)cluster_rank();
    const int g = blockIdx.y, b = blockIdx.z;
    const int G = s.H / s.Hkv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const WaitCtx wc{abort_flag, a.status, a.timeout_ns};
    const size_t plane = ((size_t)b * s.Hkv + g) * (size_t)s.N * D;
    const __nv_bfloat16 *kp = a.k + plane, *vp = a.v + plane;
    const int n_local = (a.n_chunks > r) ? (a.n_chunks - r + P - 1) / P : 0;

    if (threadIdx.x == 0) {
        for (int x = 0; x < NST; ++x) mbar_init(bar0 + 8 * x, 1);
        *abort_flag = 0u;
        tc::fence_barrier_init();
    }
    __syncthreads();

    // key list position t -> cache row
    auto key_row = [&](int t) -> int {
        return t < a.n_band ? a.lo + t : (s.N - 1) - (a.m_first + t - a.n_band) * s.period;
    };
    // chunk c of this CTA (global chunk r + c*P) into ring stage c % NST (thread 0 only)
    int issued = 0;
    auto issue = [&](int c) {
        issued = c + 1;
        const int qc = r + c * P, st = c % NST;
        const int t0 = qc * KEYS, t1 = min(t0 + KEYS, a.n_keys);
        const uint32_t sk = sbase + st * L::STAGE, sv = sk + KEYS * L::ROW;
        const uint32_t bar = bar0 + 8 * st;
        mbar_expect_tx(bar, (uint32_t)(t1 - t0) * 2u * L::ROW);
        const int tb = min(t1, a.n_band);
        if (t0 < tb) {  // band rows: one contiguous run
            const size_t row0 = (size_t)(a.lo + t0) * D;
            const uint32_t bytes = (uint32_t)(tb - t0) * L::ROW;
            bulk_g2s(sk, kp + row0, bytes, bar);
            bulk_g2s(sv, vp + row0, bytes, bar);
        }
        for (int t = max(t0, a.n_band); t < t1; ++t) {  // skip rows, one by one
            const size_t row = (size_t)key_row(t) * D;
            bulk_g2s(sk + (t - t0) * L::ROW, kp + row, L::ROW, bar);
            bulk_g2s(sv + (t - t0) * L::ROW, vp + row, L::ROW, bar);
        }
    };
    if (threadIdx.x == 0) {
        for (int c = 0; c < min(NST, n_local); ++c) issue(c);
    }

    // ---- per-warp heads: query slice, prior, online state
    constexpr int NH = KSG > 0 ? KSG : HPW;  // heads whose query slice the warp holds
    float qv[NH][E], o[NH][E], m[NH], l[NH], offb[NH], offs[NH];
#pragma unroll
    for (int j = 0; j < NH; ++j) {
        const int hh = KSG > 0 ? j : warp + WARPS * j;
        m[j] = -INFINITY;
        l[j] = 0.f;
        offb[j] = 0.f;
        offs[j] = -INFINITY;
#pragma unroll
        for (int e = 0; e < E; ++e) { qv[j][e] = 0.f; o[j][e] = 0.f; }
        if (hh < G) {
            const int h = g * G + hh;
            const __nv_bfloat16 *qr = a.q + ((size_t)b * s.H + h) * D + lane * E;
#pragma unroll
            for (int e = 0; e < E; ++e) qv[j][e] = __bfloat162float(qr[e]) * s.scale_log2;
            if (a.alpha) {
                const float al = a.alpha[(size_t)b * s.H + h];
                offb[j] = log2f(al);
                offs[j] = log2f(1.f - al);
            }
        }
    }

    bool ok = true;
    for (int c = 0; c < n_local; ++c) {
        const int st = c % NST;
        ok = wait_bar(bar0 + 8 * st, (c / NST) & 1, wc);
        ok = __syncthreads_and(ok);
        if (!ok) break;
        const int t0 = (r + c * P) * KEYS;
        const int nk = min(KEYS, a.n_keys - t0);
        const uint8_t *sk = smem + st * L::STAGE, *sv = sk + KEYS * L::ROW;
        if constexpr (KSG > 0) {
            // keys 8 warp + [0, 8) of the chunk, every head: V partial scores per lane
            constexpr int V = 8 * KSG;
            float pd[V];
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int t = 8 * warp + kk;
                float kf[E];
                if (t < nk) {
                    lds_bf16<E>(sk + t * L::ROW + lane * E * 2, kf);
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) kf[e] = 0.f;
                }
#pragma unroll
                for (int h = 0; h < KSG; ++h) {
                    float acc = 0.f;
#pragma unroll
                    for (int e = 0; e < E; ++e) acc = fmaf(qv[h][e], kf[e], acc);
                    pd[h * 8 + kk] = acc;
                }
            }
            // reduce-scatter over the low lane bits (value index h * 8 + kk = lane & (V - 1)),
            // then the sum over the others
#pragma unroll
            for (int w = V / 2; w >= 1; w >>= 1) {
                const bool up = (lane & w) != 0;
#pragma unroll
                for (int i = 0; i < w; ++i) {
                    const float send = up ? pd[i] : pd[i + w];
                    const float keep = up ? pd[i + w] : pd[i];
                    pd[i] = keep + __shfl_xor_sync(kFull, send, w);
                }
            }
#pragma unroll
            for (int w = V; w < 32; w <<= 1) pd[0] += __shfl_xor_sync(kFull, pd[0], w);
            // this lane: key kl of the warp's 8, head hl; the 8 lanes of a head share its state
            const int hl = (lane & (V - 1)) >> 3, tk = 8 * warp + (lane & 7);
            float ob = offb[0], os = offs[0];
#pragma unroll
            for (int h = 1; h < KSG; ++h)
                if (hl == h) {
                    ob = offb[h];
                    os = offs[h];
                }
            const float z = (tk < nk && hl < G) ? pd[0] + ((t0 + tk < a.n_band) ? ob : os) : -INFINITY;
            float mx = z;
#pragma unroll
            for (int w = 4; w; w >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, w));
            const float mn = fmaxf(m[0], mx);
            const float corr = (mn == -INFINITY) ? 1.f : exp2f(m[0] - mn);
            const float p = (z == -INFINITY) ? 0.f : exp2f(z - mn);
            float ps = p;
#pragma unroll
            for (int w = 4; w; w >>= 1) ps += __shfl_xor_sync(kFull, ps, w);
            l[0] = l[0] * corr + ps;
            m[0] = mn;
#pragma unroll
            for (int h = 0; h < KSG; ++h) {
                const float ch = __shfl_sync(kFull, corr, h * 8);
#pragma unroll
                for (int e = 0; e < E; ++e) o[h][e] *= ch;
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int t = 8 * warp + kk;
                if (t >= nk) break;  // uniform per warp
                float vf[E];
                lds_bf16<E>(sv + t * L::ROW + lane * E * 2, vf);
#pragma unroll
                for (int h = 0; h < KSG; ++h) {
                    const float ph = __shfl_sync(kFull, p, h * 8 + kk);
#pragma unroll
                    for (int e = 0; e < E; ++e) o[h][e] = fmaf(ph, vf[e], o[h][e]);
                }
            }
        } else {
        const bool band_key = t0 + lane < a.n_band;
#pragma unroll
        for (int j = 0; j < HPW; ++j) {
            if (warp + WARPS * j >= G) break;  // uniform per warp
            // partial dot products of the 32 keys over this lane's columns
            float pd[KEYS];
#pragma unroll
            for (int t = 0; t < KEYS; ++t) {
                float acc = 0.f;
                if (t < nk) {
                    float kf[E];
                    lds_bf16<E>(sk + t * L::ROW + lane * E * 2, kf);
#pragma unroll
                    for (int e = 0; e < E; ++e) acc = fmaf(qv[j][e], kf[e], acc);
                }
                pd[t] = acc;
            }
            // butterfly reduce-scatter: lane t ends with the full score of key t
#pragma unroll
            for (int w = 16; w >= 1; w >>= 1) {
                const bool up = (lane & w) != 0;
#pragma unroll
                for (int i = 0; i < w; ++i) {
                    const float send = up ? pd[i] : pd[i + w];
                    const float keep = up ? pd[i + w] : pd[i];
                    pd[i] = keep + __shfl_xor_sync(kFull, send, w);
                }
            }
            const float z = (lane < nk) ? pd[0] + (band_key ? offb[j] : offs[j]) : -INFINITY;
            float mx = z;
#pragma unroll
            for (int w = 16; w; w >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, w));
            const float mn = fmaxf(m[j], mx);
            if (mn == -INFINITY) continue;  // nothing finite yet (uniform)
            const float corr = exp2f(m[j] - mn);
            const float p = exp2f(z - mn);
            float ps = p;
#pragma unroll
            for (int w = 16; w; w >>= 1) ps += __shfl_xor_sync(kFull, ps, w);
            l[j] = l[j] * corr + ps;
#pragma unroll
            for (int e = 0; e < E; ++e) o[j][e] *= corr;
            for (int t = 0; t < nk; ++t) {
                const float pt = __shfl_sync(kFull, p, t);
                float vf[E];
                lds_bf16<E>(sv + t * L::ROW + lane * E * 2, vf);
#pragma unroll
                for (int e = 0; e < E; ++e) o[j][e] = fmaf(pt, vf[e], o[j][e]);
            }
            m[j] = mn;
        }
        }
        __syncthreads();  // stage st is free again
        if (threadIdx.x == 0 && c + NST < n_local) issue(c + NST);
    }
    if (!ok && threadIdx.x == 0) {  // let copies in flight (the last NST issued) land first
        volatile uint32_t zero = 0;
        WaitCtx w2{&zero, nullptr, 20000000ull};
        for (int c = max(0, issued - NST); c < issued; ++c) wait_bar(bar0 + 8 * (c % NST), (c / NST) & 1, w2);
    }

    // ---- partial states to shared memory (per head: o[D], m, l), merged across the cluster
    if constexpr (KSG > 0) {
        // the warps' states first, [warp][head] over the same space (4 x KSG <= 16 heads' room),
        // then warp h merges head h's four into slot h, which only it reads
#pragma unroll
        for (int h = 0; h < KSG; ++h) {
            if (h >= G) break;
            float *ps = part + (warp * KSG + h) * (D + 4);
#pragma unroll
            for (int e = 0; e < E; ++e) ps[lane * E + e] = ok ? o[h][e] : 0.f;
            if (lane == h * 8) {  // a lane of head h
                ps[D] = ok ? m[0] : -INFINITY;
                ps[D + 1] = ok ? l[0] : 0.f;
            }
        }
        __syncthreads();
        if (warp < G) {
            const int h = warp;
            float mw[WARPS], lw[WARPS], ow[WARPS][E];
#pragma unroll
            for (int w = 0; w < WARPS; ++w) {
                const float *ps = part + (w * KSG + h) * (D + 4);
                mw[w] = ps[D];
                lw[w] = ps[D + 1];
#pragma unroll
                for (int e = 0; e < E; ++e) ow[w][e] = ps[lane * E + e];
            }
            __syncwarp();
            float mt = -INFINITY;
#pragma unroll
            for (int w = 0; w < WARPS; ++w) mt = fmaxf(mt, mw[w]);
            float lt = 0.f, ot[E];
#pragma unroll
            for (int e = 0; e < E; ++e) ot[e] = 0.f;
            if (mt != -INFINITY) {
#pragma unroll
                for (int w = 0; w < WARPS; ++w) {
                    if (mw[w] == -INFINITY) continue;
                    const float f = exp2f(mw[w] - mt);
                    lt = fmaf(f, lw[w], lt);
#pragma unroll
                    for (int e = 0; e < E; ++e) ot[e] = fmaf(f, ow[w][e], ot[e]);
                }
            }
            float *ps = part + h * (D + 4);
#pragma unroll
            for (int e = 0; e < E; ++e) ps[lane * E + e] = ot[e];
            if (lane == 0) {
                ps[D] = mt;
                ps[D + 1] = lt;
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < HPW; ++j) {
            const int hh = warp + WARPS * j;
            if (hh >= G) break;
            float *ps = part + hh * (D + 4);
            if (lane == 0) {
                ps[D] = ok ? m[j] : -INFINITY;
                ps[D + 1] = ok ? l[j] : 0.f;
            }
#pragma unroll
            for (int e = 0; e < E; ++e) ps[lane * E + e] = ok ? o[j][e] : 0.f;
        }
    }
    cluster_sync();
    // head hh is merged by CTA hh % P of the cluster, its warps taking those heads in turn; all
    // P partial states of a head are loaded before any is used
    for (int hh = r + P * warp; hh < G; hh += P * WARPS) {
        const uint32_t pa = sbase + L::PART_OFF + hh * (D + 4) * 4;
        float mr[MAX_P], lr[MAX_P], orr[MAX_P][E];
#pragma unroll
        for (int x = 0; x < MAX_P; ++x) {
            if (x < P) {
                ld_dsmem2(dsmem_addr(pa + D * 4, x), mr[x], lr[x]);
                ld_dsmem_vec<E>(dsmem_addr(pa + lane * E * 4, x), orr[x]);
            }
        }
        float mt = -INFINITY;
#pragma unroll
        for (int x = 0; x < MAX_P; ++x)
            if (x < P) mt = fmaxf(mt, mr[x]);
        float lt = 0.f, ot[E];
#pragma unroll
        for (int e = 0; e < E; ++e) ot[e] = 0.f;
        if (mt != -INFINITY) {
#pragma unroll
            for (int x = 0; x < MAX_P; ++x) {
                if (x >= P || mr[x] == -INFINITY) continue;
                const float f = exp2f(mr[x] - mt);
                lt = fmaf(f, lr[x], lt);
#pragma unroll
                for (int e = 0; e < E; ++e) ot[e] = fmaf(f, orr[x][e], ot[e]);
            }
        }
        {
            const int h = g * G + hh;
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
            __nv_bfloat16 *orow = a.out + ((size_t)b * s.H + h) * D + lane * E;
#pragma unroll
            for (int e = 0; e < E; ++e) orow[e] = __float2bfloat16_rn(ot[e] * inv);
            if (lane == 0) a.lse[(size_t)b * s.H + h] = lt > 0.f ? (mt + log2f(lt)) * kLn2 : -INFINITY;
        }
    }
    cluster_sync();  // every CTA's shared memory stays alive until the others have read it
}

template <int D, int HPW, int KSG>
static cudaError_t launch(const DecArgs &a, int P, cudaStream_t st) {
    static PerDeviceOnce configured;  // shared memory above the 48 KB default
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured.needed(dev)) {
        const cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, HPW, KSG>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, Lay<D>::BYTES);
        if (e != cudaSuccess) return e;
        configured.mark(dev);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)P, (unsigned)a.s.Hkv, (unsigned)a.s.B);
    cfg.blockDim = dim3(THREADS, 1, 1);
    cfg.dynamicSmemBytes = Lay<D>::BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)P;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_kernel<D, HPW, KSG>, a);
}

}  // namespace dec

cudaError_t launch_decode(const LaunchDecode &L, cudaStream_t st) {
    using namespace dec;
    const Shape &s = L.s;
    const int G = s.H / s.Hkv;
    if (G > MAX_G || s.Hkv > 65535 || s.B > 65535) return cudaErrorInvalidConfiguration;
    DecArgs a{};
    a.q = static_cast<const __nv_bfloat16 *>(L.q);
    a.k = static_cast<const __nv_bfloat16 *>(L.k);
    a.v = static_cast<const __nv_bfloat16 *>(L.v);
    a.alpha = L.alpha;
    a.out = static_cast<__nv_bfloat16 *>(L.out);
    a.lse = L.lse;
    a.s = s;
    a.status = L.status;
    a.timeout_ns = L.timeout_ns;
    // the key list of row N-1: band lo .. N-1, then skips N-1 - m*period with m*period > k
    const int i = s.N - 1;
    a.lo = band_lo(i, s.mode, s.k_local);
    a.n_band = i - a.lo + 1;
    a.m_first = 1;
    int n_skip = 0;
    if (s.mode != kModeEcp && s.S > 0) {
        a.m_first = first_skip_multiple(s);
        const int m_last = min(s.S, i / s.period);
        n_skip = max(0, m_last - a.m_first + 1);
    }
    a.n_keys = a.n_band + n_skip;
    a.n_chunks = (a.n_keys + KEYS - 1) / KEYS;
    // cluster size: enough CTAs for about two per SM, at most one chunk each, at most 8 (on D4,
    // 64 sequences x 4 KV heads: 1, 2, 3 and 8 CTAs per cluster ran 31, 25, 29 and 42 us)
    static int sms = 0;
    if (sms == 0) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
            sms = 1;
    }
    const long long pairs = (long long)s.B * s.Hkv;
    int P = (int)std::min<long long>(MAX_P, std::max<long long>(1, (2LL * sms + pairs - 1) / pairs));
    P = std::max(1, std::min(P, a.n_chunks));
    // groups of up to 4 heads: key-split warps (KSG = G rounded up to a power of two); larger
    // groups: ceil(G / 4) heads per warp
    const int hpw = (G + WARPS - 1) / WARPS;
    if (s.d == 64) {
        if (G <= 1) return launch<64, 1, 1>(a, P, st);
        if (G <= 2) return launch<64, 2, 2>(a, P, st);
        if (G <= 4) return launch<64, 4, 4>(a, P, st);
        if (hpw <= 2) return launch<64, 2, 0>(a, P, st);
        return launch<64, 4, 0>(a, P, st);
    }
    if (s.d == 128) {
        if (G <= 1) return launch<128, 1, 1>(a, P, st);
        if (G <= 2) return launch<128, 2, 2>(a, P, st);
        if (G <= 4) return launch<128, 4, 4>(a, P, st);
        if (hpw <= 2) return launch<128, 2, 0>(a, P, st);
        return launch<128, 4, 0>(a, P, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pi
