// pi_fwd_tc.cu -- fused pi-Attention / ECP forward on sm_103a tensor cores.
//
// What it computes ("pi-Attention: Periodic Sparse Transformers for Efficient
// Long-Context Modeling", section 2.1-2.3; ECP page section 2; GQA from the
// GSS-Transformer hybrid page): for each query row i, one softmax over the
// causal band [lo(i), i] and the skip keys i - m*period (pi mode), with
// log2(alpha) added to band logits and log2(1 - alpha) to skip logits, and the
// softmax-weighted sum of value rows.
//
// How (one CTA = 128 query rows = the M of every MMA):
//   * GQA packing: the 128 rows are GP query heads of one KV group x R = 128/GP
//     consecutive positions, so every K/V tile staged in shared memory serves
//     all GP heads at once.
//   * Keys are walked in 32-key chunks (one TMA box each).  A chunk is either a
//     band chunk (keys lo(p0) + 32c ...) or a skip chunk: the keys i - m*period
//     of the block's rows form R consecutive keys, so one skip block is R/32
//     chunks; each row attends to exactly one column of it (the "diagonal").
//     A key tile is one chunk at d = 128 and two at d = 64 (Tiling<D>).
//   * Warp 0 (lane 0) streams Q and K tiles with TMA, warp 2 (lane 0) streams V
//     tiles; warp 1 issues S = Q K^T into one of the 128 columns of TMEM S
//     buffers (four of 32 or two of 64) and warp 3 issues O += P V with P read
//     from TMEM (each whole warp runs its loop, one elected lane issues the MMAs
//     and commits).
//   * Warps 4-7 run the softmax, one thread per row (TMEM lane = row): masks,
//     adds the prior, keeps the running max m and sum l (rescaling O in TMEM
//     only when the max grows by more than 2^8), writes P as bf16 over its S,
//     and finally normalises O, stages it in shared memory and TMA-stores it.
//   * Every wait is bounded; a wait that runs out sets the device status word
//     and the CTA unwinds without hanging.
#include <cuda.h>

#include "pi_common.cuh"
#include "pi_launch.h"
#include "pi_tc_ptx.cuh"

namespace pi {
namespace tc {

constexpr int BM = 128;           // rows per CTA (MMA M)
constexpr int CHUNK = 32;         // keys per chunk (TMA box rows)
// Chunks per key tile (the N of the S products is 32 * CPT) and S buffers, NB x TILE_N = 128
// TMEM columns.  At d = 128 the S products of 32-key tiles cost the pipe its per-instruction
// minimum, but four buffers keep S of tile t+4 from waiting on more than PV of tile t; at d = 64
// the eight S products of a 64-key tile take no longer than those of a 32-key tile, and two
// buffers suffice.
template <int D>
struct Tiling {
    static constexpr int CPT = (D == 64) ? 2 : 1;
    static constexpr int TILE_N = CPT * CHUNK;
    static constexpr int NB = 4 / CPT;
};
constexpr int NUM_THREADS = 256;
constexpr int TMEM_COLS = 256;    // S buffers [0,128), O [128, 128+d)
constexpr int O_COL = 128;
constexpr int ROW_BYTES = 128;    // one 64-element bf16 swizzle row
constexpr int BOX_BYTES = CHUNK * ROW_BYTES;  // one 64 x 32 TMA box
constexpr float kRescaleThreshold = 8.f;      // log2 units

template <int D>
struct Cfg {
    static constexpr int CPT = Tiling<D>::CPT, TILE_N = Tiling<D>::TILE_N, NB = Tiling<D>::NB;
    static constexpr int KD = D / 64;  // 64-element column blocks of d
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int KV_STAGE = TILE_N * D * 2;
    // 48 KB of K tiles (the S issuer runs furthest ahead) and 32 KB of V tiles
    static constexpr int KSTAGES = 49152 / KV_STAGE;
    static constexpr int VSTAGES = 32768 / KV_STAGE;
    static constexpr int KV_DBLK = TILE_N * ROW_BYTES;  // one 64-column block of a stage
    static constexpr int Q_DBLK = BM * ROW_BYTES;
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + Q_BYTES;
    static constexpr int V_OFF = K_OFF + KSTAGES * KV_STAGE;
    static constexpr int DATA_BYTES = V_OFF + VSTAGES * KV_STAGE;  // from a 1024-byte aligned base
    // barrier indices
    static constexpr int B_Q = 0;
    static constexpr int B_KF = 1;
    static constexpr int B_KE = B_KF + KSTAGES;
    static constexpr int B_VF = B_KE + KSTAGES;
    static constexpr int B_VE = B_VF + VSTAGES;
    static constexpr int B_SF = B_VE + VSTAGES;  // S of tile t in TMEM buffer t % NB
    static constexpr int B_PR = B_SF + NB;      // P of the tile written over its S
    // PV of tile T completes barrier B_PV + T % NB, phase T / NB: a buffer's PV barrier is
    // waited for in order, so no parity wait has two of its phases outstanding.
    static constexpr int B_PV = B_PR + NB;
    static constexpr int B_OF = B_PV + NB;  // O complete (after the last PV), single phase
    static constexpr int B_DR = B_OF + 1;  // drain of the S issuer's MMAs
    static constexpr int B_DR2 = B_DR + 1; // drain of the PV issuer's MMAs
    static constexpr int NBARS = B_DR2 + 1;
    static constexpr int BAR_BYTES = NBARS * 8 + 16;  // + TMEM address and abort flag
    static_assert(BAR_BYTES <= 512, "barriers must fit the alignment gap or its complement");
    // The data starts at the first 1024-byte boundary of the dynamic shared memory; the
    // barriers go into the gap before it when it is large enough, else after the data.
    // Either way DATA_BYTES + 1024 bytes suffice.
    static constexpr int SMEM_BYTES = DATA_BYTES + 1024;
};

// Phase 1 of a key chunk for one row: mask the scores outside [clo, chi] and return the
// chunk's largest logit in log2 units (prior included).  A skip chunk holds at most one
// valid column per row (its diagonal), read with a select tree instead of a full pass.
__device__ __forceinline__ float chunk_max(float *f, int clo, int chi, bool skip, float sc, float off) {
    if (skip) {
        if (clo > chi) return -INFINITY;
        return fmaf(select32(f, clo), sc, off);
    }
    if (!__all_sync(0xffffffffu, clo <= 0 && chi >= 31)) {
#pragma unroll
        for (int c = 0; c < 32; ++c) f[c] = (c >= clo && c <= chi) ? f[c] : -INFINITY;
    }
    // four independent partial maxima: a short dependency chain
    float m0 = max3(f[0], f[1], f[2]), m1 = max3(f[3], f[4], f[5]);
    float m2 = max3(f[6], f[7], f[8]), m3 = max3(f[9], f[10], f[11]);
#pragma unroll
    for (int c = 12; c < 32; c += 8) {
        m0 = max3(m0, f[c], f[c + 1]);
        m1 = max3(m1, f[c + 2], f[c + 3]);
        m2 = max3(m2, f[c + 4], f[c + 5]);
        m3 = max3(m3, f[c + 6], f[c + 7]);
    }
    const float mx = fmaxf(max3(m0, m1, m2), m3);
    return (mx == -INFINITY) ? -INFINITY : fmaf(mx, sc, off);
}

// Phase 2: P = exp2(logit - mu) packed as 16 bf16 pairs; returns the chunk's sum of P.
// For a skip chunk `zdiag` is the diagonal logit from phase 1 and column clo the only
// non-zero entry.
__device__ __forceinline__ float chunk_exp(const float *f, int clo, bool skip, float zdiag, float sc,
                                           float off, float mu, uint32_t *pk) {
    if (skip) {
        const float p = fast_exp2(zdiag - mu);
        __nv_bfloat16 hb = __float2bfloat16_rn(p);
        const uint32_t bits = (uint32_t)(*reinterpret_cast<uint16_t *>(&hb));
        const uint32_t word = (clo & 1) ? (bits << 16) : bits;
#pragma unroll
        for (int w = 0; w < 16; ++w) pk[w] = (w == (clo >> 1)) ? word : 0u;
        return p;
    }
    const float bo = off - mu;
    const uint64_t sc2 = pack2(sc, sc), bo2 = pack2(bo, bo);
    uint64_t acc0 = pack2(0.f, 0.f), acc1 = pack2(0.f, 0.f);  // two independent sums
#pragma unroll
    for (int c = 0; c < 32; c += 2) {
        float z0, z1;
        unpack2(fma2(pack2(f[c], f[c + 1]), sc2, bo2), z0, z1);
        const float p0 = fast_exp2(z0);
        const float p1 = fast_exp2(z1);
        if ((c >> 1) & 1) acc1 = add2(acc1, pack2(p0, p1));
        else acc0 = add2(acc0, pack2(p0, p1));
        pk[c / 2] = pack_bf16(p0, p1);
    }
    float a0, a1, b0, b1;
    unpack2(acc0, a0, a1);
    unpack2(acc1, b0, b1);
    return (a0 + a1) + (b0 + b1);
}

// Fast path of a key tile that lies inside the band of every row: P = exp2(f * sc + bo) for
// the tile's NCH x 32 scores, packed as bf16 pairs in place (word c/2 of each chunk, written
// after scores c and c+1 were read); returns the sum of the fp32 values.
template <int NCH>
__device__ __forceinline__ float exp_pack(uint32_t *ra, uint32_t *rb, float sc, float bo) {
    const uint64_t sc2 = pack2(sc, sc), bo2 = pack2(bo, bo);
    uint64_t acc[4] = {pack2(0.f, 0.f), pack2(0.f, 0.f), pack2(0.f, 0.f), pack2(0.f, 0.f)};
#pragma unroll
    for (int h = 0; h < NCH; ++h) {
        uint32_t *r = h ? rb : ra;
#pragma unroll
        for (int c = 0; c < CHUNK; c += 2) {
            float z0, z1;
            unpack2(fma2(pack2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])), sc2, bo2), z0, z1);
            const float p0 = fast_exp2(z0), p1 = fast_exp2(z1);
            acc[2 * h + ((c >> 1) & 1)] = add2(acc[2 * h + ((c >> 1) & 1)], pack2(p0, p1));
            r[c / 2] = pack_bf16(p0, p1);
        }
    }
    float a[8];
    unpack2(acc[0], a[0], a[1]);
    unpack2(acc[1], a[2], a[3]);
    unpack2(acc[2], a[4], a[5]);
    unpack2(acc[3], a[6], a[7]);
    return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
}

// Largest of the NCH x 32 raw scores of a tile (four independent chains per chunk).
template <int NCH>
__device__ __forceinline__ float max_tile(const uint32_t *ra, const uint32_t *rb) {
    float m[8];
#pragma unroll
    for (int h = 0; h < NCH; ++h) {
        const uint32_t *r = h ? rb : ra;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            m[4 * h + k] = max3(__uint_as_float(r[k]), __uint_as_float(r[k + 4]), __uint_as_float(r[k + 8]));
#pragma unroll
        for (int c = 12; c < CHUNK; c += 8) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                m[4 * h + k] = max3(m[4 * h + k], __uint_as_float(r[c + k]), __uint_as_float(r[c + 4 + k]));
        }
    }
    float mx = fmaxf(max3(m[0], m[1], m[2]), m[3]);
    if (NCH == 2) mx = fmaxf(mx, fmaxf(max3(m[4], m[5], m[6]), m[7]));
    return mx;
}

// ------------------------------------------------------------------ kernel

struct TcArgs {
    const float *alpha;
    float *lse;
    Shape s;
    int GP;       // query heads packed per CTA
    int m_first;  // smallest skip multiple m with m * period > k_local
    int *status;
    uint64_t timeout_ns;
    int *cnt;
    long long *isum;
    const float *lse_in;
    float *P;
    long long *trace;  // DBG 3: clock64() stamps, kTraceSlots per traced CTA
    int n_trace;       // DBG 3: CTAs 0 .. n_trace-1 are traced
    const float *gate_w;  // fused gate (or null): alpha = 1 / (1 + exp(-(q_i . gate_w[h] + gate_b[h])))
    const float *gate_b;
    float *alpha_out;     // [B, H, N] the gate's alpha (may be null)
};

// Trace layout (DBG 3), slots per CTA: 0 entry, 1 set-up done, 2 Q issued, 3 Q landed (MMA
// side), 4 O complete (softmax side), 5 output stored, 6 exit, 7 tile count; then per tile t
// (t < 16): 8+t K issued, 24+t V issued, 40+t S issued, 56+t PV issued, 72+t S seen by the
// softmax, 88+t P ready; and cycles spent waiting, each measured within one thread:
// 104+t S issuer on K, 120+t S issuer on the S buffer (PV of t-2), 136+t PV issuer on P,
// 152+t PV issuer on V, 168+t softmax on S; softmax (warp 4) stamps inside tile t: 184+t S
// loaded from TMEM, 200+t maxima done (full tiles: exponentials done), 216+t P written to
// TMEM (issued); 232 the SM the CTA ran on, 233 and 234 the global timer (ns) at
// entry and exit.  Absolute stamps of different warps need not share a clock; the waits are
// exact.
constexpr int kTraceSlots = 240;
constexpr int kTraceTiles = 16;

// Key chunk ci of the block: first key position, whether it is a skip chunk,
// its skip distance m*period and sub-block index u.
// Skip blocks come after the band: first the n_back blocks of keys i - m*period, then (in the
// bidirectional mode) those of keys i + m*period, both for m = m_first, m_first + 1, ...;
// `back` is the signed distance i - key.
struct ChunkWalk {
    int lo0, n_band, m_first, cpb, cpb_log2, p0, period, n_back;
    __device__ __forceinline__ int key0(int ci, int &back, int &u, bool &skip) const {
        if (ci < n_band) {
            back = 0; u = 0; skip = false;
            return lo0 + ci * CHUNK;
        }
        const int sc = ci - n_band;  // cpb = R / 32 is 1, 2 or 4
        const int blk = sc >> cpb_log2;
        u = sc & (cpb - 1);
        back = (blk < n_back) ? (m_first + blk) * period : -(m_first + blk - n_back) * period;
        skip = true;
        return p0 - back + u * CHUNK;
    }
};

template <int D, int DBG>
__global__ void __launch_bounds__(NUM_THREADS, 2)
fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
              const TcArgs args) {
    using C = Cfg<D>;
    constexpr int KST = C::KSTAGES, VST = C::VSTAGES;
    constexpr int CPT = C::CPT, TILE_N = C::TILE_N, NB = C::NB;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_addr + pad;
    const uint32_t bar_off = (pad >= (uint32_t)C::BAR_BYTES) ? 0u : pad + C::DATA_BYTES;
    const uint32_t sQ = sbase + C::Q_OFF, sK = sbase + C::K_OFF, sV = sbase + C::V_OFF;
    const uint32_t sBar = raw_addr + bar_off;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem_raw + bar_off + C::NBARS * 8);
    uint32_t *tmem_slot = misc;
    volatile uint32_t *abort_flag = misc + 1;
    auto bar = [&](int idx) -> uint32_t { return sBar + idx * 8; };

    const Shape &s = args.s;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const WaitCtx wc{abort_flag, args.status, args.timeout_ns};
    // grid (position block, head group, batch entry): positions fastest, as CTAs are launched
    const long long lin = blockIdx.x + (long long)gridDim.x * (blockIdx.y + (long long)gridDim.y * blockIdx.z);
    const bool traced = DBG == 3 && lin < args.n_trace;
    auto stamp = [&](int slot) {
        if (traced) args.trace[lin * kTraceSlots + slot] = (long long)clock64();
    };
    auto stamp_tile = [&](int base, int t) {
        if (t < kTraceTiles) stamp(base + t);
    };
    // bounded wait that also records how long it took (DBG 3)
    auto timed_wait = [&](uint32_t b, uint32_t parity, int slot_base, int t) -> bool {
        const long long c0 = (DBG == 3) ? (long long)clock64() : 0;
        const bool r = wait_bar(b, parity, wc);
        if (traced && t < kTraceTiles && lane == 0)
            args.trace[lin * kTraceSlots + slot_base + t] = (long long)clock64() - c0;
        return r;
    };
    if (threadIdx.x == 0 && traced) {
        stamp(0);
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        args.trace[lin * kTraceSlots + 232] = smid;
        args.trace[lin * kTraceSlots + 233] = (long long)global_ns();
    }

    // ---- block coordinates
    const int GP = args.GP;
    const int R = BM / GP;
    const int pb = blockIdx.x, b = blockIdx.z;
    const int h0 = blockIdx.y * GP;
    const int g = h0 / (s.H / s.Hkv);
    const int p0 = pb * R;

    // ---- Q first: its load is the longest wait of the block's set-up
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmQ);
        mbar_init(bar(C::B_Q), 1u);
        fence_barrier_init();
        mbar_expect_tx(bar(C::B_Q), C::Q_BYTES);
        for (int dc = 0; dc < C::KD; ++dc)
            tma_load_3d_hint(sQ + dc * C::Q_DBLK, &tmQ, dc * 64, p0, b * s.H + h0, bar(C::B_Q),
                             policy_evict_first());
        stamp(2);
    }

    // ---- key chunks of this block
    ChunkWalk cw;
    cw.p0 = p0;
    cw.period = s.period;
    cw.cpb = R / CHUNK;
    cw.cpb_log2 = (cw.cpb == 4) ? 2 : (cw.cpb == 2) ? 1 : 0;
    cw.lo0 = band_lo(p0, s.mode, s.k_local);
    const int blk_hi = band_hi(min(s.N - 1, p0 + R - 1), s.N, s.mode, s.k_local);
    cw.n_band = (blk_hi - cw.lo0) / CHUNK + 1;
    int n_skip_blocks = 0;
    cw.m_first = args.m_first;
    cw.n_back = 0;
    if (s.mode != kModeEcp && s.S > 0) {
        const int m_last = min(s.S, (p0 + R - 1) / s.period);  // some row has i - m*period >= 0
        cw.n_back = max(0, m_last - cw.m_first + 1);
        n_skip_blocks = cw.n_back;
        if (s.mode == kModeBidir) {
            const int m_last_f = min(s.S, (s.N - 1 - p0) / s.period);  // some row has i + m*period < N
            n_skip_blocks += max(0, m_last_f - cw.m_first + 1);
        }
    }
    const int n_chunks = cw.n_band + n_skip_blocks * cw.cpb;
    const int n_tiles = (n_chunks + CPT - 1) / CPT;
    // Band chunks full_lo .. full_hi lie inside the band of every row of the block (the block
    // has no rows past N, the chunk starts at or after the last row's first key and ends at or
    // before the first row): such chunks need no per-row range.
    int full_lo = 1, full_hi = 0;
    if (p0 + R <= s.N) {
        const int lo_last = band_lo(p0 + R - 1, s.mode, s.k_local);
        full_lo = (lo_last - cw.lo0 + CHUNK - 1) / CHUNK;
        const int span = band_hi(p0, s.N, s.mode, s.k_local) - (CHUNK - 1) - cw.lo0;
        full_hi = span >= 0 ? min(span / CHUNK, cw.n_band - 1) : -1;
    }

    // ---- setup: barriers (spread over warp 0's lanes; only the P-ready barriers count 128
    // arrivals), TMEM
    if (warp == 0) {
        for (int idx = lane; idx < C::NBARS; idx += 32)
            if (idx != C::B_Q) mbar_init(bar(idx), (idx >= C::B_PR && idx < C::B_PR + NB) ? 128u : 1u);
        if (lane == 0) *abort_flag = 0u;
        fence_barrier_init();
        __syncwarp();
    }
    // K or V tile t into stage t % nst of its ring (the stage must be free)
    auto issue_kv = [&](const CUtensorMap *tm, uint32_t sbuf, int full_bar, int nst, int t, uint64_t policy) {
        const int st = t % nst;
        const int nch = min(CPT, n_chunks - CPT * t);
        mbar_expect_tx(bar(full_bar + st), nch * C::KD * BOX_BYTES);
        for (int cc = 0; cc < nch; ++cc) {
            int back, u;
            bool sk;
            const int key0 = cw.key0(CPT * t + cc, back, u, sk);
            for (int dc = 0; dc < C::KD; ++dc)
                tma_load_3d_hint(sbuf + st * C::KV_STAGE + dc * C::KV_DBLK + cc * BOX_BYTES, tm, dc * 64,
                                 key0, b * s.Hkv + g, bar(full_bar + st), policy);
        }
    };
    // The first K tile, which the first S = Q K^T waits for, goes out before the CTA barrier, so
    // that its latency overlaps the TMEM allocation and the barrier itself.
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmK);
        stamp_tile(8, 0);
        issue_kv(&tmK, sK, C::B_KF, KST, 0, policy_evict_last());
    }
    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    if (threadIdx.x == 0) {
        stamp(1);
        if (traced) args.trace[lin * kTraceSlots + 7] = n_tiles;
    }

    if (warp == 0) {
        // ================= producer: K tiles after the first
        if (lane == 0) {
            const uint64_t reused = policy_evict_last();
            int issued = 1;
            for (int t = 1; t < n_tiles; ++t) {
                const int st = t % KST, round = t / KST;
                if (round > 0 && !wait_bar(bar(C::B_KE + st), (round - 1) & 1, wc)) break;
                stamp_tile(8, t);
                issue_kv(&tmK, sK, C::B_KF, KST, t, reused);
                issued = t + 1;
            }
            if (*abort_flag) {  // let loads in flight land before the CTA leaves
                volatile uint32_t zero = 0;
                WaitCtx w2{&zero, nullptr, 20000000ull};
                wait_bar(bar(C::B_Q), 0, w2);
                for (int t = max(0, issued - KST); t < issued; ++t)
                    wait_bar(bar(C::B_KF + t % KST), (t / KST) & 1, w2);
            }
        }
    } else if (warp == 2) {
        // ================= producer: V tiles
        if (lane == 0) {
            prefetch_tmap(&tmV);
            const uint64_t reused = policy_evict_last();
            int issued = 0;
            for (int t = 0; t < n_tiles; ++t) {
                const int st = t % VST, round = t / VST;
                if (round > 0 && !wait_bar(bar(C::B_VE + st), (round - 1) & 1, wc)) break;
                stamp_tile(24, t);
                issue_kv(&tmV, sV, C::B_VF, VST, t, reused);
                issued = t + 1;
            }
            if (*abort_flag) {
                volatile uint32_t zero = 0;
                WaitCtx w2{&zero, nullptr, 20000000ull};
                for (int t = max(0, issued - VST); t < issued; ++t)
                    wait_bar(bar(C::B_VF + t % VST), (t / VST) & 1, w2);
            }
        }
    } else if (warp == 1) {
        // ================= S issuer: S = Q K^T into the tile's TMEM buffer.  It runs ahead of
        // the PV issuer, so that a PV never waits behind a K tile still in flight.  The whole warp
        // runs the loop and its waits, so that descriptors and TMEM addresses are warp-uniform;
        // one elected lane issues the MMAs and the commits.
        bool ok = __all_sync(0xffffffffu, wait_bar(bar(C::B_Q), 0, wc));
        if (ok && lane == 0) stamp(3);
        for (int t = 0; ok && t < n_tiles; ++t) {
            const int st = t % KST, buf = t % NB;
            bool w = timed_wait(bar(C::B_KF + st), (t / KST) & 1, 104, t);
            // buffer buf last held P of tile t-NB: its PV must be done
            if (w && t >= NB) w = timed_wait(bar(C::B_PV + buf), ((t - NB) / NB) & 1, 120, t);
            if (!__all_sync(0xffffffffu, w)) break;
            tc_fence_after();
            const int nch = min(CPT, n_chunks - CPT * t);
            const uint32_t idesc = idesc_bf16(BM, CHUNK * nch, 0, 0);
            const uint32_t dS = tbase + buf * TILE_N;
            const uint64_t a0 = sdesc(sQ, 16, 1024);
            const uint64_t b0 = sdesc(sK + st * C::KV_STAGE, 16, 1024);
            if (elect_one()) {
#pragma unroll
                for (int dc = 0; dc < C::KD; ++dc) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        // the start address field counts 16-byte units
                        const uint64_t a = a0 + (uint64_t)((dc * C::Q_DBLK + ks * 32) >> 4);
                        const uint64_t bb = b0 + (uint64_t)((dc * C::KV_DBLK + ks * 32) >> 4);
                        mma_ss(dS, a, bb, idesc, (dc | ks) != 0);
                    }
                }
                tc_commit(bar(C::B_SF + buf));
                tc_commit(bar(C::B_KE + st));
            }
            __syncwarp();
            if (lane == 0) stamp_tile(40, t);
        }
        // every MMA this warp issued has finished before TMEM is released
        if (elect_one()) tc_commit(bar(C::B_DR));
        __syncwarp();
        volatile uint32_t zero = 0;
        WaitCtx w2{&zero, args.status, args.timeout_ns};
        wait_bar(bar(C::B_DR), 0, w2);
    } else if (warp == 3) {
        // ================= PV issuer: O += P V with P read from TMEM (whole warp, one elected
        // lane issuing, as for the S issuer)
        bool ok = true;
        for (int u = 0; ok && u < n_tiles; ++u) {
            const int st = u % VST, buf = u % NB;
            bool w = timed_wait(bar(C::B_PR + buf), (u / NB) & 1, 136, u);
            if (w) w = timed_wait(bar(C::B_VF + st), (u / VST) & 1, 152, u);
            if (!__all_sync(0xffffffffu, w)) break;
            tc_fence_after();
            const int nch = min(CPT, n_chunks - CPT * u);
            const uint32_t idesc = idesc_bf16(BM, D, 0, 1);
            const uint32_t aP = tbase + buf * TILE_N;
            const uint64_t b0 = sdesc(sV + st * C::KV_STAGE, C::KV_DBLK, 1024);
            if (elect_one()) {
                for (int kk = 0; kk < 2 * nch; ++kk)
                    mma_ts(tbase + O_COL, aP + kk * 8, b0 + (uint64_t)((kk * 16 * ROW_BYTES) >> 4), idesc,
                           (u > 0 || kk > 0) ? 1u : 0u);
                tc_commit(bar(C::B_PV + buf));
                tc_commit(bar(C::B_VE + st));
                if (u == n_tiles - 1) tc_commit(bar(C::B_OF));
            }
            __syncwarp();
            if (lane == 0) stamp_tile(56, u);
        }
        if (elect_one()) tc_commit(bar(C::B_DR2));
        __syncwarp();
        volatile uint32_t zero = 0;
        WaitCtx w2{&zero, args.status, args.timeout_ns};
        wait_bar(bar(C::B_DR2), 0, w2);
    } else if (warp >= 4) {
        // ================= softmax + epilogue: one thread per row
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;
        const int hh = r / R, trow = r % R;
        const int i = p0 + trow;
        const int h = h0 + hh;
        const bool row_ok = i < s.N;
        const long long row_g = ((long long)b * s.H + h) * s.N + i;
        float al = (args.alpha && row_ok) ? args.alpha[row_g] : 1.f;
        if (args.gate_w) {
            // Fused gate ("pi-Attention" page, 2.3): a per-token, per-head logistic gate on this
            // row of the Q tile, alpha = 1 / (1 + exp(-(q_i . w_h + c_h))).  The rows past N
            // read the zero fill and are not written.
            if (__all_sync(0xffffffffu, wait_bar(bar(C::B_Q), 0, wc))) {
                const float *wh = args.gate_w + (size_t)h * D;
                float z0 = args.gate_b[h], z1 = 0.f;
#pragma unroll
                for (int dc = 0; dc < C::KD; ++dc) {
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {  // 8 bf16 of the row per 16-byte chunk
                        const uint4 u = *reinterpret_cast<const uint4 *>(smem + C::Q_OFF + dc * C::Q_DBLK +
                                                                         r * ROW_BYTES + ((ch ^ (r & 7)) << 4));
                        const float4 wa = *reinterpret_cast<const float4 *>(wh + dc * 64 + ch * 8);
                        const float4 wb = *reinterpret_cast<const float4 *>(wh + dc * 64 + ch * 8 + 4);
                        z0 = fmaf(__uint_as_float(u.x << 16), wa.x, z0);
                        z1 = fmaf(__uint_as_float(u.x & 0xffff0000u), wa.y, z1);
                        z0 = fmaf(__uint_as_float(u.y << 16), wa.z, z0);
                        z1 = fmaf(__uint_as_float(u.y & 0xffff0000u), wa.w, z1);
                        z0 = fmaf(__uint_as_float(u.z << 16), wb.x, z0);
                        z1 = fmaf(__uint_as_float(u.z & 0xffff0000u), wb.y, z1);
                        z0 = fmaf(__uint_as_float(u.w << 16), wb.z, z0);
                        z1 = fmaf(__uint_as_float(u.w & 0xffff0000u), wb.w, z1);
                    }
                }
                al = 1.f / (1.f + __expf(-(z0 + z1)));
                if (args.alpha_out && row_ok) args.alpha_out[row_g] = al;
            }
        }
        const float off_band = (s.mode != kModeEcp) ? log2f(al) : 0.f;
        const float off_skip = log2f(1.f - al);
        const int lo_i = band_lo(i, s.mode, s.k_local);
        const int hi_i = band_hi(i, s.N, s.mode, s.k_local);
        const float sc = s.scale_log2;
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        float lse2_in = 0.f;
        if (DBG == 2) lse2_in = row_ok ? args.lse_in[row_g] * kLog2e : -INFINITY;

        float m_ref = -INFINITY, l = 0.f;
        long long cnt = 0, isum = 0;
        bool ok = true;

        // valid column range [clo, chi] of chunk ci for this row, and its prior
        auto chunk_range = [&](int ci, int &key0, int &clo, int &chi, float &off, bool &sk) {
            int back, u;
            key0 = cw.key0(ci, back, u, sk);
            if (!sk) {
                clo = max(lo_i - key0, 0);
                chi = min(hi_i - key0, CHUNK - 1);
                off = off_band;
            } else {
                const int jk = i - back;
                const int c = jk - key0;
                if (jk >= 0 && jk < s.N && c >= 0 && c < CHUNK) { clo = c; chi = c; }
                else { clo = CHUNK; chi = -1; }
                off = off_skip;
            }
        };

        // Rescale this row of O when the reference max moved.  PV of tile t-1 must be done.
        // The wait names that phase exactly: S of tile t-1 implied PV of tile t-3 finished,
        // and PV of tile t+1 cannot start before this thread arrives for tile t+1.
        auto rescale_o = [&](int t, bool need_o, float corr) -> bool {
            if (!__any_sync(0xffffffffu, need_o)) return true;
            const bool r_ = wait_bar(bar(C::B_PV + (t - 1) % NB), ((t - 1) / NB) & 1, wc);
            if (!__all_sync(0xffffffffu, r_)) return false;
            tc_fence_after();
            const float f = need_o ? corr : 1.f;
#pragma unroll
            for (int oc = 0; oc < D / 16; ++oc) {
                uint32_t x[16];
                tmem_ld16(tbase + lane_base + O_COL + oc * 16, x);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 16; ++c) x[c] = __float_as_uint(__uint_as_float(x[c]) * f);
                tmem_st16(tbase + lane_base + O_COL + oc * 16, x);
            }
            return true;
        };

        for (int t = 0; t < n_tiles; ++t) {
            const int buf = t % NB;
            if (warp == 4 && lane == 0) ok = timed_wait(bar(C::B_SF + buf), (t / NB) & 1, 168, t);
            else ok = wait_bar(bar(C::B_SF + buf), (t / NB) & 1, wc);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            if (warp == 4 && lane == 0) stamp_tile(72, t);
            tc_fence_after();
            __syncwarp();
            const int nch = (CPT == 1) ? 1 : min(2, n_chunks - 2 * t);
            const uint32_t tS = tbase + lane_base + buf * TILE_N;
            uint32_t ra[CHUNK], rb[CHUNK];
            tmem_ld32(tS, ra);
            if (nch > 1) tmem_ld32(tS + CHUNK, rb);
            tmem_wait_ld();
            if (warp == 4 && lane == 0) stamp_tile(184, t);

            // Full tile (the same for every thread of the CTA): P with the running reference; the
            // maximum is only needed when some P exceeds 2^8 (the lazy-rescale bound), which a
            // sum above 2^8 is the first sign of.  Rows with no reference yet take the general
            // path, as do the debug modes that record per-row ranges.
            const bool fast = (DBG == 0 || DBG == 3) && nch == CPT && CPT * t >= full_lo &&
                              CPT * t + CPT - 1 <= full_hi && __all_sync(0xffffffffu, m_ref != -INFINITY);
            float corr = 1.f, lsum;
            bool need_o = false;
            if (fast) {
                lsum = exp_pack<CPT>(ra, rb, sc, off_band - m_ref);
                if (__any_sync(0xffffffffu, !(lsum <= 256.f))) {
                    tmem_ld32(tS, ra);  // S is still in TMEM: P has not been written yet
                    if (CPT == 2) tmem_ld32(tS + CHUNK, rb);
                    tmem_wait_ld();
                    const float mt = fmaf(max_tile<CPT>(ra, rb), sc, off_band);
                    if (mt > m_ref + kRescaleThreshold) {
                        corr = fast_exp2(m_ref - mt);
                        need_o = true;  // m_ref was set by an earlier tile, so t > 0
                        m_ref = mt;
                    }
                    l *= corr;
                    lsum = exp_pack<CPT>(ra, rb, sc, off_band - m_ref);
                }
                if (warp == 4 && lane == 0) stamp_tile(200, t);
                tmem_st16(tS, ra);
                if (CPT == 2) tmem_st16(tS + CHUNK / 2, rb);
            } else {

                int key0a, cloa, chia, key0b = 0, clob = CHUNK, chib = -1;
                float offa, offb = 0.f;
                bool ska, skb = false;
                chunk_range(CPT * t, key0a, cloa, chia, offa, ska);
                if (nch > 1) chunk_range(CPT * t + 1, key0b, clob, chib, offb, skb);

                float *fa = reinterpret_cast<float *>(ra);
                float *fb = reinterpret_cast<float *>(rb);
                const float za = chunk_max(fa, cloa, chia, ska, sc, offa);
                const float zb = (nch > 1) ? chunk_max(fb, clob, chib, skb, sc, offb) : -INFINITY;
                const float mt = fmaxf(za, zb);
                if (warp == 4 && lane == 0) stamp_tile(200, t);
                if (mt > m_ref + kRescaleThreshold) {
                    if (m_ref != -INFINITY) {
                        corr = fast_exp2(m_ref - mt);
                        need_o = (t > 0);
                    }
                    m_ref = mt;
                }
                l *= corr;
                const float mu = (m_ref == -INFINITY) ? 0.f : m_ref;

                if (DBG == 1) {
                    const int na = max(0, chia - cloa + 1), nb = max(0, chib - clob + 1);
                    cnt += na + nb;
                    isum += (long long)na * key0a + (long long)(cloa + chia) * na / 2;
                    isum += (long long)nb * key0b + (long long)(clob + chib) * nb / 2;
                }
                if (DBG == 2 && row_ok && lse2_in != -INFINITY) {
                    for (int c = 0; c < CHUNK; ++c) {
                        if (c >= cloa && c <= chia)
                            args.P[row_g * s.N + key0a + c] = exp2f(fmaf(fa[c], sc, offa - lse2_in));
                        if (nch > 1 && c >= clob && c <= chib)
                            args.P[row_g * s.N + key0b + c] = exp2f(fmaf(fb[c], sc, offb - lse2_in));
                    }
                }

                // P = exp2(z - m_ref) as bf16, written over the chunk's S columns
                uint32_t pk[CHUNK / 2];
                lsum = chunk_exp(fa, cloa, ska, za, sc, offa, mu, pk);
                tmem_st16(tS, pk);
                if (nch > 1) {
                    lsum += chunk_exp(fb, clob, skb, zb, sc, offb, mu, pk);
                    tmem_st16(tS + CHUNK / 2, pk);
                }
            }
            if (warp == 4 && lane == 0) stamp_tile(216, t);
            l += lsum;
            __syncwarp();
            if (!rescale_o(t, need_o, corr)) { ok = false; break; }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(C::B_PR + buf));
            if (warp == 4 && lane == 0) stamp_tile(88, t);
        }

        // ---- epilogue: O / l -> bf16 -> shared (swizzled, reusing the Q buffer) -> TMA store
        // A parity wait names a phase only if the barrier is at most one phase away from it;
        // by now the PV barrier may be anywhere from n_tiles-2 to n_tiles phases along, so the
        // epilogue waits on its own single-phase barrier.
        if (ok) {
            ok = wait_bar(bar(C::B_OF), 0, wc);
            ok = __all_sync(0xffffffffu, ok);
        }
        if (warp == 4 && lane == 0) stamp(4);
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
        if (ok) {
            tc_fence_after();
            __syncwarp();
#pragma unroll
            for (int oh = 0; oh < D / 32; ++oh) {  // 32 fp32 columns per TMEM round trip
                uint32_t x[32];
                tmem_ld32(tbase + lane_base + O_COL + oh * 32, x);
                tmem_wait_ld();
                const int dc = oh >> 1;
                uint8_t *rowp = smem + C::Q_OFF + dc * C::Q_DBLK + r * ROW_BYTES;
#pragma unroll
                for (int w = 0; w < 4; ++w) {  // 8 columns -> one 16-byte chunk of the row
                    const int cidx = (oh & 1) * 4 + w;
                    const float *f = reinterpret_cast<const float *>(x) + 8 * w;
                    const uint4 val = make_uint4(pack_bf16(f[0] * inv_l, f[1] * inv_l), pack_bf16(f[2] * inv_l, f[3] * inv_l),
                                                 pack_bf16(f[4] * inv_l, f[5] * inv_l), pack_bf16(f[6] * inv_l, f[7] * inv_l));
                    *reinterpret_cast<uint4 *>(rowp + ((cidx ^ (r & 7)) << 4)) = val;
                }
            }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (ok && warp == 4 && lane == 0) {
            const uint64_t stream_once = policy_evict_first();
            for (int dc = 0; dc < C::KD; ++dc)
                tma_store_3d(&tmO, sQ + dc * C::Q_DBLK, dc * 64, p0, b * s.H + h0, stream_once);
            tma_store_commit_and_wait();
            stamp(5);
        }
        if (ok && row_ok) {
            args.lse[row_g] = (l > 0.f) ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
            if (DBG == 1) {
                args.cnt[row_g] = (int)cnt;
                args.isum[row_g] = isum;
            }
        }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && traced) {
        stamp(6);
        args.trace[lin * kTraceSlots + 234] = (long long)global_ns();
    }
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tbase, TMEM_COLS);
    }
}

// Bounded-wait self test: waits on a barrier that never completes.
__global__ void wait_timeout_probe_kernel(int *status, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar_storage;
    __shared__ uint32_t abort_storage;
    const uint32_t b = smem_u32(&bar_storage);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        abort_storage = 0u;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        WaitCtx w{&abort_storage, status, timeout_ns};
        wait_bar(b, 0, w);
    }
    __syncthreads();
}

// ------------------------------------------------------------------ host side

template <int D, int DBG>
static cudaError_t launch(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                          const CUtensorMap &mo, const TcArgs &a, dim3 grid, cudaStream_t st) {
    constexpr int smem = Cfg<D>::SMEM_BYTES;
    static int configured_device = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_device != dev) {
        cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel<D, DBG>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured_device = dev;
    }
    fwd_tc_kernel<D, DBG><<<grid, NUM_THREADS, smem, st>>>(mq, mk, mv, mo, a);
    return cudaGetLastError();
}

}  // namespace tc

cudaError_t launch_fwd_tc(const LaunchFwd &L, cudaStream_t st) {
    using namespace tc;
    const Shape &s = L.s;
    const int G = s.H / s.Hkv;
    const int GP = (G % 4 == 0) ? 4 : (G % 2 == 0) ? 2 : 1;
    const int R = BM / GP;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, L.q, s.d, s.N, (long long)s.B * s.H, R, GP) ||
        !make_map(&mo, L.out, s.d, s.N, (long long)s.B * s.H, R, GP) ||
        !make_map(&mk, L.k, s.d, s.N, (long long)s.B * s.Hkv, CHUNK, 1) ||
        !make_map(&mv, L.v, s.d, s.N, (long long)s.B * s.Hkv, CHUNK, 1))
        return cudaErrorNotSupported;
    int m_first = 1;
    if (s.mode != kModeEcp && s.S > 0) m_first = s.k_local / s.period + 1;  // smallest m with m*period > k
    TcArgs a{L.alpha, L.lse, s, GP, m_first, L.status, L.timeout_ns, L.cnt, L.isum, L.lse_in, L.P,
             L.trace, L.n_trace, L.gate_w, L.gate_b, L.alpha_out};
    if (s.H / GP > 65535 || s.B > 65535) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)((s.N + R - 1) / R), (unsigned)(s.H / GP), (unsigned)s.B);
    if (s.d == 64) {
        if (L.dbg == 0) return launch<64, 0>(mq, mk, mv, mo, a, grid, st);
        if (L.dbg == 1) return launch<64, 1>(mq, mk, mv, mo, a, grid, st);
        if (L.dbg == 3) return launch<64, 3>(mq, mk, mv, mo, a, grid, st);
        return launch<64, 2>(mq, mk, mv, mo, a, grid, st);
    }
    if (s.d == 128) {
        if (L.dbg == 0) return launch<128, 0>(mq, mk, mv, mo, a, grid, st);
        if (L.dbg == 1) return launch<128, 1>(mq, mk, mv, mo, a, grid, st);
        if (L.dbg == 3) return launch<128, 3>(mq, mk, mv, mo, a, grid, st);
        return launch<128, 2>(mq, mk, mv, mo, a, grid, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_wait_timeout_probe(int *status, uint64_t timeout_ns, cudaStream_t st) {
    tc::wait_timeout_probe_kernel<<<1, 32, 0, st>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace pi
