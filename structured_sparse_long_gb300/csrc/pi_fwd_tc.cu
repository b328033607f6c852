// pi_fwd_tc.cu -- fused pi-Attention / ECP forward on sm_103a tensor cores.
//
// What it computes ("pi-Attention: Periodic Sparse Transformers for Efficient
// Long-Context Modeling", section 2.1-2.3; ECP page section 2; GQA from the
// GSS-Transformer hybrid page): for each query row i, one softmax over the
// causal band [lo(i), i] and the skip keys i - m*period (pi mode), with
// log2(alpha) added to band logits and log2(1 - alpha) to skip logits, and the
// softmax-weighted sum of value rows.
//
// How (one block = 128 query rows = the M of every MMA):
//   * GQA packing: the 128 rows are GP query heads of one KV group x R = 128/GP
//     consecutive positions, so every K/V tile staged in shared memory serves
//     all GP heads at once.
//   * Keys are walked in 32-key tiles (one TMA box per 64 columns of d).  A tile
//     is either a band tile (keys lo(p0) + 32c ...) or a skip tile: the keys
//     i - m*period of the block's rows form R consecutive keys, so one skip block
//     is R/32 tiles; each row attends to exactly one column of it (the
//     "diagonal").
//   * The kernel is persistent: each CTA (two per SM) processes blocks c,
//     c + gridDim.x, ... in turn.  The next block's Q tile is loaded during the
//     current block and copied into TMEM (tcgen05.cp, by the S issuer) as soon as
//     the current block's last S product is done, so the next block's first S
//     products overlap this block's epilogue; a producer warp TMA-stores each
//     block's staged output.
//   * Warp 0 (lane 0) streams the K tiles; warp 2 (lane 0) streams the V tiles,
//     stores the staged outputs and loads the next Q tiles.  Both MMAs take their
//     A operand from TMEM: warp 1 copies each Q tile there and issues S = Q K^T
//     into one of NB TMEM S buffers, and warp 3 issues O += P V with P read from
//     TMEM (each whole warp runs its loop, one elected lane issues the copies, the
//     MMAs and the commits).
//   * Warps 4-7 run the softmax, one thread per row (TMEM lane = row): masks,
//     adds the prior, keeps the running max m and sum l (rescaling O in TMEM only
//     when the max grows by more than 2^8), writes P as bf16 over its S, and at
//     the end of the block normalises O and stages it in shared memory.
//   * The fused gate (GATE) puts one more tile in front of a block's key tiles: the
//     W1 rows of the block's heads, so that its S product is the heads' hidden
//     pre-activations; the row threads finish the MLP and take its alpha.
//   * Every wait is bounded; a wait that runs out sets the device status word and
//     the CTA unwinds without hanging.
//   * The kernel's speed is bound by latency and by instruction fetch, so the
//     per-tile code is kept small: one copy of the 32 exponentials, rare paths
//     rolled, the polling part of the waits out of line.
#include <cuda.h>

#include "pi_common.cuh"
#include "pi_launch.h"
#include "pi_tc_ptx.cuh"

namespace pi {
namespace tc {

constexpr int BM = 128;           // rows per block (MMA M)
constexpr int CHUNK = 32;         // keys per tile (TMA box rows; the N of the S products)
// S buffers in TMEM.  The query tile is the A operand of the S products and lives in TMEM,
// so that an S product reads only its K tile from shared memory: a 128 x 32 x 16 product
// with A in TMEM costs the pipe about 26 cycles, against about 59 with A in shared memory.
// P is written as bf16 over its S and is the TMEM A operand of the PV products.  TMEM columns
// (256 per CTA, two CTAs per SM):
//   d = 128: S buffers [0, 64) (two of 32 keys), Q [64, 128) (bf16 pairs), O [128, 256)
//   d = 64:  S buffers [0, 128) (four of 32 keys), O [128, 192), Q [192, 224)
template <int D>
struct Tiling {
    static constexpr int NB = (D == 64) ? 4 : 2;
    static constexpr int O_COL = 128;
    static constexpr int Q_COL = (D == 128) ? 64 : 192;
    static_assert(NB * CHUNK <= Q_COL && NB * CHUNK <= O_COL, "S buffers overlap Q or O");
    static_assert(Q_COL + D / 2 <= O_COL || Q_COL >= O_COL + D, "Q overlaps O");
    static_assert(Q_COL + D / 2 <= 256 && O_COL + D <= 256, "TMEM regions exceed 256 columns");
};
constexpr int NUM_THREADS = 256;
constexpr int TMEM_COLS = 256;
constexpr int ROW_BYTES = 128;    // one 64-element bf16 swizzle row
constexpr int BOX_BYTES = CHUNK * ROW_BYTES;  // one 64 x 32 TMA box
constexpr float kRescaleThreshold = 8.f;      // log2 units

template <int D>
struct Cfg {
    static constexpr int NB = Tiling<D>::NB;
    static constexpr int O_COL = Tiling<D>::O_COL, Q_COL = Tiling<D>::Q_COL;
    static constexpr int KD = D / 64;  // 64-element column blocks of d
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int KV_STAGE = CHUNK * D * 2;
    // 48 KB of K tiles (the S issuer runs furthest ahead) and 32 KB of V tiles
    static constexpr int KSTAGES = 49152 / KV_STAGE;
    static constexpr int VSTAGES = 32768 / KV_STAGE;
    static constexpr int KV_DBLK = CHUNK * ROW_BYTES;  // one 64-column block of a stage
    static constexpr int Q_DBLK = BM * ROW_BYTES;
    // [0, Q_BYTES): the Q tile as loaded; once it is copied into TMEM, the same bytes stage the
    // previous block's output for its TMA store, and then take the Q tile of the next block.
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + Q_BYTES;
    static constexpr int V_OFF = K_OFF + KSTAGES * KV_STAGE;
    static constexpr int DATA_BYTES = V_OFF + VSTAGES * KV_STAGE;  // from a 1024-byte aligned base
    // barrier indices.  Tiles are counted across the blocks a CTA processes; block k of the CTA
    // completes the per-block barriers in phase k.
    static constexpr int B_Q = 0;                // Q tile of the block landed in shared memory
    static constexpr int B_KF = 1;
    static constexpr int B_KE = B_KF + KSTAGES;
    static constexpr int B_VF = B_KE + KSTAGES;
    static constexpr int B_VE = B_VF + VSTAGES;
    static constexpr int B_SF = B_VE + VSTAGES;  // [NB] S of tile g in TMEM buffer g % NB
    static constexpr int B_PR = B_SF + NB;       // [NB] P of the tile written over its S (128)
    // PV of tile g completes barrier B_PV + g % NB, phase g / NB: a buffer's PV barrier is
    // waited for in order, so no parity wait has two of its phases outstanding.
    static constexpr int B_PV = B_PR + NB;
    static constexpr int B_OF = B_PV + NB;   // O of the block complete (after its last PV)
    static constexpr int B_QT = B_OF + 1;    // Q of the block copied into TMEM (its shared buffer read)
    static constexpr int B_STF = B_QT + 1;   // output of the block staged (128 arrivals)
    static constexpr int B_STR = B_STF + 1;  // staged output read by its TMA store
    static constexpr int B_DR = B_STR + 1;   // drain of the S issuer's MMAs
    static constexpr int B_DR2 = B_DR + 1;   // drain of the PV issuer's MMAs
    static constexpr int B_SD = B_DR2 + 1;   // S products of the block done (its Q no longer read)
    static constexpr int NBARS = B_SD + 1;
    static constexpr bool counts128(int idx) {
        return (idx >= B_PR && idx < B_PR + NB) || idx == B_STF;
    }
    static constexpr int BAR_BYTES = NBARS * 8 + 16;  // + TMEM address and abort flag
    static_assert(BAR_BYTES <= 512, "barriers must fit the alignment gap or its complement");
    // The data starts at the first 1024-byte boundary of the dynamic shared memory; the
    // barriers go into the gap before it when it is large enough, else after the data.
    // Either way DATA_BYTES + 1024 bytes suffice.
    static constexpr int SMEM_BYTES = DATA_BYTES + 1024;
};

// Phase 1 of a tile for one row (general path): mask the scores outside [clo, chi] and return
// the tile's largest logit in log2 units (prior included).  A skip tile holds at most one
// valid column per row (its diagonal), read with a select tree instead of a full pass.
__device__ __forceinline__ float tile_max(float *f, int clo, int chi, bool skip, float sc, float off) {
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

// P = exp2(s * sc + bo) for a tile's 32 raw scores, packed as 16 bf16 pairs in place (word
// c/2 is written after scores c and c+1 were read); returns the sum of the fp32 values.
// Masked scores (-inf) give exactly 0.
__device__ __forceinline__ float tile_exp(uint32_t *r, float sc, float bo) {
    const uint64_t sc2 = pack2(sc, sc), bo2 = pack2(bo, bo);
    uint64_t acc0 = pack2(0.f, 0.f), acc1 = pack2(0.f, 0.f);  // two independent sums
#pragma unroll
    for (int c = 0; c < 32; c += 2) {
        float z0, z1;
        unpack2(fma2(pack2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])), sc2, bo2), z0, z1);
        const float p0 = fast_exp2(z0);
        const float p1 = fast_exp2(z1);
        if ((c >> 1) & 1) acc1 = add2(acc1, pack2(p0, p1));
        else acc0 = add2(acc0, pack2(p0, p1));
        r[c / 2] = pack_bf16(p0, p1);
    }
    float a0, a1, b0, b1;
    unpack2(acc0, a0, a1);
    unpack2(acc1, b0, b1);
    return (a0 + a1) + (b0 + b1);
}

// Skip tile: P is zero except column clo, exp2(zdiag - mu); packed into words 0-15.
__device__ __forceinline__ float tile_exp_diag(uint32_t *r, int clo, float zdiag, float mu) {
    const float p = (clo < CHUNK) ? fast_exp2(zdiag - mu) : 0.f;
    __nv_bfloat16 hb = __float2bfloat16_rn(p);
    const uint32_t bits = (uint32_t)(*reinterpret_cast<uint16_t *>(&hb));
    const uint32_t word = (clo & 1) ? (bits << 16) : bits;
#pragma unroll
    for (int w = 0; w < 16; ++w) r[w] = (w == (clo >> 1)) ? word : 0u;
    return p;
}

// Largest of a tile's 32 raw scores (four independent chains).
__device__ __forceinline__ float tile_raw_max(const uint32_t *r) {
    float m[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) m[k] = max3(__uint_as_float(r[k]), __uint_as_float(r[k + 4]), __uint_as_float(r[k + 8]));
#pragma unroll
    for (int c = 12; c < CHUNK; c += 8) {
#pragma unroll
        for (int k = 0; k < 4; ++k) m[k] = max3(m[k], __uint_as_float(r[c + k]), __uint_as_float(r[c + 4 + k]));
    }
    return fmaxf(max3(m[0], m[1], m[2]), m[3]);
}

// ------------------------------------------------------------------ kernel

// Division by a divisor fixed for the launch, as a multiply and a shift (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994: with
// l = ceil(log2 d) and m = floor(2^(32+l) / d) + 1, floor(n / d) = floor(n m / 2^(32+l)) for
// every 32-bit n).  The dividends here are below 2^31, so n * m (m < 2^33) fits 64 bits.
struct FastDiv {
    uint64_t m;
    int sh;
    __device__ __forceinline__ int div(int n) const {
        return (int)(((unsigned long long)(unsigned)n * m) >> sh);
    }
};
static inline FastDiv make_fastdiv(int d) {
    int l = 0;
    while ((1LL << l) < (long long)d) ++l;
    const unsigned __int128 num = (unsigned __int128)1 << (32 + l);
    FastDiv f;
    f.m = (uint64_t)(num / (unsigned)d) + 1;
    f.sh = 32 + l;
    return f;
}

struct TcArgs {
    const float *alpha;
    float *lse;
    Shape s;
    int GP;       // query heads packed per block
    int m_first;  // smallest skip multiple m with m * period > k_local (at most S + 1)
    int nqb;      // position blocks per (batch entry, head group)
    int ngrp;     // head groups (H / GP)
    int R;        // positions per block, 128 / GP
    int cpb_log2; // log2 of the tiles per skip block (R / 32)
    FastDiv div_nqb, div_ngrp, div_G, div_period;  // by nqb, ngrp, H / Hkv, period
    int n_blocks; // blocks in all: nqb * ngrp * B; CTA c processes blocks c, c + gridDim.x, ...
    int *status;
    uint64_t timeout_ns;
    int *cnt;
    long long *isum;
    const float *lse_in;
    float *P;
    long long *trace;  // DBG 3: clock64() stamps, kTraceSlots per traced CTA
    int n_trace;       // DBG 3: CTAs 0 .. n_trace-1 are traced
    // fused gate (GATE): hid = max(0, W1_h q_i + b1_h), alpha = 1 / (1 + exp(-(w2_h . hid + b2_h)));
    // W1 [H * kGateHidden, d] bf16 reaches the kernel as a tensor map
    const float *gate_b1;  // [H, kGateHidden]
    const float *gate_w2;  // [H, kGateHidden]
    const float *gate_b2;  // [H]
    float *alpha_out;      // [B, H, N] the gate's alpha (may be null)
};

// Trace layout (DBG 3: one block per CTA), slots per CTA: 0 entry, 1 set-up done, 2 Q issued,
// 3 Q in TMEM (seen by the S issuer), 4 O complete (softmax side), 5 output staged, 6 exit,
// 7 tile count; then per tile t (t < 16): 8+t K issued, 24+t V issued, 40+t S issued, 56+t PV
// issued, 72+t S seen by the softmax, 88+t P ready; and cycles spent waiting, each measured
// within one thread: 104+t S issuer on K, 120+t S issuer on the S buffer (PV of t-NB), 136+t
// PV issuer on P, 152+t PV issuer on V, 168+t softmax on S; softmax (warp 4) stamps inside tile
// t: 184+t S loaded from TMEM, 200+t maxima done (full tiles: exponentials done), 216+t P
// written to TMEM (issued); 232 the SM the CTA ran on, 233 and 234 the global timer (ns) at
// entry and exit.  The warps of an SM read one clock.
constexpr int kTraceSlots = 240;
constexpr int kTraceTiles = 16;

// Key tile ti of a block: first key position, whether it is a skip tile, and its skip
// distance.  Skip blocks come after the band: first the n_back blocks of keys i - m*period,
// then (in the bidirectional mode) those of keys i + m*period, both for m = m_first,
// m_first + 1, ...; `back` is the signed distance i - key.
struct ChunkWalk {
    int lo0, n_band, m_first, cpb, cpb_log2, p0, period, n_back;
    __device__ __forceinline__ int key0(int ci, int &back, bool &skip) const {
        if (ci < n_band) {
            back = 0;
            skip = false;
            return lo0 + ci * CHUNK;
        }
        const int sc = ci - n_band;  // cpb = R / 32 is 1, 2 or 4
        const int blk = sc >> cpb_log2;
        const int u = sc & (cpb - 1);
        back = (blk < n_back) ? (m_first + blk) * period : -(m_first + blk - n_back) * period;
        skip = true;
        return p0 - back + u * CHUNK;
    }
};

// One block: 128 query rows = GP heads of one KV group x R = 128 / GP consecutive positions.
struct BlockDesc {
    int b, h0, g, p0;
    ChunkWalk cw;
    int n_tiles;
    int full_lo, full_hi;  // band tiles inside the band of every row of the block
};

// Block L (positions fastest, then head groups, then batch entries) and its key tiles.
__device__ __forceinline__ void describe_block(int L, const TcArgs &a, BlockDesc &d) {
    const Shape &s = a.s;
    const int R = a.R;
    const int rest = a.div_nqb.div(L);
    const int pb = L - rest * a.nqb;
    const int b = a.div_ngrp.div(rest);
    d.h0 = (rest - b * a.ngrp) * a.GP;
    d.b = b;
    d.g = a.div_G.div(d.h0);
    d.p0 = s.qoff + pb * R;  // key position of the block's first query row
    ChunkWalk &cw = d.cw;
    cw.p0 = d.p0;
    cw.period = s.period;
    cw.cpb_log2 = a.cpb_log2;
    cw.cpb = 1 << a.cpb_log2;
    cw.lo0 = band_lo(d.p0, s.mode, s.k_local);
    const int blk_hi = band_hi(min(s.N - 1, d.p0 + R - 1), s.N, s.mode, s.k_local);
    cw.n_band = (blk_hi - cw.lo0) / CHUNK + 1;
    int n_skip_blocks = 0;
    cw.m_first = a.m_first;
    cw.n_back = 0;
    if (s.mode != kModeEcp && s.S > 0) {
        const int m_last = min(s.S, a.div_period.div(d.p0 + R - 1));  // some row has i - m*period >= 0
        cw.n_back = max(0, m_last - cw.m_first + 1);
        n_skip_blocks = cw.n_back;
        if (s.mode == kModeBidir) {
            const int m_last_f = min(s.S, a.div_period.div(s.N - 1 - d.p0));  // some row has i + m*period < N
            n_skip_blocks += max(0, m_last_f - cw.m_first + 1);
        }
    }
    d.n_tiles = cw.n_band + n_skip_blocks * cw.cpb;
    // Band tiles full_lo .. full_hi lie inside the band of every row of the block (the block
    // has no rows past N, the tile starts at or after the last row's first key and ends at or
    // before the first row): such tiles need no per-row range.
    d.full_lo = 1;
    d.full_hi = 0;
    if (d.p0 + R <= s.N) {
        const int lo_last = band_lo(d.p0 + R - 1, s.mode, s.k_local);
        d.full_lo = (lo_last - cw.lo0 + CHUNK - 1) / CHUNK;
        const int span = band_hi(d.p0, s.N, s.mode, s.k_local) - (CHUNK - 1) - cw.lo0;
        d.full_hi = span >= 0 ? min(span / CHUNK, cw.n_band - 1) : -1;
    }
}

// The fused gate's output for one row ("pi-Attention" page, 2.3: a light MLP per token and per
// head): pre holds the row's hidden pre-activations W1_h q (the tensor core's product of the Q
// tile with the W1 rows of the block's heads); returns alpha = 1 / (1 + exp(-z)) with
// z = w2_h . max(0, pre + b1_h) + b2_h.  A warp's rows share one head, so the weight loads are
// warp-uniform.
__device__ __forceinline__ float gate_alpha(const uint32_t *pre, const float *b1, const float *w2, float b2) {
    float z = b2;
#pragma unroll
    for (int f = 0; f < kGateHidden; ++f) z = fmaf(w2[f], fmaxf(__uint_as_float(pre[f]) + b1[f], 0.f), z);
    return 1.f / (1.f + __expf(-z));
}

template <int D, int DBG, bool GATE>
__global__ void __launch_bounds__(NUM_THREADS, 2)
fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
              const __grid_constant__ CUtensorMap tmW, const TcArgs args) {
    using C = Cfg<D>;
    constexpr int KST = C::KSTAGES, VST = C::VSTAGES, NB = C::NB;
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
    const int L0 = blockIdx.x, LS = gridDim.x;
    // the CTA's next block, or n_blocks past its last (no int overflow near 2^31 blocks)
    auto next_block = [&](int L) -> int { return (L < args.n_blocks - LS) ? L + LS : args.n_blocks; };
    const bool traced = DBG == 3 && L0 < args.n_trace;
    auto stamp = [&](int slot) {
        if (traced) args.trace[(long long)L0 * kTraceSlots + slot] = (long long)clock64();
    };
    auto stamp_tile = [&](int base, int t) {
        if (t < kTraceTiles) stamp(base + t);
    };
    // bounded wait that also records how long it took (DBG 3)
    auto timed_wait = [&](uint32_t b, uint32_t parity, int slot_base, int t) -> bool {
        const long long c0 = (DBG == 3) ? (long long)clock64() : 0;
        const bool r = wait_bar(b, parity, wc);
        if (traced && t < kTraceTiles && lane == 0)
            args.trace[(long long)L0 * kTraceSlots + slot_base + t] = (long long)clock64() - c0;
        return r;
    };
    if (threadIdx.x == 0 && traced) {
        stamp(0);
        uint32_t smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        args.trace[(long long)L0 * kTraceSlots + 232] = smid;
        args.trace[(long long)L0 * kTraceSlots + 233] = (long long)global_ns();
    }

    BlockDesc bd0;
    describe_block(L0, args, bd0);
    auto issue_q = [&](const BlockDesc &bd) {
        mbar_expect_tx(bar(C::B_Q), C::Q_BYTES);
        for (int dc = 0; dc < C::KD; ++dc)
            tma_load_3d_hint(sQ + dc * C::Q_DBLK, &tmQ, dc * 64, bd.p0 - s.qoff, bd.b * s.H + bd.h0, bar(C::B_Q),
                             policy_evict_first());
    };

    // ---- Q of the first block first: its load is the longest wait of the set-up
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmQ);
        mbar_init(bar(C::B_Q), 1u);
        fence_barrier_init();
        issue_q(bd0);
        stamp(2);
    }

    // ---- setup: barriers (spread over warp 0's lanes), TMEM
    if (warp == 0) {
        for (int idx = lane; idx < C::NBARS; idx += 32)
            if (idx != C::B_Q) mbar_init(bar(idx), C::counts128(idx) ? 128u : 1u);
        if (lane == 0) *abort_flag = 0u;
        fence_barrier_init();
        __syncwarp();
    }
    // K or V tile t of block bd into stage st of its ring (the stage must be free)
    auto issue_kv = [&](const CUtensorMap *tm, uint32_t sbuf, int full_bar, const BlockDesc &bd, int t, int st,
                        uint64_t policy) {
        mbar_expect_tx(bar(full_bar + st), C::KD * BOX_BYTES);
        int back;
        bool sk;
        const int key0 = bd.cw.key0(t, back, sk);
        for (int dc = 0; dc < C::KD; ++dc)
            tma_load_3d_hint(sbuf + st * C::KV_STAGE + dc * C::KV_DBLK, tm, dc * 64, key0, bd.b * s.Hkv + bd.g,
                             bar(full_bar + st), policy);
    };
    // With the fused gate a block's first tile holds the W1 rows of its heads (32 rows of the
    // [H * 8, d] bf16 matrix from row h0 * 8: its S product is the heads' hidden
    // pre-activations); its key tiles follow, shifted by one.
    constexpr int G0 = GATE ? 1 : 0;
    auto issue_k = [&](const BlockDesc &bd, int t, int st, uint64_t policy) {
        if (GATE && t == 0) {
            mbar_expect_tx(bar(C::B_KF + st), C::KD * BOX_BYTES);
            for (int dc = 0; dc < C::KD; ++dc)
                tma_load_3d_hint(sK + st * C::KV_STAGE + dc * C::KV_DBLK, &tmW, dc * 64, bd.h0 * kGateHidden, 0,
                                 bar(C::B_KF + st), policy);
        } else {
            issue_kv(&tmK, sK, C::B_KF, bd, t - G0, st, policy);
        }
    };
    // The first K tile, which the first S = Q K^T waits for, goes out before the CTA barrier, so
    // that its latency overlaps the TMEM allocation and the barrier itself.
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmK);
        if (GATE) prefetch_tmap(&tmW);
        stamp_tile(8, 0);
        issue_k(bd0, 0, 0, policy_evict_last());
    }
    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;
    if (threadIdx.x == 0) {
        stamp(1);
        if (traced) args.trace[(long long)L0 * kTraceSlots + 7] = bd0.n_tiles;
    }

    if (warp == 0) {
        // ================= producer: K tiles of every block, after the first
        if (lane == 0) {
            const uint64_t reused = policy_evict_last();
            uint32_t gk = 1;  // tiles counted across blocks; tile 0 is out already
            bool ok = true;
            for (int L = L0; ok && L < args.n_blocks; L = next_block(L)) {
                BlockDesc bd;
                describe_block(L, args, bd);
                for (int t = (L == L0) ? 1 : 0; t < bd.n_tiles + G0; ++t, ++gk) {
                    const int st = (int)(gk % KST);
                    const uint32_t round = gk / KST;
                    if (round > 0 && !wait_bar(bar(C::B_KE + st), (round - 1) & 1, wc)) {
                        ok = false;
                        break;
                    }
                    if (L == L0) stamp_tile(8, t);
                    issue_k(bd, t, st, reused);
                }
            }
            if (*abort_flag) {  // let loads in flight land before the CTA leaves
                volatile uint32_t zero = 0;
                WaitCtx w2{&zero, nullptr, 20000000ull};
                for (uint32_t g = (gk > KST ? gk - KST : 0); g < gk; ++g)
                    wait_bar(bar(C::B_KF + (int)(g % KST)), (g / KST) & 1, w2);
            }
        }
    } else if (warp == 2) {
        // ================= producer: V tiles; the TMA store of each block's staged output; the
        // next block's Q tile.  At V tile t_st of block k (t_st = min(4, tiles - 1)) the output
        // of block k-1 is staged (its PV products finished long ago), so it is stored from the
        // shared buffer, and once that store has read the buffer the Q tile of block k+1 takes
        // its place (the Q tile of block k was copied into TMEM before the output was staged).
        if (lane == 0) {
            prefetch_tmap(&tmV);
            prefetch_tmap(&tmO);
            const uint64_t reused = policy_evict_last(), stream_once = policy_evict_first();
            uint32_t gv = 0;
            int k = 0, q_loads = 1;  // Q tiles loaded so far (the first by thread 0)
            bool ok = true;
            BlockDesc prev;
            auto store_out = [&](const BlockDesc &bd, int kb) -> bool {
                if (!wait_bar(bar(C::B_STF), (uint32_t)(kb & 1), wc)) return false;
                for (int dc = 0; dc < C::KD; ++dc)
                    tma_store_3d(&tmO, sQ + dc * C::Q_DBLK, dc * 64, bd.p0 - s.qoff, bd.b * s.H + bd.h0,
                                 stream_once);
                tma_store_commit_and_wait();
                mbar_arrive(bar(C::B_STR));
                return true;
            };
            for (int L = L0; ok && L < args.n_blocks; L = next_block(L), ++k) {
                BlockDesc bd;
                describe_block(L, args, bd);
                const int t_st = min(4, bd.n_tiles - 1);
                for (int t = 0; t < bd.n_tiles; ++t, ++gv) {
                    const int st = (int)(gv % VST);
                    const uint32_t round = gv / VST;
                    if (round > 0 && !wait_bar(bar(C::B_VE + st), (round - 1) & 1, wc)) {
                        ok = false;
                        break;
                    }
                    if (k == 0) stamp_tile(24, t);
                    issue_kv(&tmV, sV, C::B_VF, bd, t, st, reused);
                    if (t == t_st) {
                        if (k > 0 && !store_out(prev, k - 1)) {
                            ok = false;
                            break;
                        }
                        if (L < args.n_blocks - LS) {
                            // the Q tile of block k is in TMEM, and the buffer is free
                            if (!wait_bar(bar(C::B_QT), (uint32_t)(k & 1), wc)) {
                                ok = false;
                                break;
                            }
                            BlockDesc nx;
                            describe_block(L + LS, args, nx);  // L + LS < n_blocks
                            issue_q(nx);
                            ++q_loads;
                        }
                    }
                }
                prev = bd;
            }
            if (ok && k > 0) ok = store_out(prev, k - 1);  // the CTA's last block
            if (*abort_flag) {
                volatile uint32_t zero = 0;
                WaitCtx w2{&zero, nullptr, 20000000ull};
                wait_bar(bar(C::B_Q), (uint32_t)((q_loads - 1) & 1), w2);
                for (uint32_t g = (gv > VST ? gv - VST : 0); g < gv; ++g)
                    wait_bar(bar(C::B_VF + (int)(g % VST)), (g / VST) & 1, w2);
                tma_store_commit_and_wait();
            }
        }
    } else if (warp == 1) {
        // ================= S issuer: S = Q K^T into the tile's TMEM buffer, Q (A operand) read
        // from TMEM and the K tile (B operand) from shared memory.  It runs ahead of the PV
        // issuer, so that a PV never waits behind a K tile still in flight.  The whole warp runs
        // the loop and its waits, so that descriptors and TMEM addresses are warp-uniform; one
        // elected lane issues the MMAs and the commits.
        const uint32_t aQ = tbase + C::Q_COL;
        const uint32_t idesc = idesc_bf16(BM, CHUNK, 0, 0);
        uint32_t gs = 0;
        int k = 0;
        bool ok = true;
        for (int L = L0; ok && L < args.n_blocks; L = next_block(L), ++k) {
            BlockDesc bd;
            describe_block(L, args, bd);
            // The block's Q tile into TMEM, as the A operand of its S products: once the previous
            // block's S products are done with the old one, and the tile has landed in shared
            // memory, one copy per 16 elements of d; the S products below execute after them.
            bool w = (k == 0) || wait_bar(bar(C::B_SD), (uint32_t)((k - 1) & 1), wc);
            if (w) w = wait_bar(bar(C::B_Q), (uint32_t)(k & 1), wc);
            ok = __all_sync(0xffffffffu, w);
            if (!ok) break;
            tc_fence_after();
            if (elect_one()) {
                const uint64_t q0 = sdesc(sQ, 16, 1024);
#pragma unroll
                for (int dc = 0; dc < C::KD; ++dc)
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        tmem_cp_128x256b(aQ + (dc * 4 + ks) * 8, q0 + (uint64_t)((dc * C::Q_DBLK + ks * 32) >> 4));
                tc_commit(bar(C::B_QT));  // the shared buffer is read once the copies are done
            }
            __syncwarp();
            if (k == 0 && lane == 0) stamp(3);
            for (int t = 0; t < bd.n_tiles + G0; ++t, ++gs) {
                const int st = (int)(gs % KST), buf = (int)(gs % NB);
                bool w = timed_wait(bar(C::B_KF + st), (gs / KST) & 1, 104, t);
                // buffer buf last held P of tile gs - NB: its PV must be done
                if (w && gs >= NB) w = timed_wait(bar(C::B_PV + buf), ((gs - NB) / NB) & 1, 120, t);
                if (!__all_sync(0xffffffffu, w)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t dS = tbase + buf * CHUNK;
                const uint64_t b0 = sdesc(sK + st * C::KV_STAGE, 16, 1024);
                if (elect_one()) {
#pragma unroll
                    for (int dc = 0; dc < C::KD; ++dc) {
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            // k-step dc*4 + ks: 16 elements of d, 8 TMEM columns of bf16 pairs;
                            // the start address field of the K descriptor counts 16-byte units
                            const uint64_t bb = b0 + (uint64_t)((dc * C::KV_DBLK + ks * 32) >> 4);
                            mma_ts(dS, aQ + (dc * 4 + ks) * 8, bb, idesc, (dc | ks) != 0);
                        }
                    }
                    tc_commit(bar(C::B_SF + buf));
                    tc_commit(bar(C::B_KE + st));
                    if (t == bd.n_tiles + G0 - 1) tc_commit(bar(C::B_SD));
                }
                __syncwarp();
                if (k == 0 && lane == 0) stamp_tile(40, t);
            }
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
        const uint32_t idesc = idesc_bf16(BM, D, 0, 1);
        uint32_t gp = 0, gv = 0;  // tiles (S buffers) and V tiles, counted across blocks
        int k = 0;
        bool ok = true;
        for (int L = L0; ok && L < args.n_blocks; L = next_block(L), ++k) {
            BlockDesc bd;
            describe_block(L, args, bd);
            for (int u = 0; u < bd.n_tiles + G0; ++u, ++gp) {
                const int buf = (int)(gp % NB);
                if (GATE && u == 0) {
                    // the gate tile has no PV product: its buffer is free once the row threads
                    // have read it (a commit with nothing new behind it)
                    const bool w = wait_bar(bar(C::B_PR + buf), (gp / NB) & 1, wc);
                    if (!__all_sync(0xffffffffu, w)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (elect_one()) tc_commit(bar(C::B_PV + buf));
                    __syncwarp();
                    continue;
                }
                const int st = (int)(gv % VST);
                bool w = timed_wait(bar(C::B_PR + buf), (gp / NB) & 1, 136, u);
                if (w) w = timed_wait(bar(C::B_VF + st), (gv / VST) & 1, 152, u);
                if (!__all_sync(0xffffffffu, w)) {
                    ok = false;
                    break;
                }
                ++gv;
                tc_fence_after();
                const uint32_t aP = tbase + buf * CHUNK;
                const uint64_t b0 = sdesc(sV + st * C::KV_STAGE, C::KV_DBLK, 1024);
                if (elect_one()) {
                    // the block's first product overwrites O (the previous block's epilogue read
                    // it before this block's first P was marked ready)
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)
                        mma_ts(tbase + C::O_COL, aP + kk * 8, b0 + (uint64_t)((kk * 16 * ROW_BYTES) >> 4), idesc,
                               (u > G0 || kk > 0) ? 1u : 0u);
                    tc_commit(bar(C::B_PV + buf));
                    tc_commit(bar(C::B_VE + st));
                    if (u == bd.n_tiles + G0 - 1) tc_commit(bar(C::B_OF));
                }
                __syncwarp();
                if (k == 0 && lane == 0) stamp_tile(56, u);
            }
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
        const int R = args.R;
        const int hh = r >> (5 + args.cpb_log2), trow = r & (R - 1);  // R = 32 << cpb_log2
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        const float sc = s.scale_log2;

        // This row's input alpha in block L (1 where none is given or the row is past the
        // window; the fused gate's comes from the block's gate tile).  Each block's alpha is
        // prefetched into L2 two blocks ahead and loaded one block ahead.
        const bool use_alpha = !GATE && args.alpha != nullptr;
        auto alpha_ptr = [&](int L) -> const float * {
            const int rest = args.div_nqb.div(L);
            const int bn = args.div_ngrp.div(rest);
            const int in = (L - rest * args.nqb) * R + trow;
            if (!use_alpha || in >= s.nq) return nullptr;
            return args.alpha + ((long long)bn * s.H + (rest - bn * args.ngrp) * args.GP + hh) * s.nq + in;
        };
        const float *pa0 = alpha_ptr(L0);
        float al_next = pa0 ? *pa0 : 1.f;
        if (L0 < args.n_blocks - LS) {
            const float *pa = alpha_ptr(L0 + LS);
            if (pa) prefetch_l2(pa);
        }
        bool ok = true;
        uint32_t gsm = 0;
        int k = 0;
        for (int L = L0; ok && L < args.n_blocks; L = next_block(L), ++k) {
            BlockDesc bd;
            describe_block(L, args, bd);
            const bool has_next = L < args.n_blocks - LS;
            const int i = bd.p0 + trow, h = bd.h0 + hh, iq = i - s.qoff;
            const bool row_ok = iq < s.nq;
            const long long row_g = ((long long)bd.b * s.H + h) * s.nq + iq;
            float al = al_next;  // the fused gate sets it at the block's first tile
            if (has_next) {      // L + LS < n_blocks
                const float *pa = alpha_ptr(L + LS);
                al_next = pa ? *pa : 1.f;
            }
            if (L < args.n_blocks - 2 * LS) {
                const float *pa = alpha_ptr(L + 2 * LS);
                if (pa) prefetch_l2(pa);
            }
            float off_band = (s.mode != kModeEcp) ? log2f(al) : 0.f;
            float off_skip = log2f(1.f - al);
            const int lo_i = band_lo(i, s.mode, s.k_local);
            const int hi_i = band_hi(i, s.N, s.mode, s.k_local);
            float lse2_in = 0.f;
            if (DBG == 2) lse2_in = row_ok ? args.lse_in[row_g] * kLog2e : -INFINITY;

            float m_ref = -INFINITY, l = 0.f;
            long long cnt = 0, isum = 0;
            for (int t = 0; t < bd.n_tiles + G0; ++t, ++gsm) {
                const int buf = (int)(gsm % NB);
                if (DBG == 3 && warp == 4 && lane == 0) ok = timed_wait(bar(C::B_SF + buf), (gsm / NB) & 1, 168, t);
                else ok = wait_bar(bar(C::B_SF + buf), (gsm / NB) & 1, wc);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                if (k == 0 && warp == 4 && lane == 0) stamp_tile(72, t);
                tc_fence_after();
                __syncwarp();
                if (GATE && t == 0) {
                    // the gate tile: this row's head's 8 hidden pre-activations, then alpha
                    uint32_t pre[kGateHidden];
                    tmem_ld8(tbase + lane_base + buf * CHUNK + hh * kGateHidden, pre);
                    tmem_wait_ld();
                    tc_fence_before();
                    mbar_arrive(bar(C::B_PR + buf));  // the buffer is free for the next S
                    al = gate_alpha(pre, args.gate_b1 + h * kGateHidden, args.gate_w2 + h * kGateHidden,
                                    args.gate_b2[h]);
                    if (args.alpha_out && row_ok) args.alpha_out[row_g] = al;
                    off_band = log2f(al);
                    off_skip = log2f(1.f - al);
                    continue;
                }
                const int tk = t - G0;  // key tile of the block
                const uint32_t tS = tbase + lane_base + buf * CHUNK;
                uint32_t ra[CHUNK];
                tmem_ld32(tS, ra);
                tmem_wait_ld();
                if (k == 0 && warp == 4 && lane == 0) stamp_tile(184, t);

                // Full tile (the same for every thread of the CTA): P with the running reference;
                // the maximum is only needed when some P exceeds 2^8 (the lazy-rescale bound),
                // which a sum above 2^8 is the first sign of.  Rows with no reference yet take the
                // general path, as do the debug modes that record per-row ranges.
                const bool fast = (DBG == 0 || DBG == 3) && tk >= bd.full_lo && tk <= bd.full_hi &&
                                  __all_sync(0xffffffffu, m_ref != -INFINITY);
                float corr = 1.f, lsum, bo;
                bool need_o = false, diag = false;
                int clo = 0;
                float zdiag = 0.f, mu = 0.f;
                if (fast) {
                    bo = off_band - m_ref;
                } else {
                    int back, chi;
                    bool sk;
                    const int key0 = bd.cw.key0(tk, back, sk);
                    float off;
                    if (!sk) {
                        clo = max(lo_i - key0, 0);
                        chi = min(hi_i - key0, CHUNK - 1);
                        off = off_band;
                    } else {
                        const int jk = i - back, c = jk - key0;
                        if (jk >= 0 && jk < s.N && c >= 0 && c < CHUNK) { clo = c; chi = c; }
                        else { clo = CHUNK; chi = -1; }
                        off = off_skip;
                    }
                    float *fa = reinterpret_cast<float *>(ra);
                    const float mt = tile_max(fa, clo, chi, sk, sc, off);
                    if (k == 0 && warp == 4 && lane == 0) stamp_tile(200, t);
                    if (mt > m_ref + kRescaleThreshold) {
                        if (m_ref != -INFINITY) {
                            corr = fast_exp2(m_ref - mt);
                            need_o = (tk > 0);
                        }
                        m_ref = mt;
                    }
                    l *= corr;
                    mu = (m_ref == -INFINITY) ? 0.f : m_ref;
                    bo = off - mu;
                    diag = sk;
                    zdiag = mt;
                    if (DBG == 1) {
                        const int na = max(0, chi - clo + 1);
                        cnt += na;
                        isum += (long long)na * key0 + (long long)(clo + chi) * na / 2;
                    }
                    if (DBG == 2 && row_ok && lse2_in != -INFINITY) {
                        for (int c = 0; c < CHUNK; ++c)
                            if (c >= clo && c <= chi)
                                args.P[row_g * s.N + key0 + c] = exp2f(fmaf(fa[c], sc, off - lse2_in));
                    }
                }
                if (diag) {
                    lsum = tile_exp_diag(ra, clo, zdiag, mu);
                } else {
                    // one copy of the exponentials: on the fast path, a second pass only when the
                    // first found P above the lazy-rescale bound (S is still in TMEM)
#pragma unroll 1
                    for (int pass = 0;; ++pass) {
                        lsum = tile_exp(ra, sc, bo);
                        if (!fast || pass > 0 || !__any_sync(0xffffffffu, !(lsum <= 256.f))) break;
                        tmem_ld32(tS, ra);
                        tmem_wait_ld();
                        const float mt = fmaf(tile_raw_max(ra), sc, off_band);
                        if (mt > m_ref + kRescaleThreshold) {
                            corr = fast_exp2(m_ref - mt);
                            need_o = true;  // m_ref was set by an earlier tile, so t > 0
                            m_ref = mt;
                        }
                        l *= corr;
                        bo = off_band - m_ref;
                    }
                }
                if (fast && k == 0 && warp == 4 && lane == 0) stamp_tile(200, t);
                tmem_st16(tS, ra);  // P as bf16 pairs over the tile's first 16 S columns
                if (k == 0 && warp == 4 && lane == 0) stamp_tile(216, t);
                l += lsum;
                __syncwarp();
                // Rescale this row of O when the reference max moved (tile t > 0 of the block).
                // PV of the previous tile must be done.  The wait names that phase exactly: S of
                // the previous tile implied PV of the tile before it finished, and the next PV
                // cannot start before this thread marks the next P ready.
                if (__any_sync(0xffffffffu, need_o)) {
                    const bool r_ = wait_bar(bar(C::B_PV + (int)((gsm - 1) % NB)), ((gsm - 1) / NB) & 1, wc);
                    if (!__all_sync(0xffffffffu, r_)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const float f = need_o ? corr : 1.f;
#pragma unroll 1
                    for (int oc = 0; oc < D / 16; ++oc) {
                        uint32_t x[16];
                        tmem_ld16(tbase + lane_base + C::O_COL + oc * 16, x);
                        tmem_wait_ld();
#pragma unroll
                        for (int c = 0; c < 16; ++c) x[c] = __float_as_uint(__uint_as_float(x[c]) * f);
                        tmem_st16(tbase + lane_base + C::O_COL + oc * 16, x);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(C::B_PR + buf));
                if (k == 0 && warp == 4 && lane == 0) stamp_tile(88, t);
            }

            // ---- epilogue: O / l -> bf16 -> shared (swizzled) -> TMA store by warp 2.  A parity
            // wait names a phase only if the barrier is at most one phase away from it; by now
            // the PV barrier may be anywhere from n_tiles-2 to n_tiles phases along, so the
            // epilogue waits on the block's O barrier.  The staging buffer holds the previous
            // block's output until warp 2's store has read it, and then the next block's Q tile
            // until the S issuer's copies into TMEM have read it.  (That copy's barrier is one
            // phase on from this block's, which had completed before this block's S products:
            // the copies execute ahead of them.)
            if (ok) ok = __all_sync(0xffffffffu, wait_bar(bar(C::B_OF), (uint32_t)(k & 1), wc));
            if (ok && k > 0) ok = __all_sync(0xffffffffu, wait_bar(bar(C::B_STR), (uint32_t)((k - 1) & 1), wc));
            if (ok && has_next) ok = __all_sync(0xffffffffu, wait_bar(bar(C::B_QT), (uint32_t)((k + 1) & 1), wc));
            if (k == 0 && warp == 4 && lane == 0) stamp(4);
            if (!ok) break;
            const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
            tc_fence_after();
            __syncwarp();
#pragma unroll 1
            for (int oh = 0; oh < D / 32; oh += 2) {  // 64 fp32 columns per TMEM round trip
                uint32_t x[64];
                tmem_ld32(tbase + lane_base + C::O_COL + oh * 32, x);
                tmem_ld32(tbase + lane_base + C::O_COL + oh * 32 + 32, x + 32);
                tmem_wait_ld();
                uint8_t *rowp = smem + C::Q_OFF + (oh >> 1) * C::Q_DBLK + r * ROW_BYTES;
#pragma unroll
                for (int w = 0; w < 8; ++w) {  // 8 columns -> one 16-byte chunk of the row
                    const float *f = reinterpret_cast<const float *>(x) + 8 * w;
                    const uint4 val = make_uint4(pack_bf16(f[0] * inv_l, f[1] * inv_l), pack_bf16(f[2] * inv_l, f[3] * inv_l),
                                                 pack_bf16(f[4] * inv_l, f[5] * inv_l), pack_bf16(f[6] * inv_l, f[7] * inv_l));
                    *reinterpret_cast<uint4 *>(rowp + ((w ^ (r & 7)) << 4)) = val;
                }
            }
            // O is read: the next block's first PV may overwrite it once this thread marks that
            // block's first P ready (program order).
            fence_proxy_async_smem();
            mbar_arrive(bar(C::B_STF));
            if (k == 0 && warp == 4 && lane == 0) stamp(5);
            if (row_ok) {
                args.lse[row_g] = (l > 0.f) ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
                if (DBG == 1) {
                    args.cnt[row_g] = (int)cnt;
                    args.isum[row_g] = isum;
                }
            }
        }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && traced) {
        stamp(6);
        args.trace[(long long)L0 * kTraceSlots + 234] = (long long)global_ns();
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

template <int D, int DBG, bool GATE = false>
static cudaError_t launch(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                          const CUtensorMap &mo, const CUtensorMap &mw, const TcArgs &a, unsigned grid,
                          cudaStream_t st) {
    constexpr int smem = Cfg<D>::SMEM_BYTES;
    static PerDeviceOnce configured;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured.needed(dev)) {
        cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel<D, DBG, GATE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured.mark(dev);
    }
    fwd_tc_kernel<D, DBG, GATE><<<grid, NUM_THREADS, smem, st>>>(mq, mk, mv, mo, mw, a);
    return cudaGetLastError();
}

// Streaming multiprocessors of the current device (looked up once per device).
static int sm_count() {
    constexpr int kMaxDev = 64;
    static std::atomic<int> cache[kMaxDev];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
    int n = cache[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

}  // namespace tc

cudaError_t launch_fwd_tc(const LaunchFwd &L, cudaStream_t st) {
    using namespace tc;
    const Shape &s = L.s;
    const int G = s.H / s.Hkv;
    const int GP = (G % 4 == 0) ? 4 : (G % 2 == 0) ? 2 : 1;
    const int R = BM / GP;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, L.q, s.d, s.nq, (long long)s.B * s.H, R, GP) ||
        !make_map(&mo, L.out, s.d, s.nq, (long long)s.B * s.H, R, GP) ||
        !make_map(&mk, L.k, s.d, s.N, (long long)s.B * s.Hkv, CHUNK, 1) ||
        !make_map(&mv, L.v, s.d, s.N, (long long)s.B * s.Hkv, CHUNK, 1))
        return cudaErrorNotSupported;
    const int m_first = (s.mode != kModeEcp && s.S > 0) ? first_skip_multiple(s) : 1;
    const int nqb = (s.nq + R - 1) / R, ngrp = s.H / GP;
    const long long nb64 = (long long)nqb * ngrp * s.B;
    if (nb64 > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const int n_blocks = (int)nb64;
    const int cpb_log2 = (R == 128) ? 2 : (R == 64) ? 1 : 0;
    TcArgs a{L.alpha, L.lse, s, GP, m_first, nqb, ngrp, R, cpb_log2, make_fastdiv(nqb), make_fastdiv(ngrp),
             make_fastdiv(G), make_fastdiv(s.S > 0 && s.period > 0 ? s.period : 1), n_blocks, L.status,
             L.timeout_ns, L.cnt, L.isum, L.lse_in, L.P, L.trace, L.n_trace, L.gate_b1, L.gate_w2,
             L.gate_b2, L.alpha_out};
    // The forward runs persistent, two CTAs per SM; the debug modes take one CTA per block.
    unsigned grid = (unsigned)n_blocks;
    if (L.dbg == 0) {
        const int resident = 2 * sm_count();
        if (resident > 0 && resident < n_blocks) grid = (unsigned)resident;
    }
    if (L.gate_w1) {  // the fused gate: the forward only
        if (L.dbg != 0) return cudaErrorInvalidValue;
        CUtensorMap mw;  // W1 as [1][H * kGateHidden][d]: a block's heads are 32 (or fewer) rows
        if (!make_map(&mw, L.gate_w1, s.d, s.H * kGateHidden, 1, CHUNK, 1)) return cudaErrorNotSupported;
        if (s.d == 64) return launch<64, 0, true>(mq, mk, mv, mo, mw, a, grid, st);
        if (s.d == 128) return launch<128, 0, true>(mq, mk, mv, mo, mw, a, grid, st);
        return cudaErrorInvalidValue;
    }
    if (s.d == 64) {
        if (L.dbg == 0) return launch<64, 0>(mq, mk, mv, mo, mk, a, grid, st);
        if (L.dbg == 1) return launch<64, 1>(mq, mk, mv, mo, mk, a, grid, st);
        if (L.dbg == 3) return launch<64, 3>(mq, mk, mv, mo, mk, a, grid, st);
        return launch<64, 2>(mq, mk, mv, mo, mk, a, grid, st);
    }
    if (s.d == 128) {
        if (L.dbg == 0) return launch<128, 0>(mq, mk, mv, mo, mk, a, grid, st);
        if (L.dbg == 1) return launch<128, 1>(mq, mk, mv, mo, mk, a, grid, st);
        if (L.dbg == 3) return launch<128, 3>(mq, mk, mv, mo, mk, a, grid, st);
        return launch<128, 2>(mq, mk, mv, mo, mk, a, grid, st);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_wait_timeout_probe(int *status, uint64_t timeout_ns, cudaStream_t st) {
    tc::wait_timeout_probe_kernel<<<1, 32, 0, st>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace pi
