// pi_bwd_tc.cu -- backward of the fused pi-Attention / ECP attention on sm_103a tensor cores.
//
// The chain rule through the forward's definition ("pi-Attention: Periodic Sparse
// Transformers for Efficient Long-Context Modeling", section 2.1-2.3; ECP page section 2):
//   p_ij = exp(z_ij - lse_i),  dp_ij = dout_i . v_j,  D_i = sum_j p_ij dp_ij,
//   dz_ij = p_ij (dp_ij - D_i),
//   dq_i = tau sum_j dz_ij k_j = tau (sum_j p_ij (dp_ij - c_i) k_j - (D_i - c_i) sum_j p_ij k_j)
//          for any per-row constant c_i,
//   dk_j = tau sum_{h in group, i} dz_ij q_i,  dv_j = sum_{h in group, i} p_ij dout_i,
//   dalpha_i = -(sum_{j in P(i)} dz_ij) / (alpha_i (1 - alpha_i)).
//
// Kernel 1 (query-major, one CTA per 128 query rows laid out as in the forward):
//   per key tile, S = Q K^T and dP = dO V^T into TMEM; one thread per row forms p and p*dp,
//   keeps D_i and the skip sums of dalpha in registers and writes p and p (dp - c) (bf16)
//   back to TMEM; two MMAs accumulate A1 = sum p (dp - c) K and A2 = sum p K.  The epilogue
//   writes dq = tau (A1 - (D - c) A2), D_i (for kernel 2) and dalpha.  One sweep over the
//   keys, and D_i is exact: it never goes through the bf16-rounded out.  The centre c_i is
//   dout_i . out_i from the bf16 out, within rounding of D_i, so that the bf16 operand of A1
//   carries dz itself rather than p dp, whose cancellation against D A2 would cost accuracy.
// Kernel 2 (key-major, one CTA per 128 keys of a KV head): for every 64-query chunk of every
//   query head of the group whose band contains these keys, and every chunk of skip queries
//   j + m*period: S^T = K Q^T and dP^T = V dO^T into TMEM; one thread per key forms p and dz
//   with the chunk's per-query bias (prior - lse) and D, writes them (bf16) back to TMEM; two
//   MMAs accumulate dV += P^T dO and dK += dZ^T Q.  No atomics: deterministic.
#include <algorithm>

#include "pi_common.cuh"
#include "pi_launch.h"
#include "pi_tc_ptx.cuh"

namespace pi {
namespace tcb {

using namespace tc;

constexpr int BM = 128;     // rows per CTA (MMA M)
constexpr int CHUNK = 32;   // keys per chunk (TMA box rows)
constexpr int NUM_THREADS = 256;
constexpr int ROW_BYTES = 128;
constexpr int BOX_BYTES = CHUNK * ROW_BYTES;

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
        : "memory");
}

// Key chunk walk of a q-block: identical enumeration to the forward kernel's.  Skip blocks
// follow the band: first the n_back blocks of keys i - m*period, then (bidirectional mode)
// those of keys i + m*period, both for m = m_first, m_first + 1, ...; `back` is the distance
// i - key of the chunk's keys (negative for keys after the query).
struct QWalk {
    int lo0, n_band, m_first, cpb, cpb_log2, p0, period, n_back;
    __device__ __forceinline__ int key0(int ci, int &back, bool &skip) const {
        if (ci < n_band) {
            back = 0;
            skip = false;
            return lo0 + ci * CHUNK;
        }
        const int sc = ci - n_band;
        const int blk = sc >> cpb_log2;
        const int u = sc & (cpb - 1);
        back = (blk < n_back) ? (m_first + blk) * period : -(m_first + blk - n_back) * period;
        skip = true;
        return p0 - back + u * CHUNK;
    }
};

template <int D>
struct CfgQ {
    static constexpr int KD = D / 64;
    static constexpr int CPT = (D == 64) ? 1 : 2;  // chunks per key tile
    static constexpr int TILE = CPT * CHUNK;
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int Q_DBLK = BM * ROW_BYTES;
    static constexpr int KV_STAGE = TILE * D * 2;
    static constexpr int KV_DBLK = TILE * ROW_BYTES;
    static constexpr int ST = 32768 / KV_STAGE;  // 32 KB of K tiles and 32 KB of V tiles
    static constexpr int Q_OFF = 0;
    static constexpr int G_OFF = Q_BYTES;  // dO tile
    static constexpr int K_OFF = 2 * Q_BYTES;
    static constexpr int V_OFF = K_OFF + ST * KV_STAGE;
    static constexpr int BAR_OFF = V_OFF + ST * KV_STAGE;
    static constexpr int B_QF = 0;
    static constexpr int B_KF = 1;
    static constexpr int B_KE = B_KF + ST;
    static constexpr int B_VF = B_KE + ST;
    static constexpr int B_VE = B_VF + ST;
    // Two S/dP buffers in TMEM: tile t uses buffer t & 1.  Per buffer: S and dP written by the
    // MMAs, then p (dp - c) and p written back over them for the A1/A2 MMAs.
    static constexpr int B_SF = B_VE + ST;  // [2] S and dP of the tile in TMEM
    static constexpr int B_PR = B_SF + 2;   // [2] p and p (dp - c) written back (128 arrivals)
    static constexpr int B_BF = B_PR + 2;   // [2] A1/A2 MMAs of the tile done: buffer free
    static constexpr int B_AF = B_BF + 2;   // A1/A2 complete (single phase)
    static constexpr int B_DR = B_AF + 1;   // drain of the S/dP issuer
    static constexpr int B_DR2 = B_DR + 1;  // drain of the A1/A2 issuer
    static constexpr int NBARS = B_DR2 + 1;
    static constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16 + 1024;
    // TMEM columns
    static constexpr int BUF = 2 * TILE;  // S then dP of one buffer
    static constexpr int S_COL = 0, DP_COL = TILE, A1_COL = 2 * BUF, A2_COL = 2 * BUF + D;
    static constexpr int TMEM_COLS = (A2_COL + D <= 256) ? 256 : 512;
};

struct DqArgs {
    const __nv_bfloat16 *out, *dout;  // rows of the forward output and its gradient (centre c_i)
    const float *alpha;
    const float *lse;
    float *Dws;
    float *dalpha;
    Shape s;
    int GP;
    int *status;
    uint64_t timeout_ns;
};

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmG,
                 const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const __grid_constant__ CUtensorMap tmDQ, const DqArgs args) {
    using C = CfgQ<D>;
    constexpr int ST = C::ST;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_addr + pad;
    const uint32_t sQ = sbase + C::Q_OFF, sG = sbase + C::G_OFF, sK = sbase + C::K_OFF,
                   sV = sbase + C::V_OFF, sBar = sbase + C::BAR_OFF;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::BAR_OFF + C::NBARS * 8);
    uint32_t *tmem_slot = misc;
    volatile uint32_t *abort_flag = misc + 1;
    auto bar = [&](int idx) -> uint32_t { return sBar + idx * 8; };

    const Shape &s = args.s;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const WaitCtx wc{abort_flag, args.status, args.timeout_ns};

    // ---- q-block coordinates and key chunks (as in the forward)
    const int GP = args.GP;
    const int R = BM / GP;
    const int nqb = (s.nq + R - 1) / R;
    const int hsub = s.H / GP;
    int bid = blockIdx.x;
    const int pb = bid % nqb;
    bid /= nqb;
    const int hs = bid % hsub;
    const int b = bid / hsub;
    const int h0 = hs * GP;
    const int g = h0 / (s.H / s.Hkv);
    const int p0 = s.qoff + pb * R;  // key position of the block's first query row
    QWalk cw;
    cw.p0 = p0;
    cw.period = s.period;
    cw.cpb = R / CHUNK;
    cw.cpb_log2 = (cw.cpb == 4) ? 2 : (cw.cpb == 2) ? 1 : 0;
    cw.lo0 = band_lo(p0, s.mode, s.k_local);
    cw.n_band = (band_hi(min(s.N - 1, p0 + R - 1), s.N, s.mode, s.k_local) - cw.lo0) / CHUNK + 1;
    int n_skip_blocks = 0;
    cw.m_first = 1;
    cw.n_back = 0;
    if (s.mode != kModeEcp && s.S > 0) {
        cw.m_first = first_skip_multiple(s);
        const int m_last = min(s.S, (p0 + R - 1) / s.period);  // some row has i - m*period >= 0
        cw.n_back = max(0, m_last - cw.m_first + 1);
        n_skip_blocks = cw.n_back;
        if (s.mode == kModeBidir) {
            const int m_last_f = min(s.S, (s.N - 1 - p0) / s.period);  // some row has i + m*period < N
            n_skip_blocks += max(0, m_last_f - cw.m_first + 1);
        }
    }
    const int n_chunks = cw.n_band + n_skip_blocks * cw.cpb;
    constexpr int CPT = C::CPT;
    const int n_tiles = (n_chunks + CPT - 1) / CPT;

    if (warp == 0) {  // barriers spread over warp 0's lanes; only the P-ready ones count 128
        for (int idx = lane; idx < C::NBARS; idx += 32)
            mbar_init(bar(idx), (idx == C::B_PR || idx == C::B_PR + 1) ? 128u : 1u);
        if (lane == 0) *abort_flag = 0u;
        fence_barrier_init();
        __syncwarp();
    }
    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    if (warp == 0) {
        // ================= producer: Q, dO, K tiles
        if (lane == 0) {
            prefetch_tmap(&tmQ);
            prefetch_tmap(&tmG);
            prefetch_tmap(&tmK);
            const uint64_t once = policy_evict_first(), reused = policy_evict_last();
            mbar_expect_tx(bar(C::B_QF), 2 * C::Q_BYTES);
            for (int dc = 0; dc < C::KD; ++dc) {
                tma_load_3d_hint(sQ + dc * C::Q_DBLK, &tmQ, dc * 64, p0 - s.qoff, b * s.H + h0, bar(C::B_QF), once);
                tma_load_3d_hint(sG + dc * C::Q_DBLK, &tmG, dc * 64, p0 - s.qoff, b * s.H + h0, bar(C::B_QF), once);
            }
            int issued = 0;
            for (int t = 0; t < n_tiles; ++t) {
                const int st = t % ST, round = t / ST;
                if (round > 0 && !wait_bar(bar(C::B_KE + st), (round - 1) & 1, wc)) break;
                const int nch = min(CPT, n_chunks - CPT * t);
                mbar_expect_tx(bar(C::B_KF + st), nch * C::KD * BOX_BYTES);
                for (int cc = 0; cc < nch; ++cc) {
                    int back;
                    bool sk;
                    const int key0 = cw.key0(CPT * t + cc, back, sk);
                    for (int dc = 0; dc < C::KD; ++dc)
                        tma_load_3d_hint(sK + st * C::KV_STAGE + dc * C::KV_DBLK + cc * BOX_BYTES, &tmK,
                                         dc * 64, key0, b * s.Hkv + g, bar(C::B_KF + st), reused);
                }
                issued = t + 1;
            }
            if (*abort_flag) {
                volatile uint32_t zero = 0;
                WaitCtx w2{&zero, nullptr, 20000000ull};
                wait_bar(bar(C::B_QF), 0, w2);
                for (int t = max(0, issued - ST); t < issued; ++t)
                    wait_bar(bar(C::B_KF + t % ST), (t / ST) & 1, w2);
            }
        }
    } else if (warp == 2) {
        // ================= producer: V tiles
        if (lane == 0) {
            prefetch_tmap(&tmV);
            const uint64_t reused = policy_evict_last();
            int issued = 0;
            for (int t = 0; t < n_tiles; ++t) {
                const int st = t % ST, round = t / ST;
                if (round > 0 && !wait_bar(bar(C::B_VE + st), (round - 1) & 1, wc)) break;
                const int nch = min(CPT, n_chunks - CPT * t);
                mbar_expect_tx(bar(C::B_VF + st), nch * C::KD * BOX_BYTES);
                for (int cc = 0; cc < nch; ++cc) {
                    int back;
                    bool sk;
                    const int key0 = cw.key0(CPT * t + cc, back, sk);
                    for (int dc = 0; dc < C::KD; ++dc)
                        tma_load_3d_hint(sV + st * C::KV_STAGE + dc * C::KV_DBLK + cc * BOX_BYTES, &tmV,
                                         dc * 64, key0, b * s.Hkv + g, bar(C::B_VF + st), reused);
                }
                issued = t + 1;
            }
            if (*abort_flag) {
                volatile uint32_t zero = 0;
                WaitCtx w2{&zero, nullptr, 20000000ull};
                for (int t = max(0, issued - ST); t < issued; ++t)
                    wait_bar(bar(C::B_VF + t % ST), (t / ST) & 1, w2);
            }
        }
    } else if (warp == 1) {
        // ================= S/dP issuer: S = Q K^T and dP = dO V^T into buffer t & 1, as soon as
        // that buffer's previous A1/A2 MMAs (tile t-2) are done.  The whole warp runs the loop and
        // its waits (warp-uniform operands); one elected lane issues the MMAs and commits.
        bool ok = __all_sync(0xffffffffu, wait_bar(bar(C::B_QF), 0, wc));
        const uint64_t q0 = sdesc(sQ, 16, 1024), g0 = sdesc(sG, 16, 1024);
        for (int t = 0; ok && t < n_tiles; ++t) {
            const int st = t % ST, buf = t & 1;
            bool w = wait_bar(bar(C::B_KF + st), (t / ST) & 1, wc);
            if (w) w = wait_bar(bar(C::B_VF + st), (t / ST) & 1, wc);
            if (w && t >= 2) w = wait_bar(bar(C::B_BF + buf), ((t - 2) >> 1) & 1, wc);
            if (!__all_sync(0xffffffffu, w)) break;
            tc_fence_after();
            const int nch = min(CPT, n_chunks - CPT * t);
            const uint32_t idesc_s = idesc_bf16(BM, CHUNK * nch, 0, 0);
            const uint32_t dS = tbase + C::S_COL + buf * C::BUF, dP = tbase + C::DP_COL + buf * C::BUF;
            const uint64_t k0 = sdesc(sK + st * C::KV_STAGE, 16, 1024), v0 = sdesc(sV + st * C::KV_STAGE, 16, 1024);
            if (elect_one()) {
#pragma unroll
                for (int dc = 0; dc < C::KD; ++dc) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint32_t acc = (dc | ks) != 0;
                        // the start address field counts 16-byte units
                        const uint64_t oq = (uint64_t)((dc * C::Q_DBLK + ks * 32) >> 4);
                        const uint64_t okv = (uint64_t)((dc * C::KV_DBLK + ks * 32) >> 4);
                        mma_ss(dS, q0 + oq, k0 + okv, idesc_s, acc);
                        mma_ss(dP, g0 + oq, v0 + okv, idesc_s, acc);
                    }
                }
                tc_commit(bar(C::B_SF + buf));
                tc_commit(bar(C::B_VE + st));  // V is read by dP only
            }
            __syncwarp();
        }
        if (elect_one()) tc_commit(bar(C::B_DR));
        __syncwarp();
        volatile uint32_t zero = 0;
        WaitCtx w2{&zero, args.status, args.timeout_ns};
        wait_bar(bar(C::B_DR), 0, w2);
    } else if (warp == 3) {
        // ================= A1/A2 issuer: A1 += p (dp - c) K, A2 += p K from buffer t & 1 (whole
        // warp, one elected lane issuing)
        const uint32_t idesc_a = idesc_bf16(BM, D, 0, 1);
        for (int t = 0; t < n_tiles; ++t) {
            const int st = t % ST, buf = t & 1;
            // K of tile t landed before S of tile t, which the softmax saw before P
            if (!__all_sync(0xffffffffu, wait_bar(bar(C::B_PR + buf), (t >> 1) & 1, wc))) break;
            tc_fence_after();
            const int nch = min(CPT, n_chunks - CPT * t);
            const uint64_t k0 = sdesc(sK + st * C::KV_STAGE, C::KV_DBLK, 1024);
            if (elect_one()) {
                for (int kk = 0; kk < 2 * nch; ++kk) {
                    const uint64_t kb = k0 + (uint64_t)((kk * 16 * ROW_BYTES) >> 4);
                    const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
                    mma_ts(tbase + C::A1_COL, tbase + C::S_COL + buf * C::BUF + kk * 8, kb, idesc_a, acc);
                    mma_ts(tbase + C::A2_COL, tbase + C::DP_COL + buf * C::BUF + kk * 8, kb, idesc_a, acc);
                }
                tc_commit(bar(C::B_BF + buf));
                tc_commit(bar(C::B_KE + st));  // K is read by S and by A1/A2, which come last
                if (t == n_tiles - 1) tc_commit(bar(C::B_AF));
            }
            __syncwarp();
        }
        if (elect_one()) tc_commit(bar(C::B_DR2));
        __syncwarp();
        volatile uint32_t zero = 0;
        WaitCtx w2{&zero, args.status, args.timeout_ns};
        wait_bar(bar(C::B_DR2), 0, w2);
    } else if (warp >= 4) {
        // ================= one thread per query row
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;
        const int hh = r / R, trow = r % R;
        const int i = p0 + trow;
        const int h = h0 + hh;
        const bool row_ok = i - s.qoff < s.nq;
        const long long row_g = ((long long)b * s.H + h) * s.nq + (i - s.qoff);
        // the row's out (for the centre below) is loaded in the same round trip as its alpha
        // and lse; its dout is the staged dO tile's row
        uint4 orow_v[D / 8];
#pragma unroll
        for (int c = 0; c < D / 8; ++c)
            orow_v[c] = row_ok ? __ldg(reinterpret_cast<const uint4 *>(args.out + row_g * D) + c) : make_uint4(0u, 0u, 0u, 0u);
        const float al = (args.alpha && row_ok) ? args.alpha[row_g] : 1.f;
        const float off_band = (s.mode != kModeEcp) ? log2f(al) : 0.f;
        const float off_skip = log2f(1.f - al);
        const float lse2 = row_ok ? args.lse[row_g] * kLog2e : -INFINITY;
        const bool live = row_ok && lse2 != -INFINITY;
        const int lo_i = band_lo(i, s.mode, s.k_local);
        const int hi_i = band_hi(i, s.N, s.mode, s.k_local);
        const float sc = s.scale_log2;
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        float dsum = 0.f, skip_p = 0.f, skip_pdp = 0.f;
        bool any_skip = false;
        bool ok = true;
        // centre c_i = dout_i . out_i (bf16 rows); D_i itself is accumulated exactly below
        ok = __all_sync(0xffffffffu, wait_bar(bar(C::B_QF), 0, wc));  // the dO tile has landed
        float cen = 0.f;
        if (live) {
            const uint8_t *grow = smem + C::G_OFF + r * ROW_BYTES;
            uint64_t acc0 = pack2(0.f, 0.f), acc1 = pack2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {  // 8 elements per 16-byte chunk
                const uint4 gv = *reinterpret_cast<const uint4 *>(grow + (c >> 3) * C::Q_DBLK + (((c & 7) ^ (r & 7)) << 4));
                const uint4 ov = orow_v[c];
                acc0 = fma2(pack2(__uint_as_float(ov.x << 16), __uint_as_float(ov.x & 0xffff0000u)),
                            pack2(__uint_as_float(gv.x << 16), __uint_as_float(gv.x & 0xffff0000u)), acc0);
                acc1 = fma2(pack2(__uint_as_float(ov.y << 16), __uint_as_float(ov.y & 0xffff0000u)),
                            pack2(__uint_as_float(gv.y << 16), __uint_as_float(gv.y & 0xffff0000u)), acc1);
                acc0 = fma2(pack2(__uint_as_float(ov.z << 16), __uint_as_float(ov.z & 0xffff0000u)),
                            pack2(__uint_as_float(gv.z << 16), __uint_as_float(gv.z & 0xffff0000u)), acc0);
                acc1 = fma2(pack2(__uint_as_float(ov.w << 16), __uint_as_float(ov.w & 0xffff0000u)),
                            pack2(__uint_as_float(gv.w << 16), __uint_as_float(gv.w & 0xffff0000u)), acc1);
            }
            float x0, x1, y0, y1;
            unpack2(acc0, x0, x1);
            unpack2(acc1, y0, y1);
            cen = (x0 + x1) + (y0 + y1);
        }

        for (int t = 0; t < n_tiles; ++t) {
            const int buf = t & 1;
            const uint32_t bcol = tbase + lane_base + buf * C::BUF;
            ok = wait_bar(bar(C::B_SF + buf), (t >> 1) & 1, wc);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            __syncwarp();
            const int nch = min(CPT, n_chunks - CPT * t);
            for (int cc = 0; cc < nch; ++cc) {
                int back;
                bool sk;
                const int key0 = cw.key0(CPT * t + cc, back, sk);
                int clo, chi;
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
                    any_skip |= (clo <= chi);
                }
                if (!live) { clo = CHUNK; chi = -1; }
                const float bo = off - lse2;
                const uint32_t tS = bcol + C::S_COL + cc * CHUNK, tP = bcol + C::DP_COL + cc * CHUNK;
                const uint32_t oS = bcol + C::S_COL + cc * (CHUNK / 2), oP = bcol + C::DP_COL + cc * (CHUNK / 2);
                if (!__any_sync(0xffffffffu, clo <= chi)) {
                    // no row of the warp attends here (a skip chunk of other rows): zero operands
                    const uint32_t zw[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
                    tmem_st8(oS, zw);
                    tmem_st8(oP, zw);
                    tmem_st8(oS + 8, zw);
                    tmem_st8(oP + 8, zw);
                    continue;
                }
                if (sk) {
                    // skip chunk: one column per row (its diagonal key), read with a select tree
                    uint32_t sr[32], dr[32];
                    tmem_ld32(tS, sr);
                    tmem_ld32(tP, dr);
                    tmem_wait_ld();
                    const bool v = clo <= chi;
                    const int cs = v ? clo : 0;
                    const float p = v ? fast_exp2(fmaf(select32(reinterpret_cast<const float *>(sr), cs), sc, bo)) : 0.f;
                    const float w = p * select32(reinterpret_cast<const float *>(dr), cs);
                    dsum += w;
                    skip_p += p;
                    skip_pdp += w;
                    const float a1 = fmaf(-p, cen, w);
                    const uint32_t w1 = (cs & 1) ? pack_bf16(0.f, a1) : pack_bf16(a1, 0.f);
                    const uint32_t w2 = (cs & 1) ? pack_bf16(0.f, p) : pack_bf16(p, 0.f);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t pw[8], pp[8];
#pragma unroll
                        for (int x = 0; x < 8; ++x) {
                            const bool hit = v && (half * 8 + x == (cs >> 1));
                            pw[x] = hit ? w1 : 0u;
                            pp[x] = hit ? w2 : 0u;
                        }
                        tmem_st8(oS + half * 8, pw);
                        tmem_st8(oP + half * 8, pp);
                    }
                    continue;
                }
                if (__all_sync(0xffffffffu, clo == 0 && chi == CHUNK - 1)) {
                    // band chunk inside every row's band: no masks, f32x2 arithmetic
                    const uint64_t sc2 = pack2(sc, sc), bo2 = pack2(bo, bo), mc2 = pack2(-cen, -cen);
                    uint64_t ds2 = pack2(0.f, 0.f);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t sr[16], dr[16];
                        tmem_ld16(tS + half * 16, sr);
                        tmem_ld16(tP + half * 16, dr);
                        tmem_wait_ld();
                        uint32_t pw[8], pp[8];
#pragma unroll
                        for (int c = 0; c < 16; c += 2) {
                            float z0, z1, a0, a1;
                            unpack2(fma2(pack2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sc2, bo2), z0, z1);
                            const float p0 = fast_exp2(z0), p1 = fast_exp2(z1);
                            const uint64_t p2 = pack2(p0, p1);
                            const uint64_t w2 = mul2(p2, pack2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])));
                            ds2 = add2(ds2, w2);
                            unpack2(fma2(p2, mc2, w2), a0, a1);  // p (dp - c)
                            pp[c / 2] = pack_bf16(p0, p1);
                            pw[c / 2] = pack_bf16(a0, a1);
                        }
                        tmem_st8(oS + half * 8, pw);
                        tmem_st8(oP + half * 8, pp);
                    }
                    float d0, d1;
                    unpack2(ds2, d0, d1);
                    dsum += d0 + d1;
                    continue;
                }
                // general path: the row's valid columns [clo, chi] as a bit mask; a masked logit
                // becomes -inf, whose exp2 is 0
                const uint32_t mbits = (clo <= chi) ? ((0xffffffffu >> (31 - chi)) & (0xffffffffu << clo)) : 0u;
                const uint64_t sc2 = pack2(sc, sc), bo2 = pack2(bo, bo), mc2 = pack2(-cen, -cen);
                uint64_t ds2 = pack2(0.f, 0.f);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t sr[16], dr[16];
                    tmem_ld16(tS + half * 16, sr);
                    tmem_ld16(tP + half * 16, dr);
                    tmem_wait_ld();
                    uint32_t pw[8], pp[8];
#pragma unroll
                    for (int c = 0; c < 16; c += 2) {
                        const int c0 = half * 16 + c;
                        float z0, z1, a0, a1;
                        unpack2(fma2(pack2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sc2, bo2), z0, z1);
                        const float p0 = fast_exp2(((mbits >> c0) & 1u) ? z0 : -INFINITY);
                        const float p1 = fast_exp2(((mbits >> (c0 + 1)) & 1u) ? z1 : -INFINITY);
                        const uint64_t p2 = pack2(p0, p1);
                        const uint64_t w2 = mul2(p2, pack2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])));
                        ds2 = add2(ds2, w2);
                        unpack2(fma2(p2, mc2, w2), a0, a1);  // p (dp - c)
                        pp[c / 2] = pack_bf16(p0, p1);
                        pw[c / 2] = pack_bf16(a0, a1);
                    }
                    // A1 operand p (dp - c) over the S columns, A2 operand p over the dP columns;
                    // both chunk halves' values are already in registers
                    tmem_st8(oS + half * 8, pw);
                    tmem_st8(oP + half * 8, pp);
                }
                float d0, d1;
                unpack2(ds2, d0, d1);
                dsum += d0 + d1;
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(C::B_PR + buf));
        }

        // ---- epilogue: dq = tau (A1 - (D - c) A2) -> bf16 -> shared (Q buffer) -> TMA store
        if (ok) {
            ok = wait_bar(bar(C::B_AF), 0, wc);
            ok = __all_sync(0xffffffffu, ok);
        }
        const float tau = s.scale_log2 / kLog2e;
        const float dres = dsum - cen;
        if (ok) {
            tc_fence_after();
            __syncwarp();
#pragma unroll
            for (int oc = 0; oc < D / 16; ++oc) {
                uint32_t a1[16], a2[16];
                tmem_ld16(tbase + lane_base + C::A1_COL + oc * 16, a1);
                tmem_ld16(tbase + lane_base + C::A2_COL + oc * 16, a2);
                tmem_wait_ld();
                uint32_t pk[8];
#pragma unroll
                for (int c = 0; c < 16; c += 2) {
                    const float x0 = tau * fmaf(-dres, __uint_as_float(a2[c]), __uint_as_float(a1[c]));
                    const float x1 = tau * fmaf(-dres, __uint_as_float(a2[c + 1]), __uint_as_float(a1[c + 1]));
                    pk[c / 2] = pack_bf16(x0, x1);
                }
                const int dc = oc >> 2, quarter = oc & 3;
                uint8_t *rowp = smem + C::Q_OFF + dc * C::Q_DBLK + r * ROW_BYTES;
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    const int cidx = quarter * 2 + w;
                    *reinterpret_cast<uint4 *>(rowp + ((cidx ^ (r & 7)) << 4)) =
                        make_uint4(pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
                }
            }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (ok && warp == 4 && lane == 0) {
            const uint64_t once = policy_evict_first();
            for (int dc = 0; dc < C::KD; ++dc)
                tma_store_3d(&tmDQ, sQ + dc * C::Q_DBLK, dc * 64, p0 - s.qoff, b * s.H + h0, once);
            tma_store_commit_and_wait();
        }
        if (ok && row_ok) {
            args.Dws[row_g] = dsum;
            if (args.dalpha) {
                any_skip = any_skip && live;
                args.dalpha[row_g] =
                    (s.mode != kModeEcp && any_skip && al > 0.f && al < 1.f)
                        ? -(skip_pdp - dsum * skip_p) / (al * (1.f - al)) : 0.f;  // saturated gate: 0
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tbase, C::TMEM_COLS);
    }
}

template <int D>
static cudaError_t launch_dq(const CUtensorMap &mq, const CUtensorMap &mg, const CUtensorMap &mk,
                            const CUtensorMap &mv, const CUtensorMap &mdq, const DqArgs &a,
                            unsigned grid, cudaStream_t st) {
    constexpr int smem = CfgQ<D>::SMEM_BYTES;
    static PerDeviceOnce configured;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured.needed(dev)) {
        cudaError_t e = cudaFuncSetAttribute(bwd_dq_tc_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured.mark(dev);
    }
    bwd_dq_tc_kernel<D><<<grid, NUM_THREADS, smem, st>>>(mq, mg, mk, mv, mdq, a);
    return cudaGetLastError();
}


// ---------------------------------------------------------------------------- kernel 2

constexpr int BK = 128;     // keys per CTA (M)

// The query chunks (qc queries each) that attend to keys [j0, j0 + 128) of one KV head, for
// one query head: band chunks i0 = q0 + qc*c from the first query whose band holds key j0 to
// the last whose band holds key j0 + 127; then 128/qc chunks per skip multiple m: first the
// n_fwd multiples of queries j0 + m*period + [0, 128) (their keys i - m*period), then
// (bidirectional mode) those of queries j0 - m*period + [0, 128) (keys i + m*period).  `back` is
// the distance query - key of a skip chunk.
struct KWalk {
    int j0, q0, n_band, m_first, n_fwd, n_skip, period, per_head, qc, cps_log2;
    __device__ __forceinline__ void chunk(int ci, int &hh, int &i0, int &back, bool &skip) const {
        hh = ci / per_head;
        const int c = ci - hh * per_head;
        if (c < n_band) {
            i0 = q0 + c * qc;
            back = 0;
            skip = false;
        } else {
            const int sc = c - n_band;
            const int blk = sc >> cps_log2;
            back = (blk < n_fwd) ? (m_first + blk) * period : -(m_first + blk - n_fwd) * period;
            i0 = j0 + back + (sc & ((1 << cps_log2) - 1)) * qc;
            skip = true;
        }
    }
};

template <int D>
struct CfgK {
    static constexpr int KD = D / 64;
    static constexpr int QC = (D == 64) ? 32 : 64;  // queries per chunk (N of the transposed MMAs)
    static constexpr int CPS_LOG2 = (D == 64) ? 2 : 1;  // log2(BK / QC): chunks per skip block
    static constexpr int ST = (D == 64) ? 6 : 3;        // query-chunk stages
    static constexpr int KT_BYTES = BK * D * 2;
    static constexpr int KT_DBLK = BK * ROW_BYTES;
    static constexpr int QC_BYTES = QC * D * 2;
    static constexpr int QC_DBLK = QC * ROW_BYTES;
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = KT_BYTES;
    static constexpr int Q_OFF = 2 * KT_BYTES;                // [ST] Q chunks
    static constexpr int G_OFF = Q_OFF + ST * QC_BYTES;        // [ST] dO chunks
    static constexpr int X_OFF = G_OFF + ST * QC_BYTES;        // [ST][2][QC] fp32: bias, D
    static constexpr int BAR_OFF = X_OFF + ST * 2 * QC * 4;
    static constexpr int B_KV = 0;                 // K and V tiles landed
    static constexpr int B_QF = 1;                 // [ST] Q/dO chunk landed
    static constexpr int B_QE = B_QF + ST;         // [ST] chunk consumed by its dV/dK MMAs
    static constexpr int B_XF = B_QE + ST;         // [ST] per-query vectors ready (32 arrivals)
    static constexpr int B_XE = B_XF + ST;         // [ST] vectors consumed (128 arrivals)
    // Two S^T/dP^T buffers in TMEM: chunk ci uses buffer ci & 1.
    static constexpr int B_SF = B_XE + ST;         // [2] S^T, dP^T in TMEM
    static constexpr int B_PR = B_SF + 2;          // [2] P^T, dZ^T written back (128 arrivals)
    static constexpr int B_BF = B_PR + 2;          // [2] dV/dK MMAs of the chunk done: buffer free
    static constexpr int B_OF = B_BF + 2;          // dK, dV complete (single phase)
    static constexpr int B_DR = B_OF + 1;          // drain of the S^T/dP^T issuer
    static constexpr int B_DR2 = B_DR + 1;         // drain of the dV/dK issuer
    static constexpr int NBARS = B_DR2 + 1;
    static constexpr int SMEM_BYTES = BAR_OFF + NBARS * 8 + 16 + 1024;
    static constexpr int BUF = 2 * QC;  // S^T then dP^T of one buffer
    static constexpr int ST_COL = 0, DPT_COL = QC, DV_COL = 2 * BUF, DK_COL = 2 * BUF + D;
    static constexpr int TMEM_COLS = (DK_COL + D <= 256) ? 256 : 512;
};

struct DkvArgs {
    const float *alpha;
    const float *lse;
    const float *Dws;
    Shape s;
    int *status;
    uint64_t timeout_ns;
};

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
bwd_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const __grid_constant__ CUtensorMap tmQc, const __grid_constant__ CUtensorMap tmGc,
                   const __grid_constant__ CUtensorMap tmDK, const __grid_constant__ CUtensorMap tmDV,
                   const DkvArgs args) {
    using C = CfgK<D>;
    constexpr int ST = C::ST;
    constexpr int QC = C::QC;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_addr & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    const uint32_t sbase = raw_addr + pad;
    const uint32_t sK = sbase + C::K_OFF, sV = sbase + C::V_OFF, sQ = sbase + C::Q_OFF,
                   sG = sbase + C::G_OFF, sBar = sbase + C::BAR_OFF;
    float *xvec = reinterpret_cast<float *>(smem + C::X_OFF);
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::BAR_OFF + C::NBARS * 8);
    uint32_t *tmem_slot = misc;
    volatile uint32_t *abort_flag = misc + 1;
    auto bar = [&](int idx) -> uint32_t { return sBar + idx * 8; };

    const Shape &s = args.s;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const WaitCtx wc{abort_flag, args.status, args.timeout_ns};

    // ---- key block and its query chunks
    const int nkb = (s.N + BK - 1) / BK;
    const int kb = blockIdx.x % nkb;
    const int bg = blockIdx.x / nkb;
    const int g = bg % s.Hkv, b = bg / s.Hkv;
    const int G = s.H / s.Hkv;
    KWalk kw;
    kw.j0 = kb * BK;
    kw.period = s.period;
    kw.qc = QC;
    kw.cps_log2 = C::CPS_LOG2;
    const int qlast = band_last_query(min(s.N - 1, kw.j0 + BK - 1), s.N, s.mode, s.k_local);
    kw.q0 = band_first_query(kw.j0, s.mode, s.k_local);
    kw.n_band = (qlast - kw.q0) / QC + 1;
    kw.m_first = 1;
    kw.n_fwd = 0;
    kw.n_skip = 0;
    if (s.mode != kModeEcp && s.S > 0) {
        kw.m_first = first_skip_multiple(s);
        // multiples whose first skip query j0 + m*period is inside the sequence
        const int m_last = min(s.S, (s.N - 1 - kw.j0) / s.period);
        kw.n_fwd = max(0, m_last - kw.m_first + 1);
        int n_blocks = kw.n_fwd;
        if (s.mode == kModeBidir) {  // multiples whose last skip query j0 + 127 - m*period is >= 0
            const int m_last_b = min(s.S, min(s.N - 1, kw.j0 + BK - 1) / s.period);
            n_blocks += max(0, m_last_b - kw.m_first + 1);
        }
        kw.n_skip = (1 << C::CPS_LOG2) * n_blocks;
    }
    kw.per_head = kw.n_band + kw.n_skip;
    const int n_chunks = G * kw.per_head;

    if (warp == 0) {  // barriers spread over warp 0's lanes
        for (int idx = lane; idx < C::NBARS; idx += 32) {
            uint32_t count = 1;
            if (idx >= C::B_XF && idx < C::B_XF + ST) count = 32;
            if ((idx >= C::B_XE && idx < C::B_XE + ST) || idx == C::B_PR || idx == C::B_PR + 1) count = 128;
            mbar_init(bar(idx), count);
        }
        if (lane == 0) *abort_flag = 0u;
        fence_barrier_init();
        __syncwarp();
    }
    if (warp == 0) tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *tmem_slot;

    if (warp == 0) {
        // ================= producer: K and V tiles once, then Q/dO chunks
        if (lane == 0) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
            prefetch_tmap(&tmQc);
            prefetch_tmap(&tmGc);
            const uint64_t reused = policy_evict_last();
            mbar_expect_tx(bar(C::B_KV), 2 * C::KT_BYTES);
            for (int dc = 0; dc < C::KD; ++dc) {
                tma_load_3d_hint(sK + dc * C::KT_DBLK, &tmK, dc * 64, kw.j0, b * s.Hkv + g, bar(C::B_KV), reused);
                tma_load_3d_hint(sV + dc * C::KT_DBLK, &tmV, dc * 64, kw.j0, b * s.Hkv + g, bar(C::B_KV), reused);
            }
            int issued = 0;
            for (int ci = 0; ci < n_chunks; ++ci) {
                const int st = ci % ST, round = ci / ST;
                if (round > 0 && !wait_bar(bar(C::B_QE + st), (round - 1) & 1, wc)) break;
                int hh, i0, back;
                bool sk;
                kw.chunk(ci, hh, i0, back, sk);
                const int plane = b * s.H + g * G + hh;
                mbar_expect_tx(bar(C::B_QF + st), 2 * C::QC_BYTES);
                for (int dc = 0; dc < C::KD; ++dc) {
                    tma_load_3d_hint(sQ + st * C::QC_BYTES + dc * C::QC_DBLK, &tmQc, dc * 64, i0 - s.qoff,
                                     plane, bar(C::B_QF + st), reused);
                    tma_load_3d_hint(sG + st * C::QC_BYTES + dc * C::QC_DBLK, &tmGc, dc * 64, i0 - s.qoff,
                                     plane, bar(C::B_QF + st), reused);
                }
                issued = ci + 1;
            }
            if (*abort_flag) {
                volatile uint32_t zero = 0;
                WaitCtx w2{&zero, nullptr, 20000000ull};
                wait_bar(bar(C::B_KV), 0, w2);
                for (int ci = max(0, issued - ST); ci < issued; ++ci)
                    wait_bar(bar(C::B_QF + ci % ST), (ci / ST) & 1, w2);
            }
        }
    } else if (warp == 2) {
        // ================= per-query vectors of each chunk: bias = prior - lse (log2 units), D.
        // The loads of chunk ci + 1 are in flight while chunk ci's values are stored.
        constexpr int QL = QC / 32;  // queries per lane
        float nl[QL], na[QL], nd[QL];
        bool nsk = false;
        auto fetch = [&](int ci) {
            int hh, i0, back;
            kw.chunk(ci, hh, i0, back, nsk);
            const long long rbase = ((long long)b * s.H + g * G + hh) * s.nq;
#pragma unroll
            for (int e = 0; e < QL; ++e) {
                // skip chunks of the bidirectional mode may start before 0; positions outside the
                // query window (a sequence shard's halo) have no query and take P = 0
                const int iq = i0 + lane + 32 * e - s.qoff;  // row of the query window
                const bool in = iq >= 0 && iq < s.nq;
                nl[e] = in ? args.lse[rbase + iq] : -INFINITY;
                na[e] = (in && args.alpha) ? args.alpha[rbase + iq] : 1.f;
                nd[e] = in ? args.Dws[rbase + iq] : 0.f;
            }
        };
        if (n_chunks > 0) fetch(0);
        bool ok = true;
        for (int ci = 0; ok && ci < n_chunks; ++ci) {
            const int st = ci % ST, round = ci / ST;
            if (round > 0) {
                ok = wait_bar(bar(C::B_XE + st), (round - 1) & 1, wc);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
            }
            float cl[QL], ca[QL], cd[QL];
#pragma unroll
            for (int e = 0; e < QL; ++e) {
                cl[e] = nl[e];
                ca[e] = na[e];
                cd[e] = nd[e];
            }
            const bool sk = nsk;
            if (ci + 1 < n_chunks) fetch(ci + 1);
            float *xb = xvec + st * 2 * QC;
#pragma unroll
            for (int e = 0; e < QL; ++e) {
                const float lse2 = cl[e] * kLog2e;
                const float prior = (s.mode == kModeEcp) ? 0.f : (sk ? log2f(1.f - ca[e]) : log2f(ca[e]));
                xb[lane + 32 * e] = (lse2 != -INFINITY) ? prior - lse2 : -INFINITY;
                xb[QC + lane + 32 * e] = cd[e];
            }
            mbar_arrive(bar(C::B_XF + st));
        }
    } else if (warp == 1) {
        // ================= S^T/dP^T issuer: into buffer ci & 1 once its previous dV/dK MMAs
        // (chunk ci-2) are done (whole warp, one elected lane issuing)
        bool ok = __all_sync(0xffffffffu, wait_bar(bar(C::B_KV), 0, wc));
        const uint32_t idesc_t = idesc_bf16(BK, QC, 0, 0);  // S^T, dP^T: both operands K-major
        const uint64_t kd0 = sdesc(sK, 16, 1024), vd0 = sdesc(sV, 16, 1024);
        for (int ci = 0; ok && ci < n_chunks; ++ci) {
            const int st = ci % ST, buf = ci & 1;
            bool w = wait_bar(bar(C::B_QF + st), (ci / ST) & 1, wc);
            if (w && ci >= 2) w = wait_bar(bar(C::B_BF + buf), ((ci - 2) >> 1) & 1, wc);
            if (!__all_sync(0xffffffffu, w)) break;
            tc_fence_after();
            const uint64_t qd0 = sdesc(sQ + st * C::QC_BYTES, 16, 1024), gd0 = sdesc(sG + st * C::QC_BYTES, 16, 1024);
            const uint32_t dS = tbase + C::ST_COL + buf * C::BUF, dP = tbase + C::DPT_COL + buf * C::BUF;
            if (elect_one()) {
#pragma unroll
                for (int dc = 0; dc < C::KD; ++dc) {
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const uint32_t acc = (dc | ks) != 0;
                        // the start address field counts 16-byte units
                        const uint64_t ok_ = (uint64_t)((dc * C::KT_DBLK + ks * 32) >> 4);
                        const uint64_t oq = (uint64_t)((dc * C::QC_DBLK + ks * 32) >> 4);
                        mma_ss(dS, kd0 + ok_, qd0 + oq, idesc_t, acc);
                        mma_ss(dP, vd0 + ok_, gd0 + oq, idesc_t, acc);
                    }
                }
                tc_commit(bar(C::B_SF + buf));
            }
            __syncwarp();
        }
        if (elect_one()) tc_commit(bar(C::B_DR));
        __syncwarp();
        volatile uint32_t zero = 0;
        WaitCtx w2{&zero, args.status, args.timeout_ns};
        wait_bar(bar(C::B_DR), 0, w2);
    } else if (warp == 3) {
        // ================= dV/dK issuer: dV += P^T dO, dK += dZ^T Q from buffer ci & 1 (whole
        // warp, one elected lane issuing)
        const uint32_t idesc_a = idesc_bf16(BK, D, 0, 1);   // dV, dK: B = chunk, MN-major
        for (int ci = 0; ci < n_chunks; ++ci) {
            const int st = ci % ST, buf = ci & 1;
            // the chunk's Q/dO landed before its S^T, which the key threads saw before P^T
            if (!__all_sync(0xffffffffu, wait_bar(bar(C::B_PR + buf), (ci >> 1) & 1, wc))) break;
            tc_fence_after();
            const uint64_t qd0 = sdesc(sQ + st * C::QC_BYTES, C::QC_DBLK, 1024);
            const uint64_t gd0 = sdesc(sG + st * C::QC_BYTES, C::QC_DBLK, 1024);
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < QC / 16; ++kk) {
                    const uint32_t acc = (ci > 0 || kk > 0) ? 1u : 0u;
                    const uint64_t o = (uint64_t)((kk * 16 * ROW_BYTES) >> 4);
                    mma_ts(tbase + C::DV_COL, tbase + C::ST_COL + buf * C::BUF + kk * 8, gd0 + o, idesc_a, acc);
                    mma_ts(tbase + C::DK_COL, tbase + C::DPT_COL + buf * C::BUF + kk * 8, qd0 + o, idesc_a, acc);
                }
                tc_commit(bar(C::B_BF + buf));
                tc_commit(bar(C::B_QE + st));
                if (ci == n_chunks - 1) tc_commit(bar(C::B_OF));
            }
            __syncwarp();
        }
        if (elect_one()) tc_commit(bar(C::B_DR2));
        __syncwarp();
        volatile uint32_t zero = 0;
        WaitCtx w2{&zero, args.status, args.timeout_ns};
        wait_bar(bar(C::B_DR2), 0, w2);
    } else if (warp >= 4) {
        // ================= one thread per key
        const int q4 = warp & 3;
        const int r = q4 * 32 + lane;
        const int j = kw.j0 + r;
        const bool key_ok = j < s.N;
        const int qlast_j = key_ok ? band_last_query(j, s.N, s.mode, s.k_local) : -1;
        const int qfirst_j = band_first_query(j, s.mode, s.k_local);
        const float sc = s.scale_log2;
        const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
        bool ok = true;

        for (int ci = 0; ci < n_chunks; ++ci) {
            const int st = ci % ST, buf = ci & 1;
            const uint32_t bcol = tbase + lane_base + buf * C::BUF;
            ok = wait_bar(bar(C::B_SF + buf), (ci >> 1) & 1, wc);
            ok = ok && wait_bar(bar(C::B_XF + st), (ci / ST) & 1, wc);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();
            __syncwarp();
            int hh, i0, back;
            bool sk;
            kw.chunk(ci, hh, i0, back, sk);
            // valid query columns of this key: [clo, chi]
            int clo, chi;
            if (!sk) {
                clo = max(qfirst_j - i0, 0);
                chi = min(qlast_j - i0, QC - 1);
            } else {
                const int iq = j + back, c = iq - i0;
                if (iq >= 0 && iq < s.N && c >= 0 && c < QC) { clo = c; chi = c; }
                else { clo = QC; chi = -1; }
            }
            if (!key_ok) { clo = QC; chi = -1; }
            const float *xb = xvec + st * 2 * QC;
            const unsigned any = __ballot_sync(0xffffffffu, clo <= chi);
            if (any == 0u || sk) {
                // skip chunk (one column per key, its diagonal query) or nothing for this warp: the
                // valid columns of a warp's keys are consecutive and lie in one 32-column block
                const int qb = any ? (__shfl_sync(0xffffffffu, clo, __ffs(any) - 1) >> 5) : -1;
                const bool v = clo <= chi;
                const int cs = clo & 31;
                uint32_t w1 = 0u, w2 = 0u;
                if (qb >= 0) {
                    uint32_t sr[32], dr[32];
                    tmem_ld32(bcol + C::ST_COL + qb * 32, sr);
                    tmem_ld32(bcol + C::DPT_COL + qb * 32, dr);
                    tmem_wait_ld();
                    const int cq = v ? clo : 0;
                    const float p = v ? fast_exp2(fmaf(select32(reinterpret_cast<const float *>(sr), cs), sc, xb[cq])) : 0.f;
                    const float z = p * (select32(reinterpret_cast<const float *>(dr), cs) - xb[QC + cq]);
                    w1 = (cs & 1) ? pack_bf16(0.f, p) : pack_bf16(p, 0.f);
                    w2 = (cs & 1) ? pack_bf16(0.f, z) : pack_bf16(z, 0.f);
                }
#pragma unroll
                for (int q = 0; q < QC / 32; ++q) {
                    uint32_t pp[16], pz[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        const bool hit = v && q == qb && x == (cs >> 1);
                        pp[x] = hit ? w1 : 0u;
                        pz[x] = hit ? w2 : 0u;
                    }
                    tmem_st16(bcol + C::ST_COL + q * 16, pp);
                    tmem_st16(bcol + C::DPT_COL + q * 16, pz);
                }
            } else if (__all_sync(0xffffffffu, clo == 0 && chi == QC - 1)) {
                // band chunk inside the band of every key of the warp: no masks, f32x2 arithmetic
                const uint64_t sc2 = pack2(sc, sc), neg2 = pack2(-1.f, -1.f);
#pragma unroll
                for (int q = 0; q < QC / 32; ++q) {
                    uint32_t sr[32], dr[32];
                    tmem_ld32(bcol + C::ST_COL + q * 32, sr);
                    tmem_ld32(bcol + C::DPT_COL + q * 32, dr);
                    tmem_wait_ld();
                    uint32_t pp[16], pz[16];
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        const int c0 = q * 32 + c;
                        const uint64_t bias2 = *reinterpret_cast<const uint64_t *>(xb + c0);
                        const uint64_t dd2 = *reinterpret_cast<const uint64_t *>(xb + QC + c0);
                        float z0, z1, y0, y1;
                        unpack2(fma2(pack2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sc2, bias2), z0, z1);
                        const float p0 = fast_exp2(z0), p1 = fast_exp2(z1);
                        const uint64_t p2 = pack2(p0, p1);
                        // dz = p (dp - D)
                        unpack2(mul2(p2, fma2(dd2, neg2, pack2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])))), y0, y1);
                        pp[c / 2] = pack_bf16(p0, p1);
                        pz[c / 2] = pack_bf16(y0, y1);
                    }
                    tmem_st16(bcol + C::ST_COL + q * 16, pp);
                    tmem_st16(bcol + C::DPT_COL + q * 16, pz);
                }
            } else {
            // general path: the key's valid columns [clo, chi] as a bit mask per 32-column block; a
            // masked logit becomes -inf, whose exp2 is 0
            const uint64_t sc2 = pack2(sc, sc), neg2 = pack2(-1.f, -1.f);
#pragma unroll
            for (int q = 0; q < QC / 32; ++q) {  // 32 columns of S^T and dP^T per TMEM round trip
                const int lo = max(clo - 32 * q, 0), hi = min(chi - 32 * q, 31);
                const uint32_t mbits = (lo <= hi) ? ((0xffffffffu >> (31 - hi)) & (0xffffffffu << lo)) : 0u;
                uint32_t sr[32], dr[32];
                tmem_ld32(bcol + C::ST_COL + q * 32, sr);
                tmem_ld32(bcol + C::DPT_COL + q * 32, dr);
                tmem_wait_ld();
                uint32_t pp[16], pz[16];
#pragma unroll
                for (int c = 0; c < 32; c += 2) {
                    const int c0 = q * 32 + c;
                    const uint64_t bias2 = *reinterpret_cast<const uint64_t *>(xb + c0);
                    const uint64_t dd2 = *reinterpret_cast<const uint64_t *>(xb + QC + c0);
                    float z0, z1, y0, y1;
                    unpack2(fma2(pack2(__uint_as_float(sr[c]), __uint_as_float(sr[c + 1])), sc2, bias2), z0, z1);
                    const float p0 = fast_exp2(((mbits >> c) & 1u) ? z0 : -INFINITY);
                    const float p1 = fast_exp2(((mbits >> (c + 1)) & 1u) ? z1 : -INFINITY);
                    const uint64_t p2 = pack2(p0, p1);
                    unpack2(mul2(p2, fma2(dd2, neg2, pack2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])))), y0, y1);
                    pp[c / 2] = pack_bf16(p0, p1);
                    pz[c / 2] = pack_bf16(y0, y1);
                }
                tmem_st16(bcol + C::ST_COL + q * 16, pp);
                tmem_st16(bcol + C::DPT_COL + q * 16, pz);
            }
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(C::B_PR + buf));
            mbar_arrive(bar(C::B_XE + st));
        }

        // ---- epilogue: dK * tau, dV -> bf16 -> shared (the K and V tiles) -> TMA store
        if (ok) {
            ok = wait_bar(bar(C::B_OF), 0, wc);
            ok = __all_sync(0xffffffffu, ok);
        }
        const float tau = sc / kLog2e;
        if (ok) {
            tc_fence_after();
            __syncwarp();
#pragma unroll
            for (int oc = 0; oc < D / 16; ++oc) {
                uint32_t xk[16], xv[16];
                tmem_ld16(tbase + lane_base + C::DK_COL + oc * 16, xk);
                tmem_ld16(tbase + lane_base + C::DV_COL + oc * 16, xv);
                tmem_wait_ld();
                uint32_t pk[8], pv[8];
#pragma unroll
                for (int c = 0; c < 16; c += 2) {
                    pk[c / 2] = pack_bf16(__uint_as_float(xk[c]) * tau, __uint_as_float(xk[c + 1]) * tau);
                    pv[c / 2] = pack_bf16(__uint_as_float(xv[c]), __uint_as_float(xv[c + 1]));
                }
                const int dc = oc >> 2, quarter = oc & 3;
                uint8_t *rk = smem + C::K_OFF + dc * C::KT_DBLK + r * ROW_BYTES;
                uint8_t *rv = smem + C::V_OFF + dc * C::KT_DBLK + r * ROW_BYTES;
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    const int off = ((quarter * 2 + w) ^ (r & 7)) << 4;
                    *reinterpret_cast<uint4 *>(rk + off) = make_uint4(pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
                    *reinterpret_cast<uint4 *>(rv + off) = make_uint4(pv[4 * w], pv[4 * w + 1], pv[4 * w + 2], pv[4 * w + 3]);
                }
            }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (ok && warp == 4 && lane == 0) {
            const uint64_t once = policy_evict_first();
            for (int dc = 0; dc < C::KD; ++dc) {
                tma_store_3d(&tmDK, sK + dc * C::KT_DBLK, dc * 64, kw.j0, b * s.Hkv + g, once);
                tma_store_3d(&tmDV, sV + dc * C::KT_DBLK, dc * 64, kw.j0, b * s.Hkv + g, once);
            }
            tma_store_commit_and_wait();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tbase, C::TMEM_COLS);
    }
}

template <int D>
static cudaError_t launch_dkdv(const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mqc,
                              const CUtensorMap &mgc, const CUtensorMap &mdk, const CUtensorMap &mdv,
                              const DkvArgs &a, unsigned grid, cudaStream_t st) {
    constexpr int smem = CfgK<D>::SMEM_BYTES;
    static PerDeviceOnce configured;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured.needed(dev)) {
        cudaError_t e = cudaFuncSetAttribute(bwd_dkdv_tc_kernel<D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured.mark(dev);
    }
    bwd_dkdv_tc_kernel<D><<<grid, NUM_THREADS, smem, st>>>(mk, mv, mqc, mgc, mdk, mdv, a);
    return cudaGetLastError();
}

}  // namespace tcb

cudaError_t launch_bwd_dq_tc(const LaunchBwd &L, int *status, uint64_t timeout_ns, cudaStream_t st) {
    using namespace tcb;
    const Shape &s = L.s;
    const int G = s.H / s.Hkv;
    const int GP = (G % 4 == 0) ? 4 : (G % 2 == 0) ? 2 : 1;
    const int R = BM / GP;
    CUtensorMap mq, mg, mk, mv, mdq;
    if (!make_map(&mq, L.q, s.d, s.nq, (long long)s.B * s.H, R, GP) ||
        !make_map(&mg, L.dout, s.d, s.nq, (long long)s.B * s.H, R, GP) ||
        !make_map(&mdq, L.dq, s.d, s.nq, (long long)s.B * s.H, R, GP) ||
        !make_map(&mk, L.k, s.d, s.N, (long long)s.B * s.Hkv, CHUNK, 1) ||
        !make_map(&mv, L.v, s.d, s.N, (long long)s.B * s.Hkv, CHUNK, 1))
        return cudaErrorNotSupported;
    DqArgs a{static_cast<const __nv_bfloat16 *>(L.out), static_cast<const __nv_bfloat16 *>(L.dout), L.alpha,
             L.lse, L.Dws, L.dalpha, s, GP, status, timeout_ns};
    const long long grid = (long long)s.B * (s.H / GP) * ((s.nq + R - 1) / R);
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (s.d == 64) return launch_dq<64>(mq, mg, mk, mv, mdq, a, (unsigned)grid, st);
    if (s.d == 128) return launch_dq<128>(mq, mg, mk, mv, mdq, a, (unsigned)grid, st);
    return cudaErrorInvalidValue;
}

cudaError_t launch_bwd_dkdv_tc(const LaunchBwd &L, int *status, uint64_t timeout_ns, cudaStream_t st) {
    using namespace tcb;
    const Shape &s = L.s;
    CUtensorMap mk, mv, mqc, mgc, mdk, mdv;
    if (!make_map(&mk, L.k, s.d, s.N, (long long)s.B * s.Hkv, BK, 1) ||
        !make_map(&mv, L.v, s.d, s.N, (long long)s.B * s.Hkv, BK, 1) ||
        !make_map(&mdk, L.dk, s.d, s.N, (long long)s.B * s.Hkv, BK, 1) ||
        !make_map(&mdv, L.dv, s.d, s.N, (long long)s.B * s.Hkv, BK, 1) ||
        !make_map(&mqc, L.q, s.d, s.nq, (long long)s.B * s.H, s.d == 64 ? CfgK<64>::QC : CfgK<128>::QC, 1) ||
        !make_map(&mgc, L.dout, s.d, s.nq, (long long)s.B * s.H, s.d == 64 ? CfgK<64>::QC : CfgK<128>::QC, 1))
        return cudaErrorNotSupported;
    DkvArgs a{L.alpha, L.lse, L.Dws, s, status, timeout_ns};
    const long long grid = (long long)s.B * s.Hkv * ((s.N + BK - 1) / BK);
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (s.d == 64) return launch_dkdv<64>(mk, mv, mqc, mgc, mdk, mdv, a, (unsigned)grid, st);
    if (s.d == 128) return launch_dkdv<128>(mk, mv, mqc, mgc, mdk, mdv, a, (unsigned)grid, st);
    return cudaErrorInvalidValue;
}

}  // namespace pi
