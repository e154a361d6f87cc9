// Round attention on the 5th-generation tensor cores with the probabilities
// P kept apart from the scores S in tensor memory.
//
// Computes exactly what attn_tc.cu computes ("Wave Forcing", Sec. 3.1
// Eq. 4-5: for every active task and head, softmax(Q K^T / sqrt(D)) V over
// the task's ordered context, bidirectional inside each chunk, masked chunk
// blocks never visited), with a different pipeline.
//
// In attn_tc.cu P overwrites the first columns of S, so the next key tile's
// S = Q K^T can only be issued after P V has consumed P: the tile's own two
// MMA groups sit on the softmax's critical path.  Here key tiles are 80 keys
// (bf16) or 96 keys (e4m3), small enough that each query tile's S and P get
// separate tensor-memory regions beside the two O accumulators:
//
//   tile X: S at column 128 X (BN columns), P at 128 X + BN (BN/2 bf16 or
//   BN/4 e4m3 columns); O_X at 256 + 128 X.             (496 of 512 columns)
//
// so the issuer starts S(j+1) = Q K_{j+1}^T as soon as the softmax has read
// S(j) into registers ("S free"), and P(j) V_j when P(j) is stored.  The
// softmax of a tile then runs back to back while the tensor pipe works
// through the other tile's and its own MMAs.  Two hazards the aliasing used
// to rule out are handled by a "PV done" barrier per tile: the softmax waits
// for P(j-1) V_{j-1} to complete before it overwrites P with P(j), and before
// it rescales O (rare: only when the running maximum grows by more than 2^8).
//
// Roles (one persistent 384-thread CTA per SM, units = (task, head, pair of
// 128-row query tiles) handed out longest context first, as in attn_tc.cu):
// warp 8 one thread: TMA producer (Q tiles, then K_0, K_1, V_0, K_2, V_1, ...
// through an NST-stage ring); warp 9 one thread: tcgen05.mma issuer; warps
// 0-3 / 4-7: softmax of query tile 0 / 1, one thread per row.
//
// Every wait is bounded (%globaltimer); on a timeout the kernel records it in
// the status word, drains its own copies and MMAs, frees TMEM and returns.

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "wf_internal.h"
#include "wf_ptx.cuh"

using namespace wfptx;

namespace {

constexpr int BM = 128;             // query rows per tile
constexpr int HD = 128;             // head dim
constexpr int NUM_THREADS = 384;
constexpr uint64_t WAIT_NS = 1000000000ull;  // 1 s

template <bool F8>
struct L2 {
    static constexpr int BN = F8 ? 96 : 80;               // keys per tile
    static constexpr int NST = F8 ? 8 : 7;                // K/V ring stages
    static constexpr int PCOLS = F8 ? BN / 4 : BN / 2;   // TMEM columns of P
    static constexpr uint32_t QTILE = BM * HD * (F8 ? 1 : 2);
    static constexpr uint32_t QHALF = F8 ? QTILE : QTILE / 2;       // one 128-byte-wide block
    static constexpr uint32_t KVTILE = BN * HD * (F8 ? 1 : 2);
    static constexpr uint32_t KVHALF = F8 ? KVTILE : KVTILE / 2;
    static constexpr uint32_t Q0 = 0;
    static constexpr uint32_t Q1 = QTILE;
    static constexpr uint32_t KV = 2 * QTILE;
    static constexpr uint32_t BAR = KV + NST * KVTILE;
    // barriers
    static constexpr int B_QFULL = 0;
    static constexpr int B_KVFULL = 1;
    static constexpr int B_KVEMPTY = B_KVFULL + NST;
    static constexpr int B_SFULL = B_KVEMPTY + NST;   // S(j) computed (per tile)
    static constexpr int B_SFREE = B_SFULL + 2;       // S(j) read by the softmax
    static constexpr int B_PFULL = B_SFREE + 2;       // P(j) stored
    static constexpr int B_PVDONE = B_PFULL + 2;      // P(j) V_j completed
    static constexpr int B_DRAIN = B_PVDONE + 2;
    static constexpr int NBARS = B_DRAIN + 1;
    static constexpr uint32_t MISC = BAR + ((NBARS * 8 + 63) / 64) * 64;
    static constexpr uint32_t ALLOC = MISC + 64 + 1024;   // + alignment slack
    static_assert(QTILE % 1024 == 0 && KVTILE % 1024 == 0 && KVHALF % 1024 == 0,
                  "128-byte swizzle atoms must stay 1024-byte aligned");
    static_assert(2 * (BN + PCOLS) <= 256, "S and P of both tiles must fit beside O");
    static_assert(ALLOC <= 232448, "shared memory");
};

// Register split as in attn_tc.cu: 384 x 168 at launch; the producer/MMA
// warpgroup gives up what the softmax warpgroups take.
constexpr int LAUNCH_REGS = 168;
constexpr int REGS_SOFTMAX = 224;
constexpr int REGS_AUX = 56;
static_assert(8 * (REGS_SOFTMAX - LAUNCH_REGS) <= 4 * (LAUNCH_REGS - REGS_AUX),
              "register split exceeds the launch pool");

struct Tc2Params {
    int layer;
    int n_units;
    int qpairs;           // pairs of query tiles per (task, head)
    int tpc;              // key tiles per chunk
    float sl2;            // log2(e) / sqrt(D) (/ qk_scale^2 for e4m3 Q and K)
    float o_scale;        // 1 (bf16) or 1 / v_scale (e4m3 V)
    __nv_bfloat16 *out;   // [slot][N_C][H][D] bf16, or e4m3 bytes when out_e4m3
    int out_e4m3;
    uint32_t *ctl;        // scheduler counters (work, finished CTAs)
    uint32_t *stat;       // status and wait-site words
};

__device__ __forceinline__ int kseq(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int vseq(int j, int n) { return j == n - 1 ? 2 * n - 1 : 2 * j + 2; }

template <bool F8>
struct Ctx2 {
    uint32_t sbase;
    volatile int *abort;
    uint32_t *status, *where;
    __device__ uint32_t bar(int i) const { return sbase + L2<F8>::BAR + 8u * i; }
    __device__ bool wait(int b, uint32_t parity, uint32_t site) const {
        return mbar_wait(bar(b), parity, abort, status, where, site, WAIT_NS);
    }
};

__device__ __forceinline__ void decode_unit(int u, const WfRoundDev &rd, const Tc2Params &p, int H,
                                            int &ti, int &h, int &qp) {
    int per_task = H * p.qpairs;
    int oi = u / per_task;
    int rem = u - oi * per_task;
    ti = rd.lpt[oi];
    h = rem / p.qpairs;
    qp = rem - h * p.qpairs;
}

// ---- producer ----------------------------------------------------------------
template <bool F8>
__device__ void producer(const Ctx2<F8> &c, const CUtensorMap *tq, const CUtensorMap *tkv,
                         const WfGeom &g, const WfRoundDev &rd, const Tc2Params &p, int ti, int h,
                         int qp, int n, uint32_t seq, uint32_t *issued) {
    using L = L2<F8>;
    const int plane_q = rd.slot[ti] * g.H + h;
    mbar_arrive_expect_tx(c.bar(L::B_QFULL), 2 * L::QTILE);
    for (int x = 0; x < 2; ++x) {
        const uint32_t dst = c.sbase + (x ? L::Q1 : L::Q0);
        tma_load_3d(dst, tq, c.bar(L::B_QFULL), 0, (2 * qp + x) * BM, plane_q);
        if (!F8) tma_load_3d(dst + L::QHALF, tq, c.bar(L::B_QFULL), 64, (2 * qp + x) * BM, plane_q);
    }
    for (int i = 0; i < 2 * n; ++i) {
        int j, isv;
        if (i == 0) {
            j = 0; isv = 0;
        } else if (i == 2 * n - 1) {
            j = n - 1; isv = 1;
        } else if (i & 1) {
            j = (i + 1) / 2; isv = 0;
        } else {
            j = i / 2 - 1; isv = 1;
        }
        const uint32_t s = seq + i;
        const int st = s % L::NST;
        if (!c.wait(L::B_KVEMPTY + st, ((s / L::NST) & 1) ^ 1, 1)) return;
        const int ci = j / p.tpc;
        const int t = j - ci * p.tpc;
        const int plane = ((rd.page[ti][ci] * g.L + p.layer) * 2 + isv) * g.H + h;
        const uint32_t dst = c.sbase + L::KV + st * L::KVTILE;
        mbar_arrive_expect_tx(c.bar(L::B_KVFULL + st), L::KVTILE);
        tma_load_3d(dst, tkv, c.bar(L::B_KVFULL + st), 0, t * L::BN, plane);
        if (!F8) tma_load_3d(dst + L::KVHALF, tkv, c.bar(L::B_KVFULL + st), 64, t * L::BN, plane);
        *issued = s + 1;
    }
}

// ---- MMA issuer ----------------------------------------------------------------
// S = Q K^T: M = 128, N = BN; K = 16 per instruction for bf16 (two 64-column
// halves of Q and K, at their own offsets), 32 for e4m3.
template <bool F8>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_addr, uint32_t k_addr) {
    using L = L2<F8>;
    if constexpr (F8) {
        constexpr uint32_t idesc = idesc_e4m3_f32(BM, L::BN, false);
#pragma unroll
        for (int kk = 0; kk < HD / 32; ++kk)
            mma_ss_f8(d_tmem, sdesc_sw128(q_addr + kk * 32, 16, 1024),
                      sdesc_sw128(k_addr + kk * 32, 16, 1024), idesc, kk > 0 ? 1u : 0u);
    } else {
        constexpr uint32_t idesc = idesc_bf16_f32(BM, L::BN, false);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk)
            mma_ss(d_tmem, sdesc_sw128(q_addr + (kk >> 2) * L::QHALF + (kk & 3) * 32, 16, 1024),
                   sdesc_sw128(k_addr + (kk >> 2) * L::KVHALF + (kk & 3) * 32, 16, 1024), idesc,
                   kk > 0 ? 1u : 0u);
    }
}
// O += P V: P from TMEM (bf16: 2 keys per column, e4m3: 4), V the MN-major B
// operand (keys along K, rows of 128 bytes, 8-row groups 1 KB apart, the two
// 64-column halves of a bf16 tile KVHALF apart).
template <bool F8>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_addr, bool acc) {
    using L = L2<F8>;
    if constexpr (F8) {
        constexpr uint32_t idesc = idesc_e4m3_f32(BM, HD, true);
#pragma unroll
        for (int kk = 0; kk < L::BN / 32; ++kk)
            mma_ts_f8(d_tmem, p_tmem + kk * 8, sdesc_sw128(v_addr + kk * 4096, L::KVHALF, 1024), idesc,
                      (acc || kk > 0) ? 1u : 0u);
    } else {
        constexpr uint32_t idesc = idesc_bf16_f32(BM, HD, true);
#pragma unroll
        for (int kk = 0; kk < L::BN / 16; ++kk)
            mma_ts(d_tmem, p_tmem + kk * 8, sdesc_sw128(v_addr + kk * 2048, L::KVHALF, 1024), idesc,
                   (acc || kk > 0) ? 1u : 0u);
    }
}

// Global iteration g = it_base + j counts key tiles over the CTA's units;
// every per-tile barrier completes one phase per iteration.
template <bool F8>
__device__ void mma_issuer(const Ctx2<F8> &c, uint32_t tmem, int n, uint32_t seq, uint32_t it_base,
                           uint32_t unit_iter) {
    using L = L2<F8>;
    const uint32_t qa[2] = {c.sbase + L::Q0, c.sbase + L::Q1};
    if (!c.wait(L::B_QFULL, unit_iter & 1, 2)) return;
    tc_fence_after();
    for (int j = 0; j < n; ++j) {
        const uint32_t gi = it_base + j;
        const uint32_t ks = seq + kseq(j);
        const int kst = ks % L::NST;
        if (!c.wait(L::B_KVFULL + kst, (ks / L::NST) & 1, 3)) return;
        tc_fence_after();
        const uint32_t ka = c.sbase + L::KV + kst * L::KVTILE;
        for (int x = 0; x < 2; ++x) {
            // the softmax has read the previous S of this tile
            if (gi > 0 && !c.wait(L::B_SFREE + x, (gi - 1) & 1, 4 + x)) return;
            tc_fence_after();
            issue_qk<F8>(tmem + 128 * x, qa[x], ka);
            mma_commit(c.bar(L::B_SFULL + x));
        }
        mma_commit(c.bar(L::B_KVEMPTY + kst));
        if (j == 0) continue;
        const uint32_t vs = seq + vseq(j - 1, n);
        const int vst = vs % L::NST;
        if (!c.wait(L::B_KVFULL + vst, (vs / L::NST) & 1, 6)) return;
        const uint32_t va = c.sbase + L::KV + vst * L::KVTILE;
        for (int x = 0; x < 2; ++x) {
            if (!c.wait(L::B_PFULL + x, (gi - 1) & 1, 7 + x)) return;
            tc_fence_after();
            issue_pv<F8>(tmem + 256 + 128 * x, tmem + 128 * x + L::BN, va, j - 1 > 0);
            mma_commit(c.bar(L::B_PVDONE + x));
        }
        mma_commit(c.bar(L::B_KVEMPTY + vst));
    }
    const uint32_t gl = it_base + n - 1;
    const uint32_t vs = seq + vseq(n - 1, n);
    const int vst = vs % L::NST;
    if (!c.wait(L::B_KVFULL + vst, (vs / L::NST) & 1, 9)) return;
    const uint32_t va = c.sbase + L::KV + vst * L::KVTILE;
    for (int x = 0; x < 2; ++x) {
        if (!c.wait(L::B_PFULL + x, gl & 1, 10 + x)) return;
        tc_fence_after();
        issue_pv<F8>(tmem + 256 + 128 * x, tmem + 128 * x + L::BN, va, n - 1 > 0);
        mma_commit(c.bar(L::B_PVDONE + x));
    }
    mma_commit(c.bar(L::B_KVEMPTY + vst));
}

// ---- softmax / epilogue -------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// One row's BN scores from TMEM (columns col .. col + BN - 1).
template <bool F8>
__device__ __forceinline__ void load_scores(uint32_t tS, uint32_t (&r)[L2<F8>::BN]) {
    if constexpr (F8) {                       // 96 = 6 x 16
        tmem_ld16(tS + 0, r + 0);
        tmem_ld16(tS + 16, r + 16);
        tmem_ld16(tS + 32, r + 32);
        tmem_ld16(tS + 48, r + 48);
        tmem_ld16(tS + 64, r + 64);
        tmem_ld16(tS + 80, r + 80);
#pragma unroll
        for (int q = 0; q < 6; ++q) tmem_wait_ld16(r + 16 * q);
    } else {                                  // 80 = 5 x 16
        tmem_ld16(tS + 0, r + 0);
        tmem_ld16(tS + 16, r + 16);
        tmem_ld16(tS + 32, r + 32);
        tmem_ld16(tS + 48, r + 48);
        tmem_ld16(tS + 64, r + 64);
#pragma unroll
        for (int q = 0; q < 5; ++q) tmem_wait_ld16(r + 16 * q);
    }
}

template <bool F8>
__device__ void softmax_tile(const Ctx2<F8> &c, uint32_t tmem, const WfGeom &g, const WfRoundDev &rd,
                             const Tc2Params &p, int X, int ti, int h, int qp, int n, uint32_t it_base) {
    using L = L2<F8>;
    constexpr int BN = L::BN;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + X * 128;
    const uint32_t tP = tS + BN;
    const uint32_t tO = tmem + lane_off + 256 + X * 128;
    const float sl2 = p.sl2;
    float m_run = -INFINITY, l_run = 0.f;

    for (int j = 0; j < n; ++j) {
        const uint32_t gi = it_base + j;
        bool ok = c.wait(L::B_SFULL + X, gi & 1, 12 + X);
        if (!__all_sync(0xffffffffu, ok)) return;
        tc_fence_after();
        uint32_t r[BN];
        load_scores<F8>(tS, r);
        // S has been read: the issuer may compute the next S into it
        tc_fence_before();
        mbar_arrive(c.bar(L::B_SFREE + X));
        const int t = j % p.tpc;
        const int valid = g.NC - t * BN;
        if (valid < BN) {
#pragma unroll
            for (int i = 0; i < BN; ++i)
                if (i >= valid) r[i] = __float_as_uint(-INFINITY);
        }
        // row max: BN / 16 independent chains of 3-input max over 16 scores
        constexpr int NCH = BN / 16;
        float pm[NCH];
#pragma unroll
        for (int a = 0; a < NCH; ++a) {
            const uint32_t *v = &r[a * 16];
            float m = fmax3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
#pragma unroll
            for (int i = 3; i < 15; i += 2) m = fmax3(m, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
            pm[a] = fmaxf(m, __uint_as_float(v[15]));
        }
        float mx = pm[0];
#pragma unroll
        for (int a = 1; a < NCH; ++a) mx = fmaxf(mx, pm[a]);
        const float mnew = mx * sl2;
        float alpha = 1.f;
        if (mnew > m_run + 8.f) {
            alpha = ex2(m_run - mnew);
            m_run = mnew;
        }
        bool pv_done = gi == 0;   // nothing of this tile's earlier P V is pending
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
            // O holds P V up to tile j - 1 only once that product has completed
            ok = c.wait(L::B_PVDONE + X, (gi - 1) & 1, 14 + X);
            if (!__all_sync(0xffffffffu, ok)) return;
            tc_fence_after();
            pv_done = true;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t o[32];
                tmem_ld32(tO + q * 32, o);
                tmem_wait_ld(o);
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                tmem_st32(tO + q * 32, o);
            }
        }
        // p = 2^(s*sl2 - m_run) on packed pairs; packed partial sums
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        const uint64_t negm2 = f2_pack(-m_run, -m_run);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        uint32_t pk[L::PCOLS];
#pragma unroll
        for (int i = 0; i < BN / 2; ++i) {
            const uint64_t x = f2_fma(f2_pack(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])),
                                      sl2x2, negm2);
            float a0, a1;
            f2_unpack(x, a0, a1);
            const float p0 = ex2(a0), p1 = ex2(a1);
            acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
            if constexpr (F8) {
                const uint32_t hb = pack_e4m3x2(p0, p1);
                uint32_t &w = pk[i >> 1];
                w = (i & 1) ? (w | (hb << 16)) : hb;
            } else {
                pk[i] = pack_bf16(p0, p1);
            }
        }
        float s0, s1, s2, s3;
        f2_unpack(f2_add(acc[0], acc[1]), s0, s1);
        f2_unpack(f2_add(acc[2], acc[3]), s2, s3);
        l_run = l_run * alpha + ((s0 + s1) + (s2 + s3));
        if (!pv_done) {
            // P(j) overwrites P(j - 1): its P V must have completed
            ok = c.wait(L::B_PVDONE + X, (gi - 1) & 1, 16 + X);
            if (!__all_sync(0xffffffffu, ok)) return;
            tc_fence_after();
        }
        if constexpr (F8) {                   // 24 columns
            tmem_st16(tP, pk);
            tmem_st8(tP + 16, pk + 16);
        } else {                              // 40 columns
            tmem_st32(tP, *reinterpret_cast<const uint32_t(*)[32]>(pk));
            tmem_st8(tP + 32, pk + 32);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(c.bar(L::B_PFULL + X));
    }

    bool ok = c.wait(L::B_PVDONE + X, (it_base + n - 1) & 1, 18 + X);
    if (!__all_sync(0xffffffffu, ok)) return;
    tc_fence_after();
    const int qrow = (2 * qp + X) * BM + row;
    const float inv = p.o_scale / l_run;
    const size_t o_off = (((size_t)rd.slot[ti] * g.NC + qrow) * g.H + h) * HD;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t o[32];
        tmem_ld32(tO + q * 32, o);
        tmem_wait_ld(o);
        if (qrow < g.NC) {
            if (p.out_e4m3) {
                uint32_t w[8];
#pragma unroll
                for (int v = 0; v < 8; ++v)
                    w[v] = pack_e4m3x2(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv) |
                           (pack_e4m3x2(__uint_as_float(o[4 * v + 2]) * inv,
                                        __uint_as_float(o[4 * v + 3]) * inv) << 16);
                uint4 *d4 = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(p.out) + o_off + q * 32);
                d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
                d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
            } else {
                uint4 *d4 = reinterpret_cast<uint4 *>(p.out + o_off + q * 32);
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    uint4 w;
                    w.x = pack_bf16(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
                    w.y = pack_bf16(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
                    w.z = pack_bf16(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
                    w.w = pack_bf16(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
                    d4[v] = w;
                }
            }
        }
    }
}

template <bool F8>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_tc2_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tkv,
                    const WfGeom g, const WfRoundDev rd, const Tc2Params p) {
    using L = L2<F8>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_u32 & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    Ctx2<F8> c;
    c.sbase = raw_u32 + pad;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC);
    int *unit_slot = reinterpret_cast<int *>(smem + L::MISC + 8);
    c.abort = reinterpret_cast<volatile int *>(smem + L::MISC + 16);
    c.status = p.stat + WF_SCRATCH_STATUS / 4;
    c.where = p.stat + WF_SCRATCH_WHERE / 4;
    uint32_t *work = p.ctl + WF_SCRATCH_WORK / 4;
    uint32_t *done = p.ctl + WF_SCRATCH_DONE / 4;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(c.bar(L::B_QFULL), 1);
        for (int i = 0; i < L::NST; ++i) {
            mbar_init(c.bar(L::B_KVFULL + i), 1);
            mbar_init(c.bar(L::B_KVEMPTY + i), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(c.bar(L::B_SFULL + x), 1);
            mbar_init(c.bar(L::B_SFREE + x), 128);
            mbar_init(c.bar(L::B_PFULL + x), 128);
            mbar_init(c.bar(L::B_PVDONE + x), 1);
        }
        mbar_init(c.bar(L::B_DRAIN), 1);
        mbar_fence_init();
        *c.abort = 0;
        unit_slot[0] = blockIdx.x;
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tkv);
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    uint32_t seq = 0, it_base = 0, unit_iter = 0, issued = 0;
    auto next_unit = [&](int n) -> int {
        seq += 2 * n;
        it_base += n;
        unit_iter += 1;
        if (threadIdx.x == 0) unit_slot[unit_iter & 1] = (int)(gridDim.x + atomicAdd(work, 1u));
        tc_fence_before();
        named_bar_sync(1, NUM_THREADS);
        tc_fence_after();
        return *c.abort ? p.n_units : unit_slot[unit_iter & 1];
    };
    if (warp < 8) {
        reg_inc<REGS_SOFTMAX>();
        for (int u = unit_slot[0]; u < p.n_units;) {
            int ti, h, qp;
            decode_unit(u, rd, p, g.H, ti, h, qp);
            const int n = rd.n_ctx[ti] * p.tpc;
            softmax_tile<F8>(c, tmem, g, rd, p, warp >> 2, ti, h, qp, n, it_base);
            u = next_unit(n);
        }
    } else {
        reg_dec<REGS_AUX>();
        for (int u = unit_slot[0]; u < p.n_units;) {
            int ti, h, qp;
            decode_unit(u, rd, p, g.H, ti, h, qp);
            const int n = rd.n_ctx[ti] * p.tpc;
            if (warp == 8 && lane == 0)
                producer<F8>(c, &tq, &tkv, g, rd, p, ti, h, qp, n, seq, &issued);
            else if (warp == 9 && lane == 0)
                mma_issuer<F8>(c, tmem, n, seq, it_base, unit_iter);
            u = next_unit(n);
        }
    }

    if (*c.abort) {
        // let the copies and MMAs this CTA started land before TMEM and
        // shared memory are released
        if (warp == 8 && lane == 0) {
            uint32_t first = issued > (uint32_t)L::NST ? issued - L::NST : 0;
            for (uint32_t s = first; s < issued; ++s)
                mbar_wait(c.bar(L::B_KVFULL + s % L::NST), (s / L::NST) & 1, nullptr, nullptr, nullptr, 0,
                          WAIT_NS);
            if (unit_iter > 0)
                mbar_wait(c.bar(L::B_QFULL), (unit_iter - 1) & 1, nullptr, nullptr, nullptr, 0, WAIT_NS);
        }
        if (warp == 9 && lane == 0) {
            mma_commit(c.bar(L::B_DRAIN));
            mbar_wait(c.bar(L::B_DRAIN), 0, nullptr, nullptr, nullptr, 0, WAIT_NS);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 9) tmem_dealloc(tmem, 512);
    if (threadIdx.x == 0) {
        __threadfence();
        uint32_t prev = atomicAdd(done, 1u);
        if (prev == gridDim.x - 1) {
            atomicExch(work, 0u);
            atomicExch(done, 0u);
        }
    }
}

template <bool F8>
cudaError_t prepare_kernel() {
    static std::atomic<unsigned long long> done{0};
    return wf_once_per_device(done, [] {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, attn_tc2_kernel<F8>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != LAUNCH_REGS) return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(attn_tc2_kernel<F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    L2<F8>::ALLOC);
    });
}

}  // namespace

int wf_attn_tc2_keys(int dtype) { return dtype == WF_FP8 ? L2<true>::BN : L2<false>::BN; }

cudaError_t wf_launch_attn_tc2(const WfGeom &g, const WfRoundDev &rd, int layer, const WfTmaps &maps,
                               void *out, void *scratch, int num_sms, cudaStream_t stream, int out_e4m3) {
    if (rd.n_tasks < 1) return cudaSuccess;
    const bool f8 = g.dtype == WF_FP8;
    cudaError_t e = f8 ? prepare_kernel<true>() : prepare_kernel<false>();
    if (e != cudaSuccess) return e;
    const int bn = wf_attn_tc2_keys(g.dtype);
    Tc2Params p;
    p.layer = layer;
    p.tpc = (g.NC + bn - 1) / bn;
    p.qpairs = ((g.NC + BM - 1) / BM + 1) / 2;
    p.n_units = rd.n_tasks * g.H * p.qpairs;
    p.sl2 = 1.4426950408889634f / sqrtf((float)HD);
    p.o_scale = 1.f;
    if (f8) {
        p.sl2 /= g.qk_scale * g.qk_scale;
        p.o_scale = 1.f / g.v_scale;
    }
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.out_e4m3 = out_e4m3;
    p.ctl = static_cast<uint32_t *>(scratch);
    p.stat = static_cast<uint32_t *>(scratch);
    const int grid = p.n_units < num_sms ? p.n_units : num_sms;
    if (f8)
        attn_tc2_kernel<true><<<grid, NUM_THREADS, L2<true>::ALLOC, stream>>>(maps.q, maps.kv2, g, rd, p);
    else
        attn_tc2_kernel<false><<<grid, NUM_THREADS, L2<false>::ALLOC, stream>>>(maps.q, maps.kv2, g, rd, p);
    return cudaGetLastError();
}
