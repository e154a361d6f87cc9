// Round attention on the 5th-generation tensor cores (bf16, head_dim 128).
//
// What it computes ("Wave Forcing", Sec. 3.1 Eq. 4-5): for every active task
// of the round (chunk k - s at stage s, plus the store at stage S) and every
// head, O = softmax(Q K^T / sqrt(D)) V over the task's ordered context --
// anchor, bounded history, live store, live stages j >= s -- with full
// (bidirectional) attention inside each chunk.  The mask is applied at chunk
// granularity by construction: a task's key stream is exactly the pages of
// its context, so masked-out chunk blocks are never loaded or multiplied.
// Only the ragged last key tile of each chunk (N_C mod 128 valid keys) needs
// an element mask.
//
// Design (one persistent CTA per SM, 384 threads):
//  * work unit = (task, head, pair of 128-row query tiles); units are handed
//    out through an atomic counter in scratch, in blocks of a few heads
//    (longest context first inside a block), the block size chosen on the
//    host by simulating the hand-out: it sets how the longest units spread
//    over the waves, and a block whose pages fit in L2 lets the round's
//    tasks, which share most of their pages, read each page from DRAM once;
//  * warp 8 (one thread): TMA producer -- both Q tiles, then K_0, K_1, V_0,
//    K_2, V_1, ... through a 4-stage ring of 32 KB tiles (128B swizzle); the
//    pages are read through a 3D tensor map [plane][N_C][128], so rows past
//    N_C are zero-filled by the TMA unit;
//  * warp 9 (one thread): tcgen05.mma issuer.  S = Q K^T (SS, fp32 in TMEM)
//    and O += P V (P read from TMEM, V MN-major from shared memory), the two
//    query tiles interleaved so one tile's softmax overlaps the other tile's
//    MMAs;
//  * warps 0-3 / 4-7: softmax of tile 0 / tile 1.  Thread r owns query row r:
//    tcgen05.ld of its 128 scores, row max in registers, exp2, P packed to
//    bf16 and written back over S in TMEM.  The running max is only raised
//    when it grows by more than 2^8, and O is rescaled in TMEM only then.
//  * TMEM (512 columns): S0 | S1 | O0 | O1, P aliasing the first 64 columns of S.
//
// Every wait is bounded (%globaltimer); on a timeout the kernel records it in
// the scratch status word, drains its own copies and MMAs, frees TMEM and
// returns.

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <mutex>

#include "wf_internal.h"
#include "wf_ptx.cuh"

using namespace wfptx;

namespace {

constexpr int BM = 128;             // query rows per tile
constexpr int BN = 128;             // keys per tile
constexpr int HD = 128;             // head dim
constexpr int NST = 4;              // K/V ring stages
constexpr int NUM_THREADS = 384;

// Shared-memory layout of one CTA.  bf16: a 128 x 128 tile is two 64-column
// halves of 128-byte rows (16 KB each); e4m3: one block of 128-byte rows.
template <bool F8>
struct Lay {
    static constexpr uint32_t TILE = BM * HD * (F8 ? 1 : 2);
    static constexpr uint32_t HALF = F8 ? TILE : TILE / 2;  // one 128-byte-wide column block
    static constexpr uint32_t Q0 = 0;
    static constexpr uint32_t Q1 = TILE;
    static constexpr uint32_t KV = 2 * TILE;
    static constexpr uint32_t BAR = KV + NST * TILE;
};

constexpr int B_QFULL = 0;
constexpr int B_KVFULL = 1;
constexpr int B_KVEMPTY = B_KVFULL + NST;
constexpr int B_SFULL = B_KVEMPTY + NST;
constexpr int B_PFULL = B_SFULL + 2;
constexpr int B_ODONE = B_PFULL + 2;
constexpr int B_DRAIN = B_ODONE + 2;
constexpr int NBARS = B_DRAIN + 1;

template <bool F8>
struct LayMisc {
    static constexpr uint32_t MISC = Lay<F8>::BAR + ((NBARS * 8 + 63) / 64) * 64;
    static constexpr uint32_t ALLOC = MISC + 64 + 1024;   // + alignment slack
};

constexpr uint64_t WAIT_NS = 1000000000ull;  // 1 s

// Register split: the kernel is launched with LAUNCH_REGS per thread (384 x
// 168 = 64512 of the SM's 65536); the producer/MMA warpgroup gives up
// 4 warps x 32 x (168 - 56) registers and the two softmax warpgroups take
// 8 warps x 32 x (224 - 168) -- the same 14336, so the increase never waits.
constexpr int LAUNCH_REGS = 168;
constexpr int REGS_SOFTMAX = 224;
constexpr int REGS_AUX = 56;
static_assert(8 * (REGS_SOFTMAX - LAUNCH_REGS) <= 4 * (LAUNCH_REGS - REGS_AUX),
              "register split exceeds the launch pool");

struct TcParams {
    int layer;
    int n_units;
    int qpairs;           // pairs of query tiles per (task, head)
    int hblk;             // heads per block of the unit order
    int tpc;              // key tiles per chunk
    float sl2;            // log2(e) / sqrt(D) (/ qk_scale^2 for e4m3 Q and K)
    float o_scale;        // 1 (bf16) or 1 / v_scale (e4m3 V)
    __nv_bfloat16 *out;   // [slot][N_C][H][D] bf16, or e4m3 bytes when out_e4m3
    int out_e4m3;         // O as e4m3 (unit scale): the input of an e4m3 output projection
    uint32_t *ctl;        // scheduler counters (work, finished CTAs)
    uint32_t *stat;       // status and wait-site words (the plan's scratch, read by wf_sync_status)
};

__device__ __forceinline__ int kseq(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int vseq(int j, int n) { return j == n - 1 ? 2 * n - 1 : 2 * j + 2; }

template <bool F8>
struct Ctx {
    uint32_t sbase;
    volatile int *abort;
    uint32_t *status, *where;
    __device__ uint32_t bar(int i) const { return sbase + Lay<F8>::BAR + 8u * i; }
    __device__ bool wait(int b, uint32_t parity, uint32_t site) const {
        return mbar_wait(bar(b), parity, abort, status, where, site, WAIT_NS);
    }
};

// Unit order: blocks of hblk heads; inside a block the tasks longest
// context first (rd.lpt), then the block's heads, then the pairs of query
// tiles.  The tasks of a round share most of their context pages, so a
// block whose pages fit in L2 reads each (page, head) from DRAM about once;
// hblk = H is plain longest-first order over (task, head).
__device__ __forceinline__ void decode_unit(int u, const WfRoundDev &rd, const TcParams &p, int H,
                                            int &ti, int &h, int &qp) {
    const int per_block = rd.n_tasks * p.hblk * p.qpairs;
    const int b = u / per_block;                       // the last block may hold fewer heads
    const int h0 = b * p.hblk;
    const int nh = min(p.hblk, H - h0);
    const int rem = u - b * per_block;
    const int per_task = nh * p.qpairs;
    const int oi = rem / per_task;
    const int r2 = rem - oi * per_task;
    ti = rd.lpt[oi];
    h = h0 + r2 / p.qpairs;
    qp = r2 - (r2 / p.qpairs) * p.qpairs;
}

// ---- producer ----------------------------------------------------------------
template <bool F8>
__device__ void producer(const Ctx<F8> &c, const CUtensorMap *tq, const CUtensorMap *tkv,
                         const WfGeom &g, const WfRoundDev &rd, const TcParams &p, int ti, int h,
                         int qp, int n, uint32_t seq, uint32_t *issued) {
    using L = Lay<F8>;
    const int plane_q = rd.slot[ti] * g.H + h;
    mbar_arrive_expect_tx(c.bar(B_QFULL), 2 * L::TILE);
    for (int x = 0; x < 2; ++x) {
        const uint32_t dst = c.sbase + (x ? L::Q1 : L::Q0);
        tma_load_3d(dst, tq, c.bar(B_QFULL), 0, (2 * qp + x) * BM, plane_q);
        if (!F8) tma_load_3d(dst + L::HALF, tq, c.bar(B_QFULL), 64, (2 * qp + x) * BM, plane_q);
    }
    for (int i = 0; i < 2 * n; ++i) {
        int j;
        int isv;
        if (i == 0) {
            j = 0; isv = 0;
        } else if (i == 2 * n - 1) {
            j = n - 1; isv = 1;
        } else if (i & 1) {
            j = (i + 1) / 2; isv = 0;
        } else {
            j = i / 2 - 1; isv = 1;
        }
        uint32_t s = seq + i;
        int st = s % NST;
        if (!c.wait(B_KVEMPTY + st, ((s / NST) & 1) ^ 1, 1)) return;
        int ci = j / p.tpc;
        int t = j - ci * p.tpc;
        int plane = ((rd.page[ti][ci] * g.L + p.layer) * 2 + isv) * g.H + h;
        uint32_t dst = c.sbase + L::KV + st * L::TILE;
        mbar_arrive_expect_tx(c.bar(B_KVFULL + st), L::TILE);
        tma_load_3d(dst, tkv, c.bar(B_KVFULL + st), 0, t * BN, plane);
        if (!F8) tma_load_3d(dst + L::HALF, tkv, c.bar(B_KVFULL + st), 64, t * BN, plane);
        *issued = s + 1;
    }
}

// ---- MMA issuer ----------------------------------------------------------------
// S = Q K^T: K = 16 per instruction for bf16 (two 64-column halves), 32 for
// e4m3 (one 128-byte block); the descriptor start advances 32 bytes a step.
template <bool F8>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_addr, uint32_t k_addr) {
    if constexpr (F8) {
        constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN, false);
#pragma unroll
        for (int kk = 0; kk < HD / 32; ++kk)
            mma_ss_f8(d_tmem, sdesc_sw128(q_addr + kk * 32, 16, 1024),
                      sdesc_sw128(k_addr + kk * 32, 16, 1024), idesc, kk > 0 ? 1u : 0u);
    } else {
        constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, false);
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
            uint32_t off = (kk >> 2) * Lay<false>::HALF + (kk & 3) * 32;
            mma_ss(d_tmem, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(k_addr + off, 16, 1024),
                   idesc, kk > 0 ? 1u : 0u);
        }
    }
}
// O += P V: P from TMEM (bf16: 2 keys per column, e4m3: 4), V the MN-major B
// operand (keys along K, rows of 128 bytes; 8-row groups 1 KB apart).
template <bool F8>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_addr,
                                         bool acc) {
    if constexpr (F8) {
        constexpr uint32_t idesc = idesc_e4m3_f32(BM, HD, true);
#pragma unroll
        for (int kk = 0; kk < BN / 32; ++kk)
            mma_ts_f8(d_tmem, p_tmem + kk * 8, sdesc_sw128(v_addr + kk * 4096, Lay<true>::HALF, 1024),
                      idesc, (acc || kk > 0) ? 1u : 0u);
    } else {
        constexpr uint32_t idesc = idesc_bf16_f32(BM, HD, true);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(d_tmem, p_tmem + kk * 8, sdesc_sw128(v_addr + kk * 2048, Lay<false>::HALF, 1024),
                   idesc, (acc || kk > 0) ? 1u : 0u);
    }
}

template <bool F8>
__device__ void mma_issuer(const Ctx<F8> &c, uint32_t tmem, int n, uint32_t seq, uint32_t it_base,
                           uint32_t unit_iter) {
    const uint32_t tS0 = tmem, tS1 = tmem + 128, tO0 = tmem + 256, tO1 = tmem + 384;
    using L = Lay<F8>;
    const uint32_t q0 = c.sbase + L::Q0, q1 = c.sbase + L::Q1;
    if (!c.wait(B_QFULL, unit_iter & 1, 2)) return;
    tc_fence_after();
    for (int j = 0; j < n; ++j) {
        uint32_t ks = seq + kseq(j);
        int kst = ks % NST;
        if (!c.wait(B_KVFULL + kst, (ks / NST) & 1, 3)) return;
        tc_fence_after();
        uint32_t ka = c.sbase + L::KV + kst * L::TILE;
        if (j == 0) {
            issue_qk<F8>(tS0, q0, ka);
            mma_commit(c.bar(B_SFULL + 0));
            issue_qk<F8>(tS1, q1, ka);
            mma_commit(c.bar(B_SFULL + 1));
            mma_commit(c.bar(B_KVEMPTY + kst));
            continue;
        }
        uint32_t vs = seq + vseq(j - 1, n);
        int vst = vs % NST;
        if (!c.wait(B_KVFULL + vst, (vs / NST) & 1, 4)) return;
        uint32_t va = c.sbase + L::KV + vst * L::TILE;
        uint32_t par = (it_base + j - 1) & 1;
        if (!c.wait(B_PFULL + 0, par, 5)) return;
        tc_fence_after();
        issue_pv<F8>(tO0, tS0, va, j - 1 > 0);
        issue_qk<F8>(tS0, q0, ka);
        mma_commit(c.bar(B_SFULL + 0));
        if (!c.wait(B_PFULL + 1, par, 6)) return;
        tc_fence_after();
        issue_pv<F8>(tO1, tS1, va, j - 1 > 0);
        mma_commit(c.bar(B_KVEMPTY + vst));
        issue_qk<F8>(tS1, q1, ka);
        mma_commit(c.bar(B_SFULL + 1));
        mma_commit(c.bar(B_KVEMPTY + kst));
    }
    uint32_t vs = seq + vseq(n - 1, n);
    int vst = vs % NST;
    if (!c.wait(B_KVFULL + vst, (vs / NST) & 1, 7)) return;
    uint32_t va = c.sbase + L::KV + vst * L::TILE;
    uint32_t par = (it_base + n - 1) & 1;
    if (!c.wait(B_PFULL + 0, par, 8)) return;
    tc_fence_after();
    issue_pv<F8>(tO0, tS0, va, n - 1 > 0);
    mma_commit(c.bar(B_ODONE + 0));
    if (!c.wait(B_PFULL + 1, par, 9)) return;
    tc_fence_after();
    issue_pv<F8>(tO1, tS1, va, n - 1 > 0);
    mma_commit(c.bar(B_ODONE + 1));
    mma_commit(c.bar(B_KVEMPTY + vst));
}

// ---- softmax / epilogue -------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
// Two floats to e4m3 (round to nearest even, saturating): lo in the low byte.
__device__ __forceinline__ uint32_t pack_e4m3x2(float lo, float hi) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

template <bool F8>
__device__ void softmax_tile(const Ctx<F8> &c, uint32_t tmem, const WfGeom &g, const WfRoundDev &rd,
                             const TcParams &p, int X, int ti, int h, int qp, int n,
                             uint32_t it_base, uint32_t unit_iter) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
    const uint32_t tS = tmem + lane_off + X * 128;
    const uint32_t tO = tmem + lane_off + 256 + X * 128;
    const float sl2 = p.sl2;
    float m_run = -INFINITY, l_run = 0.f;

    for (int j = 0; j < n; ++j) {
        bool ok = c.wait(B_SFULL + X, (it_base + j) & 1, 10 + X);
        if (!__all_sync(0xffffffffu, ok)) return;
        tc_fence_after();
        uint32_t r[4][32];
        tmem_ld32(tS + 0, r[0]);
        tmem_ld32(tS + 32, r[1]);
        tmem_ld32(tS + 64, r[2]);
        tmem_ld32(tS + 96, r[3]);
        tmem_wait_ld(r[0]);
        tmem_wait_ld(r[1]);
        tmem_wait_ld(r[2]);
        tmem_wait_ld(r[3]);
        const int t = j % p.tpc;
        const int valid = g.NC - t * BN;
        if (valid < BN) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (q * 32 + i >= valid) r[q][i] = __float_as_uint(-INFINITY);
        }
        // row max: 8 independent chains of 3-input max over 16 scores each
        float pm[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) {
            const uint32_t *v = &r[a >> 1][(a & 1) * 16];
            float m = fmax3(__uint_as_float(v[0]), __uint_as_float(v[1]), __uint_as_float(v[2]));
#pragma unroll
            for (int i = 3; i < 15; i += 2) m = fmax3(m, __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
            pm[a] = fmaxf(m, __uint_as_float(v[15]));
        }
        const float mx = fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]),
                               fmaxf(pm[6], pm[7]));
        const float mnew = mx * sl2;
        float alpha = 1.f;
        if (mnew > m_run + 8.f) {
            alpha = ex2(m_run - mnew);
            m_run = mnew;
        }
        // p = 2^(s*sl2 - m_run) on packed pairs; 4 independent packed partial sums
        const uint64_t sl2x2 = f2_pack(sl2, sl2);
        const uint64_t negm2 = f2_pack(-m_run, -m_run);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        // P for the PV MMA: bf16 pairs (64 TMEM columns) or e4m3 quads (32)
        uint32_t pk[2][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                uint64_t x = f2_fma(f2_pack(__uint_as_float(r[q][2 * i]), __uint_as_float(r[q][2 * i + 1])),
                                    sl2x2, negm2);
                float a0, a1;
                f2_unpack(x, a0, a1);
                const float p0 = ex2(a0), p1 = ex2(a1);
                acc[i & 3] = f2_add(acc[i & 3], f2_pack(p0, p1));
                if constexpr (F8) {
                    const uint32_t h = pack_e4m3x2(p0, p1);
                    uint32_t &w = pk[0][q * 8 + (i >> 1)];
                    w = (i & 1) ? (w | (h << 16)) : h;
                } else {
                    pk[q >> 1][(q & 1) * 16 + i] = pack_bf16(p0, p1);
                }
            }
        }
        float s0, s1, s2, s3;
        f2_unpack(f2_add(acc[0], acc[1]), s0, s1);
        f2_unpack(f2_add(acc[2], acc[3]), s2, s3);
        const float sum = (s0 + s1) + (s2 + s3);
        l_run = l_run * alpha + sum;
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
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
        tmem_st32(tS + 0, pk[0]);
        if (!F8) tmem_st32(tS + 32, pk[1]);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(c.bar(B_PFULL + X));
    }

    bool ok = c.wait(B_ODONE + X, unit_iter & 1, 12 + X);
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
    attn_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tkv,
                   const WfGeom g, const WfRoundDev rd, const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_u32 & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    constexpr uint32_t MISC = LayMisc<F8>::MISC;
    Ctx<F8> c;
    c.sbase = raw_u32 + pad;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + MISC);
    int *unit_slot = reinterpret_cast<int *>(smem + MISC + 8);
    c.abort = reinterpret_cast<volatile int *>(smem + MISC + 16);
    c.status = p.stat + WF_SCRATCH_STATUS / 4;
    c.where = p.stat + WF_SCRATCH_WHERE / 4;
    uint32_t *work = p.ctl + WF_SCRATCH_WORK / 4;
    uint32_t *done = p.ctl + WF_SCRATCH_DONE / 4;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(c.bar(B_QFULL), 1);
        for (int i = 0; i < NST; ++i) {
            mbar_init(c.bar(B_KVFULL + i), 1);
            mbar_init(c.bar(B_KVEMPTY + i), 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(c.bar(B_SFULL + x), 1);
            mbar_init(c.bar(B_PFULL + x), 128);
            mbar_init(c.bar(B_ODONE + x), 1);
        }
        mbar_init(c.bar(B_DRAIN), 1);
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

    // Every role walks the same unit sequence; units end on named barrier 1
    // over all 384 threads, after which the next unit index (fetched by
    // thread 0) is read.  Each role has its own loop so that the register
    // budget set right before it applies to the whole loop.
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
            softmax_tile<F8>(c, tmem, g, rd, p, warp >> 2, ti, h, qp, n, it_base, unit_iter);
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
        // give the copies and MMAs this CTA started time to land before TMEM
        // and shared memory are released
        if (warp == 8 && lane == 0) {
            uint32_t first = issued > (uint32_t)NST ? issued - NST : 0;
            for (uint32_t s = first; s < issued; ++s)
                mbar_wait(c.bar(B_KVFULL + s % NST), (s / NST) & 1, nullptr, nullptr, nullptr, 0,
                          WAIT_NS);
            if (unit_iter > 0)  // the Q tiles of the unit that was cut short
                mbar_wait(c.bar(B_QFULL), (unit_iter - 1) & 1, nullptr, nullptr, nullptr, 0,
                          WAIT_NS);
        }
        if (warp == 9 && lane == 0) {
            mma_commit(c.bar(B_DRAIN));
            mbar_wait(c.bar(B_DRAIN), 0, nullptr, nullptr, nullptr, 0, WAIT_NS);
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

// Opt in to the shared-memory size and refuse to launch unless the kernel was
// compiled to exactly the register count the setmaxnreg split assumes.
template <bool F8>
cudaError_t prepare_kernel() {
    static std::atomic<unsigned long long> done{0};
    return wf_once_per_device(done, [] {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, attn_tc_kernel<F8>);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != LAUNCH_REGS) return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(attn_tc_kernel<F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    LayMisc<F8>::ALLOC);
    });
}

// ---- unit order ----------------------------------------------------------------
// Finish time of the last CTA when `workers` persistent CTAs take the units
// in decode_unit's order for blocks of hblk heads, each the next unit as
// soon as it is free; a unit costs its key tiles plus a few tiles' worth of
// Q loads and O stores.
double simulate_order(const WfRoundDev &rd, int H, int qpairs, int tpc, int hblk, int workers) {
    double heap[1024];                       // min-heap of the CTAs' busy-until times
    for (int i = 0; i < workers; ++i) heap[i] = 0.0;
    auto take = [&](double cost) {           // the earliest-free CTA takes the unit
        heap[0] += cost;
        int i = 0;
        for (;;) {
            int c = 2 * i + 1;
            if (c >= workers) break;
            if (c + 1 < workers && heap[c + 1] < heap[c]) ++c;
            if (heap[c] >= heap[i]) break;
            const double t = heap[c];
            heap[c] = heap[i];
            heap[i] = t;
            i = c;
        }
    };
    for (int h0 = 0; h0 < H; h0 += hblk) {
        const int nh = hblk < H - h0 ? hblk : H - h0;
        for (int oi = 0; oi < rd.n_tasks; ++oi) {
            const double cost = (double)rd.n_ctx[rd.lpt[oi]] * tpc + 3.0;
            for (int u = 0; u < nh * qpairs; ++u) take(cost);
        }
    }
    double end = 0.0;
    for (int i = 0; i < workers; ++i) end = heap[i] > end ? heap[i] : end;
    return end;
}

// Heads per block of the unit order.  Blocks of a few heads keep the pages
// the round's tasks share in L2, and the block size also sets how the
// longest units spread over the waves, so it is chosen by simulating the
// hand-out above for every candidate (1 .. 16 heads and H) and taking the
// shortest finish; among near-ties the blocks whose pages (K and V at bf16
// width) fit in about 80 MB of L2 win.  Cached per round shape (no
// allocation: a small fixed table).
int heads_per_block(const WfGeom &g, const WfRoundDev &rd, int qpairs, int tpc, int workers) {
    if (workers < 1 || workers > 1024 || rd.n_tasks < 1) return g.H;
    uint64_t key = 1469598103934665603ull;   // FNV-1a over the shape
    auto mix = [&](uint64_t v) { key = (key ^ v) * 1099511628211ull; };
    mix((uint64_t)g.H);
    mix((uint64_t)qpairs);
    mix((uint64_t)tpc);
    mix((uint64_t)workers);
    mix((uint64_t)g.NC);
    mix((uint64_t)rd.n_tasks);
    bool seen[256] = {};
    int distinct = 0;
    for (int i = 0; i < rd.n_tasks; ++i) {
        mix((uint64_t)rd.n_ctx[rd.lpt[i]]);
        for (int e = 0; e < rd.n_ctx[i]; ++e)
            if (!seen[rd.page[i][e]]) {
                seen[rd.page[i][e]] = true;
                ++distinct;
            }
    }
    mix((uint64_t)distinct);
    constexpr int kSlots = 64;
    static std::mutex mu;
    static uint64_t keys[kSlots];
    static int vals[kSlots];
    {
        std::lock_guard<std::mutex> lock(mu);
        const int slot = (int)(key % kSlots);
        if (vals[slot] > 0 && keys[slot] == key) return vals[slot];
    }
    const double head_bytes = (double)distinct * g.NC * HD * 2 * 2;
    const int fit = head_bytes > 0 ? (int)(80e6 / head_bytes) : g.H;
    int best = g.H;
    double best_t = 0.0;
    for (int G = 1; G <= g.H; ++G) {
        if (G > 16 && G != g.H) continue;
        double t = simulate_order(rd, g.H, qpairs, tpc, G, workers);
        if (G > fit) t *= 1.003;             // DRAM re-reads once the block leaves L2
        if (G == 1 || t < best_t) {
            best = G;
            best_t = t;
        }
    }
    std::lock_guard<std::mutex> lock(mu);
    const int slot = (int)(key % kSlots);
    keys[slot] = key;
    vals[slot] = best;
    return best;
}

// Parameters and launch of one round's attention (ctl: the scheduler
// counters; stat: the status and wait-site words).
cudaError_t launch_tc(const WfGeom &g, const WfRoundDev &rd, int layer, const WfTmaps &maps,
                      void *out, uint32_t *ctl, uint32_t *stat, int num_sms, cudaStream_t stream,
                      int out_e4m3 = 0) {
    const bool f8 = g.dtype == WF_FP8;
    cudaError_t e = f8 ? prepare_kernel<true>() : prepare_kernel<false>();
    if (e != cudaSuccess) return e;
    TcParams p;
    p.layer = layer;
    p.tpc = (g.NC + BN - 1) / BN;
    p.qpairs = ((g.NC + BM - 1) / BM + 1) / 2;
    p.n_units = rd.n_tasks * g.H * p.qpairs;
    const int grid = p.n_units < num_sms ? p.n_units : num_sms;
    p.hblk = heads_per_block(g, rd, p.qpairs, p.tpc, grid);
    p.sl2 = 1.4426950408889634f / sqrtf((float)HD);
    p.o_scale = 1.f;
    if (f8) {
        p.sl2 /= g.qk_scale * g.qk_scale;
        p.o_scale = 1.f / g.v_scale;
    }
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.out_e4m3 = out_e4m3;
    p.ctl = ctl;
    p.stat = stat;
    if (f8)
        attn_tc_kernel<true><<<grid, NUM_THREADS, LayMisc<true>::ALLOC, stream>>>(maps.q, maps.kv, g, rd, p);
    else
        attn_tc_kernel<false><<<grid, NUM_THREADS, LayMisc<false>::ALLOC, stream>>>(maps.q, maps.kv, g, rd, p);
    return cudaGetLastError();
}

}  // namespace

bool wf_attn_tc_supported(const WfGeom &g, int dtype) {
    return (dtype == WF_BF16 || dtype == WF_FP8) && g.D == HD;
}

cudaError_t wf_encode_tmaps(const WfGeom &g, void *qbuf, void *pool, WfTmaps *out, int n_req) {
    typedef CUresult (*EncodeFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    // looked up once (thread-safe static initialisation); the driver entry
    // point is the same for every device
    static const EncodeFn encode = [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            fn = nullptr;
        return reinterpret_cast<EncodeFn>(fn);
    }();
    if (!encode) return cudaErrorUnknown;
    // bf16: 64-element (128-byte) boxes, two per 128-wide tile; e4m3: one
    // 128-element (128-byte) box
    const bool f8 = g.dtype == WF_FP8;
    const cuuint64_t es = f8 ? 1 : 2;
    const CUtensorMapDataType ty = f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint32_t box[3] = {f8 ? 128u : 64u, 128, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const cuuint64_t strides[2] = {(cuuint64_t)HD * es, (cuuint64_t)g.NC * HD * es};
    cuuint64_t dq[3] = {(cuuint64_t)HD, (cuuint64_t)g.NC, (cuuint64_t)n_req * (g.S + 1) * g.H};
    if (encode(&out->q, ty, 3, qbuf, dq, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    cuuint64_t dk[3] = {(cuuint64_t)HD, (cuuint64_t)g.NC, (cuuint64_t)n_req * g.P * g.L * 2 * g.H};
    if (encode(&out->kv, ty, 3, pool, dk, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

cudaError_t wf_launch_attn_tc(const WfGeom &g, const WfRoundDev &rd, int layer,
                              const WfTmaps &maps, void *out, void *scratch, int num_sms,
                              cudaStream_t stream, int out_e4m3) {
    if (rd.n_tasks < 1) return cudaSuccess;
    return launch_tc(g, rd, layer, maps, out, static_cast<uint32_t *>(scratch),
                     static_cast<uint32_t *>(scratch), num_sms, stream, out_e4m3);
}

// ---- launch without caller scratch ------------------------------------------
// The attention kernel's scheduler counters (work counter, finished-CTA
// counter) in a fixed device block owned by the library.  Static device
// memory starts zeroed when the module loads; each call clears the counters
// on its stream before launching, so a call never inherits a previous call's
// counters.  All calls share this block: kernels that overlap on the GPU race
// on it.  A bounded-wait timeout is recorded where wf_round_attention records
// it -- the status word of the plan's scratch, which wf_sync_status reads --
// so a failed call is never hidden by the next call's clearing.
static __device__ __align__(256) uint32_t wf_noalloc_scratch[WF_NOALLOC_SCRATCH_BYTES / 4];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_addr[kMaxDevices] = {};  // device address of the block, per device
}  // namespace

cudaError_t wf_launch_attn_tc_noalloc(const WfGeom &g, const WfRoundDev &rd, int layer,
                                      const WfTmaps &maps, void *out, void *status_scratch,
                                      int num_sms, cudaStream_t stream, int *wf_err) {
    *wf_err = WF_OK;
    // bytes of scheduler counters the kernel reads and writes (work, finished CTAs)
    const size_t need = WF_SCRATCH_DONE + sizeof(uint32_t);
    if (need > WF_NOALLOC_SCRATCH_BYTES) {
        *wf_err = WF_ERANGE;
        return cudaSuccess;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) {
        *wf_err = WF_ERANGE;
        return cudaSuccess;
    }
    void *ctl = nullptr;
    {
        // once per device, with that device current: the host-side name of a
        // __device__ array is not a device address, so look the address up.
        // The address is kept for the life of the process; it is no longer
        // valid once the device's context is destroyed (cudaDeviceReset).
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_addr[dev]) {
            void *a = nullptr;
            e = cudaGetSymbolAddress(&a, wf_noalloc_scratch);
            if (e != cudaSuccess) return e;
            g_noalloc_addr[dev] = a;
        }
        ctl = g_noalloc_addr[dev];
    }
    if (rd.n_tasks < 1) return cudaSuccess;
    e = cudaMemsetAsync(ctl, 0, need, stream);
    if (e != cudaSuccess) return e;
    return launch_tc(g, rd, layer, maps, out, static_cast<uint32_t *>(ctl),
                     static_cast<uint32_t *>(status_scratch), num_sms, stream);
}
