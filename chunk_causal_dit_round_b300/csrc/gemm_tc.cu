// Linear layers of the DiT block on the 5th-generation tensor cores.
//
// out = epilogue(A W^T + b) for A [M, K] bf16 (row-major activations) and
// W [N, K] bf16 (a linear layer's weight, output-major): the QKV projection
// whose epilogue applies RoPE and publishes K/V into their page slots
// ("Wave Forcing", Sec. 4.2: K/V are published right after QKV projection and
// RoPE; App. B.2 Eq. 13 fixed-slot placement), and the "remaining block" of
// Sec. 4.1 (output projection and FFN with gated residual adds, GELU), plus
// the patch embedding and the head whose epilogue performs the stage
// transition of Sec. 2 Eq. 1.
//
// Design (one persistent CTA per SM, 320 threads, no scratch memory):
//  * tiles of 128 rows x BN columns, visited output-column-fastest so the
//    CTAs of one wave share a few rows of A and the whole weight matrix stays
//    in L2; CTA c takes tiles c, c + grid, c + 2 grid, ...;
//  * warp 0 (one thread): TMA producer of 64-wide K slices of A and W
//    (128-byte swizzle) into an NST-deep shared-memory ring;
//  * warp 1 (one thread): tcgen05.mma issuer, M = 128, N = BN, fp32
//    accumulators in TMEM, double-buffered (2 x BN columns) so the epilogue
//    of tile i runs under the MMAs of tile i + 1;
//  * warps 2-9: epilogue, two warps per TMEM lane quarter (each takes half of
//    the tile's columns), one accumulator row per thread, tcgen05.ld of 32
//    columns at a time with the next chunk's load in flight while the
//    current one is processed; fused elementwise work (packed f32x2
//    arithmetic), direct global stores -- except the gated residual, whose
//    32 x 32 blocks go through shared memory into a TMA reduce-add on x, so
//    the read-modify-write of the fp32 residual stream happens in L2.
// Every wait is bounded (%globaltimer); on a timeout the kernel records it in
// the plan's status word, drains its own copies and MMAs, frees TMEM and
// returns.

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "wf_internal.h"
#include "wf_ptx.cuh"

using namespace wfptx;

namespace {

constexpr int BM = 128;
constexpr int BK = 64;                       // one 128-byte swizzle atom of bf16
constexpr int NUM_THREADS = 320;           // producer, MMA issuer, 8 epilogue warps
constexpr int EPI_WARPS = 8;
constexpr uint64_t WAIT_NS = 1000000000ull;  // 1 s

template <int BN>
struct Cfg {
    static constexpr int NST = BN >= 256 ? 4 : 6;
    static constexpr uint32_t A_BYTES = BM * BK * 2;
    static constexpr uint32_t B_BYTES = BN * BK * 2;
    static constexpr uint32_t STAGE = A_BYTES + B_BYTES;
    static constexpr uint32_t SM_BAR = NST * STAGE;
    // full[NST], empty[NST], tfull[2], tempty[2], drain
    static constexpr int B_FULL = 0, B_EMPTY = NST, B_TFULL = 2 * NST, B_TEMPTY = 2 * NST + 2,
                         B_DRAIN = 2 * NST + 4, NBARS = 2 * NST + 5;
    static constexpr uint32_t SM_MISC = SM_BAR + ((NBARS * 8 + 63) / 64) * 64;
    // per epilogue warp: a 32 x 32 fp32 staging tile in the TMA's 128-byte
    // swizzled layout (1 KB-aligned), the source of the residual reduce-add
    static constexpr uint32_t SM_STAGE = (SM_MISC + 64 + 1023) / 1024 * 1024;
    static constexpr uint32_t SM_ALLOC = SM_STAGE + 8 * 4096 + 1024;
    static constexpr uint32_t TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;
};

struct Roles {
    uint32_t sbase;
    volatile int *abort;
    uint32_t *status, *where;
    __device__ bool wait(uint32_t bar, uint32_t parity, uint32_t site) const {
        return mbar_wait(bar, parity, abort, status, where, site, WAIT_NS);
    }
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// x[box at (c0, c1)] += the shared-memory box at src (fp32 add in L2)
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap *map, uint32_t src, int c0, int c1) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(c0), "r"(c1), "r"(src)
        : "memory");
}
// global[box at (c0, c1)] = the shared-memory box at src
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the bulk copies of this thread have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// the bulk copies of this thread are complete
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// generic-proxy shared-memory writes become visible to the async (TMA) proxy
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Packed f32x2 arithmetic, IEEE round-to-nearest without flushing.
__device__ __forceinline__ uint64_t p2(float lo, float hi) { return f2_pack(lo, hi); }
__device__ __forceinline__ uint64_t p2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t p2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t p2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// v = acc (x the e4m3 weight scale of the column when HAS_WS) + bias, as 16
// packed pairs; bias may be null.
template <bool HAS_WS>
__device__ __forceinline__ void affine_cols(const uint32_t (&u)[32], const float *ws,
                                            const __nv_bfloat16 *bias, uint64_t (&v)[16]) {
#pragma unroll
    for (int q = 0; q < 16; ++q) v[q] = p2(__uint_as_float(u[2 * q]), __uint_as_float(u[2 * q + 1]));
    if constexpr (HAS_WS) {
        const float4 *w4 = reinterpret_cast<const float4 *>(ws);
        if (bias) {
            const uint4 *b4 = reinterpret_cast<const uint4 *>(bias);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 bb = __ldg(b4 + q);
                const float4 wa = __ldg(w4 + 2 * q), wb = __ldg(w4 + 2 * q + 1);
                const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&bb);
                const float2 b0 = __bfloat1622float2(h2[0]), b1 = __bfloat1622float2(h2[1]);
                const float2 b2 = __bfloat1622float2(h2[2]), b3 = __bfloat1622float2(h2[3]);
                v[4 * q] = p2_fma(v[4 * q], p2(wa.x, wa.y), p2(b0.x, b0.y));
                v[4 * q + 1] = p2_fma(v[4 * q + 1], p2(wa.z, wa.w), p2(b1.x, b1.y));
                v[4 * q + 2] = p2_fma(v[4 * q + 2], p2(wb.x, wb.y), p2(b2.x, b2.y));
                v[4 * q + 3] = p2_fma(v[4 * q + 3], p2(wb.z, wb.w), p2(b3.x, b3.y));
            }
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float4 w = __ldg(w4 + q);
                v[2 * q] = p2_mul(v[2 * q], p2(w.x, w.y));
                v[2 * q + 1] = p2_mul(v[2 * q + 1], p2(w.z, w.w));
            }
        }
    } else if (bias) {
        const uint4 *b4 = reinterpret_cast<const uint4 *>(bias);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 bb = __ldg(b4 + q);
            const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&bb);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(h2[e]);
                v[4 * q + e] = p2_add(v[4 * q + e], p2(f.x, f.y));
            }
        }
    }
}

// GELU, tanh form 0.5 x (1 + tanh u), u = sqrt(2/pi) (x + 0.044715 x^3), on a
// packed pair, evaluated as x / (1 + 2^a) with a = -2 log2(e) u, since
// 0.5 (1 + tanh u) = 1 / (1 + e^(-2u)): accurate in relative terms also where
// GELU(x) is tiny.  a is capped at 126 so that 1 + 2^a stays finite.
__device__ __forceinline__ uint64_t gelu2(uint64_t x) {
    constexpr float G0 = -2.0f * 1.4426950408889634f * 0.7978845608028654f;
    constexpr float G1 = G0 * 0.044715f;
    const uint64_t a2 = p2_mul(x, p2_fma(p2_mul(x, x), p2(G1, G1), p2(G0, G0)));
    float a0, a1;
    f2_unpack(a2, a0, a1);
    const uint64_t d = p2_add(p2(1.f, 1.f), p2(ex2(fminf(a0, 126.f)), ex2(fminf(a1, 126.f))));
    float d0, d1;
    f2_unpack(d, d0, d1);
    return p2_mul(x, p2(rcp_approx(d0), rcp_approx(d1)));
}

// ---- epilogues -----------------------------------------------------------------
// Each receives one thread's 32 consecutive accumulator columns of one row.

template <int EPI>
struct Epi;

// out (bf16 or f32) = acc + bias;  GELU variant.
template <>
struct Epi<WF_EPI_BF16> {
    __device__ static void apply(const GemmParams &p, int row, int col, float (&v)[32]) {
        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(p.out) + (size_t)row * p.ldo + col;
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            d4[q] = make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                               pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
    }
};
template <>
struct Epi<WF_EPI_GELU_BF16> {
    __device__ static void apply2(const GemmParams &p, int row, int col, uint64_t (&v2)[16]) {
        float v[32];
#pragma unroll
        for (int q = 0; q < 16; ++q) f2_unpack(gelu2(v2[q]), v[2 * q], v[2 * q + 1]);
        Epi<WF_EPI_BF16>::apply(p, row, col, v);
    }
};
// GELU for an e4m3 output on a packed pair: 0.5 x (1 + tanh u) with the
// hardware tanh approximation (relative error about 2^-11, far below the
// e4m3 step 2^-4 and at most ~1e-3 absolute where the result is tiny).
__device__ __forceinline__ uint64_t gelu2_fast(uint64_t x) {
    constexpr float C0 = 0.7978845608028654f;
    constexpr float C1 = C0 * 0.044715f;
    const uint64_t u2 = p2_mul(x, p2_fma(p2_mul(x, x), p2(C1, C1), p2(C0, C0)));
    float u0, u1, t0, t1;
    f2_unpack(u2, u0, u1);
    asm("tanh.approx.f32 %0, %1;" : "=f"(t0) : "f"(u0));
    asm("tanh.approx.f32 %0, %1;" : "=f"(t1) : "f"(u1));
    const uint64_t hx = p2_mul(x, p2(0.5f, 0.5f));
    return p2_fma(hx, p2(t0, t1), hx);
}
__device__ __forceinline__ uint32_t e4m3x2_of(uint64_t v) {
    float a, b;
    f2_unpack(v, a, b);
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// FFN hidden layer for an e4m3 FFN2: GELU, then e4m3 bytes (unit scale)
template <>
struct Epi<WF_EPI_GELU_E4M3> {
    __device__ static void apply2(const GemmParams &p, int row, int col, uint64_t (&v2)[16]) {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            w[i] = e4m3x2_of(gelu2_fast(v2[2 * i])) | (e4m3x2_of(gelu2_fast(v2[2 * i + 1])) << 16);
        uint4 *d4 = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(p.out) + (size_t)row * p.ldo + col);
        d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
};
template <>
struct Epi<WF_EPI_F32> {
    __device__ static void apply(const GemmParams &p, int row, int col, float (&v)[32]) {
        float4 *d4 = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + (size_t)row * p.ldo + col);
#pragma unroll
        for (int q = 0; q < 8; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
};
// The gated residual add x += gate[group(row)][col] * (acc + bias) of the
// attention and FFN halves of a block is in the kernel body: it stages each
// 32 x 32 block for a TMA reduce-add.

// QKV projection epilogue: columns [0, dim) are Q, [dim, 2 dim) K, [2 dim,
// 3 dim) V, head h at columns h*D .. h*D + D - 1 of each part.  RoPE on Q and
// K at the token's absolute (t, h, w); Q -> qbuf[slot][h][n][:], K/V ->
// pool[dest page][layer][K|V][h][n][:]; the store of the anchor also keeps
// its unrotated key on the raw-anchor page (App. B.3).  WF_FP8 plans store
// e4m3 (Q and K times qk_scale, V times v_scale) instead of bf16.  With
// qk_raw set, Q and K go out unrotated in bf16 for the q/k RMSNorm kernel
// (which needs whole rows) and only V is published here.
template <>
struct Epi<WF_EPI_QKV_PUBLISH> {
    __device__ static void store32(__nv_bfloat16 *dst, const float (&v)[32]) {
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            d4[q] = make_uint4(pack_bf16(v[8 * q], v[8 * q + 1]), pack_bf16(v[8 * q + 2], v[8 * q + 3]),
                               pack_bf16(v[8 * q + 4], v[8 * q + 5]), pack_bf16(v[8 * q + 6], v[8 * q + 7]));
    }
    // e4m3 pages (WF_FP8 plans): 32 values times scale, rounded, 32 bytes
    __device__ static void store32_e4m3(uint8_t *dst, const float (&v)[32], float scale) {
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i] * scale, v[4 * i + 1] * scale),
                                                         __NV_SATFINITE, __NV_E4M3);
            const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i + 2] * scale, v[4 * i + 3] * scale),
                                                         __NV_SATFINITE, __NV_E4M3);
            w[i] = lo | (hi << 16);
        }
        uint4 *d4 = reinterpret_cast<uint4 *>(dst);
        d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
    }
    // one row of one head's 32 channels into a page plane or the query workspace
    __device__ static void put(const GemmParams &p, size_t off, const float (&v)[32], float scale) {
        if (p.g.dtype == WF_FP8)
            store32_e4m3(reinterpret_cast<uint8_t *>(p.pool) + off, v, scale);
        else
            store32(p.pool + off, v);
    }
    __device__ static void putq(const GemmParams &p, size_t off, const float (&v)[32], float scale) {
        if (p.g.dtype == WF_FP8)
            store32_e4m3(reinterpret_cast<uint8_t *>(p.qbuf) + off, v, scale);
        else
            store32(p.qbuf + off, v);
    }
    // What a row needs, computed once per tile: its slot, token, task, and
    // the offsets (in float2 units, to be added to the pair index m) of its
    // rotary rows in the t / h / w tables.
    struct Row {
        int slot, n, ti;
        int t_off, h_off, w_off;
    };
    __device__ static Row row_info(const GemmParams &p, int row) {
        const WfGeom &g = p.g;
        Row r{};
        r.slot = row / g.NC;
        r.n = row - r.slot * g.NC;
        r.ti = p.rd.task_of_slot[r.slot];
        if (r.ti < 0) return r;                     // a slot without a task: skipped
        const int hw = g.gh * g.gw;
        const int f = r.n / hw, hh = (r.n / g.gw) % g.gh, ww = r.n - (r.n / g.gw) * g.gw;
        const int t = g.gt * p.rd.chunk[r.ti] + f;
        r.t_off = g.rope_t_off + t * g.dt2;
        r.h_off = g.rope_h_off + hh * g.dh2 - g.dt2;
        r.w_off = g.rope_w_off + ww * g.dw2 - g.dt2 - g.dh2;
        return r;
    }
    __device__ static void apply(const GemmParams &p, const Row &ri, int col, float (&v)[32]) {
        const WfGeom &g = p.g;
        const int dim = g.H * g.D;
        const int part = col / dim;                 // 0 Q, 1 K, 2 V
        const int cc = col - part * dim;
        const int h = cc / g.D;
        const int d0 = cc - h * g.D;                // 32 consecutive channels d0 .. d0 + 31
        const int slot = ri.slot, n = ri.n, ti = ri.ti;
        const size_t plane = (size_t)g.NC * g.D;
        if (ti < 0) return;
        if (part < 2 && p.qk_raw) {
            // the block normalises q and k over the full width: leave the
            // unrotated row for the q/k RMSNorm kernel
            store32(p.qk_raw + ((size_t)slot * g.NC + n) * (2 * dim) + col, v);
            return;
        }
        if (part == 2) {
            size_t kvp = (((size_t)p.rd.dest[ti] * g.L + p.layer) * 2 + 1) * g.H + h;
            put(p, kvp * plane + (size_t)n * g.D + d0, v, g.v_scale);
            return;
        }
        if (part == 1 && p.rd.raw_page[ti] >= 0) {
            size_t rawp = (((size_t)p.rd.raw_page[ti] * g.L + p.layer) * 2) * g.H + h;
            put(p, rawp * plane + (size_t)n * g.D + d0, v, g.qk_scale);
        }
        const float2 *tab = p.rope;
        float2 cs[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int m = d0 / 2 + i;
            const int off = m < g.dt2 ? ri.t_off : (m < g.dt2 + g.dh2 ? ri.h_off : ri.w_off);
            cs[i] = __ldg(tab + off + m);
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float a = v[2 * i], b = v[2 * i + 1];
            v[2 * i] = a * cs[i].x - b * cs[i].y;
            v[2 * i + 1] = a * cs[i].y + b * cs[i].x;
        }
        if (part == 0) {
            putq(p, ((size_t)slot * g.H + h) * plane + (size_t)n * g.D + d0, v, g.qk_scale);
        } else {
            size_t kp = (((size_t)p.rd.dest[ti] * g.L + p.layer) * 2) * g.H + h;
            put(p, kp * plane + (size_t)n * g.D + d0, v, g.qk_scale);
        }
    }
};

// Head epilogue: the 4C outputs of a token are ordered (row offset, column
// offset, channel) of its 2 x 2 latent patch.  x0 = prediction; for a
// denoising slot s the next stage's input is Psi(x0, eps) = (1 - sigma') x0 +
// sigma' eps (Sec. 2 Eq. 1; sigma' = 0 gives x0 itself for the last stage);
// the store slot's prediction is discarded.
template <>
struct Epi<WF_EPI_HEAD> {
    __device__ static void apply(const GemmParams &p, int row, int col, float (&v)[32]) {
        const WfGeom &g = p.g;
        const int gslot = row / g.NC;               // request m, stage slot `slot`
        if (p.rd.task_of_slot[gslot] < 0) return;   // no task in this slot this round
        const int m = gslot / (g.S + 1);
        const int slot = gslot - m * (g.S + 1);
        const int n = row - gslot * g.NC;
        const int hw = g.gh * g.gw;
        const int f = n / hw, hh = (n / g.gw) % g.gh, ww = n - (n / g.gw) * g.gw;
        const int C = p.channels;
        const int Hl = 2 * g.gh, Wl = 2 * g.gw;
        const size_t cstride = (size_t)g.gt * Hl * Wl;
        const size_t lat = (size_t)C * cstride;
        const float sg = p.sigma_next[slot];
        float *x0 = p.x0_out ? p.x0_out + (size_t)gslot * lat : nullptr;
        float *zn = slot < g.S ? p.z_next[m] + (size_t)(slot + 1) * lat : nullptr;
        const float *eps = (slot < g.S && sg != 0.f) ? p.eps + ((size_t)m * g.S + slot) * lat : nullptr;
        float *emit = (slot == g.S - 1 && p.chunk_out) ? p.chunk_out + (size_t)m * lat : nullptr;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int j = col + i;              // feature index (q, r, c)
            const int qr = j / C, c = j - qr * C;
            const int q = qr >> 1, r = qr & 1;
            const size_t at = (size_t)c * cstride + ((size_t)f * Hl + 2 * hh + q) * Wl + 2 * ww + r;
            const float x = v[i];
            if (x0) x0[at] = x;
            if (zn) {
                const float z = eps ? fmaf(sg, eps[at], (1.f - sg) * x) : x;
                zn[at] = z;
                if (emit) emit[at] = z;
            }
        }
    }
};

// per-row state kept across a tile's column chunks (only the QKV epilogue has any)
struct NoRow {};
template <int EPI>
struct QkvRowT {
    using type = NoRow;
};
template <>
struct QkvRowT<WF_EPI_QKV_PUBLISH> {
    using type = Epi<WF_EPI_QKV_PUBLISH>::Row;
};

// ---- kernel -----------------------------------------------------------------------

template <int BN, int EPI, bool F8>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb,
                   const __grid_constant__ CUtensorMap tc, const __grid_constant__ CUtensorMap td,
                   const GemmParams p) {
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = smem_u32(smem_raw);
    const uint32_t pad = (1024u - (raw_u32 & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    Roles r;
    r.sbase = raw_u32 + pad;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::SM_MISC);
    r.abort = reinterpret_cast<volatile int *>(smem + C::SM_MISC + 16);
    r.status = p.status;
    r.where = p.status ? p.status + WF_SCRATCH_WHERE / 4 : nullptr;
    auto bar = [&](int i) { return r.sbase + C::SM_BAR + 8u * i; };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NST; ++i) {
            mbar_init(bar(C::B_FULL + i), 1);
            mbar_init(bar(C::B_EMPTY + i), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(C::B_TFULL + b), 1);
            mbar_init(bar(C::B_TEMPTY + b), EPI_WARPS);  // one arrival per epilogue warp
        }
        mbar_init(bar(C::B_DRAIN), 1);
        mbar_fence_init();
        *r.abort = 0;
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&ta);
        tma_prefetch_desc(&tb);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int n_tiles = p.tiles_m * p.tiles_n;
    // K elements per 128-byte stage row: 64 bf16 or 128 e4m3
    constexpr int KE = F8 ? 2 * BK : BK;
    const int kb_n = p.K / KE;
    uint32_t issued = 0;

    if (warp == 0 && lane == 0) {
        // ---- producer ----
        uint32_t it = 0;
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
            const int m0 = p.row_begin + (tile / p.tiles_n) * BM;
            const int n0 = (tile % p.tiles_n) * BN;
            for (int kb = 0; kb < kb_n; ++kb, ++it) {
                const int st = it % C::NST;
                if (!r.wait(bar(C::B_EMPTY + st), ((it / C::NST) & 1) ^ 1, 1)) goto done;
                const uint32_t sa = r.sbase + st * C::STAGE;
                mbar_arrive_expect_tx(bar(C::B_FULL + st), C::STAGE);
                tma_load_2d(sa, &ta, bar(C::B_FULL + st), kb * KE, m0);
                tma_load_2d(sa + C::A_BYTES, &tb, bar(C::B_FULL + st), kb * KE, n0);
                issued = it + 1;
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer ----
        constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(BM, BN, false) : idesc_bf16_f32(BM, BN, false);
        uint32_t it = 0, tl = 0;
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++tl) {
            const int buf = tl & 1;
            if (!r.wait(bar(C::B_TEMPTY + buf), ((tl >> 1) & 1) ^ 1, 2)) goto done;
            tc_fence_after();
            const uint32_t d = tmem + buf * BN;
            for (int kb = 0; kb < kb_n; ++kb, ++it) {
                const int st = it % C::NST;
                if (!r.wait(bar(C::B_FULL + st), (it / C::NST) & 1, 3)) goto done;
                tc_fence_after();
                const uint32_t sa = r.sbase + st * C::STAGE;
                const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk)
                    if constexpr (F8)
                        mma_ss_f8(d, sdesc_sw128(sa + kk * 32, 16, 1024), sdesc_sw128(sb + kk * 32, 16, 1024),
                                  idesc, (kb | kk) != 0 ? 1u : 0u);
                    else
                        mma_ss(d, sdesc_sw128(sa + kk * 32, 16, 1024), sdesc_sw128(sb + kk * 32, 16, 1024),
                               idesc, (kb | kk) != 0 ? 1u : 0u);
                mma_commit(bar(C::B_EMPTY + st));
            }
            mma_commit(bar(C::B_TFULL + buf));
        }
    } else if (warp >= 2) {
        // ---- epilogue ----
        constexpr int NPW = BN / 64;                // 32-column chunks per warp
        const int quarter = warp & 3;               // TMEM lanes 32*quarter .. +31
        const int half = (warp - 2) >> 2;           // which half of the columns
        uint32_t tl = 0;
        for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++tl) {
            const int buf = tl & 1;
            bool ok = r.wait(bar(C::B_TFULL + buf), (tl >> 1) & 1, 4);
            if (!__all_sync(0xffffffffu, ok)) goto done;
            tc_fence_after();
            const int rel_row0 = (tile / p.tiles_n) * BM + quarter * 32;   // warp's first row - row_begin
            const int row = p.row_begin + rel_row0 + lane;
            const int n0 = (tile % p.tiles_n) * BN + half * (BN / 2);
            const bool live = row < p.row_end;
            int grp = 0;
            if constexpr (EPI == WF_EPI_GATED_RESIDUAL) grp = live ? row / p.rows_per_group : 0;
            typename QkvRowT<EPI>::type qrow{};
            if constexpr (EPI == WF_EPI_QKV_PUBLISH)
                if (live) qrow = Epi<WF_EPI_QKV_PUBLISH>::row_info(p, row);
            const uint32_t taddr =
                tmem + ((uint32_t)(quarter * 32) << 16) + buf * BN + half * (BN / 2);
            uint32_t u[2][32];
            tmem_ld32(taddr, u[0]);
            tmem_wait_ld(u[0]);
#pragma unroll
            for (int c = 0; c < NPW; ++c) {
                if (c + 1 < NPW) {
                    tmem_ld32(taddr + (c + 1) * 32, u[(c + 1) & 1]);
                } else {
                    // the accumulator buffer is fully in registers: hand it
                    // back to the MMA issuer before the last stores
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(C::B_TEMPTY + buf));
                }
                const int col = n0 + c * 32;
                // Row-major outputs (bf16, GELU bf16 / e4m3, the QKV
                // projection's unrotated q | k rows) leave through shared
                // memory: a warp's 32 rows x 128 bytes (64 bf16 or 128 e4m3
                // columns, several 32-column chunks) are staged in the TMA's
                // 128-byte swizzled layout and written by one TMA store, so
                // the global writes are whole lines instead of one row per
                // thread; rows past row_end and columns past the output's
                // width are clipped by the map.
                constexpr bool STAGEABLE = EPI == WF_EPI_BF16 || EPI == WF_EPI_GELU_BF16 ||
                                           EPI == WF_EPI_GELU_E4M3 || EPI == WF_EPI_QKV_PUBLISH;
                constexpr int CPB = EPI == WF_EPI_GELU_E4M3 ? 4 : 2;   // chunks per staged block
                bool staged = false;
                if constexpr (STAGEABLE)
                    staged = p.staged && (EPI != WF_EPI_QKV_PUBLISH || col < 2 * p.g.H * p.g.D);
                // V of the QKV projection: a warp's 32 rows of one head's 32
                // channels go to their page plane by one TMA store when the
                // rows lie in one slot with a task (all but the block that
                // straddles two chunks); otherwise per-thread stores below
                bool vstaged = false;
                int vslot = 0, vn0 = 0;
                if constexpr (EPI == WF_EPI_QKV_PUBLISH) {
                    if (p.staged_v && col >= 2 * p.g.H * p.g.D && col < p.N) {
                        const int r0abs = p.row_begin + rel_row0;
                        vslot = r0abs / p.g.NC;
                        vn0 = r0abs - vslot * p.g.NC;
                        vstaged = vn0 + 31 < p.g.NC && r0abs + 31 < p.row_end && p.rd.task_of_slot[vslot] >= 0;
                    }
                }
                if (vstaged) {
                    uint8_t *stg = smem + C::SM_STAGE + (warp - 2) * 4096;
                    if (lane == 0) bulk_wait_read();          // the previous block has left stg
                    __syncwarp();
                    uint64_t v2[16];
                    affine_cols<F8>(u[c & 1], F8 ? p.wscale + col : nullptr, p.bias ? p.bias + col : nullptr, v2);
                    if (p.g.dtype == WF_FP8) {
                        const float sc = p.g.v_scale;
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            float a0, a1, a2, a3;
                            f2_unpack(v2[2 * i], a0, a1);
                            f2_unpack(v2[2 * i + 1], a2, a3);
                            w[i] = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a0 * sc, a1 * sc), __NV_SATFINITE, __NV_E4M3) |
                                   ((uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a2 * sc, a3 * sc), __NV_SATFINITE,
                                                                       __NV_E4M3) << 16);
                        }
                        uint4 *srow = reinterpret_cast<uint4 *>(stg + lane * 32);
                        srow[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        srow[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    } else {
                        uint4 *srow = reinterpret_cast<uint4 *>(stg + lane * 64);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            uint32_t w[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                float a, b;
                                f2_unpack(v2[4 * q + i], a, b);
                                w[i] = pack_bf16(a, b);
                            }
                            srow[q] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int ti = p.rd.task_of_slot[vslot];
                        const int cc = col - 2 * p.g.H * p.g.D;
                        const int h = cc / p.g.D;
                        const int plane = ((p.rd.dest[ti] * p.g.L + p.layer) * 2 + 1) * p.g.H + h;
                        tma_store_3d(&td, smem_u32(stg), cc - h * p.g.D, vn0, plane);
                        bulk_commit();
                    }
                } else if (staged) {
                    const int cb = c % CPB;
                    const int col0 = col - cb * 32;           // first column of the block
                    uint8_t *stg = smem + C::SM_STAGE + (warp - 2) * 4096;
                    if (cb == 0) {
                        if (lane == 0) bulk_wait_read();      // the previous block has left stg
                        __syncwarp();
                    }
                    if (col < p.N) {
                        uint64_t v2[16];
                        affine_cols<F8>(u[c & 1], F8 ? p.wscale + col : nullptr, p.bias ? p.bias + col : nullptr, v2);
                        uint4 *srow = reinterpret_cast<uint4 *>(stg + lane * 128);
                        if constexpr (EPI == WF_EPI_GELU_E4M3) {
                            uint32_t w[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                w[i] = e4m3x2_of(gelu2_fast(v2[2 * i])) | (e4m3x2_of(gelu2_fast(v2[2 * i + 1])) << 16);
                            srow[(2 * cb) ^ (lane & 7)] = make_uint4(w[0], w[1], w[2], w[3]);
                            srow[(2 * cb + 1) ^ (lane & 7)] = make_uint4(w[4], w[5], w[6], w[7]);
                        } else {
                            if constexpr (EPI == WF_EPI_GELU_BF16) {
#pragma unroll
                                for (int q = 0; q < 16; ++q) v2[q] = gelu2(v2[q]);
                            }
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                uint32_t w[4];
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    float a, b;
                                    f2_unpack(v2[4 * q + i], a, b);
                                    w[i] = pack_bf16(a, b);
                                }
                                srow[(4 * cb + q) ^ (lane & 7)] = make_uint4(w[0], w[1], w[2], w[3]);
                            }
                        }
                    }
                    if (cb == CPB - 1 || c == NPW - 1) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0 && col0 < p.N) {
                            tma_store_2d(&tc, smem_u32(stg), col0, rel_row0);
                            bulk_commit();
                        }
                    }
                } else if constexpr (EPI == WF_EPI_GATED_RESIDUAL) {
                    // y = gate[group(row)] * (acc + b) staged as a 32 x 32
                    // block (row = lane, 16-byte units swizzled by row & 7, the
                    // TMA's 128-byte pattern), then x[block] += y by a TMA
                    // reduce-add; rows past row_end are clipped by the map.
                    if (col < p.N) {
                        uint64_t v2[16];
                        affine_cols<F8>(u[c & 1], F8 ? p.wscale + col : nullptr, p.bias ? p.bias + col : nullptr, v2);
                        if (live) {
                            const float4 *g4 = reinterpret_cast<const float4 *>(
                                p.gate + (size_t)grp * p.gate_ld + col);
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float4 gv = __ldg(g4 + q);
                                v2[2 * q] = p2_mul(v2[2 * q], p2(gv.x, gv.y));
                                v2[2 * q + 1] = p2_mul(v2[2 * q + 1], p2(gv.z, gv.w));
                            }
                        }
                        float *stg = reinterpret_cast<float *>(smem + C::SM_STAGE) + (warp - 2) * 1024;
                        if (lane == 0) bulk_wait_read();      // the previous block has left stg
                        __syncwarp();
                        float4 *srow = reinterpret_cast<float4 *>(stg + lane * 32);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            float a0, a1, a2, a3;
                            f2_unpack(v2[2 * q], a0, a1);
                            f2_unpack(v2[2 * q + 1], a2, a3);
                            srow[q ^ (lane & 7)] = make_float4(a0, a1, a2, a3);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_reduce_add_2d(&tc, smem_u32(stg), col, rel_row0);
                            bulk_commit();
                        }
                    }
                } else if (live && col < p.N) {
                    uint64_t v2[16];
                    affine_cols<F8>(u[c & 1], F8 ? p.wscale + col : nullptr, p.bias ? p.bias + col : nullptr, v2);
                    if constexpr (EPI == WF_EPI_GELU_BF16 || EPI == WF_EPI_GELU_E4M3) {
                        Epi<EPI>::apply2(p, row, col, v2);
                    } else {
                        float v[32];
#pragma unroll
                        for (int q = 0; q < 16; ++q) f2_unpack(v2[q], v[2 * q], v[2 * q + 1]);
                        if constexpr (EPI == WF_EPI_QKV_PUBLISH)
                            Epi<EPI>::apply(p, qrow, col, v);
                        else
                            Epi<EPI>::apply(p, row, col, v);
                    }
                }
                if (c + 1 < NPW) tmem_wait_ld(u[(c + 1) & 1]);
            }
        }
    }
done:
    if constexpr (EPI == WF_EPI_GATED_RESIDUAL || EPI == WF_EPI_BF16 || EPI == WF_EPI_GELU_BF16 ||
                  EPI == WF_EPI_GELU_E4M3 || EPI == WF_EPI_QKV_PUBLISH) {
        // the reduce-adds / stores this warp issued have completed (shared
        // memory is released when the CTA exits)
        if (warp >= 2 && lane == 0) bulk_wait_all();
    }
    if (*r.abort) {
        if (warp == 0 && lane == 0) {
            uint32_t first = issued > (uint32_t)C::NST ? issued - C::NST : 0;
            for (uint32_t s = first; s < issued; ++s)
                mbar_wait(bar(C::B_FULL + s % C::NST), (s / C::NST) & 1, nullptr, nullptr, nullptr, 0,
                          WAIT_NS);
        }
        if (warp == 1 && lane == 0) {
            mma_commit(bar(C::B_DRAIN));
            mbar_wait(bar(C::B_DRAIN), 0, nullptr, nullptr, nullptr, 0, WAIT_NS);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int BN, int EPI, bool F8>
cudaError_t launch(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tc,
                   const CUtensorMap &td, const GemmParams &p, int num_sms, cudaStream_t stream) {
    using C = Cfg<BN>;
    static std::atomic<unsigned long long> attr_set{0};
    cudaError_t e = wf_once_per_device(attr_set, [] {
        return cudaFuncSetAttribute(gemm_tc_kernel<BN, EPI, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    C::SM_ALLOC);
    });
    if (e != cudaSuccess) return e;
    const int n_tiles = p.tiles_m * p.tiles_n;
    const int grid = n_tiles < num_sms ? n_tiles : num_sms;
    gemm_tc_kernel<BN, EPI, F8><<<grid, NUM_THREADS, C::SM_ALLOC, stream>>>(ta, tb, tc, td, p);
    return cudaGetLastError();
}

typedef CUresult (*EncodeFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                             const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                             const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                             CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once (thread-safe static
// initialisation); the entry point is the same for every device.
EncodeFn encoder() {
    static const EncodeFn fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<EncodeFn>(f);
    }();
    return fn;
}

// 2D bf16 map over a row-major [rows, cols] matrix with row pitch ld
// elements, box (64 columns, box_rows rows), 128-byte swizzle.
bool encode_2d(CUtensorMap *m, const void *base, long long rows, long long cols, long long ld,
               int box_rows, bool f8) {
    EncodeFn enc = encoder();
    if (!enc) return false;
    const int es = f8 ? 1 : 2;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * es};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / es), (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
               const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int wf_gemm_bn_for(int epi) { return epi == WF_EPI_HEAD ? 64 : 256; }

cudaError_t wf_launch_gemm(int epi, const void *a, long long a_rows, int lda, const void *w,
                           GemmParams p, int num_sms, cudaStream_t stream, bool f8) {
    const int bn = wf_gemm_bn_for(epi);
    const int ke = f8 ? 2 * BK : BK;
    if (p.K % ke || p.N % 32 || lda % (f8 ? 16 : 8) || p.row_end <= p.row_begin)
        return cudaErrorInvalidValue;
    if (f8 && !p.wscale) return cudaErrorInvalidValue;
    CUtensorMap ta, tb, tc;
    if (!encode_2d(&ta, a, a_rows, p.K, lda, BM, f8)) return cudaErrorInvalidValue;
    if (!encode_2d(&tb, w, p.N, p.K, p.K, bn, f8)) return cudaErrorInvalidValue;
    tc = ta;   // unused unless the epilogue reduces into x or stores through TMA
    p.staged = 0;
    const bool qk_rows = epi == WF_EPI_QKV_PUBLISH && p.qk_raw && (p.g.H * p.g.D) % 64 == 0;
    if (epi == WF_EPI_BF16 || epi == WF_EPI_GELU_BF16 || epi == WF_EPI_GELU_E4M3 || qk_rows) {
        // row-major output rows [row_begin, row_end), boxes of 32 rows x 128
        // bytes, 128-byte swizzle; outputs a map cannot describe keep the
        // per-thread stores
        const bool e8 = epi == WF_EPI_GELU_E4M3;
        const long long ncols = qk_rows ? 2LL * p.g.H * p.g.D : p.N;
        const long long pitch = qk_rows ? ncols : p.ldo;
        const char *base = qk_rows ? reinterpret_cast<const char *>(p.qk_raw + (size_t)p.row_begin * pitch)
                                   : static_cast<const char *>(p.out) + (size_t)p.row_begin * pitch * (e8 ? 1 : 2);
        EncodeFn enc = encoder();
        if (enc && (reinterpret_cast<uintptr_t>(base) & 15) == 0 && (pitch * (e8 ? 1 : 2)) % 16 == 0 &&
            pitch >= ncols) {
            const cuuint64_t dims[2] = {(cuuint64_t)ncols, (cuuint64_t)(p.row_end - p.row_begin)};
            const cuuint64_t strides[1] = {(cuuint64_t)pitch * (e8 ? 1 : 2)};
            const cuuint32_t box[2] = {e8 ? 128u : 64u, 32};
            const cuuint32_t estr[2] = {1, 1};
            if (enc(&tc, e8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<char *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
                p.staged = 1;
        }
    }
    CUtensorMap td = ta;   // unused unless V is stored through TMA
    p.staged_v = 0;
    if (epi == WF_EPI_QKV_PUBLISH && p.pool && p.rd.n_tasks > 0 && p.g.D % 32 == 0) {
        // the page pool as [plane][N_C][D] (plane = (page, layer, K/V, head)),
        // over the pages this round writes; boxes of 32 tokens x 32 channels
        int pages = 0;
        for (int i = 0; i < p.rd.n_tasks; ++i) pages = p.rd.dest[i] + 1 > pages ? p.rd.dest[i] + 1 : pages;
        const bool e8 = p.g.dtype == WF_FP8;
        const int es = e8 ? 1 : 2;
        EncodeFn enc = encoder();
        const cuuint64_t dims[3] = {(cuuint64_t)p.g.D, (cuuint64_t)p.g.NC,
                                    (cuuint64_t)pages * p.g.L * 2 * p.g.H};
        const cuuint64_t strides[2] = {(cuuint64_t)p.g.D * es, (cuuint64_t)p.g.NC * p.g.D * es};
        const cuuint32_t box[3] = {32, 32, 1};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (enc && (reinterpret_cast<uintptr_t>(p.pool) & 15) == 0 &&
            enc(&td, e8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.pool, dims,
                strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
            p.staged_v = 1;
    }
    if (epi == WF_EPI_GATED_RESIDUAL) {
        // fp32 x rows [row_begin, row_end), 32 x 32 boxes, 128-byte swizzle
        float *x0 = static_cast<float *>(p.out) + (size_t)p.row_begin * p.ldo;
        if (p.ldo % 4 || reinterpret_cast<uintptr_t>(x0) % 16) return cudaErrorInvalidValue;
        EncodeFn enc = encoder();
        if (!enc) return cudaErrorInvalidValue;
        const cuuint64_t dims[2] = {(cuuint64_t)p.N, (cuuint64_t)(p.row_end - p.row_begin)};
        const cuuint64_t strides[1] = {(cuuint64_t)p.ldo * 4};
        const cuuint32_t box[2] = {32, 32};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&tc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, x0, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    p.tiles_m = (p.row_end - p.row_begin + BM - 1) / BM;
    p.tiles_n = (p.N + bn - 1) / bn;
    if (f8) {
        switch (epi) {
            case WF_EPI_BF16: return launch<256, WF_EPI_BF16, true>(ta, tb, tc, td, p, num_sms, stream);
            case WF_EPI_F32: return launch<256, WF_EPI_F32, true>(ta, tb, tc, td, p, num_sms, stream);
            case WF_EPI_GELU_BF16: return launch<256, WF_EPI_GELU_BF16, true>(ta, tb, tc, td, p, num_sms, stream);
            case WF_EPI_GELU_E4M3: return launch<256, WF_EPI_GELU_E4M3, true>(ta, tb, tc, td, p, num_sms, stream);
            case WF_EPI_GATED_RESIDUAL:
                return launch<256, WF_EPI_GATED_RESIDUAL, true>(ta, tb, tc, td, p, num_sms, stream);
            case WF_EPI_QKV_PUBLISH: return launch<256, WF_EPI_QKV_PUBLISH, true>(ta, tb, tc, td, p, num_sms, stream);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (epi) {
        case WF_EPI_BF16: return launch<256, WF_EPI_BF16, false>(ta, tb, tc, td, p, num_sms, stream);
        case WF_EPI_F32: return launch<256, WF_EPI_F32, false>(ta, tb, tc, td, p, num_sms, stream);
        case WF_EPI_GELU_BF16: return launch<256, WF_EPI_GELU_BF16, false>(ta, tb, tc, td, p, num_sms, stream);
        case WF_EPI_GATED_RESIDUAL: return launch<256, WF_EPI_GATED_RESIDUAL, false>(ta, tb, tc, td, p, num_sms, stream);
        case WF_EPI_QKV_PUBLISH: return launch<256, WF_EPI_QKV_PUBLISH, false>(ta, tb, tc, td, p, num_sms, stream);
        case WF_EPI_HEAD: return launch<64, WF_EPI_HEAD, false>(ta, tb, tc, td, p, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

// ---- weight quantisation: one warp per output row ------------------------------------
namespace {
__global__ void __launch_bounds__(256) quant_rows_kernel(const __nv_bfloat16 *__restrict__ w, int N,
                                                         int K, uint8_t *__restrict__ w8,
                                                         float *__restrict__ scale) {
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= N) return;
    const __nv_bfloat16 *wr = w + (size_t)row * K;
    float amax = 0.f;
    for (int k = lane; k < K; k += 32) amax = fmaxf(amax, fabsf(__bfloat162float(wr[k])));
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    if (lane == 0) scale[row] = sc;
    uint8_t *dst = w8 + (size_t)row * K;
    for (int k = 2 * lane; k < K; k += 64) {
        const float a = __fdiv_rn(__bfloat162float(wr[k]), sc);
        const float b = __fdiv_rn(__bfloat162float(wr[k + 1]), sc);
        *reinterpret_cast<uint16_t *>(dst + k) =
            (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    }
}
}  // namespace

cudaError_t wf_launch_quant_rows(const void *w, int N, int K, void *w8, float *scale,
                                 cudaStream_t stream) {
    if (K % 2) return cudaErrorInvalidValue;
    quant_rows_kernel<<<(N * 32 + 255) / 256, 256, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(w), N, K, static_cast<uint8_t *>(w8), scale);
    return cudaGetLastError();
}
