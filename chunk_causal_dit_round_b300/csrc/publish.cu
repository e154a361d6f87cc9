// QKV publication: 3D RoPE on Q and K, then Q into the query workspace and
// K/V straight into their fixed page slots ("Wave Forcing", Sec. 4.2: K/V are
// published right after QKV projection and RoPE; App. B.2 Eq. 13: paged
// placement into final attention slots, no concatenation).  The same launch
// keeps the anchor's unrotated key when chunk 0 is stored, and re-rotates
// the anchor key from that copy when the bounded window has shifted
// (App. B.3).
//
// HBM-bound: every element is read once and written once (twice for the
// anchor copy).  One thread moves 16 bytes of each of Q, K and V for one
// (token, head); consecutive threads walk the head dimension, so loads from
// the token-major input and stores into the head-major pages are both
// contiguous 16-byte vectors.

#include <atomic>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "wf_internal.h"

namespace {

template <typename T>
struct Vec;  // 16 bytes of T
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
};
template <>
struct Vec<float> {
    static constexpr int N = 4;
};

__device__ __forceinline__ void unpack(const uint4 &u, float *f, __nv_bfloat16 *) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 x = __bfloat1622float2(h[i]);
        f[2 * i] = x.x;
        f[2 * i + 1] = x.y;
    }
}
__device__ __forceinline__ void unpack(const uint4 &u, float *f, float *) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
}
__device__ __forceinline__ uint4 pack(const float *f, __nv_bfloat16 *) {
    uint4 u;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return u;
}
__device__ __forceinline__ uint4 pack(const float *f, float *) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
}

// Rotate the interleaved pairs of one 16-byte vector starting at channel d0
// of a token at (t, h, w).
template <typename T>
__device__ __forceinline__ uint4 rope_vec(const uint4 &in, int d0, int t, int hh, int ww,
                                          const WfGeom &g, const float2 *tab) {
    constexpr int N = Vec<T>::N;
    float x[N];
    unpack(in, x, (T *)nullptr);
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        int m = d0 / 2 + i;
        float2 cs;
        if (m < g.dt2)
            cs = tab[g.rope_t_off + t * g.dt2 + m];
        else if (m < g.dt2 + g.dh2)
            cs = tab[g.rope_h_off + hh * g.dh2 + (m - g.dt2)];
        else
            cs = tab[g.rope_w_off + ww * g.dw2 + (m - g.dt2 - g.dh2)];
        float a = x[2 * i], b = x[2 * i + 1];
        x[2 * i] = a * cs.x - b * cs.y;
        x[2 * i + 1] = a * cs.y + b * cs.x;
    }
    return pack(x, (T *)nullptr);
}

template <typename T>
__global__ void __launch_bounds__(256) publish_kernel(const WfGeom g, const WfRoundDev rd,
                                                      int layer, const T *__restrict__ qkv,
                                                      T *__restrict__ qbuf, T *__restrict__ pool,
                                                      const float2 *__restrict__ tab) {
    constexpr int N = Vec<T>::N;
    const unsigned nv = g.D / N;                  // vectors per (token, head) row
    const unsigned per_task = (unsigned)g.NC * g.H * nv;
    const unsigned n_task_items = per_task * rd.n_tasks;
    const unsigned n_items = n_task_items + per_task * (unsigned)rd.n_rerot;
    const size_t plane = (size_t)g.NC * g.D;      // elements of one [NC][D] plane
    const int hw = g.gh * g.gw;

    for (unsigned it = blockIdx.x * blockDim.x + threadIdx.x; it < n_items;
         it += gridDim.x * blockDim.x) {
        unsigned r = it < n_task_items ? it : it - n_task_items;
        int v = (int)(r % nv);
        unsigned r2 = r / nv;
        int h = (int)(r2 % (unsigned)g.H);
        unsigned r3 = r2 / (unsigned)g.H;
        int n = (int)(r3 % (unsigned)g.NC);
        int ti = (int)(r3 / (unsigned)g.NC);
        int f = n / hw, hh = (n / g.gw) % g.gh, ww = n % g.gw;
        int d0 = v * N;
        if (it < n_task_items) {
            int slot = rd.slot[ti];
            int t = g.gt * rd.chunk[ti] + f;
            const T *src = qkv + (((size_t)slot * g.NC + n) * 3 * g.H + h) * g.D + d0;
            uint4 q = *reinterpret_cast<const uint4 *>(src);
            uint4 k = *reinterpret_cast<const uint4 *>(src + (size_t)g.H * g.D);
            uint4 vv = *reinterpret_cast<const uint4 *>(src + (size_t)2 * g.H * g.D);
            T *qdst = qbuf + ((size_t)slot * g.H + h) * plane + (size_t)n * g.D + d0;
            *reinterpret_cast<uint4 *>(qdst) = rope_vec<T>(q, d0, t, hh, ww, g, tab);
            size_t kv_plane = (((size_t)rd.dest[ti] * g.L + layer) * 2) * g.H + h;
            T *kdst = pool + kv_plane * plane + (size_t)n * g.D + d0;
            *reinterpret_cast<uint4 *>(kdst) = rope_vec<T>(k, d0, t, hh, ww, g, tab);
            *reinterpret_cast<uint4 *>(kdst + (size_t)g.H * plane) = vv;
            if (rd.raw_page[ti] >= 0) {
                size_t raw_plane = (((size_t)rd.raw_page[ti] * g.L + layer) * 2) * g.H + h;
                *reinterpret_cast<uint4 *>(pool + raw_plane * plane + (size_t)n * g.D + d0) = k;
            }
        } else {
            // anchor re-rotation e = ti: unrotated copy -> anchor page at the new position
            int t = g.gt * rd.rerot_tpos[ti] + f;
            size_t raw_plane = (((size_t)rd.rerot_raw[ti] * g.L + layer) * 2) * g.H + h;
            size_t anc_plane = (((size_t)rd.rerot_anchor[ti] * g.L + layer) * 2) * g.H + h;
            uint4 k = *reinterpret_cast<const uint4 *>(pool + raw_plane * plane + (size_t)n * g.D + d0);
            *reinterpret_cast<uint4 *>(pool + anc_plane * plane + (size_t)n * g.D + d0) =
                rope_vec<T>(k, d0, t, hh, ww, g, tab);
        }
    }
}

// ---- 8-bit (e4m3) pages ------------------------------------------------------------
// Same placement as publish_kernel, for WF_FP8 plans: bf16 Q/K/V in, RoPE in
// fp32, then Q and K multiplied by qk_scale and V by v_scale and rounded to
// e4m3 (nearest even, saturating).  One thread handles 8 channels of one
// (token, head): 16 bytes of each input, 8 bytes of each output.  The
// anchor re-rotation reads the 8-bit unrotated copy.

__device__ __forceinline__ void rope8(float *x, int d0, int t, int hh, int ww, const WfGeom &g,
                                      const float2 *tab) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int m = d0 / 2 + i;
        float2 cs;
        if (m < g.dt2)
            cs = tab[g.rope_t_off + t * g.dt2 + m];
        else if (m < g.dt2 + g.dh2)
            cs = tab[g.rope_h_off + hh * g.dh2 + (m - g.dt2)];
        else
            cs = tab[g.rope_w_off + ww * g.dw2 + (m - g.dt2 - g.dh2)];
        float a = x[2 * i], b = x[2 * i + 1];
        x[2 * i] = a * cs.x - b * cs.y;
        x[2 * i + 1] = a * cs.y + b * cs.x;
    }
}

__device__ __forceinline__ uint2 e4m3x8(const float *x, float scale) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(x[2 * i] * scale, x[2 * i + 1] * scale),
                                                  __NV_SATFINITE, __NV_E4M3);
    return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

__device__ __forceinline__ void from_e4m3x8(uint2 u, float *x, float inv_scale) {
    const uint32_t w[2] = {u.x, u.y};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_fp8x2_storage_t h = (__nv_fp8x2_storage_t)((w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu);
        const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(h, __NV_E4M3)));
        x[2 * i] = f.x * inv_scale;
        x[2 * i + 1] = f.y * inv_scale;
    }
}

__global__ void __launch_bounds__(256) publish_fp8_kernel(const WfGeom g, const WfRoundDev rd,
                                                          int layer,
                                                          const __nv_bfloat16 *__restrict__ qkv,
                                                          uint8_t *__restrict__ qbuf,
                                                          uint8_t *__restrict__ pool,
                                                          const float2 *__restrict__ tab) {
    const unsigned nv = g.D / 8;
    const unsigned per_task = (unsigned)g.NC * g.H * nv;
    const unsigned n_task_items = per_task * rd.n_tasks;
    const unsigned n_items = n_task_items + per_task * (unsigned)rd.n_rerot;
    const size_t plane = (size_t)g.NC * g.D;
    const int hw = g.gh * g.gw;
    const float sqk = g.qk_scale, sv = g.v_scale;
    for (unsigned it = blockIdx.x * blockDim.x + threadIdx.x; it < n_items;
         it += gridDim.x * blockDim.x) {
        unsigned r = it < n_task_items ? it : it - n_task_items;
        int v = (int)(r % nv);
        unsigned r2 = r / nv;
        int h = (int)(r2 % (unsigned)g.H);
        unsigned r3 = r2 / (unsigned)g.H;
        int n = (int)(r3 % (unsigned)g.NC);
        int ti = (int)(r3 / (unsigned)g.NC);
        int f = n / hw, hh = (n / g.gw) % g.gh, ww = n % g.gw;
        int d0 = v * 8;
        if (it < n_task_items) {
            int slot = rd.slot[ti];
            int t = g.gt * rd.chunk[ti] + f;
            const __nv_bfloat16 *src = qkv + (((size_t)slot * g.NC + n) * 3 * g.H + h) * g.D + d0;
            float q[8], k[8], vv[8];
            unpack(*reinterpret_cast<const uint4 *>(src), q, (__nv_bfloat16 *)nullptr);
            unpack(*reinterpret_cast<const uint4 *>(src + (size_t)g.H * g.D), k, (__nv_bfloat16 *)nullptr);
            unpack(*reinterpret_cast<const uint4 *>(src + (size_t)2 * g.H * g.D), vv, (__nv_bfloat16 *)nullptr);
            size_t kv_plane = (((size_t)rd.dest[ti] * g.L + layer) * 2) * g.H + h;
            uint8_t *kdst = pool + kv_plane * plane + (size_t)n * g.D + d0;
            *reinterpret_cast<uint2 *>(kdst + (size_t)g.H * plane) = e4m3x8(vv, sv);
            if (rd.raw_page[ti] >= 0) {
                size_t raw_plane = (((size_t)rd.raw_page[ti] * g.L + layer) * 2) * g.H + h;
                *reinterpret_cast<uint2 *>(pool + raw_plane * plane + (size_t)n * g.D + d0) = e4m3x8(k, sqk);
            }
            rope8(q, d0, t, hh, ww, g, tab);
            rope8(k, d0, t, hh, ww, g, tab);
            *reinterpret_cast<uint2 *>(qbuf + ((size_t)slot * g.H + h) * plane + (size_t)n * g.D + d0) =
                e4m3x8(q, sqk);
            *reinterpret_cast<uint2 *>(kdst) = e4m3x8(k, sqk);
        } else {
            int t = g.gt * rd.rerot_tpos[ti] + f;
            size_t raw_plane = (((size_t)rd.rerot_raw[ti] * g.L + layer) * 2) * g.H + h;
            size_t anc_plane = (((size_t)rd.rerot_anchor[ti] * g.L + layer) * 2) * g.H + h;
            float k[8];
            from_e4m3x8(*reinterpret_cast<const uint2 *>(pool + raw_plane * plane + (size_t)n * g.D + d0),
                        k, 1.f / sqk);
            rope8(k, d0, t, hh, ww, g, tab);
            *reinterpret_cast<uint2 *>(pool + anc_plane * plane + (size_t)n * g.D + d0) = e4m3x8(k, sqk);
        }
    }
}

// ---- q/k RMSNorm, RoPE and paged publication ---------------------------------
// The standard Wan2.1 block normalises the projected q and k over the full
// model width before RoPE ("Wave Forcing" App. D.2 keeps that architecture):
// y = x / sqrt(mean(x^2) + 1e-6) * gain.  The QKV projection's epilogue sees
// only 256 of a row's columns, so it leaves the unrotated q | k rows in bf16
// and this kernel finishes them: one warp per (token row, q or k) reads the
// row (16 bytes per lane per step, coalesced), reduces the sum of squares
// with shuffles, then scales by the gain, rotates and stores Q into the
// query workspace or K into its page (plus the normalised unrotated key of
// the anchor when chunk 0 is stored).  HBM-bound: 2 dim bf16 read and 2 dim
// elements written per token.  NV > 0 keeps the row in registers (dim =
// 256 NV, up to 3072, where a warp still needs < 128 registers); NV = 0
// handles any dim % 8 == 0 by reading the row twice (the second read hits
// the caches).

// Three 256-thread blocks per SM: the kernel is latency-bound at two (one
// warp's loads are in flight only until it starts computing), and the
// register cap this sets (85) costs at most a few bytes of spill.
template <int NV, bool F8>
__global__ void __launch_bounds__(256, 3) qk_norm_rope_kernel(const WfGeom g, const WfRoundDev rd,
                                                           const WfQkNormArgs a) {
    const int warp = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    const int row = a.row_begin + (warp >> 1);
    const int part = warp & 1;                        // 0: q, 1: k
    if (row >= a.row_end) return;
    const int dim = g.H * g.D;
    const int nvec = dim / 8;
    const __nv_bfloat16 *src = a.raw + (size_t)row * 2 * dim + (size_t)part * dim;
    const __nv_bfloat16 *gain = part ? a.gk : a.gq;
    float ss = 0.f;
    uint4 u[NV > 0 ? NV : 1];
    auto sumsq = [&](uint4 v) {
        float x[8];
        unpack(v, x, (__nv_bfloat16 *)nullptr);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(x[i], x[i], ss);
    };
    if constexpr (NV > 0) {
#pragma unroll
        for (int i = 0; i < NV; ++i) u[i] = __ldg(reinterpret_cast<const uint4 *>(src) + lane + 32 * i);
#pragma unroll
        for (int i = 0; i < NV; ++i) sumsq(u[i]);
    } else {
        for (int v = lane; v < nvec; v += 32) sumsq(__ldg(reinterpret_cast<const uint4 *>(src) + v));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float rstd = rsqrtf(ss / (float)dim + 1e-6f);

    const int slot = row / g.NC, n = row - slot * g.NC;
    const int ti = rd.task_of_slot[slot];
    if (ti < 0) return;                               // a slot without a task this round
    const int hw = g.gh * g.gw;
    const int f = n / hw, hh = (n / g.gw) % g.gh, ww = n % g.gw;
    const int t = g.gt * rd.chunk[ti] + f;
    const size_t plane = (size_t)g.NC * g.D;
    const int raw_page = part == 1 ? rd.raw_page[ti] : -1;
    const size_t kplane = (((size_t)rd.dest[ti] * g.L + a.layer) * 2) * g.H;
    const size_t rplane = (((size_t)(raw_page < 0 ? 0 : raw_page) * g.L + a.layer) * 2) * g.H;
    auto emit = [&](uint4 in, int v) {
        const int c = 8 * v;                          // channels c .. c + 7, one head
        float x[8], w[8];
        unpack(in, x, (__nv_bfloat16 *)nullptr);
        unpack(__ldg(reinterpret_cast<const uint4 *>(gain) + v), w, (__nv_bfloat16 *)nullptr);
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = x[i] * rstd * w[i];
        const int h = c / g.D, d0 = c - h * g.D;
        size_t dst;
        if (part == 0) {
            dst = ((size_t)slot * g.H + h) * plane + (size_t)n * g.D + d0;
        } else {
            dst = (kplane + h) * plane + (size_t)n * g.D + d0;
            if (raw_page >= 0) {
                const size_t raw = (rplane + h) * plane + (size_t)n * g.D + d0;
                if constexpr (F8)
                    *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(a.pool) + raw) = e4m3x8(x, g.qk_scale);
                else
                    *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(a.pool) + raw) =
                        pack(x, (__nv_bfloat16 *)nullptr);
            }
        }
        rope8(x, d0, t, hh, ww, g, a.tab);
        void *base = part == 0 ? a.qbuf : a.pool;
        if constexpr (F8)
            *reinterpret_cast<uint2 *>(static_cast<uint8_t *>(base) + dst) = e4m3x8(x, g.qk_scale);
        else
            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(base) + dst) =
                pack(x, (__nv_bfloat16 *)nullptr);
    };
    if constexpr (NV > 0) {
#pragma unroll
        for (int i = 0; i < NV; ++i) emit(u[i], lane + 32 * i);
    } else {
        for (int v = lane; v < nvec; v += 32) emit(__ldg(reinterpret_cast<const uint4 *>(src) + v), v);
    }
}

template <bool F8>
cudaError_t launch_qk_norm(const WfGeom &g, const WfRoundDev &rd, const WfQkNormArgs &a, int blocks,
                           cudaStream_t stream) {
    const int dim = g.H * g.D;
    const int nv = dim % 256 == 0 ? dim / 256 : 0;
    switch (nv) {
#define WF_QKN(NV) \
    case NV: qk_norm_rope_kernel<NV, F8><<<blocks, 256, 0, stream>>>(g, rd, a); break;
        WF_QKN(1) WF_QKN(2) WF_QKN(4) WF_QKN(6) WF_QKN(8) WF_QKN(12)
#undef WF_QKN
        default: qk_norm_rope_kernel<0, F8><<<blocks, 256, 0, stream>>>(g, rd, a); break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t wf_launch_qk_norm(const WfGeom &g, const WfRoundDev &rd, const WfQkNormArgs &a,
                              cudaStream_t stream) {
    if (g.D % 8 || (g.dtype != WF_BF16 && g.dtype != WF_FP8) || a.row_end <= a.row_begin)
        return cudaErrorInvalidValue;
    const long long warps = 2ll * (a.row_end - a.row_begin);
    const long long blocks = (warps + 7) / 8;
    if (blocks >= (1ll << 31)) return cudaErrorInvalidValue;
    return g.dtype == WF_FP8 ? launch_qk_norm<true>(g, rd, a, (int)blocks, stream)
                             : launch_qk_norm<false>(g, rd, a, (int)blocks, stream);
}

cudaError_t wf_launch_publish(const WfGeom &g, const WfRoundDev &rd, int layer, int dtype,
                              const void *qkv, void *qbuf, void *pool, const void *scratch,
                              cudaStream_t stream) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int threads = 256;
    int nvec = dtype == WF_FP32 ? 4 : 8;
    if (g.D % nvec) return cudaErrorInvalidValue;
    long long items = (long long)g.NC * g.H * (g.D / nvec) * (rd.n_tasks + rd.n_rerot);
    if (items >= (1ll << 31)) return cudaErrorInvalidValue;
    long long want = (items + threads - 1) / threads;
    // one wave of the grid-stride loop: as many blocks as fit on the SMs at
    // once (a second, partial wave of late-starting blocks would finish
    // after the first one)
    static std::atomic<int> resident[3];
    const int kind = dtype == WF_FP8 ? 0 : (dtype == WF_FP32 ? 1 : 2);
    int per_sm = resident[kind].load(std::memory_order_relaxed);
    if (per_sm < 1) {
        cudaError_t e;
        if (kind == 0)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, publish_fp8_kernel, threads, 0);
        else if (kind == 1)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, publish_kernel<float>, threads, 0);
        else
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, publish_kernel<__nv_bfloat16>, threads, 0);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) per_sm = 1;
        resident[kind].store(per_sm, std::memory_order_relaxed);
    }
    int blocks = (int)(want < (long long)sms * per_sm ? want : (long long)sms * per_sm);
    if (blocks < 1) blocks = 1;
    const float2 *tab =
        reinterpret_cast<const float2 *>(static_cast<const char *>(scratch) + WF_SCRATCH_TABLES);
    if (dtype == WF_FP8)
        publish_fp8_kernel<<<blocks, threads, 0, stream>>>(
            g, rd, layer, static_cast<const __nv_bfloat16 *>(qkv), static_cast<uint8_t *>(qbuf),
            static_cast<uint8_t *>(pool), tab);
    else if (dtype == WF_FP32)
        publish_kernel<float><<<blocks, threads, 0, stream>>>(
            g, rd, layer, static_cast<const float *>(qkv), static_cast<float *>(qbuf),
            static_cast<float *>(pool), tab);
    else
        publish_kernel<__nv_bfloat16><<<blocks, threads, 0, stream>>>(
            g, rd, layer, static_cast<const __nv_bfloat16 *>(qkv),
            static_cast<__nv_bfloat16 *>(qbuf), static_cast<__nv_bfloat16 *>(pool), tab);
    return cudaGetLastError();
}
