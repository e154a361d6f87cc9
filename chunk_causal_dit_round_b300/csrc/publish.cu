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
    const unsigned n_items = n_task_items + (rd.rerotate ? per_task : 0u);
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
            if (ti == rd.raw_copy_task) {
                size_t raw_plane = (((size_t)g.raw_anchor_page * g.L + layer) * 2) * g.H + h;
                *reinterpret_cast<uint4 *>(pool + raw_plane * plane + (size_t)n * g.D + d0) = k;
            }
        } else {
            // anchor re-rotation: unrotated copy -> anchor page 0 at the new position
            int t = g.gt * rd.anchor_tpos + f;
            size_t raw_plane = (((size_t)g.raw_anchor_page * g.L + layer) * 2) * g.H + h;
            size_t anc_plane = (((size_t)0 * g.L + layer) * 2) * g.H + h;
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
    const unsigned n_items = n_task_items + (rd.rerotate ? per_task : 0u);
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
            if (ti == rd.raw_copy_task) {
                size_t raw_plane = (((size_t)g.raw_anchor_page * g.L + layer) * 2) * g.H + h;
                *reinterpret_cast<uint2 *>(pool + raw_plane * plane + (size_t)n * g.D + d0) = e4m3x8(k, sqk);
            }
            rope8(q, d0, t, hh, ww, g, tab);
            rope8(k, d0, t, hh, ww, g, tab);
            *reinterpret_cast<uint2 *>(qbuf + ((size_t)slot * g.H + h) * plane + (size_t)n * g.D + d0) =
                e4m3x8(q, sqk);
            *reinterpret_cast<uint2 *>(kdst) = e4m3x8(k, sqk);
        } else {
            int t = g.gt * rd.anchor_tpos + f;
            size_t raw_plane = (((size_t)g.raw_anchor_page * g.L + layer) * 2) * g.H + h;
            size_t anc_plane = (((size_t)0 * g.L + layer) * 2) * g.H + h;
            float k[8];
            from_e4m3x8(*reinterpret_cast<const uint2 *>(pool + raw_plane * plane + (size_t)n * g.D + d0),
                        k, 1.f / sqk);
            rope8(k, d0, t, hh, ww, g, tab);
            *reinterpret_cast<uint2 *>(pool + anc_plane * plane + (size_t)n * g.D + d0) = e4m3x8(k, sqk);
        }
    }
}

}  // namespace

cudaError_t wf_launch_publish(const WfGeom &g, const WfRoundDev &rd, int layer, int dtype,
                              const void *qkv, void *qbuf, void *pool, const void *scratch,
                              cudaStream_t stream) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int threads = 256;
    int nvec = dtype == WF_FP32 ? 4 : 8;
    if (g.D % nvec) return cudaErrorInvalidValue;
    long long items = (long long)g.NC * g.H * (g.D / nvec) * (rd.n_tasks + (rd.rerotate ? 1 : 0));
    if (items >= (1ll << 31)) return cudaErrorInvalidValue;
    long long want = (items + threads - 1) / threads;
    int blocks = (int)(want < (long long)sms * 8 ? want : (long long)sms * 8);
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
