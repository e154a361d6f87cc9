// Round attention on the CUDA cores (fp32 path, and any head_dim that is a
// multiple of 32 up to 128).  Same semantics as the tensor-core kernel:
// for one task (chunk, stage) and head, softmax(Q K^T / sqrt(D)) V over the
// task's ordered context ("Wave Forcing", Sec. 3.1 Eq. 5), read page by page
// from the pool; chunks outside the context are never visited (Eq. 4), and
// inside a chunk attention is bidirectional.  Online softmax in fp32 with
// exact exponentials; accumulation order is fixed (context order, then key
// order), so results are deterministic.
//
// Block = 4 warps x 4 query rows; keys are staged 32 at a time in shared
// memory as fp32.  Each lane scores one key, the warp reduces max/sum with
// shuffles, and lanes own D/32 output channels.

#include <cuda_bf16.h>

#include "wf_internal.h"

namespace {

constexpr int ROWS_PER_WARP = 4;
constexpr int WARPS = 4;
constexpr int ROWS = ROWS_PER_WARP * WARPS;
constexpr int KT = 32;

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float v, float *d) { *d = v; }
__device__ __forceinline__ void from_f(float v, __nv_bfloat16 *d) { *d = __float2bfloat16_rn(v); }

template <typename T, int DV>  // DV = D / 32 channels per lane
__global__ void __launch_bounds__(128) attn_simt_kernel(const WfGeom g, const WfRoundDev rd,
                                                        int layer, const T *__restrict__ qbuf,
                                                        const T *__restrict__ pool,
                                                        T *__restrict__ out) {
    constexpr int D = DV * 32;
    extern __shared__ float sm[];
    float *Qs = sm;                   // [ROWS][D]
    float *Ks = Qs + ROWS * D;        // [KT][D + 1]
    float *Vs = Ks + KT * (D + 1);    // [KT][D]

    const int ti = blockIdx.z, h = blockIdx.y, row0 = blockIdx.x * ROWS;
    const int slot = rd.slot[ti];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t plane = (size_t)g.NC * D;
    const float scale = rsqrtf((float)D);

    const T *qsrc = qbuf + ((size_t)slot * g.H + h) * plane;
    for (int i = threadIdx.x; i < ROWS * D; i += blockDim.x) {
        int r = row0 + i / D;
        Qs[i] = r < g.NC ? to_f(qsrc[(size_t)r * D + i % D]) : 0.f;
    }

    float m[ROWS_PER_WARP], l[ROWS_PER_WARP], acc[ROWS_PER_WARP][DV];
#pragma unroll
    for (int r = 0; r < ROWS_PER_WARP; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int i = 0; i < DV; ++i) acc[r][i] = 0.f;
    }

    for (int c = 0; c < rd.n_ctx[ti]; ++c) {
        size_t kplane = (((size_t)rd.page[ti][c] * g.L + layer) * 2) * g.H + h;
        const T *kp = pool + kplane * plane;
        const T *vp = kp + (size_t)g.H * plane;
        for (int k0 = 0; k0 < g.NC; k0 += KT) {
            __syncthreads();
            for (int i = threadIdx.x; i < KT * D; i += blockDim.x) {
                int kr = i / D, d = i % D, key = k0 + kr;
                bool ok = key < g.NC;
                Ks[kr * (D + 1) + d] = ok ? to_f(kp[(size_t)key * D + d]) : 0.f;
                Vs[kr * D + d] = ok ? to_f(vp[(size_t)key * D + d]) : 0.f;
            }
            __syncthreads();
            const int nvalid = min(KT, g.NC - k0);
#pragma unroll
            for (int r = 0; r < ROWS_PER_WARP; ++r) {
                const float *q = Qs + (warp * ROWS_PER_WARP + r) * D;
                float s = -INFINITY;
                if (lane < nvalid) {
                    float dot = 0.f;
                    const float *kr = Ks + lane * (D + 1);
#pragma unroll 8
                    for (int d = 0; d < D; ++d) dot = fmaf(q[d], kr[d], dot);
                    s = dot * scale;
                }
                float mt = s;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
                float mn = fmaxf(m[r], mt);
                float alpha = expf(m[r] - mn);  // m = -inf on the first tile -> 0
                float p = lane < nvalid ? expf(s - mn) : 0.f;
                float ps = p;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
                l[r] = l[r] * alpha + ps;
#pragma unroll
                for (int i = 0; i < DV; ++i) acc[r][i] *= alpha;
                for (int kk = 0; kk < nvalid; ++kk) {
                    float pk = __shfl_sync(0xffffffffu, p, kk);
#pragma unroll
                    for (int i = 0; i < DV; ++i) acc[r][i] = fmaf(pk, Vs[kk * D + lane + 32 * i], acc[r][i]);
                }
                m[r] = mn;
            }
        }
    }

#pragma unroll
    for (int r = 0; r < ROWS_PER_WARP; ++r) {
        int row = row0 + warp * ROWS_PER_WARP + r;
        if (row < g.NC) {
            T *dst = out + (((size_t)slot * g.NC + row) * g.H + h) * D;
            float inv = 1.f / l[r];
#pragma unroll
            for (int i = 0; i < DV; ++i) from_f(acc[r][i] * inv, dst + lane + 32 * i);
        }
    }
}

template <typename T, int DV>
cudaError_t launch(const WfGeom &g, const WfRoundDev &rd, int layer, const void *qbuf,
                   const void *pool, void *out, cudaStream_t stream) {
    constexpr int D = DV * 32;
    dim3 grid((g.NC + ROWS - 1) / ROWS, g.H, rd.n_tasks);
    size_t smem = (size_t)(ROWS * D + KT * (D + 1) + KT * D) * sizeof(float);
    attn_simt_kernel<T, DV><<<grid, 128, smem, stream>>>(
        g, rd, layer, static_cast<const T *>(qbuf), static_cast<const T *>(pool),
        static_cast<T *>(out));
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch(const WfGeom &g, const WfRoundDev &rd, int layer, const void *qbuf,
                     const void *pool, void *out, cudaStream_t stream) {
    switch (g.D) {
        case 32: return launch<T, 1>(g, rd, layer, qbuf, pool, out, stream);
        case 64: return launch<T, 2>(g, rd, layer, qbuf, pool, out, stream);
        case 96: return launch<T, 3>(g, rd, layer, qbuf, pool, out, stream);
        case 128: return launch<T, 4>(g, rd, layer, qbuf, pool, out, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t wf_launch_attn_simt(const WfGeom &g, const WfRoundDev &rd, int layer, int dtype,
                                const void *qbuf, const void *pool, void *out,
                                cudaStream_t stream) {
    if (rd.n_tasks < 1) return cudaSuccess;
    if (dtype == WF_FP32) return dispatch<float>(g, rd, layer, qbuf, pool, out, stream);
    return dispatch<__nv_bfloat16>(g, rd, layer, qbuf, pool, out, stream);
}
