// Memory-bound pieces of the chunk-wise causal DiT forward ("Wave Forcing",
// Sec. 4.1: C_{s,l} performs attention and "the remaining block" of the
// standard Wan2.1 transformer, App. D.2):
//  * LayerNorm with per-task modulation, x' = LN(x) (1 + scale_s) + shift_s,
//    written as the bf16 input of the next linear layer;
//  * patchify: (1, 2, 2) latent patches of every active task into the bf16
//    rows of the patch-embedding GEMM;
//  * the timestep embedding and modulation tables, computed once per model
//    binding (each stage has a fixed timestep, App. A).

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "wf_internal.h"

namespace {

// ---- LayerNorm + modulation: one warp per row ---------------------------------
template <bool F8>
__global__ void __launch_bounds__(256) ln_mod_kernel(const float *__restrict__ x,
                                                     void *__restrict__ out, int row_begin,
                                                     int row_end, int dim, int NC,
                                                     const float *__restrict__ mod, int mod_ld,
                                                     int shift_off, int scale_off) {
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int row = row_begin + warp;
    if (row >= row_end) return;
    const float4 *xr = reinterpret_cast<const float4 *>(x + (size_t)row * dim);
    const int nv = dim >> 2;
    // two passes over the row (the second one hits L1): mean, then variance
    float s = 0.f;
    for (int i = lane; i < nv; i += 32) {
        float4 v = xr[i];
        s += (v.x + v.y) + (v.z + v.w);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float mean = s / dim;
    float q = 0.f;
    for (int i = lane; i < nv; i += 32) {
        float4 v = xr[i];
        float a = v.x - mean, b = v.y - mean, c = v.z - mean, d = v.w - mean;
        q += (a * a + b * b) + (c * c + d * d);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
    const float rstd = rsqrtf(q / dim + 1e-6f);
    const int slot = row / NC;
    const float4 *sh = reinterpret_cast<const float4 *>(mod + (size_t)slot * mod_ld + shift_off);
    const float4 *sc = reinterpret_cast<const float4 *>(mod + (size_t)slot * mod_ld + scale_off);
    for (int i = lane; i < nv; i += 32) {
        float4 v = xr[i], a = __ldg(sh + i), b = __ldg(sc + i);
        float y0 = fmaf((v.x - mean) * rstd, 1.f + b.x, a.x);
        float y1 = fmaf((v.y - mean) * rstd, 1.f + b.y, a.y);
        float y2 = fmaf((v.z - mean) * rstd, 1.f + b.z, a.z);
        float y3 = fmaf((v.w - mean) * rstd, 1.f + b.w, a.w);
        if constexpr (F8) {
            // e4m3 with unit scale: the input of an e4m3 linear layer
            const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(y0, y1), __NV_SATFINITE, __NV_E4M3);
            const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(y2, y3), __NV_SATFINITE, __NV_E4M3);
            reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(out) + (size_t)row * dim)[i] = lo | (hi << 16);
        } else {
            __nv_bfloat162 p0 = __floats2bfloat162_rn(y0, y1), p1 = __floats2bfloat162_rn(y2, y3);
            reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(out) + (size_t)row * dim)[i] =
                make_uint2(*reinterpret_cast<uint32_t *>(&p0), *reinterpret_cast<uint32_t *>(&p1));
        }
    }
}

// The same with the row held in registers (NV float4 per lane, dim = 128 NV):
// x is read from memory once, all of a lane's loads in flight together.
template <bool F8, int NV>
__global__ void __launch_bounds__(256) ln_mod_reg_kernel(const float *__restrict__ x,
                                                         void *__restrict__ out, int row_begin,
                                                         int row_end, int NC,
                                                         const float *__restrict__ mod, int mod_ld,
                                                         int shift_off, int scale_off) {
    constexpr int dim = 128 * NV;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int row = row_begin + warp;
    if (row >= row_end) return;
    const float4 *xr = reinterpret_cast<const float4 *>(x + (size_t)row * dim);
    float4 v[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) v[k] = xr[lane + 32 * k];
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) s += (v[k].x + v[k].y) + (v[k].z + v[k].w);
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float mean = s / dim;
    float q = 0.f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const float a = v[k].x - mean, b = v[k].y - mean, c = v[k].z - mean, d = v[k].w - mean;
        q += (a * a + b * b) + (c * c + d * d);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) q += __shfl_xor_sync(0xffffffffu, q, o);
    const float rstd = rsqrtf(q / dim + 1e-6f);
    const int slot = row / NC;
    const float4 *sh = reinterpret_cast<const float4 *>(mod + (size_t)slot * mod_ld + shift_off);
    const float4 *sc = reinterpret_cast<const float4 *>(mod + (size_t)slot * mod_ld + scale_off);
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        const int i = lane + 32 * k;
        const float4 a = __ldg(sh + i), b = __ldg(sc + i);
        const float y0 = fmaf((v[k].x - mean) * rstd, 1.f + b.x, a.x);
        const float y1 = fmaf((v[k].y - mean) * rstd, 1.f + b.y, a.y);
        const float y2 = fmaf((v[k].z - mean) * rstd, 1.f + b.z, a.z);
        const float y3 = fmaf((v[k].w - mean) * rstd, 1.f + b.w, a.w);
        if constexpr (F8) {
            const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(y0, y1), __NV_SATFINITE, __NV_E4M3);
            const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(y2, y3), __NV_SATFINITE, __NV_E4M3);
            reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(out) + (size_t)row * dim)[i] = lo | (hi << 16);
        } else {
            __nv_bfloat162 p0 = __floats2bfloat162_rn(y0, y1), p1 = __floats2bfloat162_rn(y2, y3);
            reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(out) + (size_t)row * dim)[i] =
                make_uint2(*reinterpret_cast<uint32_t *>(&p0), *reinterpret_cast<uint32_t *>(&p1));
        }
    }
}

// ---- patchify -------------------------------------------------------------------
// Row n of slot s: features (channel c, row offset q, column offset r) of the
// 2 x 2 patch of token (f, h, w); one thread per (token, channel).
struct SlotSrc {
    const float *p[WF_MAX_ROUND_TASKS];   // per (global) slot
};

__global__ void __launch_bounds__(256) patchify_kernel(const WfGeom g, int C, SlotSrc src, int lo,
                                                       int hi, __nv_bfloat16 *__restrict__ patches) {
    const long long total = (long long)(hi - lo + 1) * g.NC * C;
    const int Hl = 2 * g.gh, Wl = 2 * g.gw;
    const size_t cstride = (size_t)g.gt * Hl * Wl;
    for (long long it = blockIdx.x * (long long)blockDim.x + threadIdx.x; it < total;
         it += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(it % C);
        const long long tok = it / C;
        const int slot = lo + (int)(tok / g.NC);
        const int n = (int)(tok % g.NC);
        const int hw = g.gh * g.gw;
        const int f = n / hw, hh = (n / g.gw) % g.gh, ww = n % g.gw;
        float2 top = make_float2(0.f, 0.f), bot = top;     // a slot without a task: zero patches
        if (src.p[slot]) {
            const float *z = src.p[slot] + (size_t)c * cstride + ((size_t)f * Hl + 2 * hh) * Wl + 2 * ww;
            top = *reinterpret_cast<const float2 *>(z);
            bot = *reinterpret_cast<const float2 *>(z + Wl);
        }
        __nv_bfloat162 a = __floats2bfloat162_rn(top.x, top.y), b = __floats2bfloat162_rn(bot.x, bot.y);
        uint2 w = make_uint2(*reinterpret_cast<uint32_t *>(&a), *reinterpret_cast<uint32_t *>(&b));
        *reinterpret_cast<uint2 *>(patches + ((size_t)slot * g.NC + n) * 4 * C + 4 * c) = w;
    }
}

// ---- timestep embedding (run once per binding) ----------------------------------
__global__ void sinusoid_kernel(const float *__restrict__ t_model, int B, int freq, float *out,
                                int out_ld) {
    const int half = freq / 2;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < B * half; i += gridDim.x * blockDim.x) {
        const int b = i / half, j = i % half;
        const double w = pow(10000.0, -(double)j / half);
        const double a = (double)t_model[b] * w;
        out[(size_t)b * out_ld + j] = (float)cos(a);
        out[(size_t)b * out_ld + half + j] = (float)sin(a);
    }
}

// out[b][n] = sum_k W[n][k] act(in[b][k]) + bias[n]; act = SiLU when silu_in.
// One warp per output feature n, all B rows at once (B <= WF_MAX_TASKS).
__global__ void __launch_bounds__(256) gemv_kernel(const __nv_bfloat16 *__restrict__ W,
                                                   const __nv_bfloat16 *__restrict__ bias,
                                                   const float *in, int in_ld, float *out, int out_ld,
                                                   int B, int N, int K, int silu_in) {
    const int n = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (n >= N) return;
    float acc[WF_MAX_TASKS];
#pragma unroll
    for (int b = 0; b < WF_MAX_TASKS; ++b) acc[b] = 0.f;
    for (int k = lane; k < K; k += 32) {
        const float w = __bfloat162float(W[(size_t)n * K + k]);
#pragma unroll
        for (int b = 0; b < WF_MAX_TASKS; ++b) {
            if (b >= B) break;
            float v = in[(size_t)b * in_ld + k];
            if (silu_in) v = v / (1.f + expf(-v));
            acc[b] = fmaf(w, v, acc[b]);
        }
    }
#pragma unroll
    for (int b = 0; b < WF_MAX_TASKS; ++b) {
        if (b >= B) break;
        float a = acc[b];
#pragma unroll
        for (int o = 16; o; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0) out[(size_t)b * out_ld + n] = a + (bias ? __bfloat162float(bias[n]) : 0.f);
    }
}

// modtab[l][b][i][:] = mod_l[i][:] + e0[b % B][i][:];  headtab[b][i][:] = head_mod[i][:] + e[b % B][:]
// for b < B_out: the tables of the B stage slots, written once per request of
// a group (B_out = n B; slot b of the group is stage b % B).
__global__ void tables_kernel(const WfDitLayerDev *layers, int L, int B, int B_out, int dim,
                              const float *temb, int temb_ld, int e_off, int e0_off,
                              const __nv_bfloat16 *head_mod, float *modtab, float *headtab) {
    const long long n_mod = (long long)L * B_out * 6 * dim;
    const long long n_head = (long long)B_out * 2 * dim;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n_mod + n_head;
         i += (long long)gridDim.x * blockDim.x) {
        if (i < n_mod) {
            const int c = (int)(i % dim);
            const int r = (int)((i / dim) % 6);
            const int b = (int)((i / (6LL * dim)) % B_out);
            const int l = (int)(i / (6LL * dim * B_out));
            modtab[i] = __bfloat162float(layers[l].mod[r * dim + c]) +
                        temb[(size_t)(b % B) * temb_ld + e0_off + r * dim + c];
        } else {
            const long long j = i - n_mod;
            const int c = (int)(j % dim);
            const int r = (int)((j / dim) % 2);
            const int b = (int)(j / (2LL * dim));
            headtab[j] = __bfloat162float(head_mod[r * dim + c]) +
                         temb[(size_t)(b % B) * temb_ld + e_off + c];
        }
    }
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

size_t wf_dit_workspace_bytes(int S, int NC, int dim, int ffn, int C, int freq, int L, size_t latent,
                              int linear_fp8) {
    const size_t rows = (size_t)(S + 1) * NC, B = S + 1;
    const size_t hcols = ffn > 2 * dim ? ffn : 2 * dim;   // FFN hidden layer, or q | k rows
    size_t b = align256(rows * dim * 4) + align256(rows * dim * 2) + align256(rows * hcols * 2) +
               align256(rows * 4 * C * 2) + align256(2 * B * latent * 4) +
               align256((size_t)L * B * 6 * dim * 4) + align256(B * 2 * dim * 4) +
               align256(B * (size_t)(freq + 9 * dim) * 4) + align256((size_t)L * sizeof(WfDitLayerDev)) +
               align256(B * 4);
    if (linear_fp8) {
        const size_t d = dim, f = ffn;
        b += align256(rows * d) + align256(rows * f);
        b += (size_t)L * (align256(3 * d * d) + align256(d * d) + align256(f * d) + align256(d * f) +
                          align256(3 * d * 4) + align256(d * 4) + align256(f * 4) + align256(d * 4));
    }
    return b;
}

void wf_dit_carve(WfDit *d, void *ws, int S, int NC, size_t latent) {
    const size_t rows = (size_t)(S + 1) * NC, B = S + 1;
    char *p = static_cast<char *>(ws);
    auto take = [&](size_t bytes) { char *r = p; p += align256(bytes); return r; };
    d->x = reinterpret_cast<float *>(take(rows * d->dim * 4));
    d->xa = reinterpret_cast<__nv_bfloat16 *>(take(rows * d->dim * 2));
    const size_t hcols = d->ffn > 2 * d->dim ? d->ffn : 2 * d->dim;
    d->hmid = reinterpret_cast<__nv_bfloat16 *>(take(rows * hcols * 2));
    d->patches = reinterpret_cast<__nv_bfloat16 *>(take(rows * 4 * d->C * 2));
    d->lat = reinterpret_cast<float *>(take(2 * B * latent * 4));
    d->modtab = reinterpret_cast<float *>(take((size_t)d->L * B * 6 * d->dim * 4));
    d->headtab = reinterpret_cast<float *>(take(B * 2 * d->dim * 4));
    d->temb = reinterpret_cast<float *>(take(B * (size_t)(d->freq + 9 * d->dim) * 4));
    d->layers_dev = reinterpret_cast<WfDitLayerDev *>(take((size_t)d->L * sizeof(WfDitLayerDev)));
    d->tmodel = reinterpret_cast<float *>(take(B * 4));
    d->latent = latent;
    d->xa8 = d->h8 = nullptr;
    if (d->linear_fp8) {
        const size_t dm = d->dim, f = d->ffn;
        d->xa8 = reinterpret_cast<uint8_t *>(take(rows * dm));
        d->h8 = reinterpret_cast<uint8_t *>(take(rows * f));
        for (int l = 0; l < d->L; ++l) {
            WfDitLayerDev &w = d->layers[l];
            w.qkv_w8 = reinterpret_cast<uint8_t *>(take(3 * dm * dm));
            w.o_w8 = reinterpret_cast<uint8_t *>(take(dm * dm));
            w.f1_w8 = reinterpret_cast<uint8_t *>(take(f * dm));
            w.f2_w8 = reinterpret_cast<uint8_t *>(take(dm * f));
            w.qkv_s = reinterpret_cast<float *>(take(3 * dm * 4));
            w.o_s = reinterpret_cast<float *>(take(dm * 4));
            w.f1_s = reinterpret_cast<float *>(take(f * 4));
            w.f2_s = reinterpret_cast<float *>(take(dm * 4));
        }
    }
}

cudaError_t wf_launch_ln_mod(const float *x, void *out, int row_begin, int row_end, int dim, int NC,
                             const float *mod, int mod_ld, int shift_off, int scale_off,
                             cudaStream_t stream, bool out_e4m3) {
    if (dim % 4 || row_end <= row_begin) return cudaErrorInvalidValue;
    const int rows = row_end - row_begin;
    const int blocks = (rows + 7) / 8;
#define WF_LN_REG(NV)                                                                                  \
    if (dim == 128 * NV) {                                                                             \
        if (out_e4m3)                                                                                  \
            ln_mod_reg_kernel<true, NV><<<blocks, 256, 0, stream>>>(x, out, row_begin, row_end, NC, mod,  \
                                                                    mod_ld, shift_off, scale_off);     \
        else                                                                                           \
            ln_mod_reg_kernel<false, NV><<<blocks, 256, 0, stream>>>(x, out, row_begin, row_end, NC, mod, \
                                                                     mod_ld, shift_off, scale_off);    \
        return cudaGetLastError();                                                                     \
    }
    WF_LN_REG(12)   // dim 1536 (Wan2.1-1.3B)
    WF_LN_REG(16)   // dim 2048
    WF_LN_REG(2)    // dim 256
#undef WF_LN_REG
    if (out_e4m3)
        ln_mod_kernel<true><<<blocks, 256, 0, stream>>>(x, out, row_begin, row_end, dim, NC, mod, mod_ld,
                                                        shift_off, scale_off);
    else
        ln_mod_kernel<false><<<blocks, 256, 0, stream>>>(x, out, row_begin, row_end, dim, NC, mod, mod_ld,
                                                         shift_off, scale_off);
    return cudaGetLastError();
}

cudaError_t wf_launch_patchify(const WfGeom &g, int C, const float *const *src, int lo, int hi,
                               __nv_bfloat16 *patches, cudaStream_t stream) {
    if (lo < 0 || hi >= WF_MAX_ROUND_TASKS || hi < lo) return cudaErrorInvalidValue;
    SlotSrc s{};
    for (int i = lo; i <= hi; ++i) s.p[i] = src[i];
    const long long total = (long long)(hi - lo + 1) * g.NC * C;
    long long want = (total + 255) / 256;
    int blocks = (int)(want < 148 * 16 ? want : 148 * 16);
    if (blocks < 1) blocks = 1;
    patchify_kernel<<<blocks, 256, 0, stream>>>(g, C, s, lo, hi, patches);
    return cudaGetLastError();
}

cudaError_t wf_launch_time_embedding(const WfDit &d, int S, int n_req, cudaStream_t stream) {
    // temb row b: [sinusoid (freq) | h1 (dim) | e (dim) | e0 (6 dim)]
    const int B = S + 1, dim = d.dim;
    const int ld = d.freq + 9 * dim;
    const int o_h1 = d.freq, o_e = d.freq + dim, o_e0 = d.freq + 2 * dim;
    float *T = d.temb;
    sinusoid_kernel<<<8, 256, 0, stream>>>(d.tmodel, B, d.freq, T, ld);
    auto gemv = [&](const __nv_bfloat16 *W, const __nv_bfloat16 *b, int in_off, int out_off, int N,
                    int K, int silu) {
        gemv_kernel<<<(N * 32 + 255) / 256, 256, 0, stream>>>(W, b, T + in_off, ld, T + out_off, ld,
                                                              B, N, K, silu);
    };
    gemv(d.t1_w, d.t1_b, 0, o_h1, dim, d.freq, 0);
    gemv(d.t2_w, d.t2_b, o_h1, o_e, dim, dim, 1);
    gemv(d.tp_w, d.tp_b, o_e, o_e0, 6 * dim, dim, 1);
    tables_kernel<<<148 * 4, 256, 0, stream>>>(d.layers_dev, d.L, B, n_req * B, dim, T, ld, o_e, o_e0,
                                               d.head_mod, d.modtab, d.headtab);
    return cudaGetLastError();
}
