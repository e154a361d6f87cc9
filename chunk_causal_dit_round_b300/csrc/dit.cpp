// Host side of the DiT path: the generic linear-layer entry point, the QKV
// projection with its RoPE + paged-publication epilogue, and one whole
// wavefront round of the chunk-wise causal DiT forward ("Wave Forcing",
// Sec. 2 Eq. 1; Sec. 3.1 Eq. 3-5; Sec. 4.1 Eq. 8-9 dependency order; App. A
// schedules; App. B.3 store pass).
//
// On one GPU and one stream the per-layer dependencies of Eq. 8-9 hold by
// construction: every task's projection P_{s,l} (one batched GEMM over all
// active tasks) completes before the round's attention C_{s,l} for that
// layer, and C_{s,l} before P_{s,l+1}.

#include <cmath>
#include <functional>
#include <cstring>
#include <new>

#include "wf_plan_impl.h"

namespace {

bool aligned16(const void *q) { return ((uintptr_t)q & 15) == 0; }

double warp_sigma(double nu, double shift) {
    double s = nu / 1000.0;
    return shift * s / (1.0 + (shift - 1.0) * s);
}

GemmParams base_params(wf_plan_s *p, int row_begin, int row_end, int N, int K, const void *bias) {
    GemmParams gp;
    std::memset(&gp, 0, sizeof(gp));
    gp.row_begin = row_begin;
    gp.row_end = row_end;
    gp.N = N;
    gp.K = K;
    gp.bias = static_cast<const __nv_bfloat16 *>(bias);
    gp.status = static_cast<uint32_t *>(p->scratch);
    return gp;
}

}  // namespace

// Binding shared by a plan (n_req = 1) and a group of n_req plans of p's
// shape: the activations and tables are sized for n_req (S+1) slots, the
// modulation and head tables written once per request.
int wf_dit_bind_impl(WfDit *dp, const wf_plan_s *p, const wf_dit_model *m, void *workspace,
                     int n_req, cudaStream_t stream) {
    if ((p->o.dtype != WF_BF16 && p->o.dtype != WF_FP8) || p->D != 128) return WF_EUNSUPPORTED;
    if ((uintptr_t)workspace & 255) return WF_EINVAL;
    size_t need;
    int rc = wf_dit_workspace_size(const_cast<wf_plan_s *>(p), m->model_dim, m->ffn_dim, m->channels,
                                   m->freq_dim, m->linear_fp8, &need);
    if (rc != WF_OK) return rc;
    if (!(m->shift > 0.0) || !std::isfinite(m->shift) || !(m->context_noise >= 0.0) ||
        !(m->context_noise <= 1000.0))
        return WF_EINVAL;
    for (int s = 0; s < p->S; ++s)
        if (!(m->timesteps[s] > 0.0 && m->timesteps[s] <= 1000.0) ||
            (s > 0 && !(m->timesteps[s] < m->timesteps[s - 1])))
            return WF_EINVAL;
    const void *ptrs[] = {m->patch_w, m->t1_w, m->t1_b, m->t2_w, m->t2_b, m->tp_w, m->tp_b,
                          m->head_w, m->head_mod, m->layers};
    for (const void *q : ptrs)
        if (!q) return WF_EINVAL;
    const int L = p->o.layers;
    for (int l = 0; l < L; ++l) {
        const wf_dit_layer &w = m->layers[l];
        if (!w.qkv_w || !w.o_w || !w.ffn1_w || !w.ffn2_w || !w.modulation || !w.norm_q || !w.norm_k)
            return WF_EINVAL;
        const void *all[] = {w.qkv_w, w.qkv_b, w.o_w, w.o_b, w.ffn1_w, w.ffn1_b, w.ffn2_w, w.ffn2_b,
                             w.norm_q, w.norm_k};
        for (const void *q : all)
            if (q && !aligned16(q)) return WF_EINVAL;
    }
    WfDit &d = *dp;
    delete[] d.layers;
    d.layers = nullptr;
    d.dim = m->model_dim;
    d.ffn = m->ffn_dim;
    d.C = m->channels;
    d.freq = m->freq_dim;
    d.L = L;
    d.linear_fp8 = m->linear_fp8;
    d.shift = m->shift;
    d.context_noise = m->context_noise;
    for (int s = 0; s < p->S; ++s) d.nu[s] = m->timesteps[s];
    d.nu[p->S] = 0.0;
    auto B = [](const void *q) { return static_cast<const __nv_bfloat16 *>(q); };
    d.patch_w = B(m->patch_w); d.patch_b = B(m->patch_b);
    d.t1_w = B(m->t1_w); d.t1_b = B(m->t1_b);
    d.t2_w = B(m->t2_w); d.t2_b = B(m->t2_b);
    d.tp_w = B(m->tp_w); d.tp_b = B(m->tp_b);
    d.head_w = B(m->head_w); d.head_b = B(m->head_b); d.head_mod = B(m->head_mod);
    d.layers = new (std::nothrow) WfDitLayerDev[L];
    if (!d.layers) return WF_ENOMEM;
    for (int l = 0; l < L; ++l) {
        const wf_dit_layer &w = m->layers[l];
        d.layers[l] = {B(w.qkv_w), B(w.qkv_b), B(w.o_w), B(w.o_b), B(w.ffn1_w),
                       B(w.ffn1_b), B(w.ffn2_w), B(w.ffn2_b), B(w.modulation),
                       B(w.norm_q), B(w.norm_k),
                       nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};
    }
    const size_t latent = (size_t)d.C * p->g.gt * 4 * p->g.gh * p->g.gw;
    const int slots = n_req * (p->S + 1);
    wf_dit_carve(&d, workspace, slots - 1, p->NC, latent);
    // model timestep per stage slot: warped nu_s for stage s, warped context_noise for the store
    float tm[WF_MAX_TASKS];
    for (int s = 0; s < p->S; ++s) tm[s] = (float)(1000.0 * warp_sigma(d.nu[s], d.shift));
    tm[p->S] = (float)(1000.0 * warp_sigma(d.context_noise, d.shift));
    if (cudaMemcpy(d.tmodel, tm, sizeof(float) * (p->S + 1), cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(d.layers_dev, d.layers, sizeof(WfDitLayerDev) * L, cudaMemcpyHostToDevice) !=
            cudaSuccess)
        return WF_ECUDA;
    if (cudaMemsetAsync(d.lat, 0, 2 * (size_t)slots * latent * 4, stream) != cudaSuccess)
        return WF_ECUDA;
    if (wf_launch_time_embedding(d, p->S, n_req, stream) != cudaSuccess) return WF_ECUDA;
    if (d.linear_fp8) {
        const int dm = d.dim, f = d.ffn;
        for (int l = 0; l < L; ++l) {
            const WfDitLayerDev &w = d.layers[l];
            if (wf_launch_quant_rows(w.qkv_w, 3 * dm, dm, w.qkv_w8, w.qkv_s, stream) != cudaSuccess ||
                wf_launch_quant_rows(w.o_w, dm, dm, w.o_w8, w.o_s, stream) != cudaSuccess ||
                wf_launch_quant_rows(w.f1_w, f, dm, w.f1_w8, w.f1_s, stream) != cudaSuccess ||
                wf_launch_quant_rows(w.f2_w, dm, f, w.f2_w8, w.f2_s, stream) != cudaSuccess)
                return WF_ECUDA;
        }
    }
    return WF_OK;
}

// One DiT forward over the rows [r0, r1) of n_slots slot-indexed buffers
// (a plan's S+1 slots, or a group's n (S+1)), every layer's publication and
// attention through the given callbacks, then the head and the stage
// transition into each request's next-round slot buffers.
int wf_dit_pass(const WfDitPass &a, cudaStream_t stream) {
    WfDit &d = *a.d;
    const WfGeom &g = *a.g;
    const int NC = g.NC, S = g.S;
    const int dim = d.dim, mod_ld = 6 * dim;
    const long long rows = (long long)a.n_slots * NC;
    auto params = [&](int N, int K, const void *bias) {
        GemmParams gp;
        std::memset(&gp, 0, sizeof(gp));
        gp.row_begin = a.r0;
        gp.row_end = a.r1;
        gp.N = N;
        gp.K = K;
        gp.bias = static_cast<const __nv_bfloat16 *>(bias);
        gp.status = a.status;
        return gp;
    };
    // patch embedding of every active task's input latent
    if (wf_launch_patchify(g, d.C, a.src, a.lo, a.hi, d.patches, stream) != cudaSuccess) return WF_ECUDA;
    GemmParams gp = params(dim, 4 * d.C, d.patch_b);
    gp.out = d.x;
    gp.ldo = dim;
    if (wf_launch_gemm(WF_EPI_F32, d.patches, rows, 4 * d.C, d.patch_w, gp, a.num_sms, stream) !=
        cudaSuccess)
        return WF_ECUDA;

    const bool f8 = d.linear_fp8 != 0;
    for (int l = 0; l < d.L; ++l) {
        const WfDitLayerDev &w = d.layers[l];
        const float *mod = d.modtab + (size_t)l * a.n_slots * mod_ld;
        // activations of the linear layers: bf16, or e4m3 with e4m3 weights
        void *act = f8 ? static_cast<void *>(d.xa8) : static_cast<void *>(d.xa);
        // P_{s,l}: x' = LN(x)(1 + scale_a) + shift_a; QKV projection, q/k RMSNorm, RoPE, publish
        if (wf_launch_ln_mod(d.x, act, a.r0, a.r1, dim, NC, mod, mod_ld, 0, dim, stream, f8) != cudaSuccess)
            return WF_ECUDA;
        int rc = a.publish(l, act, w, f8);
        if (rc != WF_OK) return rc;
        // C_{s,l}: round attention (output over x', which is dead), then the rest of the block
        rc = a.attend(l, act, f8);
        if (rc != WF_OK) return rc;
        gp = params(dim, dim, w.o_b);
        gp.out = d.x;
        gp.ldo = dim;
        gp.gate = mod + 2 * dim;
        gp.gate_ld = mod_ld;
        gp.rows_per_group = NC;
        gp.wscale = w.o_s;
        if (wf_launch_gemm(WF_EPI_GATED_RESIDUAL, act, rows, dim, f8 ? (const void *)w.o_w8 : w.o_w, gp,
                           a.num_sms, stream, f8) != cudaSuccess)
            return WF_ECUDA;
        if (wf_launch_ln_mod(d.x, act, a.r0, a.r1, dim, NC, mod, mod_ld, 3 * dim, 4 * dim, stream, f8) !=
            cudaSuccess)
            return WF_ECUDA;
        gp = params(d.ffn, dim, w.f1_b);
        gp.out = f8 ? static_cast<void *>(d.h8) : static_cast<void *>(d.hmid);
        gp.ldo = d.ffn;
        gp.wscale = w.f1_s;
        if (wf_launch_gemm(f8 ? WF_EPI_GELU_E4M3 : WF_EPI_GELU_BF16, act, rows, dim,
                           f8 ? (const void *)w.f1_w8 : w.f1_w, gp, a.num_sms, stream, f8) != cudaSuccess)
            return WF_ECUDA;
        gp = params(dim, d.ffn, w.f2_b);
        gp.out = d.x;
        gp.ldo = dim;
        gp.gate = mod + 5 * dim;
        gp.gate_ld = mod_ld;
        gp.rows_per_group = NC;
        gp.wscale = w.f2_s;
        if (wf_launch_gemm(WF_EPI_GATED_RESIDUAL, f8 ? static_cast<const void *>(d.h8) : d.hmid, rows,
                           d.ffn, f8 ? (const void *)w.f2_w8 : w.f2_w, gp, a.num_sms, stream, f8) !=
            cudaSuccess)
            return WF_ECUDA;
    }

    // head and stage transition (Eq. 1) into next round's slot inputs
    if (wf_launch_ln_mod(d.x, d.xa, a.r0, a.r1, dim, NC, d.headtab, 2 * dim, 0, dim, stream) !=
        cudaSuccess)
        return WF_ECUDA;
    gp = params(4 * d.C, dim, d.head_b);
    gp.g = g;
    gp.rd = *a.rd;
    gp.channels = d.C;
    for (int s = 0; s <= S; ++s)
        gp.sigma_next[s] = s < S ? (float)warp_sigma(d.nu[s + 1], d.shift) : 0.f;
    gp.eps = a.eps;
    for (int m = 0; m < WF_MAX_GROUP; ++m) gp.z_next[m] = a.z_next[m];
    gp.x0_out = a.x0_out;
    gp.chunk_out = a.chunk_out;
    if (wf_launch_gemm(WF_EPI_HEAD, d.xa, rows, dim, d.head_w, gp, a.num_sms, stream) != cudaSuccess)
        return WF_ECUDA;
    return WF_OK;
}

extern "C" {

int wf_linear(wf_plan_t p, const void *a, long long a_rows, int lda, int row_begin, int row_end,
              const void *w, const void *bias, int N, int K, int epilogue, void *out, int ldo,
              const float *gate, int gate_ld, int rows_per_group, cudaStream_t stream) {
    if (!p) return WF_EINVAL;
    if (!p->bound) return WF_EUNBOUND;
    if (!a || !w || !out) return WF_EINVAL;
    if (epilogue < WF_EPI_BF16 || epilogue > WF_EPI_GATED_RESIDUAL) return WF_EINVAL;
    if (K < 64 || K % 64 || N < 32 || N % 32 || lda < K || lda % 8 || ldo < N || ldo % 8)
        return WF_EINVAL;
    if (row_begin < 0 || row_end <= row_begin || row_end > a_rows) return WF_ERANGE;
    if (!aligned16(a) || !aligned16(w) || !aligned16(out) || (bias && !aligned16(bias)))
        return WF_EINVAL;
    if (epilogue == WF_EPI_GATED_RESIDUAL &&
        (!gate || !aligned16(gate) || gate_ld % 4 || gate_ld < N || rows_per_group < 1))
        return WF_EINVAL;
    GemmParams gp = base_params(p, row_begin, row_end, N, K, bias);
    gp.out = out;
    gp.ldo = ldo;
    gp.gate = gate;
    gp.gate_ld = gate_ld;
    gp.rows_per_group = rows_per_group > 0 ? rows_per_group : 1;
    return wf_launch_gemm(epilogue, a, a_rows, lda, w, gp, p->num_sms, stream) == cudaSuccess
               ? WF_OK
               : WF_ECUDA;
}

int wf_quantize_weight_e4m3(wf_plan_t p, const void *w, int N, int K, void *w8, float *scale,
                            cudaStream_t stream) {
    if (!p) return WF_EINVAL;
    if (!p->bound) return WF_EUNBOUND;
    if (!w || !w8 || !scale || N < 1 || K < 2 || K % 2) return WF_EINVAL;
    return wf_launch_quant_rows(w, N, K, w8, scale, stream) == cudaSuccess ? WF_OK : WF_ECUDA;
}

int wf_linear_e4m3(wf_plan_t p, const void *a8, long long a_rows, int lda, int row_begin,
                   int row_end, const void *w8, const float *wscale, const void *bias, int N, int K,
                   int epilogue, void *out, int ldo, const float *gate, int gate_ld,
                   int rows_per_group, cudaStream_t stream) {
    if (!p) return WF_EINVAL;
    if (!p->bound) return WF_EUNBOUND;
    if (!a8 || !w8 || !wscale || !out) return WF_EINVAL;
    if (epilogue < WF_EPI_BF16 || epilogue > WF_EPI_GATED_RESIDUAL) return WF_EINVAL;
    if (K < 128 || K % 128 || N < 32 || N % 32 || lda < K || lda % 16 || ldo < N || ldo % 8)
        return WF_EINVAL;
    if (row_begin < 0 || row_end <= row_begin || row_end > a_rows) return WF_ERANGE;
    if (!aligned16(a8) || !aligned16(w8) || !aligned16(wscale) || !aligned16(out) ||
        (bias && !aligned16(bias)))
        return WF_EINVAL;
    if (epilogue == WF_EPI_GATED_RESIDUAL &&
        (!gate || !aligned16(gate) || gate_ld % 4 || gate_ld < N || rows_per_group < 1))
        return WF_EINVAL;
    GemmParams gp = base_params(p, row_begin, row_end, N, K, bias);
    gp.wscale = wscale;
    gp.out = out;
    gp.ldo = ldo;
    gp.gate = gate;
    gp.gate_ld = gate_ld;
    gp.rows_per_group = rows_per_group;
    return wf_launch_gemm(epilogue, a8, a_rows, lda, w8, gp, p->num_sms, stream, true) == cudaSuccess
               ? WF_OK
               : WF_ECUDA;
}

int wf_qkv_proj_rope_publish(wf_plan_t p, int layer, const void *x, const void *w_qkv,
                             const void *b_qkv, const void *norm_q, const void *norm_k,
                             void *qk_tmp, cudaStream_t stream) {
    if (!p) return WF_EINVAL;
    if (!p->bound) return WF_EUNBOUND;
    if (p->k < 0) return WF_ENOROUND;
    if (layer < 0 || layer >= p->o.layers) return WF_ERANGE;
    if (!x || !w_qkv || !aligned16(x) || !aligned16(w_qkv) || (b_qkv && !aligned16(b_qkv)))
        return WF_EINVAL;
    if ((norm_q == nullptr) != (norm_k == nullptr)) return WF_EINVAL;
    if (norm_q && (!qk_tmp || !aligned16(norm_q) || !aligned16(norm_k) || !aligned16(qk_tmp)))
        return WF_EINVAL;
    if (p->o.dtype != WF_BF16 && p->o.dtype != WF_FP8) return WF_EUNSUPPORTED;
    const int dim = p->H * p->D;
    if (dim % 64 || p->D % 32) return WF_EUNSUPPORTED;
    return wf_publish_impl(p, layer, x, w_qkv, b_qkv, nullptr, stream, nullptr, norm_q, norm_k,
                           qk_tmp);
}

int wf_dit_workspace_size(wf_plan_t p, int model_dim, int ffn_dim, int channels, int freq_dim,
                          int linear_fp8, size_t *bytes) {
    if (!p || !bytes) return WF_EINVAL;
    if (model_dim != p->H * p->D || ffn_dim < 64 || ffn_dim % 64 || channels < 1 ||
        (4 * channels) % 64 || freq_dim < 2 || freq_dim % 2 || (linear_fp8 != 0 && linear_fp8 != 1))
        return WF_EINVAL;
    // e4m3 linear layers take K in 128-element steps
    if (linear_fp8 && (model_dim % 128 || ffn_dim % 128)) return WF_EINVAL;
    const size_t latent = (size_t)channels * p->g.gt * 4 * p->g.gh * p->g.gw;
    *bytes = wf_dit_workspace_bytes(p->S, p->NC, model_dim, ffn_dim, channels, freq_dim,
                                    p->o.layers, latent, linear_fp8);
    return WF_OK;
}

int wf_dit_bind(wf_plan_t p, const wf_dit_model *m, void *workspace, cudaStream_t stream) {
    if (!p || !m || !workspace) return WF_EINVAL;
    if (!p->bound) return WF_EUNBOUND;
    p->dit_bound = false;
    const int rc = wf_dit_bind_impl(&p->dit, p, m, workspace, 1, stream);
    if (rc != WF_OK) return rc;
    p->dit_bound = true;
    return WF_OK;
}

int wf_dit_round(wf_plan_t p, const float *z_new, const float *eps, float *x0_out,
                 float *chunk_out, cudaStream_t stream) {
    if (!p) return WF_EINVAL;
    if (!p->bound) return WF_EUNBOUND;
    if (!p->dit_bound) return WF_EUNBOUND;
    if (p->k < 0) return WF_ENOROUND;
    const int S = p->S, NC = p->NC, k = p->k;
    bool new_chunk = false;                      // a task at stage 0 reads z_new
    for (int i = 0; i < p->rd.n_tasks; ++i) new_chunk |= p->rd.slot[i] == 0;
    if (new_chunk && (!z_new || ((uintptr_t)z_new & 7))) return WF_EINVAL;
    if (S > 1 && (!eps || !aligned16(eps))) return WF_EINVAL;
    if ((x0_out && !aligned16(x0_out)) || (chunk_out && ((uintptr_t)chunk_out & 3)))
        return WF_EINVAL;
    WfDit &d = p->dit;
    int lo, hi;
    wf_active_range(p, &lo, &hi);
    const size_t latent = d.latent;
    float *lat_cur = d.lat + (size_t)(k & 1) * (S + 1) * latent;
    float *lat_next = d.lat + (size_t)((k + 1) & 1) * (S + 1) * latent;

    WfDitPass a;
    a.d = &d;
    a.g = &p->g;
    a.n_slots = S + 1;
    a.lo = lo;
    a.hi = hi;
    a.r0 = lo * NC;
    a.r1 = (hi + 1) * NC;
    a.rd = &p->rd;
    a.status = static_cast<uint32_t *>(p->scratch);
    a.num_sms = p->num_sms;
    for (int i = 0; i < WF_MAX_ROUND_TASKS; ++i) a.src[i] = nullptr;
    a.src[0] = z_new;
    for (int s = 1; s <= S; ++s) a.src[s] = lat_cur + (size_t)s * latent;
    for (int m = 0; m < WF_MAX_GROUP; ++m) a.z_next[m] = m == 0 ? lat_next : nullptr;
    a.eps = eps;
    a.x0_out = x0_out;
    a.chunk_out = chunk_out;
    a.publish = [&](int l, const void *act, const WfDitLayerDev &w, bool f8) {
        // (q/k RMSNorm: the projection leaves unrotated q | k rows in hmid, free until FFN1)
        return f8 ? wf_publish_impl(p, l, act, w.qkv_w8, w.qkv_b, nullptr, stream, w.qkv_s, w.nq, w.nk,
                                    d.hmid)
                  : wf_publish_impl(p, l, act, w.qkv_w, w.qkv_b, nullptr, stream, nullptr, w.nq, w.nk,
                                    d.hmid);
    };
    a.attend = [&](int l, void *act, bool f8) {
        return wf_attention_impl(p, l, act, WF_ATTN_TC, stream, f8 ? 1 : 0);
    };
    return wf_dit_pass(a, stream);
}

}  // extern "C"
