// Several independent requests batched into one round ("Wave Forcing" Sec. 8
// and App. E name serving concurrent streams as the next step).
//
// A group holds up to WF_MAX_GROUP plans of one shape whose device buffers
// are consecutive slices of one allocation.  Each plan keeps its own
// schedule, page ring and anchor (it is advanced with wf_round_step as
// before, may start later than the others and finishes on its own); a group
// launch concatenates the current rounds of the selected plans into one
// round view -- request r's slot s becomes global slot r (S+1) + s, its page
// p global page r P + p -- so their tasks share one QKV projection, one
// publication and one attention launch.  Every kernel addresses the query
// workspace, the output and the page pool through global slots and pages, so
// the batched round computes exactly what each plan's own round computes.

#include <algorithm>
#include <cstring>
#include <new>

#include "wf_plan_impl.h"

struct wf_group_s {
    int n = 0;
    wf_plan_s *plans[WF_MAX_GROUP] = {};
    bool tmaps_ok = false;
    WfTmaps tmaps;   // over the n consecutive query workspaces and pools
    // DiT model of the group (wf_group_dit_bind): activations for n (S+1)
    // slots; member r's latent slot inputs at lat + r * 2 (S+1) latent,
    // double-buffered by that member's own round parity
    bool dit_bound = false;
    WfDit dit{};
    ~wf_group_s() { delete[] dit.layers; }
};

namespace {

bool aligned16(const void *q) { return ((uintptr_t)q & 15) == 0; }

bool same_shape(const wf_plan_s *a, const wf_plan_s *b) {
    return std::memcmp(&a->g, &b->g, sizeof(WfGeom)) == 0 && a->o.rope_theta == b->o.rope_theta;
}

// The round view of the selected plans (bit r of mask: plan r).  Returns a
// WF_* code: every selected plan must be in a round.
int group_round(const wf_group_s *gr, unsigned mask, WfRoundDev *rd) {
    std::memset(rd, 0, sizeof(*rd));
    for (int i = 0; i < WF_MAX_ROUND_TASKS; ++i) rd->task_of_slot[i] = -1;
    const WfGeom &g = gr->plans[0]->g;
    const int slots = g.S + 1;
    for (int r = 0; r < gr->n; ++r) {
        if (!((mask >> r) & 1u)) continue;
        const wf_plan_s *p = gr->plans[r];
        if (p->k < 0) return WF_ENOROUND;
        const WfRoundDev &pr = p->rd;
        const int off = r * g.P;
        for (int i = 0; i < pr.n_tasks; ++i) {
            const int o = rd->n_tasks++;
            rd->slot[o] = r * slots + pr.slot[i];
            rd->chunk[o] = pr.chunk[i];
            rd->dest[o] = off + pr.dest[i];
            rd->n_ctx[o] = pr.n_ctx[i];
            rd->raw_page[o] = pr.raw_page[i] >= 0 ? off + pr.raw_page[i] : -1;
            for (int e = 0; e < pr.n_ctx[i]; ++e) rd->page[o][e] = (uint8_t)(off + pr.page[i][e]);
            rd->task_of_slot[rd->slot[o]] = o;
            rd->lpt[o] = o;
        }
    }
    std::stable_sort(rd->lpt, rd->lpt + rd->n_tasks,
                     [&](int a, int b) { return rd->n_ctx[a] > rd->n_ctx[b]; });
    return WF_OK;
}

int check_mask(const wf_group_s *gr, unsigned mask) {
    if (mask == 0 || (gr->n < 32 && (mask >> gr->n))) return WF_EINVAL;
    return WF_OK;
}

// Publication of the selected plans' current rounds (x: projection input,
// else the given qkv), with each plan's anchor re-rotation.
int group_publish(wf_group_s *gr, unsigned mask, int layer, const void *x, const void *w_qkv,
                  const void *b_qkv, const void *nq, const void *nk, void *qk_tmp, const void *qkv,
                  cudaStream_t stream, const float *wscale = nullptr) {
    wf_plan_s *p0 = gr->plans[0];
    if (layer < 0 || layer >= p0->o.layers) return WF_ERANGE;
    WfRoundDev rd;
    int rc = group_round(gr, mask, &rd);
    if (rc != WF_OK) return rc;
    bool rerot[WF_MAX_GROUP] = {};
    int new_rot[WF_MAX_GROUP] = {};
    int lo = WF_MAX_ROUND_TASKS, hi = -1;
    for (int i = 0; i < rd.n_tasks; ++i) {
        lo = std::min(lo, rd.slot[i]);
        hi = std::max(hi, rd.slot[i]);
    }
    for (int r = 0; r < gr->n; ++r) {
        if (!((mask >> r) & 1u)) continue;
        const wf_plan_s *p = gr->plans[r];
        wf_anchor_update(p, layer, &rerot[r], &new_rot[r]);
        if (rerot[r]) {
            const int e = rd.n_rerot++;
            rd.rerot_anchor[e] = r * p0->g.P;
            rd.rerot_raw[e] = r * p0->g.P + p0->g.raw_anchor_page;
            rd.rerot_tpos[e] = p->anchor_tpos;
        }
    }
    if (rd.n_tasks > 0 || rd.n_rerot > 0) {
        WfPublishArgs a;
        std::memset(&a, 0, sizeof(a));
        a.g = p0->g;
        a.layer = layer;
        a.row_begin = (hi >= 0 ? lo : 0) * p0->NC;
        a.row_end = (hi >= 0 ? hi + 1 : 0) * p0->NC;
        a.x = rd.n_tasks > 0 ? x : nullptr;
        a.x_rows = (long long)gr->n * (p0->S + 1) * p0->NC;
        a.w_qkv = w_qkv;
        a.b_qkv = b_qkv;
        a.wscale = wscale;
        a.nq = nq;
        a.nk = nk;
        a.qk_tmp = qk_tmp;
        a.qkv = qkv;
        a.qbuf = p0->qbuf;
        a.pool = p0->pool;
        a.scratch = p0->scratch;
        a.num_sms = p0->num_sms;
        if (x && rd.n_tasks == 0) {
            // only re-rotations are due: the given-Q/K/V kernel with no tasks does them
            a.qkv = nullptr;
        }
        rc = wf_publish_launch(a, rd, stream);
        if (rc != WF_OK) return rc;
    }
    for (int r = 0; r < gr->n; ++r) {
        if (!((mask >> r) & 1u)) continue;
        gr->plans[r]->anchor_rot[layer] = new_rot[r];
        gr->plans[r]->published[layer] = gr->plans[r]->k;
    }
    return WF_OK;
}

// Round attention of the selected members' current rounds, one launch
// (out_e4m3: O as e4m3 bytes, tensor-core kernel only).
int group_attention(wf_group_s *gr, unsigned mask, int layer, void *out, int kernel,
                    cudaStream_t stream, int out_e4m3) {
    wf_plan_s *p0 = gr->plans[0];
    for (int r = 0; r < gr->n; ++r) {
        if (!((mask >> r) & 1u)) continue;
        const wf_plan_s *p = gr->plans[r];
        if (p->k < 0) return WF_ENOROUND;
        if (p->published[layer] != p->k) return WF_EORDER;
    }
    WfRoundDev rd;
    int rc = group_round(gr, mask, &rd);
    if (rc != WF_OK) return rc;
    if (rd.n_tasks == 0) return WF_OK;
    const bool tc_ok = gr->tmaps_ok && wf_attn_tc_supported(p0->g, p0->o.dtype);
    const bool simt_ok = p0->D % 32 == 0 && p0->D <= 128 && p0->o.dtype != WF_FP8 && !out_e4m3;
    if (kernel == WF_ATTN_AUTO) kernel = tc_ok ? WF_ATTN_TC : WF_ATTN_SIMT;
    cudaError_t e;
    if (kernel == WF_ATTN_TC) {
        if (!tc_ok) return WF_EUNSUPPORTED;
        e = wf_launch_attn_tc(p0->g, rd, layer, gr->tmaps, out, p0->scratch, p0->num_sms, stream,
                              out_e4m3);
    } else {
        if (!simt_ok) return WF_EUNSUPPORTED;
        e = wf_launch_attn_simt(p0->g, rd, layer, p0->o.dtype, p0->qbuf, p0->pool, out, stream);
    }
    return e == cudaSuccess ? WF_OK : WF_ECUDA;
}

}  // namespace

extern "C" {

int wf_group_create(const wf_plan_t *plans, int n, wf_group_t *out) {
    if (!out) return WF_EINVAL;
    *out = nullptr;
    if (!plans) return WF_EINVAL;
    if (n < 1 || n > WF_MAX_GROUP) return WF_ERANGE;
    for (int r = 0; r < n; ++r) {
        if (!plans[r]) return WF_EINVAL;
        for (int q = 0; q < r; ++q)
            if (plans[q] == plans[r]) return WF_EINVAL;
    }
    for (int r = 0; r < n; ++r)
        if (!plans[r]->bound) return WF_EUNBOUND;
    const wf_plan_s *p0 = plans[0];
    if (n * p0->P > 256) return WF_ERANGE;                 // global page ids are one byte
    wf_buffer_sizes sz;
    if (wf_plan_buffer_sizes(const_cast<wf_plan_s *>(p0), &sz) != WF_OK) return WF_ERANGE;
    for (int r = 1; r < n; ++r) {
        const wf_plan_s *p = plans[r];
        if (!same_shape(p0, p) || p->device != p0->device) return WF_EINVAL;
        if (static_cast<char *>(p->pool) != static_cast<char *>(p0->pool) + r * sz.pool ||
            static_cast<char *>(p->qbuf) != static_cast<char *>(p0->qbuf) + r * sz.qbuf)
            return WF_EINVAL;
    }
    wf_group_s *gr = new (std::nothrow) wf_group_s();
    if (!gr) return WF_ENOMEM;
    gr->n = n;
    for (int r = 0; r < n; ++r) gr->plans[r] = plans[r];
    if (p0->tmaps_ok) {
        if (wf_encode_tmaps(p0->g, p0->qbuf, p0->pool, &gr->tmaps, n) != cudaSuccess) {
            delete gr;
            return WF_ECUDA;
        }
        gr->tmaps_ok = true;
    }
    *out = gr;
    return WF_OK;
}

int wf_group_publish(wf_group_t gr, unsigned int plan_mask, int layer, const void *qkv,
                     cudaStream_t stream) {
    if (!gr) return WF_EINVAL;
    int rc = check_mask(gr, plan_mask);
    if (rc != WF_OK) return rc;
    if (!qkv || !aligned16(qkv)) return WF_EINVAL;
    return group_publish(gr, plan_mask, layer, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                         qkv, stream);
}

int wf_group_proj_publish(wf_group_t gr, unsigned int plan_mask, int layer, const void *x,
                          const void *w_qkv, const void *b_qkv, const void *norm_q,
                          const void *norm_k, void *qk_tmp, cudaStream_t stream) {
    if (!gr) return WF_EINVAL;
    int rc = check_mask(gr, plan_mask);
    if (rc != WF_OK) return rc;
    if (!x || !w_qkv || !aligned16(x) || !aligned16(w_qkv) || (b_qkv && !aligned16(b_qkv)))
        return WF_EINVAL;
    if ((norm_q == nullptr) != (norm_k == nullptr)) return WF_EINVAL;
    if (norm_q && (!qk_tmp || !aligned16(norm_q) || !aligned16(norm_k) || !aligned16(qk_tmp)))
        return WF_EINVAL;
    const wf_plan_s *p0 = gr->plans[0];
    if (p0->o.dtype != WF_BF16 && p0->o.dtype != WF_FP8) return WF_EUNSUPPORTED;
    if ((p0->H * p0->D) % 64 || p0->D % 32) return WF_EUNSUPPORTED;
    return group_publish(gr, plan_mask, layer, x, w_qkv, b_qkv, norm_q, norm_k, qk_tmp, nullptr,
                         stream);
}

int wf_group_attention(wf_group_t gr, unsigned int plan_mask, int layer, void *out, int kernel,
                       cudaStream_t stream) {
    if (!gr) return WF_EINVAL;
    int rc = check_mask(gr, plan_mask);
    if (rc != WF_OK) return rc;
    if (layer < 0 || layer >= gr->plans[0]->o.layers) return WF_ERANGE;
    if (!out || !aligned16(out)) return WF_EINVAL;
    if (kernel != WF_ATTN_AUTO && kernel != WF_ATTN_TC && kernel != WF_ATTN_SIMT) return WF_EINVAL;
    return group_attention(gr, plan_mask, layer, out, kernel, stream, 0);
}

int wf_group_dit_workspace_size(wf_group_t gr, int model_dim, int ffn_dim, int channels,
                                int freq_dim, int linear_fp8, size_t *bytes) {
    if (!gr || !bytes) return WF_EINVAL;
    wf_plan_s *p0 = gr->plans[0];
    size_t one;
    const int rc = wf_dit_workspace_size(p0, model_dim, ffn_dim, channels, freq_dim, linear_fp8, &one);
    if (rc != WF_OK) return rc;
    const size_t latent = (size_t)channels * p0->g.gt * 4 * p0->g.gh * p0->g.gw;
    *bytes = wf_dit_workspace_bytes(gr->n * (p0->S + 1) - 1, p0->NC, model_dim, ffn_dim, channels,
                                    freq_dim, p0->o.layers, latent, linear_fp8);
    return WF_OK;
}

int wf_group_dit_bind(wf_group_t gr, const wf_dit_model *m, void *workspace, cudaStream_t stream) {
    if (!gr || !m || !workspace) return WF_EINVAL;
    gr->dit_bound = false;
    const int rc = wf_dit_bind_impl(&gr->dit, gr->plans[0], m, workspace, gr->n, stream);
    if (rc != WF_OK) return rc;
    gr->dit_bound = true;
    return WF_OK;
}

int wf_group_dit_round(wf_group_t gr, unsigned int plan_mask, const float *z_new, const float *eps,
                       float *x0_out, float *chunk_out, cudaStream_t stream) {
    if (!gr) return WF_EINVAL;
    int rc = check_mask(gr, plan_mask);
    if (rc != WF_OK) return rc;
    if (!gr->dit_bound) return WF_EUNBOUND;
    wf_plan_s *p0 = gr->plans[0];
    const int S = p0->S, NC = p0->NC, slots = S + 1;
    WfRoundDev rd;
    rc = group_round(gr, plan_mask, &rd);
    if (rc != WF_OK) return rc;
    if (rd.n_tasks == 0) return WF_OK;
    bool new_chunk = false;                      // a task at stage 0 reads z_new
    int lo = WF_MAX_ROUND_TASKS, hi = -1;
    for (int i = 0; i < rd.n_tasks; ++i) {
        new_chunk |= rd.slot[i] % slots == 0;
        lo = std::min(lo, rd.slot[i]);
        hi = std::max(hi, rd.slot[i]);
    }
    if (new_chunk && (!z_new || ((uintptr_t)z_new & 7))) return WF_EINVAL;
    if (S > 1 && (!eps || !aligned16(eps))) return WF_EINVAL;
    if ((x0_out && !aligned16(x0_out)) || (chunk_out && ((uintptr_t)chunk_out & 3)))
        return WF_EINVAL;
    WfDit &d = gr->dit;
    const size_t latent = d.latent;

    WfDitPass a;
    a.d = &d;
    a.g = &p0->g;
    a.n_slots = gr->n * slots;
    a.lo = lo;
    a.hi = hi;
    a.r0 = lo * NC;
    a.r1 = (hi + 1) * NC;
    a.rd = &rd;
    a.status = static_cast<uint32_t *>(p0->scratch);
    a.num_sms = p0->num_sms;
    for (int i = 0; i < WF_MAX_ROUND_TASKS; ++i) a.src[i] = nullptr;
    for (int r = 0; r < WF_MAX_GROUP; ++r) a.z_next[r] = nullptr;
    for (int r = 0; r < gr->n; ++r) {
        if (!((plan_mask >> r) & 1u)) continue;
        const int k = gr->plans[r]->k;
        float *own = d.lat + (size_t)r * 2 * slots * latent;
        const float *cur = own + (size_t)(k & 1) * slots * latent;
        a.z_next[r] = own + (size_t)((k + 1) & 1) * slots * latent;
        for (int s = 0; s <= S; ++s) {
            const int gs = r * slots + s;
            if (rd.task_of_slot[gs] < 0) continue;
            a.src[gs] = s == 0 ? z_new + (size_t)r * latent : cur + (size_t)s * latent;
        }
    }
    a.eps = eps;
    a.x0_out = x0_out;
    a.chunk_out = chunk_out;
    a.publish = [&](int l, const void *act, const WfDitLayerDev &w, bool f8) {
        // (q/k RMSNorm: the projection leaves unrotated q | k rows in hmid, free until FFN1)
        return group_publish(gr, plan_mask, l, act, f8 ? (const void *)w.qkv_w8 : w.qkv_w, w.qkv_b,
                             w.nq, w.nk, d.hmid, nullptr, stream, f8 ? w.qkv_s : nullptr);
    };
    a.attend = [&](int l, void *act, bool f8) {
        return group_attention(gr, plan_mask, l, act, WF_ATTN_TC, stream, f8 ? 1 : 0);
    };
    return wf_dit_pass(a, stream);
}

void wf_group_destroy(wf_group_t gr) { delete gr; }

}  // extern "C"
