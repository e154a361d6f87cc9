// Host side of the wavefront-round library: plan, round schedule, page ring,
// argument validation and the C ABI entry points of include/wf.h.
//
// Schedule: "Wave Forcing: Towards Speed-of-Light Streaming Video
// Generation", Sec. 3.1 Eq. 3 (cell (i, s) runs in round k = i + s, store at
// (k - S, S), active set A_k), Eq. 5 (ordered context), App. B.3 Algorithm 1
// (N_chunk + S rounds; the store page is promoted into history after the
// round; the first clean chunk is a persistent anchor whose unrotated key is
// kept) and App. B.8 (fixed page capacity).  The ring is a real FIFO
// allocator: a freed page is reused by the next stored chunk.

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <deque>
#include <new>
#include <vector>

#include "wf_internal.h"

#include "wf_plan_impl.h"

using namespace wfimpl;

namespace {

// bytes of one element of the Q/K/V input and attention output, and of the
// query workspace and page pool
size_t elem_size(int dtype) { return dtype == WF_FP32 ? 4 : 2; }
size_t page_elem_size(int dtype) { return dtype == WF_FP32 ? 4 : (dtype == WF_FP8 ? 1 : 2); }

bool mul_ok(size_t a, size_t b, size_t *out) {
    if (a != 0 && b > SIZE_MAX / a) return false;
    *out = a * b;
    return true;
}

size_t tables_bytes(const WfGeom &g) {
    return (size_t)(g.t_max * g.dt2 + g.gh * g.dh2 + g.gw * g.dw2) * 8;
}

// Live (denoising) tasks of the current round: (chunk, stage), stages
// ascending.  Wavefront: chunk k - s for every s with 0 <= k - s < N
// (Sec. 3.1 Eq. 3).  Sequential: the single task of round k, if it is not
// the chunk's store pass.
int live_tasks(const wf_plan_s *p, int *chunk, int *stage) {
    int n = 0;
    if (p->o.schedule == WF_SCHED_SEQUENTIAL) {
        int i = p->k / (p->S + 1), s = p->k % (p->S + 1);
        if (s < p->S) { chunk[0] = i; stage[0] = s; n = 1; }
        return n;
    }
    for (int s = 0; s < p->S; ++s) {
        int c = p->k - s;
        if (c >= 0 && c < p->o.n_chunks) { chunk[n] = c; stage[n] = s; ++n; }
    }
    return n;
}

// Anchor position of the round (mode ADJACENT): one chunk before the oldest
// non-anchor chunk present in the round, clamped at 0.
int adjacent_anchor_pos(const wf_plan_s *p, int store_chunk, const int *live_chunk, int n_live) {
    int oldest = -1;
    auto take = [&](int c) { if (oldest < 0 || c < oldest) oldest = c; };
    for (auto &h : p->history) take(h.first);
    if (store_chunk >= 0 && !(p->o.use_anchor && store_chunk == 0)) take(store_chunk);
    for (int a = 0; a < n_live; ++a) take(live_chunk[a]);
    return oldest <= 0 ? 0 : oldest - 1;
}

void build_round(wf_plan_s *p, int store_chunk, int store_page) {
    const int S = p->S;
    int lchunk[WF_MAX_STAGES], lstage[WF_MAX_STAGES];
    const int na = live_tasks(p, lchunk, lstage);
    CtxEntry prefix[WF_MAX_CTX];
    int np = 0;
    bool anchor_in = p->o.use_anchor && p->anchor_stored;
    p->anchor_tpos = -1;
    if (anchor_in) {
        p->anchor_tpos = p->o.anchor_mode == WF_ANCHOR_ABSOLUTE
                             ? 0 : adjacent_anchor_pos(p, store_chunk, lchunk, na);
        prefix[np++] = {WF_KIND_ANCHOR, 0, S + 1, 0, p->anchor_tpos};
    }
    // the denoising tasks see the W newest history chunks; the store also the
    // E older ones it alone keeps (label S + 2)
    const int n_hist = (int)p->history.size();
    const int n_shared = p->W >= 0 ? std::min(n_hist, p->W) : n_hist;
    CtxEntry store_prefix[WF_MAX_CTX];
    int nsp = 0;
    for (int e = 0; e < np; ++e) store_prefix[nsp++] = prefix[e];   // the anchor
    int at = 0;
    for (auto &h : p->history) {
        const bool shared = at++ >= n_hist - n_shared;
        if (shared) prefix[np++] = {WF_KIND_HISTORY, h.first, S + 1, h.second, h.first};
        store_prefix[nsp++] = {WF_KIND_HISTORY, h.first, shared ? S + 1 : S + 2, h.second, h.first};
    }
    if (store_chunk >= 0) {
        prefix[np++] = {WF_KIND_STORE, store_chunk, S, store_page, store_chunk};
        store_prefix[nsp++] = prefix[np - 1];
    }

    p->n_tasks = 0;
    for (int a = 0; a < na; ++a) {
        int s = lstage[a];
        HostTask &t = p->tasks[p->n_tasks++];
        t.chunk = lchunk[a];
        t.stage = s;
        t.dest = 1 + p->R + s;
        t.n_ctx = 0;
        for (int e = 0; e < np; ++e) t.ctx[t.n_ctx++] = prefix[e];
        // Eq. 5: live K/V of stages j >= s in increasing j; the RF mask also
        // lists the noisier stages j < s
        for (int b = 0; b < na; ++b) {
            int j = lstage[b];
            if (j >= s || p->o.mask == WF_MASK_RF)
                t.ctx[t.n_ctx++] = {WF_KIND_LIVE, lchunk[b], j, 1 + p->R + j, lchunk[b]};
        }
    }
    if (store_chunk >= 0) {
        HostTask &t = p->tasks[p->n_tasks++];
        t.chunk = store_chunk;
        t.stage = S;
        t.dest = store_page;
        t.n_ctx = 0;
        for (int e = 0; e < nsp; ++e) t.ctx[t.n_ctx++] = store_prefix[e];
    }

    // device view
    WfRoundDev &rd = p->rd;
    std::memset(&rd, 0, sizeof(rd));
    rd.n_tasks = p->n_tasks;
    for (int i = 0; i < WF_MAX_ROUND_TASKS; ++i) rd.task_of_slot[i] = -1;
    for (int i = 0; i < p->n_tasks; ++i) {
        const HostTask &t = p->tasks[i];
        rd.slot[i] = t.stage;
        rd.chunk[i] = t.chunk;
        rd.dest[i] = t.dest;
        rd.n_ctx[i] = t.n_ctx;
        for (int e = 0; e < t.n_ctx; ++e) rd.page[i][e] = (uint8_t)t.ctx[e].page;
        // the store of the anchor chunk also keeps its unrotated key (App. B.3)
        rd.raw_page[i] = (t.stage == S && p->o.use_anchor && t.chunk == 0) ? p->g.raw_anchor_page : -1;
        rd.task_of_slot[t.stage] = i;
        rd.lpt[i] = i;
    }
    std::stable_sort(rd.lpt, rd.lpt + p->n_tasks,
                     [&](int a, int b) { return rd.n_ctx[a] > rd.n_ctx[b]; });
    rd.n_rerot = 0;
}

}  // namespace

namespace {
// The round restricted to the tasks whose slot bit is set in mask (longest
// context first, as in the full round).
WfRoundDev subset_round(const WfRoundDev &rd, unsigned mask) {
    WfRoundDev r = rd;
    r.n_tasks = 0;
    for (int i = 0; i < WF_MAX_ROUND_TASKS; ++i) r.task_of_slot[i] = -1;
    for (int i = 0; i < rd.n_tasks; ++i) {
        if (!((mask >> rd.slot[i]) & 1u)) continue;
        const int o = r.n_tasks++;
        r.slot[o] = rd.slot[i];
        r.chunk[o] = rd.chunk[i];
        r.dest[o] = rd.dest[i];
        r.n_ctx[o] = rd.n_ctx[i];
        r.raw_page[o] = rd.raw_page[i];
        std::memcpy(r.page[o], rd.page[i], sizeof(rd.page[i]));
        r.task_of_slot[r.slot[o]] = o;
        r.lpt[o] = o;
    }
    std::stable_sort(r.lpt, r.lpt + r.n_tasks, [&](int a, int b) { return r.n_ctx[a] > r.n_ctx[b]; });
    r.n_rerot = 0;
    return r;
}
}  // namespace

int wf_attention_impl(wf_plan_s *p, int layer, void *out, int kernel, cudaStream_t stream,
                      int out_e4m3, unsigned slot_mask) {
    const WfRoundDev rd = slot_mask == ~0u ? p->rd : subset_round(p->rd, slot_mask);
    if (rd.n_tasks == 0) return WF_OK;
    bool tc_ok = p->tmaps_ok && wf_attn_tc_supported(p->g, p->o.dtype);
    bool simt_ok = p->D % 32 == 0 && p->D <= 128 && p->o.dtype != WF_FP8 && !out_e4m3;
    if (kernel == WF_ATTN_AUTO) kernel = tc_ok ? WF_ATTN_TC : WF_ATTN_SIMT;
    cudaError_t e;
    if (kernel == WF_ATTN_TC) {
        if (!tc_ok) return WF_EUNSUPPORTED;
        e = wf_launch_attn_tc(p->g, rd, layer, p->tmaps, out, p->scratch, p->num_sms, stream,
                              out_e4m3);
    } else {
        if (!simt_ok) return WF_EUNSUPPORTED;
        e = wf_launch_attn_simt(p->g, rd, layer, p->o.dtype, p->qbuf, p->pool, out, stream);
    }
    return e == cudaSuccess ? WF_OK : WF_ECUDA;
}

// Rebuild the current round's contexts from the round state (after a state
// import): the current round's store is the one recorded for promotion.
void wf_rebuild_round(wf_plan_s *p) {
    if (p->have_prev_store)
        build_round(p, p->prev_store_chunk, p->prev_store_page);
    else
        build_round(p, -1, -1);
}

// Shared by wf_qkv_rope_publish (Q/K/V given) and the projection path
// (x and W_qkv given): one launch publishes every active task; the anchor
// key is re-rotated from its unrotated copy when the window moved.
void wf_anchor_update(const wf_plan_s *p, int layer, bool *rerotate, int *new_rot) {
    *rerotate = false;
    *new_rot = p->anchor_rot[layer];
    bool stores_anchor = false;
    for (int i = 0; i < p->rd.n_tasks; ++i) stores_anchor |= p->rd.raw_page[i] >= 0;
    if (stores_anchor) {
        *new_rot = 0;  // the store of chunk 0 writes the anchor at its own position
    } else if (p->anchor_tpos >= 0 && p->anchor_rot[layer] != p->anchor_tpos) {
        *rerotate = true;
        *new_rot = p->anchor_tpos;
    }
}

int wf_publish_launch(const WfPublishArgs &a, const WfRoundDev &rd, cudaStream_t stream) {
    const WfGeom &g = a.g;
    if (a.x) {
        GemmParams gp;
        std::memset(&gp, 0, sizeof(gp));
        gp.row_begin = a.row_begin;
        gp.row_end = a.row_end;
        gp.N = 3 * g.H * g.D;
        gp.K = g.H * g.D;
        gp.bias = static_cast<const __nv_bfloat16 *>(a.b_qkv);
        gp.status = static_cast<uint32_t *>(a.scratch);
        gp.g = g;
        gp.rd = rd;
        gp.rd.n_rerot = 0;
        gp.layer = a.layer;
        gp.qbuf = static_cast<__nv_bfloat16 *>(a.qbuf);
        gp.pool = static_cast<__nv_bfloat16 *>(a.pool);
        gp.rope = reinterpret_cast<const float2 *>(static_cast<const char *>(a.scratch) +
                                                   WF_SCRATCH_TABLES);
        gp.wscale = a.wscale;
        gp.qk_raw = a.nq ? static_cast<__nv_bfloat16 *>(a.qk_tmp) : nullptr;
        if (wf_launch_gemm(WF_EPI_QKV_PUBLISH, a.x, a.x_rows, gp.K, a.w_qkv, gp, a.num_sms, stream,
                           a.wscale != nullptr) != cudaSuccess)
            return WF_ECUDA;
        if (a.nq) {
            WfQkNormArgs n;
            std::memset(&n, 0, sizeof(n));
            n.row_begin = a.row_begin;
            n.row_end = a.row_end;
            n.layer = a.layer;
            n.raw = gp.qk_raw;
            n.gq = static_cast<const __nv_bfloat16 *>(a.nq);
            n.gk = static_cast<const __nv_bfloat16 *>(a.nk);
            n.qbuf = a.qbuf;
            n.pool = a.pool;
            n.tab = gp.rope;
            if (wf_launch_qk_norm(g, gp.rd, n, stream) != cudaSuccess) return WF_ECUDA;
        }
        if (rd.n_rerot > 0) {
            WfRoundDev rr = rd;
            rr.n_tasks = 0;
            if (wf_launch_publish(g, rr, a.layer, g.dtype, nullptr, a.qbuf, a.pool, a.scratch,
                                  stream) != cudaSuccess)
                return WF_ECUDA;
        }
    } else if (wf_launch_publish(g, rd, a.layer, g.dtype, a.qkv, a.qbuf, a.pool, a.scratch,
                                 stream) != cudaSuccess) {
        return WF_ECUDA;
    }
    return WF_OK;
}

int wf_publish_impl(wf_plan_s *p, int layer, const void *x, const void *w_qkv, const void *b_qkv,
                    const void *qkv, cudaStream_t stream, const float *wscale, const void *nq,
                    const void *nk, void *qk_tmp) {
    bool rerotate;
    int new_rot;
    wf_anchor_update(p, layer, &rerotate, &new_rot);
    WfRoundDev rd = p->rd;
    if (rerotate) {
        rd.n_rerot = 1;
        rd.rerot_anchor[0] = 0;
        rd.rerot_raw[0] = p->g.raw_anchor_page;
        rd.rerot_tpos[0] = p->anchor_tpos;
    }
    int lo, hi;
    wf_active_range(p, &lo, &hi);
    WfPublishArgs a;
    std::memset(&a, 0, sizeof(a));
    a.g = p->g;
    a.layer = layer;
    a.row_begin = lo * p->NC;
    a.row_end = (hi + 1) * p->NC;
    a.x = x;
    a.x_rows = (long long)(p->S + 1) * p->NC;
    a.w_qkv = w_qkv;
    a.b_qkv = b_qkv;
    a.wscale = wscale;
    a.nq = nq;
    a.nk = nk;
    a.qk_tmp = qk_tmp;
    a.qkv = qkv;
    a.qbuf = p->qbuf;
    a.pool = p->pool;
    a.scratch = p->scratch;
    a.num_sms = p->num_sms;
    const int rc = wf_publish_launch(a, rd, stream);
    if (rc != WF_OK) return rc;
    p->anchor_rot[layer] = new_rot;
    p->published[layer] = p->k;
    return WF_OK;
}

extern "C" {

const char *wf_strerror(int code) {
    switch (code) {
        case WF_OK: return "ok";
        case WF_EINVAL: return "invalid argument";
        case WF_ERANGE: return "size or index out of range";
        case WF_ENOMEM: return "buffer too small";
        case WF_ECUDA: return "CUDA call failed";
        case WF_ETIMEOUT: return "device-side bounded wait timed out";
        case WF_EDONE: return "request finished: no more rounds";
        case WF_EUNBOUND: return "plan has no bound device buffers";
        case WF_ENOROUND: return "no current round (call wf_round_step)";
        case WF_EUNSUPPORTED: return "kernel does not support this dtype/shape";
        case WF_EORDER: return "layer not published in the current round";
        default: return "unknown error";
    }
}

void wf_plan_opts_default(wf_plan_opts *o) {
    if (!o) return;
    std::memset(o, 0, sizeof(*o));
    o->n_chunks = 1;
    o->layers = 1;
    o->grid_t = 3;
    o->grid_h = 0;
    o->grid_w = 0;
    o->dtype = WF_BF16;
    o->use_anchor = 1;
    o->anchor_mode = WF_ANCHOR_ADJACENT;
    o->rope_theta = 10000.0;
    o->mask = WF_MASK_WF;
    o->schedule = WF_SCHED_WAVEFRONT;
    o->fp8_qk_scale = 1.0;
    o->fp8_v_scale = 1.0;
}

int wf_plan(int S, int chunk_tokens, int heads, int head_dim, int history_chunks,
            const wf_plan_opts *opts, wf_plan_t *out) {
    if (!out) return WF_EINVAL;
    *out = nullptr;
    wf_plan_opts o;
    if (opts) o = *opts; else wf_plan_opts_default(&o);
    if (S < 1 || S > WF_MAX_STAGES) return WF_ERANGE;
    if (chunk_tokens < 1 || heads < 1 || head_dim < 8 || (head_dim % 8)) return WF_EINVAL;
    if (head_dim > 256) return WF_ERANGE;
    if (history_chunks < -1) return WF_EINVAL;
    if (o.n_chunks < 1 || o.layers < 1) return WF_ERANGE;
    if (o.dtype != WF_FP32 && o.dtype != WF_BF16 && o.dtype != WF_FP8) return WF_EINVAL;
    if (o.dtype == WF_FP8 &&
        (!(o.fp8_qk_scale > 0.0) || !std::isfinite(o.fp8_qk_scale) || !(o.fp8_v_scale > 0.0) ||
         !std::isfinite(o.fp8_v_scale)))
        return WF_EINVAL;
    if (o.anchor_mode != WF_ANCHOR_ADJACENT && o.anchor_mode != WF_ANCHOR_ABSOLUTE) return WF_EINVAL;
    if (o.use_anchor != 0 && o.use_anchor != 1) return WF_EINVAL;
    if (!(o.rope_theta > 1.0) || !std::isfinite(o.rope_theta)) return WF_EINVAL;
    if (o.mask != WF_MASK_WF && o.mask != WF_MASK_RF) return WF_EINVAL;
    if (o.schedule != WF_SCHED_WAVEFRONT && o.schedule != WF_SCHED_SEQUENTIAL) return WF_EINVAL;
    const bool custom_split = o.rope_split[0] || o.rope_split[1] || o.rope_split[2];
    if (custom_split) {
        for (int a = 0; a < 3; ++a)
            if (o.rope_split[a] < 0 || o.rope_split[a] % 2) return WF_EINVAL;
        if (o.rope_split[0] + o.rope_split[1] + o.rope_split[2] != head_dim) return WF_EINVAL;
    }
    if (o.store_extra_history < 0) return WF_EINVAL;
    if (o.store_extra_history > 0 && history_chunks < 0) return WF_EINVAL;
    if (o.grid_t < 1) return WF_EINVAL;
    if (o.grid_h == 0 && o.grid_w == 0) {
        if (chunk_tokens % o.grid_t) return WF_EINVAL;
        o.grid_h = chunk_tokens / o.grid_t;
        o.grid_w = 1;
    }
    if (o.grid_h < 1 || o.grid_w < 1 ||
        (long long)o.grid_t * o.grid_h * o.grid_w != (long long)chunk_tokens)
        return WF_EINVAL;

    const int E = o.store_extra_history;
    // ring: the store's history (W + E) and the live store
    int R = history_chunks >= 0 ? history_chunks + E + 1
                                : std::max(1, o.n_chunks - (o.use_anchor ? 1 : 0));
    // longest context: anchor + history + store + S live chunks (a denoising
    // task), or anchor + W + E history + itself (the store)
    int hist_max = history_chunks >= 0 ? history_chunks : std::max(0, o.n_chunks - 1);
    if (1 + hist_max + 1 + S > WF_MAX_CTX || 1 + hist_max + E + 1 > WF_MAX_CTX) return WF_ERANGE;
    int P = 1 + R + S + 1;
    if (P > 255) return WF_ERANGE;

    wf_plan_s *p = new (std::nothrow) wf_plan_s();
    if (!p) return WF_ENOMEM;
    p->S = S; p->NC = chunk_tokens; p->H = heads; p->D = head_dim; p->W = history_chunks;
    p->o = o; p->R = R; p->P = P;
    WfGeom &g = p->g;
    g.S = S; g.NC = chunk_tokens; g.H = heads; g.D = head_dim; g.L = o.layers;
    g.gt = o.grid_t; g.gh = o.grid_h; g.gw = o.grid_w;
    g.P = P; g.raw_anchor_page = 1 + R + S;
    g.dtype = o.dtype;
    g.qk_scale = (float)o.fp8_qk_scale;
    g.v_scale = (float)o.fp8_v_scale;
    if (custom_split) {
        g.dt2 = o.rope_split[0] / 2; g.dh2 = o.rope_split[1] / 2; g.dw2 = o.rope_split[2] / 2;
    } else {
        const int q6 = head_dim / 6;
        g.dt2 = (head_dim - 4 * q6) / 2; g.dh2 = q6; g.dw2 = q6;
    }
    g.t_max = o.grid_t * o.n_chunks;
    g.rope_t_off = 0;
    g.rope_h_off = g.t_max * g.dt2;
    g.rope_w_off = g.rope_h_off + g.gh * g.dh2;
    for (int i = 1; i <= R; ++i) p->free_pages.push_back(i);
    p->anchor_rot.assign(o.layers, -1);
    p->published.assign(o.layers, -1);
    *out = p;
    return WF_OK;
}

int wf_plan_buffer_sizes(wf_plan_t p, wf_buffer_sizes *out) {
    if (!p || !out) return WF_EINVAL;
    const size_t elems = (size_t)p->NC * p->H * p->D;  // one slot, one of Q/K/V
    size_t tok = elems * elem_size(p->o.dtype);
    size_t ptok = elems * page_elem_size(p->o.dtype);
    size_t slots = (size_t)p->S + 1;
    size_t a, b;
    std::memset(out, 0, sizeof(*out));
    if (!mul_ok(tok, slots * 3, &out->qkv)) return WF_ERANGE;
    out->qbuf = ptok * slots;
    out->out = tok * slots;
    if (!mul_ok(ptok, (size_t)p->P * p->o.layers, &a) || !mul_ok(a, 2, &b)) return WF_ERANGE;
    out->pool = b;
    out->scratch = WF_SCRATCH_TABLES + tables_bytes(p->g);
    out->qk_norm_tmp = (size_t)p->NC * p->H * p->D * 2 * 2 * slots;
    out->n_pages = p->P;
    out->ring_pages = p->R;
    return WF_OK;
}

int wf_bind(wf_plan_t p, void *pool, void *qbuf, void *scratch) {
    if (!p || !pool || !qbuf || !scratch) return WF_EINVAL;
    if (((uintptr_t)pool | (uintptr_t)qbuf | (uintptr_t)scratch) & 255) return WF_EINVAL;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return WF_ECUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return WF_ECUDA;
    // RoPE tables (cos, sin) computed in double and rounded to float
    const WfGeom &g = p->g;
    std::vector<float> tab(tables_bytes(g) / 4);
    auto fill = [&](int off, int rows, int pairs, int part) {
        for (int r = 0; r < rows; ++r)
            for (int m = 0; m < pairs; ++m) {
                double inv = std::pow(p->o.rope_theta, -2.0 * m / part);
                double a = r * inv;
                tab[2 * (off + r * pairs + m)] = (float)std::cos(a);
                tab[2 * (off + r * pairs + m) + 1] = (float)std::sin(a);
            }
    };
    fill(g.rope_t_off, g.t_max, g.dt2, 2 * g.dt2);
    fill(g.rope_h_off, g.gh, g.dh2, 2 * g.dh2);
    fill(g.rope_w_off, g.gw, g.dw2, 2 * g.dw2);
    if (cudaMemset(scratch, 0, WF_SCRATCH_TABLES) != cudaSuccess) return WF_ECUDA;
    if (!tab.empty() &&
        cudaMemcpy((char *)scratch + WF_SCRATCH_TABLES, tab.data(), tab.size() * 4,
                   cudaMemcpyHostToDevice) != cudaSuccess)
        return WF_ECUDA;
    p->tmaps_ok = false;
    if (wf_attn_tc_supported(g, p->o.dtype)) {
        if (wf_encode_tmaps(g, qbuf, pool, &p->tmaps) != cudaSuccess) return WF_ECUDA;
        p->tmaps_ok = true;
    }
    p->pool = pool; p->qbuf = qbuf; p->scratch = scratch;
    p->device = dev; p->num_sms = sms;
    p->bound = true;
    std::fill(p->anchor_rot.begin(), p->anchor_rot.end(), -1);
    return WF_OK;
}

int wf_round_step(wf_plan_t p, wf_round_info *info) {
    if (!p) return WF_EINVAL;
    const int S = p->S, N = p->o.n_chunks;
    const bool seq = p->o.schedule == WF_SCHED_SEQUENTIAL;
    if (p->k + 1 >= (seq ? N * (S + 1) : N + S)) return WF_EDONE;
    p->k += 1;
    // round boundary: the previous store page becomes history (App. B.3)
    if (p->have_prev_store) {
        if (p->o.use_anchor && p->prev_store_chunk == 0) {
            p->anchor_stored = true;
        } else {
            p->history.emplace_back(p->prev_store_chunk, p->prev_store_page);
            while (p->W >= 0 && (int)p->history.size() > p->W + p->o.store_extra_history) {
                p->free_pages.push_back(p->history.front().second);
                p->history.pop_front();
            }
        }
        p->have_prev_store = false;
    }
    int u = seq ? (p->k % (S + 1) == S ? p->k / (S + 1) : -1) : p->k - S;
    int store_chunk = -1, store_page = -1;
    if (u >= 0 && u < N) {
        store_chunk = u;
        if (p->o.use_anchor && u == 0) {
            store_page = 0;
        } else {
            if (p->free_pages.empty()) return WF_ERANGE;  // cannot happen with R = W + 1
            store_page = p->free_pages.front();
            p->free_pages.pop_front();
        }
        p->have_prev_store = true;
        p->prev_store_chunk = store_chunk;
        p->prev_store_page = store_page;
    }
    build_round(p, store_chunk, store_page);
    if (info) {
        std::memset(info, 0, sizeof(*info));
        info->k = p->k;
        info->n_tasks = p->n_tasks;
        info->store_chunk = store_chunk;
        info->anchor_tpos = p->anchor_tpos;
        double fl = 0;
        for (int i = 0; i < p->n_tasks; ++i) {
            info->task_chunk[i] = p->tasks[i].chunk;
            info->task_stage[i] = p->tasks[i].stage;
            info->task_ctx[i] = p->tasks[i].n_ctx;
            fl += 4.0 * p->NC * (double)p->tasks[i].n_ctx * p->NC * p->D * p->H;
        }
        info->attn_flops = fl;
    }
    return WF_OK;
}

int wf_page_table(wf_plan_t p, int32_t *out, int cap, int *n_rows) {
    if (!p || !n_rows || (cap > 0 && !out) || cap < 0) return WF_EINVAL;
    if (p->k < 0) return WF_ENOROUND;
    int n = 0;
    for (int i = 0; i < p->n_tasks; ++i) {
        const HostTask &t = p->tasks[i];
        for (int e = 0; e < t.n_ctx; ++e, ++n) {
            if (n >= cap) continue;
            int32_t *r = out + 10 * n;
            r[0] = t.stage; r[1] = t.chunk; r[2] = t.stage; r[3] = t.dest; r[4] = e;
            r[5] = t.ctx[e].kind; r[6] = t.ctx[e].chunk; r[7] = t.ctx[e].j;
            r[8] = t.ctx[e].page; r[9] = t.ctx[e].tpos;
        }
    }
    *n_rows = n;
    return WF_OK;
}

int wf_qkv_rope_publish(wf_plan_t p, int layer, const void *qkv, cudaStream_t stream) {
    if (!p) return WF_EINVAL;
    if (!p->bound) return WF_EUNBOUND;
    if (p->k < 0) return WF_ENOROUND;
    if (layer < 0 || layer >= p->o.layers) return WF_ERANGE;
    if (!qkv || ((uintptr_t)qkv & 15)) return WF_EINVAL;
    return wf_publish_impl(p, layer, nullptr, nullptr, nullptr, qkv, stream);
}

int wf_round_attention(wf_plan_t p, int layer, void *out, int kernel, cudaStream_t stream) {
    if (!p) return WF_EINVAL;
    if (!p->bound) return WF_EUNBOUND;
    if (p->k < 0) return WF_ENOROUND;
    if (layer < 0 || layer >= p->o.layers) return WF_ERANGE;
    if (!out || ((uintptr_t)out & 15)) return WF_EINVAL;
    if (kernel != WF_ATTN_AUTO && kernel != WF_ATTN_TC && kernel != WF_ATTN_SIMT) return WF_EINVAL;
    if (p->published[layer] != p->k) return WF_EORDER;
    return wf_attention_impl(p, layer, out, kernel, stream);
}

int wf_round_attention_tasks(wf_plan_t p, int layer, void *out, int kernel, unsigned int slot_mask,
                             cudaStream_t stream) {
    if (!p) return WF_EINVAL;
    if (!p->bound) return WF_EUNBOUND;
    if (p->k < 0) return WF_ENOROUND;
    if (layer < 0 || layer >= p->o.layers) return WF_ERANGE;
    if (!out || ((uintptr_t)out & 15)) return WF_EINVAL;
    if (kernel != WF_ATTN_AUTO && kernel != WF_ATTN_TC && kernel != WF_ATTN_SIMT) return WF_EINVAL;
    if (slot_mask >> (p->S + 1)) return WF_EINVAL;
    if (p->published[layer] != p->k) return WF_EORDER;
    return wf_attention_impl(p, layer, out, kernel, stream, 0, slot_mask);
}

int wf_round_attention_noalloc(wf_plan_t p, int layer, void *out, cudaStream_t stream) {
    if (!p) return WF_EINVAL;
    if (!p->bound) return WF_EUNBOUND;
    if (p->k < 0) return WF_ENOROUND;
    if (layer < 0 || layer >= p->o.layers) return WF_ERANGE;
    if (!out || ((uintptr_t)out & 15)) return WF_EINVAL;
    if (p->published[layer] != p->k) return WF_EORDER;
    if (!(p->tmaps_ok && wf_attn_tc_supported(p->g, p->o.dtype))) return WF_EUNSUPPORTED;
    int wf_err = WF_OK;
    cudaError_t e = wf_launch_attn_tc_noalloc(p->g, p->rd, layer, p->tmaps, out, p->scratch,
                                              p->num_sms, stream, &wf_err);
    if (e != cudaSuccess) return WF_ECUDA;
    return wf_err;
}

int wf_sync_status(wf_plan_t p, cudaStream_t stream) {
    if (!p) return WF_EINVAL;
    if (!p->bound) return WF_EUNBOUND;
    uint32_t st[4] = {0, 0, 0, 0};
    if (cudaMemcpyAsync(st, p->scratch, sizeof(st), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return WF_ECUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return WF_ECUDA;
    if (st[0] != 0) {
        uint32_t z[4] = {0, 0, 0, 0};
        if (cudaMemcpy(p->scratch, z, sizeof(z), cudaMemcpyHostToDevice) != cudaSuccess)
            return WF_ECUDA;
        return WF_ETIMEOUT;
    }
    return WF_OK;
}

int wf_selftest_timeout(wf_plan_t p, unsigned int limit_us, cudaStream_t stream) {
    if (!p) return WF_EINVAL;
    if (!p->bound) return WF_EUNBOUND;
    if (limit_us < 1 || limit_us > 2000000) return WF_ERANGE;
    return wf_launch_wait_probe(p->scratch, (uint64_t)limit_us * 1000ull, stream) == cudaSuccess
               ? WF_OK
               : WF_ECUDA;
}

// ---- checkpoint / resume of the host round state ----------------------------
// Layout (int32 words): the shape words (magic, version, S, N_C, H, D, W,
// n_chunks, layers, use_anchor, anchor_mode, mask, schedule,
// store_extra_history, dtype, the three rotary pair counts d_t/2, d_h/2,
// d_w/2, rope_theta as two words of its IEEE bits, the float bits of the two
// e4m3 scales), then k, have_prev_store, prev_store_chunk, prev_store_page,
// anchor_stored, n_history, (chunk, page) x n_history, n_free,
// page x n_free, anchor_rot[layers], published[layers].
namespace {
constexpr int32_t kStateMagic = 0x57465354;  // "WFST"
constexpr int32_t kStateVersion = 3;
constexpr int kShapeWords = 22;  // words that must equal the importing plan's
constexpr int kStateHead = kShapeWords + 6;   // words before the history list

void shape_words(const wf_plan_s *p, int32_t *w) {
    uint64_t theta;
    std::memcpy(&theta, &p->o.rope_theta, 8);
    uint32_t sqk, sv;
    std::memcpy(&sqk, &p->g.qk_scale, 4);
    std::memcpy(&sv, &p->g.v_scale, 4);
    const int32_t v[kShapeWords] = {kStateMagic, kStateVersion, p->S, p->NC, p->H, p->D, p->W,
                                    p->o.n_chunks, p->o.layers, p->o.use_anchor, p->o.anchor_mode,
                                    p->o.mask, p->o.schedule, p->o.store_extra_history, p->o.dtype,
                                    p->g.dt2, p->g.dh2, p->g.dw2, (int32_t)(uint32_t)theta,
                                    (int32_t)(uint32_t)(theta >> 32), (int32_t)sqk, (int32_t)sv};
    std::memcpy(w, v, sizeof(v));
}
}  // namespace

int wf_plan_state_size(wf_plan_t p, size_t *bytes) {
    if (!p || !bytes) return WF_EINVAL;
    *bytes = sizeof(int32_t) * (kStateHead + 2 * p->history.size() + 1 + p->free_pages.size() +
                                2 * (size_t)p->o.layers);
    return WF_OK;
}

int wf_plan_export_state(wf_plan_t p, void *buf, size_t cap, size_t *written) {
    if (!p || !buf || !written) return WF_EINVAL;
    size_t need;
    wf_plan_state_size(p, &need);
    if (cap < need) return WF_ENOMEM;
    std::vector<int32_t> w(kStateHead);
    shape_words(p, w.data());
    const int32_t round[6] = {p->k, p->have_prev_store ? 1 : 0, p->prev_store_chunk,
                              p->prev_store_page, p->anchor_stored ? 1 : 0,
                              (int32_t)p->history.size()};
    std::memcpy(w.data() + kShapeWords, round, sizeof(round));
    for (auto &h : p->history) { w.push_back(h.first); w.push_back(h.second); }
    w.push_back((int32_t)p->free_pages.size());
    for (int f : p->free_pages) w.push_back(f);
    for (int l = 0; l < p->o.layers; ++l) w.push_back(p->anchor_rot[l]);
    for (int l = 0; l < p->o.layers; ++l) w.push_back(p->published[l]);
    std::memcpy(buf, w.data(), w.size() * 4);
    *written = w.size() * 4;
    return WF_OK;
}

int wf_plan_import_state(wf_plan_t p, const void *buf, size_t n) {
    if (!p || !buf || n % 4 || n < kStateHead * 4) return WF_EINVAL;
    const int32_t *w = static_cast<const int32_t *>(buf);
    const size_t nw = n / 4;
    int32_t want[kShapeWords];
    shape_words(p, want);
    for (int i = 0; i < kShapeWords; ++i)
        if (w[i] != want[i]) return WF_EINVAL;
    const int32_t *rw = w + kShapeWords;
    const int S = p->S, N = p->o.n_chunks, R = p->R;
    const bool seq = p->o.schedule == WF_SCHED_SEQUENTIAL;
    const int k = rw[0];
    if (k < -1 || k >= (seq ? N * (S + 1) : N + S)) return WF_EINVAL;
    size_t at = kStateHead;
    const int nh = rw[5];
    if (nh < 0 || nh > R || at + 2 * (size_t)nh + 1 > nw) return WF_EINVAL;
    // every ring page 1..R is in exactly one place: history, the free list,
    // or the previous round's store page awaiting promotion
    std::vector<int> owner(R + 1, 0);
    auto claim = [&](int page) {
        if (page < 1 || page > R || owner[page]) return false;
        owner[page] = 1;
        return true;
    };
    std::deque<std::pair<int, int>> hist;
    for (int i = 0; i < nh; ++i, at += 2) {
        const int c = w[at], pg = w[at + 1];
        if (c < 0 || c >= N || !claim(pg)) return WF_EINVAL;
        if (!hist.empty() && c <= hist.back().first) return WF_EINVAL;   // oldest first
        hist.emplace_back(c, pg);
    }
    const int nf = w[at++];
    if (nf < 0 || nf > R || at + (size_t)nf + 2 * (size_t)p->o.layers != nw) return WF_EINVAL;
    std::deque<int> freep;
    for (int i = 0; i < nf; ++i, ++at) {
        if (!claim(w[at])) return WF_EINVAL;
        freep.push_back(w[at]);
    }
    std::vector<int> rot(p->o.layers), pub(p->o.layers);
    for (int l = 0; l < p->o.layers; ++l) rot[l] = w[at++];
    for (int l = 0; l < p->o.layers; ++l) pub[l] = w[at++];
    const bool have_prev = rw[1] != 0;
    const int prev_chunk = rw[2], prev_page = rw[3];
    if (have_prev) {
        if (prev_chunk < 0 || prev_chunk >= N) return WF_EINVAL;
        // the store of the anchor chunk writes page 0; every other store a ring page
        const bool anchor_store = p->o.use_anchor && prev_chunk == 0;
        if (anchor_store ? prev_page != 0 : !claim(prev_page)) return WF_EINVAL;
    }
    for (int pg = 1; pg <= R; ++pg)
        if (!owner[pg]) return WF_EINVAL;
    p->k = k;
    p->have_prev_store = have_prev;
    p->prev_store_chunk = prev_chunk;
    p->prev_store_page = prev_page;
    p->anchor_stored = rw[4] != 0;
    p->history = hist;
    p->free_pages = freep;
    p->anchor_rot = rot;
    p->published = pub;
    if (k >= 0) wf_rebuild_round(p);
    return WF_OK;
}

void wf_plan_destroy(wf_plan_t p) { delete p; }

}  // extern "C"
