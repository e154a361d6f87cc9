// The plan object behind the opaque wf_plan_t handle (host state of one
// request), shared by the host files of the library.  Not part of the C ABI.
#pragma once

#include <functional>
#include <deque>
#include <utility>
#include <vector>

#include "wf_internal.h"

namespace wfimpl {

struct CtxEntry {
    int kind, chunk, j, page, tpos;
};

struct HostTask {
    int chunk, stage, dest;
    int n_ctx;
    CtxEntry ctx[WF_MAX_CTX];
};

}  // namespace wfimpl

struct wf_plan_s {
    int S, NC, H, D, W;
    wf_plan_opts o;
    int R, P;                // ring pages, total pages
    WfGeom g;

    // round state
    int k = -1;
    bool have_prev_store = false;
    int prev_store_chunk = -1, prev_store_page = -1;
    bool anchor_stored = false;               // chunk 0 clean and on page 0
    std::deque<std::pair<int, int>> history;  // (chunk, page), oldest first
    std::deque<int> free_pages;
    int n_tasks = 0;
    wfimpl::HostTask tasks[WF_MAX_TASKS];
    int anchor_tpos = -1;
    WfRoundDev rd{};
    std::vector<int> anchor_rot;              // per layer: tpos the anchor page holds, -1 none
    std::vector<int> published;               // per layer: round whose publish ran

    // binding
    bool bound = false;
    void *pool = nullptr, *qbuf = nullptr, *scratch = nullptr;
    int device = 0, num_sms = 0;
    bool tmaps_ok = false;
    WfTmaps tmaps;

    // DiT model (wf_dit_bind)
    bool dit_bound = false;
    WfDit dit{};
    ~wf_plan_s() { delete[] dit.layers; }
};

// Active slots of the current round form the contiguous range [lo, hi]:
// wavefront stage s is active iff k - N_chunk < s <= k, the store likewise
// with s = S; a sequential round has one slot.
inline void wf_active_range(const wf_plan_s *p, int *lo, int *hi) {
    int a = WF_MAX_TASKS, b = -1;
    for (int i = 0; i < p->rd.n_tasks; ++i) {
        if (p->rd.slot[i] < a) a = p->rd.slot[i];
        if (p->rd.slot[i] > b) b = p->rd.slot[i];
    }
    *lo = a;
    *hi = b;
}

// Rebuild the current round's task table from the round state.
void wf_rebuild_round(wf_plan_s *p);

// Launch the QKV publication for `layer` of the current round: either the
// projection GEMM (x != nullptr) or the given Q/K/V; the anchor re-rotation
// when the window moved.  Returns a WF_* code.
// Anchor bookkeeping of a plan's publication of `layer` in its current
// round: whether its anchor page must be re-rotated from the unrotated copy
// and the position the page holds afterwards (App. B.3).
void wf_anchor_update(const wf_plan_s *p, int layer, bool *rerotate, int *new_rot);

// The launches of one publication over a round view (a plan's or a
// group's): the projection GEMM (x set; with gains, then the q/k RMSNorm
// kernel) or the given-Q/K/V kernel, and rd's anchor re-rotations.
struct WfPublishArgs {
    WfGeom g;
    int layer;
    int row_begin, row_end;      // projection rows (slots without a task are skipped)
    const void *x;               // [x_rows][dim] or null
    long long x_rows;
    const void *w_qkv, *b_qkv;
    const float *wscale;         // e4m3 weights: per output channel scale, else null
    const void *nq, *nk;         // q / k RMSNorm gains, or null
    void *qk_tmp;
    const void *qkv;             // given Q/K/V when x is null
    void *qbuf, *pool, *scratch;
    int num_sms;
};
int wf_publish_launch(const WfPublishArgs &a, const WfRoundDev &rd, cudaStream_t stream);

// With gains nq / nk (projection path only) the projection leaves unrotated
// q | k rows in qk_tmp and the q/k RMSNorm kernel publishes them.
int wf_publish_impl(wf_plan_s *p, int layer, const void *x, const void *w_qkv, const void *b_qkv,
                    const void *qkv, cudaStream_t stream, const float *wscale = nullptr,
                    const void *nq = nullptr, const void *nk = nullptr, void *qk_tmp = nullptr);

// Round attention of `layer` after the argument checks of wf_round_attention;
// out_e4m3 writes O as e4m3 bytes (tensor-core kernel); slot_mask selects the
// tasks by slot (all by default).  Returns a WF_* code.
int wf_attention_impl(wf_plan_s *p, int layer, void *out, int kernel, cudaStream_t stream,
                      int out_e4m3 = 0, unsigned slot_mask = ~0u);

// ---- one DiT forward over slot-indexed buffers (dit.cpp) ---------------------
// Binding of the DiT model's pointers and tables for n_req requests of p's
// shape (a plan: n_req = 1; a group: its member count), activations carved
// for n_req (S+1) slots of `workspace`.  Returns a WF_* code.
int wf_dit_bind_impl(WfDit *d, const wf_plan_s *p, const wf_dit_model *m, void *workspace,
                     int n_req, cudaStream_t stream);

// What one DiT forward needs besides the model: the round view (global
// slots; request m owns slots m (S+1) .. m (S+1) + S), the rows it covers,
// the per-slot inputs, the per-request outputs and the layer steps that
// differ between a plan and a group (publication and attention).
struct WfDitPass {
    WfDit *d;
    const WfGeom *g;
    int n_slots;                              // slot rows of the activation buffers
    int lo, hi;                               // first / last slot with a task
    int r0, r1;                               // rows [lo NC, (hi+1) NC)
    const WfRoundDev *rd;
    uint32_t *status;
    int num_sms;
    const float *src[WF_MAX_ROUND_TASKS];     // per slot: input latent (null: no task)
    float *z_next[WF_MAX_GROUP];              // per request: next round's slot inputs
    const float *eps;
    float *x0_out, *chunk_out;
    std::function<int(int layer, const void *act, const WfDitLayerDev &w, bool f8)> publish;
    std::function<int(int layer, void *act, bool f8)> attend;
};
int wf_dit_pass(const WfDitPass &a, cudaStream_t stream);

