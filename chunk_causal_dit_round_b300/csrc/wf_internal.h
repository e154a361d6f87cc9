// Internal declarations shared by the host plan (wf_plan.cpp) and the CUDA
// kernels.  Not part of the public C ABI (include/wf.h).
#pragma once

#include <atomic>
#include <cstdint>
#include <cstddef>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/wf.h"

// Runs fn() -- a per-device CUDA setting such as a kernel's shared-memory
// opt-in -- once per device for the calling process; done holds one bit per
// device.  Repeating fn() is harmless, so concurrent first calls need no lock.
template <typename F>
inline cudaError_t wf_once_per_device(std::atomic<unsigned long long> &done, F &&fn) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = dev >= 0 && dev < 64 ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = fn();
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
    return e;
}

#define WF_MAX_TASKS (WF_MAX_STAGES + 1)
// A round view may batch the tasks of up to WF_MAX_GROUP requests (a
// wf_group): request r's slot s is global slot r (S+1) + s and its page p
// global page r P + p.
#define WF_MAX_GROUP WF_MAX_GROUP_PLANS
#define WF_MAX_ROUND_TASKS (WF_MAX_GROUP * WF_MAX_TASKS)

// Geometry of a plan, passed by value to every kernel.
struct WfGeom {
    int S, NC, H, D, L;        // stages, chunk tokens, heads, head dim, layers
    int gt, gh, gw;            // latent frames per chunk, patch grid
    int P;                     // pages in the pool
    int raw_anchor_page;       // page keeping the anchor's unrotated key
    int dt2, dh2, dw2;         // rotary pairs of the t / h / w parts
    int t_max;                 // rows of the temporal table (absolute frames)
    int rope_t_off, rope_h_off, rope_w_off;  // float2 offsets of the tables in scratch
    int dtype;                 // WF_FP32 / WF_BF16 / WF_FP8 (storage of Q and the K/V pages)
    float qk_scale, v_scale;   // e4m3 storage: Q, K (resp. V) multiplied by these before rounding
};

// One round as the kernels see it (host-built in wf_round_step; a group
// concatenates the rounds of its requests with global slots and pages).
struct WfRoundDev {
    int n_tasks;
    int slot[WF_MAX_ROUND_TASKS];        // q/out slot (request r, stage s: r (S+1) + s; S = store)
    int chunk[WF_MAX_ROUND_TASKS];       // chunk index (temporal position of its own tokens)
    int dest[WF_MAX_ROUND_TASKS];        // page its K/V are published to
    int n_ctx[WF_MAX_ROUND_TASKS];       // chunks in its ordered context
    int lpt[WF_MAX_ROUND_TASKS];         // task indices, longest context first
    int raw_page[WF_MAX_ROUND_TASKS];    // page that also keeps its unrotated K (the store of
                                         // an anchor chunk), or -1
    int task_of_slot[WF_MAX_ROUND_TASKS];  // slot -> task index, -1 for an inactive slot
    uint8_t page[WF_MAX_ROUND_TASKS][WF_MAX_CTX];  // ordered context page ids (Eq. 5)
    // anchor re-rotations a publish launch performs: the anchor page, the
    // page of its unrotated key, the temporal chunk position to rotate to
    int n_rerot;
    int rerot_anchor[WF_MAX_GROUP], rerot_raw[WF_MAX_GROUP], rerot_tpos[WF_MAX_GROUP];
};

// Scratch layout (bytes): control words first, then the RoPE tables.
#define WF_SCRATCH_STATUS   0   // uint32: 0 ok, else a WF_DEV_* code
#define WF_SCRATCH_WORK     4   // uint32: attention work counter
#define WF_SCRATCH_DONE     8   // uint32: attention finished-CTA counter
#define WF_SCRATCH_WHERE    12  // uint32: where a bounded wait gave up
#define WF_SCRATCH_TABLES   256

#define WF_DEV_TIMEOUT 1

// ---- kernel launchers (defined in the .cu files) ------------------------
cudaError_t wf_launch_publish(const WfGeom &g, const WfRoundDev &rd, int layer, int dtype,
                              const void *qkv, void *qbuf, void *pool, const void *scratch,
                              cudaStream_t stream);

// q/k RMSNorm over the full width, RoPE and paged publication of rows
// [row_begin, row_end) of raw = [rows][2 H D] unrotated bf16 q | k (the
// QKV projection's epilogue output when the block normalises q and k).
struct WfQkNormArgs {
    int row_begin, row_end, layer;    // rows of inactive slots in the range are skipped
    const __nv_bfloat16 *raw;
    const __nv_bfloat16 *gq, *gk;     // [H D] gains of q and k
    void *qbuf, *pool;
    const float2 *tab;                // RoPE tables in scratch
};
cudaError_t wf_launch_qk_norm(const WfGeom &g, const WfRoundDev &rd, const WfQkNormArgs &a,
                              cudaStream_t stream);

cudaError_t wf_launch_attn_simt(const WfGeom &g, const WfRoundDev &rd, int layer, int dtype,
                                const void *qbuf, const void *pool, void *out, cudaStream_t stream);

struct WfTmaps {
    CUtensorMap q;     // qbuf  [S+1][H][NC][128] bf16, box 64 x 128 x 1, 128B swizzle
    CUtensorMap kv;    // pool  [P*L*2*H][NC][128] bf16, same box
};

bool wf_attn_tc_supported(const WfGeom &g, int dtype);
// Tensor maps over n_req consecutive requests' query workspaces and pools
// (1 for a single plan).
cudaError_t wf_encode_tmaps(const WfGeom &g, void *qbuf, void *pool, WfTmaps *out, int n_req = 1);
cudaError_t wf_launch_attn_tc(const WfGeom &g, const WfRoundDev &rd, int layer,
                              const WfTmaps &maps, void *out, void *scratch, int num_sms,
                              cudaStream_t stream, int out_e4m3 = 0);

// Variant of wf_launch_attn_tc whose scheduler counters live in a static
// device block inside the library; status_scratch receives the status and
// wait-site words (the plan's scratch); see wf_round_attention_noalloc.
cudaError_t wf_launch_attn_tc_noalloc(const WfGeom &g, const WfRoundDev &rd, int layer,
                                      const WfTmaps &maps, void *out, void *status_scratch,
                                      int num_sms, cudaStream_t stream, int *wf_err);

// ---- linear layers (gemm_tc.cu) -------------------------------------------
// Internal epilogue of the QKV projection (RoPE + paged publication) and of
// the head (unpatchify + stage transition); the public ones are WF_EPI_*.
#define WF_EPI_QKV_PUBLISH 100
#define WF_EPI_HEAD        101
#define WF_EPI_GELU_E4M3   102   // GELU, e4m3 bytes out (the input of an e4m3 FFN2)

struct GemmParams {
    int row_begin, row_end;      // rows of A / out processed (absolute)
    int N, K;
    int tiles_m, tiles_n;        // filled by the launcher
    const __nv_bfloat16 *bias;   // [N] or null
    const float *wscale;         // e4m3 operands: per output column (weight row) scale
    void *out;                   // epilogue destination
    int ldo;                     // its row pitch, elements
    const float *gate;           // gated residual: gate[group][col]
    int gate_ld, rows_per_group;
    uint32_t *status;            // plan scratch control words (timeouts), or null
    int staged;                  // set by the launcher: row-major output through TMA stores
    int staged_v;                // set by the launcher: V pages through TMA stores
    // QKV publication
    WfGeom g;
    WfRoundDev rd;               // rows of slots without a task are skipped
    int layer;
    __nv_bfloat16 *qbuf, *pool;
    const float2 *rope;
    __nv_bfloat16 *qk_raw;       // non-null: Q/K columns stored unrotated here ([rows][2 dim]) for
                                 // the q/k RMSNorm kernel, which rotates and publishes them
    // head + stage transition
    int channels;
    float sigma_next[WF_MAX_TASKS];  // per stage slot: warped sigma of the next stage (0: identity)
    // request m of a group owns global slots m (S+1) .. m (S+1) + S (m = 0 for one plan)
    const float *eps;            // [n][S][latent] transition draws, or null
    float *z_next[WF_MAX_GROUP]; // per request: [S+1][latent] next round's slot inputs
    float *x0_out;               // [n][S+1][latent] predictions, or null
    float *chunk_out;            // [n][latent] emitted clean chunks, or null
};

int wf_gemm_bn_for(int epi);
cudaError_t wf_launch_gemm(int epi, const void *a, long long a_rows, int lda, const void *w,
                           GemmParams p, int num_sms, cudaStream_t stream, bool f8 = false);
// Per-row e4m3 quantisation of a bf16 weight [N][K]: scale[n] = max|w_n| / 448
// (1 for an all-zero row), w8[n][k] = e4m3(w[n][k] / scale[n]).
cudaError_t wf_launch_quant_rows(const void *w, int N, int K, void *w8, float *scale,
                                 cudaStream_t stream);

// ---- DiT block pieces (dit_ops.cu) ------------------------------------------
struct WfDitLayerDev {
    const __nv_bfloat16 *qkv_w, *qkv_b, *o_w, *o_b, *f1_w, *f1_b, *f2_w, *f2_b, *mod;
    const __nv_bfloat16 *nq, *nk;   // q / k RMSNorm gains [dim]
    // e4m3 weights and per-output-channel scales (linear_fp8), in the workspace
    uint8_t *qkv_w8, *o_w8, *f1_w8, *f2_w8;
    float *qkv_s, *o_s, *f1_s, *f2_s;
};

struct WfDit {
    int dim, ffn, C, freq, L;
    int linear_fp8;              // the block's linear layers in e4m3
    uint8_t *xa8;                // [(S+1) N_C][dim] e4m3 LN output / attention output
    uint8_t *h8;                 // [(S+1) N_C][ffn] e4m3 FFN hidden
    double shift, context_noise, nu[WF_MAX_STAGES + 1];
    const __nv_bfloat16 *patch_w, *patch_b, *t1_w, *t1_b, *t2_w, *t2_b, *tp_w, *tp_b, *head_w,
        *head_b, *head_mod;
    WfDitLayerDev *layers;       // host array (owned by the plan)
    // workspace carve-up
    float *x;                    // [(S+1) N_C][dim] residual stream
    __nv_bfloat16 *xa;           // [(S+1) N_C][dim] normalised input / attention output
    __nv_bfloat16 *hmid;         // [(S+1) N_C][max(ffn, 2 dim)]: FFN hidden layer; before the
                                 // attention, the unrotated q | k rows the q/k RMSNorm reads
    __nv_bfloat16 *patches;      // [(S+1) N_C][4 C]
    float *lat;                  // [2][S+1][latent] slot inputs, double-buffered by round parity
    float *modtab;               // [L][S+1][6][dim]
    float *headtab;              // [S+1][2][dim]
    float *temb;                 // [S+1][freq + 3 dim + 6 dim] time-embedding work area
    WfDitLayerDev *layers_dev;   // device copy of the per-layer pointers
    float *tmodel;               // [S+1] model timestep of each slot
    size_t latent;               // floats of one latent chunk
};

size_t wf_dit_workspace_bytes(int S, int NC, int dim, int ffn, int C, int freq, int L, size_t latent,
                              int linear_fp8);
void wf_dit_carve(WfDit *d, void *ws, int S, int NC, size_t latent);

cudaError_t wf_launch_ln_mod(const float *x, void *out, int row_begin, int row_end, int dim, int NC,
                             const float *mod, int mod_ld, int shift_off, int scale_off,
                             cudaStream_t stream, bool out_e4m3 = false);
cudaError_t wf_launch_patchify(const WfGeom &g, int C, const float *const *src, int lo, int hi,
                               __nv_bfloat16 *patches, cudaStream_t stream);
// Timestep embeddings of the S+1 stage slots and the modulation / head
// tables, written once per request of a group (n_req = 1 for one plan).
cudaError_t wf_launch_time_embedding(const WfDit &d, int S, int n_req, cudaStream_t stream);

// ---- failure-detection self-test (selftest.cu) --------------------------------
cudaError_t wf_launch_wait_probe(void *scratch, uint64_t limit_ns, cudaStream_t stream);
