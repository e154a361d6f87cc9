/*
 * wf.h -- C ABI of the wavefront-round library (libwf.so).
 *
 * One wavefront round of the chunk-wise causal DiT forward of "Wave Forcing:
 * Towards Speed-of-Light Streaming Video Generation" (arXiv 2611.00859), on
 * one GPU.  In round k the S+1 tasks -- chunk i = k - s at denoising stage s
 * for every active s < S, plus the store pass of chunk k - S (stage S) -- are
 * batched into the same kernels (Sec. 3.1 Eq. 3).  Each query token attends
 * bidirectionally inside its own chunk and to the paged K/V of earlier,
 * cleaner chunks under M_WF(s, j) = 1[j >= s] (Sec. 3.1 Eq. 4), in the
 * ordered context anchor, history, live store, live stages j >= s (Eq. 5).
 *
 * Conventions shared by every entry point:
 *  - Every function returns an int: WF_OK (0) on success, a negative WF_E*
 *    code otherwise.  Arguments are validated on the host before anything is
 *    launched; a rejected call launches nothing and changes no state.
 *  - Device pointers are caller-owned (the library never frees caller memory
 *    and allocates no device memory of its own: every device buffer, scratch
 *    included, is passed in through wf_bind).  The plan owns host state only.
 *  - Launching calls are asynchronous on the caller's stream; a plan is not
 *    thread-safe (one plan per host thread).
 *  - "slot" s in [0, S] indexes the fixed per-stage buffers: slot s < S holds
 *    the task at denoising stage s, slot S the store task.  Slots of inactive
 *    stages (pipeline fill/drain) are neither read nor written.
 *  - Element type of every activation buffer is the plan's dtype
 *    (WF_BF16: bfloat16, WF_FP32: float); with WF_FP8 the query workspace
 *    and the page pool hold e4m3 bytes while qkv and out are bfloat16.
 *
 * Layouts (row-major, innermost last; N_C = chunk_tokens, H = heads,
 * D = head_dim, L = layers, P = n_pages from wf_plan_buffer_sizes):
 *   qkv      [S+1][N_C][3][H][D]   raw (pre-RoPE) Q/K/V of each slot, the
 *                                   token-major order a QKV projection writes
 *   qbuf     [S+1][H][N_C][D]       RoPE-applied queries (library workspace)
 *   pool     [P][L][2][H][N_C][D]   K/V pages (index 0 = K, 1 = V); page ids
 *                                   follow wf_page_table
 *   out      [S+1][N_C][H][D]       attention output, token-major
 */
#ifndef WF_H
#define WF_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *cudaStream_t; /* identical to CUDA's own typedef */

/* ---- return codes ------------------------------------------------------ */
#define WF_OK            0
#define WF_EINVAL       -1  /* bad argument (null pointer, bad enum, misaligned) */
#define WF_ERANGE       -2  /* size or index out of the supported range */
#define WF_ENOMEM       -3  /* a caller buffer is smaller than required */
#define WF_ECUDA        -4  /* a CUDA runtime/driver call failed */
#define WF_ETIMEOUT     -5  /* a device-side bounded wait gave up (see wf_sync_status) */
#define WF_EDONE        -6  /* the request has no more rounds (k >= N_chunk + S) */
#define WF_EUNBOUND     -7  /* wf_bind has not been called */
#define WF_ENOROUND     -8  /* no current round: call wf_round_step first */
#define WF_EUNSUPPORTED -9  /* shape/dtype not supported by the requested kernel */
#define WF_EORDER      -10  /* attention before this round's publication of that layer */

#define WF_FP32 0
#define WF_BF16 1
#define WF_FP8  2  /* 8-bit attention: Q and the K/V pages stored as OCP FP8 e4m3 (1 byte;
                      Q and K multiplied by fp8_qk_scale, V by fp8_v_scale before rounding,
                      saturating at +-448); Q/K/V input and attention output stay bf16;
                      tensor-core attention only (the pages' 8-bit SageAttention backend
                      and FP8 K/V payload, Sec. 5 and App. C.6) */

#define WF_ANCHOR_ADJACENT 0 /* anchor re-rotated just before the oldest retained chunk */
#define WF_ANCHOR_ABSOLUTE 1 /* anchor keeps its own position (frames 0..grid_t-1) */

#define WF_MASK_WF 0   /* chunk-wise causal mask M_WF(s, j) = 1[j >= s] (Sec. 3.1 Eq. 4) */
#define WF_MASK_RF 1   /* Rolling Forcing's full active window: denoising tasks also read
                          noisier live chunks (the reverse edges Eq. 4 removes) */

#define WF_SCHED_WAVEFRONT  0 /* S+1 staggered tasks per round, one chunk per round (1F1C) */
#define WF_SCHED_SEQUENTIAL 1 /* one task per round: each chunk's S denoising forwards, then
                                 its store pass (NF1C, Sec. 2) */

#define WF_KIND_ANCHOR  0
#define WF_KIND_HISTORY 1
#define WF_KIND_STORE   2
#define WF_KIND_LIVE    3

#define WF_MAX_STAGES 8   /* S <= 8, so at most 9 tasks per round */
#define WF_MAX_CTX    32  /* at most 32 chunks in one task's ordered context */

#define WF_ATTN_AUTO 0    /* tensor-core kernel when supported, else the SIMT kernel */
#define WF_ATTN_TC   1    /* tcgen05/TMEM/TMA kernel (bf16, head_dim 128) */
#define WF_ATTN_SIMT 2    /* CUDA-core kernel (fp32 or bf16, head_dim 32..128, %32) */

#define WF_EPI_BF16           0 /* out bf16 = acc + bias */
#define WF_EPI_F32            1 /* out f32  = acc + bias */
#define WF_EPI_GELU_BF16      2 /* out bf16 = GELU_tanh(acc + bias) */
#define WF_EPI_GATED_RESIDUAL 3 /* out f32 += gate[row / rows_per_group][col] * (acc + bias) */

typedef struct wf_plan_s *wf_plan_t; /* opaque, library-owned host state */

typedef struct wf_plan_opts {
    int n_chunks;       /* N_chunk, chunks in the request (>= 1) */
    int layers;         /* L, transformer layers with a K/V page each (>= 1) */
    int grid_t;         /* latent frames per chunk (3 in the paper, App. A) */
    int grid_h, grid_w; /* patch grid; grid_t*grid_h*grid_w == chunk_tokens */
    int dtype;          /* WF_BF16 (default) or WF_FP32 */
    int use_anchor;     /* 1 (default): first clean chunk is a persistent anchor (App. B.3) */
    int anchor_mode;    /* WF_ANCHOR_ADJACENT (default) or WF_ANCHOR_ABSOLUTE */
    double rope_theta;  /* RoPE base, default 10000 */
    int mask;           /* WF_MASK_WF (default) or WF_MASK_RF */
    int schedule;       /* WF_SCHED_WAVEFRONT (default) or WF_SCHED_SEQUENTIAL */
    double fp8_qk_scale;  /* WF_FP8: scale of Q and K before e4m3 rounding (default 1) */
    double fp8_v_scale;   /* WF_FP8: scale of V before e4m3 rounding (default 1) */
    int store_extra_history; /* E >= 0 (default 0): the store pass keeps the E next-older
                                clean chunks besides the W all tasks see ("Wave Forcing"
                                App. B.3: the store reserves one query chunk where a
                                denoising task reserves S, so under a token budget its
                                prefix can be longer; E = S gives it the key count of a
                                stage-0 task).  Needs history_chunks >= 0.  Page-table
                                label of those entries: S + 2 (seen by the store only). */
    int rope_split[3];  /* sizes (d_t, d_h, d_w) of the temporal / height / width parts of the
                           head dimension rotated by 3D RoPE (Sec. 4.2 applies RoPE; the
                           pages give no split): all 0 (default) = D - 4 floor(D/6),
                           2 floor(D/6), 2 floor(D/6) (128 -> 44/42/42); otherwise even,
                           >= 0 and summing to head_dim, else WF_EINVAL */
} wf_plan_opts;

typedef struct wf_buffer_sizes {
    size_t qkv;      /* bytes of one round's raw Q/K/V input */
    size_t qbuf;     /* bytes of the query workspace */
    size_t pool;     /* bytes of the K/V page pool */
    size_t out;      /* bytes of one attention output */
    size_t scratch;  /* bytes of library scratch (RoPE tables, scheduler counters, status) */
    int n_pages;     /* P */
    int ring_pages;  /* R: clean-history ring incl. the live store page */
    size_t qk_norm_tmp; /* bytes of the q | k workspace wf_qkv_proj_rope_publish needs when it
                           normalises q and k: (S+1) N_C 2 H D bf16 */
} wf_buffer_sizes;

typedef struct wf_round_info {
    int k;                 /* round just entered, 0 .. N_chunk+S-1 (sequential: 0 .. N_chunk(S+1)-1) */
    int n_tasks;           /* active tasks, 1 .. S+1 */
    int store_chunk;       /* chunk whose store pass runs (its clean output B_i completes), or -1 */
    int anchor_tpos;       /* temporal chunk position of the anchor's keys this round, or -1 */
    int task_chunk[WF_MAX_STAGES + 1];  /* per active task (slot order): chunk i */
    int task_stage[WF_MAX_STAGES + 1];  /* stage s (== slot); S for the store */
    int task_ctx[WF_MAX_STAGES + 1];    /* chunks in its ordered context */
    double attn_flops;     /* algorithmic attention FLOPs of one layer: sum 4*N_C*keys*D*H */
} wf_round_info;

/* Fill *opts with the defaults listed above (n_chunks = 1, layers = 1,
 * grid_t = 3, grid_h = grid_w = 0 meaning "chunk_tokens/3 x 1"). */
void wf_plan_opts_default(wf_plan_opts *opts);

/* Create a plan for one request: S denoising stages (store = stage S),
 * chunk_tokens = N_C, heads = H, head_dim = D, history_chunks = W clean
 * chunks kept besides the anchor (-1 = all).  "Wave Forcing" Sec. 3.1
 * Eq. 3-5; App. B.2 Eq. 13 and App. B.8 (fixed page capacity: anchor,
 * W history + live store ring, S live pages, plus one page that keeps the
 * anchor's unrotated key, App. B.3).  No CUDA call is made.
 * Errors: WF_EINVAL (null out, bad enum, odd D, grid mismatch), WF_ERANGE
 * (S > WF_MAX_STAGES, context longer than WF_MAX_CTX, sizes overflow). */
int wf_plan(int S, int chunk_tokens, int heads, int head_dim, int history_chunks,
            const wf_plan_opts *opts, wf_plan_t *out);

/* Bytes of every caller-owned buffer this plan needs.  No CUDA call. */
int wf_plan_buffer_sizes(wf_plan_t plan, wf_buffer_sizes *out);

/* Attach caller-owned device memory (all 256-byte aligned, sizes from
 * wf_plan_buffer_sizes) and the current CUDA device.  Uploads the RoPE
 * tables into scratch (synchronous), zeroes the scratch control words, and
 * encodes the TMA descriptors.  May be called again to re-bind.
 * Errors: WF_EINVAL (null/misaligned), WF_ECUDA. */
int wf_bind(wf_plan_t plan, void *pool, void *qbuf, void *scratch);

/* Advance to the next round k (the first call enters k = 0).  Host only:
 * promotes the previous round's store page into history, evicts the oldest
 * history page beyond W, allocates the store page of chunk k - S, and builds
 * the ordered contexts of the round (Algorithm 1, App. B.3).  With
 * WF_SCHED_SEQUENTIAL round k runs the single task chunk k / (S+1) at stage
 * k % (S+1) (stage S = its store pass) over anchor, history and itself.
 * With WF_MASK_RF each denoising task's context also lists the noisier live
 * chunks (all live stages in increasing order).  info may be NULL.
 * Errors: WF_EDONE after the last round (state unchanged). */
int wf_round_step(wf_plan_t plan, wf_round_info *info);

/* Export the current round's table as int32 rows, one per context entry:
 *   {slot, chunk, stage, dest_page, ctx_index, kind, entry_chunk, j, page, tpos}
 * (10 ints per row, tasks in slot order, entries in Eq. 5 order).  Writes at
 * most cap rows and stores the row count in *n_rows.  Errors: WF_ENOROUND. */
int wf_page_table(wf_plan_t plan, int32_t *out, int cap, int *n_rows);

/* QKV publication of one layer (Sec. 4.2: "publishes K/V after QKV
 * projection and RoPE"; App. B.2 paged placement Eq. 13).  For every active
 * task: applies 3D RoPE to Q and K at the task chunk's absolute positions,
 * writes Q to qbuf[slot] and K/V straight into the task's fixed page (live
 * page of its stage; ring page of the stored chunk; the anchor page -- plus
 * its unrotated key -- when chunk 0 is stored).  When the anchor's position
 * differs from the one its page of this layer was last rotated at, the same
 * launch re-rotates the anchor key from its unrotated copy (App. B.3).
 * qkv: device pointer, layout above.  Errors: WF_EUNBOUND, WF_ENOROUND,
 * WF_ERANGE (layer), WF_EINVAL (null), WF_ECUDA (launch). */
int wf_qkv_rope_publish(wf_plan_t plan, int layer, const void *qkv, cudaStream_t stream);

/* Round attention of one layer: one launch computes, for every active task
 * and head, softmax(Q K^T / sqrt(D)) V over the task's ordered context
 * (Eq. 5) read from the page pool, bidirectional inside each chunk; keys of
 * chunks outside the context are never visited (Sec. 3.1 Eq. 4).
 * out: device pointer [S+1][N_C][H][D].  kernel: WF_ATTN_*.
 * Uses scratch (scheduler counters; calls that overlap on the GPU with the
 * same scratch race).  Errors: WF_EUNBOUND, WF_ENOROUND, WF_ERANGE,
 * WF_EINVAL, WF_EORDER (wf_qkv_rope_publish of this layer has not run in
 * this round: the pages would hold stale K/V), WF_EUNSUPPORTED (kernel not
 * available for dtype/head_dim), WF_ECUDA. */
int wf_round_attention(wf_plan_t plan, int layer, void *out, int kernel, cudaStream_t stream);

/* Round attention of a subset of the round's tasks: as wf_round_attention,
 * for the active tasks whose slot s has bit s set in slot_mask (other slots
 * of out are not written).  Each task's result does not depend on which
 * other tasks share the launch (every (task, head, query tile) unit reads
 * only its own context, in a fixed order), so launching the tasks one at a
 * time -- e.g. the store, then stages S-1 .. 0, the sequential replay of
 * "Wave Forcing" App. B.6 Proposition 1 -- gives bit-identical outputs to
 * the batched launch.  Lets a caller run the store pass first or split a
 * round over streams.  A mask selecting no active task launches nothing.
 * Errors: as wf_round_attention, plus WF_EINVAL (bits above slot S set). */
int wf_round_attention_tasks(wf_plan_t plan, int layer, void *out, int kernel,
                             unsigned int slot_mask, cudaStream_t stream);

/* Round attention without caller-provided scratch.  The paper has no
 * counterpart: this is a library convenience.
 *
 * Same computation, kernel and output as wf_round_attention(plan, layer, out,
 * WF_ATTN_TC, stream) -- the tensor-core kernel, so bf16 or WF_FP8 plans with
 * head_dim 128 only (else WF_EUNSUPPORTED) -- but the kernel's scheduler
 * counters live in a fixed block of WF_NOALLOC_SCRATCH_BYTES inside libwf.so
 * instead of the plan's scratch buffer.  It is meant for callers that cannot
 * allocate device memory at the point where they launch attention: code
 * running under a memory manager that owns every device byte (a caching
 * allocator or an arena sized at start-up), or a steady-state loop that must
 * not call cudaMalloc because it can synchronise the whole device.  This
 * call itself calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * - The first call on a device (the current device) looks up the block's
 *   device address once (cudaGetSymbolAddress); make that first call before
 *   any stream capture.  The address is kept for the life of the process:
 *   after the device's context is destroyed (cudaDeviceReset) it is stale,
 *   so do not call this entry point again in that process.  Every GPU that
 *   loads the library holds the block until the process exits.
 * - Each call clears the block's counters on `stream` (cudaMemsetAsync of
 *   the counter words) before the launch.  All calls share the one block,
 *   so calls whose kernels overlap on the GPU (different streams, or
 *   different plans on the same device) race; serialise them.
 * - The counters the kernel needs must fit in the block; a larger need is
 *   rejected with WF_ERANGE before anything is launched.
 * - A bounded-wait timeout inside the kernel is recorded in the status word
 *   of the plan's scratch, as wf_round_attention records it, so
 *   wf_sync_status reports it (the next call does not clear it).
 * Errors: as wf_round_attention, plus WF_ERANGE (control block too small)
 * and WF_ECUDA (symbol lookup, memset or launch failed). */
#define WF_NOALLOC_SCRATCH_BYTES 256
int wf_round_attention_noalloc(wf_plan_t plan, int layer, void *out, cudaStream_t stream);

/* ---- several requests batched into one round ------------------------------
 * "Wave Forcing" names serving concurrent streams with batching as the next
 * step (Sec. 8 Future Work; App. E).  A group batches the current rounds of
 * up to WF_MAX_GROUP_PLANS independent requests into single launches.
 *
 * Each member plan keeps its own schedule, page ring and anchor and is
 * advanced with wf_round_step as before: members may start at different
 * times and finish on their own.  A group call takes plan_mask (bit r:
 * member r takes part; a member that has not entered a round yet or has
 * finished is left out) and concatenates the selected members' rounds: the
 * tasks of member r use slot r (S+1) + s and page r P + p of the group's
 * buffers, so one launch serves all of them and every member gets exactly
 * what its own wf_qkv_rope_publish / wf_round_attention would compute.
 *
 * wf_group_create: plans[0 .. n-1] (1 <= n <= WF_MAX_GROUP_PLANS), distinct,
 *   bound, of one shape (every plan option that fixes the buffers' layout or
 *   bytes equal: S, N_C, H, D, W, n_chunks, layers, grid, dtype, RoPE, e4m3
 *   scales), on one device, whose pools and query workspaces are consecutive
 *   slices of one allocation: plan r's pool at plan 0's pool + r * pool
 *   bytes, its query workspace at plan 0's + r * qbuf bytes
 *   (wf_plan_buffer_sizes).  n * n_pages <= 256.  The group keeps the
 *   pointers: the plans must outlive it and stay bound to those buffers.
 *   Group launches use plan 0's scratch (RoPE tables, scheduler counters,
 *   status): read timeouts with wf_sync_status(plans[0]) and do not overlap
 *   them with plan 0's own launches.  Errors: WF_EINVAL (null, duplicate,
 *   shape or layout mismatch), WF_ERANGE (n, page ids), WF_EUNBOUND,
 *   WF_ECUDA (tensor maps).
 * wf_group_publish: as wf_qkv_rope_publish for every selected member, one
 *   launch (plus the members' anchor re-rotations in the same launch);
 *   qkv [n][S+1][N_C][3][H][D].
 * wf_group_proj_publish: as wf_qkv_proj_rope_publish for every selected
 *   member, one projection GEMM over their rows; x [n][S+1][N_C][dim];
 *   qk_tmp (with the q/k RMSNorm gains) n * wf_buffer_sizes.qk_norm_tmp
 *   bytes.
 * wf_group_attention: as wf_round_attention for every selected member, one
 *   launch; out [n][S+1][N_C][H][D].  WF_EORDER when a selected member has
 *   not published this layer in its current round.
 * Errors of the launching calls: as their single-plan counterparts, plus
 *   WF_EINVAL (empty mask or bits beyond n), WF_ENOROUND (a selected member
 *   has no current round). */
#define WF_MAX_GROUP_PLANS 8
typedef struct wf_group_s *wf_group_t;
int wf_group_create(const wf_plan_t *plans, int n, wf_group_t *out);
int wf_group_publish(wf_group_t group, unsigned int plan_mask, int layer, const void *qkv,
                     cudaStream_t stream);
int wf_group_proj_publish(wf_group_t group, unsigned int plan_mask, int layer, const void *x,
                          const void *w_qkv, const void *b_qkv, const void *norm_q,
                          const void *norm_k, void *qk_tmp, cudaStream_t stream);
int wf_group_attention(wf_group_t group, unsigned int plan_mask, int layer, void *out, int kernel,
                       cudaStream_t stream);
void wf_group_destroy(wf_group_t group);

/* ---- linear layers on the tensor cores -------------------------------------
 * out = epilogue(A W^T + bias) for rows row_begin .. row_end-1 of A.
 *   a     bf16 [a_rows][lda] row-major activations (device)
 *   w     bf16 [N][K] row-major weight of a linear layer, output-major (device)
 *   bias  bf16 [N] or NULL
 *   out   WF_EPI_BF16 / WF_EPI_GELU_BF16: bf16 [.][ldo]; WF_EPI_F32 and
 *         WF_EPI_GATED_RESIDUAL: float [.][ldo]; row r of out corresponds to
 *         row r of a.  For the gated residual, out[r] += gate-row * (A W^T +
 *         bias)[r]: the sum is added in place by the GPU's memory system (a
 *         tensor reduce-add per 32 x 32 block), once per element, only on
 *         rows row_begin .. row_end-1; nothing else may write those rows
 *         while the call runs
 *   gate  WF_EPI_GATED_RESIDUAL only: float rows of gate_ld values, row
 *         r / rows_per_group gates output row r (one gate vector per task slot
 *         when rows_per_group = N_C); at least (row_end - 1) / rows_per_group
 *         + 1 rows
 * These are the dense operators of one DiT block ("Wave Forcing" Sec. 4.1:
 * attention and "the remaining block" of the standard Wan2.1 transformer,
 * App. D.2): output projection and FFN with gated residual adds, GELU FFN
 * hidden layer, patch embedding.  Uses the plan's scratch status word for
 * bounded-wait timeouts (wf_sync_status) and nothing else of the plan.
 * Requirements: K % 64 == 0, N % 32 == 0, lda % 8 == 0, ldo % 8 == 0, every
 * pointer 16-byte aligned.  Errors: WF_EINVAL, WF_ERANGE (row range),
 * WF_EUNBOUND, WF_ECUDA. */
int wf_linear(wf_plan_t plan, const void *a, long long a_rows, int lda, int row_begin, int row_end,
              const void *w, const void *bias, int N, int K, int epilogue, void *out, int ldo,
              const float *gate, int gate_ld, int rows_per_group, cudaStream_t stream);

/* 8-bit linear layers (the pages' W8A8 backend, Sec. 5; the pages give no
 * recipe, so: OCP e4m3 weights with one scale per output channel, e4m3
 * activations with unit scale, fp32 accumulation).
 *
 * wf_quantize_weight_e4m3: w bf16 [N][K] -> w8 e4m3 [N][K] and scale float
 *   [N]: scale[n] = max_k |w[n][k]| / 448 (1 for an all-zero row),
 *   w8[n][k] = e4m3(w[n][k] / scale[n]) (round to nearest even, saturating).
 * wf_linear_e4m3: as wf_linear with a8 e4m3 [a_rows][lda] and w8 e4m3
 *   [N][K]; out = epilogue(scale[n] * (a8 w8^T) + bias).  K % 128 == 0,
 *   lda % 16 == 0.
 * Errors: as wf_linear. */
int wf_quantize_weight_e4m3(wf_plan_t plan, const void *w, int N, int K, void *w8, float *scale,
                            cudaStream_t stream);
int wf_linear_e4m3(wf_plan_t plan, const void *a8, long long a_rows, int lda, int row_begin,
                   int row_end, const void *w8, const float *wscale, const void *bias, int N, int K,
                   int epilogue, void *out, int ldo, const float *gate, int gate_ld,
                   int rows_per_group, cudaStream_t stream);

/* QKV projection of one layer fused with RoPE and paged publication (Sec.
 * 4.2: "publishes K/V after QKV projection and RoPE"; App. B.2 Eq. 13 direct
 * placement into fixed slots).  Same effect as wf_qkv_rope_publish applied
 * to qkv = x W_qkv^T + b_qkv, without materialising qkv:
 *   x      bf16 [S+1][N_C][dim] (dim = heads*head_dim), slot-indexed like
 *          qkv; only the active slots' rows are read
 *   w_qkv  bf16 [3 dim][dim]: rows 0..dim-1 produce Q, then K, then V; head h
 *          of each part is rows h*head_dim .. h*head_dim + head_dim - 1
 *   b_qkv  bf16 [3 dim] or NULL
 *   norm_q, norm_k  bf16 [dim] gains of the standard Wan2.1 block's q/k
 *          RMSNorm (App. D.2 keeps that architecture), or both NULL for no
 *          normalisation: q <- q / sqrt(mean(q^2) + 1e-6) * norm_q over the
 *          full width (all heads of a token), likewise k, before RoPE.  The
 *          projection then writes the unrotated q | k rows (bf16) to
 *   qk_tmp  device workspace of wf_buffer_sizes.qk_norm_tmp bytes (16-byte
 *          aligned; ignored without norms), and a second, memory-bound
 *          launch normalises, rotates and publishes them
 * bf16 or WF_FP8 plans (e4m3 pages), dim % 64 == 0, head_dim % 32 == 0.
 * Errors: as wf_qkv_rope_publish, plus WF_EUNSUPPORTED; WF_EINVAL when only
 * one gain is given or qk_tmp is missing. */
int wf_qkv_proj_rope_publish(wf_plan_t plan, int layer, const void *x, const void *w_qkv,
                             const void *b_qkv, const void *norm_q, const void *norm_k,
                             void *qk_tmp, cudaStream_t stream);

/* ---- the chunk-wise causal DiT round --------------------------------------
 * Weights of one transformer block (device pointers, bf16, linear weights
 * [out][in]; biases may be NULL). */
typedef struct wf_dit_layer {
    const void *qkv_w, *qkv_b;     /* [3 dim][dim], [3 dim] */
    const void *o_w, *o_b;         /* [dim][dim], [dim] */
    const void *ffn1_w, *ffn1_b;   /* [ffn][dim], [ffn] */
    const void *ffn2_w, *ffn2_b;   /* [dim][ffn], [dim] */
    const void *modulation;        /* [6][dim]: shift, scale, gate of attention, then of FFN */
    const void *norm_q, *norm_k;   /* [dim], [dim]: gains of the q / k RMSNorm (required) */
} wf_dit_layer;

/* A Wan2.1-style DiT without text cross-attention (the pages omit text
 * conditioning, Sec. 2).  The block, as this library computes it:
 *   (shift_a, scale_a, gate_a, shift_f, scale_f, gate_f) = modulation + e0(t)
 *   x' = LN(x)(1 + scale_a) + shift_a   (LayerNorm eps 1e-6, no affine)
 *   Q,K,V = x' W_qkv^T + b; Q = RMSNorm(Q) norm_q, K = RMSNorm(K) norm_k
 *   (over the full width, eps 1e-6); RoPE on Q, K; x += gate_a (Attn W_o^T + b_o)
 *   x += gate_f (GELU_tanh((LN(x)(1 + scale_f) + shift_f) W_1^T + b_1) W_2^T + b_2)
 * with the timestep embedding e(t) = W_t2 SiLU(W_t1 sinusoid(t) + b) + b,
 * e0 = W_tp SiLU(e) + b_tp; patch embedding of (1,2,2) patches of C
 * channels (features ordered channel, row offset, column offset); head
 * (shift, scale) = head_mod + e, y = (LN(x)(1 + scale) + shift) W_h^T + b_h,
 * 4C outputs per token ordered (row offset, column offset, channel). */
typedef struct wf_dit_model {
    int model_dim;                 /* = heads * head_dim of the plan */
    int ffn_dim;                   /* % 64 == 0 */
    int channels;                  /* latent channels C, 4C % 64 == 0 (16 for Wan2.1) */
    int freq_dim;                  /* sinusoidal timestep features (256 for Wan2.1) */
    double shift;                  /* timestep warp: sigma' = shift s / (1 + (shift-1) s), s = nu/1000 */
    double context_noise;          /* nu of the store pass (App. B.3), in [0, 1000] */
    double timesteps[WF_MAX_STAGES];  /* nu_0 > ... > nu_{S-1} in (0, 1000] (App. A) */
    const void *patch_w, *patch_b; /* [dim][4C], [dim] */
    const void *t1_w, *t1_b;       /* [dim][freq], [dim] */
    const void *t2_w, *t2_b;       /* [dim][dim], [dim] */
    const void *tp_w, *tp_b;       /* [6 dim][dim], [6 dim] */
    const void *head_w, *head_b;   /* [4C][dim], [4C] */
    const void *head_mod;          /* [2][dim]: shift, scale */
    const wf_dit_layer *layers;    /* host array of `layers` (plan option) entries */
    int linear_fp8;                /* 1: the block's four linear layers run in e4m3 (weights
                                      quantised per output channel at bind time, LN output,
                                      attention output and FFN hidden layer as e4m3 with unit
                                      scale); patch embedding and head stay bf16 */
} wf_dit_model;

/* Bytes of the DiT workspace (residual stream, normalised activations, FFN
 * hidden layer, patches, double-buffered latent slot inputs, modulation
 * tables; with linear_fp8 also the e4m3 activations and the quantised
 * weights of every layer).  No CUDA call.  Errors: WF_EINVAL (dims). */
int wf_dit_workspace_size(wf_plan_t plan, int model_dim, int ffn_dim, int channels, int freq_dim,
                          int linear_fp8, size_t *bytes);

/* Attach a model and a caller-owned workspace (256-byte aligned, size from
 * wf_dit_workspace_size) to a bound bf16 or WF_FP8 plan with head_dim 128
 * (WF_FP8: attention in e4m3, every other tensor as in the bf16 plan).  The weight
 * pointers are kept (not copied): they must stay valid while the plan is
 * used.  Computes the timestep embeddings and modulation tables of every
 * slot on `stream` (each stage has a fixed timestep) and clears the latent
 * slot buffers.  Errors: WF_EINVAL, WF_EUNBOUND, WF_EUNSUPPORTED, WF_ENOMEM,
 * WF_ECUDA. */
int wf_dit_bind(wf_plan_t plan, const wf_dit_model *model, void *workspace, cudaStream_t stream);

/* The DiT forward of the current round (enter it with wf_round_step) for
 * every active task, and the stage transition of Sec. 2 Eq. 1:
 *   Z^(s+1) = Psi_{nu_{s+1}}(G(Z^(s), nu_s | C), eps),  Psi_nu(x, e) = (1 - sigma') x + sigma' e,
 * Psi_0 = identity.  Slot 0 reads z_new (the fresh noise Z^(0) of chunk k);
 * slot s in 1..S-1 reads the latent its chunk left in the previous round;
 * the store slot reads the clean chunk finished in the previous round.
 *   z_new      float [C][grid_t][2 grid_h][2 grid_w] (device), required while
 *              chunk k < N_chunk
 *   eps        float [S][latent]: eps[s] re-noises slot s's prediction (eps[S-1]
 *              is not read); may be NULL when S == 1
 *   x0_out     float [S+1][latent] predictions of the active slots, or NULL
 *   chunk_out  float [latent]: the clean chunk B_{k-S+1} finished this round
 *              (written when stage S-1 is active), or NULL
 * All L layers run: per layer one batched QKV projection with RoPE and
 * paged publication, one round-attention launch, the output projection,
 * and the FFN; then the head.  Asynchronous on `stream`.  Errors:
 * WF_EUNBOUND (no wf_bind / wf_dit_bind), WF_ENOROUND, WF_EINVAL, WF_ECUDA. */
int wf_dit_round(wf_plan_t plan, const float *z_new, const float *eps, float *x0_out,
                 float *chunk_out, cudaStream_t stream);

/* ---- whole DiT rounds of a group -------------------------------------------
 * The DiT round of every selected member of a group (wf_group_create) in one
 * pass: one patch embedding, per layer one projection + publication, one
 * attention launch, the output projection and the FFN over all selected
 * members' tasks, then one head.  Each member computes exactly what its own
 * wf_dit_round computes (same kernels, global slots as in the group calls).
 * The group keeps its own DiT state: the members' latent slot inputs live
 * in the group workspace, double-buffered by each member's round parity, so
 * a member advanced by group rounds is not also run by wf_dit_round.
 *
 * wf_group_dit_workspace_size: bytes of the group's DiT workspace (the
 *   single-plan workspace with n (S+1) slots).  Errors: as
 *   wf_dit_workspace_size.
 * wf_group_dit_bind: as wf_dit_bind for the group (model checked against
 *   member 0; workspace 256-byte aligned, caller-owned; modulation tables
 *   written once per member; latent buffers cleared).  The weight pointers
 *   are kept.
 * wf_group_dit_round: members in plan_mask, each already entered into its
 *   current round with wf_round_step.  Request r's arguments sit at
 *   r times the single-plan sizes:
 *     z_new      float [n][latent]: member r's fresh chunk, read when member r
 *                has a stage-0 task
 *     eps        float [n][S][latent] (may be NULL when S == 1)
 *     x0_out     float [n][S+1][latent] or NULL (rows of active slots written)
 *     chunk_out  float [n][latent] or NULL (row r written when member r has a
 *                stage-(S-1) task)
 *   Launches use member 0's scratch (wf_sync_status(plans[0])).  Errors:
 *   WF_EINVAL (mask, pointers), WF_EUNBOUND (no wf_group_dit_bind),
 *   WF_ENOROUND, WF_ECUDA. */
int wf_group_dit_workspace_size(wf_group_t group, int model_dim, int ffn_dim, int channels,
                                int freq_dim, int linear_fp8, size_t *bytes);
int wf_group_dit_bind(wf_group_t group, const wf_dit_model *model, void *workspace,
                      cudaStream_t stream);
int wf_group_dit_round(wf_group_t group, unsigned int plan_mask, const float *z_new,
                       const float *eps, float *x0_out, float *chunk_out, cudaStream_t stream);

/* Read and clear the device status word in scratch (synchronises stream).
 * Returns WF_OK, WF_ETIMEOUT if a kernel's bounded wait gave up, or WF_ECUDA. */
int wf_sync_status(wf_plan_t plan, cudaStream_t stream);

/* Failure-detection self-test.  Launches one CTA that waits, with the same
 * bounded wait the library's kernels use, on a barrier that nothing ever
 * completes; after limit_us microseconds the wait gives up, records the
 * timeout in the plan's status word and the kernel returns, leaving the
 * context usable.  The following wf_sync_status returns WF_ETIMEOUT (and
 * clears the word).  Errors: WF_EUNBOUND, WF_ERANGE (limit_us outside
 * 1 .. 2,000,000), WF_ECUDA. */
int wf_selftest_timeout(wf_plan_t plan, unsigned int limit_us, cudaStream_t stream);

/* Checkpoint / resume of a request's host round state: round index,
 * history ring, free pages, anchor state and the per-layer publication and
 * anchor-rotation records (int32 words, versioned).  Together with the K/V
 * page pool (caller-owned device memory, which the caller keeps) this lets a
 * request continue in a new plan of the same shape.  Import checks the shape
 * words (S, N_C, heads, head_dim, W, n_chunks, layers, anchor, mask,
 * schedule, store history, and what fixes the pages' bytes: dtype, RoPE base
 * and split, e4m3 scales), every page and chunk id, and that each ring page
 * sits in exactly one of history (oldest first), the free list and the
 * pending store page; then it rebuilds the current round's contexts.  No
 * CUDA call.  Errors: WF_EINVAL (null, foreign or corrupt state), WF_ENOMEM
 * (cap smaller than wf_plan_state_size). */
int wf_plan_state_size(wf_plan_t plan, size_t *bytes);
int wf_plan_export_state(wf_plan_t plan, void *buf, size_t cap, size_t *written);
int wf_plan_import_state(wf_plan_t plan, const void *buf, size_t n);

void wf_plan_destroy(wf_plan_t plan);
const char *wf_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* WF_H */
