// Internal declarations shared by the host plan (wf_plan.cpp) and the CUDA
// kernels.  Not part of the public C ABI (include/wf.h).
#pragma once

#include <cstdint>
#include <cstddef>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/wf.h"

#define WF_MAX_TASKS (WF_MAX_STAGES + 1)

// Geometry of a plan, passed by value to every kernel.
struct WfGeom {
    int S, NC, H, D, L;        // stages, chunk tokens, heads, head dim, layers
    int gt, gh, gw;            // latent frames per chunk, patch grid
    int P;                     // pages in the pool
    int raw_anchor_page;       // page keeping the anchor's unrotated key
    int dt2, dh2, dw2;         // rotary pairs of the t / h / w parts
    int t_max;                 // rows of the temporal table (absolute frames)
    int rope_t_off, rope_h_off, rope_w_off;  // float2 offsets of the tables in scratch
};

// One round as the kernels see it (host-built in wf_round_step).
struct WfRoundDev {
    int n_tasks;
    int slot[WF_MAX_TASKS];        // q/out slot (== stage; S for the store)
    int chunk[WF_MAX_TASKS];       // chunk index (temporal position of its own tokens)
    int dest[WF_MAX_TASKS];        // page its K/V are published to
    int n_ctx[WF_MAX_TASKS];       // chunks in its ordered context
    int lpt[WF_MAX_TASKS];         // task indices, longest context first
    uint8_t page[WF_MAX_TASKS][WF_MAX_CTX];  // ordered context page ids (Eq. 5)
    int raw_copy_task;             // task whose K is also kept unrotated (store of the anchor), or -1
    int rerotate;                  // publish launch re-rotates the anchor page
    int anchor_tpos;               // temporal chunk position for the re-rotation
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

cudaError_t wf_launch_attn_simt(const WfGeom &g, const WfRoundDev &rd, int layer, int dtype,
                                const void *qbuf, const void *pool, void *out, cudaStream_t stream);

struct WfTmaps {
    CUtensorMap q;     // qbuf  [S+1][H][NC][128] bf16, box 64 x 128 x 1, 128B swizzle
    CUtensorMap kv;    // pool  [P*L*2*H][NC][128] bf16, same box
};

bool wf_attn_tc_supported(const WfGeom &g, int dtype);
cudaError_t wf_encode_tmaps(const WfGeom &g, void *qbuf, void *pool, WfTmaps *out);
cudaError_t wf_launch_attn_tc(const WfGeom &g, const WfRoundDev &rd, int layer,
                              const WfTmaps &maps, void *out, void *scratch, int num_sms,
                              cudaStream_t stream);

// Variant of wf_launch_attn_tc whose control words live in a static device
// block inside the library (no caller scratch); see wf_round_attention_noalloc.
cudaError_t wf_launch_attn_tc_noalloc(const WfGeom &g, const WfRoundDev &rd, int layer,
                                      const WfTmaps &maps, void *out, int num_sms,
                                      cudaStream_t stream, int *wf_err);
