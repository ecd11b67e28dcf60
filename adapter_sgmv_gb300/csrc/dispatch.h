// dispatch.h -- the sequence of kernels behind each entry point.
#pragma once

#include "internal.h"

namespace lora {

// Workspace of the packed calls: two bf16 hand-off buffers [T, rw] (see
// tc_host.h), or for a decode-size forward the shrink's fp32 slice partials,
// whichever is larger.
size_t handoff_region_bytes(int32_t T, int32_t r_max);
// the ordered backward's tickets (one int per adapter's first span and column
// range of dB and of dA), zeroed at the start of every ordered call
size_t ticket_region_bytes(const lora_adapter_table &tab, int32_t T);
// case i's partials for batches of few tiles (zero bytes otherwise), after the tickets
size_t part_region_bytes(const lora_adapter_table &tab, int32_t T);
// what the backward uses of the workspace: hand-off copies, tickets, partials
size_t bwd_workspace_bytes(const lora_adapter_table &tab, int32_t T);
size_t packed_workspace_bytes(const lora_adapter_table &tab, int32_t T);

// Optional CUDA events recorded around each kernel of a call (measurement):
// ev[2k] before and ev[2k + 1] after the k-th kernel, while room is left.
struct Marks {
    void *const *ev;
    int32_t n;
    int32_t k;
};

lora_status_t run_shrink(float *H, const void *x, const lora_adapter_table &tab, const lora_segments &segs,
                         cudaStream_t stream);
lora_status_t run_expand(void *y, const float *H, const lora_adapter_table &tab, const lora_segments &segs,
                         cudaStream_t stream);
// ws: ws_bytes >= 2 * handoff_region_bytes bytes; case i is split along d
// only when ws_bytes reaches packed_workspace_bytes(tab, T)
lora_status_t run_fwd(void *y, float *H_save, const void *x, void *ws, size_t ws_bytes, const lora_adapter_table &tab,
                      const lora_segments &segs, cudaStream_t stream, Marks *marks = nullptr);
// several projections reading the same x (tables share d_in and the adapter count)
size_t multi_workspace_bytes(int32_t n_proj, const lora_adapter_table *tabs, int32_t T);
lora_status_t run_multi_fwd(int32_t n_proj, void *const *y, float *const *H_save, const void *x, void *ws,
                            size_t ws_bytes, const lora_adapter_table *tabs, const lora_segments &segs,
                            cudaStream_t stream);
// Caller-owned streams and events on which the backward may run its
// independent products side by side (lora_packed_bwd_concurrent).
struct SideStreams {
    cudaStream_t s[2];
    cudaEvent_t ev[4];
};

lora_status_t run_bwd(void *dX, float *dA, float *dB, const void *dY, const void *X, const float *H_saved, void *ws,
                      size_t ws_bytes, const lora_adapter_table &tab, const lora_segments &segs, cudaStream_t stream,
                      Marks *marks = nullptr, const SideStreams *side = nullptr, bool ordered = false);

// one AdamW step over A and B^T (fp32 masters, moments) and their bf16 copies
// in the table (adamw.cu)
lora_status_t run_adamw(const lora_adapter_table &tab, float *wA, float *wB, const float *gA, const float *gB,
                        float *mA, float *vA, float *mB, float *vB, const float *lr, const int32_t *step, float beta1,
                        float beta2, float eps, float weight_decay, cudaStream_t stream);

}  // namespace lora
