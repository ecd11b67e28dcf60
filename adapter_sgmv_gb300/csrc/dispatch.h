// dispatch.h -- choice of kernels for each product of the LoRA delta.
#pragma once

#include "internal.h"

namespace lora {

lora_status_t run_shrink(float *H, const void *x, const lora_adapter_table &tab, const lora_segments &segs,
                         cudaStream_t stream);
lora_status_t run_expand(void *y, const float *H, const lora_adapter_table &tab, const lora_segments &segs,
                         cudaStream_t stream);
lora_status_t run_fwd(void *y, float *H, const void *x, const lora_adapter_table &tab,
                      const lora_segments &segs, cudaStream_t stream);
lora_status_t run_bwd(void *dX, float *dA, float *dB, const void *dY, const void *X, const float *H, float *dH,
                      const lora_adapter_table &tab, const lora_segments &segs, cudaStream_t stream);

}  // namespace lora
