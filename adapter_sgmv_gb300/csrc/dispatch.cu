// dispatch.cu -- choice of kernels for each product of the LoRA delta.
#include "dispatch.h"
#include "tc_host.h"

namespace lora {

lora_status_t run_shrink(float *H, const void *x, const lora_adapter_table &tab, const lora_segments &segs,
                         cudaStream_t stream)
{
    return tc_shrink(H, x, tab, segs, stream);
}

lora_status_t run_expand(void *y, const float *H, const lora_adapter_table &tab, const lora_segments &segs,
                         cudaStream_t stream)
{
    return tc_expand(y, H, tab, segs, stream);
}

lora_status_t run_fwd(void *y, float *H, const void *x, const lora_adapter_table &tab,
                      const lora_segments &segs, cudaStream_t stream)
{
    lora_status_t st = run_shrink(H, x, tab, segs, stream);
    if (st != LORA_OK) return st;
    return run_expand(y, H, tab, segs, stream);
}

lora_status_t run_bwd(void *dX, float *dA, float *dB, const void *dY, const void *X, const float *H, float *dH,
                      const lora_adapter_table &tab, const lora_segments &segs, cudaStream_t stream)
{
    lora_status_t st = tc_dh(dH, dY, tab, segs, stream);
    if (st == LORA_OK && dB != nullptr) st = tc_db(dB, dY, H, tab, segs, stream);
    if (st == LORA_OK && dA != nullptr) st = tc_da(dA, dH, X, tab, segs, stream);
    if (st == LORA_OK && dX != nullptr) st = tc_dx(dX, dH, tab, segs, stream);
    return st;
}

}  // namespace lora
