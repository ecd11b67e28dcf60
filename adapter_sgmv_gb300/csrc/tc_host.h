// tc_host.h -- host helpers and launchers of the tensor-core kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lora_sgmv.h"

namespace lora {

// Row-major bf16 matrix [rows, cols] as a 2-D TMA tensor, box [box_rows, box_cols].
bool make_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                       uint32_t box_rows, bool swizzle128);
int sm_count();

// case i: out[t, k] = c * sum_j act[t, j] W(k, j)   (shrink: W = A_i, c = 1; dh: W = B_i^T, c = s_i)
lora_status_t tc_shrink(float *H, const void *x, const lora_adapter_table &tab, const lora_segments &segs,
                        cudaStream_t stream);
lora_status_t tc_dh(float *dH, const void *dY, const lora_adapter_table &tab, const lora_segments &segs,
                    cudaStream_t stream);

// case ii: out[t, n] += c * sum_k h[t, k] W(n, k)   (expand: W = B_i, c = s_i; dX: W = A_i^T, c = 1)
lora_status_t tc_expand(void *y, const float *H, const lora_adapter_table &tab, const lora_segments &segs,
                        cudaStream_t stream);
lora_status_t tc_dx(void *dX, const float *dH, const lora_adapter_table &tab, const lora_segments &segs,
                    cudaStream_t stream);

// cases iii / iv: G_i[n, k] = c * sum_{t in i} act[t, n] h[t, k]   (dB: act = dY, h = H, c = s_i;
// dA: act = X, h = dH, c = 1); G is overwritten
lora_status_t tc_db(float *dB, const void *dY, const float *H, const lora_adapter_table &tab,
                    const lora_segments &segs, cudaStream_t stream);
lora_status_t tc_da(float *dA, const float *dH, const void *X, const lora_adapter_table &tab,
                    const lora_segments &segs, cudaStream_t stream);

}  // namespace lora
