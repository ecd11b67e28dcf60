// internal.h -- declarations shared between the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lora_sgmv.h"

namespace lora {

constexpr int32_t kMaxAdapters = 65536;
constexpr int32_t kMaxTokens = 1 << 24;
constexpr int64_t kMaxHistWords = int64_t(1) << 26;  // N * ceil(T / 32) counters
constexpr int32_t kMaxDim = 1 << 20;

// word offsets of the regions of a lora_segments storage block
struct SegLayout {
    bool ok;
    int32_t n_chunks, max_tiles, max_spans, block_sums;
    int64_t hist_words;
    int64_t off_perm, off_seg, off_tiles, off_ntiles, off_status, off_spans, off_nspans, off_scratch;
    int64_t scratch_words, total_words;
};

SegLayout seg_layout(int32_t T, int32_t N);

lora_status_t build_segments(const int32_t *ids, const int32_t *seg_offsets, int32_t T, int32_t N,
                             void *storage, size_t storage_bytes, lora_segments *out,
                             cudaStream_t stream);

// generic SIMT kernels (any rank, any routing), each launch stream-ordered
lora_status_t simt_shrink(float *H, const void *x, const lora_adapter_table &tab,
                          const lora_segments &segs, cudaStream_t stream);
lora_status_t simt_dh(float *dH, const void *dY, const lora_adapter_table &tab,
                      const lora_segments &segs, cudaStream_t stream);
lora_status_t simt_expand(void *y, const float *H, const lora_adapter_table &tab,
                          const lora_segments &segs, cudaStream_t stream);
lora_status_t simt_dx(void *dX, const float *dH, const lora_adapter_table &tab,
                      const lora_segments &segs, cudaStream_t stream);
lora_status_t simt_db(float *dB, const void *dY, const float *H, const lora_adapter_table &tab,
                      const lora_segments &segs, cudaStream_t stream);
lora_status_t simt_da(float *dA, const float *dH, const void *X, const lora_adapter_table &tab,
                      const lora_segments &segs, cudaStream_t stream);

}  // namespace lora
