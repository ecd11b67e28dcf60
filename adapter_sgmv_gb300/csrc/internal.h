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

// Host-side argument checks shared by the entry points (lora_sgmv.cu,
// noalloc.cu): each returns LORA_OK or the status to report, before anything
// is launched.
bool aligned16(const void *p);
bool aligned4(const void *p);
lora_status_t check_table(const lora_adapter_table *t);
// segs against the table (t may be null to check segs alone)
lora_status_t check_segs(const lora_segments *s, const lora_adapter_table *t);
// the current device is an sm_103 GPU (the library holds code for sm_103a only)
lora_status_t check_device();

}  // namespace lora
