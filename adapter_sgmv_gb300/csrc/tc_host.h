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
// Row-major fp32 matrix [rows, cols] as a 2-D TMA tensor (no swizzle), box [box_rows, box_cols].
// Three tensor maps over one weight matrix ([sum_r, d] bf16, 128-byte swizzle,
// 64 columns wide) with boxes of 16, 32 and 64 rows: rp rows are fetched with
// as few boxes as possible (64-row boxes first), so that one stage of a rank
// 128 adapter takes two TMA copies instead of eight.
struct WMaps {
    CUtensorMap m16, m32, m64;
};
bool make_wmaps(WMaps *maps, const void *base, uint64_t cols, uint64_t rows);

// A bf16 [rows, cols] row-major matrix (cols a multiple of 64) seen as 3-D
// (64 columns, rows, cols / 64 column blocks), 128-byte swizzle: one box of
// {64, box_rows, box_blocks} lands as box_blocks consecutive [box_rows x 128 B]
// swizzled blocks, i.e. as box_blocks separate 2-D boxes would.
bool make_tmap_bf16_blocks(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows,
                           uint32_t box_blocks);

bool make_tmap_f32_2d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
                      uint32_t box_rows);
int sm_count();

// Hand-off buffers between the kernels: bf16 [T, rw] rows in perm order (the
// position of the token in its adapter's group), zero from each adapter's rank
// up to the rank rounded to 16, unwritten past that (no product reads there).
inline int32_t handoff_cols(int32_t r_max) { return r_max <= 64 ? 64 : 128; }

// case i.  shrink: H[t, :] = A_i x_t.  Writes the fp32 H by token (H may be
// null; zero past r_i) and/or its bf16 hi (+ lo) split by perm position (null
// to skip; zero from r_i up to r_i rounded to 16, unwritten past that, where
// no product reads).
// part: null, or rowproj_splits(max_tiles, d) x T x rowproj_part_ld(r_max)
// floats of scratch, with which a batch of few tiles is cut along d into
// parts whose partials a second small kernel adds.
// zero_claims: null, or n_zero work-claim counters of kernels that follow on
// the same stream in the same call, set to zero before anything else.
// zero_out: null, or zero_out_n floats (16-byte aligned, a multiple of 4)
// that a later kernel of the call adds into, set to zero by the whole grid.
lora_status_t tc_shrink(const void *x, const lora_adapter_table &tab, const lora_segments &segs, float *H,
                        uint16_t *hi, uint16_t *lo, int32_t rw, float *part, int32_t *zero_claims, int32_t n_zero,
                        float *zero_out, int64_t zero_out_n, cudaStream_t stream);
// case i.  dh = s_i B_i^T dy as bf16 by perm position.
lora_status_t tc_dh(const void *dY, const lora_adapter_table &tab, const lora_segments &segs, uint16_t *dh_bf16,
                    int32_t rw, float *part, int32_t *zero_claims, int32_t n_zero, float *zero_out,
                    int64_t zero_out_n, cudaStream_t stream);
int32_t rowproj_splits(int32_t max_tiles, int32_t d);
int32_t rowproj_part_ld(int32_t r_max);

// A saved fp32 H (by token) converted to the bf16 hand-off rows (by perm
// position) that cases iii reads; the same values case i writes as its hi.
lora_status_t tc_h_to_bf16(const float *H, uint16_t *hb, int32_t rw, int32_t *zero_claims, int32_t n_zero,
                           float *zero_out, int64_t zero_out_n, const lora_adapter_table &tab,
                           const lora_segments &segs, cudaStream_t stream);
// case ii.  y += s_i B_i h from the bf16 hand-off buffers (lo may be null).
// claim: null (CTA b takes items b, b + grid, ...) or a counter that is zero
// when the kernel starts, from which items are claimed at run time.
lora_status_t tc_expand_bf16(void *y, const uint16_t *hi, const uint16_t *lo, int32_t rw, int32_t *claim,
                             const lora_adapter_table &tab, const lora_segments &segs, cudaStream_t stream);
// case ii.  y += s_i B_i h from an fp32 H by token (converted in the kernel).
lora_status_t tc_expand_f32(void *y, const float *H, const lora_adapter_table &tab, const lora_segments &segs,
                            cudaStream_t stream);
// case ii.  dX += A_i^T dh from the bf16 hand-off buffer.
lora_status_t tc_dx(void *dX, const uint16_t *dh_bf16, int32_t rw, int32_t *claim, const lora_adapter_table &tab,
                    const lora_segments &segs, cudaStream_t stream);

// cases iii / iv, output [sum_r, d] accumulated into (the caller zeroes it):
// dB[row_off + k, o] and dA[row_off + k, j].  tickets: null, or
// tokred_ranges(d) x segs.max_spans zeroed ints for the ordered mode (each
// adapter's span partials added in span order: bit-reproducible sums).
// claim: as for case ii.
int32_t tokred_ranges(int32_t d);
lora_status_t tc_db(float *dB, const void *dY, const uint16_t *h_bf16, int32_t rw, int32_t *tickets, int32_t *claim,
                    const lora_adapter_table &tab, const lora_segments &segs, cudaStream_t stream);
lora_status_t tc_da(float *dA, const void *X, const uint16_t *dh_bf16, int32_t rw, int32_t *tickets, int32_t *claim,
                    const lora_adapter_table &tab, const lora_segments &segs, cudaStream_t stream);

// decode-sized batches: the shrink split over d_in, one CTA per (tile, slice),
// its fp32 partials in ws, then the expand as a programmatic dependent launch
// that adds them; H_save may be null.  ws: decode_workspace_bytes(T, r_max,
// d_in) bytes.
constexpr int32_t kDecodeSlices = 16;  // most slices of d_in
constexpr int32_t kMaxProjections = LORA_MAX_PROJECTIONS;
size_t decode_workspace_bytes(int32_t T, int32_t r_max, int32_t d_in);
lora_status_t tc_decode_fwd(void *y, float *H_save, const void *x, void *ws, const lora_adapter_table &tab,
                            const lora_segments &segs, cudaStream_t stream);
// n_proj projections reading the same x in the same two launches (tables
// share d_in and the adapter count); H_save may be null, or hold null entries.
// ws: n_proj * decode_workspace_bytes(T, largest r_max, d_in) bytes.
lora_status_t tc_decode_multi(int32_t n_proj, void *const *y, float *const *H_save, const void *x, void *ws,
                              const lora_adapter_table *tabs, const lora_segments &segs, cudaStream_t stream);

// Base projection plus packed delta in one persistent launch (segment-sorted
// batches): y = x W^T + s_i (x A_i^T) B_i^T, H (fp32, may be null) = x A_i^T.
// ws: base_workspace_bytes(T, r_max, segs.max_tiles) bytes.
size_t base_workspace_bytes(int32_t T, int32_t r_max, int32_t max_tiles);
lora_status_t tc_base_fwd(void *y, float *H, const void *x, const void *W, void *ws, const lora_adapter_table &tab,
                          const lora_segments &segs, cudaStream_t stream);

}  // namespace lora
