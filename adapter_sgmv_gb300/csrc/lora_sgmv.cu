// lora_sgmv.cu -- the C ABI: argument checks, workspace layout and dispatch.
//
// Every entry point validates its arguments on the host before touching the
// GPU, then enqueues its kernels on the caller's stream.  Nothing here
// allocates, frees or synchronises (lora_query_status excepted).
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "dispatch.h"
#include "tc_host.h"

using namespace lora;

namespace lora {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

lora_status_t check_table(const lora_adapter_table *t)
{
    if (t == nullptr) return LORA_ERR_INVALID_ARG;
    if (t->rank == nullptr || t->row_off == nullptr || t->scale == nullptr || t->A == nullptr ||
        t->B == nullptr)
        return LORA_ERR_INVALID_ARG;
    if (t->n_adapters < 1 || t->n_adapters > kMaxAdapters) return LORA_ERR_SHAPE;
    if (t->d_in < 8 || t->d_in > kMaxDim || (t->d_in % 8) != 0) return LORA_ERR_SHAPE;
    if (t->d_out < 8 || t->d_out > kMaxDim || (t->d_out % 8) != 0) return LORA_ERR_SHAPE;
    if (t->r_max < 1 || t->r_max > LORA_MAX_RANK) return LORA_ERR_SHAPE;
    if (t->sum_r < t->r_max || (int64_t)t->sum_r > (int64_t)t->n_adapters * t->r_max) return LORA_ERR_SHAPE;
    if (!aligned16(t->A) || !aligned16(t->B) || !aligned4(t->rank) || !aligned4(t->row_off) ||
        !aligned4(t->scale))
        return LORA_ERR_ALIGNMENT;
    return LORA_OK;
}

// Every pointer the kernels dereference must be present: the tile and span
// counts are read on the device before anything else.
lora_status_t check_segs(const lora_segments *s, const lora_adapter_table *t)
{
    if (s == nullptr) return LORA_ERR_INVALID_ARG;
    if (s->perm == nullptr || s->seg_start == nullptr || s->tiles == nullptr || s->n_tiles == nullptr ||
        s->status == nullptr || s->spans == nullptr || s->n_spans == nullptr)
        return LORA_ERR_INVALID_ARG;
    if (s->n_tokens < 0 || s->n_tokens > kMaxTokens || s->n_adapters < 1 || s->max_tiles < 0 || s->max_spans < 0)
        return LORA_ERR_SHAPE;
    if (t != nullptr && s->n_adapters != t->n_adapters) return LORA_ERR_SHAPE;
    if (!aligned4(s->perm) || !aligned4(s->seg_start) || !aligned16(s->tiles) || !aligned16(s->spans) ||
        !aligned4(s->n_tiles) || !aligned4(s->n_spans) || !aligned4(s->status))
        return LORA_ERR_ALIGNMENT;
    return LORA_OK;
}

lora_status_t check_device()
{
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LORA_ERR_CUDA;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return LORA_ERR_CUDA;
    if (major != 10 || minor != 3) return LORA_ERR_UNSUPPORTED;  // built for sm_103a only
    return LORA_OK;
}

}  // namespace lora

namespace {

size_t workspace_bytes(const lora_adapter_table *t, int32_t T) { return packed_workspace_bytes(*t, T); }


#define LORA_TRY(expr)                          \
    do {                                        \
        lora_status_t _st = (expr);             \
        if (_st != LORA_OK) return _st;         \
    } while (0)

lora_status_t packed_fwd(void *y, float *H_save, const void *x, const lora_adapter_table *table,
                         const lora_segments *segs, void *ws, size_t ws_bytes, lora_stream_t stream, Marks *marks)
{
    LORA_TRY(check_table(table));
    LORA_TRY(check_segs(segs, table));
    if (y == nullptr || x == nullptr) return LORA_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(x) || (H_save && !aligned16(H_save)) || (ws && !aligned16(ws)))
        return LORA_ERR_ALIGNMENT;
    const size_t need = workspace_bytes(table, segs->n_tokens);
    if (need > 0 && (ws == nullptr || ws_bytes < need)) return LORA_ERR_WORKSPACE_TOO_SMALL;
    LORA_TRY(check_device());
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return run_fwd(y, H_save, x, ws, ws_bytes, *table, *segs, st, marks);
}

lora_status_t packed_bwd(void *dX, float *dA, float *dB, const void *dY, const void *X, const float *H_saved,
                         const lora_adapter_table *table, const lora_segments *segs, void *ws, size_t ws_bytes,
                         lora_stream_t stream, Marks *marks, const SideStreams *side = nullptr, bool ordered = false)
{
    LORA_TRY(check_table(table));
    LORA_TRY(check_segs(segs, table));
    if (dY == nullptr || X == nullptr) return LORA_ERR_INVALID_ARG;
    if (!aligned16(dY) || !aligned16(X) || (dX && !aligned16(dX)) || (dA && !aligned16(dA)) ||
        (dB && !aligned16(dB)) || (H_saved && !aligned16(H_saved)) || (ws && !aligned16(ws)))
        return LORA_ERR_ALIGNMENT;
    const size_t need = workspace_bytes(table, segs->n_tokens);
    if (need > 0 && (ws == nullptr || ws_bytes < need)) return LORA_ERR_WORKSPACE_TOO_SMALL;
    LORA_TRY(check_device());
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return run_bwd(dX, dA, dB, dY, X, H_saved, ws, ws_bytes, *table, *segs, st, marks, side, ordered);
}

// the caller's side streams and events, checked: distinct, none of them `stream`
lora_status_t side_streams_of(const lora_side_streams *side, lora_stream_t stream, SideStreams *out)
{
    SideStreams &sd = *out;
    for (int i = 0; i < 2; ++i) {
        if (side->stream[i] == nullptr || side->stream[i] == stream) return LORA_ERR_INVALID_ARG;
        sd.s[i] = reinterpret_cast<cudaStream_t>(side->stream[i]);
    }
    if (side->stream[0] == side->stream[1]) return LORA_ERR_INVALID_ARG;
    for (int i = 0; i < 4; ++i) {
        if (side->event[i] == nullptr) return LORA_ERR_INVALID_ARG;
        for (int j = 0; j < i; ++j)
            if (side->event[j] == side->event[i]) return LORA_ERR_INVALID_ARG;
        sd.ev[i] = static_cast<cudaEvent_t>(side->event[i]);
    }
    return LORA_OK;
}

}  // namespace

extern "C" {

int32_t lora_abi_version(void) { return LORA_SGMV_ABI_VERSION; }

const char *lora_status_string(lora_status_t s)
{
    switch (s) {
    case LORA_OK: return "LORA_OK";
    case LORA_ERR_INVALID_ARG: return "LORA_ERR_INVALID_ARG";
    case LORA_ERR_SHAPE: return "LORA_ERR_SHAPE";
    case LORA_ERR_ALIGNMENT: return "LORA_ERR_ALIGNMENT";
    case LORA_ERR_BAD_ADAPTER_ID: return "LORA_ERR_BAD_ADAPTER_ID";
    case LORA_ERR_WORKSPACE_TOO_SMALL: return "LORA_ERR_WORKSPACE_TOO_SMALL";
    case LORA_ERR_UNSUPPORTED: return "LORA_ERR_UNSUPPORTED";
    case LORA_ERR_TIMEOUT: return "LORA_ERR_TIMEOUT";
    case LORA_ERR_BAD_TABLE: return "LORA_ERR_BAD_TABLE";
    case LORA_ERR_BAD_SEGMENTS: return "LORA_ERR_BAD_SEGMENTS";
    case LORA_ERR_CUDA: return "LORA_ERR_CUDA";
    case LORA_ERR_INDEX: return "LORA_ERR_INDEX";
    }
    return "LORA_ERR_UNKNOWN";
}

size_t lora_segments_bytes(int32_t n_tokens, int32_t n_adapters)
{
    const SegLayout L = seg_layout(n_tokens, n_adapters);
    return L.ok ? (size_t)L.total_words * 4 : 0;
}

lora_status_t lora_build_segments(const int32_t *ids, const int32_t *seg_offsets, int32_t n_tokens,
                                  int32_t n_adapters, void *storage, size_t storage_bytes,
                                  lora_segments *out, lora_stream_t stream)
{
    if (out == nullptr || storage == nullptr) return LORA_ERR_INVALID_ARG;
    if (n_tokens < 0 || n_adapters < 1) return LORA_ERR_SHAPE;
    if ((ids == nullptr) == (seg_offsets == nullptr) && !(n_tokens == 0 && seg_offsets == nullptr))
        return LORA_ERR_INVALID_ARG;
    if (!aligned16(storage) || (ids && !aligned4(ids)) || (seg_offsets && !aligned4(seg_offsets)))
        return LORA_ERR_ALIGNMENT;
    const SegLayout L = seg_layout(n_tokens, n_adapters);
    if (!L.ok) return LORA_ERR_SHAPE;
    if ((size_t)L.total_words * 4 > storage_bytes) return LORA_ERR_WORKSPACE_TOO_SMALL;
    LORA_TRY(check_device());
    return build_segments(ids, seg_offsets, n_tokens, n_adapters, storage, storage_bytes, out,
                          reinterpret_cast<cudaStream_t>(stream));
}

size_t lora_workspace_bytes(const lora_adapter_table *table, int32_t n_tokens)
{
    if (check_table(table) != LORA_OK || n_tokens < 0 || n_tokens > kMaxTokens) return 0;
    return workspace_bytes(table, n_tokens);
}

lora_status_t lora_sgmv_shrink(float *H, const void *x, const lora_adapter_table *table,
                               const lora_segments *segs, lora_stream_t stream)
{
    LORA_TRY(check_table(table));
    LORA_TRY(check_segs(segs, table));
    if (H == nullptr || x == nullptr) return LORA_ERR_INVALID_ARG;
    if (!aligned16(H) || !aligned16(x)) return LORA_ERR_ALIGNMENT;
    LORA_TRY(check_device());
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return run_shrink(H, x, *table, *segs, st);
}

lora_status_t lora_sgmv_expand(void *y, const float *H, const lora_adapter_table *table,
                               const lora_segments *segs, lora_stream_t stream)
{
    LORA_TRY(check_table(table));
    LORA_TRY(check_segs(segs, table));
    if (H == nullptr || y == nullptr) return LORA_ERR_INVALID_ARG;
    if (!aligned16(H) || !aligned16(y)) return LORA_ERR_ALIGNMENT;
    LORA_TRY(check_device());
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return run_expand(y, H, *table, *segs, st);
}

lora_status_t lora_packed_fwd(void *y, float *H_save, const void *x, const lora_adapter_table *table,
                              const lora_segments *segs, void *ws, size_t ws_bytes, lora_stream_t stream)
{
    return packed_fwd(y, H_save, x, table, segs, ws, ws_bytes, stream, nullptr);
}

lora_status_t lora_packed_bwd(void *dX, float *dA, float *dB, const void *dY, const void *X,
                              const float *H_saved, const lora_adapter_table *table,
                              const lora_segments *segs, void *ws, size_t ws_bytes, lora_stream_t stream)
{
    return packed_bwd(dX, dA, dB, dY, X, H_saved, table, segs, ws, ws_bytes, stream, nullptr);
}

lora_status_t lora_side_streams_destroy(lora_side_streams *side)
{
    if (side == nullptr) return LORA_ERR_INVALID_ARG;
    bool ok = true;
    for (auto &st : side->stream) {
        if (st != nullptr && cudaStreamDestroy(reinterpret_cast<cudaStream_t>(st)) != cudaSuccess) ok = false;
        st = nullptr;
    }
    for (auto &ev : side->event) {
        if (ev != nullptr && cudaEventDestroy(static_cast<cudaEvent_t>(ev)) != cudaSuccess) ok = false;
        ev = nullptr;
    }
    return ok ? LORA_OK : LORA_ERR_CUDA;
}

lora_status_t lora_side_streams_create(lora_side_streams *side)
{
    if (side == nullptr) return LORA_ERR_INVALID_ARG;
    *side = lora_side_streams{};
    for (auto &st : side->stream) {
        cudaStream_t s = nullptr;
        if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) {
            cudaGetLastError();
            lora_side_streams_destroy(side);
            return LORA_ERR_CUDA;
        }
        st = reinterpret_cast<lora_stream_t>(s);
    }
    for (auto &ev : side->event) {
        cudaEvent_t e = nullptr;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            lora_side_streams_destroy(side);
            return LORA_ERR_CUDA;
        }
        ev = e;
    }
    return LORA_OK;
}

lora_status_t lora_packed_bwd_concurrent(void *dX, float *dA, float *dB, const void *dY, const void *X,
                                         const float *H_saved, const lora_adapter_table *table,
                                         const lora_segments *segs, void *ws, size_t ws_bytes,
                                         const lora_side_streams *side, lora_stream_t stream)
{
    if (side == nullptr) return LORA_ERR_INVALID_ARG;
    SideStreams sd;
    LORA_TRY(side_streams_of(side, stream, &sd));
    return packed_bwd(dX, dA, dB, dY, X, H_saved, table, segs, ws, ws_bytes, stream, nullptr, &sd);
}

lora_status_t lora_packed_bwd_ex(void *dX, float *dA, float *dB, const void *dY, const void *X, const float *H_saved,
                                 const lora_adapter_table *table, const lora_segments *segs, void *ws,
                                 size_t ws_bytes, const lora_side_streams *side, uint32_t flags, lora_stream_t stream)
{
    if ((flags & ~(uint32_t)LORA_BWD_DETERMINISTIC) != 0) return LORA_ERR_INVALID_ARG;
    SideStreams sd;
    if (side != nullptr) LORA_TRY(side_streams_of(side, stream, &sd));
    return packed_bwd(dX, dA, dB, dY, X, H_saved, table, segs, ws, ws_bytes, stream, nullptr,
                      side != nullptr ? &sd : nullptr, (flags & LORA_BWD_DETERMINISTIC) != 0);
}

lora_status_t lora_packed_fwd_marked(void *y, float *H_save, const void *x, const lora_adapter_table *table,
                                     const lora_segments *segs, void *ws, size_t ws_bytes, lora_stream_t stream,
                                     void *const *events, int32_t n_events, int32_t *n_recorded)
{
    if (n_events < 0 || (n_events > 0 && events == nullptr)) return LORA_ERR_INVALID_ARG;
    Marks m{events, n_events, 0};
    const lora_status_t st = packed_fwd(y, H_save, x, table, segs, ws, ws_bytes, stream, &m);
    if (n_recorded != nullptr) *n_recorded = m.k;
    return st;
}

lora_status_t lora_packed_bwd_marked(void *dX, float *dA, float *dB, const void *dY, const void *X,
                                     const float *H_saved, const lora_adapter_table *table,
                                     const lora_segments *segs, void *ws, size_t ws_bytes, lora_stream_t stream,
                                     void *const *events, int32_t n_events, int32_t *n_recorded)
{
    if (n_events < 0 || (n_events > 0 && events == nullptr)) return LORA_ERR_INVALID_ARG;
    Marks m{events, n_events, 0};
    const lora_status_t st = packed_bwd(dX, dA, dB, dY, X, H_saved, table, segs, ws, ws_bytes, stream, &m);
    if (n_recorded != nullptr) *n_recorded = m.k;
    return st;
}

lora_status_t lora_adamw_step(const lora_adapter_table *table, float *wA, float *wB, const float *gA, const float *gB,
                              float *mA, float *vA, float *mB, float *vB, const float *lr, const int32_t *step,
                              float beta1, float beta2, float eps, float weight_decay, lora_stream_t stream)
{
    LORA_TRY(check_table(table));
    const void *f32[] = {wA, wB, gA, gB, mA, vA, mB, vB};
    for (const void *p : f32) {
        if (p == nullptr) return LORA_ERR_INVALID_ARG;
        if (!aligned16(p)) return LORA_ERR_ALIGNMENT;
    }
    if (lr == nullptr || step == nullptr) return LORA_ERR_INVALID_ARG;
    if (!aligned4(lr) || !aligned4(step)) return LORA_ERR_ALIGNMENT;
    if (!(beta1 >= 0.f && beta1 < 1.f) || !(beta2 >= 0.f && beta2 < 1.f) || !(eps >= 0.f) ||
        !(weight_decay >= 0.f))
        return LORA_ERR_INVALID_ARG;
    LORA_TRY(check_device());
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return run_adamw(*table, wA, wB, gA, gB, mA, vA, mB, vB, lr, step, beta1, beta2, eps, weight_decay, st);
}

size_t lora_multi_workspace_bytes(int32_t n_proj, const lora_adapter_table *tables, int32_t n_tokens)
{
    if (tables == nullptr || n_proj < 1 || n_proj > LORA_MAX_PROJECTIONS || n_tokens < 0 || n_tokens > kMaxTokens)
        return 0;
    for (int32_t p = 0; p < n_proj; ++p)
        if (check_table(&tables[p]) != LORA_OK) return 0;
    return multi_workspace_bytes(n_proj, tables, n_tokens);
}

lora_status_t lora_multi_fwd(int32_t n_proj, void *const *y, float *const *H_save, const void *x,
                             const lora_adapter_table *tables, const lora_segments *segs, void *ws, size_t ws_bytes,
                             lora_stream_t stream)
{
    if (y == nullptr || tables == nullptr || x == nullptr) return LORA_ERR_INVALID_ARG;
    if (n_proj < 1 || n_proj > LORA_MAX_PROJECTIONS) return LORA_ERR_SHAPE;
    for (int32_t p = 0; p < n_proj; ++p) {
        LORA_TRY(check_table(&tables[p]));
        LORA_TRY(check_segs(segs, &tables[p]));
        if (tables[p].d_in != tables[0].d_in) return LORA_ERR_SHAPE;
        if (y[p] == nullptr) return LORA_ERR_INVALID_ARG;
        if (!aligned16(y[p]) || (H_save != nullptr && H_save[p] != nullptr && !aligned16(H_save[p])))
            return LORA_ERR_ALIGNMENT;
    }
    if (!aligned16(x) || (ws && !aligned16(ws))) return LORA_ERR_ALIGNMENT;
    const size_t need = multi_workspace_bytes(n_proj, tables, segs->n_tokens);
    if (need > 0 && (ws == nullptr || ws_bytes < need)) return LORA_ERR_WORKSPACE_TOO_SMALL;
    LORA_TRY(check_device());
    return run_multi_fwd(n_proj, y, H_save, x, ws, ws_bytes, tables, *segs, reinterpret_cast<cudaStream_t>(stream));
}

size_t lora_fused_base_workspace_bytes(const lora_adapter_table *table, int32_t n_tokens)
{
    if (check_table(table) != LORA_OK || n_tokens < 0) return 0;
    const SegLayout L = seg_layout(n_tokens, table->n_adapters);
    return L.ok ? base_workspace_bytes(n_tokens, table->r_max, L.max_tiles) : 0;
}

lora_status_t lora_fused_base_fwd(void *y, float *H_save, const void *x, const void *W,
                                  const lora_adapter_table *table, const lora_segments *segs, void *ws,
                                  size_t ws_bytes, lora_stream_t stream)
{
    LORA_TRY(check_table(table));
    LORA_TRY(check_segs(segs, table));
    if (y == nullptr || x == nullptr || W == nullptr) return LORA_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(x) || !aligned16(W) || (H_save && !aligned16(H_save)) ||
        (ws && !aligned16(ws)))
        return LORA_ERR_ALIGNMENT;
    if (segs->n_tokens > 0 && segs->sorted == 0) return LORA_ERR_UNSUPPORTED;
    const size_t need = base_workspace_bytes(segs->n_tokens, table->r_max, segs->max_tiles);
    if (segs->n_tokens > 0 && (ws == nullptr || ws_bytes < need)) return LORA_ERR_WORKSPACE_TOO_SMALL;
    LORA_TRY(check_device());
    return tc_base_fwd(y, H_save, x, W, ws, *table, *segs, reinterpret_cast<cudaStream_t>(stream));
}

int32_t lora_debug_checks(void) { return LORA_DEBUG_CHECKS ? 1 : 0; }

lora_status_t lora_query_index_check(const lora_segments *segs, lora_stream_t stream, int32_t *where)
{
    if (segs == nullptr || segs->status == nullptr || where == nullptr) return LORA_ERR_INVALID_ARG;
    int32_t h[2] = {0, 0};
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(h, segs->status, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return LORA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return LORA_ERR_CUDA;
    *where = h[1];
    return static_cast<lora_status_t>(h[0]);
}

lora_status_t lora_query_status(const lora_segments *segs, lora_stream_t stream)
{
    if (segs == nullptr || segs->status == nullptr) return LORA_ERR_INVALID_ARG;
    int32_t h = 0;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&h, segs->status, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return LORA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return LORA_ERR_CUDA;
    return static_cast<lora_status_t>(h);
}

lora_status_t lora_reset_status(const lora_segments *segs, lora_stream_t stream)
{
    if (segs == nullptr || segs->status == nullptr) return LORA_ERR_INVALID_ARG;
    if (cudaMemsetAsync(segs->status, 0, 2 * sizeof(int32_t), reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return LORA_ERR_CUDA;
    return LORA_OK;
}

}  // extern "C"
