// dispatch.cu -- the sequence of kernels behind each entry point.
//
//   forward:  case i (shrink) writes H (optional fp32 copy for the caller) and
//             its bf16 hi + lo split in perm order; case ii (expand) reads them.
//   backward: a small kernel converts the saved H to bf16 in perm order (or
//             case i recomputes it from X); case i (dh) writes bf16 dH in perm
//             order; case iii (dB), case iv (dA) and case ii (dX) read those.
#include "dispatch.h"
#include "tc_host.h"

namespace lora {

size_t handoff_region_bytes(int32_t T, int32_t r_max)
{
    const int64_t b = (int64_t)T * handoff_cols(r_max) * 2;
    return (size_t)((b + 255) & ~int64_t(255));
}

// batches up to this many tokens take the decode kernels
constexpr int32_t kDecodeMaxTokens = 512;

// Work-claim counters, 256 bytes after the two hand-off regions: one int per
// claiming launch of a call.  The kernel before a claiming one on the same
// stream zeroes its counter (forward: the shrink zeroes the expand's;
// backward: the bf16 copy of H, or the recomputing shrink, zeroes dB's, and
// dh zeroes dA's and dX's), so no memset is needed.  Items are claimed at run
// time when their costs differ (id-routed batches: gathered and TMA tiles,
// tiles and spans of any length) and in the ordered backward (whose waits
// rely on it); the uniform items of segment-sorted batches are split evenly
// ahead of time (CTA b takes b, b + grid, ...), which ends every CTA's share
// together where run-time claims would leave the last items to CTAs that are
// still finishing others.
constexpr size_t kClaimRegionBytes = 256;
enum ClaimSlot { kClaimExpand = 0, kClaimDB = 1, kClaimDA = 2, kClaimDX = 3 };

size_t ticket_region_bytes(const lora_adapter_table &tab, int32_t T)
{
    const SegLayout L = seg_layout(T, tab.n_adapters);
    if (!L.ok) return 0;
    const int64_t words = (int64_t)L.max_spans * (tokred_ranges(tab.d_out) + tokred_ranges(tab.d_in));
    return (size_t)((words * 4 + 255) & ~int64_t(255));
}

namespace {
// the claim counters, when the workspace holds them (null: items by CTA index)
int32_t *claim_region(void *ws, size_t ws_bytes, int32_t T, int32_t r_max)
{
    const size_t off = 2 * handoff_region_bytes(T, r_max);
    if (ws_bytes < off + kClaimRegionBytes) return nullptr;
    return reinterpret_cast<int32_t *>(static_cast<char *>(ws) + off);
}
}  // namespace

size_t part_region_bytes(const lora_adapter_table &tab, int32_t T)
{
    const SegLayout L = seg_layout(T, tab.n_adapters);
    if (!L.ok) return 0;
    const int32_t a = rowproj_splits(L.max_tiles, tab.d_in), b = rowproj_splits(L.max_tiles, tab.d_out);
    const int32_t sp = a > b ? a : b;
    if (sp <= 1) return 0;
    const int64_t bytes = (int64_t)sp * T * rowproj_part_ld(tab.r_max) * 4;
    return (size_t)((bytes + 255) & ~int64_t(255));
}

namespace {
// case i's partials in the workspace, when the workspace holds them
float *part_region(void *ws, size_t ws_bytes, const lora_adapter_table &tab, int32_t T)
{
    const size_t off = 2 * handoff_region_bytes(T, tab.r_max) + kClaimRegionBytes + ticket_region_bytes(tab, T);
    const size_t need = part_region_bytes(tab, T);
    if (need == 0 || ws_bytes < off + need) return nullptr;
    return reinterpret_cast<float *>(static_cast<char *>(ws) + off);
}
}  // namespace

size_t bwd_workspace_bytes(const lora_adapter_table &tab, int32_t T)
{
    return 2 * handoff_region_bytes(T, tab.r_max) + kClaimRegionBytes + ticket_region_bytes(tab, T) +
           part_region_bytes(tab, T);
}

size_t packed_workspace_bytes(const lora_adapter_table &tab, int32_t T)
{
    const size_t packed = bwd_workspace_bytes(tab, T);
    const size_t decode = T <= kDecodeMaxTokens ? decode_workspace_bytes(T, tab.r_max, tab.d_in) : 0;
    return packed > decode ? packed : decode;
}

lora_status_t run_shrink(float *H, const void *x, const lora_adapter_table &tab, const lora_segments &segs,
                         cudaStream_t stream)
{
    return tc_shrink(x, tab, segs, H, nullptr, nullptr, 0, nullptr, nullptr, 0, nullptr, 0, stream);  // not split
}

lora_status_t run_expand(void *y, const float *H, const lora_adapter_table &tab, const lora_segments &segs,
                         cudaStream_t stream)
{
    return tc_expand_f32(y, H, tab, segs, stream);
}

namespace {

void mark(Marks *m, cudaStream_t stream)
{
    if (m != nullptr && m->k < m->n) cudaEventRecord(static_cast<cudaEvent_t>(m->ev[m->k++]), stream);
}

// launch `f` between a pair of marks
template <class F>
lora_status_t marked(Marks *m, cudaStream_t stream, F f)
{
    mark(m, stream);
    const lora_status_t st = f();
    mark(m, stream);
    return st;
}

}  // namespace

lora_status_t run_fwd(void *y, float *H_save, const void *x, void *ws, size_t ws_bytes, const lora_adapter_table &tab,
                      const lora_segments &segs, cudaStream_t stream, Marks *marks)
{
    if (segs.n_tokens <= kDecodeMaxTokens)  // one pair of marks around both decode launches
        return marked(marks, stream, [&] { return tc_decode_fwd(y, H_save, x, ws, tab, segs, stream); });
    const int32_t rw = handoff_cols(tab.r_max);
    uint16_t *hi = static_cast<uint16_t *>(ws);
    uint16_t *lo = reinterpret_cast<uint16_t *>(static_cast<char *>(ws) + handoff_region_bytes(segs.n_tokens, tab.r_max));
    float *part = part_region(ws, ws_bytes, tab, segs.n_tokens);
    int32_t *claims = claim_region(ws, ws_bytes, segs.n_tokens, tab.r_max);
    int32_t *c_expand = claims != nullptr ? claims + kClaimExpand : nullptr;
    lora_status_t st = marked(
        marks, stream,
        [&] { return tc_shrink(x, tab, segs, H_save, hi, lo, rw, part, c_expand, 1, nullptr, 0, stream); });
    if (st != LORA_OK) return st;
    int32_t *use = segs.sorted != 0 ? nullptr : c_expand;
    return marked(marks, stream, [&] { return tc_expand_bf16(y, hi, lo, rw, use, tab, segs, stream); });
}

size_t multi_workspace_bytes(int32_t n_proj, const lora_adapter_table *tabs, int32_t T)
{
    size_t need = 0;
    int32_t r_max = 0;
    for (int32_t p = 0; p < n_proj; ++p) {
        r_max = tabs[p].r_max > r_max ? tabs[p].r_max : r_max;
        const size_t one = packed_workspace_bytes(tabs[p], T);  // the per-projection path
        need = one > need ? one : need;
    }
    if (T <= kDecodeMaxTokens) {  // the shared decode launches: one h buffer per projection
        const size_t dec = (size_t)n_proj * decode_workspace_bytes(T, r_max, tabs[0].d_in);
        need = dec > need ? dec : need;
    }
    return need;
}

lora_status_t run_multi_fwd(int32_t n_proj, void *const *y, float *const *H_save, const void *x, void *ws,
                            size_t ws_bytes, const lora_adapter_table *tabs, const lora_segments &segs,
                            cudaStream_t stream)
{
    if (segs.n_tokens <= kDecodeMaxTokens) return tc_decode_multi(n_proj, y, H_save, x, ws, tabs, segs, stream);
    for (int32_t p = 0; p < n_proj; ++p) {  // large batches: the packed kernels, one projection after another
        const lora_status_t st =
            run_fwd(y[p], H_save != nullptr ? H_save[p] : nullptr, x, ws, ws_bytes, tabs[p], segs, stream, nullptr);
        if (st != LORA_OK) return st;
    }
    return LORA_OK;
}

lora_status_t run_bwd(void *dX, float *dA, float *dB, const void *dY, const void *X, const float *H_saved, void *ws,
                      size_t ws_bytes, const lora_adapter_table &tab, const lora_segments &segs, cudaStream_t stream,
                      Marks *marks, const SideStreams *side, bool ordered)
{
    const int32_t rw = handoff_cols(tab.r_max);
    const size_t hreg = handoff_region_bytes(segs.n_tokens, tab.r_max);
    uint16_t *hb = static_cast<uint16_t *>(ws);
    uint16_t *dhb = reinterpret_cast<uint16_t *>(static_cast<char *>(ws) + hreg);
    float *part = part_region(ws, ws_bytes, tab, segs.n_tokens);  // case i split along d (few tiles)
    int32_t *claims = claim_region(ws, ws_bytes, segs.n_tokens, tab.r_max);
    auto claim = [&](ClaimSlot k) { return claims != nullptr ? claims + k : nullptr; };
    // the counters the launches claim from (null: items split ahead of time)
    const bool dyn = segs.sorted == 0;
    auto use = [&](ClaimSlot k, bool on) { return on ? claim(k) : nullptr; };
    // ordered mode: tickets of dB, then of dA, after the claim counters
    int32_t *tk_B = nullptr, *tk_A = nullptr;
    if (ordered && (dA != nullptr || dB != nullptr)) {
        if (claims == nullptr) return LORA_ERR_WORKSPACE_TOO_SMALL;
        tk_B = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + 2 * hreg + kClaimRegionBytes);
        tk_A = tk_B + (int64_t)segs.max_spans * tokred_ranges(tab.d_out);
        if (cudaMemsetAsync(tk_B, 0, ticket_region_bytes(tab, segs.n_tokens), stream) != cudaSuccess)
            return LORA_ERR_CUDA;
    }
    // dA and dB are sums over token spans added into zeroed outputs.  dA is
    // cleared by dh, the kernel before it (its full grid zeroes it in a few
    // us, where a separate memset launch would sit on the critical path).  dB
    // is cleared the same way by the kernel before it on its stream (the
    // small bf16 copy of H, or the recomputing shrink) when it is small; a
    // large dB goes to a memset at the start, faster than that small grid.
    // With no tokens no kernel runs: memsets.
    const int64_t nB = (int64_t)tab.sum_r * tab.d_out, nA = (int64_t)tab.sum_r * tab.d_in;
    const bool empty = segs.n_tokens == 0 || segs.max_tiles == 0;
    constexpr int64_t kFoldMaxFloats = (int64_t)4 << 20;  // 16 MB
    float *zero_B = dB != nullptr && !empty && nB <= kFoldMaxFloats ? dB : nullptr;
    if (dB != nullptr && zero_B == nullptr &&
        cudaMemsetAsync(dB, 0, (size_t)nB * sizeof(float), stream) != cudaSuccess)
        return LORA_ERR_CUDA;
    if (dA != nullptr && empty && cudaMemsetAsync(dA, 0, (size_t)nA * sizeof(float), stream) != cudaSuccess)
        return LORA_ERR_CUDA;
    lora_status_t st = LORA_OK;
    // dB needs only dY and the bf16 rows of H, so with side streams it runs
    // beside case i (dh); dA and dX need dh.  Side stream 0: [H to bf16], dB;
    // the caller's stream: [the shrink, when H is not saved], dh, dX; side
    // stream 1: dA after dh.  Without side streams (and in a marked call, so
    // that each event pair brackets one kernel alone) everything runs one
    // after another on the caller's stream.
    const bool par = side != nullptr && marks == nullptr && (dB != nullptr || dA != nullptr);
    cudaStream_t sB = par ? side->s[0] : stream, sA = par ? side->s[1] : stream;
    // fork: the side stream waits for what the caller's stream has issued so far
    auto fork = [&](cudaEvent_t ev, cudaStream_t on) {
        return cudaEventRecord(ev, stream) == cudaSuccess && cudaStreamWaitEvent(on, ev, 0) == cudaSuccess;
    };
    bool forked_B = false, forked_A = false;
    if (H_saved == nullptr)
        st = marked(marks, stream, [&] {
            return tc_shrink(X, tab, segs, nullptr, hb, nullptr, rw, part, claim(kClaimDB), 1, zero_B, nB, stream);
        });
    if (st == LORA_OK && par && dB != nullptr) {  // fork B once the outputs are zeroed (and H recomputed)
        forked_B = fork(side->ev[0], sB);
        if (!forked_B) st = LORA_ERR_CUDA;
    }
    if (st == LORA_OK && dB != nullptr) {
        if (H_saved != nullptr)
            st = marked(marks, sB,
                        [&] { return tc_h_to_bf16(H_saved, hb, rw, claim(kClaimDB), 1, zero_B, nB, tab, segs, sB); });
        if (st == LORA_OK)
            st = marked(marks, sB, [&] { return tc_db(dB, dY, hb, rw, tk_B, use(kClaimDB, dyn || ordered), tab, segs, sB); });
    }
    if (st == LORA_OK)
        st = marked(marks, stream,
                    [&] { return tc_dh(dY, tab, segs, dhb, rw, part, claim(kClaimDA), 2, dA, nA, stream); });
    if (st == LORA_OK && par && dA != nullptr) {  // fork A after dh
        forked_A = fork(side->ev[3], sA);
        if (!forked_A) st = LORA_ERR_CUDA;
    }
    if (st == LORA_OK && dA != nullptr)
        st = marked(marks, sA, [&] { return tc_da(dA, X, dhb, rw, tk_A, use(kClaimDA, dyn || ordered), tab, segs, sA); });
    if (st == LORA_OK && dX != nullptr)
        st = marked(marks, stream, [&] { return tc_dx(dX, dhb, rw, use(kClaimDX, dyn), tab, segs, stream); });
    // join: the caller's stream waits for every side stream that was forked,
    // after an error too, so that no work of this call outlives it unordered
    // with the caller's stream (and a capture is never left with an open fork)
    auto join = [&](cudaEvent_t ev, cudaStream_t on) {
        return cudaEventRecord(ev, on) == cudaSuccess && cudaStreamWaitEvent(stream, ev, 0) == cudaSuccess;
    };
    if (forked_B && !join(side->ev[1], sB) && st == LORA_OK) st = LORA_ERR_CUDA;
    if (forked_A && !join(side->ev[2], sA) && st == LORA_OK) st = LORA_ERR_CUDA;
    return st;
}

}  // namespace lora
