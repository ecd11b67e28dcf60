// tc_tokred.cu -- cases iii and iv on the 5th-generation tensor cores: the
// reductions over tokens that produce the adapters' weight gradients, tiled
// along the hidden dimension and split along tokens (PLoRA technical summary,
// "2. LoRA Execution Engine").
//
//   dB  dB_i[o, k] = s_i sum_{t in i} dY[t, o] H[t, k]   stored at dB[row_off[i] + k, o]
//   dA  dA_i[k, j] =     sum_{t in i} dH[t, k] X[t, j]   stored at dA[row_off[i] + k, j]
//
// One MMA shape serves both: D[n, k] (M = 128 columns n of d, N = r_pad,
// K = tokens) = act^T x h.  The activations are the MN-major A operand read
// as stored (TMA with 128-byte swizzle; cp.async gather for non-consecutive
// tokens), h is the MN-major B operand read by TMA from the perm-ordered bf16
// hand-off buffer the case i kernel wrote (a span's last, partial stage is
// copied with cp.async and zero-filled so that rows past the span add
// nothing).  A work item is (span of <= LORA_SPAN_TOKENS tokens of one
// adapter, 512 columns of d): four TMEM accumulators of up to 128 columns
// accumulate over the span in 32-token stages; the epilogue moves each
// warp's 32 x r_pad block 16 rows at a time through two small shared-memory
// buffers and adds it into the zero-initialised output with TMA bulk
// reductions (spans of an adapter sum).  With the staging that small the
// ring holds five stages, 160 KB of activations in flight per SM.  Segment-
// sorted batches in the default order run a second shape (struct Shape): two
// CTAs per SM, each with three stages of 256-column items and two
// accumulators.
//
// Warp roles (32 (S + 5) threads for S stages): 0..S-1 load, warp w filling
// every stage of ring slot w (a gathered stage's copies are waited for by the
// warp that issued them, which makes them visible to the tensor cores and
// releases the stage at once, so all S stages can be in flight); S MMA + TMEM
// owner; S+1..S+4 epilogue.
#define LORA_DBG_FILE 4
#include "internal.h"
#include "tc_common.cuh"
#include "tc_host.h"

namespace lora {
namespace {

using namespace tc;

constexpr int kTok = 32;                                  // tokens per stage
constexpr uint32_t kBox = kTok * 64 * 2;                  // one [64 x 32] box
constexpr uint32_t kHBytes = 2 * kBox;                    // h: up to 128 columns
constexpr uint32_t kRedBlock = 16 * 32 * 4;  // one reduction box: [16 rows x 32 columns] fp32
constexpr uint32_t kRedBytes = 2 * kRedBlock;  // per epilogue warp: two boxes in turn

// Two shapes.  One CTA per SM: five stages of 32 tokens x 512 columns, four
// TMEM accumulators (512 columns).  Two CTAs per SM (segment-sorted batches in
// the default order): three stages of 32 tokens x 256 columns and two
// accumulators each, so that one CTA's item changes and epilogue are covered
// by the other's loads.
template <bool kTwo>
struct Shape {
    static constexpr int kStages = kTwo ? 3 : 5;
    static constexpr int kProd = kStages;  // producer warps, one per ring slot
    static constexpr int kMmaWarp = kProd;
    static constexpr int kEpi0 = kProd + 1;  // first epilogue warp
    static constexpr int kThreads = 32 * (kProd + 1 + 4);
    static constexpr int kRange = kTwo ? 256 : 512;  // most columns of d per work item
    static constexpr uint32_t kActBytes = kTok * kRange * 2;  // kRange / 64 boxes of [64 cols x 32 tokens]
    static constexpr uint32_t kStageBytes = kActBytes + kHBytes;
    static constexpr uint32_t kTmemCols = kRange;  // one accumulator of up to 128 columns per 128 of d
    static constexpr size_t kSmemBytes = 1024 + kStages * (size_t)kStageBytes + 4 * (size_t)kRedBytes + 256;
};

struct Smem {
    uint8_t *act, *h, *red;
    uint64_t *full, *empty, *tfull, *tempty, *done, *tk_go, *tk_done;
    uint32_t *tmem_holder;
    volatile int32_t *abort;
    ClaimRing claims;  // items claimed at run time
};

template <bool kTwo>
LORA_DEV Smem carve(uint8_t *raw)
{
    constexpr int kStages = Shape<kTwo>::kStages;
    constexpr uint32_t kActBytes = Shape<kTwo>::kActBytes;
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    Smem s;
    s.act = base;
    s.h = base + kStages * kActBytes;
    s.red = s.h + kStages * kHBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(s.red + 4 * kRedBytes);
    s.full = bars;
    s.empty = bars + kStages;
    s.tfull = bars + 2 * kStages;
    s.tempty = s.tfull + 1;
    s.done = s.tempty + 1;
    s.tk_go = s.done + 1;
    s.tk_done = s.tk_go + 1;
    s.tmem_holder = reinterpret_cast<uint32_t *>(s.tk_done + 1);
    s.abort = reinterpret_cast<volatile int32_t *>(s.tmem_holder + 1);
    s.claims.full = reinterpret_cast<uint64_t *>(s.tmem_holder + 8);
    s.claims.empty = s.claims.full + kClaimSlots;
    s.claims.slot = reinterpret_cast<volatile int32_t *>(s.claims.empty + kClaimSlots);
    return s;
}

LORA_DEV int32_t rpad16(int32_t r) { return (r + 15) & ~15; }

struct Item {
    Tile span;
    AdapterInfo ad;
    int32_t n_base, n_chunks, n_stages;
};

LORA_DEV Item load_item(const lora_adapter_table &tab, const lora_segments &segs, int32_t it, int32_t n_ranges,
                        int32_t d, int32_t rng)
{
    Item I;
    I.span = LOAD_SPAN(segs, it / n_ranges);
    I.ad = load_adapter(tab, I.span.adapter, segs.status);
    I.n_base = (it % n_ranges) * rng;
    I.n_chunks = min(rng / 128, (d - I.n_base + 127) / 128);
    I.n_stages = (I.span.rows + kTok - 1) / kTok;
    return I;
}

LORA_DEV void tma_reduce_add_2d(const CUtensorMap *map, const void *smem_src, int32_t c0, int32_t c1)
{
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map),
                 "r"(smem_u32(smem_src)), "r"(c0), "r"(c1)
                 : "memory");
}
LORA_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// orders memory accesses between the generic and the async proxy (all state spaces)
LORA_DEV void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }

// Ordered adds.  An item of the ordered mode adds its span's partial only
// after the partials of the adapter's earlier spans (same column range) are in
// the output: the span's ticket holds the number of spans already added.  The
// wait is bounded like every pipeline wait; on time-out the CTA's abort flag
// and LORA_ERR_TIMEOUT are set.  The ordered mode claims its items at run
// time, in index order, so every item below a claimed one is held by a
// running CTA; an earlier span of the same adapter and range has the lower
// index, and a CTA works through its claims in order, so the unfinished item
// with the lowest index can always proceed.
LORA_DEV bool wait_ticket(const int32_t *tk, int32_t want, volatile int32_t *abort_flag, int32_t *status)
{
    const long long t0 = clock64();
    for (;;) {
        int32_t v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(tk) : "memory");
        if (v == want) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            *abort_flag = 1;
            set_status(status, LORA_ERR_TIMEOUT);
            return false;
        }
        __nanosleep(128);
    }
}
LORA_DEV void release_ticket(int32_t *tk, int32_t v)
{
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(tk), "r"(v) : "memory");
}
// all but the newest bulk group of this thread have read their source
LORA_DEV void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

// kClaim: items claimed at run time from `claim` (id-routed batches and the
// ordered mode), else CTA b takes items b, b + gridDim.x, ...
template <bool kClaim, bool kTwo>
__global__ void __launch_bounds__(Shape<kTwo>::kThreads, kTwo ? 2 : 1)
tc_tokred_kernel(const __grid_constant__ CUtensorMap map_act, const __grid_constant__ CUtensorMap map_act3,
                 const __grid_constant__ CUtensorMap map_h,
                 const __grid_constant__ CUtensorMap map_g, const uint16_t *__restrict__ act, int32_t d,
                 const uint16_t *__restrict__ hbuf, int32_t rw, float use_scale, int32_t blocks3, int32_t rng,
                 int32_t *__restrict__ tickets, int32_t *claim, lora_adapter_table tab, lora_segments segs)
{
    extern __shared__ uint8_t smem_raw[];
    using Sh = Shape<kTwo>;
    constexpr int kStages = Sh::kStages, kProd = Sh::kProd, kMmaWarp = Sh::kMmaWarp, kEpi0 = Sh::kEpi0;
    constexpr uint32_t kActBytes = Sh::kActBytes, kTmemCols = Sh::kTmemCols;
    const Smem S = carve<kTwo>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the claimer's first item, claimed before the set-up so that its round trip overlaps it
    const int32_t first = kClaim && warp == 0 && lane == 0 ? claim_first(claim) : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&S.full[i], 33);
            mbar_init(&S.empty[i], 1);
        }
        mbar_init(S.tfull, 1);
        mbar_init(S.tempty, 4);
        mbar_init(S.done, 1);
        mbar_init(S.tk_go, 1);    // ordered mode: the ticket says the earlier spans are added
        mbar_init(S.tk_done, 4);  // ordered mode: every epilogue warp's adds are complete
        if (kClaim)
            for (int i = 0; i < kClaimSlots; ++i) {  // claimed by producer warp 0, read by the other warps
                mbar_init(&S.claims.full[i], 1);
                mbar_init(&S.claims.empty[i], (kProd - 1) + 1 + 4);
            }
        *S.abort = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(S.tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *S.tmem_holder;
    const int32_t n_ranges = (d + rng - 1) / rng;  // rng: 512 or, when spans are few, 128 columns
    const int32_t n_items = N_SPANS(segs) * n_ranges;

    if (warp < kProd) {
        // ------------------------------------------------------------ producers
        // Stage g of the whole sequence goes to ring slot g % kStages = warp.
        if (lane == 0 && warp == 0) {
            prefetch_tensormap(blocks3 ? &map_act3 : &map_act);
            prefetch_tensormap(&map_h);
        }
        uint32_t g = 0, last = 0xffffffffu;
        bool ok = true;
        uint32_t q = 0;
        for (int32_t it = blockIdx.x; (kClaim || it < n_items) && ok; it += gridDim.x, ++q) {
            if (kClaim) {
                bool got = true;
                if (warp == 0) {  // the claimer
                    if (lane == 0) got = claim_next(S.claims, q, claim, first, &it, S.abort, segs.status);
                    got = __shfl_sync(0xffffffffu, got, 0);
                    it = __shfl_sync(0xffffffffu, it, 0);
                } else {
                    got = claim_read_warp(S.claims, q, &it, S.abort, segs.status);
                }
                if (!got) {
                    ok = false;
                    break;
                }
                if (it < 0 || it >= n_items) break;
            }
            const Item I = load_item(tab, segs, it, n_ranges, d, rng);
            if (!I.ad.ok) continue;
            // this warp's first stage of the item, and whether it has one at all
            const int32_t st0 = (warp - (int)(g % kStages) + kStages) % kStages;
            if (st0 >= I.n_stages) {
                g += (uint32_t)I.n_stages;
                continue;
            }
            const int32_t rp = rpad16(I.ad.rank);
            const int natoms = (rp + 63) / 64;
            const int32_t p0 = I.span.begin;
            const bool contiguous = (I.span.flags & 1) != 0;
            const int32_t t0 = PERM_AT(segs, p0);
            for (int32_t st = st0; st < I.n_stages; st += kStages) {
                const uint32_t gs = g + (uint32_t)st;
                const uint32_t s = gs % kStages, ph = (gs / kStages) & 1u;
                // a gathered stage: lane m holds the token of row m (loaded before the wait)
                const int valid = min(kTok, I.span.rows - kTok * st);  // rows of this stage in the span
                const int32_t tl = !contiguous && lane < valid ? PERM_AT(segs, p0 + kTok * st + lane) : -1;
                if (!mbar_wait(&S.empty[s], ph ^ 1u, S.abort, segs.status)) {
                    ok = false;
                    break;
                }
                uint8_t *act_s = S.act + s * kActBytes;
                uint8_t *h_s = S.h + s * kHBytes;
                const bool h_tma = valid == kTok;
                if (lane == 0) {
                    // a 3-D box always moves all eight blocks (past d: zero-filled)
                    const uint32_t act_bytes = blocks3 ? (uint32_t)(rng / 64) * kBox : (uint32_t)I.n_chunks * 2u * kBox;
                    const uint32_t bytes = (contiguous ? act_bytes : 0u) +
                                           (h_tma ? (uint32_t)natoms * kBox : 0u);
                    mbar_arrive_expect_tx(&S.full[s], bytes);
                    if (contiguous) {
                        if (blocks3)  // all 2 n_chunks 64-column blocks of the stage in one copy
                            tma_load_3d(act_s, &map_act3, &S.full[s], 0, t0 + kTok * st, I.n_base / 64);
                        else
                            for (int b = 0; b < 2 * I.n_chunks; ++b)
                                tma_load_2d(act_s + b * kBox, &map_act, &S.full[s], I.n_base + 64 * b,
                                            t0 + kTok * st);
                    }
                    if (h_tma)
                        for (int a = 0; a < natoms; ++a)
                            tma_load_2d(h_s + a * kBox, &map_h, &S.full[s], 64 * a, p0 + kTok * st);
                }
                if (!contiguous) {
                    // token row m, 16-byte chunk c of the 512 columns: box b = c / 8 holds
                    // columns 64 b .. 64 b + 63 as a [32 x 128 B] 128-byte-swizzled block;
                    // lanes take chunks lane, lane + 32
                    const int nch = I.n_chunks * 16;
#pragma unroll 4
                    for (int m = 0; m < kTok; ++m) {
                        const int32_t t = __shfl_sync(0xffffffffu, tl, m);
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const int c = lane + 32 * j;
                            if (c < nch) {
                                const bool v = t >= 0 && I.n_base + 8 * c < d;
                                const uint16_t *src = v ? act + (int64_t)t * d + I.n_base + 8 * c : act;
                                cp_async_16(act_s + (c >> 3) * kBox + sw128_offset((uint32_t)m, (uint32_t)(c & 7)), src,
                                            v);
                            }
                        }
                    }
                }
                if (!h_tma) {
                    // partial last stage: rows past the span are zero so they add nothing
                    const int nch = natoms * 8;
                    for (int e = lane; e < kTok * nch; e += 32) {
                        const int m = e / nch, c = e % nch;
                        const bool v = m < valid;
                        const uint16_t *src = v ? hbuf + (int64_t)(p0 + kTok * st + m) * rw + 8 * c : hbuf;
                        cp_async_16(h_s + (c >> 3) * kBox + sw128_offset((uint32_t)m, (uint32_t)(c & 7)), src, v);
                    }
                }
                if (!contiguous || !h_tma) {  // this lane's copies have landed; visible to the tensor cores
                    cp_async_commit();
                    cp_async_wait<0>();
                    fence_proxy_async();
                }
                mbar_arrive(&S.full[s]);
                last = gs;
            }
            g += (uint32_t)I.n_stages;
        }
        if (!ok && lane == 0 && last != 0xffffffffu) {  // aborted: let the last stage's TMA copies land
            uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(&S.full[last % kStages], (last / kStages) & 1u) &&
                   globaltimer_ns() - t0 < kWaitLimitNs / 8) {
            }
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t g = 0, nitem = 0;
            bool ok = true;
            uint32_t q = 0;
            for (int32_t it = blockIdx.x; (kClaim || it < n_items) && ok; it += gridDim.x, ++q) {
                if (kClaim) {
                    if (!claim_read(S.claims, q, &it, S.abort, segs.status)) break;
                    if (it < 0 || it >= n_items) break;
                }
                const Item I = load_item(tab, segs, it, n_ranges, d, rng);
                if (!I.ad.ok) continue;
                const uint32_t rp = (uint32_t)rpad16(I.ad.rank);
                const uint32_t idesc = make_idesc_bf16(128, rp, true, true);
                if (!mbar_wait(S.tempty, (nitem & 1u) ^ 1u, S.abort, segs.status)) break;
                tc_fence_after();
                for (int32_t st = 0; st < I.n_stages; ++st) {
                    const uint32_t s = g % kStages, ph = (g / kStages) & 1u;
                    if (!mbar_wait(&S.full[s], ph, S.abort, segs.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(S.act + s * kActBytes);
                    const uint32_t h_base = smem_u32(S.h + s * kHBytes);
                    for (int q = 0; q < I.n_chunks; ++q) {
#pragma unroll
                        for (int kk = 0; kk < kTok / 16; ++kk) {
                            const uint64_t adesc = make_desc(a_base + 2u * kBox * q + 2048u * kk, kBox, 1024, kSwizzle128);
                            const uint64_t bdesc = make_desc(h_base + 2048u * kk, kBox, 1024, kSwizzle128);
                            umma_bf16(tmem_base + 128u * q, adesc, bdesc, idesc, (st > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    umma_commit(&S.empty[s]);
                    ++g;
                }
                if (!ok) break;
                umma_commit(S.tfull);
                ++nitem;
            }
            umma_commit(S.done);
            uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(S.done, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        // Each warp owns 32 columns n (its TMEM lanes) of every chunk: 16 rows k
        // at a time it writes c * acc as [16 x 32] fp32 into one of its two
        // staging boxes and adds the box into G (rows row_off + k, columns n)
        // with a TMA bulk reduction.  Rows k in [r_i, r_pad) add exact zeros (h
        // is zero there); rows and columns past G's edge are clipped by the
        // TMA.  The accumulators go back to the MMA issuer once the last of
        // them is read.
        const uint32_t lane_base = 32u * (warp & 3);
        float *red = reinterpret_cast<float *>(S.red + (warp - kEpi0) * kRedBytes);
        uint32_t nitem = 0, n_ord = 0, nbox = 0;
        uint32_t q = 0;
        for (int32_t it = blockIdx.x; kClaim || it < n_items; it += gridDim.x, ++q) {
            if (kClaim) {
                if (q > 0) claim_release_warp(S.claims, q - 1);  // the previous item is done
                if (!claim_read_warp(S.claims, q, &it, S.abort, segs.status, true)) break;
                if (it < 0 || it >= n_items) {
                    claim_release_warp(S.claims, q);
                    break;
                }
            }
            const Item I = load_item(tab, segs, it, n_ranges, d, rng);
            if (!I.ad.ok) continue;
            const int32_t rp = rpad16(I.ad.rank);
            if (!mbar_wait_warp(S.tfull, nitem & 1u, S.abort, segs.status)) break;
            tc_fence_after();
            const float c = use_scale != 0.f ? I.ad.scale : 1.0f;
            // ordered mode, adapters of three spans or more (with two, the two adds
            // to zero commute exactly): span j of the adapter, its ticket
            int32_t *tk = nullptr;
            int32_t tj = 0;
            if (tickets != nullptr) {
                const int32_t g0 = segs.seg_start[I.span.adapter], g1 = segs.seg_start[I.span.adapter + 1];
                if (g1 - g0 > 2 * LORA_SPAN_TOKENS) {
                    tj = (I.span.begin - g0) / LORA_SPAN_TOKENS;
                    tk = tickets + LORA_DBG_INDEX((int64_t)(it / n_ranges - tj) * n_ranges + it % n_ranges,
                                                  (int64_t)segs.max_spans * n_ranges, segs.status);
                }
            }
            if (tk != nullptr) {
                if (warp == kEpi0 && lane == 0 && wait_ticket(tk, tj, S.abort, segs.status)) {
                    fence_proxy_async_all();
                    mbar_arrive(S.tk_go);
                }
                if (!mbar_wait_warp(S.tk_go, n_ord & 1u, S.abort, segs.status)) break;
                if (lane == 0) fence_proxy_async_all();
            }
            for (int q = 0; q < 4; ++q) {
                if (q >= I.n_chunks) break;
                const int32_t n0 = I.n_base + 128 * q + (int32_t)lane_base;
                const bool live = n0 < d;  // a box wholly past column d - 1 is not added
                for (int c0 = 0; c0 < rp; c0 += 16) {
                    float *buf = red + (nbox & 1u) * (kRedBlock / 4);
                    if (live) {
                        if (lane == 0) bulk_wait_read1();  // the reduction of this buffer's last box has read it
                        __syncwarp();
                    }
                    uint32_t v[16];
                    tmem_ld16(tmem_base + (lane_base << 16) + 128u * q + (uint32_t)c0, v);
                    tmem_ld_wait();
                    if (live) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) buf[e * 32 + lane] = c * __uint_as_float(v[e]);
                    }
                    if (q == I.n_chunks - 1 && c0 + 16 >= rp) {  // every accumulator is read: free them
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(S.tempty);
                    }
                    if (live) {
                        fence_proxy_async();
                        __syncwarp();
                        if (lane == 0) {
                            tma_reduce_add_2d(&map_g, buf, n0, I.ad.row_off + c0);
                            bulk_commit();
                        }
                        ++nbox;
                    }
                }
            }
            ++nitem;
            if (tk != nullptr) {  // the span's adds are complete in every warp: pass the ticket on
                if (lane == 0) {
                    bulk_wait0();
                    fence_proxy_async_all();
                    mbar_arrive(S.tk_done);
                }
                if (warp == kEpi0) {
                    if (!mbar_wait_warp(S.tk_done, n_ord & 1u, S.abort, segs.status)) break;
                    if (lane == 0) release_ticket(tk, tj + 1);
                }
                ++n_ord;
            }
        }
        if (lane == 0) bulk_wait0();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

lora_status_t launch_tokred(float *G, const void *act, int32_t d, const uint16_t *hbuf, int32_t rw, float use_scale,
                            int32_t *tickets, int32_t *claim, const lora_adapter_table &tab, const lora_segments &segs,
                            cudaStream_t stream)
{
    if (tickets != nullptr && claim == nullptr) return LORA_ERR_INVALID_ARG;  // the ordered adds need claimed items
    if (segs.n_tokens == 0 || segs.max_spans == 0) return LORA_OK;
    CUtensorMap map_act, map_act3, map_h, map_g;
    // 512-column items (256 in the two-CTA shape), or 128-column ones when the
    // wide items would leave half the SMs idle (few spans: a narrow batch of
    // large adapters); in between, the wider items' fewer reads of h win
    const int sms = sm_count();
    auto range_for = [&](int32_t wide) {
        return 2 * (int64_t)segs.max_spans * ((d + wide - 1) / wide) < sms ? 128 : wide;
    };
    // Two CTAs per SM for segment-sorted batches in the default order (no
    // claim counter given) with 1.5 to 3 items of the one-CTA shape per SM:
    // packed4096 (1.7) dB 70.0 -> 64.2 us, dA 60.6 -> 54.9 us.  Id-routed
    // batches gather their stages and lost with it (skewed dB 125 -> 139 us);
    // with about one item per SM most SMs would hold a single three-stage CTA
    // (sweep N = 2, dA 18.3 -> 21.4 us); with many items per SM the kernel
    // still gained but the step, where dB runs beside dh, lost (sweep N = 32,
    // 1.83 -> 1.86 ms).  The ordered mode claims its spans.
    const int64_t items1 = (int64_t)segs.max_spans * ((d + range_for(Shape<false>::kRange) - 1) /
                                                      range_for(Shape<false>::kRange));
    const bool two = claim == nullptr && tickets == nullptr && 2 * items1 >= 3 * (int64_t)sms &&
                     items1 < 3 * (int64_t)sms;
    const int32_t rng = range_for(two ? Shape<true>::kRange : Shape<false>::kRange);
    // d a multiple of 64: a stage's column blocks come in one 3-D copy
    const int32_t blocks3 = (d % 64 == 0 && make_tmap_bf16_blocks(&map_act3, act, (uint64_t)d,
                                                                   (uint64_t)segs.n_tokens, kTok, rng / 64))
                                ? 1
                                : 0;
    if (!make_tmap_bf16_2d(&map_act, act, (uint64_t)d, (uint64_t)segs.n_tokens, 64, kTok, true) ||
        !make_tmap_bf16_2d(&map_h, hbuf, (uint64_t)rw, (uint64_t)segs.n_tokens, 64, kTok, true) ||
        !make_tmap_f32_2d(&map_g, G, (uint64_t)d, (uint64_t)tab.sum_r, 32, 16))
        return LORA_ERR_CUDA;
    const int n_ranges = (d + rng - 1) / rng;
    const int64_t items = (int64_t)segs.max_spans * n_ranges;
    // run-time claims balance uneven items once every CTA has several to
    // take; with fewer than three per CTA (at most) the split by CTA index did
    // better (skewed batch, dA: 50 against 55 us).  The ordered mode always
    // claims: its waits rely on it.
    if (tickets == nullptr && items < 3 * (int64_t)sms) claim = nullptr;
    if (!blocks3) map_act3 = map_act;
    auto *kernel = claim != nullptr ? tc_tokred_kernel<true, false>
                   : two            ? tc_tokred_kernel<false, true>
                                    : tc_tokred_kernel<false, false>;
    const size_t smem = two ? Shape<true>::kSmemBytes : Shape<false>::kSmemBytes;
    const int threads = two ? Shape<true>::kThreads : Shape<false>::kThreads;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return LORA_ERR_CUDA;
    const int per_sm = two ? 2 : 1;
    const int grid = items < per_sm * sms ? (int)items : per_sm * sms;
    kernel<<<grid, threads, smem, stream>>>(map_act, map_act3, map_h, map_g, static_cast<const uint16_t *>(act), d,
                                            hbuf, rw, use_scale, blocks3, rng, tickets, claim, tab, segs);
    return cudaGetLastError() == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

}  // namespace

int32_t tokred_ranges(int32_t d) { return (d + 127) / 128; }  // the most column ranges of an item list

lora_status_t tc_db(float *dB, const void *dY, const uint16_t *h_bf16, int32_t rw, int32_t *tickets, int32_t *claim,
                    const lora_adapter_table &tab, const lora_segments &segs, cudaStream_t stream)
{
    return launch_tokred(dB, dY, tab.d_out, h_bf16, rw, 1.f, tickets, claim, tab, segs, stream);
}

lora_status_t tc_da(float *dA, const void *X, const uint16_t *dh_bf16, int32_t rw, int32_t *tickets, int32_t *claim,
                    const lora_adapter_table &tab, const lora_segments &segs, cudaStream_t stream)
{
    return launch_tokred(dA, X, tab.d_in, dh_bf16, rw, 0.f, tickets, claim, tab, segs, stream);
}

}  // namespace lora
