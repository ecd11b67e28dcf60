// tc_colproj.cu -- case ii on the 5th-generation tensor cores: a reduction over
// the rank into a T x d result that is accumulated into a bf16 tensor, tiled
// along tokens and the hidden dimension (PLoRA technical summary, "2. LoRA
// Execution Engine").
//
//   expand  y[t, o]  += s_i sum_k H[t, k]  B_i[o, k]
//   dX      dX[t, j] +=     sum_k dH[t, k] A_i[k, j]
//
// A work item is (tile of up to 128 tokens of one adapter, a 1024-column part
// of d).  The A operand is the tile's 128 x r_pad block of h in bf16: read by
// TMA from the perm-ordered hand-off buffers the case i kernel wrote (expand
// uses h = hi + lo, both multiplied, so H enters at ~16 significant bits), or,
// for the standalone expand of an fp32 H, converted by four loader warps.  The
// weights of every 128-column chunk (B_i^T or A_i rows, stacked alike) are the
// MN-major B operand, by TMA with 128-byte swizzle.  tcgen05.mma (M = 128,
// N = 128, K = 16) accumulates in a ring of four TMEM accumulators.  The bf16
// rows being updated are staged through a ring of 128 x 64 shared-memory
// blocks (TMA for consecutive tokens, cp.async gather otherwise); the epilogue
// adds c * acc in fp32, rounds once, and writes back with a TMA store (full
// tiles of consecutive tokens) or, from the same staged block, plain stores
// of the valid rows in which eight lanes cover one row's 128 bytes (a lane
// per row stored 16 bytes to each of 32 rows per instruction: skewed batch
// expand 207 -> 178 us, dX 70 -> 60 us).
//
// Warp roles: 0 loads (TMA / cp.async), 1 MMA + TMEM owner, then the
// epilogue: warps 2..9 for sorted batches (both column halves of a chunk at
// once), else 2..5; in the loader variant 2..5 epilogue and 6..9 fp32 -> bf16
// conversion of the h block.
#define LORA_DBG_FILE 3
#include "internal.h"
#include "tc_common.cuh"
#include "tc_host.h"

namespace lora {
namespace {

using namespace tc;

constexpr int kWStages = 2;
constexpr int kYStages = 6;
constexpr int kLook = 2;  // gathered tiles: chunks of y an epilogue warp copies ahead (kLook + 1 <= kYStages / 2)
constexpr int kNC = 128;                              // columns per MMA chunk
constexpr int kNPart = 1024;                          // columns per work item
constexpr uint32_t kWBytes = kNC * LORA_MAX_RANK * 2;  // one weight chunk
constexpr uint32_t kABytes = 128 * LORA_MAX_RANK * 2;  // one bf16 copy of the h block
constexpr uint32_t kYBytes = 128 * 64 * 2;             // one staged 128 x 64 block of y
constexpr uint32_t kAcc = 4;
constexpr uint32_t kTmemCols = 512;
constexpr size_t kSmemBytes = 1024 + kWStages * (size_t)kWBytes + 2 * (size_t)kABytes + kYStages * (size_t)kYBytes + 768;

struct Smem {
    uint8_t *w, *a, *y;
    uint64_t *wfull, *wempty, *yfull, *yempty, *ysync, *tfull, *tempty, *afull, *aempty, *done;
    uint32_t *tmem_holder;
    volatile int32_t *abort;
    ClaimRing claims;  // items claimed at run time
};

LORA_DEV Smem carve(uint8_t *raw)
{
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    Smem s;
    s.w = base;
    s.a = s.w + kWStages * kWBytes;
    s.y = s.a + 2 * kABytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(s.y + kYStages * kYBytes);
    s.wfull = bars;
    s.wempty = s.wfull + kWStages;
    s.yfull = s.wempty + kWStages;
    s.yempty = s.yfull + kYStages;
    s.ysync = s.yempty + kYStages;
    s.tfull = s.ysync + kYStages;
    s.tempty = s.tfull + kAcc;
    s.afull = s.tempty + kAcc;
    s.aempty = s.afull + 1;
    s.done = s.aempty + 1;
    s.tmem_holder = reinterpret_cast<uint32_t *>(s.done + 1);
    s.abort = reinterpret_cast<volatile int32_t *>(s.tmem_holder + 1);
    s.claims.full = reinterpret_cast<uint64_t *>(s.tmem_holder + 8);
    s.claims.empty = s.claims.full + kClaimSlots;
    s.claims.slot = reinterpret_cast<volatile int32_t *>(s.claims.empty + kClaimSlots);
    return s;
}

LORA_DEV int32_t rpad16(int32_t r) { return (r + 15) & ~15; }

struct Item {
    Tile tile;
    AdapterInfo ad;
    int32_t n_lo, n_hi;
    bool full;  // 128 consecutive tokens: TMA load and store of y
};

LORA_DEV Item load_item(const lora_adapter_table &tab, const lora_segments &segs, int32_t it, int32_t n_parts,
                        int32_t d)
{
    Item I;
    I.tile = LOAD_TILE(segs, it / n_parts);
    I.ad = load_adapter(tab, I.tile.adapter, segs.status);
    I.n_lo = (it % n_parts) * kNPart;
    I.n_hi = min(d, I.n_lo + kNPart);
    I.full = (I.tile.flags & 1) != 0 && I.tile.rows == 128;
    return I;
}

template <int N>
LORA_DEV void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory"); }
// Per store leader, the TMA stores whose shared-memory reads may still be
// pending: none with eight epilogue warps (one leader per column half), one
// with four (one leader for both halves).
template <int kEpi>
__host__ __device__ constexpr int store_lag() { return kEpi == 8 ? 0 : 1; }
// Threads: producer and MMA warps, the epilogue, and the loader warps.
template <bool kLoader, int kEpi>
__host__ __device__ constexpr int threads_of() { return 64 + 32 * kEpi + (kLoader ? 128 : 0); }

struct ColIn {
    const float *h32;  // loader variant: fp32 h by token, stride r_max
    float use_scale;   // 1: c = s_i, 0: c = 1
    int32_t split;     // 1: the A operand is hi + lo
    int32_t *claim;    // kClaim: the work-claim counter, zero at launch
};

// kGather: tiles of non-consecutive tokens occur (id-routed batches); their
// rows of y are copied into the stages by the epilogue warps that use them.
// kClaim: items claimed at run time from in.claim (id-routed batches, whose
// items differ in cost), else CTA b takes items b, b + gridDim.x, ...
template <bool kLoader, int kEpi, bool kGather, bool kClaim>
__global__ void __launch_bounds__(threads_of<kLoader, kEpi>(), 1)
tc_colproj_kernel(const __grid_constant__ WMaps map_w, const __grid_constant__ CUtensorMap map_hi,
                  const __grid_constant__ CUtensorMap map_lo, const __grid_constant__ CUtensorMap map_y,
                  uint16_t *__restrict__ out, int32_t d, ColIn in, lora_adapter_table tab, lora_segments segs)
{
    // epilogue warps: eight (sorted batches: every tile is a run of consecutive
    // tokens), else four; four when warps 6..9 convert the fp32 h block
    static_assert((kEpi == 4 || kEpi == 8) && !(kLoader && kEpi == 8), "epilogue of four or eight warps");
    static_assert(!(kLoader && kClaim), "the loader variant takes its items by CTA index");
    constexpr int kHStep = kEpi / 4;
    constexpr int kStoreLag = store_lag<kEpi>();
    // A stage of a full tile is freed once its leader has issued kStoreLag more
    // stores, i.e. after stage g + kStoreLag (four warps: one leader for both
    // halves) or g + 2 kStoreLag (eight: one leader per half) is worked on; TMA
    // stages arrive when issued, so the producer can fill that stage once an
    // earlier one is freed.  The stages of a gathered tile are handed to the
    // epilogue empty: each epilogue warp copies its own 32 rows of the chunk
    // kLook chunks ahead of the one it works on (cp.async, its own copy groups,
    // no barrier between warps), and the stage is freed without a store.
    // Tiles of the two kinds never share an item, and every item ends with its
    // stores drained.
    static_assert((kEpi / 4) * kStoreLag < kYStages, "y-stage ring too shallow for the store lag");
    extern __shared__ uint8_t smem_raw[];
    const Smem S = carve(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool split = in.split != 0;
    // the claimer's first item, claimed before the set-up so that its round trip overlaps it
    const int32_t first = kClaim && warp == 0 && lane == 0 ? claim_first(in.claim) : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kWStages; ++i) {
            mbar_init(&S.wfull[i], 1);
            mbar_init(&S.wempty[i], 1);
        }
        for (int i = 0; i < kYStages; ++i) {
            mbar_init(&S.yfull[i], 33);
            mbar_init(&S.yempty[i], 1);
            mbar_init(&S.ysync[i], 4);  // one arrive per warp of the group once its rows are done
        }
        for (uint32_t i = 0; i < kAcc; ++i) {
            mbar_init(&S.tfull[i], 1);
            mbar_init(&S.tempty[i], kEpi);
        }
        mbar_init(S.afull, kLoader ? 4 : 1);
        mbar_init(S.aempty, 1);
        mbar_init(S.done, 1);
        if (kClaim)
            for (int i = 0; i < kClaimSlots; ++i) {  // claimed by warp 0; read by the MMA thread and the epilogue
                mbar_init(&S.claims.full[i], 1);
                mbar_init(&S.claims.empty[i], 1 + kEpi);
            }
        *S.abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(S.tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *S.tmem_holder;
    const int32_t n_parts = (d + kNPart - 1) / kNPart;
    const int32_t n_items = N_TILES(segs) * n_parts;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&map_w.m16);
            prefetch_tensormap(&map_w.m32);
            prefetch_tensormap(&map_w.m64);
            prefetch_tensormap(&map_y);
            if (!kLoader) {
                prefetch_tensormap(&map_hi);
                if (split) prefetch_tensormap(&map_lo);
            }
        }
        uint32_t gw = 0, gy = 0, na = 0;
        bool ok = true;
        uint32_t q = 0;
        for (int32_t it = blockIdx.x; (kClaim || it < n_items) && ok; it += gridDim.x, ++q) {
            if (kClaim) {
                bool got = true;
                if (lane == 0) got = claim_next(S.claims, q, in.claim, first, &it, S.abort, segs.status);
                got = __shfl_sync(0xffffffffu, got, 0);
                it = __shfl_sync(0xffffffffu, it, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                if (it < 0 || it >= n_items) break;
            }
            const Item I = load_item(tab, segs, it, n_parts, d);
            if (!I.ad.ok) continue;
            const int32_t rp = rpad16(I.ad.rank);
            const bool contiguous = (I.tile.flags & 1) != 0;
            const int32_t t0 = PERM_AT(segs, I.tile.begin);
            if (!kLoader) {
                if (!mbar_wait(S.aempty, (na & 1u) ^ 1u, S.abort, segs.status)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const int natoms = (rp + 63) / 64;
                    mbar_arrive_expect_tx(S.afull, (uint32_t)natoms * kYBytes * (split ? 2u : 1u));
                    for (int a = 0; a < natoms; ++a) {
                        tma_load_2d(S.a + a * kYBytes, &map_hi, S.afull, 64 * a, I.tile.begin);
                        if (split) tma_load_2d(S.a + kABytes + a * kYBytes, &map_lo, S.afull, 64 * a, I.tile.begin);
                    }
                }
                ++na;
            }
            for (int32_t n0 = I.n_lo; n0 < I.n_hi && ok; n0 += kNC) {
                // weights of the chunk: A_i / B_i^T rows k, columns n0 .. n0+127, MN-major atoms
                {
                    const uint32_t s = gw % kWStages, ph = (gw / kWStages) & 1u;
                    if (!mbar_wait(&S.wempty[s], ph ^ 1u, S.abort, segs.status)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        uint8_t *w_s = S.w + s * kWBytes;
                        mbar_arrive_expect_tx(&S.wfull[s], (uint32_t)rp * 256u);
                        for (int a = 0; a < 2; ++a)
                            tma_load_rows(w_s + a * rp * 128, map_w, &S.wfull[s], n0 + 64 * a, I.ad.row_off, rp);
                    }
                    ++gw;
                }
                // the two 64-column halves of the chunk's rows of y
                for (int h = 0; h < 2; ++h) {
                    const int32_t c0 = n0 + 64 * h;
                    const uint32_t s = gy % kYStages, ph = (gy / kYStages) & 1u;
                    if (!mbar_wait(&S.yempty[s], ph ^ 1u, S.abort, segs.status)) {
                        ok = false;
                        break;
                    }
                    uint8_t *y_s = S.y + s * kYBytes;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&S.yfull[s], contiguous ? kYBytes : 0u);
                        if (contiguous) tma_load_2d(y_s, &map_y, &S.yfull[s], c0, t0);
                    }
                    // every lane's arrival: a gathered tile's stage goes to the
                    // epilogue warps empty (they copy their own rows into it)
                    mbar_arrive(&S.yfull[s]);
                    ++gy;
                }
            }
        }
        if (!ok && lane == 0) {  // aborted: let issued copies land before the CTA leaves
            for (uint32_t u = gy > (uint32_t)kYStages ? gy - kYStages : 0u; u < gy; ++u) {
                uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&S.yfull[u % kYStages], (u / kYStages) & 1u) &&
                       globaltimer_ns() - t0 < kWaitLimitNs / 8) {
                }
            }
            for (uint32_t u = gw > (uint32_t)kWStages ? gw - kWStages : 0u; u < gw; ++u) {
                uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&S.wfull[u % kWStages], (u / kWStages) & 1u) &&
                       globaltimer_ns() - t0 < kWaitLimitNs / 8) {
                }
            }
            if (!kLoader && na > 0) {
                uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(S.afull, (na - 1) & 1u) && globaltimer_ns() - t0 < kWaitLimitNs / 8) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t gw = 0, a = 0, na = 0;
            bool ok = true;
            const uint32_t idesc = make_idesc_bf16(128, kNC, false, true);
            const uint32_t abase = smem_u32(S.a);
            uint32_t q = 0;
            for (int32_t it = blockIdx.x; (kClaim || it < n_items) && ok; it += gridDim.x, ++q) {
                if (kClaim) {
                    if (!claim_read(S.claims, q, &it, S.abort, segs.status)) break;
                    if (it < 0 || it >= n_items) break;
                }
                const Item I = load_item(tab, segs, it, n_parts, d);
                if (!I.ad.ok) continue;
                const int32_t rp = rpad16(I.ad.rank);
                if (!mbar_wait(S.afull, na & 1u, S.abort, segs.status)) break;
                tc_fence_after();
                for (int32_t n0 = I.n_lo; n0 < I.n_hi; n0 += kNC) {
                    const uint32_t s = gw % kWStages, ph = (gw / kWStages) & 1u;
                    const uint32_t acc = a % kAcc, aph = (a / kAcc) & 1u;
                    if (!mbar_wait(&S.tempty[acc], aph ^ 1u, S.abort, segs.status) ||
                        !mbar_wait(&S.wfull[s], ph, S.abort, segs.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t w_base = smem_u32(S.w + s * kWBytes);
                    const uint32_t d_tmem = tmem_base + acc * 128u;
                    for (int kk = 0; kk < rp / 16; ++kk) {
                        const uint32_t aoff = (uint32_t)(kk >> 2) * kYBytes + (uint32_t)(kk & 3) * 32u;
                        const uint64_t bdesc = make_desc(w_base + 2048u * kk, (uint32_t)rp * 128u, 1024, kSwizzle128);
                        umma_bf16(d_tmem, make_desc(abase + aoff, 16, 1024, kSwizzle128), bdesc, idesc,
                                  kk > 0 ? 1u : 0u);
                        if (split)
                            umma_bf16(d_tmem, make_desc(abase + kABytes + aoff, 16, 1024, kSwizzle128), bdesc, idesc,
                                      1u);
                    }
                    umma_commit(&S.wempty[s]);
                    umma_commit(&S.tfull[acc]);
                    ++gw;
                    ++a;
                }
                if (!ok) break;
                umma_commit(S.aempty);
                ++na;
            }
            umma_commit(S.done);
            uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(S.done, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else if (kLoader && warp >= 6) {
        // ------------------------------------------------------------ fp32 h -> bf16 A operand
        const int m = threadIdx.x - 6 * 32;  // row 0..127 of the tile
        const int32_t r_max = tab.r_max;
        uint32_t na = 0;
        for (int32_t it = blockIdx.x; it < n_items; it += gridDim.x) {
            const Item I = load_item(tab, segs, it, n_parts, d);
            if (!I.ad.ok) continue;
            const int32_t r = I.ad.rank, rp = rpad16(r);
            if (!mbar_wait_warp(S.aempty, (na & 1u) ^ 1u, S.abort, segs.status)) break;
            const int32_t t = m < I.tile.rows ? PERM_AT(segs, I.tile.begin + m) : -1;
            const float *hr = in.h32 + (int64_t)(t < 0 ? 0 : t) * r_max;
#pragma unroll 4
            for (int kc = 0; kc < rp / 8; ++kc) {
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = (t >= 0 && 8 * kc + e < r) ? hr[8 * kc + e] : 0.f;
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    hi[e / 2] = pack_bf16(f[e], f[e + 1]);
                    lo[e / 2] = pack_bf16(f[e] - bf16lo(hi[e / 2]), f[e + 1] - bf16hi(hi[e / 2]));
                }
                const uint32_t off = (uint32_t)(kc >> 3) * kYBytes + sw128_offset((uint32_t)m, (uint32_t)(kc & 7));
                *reinterpret_cast<uint4 *>(S.a + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                if (split) *reinterpret_cast<uint4 *>(S.a + kABytes + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(S.afull);
            ++na;
        }
    } else if (warp >= 2 && warp < 2 + kEpi) {
        // ------------------------------------------------------------ epilogue
        // Group hg of four warps (one per TMEM sub-partition) takes the column
        // halves h = hg, hg + kHStep of every chunk: with eight epilogue warps
        // both halves of a chunk are worked on at once, each with its own
        // store leader (lane 0 of the group's first warp).
        const int hg = (warp - 2) >> 2;
        const uint32_t lane_base = 32u * (warp & 3);
        const int m = (int)lane_base + lane;
        const bool leader = (warp & 3) == 2 && lane == 0;
        const bool lead_warp = (warp & 3) == 2;
        uint32_t a = 0;
        bool ok = true;
        // leader only: stages whose TMA store may still be reading shared memory,
        // oldest first; a stage goes back to the producer once its store has read it
        int32_t pend[kStoreLag + 1];
        int npend = 0;
        uint32_t q = 0;
        for (int32_t it = blockIdx.x; (kClaim || it < n_items) && ok; it += gridDim.x, ++q) {
            if (kClaim) {
                if (q > 0) claim_release_warp(S.claims, q - 1);  // the previous item is done
                if (!claim_read_warp(S.claims, q, &it, S.abort, segs.status, true)) break;
                if (it < 0 || it >= n_items) {
                    claim_release_warp(S.claims, q);
                    break;
                }
            }
            const Item I = load_item(tab, segs, it, n_parts, d);
            if (!I.ad.ok) continue;
            const float c = in.use_scale != 0.f ? I.ad.scale : 1.0f;
            const int32_t t = m < I.tile.rows ? PERM_AT(segs, I.tile.begin + m) : -1;
            const int32_t t0 = PERM_AT(segs, I.tile.begin);
            // a gathered tile: this warp copies its own 32 rows of each chunk's
            // halves into the chunk's stages, kLook chunks ahead; lane l copies
            // 16 bytes (piece l & 7) of rows (l >> 3) + 4 q, q < 8, of the warp
            const bool gathered = kGather && (I.tile.flags & 1) == 0;
            const uint32_t a0 = a;
            const int32_t n_chunks = (I.n_hi - I.n_lo + kNC - 1) / kNC;
            // tokens of rows (l >> 3) + 4 q, q < 8, of the warp (-1 past the tile):
            // a gathered tile's copies and any tile that is not full move rows in
            // that pattern, four rows of 128 bytes per warp instruction
            int32_t tg[8];
            if (gathered || !I.full) {
#pragma unroll
                for (int q = 0; q < 8; ++q) tg[q] = __shfl_sync(0xffffffffu, t, (lane >> 3) + 4 * q);
            }
            auto copy_rows = [&](int32_t j) -> bool {
                for (int h = hg; h < 2; h += kHStep) {
                    const uint32_t gy = 2u * (a0 + (uint32_t)j) + (uint32_t)h;
                    const uint32_t s = gy % kYStages, ph = (gy / kYStages) & 1u;
                    if (!mbar_wait_warp(&S.yfull[s], ph, S.abort, segs.status)) return false;  // handed over
                    uint8_t *y_s = S.y + s * kYBytes;
                    const int32_t c0 = I.n_lo + j * kNC + 64 * h;
                    const int cc = lane & 7;
                    const bool cin = c0 + 8 * cc < d;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const bool v = tg[q] >= 0 && cin;
                        cp_async_16(y_s + sw128_offset(lane_base + (uint32_t)((lane >> 3) + 4 * q), (uint32_t)cc),
                                    v ? out + (int64_t)tg[q] * d + c0 + 8 * cc : out, v);
                    }
                }
                cp_async_commit();
                return true;
            };
            if (gathered) {
                for (int32_t j = 0; j < kLook && j < n_chunks && ok; ++j) ok = copy_rows(j);
                if (!ok) break;
            }
            for (int32_t n0 = I.n_lo; n0 < I.n_hi; n0 += kNC) {
                const int32_t j = (n0 - I.n_lo) / kNC;
                if (gathered && j + kLook < n_chunks && !copy_rows(j + kLook)) {
                    ok = false;
                    break;
                }
                const uint32_t acc = a % kAcc, aph = (a / kAcc) & 1u;
                if (!mbar_wait_warp(&S.tfull[acc], aph, S.abort, segs.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (gathered) {  // this warp's copies of chunk j have landed (later chunks' may not have)
                    const int32_t later = min(kLook, n_chunks - 1 - j);
                    if (later >= 2)
                        cp_async_wait<2>();
                    else if (later == 1)
                        cp_async_wait<1>();
                    else
                        cp_async_wait<0>();
                    __syncwarp();
                }
#pragma unroll 1
                for (int h = hg; h < 2; h += kHStep) {
                    const int32_t c0 = n0 + 64 * h;
                    const uint32_t gy = 2u * a + (uint32_t)h;  // the producer fills two stages per chunk
                    const uint32_t s = gy % kYStages, ph = (gy / kYStages) & 1u;
                    if (!gathered && !mbar_wait_warp(&S.yfull[s], ph, S.abort, segs.status)) {
                        ok = false;
                        break;
                    }
                    uint8_t *y_s = S.y + s * kYBytes;
                    uint4 yv[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        yv[q] = *reinterpret_cast<const uint4 *>(y_s + sw128_offset((uint32_t)m, (uint32_t)q));
                    uint32_t v[4][16];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        tmem_ld16(tmem_base + (lane_base << 16) + acc * 128u + 64u * h + 16u * q, v[q]);
                    tmem_ld_wait();
                    if (h + kHStep >= 2) {  // this warp's last read of the accumulator
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&S.tempty[acc]);
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint32_t *acc8 = &v[q >> 1][(q & 1) * 8];
                        uint32_t w[4] = {yv[q].x, yv[q].y, yv[q].z, yv[q].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float lo = bf16lo(w[e]) + c * __uint_as_float(acc8[2 * e]);
                            const float hi = bf16hi(w[e]) + c * __uint_as_float(acc8[2 * e + 1]);
                            w[e] = pack_bf16(lo, hi);
                        }
                        *reinterpret_cast<uint4 *>(y_s + sw128_offset((uint32_t)m, (uint32_t)q)) =
                            make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    if (I.full) fence_proxy_async();
                    __syncwarp();
                    if (!I.full) {  // the warp's rows back to their tokens, 128 contiguous bytes per row and lane octet
                        const int cc = lane & 7;
                        if (c0 + 8 * cc < d) {
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                if (tg[q] >= 0)
                                    *reinterpret_cast<uint4 *>(out + (int64_t)tg[q] * d + c0 + 8 * cc) =
                                        *reinterpret_cast<const uint4 *>(
                                            y_s + sw128_offset(lane_base + (uint32_t)((lane >> 3) + 4 * q), (uint32_t)cc));
                        }
                        __syncwarp();
                    }
                    if (lane == 0) mbar_arrive(&S.ysync[s]);
                    if (lead_warp) {  // the group's four warps have their rows in place: store, free stages
                        if (!mbar_wait_warp(&S.ysync[s], ph, S.abort, segs.status)) {
                            ok = false;
                        } else if (leader) {
                            if (I.full) {
                                tma_store_2d(&map_y, y_s, c0, t0);
                                pend[npend++] = (int32_t)s;
                                if (npend > kStoreLag) {  // the oldest store has read its stage
                                    bulk_wait_read<kStoreLag>();
                                    mbar_arrive(&S.yempty[pend[0]]);
                                    for (int q = 1; q < npend; ++q) pend[q - 1] = pend[q];
                                    --npend;
                                }
                            } else {
                                mbar_arrive(&S.yempty[s]);
                            }
                        }
                        __syncwarp();
                    }
                    if (!ok) break;
                }
                if (!ok) break;
                ++a;
            }
            // end of the item: every pending store finishes reading and its stage is
            // handed back, so the producer never waits on a stage held across items
            if (leader) {
                bulk_wait_read<0>();
                for (int q = 0; q < npend; ++q) mbar_arrive(&S.yempty[pend[q]]);
                npend = 0;
            }
            __syncwarp();
        }
        if (leader) {
            bulk_wait0();
            for (int q = 0; q < npend; ++q) mbar_arrive(&S.yempty[pend[q]]);
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <bool kLoader, int kEpi, bool kGather, bool kClaim>
lora_status_t launch_colproj(uint16_t *out, int32_t d, const void *w, const uint16_t *hi, const uint16_t *lo,
                             int32_t rw, const ColIn &in, const lora_adapter_table &tab, const lora_segments &segs,
                             cudaStream_t stream)
{
    if (segs.n_tokens == 0 || segs.max_tiles == 0) return LORA_OK;
    WMaps map_w;
    CUtensorMap map_hi, map_lo, map_y;
    if (!make_wmaps(&map_w, w, (uint64_t)d, (uint64_t)tab.sum_r) ||
        !make_tmap_bf16_2d(&map_y, out, (uint64_t)d, (uint64_t)segs.n_tokens, 64, 128, true))
        return LORA_ERR_CUDA;
    if (!kLoader) {
        if (!make_tmap_bf16_2d(&map_hi, hi, (uint64_t)rw, (uint64_t)segs.n_tokens, 64, 128, true))
            return LORA_ERR_CUDA;
        if (lo != nullptr) {
            if (!make_tmap_bf16_2d(&map_lo, lo, (uint64_t)rw, (uint64_t)segs.n_tokens, 64, 128, true))
                return LORA_ERR_CUDA;
        } else {
            map_lo = map_hi;
        }
    } else {
        map_hi = map_y;
        map_lo = map_y;
    }
    if (cudaFuncSetAttribute(tc_colproj_kernel<kLoader, kEpi, kGather, kClaim>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
        return LORA_ERR_CUDA;
    const int n_parts = (d + kNPart - 1) / kNPart;
    const int64_t items = (int64_t)segs.max_tiles * n_parts;
    const int sms = sm_count();
    const int grid = items < sms ? (int)items : sms;
    tc_colproj_kernel<kLoader, kEpi, kGather, kClaim><<<grid, threads_of<kLoader, kEpi>(), kSmemBytes, stream>>>(
        map_w, map_hi, map_lo, map_y, out, d, in, tab, segs);
    return cudaGetLastError() == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

}  // namespace

// Segment-sorted batches: every tile a run of consecutive tokens, items split
// ahead of time (they cost the same but for the last tile of each adapter).
// Id-routed batches: gathered tiles too, items claimed at run time when a
// counter is given (gathered and TMA tiles, tiles of any length).
lora_status_t launch_bf16(uint16_t *out, int32_t d, const void *w, const uint16_t *hi, const uint16_t *lo, int32_t rw,
                          const ColIn &in, const lora_adapter_table &tab, const lora_segments &segs,
                          cudaStream_t stream)
{
    if (segs.sorted != 0) return launch_colproj<false, 8, false, false>(out, d, w, hi, lo, rw, in, tab, segs, stream);
    if (in.claim != nullptr) return launch_colproj<false, 8, true, true>(out, d, w, hi, lo, rw, in, tab, segs, stream);
    return launch_colproj<false, 8, true, false>(out, d, w, hi, lo, rw, in, tab, segs, stream);
}

lora_status_t tc_expand_bf16(void *y, const uint16_t *hi, const uint16_t *lo, int32_t rw, int32_t *claim,
                             const lora_adapter_table &tab, const lora_segments &segs, cudaStream_t stream)
{
    const ColIn in{nullptr, 1.f, lo != nullptr ? 1 : 0, claim};
    return launch_bf16(static_cast<uint16_t *>(y), tab.d_out, tab.B, hi, lo, rw, in, tab, segs, stream);
}

lora_status_t tc_expand_f32(void *y, const float *H, const lora_adapter_table &tab, const lora_segments &segs,
                            cudaStream_t stream)
{
    const ColIn in{H, 1.f, 1, nullptr};
    return launch_colproj<true, 4, true, false>(static_cast<uint16_t *>(y), tab.d_out, tab.B, nullptr, nullptr, 0, in,
                                                tab, segs, stream);
}

lora_status_t tc_dx(void *dX, const uint16_t *dh_bf16, int32_t rw, int32_t *claim, const lora_adapter_table &tab,
                    const lora_segments &segs, cudaStream_t stream)
{
    const ColIn in{nullptr, 0.f, 0, claim};
    return launch_bf16(static_cast<uint16_t *>(dX), tab.d_in, tab.A, dh_bf16, nullptr, rw, in, tab, segs, stream);
}

}  // namespace lora
