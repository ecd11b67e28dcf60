// tc_base.cu -- a LoRA layer's forward over a packed, segment-sorted batch in
// one persistent launch on the 5th-generation tensor cores:
//
//   y_t = W x_t + s_i B_i (A_i x_t)        (token t of adapter i)
//
// The frozen base weight W is shared by every adapter of the batch, which is
// what packing amortises (PLoRA technical summary, "2. LoRA Execution
// Engine"); the delta rides on the base GEMM's accumulators instead of
// making another pass over y.
//
// Work is a list of tasks that the CTAs (one per SM) claim in index order
// from a global atomic counter:
//   h task (routing tile m of up to 128 tokens of adapter i): h = x A_i^T
//     accumulated in TMEM over d_in (M = 128, N = r_i rounded up to 16), then
//     written as fp32 H (optional, for the backward) and as bf16 s_i h to a
//     hand-off buffer; a release counter per routing tile says it is there.
//   tile task (pair of routing tiles p = 2q, 2q + 1; 256 output columns j):
//     two 128 x 256 fp32 accumulators (all 512 TMEM columns), K-loop over d_in
//     with both halves' x blocks and one W block per stage; then, per half, the
//     delta as extra K steps: A operand = the hand-off rows of s_i h, B operand
//     = rows of B_i^T (MN-major) -- the same accumulator, so y is rounded to
//     bf16 once, straight from TMEM.
// h tasks run a fixed number of pairs ahead of the tile tasks that need them,
// so a tile's wait for its h is normally already satisfied; the launch is
// cooperative (every CTA resident), and a task only ever waits for tasks of
// lower index, so the waits always end (each is bounded all the same).  Tiles
// of one pair and its 16 column blocks run at about the same time on
// neighbouring CTAs, so x is read from HBM about once (by the h task) and W
// stays in L2.
//
// Warp roles: 0 TMA producer, 1 MMA issuer + TMEM owner, 2..9 epilogue
// (2..5 the first half's rows, 6..9 the second's, one TMEM sub-partition per
// warp).
#define LORA_DBG_FILE 6
#include "internal.h"
#include "tc_common.cuh"
#include "tc_host.h"

namespace lora {
namespace {

using namespace tc;

constexpr int kStages = 3;
constexpr int kBN = 256;                                   // output columns per tile
constexpr uint32_t kXBytes = 128 * 128;                    // 128 rows x 64 bf16 (16 KB)
constexpr uint32_t kWBytes = 256 * 128;                    // 256 rows x 64 bf16 (32 KB)
constexpr uint32_t kStageBytes = 2 * kXBytes + kWBytes;    // both halves' x + one W block
constexpr uint32_t kYBytes = 128 * 128;                    // y staging: 128 rows x 64 bf16, one per half
constexpr int kRing = 4;                                   // claimed tasks in flight per CTA
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
constexpr size_t kSmemBytes = 1024 + kStages * (size_t)kStageBytes + 2 * (size_t)kYBytes + 256;
constexpr int32_t kHandoffReady = 4;  // one release increment per epilogue warp of the half

struct Smem {
    uint8_t *stage, *ybuf;
    uint64_t *full, *empty, *tfull, *tempty, *done, *qfull, *qempty, *sfull, *sfree;
    int64_t *ring;
    uint32_t *tmem_holder;
    volatile int32_t *abort;
};

LORA_DEV Smem carve(uint8_t *raw)
{
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    Smem s;
    s.stage = base;
    s.ybuf = base + kStages * kStageBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(s.ybuf + 2 * kYBytes);
    s.full = bars;
    s.empty = s.full + kStages;
    s.tfull = s.empty + kStages;
    s.tempty = s.tfull + 1;
    s.done = s.tempty + 1;
    s.qfull = s.done + 1;
    s.qempty = s.qfull + kRing;
    s.sfull = s.qempty + kRing;
    s.sfree = s.sfull + 2;
    s.ring = reinterpret_cast<int64_t *>(s.sfree + 2);
    s.tmem_holder = reinterpret_cast<uint32_t *>(s.ring + kRing);
    s.abort = reinterpret_cast<volatile int32_t *>(s.tmem_holder + 1);
    return s;
}

LORA_DEV int32_t rpad16(int32_t r) { return (r + 15) & ~15; }

struct BaseArgs {
    uint16_t *y;       // [T, d_out] bf16 (out)
    float *H;          // [T, r_max] fp32 (out) or null
    uint16_t *hs;      // [T, rw] bf16 hand-off: s_i h, zero beyond r_i
    int32_t *ready;    // per routing tile: kHandoffReady once its hand-off rows are written
    int32_t *claim;    // next unclaimed task (zero at launch)
    int32_t rw;
    int32_t n_col;     // column blocks of 256 per pair
    int32_t ahead;     // pairs whose h tasks come before the tile tasks that read them
};

// Task k of the list: the first 2 * ahead are h(0 .. 2 ahead - 1); after them
// come groups of (2 + n_col): h tasks of pair g + ahead, then the tiles of
// pair g.  Every h(m) precedes all the tiles that read it.
struct Task {
    int32_t kind;  // 0 none, 1 h task, 2 tile task
    int32_t m;     // routing tile (h) or pair (tile)
    int32_t j;     // column block (tile)
};

LORA_DEV Task task_of(int64_t k, int32_t n_tiles, const BaseArgs &a)
{
    Task t{0, 0, 0};
    const int64_t pre = 2 * (int64_t)a.ahead;
    if (k < pre) {
        t.m = (int32_t)k;
        t.kind = t.m < n_tiles ? 1 : 0;
        return t;
    }
    const int64_t g = (k - pre) / (2 + a.n_col), q = (k - pre) % (2 + a.n_col);
    if (q < 2) {
        const int64_t m = 2 * (g + a.ahead) + q;
        t.m = (int32_t)m;
        t.kind = m < n_tiles ? 1 : 0;
    } else {
        t.m = (int32_t)g;
        t.j = (int32_t)(q - 2);
        t.kind = 2 * g < n_tiles ? 2 : 0;
    }
    return t;
}

LORA_DEV int64_t n_tasks(int32_t n_tiles, const BaseArgs &a)
{
    const int64_t pairs = (n_tiles + 1) / 2;
    return 2 * (int64_t)a.ahead + pairs * (2 + a.n_col);
}

// the pair's halves: present, and whether the delta applies (adapter valid)
struct Pair {
    Tile t[2];
    AdapterInfo ad[2];
    bool has1;
};

LORA_DEV Pair load_pair(const lora_adapter_table &tab, const lora_segments &segs, int32_t p, int32_t n_tiles)
{
    Pair P;
    P.has1 = 2 * p + 1 < n_tiles;
    P.t[0] = LOAD_TILE(segs, 2 * p);
    P.ad[0] = load_adapter(tab, P.t[0].adapter, nullptr);  // the h task reports a bad entry
    if (P.has1) {
        P.t[1] = LOAD_TILE(segs, 2 * p + 1);
        P.ad[1] = load_adapter(tab, P.t[1].adapter, nullptr);
    } else {
        P.t[1] = P.t[0];
        P.ad[1] = P.ad[0];
        P.ad[1].ok = false;
    }
    return P;
}

// k-steps of the delta for one half: ceil(r_pad / 64) stages of up to 64 ranks
LORA_DEV int32_t delta_stages(const AdapterInfo &ad) { return ad.ok ? (rpad16(ad.rank) + 63) / 64 : 0; }

LORA_DEV bool wait_ready(const int32_t *flag, volatile int32_t *abort_flag, int32_t *status)
{
    long long t0 = 0;
    for (uint32_t it = 0;; ++it) {
        int32_t v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v >= kHandoffReady) {
            asm volatile("fence.proxy.async.global;" ::: "memory");  // the TMA reads that follow see the rows
            return true;
        }
        if ((it & 63u) == 0u) {
            if (*abort_flag) return false;
            const long long now = clock64();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kWaitLimitCycles) {
                *abort_flag = 1;
                set_status(status, LORA_ERR_TIMEOUT);
                return false;
            }
        }
        __nanosleep(100);
    }
}

LORA_DEV void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// The next claimed task from the CTA's ring (every consumer sees every task
// in claim order); -1 at the end, -2 on abort.
LORA_DEV int64_t next_task_warp(const Smem &S, uint32_t i, int32_t *status)
{
    const uint32_t slot = i % kRing, ph = (i / kRing) & 1u;
    if (!mbar_wait_warp(&S.qfull[slot], ph, S.abort, status)) return -2;
    const int64_t k = S.ring[slot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&S.qempty[slot]);
    return k;
}

__global__ void __launch_bounds__(kThreads, 1)
tc_base_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
               const __grid_constant__ CUtensorMap map_hs, const __grid_constant__ CUtensorMap map_y,
               const __grid_constant__ WMaps map_a, const __grid_constant__ WMaps map_b, BaseArgs args,
               lora_adapter_table tab, lora_segments segs)
{
    extern __shared__ uint8_t smem_raw[];
    const Smem S = carve(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], 1);
        }
        mbar_init(S.tfull, 1);
        mbar_init(S.tempty, 8);  // one arrive per epilogue warp
        mbar_init(S.done, 1);
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&S.qfull[i], 1);
            mbar_init(&S.qempty[i], 9);  // the MMA warp and the eight epilogue warps
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&S.sfull[h], 4);  // the half's four warps have staged their rows
            mbar_init(&S.sfree[h], 1);  // the half's store has read the staging buffer
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
    const int32_t n_tiles = N_TILES(segs);
    const int64_t total = n_tasks(n_tiles, args);
    const int32_t kb_n = (tab.d_in + 63) / 64;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Claims tasks from the global counter (so CTAs stay balanced), passes
        // each to the MMA and epilogue warps through the ring, and loads its
        // operands.  Claims are handed out in increasing order, so every h
        // task a tile waits for has already been claimed by a running CTA.
        if (lane == 0) {
            prefetch_tensormap(&map_x);
            prefetch_tensormap(&map_w);
            prefetch_tensormap(&map_hs);
            uint32_t g = 0;
            bool ok = true;
            auto next_stage = [&](uint32_t bytes) -> uint8_t * {
                const uint32_t s = g % kStages, ph = (g / kStages) & 1u;
                if (!mbar_wait(&S.empty[s], ph ^ 1u, S.abort, segs.status)) return nullptr;
                mbar_arrive_expect_tx(&S.full[s], bytes);
                return S.stage + s * kStageBytes;
            };
            for (uint32_t i = 0; ok; ++i) {
                // claim the next task that has work (h tasks of a bad table entry are dropped)
                int64_t k;
                Task t{};
                for (;;) {
                    k = atomicAdd(args.claim, 1);
                    if (k >= total) {
                        k = -1;
                        break;
                    }
                    t = task_of(k, n_tiles, args);
                    if (t.kind == 2) break;
                    if (t.kind == 1 && load_adapter(tab, LOAD_TILE(segs, t.m).adapter, segs.status).ok) break;
                }
                const uint32_t slot = i % kRing, ph = (i / kRing) & 1u;
                if (!mbar_wait(&S.qempty[slot], ph ^ 1u, S.abort, segs.status)) break;
                S.ring[slot] = k;
                mbar_arrive(&S.qfull[slot]);
                if (k < 0) break;
                if (t.kind == 1) {
                    const Tile T = LOAD_TILE(segs, t.m);
                    const AdapterInfo ad = load_adapter(tab, T.adapter, nullptr);
                    const int32_t rp = rpad16(ad.rank);
                    for (int32_t kb = 0; kb < kb_n; ++kb) {
                        uint8_t *st = next_stage(kXBytes + (uint32_t)rp * 128u);
                        if (st == nullptr) {
                            ok = false;
                            break;
                        }
                        uint64_t *bar = &S.full[g % kStages];
                        tma_load_2d(st, &map_x, bar, 64 * kb, T.begin);
                        tma_load_rows(st + 2 * kXBytes, map_a, bar, 64 * kb, ad.row_off, rp);
                        ++g;
                    }
                } else {
                    const Pair P = load_pair(tab, segs, t.m, n_tiles);
                    const int32_t n0 = kBN * t.j;
                    for (int32_t kb = 0; kb < kb_n; ++kb) {
                        uint8_t *st = next_stage(kXBytes * (P.has1 ? 2u : 1u) + kWBytes);
                        if (st == nullptr) {
                            ok = false;
                            break;
                        }
                        uint64_t *bar = &S.full[g % kStages];
                        tma_load_2d(st, &map_x, bar, 64 * kb, P.t[0].begin);
                        if (P.has1) tma_load_2d(st + kXBytes, &map_x, bar, 64 * kb, P.t[1].begin);
                        tma_load_2d(st + 2 * kXBytes, &map_w, bar, 64 * kb, n0);
                        ++g;
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int32_t ns = ok ? delta_stages(P.ad[h]) : 0;
                        if (ns == 0) continue;
                        if (!wait_ready(args.ready + 2 * t.m + h, S.abort, segs.status)) {
                            ok = false;
                            break;
                        }
                        const int32_t rp = rpad16(P.ad[h].rank);
                        for (int32_t ks = 0; ks < ns; ++ks) {
                            const int32_t kr = min(64, rp - 64 * ks);
                            uint8_t *st = next_stage(kXBytes + (uint32_t)kr * 512u);
                            if (st == nullptr) {
                                ok = false;
                                break;
                            }
                            uint64_t *bar = &S.full[g % kStages];
                            tma_load_2d(st, &map_hs, bar, 64 * ks, P.t[h].begin);
                            for (int a = 0; a < 4; ++a)
                                tma_load_rows(st + 2 * kXBytes + a * kr * 128, map_b, bar, n0 + 64 * a,
                                              P.ad[h].row_off + 64 * ks, kr);
                            ++g;
                        }
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        uint32_t g = 0, u = 0;
        bool ok = true;
        auto take_stage = [&]() -> uint32_t {  // smem address of the stage, 0 on abort
            const uint32_t s = g % kStages, ph = (g / kStages) & 1u;
            if (!mbar_wait(&S.full[s], ph, S.abort, segs.status)) return 0u;
            tc_fence_after();
            return smem_u32(S.stage + s * kStageBytes);
        };
        auto release_stage = [&]() {
            umma_commit(&S.empty[g % kStages]);
            ++g;
        };
        // one task's MMAs (lane 0); false on abort
        auto mma_task = [&](int64_t k) -> bool {
            bool ok = true;
            const Task t = task_of(k, n_tiles, args);
            // every earlier task's epilogue has read TMEM
            if (!mbar_wait(S.tempty, (u & 1u) ^ 1u, S.abort, segs.status)) return false;
            tc_fence_after();
            if (t.kind == 1) {
                const AdapterInfo ad = load_adapter(tab, LOAD_TILE(segs, t.m).adapter, nullptr);
                const int32_t rp = rpad16(ad.rank);
                const uint32_t idesc = make_idesc_bf16(128, (uint32_t)rp, false, false);
                for (int32_t kb = 0; kb < kb_n; ++kb) {
                    const uint32_t st = take_stage();
                    if (st == 0u) {
                        ok = false;
                        break;
                    }
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tmem_base, make_desc(st + 32u * kk, 16, 1024, kSwizzle128),
                                  make_desc(st + 2 * kXBytes + 32u * kk, 16, 1024, kSwizzle128), idesc,
                                  (kb | kk) != 0 ? 1u : 0u);
                    release_stage();
                }
            } else {
                const Pair P = load_pair(tab, segs, t.m, n_tiles);
                const uint32_t idesc = make_idesc_bf16(128, kBN, false, false);
                for (int32_t kb = 0; kb < kb_n; ++kb) {
                    const uint32_t st = take_stage();
                    if (st == 0u) {
                        ok = false;
                        break;
                    }
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bdesc = make_desc(st + 2 * kXBytes + 32u * kk, 16, 1024, kSwizzle128);
                        const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
                        umma_bf16(tmem_base, make_desc(st + 32u * kk, 16, 1024, kSwizzle128), bdesc, idesc, acc);
                        if (P.has1)
                            umma_bf16(tmem_base + 256u, make_desc(st + kXBytes + 32u * kk, 16, 1024, kSwizzle128),
                                      bdesc, idesc, acc);
                    }
                    release_stage();
                }
                const uint32_t idesc_d = make_idesc_bf16(128, kBN, false, true);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int32_t ns = ok ? delta_stages(P.ad[h]) : 0;
                    const int32_t rp = rpad16(P.ad[h].rank);
                    for (int32_t ks = 0; ks < ns; ++ks) {
                        const int32_t kr = min(64, rp - 64 * ks);
                        const uint32_t st = take_stage();
                        if (st == 0u) {
                            ok = false;
                            break;
                        }
                        for (int kk = 0; kk < kr / 16; ++kk)
                            umma_bf16(tmem_base + 256u * h, make_desc(st + 32u * kk, 16, 1024, kSwizzle128),
                                      make_desc(st + 2 * kXBytes + 2048u * kk, (uint32_t)kr * 128u, 1024,
                                                kSwizzle128),
                                      idesc_d, 1u);
                        release_stage();
                    }
                }
            }
            if (!ok) return false;
            umma_commit(S.tfull);
            ++u;
            return true;
        };
        // the whole warp walks the ring (warp-uniform waits); lane 0 issues
        for (uint32_t i = 0; ok; ++i) {
            const int64_t k = next_task_warp(S, i, segs.status);
            if (k < 0) break;
            if (lane == 0) ok = mma_task(k);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
        if (lane == 0) {
            umma_commit(S.done);
            uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(S.done, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        // Each warp reads its 32 rows of the accumulator and hands TMEM back to
        // the MMA warp as soon as its last read is done.  Full tiles leave
        // through a 128 x 64 staging block per half and TMA stores (one store
        // leader per half); short tiles (the end of a segment) with plain
        // stores of the valid rows.
        const int half = (warp - 2) >> 2;
        const uint32_t lane_base = 32u * (warp & 3);
        const int32_t row = (int32_t)lane_base + lane;
        const uint32_t tb = tmem_base + (lane_base << 16);
        const int32_t d_out = tab.d_out, r_max = tab.r_max;
        const bool leader = (warp & 3) == 2 && lane == 0;
        uint8_t *ybuf = S.ybuf + half * kYBytes;
        uint32_t u = 0, js = 0;  // tasks seen; stores of this half issued
        for (uint32_t i = 0;; ++i) {
            const int64_t k = next_task_warp(S, i, segs.status);
            if (k < 0) break;
            const Task t = task_of(k, n_tiles, args);
            if (!mbar_wait_warp(S.tfull, u & 1u, S.abort, segs.status)) break;
            tc_fence_after();
            ++u;
            if (t.kind == 1) {
                const Tile T = LOAD_TILE(segs, t.m);
                const AdapterInfo ad = load_adapter(tab, T.adapter, nullptr);
                if (half == 0) {
                    // h of this warp's 32 rows: fp32 H by token and bf16 s_i h hand-off,
                    // 64 columns at a time; TMEM goes back after the last block's reads
                    const int32_t rp = rpad16(ad.rank);
                    const int32_t n_blk = rp > 64 ? 2 : 1;
                    const bool valid = row < T.rows;
                    const int64_t tok = (int64_t)T.begin + row;
                    const float sc = ad.scale;
                    for (int32_t blk = 0; blk < 2; ++blk) {
                        const int32_t c0 = 64 * blk;
                        uint32_t hv[4][16];
                        if (blk < n_blk) {
#pragma unroll
                            for (int c = 0; c < 4; ++c)
                                if (c0 + 16 * c < rp) tmem_ld16(tb + (uint32_t)(c0 + 16 * c), hv[c]);
                            tmem_ld_wait();
                        }
                        if (blk == n_blk - 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(S.tempty);
                        }
                        if (!valid || c0 >= args.rw) continue;
                        // columns at or past rp were not loaded: every value is masked by col < rank
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                hv[c][e] = c0 + 16 * c + e < ad.rank ? hv[c][e] : 0u;
                        if (args.H != nullptr) {
                            float *hr = args.H + tok * r_max + c0;
                            if ((r_max & 3) == 0) {
#pragma unroll
                                for (int c = 0; c < 4; ++c)
#pragma unroll
                                    for (int q = 0; q < 4; ++q)
                                        if (c0 + 16 * c + 4 * q < r_max)
                                            *reinterpret_cast<uint4 *>(hr + 16 * c + 4 * q) =
                                                make_uint4(hv[c][4 * q], hv[c][4 * q + 1], hv[c][4 * q + 2],
                                                           hv[c][4 * q + 3]);
                            } else {
#pragma unroll
                                for (int c = 0; c < 4; ++c)
#pragma unroll
                                    for (int e = 0; e < 16; ++e)
                                        if (c0 + 16 * c + e < r_max) hr[16 * c + e] = __uint_as_float(hv[c][e]);
                            }
                        }
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint32_t w[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e)
                                w[e] = pack_bf16(sc * __uint_as_float(hv[c][2 * e]), sc * __uint_as_float(hv[c][2 * e + 1]));
                            uint4 *dst = reinterpret_cast<uint4 *>(args.hs + tok * args.rw + c0 + 16 * c);
                            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                        }
                    }
                    asm volatile("fence.proxy.async.global;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        __threadfence();
                        asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(args.ready + t.m) : "memory");
                    }
                } else {
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(S.tempty);
                }
                continue;
            }
            const Pair P = load_pair(tab, segs, t.m, n_tiles);
            const bool present = half == 0 || P.has1;
            const Tile Th = half ? P.t[1] : P.t[0];
            const int32_t n0 = kBN * t.j;
            if (present && Th.rows == 128) {
                // full tile: four 64-column chunks through the staging block
                const int32_t n_chunks = min(4, (d_out - n0 + 63) / 64);
                bool sok = true;
                for (int32_t c = 0; c < n_chunks; ++c) {
                    uint32_t v[4][16];
#pragma unroll
                    for (int q = 0; q < 4; ++q) tmem_ld16(tb + 256u * half + 64u * c + 16u * q, v[q]);
                    tmem_ld_wait();
                    if (c == n_chunks - 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(S.tempty);
                    }
                    // the previous store of this half has finished reading the block
                    if (!mbar_wait_warp(&S.sfree[half], (js & 1u) ^ 1u, S.abort, segs.status)) {
                        sok = false;
                        if (c < n_chunks - 1) {  // TMEM still goes back
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(S.tempty);
                        }
                        break;
                    }
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint32_t *a8 = &v[q >> 1][(q & 1) * 8];
                        *reinterpret_cast<uint4 *>(ybuf + sw128_offset((uint32_t)row, (uint32_t)q)) =
                            make_uint4(pack_bf16(__uint_as_float(a8[0]), __uint_as_float(a8[1])),
                                       pack_bf16(__uint_as_float(a8[2]), __uint_as_float(a8[3])),
                                       pack_bf16(__uint_as_float(a8[4]), __uint_as_float(a8[5])),
                                       pack_bf16(__uint_as_float(a8[6]), __uint_as_float(a8[7])));
                    }
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&S.sfull[half]);
                    if (leader) {
                        if (mbar_wait(&S.sfull[half], js & 1u, S.abort, segs.status)) {
                            tma_store_2d(&map_y, ybuf, n0 + 64 * c, Th.begin);
                            bulk_wait_read0();
                        }
                        mbar_arrive(&S.sfree[half]);
                    }
                    __syncwarp();
                    ++js;
                }
                if (!sok) break;
            } else if (present) {
                // short tile: plain stores of the valid rows
                const bool valid = row < Th.rows;
                uint16_t *yr = args.y + ((int64_t)Th.begin + row) * d_out + n0;
#pragma unroll 1
                for (int32_t c0 = 0; c0 < kBN; c0 += 32) {
                    uint32_t v[2][16];
                    tmem_ld16(tb + 256u * half + (uint32_t)c0, v[0]);
                    tmem_ld16(tb + 256u * half + (uint32_t)c0 + 16u, v[1]);
                    tmem_ld_wait();
                    if (!valid) continue;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (n0 + c0 + 8 * q >= d_out) break;
                        const uint32_t *a8 = &v[q >> 1][(q & 1) * 8];
                        *reinterpret_cast<uint4 *>(yr + c0 + 8 * q) =
                            make_uint4(pack_bf16(__uint_as_float(a8[0]), __uint_as_float(a8[1])),
                                       pack_bf16(__uint_as_float(a8[2]), __uint_as_float(a8[3])),
                                       pack_bf16(__uint_as_float(a8[4]), __uint_as_float(a8[5])),
                                       pack_bf16(__uint_as_float(a8[6]), __uint_as_float(a8[7])));
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(S.tempty);
            } else {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(S.tempty);
            }
        }
        if (leader) bulk_wait0();  // every store of this half has landed
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

size_t base_workspace_bytes(int32_t T, int32_t r_max, int32_t max_tiles)
{
    const size_t hs = ((size_t)T * handoff_cols(r_max) * 2 + 255) & ~size_t(255);
    return hs + (((size_t)(max_tiles + 1) * 4 + 255) & ~size_t(255));  // ready counters + claim counter
}

lora_status_t tc_base_fwd(void *y, float *H, const void *x, const void *W, void *ws, const lora_adapter_table &tab,
                          const lora_segments &segs, cudaStream_t stream)
{
    if (segs.n_tokens == 0 || segs.max_tiles == 0) return LORA_OK;
    const int32_t T = segs.n_tokens;
    const int32_t rw = handoff_cols(tab.r_max);
    BaseArgs args;
    args.y = static_cast<uint16_t *>(y);
    args.H = H;
    args.hs = static_cast<uint16_t *>(ws);
    args.ready = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(ws) +
                                             (((size_t)T * rw * 2 + 255) & ~size_t(255)));
    args.claim = args.ready + segs.max_tiles;
    args.rw = rw;
    args.n_col = (tab.d_out + kBN - 1) / kBN;

    CUtensorMap map_x, map_w, map_hs, map_y;
    WMaps map_a, map_b;
    if (!make_tmap_bf16_2d(&map_x, x, (uint64_t)tab.d_in, (uint64_t)T, 64, 128, true) ||
        !make_tmap_bf16_2d(&map_w, W, (uint64_t)tab.d_in, (uint64_t)tab.d_out, 64, 256, true) ||
        !make_tmap_bf16_2d(&map_hs, args.hs, (uint64_t)rw, (uint64_t)T, 64, 128, true) ||
        !make_tmap_bf16_2d(&map_y, y, (uint64_t)tab.d_out, (uint64_t)T, 64, 128, true) ||
        !make_wmaps(&map_a, tab.A, (uint64_t)tab.d_in, (uint64_t)tab.sum_r) ||
        !make_wmaps(&map_b, tab.B, (uint64_t)tab.d_out, (uint64_t)tab.sum_r))
        return LORA_ERR_CUDA;
    if (cudaFuncSetAttribute(tc_base_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
        cudaSuccess)
        return LORA_ERR_CUDA;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc_base_kernel, kThreads, kSmemBytes) != cudaSuccess ||
        per_sm < 1)
        return LORA_ERR_UNSUPPORTED;
    const int sms = sm_count();
    const int64_t pairs = (segs.max_tiles + 1) / 2;
    const int64_t want = pairs * (2 + args.n_col);
    const int grid = (int)(want < sms ? want : sms);  // one CTA per SM (all resident: cooperative)
    args.ahead = (grid + args.n_col - 1) / args.n_col + 1;

    if (cudaMemsetAsync(args.ready, 0, (size_t)(segs.max_tiles + 1) * 4, stream) != cudaSuccess)
        return LORA_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, tc_base_kernel, map_x, map_w, map_hs, map_y, map_a, map_b, args, tab, segs) !=
        cudaSuccess)
        return LORA_ERR_CUDA;
    return LORA_OK;
}

}  // namespace lora
