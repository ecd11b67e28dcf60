// tc_fwd.cu -- the packed forward in one persistent launch (PLoRA technical
// summary, "2. LoRA Execution Engine", Packed LoRA Kernels: the adapters of a
// packed batch run as one kernel): the shrink of every routing tile (case i)
// and then the expand of every (tile, 1024-column part) item (case ii).
//
// Run as two launches, the expand cannot start before the last shrink tile
// is done: with 256 tiles on 152 SMs the shrink's second wave leaves a third
// of the SMs idle, and the expand's first loads wait for the launch boundary.
// Here every CTA claims tasks from one counter in index order: the tiles
// (0 .. n_tiles - 1) first, then the expand items.  A CTA runs the case i body
// for the tiles it claims; the first index past the tiles that its claimer
// takes ends that phase, and after a CTA-wide barrier the same CTA runs the
// case ii body for that index and the items it claims next.  An expand item
// waits (bounded) for its tile's ready count, which each of the four case i
// epilogue warps raises once its rows of the tile's bf16 hand-off rows are
// written.  The tile has a lower index than every item that reads it and is
// claimed by a CTA that is running, so the unfinished task with the lowest
// index can always proceed: the waits cannot form a cycle, whether or not all
// CTAs are resident.
//
// Shared memory: the two bodies use the same data region one after the other
// (case ii's layout, the larger), each with its own barriers; TMEM: 512
// columns (case i uses the first 256).  Warps: case i's 11 (six producers,
// the MMA warp, four epilogue warps); case ii uses warps 0..9.
#define LORA_DBG_FILE 8
#include "tc_colproj.cuh"
#include "tc_rowproj.cuh"

namespace lora {
namespace {

using namespace tc;

constexpr int kThreads = rowproj::kThreads;
static_assert(colproj::threads_of<false, 8>() <= kThreads, "case ii's roles fit in case i's warps");
static_assert(rowproj::kStages * (size_t)rowproj::kStageBytes <=
                  colproj::kWStages * (size_t)colproj::kWBytes + 2 * (size_t)colproj::kABytes +
                      colproj::kYStages * (size_t)colproj::kYBytes,
              "case i's stages fit in case ii's data region");
constexpr size_t kSmemBytes = colproj::kSmemBytes;
constexpr uint32_t kTmemCols = 512;
constexpr int kTmemWarp = rowproj::kMmaWarp;

struct FwdArgs {
    int32_t *claim;  // the task counter, zero at launch
    int32_t *ready;  // [max_tiles] ready counts, zero at launch
};

template <bool kGather>
__global__ void __launch_bounds__(kThreads, 1)
tc_fwd_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ WMaps map_a,
              const __grid_constant__ WMaps map_b, const __grid_constant__ CUtensorMap map_hi,
              const __grid_constant__ CUtensorMap map_lo, const __grid_constant__ CUtensorMap map_y,
              const uint16_t *__restrict__ x, uint16_t *__restrict__ y, rowproj::RowOut o, colproj::ColIn in,
              FwdArgs f, lora_adapter_table tab, lora_segments segs)
{
    extern __shared__ uint8_t smem_raw[];
    const colproj::Smem CS = colproj::carve(smem_raw);
    // case i's view: its stages at the start of the data region, its barriers,
    // its claim ring and the hand-over index in the spare end of case ii's
    // barrier block
    rowproj::Smem RS;
    RS.act = CS.w;
    RS.w = CS.w + rowproj::kStages * rowproj::kActBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(CS.wfull) + 512);
    RS.full = bars;
    RS.empty = RS.full + rowproj::kStages;
    RS.tfull = RS.empty + rowproj::kStages;
    RS.tempty = RS.tfull + 2;
    RS.done = RS.tempty + 2;
    RS.tmem_holder = CS.tmem_holder;
    RS.abort = CS.abort;
    rowproj::Fused F1;
    F1.ring.full = RS.done + 1;
    F1.ring.empty = F1.ring.full + kClaimSlots;
    F1.ring.slot = reinterpret_cast<volatile int32_t *>(F1.ring.empty + kClaimSlots);
    F1.carry = F1.ring.slot + kClaimSlots;
    F1.claim = f.claim;
    F1.ready = f.ready;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the claimer's first task, claimed before the set-up so that its round trip overlaps it
    F1.first = warp == 0 && lane == 0 ? claim_first(f.claim) : 0;

    if (threadIdx.x == 0) {
        for (int i = 0; i < rowproj::kStages; ++i) {
            mbar_init(&RS.full[i], 33);
            mbar_init(&RS.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&RS.tfull[i], 1);
            mbar_init(&RS.tempty[i], 4);
        }
        mbar_init(RS.done, 1);
        for (int i = 0; i < kClaimSlots; ++i) {  // case i: claimed by warp 0, read by the other ten warps
            mbar_init(&F1.ring.full[i], 1);
            mbar_init(&F1.ring.empty[i], (rowproj::kProd - 1) + 1 + 4);
        }
        for (int i = 0; i < colproj::kWStages; ++i) {
            mbar_init(&CS.wfull[i], 1);
            mbar_init(&CS.wempty[i], 1);
        }
        for (int i = 0; i < colproj::kYStages; ++i) {
            mbar_init(&CS.yfull[i], 33);
            mbar_init(&CS.yempty[i], 1);
            mbar_init(&CS.ysync[i], 4);
        }
        for (uint32_t i = 0; i < colproj::kAcc; ++i) {
            mbar_init(&CS.tfull[i], 1);
            mbar_init(&CS.tempty[i], 8);
        }
        mbar_init(CS.afull, 1);
        mbar_init(CS.aempty, 1);
        mbar_init(CS.done, 1);
        for (int i = 0; i < kClaimSlots; ++i) {  // case ii: claimed by warp 0, read by the MMA thread and 8 warps
            mbar_init(&CS.claims.full[i], 1);
            mbar_init(&CS.claims.empty[i], 1 + 8);
        }
        *CS.abort = 0;
        *F1.carry = 0x7fffffff;  // no task past the tiles (yet)
        fence_barrier_init();
    }
    if (warp == kTmemWarp) {
        tmem_alloc(CS.tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *CS.tmem_holder;

    // tiles: shrink, H and the hand-off rows, each tile's ready count raised
    rowproj::body<true>(RS, tmem_base, map_x, map_a, x, tab.d_in, o, tab, segs, F1);

    tc_fence_before();
    __syncthreads();  // every role is done with the case i stages, barriers and accumulators
    tc_fence_after();
    const int32_t first = *F1.carry;

    // expand items, indices n_tiles and up
    const colproj::Fused F2{N_TILES(segs), f.ready};
    colproj::body<false, 8, kGather, true, true>(CS, tmem_base, map_b, map_hi, map_lo, map_y, y, tab.d_out, in, tab,
                                                 segs, first, F2);

    tc_fence_before();
    __syncthreads();
    if (warp == kTmemWarp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

lora_status_t tc_fwd_fused(void *y, float *H_save, const void *x, uint16_t *hi, uint16_t *lo, int32_t rw,
                           int32_t *counters, const lora_adapter_table &tab, const lora_segments &segs,
                           cudaStream_t stream)
{
    if (segs.n_tokens == 0 || segs.max_tiles == 0) return LORA_OK;
    CUtensorMap map_x, map_hi, map_lo, map_y;
    WMaps map_a, map_b;
    const uint64_t T = (uint64_t)segs.n_tokens;
    if (!make_tmap_bf16_2d(&map_x, x, (uint64_t)tab.d_in, T, 64, 128, true) ||
        !make_wmaps(&map_a, tab.A, (uint64_t)tab.d_in, (uint64_t)tab.sum_r) ||
        !make_wmaps(&map_b, tab.B, (uint64_t)tab.d_out, (uint64_t)tab.sum_r) ||
        !make_tmap_bf16_2d(&map_hi, hi, (uint64_t)rw, T, 64, 128, true) ||
        !make_tmap_bf16_2d(&map_lo, lo, (uint64_t)rw, T, 64, 128, true) ||
        !make_tmap_bf16_2d(&map_y, y, (uint64_t)tab.d_out, T, 64, 128, true))
        return LORA_ERR_CUDA;
    // the task counter and the tiles' ready counts start at zero
    if (cudaMemsetAsync(counters, 0, (size_t)(1 + segs.max_tiles) * sizeof(int32_t), stream) != cudaSuccess)
        return LORA_ERR_CUDA;
    const rowproj::RowOut o{H_save, hi, lo, rw, 0.f, 1, 0, nullptr, nullptr, 0};
    const colproj::ColIn in{nullptr, 1.f, 1, counters};
    const FwdArgs f{counters, counters + 1};
    const int grid = sm_count();
    auto *kernel = segs.sorted != 0 ? tc_fwd_kernel<false> : tc_fwd_kernel<true>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess)
        return LORA_ERR_CUDA;
    kernel<<<grid, kThreads, kSmemBytes, stream>>>(map_x, map_a, map_b, map_hi, map_lo, map_y,
                                                   static_cast<const uint16_t *>(x), static_cast<uint16_t *>(y), o,
                                                   in, f, tab, segs);
    return cudaGetLastError() == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

}  // namespace lora
