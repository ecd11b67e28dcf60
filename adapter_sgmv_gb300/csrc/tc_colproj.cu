// tc_colproj.cu -- case ii (expand, dX): the kernel and its launchers.  The
// kernel body and its design are in tc_colproj.cuh.
#define LORA_DBG_FILE 3
#include "tc_colproj.cuh"

namespace lora {
namespace {

using namespace colproj;

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
    extern __shared__ uint8_t smem_raw[];
    const Smem S = carve(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
    body<kLoader, kEpi, kGather, kClaim, false>(S, tmem_base, map_w, map_hi, map_lo, map_y, out, d, in, tab, segs,
                                               first, Fused{});

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
