// tc_rowproj.cu -- case i (shrink, dh): the kernel, the combine kernel of the
// split along d, the bf16 copy of a saved H, and their launchers.  The kernel
// body and its design are in tc_rowproj.cuh.
#define LORA_DBG_FILE 2
#include "tc_rowproj.cuh"

namespace lora {
namespace {

using namespace rowproj;

__global__ void __launch_bounds__(kThreads, 1)
tc_rowproj_kernel(const __grid_constant__ CUtensorMap map_act, const __grid_constant__ WMaps map_w,
                  const uint16_t *__restrict__ act, int32_t d, RowOut o, lora_adapter_table tab,
                  lora_segments segs)
{
    extern __shared__ uint8_t smem_raw[];
    const Smem S = carve(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    zero_claims(o.zero_claims, o.n_zero);

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&S.full[i], 33);  // lane 0's expect-tx arrive + one per lane of the slot's producer warp
            mbar_init(&S.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&S.tfull[i], 1);
            mbar_init(&S.tempty[i], 4);
        }
        mbar_init(S.done, 1);
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
    body<false>(S, tmem_base, map_act, map_w, act, d, o, tab, segs, Fused{});

    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// Split case i: the parts' partials added in part order (the sum does not
// depend on timing) and written as the unsplit epilogue writes them.  One CTA
// per tile, one thread per (row, 4 columns).
__global__ void __launch_bounds__(256) rowproj_combine_kernel(RowOut o, lora_adapter_table tab, lora_segments segs)
{
    const int32_t n_tiles = N_TILES(segs), r_max = tab.r_max, T_all = segs.n_tokens;
    for (int32_t ti = blockIdx.x; ti < n_tiles; ti += gridDim.x) {
        const Tile T = LOAD_TILE(segs, ti);
        const AdapterInfo ad = load_adapter(tab, T.adapter, nullptr);
        if (!ad.ok) continue;
        const int32_t r = ad.rank, rp = rpad16(r), n4 = rp / 4;
        for (int32_t i = threadIdx.x; i < T.rows * n4; i += blockDim.x) {
            const int32_t m = i / n4, k = 4 * (i % n4);
            const int64_t p = (int64_t)T.begin + m;
            float4 v = __ldcs(reinterpret_cast<const float4 *>(o.part + p * o.part_ld + k));
            for (int32_t q = 1; q < o.splits; ++q) {
                const float4 w = __ldcs(reinterpret_cast<const float4 *>(o.part + ((int64_t)q * T_all + p) * o.part_ld + k));
                v.x += w.x;
                v.y += w.y;
                v.z += w.z;
                v.w += w.w;
            }
            const float f[4] = {v.x, v.y, v.z, v.w};
            if (o.f32 != nullptr) {
                float *row = o.f32 + (int64_t)PERM_AT(segs, p) * r_max;
                for (int e = 0; e < 4; ++e)
                    if (k + e < r_max) row[k + e] = f[e];
                if (k + 4 == rp)  // the row's zero tail past the rank rounded up to 16
                    for (int32_t e = rp; e < r_max; ++e) row[e] = 0.f;
            }
            if (o.hi != nullptr) {
                const uint32_t h01 = pack_bf16(f[0], f[1]), h23 = pack_bf16(f[2], f[3]);
                *reinterpret_cast<uint2 *>(o.hi + p * o.rw + k) = make_uint2(h01, h23);
                if (o.lo != nullptr)
                    *reinterpret_cast<uint2 *>(o.lo + p * o.rw + k) =
                        make_uint2(pack_bf16(f[0] - bf16lo(h01), f[1] - bf16hi(h01)),
                                   pack_bf16(f[2] - bf16lo(h23), f[3] - bf16hi(h23)));
            }
        }
    }
}

lora_status_t launch_rowproj(const void *act, const void *w, int32_t d, RowOut o, const lora_adapter_table &tab,
                             const lora_segments &segs, float *part, cudaStream_t stream)
{
    if (segs.n_tokens == 0 || segs.max_tiles == 0) return LORA_OK;
    o.splits = part != nullptr ? rowproj_splits(segs.max_tiles, d) : 1;
    o.part_ld = rowproj_part_ld(tab.r_max);
    o.part = part;
    CUtensorMap map_act;
    WMaps map_w;
    if (!make_tmap_bf16_2d(&map_act, act, (uint64_t)d, (uint64_t)segs.n_tokens, 64, 128, true) ||
        !make_wmaps(&map_w, w, (uint64_t)d, (uint64_t)tab.sum_r))
        return LORA_ERR_CUDA;
    if (cudaFuncSetAttribute(tc_rowproj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
        cudaSuccess)
        return LORA_ERR_CUDA;
    const int sms = sm_count();
    const int64_t units = (int64_t)segs.max_tiles * o.splits;
    const int grid = units < sms ? (int)units : sms;
    tc_rowproj_kernel<<<grid, kThreads, kSmemBytes, stream>>>(map_act, map_w, static_cast<const uint16_t *>(act), d,
                                                              o, tab, segs);
    if (cudaGetLastError() != cudaSuccess) return LORA_ERR_CUDA;
    if (o.splits > 1) {
        const int cgrid = segs.max_tiles < 4 * sms ? segs.max_tiles : 4 * sms;
        rowproj_combine_kernel<<<cgrid, 256, 0, stream>>>(o, tab, segs);
        if (cudaGetLastError() != cudaSuccess) return LORA_ERR_CUDA;
    }
    return LORA_OK;
}

}  // namespace

namespace {

// A saved fp32 H (by token, stride r_max) to the bf16 hand-off rows (by perm
// position, stride rw, zero from each adapter's rank up to the rank rounded to
// 16, unwritten past that): one CTA per tile,
// one thread per (row, 8 columns).  It runs beside case i (dh), so its CTAs
// are kept small (1024-thread CTAs converted faster alone but crowded out dh's).
__global__ void __launch_bounds__(256) h_to_bf16_kernel(const float *__restrict__ H, uint16_t *__restrict__ hb,
                                                        int32_t rw, int32_t *zero, int32_t n_zero,
                                                        lora_adapter_table tab, lora_segments segs)
{
    zero_claims(zero, n_zero);  // the counters of the kernels after this one in the call
    const int32_t n_tiles = N_TILES(segs);
    const int32_t r_max = tab.r_max;
    const bool vec = (r_max & 3) == 0 && (reinterpret_cast<uintptr_t>(H) & 15u) == 0;
    for (int32_t ti = blockIdx.x; ti < n_tiles; ti += gridDim.x) {
        const Tile T = LOAD_TILE(segs, ti);
        const AdapterInfo ad = load_adapter(tab, T.adapter, nullptr);
        const int32_t r = ad.ok ? ad.rank : 0;
        const int32_t rp8 = (r + 15) / 16 * 2;  // 8-column pieces up to the rank rounded to 16; past it no product reads
        for (int32_t i = threadIdx.x; i < T.rows * rp8; i += blockDim.x) {
            const int32_t m = i / rp8, k = 8 * (i % rp8);
            const int64_t p = (int64_t)T.begin + m;
            const float *src = H + (int64_t)PERM_AT(segs, p) * r_max;
            float f[8];
            if (vec && k + 8 <= r) {  // two 16-byte loads
                const float4 a = __ldcs(reinterpret_cast<const float4 *>(src + k));
                const float4 b = __ldcs(reinterpret_cast<const float4 *>(src + k + 4));
                f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
                f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = k + e < r ? src[k + e] : 0.f;
            }
            *reinterpret_cast<uint4 *>(hb + p * rw + k) = make_uint4(pack_bf16(f[0], f[1]), pack_bf16(f[2], f[3]),
                                                                     pack_bf16(f[4], f[5]), pack_bf16(f[6], f[7]));
        }
    }
}

}  // namespace

lora_status_t tc_h_to_bf16(const float *H, uint16_t *hb, int32_t rw, int32_t *zero_claims, int32_t n_zero,
                           const lora_adapter_table &tab, const lora_segments &segs, cudaStream_t stream)
{
    if (segs.n_tokens == 0 || segs.max_tiles == 0) return LORA_OK;
    const int sms = sm_count();
    const int grid = segs.max_tiles < 4 * sms ? segs.max_tiles : 4 * sms;
    h_to_bf16_kernel<<<grid, 256, 0, stream>>>(H, hb, rw, zero_claims, n_zero, tab, segs);
    return cudaGetLastError() == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

int32_t rowproj_splits(int32_t max_tiles, int32_t d)
{
    // 2 or 4 parts when there are too few tiles to fill GB300's 152 SMs, each
    // at least 8 blocks of 64 columns deep (the choice depends on the sizes alone)
    const int32_t nk = (d + 63) / 64;
    int32_t sp = max_tiles <= 38 ? 4 : max_tiles <= 76 ? 2 : 1;
    while (sp > 1 && nk < 8 * sp) sp /= 2;
    return sp;
}
int32_t rowproj_part_ld(int32_t r_max) { return (r_max + 15) & ~15; }

lora_status_t tc_shrink(const void *x, const lora_adapter_table &tab, const lora_segments &segs, float *H,
                        uint16_t *hi, uint16_t *lo, int32_t rw, float *part, int32_t *zero_claims, int32_t n_zero,
                        cudaStream_t stream)
{
    RowOut o{H, hi, lo, rw, 0.f, 1, 0, nullptr, zero_claims, n_zero};
    return launch_rowproj(x, tab.A, tab.d_in, o, tab, segs, part, stream);
}

lora_status_t tc_dh(const void *dY, const lora_adapter_table &tab, const lora_segments &segs, uint16_t *dh_bf16,
                    int32_t rw, float *part, int32_t *zero_claims, int32_t n_zero, cudaStream_t stream)
{
    RowOut o{nullptr, dh_bf16, nullptr, rw, 1.f, 1, 0, nullptr, zero_claims, n_zero};
    return launch_rowproj(dY, tab.B, tab.d_out, o, tab, segs, part, stream);
}

}  // namespace lora
