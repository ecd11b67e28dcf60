// tc_tokred.cu -- cases iii and iv on the 5th-generation tensor cores: the
// reductions over tokens that produce the adapters' weight gradients, tiled
// along the hidden dimension and split along tokens (PLoRA technical summary,
// "2. LoRA Execution Engine").
//
//   dB  dB_i[o, k] = s_i sum_{t in i} dY[t, o] H[t, k]     (B layout [d_out, r_i])
//   dA  dA_i[k, j] =     sum_{t in i} dH[t, k] X[t, j]     (A layout [r_i, d_in])
//
// The MMA is G^T-free: D[n, k] (M = 128 columns n of d, N = r_pad, K = tokens)
// = act^T (MN-major: the activation block read as stored, 128-byte swizzle) x
// h (MN-major interleaved, converted from fp32 to bf16 by loader warps).  A
// work item is (span of <= LORA_SPAN_TOKENS tokens of one adapter, 512 columns
// of d): four TMEM accumulators of up to 128 columns, one per 128-column
// chunk, accumulate over the span in 32-token stages, then are added into the
// zero-initialised output with fp32 reductions (spans of one adapter add up).
//
// Warp roles (256 threads): 0 activation loads (TMA, or cp.async gather for
// non-consecutive tokens), 1 MMA + TMEM owner, 2..5 epilogue, 6..7 h loaders.
#include "internal.h"
#include "tc_common.cuh"
#include "tc_host.h"

namespace lora {
namespace {

using namespace tc;

constexpr int kThreads = 256;
constexpr int kStages = 4;
constexpr int kLag = 2;
constexpr int kTok = 32;                                  // tokens per stage
constexpr int kRange = 512;                               // columns of d per work item
constexpr uint32_t kActBytes = kTok * kRange * 2;         // 8 boxes of [64 cols x 32 tokens]
constexpr uint32_t kHBytes = kTok * LORA_MAX_RANK * 2;
constexpr uint32_t kStageBytes = kActBytes + kHBytes;
constexpr uint32_t kTmemCols = 512;
constexpr size_t kSmemBytes = 1024 + kStages * (size_t)kStageBytes + 256;

struct Smem {
    uint8_t *act, *h;
    uint64_t *afull, *hfull, *empty, *tfull, *tempty, *done;
    uint32_t *tmem_holder;
    volatile int32_t *abort;
};

LORA_DEV Smem carve(uint8_t *raw)
{
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    Smem s;
    s.act = base;
    s.h = base + kStages * kActBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(s.h + kStages * kHBytes);
    s.afull = bars;
    s.hfull = bars + kStages;
    s.empty = bars + 2 * kStages;
    s.tfull = bars + 3 * kStages;
    s.tempty = s.tfull + 1;
    s.done = s.tempty + 1;
    s.tmem_holder = reinterpret_cast<uint32_t *>(s.done + 1);
    s.abort = reinterpret_cast<volatile int32_t *>(s.tmem_holder + 1);
    return s;
}

LORA_DEV int32_t rpad16(int32_t r) { return (r + 15) & ~15; }

struct Item {
    Tile span;
    AdapterInfo ad;
    int32_t n_base, n_chunks, n_stages;
};

LORA_DEV Item load_item(const lora_adapter_table &tab, const lora_segments &segs, int32_t it, int32_t n_ranges,
                        int32_t d)
{
    Item I;
    I.span = load_tile(segs.spans, it / n_ranges);
    I.ad = load_adapter(tab, I.span.adapter, segs.status);
    I.n_base = (it % n_ranges) * kRange;
    I.n_chunks = min(4, (d - I.n_base + 127) / 128);
    I.n_stages = (I.span.rows + kTok - 1) / kTok;
    return I;
}

template <bool kDA>
__global__ void __launch_bounds__(kThreads, 1)
tc_tokred_kernel(const __grid_constant__ CUtensorMap map_act, float *__restrict__ G,
                 const uint16_t *__restrict__ act, const float *__restrict__ h, lora_adapter_table tab,
                 lora_segments segs)
{
    extern __shared__ uint8_t smem_raw[];
    const Smem S = carve(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&S.afull[i], 33);
            mbar_init(&S.hfull[i], 2);
            mbar_init(&S.empty[i], 1);
        }
        mbar_init(S.tfull, 1);
        mbar_init(S.tempty, 4);
        mbar_init(S.done, 1);
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
    const int32_t d = kDA ? tab.d_in : tab.d_out;
    const int32_t n_ranges = (d + kRange - 1) / kRange;
    const int32_t n_items = *segs.n_spans * n_ranges;
    const int32_t r_max = tab.r_max;

    if (warp == 0) {
        // ------------------------------------------------------------ activation producer
        if (lane == 0) prefetch_tensormap(&map_act);
        uint32_t g = 0;
        bool ok = true;
        for (int32_t it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            const Item I = load_item(tab, segs, it, n_ranges, d);
            if (!I.ad.ok) continue;
            const int32_t p0 = I.span.begin;
            const bool contiguous = (I.span.flags & 1) != 0;
            const int32_t t0 = segs.perm[p0];
            for (int32_t st = 0; st < I.n_stages; ++st) {
                const uint32_t s = g % kStages, ph = (g / kStages) & 1u;
                if (!mbar_wait(&S.empty[s], ph ^ 1u, S.abort, segs.status)) {
                    ok = false;
                    break;
                }
                uint8_t *act_s = S.act + s * kActBytes;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&S.afull[s], contiguous ? (uint32_t)I.n_chunks * 8192u : 0u);
                    if (contiguous)
                        for (int b = 0; b < 2 * I.n_chunks; ++b)
                            tma_load_2d(act_s + b * 4096, &map_act, &S.afull[s], I.n_base + 64 * b,
                                        t0 + kTok * st);
                }
                if (!contiguous) {
                    // token row m, 16-byte chunk c of the 512 columns: box b = c / 8 holds
                    // columns 64 b .. 64 b + 63 as a [32 x 128 B] 128-byte-swizzled block
                    const int nch = I.n_chunks * 16;
                    for (int e = lane; e < kTok * nch; e += 32) {
                        const int m = e / nch, c = e % nch;
                        const int p = p0 + kTok * st + m;
                        const bool v = (kTok * st + m < I.span.rows) && (I.n_base + 8 * c < d);
                        const int32_t t = v ? segs.perm[p] : 0;
                        const uint16_t *src = v ? act + (int64_t)t * d + I.n_base + 8 * c : act;
                        cp_async_16(act_s + (c >> 3) * 4096 + sw128_offset((uint32_t)m, (uint32_t)(c & 7)), src, v);
                    }
                }
                cp_async_commit();
                if (g >= (uint32_t)kLag) {
                    cp_async_wait<kLag>();
                    fence_proxy_async();
                    mbar_arrive(&S.afull[(g - kLag) % kStages]);
                }
                ++g;
            }
        }
        cp_async_wait<0>();
        fence_proxy_async();
        for (uint32_t u = g > (uint32_t)kLag ? g - kLag : 0u; u < g; ++u) mbar_arrive(&S.afull[u % kStages]);
        if (!ok && lane == 0) {
            for (uint32_t u = g > (uint32_t)kStages ? g - kStages : 0u; u < g; ++u) {
                uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&S.afull[u % kStages], (u / kStages) & 1u) &&
                       globaltimer_ns() - t0 < kWaitLimitNs / 8) {
                }
            }
        }
    } else if (warp >= 6) {
        // ------------------------------------------------------------ h loaders (64 threads)
        // stage layout: MN-major interleaved, N = k, K = token: chunk (m, k/8) at
        // (k/8) * 512 + (m/8) * 128 + (m%8) * 16
        const int u = threadIdx.x - 6 * 32;
        const int m = u & 31;
        const bool vec = (r_max & 3) == 0;
        uint32_t g = 0;
        bool ok = true;
        for (int32_t it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            const Item I = load_item(tab, segs, it, n_ranges, d);
            if (!I.ad.ok) continue;
            const int32_t r = I.ad.rank, rp = rpad16(r);
            for (int32_t st = 0; st < I.n_stages; ++st) {
                const uint32_t s = g % kStages, ph = (g / kStages) & 1u;
                if (!mbar_wait(&S.empty[s], ph ^ 1u, S.abort, segs.status)) {
                    ok = false;
                    break;
                }
                const bool valid = kTok * st + m < I.span.rows;
                const int32_t t = valid ? segs.perm[I.span.begin + kTok * st + m] : 0;
                const float *hr = h + (int64_t)t * r_max;
                uint8_t *h_s = S.h + s * kHBytes;
                for (int kc = u >> 5; kc < rp / 8; kc += 2) {
                    float f[8];
                    if (valid && vec && 8 * kc + 8 <= r_max) {
                        const float4 a0 = *reinterpret_cast<const float4 *>(hr + 8 * kc);
                        const float4 a1 = *reinterpret_cast<const float4 *>(hr + 8 * kc + 4);
                        f[0] = a0.x; f[1] = a0.y; f[2] = a0.z; f[3] = a0.w;
                        f[4] = a1.x; f[5] = a1.y; f[6] = a1.z; f[7] = a1.w;
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = (valid && 8 * kc + e < r_max) ? hr[8 * kc + e] : 0.f;
                    }
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 8; e += 2)
                        w[e / 2] = pack_bf16(8 * kc + e < r ? f[e] : 0.f, 8 * kc + e + 1 < r ? f[e + 1] : 0.f);
                    *reinterpret_cast<uint4 *>(h_s + kc * 512 + (m >> 3) * 128 + (m & 7) * 16) =
                        make_uint4(w[0], w[1], w[2], w[3]);
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(&S.hfull[s]);
                ++g;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t g = 0, nitem = 0;
            bool ok = true;
            for (int32_t it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
                const Item I = load_item(tab, segs, it, n_ranges, d);
                if (!I.ad.ok) continue;
                const uint32_t rp = (uint32_t)rpad16(I.ad.rank);
                const uint32_t idesc = make_idesc_bf16(128, rp, true, true);
                if (!mbar_wait(S.tempty, (nitem & 1u) ^ 1u, S.abort, segs.status)) break;
                tc_fence_after();
                for (int32_t st = 0; st < I.n_stages; ++st) {
                    const uint32_t s = g % kStages, ph = (g / kStages) & 1u;
                    if (!mbar_wait(&S.afull[s], ph, S.abort, segs.status) ||
                        !mbar_wait(&S.hfull[s], ph, S.abort, segs.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(S.act + s * kActBytes);
                    const uint32_t h_base = smem_u32(S.h + s * kHBytes);
                    for (int q = 0; q < I.n_chunks; ++q) {
#pragma unroll
                        for (int kk = 0; kk < kTok / 16; ++kk) {
                            const uint64_t adesc = make_desc(a_base + 8192u * q + 2048u * kk, 4096, 1024, kSwizzle128);
                            const uint64_t bdesc = make_desc(h_base + 256u * kk, 128, 512, kInterleave);
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
        const uint32_t lane_base = 32u * (warp & 3);
        uint32_t nitem = 0;
        for (int32_t it = blockIdx.x; it < n_items; it += gridDim.x) {
            const Item I = load_item(tab, segs, it, n_ranges, d);
            if (!I.ad.ok) continue;
            const int32_t r = I.ad.rank, rp = rpad16(r);
            if (!mbar_wait(S.tfull, nitem & 1u, S.abort, segs.status)) break;
            tc_fence_after();
            const float c = kDA ? 1.0f : I.ad.scale;
            for (int q = 0; q < 4; ++q) {
                if (q >= I.n_chunks) break;
                const int32_t n = I.n_base + 128 * q + (int32_t)lane_base + lane;
                for (int c0 = 0; c0 < rp; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(tmem_base + (lane_base << 16) + 128u * q + (uint32_t)c0, v);
                    tmem_ld_wait();
                    if (n >= d) continue;
                    if (kDA) {
                        float *col = G + ((int64_t)I.ad.row_off) * d + n;
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (c0 + e < r) red_add_f32(col + (int64_t)(c0 + e) * d, c * __uint_as_float(v[e]));
                    } else {
                        float *row = G + (int64_t)I.ad.row_off * d + (int64_t)n * r;
                        if ((r & 3) == 0) {
#pragma unroll
                            for (int e = 0; e < 16; e += 4)
                                if (c0 + e < r)
                                    red_add_v4(row + c0 + e, c * __uint_as_float(v[e]), c * __uint_as_float(v[e + 1]),
                                               c * __uint_as_float(v[e + 2]), c * __uint_as_float(v[e + 3]));
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                if (c0 + e < r) red_add_f32(row + c0 + e, c * __uint_as_float(v[e]));
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(S.tempty);
            ++nitem;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <bool kDA>
lora_status_t launch_tokred(float *G, const void *act, const float *h, const lora_adapter_table &tab,
                            const lora_segments &segs, cudaStream_t stream)
{
    const int32_t d = kDA ? tab.d_in : tab.d_out;
    const size_t gbytes = (size_t)tab.sum_r * (size_t)d * sizeof(float);
    if (cudaMemsetAsync(G, 0, gbytes, stream) != cudaSuccess) return LORA_ERR_CUDA;
    if (segs.n_tokens == 0 || segs.max_spans == 0) return LORA_OK;
    CUtensorMap map_act;
    if (!make_tmap_bf16_2d(&map_act, act, (uint64_t)d, (uint64_t)segs.n_tokens, 64, kTok, true))
        return LORA_ERR_CUDA;
    if (cudaFuncSetAttribute(tc_tokred_kernel<kDA>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
        return LORA_ERR_CUDA;
    const int n_ranges = (d + kRange - 1) / kRange;
    const int64_t items = (int64_t)segs.max_spans * n_ranges;
    const int sms = sm_count();
    const int grid = items < sms ? (int)items : sms;
    tc_tokred_kernel<kDA><<<grid, kThreads, kSmemBytes, stream>>>(map_act, G, static_cast<const uint16_t *>(act), h,
                                                                   tab, segs);
    return cudaGetLastError() == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

}  // namespace

lora_status_t tc_db(float *dB, const void *dY, const float *H, const lora_adapter_table &tab,
                    const lora_segments &segs, cudaStream_t stream)
{
    return launch_tokred<false>(dB, dY, H, tab, segs, stream);
}

lora_status_t tc_da(float *dA, const float *dH, const void *X, const lora_adapter_table &tab,
                    const lora_segments &segs, cudaStream_t stream)
{
    return launch_tokred<true>(dA, X, dH, tab, segs, stream);
}

}  // namespace lora
