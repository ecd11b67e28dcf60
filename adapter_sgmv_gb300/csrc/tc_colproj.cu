// tc_colproj.cu -- case ii on the 5th-generation tensor cores: a reduction over
// the rank into a T x d result that is accumulated into a bf16 tensor, tiled
// along tokens and the hidden dimension (PLoRA technical summary, "2. LoRA
// Execution Engine").
//
//   expand  y[t, o]  += s_i sum_k H[t, k]  B_i[o, k]
//   dX      dX[t, j] +=     sum_k dH[t, k] A_i[k, j]
//
// A work item is (tile of up to 128 tokens of one adapter, a 1024-column part
// of d).  The 128 x r_pad block of H (fp32) is converted once per item into a
// bf16 A operand; for expand it is split as h = hi + lo (both bf16) and both
// halves are multiplied, so H enters the product at ~16-bit precision.  The
// weight block of every 128-column chunk is the B operand: B_i rows (K-major,
// by cp.async) for expand, A_i columns (MN-major, 128-byte swizzle, by TMA)
// for dX.  tcgen05.mma (M = 128, N = 128, K = 16) accumulates in a ring of
// four TMEM accumulators; the epilogue adds c * acc to the bf16 rows in place
// (fp32 sum, one rounding).
//
// Warp roles (320 threads): 0 weight loads, 1 MMA + TMEM owner, 2..5 epilogue,
// 6..9 load and convert the H block.
#include "internal.h"
#include "tc_common.cuh"
#include "tc_host.h"

namespace lora {
namespace {

using namespace tc;

constexpr int kThreads = 320;
constexpr int kWStages = 4;
constexpr int kLag = 2;
constexpr int kNC = 128;                              // columns per MMA chunk
constexpr int kNPart = 1024;                          // columns per work item
constexpr uint32_t kWBytes = kNC * LORA_MAX_RANK * 2;  // one weight chunk
constexpr uint32_t kHBytes = 128 * LORA_MAX_RANK * 2;  // one bf16 copy of the H block
constexpr uint32_t kAcc = 4;                          // TMEM accumulators of 128 columns
constexpr uint32_t kTmemCols = 512;
constexpr size_t kSmemBytes = 1024 + kWStages * (size_t)kWBytes + 2 * (size_t)kHBytes + 256;

struct Smem {
    uint8_t *w, *hhi, *hlo;
    uint64_t *wfull, *wempty, *tfull, *tempty, *hfull, *hempty, *done;
    uint32_t *tmem_holder;
    volatile int32_t *abort;
};

LORA_DEV Smem carve(uint8_t *raw)
{
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    Smem s;
    s.w = base;
    s.hhi = base + kWStages * kWBytes;
    s.hlo = s.hhi + kHBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(s.hlo + kHBytes);
    s.wfull = bars;
    s.wempty = bars + kWStages;
    s.tfull = bars + 2 * kWStages;
    s.tempty = s.tfull + kAcc;
    s.hfull = s.tempty + kAcc;
    s.hempty = s.hfull + 1;
    s.done = s.hempty + 1;
    s.tmem_holder = reinterpret_cast<uint32_t *>(s.done + 1);
    s.abort = reinterpret_cast<volatile int32_t *>(s.tmem_holder + 1);
    return s;
}

LORA_DEV int32_t rpad16(int32_t r) { return (r + 15) & ~15; }

struct Item {
    Tile tile;
    AdapterInfo ad;
    int32_t n_lo, n_hi;
};

LORA_DEV Item load_item(const lora_adapter_table &tab, const lora_segments &segs, int32_t it, int32_t n_parts,
                        int32_t d)
{
    Item I;
    I.tile = load_tile(segs.tiles, it / n_parts);
    I.ad = load_adapter(tab, I.tile.adapter, segs.status);
    I.n_lo = (it % n_parts) * kNPart;
    I.n_hi = min(d, I.n_lo + kNPart);
    return I;
}

template <bool kDX>
__global__ void __launch_bounds__(kThreads, 1)
tc_colproj_kernel(const __grid_constant__ CUtensorMap map_w, uint16_t *__restrict__ out,
                  const float *__restrict__ h, lora_adapter_table tab, lora_segments segs)
{
    constexpr bool kSplit = !kDX;  // expand feeds H as hi + lo
    extern __shared__ uint8_t smem_raw[];
    const Smem S = carve(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kWStages; ++i) {
            mbar_init(&S.wfull[i], 33);
            mbar_init(&S.wempty[i], 1);
        }
        for (uint32_t i = 0; i < kAcc; ++i) {
            mbar_init(&S.tfull[i], 1);
            mbar_init(&S.tempty[i], 4);
        }
        mbar_init(S.hfull, 4);
        mbar_init(S.hempty, 1);
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
    const int32_t d = kDX ? tab.d_in : tab.d_out;
    const int32_t n_parts = (d + kNPart - 1) / kNPart;
    const int32_t n_items = *segs.n_tiles * n_parts;
    const int32_t r_max = tab.r_max;

    if (warp == 0) {
        // ------------------------------------------------------------ weight producer
        if (lane == 0 && kDX) prefetch_tensormap(&map_w);
        const uint16_t *Bw = static_cast<const uint16_t *>(tab.B);
        uint32_t g = 0;
        bool ok = true;
        for (int32_t it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
            const Item I = load_item(tab, segs, it, n_parts, d);
            if (!I.ad.ok) continue;
            const int32_t r = I.ad.rank, rp = rpad16(r);
            for (int32_t n0 = I.n_lo; n0 < I.n_hi; n0 += kNC) {
                const uint32_t s = g % kWStages, ph = (g / kWStages) & 1u;
                if (!mbar_wait(&S.wempty[s], ph ^ 1u, S.abort, segs.status)) {
                    ok = false;
                    break;
                }
                uint8_t *w_s = S.w + s * kWBytes;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&S.wfull[s], kDX ? (uint32_t)rp * 256u : 0u);
                    if (kDX) {
                        // A_i[k, n0 + 64a ..] as MN-major 128B-swizzled atoms: column a at
                        // a * (rp * 128), rows k in 16-row boxes
                        for (int a = 0; a < 2; ++a)
                            for (int q = 0; q < rp / 16; ++q)
                                tma_load_2d(w_s + a * rp * 128 + q * 2048, &map_w, &S.wfull[s], n0 + 64 * a,
                                            I.ad.row_off + 16 * q);
                    }
                }
                if (!kDX) {
                    // B_i rows o = n0 .. n0+127 as the K-major operand (N = o, K = k):
                    // chunk (o, k/8) -> (k/8) * 2048 + (o/8) * 128 + (o%8) * 16
                    const uint16_t *Bi = Bw + (int64_t)I.ad.row_off * d;
                    const int nchunks = kNC * (rp / 8);
                    for (int e = lane; e < nchunks; e += 32) {
                        const int o = e & (kNC - 1), c = e >> 7;
                        const bool v = (n0 + o < d) && (8 * c < r);
                        uint8_t *dst = w_s + c * 2048 + (o >> 3) * 128 + (o & 7) * 16;
                        if ((r & 7) == 0) {
                            cp_async_16(dst, v ? Bi + (int64_t)(n0 + o) * r + 8 * c : Bw, v);
                        } else {
                            uint32_t wv[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const int k0 = 8 * c + 2 * q;
                                const uint16_t lo = (v && k0 < r) ? Bi[(int64_t)(n0 + o) * r + k0] : 0;
                                const uint16_t hi = (v && k0 + 1 < r) ? Bi[(int64_t)(n0 + o) * r + k0 + 1] : 0;
                                wv[q] = (uint32_t)lo | ((uint32_t)hi << 16);
                            }
                            *reinterpret_cast<uint4 *>(dst) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                        }
                    }
                }
                cp_async_commit();
                if (g >= (uint32_t)kLag) {
                    cp_async_wait<kLag>();
                    fence_proxy_async();
                    mbar_arrive(&S.wfull[(g - kLag) % kWStages]);
                }
                ++g;
            }
        }
        cp_async_wait<0>();
        fence_proxy_async();
        for (uint32_t u = g > (uint32_t)kLag ? g - kLag : 0u; u < g; ++u) mbar_arrive(&S.wfull[u % kWStages]);
        if (!ok && lane == 0) {
            for (uint32_t u = g > (uint32_t)kWStages ? g - kWStages : 0u; u < g; ++u) {
                uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&S.wfull[u % kWStages], (u / kWStages) & 1u) &&
                       globaltimer_ns() - t0 < kWaitLimitNs / 8) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t g = 0, a = 0, hn = 0;
            bool ok = true;
            const uint32_t idesc = make_idesc_bf16(128, kNC, false, kDX);
            const uint32_t hhi = smem_u32(S.hhi), hlo = smem_u32(S.hlo);
            for (int32_t it = blockIdx.x; it < n_items && ok; it += gridDim.x) {
                const Item I = load_item(tab, segs, it, n_parts, d);
                if (!I.ad.ok) continue;
                const int32_t rp = rpad16(I.ad.rank);
                if (!mbar_wait(S.hfull, hn & 1u, S.abort, segs.status)) break;
                tc_fence_after();
                for (int32_t n0 = I.n_lo; n0 < I.n_hi; n0 += kNC) {
                    const uint32_t s = g % kWStages, ph = (g / kWStages) & 1u;
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
                        const uint64_t bdesc = kDX ? make_desc(w_base + 2048u * kk, (uint32_t)rp * 128u, 1024,
                                                               kSwizzle128)
                                                   : make_desc(w_base + 4096u * kk, 2048, 128, kInterleave);
                        umma_bf16(d_tmem, make_desc(hhi + 4096u * kk, 2048, 128, kInterleave), bdesc, idesc,
                                  kk > 0 ? 1u : 0u);
                        if (kSplit)
                            umma_bf16(d_tmem, make_desc(hlo + 4096u * kk, 2048, 128, kInterleave), bdesc, idesc, 1u);
                    }
                    umma_commit(&S.wempty[s]);
                    umma_commit(&S.tfull[acc]);
                    ++g;
                    ++a;
                }
                if (!ok) break;
                umma_commit(S.hempty);
                ++hn;
            }
            umma_commit(S.done);
            uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(S.done, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else if (warp >= 6) {
        // ------------------------------------------------------------ H block loader
        const int m = threadIdx.x - 6 * 32;  // row 0..127 of the tile
        const bool vec = (r_max & 3) == 0;
        uint32_t hn = 0;
        for (int32_t it = blockIdx.x; it < n_items; it += gridDim.x) {
            const Item I = load_item(tab, segs, it, n_parts, d);
            if (!I.ad.ok) continue;
            const int32_t r = I.ad.rank, rp = rpad16(r);
            if (!mbar_wait(S.hempty, (hn & 1u) ^ 1u, S.abort, segs.status)) break;
            const int32_t t = m < I.tile.rows ? segs.perm[I.tile.begin + m] : -1;
            const float *hr = h + (int64_t)(t < 0 ? 0 : t) * r_max;
            for (int kc = 0; kc < rp / 8; ++kc) {
                float f[8];
                if (t >= 0 && vec && 8 * kc + 8 <= r_max) {
                    const float4 u0 = *reinterpret_cast<const float4 *>(hr + 8 * kc);
                    const float4 u1 = *reinterpret_cast<const float4 *>(hr + 8 * kc + 4);
                    f[0] = u0.x; f[1] = u0.y; f[2] = u0.z; f[3] = u0.w;
                    f[4] = u1.x; f[5] = u1.y; f[6] = u1.z; f[7] = u1.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = (t >= 0 && 8 * kc + e < r_max) ? hr[8 * kc + e] : 0.f;
                }
                uint32_t hi[4], lo[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const float a0 = (8 * kc + e < r) ? f[e] : 0.f;
                    const float a1 = (8 * kc + e + 1 < r) ? f[e + 1] : 0.f;
                    hi[e / 2] = pack_bf16(a0, a1);
                    lo[e / 2] = pack_bf16(a0 - bf16lo(hi[e / 2]), a1 - bf16hi(hi[e / 2]));
                }
                const uint32_t off = (uint32_t)kc * 2048u + (uint32_t)m * 16u;
                *reinterpret_cast<uint4 *>(S.hhi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                if (kSplit) *reinterpret_cast<uint4 *>(S.hlo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(S.hfull);
            ++hn;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const uint32_t lane_base = 32u * (warp & 3);
        const int m = (int)lane_base + lane;
        uint32_t a = 0;
        for (int32_t it = blockIdx.x; it < n_items; it += gridDim.x) {
            const Item I = load_item(tab, segs, it, n_parts, d);
            if (!I.ad.ok) continue;
            const float c = kDX ? 1.0f : I.ad.scale;
            const int32_t t = m < I.tile.rows ? segs.perm[I.tile.begin + m] : -1;
            uint16_t *row = out + (int64_t)(t < 0 ? 0 : t) * d;
            bool ok = true;
            for (int32_t n0 = I.n_lo; n0 < I.n_hi; n0 += kNC) {
                const uint32_t acc = a % kAcc, aph = (a / kAcc) & 1u;
                if (!mbar_wait(&S.tfull[acc], aph, S.abort, segs.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int half = 0; half < 2; ++half) {
                    const int32_t c0 = n0 + 64 * half;
                    uint4 yv[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        yv[q] = (t >= 0 && c0 + 8 * q < d) ? *reinterpret_cast<const uint4 *>(row + c0 + 8 * q)
                                                           : make_uint4(0, 0, 0, 0);
                    uint32_t v[4][16];
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        tmem_ld16(tmem_base + (lane_base << 16) + acc * 128u + 64u * half + 16u * q, v[q]);
                    tmem_ld_wait();
                    if (half == 1) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&S.tempty[acc]);
                    }
                    if (t >= 0) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            if (c0 + 8 * q >= d) continue;
                            const uint32_t *acc8 = &v[q >> 1][(q & 1) * 8];
                            uint32_t w[4] = {yv[q].x, yv[q].y, yv[q].z, yv[q].w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float lo = bf16lo(w[e]) + c * __uint_as_float(acc8[2 * e]);
                                const float hi = bf16hi(w[e]) + c * __uint_as_float(acc8[2 * e + 1]);
                                w[e] = pack_bf16(lo, hi);
                            }
                            *reinterpret_cast<uint4 *>(row + c0 + 8 * q) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
                ++a;
            }
            if (!ok) break;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <bool kDX>
lora_status_t launch_colproj(void *out, const float *h, const lora_adapter_table &tab, const lora_segments &segs,
                             cudaStream_t stream)
{
    if (segs.n_tokens == 0 || segs.max_tiles == 0) return LORA_OK;
    const int32_t d = kDX ? tab.d_in : tab.d_out;
    CUtensorMap map_w;
    if (!make_tmap_bf16_2d(&map_w, tab.A, (uint64_t)tab.d_in, (uint64_t)tab.sum_r, 64, 16, true))
        return LORA_ERR_CUDA;
    if (cudaFuncSetAttribute(tc_colproj_kernel<kDX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kSmemBytes) != cudaSuccess)
        return LORA_ERR_CUDA;
    const int n_parts = (d + kNPart - 1) / kNPart;
    const int64_t items = (int64_t)segs.max_tiles * n_parts;
    const int sms = sm_count();
    const int grid = items < sms ? (int)items : sms;
    tc_colproj_kernel<kDX><<<grid, kThreads, kSmemBytes, stream>>>(map_w, static_cast<uint16_t *>(out), h, tab,
                                                                    segs);
    return cudaGetLastError() == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

}  // namespace

lora_status_t tc_expand(void *y, const float *H, const lora_adapter_table &tab, const lora_segments &segs,
                        cudaStream_t stream)
{
    return launch_colproj<false>(y, H, tab, segs, stream);
}

lora_status_t tc_dx(void *dX, const float *dH, const lora_adapter_table &tab, const lora_segments &segs,
                    cudaStream_t stream)
{
    return launch_colproj<true>(dX, dH, tab, segs, stream);
}

}  // namespace lora
