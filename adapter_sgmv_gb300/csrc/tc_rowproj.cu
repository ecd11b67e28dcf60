// tc_rowproj.cu -- case i on the 5th-generation tensor cores: a reduction over
// the hidden dimension into a T x r result, tiled along tokens (PLoRA
// technical summary, "2. LoRA Execution Engine": tile the concatenated LoRA
// tensors along the sequence or hidden dimension, never along the rank).
//
//   shrink  H[t, k]  = sum_j x[t, j]  A_i[k, j]          (c = 1)
//   dh      dH[t, k] = s_i sum_o dY[t, o] B_i[o, k]       (c = s_i)
//
// A and B are stored alike (A_i and B_i^T stacked, [sum_r, d]), so both
// products read their weights the same way: r_pad x 64 blocks by TMA as the
// K-major B operand.  One work tile = up to 128 tokens of one adapter.  Per
// 64-wide slice of d a stage holds the 128 x 64 activation block (K-major,
// 128-byte swizzle: TMA when the rows are consecutive tokens, else cp.async
// gather) and the weight block; one thread issues tcgen05.mma (M = 128,
// N = r_pad, K = 16) into a TMEM accumulator; four epilogue warps write
//   - out_f32[t, :]  = c * acc   (fp32, stride r_max; optional), zero in
//     columns r_i .. r_max - 1
//   - out_hi[p, :]   = bf16(c * acc), out_lo[p, :] = bf16(c * acc - hi)
//     (row p = the token's position in perm, stride rw; both optional), zero
//     in columns r_i .. r_pad - 1 and not written past r_pad
// The perm-ordered bf16 rows are what the case ii / iii / iv kernels read by
// TMA; their products stop at r_pad.  A small kernel beside them converts a
// saved fp32 H into the same hand-off rows for the backward.
//
// Warp roles (32 (S + 5) threads for a ring of S stages): 0..S-1 load, warp w
// filling every stage of ring slot w (a gathered stage's copies are waited for
// by the warp that issued them, which makes them visible to the tensor cores
// and releases the stage at once, so all S stages can be in flight); S issues
// MMAs and owns TMEM; S+1..S+4 epilogue.  Every wait is bounded
// (tc::mbar_wait).  Two ring depths: six stages with one CTA per SM, or three
// stages with two CTAs per SM, taken when there are enough tiles to give most
// SMs two; the two CTAs of an SM then stream two tiles side by side and each
// one's tile changes and epilogues are covered by the other's loads.
#define LORA_DBG_FILE 2
#include "internal.h"
#include "tc_common.cuh"
#include "tc_host.h"

namespace lora {
namespace {

using namespace tc;

constexpr uint32_t kActBytes = 128 * 64 * 2;
constexpr uint32_t kWBytes = LORA_MAX_RANK * 64 * 2;
constexpr uint32_t kStageBytes = kActBytes + kWBytes;
constexpr uint32_t kTmemCols = 256;  // two accumulators of up to 128 columns (two CTAs fill an SM's 512)
template <int kStages>
constexpr int threads_of() { return 32 * (kStages + 1 + 4); }
template <int kStages>
constexpr size_t smem_of() { return 1024 + kStages * (size_t)kStageBytes + 256; }

struct Smem {
    uint8_t *act, *w;
    uint64_t *full, *empty, *tfull, *tempty, *done;
    uint32_t *tmem_holder;
    volatile int32_t *abort;
};

template <int kStages>
LORA_DEV Smem carve(uint8_t *raw)
{
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    Smem s;
    s.act = base;
    s.w = base + kStages * kActBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(base + kStages * kStageBytes);
    s.full = bars;
    s.empty = bars + kStages;
    s.tfull = bars + 2 * kStages;
    s.tempty = s.tfull + 2;
    s.done = s.tempty + 2;
    s.tmem_holder = reinterpret_cast<uint32_t *>(s.done + 1);
    s.abort = reinterpret_cast<volatile int32_t *>(s.tmem_holder + 1);
    return s;
}

LORA_DEV int32_t rpad16(int32_t r) { return (r + 15) & ~15; }

struct RowOut {
    float *f32;           // [T, r_max] by token, or null
    uint16_t *hi, *lo;    // [T, rw] by perm position, or null
    int32_t rw;
    float scale_is_adapter;  // 1: c = s_i, 0: c = 1
    // split along d (few tiles): the kernel writes fp32 partials c * acc of
    // each part to part[(q * T + p) * part_ld + k], k < r_pad, and a combine
    // kernel adds them in part order and writes the outputs above
    int32_t splits;
    int32_t part_ld;
    float *part;
    // work-claim counters of the kernels that follow in the same call, zeroed
    // here before anything else (null: none)
    int32_t *zero_claims;
    int32_t n_zero;
    // an output of a later kernel of the call that accumulates into zeros
    // (dA, dB), cleared here by the whole grid (null: none)
    float *zero_out;
    int64_t zero_out_n;
};

// the k-blocks [lo, hi) of part q of a d of nk blocks cut into `splits` parts
LORA_DEV int32_t part_lo(int32_t q, int32_t nk, int32_t splits) { return (int32_t)((int64_t)q * nk / splits); }

template <int kStages>
__global__ void __launch_bounds__(threads_of<kStages>(), kStages <= 3 ? 2 : 1)
tc_rowproj_kernel(const __grid_constant__ CUtensorMap map_act, const __grid_constant__ WMaps map_w,
                  const uint16_t *__restrict__ act, int32_t d, RowOut o, lora_adapter_table tab,
                  lora_segments segs)
{
    constexpr int kProd = kStages;  // producer warps, one per ring slot
    constexpr int kMmaWarp = kProd;
    extern __shared__ uint8_t smem_raw[];
    const Smem S = carve<kStages>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    zero_claims(o.zero_claims, o.n_zero);
    zero_grid(o.zero_out, o.zero_out_n);

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
    const int32_t n_units = N_TILES(segs) * o.splits;  // (tile, part of d)
    const int32_t nk = (d + 63) / 64;

    if (warp < kProd) {
        // ------------------------------------------------------------ producers
        // Stage g of the whole sequence goes to ring slot g % kStages = warp.
        if (lane == 0 && warp == 0) {
            prefetch_tensormap(&map_act);
            prefetch_tensormap(&map_w.m16);
            prefetch_tensormap(&map_w.m32);
            prefetch_tensormap(&map_w.m64);
        }
        uint32_t g = 0, last = 0xffffffffu;
        bool ok = true;
        for (int32_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
            const int32_t ti = u / o.splits, q = u % o.splits;
            const int32_t kb_lo = part_lo(q, nk, o.splits), kb_n = part_lo(q + 1, nk, o.splits) - kb_lo;
            const Tile T = LOAD_TILE(segs, ti);
            const AdapterInfo ad = load_adapter(tab, T.adapter, segs.status);
            if (!ad.ok) continue;
            const int32_t rp = rpad16(ad.rank);
            const bool contiguous = (T.flags & 1) != 0;
            // this warp's first stage of the unit, and whether it has one at all
            const uint32_t k0 = (uint32_t)((warp - (int)(g % kStages) + kStages) % kStages);
            if ((int32_t)k0 >= kb_n) {
                g += (uint32_t)kb_n;
                continue;
            }
            const int32_t t0 = PERM_AT(segs, T.begin);
            int32_t tok[32];  // rows (lane >> 3) + 4 q of a gathered tile
            if (!contiguous) {
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const int m = (lane >> 3) + 4 * q;
                    tok[q] = m < T.rows ? PERM_AT(segs, T.begin + m) : -1;
                }
            }
            for (int32_t kq = (int32_t)k0; kq < kb_n; kq += kStages) {
                const int32_t kb = kb_lo + kq;
                const uint32_t gs = g + (uint32_t)kq;
                const uint32_t s = gs % kStages, ph = (gs / kStages) & 1u;
                if (!mbar_wait(&S.empty[s], ph ^ 1u, S.abort, segs.status)) {
                    ok = false;
                    break;
                }
                const int32_t j0 = kb * 64;
                uint8_t *act_s = S.act + s * kActBytes;
                uint8_t *w_s = S.w + s * kWBytes;
                if (lane == 0) {
                    mbar_arrive_expect_tx(&S.full[s], (contiguous ? kActBytes : 0u) + (uint32_t)rp * 128u);
                    if (contiguous) tma_load_2d(act_s, &map_act, &S.full[s], j0, t0);
                    tma_load_rows(w_s, map_w, &S.full[s], j0, ad.row_off, rp);
                }
                if (!contiguous) {
                    const int c = lane & 7;
                    const bool cin = j0 + 8 * c < d;
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const int m = (lane >> 3) + 4 * q;
                        const bool v = tok[q] >= 0 && cin;
                        const uint16_t *src = v ? act + (int64_t)tok[q] * d + j0 + 8 * c : act;
                        cp_async_16(act_s + sw128_offset(m, c), src, v);
                    }
                    // this lane's copies have landed; visible to the tensor cores
                    cp_async_commit();
                    cp_async_wait<0>();
                    fence_proxy_async();
                }
                mbar_arrive(&S.full[s]);
                last = gs;
            }
            g += (uint32_t)kb_n;
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
            uint32_t g = 0, acc_n = 0;
            bool ok = true;
            for (int32_t u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
                const int32_t ti = u / o.splits, q = u % o.splits;
                const int32_t kb_lo = part_lo(q, nk, o.splits), kb_hi = part_lo(q + 1, nk, o.splits);
                const Tile T = LOAD_TILE(segs, ti);
                const AdapterInfo ad = load_adapter(tab, T.adapter, segs.status);
                if (!ad.ok) continue;
                const uint32_t rp = (uint32_t)rpad16(ad.rank);
                const uint32_t acc = acc_n & 1u, aph = (acc_n >> 1) & 1u;
                if (!mbar_wait(&S.tempty[acc], aph ^ 1u, S.abort, segs.status)) break;
                tc_fence_after();
                const uint32_t idesc = make_idesc_bf16(128, rp, false, false);
                const uint32_t d_tmem = tmem_base + acc * 128u;
                for (int32_t kb = kb_lo; kb < kb_hi; ++kb) {
                    const uint32_t s = g % kStages, ph = (g / kStages) & 1u;
                    if (!mbar_wait(&S.full[s], ph, S.abort, segs.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(S.act + s * kActBytes);
                    const uint32_t w_base = smem_u32(S.w + s * kWBytes);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        umma_bf16(d_tmem, make_desc(a_base + 32u * k, 16, 1024, kSwizzle128),
                                  make_desc(w_base + 32u * k, 16, 1024, kSwizzle128), idesc,
                                  (kb != kb_lo || k != 0) ? 1u : 0u);
                    umma_commit(&S.empty[s]);
                    ++g;
                }
                if (!ok) break;
                umma_commit(&S.tfull[acc]);
                ++acc_n;
            }
            umma_commit(S.done);  // every MMA issued above has completed once this fires
            uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(S.done, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const uint32_t lane_base = 32u * (warp & 3);
        const int32_t r_max = tab.r_max;
        const bool vec = (r_max & 3) == 0;
        uint32_t acc_n = 0;
        for (int32_t u = blockIdx.x; u < n_units; u += gridDim.x) {
            const int32_t ti = u / o.splits, q = u % o.splits;
            const Tile T = LOAD_TILE(segs, ti);
            const AdapterInfo ad = load_adapter(tab, T.adapter, segs.status);
            if (!ad.ok) continue;
            const int32_t r = ad.rank, rp = rpad16(r);
            const uint32_t acc = acc_n & 1u, aph = (acc_n >> 1) & 1u;
            if (!mbar_wait_warp(&S.tfull[acc], aph, S.abort, segs.status)) break;
            tc_fence_after();
            const int m = (int)lane_base + lane;
            const bool valid = m < T.rows;
            const int64_t p = (int64_t)T.begin + m;
            const int32_t t = valid ? PERM_AT(segs, p) : -1;
            const float c = o.scale_is_adapter != 0.f ? ad.scale : 1.0f;
            const bool whole = o.splits == 1;  // else this unit's part goes to the partials
            float *row = whole && o.f32 != nullptr ? o.f32 + (int64_t)(t < 0 ? 0 : t) * r_max : nullptr;
            uint16_t *rhi = whole && o.hi != nullptr ? o.hi + p * o.rw : nullptr;
            uint16_t *rlo = whole && o.lo != nullptr ? o.lo + p * o.rw : nullptr;
            float *prow = whole ? nullptr : o.part + ((int64_t)q * segs.n_tokens + p) * o.part_ld;
            for (int c0 = 0; c0 < rp; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(tmem_base + (lane_base << 16) + acc * 128u + (uint32_t)c0, v);
                tmem_ld_wait();
                if (!valid) continue;
                float f[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) f[e] = (c0 + e < r) ? c * __uint_as_float(v[e]) : 0.f;
                if (prow != nullptr) {
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        *reinterpret_cast<float4 *>(prow + c0 + e) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
                }
                if (row != nullptr) {
                    if (vec && c0 + 16 <= r_max) {
#pragma unroll
                        for (int e = 0; e < 16; e += 4)
                            *reinterpret_cast<float4 *>(row + c0 + e) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (c0 + e < r_max) row[c0 + e] = f[e];
                    }
                }
                if (rhi != nullptr) {
                    uint32_t hw[8], lw[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        hw[e] = pack_bf16(f[2 * e], f[2 * e + 1]);
                        lw[e] = pack_bf16(f[2 * e] - bf16lo(hw[e]), f[2 * e + 1] - bf16hi(hw[e]));
                    }
                    *reinterpret_cast<uint4 *>(rhi + c0) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                    *reinterpret_cast<uint4 *>(rhi + c0 + 8) = make_uint4(hw[4], hw[5], hw[6], hw[7]);
                    if (rlo != nullptr) {
                        *reinterpret_cast<uint4 *>(rlo + c0) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                        *reinterpret_cast<uint4 *>(rlo + c0 + 8) = make_uint4(lw[4], lw[5], lw[6], lw[7]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&S.tempty[acc]);
            ++acc_n;
            // the fp32 output is zero past the rank rounded up to 16 (its
            // contract); the hand-off rows are not written there, because every
            // product that reads them stops at that rounded rank
            if (!valid || row == nullptr) continue;
            if (vec) {
                for (int k = rp; k < r_max; k += 4) *reinterpret_cast<float4 *>(row + k) = make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
                for (int k = rp; k < r_max; ++k) row[k] = 0.f;
            }
        }
    }

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
    const int sms = sm_count();
    const int64_t units = (int64_t)segs.max_tiles * o.splits;
    // two CTAs per SM once there are at least 1.5 tiles per SM (packed
    // 4096-token adapters, 256 tiles: dh 61.9 -> 54.8 us); with about one
    // per SM most SMs would hold a single three-stage CTA (skewed batch, 160
    // gathered tiles: dh 114 -> 142 us)
    const bool two = 2 * units >= 3 * (int64_t)sms;
    auto *kernel = two ? tc_rowproj_kernel<3> : tc_rowproj_kernel<6>;
    const size_t smem = two ? smem_of<3>() : smem_of<6>();
    const int per_sm = two ? 2 : 1;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return LORA_ERR_CUDA;
    const int grid = units < per_sm * sms ? (int)units : per_sm * sms;
    kernel<<<grid, two ? threads_of<3>() : threads_of<6>(), smem, stream>>>(
        map_act, map_w, static_cast<const uint16_t *>(act), d, o, tab, segs);
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
// 16, unwritten past that): one CTA per tile, each thread four (row, 8
// columns) pieces at a time with all their loads issued before any store (one
// round trip for the four instead of two each), the tokens of a run of
// consecutive ones from its first.  It runs beside case i (dh), so its CTAs
// are kept small (1024-thread CTAs converted faster alone but crowded out dh's).
__global__ void __launch_bounds__(256) h_to_bf16_kernel(const float *__restrict__ H, uint16_t *__restrict__ hb,
                                                        int32_t rw, int32_t *zero, int32_t n_zero,
                                                        float *zero_out, int64_t zero_out_n,
                                                        lora_adapter_table tab, lora_segments segs)
{
    zero_claims(zero, n_zero);  // the counters of the kernels after this one in the call
    zero_grid(zero_out, zero_out_n);  // and the output they add into
    const int32_t n_tiles = N_TILES(segs);
    const int32_t r_max = tab.r_max;
    const bool vec = (r_max & 3) == 0 && (reinterpret_cast<uintptr_t>(H) & 15u) == 0;
    constexpr int kBatch = 4;  // pieces a thread loads before it stores any (their round trips overlap)
    for (int32_t ti = blockIdx.x; ti < n_tiles; ti += gridDim.x) {
        const Tile T = LOAD_TILE(segs, ti);
        const AdapterInfo ad = load_adapter(tab, T.adapter, nullptr);
        const int32_t r = ad.ok ? ad.rank : 0;
        const int32_t rp8 = (r + 15) / 16 * 2;  // 8-column pieces up to the rank rounded to 16; past it no product reads
        const int32_t n = T.rows * rp8;
        // a run of consecutive tokens needs only its first token
        const bool contiguous = (T.flags & 1) != 0;
        const int32_t t0 = contiguous ? PERM_AT(segs, T.begin) : 0;
        for (int32_t i0 = threadIdx.x; i0 < n; i0 += kBatch * blockDim.x) {
            int32_t tok[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int32_t i = i0 + j * (int32_t)blockDim.x, m = i / rp8;
                tok[j] = i < n ? (contiguous ? t0 + m : PERM_AT(segs, (int64_t)T.begin + m)) : -1;
            }
            float f[kBatch][8];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int32_t i = i0 + j * (int32_t)blockDim.x, k = 8 * (i % rp8);
                const float *src = H + (int64_t)(tok[j] < 0 ? 0 : tok[j]) * r_max;
                if (tok[j] >= 0 && vec && k + 8 <= r) {  // two 16-byte loads
                    const float4 a = __ldcs(reinterpret_cast<const float4 *>(src + k));
                    const float4 b = __ldcs(reinterpret_cast<const float4 *>(src + k + 4));
                    f[j][0] = a.x; f[j][1] = a.y; f[j][2] = a.z; f[j][3] = a.w;
                    f[j][4] = b.x; f[j][5] = b.y; f[j][6] = b.z; f[j][7] = b.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[j][e] = tok[j] >= 0 && k + e < r ? src[k + e] : 0.f;
                }
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int32_t i = i0 + j * (int32_t)blockDim.x;
                if (tok[j] < 0) continue;
                const int32_t m = i / rp8, k = 8 * (i % rp8);
                *reinterpret_cast<uint4 *>(hb + ((int64_t)T.begin + m) * rw + k) =
                    make_uint4(pack_bf16(f[j][0], f[j][1]), pack_bf16(f[j][2], f[j][3]), pack_bf16(f[j][4], f[j][5]),
                               pack_bf16(f[j][6], f[j][7]));
            }
        }
    }
}

}  // namespace

lora_status_t tc_h_to_bf16(const float *H, uint16_t *hb, int32_t rw, int32_t *zero_claims, int32_t n_zero,
                           float *zero_out, int64_t zero_out_n, const lora_adapter_table &tab,
                           const lora_segments &segs, cudaStream_t stream)
{
    if (segs.n_tokens == 0 || segs.max_tiles == 0) return LORA_OK;
    const int sms = sm_count();
    const int grid = segs.max_tiles < 4 * sms ? segs.max_tiles : 4 * sms;
    h_to_bf16_kernel<<<grid, 256, 0, stream>>>(H, hb, rw, zero_claims, n_zero, zero_out, zero_out_n, tab, segs);
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
                        float *zero_out, int64_t zero_out_n, cudaStream_t stream)
{
    RowOut o{H, hi, lo, rw, 0.f, 1, 0, nullptr, zero_claims, n_zero, zero_out, zero_out_n};
    return launch_rowproj(x, tab.A, tab.d_in, o, tab, segs, part, stream);
}

lora_status_t tc_dh(const void *dY, const lora_adapter_table &tab, const lora_segments &segs, uint16_t *dh_bf16,
                    int32_t rw, float *part, int32_t *zero_claims, int32_t n_zero, float *zero_out,
                    int64_t zero_out_n, cudaStream_t stream)
{
    RowOut o{nullptr, dh_bf16, nullptr, rw, 1.f, 1, 0, nullptr, zero_claims, n_zero, zero_out, zero_out_n};
    return launch_rowproj(dY, tab.B, tab.d_out, o, tab, segs, part, stream);
}

}  // namespace lora
