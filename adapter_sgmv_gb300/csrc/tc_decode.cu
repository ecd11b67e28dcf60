// tc_decode.cu -- SGMV for decode-sized batches: shrink and expand of every
// adapter of the batch in one launch (C-LoRA report, "Come funziona
// l'architettura": the decode kernel fuses the per-adapter matrix-vector work
// into a single GPU launch per decode step).
//
// A decode batch has few tokens per adapter, so the tokens sit on the N side
// of every tensor-core product (N = 48) and the long dimensions on M and K:
//   phase 1  D1[k, t] = sum_j A_i[k, j] x[t, j]    (M = 128 rank rows, N = 48
//            tokens, K = this CTA's share of d_in: split-K over the cluster)
//   phase 2  the cluster's eight partial D1 are summed through distributed
//            shared memory (each CTA sums r_pad / 8 rank rows and scatters the
//            bf16 hi + lo result into all eight CTAs)
//   phase 3  D3[o, t] = sum_k B_i[o, k] h[t, k]    (M = 128 output columns,
//            N = 48 tokens, K = r_pad) for this CTA's 128-column chunks, and
//            y[t, o] += s_i * D3[o, t] straight from TMEM (a warp's 32 lanes
//            are 32 consecutive columns of one token row).
// Work item = (tile, 48-token sub-tile, column part); clusters of eight CTAs
// walk the items; every CTA of a cluster sees the same items.  The weights of
// a CTA's first two output chunks and its first chunk's y values are fetched
// while phase 1 runs, so phase 3 starts from data already on chip.
//
// All mbarrier waits are bounded and no CTA leaves the item loop early: a
// time-out only makes the kernel skip work, and every CTA of a cluster still
// reaches every cluster barrier (the hardware one) after a bounded time.
#include "internal.h"
#include "tc_common.cuh"
#include "tc_host.h"

namespace lora {
namespace {

using namespace tc;

constexpr int kCS = 8;          // CTAs per cluster
constexpr int kThreads = 128;
constexpr int kStages = 4;
constexpr int kLag = 2;
constexpr int kTok = 48;        // tokens per work item (MMA N)
constexpr uint32_t kABytes = 128 * 64 * 2;   // phase-1 A block: up to 128 rank rows x 64
constexpr uint32_t kXBytes = kTok * 64 * 2;  // phase-1 B block: 48 token rows x 64 (one h atom too)
constexpr uint32_t kWBytes = LORA_MAX_RANK * 128 * 2;  // phase-3 A block: r_pad x 128 columns
constexpr uint32_t kHBytes = kTok * LORA_MAX_RANK * 2; // bf16 h, one copy
constexpr int kPStride = kTok + 1;                      // fp32 partial row stride
constexpr uint32_t kPBytes = LORA_MAX_RANK * kPStride * 4;
constexpr uint32_t kTmemCols = 256;  // D1: 48 columns at 0; D3: two slots of 48 at 64 and 128
constexpr size_t kSmemBytes =
    1024 + kStages * (size_t)(kABytes + kXBytes) + 2 * (size_t)kWBytes + 2 * (size_t)kHBytes + kPBytes + 512;

struct Smem {
    uint8_t *a, *x, *w, *hhi, *hlo;
    float *part;
    uint64_t *full, *empty, *p1done, *wfull, *d3full, *cbar;
    int32_t *tok;
    uint32_t *tmem_holder;
    volatile int32_t *abort;
};

LORA_DEV Smem carve(uint8_t *raw)
{
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    Smem s;
    s.a = base;
    s.x = s.a + kStages * kABytes;
    s.w = s.x + kStages * kXBytes;
    s.hhi = s.w + 2 * kWBytes;
    s.hlo = s.hhi + kHBytes;
    s.part = reinterpret_cast<float *>(s.hlo + kHBytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(s.part) + kPBytes);
    s.full = bars;
    s.empty = bars + kStages;
    s.p1done = s.empty + kStages;
    s.wfull = s.p1done + 1;
    s.d3full = s.wfull + 2;
    s.cbar = s.d3full + 2;
    s.tok = reinterpret_cast<int32_t *>(s.cbar + 1);
    s.tmem_holder = reinterpret_cast<uint32_t *>(s.tok + kTok);
    s.abort = reinterpret_cast<volatile int32_t *>(s.tmem_holder + 1);
    return s;
}

LORA_DEV int32_t rpad16(int32_t r) { return (r + 15) & ~15; }

LORA_DEV uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
LORA_DEV uint32_t cluster_id()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}
LORA_DEV uint32_t n_clusters()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}
// address of the same shared variable in CTA `rank` of this cluster
LORA_DEV uint32_t map_rank(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
LORA_DEV void remote_arrive(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
LORA_DEV bool cbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// the same shared fp32 word in all eight CTAs of the cluster, summed; the
// eight remote loads are issued back to back in one statement
LORA_DEV float sum_cluster_f32(uint32_t saddr)
{
    float v0, v1, v2, v3, v4, v5, v6, v7;
    asm volatile(
        "{\n\t.reg .b32 a<8>;\n\t"
        "mapa.shared::cluster.u32 a0, %8, 0;\n\tmapa.shared::cluster.u32 a1, %8, 1;\n\t"
        "mapa.shared::cluster.u32 a2, %8, 2;\n\tmapa.shared::cluster.u32 a3, %8, 3;\n\t"
        "mapa.shared::cluster.u32 a4, %8, 4;\n\tmapa.shared::cluster.u32 a5, %8, 5;\n\t"
        "mapa.shared::cluster.u32 a6, %8, 6;\n\tmapa.shared::cluster.u32 a7, %8, 7;\n\t"
        "ld.shared::cluster.f32 %0, [a0];\n\tld.shared::cluster.f32 %1, [a1];\n\t"
        "ld.shared::cluster.f32 %2, [a2];\n\tld.shared::cluster.f32 %3, [a3];\n\t"
        "ld.shared::cluster.f32 %4, [a4];\n\tld.shared::cluster.f32 %5, [a5];\n\t"
        "ld.shared::cluster.f32 %6, [a6];\n\tld.shared::cluster.f32 %7, [a7];\n\t}"
        : "=f"(v0), "=f"(v1), "=f"(v2), "=f"(v3), "=f"(v4), "=f"(v5), "=f"(v6), "=f"(v7)
        : "r"(saddr)
        : "memory");
    return ((v0 + v1) + (v2 + v3)) + ((v4 + v5) + (v6 + v7));
}
LORA_DEV void st_cluster_u16(uint32_t cluster_addr, uint16_t v)
{
    asm volatile("st.shared::cluster.u16 [%0], %1;" ::"r"(cluster_addr), "h"(v) : "memory");
}
// hardware cluster barrier: used only where every CTA of the cluster arrives
// unconditionally (start and end of the kernel), so it cannot be left waiting
LORA_DEV void hw_cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// generic-proxy writes, local or to other CTAs of the cluster -> async proxy
LORA_DEV void fence_proxy_async_all() { asm volatile("fence.proxy.async;" ::: "memory"); }

// Cluster-wide barrier inside the work loop.  Every CTA of a cluster walks the
// same items and every wait between two of these barriers is bounded, so all
// CTAs reach each barrier after a bounded time; the hardware cluster barrier
// (release / acquire) is then safe and much cheaper than an mbarrier handshake.
LORA_DEV bool cluster_sync(const Smem &, uint32_t &phase, int32_t *)
{
    hw_cluster_sync();
    phase ^= 1u;
    return true;
}

constexpr int kSubs = (LORA_TILE_M + kTok - 1) / kTok;  // token sub-tiles per tile

struct Item {
    Tile tile;
    AdapterInfo ad;
    int32_t sub_begin, rows;  // this item's tokens: perm[tile.begin + sub_begin ...], rows of them
    int32_t n_lo, n_hi;       // column part of d_out
    bool live;
};

LORA_DEV Item load_item(const lora_adapter_table &tab, const lora_segments &segs, int32_t it, int32_t n_parts,
                        int32_t part_cols)
{
    Item I;
    const int32_t per_tile = kSubs * n_parts;
    I.tile = load_tile(segs.tiles, it / per_tile);
    const int32_t sub = (it % per_tile) / n_parts, part = it % n_parts;
    I.sub_begin = sub * kTok;
    I.rows = min(kTok, I.tile.rows - I.sub_begin);
    I.n_lo = part * part_cols;
    I.n_hi = min(tab.d_out, I.n_lo + part_cols);
    I.ad = load_adapter(tab, I.tile.adapter, segs.status);
    I.live = I.rows > 0 && I.n_lo < I.n_hi && I.ad.ok;
    return I;
}

// phase-3 weights of output chunk c (columns o0 .. o0+127): B_i^T rows k as the
// MN-major A operand, two 64-column atoms of r_pad rows
LORA_DEV void load_w(const Smem &S, const CUtensorMap *map_b, uint32_t slot, int32_t o0, int32_t row_off, int32_t rp)
{
    uint8_t *w_s = S.w + slot * kWBytes;
    mbar_arrive_expect_tx(&S.wfull[slot], (uint32_t)rp * 256u);
    for (int a = 0; a < 2; ++a)
        for (int q = 0; q < rp / 16; ++q)
            tma_load_2d(w_s + a * rp * 128 + q * 2048, map_b, &S.wfull[slot], o0 + 64 * a, row_off + 16 * q);
}

__global__ void __cluster_dims__(kCS, 1, 1) __launch_bounds__(kThreads, 1)
tc_decode_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                 uint16_t *__restrict__ y, const uint16_t *__restrict__ x, float *__restrict__ H_save,
                 int32_t n_parts, int32_t part_cols, lora_adapter_table tab, lora_segments segs)
{
    extern __shared__ uint8_t smem_raw[];
    const Smem S = carve(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rho = cluster_rank();
    const int32_t d_in = tab.d_in, d_out = tab.d_out, r_max = tab.r_max;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&S.full[i], kThreads + 1);
            mbar_init(&S.empty[i], 1);
        }
        mbar_init(S.p1done, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&S.wfull[i], 1);
            mbar_init(&S.d3full[i], 1);
        }
        mbar_init(S.cbar, kCS);
        *S.abort = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(S.tmem_holder, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *S.tmem_holder;
    const uint32_t tmem_lane = (32u * warp) << 16;
    uint32_t cphase = 0;
    // every CTA of the cluster has initialised its barriers before anyone arrives remotely
    hw_cluster_sync();

    const int32_t n_items = *segs.n_tiles * kSubs * n_parts;
    const int32_t nkb = (d_in + 63) / 64;
    const int32_t kb_per = (nkb + kCS - 1) / kCS;
    const int32_t kb0 = min(nkb, (int32_t)rho * kb_per), kb1 = min(nkb, kb0 + kb_per);
    const int32_t nmy = kb1 - kb0;
    uint32_t g = 0, np1 = 0, gw = 0;  // phase-1 stages issued, phase-1 commits, phase-3 chunks

    for (int32_t it = cluster_id(); it < n_items; it += n_clusters()) {
        const Item I = load_item(tab, segs, it, n_parts, part_cols);
        if (!I.live) continue;  // uniform across the cluster: same item, same decision
        const int32_t r = I.ad.rank, rp = rpad16(r);
        const int32_t nch = (I.n_hi - I.n_lo + 127) / 128;  // 128-column chunks of the part
        if (threadIdx.x < kTok)
            S.tok[threadIdx.x] = threadIdx.x < I.rows ? segs.perm[I.tile.begin + I.sub_begin + threadIdx.x] : -1;
        __syncthreads();
        const bool run = *S.abort == 0;
        __syncthreads();
        // this CTA's chunks are c = rho, rho + 8, ...: fetch the first two chunks' weights now
        if (threadIdx.x == 0 && run)
            for (int32_t j = 0; j < 2 && (int32_t)rho + kCS * j < nch; ++j)
                load_w(S, &map_b, (gw + j) & 1u, I.n_lo + 128 * ((int32_t)rho + kCS * j), I.ad.row_off, rp);

        // ---------------------------------------------------------------- phase 1 (split-K shrink)
        if (run) {
            const uint32_t idesc1 = make_idesc_bf16(128, kTok, false, false);
            for (int32_t i = 0; i < nmy + kLag; ++i) {
                if (i < nmy) {
                    const uint32_t s = (g + i) % kStages, ph = ((g + i) / kStages) & 1u;
                    mbar_wait(&S.empty[s], ph ^ 1u, S.abort, segs.status);
                    const int32_t j0 = (kb0 + i) * 64;
                    if (threadIdx.x == 0) {
                        mbar_arrive_expect_tx(&S.full[s], (uint32_t)rp * 128u);
                        for (int q = 0; q < rp / 16; ++q)
                            tma_load_2d(S.a + s * kABytes + q * 2048, &map_a, &S.full[s], j0, I.ad.row_off + 16 * q);
                    }
                    // kTok token rows x 8 chunks of 16 bytes
                    for (int e = threadIdx.x; e < kTok * 8; e += kThreads) {
                        const int m = e >> 3, c = e & 7;
                        const int32_t t = S.tok[m];
                        const bool v = t >= 0 && j0 + 8 * c < d_in;
                        cp_async_16(S.x + s * kXBytes + sw128_offset((uint32_t)m, (uint32_t)c),
                                    v ? x + (int64_t)t * d_in + j0 + 8 * c : x, v);
                    }
                }
                cp_async_commit();
                if (i >= kLag) {
                    const uint32_t u = g + i - kLag;
                    const uint32_t s = u % kStages, ph = (u / kStages) & 1u;
                    cp_async_wait<kLag>();
                    fence_proxy_async();
                    mbar_arrive(&S.full[s]);
                    if (threadIdx.x == 0 && mbar_wait(&S.full[s], ph, S.abort, segs.status)) {
                        tc_fence_after();
                        const uint32_t ab = smem_u32(S.a + s * kABytes), xb = smem_u32(S.x + s * kXBytes);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            umma_bf16(tmem_base, make_desc(ab + 32u * k, 16, 1024, kSwizzle128),
                                      make_desc(xb + 32u * k, 16, 1024, kSwizzle128), idesc1,
                                      (i - kLag) > 0 || k > 0 ? 1u : 0u);
                        umma_commit(&S.empty[s]);
                    }
                }
            }
            if (threadIdx.x == 0) umma_commit(S.p1done);
            g += (uint32_t)nmy;
        }
        // y values of this CTA's first chunk (this thread's column, every token), fetched early
        uint16_t yv[kTok];
        {
            const int32_t o = I.n_lo + 128 * (int32_t)rho + 32 * warp + lane;
            const bool col = (int32_t)rho < nch && o < I.n_hi;
#pragma unroll
            for (int t = 0; t < kTok; ++t) yv[t] = (col && S.tok[t] >= 0) ? y[(int64_t)S.tok[t] * d_out + o] : 0;
        }
        // partial D1 (lanes = rank rows, columns = tokens) -> shared memory
        {
            const bool have =
                __syncthreads_and(run && nmy > 0 && mbar_wait(S.p1done, np1 & 1u, S.abort, segs.status)) != 0;
            tc_fence_after();
            uint32_t v[3][16];
#pragma unroll
            for (int q = 0; q < 3; ++q) tmem_ld16(tmem_base + tmem_lane + 16u * q, v[q]);
            tmem_ld_wait();
            tc_fence_before();
            const int k = 32 * warp + lane;
#pragma unroll
            for (int t = 0; t < kTok; ++t) S.part[k * kPStride + t] = have ? __uint_as_float(v[t >> 4][t & 15]) : 0.f;
        }
        if (run) ++np1;
        cluster_sync(S, cphase, segs.status);

        // ---------------------------------------------------------------- phase 2 (reduce-scatter, gather)
        {
            const int kr = rp / kCS;  // rank rows owned by this CTA (r_pad is a multiple of 16)
            for (int e = threadIdx.x; e < kr * kTok; e += kThreads) {
                const int k = (int)rho * kr + e / kTok, t = e % kTok;
                float acc = sum_cluster_f32(smem_u32(S.part + k * kPStride + t));
                if (k >= r) acc = 0.f;
                const uint16_t hi = f32_to_bf16(acc);
                const uint16_t lo = f32_to_bf16(acc - bf16_to_f32(hi));
                // element (t, k) of the K-major 128-byte-swizzled h block [kTok x 64] atoms
                const uint32_t off = (uint32_t)(k >> 6) * kXBytes + sw128_offset((uint32_t)t, (uint32_t)((k & 63) >> 3)) +
                                     (uint32_t)(k & 7) * 2u;
#pragma unroll
                for (int c = 0; c < kCS; ++c) {
                    st_cluster_u16(map_rank(smem_u32(S.hhi + off), (uint32_t)c), hi);
                    st_cluster_u16(map_rank(smem_u32(S.hlo + off), (uint32_t)c), lo);
                }
                if (H_save != nullptr && S.tok[t] >= 0 && k < r_max)
                    H_save[(int64_t)S.tok[t] * r_max + k] = acc;
            }
            if (H_save != nullptr)  // columns past r_pad
                for (int e = threadIdx.x; e < kTok * r_max; e += kThreads) {
                    const int t = e / r_max, k = e % r_max;
                    if (k >= rp && (k - rp) % kCS == (int)rho && S.tok[t] >= 0) H_save[(int64_t)S.tok[t] * r_max + k] = 0.f;
                }
        }
        fence_proxy_async_all();
        cluster_sync(S, cphase, segs.status);
        fence_proxy_async();

        // ---------------------------------------------------------------- phase 3 (expand, this CTA's chunks)
        const uint32_t idesc3 = make_idesc_bf16(128, kTok, true, false);
        for (int32_t c = (int32_t)rho, j = 0; c < nch; c += kCS, ++j) {
            const int32_t o0 = I.n_lo + 128 * c;
            const uint32_t slot = gw & 1u, ph = (gw >> 1) & 1u;
            const uint32_t d3 = tmem_base + 64u + 64u * slot;
            if (threadIdx.x == 0 && run) {
                if (mbar_wait(&S.wfull[slot], ph, S.abort, segs.status)) {
                    tc_fence_after();
                    const uint32_t wb = smem_u32(S.w + slot * kWBytes), hh = smem_u32(S.hhi), hl = smem_u32(S.hlo);
                    for (int kk = 0; kk < rp / 16; ++kk) {
                        const uint64_t adesc = make_desc(wb + 2048u * kk, (uint32_t)rp * 128u, 1024, kSwizzle128);
                        const uint32_t hoff = (uint32_t)(kk >> 2) * kXBytes + (uint32_t)(kk & 3) * 32u;
                        umma_bf16(d3, adesc, make_desc(hh + hoff, 16, 1024, kSwizzle128), idesc3, kk > 0 ? 1u : 0u);
                        umma_bf16(d3, adesc, make_desc(hl + hoff, 16, 1024, kSwizzle128), idesc3, 1u);
                    }
                }
                umma_commit(&S.d3full[slot]);
            }
            const int32_t o = o0 + 32 * warp + lane;
            if (j > 0) {  // later chunks: fetch y while the MMA runs
#pragma unroll
                for (int t = 0; t < kTok; ++t)
                    yv[t] = (o < I.n_hi && S.tok[t] >= 0) ? y[(int64_t)S.tok[t] * d_out + o] : 0;
            }
            const bool have = __syncthreads_and(run && mbar_wait(&S.d3full[slot], ph, S.abort, segs.status) &&
                                                *S.abort == 0) != 0;
            tc_fence_after();
            uint32_t v[3][16];
#pragma unroll
            for (int q = 0; q < 3; ++q) tmem_ld16(d3 + tmem_lane + 16u * q, v[q]);
            tmem_ld_wait();
            tc_fence_before();
            if (have && o < I.n_hi) {
#pragma unroll
                for (int t = 0; t < kTok; ++t)
                    if (S.tok[t] >= 0)
                        y[(int64_t)S.tok[t] * d_out + o] =
                            f32_to_bf16(bf16_to_f32(yv[t]) + I.ad.scale * __uint_as_float(v[t >> 4][t & 15]));
            }
            ++gw;
            __syncthreads();  // TMEM slot and weight slot free again
            if (threadIdx.x == 0 && run && c + 2 * kCS < nch)  // weights of this slot's next chunk
                load_w(S, &map_b, slot, I.n_lo + 128 * (c + 2 * kCS), I.ad.row_off, rp);
        }
        __syncthreads();
    }

    hw_cluster_sync();  // no CTA leaves while others may still read its shared memory
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

}  // namespace

lora_status_t tc_decode_fwd(void *y, float *H_save, const void *x, const lora_adapter_table &tab,
                            const lora_segments &segs, cudaStream_t stream)
{
    if (segs.n_tokens == 0 || segs.max_tiles == 0) return LORA_OK;
    CUtensorMap map_a, map_b;
    if (!make_tmap_bf16_2d(&map_a, tab.A, (uint64_t)tab.d_in, (uint64_t)tab.sum_r, 64, 16, true) ||
        !make_tmap_bf16_2d(&map_b, tab.B, (uint64_t)tab.d_out, (uint64_t)tab.sum_r, 64, 16, true))
        return LORA_ERR_CUDA;
    if (cudaFuncSetAttribute(tc_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
        cudaSuccess)
        return LORA_ERR_CUDA;
    // as many clusters as can be resident at once (eight-SM clusters must fit in
    // one GPC, so this is below SMs / 8), so that no cluster waits for a second wave
    const int sms = sm_count();
    int clusters = sms / kCS > 0 ? sms / kCS : 1;
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(clusters * kCS);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemBytes;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = kCS;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, tc_decode_kernel, &cfg) == cudaSuccess && active > 0 &&
            active < clusters)
            clusters = active;
        cudaGetLastError();
    }
    // column parts: enough items to give every cluster one (sub-tiles ~ T / kTok + 1)
    const int est = (segs.n_tokens + kTok - 1) / kTok + 1;
    int n_parts = clusters / est;
    n_parts = n_parts < 1 ? 1 : n_parts;
    const int chunks = (tab.d_out + 127) / 128;
    if (n_parts > chunks) n_parts = chunks;
    const int part_cols = ((chunks + n_parts - 1) / n_parts) * 128;
    n_parts = (tab.d_out + part_cols - 1) / part_cols;
    tc_decode_kernel<<<clusters * kCS, kThreads, kSmemBytes, stream>>>(
        map_a, map_b, static_cast<uint16_t *>(y), static_cast<const uint16_t *>(x), H_save, n_parts, part_cols, tab,
        segs);
    return cudaGetLastError() == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

}  // namespace lora
