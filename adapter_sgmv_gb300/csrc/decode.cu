// decode.cu -- SGMV for decode-sized batches: the shrink and expand of every
// adapter in the batch, grouped by adapter (C-LoRA report, "Come funziona
// l'architettura": the decode kernel applies every token's adapter in one
// grouped launch instead of one launch per adapter).
//
// A decode batch has a few tokens per adapter, so every product is skinny and
// the step is bound by latency (the working set is a few MB).  Two launches,
// each over all adapters, chained by programmatic dependent launch:
//
//   shrink  a CTA per (tile of <= 128 tokens of one adapter, slice s of d_in):
//           P_s[t, k] = sum_{j in slice s} x[t, j] A_i[k, j]   (fp32)
//           written to the workspace; no CTA waits for another
//   expand  work item = (tile, 256-column slice of d_out)
//           h[t, k]   = sum_s P_s[t, k]   (slice order, the same in every item)
//           y[t, o]  += s_i sum_k h[t, k] B_i[o, k]
//
// The expand kernel is launched as a programmatic dependent of the shrink: its
// CTAs start while the shrink runs and fetch their B_i^T block and the y rows
// they update (inputs the shrink does not write) before waiting for the shrink
// grid to complete; the partials are then read from L2.  The shrink is an
// ordinary launch: it reads the routing and A_i before anything else, and the
// kernel before it on the stream may have written them (a routing build, an
// optimizer step that refreshed A_i); only a completed predecessor is
// visible without a grid-dependency wait.
//
// Several projections that read the same x (q / k / v, gate / up) go through
// the same two launches: blockIdx.y selects the projection, each with its own
// adapter table, output and h buffer, so a layer's decode LoRA work costs two
// launches however many projections share the input.
//
// The products are warp-level bf16 tensor-core MMAs (m16n8k16, fp32
// accumulate): with 16..128 tokens per tile and rank 16..128 the operand
// tiles are far below the 128-row tcgen05 shapes, and TMEM allocation and
// commit round trips would cost more than the MMA time they save.  h enters
// the expand as bf16 hi + lo (about 16 significant bits), y is updated in fp32
// and rounded once.
#define LORA_DBG_FILE 5
#include <algorithm>

#include "internal.h"
#include "tc_common.cuh"
#include "tc_host.h"

namespace lora {
namespace {

using tc::cp_async_16;
using tc::cp_async_commit;
using tc::smem_u32;

constexpr int kThreads = 256;
constexpr int kKC = 128;           // shrink: columns of d_in per pipeline chunk
constexpr int kXStride = kKC + 8;  // bf16 per shared row: a 16-byte skew keeps ldmatrix conflict-free
constexpr int kNW = 256;           // expand: columns of d_out per work item
constexpr int kYStride = kNW + 8;
constexpr int kMaxStages = 6;
constexpr int kPRows = 128;        // shrink: k-groups x tile rows of per-warp sums (8 / mg x 16 mg at most)

// The projections of one call (blockIdx.y): tables share d_in and the adapter
// count; ranks, scales, B and d_out are per projection.
struct ProjSet {
    lora_adapter_table tab[kMaxProjections];
    uint16_t *y[kMaxProjections];
    float *H[kMaxProjections];     // fp32 H by token, or null
    float *part[kMaxProjections];  // [ks, T, rp_cap] fp32 slice partials of h
    int32_t n;
};

struct Geom {
    int32_t rows_cap;  // tile rows the shared buffers hold (multiple of 16, <= 128)
    int32_t rp_cap;    // rank rows they hold: the largest r_max rounded up to 16
    int32_t kw;        // shrink: columns per slice of d_in (multiple of kKC)
    int32_t ks;        // shrink: slices of d_in (<= kDecodeSlices)
    int32_t stages;    // shrink: stages of rows_cap + rp_cap rows the ring holds (>= 2)
    int32_t ns;        // expand: slices of the widest d_out
};

LORA_DEV int32_t rpad16(int32_t r) { return (r + 15) & ~15; }

LORA_DEV void cp_async_wait_n(int n)
{
    switch (n) {
    case 0: tc::cp_async_wait<0>(); break;
    case 1: tc::cp_async_wait<1>(); break;
    case 2: tc::cp_async_wait<2>(); break;
    case 3: tc::cp_async_wait<3>(); break;
    case 4: tc::cp_async_wait<4>(); break;
    default: tc::cp_async_wait<5>(); break;
    }
}

LORA_DEV void ldsm_x4(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
LORA_DEV void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4])
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// D[16 x 8] += A[16 x 16] B[16 x 8], bf16 operands, fp32 accumulators
LORA_DEV void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A work item's tile, its adapter's table entry and the token of row
// threadIdx.x, read in two rounds of memory latency instead of four: the tile
// alongside the tile count, the table entry alongside the token.  For a tile
// index past the count the dependent reads use clamped indexes (so they stay
// in bounds) and their values are discarded.
struct DecTile {
    Tile T;
    AdapterInfo ad;
    int32_t my_tok;
    bool run;
};

LORA_DEV DecTile dec_tile(const lora_adapter_table &tab, const lora_segments &segs, int32_t ti)
{
    DecTile d;
    const int32_t n_tiles = N_TILES(segs);
    d.run = ti < n_tiles;
    d.T = d.run ? LOAD_TILE(segs, ti) : Tile{0, 0, 1, 0};
    const int32_t a = min(max(d.T.adapter, 0), tab.n_adapters - 1);
    const int32_t b = min(max(d.T.begin, 0), segs.n_tokens - 1);
    d.ad.rank = __ldg(tab.rank + a);
    d.ad.row_off = __ldg(tab.row_off + a);
    d.ad.scale = __ldg(tab.scale + a);
    // only a row of the tile has a token (perm past the valid entries is unwritten)
    d.my_tok = d.run && (int32_t)threadIdx.x < d.T.rows
                   ? PERM_AT(segs, min(b + (int32_t)threadIdx.x, segs.n_tokens - 1))
                   : 0;
    d.ad.ok = d.ad.rank >= 1 && d.ad.rank <= tab.r_max && d.ad.row_off >= 0 &&
              (int64_t)d.ad.row_off + d.ad.rank <= (int64_t)tab.sum_r;
    if (d.run && !d.ad.ok) set_status(segs.status, LORA_ERR_BAD_TABLE);
    return d;
}

size_t shrink_smem(const Geom &g)
{
    return (size_t)g.stages * (g.rows_cap + g.rp_cap) * kXStride * 2 + (size_t)kPRows * g.rp_cap * 4 +
           (size_t)g.rows_cap * 4;
}
size_t expand_smem(const Geom &g)
{
    return (size_t)g.rp_cap * kYStride * 2 + (size_t)g.rows_cap * kYStride * 2 +
           2 * (size_t)g.rows_cap * (g.rp_cap + 8) * 2 + (size_t)g.rows_cap * 4;
}

// ------------------------------------------------------------------ shrink
// Warps split a tile as (16-row m-tile) x (k16 steps of each chunk): with mt
// m-tiles (rounded up to a power of two, mg) there are 8 / mg warps per
// m-tile, each taking every (8 / mg)-th k16 step, all rank columns.  Each
// k-group leaves its sums in shared memory; they are added in a fixed order
// and the tile's partial goes to P_s in perm order.
__global__ void __launch_bounds__(kThreads, 2) dec_shrink_kernel(const uint16_t *__restrict__ x,
                                                              const __grid_constant__ ProjSet ps, Geom g,
                                                              lora_segments segs)
{
    // an ordinary launch: everything earlier on the stream is complete and
    // visible.  The expand, a programmatic dependent of this grid, may start
    // its own loads of B and y now (this kernel writes neither)
    pdl_launch_dependents();
    const int32_t ti = blockIdx.x / g.ks, sl = blockIdx.x % g.ks;
    const lora_adapter_table &tab = ps.tab[blockIdx.y];
    float *__restrict__ part = ps.part[blockIdx.y];
    const DecTile D = dec_tile(tab, segs, ti);
    if (!D.run || !D.ad.ok) return;
    const Tile &T = D.T;
    const AdapterInfo &ad = D.ad;
    const int32_t d_in = tab.d_in;
    const int rows = T.rows, r = ad.rank, rp = rpad16(r), rows16 = (rows + 15) & ~15;

    extern __shared__ __align__(16) uint8_t smem[];
    // ring of stages sized for this tile: [rows16 x rows of x | rp rows of A_i] x kXStride
    uint16_t *ring = reinterpret_cast<uint16_t *>(smem);
    float *P = reinterpret_cast<float *>(ring + (size_t)g.stages * (g.rows_cap + g.rp_cap) * kXStride);  // [kg][rows16][rp]
    int32_t *tok = reinterpret_cast<int32_t *>(P + (size_t)kPRows * g.rp_cap);          // [rows16]

    const int32_t j_lo = sl * g.kw, j_hi = min(d_in, j_lo + g.kw);
    const int nchunks = (j_hi - j_lo + kKC - 1) / kKC;
    // as many stages as fit the ring for this tile's rows and rank (the host
    // sized it for at least two of the largest), all chunks at once if possible
    const int stage_elems = (rows16 + rp) * kXStride;
    const int stages =
        max(2, min(min(kMaxStages, nchunks + 1), (int)((size_t)g.stages * (g.rows_cap + g.rp_cap) / (rows16 + rp))));
    uint16_t *xs = ring;             // stage s: xs + s * stage_elems, rows16 rows
    uint16_t *as = ring + rows16 * kXStride;  // stage s: as + s * stage_elems, rp rows
    // chunk c -> stage s: x rows (gathered) and A_i rows, 16-byte pieces; past the
    // slice, the tile or the rank the pieces are zero-filled
    auto load_x = [&](int c, int s) {
        const int32_t j0 = j_lo + c * kKC;
        uint16_t *xd = xs + (size_t)s * stage_elems;
        for (int i = threadIdx.x; i < rows16 * (kKC / 8); i += kThreads) {
            const int m = i / (kKC / 8), p = i % (kKC / 8);
            const int32_t t = tok[m], j = j0 + 8 * p;
            const bool v = t >= 0 && j < j_hi;
            cp_async_16(xd + m * kXStride + 8 * p, v ? x + (int64_t)t * d_in + j : x, v);
        }
    };
    auto load_a = [&](int c, int s) {
        const int32_t j0 = j_lo + c * kKC;
        const uint16_t *A = static_cast<const uint16_t *>(tab.A);
        uint16_t *wd = as + (size_t)s * stage_elems;
        for (int i = threadIdx.x; i < rp * (kKC / 8); i += kThreads) {
            const int k = i / (kKC / 8), p = i % (kKC / 8);
            const int32_t j = j0 + 8 * p;
            const bool v = k < r && j < j_hi;
            cp_async_16(wd + k * kXStride + 8 * p, v ? A + (int64_t)(ad.row_off + k) * d_in + j : A, v);
        }
    };
    // the first stages' weights need no tokens: they go out before the tokens
    // land; each chunk's weights sit in its own or an earlier copy group
    for (int c = 0; c < stages - 1; ++c)
        if (c < nchunks) load_a(c, c);
    if (threadIdx.x < rows16) tok[threadIdx.x] = (int)threadIdx.x < rows ? D.my_tok : -1;
    __syncthreads();
    for (int c = 0; c < stages - 1; ++c) {
        if (c < nchunks) load_x(c, c);
        cp_async_commit();
    }

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int mt = rows16 / 16;
    const int mg = mt <= 1 ? 1 : mt <= 2 ? 2 : mt <= 4 ? 4 : 8;
    const int kg = 8 / mg;
    const int my_m = warp % mg, my_k = warp / mg;
    const bool active = my_m < mt;
    const int np = rp / 16;  // pairs of 8-column n-tiles
    const int lj = lane >> 3, lr = lane & 7;
    float acc[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;

    for (int c = 0; c < nchunks; ++c) {
        cp_async_wait_n(stages - 2);
        __syncthreads();  // chunk c landed for every thread; stage (c - 1) % stages is free
        {
            const int cn = c + stages - 1;
            if (cn < nchunks) {
                load_a(cn, cn % stages);
                load_x(cn, cn % stages);
            }
            cp_async_commit();
        }
        if (!active) continue;
        const int s = c % stages;
        const uint16_t *xt = xs + (size_t)s * stage_elems;
        const uint16_t *at = as + (size_t)s * stage_elems;
        for (int kk = my_k; kk < kKC / 16; kk += kg) {
            uint32_t a[4];
            ldsm_x4(smem_u32(xt + (16 * my_m + lr + 8 * (lj & 1)) * kXStride + 16 * kk + 8 * (lj >> 1)), a);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (q < np) {
                    uint32_t b[4];  // n-tiles 2q, 2q + 1: rank rows 16 q .., k16 step kk
                    ldsm_x4(smem_u32(at + (16 * q + lr + 8 * (lj >> 1)) * kXStride + 16 * kk + 8 * (lj & 1)), b);
                    mma16816(acc[2 * q], a, b[0], b[1]);
                    mma16816(acc[2 * q + 1], a, b[2], b[3]);
                }
            }
        }
    }
    tc::cp_async_wait<0>();
    if (active) {  // k-group my_k's sums: P[my_k][row][col]
        float *Pk = P + (size_t)my_k * rows16 * rp;
        const int row = 16 * my_m + (lane >> 2), col = 2 * (lane & 3);
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            if (n < 2 * np) {
                *reinterpret_cast<float2 *>(Pk + row * rp + 8 * n + col) = make_float2(acc[n][0], acc[n][1]);
                *reinterpret_cast<float2 *>(Pk + (row + 8) * rp + 8 * n + col) = make_float2(acc[n][2], acc[n][3]);
            }
        }
    }
    __syncthreads();
    // this CTA's slice partial: the k-groups added in a fixed order (the result
    // does not depend on timing), rows of the tile in perm order, to the workspace
    float *pout = part + ((int64_t)sl * segs.n_tokens + T.begin) * g.rp_cap;
    for (int i = threadIdx.x; i < rows * (rp / 4); i += kThreads) {
        const int m = i / (rp / 4), k4 = i % (rp / 4);
        float4 v = *reinterpret_cast<const float4 *>(P + m * rp + 4 * k4);
        for (int q = 1; q < kg; ++q) {
            const float4 u = *reinterpret_cast<const float4 *>(P + ((size_t)q * rows16 + m) * rp + 4 * k4);
            v.x += u.x;
            v.y += u.y;
            v.z += u.z;
            v.w += u.w;
        }
        *reinterpret_cast<float4 *>(pout + (int64_t)m * g.rp_cap + 4 * k4) = v;
    }
}

// ------------------------------------------------------------------ expand
// Warp w owns columns 32 w .. 32 w + 31 of the slice (four n-tiles) and walks
// the tile's m-tiles; y is updated in shared memory and written back in
// 16-byte pieces.
__global__ void __launch_bounds__(kThreads, 2) dec_expand_kernel(const __grid_constant__ ProjSet ps, Geom g,
                                                              lora_segments segs)
{
    const int32_t ti = blockIdx.x / g.ns, nsl = blockIdx.x % g.ns;
    const lora_adapter_table &tab = ps.tab[blockIdx.y];
    uint16_t *__restrict__ y = ps.y[blockIdx.y];
    const float *__restrict__ part = ps.part[blockIdx.y];
    float *__restrict__ H_save = ps.H[blockIdx.y];
    if (nsl * kNW >= tab.d_out) return;  // a narrower projection has fewer slices
    // the routing was complete before the shrink started, so it can be read
    // before the wait; so can B and y, which the shrink does not write
    const DecTile D = dec_tile(tab, segs, ti);
    if (!D.run || !D.ad.ok) return;
    const Tile &T = D.T;
    const AdapterInfo &ad = D.ad;
    const int32_t d_out = tab.d_out;
    const int rows = T.rows, r = ad.rank, rp = rpad16(r), rows16 = (rows + 15) & ~15;
    const int hs = g.rp_cap + 8;  // bf16 per row of the h operand

    extern __shared__ __align__(16) uint8_t smem[];
    uint16_t *bs = reinterpret_cast<uint16_t *>(smem);            // [rp_cap][kYStride]: B_i^T rows k
    uint16_t *ys = bs + (size_t)g.rp_cap * kYStride;              // [rows_cap][kYStride]
    uint16_t *hh = ys + (size_t)g.rows_cap * kYStride;            // [rows_cap][hs] bf16 hi of h
    uint16_t *hl = hh + (size_t)g.rows_cap * hs;                  // [rows_cap][hs] bf16 lo of h
    int32_t *tok = reinterpret_cast<int32_t *>(hl + (size_t)g.rows_cap * hs);

    const int32_t o_lo = nsl * kNW;
    for (int i = threadIdx.x; i < rp * (kNW / 8); i += kThreads) {
        const int k = i / (kNW / 8), p = i % (kNW / 8);
        const int32_t o = o_lo + 8 * p;
        const bool v = k < r && o < d_out;
        const uint16_t *B = static_cast<const uint16_t *>(tab.B);
        cp_async_16(bs + k * kYStride + 8 * p, v ? B + (int64_t)(ad.row_off + k) * d_out + o : B, v);
    }
    if (threadIdx.x < rows16) tok[threadIdx.x] = (int)threadIdx.x < rows ? D.my_tok : -1;
    __syncthreads();
    for (int i = threadIdx.x; i < rows * (kNW / 8); i += kThreads) {
        const int m = i / (kNW / 8), p = i % (kNW / 8);
        const int32_t o = o_lo + 8 * p;
        const bool v = o < d_out;
        cp_async_16(ys + m * kYStride + 8 * p, v ? y + (int64_t)tok[m] * d_out + o : y, v);
    }
    cp_async_commit();

    pdl_wait();  // the shrink grid has completed and its partials are visible

    // h = the slice partials added in slice order (every item of the tile
    // adds them alike); the tile's first item also writes the fp32 H
    const int32_t T_all = segs.n_tokens, r_max = tab.r_max;
    const bool write_h = H_save != nullptr && nsl == 0;
    for (int i = threadIdx.x; i < rows16 * (rp / 4); i += kThreads) {
        const int m = i / (rp / 4), k4 = i % (rp / 4);
        float e[4] = {0.f, 0.f, 0.f, 0.f};
        if (m < rows) {
            const float *src = part + ((int64_t)T.begin + m) * g.rp_cap + 4 * k4;
            float4 v[kDecodeSlices];
#pragma unroll
            for (int q = 0; q < kDecodeSlices; ++q)
                if (q < g.ks) v[q] = __ldcg(reinterpret_cast<const float4 *>(src + (int64_t)q * T_all * g.rp_cap));
#pragma unroll
            for (int q = 0; q < kDecodeSlices; ++q) {
                if (q < g.ks) {
                    e[0] += v[q].x;
                    e[1] += v[q].y;
                    e[2] += v[q].z;
                    e[3] += v[q].w;
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (4 * k4 + u >= r) e[u] = 0.f;
            if (write_h) {
                float *hrow = H_save + (int64_t)tok[m] * r_max;
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (4 * k4 + u < r_max) hrow[4 * k4 + u] = e[u];
            }
        }
        const uint32_t h01 = pack_bf16(e[0], e[1]), h23 = pack_bf16(e[2], e[3]);
        const uint32_t l01 = pack_bf16(e[0] - bf16lo(h01), e[1] - bf16hi(h01));
        const uint32_t l23 = pack_bf16(e[2] - bf16lo(h23), e[3] - bf16hi(h23));
        *reinterpret_cast<uint2 *>(hh + m * hs + 4 * k4) = make_uint2(h01, h23);
        *reinterpret_cast<uint2 *>(hl + m * hs + 4 * k4) = make_uint2(l01, l23);
    }
    if (write_h)  // columns r_pad .. r_max - 1
        for (int i = threadIdx.x; i < rows * r_max; i += kThreads) {
            const int m = i / r_max, k = i % r_max;
            if (k >= rp) H_save[(int64_t)tok[m] * r_max + k] = 0.f;
        }
    tc::cp_async_wait<0>();
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int lj = lane >> 3, lr = lane & 7;
    const float c = ad.scale;
    for (int mi = 0; mi < rows16 / 16; ++mi) {
        float acc[4][4];
#pragma unroll
        for (int n = 0; n < 4; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
        for (int kk = 0; kk < rp / 16; ++kk) {
            uint32_t ah[4], al[4];
            const int arow = 16 * mi + lr + 8 * (lj & 1), acol = 16 * kk + 8 * (lj >> 1);
            ldsm_x4(smem_u32(hh + arow * hs + acol), ah);
            ldsm_x4(smem_u32(hl + arow * hs + acol), al);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                uint32_t b[4];  // n-tiles at columns 32 w + 16 q and + 8: k rows 16 kk ..
                ldsm_x4_trans(smem_u32(bs + (16 * kk + lr + 8 * (lj & 1)) * kYStride + 32 * warp + 16 * q + 8 * (lj >> 1)),
                              b);
                mma16816(acc[2 * q], ah, b[0], b[1]);
                mma16816(acc[2 * q], al, b[0], b[1]);
                mma16816(acc[2 * q + 1], ah, b[2], b[3]);
                mma16816(acc[2 * q + 1], al, b[2], b[3]);
            }
        }
        const int row = 16 * mi + (lane >> 2);
#pragma unroll
        for (int n = 0; n < 4; ++n) {
            const int col = 32 * warp + 8 * n + 2 * (lane & 3);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t *p = reinterpret_cast<uint32_t *>(ys + (row + 8 * hf) * kYStride + col);
                const uint32_t w = *p;
                *p = pack_bf16(bf16lo(w) + c * acc[n][2 * hf], bf16hi(w) + c * acc[n][2 * hf + 1]);
            }
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < rows * (kNW / 8); i += kThreads) {
        const int m = i / (kNW / 8), p = i % (kNW / 8);
        const int32_t o = o_lo + 8 * p;
        if (o < d_out)
            *reinterpret_cast<uint4 *>(y + (int64_t)tok[m] * d_out + o) =
                *reinterpret_cast<const uint4 *>(ys + m * kYStride + 8 * p);
    }
}

// slices of d_in of at least 256 columns, at most kDecodeSlices of them
int32_t slice_width(int32_t d_in)
{
    const int32_t per = (d_in + kDecodeSlices - 1) / kDecodeSlices;
    return std::max<int32_t>(2 * kKC, ((per + kKC - 1) / kKC) * kKC);
}

Geom make_geom(const ProjSet &ps, const lora_segments &segs)
{
    Geom g;
    const lora_adapter_table &tab = ps.tab[0];  // d_in is common to the set
    const int32_t T = segs.n_tokens;
    int32_t r_max = 0, d_out = 0;
    for (int p = 0; p < ps.n; ++p) {
        r_max = std::max(r_max, ps.tab[p].r_max);
        d_out = std::max(d_out, ps.tab[p].d_out);
    }
    g.rows_cap = std::min<int32_t>(LORA_TILE_M, (T + 15) & ~15);
    g.rp_cap = (r_max + 15) & ~15;
    g.kw = slice_width(tab.d_in);
    g.ks = (tab.d_in + g.kw - 1) / g.kw;
    // as many stages as the slice has chunks, within ~100 KB (two CTAs of the
    // two kernels then fit one SM), at least two
    const int32_t chunks = g.kw / kKC;
    const size_t stage = (size_t)(g.rows_cap + g.rp_cap) * kXStride * 2;
    const size_t fixed = (size_t)kPRows * g.rp_cap * 4 + (size_t)g.rows_cap * 4;
    int32_t st = (int32_t)((100u * 1024u > fixed ? 100u * 1024u - fixed : 0) / stage);
    st = std::min<int32_t>(std::min<int32_t>(st, chunks), kMaxStages);
    g.stages = std::max<int32_t>(st, 2);
    g.ns = (d_out + kNW - 1) / kNW;
    return g;
}

}  // namespace

size_t decode_workspace_bytes(int32_t T, int32_t r_max, int32_t d_in)
{
    const int32_t kw = slice_width(d_in);
    const size_t ks = (size_t)((d_in + kw - 1) / kw);
    return ks * (size_t)T * (size_t)((r_max + 15) & ~15) * sizeof(float);
}

lora_status_t tc_decode_multi(int32_t n_proj, void *const *y, float *const *H_save, const void *x, void *ws,
                              const lora_adapter_table *tabs, const lora_segments &segs, cudaStream_t stream)
{
    if (segs.n_tokens == 0 || segs.max_tiles == 0 || n_proj == 0) return LORA_OK;
    if (n_proj < 0 || n_proj > kMaxProjections) return LORA_ERR_SHAPE;
    ProjSet ps = {};
    ps.n = n_proj;
    int32_t r_max = 0;
    for (int p = 0; p < n_proj; ++p) r_max = std::max(r_max, tabs[p].r_max);
    const size_t per = decode_workspace_bytes(segs.n_tokens, r_max, tabs[0].d_in);
    for (int p = 0; p < n_proj; ++p) {
        ps.tab[p] = tabs[p];
        ps.y[p] = static_cast<uint16_t *>(y[p]);
        ps.H[p] = H_save != nullptr ? H_save[p] : nullptr;
        ps.part[p] = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + (size_t)p * per);
    }
    const Geom g = make_geom(ps, segs);
    const size_t s1 = shrink_smem(g), s2 = expand_smem(g);
    if (cudaFuncSetAttribute(dec_shrink_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1) != cudaSuccess ||
        cudaFuncSetAttribute(dec_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s2) != cudaSuccess)
        return LORA_ERR_CUDA;
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(segs.max_tiles * g.ks), (unsigned)n_proj);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = s1;
        cfg.stream = stream;
        // an ordinary (not programmatic) launch: the shrink reads the routing
        // and A_i, which the kernel before it may have written (a routing
        // build, an optimizer step), and only a completed predecessor is
        // guaranteed visible without a grid-dependency wait
        if (cudaLaunchKernelEx(&cfg, dec_shrink_kernel, static_cast<const uint16_t *>(x), ps, g, segs) != cudaSuccess)
            return LORA_ERR_CUDA;
    }
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(segs.max_tiles * g.ns), (unsigned)n_proj);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = s2;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, dec_expand_kernel, ps, g, segs) != cudaSuccess) return LORA_ERR_CUDA;
    }
    return LORA_OK;
}

lora_status_t tc_decode_fwd(void *y, float *H_save, const void *x, void *ws, const lora_adapter_table &tab,
                            const lora_segments &segs, cudaStream_t stream)
{
    void *ys[1] = {y};
    float *hs[1] = {H_save};
    return tc_decode_multi(1, ys, hs, x, ws, &tab, segs, stream);
}

}  // namespace lora
