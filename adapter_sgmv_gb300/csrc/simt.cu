// simt.cu -- generic CUDA-core kernels for all six products.
//
// These take any rank (1..LORA_MAX_RANK), any routing (sorted or gathered
// rows) and any d that is a multiple of 8.  They accumulate in fp32 with
// plain FMAs, one output per thread register, with shared-memory staging of
// 32-token x 64-column activation blocks and the matching weight block.  The
// tensor-core kernels cover the bulk of the packed path; these cover what
// they do not (ranks that are not a multiple of 16, and small batches), and
// serve as an independent second implementation in the tests.
//
// Products (PLoRA technical summary, "2. LoRA Execution Engine": four cases
// over concatenated adapter tensors; shrink/expand as in C-LoRA's SGMV):
//   rowproj   case i    out[t, k] = c * sum_j W(k, j) act[t, j]   (shrink, dh)
//   colproj   case ii   out[t, n] += c * sum_k W(n, k) h[t, k]    (expand, dX)
//   tokred    iii / iv  G_i[n, k] = c * sum_{t in i} act[t, n] h[t, k]   (dB, dA)
#include "common.cuh"
#include "internal.h"

namespace lora {

namespace {

constexpr int kThreads = 256;
constexpr int kRows = 32;   // token rows per sub-block
constexpr int kCols = 64;   // reduction / output columns per step
constexpr int kPad = kCols + 1;

template <bool kDH>
__global__ void __launch_bounds__(kThreads)
simt_rowproj_kernel(float *__restrict__ out, const uint16_t *__restrict__ act, lora_adapter_table tab,
                    lora_segments segs)
{
    __shared__ float act_s[kRows][kPad];
    __shared__ float w_s[LORA_MAX_RANK][kPad];
    __shared__ int32_t tok_s[kRows];
    const int tile_idx = blockIdx.x;
    if (tile_idx >= *segs.n_tiles) return;
    const Tile tile = load_tile(segs.tiles, tile_idx);
    const AdapterInfo ad = load_adapter(tab, tile.adapter, segs.status);
    if (!ad.ok) return;
    const int32_t d = kDH ? tab.d_out : tab.d_in;
    const int32_t r = ad.rank, r_max = tab.r_max;
    const float c = kDH ? ad.scale : 1.0f;
    // W(k, j): shrink A_i[k, j]; dh B_i[j, k], i.e. row k of the stacked B_i^T
    const uint16_t *W = static_cast<const uint16_t *>(kDH ? tab.B : tab.A) + (int64_t)ad.row_off * d;
    const int row = threadIdx.x % kRows, kg = threadIdx.x / kRows;  // k = kg + 8 q

    for (int m0 = 0; m0 < tile.rows; m0 += kRows) {
        const int nrows = min(kRows, tile.rows - m0);
        __syncthreads();
        if (threadIdx.x < kRows)
            tok_s[threadIdx.x] = threadIdx.x < nrows ? segs.perm[tile.begin + m0 + threadIdx.x] : -1;
        float acc[LORA_MAX_RANK / 8];
#pragma unroll
        for (int q = 0; q < LORA_MAX_RANK / 8; ++q) acc[q] = 0.f;
        for (int j0 = 0; j0 < d; j0 += kCols) {
            __syncthreads();
            for (int e = threadIdx.x; e < kRows * kCols; e += kThreads) {
                const int m = e / kCols, j = e % kCols;
                const int32_t t = tok_s[m];
                act_s[m][j] = (t >= 0 && j0 + j < d) ? bf16_to_f32(act[(int64_t)t * d + j0 + j]) : 0.f;
            }
            for (int e = threadIdx.x; e < r * kCols; e += kThreads) {
                const int k = e / kCols, j = e % kCols;
                w_s[k][j] = (j0 + j < d) ? bf16_to_f32(W[(int64_t)k * d + j0 + j]) : 0.f;
            }
            __syncthreads();
#pragma unroll 4
            for (int j = 0; j < kCols; ++j) {
                const float a = act_s[row][j];
#pragma unroll
                for (int q = 0; q < LORA_MAX_RANK / 8; ++q) {
                    const int k = kg + 8 * q;
                    if (k < r) acc[q] = fmaf(w_s[k][j], a, acc[q]);
                }
            }
        }
        const int32_t t = tok_s[row];
        if (row < nrows && t >= 0) {
#pragma unroll
            for (int q = 0; q < LORA_MAX_RANK / 8; ++q) {
                const int k = kg + 8 * q;
                if (k < r_max) out[(int64_t)t * r_max + k] = k < r ? c * acc[q] : 0.f;
            }
        }
    }
}

// W(n, k): expand B_i[n, k] (row k of the stacked B_i^T); dX A_i[k, n]
template <bool kDX>
__global__ void __launch_bounds__(kThreads)
simt_colproj_kernel(uint16_t *__restrict__ out, const float *__restrict__ h, lora_adapter_table tab,
                    lora_segments segs)
{
    __shared__ float h_s[kRows][kPad];
    __shared__ float w_s[kCols][kPad];
    __shared__ int32_t tok_s[kRows];
    const int tile_idx = blockIdx.x;
    if (tile_idx >= *segs.n_tiles) return;
    const Tile tile = load_tile(segs.tiles, tile_idx);
    const AdapterInfo ad = load_adapter(tab, tile.adapter, segs.status);
    if (!ad.ok) return;
    const int32_t d = kDX ? tab.d_in : tab.d_out;
    const int32_t n0 = blockIdx.y * kCols;
    if (n0 >= d) return;
    const int32_t r = ad.rank, r_max = tab.r_max;
    const float c = kDX ? 1.0f : ad.scale;
    const uint16_t *W = static_cast<const uint16_t *>(kDX ? tab.A : tab.B) + (int64_t)ad.row_off * d;
    const int n = threadIdx.x % kCols, rg = threadIdx.x / kCols;  // rows rg + 4 q

    for (int m0 = 0; m0 < tile.rows; m0 += kRows) {
        const int nrows = min(kRows, tile.rows - m0);
        __syncthreads();
        if (threadIdx.x < kRows)
            tok_s[threadIdx.x] = threadIdx.x < nrows ? segs.perm[tile.begin + m0 + threadIdx.x] : -1;
        float acc[kRows / 4];
#pragma unroll
        for (int q = 0; q < kRows / 4; ++q) acc[q] = 0.f;
        for (int k0 = 0; k0 < r; k0 += kCols) {
            const int kn = min(kCols, r - k0);
            __syncthreads();
            for (int e = threadIdx.x; e < kRows * kCols; e += kThreads) {
                const int m = e / kCols, k = e % kCols;
                const int32_t t = tok_s[m];
                h_s[m][k] = (t >= 0 && k < kn) ? h[(int64_t)t * r_max + k0 + k] : 0.f;
            }
            for (int e = threadIdx.x; e < kCols * kCols; e += kThreads) {
                const int k = e / kCols, nn = e % kCols;
                w_s[nn][k] = (k < kn && n0 + nn < d) ? bf16_to_f32(W[(int64_t)(k0 + k) * d + n0 + nn]) : 0.f;
            }
            __syncthreads();
            for (int k = 0; k < kn; ++k) {
                const float w = w_s[n][k];
#pragma unroll
                for (int q = 0; q < kRows / 4; ++q) acc[q] = fmaf(h_s[rg + 4 * q][k], w, acc[q]);
            }
        }
        if (n0 + n < d) {
#pragma unroll
            for (int q = 0; q < kRows / 4; ++q) {
                const int m = rg + 4 * q;
                const int32_t t = tok_s[m];
                if (m < nrows && t >= 0) {
                    uint16_t *p = out + (int64_t)t * d + n0 + n;
                    *p = f32_to_bf16(bf16_to_f32(*p) + c * acc[q]);
                }
            }
        }
    }
}

// token reductions: G_i[n, k] = c * sum_{t in i} act[t, n] h[t, k], stored at
// row row_off[i] + k, column n of a [sum_r, d] array --------------------------
//   dB: act = dY (n = o), h = H,  c = s_i  (dB_i^T stacked like B)
//   dA: act = X  (n = j), h = dH, c = 1    (dA_i stacked like A)
template <bool kDA>
__global__ void __launch_bounds__(kThreads)
simt_tokred_kernel(float *__restrict__ G, const uint16_t *__restrict__ act, const float *__restrict__ h,
                   lora_adapter_table tab, lora_segments segs)
{
    __shared__ float a_s[kRows][kPad];
    __shared__ float h_s[kRows][LORA_MAX_RANK + 1];
    __shared__ int32_t tok_s[kRows];
    const int32_t i = blockIdx.x;
    const AdapterInfo ad = load_adapter(tab, i, segs.status);
    if (!ad.ok) return;
    const int32_t d = kDA ? tab.d_in : tab.d_out;
    const int32_t n0 = blockIdx.y * kCols;
    if (n0 >= d) return;
    const int32_t r = ad.rank, r_max = tab.r_max;
    const float c = kDA ? 1.0f : ad.scale;
    const int n = threadIdx.x % kCols, kg = threadIdx.x / kCols;  // k = kg + 4 q
    const int32_t g0 = segs.seg_start[i], g1 = segs.seg_start[i + 1];
    float acc[LORA_MAX_RANK / 4];
#pragma unroll
    for (int q = 0; q < LORA_MAX_RANK / 4; ++q) acc[q] = 0.f;
    for (int32_t p0 = g0; p0 < g1; p0 += kRows) {
        const int nrows = min(kRows, g1 - p0);
        __syncthreads();
        if (threadIdx.x < kRows) tok_s[threadIdx.x] = threadIdx.x < nrows ? segs.perm[p0 + threadIdx.x] : -1;
        __syncthreads();
        for (int e = threadIdx.x; e < kRows * kCols; e += kThreads) {
            const int m = e / kCols, nn = e % kCols;
            const int32_t t = tok_s[m];
            a_s[m][nn] = (t >= 0 && n0 + nn < d) ? bf16_to_f32(act[(int64_t)t * d + n0 + nn]) : 0.f;
        }
        for (int e = threadIdx.x; e < kRows * r; e += kThreads) {
            const int m = e / r, k = e % r;
            const int32_t t = tok_s[m];
            h_s[m][k] = t >= 0 ? h[(int64_t)t * r_max + k] : 0.f;
        }
        __syncthreads();
        for (int m = 0; m < nrows; ++m) {
            const float a = a_s[m][n];
#pragma unroll
            for (int q = 0; q < LORA_MAX_RANK / 4; ++q) {
                const int k = kg + 4 * q;
                if (k < r) acc[q] = fmaf(a, h_s[m][k], acc[q]);
            }
        }
    }
    if (n0 + n < d) {
#pragma unroll
        for (int q = 0; q < LORA_MAX_RANK / 4; ++q) {
            const int k = kg + 4 * q;
            if (k < r) G[((int64_t)ad.row_off + k) * d + n0 + n] = c * acc[q];
        }
    }
}

lora_status_t launched()
{
    return cudaGetLastError() == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

}  // namespace

lora_status_t simt_shrink(float *H, const void *x, const lora_adapter_table &tab, const lora_segments &segs,
                          cudaStream_t stream)
{
    if (segs.max_tiles <= 0 || segs.n_tokens == 0) return LORA_OK;
    simt_rowproj_kernel<false><<<segs.max_tiles, kThreads, 0, stream>>>(
        H, static_cast<const uint16_t *>(x), tab, segs);
    return launched();
}

lora_status_t simt_dh(float *dH, const void *dY, const lora_adapter_table &tab, const lora_segments &segs,
                      cudaStream_t stream)
{
    if (segs.max_tiles <= 0 || segs.n_tokens == 0) return LORA_OK;
    simt_rowproj_kernel<true><<<segs.max_tiles, kThreads, 0, stream>>>(
        dH, static_cast<const uint16_t *>(dY), tab, segs);
    return launched();
}

lora_status_t simt_expand(void *y, const float *H, const lora_adapter_table &tab, const lora_segments &segs,
                          cudaStream_t stream)
{
    if (segs.max_tiles <= 0 || segs.n_tokens == 0) return LORA_OK;
    dim3 grid(segs.max_tiles, (tab.d_out + kCols - 1) / kCols);
    simt_colproj_kernel<false><<<grid, kThreads, 0, stream>>>(static_cast<uint16_t *>(y), H, tab, segs);
    return launched();
}

lora_status_t simt_dx(void *dX, const float *dH, const lora_adapter_table &tab, const lora_segments &segs,
                      cudaStream_t stream)
{
    if (segs.max_tiles <= 0 || segs.n_tokens == 0) return LORA_OK;
    dim3 grid(segs.max_tiles, (tab.d_in + kCols - 1) / kCols);
    simt_colproj_kernel<true><<<grid, kThreads, 0, stream>>>(static_cast<uint16_t *>(dX), dH, tab, segs);
    return launched();
}

lora_status_t simt_db(float *dB, const void *dY, const float *H, const lora_adapter_table &tab,
                      const lora_segments &segs, cudaStream_t stream)
{
    dim3 grid(tab.n_adapters, (tab.d_out + kCols - 1) / kCols);
    simt_tokred_kernel<false><<<grid, kThreads, 0, stream>>>(dB, static_cast<const uint16_t *>(dY), H, tab, segs);
    return launched();
}

lora_status_t simt_da(float *dA, const float *dH, const void *X, const lora_adapter_table &tab,
                      const lora_segments &segs, cudaStream_t stream)
{
    dim3 grid(tab.n_adapters, (tab.d_in + kCols - 1) / kCols);
    simt_tokred_kernel<true><<<grid, kThreads, 0, stream>>>(dA, static_cast<const uint16_t *>(X), dH, tab, segs);
    return launched();
}

}  // namespace lora
