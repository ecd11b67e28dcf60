// adamw.cu -- the per-adapter optimizer step over the concatenated adapter
// weights, fused with the refresh of the bf16 copies the forward reads.
//
// Every tenant keeps FP32 master weights, optimizer moments and gradient
// buffers beside its LoRA parameters (C-LoRA report, "Come funziona
// l'architettura": the AdapterStore).  The pages name no optimizer; the step
// is AdamW (Adam moments with bias correction, weight decay decoupled from
// the gradient), each adapter with its own learning rate and step number:
//
//   w <- w - lr wd w;  m <- b1 m + (1 - b1) g;  v <- b2 v + (1 - b2) g^2
//   w <- w - lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps)
//   bf16 copy <- round-to-nearest-even(w)
//
// A and B^T are both [sum_r, d] row-major with adapter i on rows row_off[i] ..
// row_off[i] + r_i - 1, so one launch walks both matrices as one array of
// 16-byte groups; a group's adapter follows from its row.  The step is
// HBM-bound (30 bytes per weight: w, g, m, v read, w, m, v written in fp32 and
// the bf16 copy written), so the kernel is a grid-stride stream of 16-byte
// loads and stores over whole rows, sized to the SM count.
#include "common.cuh"
#include "internal.h"
#include "tc_host.h"

namespace lora {
namespace {

constexpr int kThreads = 256;

struct AdamwArgs {
    float *w[2];
    const float *g[2];
    float *m[2], *v[2];
    uint16_t *wb[2];   // the table's bf16 A and B^T
    int32_t d[2];      // d_in, d_out
    int64_t groups[2]; // 16-byte groups of fp32 per matrix: sum_r * d / 4
    const float *lr;
    const int32_t *step;
    float beta1, beta2, eps, wd;
};

// adapter owning `row`: the last i with row_off[i] <= row (row_off ascending)
LORA_DEV int32_t adapter_of_row(const int32_t *row_off, int32_t n, int32_t row)
{
    int32_t lo = 0, hi = n - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (__ldg(row_off + mid) <= row)
            lo = mid;
        else
            hi = mid - 1;
    }
    return lo;
}

constexpr int kU = 2;  // 16-byte groups per thread in flight per iteration

__global__ void __launch_bounds__(kThreads) adamw_kernel(AdamwArgs a, lora_adapter_table tab)
{
    const int64_t total = a.groups[0] + a.groups[1];
    const int64_t stride = (int64_t)gridDim.x * kThreads;
    // the adapter of the last row seen, with its per-step constants
    int32_t cur_mat = -1, row_lo = 0, row_hi = -1;
    float lr = 0.f, inv_bc1 = 1.f, inv_sqrt_bc2 = 1.f;
    for (int64_t q0 = (int64_t)blockIdx.x * kThreads + threadIdx.x; q0 < total; q0 += kU * stride) {
        float4 w[kU], g[kU], m[kU], v[kU];
        int mat[kU];
        int64_t e[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {  // all loads first
            const int64_t q = q0 + u * stride;
            mat[u] = -1;
            if (q >= total) continue;
            mat[u] = q < a.groups[0] ? 0 : 1;
            e[u] = (q - (mat[u] ? a.groups[0] : 0)) * 4;  // first element of the group
            w[u] = *reinterpret_cast<const float4 *>(a.w[mat[u]] + e[u]);
            g[u] = __ldcs(reinterpret_cast<const float4 *>(a.g[mat[u]] + e[u]));
            m[u] = *reinterpret_cast<const float4 *>(a.m[mat[u]] + e[u]);
            v[u] = *reinterpret_cast<const float4 *>(a.v[mat[u]] + e[u]);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (mat[u] < 0) continue;
            const int32_t row = (int32_t)(e[u] / a.d[mat[u]]);
            if (mat[u] != cur_mat || row < row_lo || row > row_hi) {
                const int32_t i = adapter_of_row(tab.row_off, tab.n_adapters, row);
                row_lo = __ldg(tab.row_off + i);
                row_hi = row_lo + __ldg(tab.rank + i) - 1;
                cur_mat = mat[u];
                const float t = (float)__ldg(a.step + i);
                lr = __ldg(a.lr + i);
                inv_bc1 = 1.f / (1.f - powf(a.beta1, t));
                inv_sqrt_bc2 = 1.f / sqrtf(1.f - powf(a.beta2, t));
            }
            float *wp = &w[u].x, *mp = &m[u].x, *vp = &v[u].x;
            const float *gp = &g[u].x;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float x = wp[c];
                x -= lr * a.wd * x;
                mp[c] = a.beta1 * mp[c] + (1.f - a.beta1) * gp[c];
                vp[c] = a.beta2 * vp[c] + (1.f - a.beta2) * gp[c] * gp[c];
                x -= lr * (mp[c] * inv_bc1) / (sqrtf(vp[c]) * inv_sqrt_bc2 + a.eps);
                wp[c] = x;
            }
            *reinterpret_cast<float4 *>(a.w[mat[u]] + e[u]) = w[u];
            *reinterpret_cast<float4 *>(a.m[mat[u]] + e[u]) = m[u];
            *reinterpret_cast<float4 *>(a.v[mat[u]] + e[u]) = v[u];
            *reinterpret_cast<uint2 *>(a.wb[mat[u]] + e[u]) =
                make_uint2(pack_bf16(w[u].x, w[u].y), pack_bf16(w[u].z, w[u].w));
        }
    }
}

}  // namespace

lora_status_t run_adamw(const lora_adapter_table &tab, float *wA, float *wB, const float *gA, const float *gB,
                        float *mA, float *vA, float *mB, float *vB, const float *lr, const int32_t *step, float beta1,
                        float beta2, float eps, float weight_decay, cudaStream_t stream)
{
    AdamwArgs a;
    a.w[0] = wA;
    a.w[1] = wB;
    a.g[0] = gA;
    a.g[1] = gB;
    a.m[0] = mA;
    a.m[1] = mB;
    a.v[0] = vA;
    a.v[1] = vB;
    a.wb[0] = static_cast<uint16_t *>(const_cast<void *>(tab.A));
    a.wb[1] = static_cast<uint16_t *>(const_cast<void *>(tab.B));
    a.d[0] = tab.d_in;
    a.d[1] = tab.d_out;
    a.groups[0] = (int64_t)tab.sum_r * tab.d_in / 4;
    a.groups[1] = (int64_t)tab.sum_r * tab.d_out / 4;
    a.lr = lr;
    a.step = step;
    a.beta1 = beta1;
    a.beta2 = beta2;
    a.eps = eps;
    a.wd = weight_decay;
    const int sms = sm_count();
    const int64_t total = a.groups[0] + a.groups[1];
    const int64_t want = (total + kThreads - 1) / kThreads;
    const int grid = (int)(want < 8LL * sms ? want : 8LL * sms);  // eight 256-thread blocks per SM
    // (each thread keeps kU groups in flight; the grid-stride loop covers the rest)
    if (grid <= 0) return LORA_OK;
    adamw_kernel<<<grid, kThreads, 0, stream>>>(a, tab);
    return cudaGetLastError() == cudaSuccess ? LORA_OK : LORA_ERR_CUDA;
}

}  // namespace lora
