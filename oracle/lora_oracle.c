/*
 * lora_oracle.c -- plain, slow fp64 CPU oracle for the multi-adapter LoRA delta.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg load this file's library; the CUDA library never links,
 * includes or calls it, and it shares no code with the CUDA kernels.
 *
 * What it computes (all arithmetic in IEEE double, inputs are bf16 values
 * widened exactly to double by the caller):
 *
 *   Routing.  Every token t carries an adapter id i = ids[t].  Tokens of
 *   different adapters are mixed in one batch and each token is served by its
 *   own adapter, all adapters being resident at once
 *   [C-LoRA report, vivodigitale.it, "Come funziona l'architettura": mixed-
 *   adapter decode batches, one fused SGMV launch per decode step].
 *   route(): a stable counting sort of token indices by adapter id (ties keep
 *   the original token order), plus the start of every adapter's group.
 *
 *   The per-token LoRA delta for adapter i with A_i (r_i x d_in),
 *   B_i (d_out x r_i) and scale s_i = alpha_i / r_i (standard LoRA algebra;
 *   the pages print no formula, so this is the plain reading of the method
 *   they describe):
 *     shrink   h_t      = A_i x_t                      (length r_i)
 *     expand   y_t     += s_i B_i h_t                  (length d_out)
 *   and its backward pass, i.e. the "four cases" of the packed kernels
 *   [PLoRA technical summary, gist.science, "2. LoRA Execution Engine",
 *   Kernelontwerp]:
 *     dh       dh_t     = s_i B_i^T dy_t               (reduce over d_out)
 *     dB       dB_i     = s_i sum_{t in i} dy_t h_t^T  (reduce over tokens)
 *     dA       dA_i     = sum_{t in i} dh_t x_t^T      (reduce over tokens)
 *     dX       dx_t    += A_i^T dh_t                   (reduce over r_i)
 *
 * Layouts (row-major, the same ones the CUDA library documents):
 *   A_cat  [sum_r, d_in]       A_i occupies rows row_off[i] .. row_off[i]+r_i-1
 *   Bt_cat [sum_r, d_out]      B_i transposed, stacked like A_cat: row
 *                              row_off[i]+k holds column k of B_i, so
 *                              B_i[o, k] = Bt_cat[row_off[i]+k, o]
 *   H, dH  [T, r_max]          columns >= r_i of token t are zero
 *   dA     like A_cat, dBt like Bt_cat
 * Tokens whose id lies outside [0, N) belong to no adapter: they contribute
 * nothing, their H/dH rows are zero and their y/dX rows are left unchanged.
 *
 *   Optimizer step.  Every tenant keeps FP32 master weights, optimizer
 *   moments and gradient buffers beside its LoRA parameters [C-LoRA report,
 *   vivodigitale.it, "Come funziona l'architettura": the AdapterStore].  The
 *   pages name no optimizer; the reading taken is AdamW (Adam moments with
 *   bias correction, weight decay decoupled from the gradient), per adapter
 *   with its own learning rate and step number:
 *     w <- w - lr wd w;  m <- b1 m + (1 - b1) g;  v <- b2 v + (1 - b2) g^2
 *     w <- w - lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps)
 *
 *   Base projection with the delta.  The frozen base weight W (d_out x d_in)
 *   is shared by every adapter of a packed batch, which is what packing
 *   amortises [PLoRA technical summary, gist.science, "2. LoRA Execution
 *   Engine"]; a LoRA layer's output is the base projection plus the delta:
 *     base     y_t      = W x_t                        (every token)
 *   and the layer output is base followed by expand(shrink) above.
 *
 * Each function is the per-token (or per-adapter) definition written out as
 * loops, with no blocking, fusion or reordering; OpenMP only splits the
 * independent outputs across threads, every sum runs in a fixed order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static int valid_id(int32_t i, int32_t n) { return i >= 0 && i < n; }

int lora_oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void lora_oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Stable counting sort of tokens by adapter id.
 * perm receives the valid tokens grouped by adapter, ascending id, original
 * order inside a group; seg_start[N+1] the group starts (seg_start[N] is the
 * number of valid tokens).  Returns the number of tokens with an id outside
 * [0, N). */
int64_t lora_oracle_route(int64_t T, int32_t N, const int32_t *ids,
                          int32_t *perm, int32_t *seg_start)
{
    int64_t *count = (int64_t *)calloc((size_t)N, sizeof(int64_t));
    int64_t *cursor = (int64_t *)calloc((size_t)N, sizeof(int64_t));
    int64_t bad = 0;
    for (int64_t t = 0; t < T; ++t) {
        if (valid_id(ids[t], N)) count[ids[t]] += 1;
        else bad += 1;
    }
    seg_start[0] = 0;
    for (int32_t i = 0; i < N; ++i) seg_start[i + 1] = seg_start[i] + (int32_t)count[i];
    for (int32_t i = 0; i < N; ++i) cursor[i] = seg_start[i];
    for (int64_t t = 0; t < T; ++t) {
        int32_t i = ids[t];
        if (!valid_id(i, N)) continue;
        perm[cursor[i]] = (int32_t)t;
        cursor[i] += 1;
    }
    free(count);
    free(cursor);
    return bad;
}

/* shrink: H[t, k] = sum_j A_i[k, j] * x[t, j] for k < r_i, zero for k >= r_i. */
void lora_oracle_shrink(int64_t T, int32_t N, int32_t d_in, int32_t r_max,
                        const int32_t *rank, const int64_t *row_off,
                        const int32_t *ids, const double *A, const double *x,
                        double *H)
{
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t t = 0; t < T; ++t) {
        double *h = H + t * r_max;
        for (int32_t k = 0; k < r_max; ++k) h[k] = 0.0;
        int32_t i = ids[t];
        if (!valid_id(i, N)) continue;
        const double *xt = x + t * (int64_t)d_in;
        for (int32_t k = 0; k < rank[i]; ++k) {
            const double *a = A + (row_off[i] + k) * (int64_t)d_in;
            double acc = 0.0;
            for (int32_t j = 0; j < d_in; ++j) acc += a[j] * xt[j];
            h[k] = acc;
        }
    }
}

/* expand: y[t, o] += s_i * sum_k B_i[o, k] * H[t, k]. */
void lora_oracle_expand(int64_t T, int32_t N, int32_t d_out, int32_t r_max,
                        const int32_t *rank, const int64_t *row_off,
                        const double *scale, const int32_t *ids,
                        const double *Bt, const double *H, double *y)
{
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t t = 0; t < T; ++t) {
        int32_t i = ids[t];
        if (!valid_id(i, N)) continue;
        const int32_t r = rank[i];
        const double *h = H + t * r_max;
        double *yt = y + t * (int64_t)d_out;
        for (int32_t o = 0; o < d_out; ++o) {
            double acc = 0.0;
            for (int32_t k = 0; k < r; ++k) acc += Bt[(row_off[i] + k) * (int64_t)d_out + o] * h[k];
            yt[o] += scale[i] * acc;
        }
    }
}

/* dh: dH[t, k] = s_i * sum_o B_i[o, k] * dY[t, o] for k < r_i, zero beyond. */
void lora_oracle_dh(int64_t T, int32_t N, int32_t d_out, int32_t r_max,
                    const int32_t *rank, const int64_t *row_off,
                    const double *scale, const int32_t *ids, const double *Bt,
                    const double *dY, double *dH)
{
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t t = 0; t < T; ++t) {
        double *g = dH + t * r_max;
        for (int32_t k = 0; k < r_max; ++k) g[k] = 0.0;
        int32_t i = ids[t];
        if (!valid_id(i, N)) continue;
        const int32_t r = rank[i];
        const double *dy = dY + t * (int64_t)d_out;
        for (int32_t k = 0; k < r; ++k) {
            const double *b = Bt + (row_off[i] + k) * (int64_t)d_out;
            double acc = 0.0;
            for (int32_t o = 0; o < d_out; ++o) acc += b[o] * dy[o];
            g[k] = scale[i] * acc;
        }
    }
}

/* dB: dB_i[o, k] = s_i * sum_{t : ids[t] = i} dY[t, o] * H[t, k].
 * Output uses the Bt_cat layout: dBt[row_off[i]+k, o] = dB_i[o, k]; adapters
 * without tokens get zeros. */
void lora_oracle_db(int64_t T, int32_t N, int32_t d_out, int32_t r_max,
                    const int32_t *rank, const int64_t *row_off,
                    const double *scale, const int32_t *ids, const double *dY,
                    const double *H, double *dBt)
{
    const int64_t sum_r = row_off[N];
    #pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)sum_r * sizeof(double));
        #pragma omp for schedule(dynamic, 8)
        for (int32_t o = 0; o < d_out; ++o) {
            for (int64_t q = 0; q < sum_r; ++q) acc[q] = 0.0;
            for (int64_t t = 0; t < T; ++t) {
                int32_t i = ids[t];
                if (!valid_id(i, N)) continue;
                const double g = dY[t * (int64_t)d_out + o];
                const double *h = H + t * r_max;
                for (int32_t k = 0; k < rank[i]; ++k) acc[row_off[i] + k] += g * h[k];
            }
            for (int32_t i = 0; i < N; ++i)
                for (int32_t k = 0; k < rank[i]; ++k)
                    dBt[(row_off[i] + k) * (int64_t)d_out + o] = scale[i] * acc[row_off[i] + k];
        }
        free(acc);
    }
}

/* dA: dA_i[k, j] = sum_{t : ids[t] = i} dH[t, k] * X[t, j]  (A_cat layout). */
void lora_oracle_da(int64_t T, int32_t N, int32_t d_in, int32_t r_max,
                    const int32_t *rank, const int64_t *row_off,
                    const int32_t *ids, const double *dH, const double *X,
                    double *dA)
{
    const int64_t sum_r = row_off[N];
    #pragma omp parallel
    {
        double *acc = (double *)malloc((size_t)sum_r * sizeof(double));
        #pragma omp for schedule(dynamic, 8)
        for (int32_t j = 0; j < d_in; ++j) {
            for (int64_t q = 0; q < sum_r; ++q) acc[q] = 0.0;
            for (int64_t t = 0; t < T; ++t) {
                int32_t i = ids[t];
                if (!valid_id(i, N)) continue;
                const double xv = X[t * (int64_t)d_in + j];
                const double *g = dH + t * r_max;
                for (int32_t k = 0; k < rank[i]; ++k) acc[row_off[i] + k] += g[k] * xv;
            }
            for (int64_t q = 0; q < sum_r; ++q) dA[q * (int64_t)d_in + j] = acc[q];
        }
        free(acc);
    }
}

/* dX: dX[t, j] += sum_k A_i[k, j] * dH[t, k]. */
void lora_oracle_dx(int64_t T, int32_t N, int32_t d_in, int32_t r_max,
                    const int32_t *rank, const int64_t *row_off,
                    const int32_t *ids, const double *A, const double *dH,
                    double *dX)
{
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t t = 0; t < T; ++t) {
        int32_t i = ids[t];
        if (!valid_id(i, N)) continue;
        const double *g = dH + t * r_max;
        double *dx = dX + t * (int64_t)d_in;
        for (int32_t j = 0; j < d_in; ++j) {
            double acc = 0.0;
            for (int32_t k = 0; k < rank[i]; ++k)
                acc += A[(row_off[i] + k) * (int64_t)d_in + j] * g[k];
            dx[j] += acc;
        }
    }
}

/* AdamW: one step over a weight matrix laid out like A_cat / Bt_cat
 * ([sum_r, d] rows, adapter i = rows row_off[i] .. row_off[i]+rank[i]-1),
 * adapter i with learning rate lr[i] and step number t = step[i] >= 1.
 * w, m, v are updated in place; g is the gradient. */
void lora_oracle_adamw(int32_t N, int32_t d, const int32_t *rank, const int64_t *row_off,
                       const double *lr, const int32_t *step, double beta1, double beta2,
                       double eps, double weight_decay, double *w, const double *g,
                       double *m, double *v)
{
    for (int32_t i = 0; i < N; ++i) {
        const double bc1 = 1.0 - pow(beta1, (double)step[i]);
        const double bc2 = 1.0 - pow(beta2, (double)step[i]);
        const int64_t e0 = row_off[i] * (int64_t)d, e1 = (row_off[i] + rank[i]) * (int64_t)d;
        #pragma omp parallel for schedule(static)
        for (int64_t e = e0; e < e1; ++e) {
            w[e] -= lr[i] * weight_decay * w[e];
            m[e] = beta1 * m[e] + (1.0 - beta1) * g[e];
            v[e] = beta2 * v[e] + (1.0 - beta2) * g[e] * g[e];
            w[e] -= lr[i] * (m[e] / bc1) / (sqrt(v[e] / bc2) + eps);
        }
    }
}

/* base: y[t, o] = sum_j W[o, j] * x[t, j] for every token (W row-major
 * [d_out, d_in]), overwriting y. */
void lora_oracle_base(int64_t T, int32_t d_in, int32_t d_out, const double *W,
                      const double *x, double *y)
{
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t t = 0; t < T; ++t) {
        const double *xt = x + t * (int64_t)d_in;
        double *yt = y + t * (int64_t)d_out;
        for (int32_t o = 0; o < d_out; ++o) {
            const double *w = W + (int64_t)o * d_in;
            double acc = 0.0;
            for (int32_t j = 0; j < d_in; ++j) acc += w[j] * xt[j];
            yt[o] = acc;
        }
    }
}
