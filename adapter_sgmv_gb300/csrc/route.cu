// route.cu -- segment-metadata builder: group a mixed-adapter batch by adapter.
//
// A decode or training batch mixes tokens of many adapters (C-LoRA report,
// "Come funziona l'architettura"); the packed kernels want every adapter's
// tokens together so that one tile reads one adapter's weights (PLoRA
// technical summary, "2. LoRA Execution Engine").  This file builds, on the
// device and without a host round trip:
//   perm       the stable grouping of token indices by adapter id,
//   seg_start  each adapter's start in perm,
//   tiles      work tiles of at most LORA_TILE_M rows that never straddle adapters.
//
// Unsorted ids: a stable counting sort in warp-sized chunks.  Chunk c holds
// tokens 32c .. 32c+31; hist[i][c] counts the tokens of adapter i in chunk c.
// An exclusive scan of hist in adapter-major order gives, for every (i, c),
// the first perm slot of adapter i's tokens of chunk c, and a token's rank
// inside its chunk is the number of lower lanes with the same id
// (__match_any_sync).  All of it is integer work and is bit-exact.
#define LORA_DBG_FILE 1
#include "common.cuh"
#include "internal.h"

namespace lora {

constexpr int kScanThreads = 1024;
constexpr int kScanPerThread = 4;
constexpr int kScanBlock = kScanThreads * kScanPerThread;

// Block-wide exclusive scan of one value per thread (blockDim.x == 1024).
// Returns the exclusive prefix; *block_total receives the block's sum.
__device__ int32_t block_exclusive_scan(int32_t v, int32_t *block_total)
{
    __shared__ int32_t warp_sums[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int32_t y = __shfl_up_sync(0xffffffffu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int32_t w = warp_sums[lane];
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int32_t y = __shfl_up_sync(0xffffffffu, w, d);
            if (lane >= d) w += y;
        }
        warp_sums[lane] = w;  // inclusive
    }
    __syncthreads();
    int32_t excl = x - v + (warp > 0 ? warp_sums[warp - 1] : 0);
    int32_t total = warp_sums[31];
    __syncthreads();  // warp_sums may be reused by the caller's next scan
    *block_total = total;
    return excl;
}

// ---------------------------------------------------------------- unsorted ids
__global__ void route_hist_kernel(const int32_t *__restrict__ ids, int32_t T, int32_t N,
                                  int32_t n_chunks, int32_t *__restrict__ hist,
                                  int32_t *__restrict__ status)
{
    const int32_t chunk = (int32_t)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (chunk >= n_chunks) return;  // whole warps exit together
    const int64_t t = (int64_t)chunk * 32 + lane;
    int32_t id = -1;
    if (t < T) {
        id = ids[t];
        if (id < 0 || id >= N) {
            set_status(status, LORA_ERR_BAD_ADAPTER_ID);
            id = -1;
        }
    }
    const uint32_t same = __match_any_sync(0xffffffffu, id);
    if (id >= 0 && lane == __ffs(same) - 1) hist[(int64_t)id * n_chunks + chunk] = __popc(same);
}

__global__ void route_scatter_kernel(const int32_t *__restrict__ ids, int32_t T, int32_t N,
                                     int32_t n_chunks, const int32_t *__restrict__ offs,
                                     int32_t *__restrict__ perm, int32_t *__restrict__ status)
{
    const int32_t chunk = (int32_t)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (chunk >= n_chunks) return;
    const int64_t t = (int64_t)chunk * 32 + lane;
    int32_t id = -1;
    if (t < T) {
        id = ids[t];
        if (id < 0 || id >= N) id = -1;
    }
    const uint32_t same = __match_any_sync(0xffffffffu, id);
    if (id >= 0) {
        const int32_t rank = __popc(same & ((1u << lane) - 1u));
        perm[LORA_DBG_INDEX((int64_t)offs[(int64_t)id * n_chunks + chunk] + rank, T, status)] = (int32_t)t;
    }
}

// exclusive scan of data[0..M) in place: reduce / top / apply
__global__ void scan_reduce_kernel(const int32_t *__restrict__ data, int64_t M,
                                   int32_t *__restrict__ block_sums)
{
    const int64_t base = (int64_t)blockIdx.x * kScanBlock + (int64_t)threadIdx.x * kScanPerThread;
    int32_t s = 0;
#pragma unroll
    for (int q = 0; q < kScanPerThread; ++q)
        if (base + q < M) s += data[base + q];
    int32_t total;
    block_exclusive_scan(s, &total);
    if (threadIdx.x == 0) block_sums[blockIdx.x] = total;
}

__global__ void scan_top_kernel(int32_t *__restrict__ block_sums, int32_t nb,
                                int32_t *__restrict__ total_out)
{
    int32_t carry = 0;
    for (int32_t b0 = 0; b0 < nb; b0 += kScanThreads) {
        const int32_t b = b0 + threadIdx.x;
        const int32_t v = b < nb ? block_sums[b] : 0;
        int32_t tot;
        const int32_t e = block_exclusive_scan(v, &tot);
        if (b < nb) block_sums[b] = carry + e;
        carry += tot;
    }
    if (threadIdx.x == 0) *total_out = carry;
}

__global__ void scan_apply_kernel(int32_t *__restrict__ data, int64_t M,
                                  const int32_t *__restrict__ block_sums)
{
    const int64_t base = (int64_t)blockIdx.x * kScanBlock + (int64_t)threadIdx.x * kScanPerThread;
    int32_t v[kScanPerThread];
    int32_t s = 0;
#pragma unroll
    for (int q = 0; q < kScanPerThread; ++q) {
        v[q] = base + q < M ? data[base + q] : 0;
        s += v[q];
    }
    int32_t total;
    int32_t e = block_exclusive_scan(s, &total) + block_sums[blockIdx.x];
#pragma unroll
    for (int q = 0; q < kScanPerThread; ++q) {
        if (base + q < M) data[base + q] = e;
        e += v[q];
    }
}

// ---------------------------------------------------------------- sorted input
__global__ void route_sorted_kernel(const int32_t *__restrict__ seg_offsets, int32_t T, int32_t N,
                                    int32_t *__restrict__ perm, int32_t *__restrict__ seg_start,
                                    int32_t *__restrict__ status)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < T; t += stride)
        perm[t] = (int32_t)t;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i <= N; i += stride) {
        const int32_t v = seg_offsets[i];
        seg_start[i] = v;
        bool bad = (i == 0 && v != 0) || (i == N && v != T) || v < 0 || v > T;
        if (i < N && seg_offsets[i + 1] < v) bad = true;
        if (bad) set_status(status, LORA_ERR_BAD_SEGMENTS);
    }
}

// ---------------------------------------------------------------- tiles and spans
// Cut every adapter's group into pieces of at most `len` tokens; one record
// {adapter, begin, rows, flags} per piece, flags bit 0 = consecutive tokens.
// Phase 1 scans the per-adapter piece counts into base[0..N] (scratch);
// phase 2 lets every thread emit pieces, finding the owning adapter of piece
// q by binary search (base[i] <= q < base[i+1]; empty adapters never match).
__device__ void emit_pieces(const int32_t *__restrict__ seg_start, int32_t N, const int32_t *__restrict__ perm,
                            int32_t len, int32_t *__restrict__ out, int32_t *__restrict__ n_out, int32_t max_out,
                            int32_t *__restrict__ base, int32_t T, int32_t *__restrict__ status)
{
    int32_t carry = 0;
    for (int32_t i0 = 0; i0 < N; i0 += blockDim.x) {
        const int32_t i = i0 + threadIdx.x;
        const int32_t n = i < N ? seg_start[i + 1] - seg_start[i] : 0;
        const int32_t cnt = n > 0 ? (n + len - 1) / len : 0;
        int32_t tot;
        const int32_t e = block_exclusive_scan(cnt, &tot);
        if (i < N) base[i] = carry + e;
        carry += tot;
    }
    if (threadIdx.x == 0) base[N] = carry;
    __syncthreads();
    const int32_t total = min(carry, max_out);
    for (int32_t q = threadIdx.x; q < total; q += blockDim.x) {
        int32_t lo = 0, hi = N;
        while (hi - lo > 1) {
            const int32_t mid = (lo + hi) >> 1;
            if (base[mid] <= q) lo = mid;
            else hi = mid;
        }
        const int32_t j = q - base[lo];
        const int32_t n = seg_start[lo + 1] - seg_start[lo];
        const int32_t b = seg_start[lo] + j * len;
        const int32_t rows = min(len, n - j * len);
        const int32_t contiguous =
            (perm[LORA_DBG_INDEX((int64_t)b + rows - 1, T, status)] - perm[LORA_DBG_INDEX(b, T, status)] == rows - 1)
                ? 1
                : 0;
        reinterpret_cast<int4 *>(out)[q] = make_int4(lo, b, rows, contiguous);
    }
    if (threadIdx.x == 0) *n_out = total;
    __syncthreads();  // base is reused by the next call
}

// One block: seg_start (from the scan, when unsorted), then the tile and span
// lists.  Inconsistent segments yield no work.
__global__ void route_tiles_kernel(const int32_t *__restrict__ offs, int32_t n_chunks,
                                   const int32_t *__restrict__ total, int32_t *__restrict__ seg_start,
                                   int32_t N, const int32_t *__restrict__ perm, lora_segments s)
{
    if (offs != nullptr) {  // unsorted: seg_start[i] = offs[i][0], seg_start[N] = total
        for (int32_t i = threadIdx.x; i <= N; i += blockDim.x)
            seg_start[i] = i < N ? offs[(int64_t)i * n_chunks] : *total;
        __syncthreads();
    }
    if (*s.status == LORA_ERR_BAD_SEGMENTS) {
        for (int32_t i = threadIdx.x; i <= N; i += blockDim.x) seg_start[i] = 0;
        if (threadIdx.x == 0) {
            *s.n_tiles = 0;
            *s.n_spans = 0;
        }
        return;
    }
    int32_t *base = s.scratch + (s.scratch_words - (((int64_t)N + 1 + 63) & ~int64_t(63)));
    emit_pieces(seg_start, N, perm, LORA_TILE_M, s.tiles, s.n_tiles, s.max_tiles, base, s.n_tokens, s.status);
    emit_pieces(seg_start, N, perm, LORA_SPAN_TOKENS, s.spans, s.n_spans, s.max_spans, base, s.n_tokens, s.status);
}

// ---------------------------------------------------------------- unsorted ids, one launch
// When the ids, their permutation and a table of N x 32 counts fit in shared
// memory, one block of 1024 threads does the whole build in one launch
// instead of six.  Warp w takes a contiguous run of warp-sized chunks (so the
// warps cover the batch in token order); pass 1 counts each adapter's tokens
// per warp, one exclusive scan of the counts (adapter-major, then warp) gives
// every (adapter, warp) its first slot, and pass 2 walks the same chunks again
// placing each token at its slot plus its rank among the chunk's lanes of the
// same adapter.  That is the same stable order as the six-launch build, so
// the same perm bit for bit.  The permutation is built in shared memory, cut
// into tiles and spans there, then copied out.
constexpr int64_t kSmallSmemWords = (200 * 1024) / 4;

__device__ void emit_pieces_local(const int32_t *seg, int32_t N, const int32_t *perm, int32_t len,
                                  int32_t *__restrict__ out, int32_t *__restrict__ n_out, int32_t max_out,
                                  int32_t *base, int32_t T, int32_t *__restrict__ status)
{
    int32_t carry = 0;
    for (int32_t i0 = 0; i0 < N; i0 += blockDim.x) {
        const int32_t i = i0 + threadIdx.x;
        const int32_t n = i < N ? seg[i + 1] - seg[i] : 0;
        const int32_t cnt = n > 0 ? (n + len - 1) / len : 0;
        int32_t tot;
        const int32_t e = block_exclusive_scan(cnt, &tot);
        if (i < N) base[i] = carry + e;
        carry += tot;
    }
    if (threadIdx.x == 0) base[N] = carry;
    __syncthreads();
    const int32_t total = min(carry, max_out);
    for (int32_t q = threadIdx.x; q < total; q += blockDim.x) {
        int32_t lo = 0, hi = N;
        while (hi - lo > 1) {
            const int32_t mid = (lo + hi) >> 1;
            if (base[mid] <= q) lo = mid;
            else hi = mid;
        }
        const int32_t j = q - base[lo];
        const int32_t n = seg[lo + 1] - seg[lo];
        const int32_t b = seg[lo] + j * len;
        const int32_t rows = min(len, n - j * len);
        const int32_t contiguous =
            (perm[LORA_DBG_INDEX((int64_t)b + rows - 1, T, status)] - perm[LORA_DBG_INDEX(b, T, status)] == rows - 1)
                ? 1
                : 0;
        reinterpret_cast<int4 *>(out)[q] = make_int4(lo, b, rows, contiguous);
    }
    if (threadIdx.x == 0) *n_out = total;
    __syncthreads();  // base is reused by the next call
}

int64_t small_build_words(int32_t T, int32_t N) { return 2 * (int64_t)T + 32 * (int64_t)N + 2 * ((int64_t)N + 1); }

__global__ void __launch_bounds__(1024) route_small_kernel(const int32_t *__restrict__ ids_g, int32_t T, int32_t N,
                                                           int32_t n_chunks, lora_segments s)
{
    // ids [T], perm [T], counts [N][32] (then each (adapter, warp)'s next slot), seg [N+1], base [N+1]
    extern __shared__ int32_t sm[];
    int32_t *ids = sm;
    int32_t *perm = ids + T;
    int32_t *cnt = perm + T;
    int32_t *seg = cnt + 32 * (int64_t)N;
    int32_t *base = seg + N + 1;
    if ((reinterpret_cast<uintptr_t>(ids_g) & 15u) == 0) {  // 16-byte loads, the ragged end one by one
        const int32_t T4 = T / 4;
#pragma unroll 4
        for (int32_t i = threadIdx.x; i < T4; i += blockDim.x)
            reinterpret_cast<int4 *>(ids)[i] = __ldg(reinterpret_cast<const int4 *>(ids_g) + i);
        for (int32_t i = 4 * T4 + threadIdx.x; i < T; i += blockDim.x) ids[i] = ids_g[i];
    } else {
#pragma unroll 8
        for (int32_t i = threadIdx.x; i < T; i += blockDim.x) ids[i] = ids_g[i];
    }
    for (int32_t i = threadIdx.x; i < 32 * N; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t per = (n_chunks + 31) / 32;
    const int32_t c_lo = warp * per, c_hi = min(n_chunks, c_lo + per);
    // the id of lane `lane` in chunk c (-1 past T or for an id out of range, which is reported)
    auto chunk_id = [&](int32_t c, bool report) {
        const int32_t t = c * 32 + lane;
        int32_t id = -1;
        if (c < c_hi && t < T) {
            id = ids[t];
            if (id < 0 || id >= N) {
                if (report) set_status(s.status, LORA_ERR_BAD_ADAPTER_ID);
                id = -1;
            }
        }
        return id;
    };
    // two chunks per step: both match operations are in flight before either
    // chunk's leaders add their counts (in chunk order, one after the other)
    for (int32_t c = c_lo; c < c_hi; c += 2) {  // warp-uniform
        const int32_t id0 = chunk_id(c, true), id1 = chunk_id(c + 1, true);
        const uint32_t same0 = __match_any_sync(0xffffffffu, id0), same1 = __match_any_sync(0xffffffffu, id1);
        if (id0 >= 0 && lane == __ffs(same0) - 1) cnt[id0 * 32 + warp] += __popc(same0);  // only this warp's column
        __syncwarp();
        if (id1 >= 0 && lane == __ffs(same1) - 1) cnt[id1 * 32 + warp] += __popc(same1);
        __syncwarp();
    }
    __syncthreads();
    int32_t carry = 0;  // exclusive scan in place, a 1024-wide row at a time
    for (int32_t r0 = 0; r0 < 32 * N; r0 += blockDim.x) {
        const int32_t i = r0 + threadIdx.x;
        const int32_t v = i < 32 * N ? cnt[i] : 0;
        int32_t tot;
        const int32_t e = block_exclusive_scan(v, &tot);
        if (i < 32 * N) cnt[i] = carry + e;
        carry += tot;
    }
    for (int32_t i = threadIdx.x; i <= N; i += blockDim.x) seg[i] = i < N ? cnt[i * 32] : carry;
    __syncthreads();
    for (int32_t c = c_lo; c < c_hi; c += 2) {
        const int32_t id0 = chunk_id(c, false), id1 = chunk_id(c + 1, false);
        const uint32_t same0 = __match_any_sync(0xffffffffu, id0), same1 = __match_any_sync(0xffffffffu, id1);
#pragma unroll
        for (int k = 0; k < 2; ++k) {  // chunk c, then c + 1
            const int32_t id = k ? id1 : id0;
            const uint32_t same = k ? same1 : same0;
            const int32_t slot = id >= 0 ? cnt[id * 32 + warp] : 0;
            __syncwarp();  // every lane has read its adapter's slot before the group's leader moves it on
            if (id >= 0) {
                perm[LORA_DBG_INDEX((int64_t)slot + __popc(same & ((1u << lane) - 1u)), T, s.status)] =
                    (c + k) * 32 + lane;
                if (lane == __ffs(same) - 1) cnt[id * 32 + warp] = slot + __popc(same);
            }
            __syncwarp();
        }
    }
    __syncthreads();
    const int32_t n_valid = seg[N];
    if ((T & 3) == 0 && (reinterpret_cast<uintptr_t>(s.perm) & 15u) == 0) {  // the shared perm is 16-byte aligned too
        const int32_t n4 = n_valid / 4;
        for (int32_t i = threadIdx.x; i < n4; i += blockDim.x)
            reinterpret_cast<int4 *>(s.perm)[i] = reinterpret_cast<const int4 *>(perm)[i];
        for (int32_t i = 4 * n4 + threadIdx.x; i < n_valid; i += blockDim.x) s.perm[i] = perm[i];
    } else {
        for (int32_t i = threadIdx.x; i < n_valid; i += blockDim.x) s.perm[i] = perm[i];
    }
    for (int32_t i = threadIdx.x; i <= N; i += blockDim.x) s.seg_start[i] = seg[i];
    emit_pieces_local(seg, N, perm, LORA_TILE_M, s.tiles, s.n_tiles, s.max_tiles, base, T, s.status);
    emit_pieces_local(seg, N, perm, LORA_SPAN_TOKENS, s.spans, s.n_spans, s.max_spans, base, T, s.status);
}

// ---------------------------------------------------------------- sorted input, one launch
// For tokens already grouped by adapter the permutation is the identity and
// every piece is a run of consecutive tokens, so the whole builder is one
// launch: block 0 (1024 threads) resets the status word, checks the offsets,
// and cuts the tiles and spans with the per-adapter piece bases kept in shared
// memory; the other blocks write perm[t] = t.  Used when N + 1 offsets fit the
// shared-memory table (kSortedSmemAdapters).
constexpr int32_t kSortedSmemAdapters = 4095;  // two tables of N + 1 ints: 32 KB of static shared memory

__device__ void emit_sorted_pieces(const int32_t *off, int32_t N, int32_t len, int32_t *out, int32_t *n_out,
                                   int32_t max_out, int32_t *base)
{
    int32_t carry = 0;
    for (int32_t i0 = 0; i0 < N; i0 += blockDim.x) {
        const int32_t i = i0 + threadIdx.x;
        const int32_t n = i < N ? off[i + 1] - off[i] : 0;
        const int32_t cnt = n > 0 ? (n + len - 1) / len : 0;
        int32_t tot;
        const int32_t e = block_exclusive_scan(cnt, &tot);
        if (i < N) base[i] = carry + e;
        carry += tot;
    }
    if (threadIdx.x == 0) base[N] = carry;
    __syncthreads();
    const int32_t total = min(carry, max_out);
    for (int32_t q = threadIdx.x; q < total; q += blockDim.x) {
        int32_t lo = 0, hi = N;
        while (hi - lo > 1) {
            const int32_t mid = (lo + hi) >> 1;
            if (base[mid] <= q) lo = mid;
            else hi = mid;
        }
        const int32_t j = q - base[lo];
        const int32_t b = off[lo] + j * len;
        const int32_t rows = min(len, off[lo + 1] - off[lo] - j * len);
        reinterpret_cast<int4 *>(out)[q] = make_int4(lo, b, rows, 1);
    }
    if (threadIdx.x == 0) *n_out = total;
    __syncthreads();  // base is reused by the next call
}

__global__ void __launch_bounds__(1024) route_sorted_one_kernel(const int32_t *__restrict__ seg_offsets, int32_t T,
                                                                int32_t N, lora_segments s)
{
    if (blockIdx.x > 0) {
        const int64_t stride = (int64_t)(gridDim.x - 1) * blockDim.x;
        for (int64_t t = (blockIdx.x - 1) * (int64_t)blockDim.x + threadIdx.x; t < T; t += stride)
            s.perm[t] = (int32_t)t;
        return;
    }
    __shared__ int32_t off[kSortedSmemAdapters + 1];
    __shared__ int32_t base[kSortedSmemAdapters + 1];
    __shared__ int bad;
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    for (int32_t i = threadIdx.x; i <= N; i += blockDim.x) {
        const int32_t v = seg_offsets[i];
        off[i] = v;
        if ((i == 0 && v != 0) || (i == N && v != T) || v < 0 || v > T) bad = 1;
    }
    __syncthreads();
    for (int32_t i = threadIdx.x; i < N; i += blockDim.x)
        if (off[i + 1] < off[i]) bad = 1;
    __syncthreads();
    if (bad) {  // inconsistent segments: no work, the status says why
        for (int32_t i = threadIdx.x; i <= N; i += blockDim.x) s.seg_start[i] = 0;
        if (threadIdx.x == 0) {
            s.status[0] = LORA_ERR_BAD_SEGMENTS;
            s.status[1] = 0;
            *s.n_tiles = 0;
            *s.n_spans = 0;
        }
        return;
    }
    if (threadIdx.x == 0) {
        s.status[0] = LORA_OK;
        s.status[1] = 0;  // the debug build's check site
    }
    for (int32_t i = threadIdx.x; i <= N; i += blockDim.x) s.seg_start[i] = off[i];
    emit_sorted_pieces(off, N, LORA_TILE_M, s.tiles, s.n_tiles, s.max_tiles, base);
    emit_sorted_pieces(off, N, LORA_SPAN_TOKENS, s.spans, s.n_spans, s.max_spans, base);
}

// ---------------------------------------------------------------- host side
SegLayout seg_layout(int32_t T, int32_t N)
{
    SegLayout L{};
    if (T < 0 || N < 1 || N > kMaxAdapters || T > kMaxTokens) return L;
    auto up = [](int64_t words) { return (words + 63) & ~int64_t(63); };  // 256-byte regions
    L.n_chunks = (T + 31) / 32;
    L.max_tiles = T / LORA_TILE_M + N + 1;
    L.max_spans = T / LORA_SPAN_TOKENS + N + 1;
    L.hist_words = (int64_t)N * L.n_chunks;
    if (L.hist_words > kMaxHistWords) return L;
    L.block_sums = (int32_t)((L.hist_words + kScanBlock - 1) / kScanBlock);
    int64_t o = 0;
    L.off_perm = o;       o += up(T > 0 ? T : 1);
    L.off_seg = o;        o += up(N + 1);
    L.off_tiles = o;      o += up(4 * (int64_t)L.max_tiles);
    L.off_ntiles = o;     o += up(1);
    L.off_status = o;     o += up(1);
    L.off_spans = o;      o += up(4 * (int64_t)L.max_spans);
    L.off_nspans = o;     o += up(1);
    L.off_scratch = o;
    L.scratch_words = up(L.hist_words) + up(L.block_sums) + up(1) + up((int64_t)N + 1);  // + piece bases
    o += L.scratch_words;
    L.total_words = o;
    L.ok = true;
    return L;
}

lora_status_t build_segments(const int32_t *ids, const int32_t *seg_offsets, int32_t T, int32_t N,
                             void *storage, size_t storage_bytes, lora_segments *out,
                             cudaStream_t stream)
{
    const SegLayout L = seg_layout(T, N);
    if (!L.ok) return LORA_ERR_SHAPE;
    if ((size_t)L.total_words * 4 > storage_bytes) return LORA_ERR_WORKSPACE_TOO_SMALL;
    int32_t *w = static_cast<int32_t *>(storage);
    lora_segments s{};
    s.n_tokens = T;
    s.n_adapters = N;
    s.max_tiles = L.max_tiles;
    s.sorted = seg_offsets != nullptr ? 1 : 0;
    s.perm = w + L.off_perm;
    s.seg_start = w + L.off_seg;
    s.tiles = w + L.off_tiles;
    s.n_tiles = w + L.off_ntiles;
    s.status = w + L.off_status;
    s.scratch = w + L.off_scratch;
    s.scratch_words = L.scratch_words;
    s.max_spans = L.max_spans;
    s.spans = w + L.off_spans;
    s.n_spans = w + L.off_nspans;

    if (seg_offsets != nullptr && N <= kSortedSmemAdapters) {
        const int64_t perm_blocks = ((int64_t)T + 1023) / 1024;
        const int blocks = 1 + (int)(perm_blocks < 296 ? perm_blocks : 296);
        route_sorted_one_kernel<<<blocks, 1024, 0, stream>>>(seg_offsets, T, N, s);
        if (cudaGetLastError() != cudaSuccess) return LORA_ERR_CUDA;
        *out = s;
        return LORA_OK;
    }
    if (cudaMemsetAsync(s.status, 0, 8, stream) != cudaSuccess) return LORA_ERR_CUDA;
    if (seg_offsets != nullptr) {
        const int threads = 256;
        const int64_t work = (int64_t)(T > N + 1 ? T : N + 1);
        const int blocks = (int)((work + threads - 1) / threads < 1184 ? (work + threads - 1) / threads : 1184);
        route_sorted_kernel<<<blocks > 0 ? blocks : 1, threads, 0, stream>>>(seg_offsets, T, N, s.perm,
                                                                              s.seg_start, s.status);
        route_tiles_kernel<<<1, 1024, 0, stream>>>(nullptr, 0, nullptr, s.seg_start, N, s.perm, s);
    } else {
        int32_t *hist = s.scratch;
        int32_t *bsum = hist + ((L.hist_words + 63) & ~int64_t(63));
        int32_t *total = bsum + ((L.block_sums + 63) & ~int64_t(63));
        // one launch when the ids, their permutation and N x 32 counts fit in
        // shared memory
        const int64_t small_words = small_build_words(T, N);
        if (L.hist_words > 0 && small_words <= kSmallSmemWords) {
            const int smem = (int)(small_words * 4);
            if (cudaFuncSetAttribute(route_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
                cudaSuccess)
                return LORA_ERR_CUDA;
            route_small_kernel<<<1, 1024, smem, stream>>>(ids, T, N, L.n_chunks, s);
        } else if (L.hist_words > 0) {
            if (cudaMemsetAsync(hist, 0, (size_t)L.hist_words * 4, stream) != cudaSuccess) return LORA_ERR_CUDA;
            const int threads = 256;
            const int blocks = (int)(((int64_t)L.n_chunks * 32 + threads - 1) / threads);
            route_hist_kernel<<<blocks, threads, 0, stream>>>(ids, T, N, L.n_chunks, hist, s.status);
            scan_reduce_kernel<<<L.block_sums, kScanThreads, 0, stream>>>(hist, L.hist_words, bsum);
            scan_top_kernel<<<1, kScanThreads, 0, stream>>>(bsum, L.block_sums, total);
            scan_apply_kernel<<<L.block_sums, kScanThreads, 0, stream>>>(hist, L.hist_words, bsum);
            route_scatter_kernel<<<blocks, threads, 0, stream>>>(ids, T, N, L.n_chunks, hist, s.perm, s.status);
            route_tiles_kernel<<<1, 1024, 0, stream>>>(hist, L.n_chunks, total, s.seg_start, N, s.perm, s);
        } else {  // empty batch: every group empty, no tiles
            if (cudaMemsetAsync(s.seg_start, 0, (size_t)(N + 1) * 4, stream) != cudaSuccess ||
                cudaMemsetAsync(s.n_tiles, 0, 4, stream) != cudaSuccess ||
                cudaMemsetAsync(s.n_spans, 0, 4, stream) != cudaSuccess)
                return LORA_ERR_CUDA;
        }
    }
    if (cudaGetLastError() != cudaSuccess) return LORA_ERR_CUDA;
    *out = s;
    return LORA_OK;
}

}  // namespace lora
