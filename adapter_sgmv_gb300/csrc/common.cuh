// common.cuh -- small device helpers shared by the library's kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "lora_sgmv.h"

#define LORA_DEV __device__ __forceinline__

namespace lora {

// ---------------------------------------------------------------- status word
// First error wins: a kernel that detects a problem records its code once.
LORA_DEV void set_status(int32_t *status, int32_t code)
{
    if (status != nullptr) atomicCAS(status, (int32_t)LORA_OK, code);
}

// ---------------------------------------------------------------- chained launches
// A kernel launched with programmatic stream serialisation may start while
// the kernel before it in the stream is still running.  pdl_wait() returns
// once that kernel has completed and its writes are visible; a dependent
// kernel reads nothing an earlier kernel may have written before it.
// pdl_launch_dependents() lets the next such kernel start; it is issued only
// after this kernel's own pdl_wait() (or by a kernel that is not itself a
// dependent), so a dependent that starts early knows that every kernel before
// its predecessor has completed.
LORA_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
LORA_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- bf16 words
// bf16 is carried as raw 16-bit words; widening is exact, narrowing rounds to
// nearest-even (cvt.rn: NaN stays NaN).
LORA_DEV float bf16_to_f32(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }

// two bf16 packed in a 32-bit word: low half is the lower-addressed element
LORA_DEV float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
LORA_DEV float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
// one instruction for both halves (the epilogues round millions of elements)
LORA_DEV uint32_t pack_bf16(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// ---------------------------------------------------------------- debug index checks
// The library's debug build (compiled with LORA_DEBUG_CHECKS=1) checks every
// index it reads from the routing metadata before that index addresses
// memory: the tile and span lists, their counts, perm, and the slots derived
// from them.  A value out of range sets LORA_ERR_INDEX in the status word,
// records in the word after it where the check sits (LORA_DBG_FILE << 16 |
// source line; first failure wins) and is replaced by an in-range value, so
// the access stays inside its buffer: results are then unspecified, but the
// kernel neither faults nor traps and its pipelines keep their protocol.  In
// the release build every check compiles to its argument.
#ifndef LORA_DEBUG_CHECKS
#define LORA_DEBUG_CHECKS 0
#endif
#ifndef LORA_DBG_FILE
#define LORA_DBG_FILE 0
#endif
#define LORA_DBG_HERE ((int32_t)((LORA_DBG_FILE << 16) | (__LINE__ & 0xffff)))

LORA_DEV void dbg_fail(int32_t *status, int32_t where)
{
    if (status != nullptr && atomicCAS(status, (int32_t)LORA_OK, (int32_t)LORA_ERR_INDEX) == (int32_t)LORA_OK)
        atomicExch(status + 1, where);
}

// v if 0 <= v < n, else (debug build) the failure is recorded and 0 returned
LORA_DEV int64_t dbg_index(int64_t v, int64_t n, int32_t *status, int32_t where)
{
#if LORA_DEBUG_CHECKS
    if (v < 0 || v >= n) {
        dbg_fail(status, where);
        return 0;
    }
#endif
    return v;
}
#define LORA_DBG_INDEX(v, n, status) ::lora::dbg_index((v), (n), (status), LORA_DBG_HERE)

// ---------------------------------------------------------------- work tiles
struct Tile {
    int32_t adapter, begin, rows, flags;
};

// entry idx of a tile list (tiles: rows <= LORA_TILE_M) or span list (rows <=
// LORA_SPAN_TOKENS); the debug build checks the index against the list's
// capacity and the entry against the batch (adapter in [0, N), 1 <= rows <=
// cap, begin >= 0, begin + rows <= T), and replaces a bad entry by the first
// token of adapter 0 gathered alone
LORA_DEV Tile load_piece(const int32_t *list, int32_t idx, int32_t max, int32_t cap, const lora_segments &s,
                         int32_t where)
{
#if LORA_DEBUG_CHECKS
    if (idx < 0 || idx >= max) {
        dbg_fail(s.status, where);
        idx = 0;
    }
#endif
    int4 v = reinterpret_cast<const int4 *>(list)[idx];
    Tile t{v.x, v.y, v.z, v.w};
#if LORA_DEBUG_CHECKS
    if (t.adapter < 0 || t.adapter >= s.n_adapters || t.rows < 1 || t.rows > cap || t.begin < 0 ||
        (int64_t)t.begin + t.rows > (int64_t)s.n_tokens) {
        dbg_fail(s.status, where);
        t = Tile{0, 0, 1, 0};
    }
#else
    (void)max, (void)cap, (void)s, (void)where;
#endif
    return t;
}
#define LOAD_TILE(segs, idx) \
    ::lora::load_piece((segs).tiles, (idx), (segs).max_tiles, LORA_TILE_M, (segs), LORA_DBG_HERE)
#define LOAD_SPAN(segs, idx) \
    ::lora::load_piece((segs).spans, (idx), (segs).max_spans, LORA_SPAN_TOKENS, (segs), LORA_DBG_HERE)

// perm[p], a token index; the debug build checks p and the value against T
LORA_DEV int32_t perm_at(const lora_segments &s, int64_t p, int32_t where)
{
#if LORA_DEBUG_CHECKS
    if (p < 0 || p >= s.n_tokens) {
        dbg_fail(s.status, where);
        p = 0;
    }
    const int32_t t = s.perm[p];
    if (t < 0 || t >= s.n_tokens) {
        dbg_fail(s.status, where);
        return 0;
    }
    return t;
#else
    (void)where;
    return s.perm[p];
#endif
}
#define PERM_AT(segs, p) ::lora::perm_at((segs), (p), LORA_DBG_HERE)

// the number of valid entries of a list, checked against its capacity
LORA_DEV int32_t dbg_count(int32_t n, int32_t max, int32_t *status, int32_t where)
{
#if LORA_DEBUG_CHECKS
    if (n < 0 || n > max) {
        dbg_fail(status, where);
        return n < 0 ? 0 : max;
    }
#else
    (void)max, (void)status, (void)where;
#endif
    return n;
}
#define N_TILES(segs) ::lora::dbg_count(*(segs).n_tiles, (segs).max_tiles, (segs).status, LORA_DBG_HERE)
#define N_SPANS(segs) ::lora::dbg_count(*(segs).n_spans, (segs).max_spans, (segs).status, LORA_DBG_HERE)

// per-adapter table entry, validated against the host-side sizes
struct AdapterInfo {
    int32_t rank;
    int32_t row_off;
    float scale;
    bool ok;
};

LORA_DEV AdapterInfo load_adapter(const lora_adapter_table &tab, int32_t i, int32_t *status)
{
    AdapterInfo a;
    a.rank = __ldg(tab.rank + i);
    a.row_off = __ldg(tab.row_off + i);
    a.scale = __ldg(tab.scale + i);
    a.ok = a.rank >= 1 && a.rank <= tab.r_max && a.row_off >= 0 &&
           (int64_t)a.row_off + a.rank <= (int64_t)tab.sum_r;
    if (!a.ok) set_status(status, LORA_ERR_BAD_TABLE);
    return a;
}

}  // namespace lora
