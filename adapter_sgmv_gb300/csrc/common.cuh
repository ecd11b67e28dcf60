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

// ---------------------------------------------------------------- work tiles
struct Tile {
    int32_t adapter, begin, rows, flags;
};

LORA_DEV Tile load_tile(const int32_t *tiles, int32_t idx)
{
    int4 v = reinterpret_cast<const int4 *>(tiles)[idx];
    return Tile{v.x, v.y, v.z, v.w};
}

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
