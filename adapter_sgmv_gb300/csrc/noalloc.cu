// noalloc.cu -- lora_packed_bwd_noalloc: the packed backward for callers that
// cannot allocate device memory.
//
// lora_packed_bwd takes its scratch (the bf16 hand-off copies of H and dH,
// T x 64 or T x 128 each, and for batches of few tiles fp32 partial sums) from
// a caller-provided workspace.  Some callers have no way to get
// one: code that runs where cudaMalloc is not allowed or not wanted (inside a
// custom allocator's own callbacks, in a plugin that must not touch the host
// framework's memory pool, in a process whose device memory is fully reserved
// by another runtime).  This entry point keeps that scratch in a fixed array
// in the library's own device memory instead, so it needs no workspace
// argument and allocates nothing.
//
// Costs and rules:
//  - The array is a file-scope __device__ variable of kScratchBytes (8 MiB);
//    every GPU that loads the library holds it until the process exits.
//  - The scratch is laid out as lora_packed_bwd lays out its workspace, so the
//    two compute the same bits.  Problems whose backward scratch exceeds the
//    array (2 * T * rw * 2 bytes, rw = 64 when r_max <= 64 else 128, each half
//    rounded up to 256 bytes, plus counters and partial sums) are rejected
//    with LORA_ERR_WORKSPACE_TOO_SMALL before anything is launched.
//  - All calls share the one array and the last call's contents stay in it.
//    Nothing in it has to start at zero: every scratch value a product uses
//    is written earlier in the same call (hand-off columns past a tile's rank
//    rounded up to 16 may reach shared memory with the rest of a row, but no
//    product reads them).  Calls whose work overlaps on the GPU
//    (different streams, or different host threads, same device) race on the
//    array: serialise them.
//  - In host code the array's name stands for a host-side shadow, not a
//    device address.  The first call on each device, with that device
//    current, resolves the device address once with cudaGetSymbolAddress and
//    caches it; make that first call before any stream capture.
#include <mutex>

#include "dispatch.h"
#include "internal.h"

namespace lora {
namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// device address of g_bwd_scratch on the current device (nullptr on failure)
void *scratch_address()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess) return nullptr;
        g_addr[dev] = p;
    }
    return g_addr[dev];
}

}  // namespace
}  // namespace lora

using namespace lora;

extern "C" LORA_API lora_status_t lora_packed_bwd_noalloc(void *dX, float *dA, float *dB, const void *dY,
                                                          const void *X, const float *H_saved,
                                                          const lora_adapter_table *table,
                                                          const lora_segments *segs, lora_stream_t stream)
{
    // the checks lora_packed_bwd makes, in the same order, so that a caller
    // error gives the same status here and never reaches the device
    lora_status_t st = check_table(table);
    if (st == LORA_OK) st = check_segs(segs, table);
    if (st != LORA_OK) return st;
    if (dY == nullptr || X == nullptr) return LORA_ERR_INVALID_ARG;
    if (!aligned16(dY) || !aligned16(X) || (dX && !aligned16(dX)) || (dA && !aligned16(dA)) ||
        (dB && !aligned16(dB)) || (H_saved && !aligned16(H_saved)))
        return LORA_ERR_ALIGNMENT;
    // the backward's scratch, laid out as in lora_packed_bwd's workspace: the two
    // bf16 hand-off copies (of H and dH), then counters and partial sums
    if (bwd_workspace_bytes(*table, segs->n_tokens) > kScratchBytes) return LORA_ERR_WORKSPACE_TOO_SMALL;
    st = check_device();
    if (st != LORA_OK) return st;
    void *base = scratch_address();
    if (base == nullptr) return LORA_ERR_CUDA;
    return run_bwd(dX, dA, dB, dY, X, H_saved, base, kScratchBytes, *table, *segs,
                   reinterpret_cast<cudaStream_t>(stream));
}
