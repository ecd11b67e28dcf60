// tc_common.cuh -- inline-PTX building blocks of the sm_103a tensor-core kernels:
// mbarriers with bounded waits, TMA tile loads, cp.async, the tcgen05 MMA with
// its shared-memory matrix descriptors, and tensor-memory (TMEM) management.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"
#include "tc_host.h"

namespace lora {
namespace tc {

// ---------------------------------------------------------------- addresses
LORA_DEV uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

LORA_DEV uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier
LORA_DEV void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

LORA_DEV void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

LORA_DEV void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

LORA_DEV void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

LORA_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, for a bounded time.
// The bound is counted in SM clock cycles (kWaitLimitCycles, about 2-3 s at
// GB300 clocks), read only every 1024 polls so that a wait that completes
// soon costs nothing but the polls.  On time-out the CTA-wide abort flag and
// the status word are set and false is returned; callers then stop issuing
// work and leave.
constexpr uint64_t kWaitLimitNs = 2000000000ull;      // bound of the rare clean-up waits (globaltimer)
constexpr long long kWaitLimitCycles = 4000000000ll;  // bound of pipeline waits (SM clock)

LORA_DEV bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int32_t *abort_flag, int32_t *status)
{
    if (mbar_try_wait(bar, parity)) return true;
    long long t0 = 0;
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 1023u) == 0u) {
            if (*abort_flag) return false;
            const long long now = clock64();
            if (t0 == 0) {
                t0 = now;
            } else if (now - t0 > kWaitLimitCycles) {
                *abort_flag = 1;
                set_status(status, LORA_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Warp-uniform bounded wait: every lane of the warp calls it and every lane
// gets the same answer, so a time-out can never split a warp in front of a
// .sync.aligned instruction (tcgen05.ld / alloc / dealloc), which would wait
// for the missing lanes forever.
LORA_DEV bool mbar_wait_warp(uint64_t *bar, uint32_t parity, volatile int32_t *abort_flag, int32_t *status)
{
    const bool ok = mbar_wait(bar, parity, abort_flag, status);
    return __all_sync(0xffffffffu, ok);
}

// ---------------------------------------------------------------- TMA
LORA_DEV void tma_load_2d(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int32_t c0, int32_t c1)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], "
        "[%2];" ::"r"(smem_u32(smem_dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

LORA_DEV void tma_load_3d(void *smem_dst, const CUtensorMap *map, uint64_t *bar, int32_t c0, int32_t c1, int32_t c2)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], "
        "[%2];" ::"r"(smem_u32(smem_dst)),
        "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

// TMA store of one box from shared memory (its own bulk group); c0 must not
// be negative and c0 * element size must be a multiple of 16 bytes.  Parts of
// the box outside the tensor are not written.
LORA_DEV void tma_store_2d(const CUtensorMap *map, const void *smem_src, int32_t c0, int32_t c1)
{
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(map),
                 "r"(smem_u32(smem_src)), "r"(c0), "r"(c1)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// every bulk group this thread committed has completed (writes performed)
LORA_DEV void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

LORA_DEV void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// rows row0 .. row0 + rp - 1 (rp a multiple of 16), columns col .. col + 63,
// to dst as consecutive 1 KB atoms of eight 128-byte rows
LORA_DEV void tma_load_rows(uint8_t *dst, const WMaps &wm, uint64_t *bar, int32_t col, int32_t row0, int32_t rp)
{
    for (int32_t k0 = 0; k0 < rp;) {
        const int32_t rem = rp - k0;
        const CUtensorMap *m = rem >= 64 ? &wm.m64 : rem >= 32 ? &wm.m32 : &wm.m16;
        tma_load_2d(dst + k0 * 128, m, bar, col, row0 + k0);
        k0 += rem >= 64 ? 64 : rem >= 32 ? 32 : 16;
    }
}

// ---------------------------------------------------------------- cp.async (16 B, zero-fill when !pred)
LORA_DEV void cp_async_16(void *smem_dst, const void *gmem_src, bool pred)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src),
                 "r"(pred ? 16 : 0)
                 : "memory");
}
LORA_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// Arrive on `bar` once every cp.async this thread has issued so far has
// completed.  The arrive does not raise the barrier's pending count: it is one
// of the arrivals the barrier was initialised with, so the thread never waits
// for its own copies.  Consumers that read the stage with ordinary loads see
// the data once the barrier's phase completes.
LORA_DEV void cp_async_mbar_arrive(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
template <int N>
LORA_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// generic-proxy shared-memory writes -> visible to the async proxy (tcgen05.mma, TMA)
LORA_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---------------------------------------------------------------- work claims
// The roles of a persistent CTA (producers, MMA issuer, epilogue) walk the
// same sequence of work items.  Items split ahead of time: CTA b takes b,
// b + gridDim.x, ..., which every role computes by itself.  Items claimed at
// run time: one thread, the claimer, takes each next index from a counter in
// global memory (zero when the launch starts) with atomicAdd and passes it to
// the other roles through a ring of kClaimSlots slots in shared memory.  Items
// then go out in index order to whichever CTA asks first, so items of uneven
// cost spread evenly over the SMs, and every item below a claimed one is held
// by a running CTA.  The last index a CTA passes on is >= n_items, which ends
// every role's walk.
//
// The epilogue hands its slot back only when it comes for the next claim,
// i.e. once it has finished the item: with two slots the claimer takes item
// q + 1 only after the epilogue has finished item q - 1, so a CTA holds at
// most one item beyond the one its epilogue works on (the producer's
// look-ahead) and the last items go to CTAs that are about to be free.
constexpr int kClaimSlots = 2;

struct ClaimRing {
    volatile int32_t *slot;  // [kClaimSlots]
    uint64_t *full;          // [kClaimSlots], count 1: the claimer's arrive
    uint64_t *empty;         // [kClaimSlots], count: one arrive per reader (a thread or a warp)
};

// the claimer's first item, taken before the CTA's set-up so that the
// atomic's round trip overlaps it (0 without a counter: unused)
LORA_DEV int32_t claim_first(int32_t *counter) { return counter != nullptr ? atomicAdd(counter, 1) : 0; }

// claimer (one thread): the CTA's claim number q = 0, 1, ...; false on time-out
LORA_DEV bool claim_next(const ClaimRing &R, uint32_t q, int32_t *counter, int32_t first, int32_t *it,
                         volatile int32_t *abort_flag, int32_t *status)
{
    const uint32_t s = q % kClaimSlots;
    if (!mbar_wait(&R.empty[s], ((q / kClaimSlots) & 1u) ^ 1u, abort_flag, status)) return false;
    *it = q == 0 ? first : atomicAdd(counter, 1);
    R.slot[s] = *it;
    mbar_arrive(&R.full[s]);  // release: the slot is visible to a reader once its wait returns
    return true;
}

// a reading thread: claim q of this CTA, its slot handed back at once; false on time-out
LORA_DEV bool claim_read(const ClaimRing &R, uint32_t q, int32_t *it, volatile int32_t *abort_flag, int32_t *status)
{
    const uint32_t s = q % kClaimSlots;
    if (!mbar_wait(&R.full[s], (q / kClaimSlots) & 1u, abort_flag, status)) return false;
    *it = R.slot[s];
    mbar_arrive(&R.empty[s]);
    return true;
}

// a reading warp (every lane calls it and gets the same answer).  `keep`:
// the slot is handed back later, by claim_release_warp(q), once the warp has
// finished the item (the epilogue)
LORA_DEV bool claim_read_warp(const ClaimRing &R, uint32_t q, int32_t *it, volatile int32_t *abort_flag,
                              int32_t *status, bool keep = false)
{
    const uint32_t s = q % kClaimSlots;
    if (!mbar_wait_warp(&R.full[s], (q / kClaimSlots) & 1u, abort_flag, status)) return false;
    *it = R.slot[s];
    __syncwarp();
    if (!keep && (threadIdx.x & 31) == 0) mbar_arrive(&R.empty[s]);
    return true;
}
LORA_DEV void claim_release_warp(const ClaimRing &R, uint32_t q)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&R.empty[q % kClaimSlots]);
}

// n floats at p (16-byte aligned, n a multiple of 4) set to zero by every
// thread of the grid: a kernel that runs before the one accumulating into
// them, on the same stream, clears them (no separate memset launch).
LORA_DEV void zero_grid(float *p, int64_t n)
{
    if (p == nullptr) return;
    float4 *q = reinterpret_cast<float4 *>(p);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n / 4; i += stride)
        q[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// A kernel that runs before the claiming kernels of the same call, on the
// same stream, zeroes their counters (block 0, before anything else).
LORA_DEV void zero_claims(int32_t *claims, int32_t n)
{
    if (claims != nullptr && blockIdx.x == 0 && (int32_t)threadIdx.x < n) claims[threadIdx.x] = 0;
}

// ---------------------------------------------------------------- tcgen05
// Shared-memory matrix descriptor (tcgen05 "matrix descriptor"):
//   [0,14)  start address >> 4      [16,30) leading-dimension byte offset >> 4
//   [32,46) stride-dimension byte offset >> 4    [46,48) version = 1
//   [49,52) base offset (0: atoms 1024-byte aligned)    [52] LBO mode = 0
//   [61,64) layout: 0 none (interleaved core matrices), 2 128-byte swizzle
enum Layout : uint32_t { kInterleave = 0, kSwizzle128 = 2 };

LORA_DEV uint64_t make_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes, Layout layout)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3ffffu) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3fffu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3fffu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)layout << 61;
    return d;
}

// Instruction descriptor, kind::f16 with bf16 inputs and fp32 accumulation.
//   [4,6) D format (1 = f32)   [7,10) A format (1 = bf16)   [10,13) B format (1 = bf16)
//   [15] A major (0 = K)   [16] B major (0 = K, 1 = MN)   [17,23) N >> 3   [24,29) M >> 4
LORA_DEV uint32_t make_idesc_bf16(uint32_t M, uint32_t N, bool a_mn_major, bool b_mn_major)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
           ((N >> 3) << 17) | ((M >> 4) << 24);
}

LORA_DEV void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// arrive on `bar` once every tcgen05.mma issued so far by this thread has completed
LORA_DEV void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

LORA_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
LORA_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// TMEM allocation (one whole warp); the column base is written to smem
LORA_DEV void tmem_alloc(uint32_t *dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
LORA_DEV void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;"); }
LORA_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 32 lanes x 16 columns of 32-bit words: thread i receives lane (base + i)
LORA_DEV void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
LORA_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- layouts
// K-major, 128-byte swizzle: rows of 64 bf16 (128 B), 8-row atoms of 1024 B.
// Byte offset of the 16-byte chunk c (0..7) of row m.
LORA_DEV uint32_t sw128_offset(uint32_t m, uint32_t c) { return (m >> 3) * 1024u + (m & 7u) * 128u + ((c ^ (m & 7u)) << 4); }

// red.global.add of 4 consecutive floats (16-byte aligned)
LORA_DEV void red_add_v4(float *p, float a, float b, float c, float d)
{
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}
LORA_DEV void red_add_f32(float *p, float a) { asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(a) : "memory"); }

}  // namespace tc
}  // namespace lora
