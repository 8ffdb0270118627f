// nm_common.cuh -- internal helpers shared by the library's kernels.
//
// Inline PTX wrappers for the sm_100-family features the kernels use
// (mbarrier, TMA tensor copies, programmatic dependent launch), bf16 bit
// helpers, and the per-device scratch layout. Written from the public PTX ISA.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "nmspmv.h"

namespace nm {

// ---------------------------------------------------------------------------
// Per-device scratch (allocated once per device by the host side).
// ---------------------------------------------------------------------------

// Stream-K CTAs that one launch may use; bounds the scratch size.
constexpr int kMaxCtas = 1024;
// Partial sums per CTA: 2 slots (first and last row block) x 8 batch x 32 rows.
constexpr int kPartialFloats = 2 * 8 * 32;

// status[0]: NM_ERR_TIMEOUT bit set by a bounded wait that ran out.
// status[1]: nonzero when nm_pack found more than N nonzeros in a subgroup.
struct Scratch {
    uint32_t *status;   // [4]
    uint32_t *counters; // [kMaxCtas], zero between launches
    float *partials;    // [kMaxCtas][kPartialFloats]
};

constexpr size_t kScratchStatusBytes = 256;
constexpr size_t kScratchCounterBytes = sizeof(uint32_t) * kMaxCtas;
constexpr size_t kScratchPartialBytes = sizeof(float) * (size_t)kMaxCtas * kPartialFloats;
constexpr size_t kScratchBytes = kScratchStatusBytes + kScratchCounterBytes + kScratchPartialBytes;

inline Scratch scratch_from_base(void *base)
{
    Scratch s;
    char *p = (char *)base;
    s.status = (uint32_t *)p;
    s.counters = (uint32_t *)(p + kScratchStatusBytes);
    s.partials = (float *)(p + kScratchStatusBytes + kScratchCounterBytes);
    return s;
}

// ---------------------------------------------------------------------------
// Bounds-checking build
// ---------------------------------------------------------------------------

// With -DNM_BOUNDS_CHECK, NM_IN_BOUNDS(status, cond) checks an index that
// depends on data or on the work split against its buffer: when cond fails it
// sets the NM_ERR_BOUNDS bit of the status word and yields false, and the
// caller skips the access. No trap, no assert. In the normal build it is the
// constant true and compiles away.
__device__ __forceinline__ bool bounds_ok(uint32_t *status, bool cond)
{
    if (!cond)
        atomicOr(status, 1u << NM_ERR_BOUNDS);
    return cond;
}
#ifdef NM_BOUNDS_CHECK
#define NM_IN_BOUNDS(status, cond) ::nm::bounds_ok((status), (cond))
#else
#define NM_IN_BOUNDS(status, cond) true
#endif

// ---------------------------------------------------------------------------
// bf16 bits
// ---------------------------------------------------------------------------

__device__ __forceinline__ float bf16lo_to_f32(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t pair) { return __uint_as_float(pair & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// fp32 -> bf16, round to nearest even (NaN stays NaN).
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float f)
{
    uint16_t r;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(f));
    return r;
}

// acc + w * x, where w and x are bf16 values held in the low (H = 0) or high
// (H = 1) half of 32-bit registers. The product of two bf16 values is exact in
// fp32, so this equals fmaf(float(w), float(x), acc) bit for bit; the
// mixed-precision form reads the halves directly, with no conversion.
template <int WH, int XH>
__device__ __forceinline__ float fma_bf16(uint32_t w, uint32_t x, float acc)
{
    asm("{\n\t.reg .b16 w0, w1, x0, x1;\n\t"
        "mov.b32 {w0, w1}, %1;\n\t"
        "mov.b32 {x0, x1}, %2;\n\t"
        "fma.rn.f32.bf16 %0, w%3, x%4, %0;\n\t}"
        : "+f"(acc)
        : "r"(w), "r"(x), "n"(WH), "n"(XH));
    return acc;
}

// ---------------------------------------------------------------------------
// Shared-memory access by 32-bit shared address
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Position of the most significant set bit, or -1 (0xFFFFFFFF) for zero.
__device__ __forceinline__ int bfind_u32(uint32_t m)
{
    int r;
    asm("bfind.u32 %0, %1;" : "=r"(r) : "r"(m));
    return r;
}

// 1 << s with the PTX rule for large shifts: s >= 32 (including -1 read as
// unsigned) gives 0.
__device__ __forceinline__ uint32_t bit_at(int s)
{
    uint32_t r;
    asm("shl.b32 %0, %1, %2;" : "=r"(r) : "r"(1u), "r"(s));
    return r;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: about one second, then record NM_ERR_TIMEOUT and give up.
// Once a wait of this thread has run out (`dead`), later waits only poll once,
// so a kernel that lost its data ends within about a second in total.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, uint32_t *status, bool &dead)
{
    if (mbar_try_wait(bar, parity))
        return true;
    if (dead)
        return false;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            atomicOr(status, 1u << NM_ERR_TIMEOUT);
            dead = true;
            return false;
        }
    }
    return true;
}

// ---------------------------------------------------------------------------
// TMA (tensor copies global -> shared, completion counted on an mbarrier)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Orders this thread's earlier view of global memory (generic proxy) before
// its later TMA reads of global memory (async proxy).
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t c0, int32_t c1,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, int32_t c0,
                                                 int32_t c1, uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}

// ---------------------------------------------------------------------------
// Thread-block clusters (distributed shared memory)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t smem_addr_local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr_local), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v)
{
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// All threads of every CTA of the cluster: stores before are visible to loads after.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch (no-ops when the launch does not use it)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void pdl_wait_upstream()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Global loads
// ---------------------------------------------------------------------------

// 128-bit read-only load that does not allocate in L1 (streamed data).
__device__ __forceinline__ uint4 ldg_stream128(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_stream32(const void *p)
{
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Atomic add with acquire-release semantics at GPU scope: the caller's
// earlier writes (and those ordered before them, e.g. by __syncwarp) become
// visible to a thread that later reads the counter with acquire semantics.
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ float ldcg_f32(const float *p)
{
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

} // namespace nm
