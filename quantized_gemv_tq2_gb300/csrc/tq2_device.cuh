// tq2_device.cuh -- device helpers shared by the tensor-core matvec kernels:
// mbarrier waits with a time limit, TMA copies, the m16n8k16 MMA, shared-
// memory loads through 32-bit addresses and the fake-quant rounding.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/tq2.h"

namespace tq2 {
namespace dev {

// Longest any mbarrier wait may take before the kernel gives up and reports
// TQ2_FLAG_TIMEOUT (normal waits are microseconds).
constexpr unsigned long long kTimeoutNs = 200ull * 1000 * 1000;

// Checked indexing of the debug build (TQ2_BOUNDS_CHECK): TQ2_IN(cond, status)
// is cond, and when cond is false it also sets TQ2_FLAG_BOUNDS in the status
// word (if any), so that the caller skips the access and the host learns of
// it; nothing traps.  The release build compiles every check to true.
__device__ __forceinline__ bool flag_bounds(uint32_t *status)
{
    if (status) atomicOr(status, TQ2_FLAG_BOUNDS);
    return false;
}
#ifdef TQ2_BOUNDS_CHECK
#define TQ2_IN(cond, status) ((cond) ? true : ::tq2::dev::flag_bounds(status))
#else
#define TQ2_IN(cond, status) true
#endif

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// try_wait suspends the thread until the phase completes or the hint (ns)
// runs out, so waiting warps do not take issue slots from working ones.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "n"(20000)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long globaltimer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity; give up after limit_ns.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, unsigned long long limit_ns)
{
    if (mbar_test_wait(bar, parity)) return true;  // non-blocking fast path
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > limit_ns) return false;
    }
}

// Wait for the phase with the given parity; give up after kTimeoutNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    return mbar_wait_for(bar, parity, kTimeoutNs);
}

// The same wait with cluster-scope acquire: for barriers that CTAs of a
// thread-block cluster arrive on remotely (their earlier shared-memory writes
// are then visible to the waiter).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "n"(20000)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster_for(uint32_t bar, uint32_t parity, unsigned long long limit_ns)
{
    const unsigned long long t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (globaltimer() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity)
{
    return mbar_wait_cluster_for(bar, parity, kTimeoutNs);
}

// For short producer/consumer hand-offs: spin on the non-blocking test
// first; only a long wait falls back to the suspending try_wait.  Gives up
// after kTimeoutNs like mbar_wait.
__device__ __forceinline__ bool mbar_wait_spin(uint32_t bar, uint32_t parity)
{
#pragma unroll 1
    for (int i = 0; i < 2048; ++i)
        if (mbar_test_wait(bar, parity)) return true;
    return mbar_wait(bar, parity);
}

__device__ __forceinline__ uint64_t evict_last_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void tensor2d_g2s(uint32_t dst, const CUtensorMap *map, int x, int y,
                                             uint32_t bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void tensor3d_g2s(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                             uint32_t bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void named_barrier(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// D = A * B + D
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A * B (accumulator starts at zero: no register moves to clear C)
__device__ __forceinline__ void mma_16816_zero(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {0f00000000,0f00000000,0f00000000,0f00000000};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A * B + c (the same scalar in all four accumulator registers)
__device__ __forceinline__ void mma_16816_init(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1, float c)
{
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c));
}

// shared-memory loads through 32-bit shared-window addresses (volatile:
// they stay ordered after the mbarrier waits that publish the data)
__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ float lds_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// Phase trace of the trace build (TQ2_TRACE): globaltimer stamps of the
// class-column kernel per CTA, in two slots that consecutive launches take in
// turn (a launch's parity), read by tq2_trace_read.  Phases: 0 entry, 1 the
// wait on the previous kernel returned, 2 x staged, 3 the first stage's
// codes read, 4 the stage loop done, 5 y stored, 6 the producer's last copy
// issued.  Release builds compile the stamps out.
constexpr int kTraceCtas = 1024, kTracePhases = 8;
#ifdef TQ2_TRACE
// (g_trace is defined in the translation unit of the traced kernel)
#define TQ2_STAMP(seq, phase)                                                                      \
    do {                                                                                           \
        if (blockIdx.x < ::tq2::dev::kTraceCtas)                                                    \
            ::tq2::dev::g_trace[(seq) & 1][blockIdx.x][phase] = ::tq2::dev::globaltimer();         \
    } while (0)
#else
#define TQ2_STAMP(seq, phase) \
    do {                      \
    } while (0)
#endif

// Shared-memory reads checked, in debug builds (TQ2_BOUNDS_CHECK), against a
// CTA's dynamic shared memory [lo, hi): an address outside gives zero and
// TQ2_FLAG_BOUNDS.  Release builds compile them to the plain loads.
struct SmemWindow {
    uint32_t lo, hi;
    uint32_t *status;
};

__device__ __forceinline__ uint4 lds128_c(const SmemWindow &w, uint32_t addr)
{
    return TQ2_IN(addr >= w.lo && addr + 16u <= w.hi, w.status) ? lds128(addr) : make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ float lds_f32_c(const SmemWindow &w, uint32_t addr)
{
    return TQ2_IN(addr >= w.lo && addr + 4u <= w.hi, w.status) ? lds_f32(addr) : 0.0f;
}

// Static int8 fake-quant code (gemma4 wNa8o8 page, "Implemented"):
// rint(x * (1/s)) in fp32, ties to even, clamped to [-128, 127]; NaN -> 0.
// One conversion does the rounding, the clamp and the NaN case: cvt to s8
// with round-to-nearest-even and saturation (PTX: a NaN source gives 0).
__device__ __forceinline__ float fq_code(float x, float inv_s)
{
    const float t = __fmul_rn(x, inv_s);
    int q;
    asm("cvt.rni.sat.s8.f32 %0, %1;" : "=r"(q) : "f"(t));
    return (float)q;
}

// Output requantisation at store (gemma4 wNa8o8 page, "Implemented": the
// same fake-quant at a linear's output): y -> s * clamp(rint(y * (1/s)),
// -128, 127) on the fp32 result; s == 0 leaves y as computed.
__device__ __forceinline__ float requant_out(float y, float s, float inv_s)
{
    return (s != 0.0f) ? s * fq_code(y, inv_s) : y;
}

}  // namespace dev
}  // namespace tq2
