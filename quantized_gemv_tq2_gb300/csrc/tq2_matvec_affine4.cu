// tq2_matvec_affine4.cu -- affine-int4 matvec (zero point factored out),
// M <= 2 activation rows per launch, sm_103a.
//
// What it computes ("Custom Metal kernels" page, the note on asymmetric
// (zero-point) int4: a fused affine-int4 matvec keeps the fast path by
// factoring the zero point out, acc += s * (dot - z * sum x)):
//   W[n][k] = s[n][g] * (q[n][k] - z[n][g]),  g = k / G,  q in [0, 15]
//   y[m][n] = sum_g s[n][g] * (sum_{k in g} x[m][k] q[n][k] - z[n][g] * sum_{k in g} x[m][k])
// Codes are 4 bits, two per byte, code k at bits 4*(k%2) of byte k/2 of its
// row (qs [N][K/2]); s and z are fp16 [N][K/G]; G is 64, 128 or 256.
//
// How (the ternary mma.sync kernel's skeleton, re-cut for nibbles):
//   * a producer warp streams 16-row x 2048-code chunks of the codes with
//     TMA into a ring of 16 KB stages, before the PDL wait: one copy per
//     stage through a 3-D view of the codes (16 words of a 256-code block,
//     rows, blocks), laid out block-major, 128 bytes per row, with the
//     128-byte swizzle (rows past N and blocks past K read as zero);
//   * the (s, z) pairs of the CTA's rows are staged once as half2;
//   * x is staged once per CTA in mma B-fragment order, plus the group sums
//     sum_{k in g} x_k for the zero-point term (fixed-order shuffle trees);
//   * unpack: a code word holds 8 nibbles; w & 0x000F000F (classes 0 and 2
//     after w >> 8) leaves two fp16 lanes whose bit patterns are the codes,
//     i.e. exactly q * 2^-24, and w & 0x00F000F0 leaves 16 q, i.e. q * 2^-20
//     (subnormal range, exact): one LOP3 per two codes, no conversion;
//   * the four nibble classes of a word each get an m16n8k16 MMA (f16 in,
//     f32 accumulate) whose B column c holds x at the class-c positions, so
//     column c of accumulator c is that class's sum; per group the classes
//     are combined (powers of 16), multiplied by s and the zero-point term
//     s * z * sum x is subtracted; warps' partials meet in shared memory and
//     are summed in a fixed order.  Bounded waits report TQ2_FLAG_TIMEOUT.
#include <cuda.h>
#include <cuda_fp16.h>

#include <cudaTypedefs.h>

#include <atomic>

#include "tq2_device.cuh"
#include "tq2_internal.cuh"

namespace tq2 {
namespace {

using namespace dev;

constexpr int kWarps = 8;                    // consumer warps: one 256-code block of a chunk each
constexpr int kConsumers = kWarps * 32;
constexpr int kThreads = kConsumers + 32;   // + the producer warp
constexpr int kChunkCodes = 2048;            // codes of a row per stage
constexpr int kStageBytes = 16 * kChunkCodes / 2;  // 16 rows x 1 KB
constexpr int kMaxStages = 8;
constexpr int kTwoPerSm = 112 * 1024;

struct A4Params {
    CUtensorMap tq;       // codes as uint64 {16 per block, N rows, K/256 blocks}, box 16 x 16 x 8, 128-byte swizzle
    const uint16_t *x;    // [M][K] fp16 bits (this launch's first activation row)
    const uint16_t *s;    // [N][K/G] fp16 bits
    const uint16_t *z;    // [N][K/G] fp16 bits
    void *y;              // [M][N] fp32 or fp16 (this launch's first row)
    uint32_t *status;
    int64_t N, K;
    int y_f16;
    int G;                // CTAs
    int ngr;              // row groups of 16 (the last one may be partial)
    int B;                // 256-code blocks per row
    int nkc;              // 2048-code chunks per row
    int ng;               // zero-point groups per row (K / group size)
    int max_rg;           // row groups of the largest CTA
    int stages;
    int off_bar, off_red, off_sz, off_xf, off_xg, off_ring, smem_total;
};

__device__ __forceinline__ void consumers_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

__device__ __forceinline__ void report_timeout(const A4Params &p, volatile int *abort_flag)
{
    *abort_flag = 1;
    if (p.status) atomicOr(p.status, TQ2_FLAG_TIMEOUT);
}

__device__ __forceinline__ uint2 lds64(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// checked forms for the debug build (TQ2_BOUNDS_CHECK); plain loads otherwise
__device__ __forceinline__ uint2 lds64_c(const SmemWindow &w, uint32_t addr)
{
    return TQ2_IN(addr >= w.lo && addr + 8u <= w.hi, w.status) ? lds64(addr) : make_uint2(0u, 0u);
}

__device__ __forceinline__ uint32_t lds32_c(const SmemWindow &w, uint32_t addr)
{
    return TQ2_IN(addr >= w.lo && addr + 4u <= w.hi, w.status) ? lds32(addr) : 0u;
}

__device__ __forceinline__ uint32_t pack_h2(uint16_t lo, uint16_t hi) { return (uint32_t)lo | ((uint32_t)hi << 16); }

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// ------------------------------------------------------------------ kernel
// kM: activation rows (1 or 2); kG: codes per zero-point group (64/128/256).
template <int kM, int kG>
__global__ void __launch_bounds__(kThreads, 2) matvec_affine4_kernel(const __grid_constant__ A4Params p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int abort_shared;
    volatile int *abort_flag = &abort_shared;

    constexpr int kJpg = kG / 64;    // 64-code slices (jw) per group
    constexpr int kGpb = 256 / kG;   // groups per 256-code block
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g0r = (int)((int64_t)blockIdx.x * p.ngr / p.G);
    const int g1r = (int)((int64_t)(blockIdx.x + 1) * p.ngr / p.G);
    const int nrg = g1r - g0r;
    const int64_t r0 = (int64_t)g0r * 16;
    const int64_t N = p.N, K = p.K;
    const int64_t rend = (int64_t)g1r * 16;
    const int nrows = (int)((rend < N ? rend : N) - r0);
    const int n_stages = nrg * p.nkc;
    const int S = p.stages;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.off_bar);  // full[S], empty[S]
    // ring start rounded up to 1024 bytes (the 128-byte swizzle pattern repeats every 1 KB)
    const uint32_t ring = (smem_addr(smem + p.off_ring) + 1023u) & ~1023u;

    uint32_t *const st_w = p.status;  // TQ2_FLAG_BOUNDS of debug builds
    const SmemWindow win{smem_addr(smem), smem_addr(smem) + (uint32_t)p.smem_total, st_w};
    const uint32_t ring_end = ring + (uint32_t)(S * kStageBytes);

    asm volatile("griddepcontrol.launch_dependents;");

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_addr(&bars[s]), 1);
            mbar_init(smem_addr(&bars[S + s]), kWarps);
        }
        abort_shared = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == kWarps) {
        // ------------------------------------------------------ producer warp
        const uint64_t pol = evict_first_policy();
        int issued = 0, kc = 0, rg = 0;
        for (int s = 0; s < n_stages; ++s) {
            const int slot = s % S;
            const int round = s / S;
            if (round > 0 &&
                !__all_sync(0xffffffffu, mbar_wait(smem_addr(&bars[S + slot]), (round - 1) & 1))) {
                if (lane == 0) report_timeout(p, abort_flag);
                break;
            }
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            // one 16 KB copy: 8 blocks x 16 rows x 128 bytes (blocks past K
            // and rows past N read as zero and count in full)
            const uint32_t full = smem_addr(&bars[slot]);
            if (lane == 0 && TQ2_IN(ring + (uint32_t)((slot + 1) * kStageBytes) <= ring_end && ring_end <= win.hi,
                                    st_w)) {
                mbar_arrive_expect_tx(full, (uint32_t)kStageBytes);
                tensor3d_g2s(ring + (uint32_t)(slot * kStageBytes), &p.tq, 0, (int)(r0 + rg * 16), kc * 8, full, pol);
            }
            __syncwarp();
            issued = s + 1;
            if (++kc == p.nkc) {
                kc = 0;
                ++rg;
            }
        }
        // No copy may still be writing shared memory when the CTA exits.
        for (int slot = 0; slot < S && slot < issued; ++slot) {
            const int last = slot + ((issued - 1 - slot) / S) * S;
            if (!mbar_wait(smem_addr(&bars[slot]), (last / S) & 1) && lane == 0) report_timeout(p, abort_flag);
        }
        return;
    }

    // ---------------------------------------------------------- consumer warps
    const int ng = p.ng;
    const int szstr = ng + 1;  // words per row of the (s, z) slice: rows g and g + 1 in different banks
    const uint32_t szs = smem_addr(smem + p.off_sz);
    const uint32_t xf = smem_addr(smem + p.off_xf);
    float *xg = reinterpret_cast<float *>(smem + p.off_xg);  // [kM][ng] group sums of x
    float *red = reinterpret_cast<float *>(smem + p.off_red);

    // (s, z) of this CTA's rows as half2, rows padded to ng + 1 words.  The
    // rows' slices of s and z are contiguous (and 16-byte aligned: s, z are,
    // and r0 is a multiple of 16), so they are read as 16-byte vectors, all
    // of a thread's loads in flight together; rows past N get s = 0 (no
    // contribution).
    {
        constexpr int kSzBatch = 4;
        const int ne = nrows * ng;
        const int nvec = ne >> 3;
        const uint4 *sv4 = reinterpret_cast<const uint4 *>(p.s + r0 * ng);
        const uint4 *zv4 = reinterpret_cast<const uint4 *>(p.z + r0 * ng);
        auto put = [&](int e, uint16_t sh, uint16_t zh) {
            const int r = e / ng;
            if (TQ2_IN(r * szstr + (e - r * ng) < p.max_rg * 16 * szstr, st_w))
                asm volatile("st.shared.u32 [%0], %1;" ::"r"(szs + (uint32_t)(r * szstr + (e - r * ng)) * 4u),
                             "r"(pack_h2(sh, zh))
                             : "memory");
        };
        for (int base = 0; base < nvec; base += kConsumers * kSzBatch) {
            uint4 a[kSzBatch], b[kSzBatch];
#pragma unroll
            for (int j = 0; j < kSzBatch; ++j) {
                const int v = base + j * kConsumers + tid;
                const bool in = v < nvec && TQ2_IN(r0 * ng + 8 * (int64_t)v + 8 <= N * ng, st_w);
                a[j] = in ? sv4[v] : make_uint4(0, 0, 0, 0);
                b[j] = in ? zv4[v] : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int j = 0; j < kSzBatch; ++j) {
                const int v = base + j * kConsumers + tid;
                if (v < nvec) {
                    const uint32_t aw[4] = {a[j].x, a[j].y, a[j].z, a[j].w};
                    const uint32_t bw[4] = {b[j].x, b[j].y, b[j].z, b[j].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        put(v * 8 + 2 * i, (uint16_t)(aw[i] & 0xffffu), (uint16_t)(bw[i] & 0xffffu));
                        put(v * 8 + 2 * i + 1, (uint16_t)(aw[i] >> 16), (uint16_t)(bw[i] >> 16));
                    }
                }
            }
        }
        for (int e = nvec * 8 + tid; e < ne; e += kConsumers)
            if (TQ2_IN(r0 * ng + e < N * ng, st_w)) put(e, p.s[r0 * ng + e], p.z[r0 * ng + e]);
        for (int e = ne + tid; e < nrg * 16 * ng; e += kConsumers) put(e, 0, 0);
    }

    // x depends on the previous kernel in the stream.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // x -> B-fragment order.  Task (m, block b, slice j, t) takes the 16
    // codes 64 j + 16 t .. +15 of block b; for class c it writes the entry
    // of lane (4 m + c) * 4 + t: b0 = (x[c], x[c + 4]), b1 = (x[8 + c],
    // x[12 + c]).  The 4 lanes of a slice, then the kG / 64 slices of a
    // group, are summed by a fixed shuffle tree into the group sum of x.
    {
        constexpr int kXBatch = 4;  // tasks per thread whose loads are in flight together
        const int ntask = kM * p.B * 16;
        for (int base0 = warp * 32; base0 < ntask; base0 += kConsumers * kXBatch) {
            uint4 lo[kXBatch], hi[kXBatch];
#pragma unroll
            for (int u = 0; u < kXBatch; ++u) {
                const int task = base0 + u * kConsumers + lane;
                lo[u] = hi[u] = make_uint4(0, 0, 0, 0);
                if (task < ntask) {
                    const int t = task & 3, j = (task >> 2) & 3, mb = task >> 4;
                    const int m = (kM == 2 && mb >= p.B) ? 1 : 0;
                    const int b = mb - m * p.B;
                    const uint16_t *src = p.x + (int64_t)m * K + (int64_t)b * 256 + j * 64 + t * 16;
                    if (!TQ2_IN(src + 16 <= p.x + (int64_t)kM * K, st_w)) src = p.x;
                    lo[u] = *reinterpret_cast<const uint4 *>(src);
                    hi[u] = *reinterpret_cast<const uint4 *>(src + 8);
                }
            }
#pragma unroll
            for (int u = 0; u < kXBatch; ++u) {
                const int task = base0 + u * kConsumers + lane;
                if (base0 + u * kConsumers >= ntask) break;  // warp-uniform
                const bool valid = task < ntask;
                const int t = task & 3, j = (task >> 2) & 3, mb = task >> 4;
                const int m = (kM == 2 && mb >= p.B) ? 1 : 0;
                const int b = mb - m * p.B;
                const uint32_t w[8] = {lo[u].x, lo[u].y, lo[u].z, lo[u].w, hi[u].x, hi[u].y, hi[u].z, hi[u].w};
                uint16_t h[16];
                float sum = 0.0f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    h[2 * i] = (uint16_t)(w[i] & 0xffffu);
                    h[2 * i + 1] = (uint16_t)(w[i] >> 16);
                    sum += h2f(h[2 * i]) + h2f(h[2 * i + 1]);
                }
                if (valid) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t e = (uint32_t)((4 * m + c) * 4 + t);
                        const uint32_t dst = xf + ((uint32_t)((b * 4 + j) * 16 * kM) + e) * 8u;
                        if (TQ2_IN(dst + 8u <= xf + (uint32_t)(p.B * 4 * 16 * kM * 8), st_w))
                        asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(dst), "r"(pack_h2(h[c], h[c + 4])),
                                     "r"(pack_h2(h[8 + c], h[12 + c]))
                                     : "memory");
                    }
                }
                sum += __shfl_xor_sync(0xffffffffu, sum, 1);
                sum += __shfl_xor_sync(0xffffffffu, sum, 2);
                if (kJpg >= 2) sum += __shfl_xor_sync(0xffffffffu, sum, 4);
                if (kJpg >= 4) sum += __shfl_xor_sync(0xffffffffu, sum, 8);
                if (valid && t == 0 && j % kJpg == 0 && TQ2_IN(m * ng + (b * 256 + j * 64) / kG < kM * ng, st_w))
                    xg[m * ng + (b * 256 + j * 64) / kG] = sum;
            }
        }
    }
    consumers_sync();

    // Lane (g, t): A rows g and g + 8; B column / accumulator columns 2t and
    // 2t + 1, i.e. activation row t >> 1 and classes 2 (t & 1), 2 (t & 1) + 1.
    // A row g is stage row rw = 2 (g & 3) + (g >> 2) (and rw + 8): a
    // half-warp then reads rows 0, 2, 4, 6 (or 1, 3, 5, 7), whose swizzled
    // 16-byte chunks are 8 distinct ones, so the code loads are free of bank
    // conflicts.
    const int g = lane >> 2, t = lane & 3;
    const int rw = 2 * (g & 3) + (g >> 2);
    const int pcls = t & 1;
    const int mrow = t >> 1;
    const bool mine = mrow < kM;
    constexpr uint32_t kLo = 0x000F000Fu, kHi = 0x00F000F0u;
    float acc_lo = 0.0f, acc_hi = 0.0f;

    int slot = 0, phase = 0, kc = 0, rg = 0;
    bool alive = true;  // false after this warp's wait ran out: no more waits
    for (int s = 0; s < n_stages; ++s) {
        bool ok = alive;
        if (ok && !__all_sync(0xffffffffu, mbar_wait(smem_addr(&bars[slot]), (uint32_t)phase))) {
            if (lane == 0) report_timeout(p, abort_flag);
            ok = alive = false;
        }
        const int nb = min(8, p.B - kc * 8);
        if (ok && warp < nb) {
            const int kb = kc * 8 + warp;  // this warp's 256-code block of the row
            const uint32_t cb = ring + (uint32_t)(slot * kStageBytes + warp * 2048);
            // words 8j + 2t, 8j + 2t + 1 of rows g, g + 8 (bytes 32j + 8t of
            // the 128-byte row, whose 16-byte chunks are swizzled by row & 7)
            uint2 wl[4], wh[4], bx[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t off = (uint32_t)((((2 * j + (t >> 1)) ^ rw) << 4) + (t & 1) * 8);
                wl[j] = lds64_c(win, cb + (uint32_t)rw * 128u + off);
                wh[j] = lds64_c(win, cb + (uint32_t)(rw + 8) * 128u + off);
                bx[j] = (lane < 16 * kM) ? lds64_c(win, xf + ((uint32_t)((kb * 4 + j) * 16 * kM) + (uint32_t)lane) * 8u)
                                         : make_uint2(0u, 0u);
            }
#pragma unroll
            for (int gi = 0; gi < kGpb; ++gi) {
                float c[4][4];
#pragma unroll
                for (int jj = 0; jj < kJpg; ++jj) {
                    const int j = gi * kJpg + jj;
                    const uint32_t a0 = wl[j].x, a1 = wh[j].x, a2 = wl[j].y, a3 = wh[j].y;
                    const uint32_t e0 = a0 >> 8, e1 = a1 >> 8, e2 = a2 >> 8, e3 = a3 >> 8;
                    if (jj == 0) {
                        mma_16816_zero(c[0], a0 & kLo, a1 & kLo, a2 & kLo, a3 & kLo, bx[j].x, bx[j].y);
                        mma_16816_zero(c[1], a0 & kHi, a1 & kHi, a2 & kHi, a3 & kHi, bx[j].x, bx[j].y);
                        mma_16816_zero(c[2], e0 & kLo, e1 & kLo, e2 & kLo, e3 & kLo, bx[j].x, bx[j].y);
                        mma_16816_zero(c[3], e0 & kHi, e1 & kHi, e2 & kHi, e3 & kHi, bx[j].x, bx[j].y);
                    } else {
                        mma_16816(c[0], a0 & kLo, a1 & kLo, a2 & kLo, a3 & kLo, bx[j].x, bx[j].y);
                        mma_16816(c[1], a0 & kHi, a1 & kHi, a2 & kHi, a3 & kHi, bx[j].x, bx[j].y);
                        mma_16816(c[2], e0 & kLo, e1 & kLo, e2 & kLo, e3 & kLo, bx[j].x, bx[j].y);
                        mma_16816(c[3], e0 & kHi, e1 & kHi, e2 & kHi, e3 & kHi, bx[j].x, bx[j].y);
                    }
                }
                // sum of q x over the group, in units of 2^-24: the low-nibble
                // classes carry q 2^-24, the high-nibble ones q 2^-20
                const float dlo = pcls ? (c[2][0] + c[3][1] * 0.0625f) : (c[0][0] + c[1][1] * 0.0625f);
                const float dhi = pcls ? (c[2][2] + c[3][3] * 0.0625f) : (c[0][2] + c[1][3] * 0.0625f);
                const int grp = kb * kGpb + gi;
                const uint32_t plo = lds32_c(win, szs + (uint32_t)((rg * 16 + rw) * szstr + grp) * 4u);
                const uint32_t phi = lds32_c(win, szs + (uint32_t)((rg * 16 + rw + 8) * szstr + grp) * 4u);
                const float slo = h2f((uint16_t)(plo & 0xffffu)), zlo = h2f((uint16_t)(plo >> 16));
                const float shi = h2f((uint16_t)(phi & 0xffffu)), zhi = h2f((uint16_t)(phi >> 16));
                // the zero-point term once per row and activation row (class pair 0)
                const float xs = (mine && pcls == 0 && TQ2_IN(mrow * ng + grp < kM * ng, st_w))
                                     ? xg[(mine ? mrow : 0) * ng + grp] : 0.0f;
                acc_lo = fmaf(slo * 16777216.0f, dlo, acc_lo);
                acc_lo = fmaf(-(slo * zlo), xs, acc_lo);
                acc_hi = fmaf(shi * 16777216.0f, dhi, acc_hi);
                acc_hi = fmaf(-(shi * zhi), xs, acc_hi);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&bars[S + slot]));
        if (++slot == S) {
            slot = 0;
            phase ^= 1;
        }
        if (++kc == p.nkc) {
            // row group done: the two class pairs (lanes t, t ^ 1) meet, and
            // this warp's partial of each (activation row, row) goes to red
            const float vlo = acc_lo + __shfl_xor_sync(0xffffffffu, acc_lo, 1);
            const float vhi = acc_hi + __shfl_xor_sync(0xffffffffu, acc_hi, 1);
            if (pcls == 0 && mine && TQ2_IN(((rg * kWarps + warp) * kM + mrow + 1) * 16 <= p.max_rg * kWarps * kM * 16,
                                            st_w)) {
                red[((rg * kWarps + warp) * kM + mrow) * 16 + rw] = vlo;
                red[((rg * kWarps + warp) * kM + mrow) * 16 + rw + 8] = vhi;
            }
            acc_lo = acc_hi = 0.0f;
            kc = 0;
            ++rg;
        }
    }
    consumers_sync();
    if (*abort_flag) return;  // y is invalid; TQ2_FLAG_TIMEOUT was reported

    // y[m][r0 + r] = sum over the warps (fixed order) of their partials
    for (int i = tid; i < kM * nrows; i += kConsumers) {
        const int m = (kM == 2 && i >= nrows) ? 1 : 0;
        const int r = i - m * nrows;
        const int rgi = r >> 4, ri = r & 15;
        float v = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) v += red[((rgi * kWarps + w) * kM + m) * 16 + ri];
        const int64_t o = (int64_t)m * N + r0 + r;
        if (!TQ2_IN(o < (int64_t)kM * N && rgi < p.max_rg, st_w)) continue;
        if (p.y_f16)
            reinterpret_cast<__half *>(p.y)[o] = __float2half_rn(v);
        else
            reinterpret_cast<float *>(p.y)[o] = v;
    }
}

// ------------------------------------------------------------------ host side
int align_up(int v, int a) { return (v + a - 1) / a * a; }

using KernelFn = void (*)(A4Params);

KernelFn kernel_for(int kM, int grp)
{
    if (kM == 1) {
        if (grp == 64) return matvec_affine4_kernel<1, 64>;
        if (grp == 128) return matvec_affine4_kernel<1, 128>;
        if (grp == 256) return matvec_affine4_kernel<1, 256>;
    } else if (kM == 2) {
        if (grp == 64) return matvec_affine4_kernel<2, 64>;
        if (grp == 128) return matvec_affine4_kernel<2, 128>;
        if (grp == 256) return matvec_affine4_kernel<2, 256>;
    }
    return nullptr;
}

int kernel_index(int kM, int grp) { return (kM - 1) * 3 + (grp == 64 ? 0 : grp == 128 ? 1 : 2); }

// Largest dynamic shared memory of one instantiation on `device` (the
// opt-in limit minus its static shared memory); the attribute is raised to
// it once.  0 on failure.
std::atomic<int> g_max_dyn[6][64];

int max_dynamic_smem(int kM, int grp, int device)
{
    if (device < 0 || device >= 64) return 0;
    KernelFn k = kernel_for(kM, grp);
    if (!k) return 0;
    const int idx = kernel_index(kM, grp);
    int v = g_max_dyn[idx][device].load();
    if (v > 0) return v;
    int optin = 0;
    cudaFuncAttributes fa;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, k) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    v = optin - (int)fa.sharedSizeBytes;
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, v) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    g_max_dyn[idx][device].store(v);
    return v;
}

// Shared-memory plan for G CTAs; false if it cannot fit in max_dyn bytes.
bool make_plan(int kM, int64_t N, int64_t K, int grp, int G, int max_dyn, A4Params &p)
{
    p.N = N;
    p.K = K;
    p.B = (int)(K / 256);
    p.nkc = (p.B + 7) / 8;
    p.ng = (int)(K / grp);
    p.ngr = (int)((N + 15) / 16);
    p.G = G;
    p.max_rg = (p.ngr + G - 1) / G;
    int64_t off = 0;
    p.off_bar = 0;
    off += 2 * kMaxStages * 8;
    p.off_red = (int)off;
    off += align_up(p.max_rg * kWarps * kM * 16 * 4, 16);
    p.off_sz = (int)off;
    off += (int64_t)p.max_rg * 16 * (p.ng + 1) * 4;
    off = (off + 15) / 16 * 16;
    p.off_xf = (int)off;
    off += (int64_t)p.B * 4 * 16 * kM * 8;
    p.off_xg = (int)off;
    off += (int64_t)kM * p.ng * 4;
    off = (off + 15) / 16 * 16;
    p.off_ring = (int)off;
    const int64_t fixed = off + 1024;  // the ring is aligned to 1 KB inside the kernel
    int64_t cap = kTwoPerSm;           // two CTAs per SM (the next call's CTA overlaps this one's tail)
    if (fixed + 2 * (int64_t)kStageBytes > cap) cap = max_dyn;
    if (fixed + 2 * (int64_t)kStageBytes > cap) return false;
    int S = (int)((cap - fixed) / kStageBytes);
    if (S > kMaxStages) S = kMaxStages;
    p.stages = S;
    p.smem_total = (int)(fixed + (int64_t)S * kStageBytes);
    return p.smem_total <= max_dyn;
}

// One CTA per SM (at most one per 16-row group) while the per-CTA share
// fits, more CTAs otherwise.
bool plan_for(int kM, int64_t N, int64_t K, int grp, int device, A4Params &p)
{
    const int max_dyn = max_dynamic_smem(kM, grp, device);
    if (max_dyn <= 0) return false;
    const int64_t ngr = (N + 15) / 16;
    const int nsm = sm_count(device);
    int G = (int)(ngr < nsm ? ngr : nsm);
    while (!make_plan(kM, N, K, grp, G, max_dyn, p)) {
        if (G >= ngr) return false;
        G = (int)(2 * (int64_t)G < ngr ? 2 * G : ngr);
    }
    return true;
}

// codes as uint64 {16 words of a 256-code block, N rows, K/256 blocks}
// (strides K/2 bytes for a row, 128 bytes for a block): a box of 16 x 16 x 8
// is one stage, 16 KB, block-major in shared memory with 128-byte rows
cudaError_t encode_codes(const uint8_t *qs, int64_t N, int64_t K, A4Params &p)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {16, (cuuint64_t)N, (cuuint64_t)(K / 256)};
    const cuuint64_t strides[2] = {(cuuint64_t)(K / 2), 128};
    const cuuint32_t box[3] = {16, 16, 8};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(&p.tq, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint8_t *>(qs), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

bool affine4_supported(int64_t M, int64_t N, int64_t K, int64_t grp, int device)
{
    if (M < 1 || N < 1 || K < 256 || K % 256 != 0 || (grp != 64 && grp != 128 && grp != 256)) return false;
    A4Params p{};
    // the launches take activation rows two at a time, the last one alone when M is odd
    if (M >= 2 && !plan_for(2, N, K, (int)grp, device, p)) return false;
    return (M % 2 == 0) || plan_for(1, N, K, (int)grp, device, p);
}

cudaError_t launch_affine4(const Affine4Args &a, int device)
{
    const int grp = (int)a.G;
    for (int64_t m0 = 0; m0 < a.M; m0 += 2) {
        const int kM = (a.M - m0 >= 2) ? 2 : 1;
        A4Params p{};
        if (!plan_for(kM, a.N, a.K, grp, device, p)) return cudaErrorInvalidConfiguration;
        cudaError_t e = encode_codes(a.qs, a.N, a.K, p);
        if (e != cudaSuccess) return e;
        p.x = a.x + m0 * a.K;
        p.s = a.s;
        p.z = a.z;
        p.y = static_cast<uint8_t *>(a.y) + (size_t)(m0 * a.N) * (a.y_f16 ? 2 : 4);
        p.status = a.status;
        p.y_f16 = a.y_f16;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)p.G);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = (size_t)p.smem_total;
        cfg.stream = a.stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, kernel_for(kM, grp), p);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace tq2
