// tq2_matvec_ps.cu -- tensor-core ternary matvec for M = 1..16 activation
// rows with pre-scaled x (sm_103a).
//
// What it computes (BitCPM ternary page, linear-factoring paragraph):
//   y[m][n] = sum_b d[n][b] * sum_{k in b} x'[m][k] * (q[n][k] - 1)
//
// The unpack is the one of the M <= 2 kernel: ANDing a packed 32-bit word
// (16 codes of one row) with 0x00030003 << 2c leaves two fp16 lanes whose bit
// patterns are q * 4^c, i.e. the exact values q * 2^(2c - 24); the same on the
// word shifted right by 8 gives the other two bytes.  Here the B operand is
// pre-scaled per class instead of giving each class its own accumulator:
// B_c = x * 4^(3 - c), so every product is q * x * 2^-18 whatever the class,
// and all four classes of a word accumulate into one MMA accumulator whose 8
// columns are 8 activation rows (two n-tiles for M = 9..16).  The unpack cost
// (one LOP3 per two codes) is then shared by all M rows.
//
// x * 64 is exact in fp16 while |x| <= 1023.5.  A block whose x reaches 1024
// uses B_c = x * 4^-c instead (products q * x * 2^-24); the few low bits that
// x / 64 can lose in the subnormal range are below 2^-19 per element, far
// inside the tolerance of a block that holds a value >= 1024.  The block's
// "-1" term (sum_k x_k) starts the accumulator; the result is scaled back by
// the block's power of two and by d_b with one multiply each per lane.
//
// Data path per CTA (one CTA per SM, a contiguous range of output rows):
//   * a producer warp streams the rows into a ring of 16 KB stages with TMA
//     (whole rows in one 1-D bulk copy when K <= 4096, else 2-D boxes of
//     16 rows x up to 4096 codes), before griddepcontrol.wait;
//   * the d slice of the CTA's rows is staged to shared memory as fp32;
//   * after griddepcontrol.wait, x is turned into B fragments in shared
//     memory: all of K when it fits (stages then go row group by row group),
//     else one K range at a time (stages go K range by K range, x is
//     re-staged between ranges);
//   * 8 consumer warps take (16-row group, 256-block) units of each stage and
//     keep per-warp partials per row group; the partials are summed in a
//     fixed order at the end (run-to-run deterministic).
#include <cuda.h>
#include <cuda_fp16.h>

#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>

#include "tq2_device.cuh"
#include "tq2_internal.cuh"

namespace tq2 {
namespace {

using namespace dev;

constexpr int kWarps = 8;                      // consumer warps
constexpr int kConsumers = kWarps * 32;
constexpr int kThreads = kConsumers + 32;      // + one producer warp
constexpr int kMaxStages = 8;
constexpr int kTwoPerSm = 112 * 1024;          // shared memory that lets two CTAs share an SM

// One weight matrix of a launch.  A single call has one; a grouped call
// (several matrices sharing x) gives each matrix a contiguous range of CTAs
// [g0, g0 + G) in proportion to its rows, and its own output scale.
constexpr int kMaxGroup = 4;
struct PsMat {
    const uint8_t *qs;   // [N, K/4]
    const uint16_t *d;   // [N, K/256]
    void *y;             // [M, N]
    int64_t N;
    int g0, G;
    float out_scale;     // 0: y as computed; else requantised at store
    float inv_out;       // fp32(1/out_scale)
};

// The launch plan: arguments, grid and shared-memory layout.
struct PsPlan {
    MatvecArgs a;
    int G;        // CTAs
    int B;        // 256-blocks along K
    int NT;       // n-tiles of 8 activation rows
    int kcb;      // 256-blocks per stage K range (<= 16)
    int n_kc;     // K ranges
    int xkc;      // K ranges per x chunk (all of them, or 1)
    int R;        // 16-row groups per stage
    int tma2d;    // 0: a stage is R*16 whole rows (n_kc == 1), one 1-D bulk copy
    int rb;       // bytes per stage row in shared memory (kcb * 64)
    int stage_bytes, stages;
    int max_rg;   // row groups of the largest CTA
    int dstr;     // floats per row of the d slice (B + 1: odd, conflict-free)
    int xblocks;  // 256-blocks per x chunk (kcb * xkc)
    int off_bar, off_red, off_dsm, off_xinfo, off_frag, off_ring, smem_total;
    int n_mats;
};

// Kernel parameters for up to kG matrices (1 for a single call, so that its
// parameters stay small: every launch copies them).
template <int kG>
struct PsParams : PsPlan {
    // each matrix's qs as uint64 [N][K/32], boxes (kcb*8) x {16, 8, 4, 2, 1} rows
    CUtensorMap tmap[kG][5];
    PsMat mats[kG];
};

__device__ __forceinline__ void consumers_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

__device__ __forceinline__ void report_timeout(const PsPlan &p, volatile int *abort_flag)
{
    *abort_flag = 1;
    if (p.a.status) atomicOr(p.a.status, TQ2_FLAG_TIMEOUT);
}


// Byte offsets of one block's B fragments and per-column scalars.
//   frag:  block bx (within the x chunk) holds 512*M bytes; n-tile nt starts
//          at 4096*nt and has Mt = min(8, M - 8nt) columns; word slot jw
//          (0..3) is a 128*Mt region; in it, (half h, quad t, column g) is a
//          16-byte entry at (h*4*Mt + t*Mt + col)*16, col = g for a partial
//          n-tile and g ^ sw(t, jw) for a full one (Mt = 8).  Half 0 holds
//          classes 0, 1, half 1 classes 2, 3, each class as the (b0, b1)
//          register pair.
//   xinfo: float2 (C init, rescale) per (block, column), 8*NT columns a block.
// The swizzle of a full n-tile: shared memory serves a 16-byte access of 8
// lanes at a time, one 16-byte slot of each 128-byte row per lane.  The MMA
// reads (lanes g in {2q, 2q+1} x t in 0..3, fixed jw) and the staging writes
// (lanes t in {2p, 2p+1} x jw in 0..3, fixed g) each need 8 distinct slots
// mod 8; with col = g, Mt = 8 gives 4 and 1 (measured at M = 8: 560 K load
// and 557 K store bank conflicts per q/o call, 55 K and 188 K at M = 6).
// sw = (jw & 1) | (t & 1) << 1 | ((t >> 1) ^ (jw >> 1)) << 2 puts g's bits,
// t's and jw's each on their own bit of the slot, so both read 8.
__device__ __forceinline__ int col_slot(int t, int g, int jw, int Mt)
{
    const int sw = (jw & 1) | ((t & 1) << 1) | (((t >> 1) ^ (jw >> 1)) << 2);
    return t * Mt + (Mt == 8 ? (g ^ sw) : g);
}

__device__ __forceinline__ uint32_t frag_off(int bx, int nt, int jw, int h, int t, int g, int M)
{
    const int Mt = min(8, M - 8 * nt);
    return (uint32_t)(bx * 512 * M + nt * 4096 + jw * 128 * Mt + (h * 4 * Mt + col_slot(t, g, jw, Mt)) * 16);
}

// Turn x (rows m, blocks [kb0, kb0 + nbx)) into B fragments and xinfo.
// A half-warp takes one (row, block) pair, lane wi of it the 16-code word wi
// of the block (16 x values, two 16-byte loads): it writes that word's whole
// B entry (both halves, all four classes), so no value crosses lanes; the
// block sum and the "big" test are half-warp reductions.
template <int NT>
__device__ __forceinline__ void stage_x(const PsPlan &p, int kb0, int nbx, uint32_t frag, float2 *xinfo,
                                        int warp, int lane)
{
    const int M = p.a.M;
    const int64_t K = p.a.K;
    const bool convert = p.a.act_scale != 0.0f && !p.a.x_codes;  // x holds fp16 values, not yet codes
    const int hw = lane >> 4, wi = lane & 15;
    const int t = wi >> 2, jw = wi & 3;
    const uint32_t half_mask = hw ? 0xFFFF0000u : 0x0000FFFFu;
    constexpr int kBatch = 2;                 // pairs per half-warp per pass
    constexpr int kStep = kWarps * 2;         // pairs per pass of all warps
    const int npairs = nbx * M;
    // pair index pr -> (m = pr / nbx, bx = pr - m * nbx), stepped without division
    int m0 = 0, bx0 = 2 * warp + hw;
    while (bx0 >= nbx && m0 < M) {
        bx0 -= nbx;
        ++m0;
    }
    for (int pr0 = 2 * warp; pr0 < npairs; pr0 += kStep * kBatch) {
        uint4 v[kBatch][2];
        int mm[kBatch], bb[kBatch];
        int m = m0, bx = bx0;
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            mm[i] = m;
            bb[i] = bx;
            if (m < M) {
                const uint16_t *src = p.a.x + (int64_t)m * K + (int64_t)(kb0 + bx) * 256 + 16 * wi;
                if (!TQ2_IN(src + 16 <= p.a.x + (int64_t)M * K, p.a.status)) src = p.a.x;
                v[i][0] = *reinterpret_cast<const uint4 *>(src);
                v[i][1] = *reinterpret_cast<const uint4 *>(src + 8);
            }
            bx += kStep;
            while (bx >= nbx && m < M) {
                bx -= nbx;
                ++m;
            }
        }
        m0 = m;
        bx0 = bx;
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const bool live = mm[i] < M;  // uniform over each half-warp
            if (!__any_sync(0xffffffffu, live)) break;
            uint32_t r[8] = {v[i][0].x, v[i][0].y, v[i][0].z, v[i][0].w,
                             v[i][1].x, v[i][1].y, v[i][1].z, v[i][1].w};
            if (!live) {
#pragma unroll
                for (int q = 0; q < 8; ++q) r[q] = 0u;
            }
            if (convert) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&r[q]));
                    const __half2 c2 = __floats2half2_rn(fq_code(f.x, p.a.inv_scale), fq_code(f.y, p.a.inv_scale));
                    r[q] = *reinterpret_cast<const uint32_t *>(&c2);
                }
            }
            float s2[2] = {0.0f, 0.0f};
            uint32_t mx = 0u;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&r[q]));
                s2[q & 1] += f.x + f.y;
                mx = __vmaxu2(mx, r[q] & 0x7FFF7FFFu);
            }
            float sum = s2[0] + s2[1];
            const bool big_lane = ((mx & 0xFFFFu) >= 0x6400u) || ((mx >> 16) >= 0x6400u);
            const bool big = (__ballot_sync(0xffffffffu, big_lane) & half_mask) != 0u;
            // class scales: r[q] holds positions (2q, 2q+1), classes (0,1) for even q, (2,3) for odd q
            const __half2 s01 = big ? __floats2half2_rn(1.0f, 0.25f) : __floats2half2_rn(64.0f, 16.0f);
            const __half2 s23 = big ? __floats2half2_rn(0.0625f, 0.015625f) : __floats2half2_rn(4.0f, 1.0f);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const __half2 prod = __hmul2(*reinterpret_cast<const __half2 *>(&r[q]), (q & 1) ? s23 : s01);
                r[q] = *reinterpret_cast<const uint32_t *>(&prod);
            }
            // class c: b0 = (x[c], x[8+c]), b1 = (x[4+c], x[12+c]) of the word
            uint32_t e[8];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t sel = (c & 1) ? 0x7632u : 0x5410u;
                e[2 * c] = __byte_perm(r[c >> 1], r[4 + (c >> 1)], sel);
                e[2 * c + 1] = __byte_perm(r[2 + (c >> 1)], r[6 + (c >> 1)], sel);
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            if (live) {
                const int mi = mm[i], nt = mi >> 3, Mt = min(8, M - 8 * nt);
                const uint32_t dst = frag + frag_off(bb[i], nt, jw, 0, t, mi & 7, M);
                if (TQ2_IN(dst + (uint32_t)(64 * Mt) + 16u <= frag + (uint32_t)(p.xblocks * 512 * M), p.a.status)) {
                    sts128(dst, e[0], e[1], e[2], e[3]);                          // classes 0, 1
                    sts128(dst + (uint32_t)(64 * Mt), e[4], e[5], e[6], e[7]);  // classes 2, 3
                }
                if (wi == 0 && TQ2_IN(bb[i] * 8 * NT + mi < p.xblocks * 8 * NT, p.a.status)) {
                    const float sc = big ? 5.9604644775390625e-08f : 3.814697265625e-06f;  // 2^-24, 2^-18
                    const float rs = big ? 16777216.0f : 262144.0f;
                    xinfo[bb[i] * 8 * NT + mi] = make_float2(-sum * sc, rs);
                }
            }
        }
    }
}

// 16 HMMA of one (16-row group, 256-block) unit for n-tile nt: words jw of
// rows g and g + 8 are (wa, wb); the block's B fragments start at fb, this
// lane's entry of word jw, half 0, at fb + xo[jw], of half 1 at + h1; two
// accumulator chains, merged on return.
__device__ __forceinline__ void unit_mma(const SmemWindow &win, float (&c)[4], const uint32_t (&wa)[4],
                                         const uint32_t (&wb)[4],
                                         uint32_t fb, const uint32_t (&xo)[4], uint32_t h1, float2 init)
{
    float ca[4] = {init.x, init.y, init.x, init.y};
    float cb[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int jw = 0; jw < 4; ++jw) {
        const uint32_t w0 = wa[jw], w1 = wb[jw], s0 = w0 >> 8, s1 = w1 >> 8;
        const uint4 f0 = lds128_c(win, fb + xo[jw]);
        const uint4 f1 = lds128_c(win, fb + xo[jw] + h1);
        float (&cc)[4] = (jw < 2) ? ca : cb;
        mma_16816(cc, w0 & 0x00030003u, w1 & 0x00030003u, s0 & 0x00030003u, s1 & 0x00030003u, f0.x, f0.y);
        mma_16816(cc, w0 & 0x000C000Cu, w1 & 0x000C000Cu, s0 & 0x000C000Cu, s1 & 0x000C000Cu, f0.z, f0.w);
        mma_16816(cc, w0 & 0x00300030u, w1 & 0x00300030u, s0 & 0x00300030u, s1 & 0x00300030u, f1.x, f1.y);
        mma_16816(cc, w0 & 0x00C000C0u, w1 & 0x00C000C0u, s0 & 0x00C000C0u, s1 & 0x00C000C0u, f1.z, f1.w);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = ca[i] + cb[i];
}

template <int NT, int kG>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 2 : 1) matvec_ps_kernel(const __grid_constant__ PsParams<kG> p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int abort_shared;
    volatile int *abort_flag = &abort_shared;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int M = p.a.M;
    // this CTA's matrix and rows
    int mi = 0;
    if constexpr (kG > 1)
        while (mi + 1 < p.n_mats && (int)blockIdx.x >= p.mats[mi + 1].g0) ++mi;
    const uint8_t *const qs_g = p.mats[mi].qs;
    const uint16_t *const d_g = p.mats[mi].d;
    void *const y_g = p.mats[mi].y;
    const int64_t N = p.mats[mi].N, K = p.a.K;
    const int cta = (int)blockIdx.x - p.mats[mi].g0, G_m = p.mats[mi].G;
    const int64_t r0 = (int64_t)cta * N / G_m;
    const int64_t r1 = (int64_t)(cta + 1) * N / G_m;
    const int nrows = (int)(r1 - r0);
    const int nrg = (nrows + 15) >> 4;
    const int n_rgs = (nrg + p.R - 1) / p.R;  // stage row steps
    const int n_xc = (p.n_kc + p.xkc - 1) / p.xkc;
    const int n_stages = n_rgs * p.n_kc;      // every (row step, K range) once
    const int S = p.stages;
    const int B = p.B;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.off_bar);  // full[S], empty[S]
    uint8_t *ring = smem + p.off_ring;
    uint32_t *const st_w = p.a.status;  // TQ2_FLAG_BOUNDS of debug builds
    const SmemWindow win{smem_addr(smem), smem_addr(smem) + (uint32_t)p.smem_total, st_w};
    const uint32_t ring_end = smem_addr(ring) + (uint32_t)(S * p.stage_bytes);

    // Let the next kernel in the stream start its own weight prefetch.
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
        // Stage order: x chunk, then row step, then K range within the chunk.
        const uint64_t pol = evict_first_policy();
        const int64_t row_bytes = K / 4;
        int issued = 0;
        int xc = 0, rgi = 0, kci = 0;
        for (int s = 0; s < n_stages; ++s) {
            const int slot = s % S;
            const int round = s / S;
            if (round > 0 &&
                !__all_sync(0xffffffffu, mbar_wait(smem_addr(&bars[S + slot]), (round - 1) & 1))) {
                if (lane == 0) report_timeout(p, abort_flag);
                break;
            }
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            const int kc = xc * p.xkc + kci;
            const int rg0 = rgi * p.R;
            const int rows = min(p.R * 16, nrows - rg0 * 16);
            const uint32_t full = smem_addr(&bars[slot]);
            const uint32_t dst0 = smem_addr(ring + (size_t)slot * p.stage_bytes);
            if (!p.tma2d) {
                const uint32_t bytes = (uint32_t)rows * (uint32_t)row_bytes;
                if (lane == 0 && TQ2_IN((r0 + rg0 * 16) * row_bytes + bytes <= N * row_bytes && dst0 + bytes <= ring_end,
                                        st_w)) {
                    mbar_arrive_expect_tx(full, bytes);
                    bulk_g2s(dst0, qs_g + (r0 + rg0 * 16) * row_bytes, bytes, full, pol);
                }
            } else {
                // boxes of 16 rows x (kcb*64) bytes; the last group split into 8/4/2/1
                const bool in = TQ2_IN(dst0 + (uint32_t)rows * (uint32_t)p.rb <= ring_end, st_w);
                if (lane == 0 && in) mbar_arrive_expect_tx(full, (uint32_t)rows * (uint32_t)p.rb);
                __syncwarp();
                const int x = kc * p.kcb * 8;
                int roff = 0, box = 0;
                while (in && roff + 16 <= rows) {
                    if (lane == box) tensor2d_g2s(dst0 + roff * p.rb, &p.tmap[mi][0], x, (int)(r0 + rg0 * 16 + roff), full, pol);
                    roff += 16;
                    ++box;
                }
#pragma unroll
                for (int i = 1; i < 5; ++i) {
                    const int hh = 16 >> i;
                    if ((rows - roff) & hh) {
                        if (lane == box) tensor2d_g2s(dst0 + roff * p.rb, &p.tmap[mi][i], x, (int)(r0 + rg0 * 16 + roff), full, pol);
                        roff += hh;
                        ++box;
                    }
                }
            }
            __syncwarp();
            issued = s + 1;
            // advance (xc, rgi, kci)
            const int xkc_here = min(p.xkc, p.n_kc - xc * p.xkc);
            if (++kci == xkc_here) {
                kci = 0;
                if (++rgi == n_rgs) {
                    rgi = 0;
                    ++xc;
                }
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
    float *red = reinterpret_cast<float *>(smem + p.off_red);  // [max_rg][8 warps][16 rows][M]
    float *dsm = reinterpret_cast<float *>(smem + p.off_dsm);
    float2 *xinfo = reinterpret_cast<float2 *>(smem + p.off_xinfo);
    const uint32_t frag = smem_addr(smem + p.off_frag);
    const bool prologue = p.a.act_scale != 0.0f;

    for (int i = tid; i < nrg * kWarps * 16 * M; i += kConsumers)
        if (TQ2_IN(i < p.max_rg * kWarps * 16 * M, st_w)) red[i] = 0.0f;
    for (int i = tid; i < p.xblocks * 8 * NT; i += kConsumers) xinfo[i] = make_float2(0.0f, 0.0f);
    {
        const int nd = nrows * B;
        const uint16_t *dsrc = d_g + r0 * B;
        for (int base = 0; base < nd; base += kConsumers * 8) {
            uint16_t v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = base + j * kConsumers + tid;
                v[j] = (i < nd && TQ2_IN(r0 * B + i < N * B, st_w)) ? dsrc[i] : (uint16_t)0;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = base + j * kConsumers + tid;
                if (i < nd) {
                    const int r = i / B, b = i - r * B;
                    if (TQ2_IN(r * p.dstr + b < p.max_rg * 16 * p.dstr, st_w))
                        dsm[r * p.dstr + b] = __half2float(__ushort_as_half(v[j]));
                }
            }
        }
    }

    const int g = lane >> 2, t = lane & 3;
    const uint32_t ring_thr = smem_addr(ring) + (uint32_t)(g * p.rb + t * 16);
    const uint32_t a_half = (uint32_t)(8 * p.rb);
    // K = 4096 fast path (below): with one n-tile (M <= 8) stage 0's codes
    // are read before the wait on the previous kernel (the weights never
    // depend on it, and the consumer warps would only idle there), and its
    // slot released: M = 3..8 2-4 % faster; with two n-tiles no faster, so
    // they are read after x there.
    const bool fast = p.n_kc == 1 && p.R == 1 && p.kcb == 16 && p.xkc == 1;
    constexpr bool kEarly = NT == 1;
    constexpr int kU = 16 / kWarps;  // fast path: blocks per warp and stage
    const uint32_t au0 = ring_thr + (uint32_t)(warp * 64);
#define au(u) (au0 + (uint32_t)((u) * kWarps * 64))
    uint32_t W[kU][4], V[kU][4];
    // a stage's codes to registers; the slot is released once they are read
#define TQ2_PS_LOAD_CODES(SL)                                                              \
        do {                                                                               \
            _Pragma("unroll") for (int u_ = 0; u_ < kU; ++u_) {                            \
                const uint32_t pa_ = au(u_) + (uint32_t)((SL) * p.stage_bytes);           \
                const uint4 va_ = lds128_c(win, pa_), vb_ = lds128_c(win, pa_ + a_half);                 \
                W[u_][0] = va_.x; W[u_][1] = va_.y; W[u_][2] = va_.z; W[u_][3] = va_.w;    \
                V[u_][0] = vb_.x; V[u_][1] = vb_.y; V[u_][2] = vb_.z; V[u_][3] = vb_.w;    \
            }                                                                              \
            __syncwarp();                                                                  \
            if (lane == 0) mbar_arrive(smem_addr(&bars[S + (SL)]));                        \
        } while (0)
    bool fast_ok = false;
    auto fast_first = [&]() {  // stage 0's codes to registers
        fast_ok = n_stages > 0;
        if (fast_ok && !__all_sync(0xffffffffu, mbar_wait(smem_addr(&bars[0]), 0u))) {
            if (lane == 0) report_timeout(p, abort_flag);
            fast_ok = false;
        }
        if (fast_ok) TQ2_PS_LOAD_CODES(0);
    };
    if (kEarly && fast) fast_first();

    // x depends on the previous kernel in the stream.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    consumers_sync();  // xinfo zeroed before it is written
    stage_x<NT>(p, 0, min(p.xblocks, B), frag, xinfo, warp, lane);
    consumers_sync();

    uint32_t xo[NT][4];  // this lane's B entry of word jw within a block, per n-tile
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int gsel = (8 * nt + g < M) ? g : 0;
#pragma unroll
        for (int jw = 0; jw < 4; ++jw) xo[nt][jw] = frag_off(0, nt, jw, 0, t, gsel, M);
    }
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
    int cur_rg = -1;

    auto flush = [&](int rg) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int col = 8 * nt + 2 * t;
            float *rp = red + ((rg * kWarps + warp) * 16) * M;
            if (!TQ2_IN(rg < p.max_rg, st_w)) continue;
            if (col < M) {
                rp[g * M + col] += acc[nt][0];
                rp[(g + 8) * M + col] += acc[nt][2];
            }
            if (col + 1 < M) {
                rp[g * M + col + 1] += acc[nt][1];
                rp[(g + 8) * M + col + 1] += acc[nt][3];
            }
        }
    };

    // K = 4096 with x resident: every stage is one 16-row group x all 16
    // blocks, and warp w takes blocks w and w + 8 of every stage, so its B
    // fragment bases and per-column block terms stay in registers for the
    // whole call.  A stage's codes go to registers as soon as its copy has
    // landed and the slot is released at once; the next stage's codes are
    // read once this stage's last MMAs are issued.  Four accumulator chains
    // (one per code class) per block.
    if (fast) {
        // shared-memory bases of block warp + u * kWarps, recomputed from the
        // u = 0 ones at each use (holding all of them spills registers)
        const uint32_t fb0 = frag + (uint32_t)(warp * 512 * M), fb_step = (uint32_t)(kWarps * 512 * M);
        const uint32_t du0 = smem_addr(dsm) + (uint32_t)(g * p.dstr + warp) * 4u;
        const uint32_t xi0 = smem_addr(xinfo) + (uint32_t)(warp * 8 * NT + 2 * t) * 8u;  // + 64 per n-tile
#define fbu(u) (fb0 + (uint32_t)(u) * fb_step)
#define du(u) (du0 + (uint32_t)((u) * kWarps * 4))
#define xiu(u) (xi0 + (uint32_t)((u) * kWarps * 8 * NT * 8))
        uint32_t h1[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) h1[nt] = (uint32_t)(64 * min(8, M - 8 * nt));
        const uint32_t d_half = (uint32_t)(8 * p.dstr) * 4u, d_rg = (uint32_t)(16 * p.dstr) * 4u;
        float dg[kU], dg8[kU];
#define TQ2_PS_LOAD_SCALES(RG)                                                             \
        do {                                                                               \
            _Pragma("unroll") for (int u_ = 0; u_ < kU; ++u_) {                            \
                dg[u_] = lds_f32_c(win, du(u_) + (uint32_t)(RG) * d_rg);                          \
                dg8[u_] = lds_f32_c(win, du(u_) + (uint32_t)(RG) * d_rg + d_half);                \
            }                                                                              \
        } while (0)
        int sl = 0, ph = 0;
        if (!kEarly) fast_first();
        bool ok = fast_ok;  // stage 0's codes are in registers
        if (ok) TQ2_PS_LOAD_SCALES(0);
        for (int s = 0; ok && s < n_stages; ++s) {
            const int nsl = (sl + 1 == S) ? 0 : sl + 1;
            const int nph = (sl + 1 == S) ? (ph ^ 1) : ph;
            float acc[NT][4];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint4 xw = lds128_c(win, xiu(u) + (uint32_t)(64 * nt));
                    const float4 xi = make_float4(__uint_as_float(xw.x), __uint_as_float(xw.y),
                                                  __uint_as_float(xw.z), __uint_as_float(xw.w));
                    float c0[4] = {xi.x, xi.z, xi.x, xi.z};
                    float c1[4] = {0.0f, 0.0f, 0.0f, 0.0f}, c2[4] = {0.0f, 0.0f, 0.0f, 0.0f},
                          c3[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int jw = 0; jw < 4; ++jw) {
                        const uint32_t w0 = W[u][jw], w1 = V[u][jw], s0 = w0 >> 8, s1 = w1 >> 8;
                        const uint4 f0 = lds128_c(win, fbu(u) + xo[nt][jw]);
                        const uint4 f1 = lds128_c(win, fbu(u) + xo[nt][jw] + h1[nt]);
                        mma_16816(c0, w0 & 0x00030003u, w1 & 0x00030003u, s0 & 0x00030003u, s1 & 0x00030003u, f0.x, f0.y);
                        mma_16816(c1, w0 & 0x000C000Cu, w1 & 0x000C000Cu, s0 & 0x000C000Cu, s1 & 0x000C000Cu, f0.z, f0.w);
                        mma_16816(c2, w0 & 0x00300030u, w1 & 0x00300030u, s0 & 0x00300030u, s1 & 0x00300030u, f1.x, f1.y);
                        mma_16816(c3, w0 & 0x00C000C0u, w1 & 0x00C000C0u, s0 & 0x00C000C0u, s1 & 0x00C000C0u, f1.z, f1.w);
                    }
                    const float e0 = xi.y * dg[u], e1 = xi.w * dg[u], e2 = xi.y * dg8[u], e3 = xi.w * dg8[u];
                    acc[nt][0] = fmaf((c0[0] + c1[0]) + (c2[0] + c3[0]), e0, u ? acc[nt][0] : 0.0f);
                    acc[nt][1] = fmaf((c0[1] + c1[1]) + (c2[1] + c3[1]), e1, u ? acc[nt][1] : 0.0f);
                    acc[nt][2] = fmaf((c0[2] + c1[2]) + (c2[2] + c3[2]), e2, u ? acc[nt][2] : 0.0f);
                    acc[nt][3] = fmaf((c0[3] + c1[3]) + (c2[3] + c3[3]), e3, u ? acc[nt][3] : 0.0f);
                }
                if (u + 1 == kU && s + 1 < n_stages) {
                    // this stage's codes are all in MMA operands: read the next stage's
                    if (__all_sync(0xffffffffu, mbar_wait(smem_addr(&bars[nsl]), (uint32_t)nph))) {
                        TQ2_PS_LOAD_CODES(nsl);
                    } else {
                        if (lane == 0) report_timeout(p, abort_flag);
                        ok = false;
                    }
                }
            }
            if (ok && s + 1 < n_stages) TQ2_PS_LOAD_SCALES(s + 1);
            // row group s: this warp's partials (each row group once per warp)
            float *rp = red + ((s * kWarps + warp) * 16) * M;
            if (!TQ2_IN(s < p.max_rg, st_w)) rp = red;  // (flagged: y is not stored)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int col = 8 * nt + 2 * t;
                if (col < M) {
                    rp[g * M + col] = acc[nt][0];
                    rp[(g + 8) * M + col] = acc[nt][2];
                }
                if (col + 1 < M) {
                    rp[g * M + col + 1] = acc[nt][1];
                    rp[(g + 8) * M + col + 1] = acc[nt][3];
                }
            }
            sl = nsl;
            ph = nph;
        }
#undef TQ2_PS_LOAD_CODES
#undef TQ2_PS_LOAD_SCALES
#undef fbu
#undef au
#undef du
#undef xiu
    } else {
    int slot = 0, phase = 0;
    int xc = 0, rgi = 0, kci = 0;
    bool alive = true;
    for (int s = 0; s < n_stages; ++s) {
        if (s > 0 && kci == 0 && rgi == 0) {
            // a new x chunk: every warp is done with the previous one
            consumers_sync();
            stage_x<NT>(p, xc * p.xblocks, min(p.xblocks, B - xc * p.xblocks), frag, xinfo, warp, lane);
            consumers_sync();
        }
        bool ok = alive;
        if (ok && !__all_sync(0xffffffffu, mbar_wait(smem_addr(&bars[slot]), (uint32_t)phase))) {
            if (lane == 0) report_timeout(p, abort_flag);
            ok = alive = false;
        }
        if (ok) {
            const int kc = xc * p.xkc + kci;
            const int rg0 = rgi * p.R;
            const int Rs = min(p.R, nrg - rg0);
            const int kb0 = kc * p.kcb;
            const int nbk = min(p.kcb, B - kb0);
            const int units = Rs * nbk;
            const int kbx0 = kb0 - xc * p.xblocks;  // first block of this K range within the x chunk
            const uint32_t st = ring_thr + (uint32_t)(slot * p.stage_bytes);
            int j = 0, bl = warp;
            while (bl >= nbk) {
                bl -= nbk;
                ++j;
            }
            for (int u = warp; u < units; u += kWarps) {
                const int rg = rg0 + j;
                if (rg != cur_rg) {
                    if (cur_rg >= 0) flush(cur_rg);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.0f;
                    cur_rg = rg;
                }
                const uint32_t pa = st + (uint32_t)(j * 16 * p.rb + bl * 64);
                const uint4 va = lds128_c(win, pa), vb = lds128_c(win, pa + a_half);
                const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
                const int kb = kb0 + bl, bx = kbx0 + bl;
                const float d0 = lds_f32_c(win, smem_addr(dsm + (rg * 16 + g) * p.dstr + kb));
                const float d8 = lds_f32_c(win, smem_addr(dsm + (rg * 16 + g + 8) * p.dstr + kb));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int Mt = min(8, M - 8 * nt);
                    const uint32_t fb = frag + (uint32_t)(bx * 512 * M);
                    const uint4 xw = lds128_c(win, smem_addr(&xinfo[bx * 8 * NT + 8 * nt + 2 * t]));
                    const float4 xi = make_float4(__uint_as_float(xw.x), __uint_as_float(xw.y),
                                                  __uint_as_float(xw.z), __uint_as_float(xw.w));
                    float c[4];
                    unit_mma(win, c, wa, wb, fb, xo[nt], (uint32_t)(64 * Mt), make_float2(xi.x, xi.z));
                    acc[nt][0] = fmaf(c[0], xi.y * d0, acc[nt][0]);
                    acc[nt][1] = fmaf(c[1], xi.w * d0, acc[nt][1]);
                    acc[nt][2] = fmaf(c[2], xi.y * d8, acc[nt][2]);
                    acc[nt][3] = fmaf(c[3], xi.w * d8, acc[nt][3]);
                }
                // next unit of this warp: u + 8
                bl += kWarps;
                while (bl >= nbk) {
                    bl -= nbk;
                    ++j;
                }
            }
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(smem_addr(&bars[S + slot]));  // none after a wait ran out
        if (++slot == S) {
            slot = 0;
            phase ^= 1;
        }
        const int xkc_here = min(p.xkc, p.n_kc - xc * p.xkc);
        if (++kci == xkc_here) {
            kci = 0;
            if (++rgi == n_rgs) {
                rgi = 0;
                ++xc;
            }
        }
    }
    (void)n_xc;
    if (cur_rg >= 0) flush(cur_rg);
    }
    consumers_sync();
    if (*abort_flag) return;  // y is invalid; TQ2_FLAG_TIMEOUT was reported

    // y[m][r0 + r] = sum over warps (fixed order) of the partials
    for (int i = tid; i < M * nrows; i += kConsumers) {
        const int m = i / nrows, r = i - m * nrows;
        const int rg = r >> 4, ri = r & 15;
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += red[((rg * kWarps + w) * 16 + ri) * M + m];
        if (prologue) s *= p.a.act_scale;
        s = requant_out(s, p.mats[mi].out_scale, p.mats[mi].inv_out);
        const int64_t o = (int64_t)m * N + r0 + r;
        if (!TQ2_IN(o < (int64_t)M * N && rg < p.max_rg, st_w)) continue;
        if (p.a.y_f16)
            reinterpret_cast<__half *>(y_g)[o] = __float2half_rn(s);
        else
            reinterpret_cast<float *>(y_g)[o] = s;
    }
}

// ------------------------------------------------------------------ host side
int align_up(int v, int a) { return (v + a - 1) / a * a; }

// Shared-memory plan for CTAs of at most max_rows rows within `cap` bytes;
// false if it cannot fit.
bool make_plan(int M, int64_t max_rows, int64_t K, int cap, bool resident, int kcb_try, PsPlan &p)
{
    const int64_t B = K / 256;
    if (B < 1 || B > (1 << 20)) return false;
    p.B = (int)B;
    p.NT = (M + 7) / 8;
    p.max_rg = (int)((max_rows + 15) / 16);
    if (resident) {
        if (B <= 16) {
            p.kcb = (int)B;
            p.n_kc = 1;
            p.tma2d = 0;
            p.R = 16 / (int)B;
        } else {
            p.kcb = 16;
            p.n_kc = (int)((B + 15) / 16);
            p.tma2d = 1;
            p.R = 1;
        }
        p.xkc = p.n_kc;
        p.xblocks = (int)B;
    } else {
        if (kcb_try > B) return false;
        p.kcb = kcb_try;
        p.n_kc = (int)((B + kcb_try - 1) / kcb_try);
        p.tma2d = (p.n_kc > 1) ? 1 : 0;
        p.R = 16 / kcb_try;
        p.xkc = 1;
        p.xblocks = kcb_try;
    }
    if (p.R > p.max_rg) p.R = p.max_rg;
    p.rb = p.kcb * 64;
    p.stage_bytes = p.R * 16 * p.rb;
    p.dstr = (int)B + 1;
    int64_t off = 0;
    p.off_bar = 0;
    off += 2 * kMaxStages * 8;
    p.off_red = (int)off;
    off += align_up(p.max_rg * kWarps * 16 * M * 4, 16);
    p.off_dsm = (int)off;
    off += (int64_t)p.max_rg * 16 * p.dstr * 4;
    off = (off + 15) / 16 * 16;
    p.off_xinfo = (int)off;
    off += (int64_t)p.xblocks * 8 * p.NT * 8;
    p.off_frag = (int)off;
    off += (int64_t)p.xblocks * 512 * M;
    off = (off + 127) / 128 * 128;
    p.off_ring = (int)off;
    if (off + 2 * (int64_t)p.stage_bytes > cap) return false;
    int S = (int)((cap - off) / p.stage_bytes);
    if (S > kMaxStages) S = kMaxStages;
    p.stages = S;
    p.smem_total = (int)off + S * p.stage_bytes;
    return true;
}

std::atomic<int> g_max_dyn[2][64];

template <int NT>
int max_dynamic_smem(int device)
{
    if (device < 0 || device >= 64) return 0;
    int v = g_max_dyn[NT - 1][device].load();
    if (v > 0) return v;
    int optin = 0;
    cudaFuncAttributes fa;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, matvec_ps_kernel<NT, 1>) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    v = optin - (int)fa.sharedSizeBytes;
    if (cudaFuncSetAttribute(matvec_ps_kernel<NT, kMaxGroup>, cudaFuncAttributeMaxDynamicSharedMemorySize, v) !=
            cudaSuccess ||
        cudaFuncSetAttribute(matvec_ps_kernel<NT, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, v) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    g_max_dyn[NT - 1][device].store(v);
    return v;
}

// Prefer resident x (staged once) over K-chunked x, then a plan that lets two
// CTAs share an SM (the next call's weights then stream while this one
// computes) over one CTA per SM, and one CTA per SM before more.  Resident x
// on one CTA per SM beats K-chunked x on two where both fit (measured on
// GB300, back-to-back calls: down 4096x16384 at M = 3 / 4 / 5: 15.7 / 17.7 /
// 18.9 against 16.4 / 18.3 / 19.7 us; gate/up 16384x4096 at M = 7 / 8: 14.2
// / 18.7 against 14.7 / 19.0 us): K-chunked x is re-staged per K range
// behind two barriers that drain the stage ring.
bool plan_rows(int M, int64_t max_rows, int64_t K, int max_dyn, PsPlan &p)
{
    for (int cap : {kTwoPerSm, max_dyn}) {
        if (cap > max_dyn) continue;
        if (make_plan(M, max_rows, K, cap, true, 0, p)) return true;
    }
    for (int cap : {kTwoPerSm, max_dyn}) {
        if (cap > max_dyn) continue;
        for (int kcb : {16, 8, 4, 2, 1})
            if (make_plan(M, max_rows, K, cap, false, kcb, p)) return true;
    }
    return false;
}

int max_dyn_for(int M, int device)
{
    return (M <= 8) ? max_dynamic_smem<1>(device) : max_dynamic_smem<2>(device);
}

bool plan_for(int M, int64_t N, int64_t K, int device, PsPlan &p)
{
    const int max_dyn = max_dyn_for(M, device);
    if (max_dyn <= 0 || M < 1 || M > 16) return false;
    const int nsm = sm_count(device);
    int G = (int)((N < (int64_t)nsm) ? N : nsm);
    for (;;) {
        if (plan_rows(M, (N + G - 1) / G, K, max_dyn, p)) {
            p.G = G;
            p.n_mats = 1;
            return true;
        }
        if (G >= N) return false;
        G = (int)((2 * (int64_t)G < N) ? 2 * G : N);
    }
}

// CTAs of a group in proportion to the matrices' rows (at least one each,
// one per SM in total first, then twice as many while no plan fits), then
// the plan for the largest per-CTA row count.
bool group_plan(int M, int n, const int64_t *N, int64_t K, int device, PsParams<kMaxGroup> &p)
{
    const int max_dyn = max_dyn_for(M, device);
    if (max_dyn <= 0 || M < 1 || M > 16 || n < 1 || n > kMaxGroup) return false;
    int64_t total = 0;
    for (int j = 0; j < n; ++j) {
        if (N[j] < 1) return false;
        total += N[j];
    }
    const int nsm = sm_count(device);
    for (int cap = nsm; cap <= 64 * nsm; cap *= 2) {
        int G[kMaxGroup], sum = 0;
        for (int j = 0; j < n; ++j) {
            int64_t g = (int64_t)cap * N[j] / total;
            if (g < 1) g = 1;
            if (g > N[j]) g = (int)N[j];
            G[j] = (int)g;
            sum += G[j];
        }
        while (sum < cap) {  // leftover CTAs to the matrix with the most rows per CTA
            int best = -1;
            double worst = 0.0;
            for (int j = 0; j < n; ++j)
                if (G[j] < N[j] && (double)N[j] / G[j] > worst) {
                    worst = (double)N[j] / G[j];
                    best = j;
                }
            if (best < 0) break;
            ++G[best];
            ++sum;
        }
        int64_t max_rows = 0;
        int g0 = 0;
        for (int j = 0; j < n; ++j) {
            max_rows = std::max<int64_t>(max_rows, (N[j] + G[j] - 1) / G[j]);
            p.mats[j].N = N[j];
            p.mats[j].g0 = g0;
            p.mats[j].G = G[j];
            g0 += G[j];
        }
        if (plan_rows(M, max_rows, K, max_dyn, p)) {
            p.n_mats = n;
            p.G = g0;
            return true;
        }
    }
    return false;
}

// qs as uint64 [N][K/32]; boxes (kcb*8) x {16, 8, 4, 2, 1}
cudaError_t encode_maps(const uint8_t *qs, int64_t N, int64_t K, int kcb, CUtensorMap (&tmap)[5])
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)(K / 32), (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)(K / 4)};
    const cuuint32_t estr[2] = {1, 1};
    for (int i = 0; i < 5; ++i) {
        const cuuint32_t box[2] = {(cuuint32_t)(kcb * 8), (cuuint32_t)(16 >> i)};
        CUresult r = enc(&tmap[i], CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint8_t *>(qs), dims, strides,
                         box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

template <int NT, int kG>
cudaError_t launch_params(const PsParams<kG> &p, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)p.smem_total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, matvec_ps_kernel<NT, kG>, p);
}

template <int NT>
cudaError_t launch_impl(const MatvecArgs &a, int device)
{
    PsParams<1> p{};
    p.a = a;
    if (!plan_for(a.M, a.N, a.K, device, p)) return cudaErrorInvalidConfiguration;
    p.mats[0].N = a.N;
    p.mats[0].g0 = 0;
    p.mats[0].G = p.G;
    p.mats[0].qs = a.qs;
    p.mats[0].d = a.d;
    p.mats[0].y = a.y;
    p.mats[0].out_scale = a.out_scale;
    p.mats[0].inv_out = a.inv_out;
    if (p.tma2d) {
        cudaError_t e = encode_maps(a.qs, a.N, a.K, p.kcb, p.tmap[0]);
        if (e != cudaSuccess) return e;
    }
    return launch_params<NT, 1>(p, a.stream);
}

template <int NT>
cudaError_t launch_group_impl(const MatvecArgs &a, int n, const uint8_t *const *qs, const uint16_t *const *d,
                              void *const *y, const int64_t *N, const float *out_scale, const float *inv_out,
                              int device)
{
    PsParams<kMaxGroup> p{};
    p.a = a;
    if (!group_plan(a.M, n, N, a.K, device, p)) return cudaErrorInvalidConfiguration;
    for (int j = 0; j < n; ++j) {
        p.mats[j].qs = qs[j];
        p.mats[j].d = d[j];
        p.mats[j].y = y[j];
        p.mats[j].out_scale = out_scale ? out_scale[j] : 0.0f;
        p.mats[j].inv_out = inv_out ? inv_out[j] : 0.0f;
        if (p.tma2d) {
            cudaError_t e = encode_maps(qs[j], N[j], a.K, p.kcb, p.tmap[j]);
            if (e != cudaSuccess) return e;
        }
    }
    return launch_params<NT, kMaxGroup>(p, a.stream);
}

}  // namespace

bool ps_matvec_supported(int M, int64_t N, int64_t K, int device)
{
    if (M < 1 || M > 16 || N < 1 || K < 256) return false;
    PsPlan p{};
    return plan_for(M, N, K, device, p);
}

bool ps_group_supported(int M, int n, const int64_t *N, int64_t K, int device)
{
    if (M < 1 || M > 16 || K < 256) return false;
    PsParams<kMaxGroup> p{};
    return group_plan(M, n, N, K, device, p);
}

cudaError_t launch_matvec_ps_group(const MatvecArgs &a, int n, const uint8_t *const *qs, const uint16_t *const *d,
                                   void *const *y, const int64_t *N, const float *out_scale,
                                   const float *inv_out, int device)
{
    if (a.M >= 1 && a.M <= 8) return launch_group_impl<1>(a, n, qs, d, y, N, out_scale, inv_out, device);
    if (a.M >= 9 && a.M <= 16) return launch_group_impl<2>(a, n, qs, d, y, N, out_scale, inv_out, device);
    return cudaErrorInvalidValue;
}

cudaError_t launch_matvec_ps(const MatvecArgs &a, int device)
{
    if (a.M >= 1 && a.M <= 8) return launch_impl<1>(a, device);
    if (a.M >= 9 && a.M <= 16) return launch_impl<2>(a, device);
    return cudaErrorInvalidValue;
}

}  // namespace tq2
