// tq2_matvec_dp4.cu -- integer-dot ternary matvec for one activation row
// (M = 1), sm_103a.
//
// What it computes (BitCPM ternary page, linear-factoring paragraph):
//   y[n] = sum_b d[n][b] * sum_{k in b} x'[k] * (q[n][k] - 1)
//
// The block sums run as 8-bit dot products (dp4a: four u8 x s8 products and
// an add per instruction) on integer x.  x is turned into integers per
// 256-block with a power-of-two scale 2^S_b and split into P 8-bit pieces:
//   * with the static int8 fake-quant prologue (gemma4 wNa8o8 page) x' is
//     already an int8 code: P = 1, S_b = 0, exact;
//   * otherwise X_k = round(x_k * 2^S_b) with |X_k| < 2^15 (S_b = 14 - E_b,
//     E_b the exponent of the block's largest |x|) in two pieces, when the
//     rounding bound 256 * 2^(E_b - 15) * |d_b| is at most half of the
//     block's tolerance term 1e-3 * |d_b| * sum_k |x_k|; if any block of the
//     vector misses that bound, all blocks use three pieces (S_b = 21 - E_b,
//     bound 2^-14 of the block maximum, far inside the tolerance).
// The codes of one packed 32-bit word are read as four bytes per class c
// ((w >> 2c) & 0x03030303, one code per byte); the matching x bytes (the
// positions 4i + c of the word) were laid out per class at staging.  The
// "-1" of q - 1 is the block's integer sum of X, subtracted before the one
// conversion to fp32 and the one multiply by d_b * 2^-S_b.
//
// Why: the legacy m16n8k16 MMA holds its SM sub-partition's issue slot for
// ~8 cycles per instruction (measured on this part), which caps an mma.sync
// ternary matvec near the HBM rate; dp4a runs on the FMA-heavy pipe at half
// rate and overlaps with the unpack's logic ops on the ALU pipe.
//
// Data path per CTA (a contiguous range of output rows, all of K):
//   * a producer warp streams the rows with TMA into a ring of 16 KB stages
//     (whole rows in one 1-D bulk copy when K <= 4096, else 16 rows x 4096
//     codes in 2-D boxes), before griddepcontrol.wait;
//   * the d slice is staged as fp32;
//   * after griddepcontrol.wait x is staged (two passes: block statistics,
//     then pieces);
//   * warp items are (row, group of 8 blocks); lane l takes block
//     8*group + l/4, quarter l%4 (4 words); the lane's x pieces stay in
//     registers for the K range; per row: one 16-byte shared load, 28 logic
//     ops, 16*P dp4a, then a warp reduction of the d-scaled fp32 partials.
#include <cuda.h>
#include <cuda_fp16.h>

#include <cudaTypedefs.h>

#include <atomic>

#include "tq2_device.cuh"
#include "tq2_internal.cuh"

namespace tq2 {
namespace {

using namespace dev;

constexpr int kWarps = 8;
constexpr int kConsumers = kWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kMaxStages = 8;
constexpr int kTwoPerSm = 112 * 1024;
constexpr int kMaxP = 3;

struct Dp4Params {
    CUtensorMap tmap[5];  // K > 4096: qs as uint64 [N][K/32], boxes 128 x {16, 8, 4, 2, 1}
    MatvecArgs a;
    int G;         // CTAs
    int B;         // 256-blocks per row
    int tma2d;     // 0: stage = SR whole rows, one 1-D bulk copy
    int SR;        // rows per stage
    int nbk;       // 256-blocks per stage row (16, or B when K <= 4096)
    int n_kc;      // K ranges per row step
    int ngrp;      // groups of 8 blocks per stage row (1 or 2)
    int rb;        // shared-memory bytes per stage row
    int stage_bytes, stages;
    int max_rows;  // rows of the largest CTA
    int dstr;      // floats per row of the d slice
    int off_bar, off_red, off_dsm, off_binfo, off_xsq, off_xq, off_flag, off_ring, smem_total;
};

__device__ __forceinline__ void consumers_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

__device__ __forceinline__ void report_timeout(const Dp4Params &p, volatile int *abort_flag)
{
    *abort_flag = 1;
    if (p.a.status) atomicOr(p.a.status, TQ2_FLAG_TIMEOUT);
}

__device__ __forceinline__ uint32_t dp4a_us(uint32_t a, uint32_t b, uint32_t c)  // u8 x s8
{
    uint32_t d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c)  // u8 x u8
{
    uint32_t d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// 2^e as fp32 for e in [-126, 127]
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// Round-to-nearest-even integer of v, |v| < 2^22 (fp32 magic-number add).
__device__ __forceinline__ int rint_small(float v)
{
    return __float_as_int(v + 12582912.0f) - 0x4B400000;
}

// x bytes of one (block, quarter, piece, word) as one uint4: classes 0..3.
// Blocks go in groups of 8 (one warp item); within a (group, piece, word)
// the 32 lanes' entries are contiguous, so a warp's load is one 512-byte,
// conflict-free read.
__device__ __forceinline__ uint32_t xq_off(int b, int qd, int piece, int jw, int P)
{
    return (uint32_t)(((((b >> 3) * P + piece) * 4 + jw) * 32 + (b & 7) * 4 + qd) * 16);
}

// Consumer main loop for P = 1 or 2 pieces, held in registers.
template <int P>
__device__ __forceinline__ void consume(const Dp4Params &p, uint8_t *smem, uint64_t *bars, volatile int *abort_flag,
                                        int nrows, int warp, int lane)
{
    const int S = p.stages;
    const int B = p.B;
    float *red = reinterpret_cast<float *>(smem + p.off_red);
    const float *dsm = reinterpret_cast<const float *>(smem + p.off_dsm);
    const float *binfo = reinterpret_cast<const float *>(smem + p.off_binfo);  // 2^-S_b
    const int *xsq = reinterpret_cast<const int *>(smem + p.off_xsq);          // [B][4]
    const uint32_t xq = smem_addr(smem + p.off_xq);
    const uint32_t ring = smem_addr(smem + p.off_ring);

    const int grp = (p.ngrp == 2) ? (warp & 1) : 0;
    const int row_step = kWarps / p.ngrp;
    const int row_w = (p.ngrp == 2) ? (warp >> 1) : warp;
    const int bl = grp * 8 + (lane >> 2), qd = lane & 3;
    const int n_rs = (nrows + p.SR - 1) / p.SR;
    constexpr int kRegP = (P < 2) ? P : 2;

    uint4 xr[kRegP][4];
    int xs = 0;
    float sc = 0.0f;
    float racc = 0.0f;  // K > 4096: the sum over K ranges of the row this lane holds
    int cur_kc = -1;

    int slot = 0, phase = 0, kc = 0, rs = 0;
    bool alive = true;
    const int n_stages = n_rs * p.n_kc;
    for (int s = 0; s < n_stages; ++s) {
        bool ok = alive;
        if (ok && !__all_sync(0xffffffffu, mbar_wait(smem_addr(&bars[slot]), (uint32_t)phase))) {
            if (lane == 0) report_timeout(p, abort_flag);
            ok = alive = false;
        }
        if (ok) {
            const int kb0 = kc * p.nbk;
            const int nbk = min(p.nbk, B - kb0);
            const bool active = bl < nbk;
            const int kb = kb0 + (active ? bl : 0);
            if (kc != cur_kc) {
                // this lane's x pieces, quarter sum and scale for the K range
#pragma unroll
                for (int pc = 0; pc < kRegP; ++pc)
#pragma unroll
                    for (int jw = 0; jw < 4; ++jw) xr[pc][jw] = lds128(xq + xq_off(kb, qd, pc, jw, P));
                xs = xsq[kb * 4 + qd];
                sc = binfo[kb];
                cur_kc = kc;
            }
            const int row_base = rs * p.SR;
            const int rows_here = min(p.SR, nrows - row_base);
            const uint32_t st = ring + (uint32_t)(slot * p.stage_bytes) + (uint32_t)(bl * 64 + qd * 16);
            // Rows of this warp in groups of four: the four rows' dot-product
            // chains interleave, and one transposing reduction (6 shuffles)
            // leaves row k's sum over the warp's 8 blocks in lanes
            // 8k .. 8k+7.
            const int nr = (rows_here > row_w) ? (rows_here - row_w + row_step - 1) / row_step : 0;
            const int my_k = (lane >> 3) & 3;
            for (int k0 = 0; k0 < nr; k0 += 4) {
                float f[4];
                uint4 wv[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const bool v = active && (k0 + k < nr);
                    wv[k] = v ? lds128(st + (uint32_t)((row_w + (k0 + k) * row_step) * p.rb)) : make_uint4(0, 0, 0, 0);
                }
                uint32_t a0[4] = {0, 0, 0, 0}, a1[4] = {0, 0, 0, 0}, a2[4] = {0, 0, 0, 0};
#pragma unroll
                for (int jw = 0; jw < 4; ++jw) {
                    uint4 x2 = make_uint4(0, 0, 0, 0);
                    if (P == 3) x2 = lds128(xq + xq_off(kb, qd, 2, jw, P));
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t w = (jw == 0) ? wv[k].x : (jw == 1) ? wv[k].y : (jw == 2) ? wv[k].z : wv[k].w;
                        const uint32_t c0 = w & 0x03030303u, c1 = (w >> 2) & 0x03030303u,
                                       c2 = (w >> 4) & 0x03030303u, c3 = (w >> 6) & 0x03030303u;
                        if (P == 1) {
                            a0[k] = dp4a_us(c0, xr[0][jw].x, a0[k]);
                            a0[k] = dp4a_us(c1, xr[0][jw].y, a0[k]);
                            a0[k] = dp4a_us(c2, xr[0][jw].z, a0[k]);
                            a0[k] = dp4a_us(c3, xr[0][jw].w, a0[k]);
                        } else {
                            // piece 0 unsigned (low byte); the top piece signed
                            a0[k] = dp4a_uu(c0, xr[0][jw].x, a0[k]);
                            a0[k] = dp4a_uu(c1, xr[0][jw].y, a0[k]);
                            a0[k] = dp4a_uu(c2, xr[0][jw].z, a0[k]);
                            a0[k] = dp4a_uu(c3, xr[0][jw].w, a0[k]);
                            if (P == 2) {
                                a1[k] = dp4a_us(c0, xr[kRegP - 1][jw].x, a1[k]);
                                a1[k] = dp4a_us(c1, xr[kRegP - 1][jw].y, a1[k]);
                                a1[k] = dp4a_us(c2, xr[kRegP - 1][jw].z, a1[k]);
                                a1[k] = dp4a_us(c3, xr[kRegP - 1][jw].w, a1[k]);
                            } else {
                                a1[k] = dp4a_uu(c0, xr[kRegP - 1][jw].x, a1[k]);
                                a1[k] = dp4a_uu(c1, xr[kRegP - 1][jw].y, a1[k]);
                                a1[k] = dp4a_uu(c2, xr[kRegP - 1][jw].z, a1[k]);
                                a1[k] = dp4a_uu(c3, xr[kRegP - 1][jw].w, a1[k]);
                                a2[k] = dp4a_us(c0, x2.x, a2[k]);
                                a2[k] = dp4a_us(c1, x2.y, a2[k]);
                                a2[k] = dp4a_us(c2, x2.z, a2[k]);
                                a2[k] = dp4a_us(c3, x2.w, a2[k]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    int tot;
                    if (P == 1) tot = (int)a0[k];
                    else if (P == 2) tot = (int)a0[k] + (int)a1[k] * 256;
                    else tot = (int)a0[k] + (int)a1[k] * 256 + (int)a2[k] * 65536;
                    const int rl = row_w + min(k0 + k, nr - 1) * row_step;
                    const float dv = dsm[(row_base + rl) * p.dstr + kb];
                    f[k] = (active && k0 + k < nr) ? (float)(tot - xs) * (dv * sc) : 0.0f;
                }
                // transposing reduction: lanes with bit 4 keep rows 2, 3, else 0, 1;
                // then bit 3 picks one of the two; then the 8-lane sum
                const bool b4 = (lane & 16) != 0, b3 = (lane & 8) != 0;
                const float r0 = __shfl_xor_sync(0xffffffffu, b4 ? f[0] : f[2], 16);
                const float r1 = __shfl_xor_sync(0xffffffffu, b4 ? f[1] : f[3], 16);
                const float g0 = (b4 ? f[2] : f[0]) + r0, g1 = (b4 ? f[3] : f[1]) + r1;
                const float rr = __shfl_xor_sync(0xffffffffu, b3 ? g0 : g1, 8);
                float hsum = (b3 ? g1 : g0) + rr;
                hsum += __shfl_xor_sync(0xffffffffu, hsum, 4);
                hsum += __shfl_xor_sync(0xffffffffu, hsum, 2);
                hsum += __shfl_xor_sync(0xffffffffu, hsum, 1);
                // this lane now holds row k0 + my_k
                const bool mine = (lane & 7) == 0 && k0 + my_k < nr;
                const int rl = row_w + (k0 + my_k) * row_step;
                if (p.n_kc == 1) {
                    if (mine) red[(row_base + rl) * 2 + grp] = hsum;
                } else {
                    // n_kc > 1: at most 4 rows per warp and stage (k0 == 0)
                    racc += hsum;
                    if (kc == p.n_kc - 1) {
                        if (mine) red[(row_base + rl) * 2 + grp] = racc;
                        racc = 0.0f;
                    }
                }
            }
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(smem_addr(&bars[S + slot]));  // none after a wait ran out
        if (++slot == S) {
            slot = 0;
            phase ^= 1;
        }
        if (++kc == p.n_kc) {
            kc = 0;
            ++rs;
        }
    }
}

// Three pieces (x with outliers): correct but plain -- one row at a time,
// pieces 0, 1 from registers, piece 2 from shared memory.  Kept compact so
// that it does not crowd the instruction cache of the fast paths.
__device__ __noinline__ void consume3(const Dp4Params &p, uint8_t *smem, uint64_t *bars, volatile int *abort_flag,
                                      int nrows, int warp, int lane)
{
    constexpr int P = 3;
    const int S = p.stages;
    const int B = p.B;
    float *red = reinterpret_cast<float *>(smem + p.off_red);
    const float *dsm = reinterpret_cast<const float *>(smem + p.off_dsm);
    const float *binfo = reinterpret_cast<const float *>(smem + p.off_binfo);
    const int *xsq = reinterpret_cast<const int *>(smem + p.off_xsq);
    const uint32_t xq = smem_addr(smem + p.off_xq);
    const uint32_t ring = smem_addr(smem + p.off_ring);
    const int grp = (p.ngrp == 2) ? (warp & 1) : 0;
    const int row_step = kWarps / p.ngrp;
    const int row_w = (p.ngrp == 2) ? (warp >> 1) : warp;
    const int bl = grp * 8 + (lane >> 2), qd = lane & 3;
    const int n_rs = (nrows + p.SR - 1) / p.SR;
    int slot = 0, phase = 0, kc = 0, rs = 0;
    bool alive = true;
    float racc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const int n_stages = n_rs * p.n_kc;
    for (int s = 0; s < n_stages; ++s) {
        bool ok = alive;
        if (ok && !__all_sync(0xffffffffu, mbar_wait(smem_addr(&bars[slot]), (uint32_t)phase))) {
            if (lane == 0) report_timeout(p, abort_flag);
            ok = alive = false;
        }
        if (ok) {
            const int kb0 = kc * p.nbk;
            const int nbk = min(p.nbk, B - kb0);
            const bool active = bl < nbk;
            const int kb = kb0 + (active ? bl : 0);
            const int xs = xsq[kb * 4 + qd];
            const float sc = binfo[kb];
            const int row_base = rs * p.SR;
            const int rows_here = min(p.SR, nrows - row_base);
            const uint32_t st = ring + (uint32_t)(slot * p.stage_bytes) + (uint32_t)(bl * 64 + qd * 16);
            int k = 0;
#pragma unroll 1
            for (int rl = row_w; rl < rows_here; rl += row_step, ++k) {
                float f = 0.0f;
                if (active) {
                    const uint4 wv = lds128(st + (uint32_t)(rl * p.rb));
                    uint32_t a0 = 0, a1 = 0, a2 = 0;
#pragma unroll
                    for (int jw = 0; jw < 4; ++jw) {
                        const uint32_t w = (jw == 0) ? wv.x : (jw == 1) ? wv.y : (jw == 2) ? wv.z : wv.w;
                        const uint4 x0 = lds128(xq + xq_off(kb, qd, 0, jw, P));
                        const uint4 x1 = lds128(xq + xq_off(kb, qd, 1, jw, P));
                        const uint4 x2 = lds128(xq + xq_off(kb, qd, 2, jw, P));
                        const uint32_t c[4] = {w & 0x03030303u, (w >> 2) & 0x03030303u, (w >> 4) & 0x03030303u,
                                               (w >> 6) & 0x03030303u};
                        a0 = dp4a_uu(c[0], x0.x, a0); a0 = dp4a_uu(c[1], x0.y, a0);
                        a0 = dp4a_uu(c[2], x0.z, a0); a0 = dp4a_uu(c[3], x0.w, a0);
                        a1 = dp4a_uu(c[0], x1.x, a1); a1 = dp4a_uu(c[1], x1.y, a1);
                        a1 = dp4a_uu(c[2], x1.z, a1); a1 = dp4a_uu(c[3], x1.w, a1);
                        a2 = dp4a_us(c[0], x2.x, a2); a2 = dp4a_us(c[1], x2.y, a2);
                        a2 = dp4a_us(c[2], x2.z, a2); a2 = dp4a_us(c[3], x2.w, a2);
                    }
                    const int tot = (int)a0 + (int)a1 * 256 + (int)a2 * 65536 - xs;
                    f = (float)tot * (dsm[(row_base + rl) * p.dstr + kb] * sc);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) f += __shfl_xor_sync(0xffffffffu, f, off);
                if (p.n_kc == 1) {
                    if (lane == 0) red[(row_base + rl) * 2 + grp] = f;
                } else {
                    const int kk = k & 3;  // at most 4 rows per warp and stage when n_kc > 1
                    float acc = (kk == 0) ? racc[0] : (kk == 1) ? racc[1] : (kk == 2) ? racc[2] : racc[3];
                    acc += f;
                    if (kc == p.n_kc - 1) {
                        if (lane == 0) red[(row_base + rl) * 2 + grp] = acc;
                        acc = 0.0f;
                    }
                    if (kk == 0) racc[0] = acc;
                    else if (kk == 1) racc[1] = acc;
                    else if (kk == 2) racc[2] = acc;
                    else racc[3] = acc;
                }
            }
        }
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(smem_addr(&bars[S + slot]));  // none after a wait ran out
        if (++slot == S) {
            slot = 0;
            phase ^= 1;
        }
        if (++kc == p.n_kc) {
            kc = 0;
            ++rs;
        }
    }
}

__global__ void __launch_bounds__(kThreads, 2) matvec_dp4_kernel(const __grid_constant__ Dp4Params p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int abort_shared;
    volatile int *abort_flag = &abort_shared;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t N = p.a.N, K = p.a.K;
    const int64_t r0 = (int64_t)blockIdx.x * N / p.G;
    const int64_t r1 = (int64_t)(blockIdx.x + 1) * N / p.G;
    const int nrows = (int)(r1 - r0);
    const int n_rs = (nrows + p.SR - 1) / p.SR;
    const int n_stages = n_rs * p.n_kc;
    const int S = p.stages;
    const int B = p.B;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.off_bar);  // full[S], empty[S]

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
        const int64_t row_bytes = K / 4;
        const uint32_t ring = smem_addr(smem + p.off_ring);
        int issued = 0, kc = 0, rs = 0;
        for (int s = 0; s < n_stages; ++s) {
            const int slot = s % S;
            const int round = s / S;
            if (round > 0 &&
                !__all_sync(0xffffffffu, mbar_wait(smem_addr(&bars[S + slot]), (round - 1) & 1))) {
                if (lane == 0) report_timeout(p, abort_flag);
                break;
            }
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            const int row0 = rs * p.SR;
            const int rows = min(p.SR, nrows - row0);
            const uint32_t full = smem_addr(&bars[slot]);
            const uint32_t dst0 = ring + (uint32_t)(slot * p.stage_bytes);
            if (!p.tma2d) {
                const uint32_t bytes = (uint32_t)rows * (uint32_t)row_bytes;
                if (lane == 0) {
                    mbar_arrive_expect_tx(full, bytes);
                    bulk_g2s(dst0, p.a.qs + (r0 + row0) * row_bytes, bytes, full, pol);
                }
            } else {
                if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)rows * 1024u);
                __syncwarp();
                const int y0 = (int)(r0 + row0);
                const int x = kc * 128;
                if (rows == 16) {
                    if (lane == 0) tensor2d_g2s(dst0, &p.tmap[0], x, y0, full, pol);
                } else {
                    int roff = 0, box = 0;
#pragma unroll
                    for (int i = 1; i < 5; ++i) {
                        const int h = 16 >> i;
                        if (rows & h) {
                            if (lane == box) tensor2d_g2s(dst0 + roff * 1024, &p.tmap[i], x, y0 + roff, full, pol);
                            roff += h;
                            ++box;
                        }
                    }
                }
            }
            __syncwarp();
            issued = s + 1;
            if (++kc == p.n_kc) {
                kc = 0;
                ++rs;
            }
        }
        for (int slot = 0; slot < S && slot < issued; ++slot) {
            const int last = slot + ((issued - 1 - slot) / S) * S;
            if (!mbar_wait(smem_addr(&bars[slot]), (last / S) & 1) && lane == 0) report_timeout(p, abort_flag);
        }
        return;
    }

    // ---------------------------------------------------------- consumer warps
    float *red = reinterpret_cast<float *>(smem + p.off_red);
    float *dsm = reinterpret_cast<float *>(smem + p.off_dsm);
    float *binfo = reinterpret_cast<float *>(smem + p.off_binfo);
    int *xsq = reinterpret_cast<int *>(smem + p.off_xsq);
    int *flag = reinterpret_cast<int *>(smem + p.off_flag);
    const uint32_t xq = smem_addr(smem + p.off_xq);
    const bool prologue = p.a.act_scale != 0.0f;

    if (tid == 0) *flag = 0;
    // d slice (contiguous rows r0..r1), fp32, (row, block) stepped without division
    {
        const int nd = nrows * B;
        const uint16_t *dsrc = p.a.d + r0 * B;
        const int q_step = kConsumers / B, r_step = kConsumers - q_step * B;
        int r = tid / B, b = tid - (tid / B) * B;
        for (int base = 0; base < nd; base += kConsumers * 8) {
            uint16_t v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = base + j * kConsumers + tid;
                v[j] = (i < nd) ? dsrc[i] : (uint16_t)0;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = base + j * kConsumers + tid;
                if (i < nd) dsm[r * p.dstr + b] = __half2float(__ushort_as_half(v[j]));
                r += q_step;
                b += r_step;
                if (b >= B) {
                    b -= B;
                    ++r;
                }
            }
        }
    }

    // x depends on the previous kernel in the stream.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    consumers_sync();  // flag cleared

    // x staging, pass 1: per block (one warp each), lane l holds x[8l .. 8l+7]
    // (as int8 codes with the prologue); block exponent and the 2-piece test.
    constexpr int kMaxBlocksPerWarp = 8;  // K <= 16384 keeps x in registers
    uint4 xv[kMaxBlocksPerWarp];
    int ebits[kMaxBlocksPerWarp];
    const int nbw = (B - warp + kWarps - 1) / kWarps;  // blocks of this warp
#pragma unroll
    for (int i = 0; i < kMaxBlocksPerWarp; ++i)
        if (i < nbw) xv[i] = *reinterpret_cast<const uint4 *>(p.a.x + (int64_t)(warp + i * kWarps) * 256 + 8 * lane);
    int need3 = 0;
#pragma unroll
    for (int i = 0; i < kMaxBlocksPerWarp; ++i) {
        if (i >= nbw) break;
        uint32_t r[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
        if (prologue) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&r[q]));
                const __half2 c2 = __floats2half2_rn(fq_code(f.x, p.a.inv_scale), fq_code(f.y, p.a.inv_scale));
                r[q] = *reinterpret_cast<const uint32_t *>(&c2);
            }
            xv[i] = make_uint4(r[0], r[1], r[2], r[3]);
            ebits[i] = 0;
            continue;
        }
        uint32_t mb = 0;
        float sa = 0.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            mb = max(mb, max(r[q] & 0x7FFFu, (r[q] >> 16) & 0x7FFFu));
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&r[q]));
            sa += fabsf(f.x) + fabsf(f.y);
        }
        mb = __reduce_max_sync(0xffffffffu, mb);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sa += __shfl_xor_sync(0xffffffffu, sa, off);
        // exponent of the largest |x|: normal (mb >> 10) - 15, subnormal from the leading bit
        const int E = (mb >= 0x400u) ? (int)(mb >> 10) - 15 : (mb ? (31 - __clz((int)mb)) - 24 : -200);
        ebits[i] = E;
        // two pieces when 256 * 2^(E - 15) <= 0.5e-3 * sum|x|
        if (mb && pow2f(max(E - 7, -126)) > 5.0e-4f * sa) need3 = 1;
    }
    if (__any_sync(0xffffffffu, need3) && lane == 0) atomicOr(flag, 1);
    consumers_sync();
    const int P = prologue ? 1 : (*flag ? 3 : 2);

    // pass 2: integers, pieces and per-class byte layout
    const int h = lane & 1, wd = lane >> 1, qd = wd >> 2, jw = wd & 3;
#pragma unroll
    for (int i = 0; i < kMaxBlocksPerWarp; ++i) {
        if (i >= nbw) break;
        const int b = warp + i * kWarps;
        const uint32_t r[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
        int X[8];
        int Sb = 0;
        if (prologue) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&r[q]));
                X[2 * q] = (int)f.x;
                X[2 * q + 1] = (int)f.y;
            }
        } else {
            const int E = ebits[i];
            Sb = (E <= -200) ? 0 : ((P == 2) ? 14 - E : 21 - E);
            const float sc = pow2f(min(max(Sb, -126), 127));
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&r[q]));
                X[2 * q] = rint_small(f.x * sc);
                X[2 * q + 1] = rint_small(f.y * sc);
            }
        }
        // quarter sum of X (lanes 8qd .. 8qd+7)
        int xsum = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) xsum += X[j];
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) xsum += __shfl_xor_sync(0xffffffffu, xsum, off);
        if ((lane & 7) == 0) xsq[b * 4 + qd] = xsum;
        if (lane == 0) binfo[b] = pow2f(min(max(-Sb, -126), 127));
        // piece bytes: lane holds positions 8h + j, j = 0..7 -> byte index 2h + (j >> 2), class j & 3
#pragma unroll
        for (int pc = 0; pc < kMaxP; ++pc) {
            if (pc >= P) break;
            uint32_t mine[4];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int v0 = (P == 1) ? X[c] : ((pc == P - 1) ? (X[c] >> (8 * pc)) : ((X[c] >> (8 * pc)) & 0xFF));
                const int v1 = (P == 1) ? X[4 + c] : ((pc == P - 1) ? (X[4 + c] >> (8 * pc)) : ((X[4 + c] >> (8 * pc)) & 0xFF));
                mine[c] = ((uint32_t)v0 & 0xFFu) | (((uint32_t)v1 & 0xFFu) << 8);
            }
            // lane h=0 writes classes 0, 1 needs partner's (bytes 2, 3) of them; h=1 writes 2, 3
            const uint32_t send0 = h ? mine[0] : mine[2], send1 = h ? mine[1] : mine[3];
            const uint32_t recv0 = __shfl_xor_sync(0xffffffffu, send0, 1);
            const uint32_t recv1 = __shfl_xor_sync(0xffffffffu, send1, 1);
            const uint32_t own0 = h ? mine[2] : mine[0], own1 = h ? mine[3] : mine[1];
            // full class word: bytes (0, 1) from the h = 0 lane, (2, 3) from the h = 1 lane
            const uint32_t w0 = h ? (recv0 | (own0 << 16)) : (own0 | (recv0 << 16));
            const uint32_t w1 = h ? (recv1 | (own1 << 16)) : (own1 | (recv1 << 16));
            const uint32_t dst = xq + xq_off(b, qd, pc, jw, P) + (uint32_t)(h * 8);
            asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(dst), "r"(w0), "r"(w1) : "memory");
        }
    }
    consumers_sync();

    if (P == 1) consume<1>(p, smem, bars, abort_flag, nrows, warp, lane);
    else if (P == 2) consume<2>(p, smem, bars, abort_flag, nrows, warp, lane);
    else consume3(p, smem, bars, abort_flag, nrows, warp, lane);

    consumers_sync();
    if (*abort_flag) return;  // y is invalid; TQ2_FLAG_TIMEOUT was reported
    for (int r = tid; r < nrows; r += kConsumers) {
        float s = red[r * 2];
        if (p.ngrp == 2) s += red[r * 2 + 1];
        if (prologue) s *= p.a.act_scale;
        s = requant_out(s, p.a.out_scale, p.a.inv_out);
        if (p.a.y_f16)
            reinterpret_cast<__half *>(p.a.y)[r0 + r] = __float2half_rn(s);
        else
            reinterpret_cast<float *>(p.a.y)[r0 + r] = s;
    }
}

// ------------------------------------------------------------------ host side
int align_up(int v, int a) { return (v + a - 1) / a * a; }

bool make_plan(int64_t N, int64_t K, int G, int cap, Dp4Params &p)
{
    const int64_t B = K / 256;
    if (B < 1 || B > 64) return false;  // x staging keeps <= 8 blocks per warp in registers
    p.G = G;
    p.B = (int)B;
    const int64_t max_rows = (N + G - 1) / G;
    p.max_rows = (int)max_rows;
    if (B <= 16) {
        p.tma2d = 0;
        p.nbk = (int)B;
        p.n_kc = 1;
        p.SR = (int)(65536 / K);  // 16 KB of whole rows
        p.rb = (int)(K / 4);
    } else {
        p.tma2d = 1;
        p.nbk = 16;
        p.n_kc = (int)((B + 15) / 16);
        p.SR = 16;
        p.rb = 1024;
    }
    if (p.SR > max_rows) p.SR = (int)max_rows;
    p.ngrp = (p.nbk > 8) ? 2 : 1;
    if (p.n_kc > 1 && p.SR / (kWarps / p.ngrp) > 4) return false;  // racc holds 4 rows per warp
    p.stage_bytes = p.SR * p.rb;
    p.dstr = (int)B + 1;
    int64_t off = 2 * kMaxStages * 8;
    p.off_bar = 0;
    p.off_red = (int)off;
    off += align_up((int)max_rows * 2 * 4, 16);
    p.off_dsm = (int)off;
    off += (int64_t)max_rows * p.dstr * 4;
    off = (off + 15) / 16 * 16;
    p.off_binfo = (int)off;
    off += align_up((int)B * 4, 16);
    p.off_xsq = (int)off;
    off += B * 16;
    p.off_flag = (int)off;
    off += 16;
    p.off_xq = (int)off;
    off += (int64_t)((B + 7) / 8 * 8) * 256 * kMaxP;
    off = (off + 127) / 128 * 128;
    p.off_ring = (int)off;
    if (off + 2 * (int64_t)p.stage_bytes > cap) return false;
    int S = (int)((cap - off) / p.stage_bytes);
    if (S > kMaxStages) S = kMaxStages;
    p.stages = S;
    p.smem_total = (int)off + S * p.stage_bytes;
    return true;
}

std::atomic<int> g_max_dyn[64];

int max_dynamic_smem(int device)
{
    if (device < 0 || device >= 64) return 0;
    int v = g_max_dyn[device].load();
    if (v > 0) return v;
    int optin = 0;
    cudaFuncAttributes fa;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, matvec_dp4_kernel) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    v = optin - (int)fa.sharedSizeBytes;
    if (cudaFuncSetAttribute(matvec_dp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, v) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    g_max_dyn[device].store(v);
    return v;
}

bool plan_for(int64_t N, int64_t K, int device, Dp4Params &p)
{
    const int max_dyn = max_dynamic_smem(device);
    if (max_dyn <= 0) return false;
    const int nsm = sm_count(device);
    int G = (int)((N < (int64_t)nsm) ? N : nsm);
    for (;;) {
        for (int cap : {kTwoPerSm, max_dyn}) {
            if (cap > max_dyn) continue;
            if (make_plan(N, K, G, cap, p)) return true;
        }
        if (G >= N) return false;
        G = (int)((2 * (int64_t)G < N) ? 2 * G : N);
    }
}

cudaError_t encode_maps(const MatvecArgs &a, Dp4Params &p)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)(a.K / 32), (cuuint64_t)a.N};
    const cuuint64_t strides[1] = {(cuuint64_t)(a.K / 4)};
    const cuuint32_t estr[2] = {1, 1};
    for (int i = 0; i < 5; ++i) {
        const cuuint32_t box[2] = {128, (cuuint32_t)(16 >> i)};
        CUresult r = enc(&p.tmap[i], CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint8_t *>(a.qs), dims, strides,
                         box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

}  // namespace

bool dp4_matvec_supported(int M, int64_t N, int64_t K, int device)
{
    if (M != 1 || N < 1 || K < 256) return false;
    Dp4Params p{};
    return plan_for(N, K, device, p);
}

cudaError_t launch_matvec_dp4(const MatvecArgs &a, int device)
{
    if (a.M != 1) return cudaErrorInvalidValue;
    Dp4Params p{};
    p.a = a;
    if (!plan_for(a.N, a.K, device, p)) return cudaErrorInvalidConfiguration;
    if (p.tma2d) {
        cudaError_t e = encode_maps(a, p);
        if (e != cudaSuccess) return e;
    }
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
    return cudaLaunchKernelEx(&cfg, matvec_dp4_kernel, p);
}

}  // namespace tq2
