// tq2_matvec_mma.cu -- tensor-core ternary matvec for M <= 2 (sm_103a).
//
// What it computes (BitCPM ternary page, linear-factoring paragraph):
//   y[m][n] = sum_b d[n][b] * sum_{k in b} x'[m][k] * (q[n][k] - 1)
// with one multiply by d_b per block partial and adds/subtracts only inside
// a block.  The page's Metal kernel does the block sums on SIMD lanes; here
// the adds are issued to the tensor pipe so that unpacking stays near one
// integer instruction per two codes (the custom-Metal-kernels page notes that
// unpack ALU, not memory, capped its "memory-bound" int4 matvec).
//
// Data path per CTA (one CTA owns a contiguous range of output rows, all K):
//   * a producer warp streams the CTA's packed rows into a shared-memory ring
//     of 16 KB stages with TMA, L2 evict-first: for K <= 4096 a stage is whole
//     rows, contiguous in memory, fetched with one 1-D bulk copy
//     (cp.async.bulk); for K > 4096 a stage is 16 rows x 4096 codes, fetched
//     with one 2-D tensor copy of a 16-row box (8/4/2/1-row boxes for the
//     CTA's last rows, so no other CTA's rows are read).  TMA throughput on
//     this part scales with the size of each copy (1 KB copies cap a CTA at a
//     few GB/s), hence one large copy per stage.  The producer starts before
//     the kernel waits on the previous grid (programmatic dependent launch),
//     because weights never depend on earlier kernels;
//   * the d slice of the CTA's rows is staged to shared memory as fp32;
//   * after griddepcontrol.wait, x (or its int8 fake-quant codes) is staged
//     to shared memory in MMA-fragment order, with per-block sums X_b;
//   * 8 consumer warps take (16-row group, 256-block) units of each stage.
//
// The unpack.  A packed 32-bit word holds 16 codes of one row; code j of the
// low half sits at bits 2j, code 8+j at bits 16+2j.  ANDing the word with
// 0x00030003 << 2c keeps codes c and 8+c as two fp16 lanes whose bit patterns
// are q*4^c; bit patterns below 2048 are the fp16 values pattern*2^-24
// (subnormal/first binade), so each lane is exactly q * 2^(2c-24).  The same
// on (word >> 8) keeps codes 4+c and 12+c.  One LOP3 per two codes, no
// conversion.  The four "classes" c carry different powers of two, so each
// class gets its own accumulator, and the B operand places x values of class
// c in column c (columns 4..7 hold the second activation row when M == 2).
// Column c of accumulator c is exact: sum_k q_k x_k * 2^(2c-24); the other
// columns are ignored.  Subtracting sum_k x_k (the "-1" of q-1) is folded into
// the class-0 accumulator's initial value, -X_b * 2^-24.  Per block, each
// class result is scaled by d_b (one FMA per class and row); at the end the
// classes are combined with their powers of two.  Every step is exact except
// fp32 accumulation, far inside the 1e-3 * sum|d x| tolerance.
//
// Layout of one 16-row A tile: mma row g <- smem row g, row g+8 <- g+8, rows
// dense in shared memory as TMA writes them.
#include <cuda.h>
#include <cuda_fp16.h>

#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>

#include "tq2_device.cuh"
#include "tq2_internal.cuh"

#ifdef TQ2_TRACE
namespace tq2 {
namespace dev {
__device__ unsigned long long g_trace[2][kTraceCtas][kTracePhases];
}  // namespace dev
}  // namespace tq2
#endif

namespace tq2 {
namespace {

using namespace dev;

#ifndef TQ2_MMA_WARPS
#define TQ2_MMA_WARPS 8
#endif
constexpr int kConsumerWarps = TQ2_MMA_WARPS;
constexpr int kUpw = 16 / kConsumerWarps;           // fast path: 256-blocks per warp and stage
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kMmaThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kChunkBlocks = 16;                    // 256-blocks per stage row (4096 codes)
constexpr int kTargetSmem = 112 * 1024;             // two CTAs per SM (PDL overlap)

// One weight matrix of a launch.  A single call has one; a grouped call
// (several matrices sharing x) gives each matrix a contiguous range of CTAs
// [g0, g0 + G) in proportion to its rows, and its own output scale.
constexpr int kMaxGroup = 4;
struct GroupMat {
    const uint8_t *qs;   // [N, K/4]
    const uint16_t *d;   // [N, K/256]
    void *y;             // [M, N]
    int64_t N;
    int g0, G;
    float out_scale;     // 0: y as computed; else requantised at store
    float inv_out;       // fp32(1/out_scale)
};

// The launch plan: arguments, grid and shared-memory layout.
struct MmaPlan {
    MatvecArgs a;
    int tma2d;       // 0: 1-D bulk copies of whole rows; 1: 2-D tensor boxes
    int G;           // CTAs; CTA i owns rows [i*N/G, (i+1)*N/G)
    int B;           // 256-blocks per row
    int nbk_full;    // 256-blocks per stage row
    int n_kc;        // stages per row-group along K
    int rg_s;        // 16-row groups per stage
    int rb;          // smem row stride of a stage (bytes)
    int stage_bytes;
    int stages;      // ring depth
    int max_rg;      // 16-row groups per CTA (max)
    int dstr;        // fp32 stride of the d slice rows (B + 1, odd)
    int off_bar, off_red, off_dsm, off_xsum, off_xs, off_ring, smem_total;
    int n_mats;
    int seq;         // launch sequence number (the trace build's slot parity)
};

// Kernel parameters for up to kG matrices with kT sets of tensor maps (1, or
// kG for a group at K > 4096): every launch copies its parameters, so a
// single call carries one matrix and a group without 2-D boxes one map set.
template <int kG, int kT>
struct MmaParams : MmaPlan {
    // K > 4096 only: each matrix's qs as a 2-D tensor of uint64 [N][K/32],
    // boxes of 128 x {16, 8, 4, 2, 1} rows
    CUtensorMap tmap[kT][5];  // 64-byte aligned by its type
    GroupMat mats[kG];
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ void consumer_barrier()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

// One class c of one 16-code word pair: A lanes are q * 4^c * 2^-24.
#define TQ2_MMA_CLASS(FIRST, C, MASK, CINIT)                                                   \
    do {                                                                                       \
        if (FIRST)                                                                             \
            mma_16816_init(C, w0 & (MASK), w1 & (MASK), s0 & (MASK), s1 & (MASK), b0, b1, CINIT); \
        else                                                                                   \
            mma_16816(C, w0 & (MASK), w1 & (MASK), s0 & (MASK), s1 & (MASK), b0, b1);          \
    } while (0)

__device__ __forceinline__ void report_timeout(const MmaPlan &p, volatile int *abort_flag)
{
    *abort_flag = 1;
    if (p.a.status) atomicOr(p.a.status, TQ2_FLAG_TIMEOUT);
}

// ------------------------------------------------------------------ kernel
// kHook: the test instantiation (a per-call wait limit and a stage whose copy
// the producer skips, MatvecArgs::wait_limit_ns / stall_stage); product
// launches use kHook = false, with the constant limit and no stall check.
template <int kM, int kG, int kT, bool kHook>
__global__ void __launch_bounds__(kMmaThreads, 2)
matvec_mma_kernel(const __grid_constant__ MmaParams<kG, kT> p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int abort_shared;
    volatile int *abort_flag = &abort_shared;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
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
    const int n_stages = ((nrg + p.rg_s - 1) / p.rg_s) * p.n_kc;
    const int S = p.stages;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.off_bar);  // full[S], empty[S]
    uint8_t *ring = smem + p.off_ring;
    uint32_t *const st_w = p.a.status;  // TQ2_FLAG_BOUNDS of debug builds
    const SmemWindow win{smem_addr(smem), smem_addr(smem) + (uint32_t)p.smem_total, st_w};
    const uint32_t ring_end = smem_addr(ring) + (uint32_t)(S * p.stage_bytes);
    const unsigned long long lim = (kHook && p.a.wait_limit_ns) ? p.a.wait_limit_ns : kTimeoutNs;

    if (tid == 0) TQ2_STAMP(p.seq, 0);
    // Let the next kernel in the stream start its own weight prefetch.
    asm volatile("griddepcontrol.launch_dependents;");

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_addr(&bars[s]), 1);
            mbar_init(smem_addr(&bars[S + s]), kConsumerWarps);
        }
        abort_shared = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------ producer warp
        const uint64_t pol = evict_first_policy();
        const int64_t row_bytes = K / 4;
        int issued = 0;
        for (int s = 0; s < n_stages; ++s) {
            const int slot = s % S;
            const int round = s / S;
            // every lane waits (acquire); the decision is made warp-uniform
            if (round > 0 &&
                !__all_sync(0xffffffffu, mbar_wait_for(smem_addr(&bars[S + slot]), (round - 1) & 1, lim))) {
                if (lane == 0) report_timeout(p, abort_flag);
                break;
            }
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            if (kHook && s == p.a.stall_stage) {  // test hook: no copy for this stage
                issued = s + 1;
                continue;
            }
            const int rgb = s / p.n_kc, kc = s % p.n_kc;
            const int rg0 = rgb * p.rg_s;
            const int rows = min(p.rg_s * 16, nrows - rg0 * 16);
            const uint32_t full = smem_addr(&bars[slot]);
            const uint32_t dst0 = smem_addr(ring + (size_t)slot * p.stage_bytes);
            if (!p.tma2d) {
                // whole rows [rg0*16, rg0*16 + rows): one contiguous copy
                const uint32_t bytes = (uint32_t)rows * (uint32_t)row_bytes;
                if (lane == 0 && TQ2_IN((r0 + rg0 * 16) * row_bytes + bytes <= N * row_bytes && dst0 + bytes <= ring_end,
                                        st_w)) {
                    mbar_arrive_expect_tx(full, bytes);
                    bulk_g2s(dst0, qs_g + (r0 + rg0 * 16) * row_bytes, bytes, full, pol);
                }
            } else {
                // 16 rows x 1024 bytes (columns past the row end read as zero);
                // a partial group is split into boxes of 8, 4, 2, 1 rows
                const bool in = TQ2_IN(dst0 + (uint32_t)rows * 1024u <= ring_end, st_w);
                if (lane == 0 && in) mbar_arrive_expect_tx(full, (uint32_t)rows * 1024u);
                __syncwarp();
                const int y0 = (int)(r0 + rg0 * 16);
                const int x = kc * 128;
                if (!in) {
                } else if (rows == 16) {
                    if (lane == 0) tensor2d_g2s(dst0, &p.tmap[kT > 1 ? mi : 0][0], x, y0, full, pol);
                } else {
                    int roff = 0, box = 0;
#pragma unroll
                    for (int i = 1; i < 5; ++i) {
                        const int h = 16 >> i;
                        if (rows & h) {
                            if (lane == box)
                                tensor2d_g2s(dst0 + roff * 1024, &p.tmap[kT > 1 ? mi : 0][i], x, y0 + roff, full, pol);
                            roff += h;
                            ++box;
                        }
                    }
                }
            }
            __syncwarp();
            issued = s + 1;
        }
        if (lane == 0) TQ2_STAMP(p.seq, 6);
        // No copy may still be writing shared memory when the CTA exits.
        // (Slots are refilled only after every consumer has waited for and
        // read the previous stage, so the last copy of a slot is the only one
        // that can be in flight; a skipped stage had none: its slot's last
        // copy is the one before it.)
        for (int slot = 0; slot < S && slot < issued; ++slot) {
            int last = slot + ((issued - 1 - slot) / S) * S;
            if (kHook && last == p.a.stall_stage) last -= S;
            if (last >= 0 && !mbar_wait_for(smem_addr(&bars[slot]), (last / S) & 1, lim) && lane == 0)
                report_timeout(p, abort_flag);
        }
        return;
    }

    // ---------------------------------------------------------- consumer warps
    float *red = reinterpret_cast<float *>(smem + p.off_red);
    float *dsm = reinterpret_cast<float *>(smem + p.off_dsm);
    float *xsum = reinterpret_cast<float *>(smem + p.off_xsum);
    uint8_t *xs = smem + p.off_xs;
    const int B = p.B;
    const bool prologue = p.a.act_scale != 0.0f;
    const bool convert = prologue && !p.a.x_codes;  // x holds fp16 values, not yet codes

    // zero this warp's slots of the cross-warp partial sums
    for (int i = lane; i < nrg * kM * 16; i += 32) {
        const int rg = i / (kM * 16), rest = i - rg * (kM * 16);
        const int ri = (rg * kConsumerWarps + warp) * kM * 16 + rest;
        if (TQ2_IN(ri < p.max_rg * kConsumerWarps * kM * 16, st_w)) red[ri] = 0.0f;
    }
    // d slice of this CTA's rows (contiguous in memory), fp32.  All loads of
    // a batch are issued before the first store so their latencies overlap;
    // element i = tid + 256 j sits at (row, block) stepped without division.
    {
        const int nd = nrows * B;
        const uint16_t *dsrc = d_g + r0 * B;
        const int q_step = kConsumerThreads / B, r_step = kConsumerThreads - q_step * B;
        int r = tid / B, b = tid - (tid / B) * B;
        for (int base = 0; base < nd; base += kConsumerThreads * 8) {
            uint16_t v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = base + j * kConsumerThreads + tid;
                v[j] = (i < nd && TQ2_IN(r0 * B + i < N * B, st_w)) ? dsrc[i] : (uint16_t)0;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = base + j * kConsumerThreads + tid;
                if (i < nd && TQ2_IN(r * p.dstr + b < p.max_rg * 16 * p.dstr, st_w))
                    dsm[r * p.dstr + b] = __half2float(__ushort_as_half(v[j]));
                r += q_step;
                b += r_step;
                if (b >= B) {
                    b -= B;
                    ++r;
                }
            }
        }
    }

    const int g = lane >> 2, t = lane & 3;
    const int gg = g % (4 * kM);          // x-fragment column this thread supplies
    const int mcol = (kM == 2) ? (t >> 1) : 0;  // activation row of columns 2t, 2t+1
    // per-thread shared-memory byte offsets, hoisted out of the loops
    const uint32_t a_thr = smem_addr(ring) + (uint32_t)(g * p.rb + t * 16);
    const uint32_t a_half = (uint32_t)(8 * p.rb);             // row g -> row g + 8
    const uint32_t x_thr = smem_addr(xs) + (uint32_t)(gg * 64 + t * 16);
    const uint32_t x_blk = 512u * kM;                          // per 256-block
    const uint32_t x_half = 256u * kM;                         // words 0,1 -> 2,3
    const uint32_t d_thr = smem_addr(dsm) + (uint32_t)(g * p.dstr) * 4u;
    const uint32_t d_half = (uint32_t)(8 * p.dstr) * 4u;
    const uint32_t xs_thr = smem_addr(xsum) + (uint32_t)mcol * 4u;
    const uint32_t rg_stride_d = (uint32_t)(16 * p.dstr) * 4u;

    // K = 4096 fast path (below): this warp's codes and scales of a stage
    // in registers.  Stage 0's codes are read before the wait on the
    // previous kernel -- the weights never depend on it, and the warps would
    // only idle there -- so that the first MMAs issue as soon as x is staged.
    const bool fast = p.n_kc == 1 && p.rg_s == 1 && p.nbk_full == kUpw * kConsumerWarps;
    const uint32_t a_warp = a_thr + (uint32_t)(warp * 64);
    const uint32_t d_warp = d_thr + (uint32_t)(warp * 4);
    uint32_t W0[kUpw][4], W1[kUpw][4];
    float dg[kUpw], dg8[kUpw];
    auto load_codes = [&](int sl) {
#pragma unroll
        for (int u = 0; u < kUpw; ++u) {
            const uint32_t pa = a_warp + (uint32_t)(sl * p.stage_bytes + u * kConsumerWarps * 64);
            const uint4 wa = lds128_c(win, pa), wb = lds128_c(win, pa + a_half);
            W0[u][0] = wa.x; W0[u][1] = wa.y; W0[u][2] = wa.z; W0[u][3] = wa.w;
            W1[u][0] = wb.x; W1[u][1] = wb.y; W1[u][2] = wb.z; W1[u][3] = wb.w;
        }
    };
    auto load_scales = [&](int rg) {
#pragma unroll
        for (int u = 0; u < kUpw; ++u) {
            const uint32_t pd = d_warp + (uint32_t)rg * rg_stride_d + (uint32_t)(u * kConsumerWarps * 4);
            dg[u] = lds_f32_c(win, pd);
            dg8[u] = lds_f32_c(win, pd + d_half);
        }
    };
    bool fast_ok = false;
    if (fast) {
        fast_ok = n_stages > 0;
        if (fast_ok && !__all_sync(0xffffffffu, mbar_wait_for(smem_addr(&bars[0]), 0u, lim))) {
            if (lane == 0) report_timeout(p, abort_flag);
            fast_ok = false;
        }
        if (fast_ok) load_codes(0);
    }

    // x depends on the previous kernel in the stream.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0) TQ2_STAMP(p.seq, 1);

    // x -> fragment order.  Entry (block b, half h, column cc = 4m + c, t)
    // is 16 bytes = words 2h and 2h+1 of the t-th quarter of the block, each
    // as (x[c], x[8+c], x[4+c], x[12+c]) of that 16-code word.
    // K <= 4096 (one 4096-code chunk): a single pass, thread tid taking word
    // tid of each activation row, so a half-warp's 16 words are one block,
    // summed by a shuffle tree (with its bounds known the pass schedules
    // better than the general loop: q/o 3.07 -> 2.94-2.97 us, gate/up
    // 6.40 -> 6.24-6.31 us).  Longer K: every word of all chunks, the loads of a batch of words
    // in flight together (staging chunks later, inside the stage loop, was
    // slower: down 8.19 -> 9.29 us).
    static_assert(kConsumerThreads == 16 * kChunkBlocks, "one 16-code word of a chunk per consumer thread");
    auto x_src = [&](int c, int m) {
        return p.a.x + (int64_t)m * K + (int64_t)c * (256 * kChunkBlocks) + tid * 16;
    };
    auto x_store = [&](int c) {
        const int nw = min(kChunkBlocks, B - kChunkBlocks * c) * 16;
        uint4 xpre[kM][2];
#pragma unroll
        for (int m = 0; m < kM; ++m) {
            if (tid < nw && TQ2_IN((int64_t)m * K + (int64_t)c * (256 * kChunkBlocks) + tid * 16 + 16 <= kM * K, st_w)) {
                xpre[m][0] = *reinterpret_cast<const uint4 *>(x_src(c, m));
                xpre[m][1] = *reinterpret_cast<const uint4 *>(x_src(c, m) + 8);
            } else {
                xpre[m][0] = xpre[m][1] = make_uint4(0, 0, 0, 0);
            }
        }
        const int rem = c * (16 * kChunkBlocks) + tid;  // word of the row
        const int b = rem >> 4, wib = rem & 15;
        const int t4 = wib >> 2, i4 = wib & 3;
        float sum[kM];
#pragma unroll
        for (int m = 0; m < kM; ++m) {
            sum[m] = 0.0f;
            if (tid < nw) {
                uint32_t raw[8] = {xpre[m][0].x, xpre[m][0].y, xpre[m][0].z, xpre[m][0].w,
                                   xpre[m][1].x, xpre[m][1].y, xpre[m][1].z, xpre[m][1].w};
                if (convert) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&raw[q]));
                        const __half2 h2 = __floats2half2_rn(fq_code(f.x, p.a.inv_scale),
                                                             fq_code(f.y, p.a.inv_scale));  // exact
                        raw[q] = *reinterpret_cast<const uint32_t *>(&h2);
                    }
                }
                float s2[2] = {0.0f, 0.0f};
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&raw[q]));
                    s2[q & 1] += f.x + f.y;
                }
                sum[m] = s2[0] + s2[1];
                const uint32_t dst = smem_addr(xs) + (uint32_t)(b * 512 * kM + (i4 >> 1) * (4 * kM * 64) +
                                                              t4 * 16 + (i4 & 1) * 8 + m * 4 * 64);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    // (x[c], x[8+c]) and (x[4+c], x[12+c]): halves (c & 1) of the raw words
                    const uint32_t sel = (cc & 1) ? 0x7632u : 0x5410u;
                    const uint32_t lo = __byte_perm(raw[cc >> 1], raw[4 + (cc >> 1)], sel);
                    const uint32_t hi = __byte_perm(raw[2 + (cc >> 1)], raw[6 + (cc >> 1)], sel);
                    if (TQ2_IN(dst + (uint32_t)(cc * 64) + 8u <= smem_addr(xs) + (uint32_t)(B * 512 * kM), st_w))
                    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(dst + (uint32_t)(cc * 64)), "r"(lo),
                                 "r"(hi)
                                 : "memory");
                }
            }
        }
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) {
#pragma unroll
            for (int m = 0; m < kM; ++m) sum[m] += __shfl_xor_sync(0xffffffffu, sum[m], off);
        }
#pragma unroll
        for (int m = 0; m < kM; ++m)
            if (tid < nw && (lane & 15) == 0 && TQ2_IN(b * kM + m < B * kM, st_w)) xsum[b * kM + m] = sum[m];
    };
    if (p.n_kc == 1) {
        x_store(0);
    } else
    {
        // 16-code words of x; a thread takes words L = base0 + j*256 + lane
        // (j < 4) and issues the loads of all four before using any.
        constexpr int kXBatch = (kConsumerWarps >= 16) ? 2 : 4;
        const int total = kM * B * 16;
        for (int base0 = warp * 32; base0 < total; base0 += kConsumerThreads * kXBatch) {
          uint4 xv[kXBatch][2];
#pragma unroll
          for (int j = 0; j < kXBatch; ++j) {
              const int L = base0 + j * kConsumerThreads + lane;
              if (L < total) {
                  const int m = (kM == 2 && L >= B * 16) ? 1 : 0;  // kM <= 2: no division
                  const int rem = L - m * B * 16;
                  const uint16_t *src = p.a.x + (int64_t)m * K + (int64_t)(rem >> 4) * 256 + (rem & 15) * 16;
                  if (!TQ2_IN(src + 16 <= p.a.x + kM * K, st_w)) src = p.a.x;
                  xv[j][0] = *reinterpret_cast<const uint4 *>(src);
                  xv[j][1] = *reinterpret_cast<const uint4 *>(src + 8);
              }
          }
          // per-thread partial sums of the batch first, then all four
          // half-warp reductions together (their shuffle latencies overlap)
          float sum[kXBatch];
          int bm[kXBatch];
#pragma unroll
          for (int j = 0; j < kXBatch; ++j) {
            const int L = base0 + j * kConsumerThreads + lane;
            const bool act = L < total;  // uniform over each half-warp (total % 16 == 0)
            sum[j] = 0.0f;
            bm[j] = -1;
            if (act) {
                const int m = (kM == 2 && L >= B * 16) ? 1 : 0;
                const int rem = L - m * B * 16;
                const int b = rem >> 4, wib = rem & 15;
                bm[j] = b * kM + m;
                uint32_t raw[8] = {xv[j][0].x, xv[j][0].y, xv[j][0].z, xv[j][0].w,
                                   xv[j][1].x, xv[j][1].y, xv[j][1].z, xv[j][1].w};
                if (convert) {
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&raw[q]));
                        const __half2 h2 = __floats2half2_rn(fq_code(f.x, p.a.inv_scale),
                                                             fq_code(f.y, p.a.inv_scale));  // exact
                        raw[q] = *reinterpret_cast<const uint32_t *>(&h2);
                    }
                }
                float s2[2] = {0.0f, 0.0f};
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&raw[q]));
                    s2[q & 1] += f.x + f.y;
                }
                sum[j] = s2[0] + s2[1];
                const int t4 = wib >> 2, i4 = wib & 3;
                const uint32_t dst = smem_addr(xs) + (uint32_t)(b * 512 * kM + (i4 >> 1) * (4 * kM * 64) +
                                                              t4 * 16 + (i4 & 1) * 8 + m * 4 * 64);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    // (x[c], x[8+c]) and (x[4+c], x[12+c]): halves (c & 1) of the raw words
                    const uint32_t sel = (c & 1) ? 0x7632u : 0x5410u;
                    const uint32_t lo = __byte_perm(raw[c >> 1], raw[4 + (c >> 1)], sel);
                    const uint32_t hi = __byte_perm(raw[2 + (c >> 1)], raw[6 + (c >> 1)], sel);
                    if (TQ2_IN(dst + (uint32_t)(c * 64) + 8u <= smem_addr(xs) + (uint32_t)(B * 512 * kM), st_w))
                    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(dst + (uint32_t)(c * 64)), "r"(lo),
                                 "r"(hi)
                                 : "memory");
                }
            }
          }
#pragma unroll
          for (int off = 8; off > 0; off >>= 1) {
#pragma unroll
            for (int j = 0; j < kXBatch; ++j) sum[j] += __shfl_xor_sync(0xffffffffu, sum[j], off);
          }
#pragma unroll
          for (int j = 0; j < kXBatch; ++j)
            if (bm[j] >= 0 && (lane & 15) == 0 && TQ2_IN(bm[j] < B * kM, st_w)) xsum[bm[j]] = sum[j];
        }
    }
    consumer_barrier();
    if (tid == 0) TQ2_STAMP(p.seq, 2);

    float acc[4][2];
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[c][0] = acc[c][1] = 0.0f;
    int cur_rg = -1;

    auto flush = [&](int rg) {
        float vg = (t & 1) ? (acc[2][0] * 1048576.0f + acc[3][0] * 262144.0f)
                           : (acc[0][0] * 16777216.0f + acc[1][0] * 4194304.0f);
        float vg8 = (t & 1) ? (acc[2][1] * 1048576.0f + acc[3][1] * 262144.0f)
                            : (acc[0][1] * 16777216.0f + acc[1][1] * 4194304.0f);
        vg += __shfl_xor_sync(0xffffffffu, vg, 1);
        vg8 += __shfl_xor_sync(0xffffffffu, vg8, 1);
        if ((t & 1) == 0 && (t >> 1) < kM) {
            float *rp = red + ((rg * kConsumerWarps + warp) * kM + (t >> 1)) * 16;
            if (TQ2_IN(((rg * kConsumerWarps + warp) * kM + (t >> 1) + 1) * 16 <= p.max_rg * kConsumerWarps * kM * 16,
                       st_w)) {
                rp[g] = vg;
                rp[g + 8] = vg8;
            }
        }
    };

    if (fast) {
        // K = 4096: every stage is one 16-row group, all 16 blocks.  This
        // warp takes blocks warp + u * kConsumerWarps of every stage, so their
        // x sums stay in registers.  The next stage's codes are read as soon
        // as this stage's are in MMA operands: their latency overlaps the
        // MMAs draining and the scaled sums.
        float xi[kUpw];
#pragma unroll
        for (int u = 0; u < kUpw; ++u)
            xi[u] = -lds_f32_c(win, xs_thr + (uint32_t)(warp + u * kConsumerWarps) * (4u * kM)) * 5.9604644775390625e-08f;
        const uint32_t x_warp = x_thr + (uint32_t)warp * x_blk;
        int sl = 0, ph = 0;
        bool ok = fast_ok;  // stage 0's codes are in registers already
        if (ok) load_scales(0);
        if (tid == 0) TQ2_STAMP(p.seq, 3);
        for (int s = 0; ok && s < n_stages; ++s) {
            // unit by unit: four class accumulators starting at zero, then
            // their scaled sums (the "-1" of q - 1 enters as d_b * (-X_b *
            // 2^-24) on class 0); the next stage's codes are read once this
            // stage's are all in MMA operands
            const int nsl = (sl + 1 == S) ? 0 : sl + 1;
            const int nph = (sl + 1 == S) ? (ph ^ 1) : ph;
#pragma unroll
            for (int u = 0; u < kUpw; ++u) {
                const uint32_t px = x_warp + (uint32_t)(u * kConsumerWarps) * x_blk;
                const uint4 xa = lds128_c(win, px), xb = lds128_c(win, px + x_half);
                const uint32_t BX[4][2] = {{xa.x, xa.y}, {xa.z, xa.w}, {xb.x, xb.y}, {xb.z, xb.w}};
                float c[4][4];
#pragma unroll
                for (int jw = 0; jw < 4; ++jw) {
                    const uint32_t w0 = W0[u][jw], w1 = W1[u][jw], s0 = w0 >> 8, s1 = w1 >> 8;
#pragma unroll
                    for (int cl = 0; cl < 4; ++cl) {
                        const uint32_t m = 0x00030003u << (2 * cl);
                        if (jw == 0)
                            mma_16816_zero(c[cl], w0 & m, w1 & m, s0 & m, s1 & m, BX[jw][0], BX[jw][1]);
                        else
                            mma_16816(c[cl], w0 & m, w1 & m, s0 & m, s1 & m, BX[jw][0], BX[jw][1]);
                    }
                }
                if (u + 1 == kUpw && s + 1 < n_stages) {
                    if (__all_sync(0xffffffffu, mbar_wait_for(smem_addr(&bars[nsl]), (uint32_t)nph, lim))) {
                        load_codes(nsl);
                    } else {
                        if (lane == 0) report_timeout(p, abort_flag);
                        ok = false;
                    }
                }
                const float e = dg[u], e8 = dg8[u];
                acc[0][0] = fmaf(e, c[0][0] + xi[u], u ? acc[0][0] : 0.0f);
                acc[0][1] = fmaf(e8, c[0][2] + xi[u], u ? acc[0][1] : 0.0f);
                acc[1][0] = fmaf(e, c[1][1], u ? acc[1][0] : 0.0f);
                acc[1][1] = fmaf(e8, c[1][3], u ? acc[1][1] : 0.0f);
                acc[2][0] = fmaf(e, c[2][0], u ? acc[2][0] : 0.0f);
                acc[2][1] = fmaf(e8, c[2][2], u ? acc[2][1] : 0.0f);
                acc[3][0] = fmaf(e, c[3][1], u ? acc[3][0] : 0.0f);
                acc[3][1] = fmaf(e8, c[3][3], u ? acc[3][1] : 0.0f);
            }
            if (ok && s + 1 < n_stages) load_scales(s + 1);
            flush(s);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&bars[S + sl]));
            sl = nsl;
            ph = nph;
        }
    } else {
    int slot = 0, phase = 0, kc = 0, rg0 = 0;  // stage iterator (no divisions)
    bool alive = true;        // false after this warp's wait ran out: no more waits
    bool ready_lane = false;  // early, non-blocking test of this stage's barrier
    for (int s = 0; s < n_stages; ++s) {
        // every lane waits (acquire); the decision is made warp-uniform
        bool ok = alive;
        if (ok && !__all_sync(0xffffffffu, ready_lane) &&
            !__all_sync(0xffffffffu, mbar_wait_for(smem_addr(&bars[slot]), (uint32_t)phase, lim))) {
            if (lane == 0) report_timeout(p, abort_flag);
            ok = alive = false;
        }
        ready_lane = false;
        if (tid == 0 && s == 0) TQ2_STAMP(p.seq, 3);
        if (ok && s + 1 < n_stages) {
            // test the next stage now; its latency overlaps this stage's math
            const int nslot = (slot + 1 == S) ? 0 : slot + 1;
            const int nphase = (slot + 1 == S) ? (phase ^ 1) : phase;
            ready_lane = mbar_test_wait(smem_addr(&bars[nslot]), (uint32_t)nphase);
        }
        if (ok) {
            const int nrg_s = min(p.rg_s, nrg - rg0);
            const int kb0 = kc * p.nbk_full;
            const int nbk = min(p.nbk_full, B - kb0);
            const uint32_t st = a_thr + (uint32_t)(slot * p.stage_bytes);
            if (nrg_s == 1 && nbk == kUpw * kConsumerWarps) {
                // Full 16-row x 16-block stage: this warp takes blocks
                // warp + u * kConsumerWarps (u < kUpw) of row group rg0,
                // computed together (4 * kUpw independent MMA chains).
                const int rg = rg0;
                if (rg != cur_rg) {
                    if (cur_rg >= 0) flush(cur_rg);
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[c][0] = acc[c][1] = 0.0f;
                    cur_rg = rg;
                }
                uint32_t W0[kUpw][4], W1[kUpw][4], BX[kUpw][4][2];
                float dg[kUpw], dg8[kUpw], xi[kUpw];
#pragma unroll
                for (int u = 0; u < kUpw; ++u) {
                    const int kb = kb0 + warp + u * kConsumerWarps;
                    const uint32_t pa = st + (uint32_t)((warp + u * kConsumerWarps) * 64);
                    const uint4 wa = lds128_c(win, pa), wb = lds128_c(win, pa + a_half);
                    const uint32_t px = x_thr + (uint32_t)kb * x_blk;
                    const uint4 xa = lds128_c(win, px), xb = lds128_c(win, px + x_half);
                    const uint32_t pd = d_thr + (uint32_t)rg * rg_stride_d + (uint32_t)kb * 4u;
                    dg[u] = lds_f32_c(win, pd);
                    dg8[u] = lds_f32_c(win, pd + d_half);
                    xi[u] = -lds_f32_c(win, xs_thr + (uint32_t)kb * (4u * kM)) * 5.9604644775390625e-08f;
                    W0[u][0] = wa.x; W0[u][1] = wa.y; W0[u][2] = wa.z; W0[u][3] = wa.w;
                    W1[u][0] = wb.x; W1[u][1] = wb.y; W1[u][2] = wb.z; W1[u][3] = wb.w;
                    BX[u][0][0] = xa.x; BX[u][0][1] = xa.y; BX[u][1][0] = xa.z; BX[u][1][1] = xa.w;
                    BX[u][2][0] = xb.x; BX[u][2][1] = xb.y; BX[u][3][0] = xb.z; BX[u][3][1] = xb.w;
                }
                // four class accumulators per unit, starting at zero; the "-1"
                // of q - 1 is added below as d_b * (-X_b * 2^-24) to class 0
                float c[kUpw][4][4];
#pragma unroll
                for (int jw = 0; jw < 4; ++jw) {
#pragma unroll
                    for (int u = 0; u < kUpw; ++u) {
                        const uint32_t w0 = W0[u][jw], w1 = W1[u][jw], s0 = w0 >> 8, s1 = w1 >> 8;
#pragma unroll
                        for (int cl = 0; cl < 4; ++cl) {
                            const uint32_t m = 0x00030003u << (2 * cl);
                            if (jw == 0)
                                mma_16816_zero(c[u][cl], w0 & m, w1 & m, s0 & m, s1 & m, BX[u][jw][0], BX[u][jw][1]);
                            else
                                mma_16816(c[u][cl], w0 & m, w1 & m, s0 & m, s1 & m, BX[u][jw][0], BX[u][jw][1]);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < kUpw; ++u) {
                    acc[0][0] = fmaf(dg[u], c[u][0][0] + xi[u], acc[0][0]);
                    acc[0][1] = fmaf(dg8[u], c[u][0][2] + xi[u], acc[0][1]);
                    acc[1][0] = fmaf(dg[u], c[u][1][1], acc[1][0]);
                    acc[1][1] = fmaf(dg8[u], c[u][1][3], acc[1][1]);
                    acc[2][0] = fmaf(dg[u], c[u][2][0], acc[2][0]);
                    acc[2][1] = fmaf(dg8[u], c[u][2][2], acc[2][1]);
                    acc[3][0] = fmaf(dg[u], c[u][3][1], acc[3][0]);
                    acc[3][1] = fmaf(dg8[u], c[u][3][3], acc[3][1]);
                }
            } else {
            int j = 0, bl = warp;  // unit u = warp + 8 i  ->  (16-row group j, block bl)
            while (bl >= nbk) {
                bl -= nbk;
                ++j;
            }
            while (j < nrg_s) {
                const int rg = rg0 + j, kb = kb0 + bl;
                if (rg != cur_rg) {
                    if (cur_rg >= 0) flush(cur_rg);
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[c][0] = acc[c][1] = 0.0f;
                    cur_rg = rg;
                }
                const uint32_t pa = st + (uint32_t)(j * 16 * p.rb + bl * 64);
                const uint4 wa = lds128_c(win, pa);
                const uint4 wb = lds128_c(win, pa + a_half);
                const uint32_t px = x_thr + (uint32_t)kb * x_blk;
                const uint4 xa = lds128_c(win, px);
                const uint4 xb = lds128_c(win, px + x_half);
                const uint32_t pd = d_thr + (uint32_t)rg * rg_stride_d + (uint32_t)kb * 4u;
                const float dg = lds_f32_c(win, pd);
                const float dg8 = lds_f32_c(win, pd + d_half);
                const float xi = -lds_f32_c(win, xs_thr + (uint32_t)kb * (4u * kM)) * 5.9604644775390625e-08f;
                float c0[4], c1[4], c2[4], c3[4];
                {
                    const uint32_t w0 = wa.x, w1 = wb.x, s0 = w0 >> 8, s1 = w1 >> 8;
                    const uint32_t b0 = xa.x, b1 = xa.y;
                    TQ2_MMA_CLASS(true, c0, 0x00030003u, xi);
                    TQ2_MMA_CLASS(true, c1, 0x000C000Cu, 0.0f);
                    TQ2_MMA_CLASS(true, c2, 0x00300030u, 0.0f);
                    TQ2_MMA_CLASS(true, c3, 0x00C000C0u, 0.0f);
                }
                {
                    const uint32_t w0 = wa.y, w1 = wb.y, s0 = w0 >> 8, s1 = w1 >> 8;
                    const uint32_t b0 = xa.z, b1 = xa.w;
                    TQ2_MMA_CLASS(false, c0, 0x00030003u, 0.0f);
                    TQ2_MMA_CLASS(false, c1, 0x000C000Cu, 0.0f);
                    TQ2_MMA_CLASS(false, c2, 0x00300030u, 0.0f);
                    TQ2_MMA_CLASS(false, c3, 0x00C000C0u, 0.0f);
                }
                {
                    const uint32_t w0 = wa.z, w1 = wb.z, s0 = w0 >> 8, s1 = w1 >> 8;
                    const uint32_t b0 = xb.x, b1 = xb.y;
                    TQ2_MMA_CLASS(false, c0, 0x00030003u, 0.0f);
                    TQ2_MMA_CLASS(false, c1, 0x000C000Cu, 0.0f);
                    TQ2_MMA_CLASS(false, c2, 0x00300030u, 0.0f);
                    TQ2_MMA_CLASS(false, c3, 0x00C000C0u, 0.0f);
                }
                {
                    const uint32_t w0 = wa.w, w1 = wb.w, s0 = w0 >> 8, s1 = w1 >> 8;
                    const uint32_t b0 = xb.z, b1 = xb.w;
                    TQ2_MMA_CLASS(false, c0, 0x00030003u, 0.0f);
                    TQ2_MMA_CLASS(false, c1, 0x000C000Cu, 0.0f);
                    TQ2_MMA_CLASS(false, c2, 0x00300030u, 0.0f);
                    TQ2_MMA_CLASS(false, c3, 0x00C000C0u, 0.0f);
                }
                acc[0][0] = fmaf(dg, c0[0], acc[0][0]);
                acc[0][1] = fmaf(dg8, c0[2], acc[0][1]);
                acc[1][0] = fmaf(dg, c1[1], acc[1][0]);
                acc[1][1] = fmaf(dg8, c1[3], acc[1][1]);
                acc[2][0] = fmaf(dg, c2[0], acc[2][0]);
                acc[2][1] = fmaf(dg8, c2[2], acc[2][1]);
                acc[3][0] = fmaf(dg, c3[1], acc[3][0]);
                acc[3][1] = fmaf(dg8, c3[3], acc[3][1]);
                bl += kConsumerWarps;
                while (bl >= nbk) {
                    bl -= nbk;
                    ++j;
                }
            }
            }
        }
        // a warp that gave up releases no more slots: the producer's next
        // wait for them runs out too, and no copy is issued into a slot whose
        // stage was not waited for
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(smem_addr(&bars[S + slot]));
        if (++slot == S) {
            slot = 0;
            phase ^= 1;
        }
        if (++kc == p.n_kc) {
            kc = 0;
            rg0 += p.rg_s;
        }
    }
    if (cur_rg >= 0) flush(cur_rg);
    }
    if (tid == 0) TQ2_STAMP(p.seq, 4);
    consumer_barrier();
    if (*abort_flag) return;  // y is invalid; TQ2_FLAG_TIMEOUT was reported

    // y[m][r0 + r] = sum over warps (fixed order) of the partials
    for (int i = tid; i < kM * nrows; i += kConsumerThreads) {
        const int m = (kM == 2 && i >= nrows) ? 1 : 0;  // kM <= 2: no division
        const int r = i - m * nrows;
        const int rg = r >> 4, ri = r & 15;
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) s += red[((rg * kConsumerWarps + w) * kM + m) * 16 + ri];
        if (prologue) s *= p.a.act_scale;
        s = requant_out(s, p.mats[mi].out_scale, p.mats[mi].inv_out);
        const int64_t o = (int64_t)m * N + r0 + r;
        if (!TQ2_IN(o < kM * N && rg < p.max_rg, st_w)) continue;
        if (p.a.y_f16)
            reinterpret_cast<__half *>(y_g)[o] = __float2half_rn(s);
        else
            reinterpret_cast<float *>(y_g)[o] = s;
    }
#ifdef TQ2_TRACE
    consumer_barrier();  // every y store of the CTA issued
    if (tid == 0) TQ2_STAMP(p.seq, 5);
#endif
}

// ------------------------------------------------------------------ host side
static int align_up(int v, int a) { return (v + a - 1) / a * a; }

// Launch sequence numbers (the parity picks a trace slot; in a CUDA graph
// every node keeps the number it was captured with).
std::atomic<int> g_seq{0};
int next_seq() { return g_seq.fetch_add(1, std::memory_order_relaxed); }

// Shared-memory plan for G CTAs within max_dyn bytes of dynamic shared
// memory; returns false if it cannot fit.
bool make_plan_rows(int M, int64_t max_rows, int64_t K, int max_dyn, MmaPlan &p)
{
    const int kMaxSmem = max_dyn;
    const int64_t B = K / 256;
    if (B > (1 << 20)) return false;
    p.B = (int)B;
    if (B > kChunkBlocks) {  // 16 rows x 4096 codes per stage, 2-D tensor boxes
        p.tma2d = 1;
        p.nbk_full = kChunkBlocks;
        p.n_kc = (int)((B + kChunkBlocks - 1) / kChunkBlocks);
        p.rg_s = 1;
    } else {                 // whole rows, contiguous: 1-D bulk copies
        p.tma2d = 0;
        p.nbk_full = (int)B;
        p.n_kc = 1;
        p.rg_s = kChunkBlocks / (int)B;
    }
    p.max_rg = (int)((max_rows + 15) / 16);
    if (p.rg_s > p.max_rg) p.rg_s = p.max_rg;
    p.rb = p.nbk_full * 64;  // dense rows, as TMA writes them
    p.stage_bytes = p.rg_s * 16 * p.rb;
    p.dstr = (int)B + 1;
    int off = 0;
    p.off_bar = off;  // filled after the ring depth is known (<= 16 barriers)
    off += 16 * 8;
    p.off_red = off;
    off += align_up(p.max_rg * kConsumerWarps * M * 16 * 4, 16);
    p.off_dsm = off;
    off += align_up((int)(p.max_rg * 16 * (int64_t)p.dstr * 4), 16);
    p.off_xsum = off;
    off += align_up((int)(B * M * 4), 16);
    p.off_xs = off;
    off += (int)(B * 512 * M);
    off = align_up(off, 128);
    p.off_ring = off;
    const int fixed = off;
    int S;
    if (fixed + 2 * p.stage_bytes <= kTargetSmem)
        S = (kTargetSmem - fixed) / p.stage_bytes;
    else
        S = (kMaxSmem - fixed) / p.stage_bytes;
    if (S > 8) S = 8;
    if (S < 2) return false;
    p.stages = S;
    p.smem_total = fixed + S * p.stage_bytes;
    return p.smem_total <= kMaxSmem;
}

bool make_plan(int M, int64_t N, int64_t K, int G, int max_dyn, MmaPlan &p)
{
    p.G = G;
    return make_plan_rows(M, (N + G - 1) / G, K, max_dyn, p);
}

// Largest dynamic shared memory the kernel for kM may use on `device`
// (the per-block opt-in limit minus the kernel's static shared memory);
// the kernel attribute is raised to it once per device.  0 on failure.
std::atomic<int> g_max_dyn[2][64];

template <int kM>
int max_dynamic_smem(int device)
{
    if (device < 0 || device >= 64) return 0;
    int v = g_max_dyn[kM - 1][device].load();
    if (v > 0) return v;
    int optin = 0;
    cudaFuncAttributes fa;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, matvec_mma_kernel<kM, 1, 1, false>) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    v = optin - (int)fa.sharedSizeBytes;  // the same static shared memory for both instantiations
    const auto attr = cudaFuncAttributeMaxDynamicSharedMemorySize;
    if (cudaFuncSetAttribute(matvec_mma_kernel<kM, 1, 1, false>, attr, v) != cudaSuccess ||
        cudaFuncSetAttribute(matvec_mma_kernel<kM, 1, 1, true>, attr, v) != cudaSuccess ||
        cudaFuncSetAttribute(matvec_mma_kernel<kM, kMaxGroup, 1, false>, attr, v) != cudaSuccess ||
        cudaFuncSetAttribute(matvec_mma_kernel<kM, kMaxGroup, kMaxGroup, false>, attr, v) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    g_max_dyn[kM - 1][device].store(v);
    return v;
}

// Grid and plan: one CTA per SM while the per-CTA share fits, more CTAs otherwise.
bool plan_for(int M, int64_t N, int64_t K, int device, int max_dyn, MmaPlan &p)
{
    if (max_dyn <= 0) return false;
    int G = (int)((N < (int64_t)sm_count(device)) ? N : sm_count(device));
    while (!make_plan(M, N, K, G, max_dyn, p)) {
        if (G >= N) return false;
        G = (int)((2 * (int64_t)G < N) ? 2 * G : N);
    }
    return true;
}

// CTAs of a group in proportion to the matrices' rows (at least one each,
// at most one per SM in total while that fits), then the shared-memory plan
// for the largest per-CTA row count.
template <int kT>
bool group_plan(int M, int n, const int64_t *N, int64_t K, int device, int max_dyn, MmaParams<kMaxGroup, kT> &p)
{
    if (max_dyn <= 0 || n < 1 || n > kMaxGroup) return false;
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
        // leftover CTAs to the matrix with the most rows per CTA
        while (sum < cap) {
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
        p.n_mats = n;
        p.G = g0;
        if (make_plan_rows(M, max_rows, K, max_dyn, p)) return true;
    }
    return false;
}

// qs as uint64 [N][K/32]; boxes 128 x {16, 8, 4, 2, 1}
cudaError_t encode_qs_maps(const uint8_t *qs, int64_t N, int64_t K, CUtensorMap (&tmap)[5])
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)(K / 32), (cuuint64_t)N};
    const cuuint64_t strides[1] = {(cuuint64_t)(K / 4)};
    const cuuint32_t estr[2] = {1, 1};
    for (int i = 0; i < 5; ++i) {
        const cuuint32_t box[2] = {128, (cuuint32_t)(16 >> i)};
        CUresult r = enc(&tmap[i], CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint8_t *>(qs), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

template <int kM>
cudaError_t launch_impl(const MatvecArgs &a, int device)
{
    MmaParams<1, 1> p{};
    p.a = a;
    p.seq = next_seq();
    if (!plan_for(kM, a.N, a.K, device, max_dynamic_smem<kM>(device), p))
        return cudaErrorInvalidConfiguration;
    p.n_mats = 1;
    p.mats[0] = GroupMat{a.qs, a.d, a.y, a.N, 0, p.G, a.out_scale, a.inv_out};
    if (p.tma2d) {
        cudaError_t e = encode_qs_maps(a.qs, a.N, a.K, p.tmap[0]);
        if (e != cudaSuccess) return e;
    }
    const bool hook = a.stall_stage >= 0 || a.wait_limit_ns != 0;
    auto kern = hook ? matvec_mma_kernel<kM, 1, 1, true> : matvec_mma_kernel<kM, 1, 1, false>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.G);
    cfg.blockDim = dim3(kMmaThreads);
    cfg.dynamicSmemBytes = (size_t)p.smem_total;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int kM, int kT>
cudaError_t launch_group_kt(const MatvecArgs &a, int n, const uint8_t *const *qs, const uint16_t *const *d,
                            void *const *y, const int64_t *N, const float *out_scale, const float *inv_out,
                            int device, int max_dyn)
{
    MmaParams<kMaxGroup, kT> p{};
    p.a = a;
    if (!group_plan(kM, n, N, a.K, device, max_dyn, p)) return cudaErrorInvalidConfiguration;
    for (int j = 0; j < n; ++j) {
        p.mats[j].qs = qs[j];
        p.mats[j].d = d[j];
        p.mats[j].y = y[j];
        p.mats[j].out_scale = out_scale ? out_scale[j] : 0.0f;
        p.mats[j].inv_out = inv_out ? inv_out[j] : 0.0f;
        if (p.tma2d) {
            if (kT < kMaxGroup) return cudaErrorInvalidConfiguration;  // not reached: see the caller
            cudaError_t e = encode_qs_maps(qs[j], N[j], a.K, p.tmap[kT > 1 ? j : 0]);
            if (e != cudaSuccess) return e;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.G);
    cfg.blockDim = dim3(kMmaThreads);
    cfg.dynamicSmemBytes = (size_t)p.smem_total;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, matvec_mma_kernel<kM, kMaxGroup, kT, false>, p);
}

// One map set unless the plan uses 2-D boxes (K > 4096).
template <int kM>
cudaError_t launch_group_impl(const MatvecArgs &a, int n, const uint8_t *const *qs, const uint16_t *const *d,
                              void *const *y, const int64_t *N, const float *out_scale, const float *inv_out,
                              int device)
{
    const int max_dyn = max_dynamic_smem<kM>(device);
    if (a.K > 256 * kChunkBlocks)
        return launch_group_kt<kM, kMaxGroup>(a, n, qs, d, y, N, out_scale, inv_out, device, max_dyn);
    return launch_group_kt<kM, 1>(a, n, qs, d, y, N, out_scale, inv_out, device, max_dyn);
}

}  // namespace

bool mma_group_supported(int M, int n, const int64_t *N, int64_t K, int device)
{
    if (M < 1 || M > 2 || K < 256) return false;
    MmaParams<kMaxGroup, 1> p{};
    const int max_dyn = (M == 1) ? max_dynamic_smem<1>(device) : max_dynamic_smem<2>(device);
    return group_plan(M, n, N, K, device, max_dyn, p);
}

cudaError_t launch_matvec_mma_group(const MatvecArgs &a, int n, const uint8_t *const *qs, const uint16_t *const *d,
                                    void *const *y, const int64_t *N, const float *out_scale,
                                    const float *inv_out, int device)
{
    if (a.M == 1) return launch_group_impl<1>(a, n, qs, d, y, N, out_scale, inv_out, device);
    if (a.M == 2) return launch_group_impl<2>(a, n, qs, d, y, N, out_scale, inv_out, device);
    return cudaErrorInvalidValue;
}

bool mma_matvec_supported(int M, int64_t N, int64_t K, int device)
{
    if (M < 1 || M > 2 || N < 1 || K < 256) return false;
    MmaPlan p{};
    const int max_dyn = (M == 1) ? max_dynamic_smem<1>(device) : max_dynamic_smem<2>(device);
    return plan_for(M, N, K, device, max_dyn, p);
}

cudaError_t launch_matvec_mma(const MatvecArgs &a, int device)
{
    if (a.M == 1) return launch_impl<1>(a, device);
    if (a.M == 2) return launch_impl<2>(a, device);
    return cudaErrorInvalidValue;
}

size_t trace_bytes()
{
#ifdef TQ2_TRACE
    return sizeof(unsigned long long) * 2 * dev::kTraceCtas * dev::kTracePhases;
#else
    return 0;
#endif
}

cudaError_t trace_read(void *dst, size_t bytes)
{
#ifdef TQ2_TRACE
    if (bytes < trace_bytes()) return cudaErrorInvalidValue;
    return cudaMemcpyFromSymbol(dst, dev::g_trace, trace_bytes());
#else
    (void)dst;
    (void)bytes;
    return cudaErrorNotSupported;
#endif
}

}  // namespace tq2
