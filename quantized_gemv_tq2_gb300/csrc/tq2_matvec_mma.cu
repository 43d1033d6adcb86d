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
//     with 1-D TMA bulk copies (cp.async.bulk + mbarrier complete_tx), one
//     copy per row segment, L2 evict-first; it starts before the kernel waits
//     on the previous grid (programmatic dependent launch), because weights
//     never depend on earlier kernels;
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
// Layout of one 16-row A tile: mma row g <- smem row g, row g+8 <- g+8; the
// smem row stride is padded so that rows g and g+1 fall 64 bytes apart in the
// bank space, which makes the 16-byte fragment loads conflict-free.
#include <cuda_fp16.h>

#include <atomic>

#include "tq2_internal.cuh"

namespace tq2 {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kMmaThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kChunkBlocks = 16;                    // 256-blocks per stage row (4096 codes)
constexpr int kTargetSmem = 112 * 1024;             // two CTAs per SM (PDL overlap)
constexpr int kMaxSmem = 227 * 1024;
constexpr unsigned long long kTimeoutNs = 200ull * 1000 * 1000;

struct MmaParams {
    MatvecArgs a;
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
};

// ------------------------------------------------------------------ PTX helpers
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

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long globaltimer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity; give up after kTimeoutNs.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer() - t0 > kTimeoutNs) return false;
    }
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

__device__ __forceinline__ void consumer_barrier()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
}

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Static int8 fake-quant code (gemma4 wNa8o8 page, "Implemented"):
// rint(x * (1/s)) in fp32, ties to even, clamped to [-128, 127]; NaN -> 0.
__device__ __forceinline__ float fq_code(float x, float inv_s)
{
    float t = __fmul_rn(x, inv_s);
    if (t != t) return 0.0f;
    return fminf(fmaxf(rintf(t), -128.0f), 127.0f);
}

__device__ __forceinline__ void report_timeout(const MmaParams &p, volatile int *abort_flag)
{
    *abort_flag = 1;
    if (p.a.status) atomicOr(p.a.status, TQ2_FLAG_TIMEOUT);
}

// ------------------------------------------------------------------ kernel
template <int kM>
__global__ void __launch_bounds__(kMmaThreads, 2)
matvec_mma_kernel(const __grid_constant__ MmaParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int abort_shared;
    volatile int *abort_flag = &abort_shared;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t N = p.a.N, K = p.a.K;
    const int64_t r0 = (int64_t)blockIdx.x * N / p.G;
    const int64_t r1 = (int64_t)(blockIdx.x + 1) * N / p.G;
    const int nrows = (int)(r1 - r0);
    const int nrg = (nrows + 15) >> 4;
    const int n_stages = ((nrg + p.rg_s - 1) / p.rg_s) * p.n_kc;
    const int S = p.stages;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.off_bar);  // full[S], empty[S]
    uint8_t *ring = smem + p.off_ring;

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
                !__all_sync(0xffffffffu, mbar_wait(smem_addr(&bars[S + slot]), (round - 1) & 1))) {
                if (lane == 0) report_timeout(p, abort_flag);
                break;
            }
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            const int rgb = s / p.n_kc, kc = s % p.n_kc;
            const int rg0 = rgb * p.rg_s;
            const int rows = min(p.rg_s * 16, nrows - rg0 * 16);
            const int kb0 = kc * p.nbk_full;
            const int nbk = min(p.nbk_full, p.B - kb0);
            const uint32_t seg = (uint32_t)nbk * 64u;
            const uint32_t full = smem_addr(&bars[slot]);
            if (lane == 0) mbar_arrive_expect_tx(full, seg * (uint32_t)rows);
            __syncwarp();
            const uint32_t dst0 = smem_addr(ring + (size_t)slot * p.stage_bytes);
            for (int r = lane; r < rows; r += 32) {
                const uint8_t *src = p.a.qs + (r0 + rg0 * 16 + r) * row_bytes + (int64_t)kb0 * 64;
                bulk_g2s(dst0 + (uint32_t)(r * p.rb), src, seg, full, pol);
            }
            issued = s + 1;
        }
        // No copy may still be writing shared memory when the CTA exits.
        for (int slot = 0; slot < S && slot < issued; ++slot) {
            const int last = slot + ((issued - 1 - slot) / S) * S;
            if (!mbar_wait(smem_addr(&bars[slot]), (last / S) & 1) && lane == 0)
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

    // zero this warp's slots of the cross-warp partial sums
    for (int i = lane; i < nrg * kM * 16; i += 32) {
        const int rg = i / (kM * 16), rest = i - rg * (kM * 16);
        red[(rg * kConsumerWarps + warp) * kM * 16 + rest] = 0.0f;
    }
    // d slice of this CTA's rows, fp32
    for (int i = tid; i < nrows * B; i += kConsumerThreads) {
        const int r = i / B, b = i - r * B;
        dsm[r * p.dstr + b] = __half2float(__ushort_as_half(p.a.d[(r0 + r) * B + b]));
    }

    // x depends on the previous kernel in the stream.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    // x -> fragment order.  Entry (block b, half h, column cc = 4m + c, t)
    // is 16 bytes = words 2h and 2h+1 of the t-th quarter of the block, each
    // as (x[c], x[8+c], x[4+c], x[12+c]) of that 16-code word.
    {
        const int total = kM * B * 16;  // 16-code words
        for (int base = warp * 32; base < total; base += kConsumerThreads) {
            const int L = base + lane;
            const bool act = L < total;
            float sum = 0.0f;
            int m = 0, b = 0, wib = 0;
            if (act) {
                m = L / (B * 16);
                const int rem = L - m * B * 16;
                b = rem >> 4;
                wib = rem & 15;
                const uint16_t *src = p.a.x + (int64_t)m * K + (int64_t)b * 256 + wib * 16;
                const uint4 v0 = *reinterpret_cast<const uint4 *>(src);
                const uint4 v1 = *reinterpret_cast<const uint4 *>(src + 8);
                const uint32_t raw[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                uint16_t h[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    uint16_t hb = (uint16_t)(raw[j >> 1] >> (16 * (j & 1)));
                    float f = __half2float(__ushort_as_half(hb));
                    if (prologue) {
                        f = fq_code(f, p.a.inv_scale);
                        hb = __half_as_ushort(__float2half_rn(f));  // exact: |f| <= 128
                    }
                    h[j] = hb;
                    sum += f;
                }
                const int t4 = wib >> 2, i4 = wib & 3;
                uint8_t *dst = xs + (size_t)b * 512 * kM + (i4 >> 1) * (4 * kM * 64) + t4 * 16 +
                               (i4 & 1) * 8;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint2 e;
                    e.x = (uint32_t)h[c] | ((uint32_t)h[8 + c] << 16);
                    e.y = (uint32_t)h[4 + c] | ((uint32_t)h[12 + c] << 16);
                    *reinterpret_cast<uint2 *>(dst + (4 * m + c) * 64) = e;
                }
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
            if (act && (lane & 15) == 0) xsum[b * kM + m] = sum;
        }
    }
    consumer_barrier();

    const int g = lane >> 2, t = lane & 3;
    const int gg = g % (4 * kM);          // x-fragment column this thread supplies
    const int mcol = (kM == 2) ? (t >> 1) : 0;  // activation row of columns 2t, 2t+1
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
            rp[g] = vg;
            rp[g + 8] = vg8;
        }
    };

    for (int s = 0; s < n_stages; ++s) {
        const int slot = s % S;
        // every lane waits (acquire); the decision is made warp-uniform
        bool ok = !__any_sync(0xffffffffu, *abort_flag != 0);
        if (ok && !__all_sync(0xffffffffu, mbar_wait(smem_addr(&bars[slot]), (s / S) & 1))) {
            if (lane == 0) report_timeout(p, abort_flag);
            ok = false;
        }
        if (ok) {
            const int rgb = s / p.n_kc, kc = s % p.n_kc;
            const int rg0 = rgb * p.rg_s;
            const int nrg_s = min(p.rg_s, nrg - rg0);
            const int kb0 = kc * p.nbk_full;
            const int nbk = min(p.nbk_full, B - kb0);
            const uint8_t *st = ring + (size_t)slot * p.stage_bytes;
            const int units = nrg_s * nbk;
            for (int u = warp; u < units; u += kConsumerWarps) {
                const int j = u / nbk, bl = u - j * nbk;
                const int rg = rg0 + j, kb = kb0 + bl;
                if (rg != cur_rg) {
                    if (cur_rg >= 0) flush(cur_rg);
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[c][0] = acc[c][1] = 0.0f;
                    cur_rg = rg;
                }
                const uint8_t *pa = st + (j * 16 + g) * p.rb + bl * 64 + t * 16;
                const uint4 wa = *reinterpret_cast<const uint4 *>(pa);
                const uint4 wb = *reinterpret_cast<const uint4 *>(pa + 8 * p.rb);
                const uint8_t *px = xs + (size_t)kb * 512 * kM + gg * 64 + t * 16;
                const uint4 xa = *reinterpret_cast<const uint4 *>(px);
                const uint4 xb = *reinterpret_cast<const uint4 *>(px + 4 * kM * 64);
                const float dg = dsm[(rg * 16 + g) * p.dstr + kb];
                const float dg8 = dsm[(rg * 16 + g + 8) * p.dstr + kb];
                const float xi = -xsum[kb * kM + mcol] * 5.9604644775390625e-08f;  // 2^-24
                float c0[4] = {xi, xi, xi, xi};
                float c1[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f},
                      c3[4] = {0.f, 0.f, 0.f, 0.f};
                const uint32_t w0[4] = {wa.x, wa.y, wa.z, wa.w};
                const uint32_t w1[4] = {wb.x, wb.y, wb.z, wb.w};
                const uint32_t bx[4][2] = {{xa.x, xa.y}, {xa.z, xa.w}, {xb.x, xb.y}, {xb.z, xb.w}};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t s0 = w0[i] >> 8, s1 = w1[i] >> 8;
                    mma_16816(c0, w0[i] & 0x00030003u, w1[i] & 0x00030003u, s0 & 0x00030003u,
                              s1 & 0x00030003u, bx[i][0], bx[i][1]);
                    mma_16816(c1, w0[i] & 0x000C000Cu, w1[i] & 0x000C000Cu, s0 & 0x000C000Cu,
                              s1 & 0x000C000Cu, bx[i][0], bx[i][1]);
                    mma_16816(c2, w0[i] & 0x00300030u, w1[i] & 0x00300030u, s0 & 0x00300030u,
                              s1 & 0x00300030u, bx[i][0], bx[i][1]);
                    mma_16816(c3, w0[i] & 0x00C000C0u, w1[i] & 0x00C000C0u, s0 & 0x00C000C0u,
                              s1 & 0x00C000C0u, bx[i][0], bx[i][1]);
                }
                acc[0][0] = fmaf(dg, c0[0], acc[0][0]);
                acc[0][1] = fmaf(dg8, c0[2], acc[0][1]);
                acc[1][0] = fmaf(dg, c1[1], acc[1][0]);
                acc[1][1] = fmaf(dg8, c1[3], acc[1][1]);
                acc[2][0] = fmaf(dg, c2[0], acc[2][0]);
                acc[2][1] = fmaf(dg8, c2[2], acc[2][1]);
                acc[3][0] = fmaf(dg, c3[1], acc[3][0]);
                acc[3][1] = fmaf(dg8, c3[3], acc[3][1]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&bars[S + slot]));
    }
    if (cur_rg >= 0) flush(cur_rg);
    consumer_barrier();
    if (*abort_flag) return;  // y is invalid; TQ2_FLAG_TIMEOUT was reported

    // y[m][r0 + r] = sum over warps (fixed order) of the partials
    for (int i = tid; i < kM * nrows; i += kConsumerThreads) {
        const int m = i / nrows, r = i - m * nrows;
        const int rg = r >> 4, ri = r & 15;
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) s += red[((rg * kConsumerWarps + w) * kM + m) * 16 + ri];
        if (prologue) s *= p.a.act_scale;
        const int64_t o = (int64_t)m * N + r0 + r;
        if (p.a.y_f16)
            reinterpret_cast<__half *>(p.a.y)[o] = __float2half_rn(s);
        else
            reinterpret_cast<float *>(p.a.y)[o] = s;
    }
}

// ------------------------------------------------------------------ host side
static int align_up(int v, int a) { return (v + a - 1) / a * a; }

// Shared-memory plan for G CTAs; returns false if it cannot fit.
bool make_plan(int M, int64_t N, int64_t K, int G, MmaParams &p)
{
    const int64_t B = K / 256;
    if (B > (1 << 20)) return false;
    p.G = G;
    p.B = (int)B;
    if (B >= kChunkBlocks) {
        p.nbk_full = kChunkBlocks;
        p.n_kc = (int)((B + kChunkBlocks - 1) / kChunkBlocks);
        p.rg_s = 1;
    } else {
        p.nbk_full = (int)B;
        p.n_kc = 1;
        p.rg_s = kChunkBlocks / (int)B;
    }
    const int64_t max_rows = (N + G - 1) / G;
    p.max_rg = (int)((max_rows + 15) / 16);
    if (p.rg_s > p.max_rg) p.rg_s = p.max_rg;
    // row stride = nbk*64 (+64 when nbk is even) keeps rows g, g+1 64 bytes
    // apart modulo 128 -> conflict-free 16-byte fragment loads
    p.rb = p.nbk_full * 64 + ((p.nbk_full % 2 == 0) ? 64 : 0);
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

std::atomic<int> g_smem_attr_set[2][64];

template <int kM>
cudaError_t launch_impl(const MatvecArgs &a, int device)
{
    MmaParams p{};
    p.a = a;
    int G = (int)((a.N < (int64_t)sm_count(device)) ? a.N : sm_count(device));
    while (!make_plan(kM, a.N, a.K, G, p)) {
        if (G >= a.N) return cudaErrorInvalidConfiguration;
        G = (int)((2 * (int64_t)G < a.N) ? 2 * G : a.N);
    }
    auto kern = matvec_mma_kernel<kM>;
    if (device >= 0 && device < 64 && !g_smem_attr_set[kM - 1][device].load()) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmem);
        if (e != cudaSuccess) return e;
        g_smem_attr_set[kM - 1][device].store(1);
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
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

bool mma_matvec_supported(int M, int64_t N, int64_t K, int device)
{
    if (M < 1 || M > 2 || N < 1 || K < 256) return false;
    MmaParams p{};
    int G = (int)((N < (int64_t)sm_count(device)) ? N : sm_count(device));
    while (!make_plan(M, N, K, G, p)) {
        if (G >= N) return false;
        G = (int)((2 * (int64_t)G < N) ? 2 * G : N);
    }
    return true;
}

cudaError_t launch_matvec_mma(const MatvecArgs &a, int device)
{
    if (a.M == 1) return launch_impl<1>(a, device);
    if (a.M == 2) return launch_impl<2>(a, device);
    return cudaErrorInvalidValue;
}

}  // namespace tq2
