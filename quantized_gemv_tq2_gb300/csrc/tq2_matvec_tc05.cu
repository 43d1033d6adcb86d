// tq2_matvec_tc05.cu -- ternary matvec on the 5th-generation tensor cores
// (tcgen05 / UMMA with the A operand in tensor memory), M = 1 or 2.
//
// What it computes (BitCPM ternary page, linear-factoring paragraph):
//   y[m][n] = sum_b d[n][b] * sum_{k in b} x'[m][k] * (q[n][k] - 1)
//
// Unpack.  A packed 32-bit word holds codes 0..15 of a row (code j at bits
// 2j of the low half, code 8+j at bits 16+2j).  w & (0x00030003 << 2c)
// keeps codes c and 8+c as two fp16 lanes with bit patterns q * 4^c, i.e.
// the exact fp16 values q * 4^c * 2^-24 (patterns below 2048 are
// pattern * 2^-24); (w >> 8) & (...) keeps codes 4+c and 12+c.  Eight LOP3
// per 16 codes, no conversion.  The four bit positions c differ only by the
// power 4^c, so x is stored pre-scaled by 4^(3-c) (exact in fp16 when the
// block's max |x| <= 1023.5; otherwise also by 2^-6, whose rounding error
// stays below 2^-19 |d| per element against a tolerance of at least 1e-3 |d|
// * 1023 for that block): every product is then q * x * 2^-18, and one MMA
// with K = 16 consumes all 16 codes of a word.
//
// Mapping onto tcgen05.mma.cta_group::1.kind::f16, M = 128, N = 16, K = 16:
//   * TMEM lane = (K-segment s, row r): the CTA's R rows are split along K
//     into S segments (S in {1,2,4}, R * S <= 128) so that CTAs with few rows
//     still fill the lanes;
//   * A (TMEM): per k-step (one 16-code word of each lane's segment) 8
//     columns = the 8 masked sub-words, written by the unpack warps with
//     tcgen05.st into a 4-slot ring of 64 columns (8 k-steps per slot);
//   * B (shared memory, no swizzle, K-major): column n = s * M + m holds the
//     pre-scaled x of segment s, row m, at the word's positions in the A lane
//     order.  Tiles of consecutive k-steps overlap in their unused columns, so
//     B costs exactly 2 * M * K bytes;
//   * D (TMEM): one 16-column region per 256-block of a segment; the first
//     MMA of a block overwrites, the rest accumulate.  No readout between
//     blocks: the epilogue reads D once and applies d_b, the 2^18 scale and
//     the "-1" of (q - 1) as -X_b = -sum_{k in b} x'_k.
//
// Data path per CTA (one CTA owns R consecutive rows, all K):
//   * warp 0 (producer) streams the weights with 3-D TMA boxes of
//     {128 bytes, R rows, C chunks} (~14 KB per copy), 128-byte swizzle so
//     the per-row 16-byte reads of the unpack warps are conflict-free; it
//     starts before griddepcontrol.wait (weights never depend on earlier
//     kernels);
//   * warp 1 allocates 512 TMEM columns after griddepcontrol.wait (so the
//     previous call's CTA on this SM has released them) and one lane issues
//     the MMAs;
//   * warps 2..9 (two per TMEM lane quadrant) stage d before the wait, x
//     after it, then unpack 16 bytes per lane per step into TMEM, and finally
//     read D out (tcgen05.ld), sum the K-segments of each row and store y.
// Every mbarrier wait is bounded; a wait that runs out sets TQ2_FLAG_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <atomic>

#include "tq2_device.cuh"
#include "tq2_internal.cuh"
#include "tq2_tcgen05.cuh"

namespace tq2 {
namespace {

constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kFirstUnpackWarp = 2;
constexpr int kUnpackWarps = 8;
constexpr int kThreads = (kFirstUnpackWarp + kUnpackWarps) * 32;  // 320
constexpr int kTmemCols = 512;
constexpr int kAColsPerSlot = 64;  // 8 k-steps x 8 columns (32 bytes of codes per lane)
constexpr int kASlots = 4;
constexpr int kDCol = 256;          // D regions start here (16 columns per 256-block)
constexpr int kTargetSmem = 112 * 1024;

struct Tc05Params {
    CUtensorMap wmap;  // qs as uint64 [K/512 chunks][N rows][16]; box {16, R, C}; 128B swizzle
    MatvecArgs a;
    int R;             // rows per CTA (the last CTA may have fewer)
    int S;             // K segments per row (lanes = R * S <= 128)
    int lanes_per_seg; // 128 / S
    int kseg;          // codes per segment (multiple of 512, <= 4096)
    int B;             // 256-blocks per row
    int C;             // 128-byte chunks per weight stage
    int stage_bytes;   // C * R * 128 rounded up to 1024
    int stages;        // weight ring depth
    int n_stages;      // S * (kseg / 512) / C
    int dstr;          // fp32 stride of the d slice rows (B + 1)
    int off_bar, off_b0, off_b1, off_xsum, off_rscale, off_dsm, off_red, off_ring, smem_total;
    uint32_t b_lbo;    // byte distance from the B0 to the B1 array
};

// ------------------------------------------------------------------ helpers
using namespace dev;

__device__ __forceinline__ void report_timeout(const Tc05Params &p, volatile int *flag)
{
    *flag = 1;
    if (p.a.status) atomicOr(p.a.status, TQ2_FLAG_TIMEOUT);
}

// ------------------------------------------------------------------ kernel
template <int kM>
__global__ void __launch_bounds__(kThreads, 2) matvec_tc05_kernel(const __grid_constant__ Tc05Params p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    volatile int *abort_flag = &abort_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t N = p.a.N, K = p.a.K;
    const int64_t row0 = (int64_t)blockIdx.x * p.R;
    const int R_cta = (int)((N - row0 < (int64_t)p.R) ? (N - row0) : (int64_t)p.R);
    const int S = p.S, SW = p.stages;
    const int kgroups = p.kseg / 128;  // 32-byte groups (8 k-steps) per lane
    const int nregions = p.kseg / 256;

    // barriers: wfull[SW], wempty[SW], afull[4], aempty[4], dfull
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    const uint32_t wfull0 = smem_addr(bars), wempty0 = wfull0 + 8u * SW;
    const uint32_t afull0 = wempty0 + 8u * SW, aempty0 = afull0 + 8u * kASlots;
    const uint32_t dfull = aempty0 + 8u * kASlots;

    // the weight ring is 1024-byte aligned (the 128-byte swizzle pattern is a
    // function of address bits 7..9); the plan reserves the slack
    const uint32_t ring_base = (smem_addr(smem + p.off_ring) + 1023u) & ~1023u;

    asm volatile("griddepcontrol.launch_dependents;");
    if (tid == 0) {
        for (int i = 0; i < SW; ++i) {
            mbar_init(wfull0 + 8u * i, 1);
            mbar_init(wempty0 + 8u * i, (uint32_t)(kUnpackWarps / S));
        }
        for (int i = 0; i < kASlots; ++i) {
            mbar_init(afull0 + 8u * i, 4);
            mbar_init(aempty0 + 8u * i, 1);
        }
        mbar_init(dfull, 1);
        abort_sh = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    if (warp == kProducerWarp) {
        // -------------------------------------------------- weights -> shared memory
        const uint64_t pol = evict_first_policy();
        const int kc = p.kseg / 512;  // chunks per segment
        int issued = 0;
        for (int st = 0; st < p.n_stages; ++st) {
            const int slot = st % SW, round = st / SW;
            if (round > 0 && !__all_sync(0xffffffffu, mbar_wait_spin(wempty0 + 8u * slot, (uint32_t)((round - 1) & 1)))) {
                if (lane == 0) report_timeout(p, abort_flag);
                break;
            }
            const int cg = st / S, s = st - cg * S;
            if (lane == 0) {
                const uint32_t full = wfull0 + 8u * slot;
                mbar_arrive_expect_tx(full, (uint32_t)(p.C * p.R * 128));
                tensor3d_g2s(ring_base + (uint32_t)(slot * p.stage_bytes), &p.wmap, 0,
                             (int)row0, s * kc + cg * p.C, full, pol);
            }
            __syncwarp();
            issued = st + 1;
        }
        for (int slot = 0; slot < SW && slot < issued; ++slot) {  // no copy in flight at exit
            const int last = slot + ((issued - 1 - slot) / SW) * SW;
            if (!mbar_wait_spin(wfull0 + 8u * slot, (uint32_t)((last / SW) & 1)) && lane == 0) report_timeout(p, abort_flag);
        }
        return;
    }

    if (warp == kMmaWarp) {
        // -------------------------------------------------- TMEM + MMA issue
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(&tmem_base_sh)),
                     "n"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        tc_fence_before();
        named_barrier(1, kThreads - 32);  // (a) TMEM address and B published
        tc_fence_after();
        const uint32_t tbase = tmem_base_sh;
        if (lane == 0) {
            const uint32_t idesc = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);
            const uint32_t b0 = smem_addr(smem + p.off_b0);
            const uint64_t desc_hi = ((uint64_t)((p.b_lbo & 0x3FFFFu) >> 4) << 16) | ((uint64_t)(128 >> 4) << 32) |
                                     ((uint64_t)1 << 46);
            const uint32_t tile_stride = 16u * (uint32_t)(S * kM);
            bool ok = true;
            for (int g = 0; g < kgroups && ok; ++g) {
                const int a = g & (kASlots - 1);
                if (!mbar_wait_spin(afull0 + 8u * a, (uint32_t)((g / kASlots) & 1))) {
                    report_timeout(p, abort_flag);
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int ks = 8 * g + i;
                    const uint64_t desc = desc_hi | (uint64_t)(((b0 + tile_stride * (uint32_t)ks) & 0x3FFFFu) >> 4);
                    umma_f16(tbase + kDCol + 16u * (uint32_t)(ks >> 4), tbase + (uint32_t)(a * kAColsPerSlot + 8 * i),
                             desc, idesc, (uint32_t)((ks & 15) != 0));
                }
                umma_commit(aempty0 + 8u * a);  // the slot is free once these MMAs completed
            }
            umma_commit(dfull);  // all MMAs issued above have completed
        }
        __syncwarp();
        named_barrier(2, kThreads - 32);  // (b) epilogue finished reading TMEM
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "n"(kTmemCols));
        return;
    }

    // ------------------------------------------------------ unpack / epilogue warps
    const int uw = warp - kFirstUnpackWarp;  // 0..7
    const int q = warp & 3;                  // TMEM lane quadrant this warp may access
    const int half = uw >> 2;                // groups g with g % 2 == half
    const int utid = uw * 32 + lane;         // 0..255
    const int tl = q * 32 + lane;            // TMEM lane
    const int s_lane = tl / p.lanes_per_seg;
    const int r_lane = tl - s_lane * p.lanes_per_seg;
    const bool lane_valid = r_lane < R_cta;
    const int B = p.B;
    const bool prologue = p.a.act_scale != 0.0f;
    float *xsum = reinterpret_cast<float *>(smem + p.off_xsum);
    float *rscale = reinterpret_cast<float *>(smem + p.off_rscale);
    float *dsm = reinterpret_cast<float *>(smem + p.off_dsm);
    float *red = reinterpret_cast<float *>(smem + p.off_red);

    // d slice of this CTA's rows (contiguous), fp32, loads batched before use
    {
        const int nd = R_cta * B;
        const uint16_t *dsrc = p.a.d + row0 * B;
        for (int base = 0; base < nd; base += 256 * 8) {
            uint16_t v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = base + j * 256 + utid;
                v[j] = (i < nd) ? dsrc[i] : (uint16_t)0;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int i = base + j * 256 + utid;
                if (i < nd) {
                    const int r = i / B, b = i - r * B;
                    dsm[r * p.dstr + b] = __half2float(__ushort_as_half(v[j]));
                }
            }
        }
    }

    asm volatile("griddepcontrol.wait;" ::: "memory");

    // x -> B arrays.  Word (m, block bg, word wb) -> k-step ks = 16 * (bg % nregions) + wb
    // of segment s = bg / nregions; 16 bytes at B0/B1 + 16 * (ks * S * M + s * M + m).
    {
        const uint32_t b0s = smem_addr(smem + p.off_b0), b1s = smem_addr(smem + p.off_b1);
        const int total = kM * B * 16;
        for (int base = uw * 32; base < total; base += 256) {
            const int L = base + lane;
            const bool act = L < total;  // uniform per half-warp (total % 16 == 0)
            uint32_t raw[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            int m = 0, bg = 0, wb = 0;
            if (act) {
                m = L / (B * 16);
                const int rem = L - m * B * 16;
                bg = rem >> 4;
                wb = rem & 15;
                const uint16_t *src = p.a.x + (int64_t)m * K + (int64_t)bg * 256 + wb * 16;
                const uint4 v0 = *reinterpret_cast<const uint4 *>(src);
                const uint4 v1 = *reinterpret_cast<const uint4 *>(src + 8);
                raw[0] = v0.x; raw[1] = v0.y; raw[2] = v0.z; raw[3] = v0.w;
                raw[4] = v1.x; raw[5] = v1.y; raw[6] = v1.z; raw[7] = v1.w;
                if (prologue) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&raw[j]));
                        const __half2 h2 = __floats2half2_rn(fq_code(f.x, p.a.inv_scale), fq_code(f.y, p.a.inv_scale));
                        raw[j] = *reinterpret_cast<const uint32_t *>(&h2);
                    }
                }
            }
            float sum = 0.0f, amax = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&raw[j]));
                sum += f.x + f.y;
                amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) {
                sum += __shfl_xor_sync(0xffffffffu, sum, off);
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            }
            if (act) {
                // 4^(3-c) exact unless 64 * max|x| would overflow fp16; then also 2^-6
                const bool big = amax > 1023.5f;
                const __half2 s64 = big ? __float2half2_rn(1.0f) : __float2half2_rn(64.0f);
                const __half2 s16 = big ? __float2half2_rn(0.25f) : __float2half2_rn(16.0f);
                const __half2 s4 = big ? __float2half2_rn(0.0625f) : __float2half2_rn(4.0f);
                const __half2 s1 = big ? __float2half2_rn(0.015625f) : __float2half2_rn(1.0f);
                auto pk = [&](uint32_t a_, uint32_t b_, uint32_t sel, __half2 sc) {
                    uint32_t v = __byte_perm(a_, b_, sel);
                    __half2 h = __hmul2(*reinterpret_cast<__half2 *>(&v), sc);
                    return *reinterpret_cast<uint32_t *>(&h);
                };
                // chunk0: (x0,x8) (x4,x12) x64 | (x1,x9) (x5,x13) x16 ; chunk1: (x2,x10) (x6,x14) x4 | (x3,x11) (x7,x15) x1
                const uint32_t c00 = pk(raw[0], raw[4], 0x5410u, s64), c01 = pk(raw[2], raw[6], 0x5410u, s64);
                const uint32_t c02 = pk(raw[0], raw[4], 0x7632u, s16), c03 = pk(raw[2], raw[6], 0x7632u, s16);
                const uint32_t c10 = pk(raw[1], raw[5], 0x5410u, s4), c11 = pk(raw[3], raw[7], 0x5410u, s4);
                const uint32_t c12 = pk(raw[1], raw[5], 0x7632u, s1), c13 = pk(raw[3], raw[7], 0x7632u, s1);
                const int s = bg / nregions, ks = 16 * (bg - s * nregions) + wb;
                const uint32_t off = 16u * (uint32_t)((ks * S + s) * kM + m);
                sts128(b0s + off, c00, c01, c02, c03);
                sts128(b1s + off, c10, c11, c12, c13);
                if ((lane & 15) == 0) {
                    xsum[bg * kM + m] = sum;
                    rscale[bg * kM + m] = big ? 16777216.0f : 262144.0f;  // 2^24 or 2^18
                }
            }
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // B: generic writes -> MMA reads
    named_barrier(1, kThreads - 32);                                // (a)
    tc_fence_after();
    const uint32_t tbase = tmem_base_sh;
    const uint32_t tlane = tbase + ((uint32_t)(q * 32) << 16);

    // unpack: group g (32 bytes per lane = 8 k-steps) of this lane's segment
    {
        const uint32_t ring = ring_base;
        bool alive = true;
        int cur_stage = -1;
        for (int g = half; g < kgroups; g += 2) {
            const int cs = g >> 2, u0 = (g & 3) * 2;  // 128-byte chunk, first 16-byte unit in it
            const int cg = cs / p.C, cc = cs - cg * p.C;
            const int sid = cg * S + s_lane;  // all lanes of a warp share s_lane
            const int slot = sid % SW;
            if (sid != cur_stage) {
                if (cur_stage >= 0 && lane == 0) mbar_arrive(wempty0 + 8u * (cur_stage % SW));
                cur_stage = sid;
                if (alive && !__all_sync(0xffffffffu, mbar_wait_spin(wfull0 + 8u * slot, (uint32_t)((sid / SW) & 1)))) {
                    if (lane == 0) report_timeout(p, abort_flag);
                    alive = false;
                }
            }
            const int a = g & (kASlots - 1);
            if (alive && g >= kASlots &&
                !__all_sync(0xffffffffu, mbar_wait_spin(aempty0 + 8u * a, (uint32_t)(((g / kASlots) - 1) & 1)))) {
                if (lane == 0) report_timeout(p, abort_flag);
                alive = false;
            }
            uint4 w0 = make_uint4(0u, 0u, 0u, 0u), w1 = w0;
            if (alive && lane_valid) {
                const int line = cc * p.R + r_lane;
                const uint32_t lbase = ring + (uint32_t)(slot * p.stage_bytes + line * 128);
                w0 = lds128(lbase + (((u0) ^ (line & 7)) << 4));
                w1 = lds128(lbase + (((u0 + 1) ^ (line & 7)) << 4));
            }
            const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            uint32_t v[32];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t lo = ws[4 * h2 + i], hi = lo >> 8;
                    v[8 * i + 0] = lo & 0x00030003u;
                    v[8 * i + 1] = hi & 0x00030003u;
                    v[8 * i + 2] = lo & 0x000C000Cu;
                    v[8 * i + 3] = hi & 0x000C000Cu;
                    v[8 * i + 4] = lo & 0x00300030u;
                    v[8 * i + 5] = hi & 0x00300030u;
                    v[8 * i + 6] = lo & 0x00C000C0u;
                    v[8 * i + 7] = hi & 0x00C000C0u;
                }
                if (alive) tmem_st32(tlane + (uint32_t)(a * kAColsPerSlot + 32 * h2), v);
            }
            if (alive) {
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(afull0 + 8u * a);
        }
        if (cur_stage >= 0 && lane == 0) mbar_arrive(wempty0 + 8u * (cur_stage % SW));
    }

    // epilogue: D -> per-lane partial -> per-row sum over the K segments
    const bool dok = __all_sync(0xffffffffu, mbar_wait_spin(dfull, 0u));
    if (!dok && lane == 0) report_timeout(p, abort_flag);
    tc_fence_after();
    if (half == 0) {
        float acc[kM];
#pragma unroll
        for (int m = 0; m < kM; ++m) acc[m] = 0.0f;
        for (int b = 0; b < nregions; ++b) {
            const int bg = s_lane * nregions + b;
            const float db = lane_valid ? dsm[r_lane * p.dstr + bg] : 0.0f;
#pragma unroll
            for (int m = 0; m < kM; ++m) {
                const uint32_t raw = tmem_ld1(tlane + (uint32_t)(kDCol + 16 * b + s_lane * kM + m));
                tmem_ld_wait();
                const float dv = __uint_as_float(raw);
                acc[m] = fmaf(db, fmaf(dv, rscale[bg * kM + m], -xsum[bg * kM + m]), acc[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < kM; ++m) red[(s_lane * p.lanes_per_seg + r_lane) * kM + m] = lane_valid ? acc[m] : 0.0f;
    }
    tc_fence_before();
    named_barrier(2, kThreads - 32);  // (b): TMEM reads done, red complete
    if (*abort_flag) return;
    for (int i = utid; i < kM * R_cta; i += 256) {
        const int m = i / R_cta, r = i - m * R_cta;
        float v = 0.0f;
        for (int s = 0; s < S; ++s) v += red[(s * p.lanes_per_seg + r) * kM + m];
        if (prologue) v *= p.a.act_scale;
        v = requant_out(v, p.a.out_scale, p.a.inv_out);
        const int64_t o = (int64_t)m * N + row0 + r;
        if (p.a.y_f16)
            reinterpret_cast<__half *>(p.a.y)[o] = __float2half_rn(v);
        else
            reinterpret_cast<float *>(p.a.y)[o] = v;
    }
}

// ------------------------------------------------------------------ host side
int align_up(int v, int a) { return (v + a - 1) / a * a; }

// Plan: rows per CTA, K segments, stage geometry, shared-memory layout.
bool make_plan(int M, int64_t N, int64_t K, int nsm, int max_dyn, Tc05Params &p)
{
    if (M < 1 || M > 2 || N < 1 || K < 512 || K % 512 != 0) return false;
    int64_t R = (N + nsm - 1) / nsm;
    if (R < 1) R = 1;
    int S = 4;
    while (S > 1 && (R * S > 128 || (K / S) % 512 != 0 || S * M > 8)) S >>= 1;
    if (R * S > 128) R = 128 / S;  // more CTAs (several waves) for very large N
    const int64_t kseg = K / S;
    if (kseg > 4096 || kseg % 512 != 0) return false;
    p.R = (int)R;
    p.S = S;
    p.lanes_per_seg = 128 / S;
    p.kseg = (int)kseg;
    p.B = (int)(K / 256);
    int C = 1;
    while (C * 2 <= (int)(kseg / 512) && (C * 2) * p.R * 128 <= 16384) C *= 2;
    p.C = C;
    p.stage_bytes = align_up(C * p.R * 128, 1024);
    p.n_stages = S * (int)(kseg / 512) / C;
    p.dstr = p.B + 1;
    int off = 0;
    p.off_bar = off;
    off += 8 * (2 * 8 + 2 * kASlots + 1);
    off = align_up(off, 128);
    const int bbytes = 2 * M * (int)K / 2 + 256;  // one of the two arrays: M*K bytes + padding
    p.off_b0 = off;
    off += align_up(bbytes, 128);
    p.off_b1 = off;
    off += align_up(bbytes, 128);
    p.b_lbo = (uint32_t)(p.off_b1 - p.off_b0);
    p.off_xsum = off;
    off += align_up(p.B * M * 4, 16);
    p.off_rscale = off;
    off += align_up(p.B * M * 4, 16);
    p.off_dsm = off;
    off += align_up(p.R * p.dstr * 4, 16);
    p.off_red = off;
    off += align_up(128 * M * 4, 16);
    off = align_up(off, 1024);
    p.off_ring = off;
    off += 1024;  // runtime alignment slack of the ring base
    // The S segments advance together (they share the TMEM A slots), so all S
    // stages of a chunk group must fit in the ring at once: depth >= S.
    const int need = (S < 2) ? 2 : S;
    int SW = (kTargetSmem - off) / p.stage_bytes;
    if (SW > 8) SW = 8;
    if (SW < need) SW = (max_dyn - off) / p.stage_bytes;
    if (SW > 8) SW = 8;
    if (SW < need) return false;
    p.stages = SW;
    p.smem_total = off + SW * p.stage_bytes;
    return p.smem_total <= max_dyn;
}

std::atomic<int> g_tc05_dyn[2][64];

template <int kM>
int tc05_max_dyn(int device)
{
    if (device < 0 || device >= 64) return 0;
    int v = g_tc05_dyn[kM - 1][device].load();
    if (v > 0) return v;
    int optin = 0;
    cudaFuncAttributes fa;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, matvec_tc05_kernel<kM>) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    v = optin - (int)fa.sharedSizeBytes;
    if (cudaFuncSetAttribute(matvec_tc05_kernel<kM>, cudaFuncAttributeMaxDynamicSharedMemorySize, v) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    g_tc05_dyn[kM - 1][device].store(v);
    return v;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder()
{
    static std::atomic<void *> fn{nullptr};
    void *f = fn.load();
    if (f) return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || f == nullptr) {
        cudaGetLastError();
        return nullptr;
    }
    fn.store(f);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

template <int kM>
cudaError_t launch_tc05(const MatvecArgs &a, int device)
{
    Tc05Params p{};
    p.a = a;
    if (!make_plan(kM, a.N, a.K, sm_count(device), tc05_max_dyn<kM>(device), p)) return cudaErrorInvalidConfiguration;
    PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    // qs viewed as uint64 [K/512][N][16]: dim0 16 words of a 128-byte chunk, dim1 rows, dim2 chunks
    const cuuint64_t dims[3] = {16, (cuuint64_t)a.N, (cuuint64_t)(a.K / 512)};
    const cuuint64_t strides[2] = {(cuuint64_t)(a.K / 4), 128};
    const cuuint32_t box[3] = {16, (cuuint32_t)p.R, (cuuint32_t)p.C};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&p.wmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint8_t *>(a.qs), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int G = (int)((a.N + p.R - 1) / p.R);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)p.smem_total;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, matvec_tc05_kernel<kM>, p);
}

}  // namespace

bool tc05_matvec_supported(int M, int64_t N, int64_t K, int device)
{
    if (M < 1 || M > 2) return false;
    Tc05Params p{};
    const int dyn = (M == 1) ? tc05_max_dyn<1>(device) : tc05_max_dyn<2>(device);
    return dyn > 0 && make_plan(M, N, K, sm_count(device), dyn, p);
}

cudaError_t launch_matvec_tc05(const MatvecArgs &a, int device)
{
    if (a.M == 1) return launch_tc05<1>(a, device);
    if (a.M == 2) return launch_tc05<2>(a, device);
    return cudaErrorInvalidValue;
}

}  // namespace tq2
