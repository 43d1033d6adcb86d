// tq2_gemm_tc05.cu -- ternary GEMM for prefill-sized M on the 5th-generation
// tensor cores (sm_103a): tcgen05.mma with the weights in tensor memory, x
// tiles brought by TMA, one fp32 accumulator in tensor memory.
//
// What it computes (BitCPM ternary page, linear-factoring paragraph), for any
// number M of activation rows:
//   y[m][n] = sum_b d[n][b] * sum_{k in b} x[m][k] * (q[n][k] - 1)
// Each (q - 1) * d_b is one of -d_b, 0, +d_b and therefore exact in fp16, and
// an fp16 x fp16 product is exact in fp32, so with many activation rows the
// matvec becomes a plain dense contraction W' x^T with W'[n][k] = (q - 1) d_b:
// the weights are expanded once per tile and the tensor cores accumulate over
// all of K with no per-block epilogue (the d_b and the "-1" live in W').
//
// Tile: 128 weight rows (the MMA's M, one TMEM lane each) x BN activation rows
// (the MMA's N: 16, 32 or 64 for up to 64 rows -- an MMA with N <= 64 costs
// about the same as with N = 16 -- else 128 or 256), all of K;
// tcgen05.mma.cta_group::1.kind::f16, K = 16 per instruction.
//   * warp 0 streams the packed codes: 2-D TMA boxes of 128 rows x 64 bytes
//     (one 256-block), before griddepcontrol.wait (weights never depend on
//     earlier kernels);
//   * warp 1 streams x after griddepcontrol.wait: per stage (8 k-steps) two
//     TMA boxes of 64 values x BN rows, 128 bytes per row with the 128-byte
//     swizzle, which is the K-major SWIZZLE_128B operand layout the MMA reads
//     (8-row groups 1024 bytes apart; k-step j of a box starts 32 j bytes
//     into the row); rows past M read as 0;
//   * warp 2 allocates the TMEM columns (after the wait, so the previous
//     kernel's tensor memory is free: 256 for tiles of up to 64 columns, so
//     that two CTAs share an SM, else 512); one lane issues the MMAs of a
//     stage and releases its A slot and x buffer with one commit (a commit
//     stalls the issuing thread for hundreds of cycles on this part, so
//     there is one per stage).  For tiles of up to 128 columns a lane of
//     warp 11 issues every other k-step into a second accumulator (one
//     thread issues an MMA only every ~126 cycles), and the epilogue sums
//     the two;
//   * warps 3..10 (two per TMEM lane quadrant) stage d, then expand 8 k-steps
//     at a time: for code pair (2j, 2j+1) of a 16-code word, the fp16 pair
//     (1024 + q) - 1025 = q - 1 (exact) times d_b, written with tcgen05.st
//     into a ring of 64-column TMEM slots (one per stage); with the int8
//     prologue and no workspace (given one, x arrives as codes from the
//     conversion pass) they also fake-quantise each x stage in shared memory first
//     (element-wise, by the half of the warps that expands the stage, a
//     quarter each, so the halves stay independent) and release it to the MMA
//     issuer (a generic-to-async proxy fence, then an mbarrier); at the end
//     they read D (one
//     column per activation row; the accumulators summed) and store y, with
//     the optional int8 requantisation at store.
// Split K: when the tiles alone would leave SMs idle, a thread-block cluster
// of S CTAs shares a tile, CTA r taking 256-blocks [r B / S, (r+1) B / S).
// Each writes its fp32 partial tile to its own shared memory; CTA r then sums
// its 1/S of the columns over the S partials (distributed shared memory, a
// fixed order, so the result is the same on every run) and stores them.  The
// cross-CTA hand-offs are mbarriers with remote arrivals and bounded waits.
// Every mbarrier wait is bounded; a wait that runs out sets TQ2_FLAG_TIMEOUT.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>

#include "tq2_device.cuh"
#include "tq2_internal.cuh"
#include "tq2_tcgen05.cuh"

namespace tq2 {
namespace {

using namespace dev;

constexpr int kWProducerWarp = 0;
constexpr int kBProducerWarp = 1;
constexpr int kMmaWarp = 2;               // tensor memory, MMA issue (even k-steps)
constexpr int kFirstUnpackWarp = 3;
constexpr int kUnpackWarps = 8;
constexpr int kMmaWarp2 = kFirstUnpackWarp + kUnpackWarps;  // MMA issue (odd k-steps), 11, if two issuers
constexpr int kRows = 128;               // weight rows per tile (MMA M, TMEM lanes)
constexpr int kKs = 8;                   // k-steps (16 codes) per stage: one A slot, two x boxes
constexpr int kWStageBytes = 8192;       // 128 rows x 64 bytes of codes (16 k-steps, one 256-block)
constexpr int kASlots = 4;               // TMEM A ring, at most
constexpr int kAColsPerSlot = 64;        // 8 k-steps x 8 columns

// MMA issue: one thread issues a tcgen05.mma about every 126 cycles on this
// part, whatever the operands' source or the accumulator (measured), while
// a 128 x BN x 16 MMA takes the tensor cores ~BN / 1.7 cycles: one issuing
// thread bounds every tile narrower than ~200 columns.  So two warps issue:
// warp kMmaWarp the even k-steps of each stage, warp kMmaWarp2 the odd ones,
// each into its own accumulator tile (tcgen05 MMAs of different threads are
// not ordered with one another), and the epilogue sums the two tiles in tile
// order.  A 256-column tile has room for one accumulator and a long enough
// MMA: one issuer.
//
// Tensor memory per CTA.  A tile of up to 64 activation rows takes half of
// the SM's 512 columns -- the accumulators first, then the A slots -- so
// that two CTAs fit on an SM (the next call's CTA starts beside the current
// one and streams its weights early); wider tiles take all 512 (four A
// slots at 0..255, the accumulators from 256), one CTA per SM.  The host
// sizes shared memory so that no more CTAs than that fit on an SM
// (tcgen05.alloc would otherwise wait for columns that a CTA of another
// cluster holds).  The epilogue's 32-column loads of a narrow tile run on
// into later columns, inside the allocation, which no MMA writes by then
// (masked).
template <int BN>
struct Tmem {
    static constexpr int issuers = BN <= 128 ? 2 : 1;
    static constexpr int threads = (kMmaWarp2 + issuers - 1) * 32;           // 384 or 352
    static constexpr int tmem_threads = (kUnpackWarps + issuers) * 32;       // MMA warps + unpack warps
    static constexpr int nd = issuers;                      // accumulator tiles
    static constexpr int cols = BN <= 64 ? 256 : 512;
    static constexpr int dcol = BN <= 64 ? 0 : 256;         // accumulator tile 0
    static constexpr int acol = BN <= 32 ? 64 : BN <= 64 ? 128 : 0;  // A slot 0
    static constexpr int slots = BN <= 64 ? (cols - acol) / 64 : 4;
    static_assert(dcol + (nd - 1) * BN + (BN < 64 ? BN / 2 + 32 : BN) <= cols, "epilogue loads past the columns");
    static_assert(BN <= 64 ? nd * BN <= acol : acol + slots * 64 <= dcol, "A slots overlap the accumulators");
    static_assert(acol + slots * 64 <= cols && dcol + nd * BN <= cols, "past the columns");
    static_assert(slots >= 2 && slots <= 4, "A ring depth");
};

int tmem_slots(int BN)
{
    return BN <= 16 ? Tmem<16>::slots : BN <= 32 ? Tmem<32>::slots : BN <= 64 ? Tmem<64>::slots
         : BN <= 128 ? Tmem<128>::slots : Tmem<256>::slots;
}
constexpr int kMaxStages = 8;

struct GemmParams {
    CUtensorMap wmap;  // qs as uint64 [N][K/32]; box {8, 128}; no swizzle
    CUtensorMap xmap;  // x as fp16 [M][K]; box {64, BN}; 128-byte swizzle
    MatvecArgs a;
    int n_tiles;       // weight-row tiles (ceil(N / 128)); tile = m_tile * n_tiles + n_tile
    int S;             // CTAs per tile (cluster size; split of K), blockIdx = tile * S + rank
    int B;             // 256-blocks per row
    int sw, sb;        // ring depths: codes; stages (A slots and x buffers, <= 4)
    int off_bar, off_dsm, off_w, off_b, smem_total;  // the x ring also holds the partial tile when S > 1
};

__device__ __forceinline__ void report_timeout(const GemmParams &p, volatile int *flag)
{
    *flag = 1;
    if (p.a.status) atomicOr(p.a.status, TQ2_FLAG_TIMEOUT);
}

// The 8 TMEM columns of one k-step for one weight row: column j holds the
// fp16 pair ((q[2j] - 1) d, (q[2j+1] - 1) d) of the 16-code word w.
__device__ __forceinline__ void expand_word(uint32_t w, __half2 dd, uint32_t *o)
{
    const uint32_t src[4] = {w, w >> 2, w >> 4, w >> 6};  // code pairs at bits 0-1 of each byte
    const __half2 bias = __float2half2_rn(-1025.0f);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t byte = (uint32_t)(j >> 1), odd = (uint32_t)(j & 1);
        // q[2j] -> bits 0-1 of lane 0, q[2j+1] -> bits 16-17 of lane 1
        const uint32_t t = __byte_perm(src[2 * odd], src[2 * odd + 1], byte | ((4u + byte) << 8));
        const uint32_t f = (t & 0x00030003u) | 0x64006400u;  // fp16 (1024 + q, 1024 + q')
        const __half2 h = __hmul2(__hadd2(*reinterpret_cast<const __half2 *>(&f), bias), dd);
        o[j] = *reinterpret_cast<const uint32_t *>(&h);
    }
}

// ------------------------------------------------------------------ kernel
template <int BN>
__global__ void __launch_bounds__(Tmem<BN>::threads, 1) gemm_tc05_kernel(const __grid_constant__ GemmParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    volatile int *abort_flag = &abort_sh;
    constexpr uint32_t kBoxBytes = (uint32_t)BN * 128u;     // 64 values per row
    constexpr uint32_t kBStageBytes = 2u * kBoxBytes;       // kKs = 8 k-steps

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t N = p.a.N;
    const int M = p.a.M;
    const int S = p.S;
    const int rank = (int)(blockIdx.x % (unsigned)S), tile = (int)(blockIdx.x / (unsigned)S);
    const int ntile = tile % p.n_tiles, mtile = tile / p.n_tiles;
    const int64_t n0 = (int64_t)ntile * kRows;
    const int m0 = mtile * BN;
    // this CTA's 256-blocks [w0, w1) of K; all indices below are local to it
    const int w0 = (int)((int64_t)rank * p.B / S), w1 = (int)((int64_t)(rank + 1) * p.B / S);
    const int nwst = w1 - w0;                    // code stages (one 256-block each)
    const int ngroups = 2 * nwst;                // stages of 8 k-steps (TMEM A fills, x buffers)
    const int nbst = ngroups;
    const int SW = p.sw, SB = p.sb;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + p.off_bar);
    const uint32_t wfull0 = smem_addr(bars), wempty0 = wfull0 + 8u * SW;
    // stage slot r: bfull (x landed), bconv (x fake-quantised, prologue
    // only), afull (A slot written), sempty (the MMAs of the stage completed:
    // both the A slot and the x buffer are free)
    const uint32_t bfull0 = wempty0 + 8u * SW, bconv0 = bfull0 + 8u * SB, afull0 = bconv0 + 8u * SB;
    const uint32_t sempty0 = afull0 + 8u * SB;
    const uint32_t dfull = sempty0 + 8u * SB;
    const uint32_t pready = dfull + 8u, pdone = pready + 8u;  // split K: peers' partials written / read
    // the x tiles are fake-quantised here unless x already holds the codes
    const bool prologue = p.a.act_scale != 0.0f && !p.a.x_codes;
    // the x ring must be 1024-byte aligned for the 128-byte swizzle (the plan
    // reserves the slack; both rings move together)
    const uint32_t wring = (smem_addr(smem + p.off_w) + 1023u) & ~1023u;
    const uint32_t bring = (smem_addr(smem + p.off_b) + 1023u) & ~1023u;
    // limit of the stage-ring waits (the completion, tensor-memory and
    // cluster hand-off waits keep kTimeoutNs, so that a short test limit
    // never lets a CTA leave while its peers or its MMAs still need it)
    const unsigned long long lim = p.a.wait_limit_ns ? p.a.wait_limit_ns : kTimeoutNs;
    uint32_t *const st_w = p.a.status;  // TQ2_FLAG_BOUNDS of debug builds
    const SmemWindow win{smem_addr(smem), smem_addr(smem) + (uint32_t)p.smem_total, st_w};

    asm volatile("griddepcontrol.launch_dependents;");
    if (tid == 0) {
        for (int i = 0; i < SW; ++i) {
            mbar_init(wfull0 + 8u * i, 1);
            mbar_init(wempty0 + 8u * i, kUnpackWarps);
        }
        for (int i = 0; i < SB; ++i) {
            mbar_init(bfull0 + 8u * i, 1);
            mbar_init(bconv0 + 8u * i, kUnpackWarps / 2);  // the half that expands the stage converts it
            mbar_init(afull0 + 8u * i, 4);
            mbar_init(sempty0 + 8u * i, Tmem<BN>::issuers);  // one commit per issuer
        }
        mbar_init(dfull, Tmem<BN>::issuers);
        if (S > 1) {
            mbar_init(pready, (uint32_t)(S - 1));
            mbar_init(pdone, (uint32_t)(S - 1));
        }
        abort_sh = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (S > 1) {  // every CTA's barriers exist before any peer arrives on them
        asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    }

    if (warp == kWProducerWarp) {
        // -------------------------------------------------- codes -> shared memory
        const uint64_t pol = evict_first_policy();
        int issued = 0;
        for (int s = 0; s < nwst; ++s) {
            const int slot = s % SW, round = s / SW;
            if (round > 0 && !__all_sync(0xffffffffu, mbar_wait_for(wempty0 + 8u * slot, (uint32_t)((round - 1) & 1), lim))) {
                if (lane == 0) report_timeout(p, abort_flag);
                break;
            }
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            if (lane == 0 && TQ2_IN(wring + (uint32_t)((slot + 1) * kWStageBytes) <= win.hi, st_w)) {
                const uint32_t full = wfull0 + 8u * slot;
                mbar_arrive_expect_tx(full, (uint32_t)kWStageBytes);
                tensor2d_g2s(wring + (uint32_t)(slot * kWStageBytes), &p.wmap, 8 * (w0 + s), (int)n0, full, pol);
            }
            __syncwarp();
            issued = s + 1;
        }
        for (int slot = 0; slot < SW && slot < issued; ++slot) {  // no copy in flight at exit
            const int last = slot + ((issued - 1 - slot) / SW) * SW;
            if (!mbar_wait_for(wfull0 + 8u * slot, (uint32_t)((last / SW) & 1), lim) && lane == 0) report_timeout(p, abort_flag);
        }
        return;
    }

    if (warp == kBProducerWarp) {
        // -------------------------------------------------- x -> shared memory
        asm volatile("griddepcontrol.wait;" ::: "memory");  // x may come from the previous kernel
        const uint64_t pol = evict_last_policy();           // every weight tile reads it again
        int issued = 0;
        for (int s = 0; s < nbst; ++s) {
            const int slot = s % SB, round = s / SB;
            if (round > 0 && !__all_sync(0xffffffffu, mbar_wait_for(sempty0 + 8u * slot, (uint32_t)((round - 1) & 1), lim))) {
                if (lane == 0) report_timeout(p, abort_flag);
                break;
            }
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            if (s == p.a.stall_stage) {  // test hook: no copy for this stage
                issued = s + 1;
                continue;
            }
            const uint32_t full = bfull0 + 8u * slot;
            const bool in = TQ2_IN(bring + (uint32_t)(slot + 1) * kBStageBytes <= win.hi, st_w);
            if (lane == 0 && in) mbar_arrive_expect_tx(full, kBStageBytes);
            __syncwarp();
            if (lane < 2 && in)
                tensor2d_g2s(bring + (uint32_t)slot * kBStageBytes + (uint32_t)lane * kBoxBytes, &p.xmap,
                             256 * w0 + 16 * kKs * s + 64 * lane, m0, full, pol);
            __syncwarp();
            issued = s + 1;
        }
        // (a slot is refilled only after the MMAs that read its previous
        // stage completed, so only its last copy can be in flight; a skipped
        // stage had none: its slot's last copy is the one before it)
        for (int slot = 0; slot < SB && slot < issued; ++slot) {
            int last = slot + ((issued - 1 - slot) / SB) * SB;
            if (last == p.a.stall_stage) last -= SB;
            if (last >= 0 && !mbar_wait_for(bfull0 + 8u * slot, (uint32_t)((last / SB) & 1), lim) && lane == 0)
                report_timeout(p, abort_flag);
        }
        return;
    }

    if (warp == kMmaWarp || warp == kMmaWarp2) {
        // -------------------------------------------------- TMEM + MMA issue
        const int w = (warp == kMmaWarp) ? 0 : 1;  // this issuer's k-steps: i % issuers == w
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (w == 0) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                             smem_addr(&tmem_base_sh)),
                         "n"(Tmem<BN>::cols));
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
        }
        tc_fence_before();
        named_barrier(1, Tmem<BN>::tmem_threads);  // (a) TMEM address published
        tc_fence_after();
        const uint32_t tbase = tmem_base_sh;
        if (lane == 0 && w < Tmem<BN>::issuers) {
            const uint32_t idesc = (1u << 4) | ((uint32_t)(BN >> 3) << 17) | ((128u >> 4) << 24);
            // K-major, 128-byte swizzle: 8-row groups 1024 bytes apart (the
            // leading offset is unused in this mode), layout type 2
            const uint64_t desc_hi = ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) |
                                     ((uint64_t)2 << 61);
            for (int g = 0; g < ngroups; ++g) {
                const int r = g % SB;
                const uint32_t par = (uint32_t)((g / SB) & 1);
                if (!mbar_wait_for(afull0 + 8u * r, par, lim) || !mbar_wait_for((prologue ? bconv0 : bfull0) + 8u * r, par, lim)) {
                    report_timeout(p, abort_flag);
                    break;
                }
                tc_fence_after();
                const uint32_t b0 = bring + (uint32_t)r * kBStageBytes;
                constexpr int ni = Tmem<BN>::issuers;
#pragma unroll
                for (int i0 = 0; i0 < kKs; i0 += ni) {
                    const int i = i0 + w;
                    const uint32_t baddr = b0 + (uint32_t)(i >> 2) * kBoxBytes + (uint32_t)(32 * (i & 3));
                    const uint64_t desc = desc_hi | (uint64_t)((baddr & 0x3FFFFu) >> 4);
                    umma_f16(tbase + (uint32_t)(Tmem<BN>::dcol + w * BN),
                             tbase + (uint32_t)(Tmem<BN>::acol + r * kAColsPerSlot + 8 * i), desc, idesc,
                             (uint32_t)(g != 0 || i0 != 0));  // this issuer's first k-step overwrites its tile
                }
                umma_commit(sempty0 + 8u * r);  // A slot and x buffer free once these MMAs completed
            }
            umma_commit(dfull);  // every MMA issued above has completed
            // tensor memory is freed only once those MMAs are done, even if
            // the epilogue's own wait for them ran out
            if (!mbar_wait(dfull, 0u)) report_timeout(p, abort_flag);
        }
        __syncwarp();
        named_barrier(2, Tmem<BN>::tmem_threads);  // (b) the epilogue has read D
        tc_fence_after();
        if (w == 0)
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "n"(Tmem<BN>::cols));
        return;
    }

    // ------------------------------------------------------ expand / epilogue warps
    const int uw = warp - kFirstUnpackWarp;  // 0..7
    const int q = warp & 3;                  // TMEM lane quadrant this warp may access
    const int half = uw >> 2;                // expands the groups g with g % 2 == half
    const int row = q * 32 + lane;           // weight row in the tile = TMEM lane
    const int64_t n = n0 + row;
    const int B = p.B;
    uint16_t *dsm = reinterpret_cast<uint16_t *>(smem + p.off_dsm);  // [B][128] fp16, 0 past N

    for (int i = uw * 32 + lane; i < kRows * B; i += kUnpackWarps * 32) {
        const int r = i / B, b = i - r * B;  // row-major reads of d
        if (TQ2_IN(i < p.B * kRows, st_w))
            dsm[b * kRows + r] = (n0 + r < N) ? p.a.d[(n0 + r) * (int64_t)B + b] : (uint16_t)0;
    }
    named_barrier(3, kUnpackWarps * 32);  // d staged
    named_barrier(1, Tmem<BN>::tmem_threads);       // (a)
    tc_fence_after();
    const uint32_t tbase = tmem_base_sh;
    const uint32_t tlane = tbase + ((uint32_t)(q * 32) << 16);

    {
        bool alive = true;
        int cur_w = -1;
        for (int g = half; g < ngroups; g += 2) {
            if (prologue) {
                // x' = clamp(rint(x * (1/s)), -128, 127) (times s at the store),
                // in place, by the half of the warps that expands stage g (a
                // quarter each): the two halves stay independent, as without
                // the prologue
                const int r = g % SB;
                if (alive &&
                    !__all_sync(0xffffffffu, mbar_wait_for(bfull0 + 8u * (uint32_t)r, (uint32_t)((g / SB) & 1), lim))) {
                    if (lane == 0) report_timeout(p, abort_flag);
                    alive = false;
                }
                if (alive) {
                    const uint32_t xb = bring + (uint32_t)r * (2u * BN * 128u);
                    for (int c = (uw & 3) * 32 + lane; c < 2 * BN * 8; c += (kUnpackWarps / 2) * 32) {
                        const uint4 v = lds128_c(win, xb + (uint32_t)c * 16u);
                        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[e]));
                            const __half2 h = __floats2half2_rn(fq_code(f.x, p.a.inv_scale), fq_code(f.y, p.a.inv_scale));
                            w[e] = *reinterpret_cast<const uint32_t *>(&h);
                        }
                        if (TQ2_IN(xb + (uint32_t)c * 16u + 16u <= win.hi, st_w))
                        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(xb + (uint32_t)c * 16u),
                                     "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                                     : "memory");
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic writes -> MMA reads
                }
                __syncwarp();
                if (alive && lane == 0) mbar_arrive(bconv0 + 8u * (uint32_t)r);
            }
            const int ws = g >> 1;           // code stage (2 groups)
            const int u0 = (g & 1) * 2;      // first 16-byte unit of the group in the row
            const int slot = ws % SW;
            if (ws != cur_w) {
                if (alive && cur_w >= 0 && lane == 0) mbar_arrive(wempty0 + 8u * (cur_w % SW));
                cur_w = ws;
                if (alive && !__all_sync(0xffffffffu, mbar_wait_for(wfull0 + 8u * slot, (uint32_t)((ws / SW) & 1), lim))) {
                    if (lane == 0) report_timeout(p, abort_flag);
                    alive = false;
                }
            }
            const int a = g % SB;  // stage slot: TMEM A slot a
            if (alive && g >= SB &&
                !__all_sync(0xffffffffu, mbar_wait_for(sempty0 + 8u * a, (uint32_t)(((g / SB) - 1) & 1), lim))) {
                if (lane == 0) report_timeout(p, abort_flag);
                alive = false;
            }
            uint4 c0 = make_uint4(0u, 0u, 0u, 0u), c1 = c0;
            if (alive) {
                const uint32_t lbase = wring + (uint32_t)(slot * kWStageBytes + row * 64);
                c0 = lds128_c(win, lbase + (uint32_t)(u0 << 4));
                c1 = lds128_c(win, lbase + (uint32_t)((u0 + 1) << 4));
            }
            const __half hd = __ushort_as_half(dsm[(w0 + (g >> 1)) * kRows + row]);  // block of the group
            const __half2 dd = __halves2half2(hd, hd);
            const uint32_t wd[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t v[32];
#pragma unroll
                for (int i = 0; i < 4; ++i) expand_word(wd[4 * h2 + i], dd, &v[8 * i]);
                if (alive && TQ2_IN(a < Tmem<BN>::slots, st_w))
                    tmem_st32(tlane + (uint32_t)(Tmem<BN>::acol + a * kAColsPerSlot + 32 * h2), v);
            }
            if (alive) {
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                tc_fence_before();
            }
            // a warp whose wait ran out releases nothing it did not wait
            // for: no slot is refilled while its last copy may be in flight,
            // and no barrier runs a phase ahead of its waiters
            __syncwarp();
            if (alive && lane == 0) mbar_arrive(afull0 + 8u * a);
        }
        if (alive && cur_w >= 0 && lane == 0) mbar_arrive(wempty0 + 8u * (cur_w % SW));
    }

    // epilogue: D column c is activation row m0 + c; this warp takes half of them
    const bool dok = __all_sync(0xffffffffu, mbar_wait(dfull, 0u));
    if (!dok && lane == 0) report_timeout(p, abort_flag);
    tc_fence_after();
    auto store_y = [&](int m, int64_t nn, float v) {
        if (p.a.act_scale != 0.0f) v *= p.a.act_scale;
        v = requant_out(v, p.a.out_scale, p.a.inv_out);
        const int64_t o = (int64_t)m * N + nn;
        if (!TQ2_IN(o < (int64_t)M * N, st_w)) return;
        if (p.a.y_f16)
            reinterpret_cast<__half *>(p.a.y)[o] = __float2half_rn(v);
        else
            reinterpret_cast<float *>(p.a.y)[o] = v;
    };
    // each half of the warps reads BN / 2 columns, 32 at a time (the load of
    // a narrow tile's last chunk runs past BN into unused columns: masked),
    // summed over the accumulator tiles in tile order
    const int c_beg = half * (BN / 2), c_end = c_beg + BN / 2;
    auto load_d = [&](int c0, float *v) {
        uint32_t r[32];
        tmem_ld32(tlane + (uint32_t)(Tmem<BN>::dcol + c0), r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
#pragma unroll 1
        for (int t = 1; t < Tmem<BN>::nd; ++t) {
            tmem_ld32(tlane + (uint32_t)(Tmem<BN>::dcol + t * BN + c0), r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += __uint_as_float(r[j]);
        }
    };
    if (S == 1) {
        const bool store = (*abort_flag == 0) && n < N;
#pragma unroll 1
        for (int c0 = c_beg; c0 < c_end; c0 += 32) {
            float v[32];
            load_d(c0, v);
            if (store) {
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (c0 + j < c_end && m0 + c0 + j < M) store_y(m0 + c0 + j, n, v[j]);
            }
        }
        tc_fence_before();
        named_barrier(2, Tmem<BN>::tmem_threads);  // (b)
        return;
    }

    // split K: partial tile -> own shared memory (the x ring, idle now),
    // column-major [BN][128] fp32
    float *part = reinterpret_cast<float *>(smem + p.off_b);
#pragma unroll 1
    for (int c0 = c_beg; c0 < c_end; c0 += 32) {
        float v[32];
        load_d(c0, v);
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (c0 + j < c_end && TQ2_IN(smem_addr(&part[(c0 + j) * kRows + row]) + 4u <= win.hi, st_w))
                part[(c0 + j) * kRows + row] = v[j];
    }
    tc_fence_before();
    named_barrier(2, Tmem<BN>::tmem_threads);       // (b): TMEM read, the MMA warp may free it
    named_barrier(3, kUnpackWarps * 32);  // every partial of this CTA written
    const uint32_t part_s = smem_addr(part);
    if (uw == 0 && lane < S && lane != rank) {  // tell every peer: my partial is ready
        // A CTA that gave up (a bounded wait ran out) first sets every peer's
        // abort flag, so that no peer reads its partial: its shared memory
        // must not be touched once it may exit (ordered before the arrival
        // by the release fence).
        if (*abort_flag != 0) {
            uint32_t rflag;
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rflag) : "r"(smem_addr(&abort_sh)), "r"(lane));
            asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(rflag), "r"(1u) : "memory");
        }
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(pready), "r"(lane));
        asm volatile("fence.acq_rel.cluster;\n\tmbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];"
                     ::"r"(remote) : "memory");
    }
    bool ok = __all_sync(0xffffffffu, mbar_wait_cluster(pready, 0u));
    if (!ok && lane == 0) report_timeout(p, abort_flag);
    // a peer that gave up has set this CTA's flag before its arrival: no remote
    // reads then (the result is invalid and TQ2_FLAG_TIMEOUT reported anyway)
    ok = ok && !__any_sync(0xffffffffu, *abort_flag != 0);
    // this CTA's columns [rank BN/S, (rank+1) BN/S), summed over the S partials in rank order
    const int cols = BN / S, c_lo = rank * cols;
    const int tid_u = uw * 32 + lane;
    if (ok) {
        for (int i = tid_u; i < cols * kRows; i += kUnpackWarps * 32) {
            const int c = c_lo + i / kRows, rr = i % kRows;
            const uint32_t off = (uint32_t)((c * kRows + rr) * 4);
            if (!TQ2_IN(off + 4u <= (uint32_t)(BN * kRows * 4) && part_s + off + 4u <= win.hi, st_w)) continue;
            float v = 0.0f;
            for (int q2 = 0; q2 < S; ++q2) {
                uint32_t ra;
                float t;
                asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(part_s + off), "r"(q2));
                asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(t) : "r"(ra) : "memory");
                v += t;
            }
            const int m = m0 + c;
            const int64_t nn = n0 + rr;
            if (*abort_flag == 0 && m < M && nn < N) store_y(m, nn, v);
        }
    }
    named_barrier(3, kUnpackWarps * 32);  // this CTA has read every peer's partial
    if (uw == 0 && lane < S && lane != rank) {  // tell every peer: done reading yours
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(pdone), "r"(lane));
        asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
    }
    // keep this CTA's shared memory alive until every peer has read it
    if (!__all_sync(0xffffffffu, mbar_wait_cluster(pdone, 0u)) && lane == 0) report_timeout(p, abort_flag);
}

// ------------------------------------------------------------------ host side
int align_up(int v, int a) { return (v + a - 1) / a * a; }

// CTAs of a tile width that may share an SM (their tensor memory: Tmem<BN>).
int ctas_per_sm(int BN) { return BN <= 64 ? 2 : 1; }

// The least dynamic shared memory with which no more than ctas_per_sm(BN)
// CTAs fit on an SM (static shared memory and the per-CTA reservation only
// add to it).
int min_dyn_smem(int BN, int device)
{
    static std::atomic<int> smem_per_sm[64];
    int v = (device >= 0 && device < 64) ? smem_per_sm[device].load() : 0;
    if (v <= 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device) != cudaSuccess ||
            v <= 0) {
            cudaGetLastError();
            v = 233472;  // sm_100 / sm_103: 228 KB
        }
        if (device >= 0 && device < 64) smem_per_sm[device].store(v);
    }
    return v / (ctas_per_sm(BN) + 1) + 1;
}

bool make_plan(int BN, int S, int64_t M, int64_t N, int64_t K, int max_dyn, int min_dyn, GemmParams &p)
{
    if (M < 1 || N < 1 || K < 256 || K % 256 != 0 || M > (int64_t)1 << 30) return false;
    if (K > (int64_t)1 << 24) return false;  // d slice and k-step counts stay small
    p.B = (int)(K / 256);
    if (S < 1 || S > 8 || S > p.B || BN % S != 0) return false;
    p.S = S;
    p.n_tiles = (int)((N + kRows - 1) / kRows);
    const int64_t tiles = (int64_t)p.n_tiles * ((M + BN - 1) / BN);
    if (tiles * S > 0x7FFFFFFF) return false;
    const int bstage = 2 * BN * 128;
    int off = 0;
    p.off_bar = off;
    off += 8 * (2 * kMaxStages + 4 * kASlots + 3);  // code ring 2 x sw, stage ring 4 x sb, dfull, pready, pdone
    off = align_up(off, 128);
    p.off_dsm = off;
    off += p.B * kRows * 2;
    // both rings at multiples of 1024 from the base: the runtime rounding of
    // the base then shifts them alike, and one 1024-byte slack covers it
    off = align_up(off, 1024);
    p.off_b = off;
    int sb = (max_dyn - off - 1024 - 2 * kWStageBytes) / bstage;
    const int slots = tmem_slots(BN);
    if (sb > slots) sb = slots;  // one TMEM A slot per stage
    if (sb < 2) return false;
    p.sb = sb;
    off += sb * bstage;
    p.off_w = off;
    int sw = (max_dyn - off - 1024) / kWStageBytes;
    if (sw > 4) sw = 4;
    if (sw < 2) return false;
    p.sw = sw;
    p.smem_total = off + sw * kWStageBytes + 1024;
    if (p.smem_total < min_dyn) p.smem_total = min_dyn;  // at most ctas_per_sm(BN) CTAs per SM
    return p.smem_total <= max_dyn;
}

std::atomic<int> g_gemm_dyn[5][64];

constexpr int bn_index(int BN) { return BN == 16 ? 0 : BN == 32 ? 1 : BN == 64 ? 2 : BN == 128 ? 3 : 4; }

template <int BN>
int gemm_max_dyn(int device)
{
    if (device < 0 || device >= 64) return 0;
    const int bi = bn_index(BN);
    int v = g_gemm_dyn[bi][device].load();
    if (v > 0) return v;
    int optin = 0;
    cudaFuncAttributes fa;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess ||
        cudaFuncGetAttributes(&fa, gemm_tc05_kernel<BN>) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    v = optin - (int)fa.sharedSizeBytes;
    if (cudaFuncSetAttribute(gemm_tc05_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, v) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    g_gemm_dyn[bi][device].store(v);
    return v;
}

// Up to 64 activation rows: the narrowest tile that holds them (an MMA with
// N <= 64 costs about the same as one with N = 16).  Beyond: BN = 256 (full
// tensor-core rate) when that still gives every SM a tile, else 128.
int pick_bn(int64_t M, int64_t N, int device)
{
    if (M <= 16) return 16;
    if (M <= 32) return 32;
    if (M <= 64) return 64;
    const int64_t nt = (N + kRows - 1) / kRows;
    return (nt * ((M + 255) / 256) >= (int64_t)sm_count(device)) ? 256 : 128;
}

// Split of K (cluster size): the largest power of two up to 8 with which the
// tiles still fit on the SMs at once, one CTA each (a second CTA on an SM
// shares its tensor cores: splitting further measured slower), and at least
// one 256-block per CTA.
int pick_split(int BN, int64_t M, int64_t N, int64_t K, int device)
{
    (void)BN;
    const int64_t tiles = ((N + kRows - 1) / kRows) * ((M + BN - 1) / BN);
    const int64_t slots = sm_count(device);
    int S = 1;
    while (S < 8 && tiles * (2 * S) <= slots && 2 * S <= K / 256) S *= 2;
    return S;
}

template <int BN>
cudaError_t launch_gemm(const MatvecArgs &a, int device)
{
    GemmParams p{};
    p.a = a;
    const int S = pick_split(BN, a.M, a.N, a.K, device);
    if (!make_plan(BN, S, a.M, a.N, a.K, gemm_max_dyn<BN>(device), min_dyn_smem(BN, device), p))
        return cudaErrorInvalidConfiguration;
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)(a.K / 32), (cuuint64_t)a.N};
        const cuuint64_t strides[1] = {(cuuint64_t)(a.K / 4)};
        const cuuint32_t box[2] = {8, (cuuint32_t)kRows};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&p.wmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<uint8_t *>(a.qs), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
        const cuuint64_t strides[1] = {(cuuint64_t)(a.K * 2)};
        const cuuint32_t box[2] = {64, (cuuint32_t)BN};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&p.xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t *>(a.x), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const int64_t G = (int64_t)p.n_tiles * ((a.M + BN - 1) / BN) * S;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(Tmem<BN>::threads);
    cfg.dynamicSmemBytes = (size_t)p.smem_total;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)S;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (S > 1) ? 2 : 1;  // a cluster launch only when K is split
    return cudaLaunchKernelEx(&cfg, gemm_tc05_kernel<BN>, p);
}

}  // namespace

bool gemm_tc05_supported(int64_t M, int64_t N, int64_t K, int device)
{
    GemmParams p{};
    const int bn = pick_bn(M, N, device);
    const int dyn = bn == 16 ? gemm_max_dyn<16>(device) : bn == 32 ? gemm_max_dyn<32>(device)
                  : bn == 64 ? gemm_max_dyn<64>(device) : bn == 128 ? gemm_max_dyn<128>(device)
                  : gemm_max_dyn<256>(device);
    return dyn > 0 && make_plan(bn, pick_split(bn, M, N, K, device), M, N, K, dyn, min_dyn_smem(bn, device), p);
}

cudaError_t launch_gemm_tc05(const MatvecArgs &a, int device)
{
    switch (pick_bn(a.M, a.N, device)) {
    case 16: return launch_gemm<16>(a, device);
    case 32: return launch_gemm<32>(a, device);
    case 64: return launch_gemm<64>(a, device);
    case 128: return launch_gemm<128>(a, device);
    default: return launch_gemm<256>(a, device);
    }
}

}  // namespace tq2
