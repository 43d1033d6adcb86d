// tq2_matvec_smalln.cu -- ternary matvec for a handful of output rows per
// CTA (k/v-sized N), M <= 2, sm_103a.
//
// What it computes (BitCPM ternary page, linear-factoring paragraph):
//   y[m][n] = sum_b d[n][b] * sum_{k in b} x'[m][k] * (q[n][k] - 1)
// with x' = x, or its static int8 fake-quant code (gemma4 wNa8o8 page; the
// sum is then multiplied by act_scale once), and the optional int8
// requantisation of y at store.
//
// Why a separate kernel: with N of a few hundred rows, each of the SMs' CTAs
// owns one to four rows, and a call is all latency -- the wait for the
// previous kernel, one read of x, a short sum, one reduction.  The tensor-core
// kernels spend that time staging all of x into MMA-fragment order behind a
// CTA barrier and computing 16-row MMAs for 1-2 valid rows.  Here:
//   * the CTA's codes (one 32-bit word of 16 codes per thread and row, K up
//     to 16384 in four words) and their scales go to registers before the
//     PDL wait -- weights never depend on the previous kernel;
//   * after the wait each thread reads only the 16 x values of its words,
//     all loads in flight together;
//   * per word: sum_j x_j q_j (q_j as an exact float) minus sum_j x_j, times
//     d_b; per row a warp shuffle tree and a fixed-order sum over the warps.
// Residency: in a chain of programmatic dependent launches every call here
// must occupy the SMs the way the tensor-core kernels do -- one CTA per SM
// (min(N, SMs) CTAs) and room for only two CTAs per SM -- or the next calls'
// CTAs pile up unevenly (measured on a 224-call chain: 1.37 ms per step with
// this kernel unconstrained, or reserving 72 KB of shared memory, against
// 0.988 ms reserving 100 KB).  So it reserves half an SM's shared memory
// less 14 KB (dynamic, unused) besides its 0.25 KB of partial sums.
#include <cuda_fp16.h>

#include <atomic>

#include "tq2_device.cuh"
#include "tq2_internal.cuh"

namespace tq2 {
namespace {

using namespace dev;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxRows = 4;   // output rows per CTA
constexpr int kMaxWords = 4;  // 16-code words per thread and row: K <= 16384

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }

template <int kM, int kW>
__global__ void __launch_bounds__(kThreads, 2) matvec_smalln_kernel(const MatvecArgs a, int G)
{
    __shared__ float red[kMaxRows][kM][kWarps];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t N = a.N, K = a.K;
    const int64_t r0 = (int64_t)blockIdx.x * N / G;
    const int nrows = (int)((int64_t)(blockIdx.x + 1) * N / G - r0);  // 1 .. kMaxRows (host-checked)
    const int nw = (int)(K / 16);   // 16-code words per row
    const int B = (int)(K / 256);
    const bool prologue = a.act_scale != 0.0f;
    const bool convert = prologue && !a.x_codes;  // x holds fp16 values, not yet codes

    asm volatile("griddepcontrol.launch_dependents;");

    // this thread's words of the CTA's rows and their block scales; a word
    // past the row (or a row past the CTA's) reads as codes 1 (value 0)
    uint32_t cw[kMaxRows][kW];
    float dv[kMaxRows][kW];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r)
#pragma unroll
        for (int i = 0; i < kW; ++i) {
            const int w = tid + i * kThreads;
            const bool v = r < nrows && w < nw && TQ2_IN(r0 + r < N, a.status);
            cw[r][i] = v ? __ldg(reinterpret_cast<const uint32_t *>(a.qs + (r0 + r) * (K / 4)) + w) : 0x55555555u;
            dv[r][i] = v ? h2f(__ldg(a.d + (r0 + r) * B + (w >> 4))) : 0.0f;
        }

    // x depends on the previous kernel in the stream.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    uint4 xv[kM][kW][2];
#pragma unroll
    for (int m = 0; m < kM; ++m)
#pragma unroll
        for (int i = 0; i < kW; ++i) {
            const int w = tid + i * kThreads;
            if (w < nw && TQ2_IN((int64_t)m * K + (int64_t)w * 16 + 16 <= (int64_t)kM * K, a.status)) {
                const uint4 *src = reinterpret_cast<const uint4 *>(a.x + (int64_t)m * K + (int64_t)w * 16);
                xv[m][i][0] = src[0];
                xv[m][i][1] = src[1];
            } else {
                xv[m][i][0] = xv[m][i][1] = make_uint4(0, 0, 0, 0);
            }
        }

    float part[kMaxRows][kM];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r)
#pragma unroll
        for (int m = 0; m < kM; ++m) part[r][m] = 0.0f;

#pragma unroll
    for (int i = 0; i < kW; ++i) {
#pragma unroll
        for (int m = 0; m < kM; ++m) {
            const uint32_t hw[8] = {xv[m][i][0].x, xv[m][i][0].y, xv[m][i][0].z, xv[m][i][0].w,
                                    xv[m][i][1].x, xv[m][i][1].y, xv[m][i][1].z, xv[m][i][1].w};
            float xf[16];
            float sx = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float lo = h2f((uint16_t)(hw[j] & 0xffffu)), hi = h2f((uint16_t)(hw[j] >> 16));
                if (convert) {
                    lo = fq_code(lo, a.inv_scale);
                    hi = fq_code(hi, a.inv_scale);
                }
                xf[2 * j] = lo;
                xf[2 * j + 1] = hi;
                sx += lo + hi;
            }
#pragma unroll
            for (int r = 0; r < kMaxRows; ++r) {
                if (r >= nrows) break;
                const uint32_t c = cw[r][i];
                float sq = 0.0f;  // sum_j x_j q_j, q_j = bits 2j..2j+1 of the word, exact as a float
#pragma unroll
                for (int j = 0; j < 16; ++j) sq = fmaf(xf[j], (float)((c >> (2 * j)) & 3u), sq);
                part[r][m] = fmaf(dv[r][i], sq - sx, part[r][m]);
            }
        }
    }

    // per row: warp shuffle tree, then the warps in a fixed order
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
        if (r >= nrows) break;
#pragma unroll
        for (int m = 0; m < kM; ++m) {
            float v = part[r][m];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            if (lane == 0) red[r][m][warp] = v;
        }
    }
    __syncthreads();
    if (tid < nrows * kM) {
        const int r = tid / kM, m = tid - (tid / kM) * kM;
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += red[r][m][w];
        if (prologue) s *= a.act_scale;
        s = requant_out(s, a.out_scale, a.inv_out);
        const int64_t o = (int64_t)m * N + r0 + r;
        if (!TQ2_IN(o < (int64_t)kM * N, a.status)) return;
        if (a.y_f16)
            reinterpret_cast<__half *>(a.y)[o] = __float2half_rn(s);
        else
            reinterpret_cast<float *>(a.y)[o] = s;
    }
}

template <int kM>
void *kernel_for_words(int words)
{
    switch (words) {
    case 1: return reinterpret_cast<void *>(matvec_smalln_kernel<kM, 1>);
    case 2: return reinterpret_cast<void *>(matvec_smalln_kernel<kM, 2>);
    case 3: return reinterpret_cast<void *>(matvec_smalln_kernel<kM, 3>);
    case 4: return reinterpret_cast<void *>(matvec_smalln_kernel<kM, 4>);
    default: return nullptr;
    }
}

}  // namespace

bool smalln_matvec_supported(int M, int64_t N, int64_t K, int device)
{
    if (M < 1 || M > 2 || N < 1 || K < 256 || K % 256 != 0 || K > 256 * 16 * kMaxWords) return false;
    const int64_t nsm = sm_count(device);
    if (nsm <= 0) return false;
    const int64_t G = N < nsm ? N : nsm;
    return (N + G - 1) / G <= kMaxRows;
}

// Where it beats the tensor-core kernel (measured per call on GB300, M = 1
// and 2): while a thread's rows x words stay <= 8 -- k/v (256 rows) at
// K = 4096 (1.54 against 2.27 us) and K = 16384 (2.89 against 5.09 us), up to
// ~600 rows at K = 4096 -- but not 512 rows at K = 16384 (16: 5.60 against
// 5.09 us).
bool smalln_matvec_preferred(int M, int64_t N, int64_t K, int device)
{
    if (!smalln_matvec_supported(M, N, K, device)) return false;
    const int64_t nsm = sm_count(device);
    const int64_t G = N < nsm ? N : nsm;
    const int64_t rows = (N + G - 1) / G, words = (K / 16 + kThreads - 1) / kThreads;
    return rows * words <= 8;
}

// Dynamic shared memory that leaves room for two CTAs per SM, never three:
// half the SM's capacity less 14 KB (100 KB on a 228 KB SM).  Raised on the
// instantiation once per device; 0 on failure.
std::atomic<int> g_reserve[2][kMaxWords + 1][64];

int reserve_bytes(void *k, int kM, int words, int device)
{
    if (device < 0 || device >= 64) return 0;
    int v = g_reserve[kM - 1][words][device].load();
    if (v > 0) return v;
    int per_sm = 0, optin = 0;
    if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    v = per_sm / 2 - 14 * 1024;
    if (v > optin - 1024) v = optin - 1024;
    if (v <= 0 || cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, v) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    g_reserve[kM - 1][words][device].store(v);
    return v;
}

cudaError_t launch_matvec_smalln(const MatvecArgs &a, int device)
{
    if (!smalln_matvec_supported(a.M, a.N, a.K, device)) return cudaErrorInvalidValue;
    const int nsm = sm_count(device);
    int G = (int)(a.N < nsm ? a.N : nsm);
    const int words = (int)((a.K / 16 + kThreads - 1) / kThreads);
    void *k = (a.M == 1) ? kernel_for_words<1>(words) : kernel_for_words<2>(words);
    if (!k) return cudaErrorInvalidValue;
    const int reserve = reserve_bytes(k, a.M, words, device);
    if (reserve <= 0) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = (size_t)reserve;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<MatvecArgs *>(&a), &G};
    return cudaLaunchKernelExC(&cfg, k, args);
}

}  // namespace tq2
