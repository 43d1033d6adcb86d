// tq2_matvec_simt.cu -- CUDA-core ternary matvec (fp32 FMA per code).
//
// The plain SIMT form of the BitCPM ternary page's sign-add matvec (linear
// factoring paragraph): each lane sums x_k * (q_k - 1) over 64 codes of one
// 256-block, multiplies the partial by that block's d, and the warp reduces.
// One warp per output row, all M activation rows at once.  It serves every
// M in 1..16 and is the CUDA-core variant the tensor-core kernel is measured
// against.
#include <cuda_fp16.h>

#include "tq2_device.cuh"
#include "tq2_internal.cuh"

namespace tq2 {
namespace {

constexpr int kSimtThreads = 256;

using dev::fq_code;  // rint(x * (1/s)) in fp32, clamped (gemma4 wNa8o8 page)

template <int kM>
__global__ void __launch_bounds__(kSimtThreads)
matvec_simt_kernel(MatvecArgs a)
{
    const int lane = threadIdx.x & 31;
    const int warps = kSimtThreads / 32;
    const int64_t KB = a.K / 4;       // bytes per packed row
    const int64_t B = a.K / 256;      // blocks per row
    const int64_t nchunks = a.K / 64; // 16-byte chunks (64 codes) per row
    const bool prologue = a.act_scale != 0.0f;
    const bool convert = prologue && !a.x_codes;  // x holds fp16 values, not yet codes
    for (int64_t n = (int64_t)blockIdx.x * warps + (threadIdx.x >> 5); n < a.N;
         n += (int64_t)gridDim.x * warps) {
        float acc[kM];
#pragma unroll
        for (int m = 0; m < kM; ++m) acc[m] = 0.0f;
        for (int64_t c = lane; c < nchunks; c += 32) {
            if (!TQ2_IN(n * KB + c * 16 + 16 <= a.N * KB && n * B + c / 4 < a.N * B, a.status)) continue;
            const uint4 v = *reinterpret_cast<const uint4 *>(a.qs + n * KB + c * 16);
            const float dv = __half2float(__ushort_as_half(a.d[n * B + c / 4]));
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int m = 0; m < kM; ++m) {
                const uint16_t *xr = a.x + (int64_t)m * a.K + c * 64;
                if (!TQ2_IN((int64_t)m * a.K + c * 64 + 64 <= (int64_t)a.M * a.K, a.status)) continue;
                float part = 0.0f;
#pragma unroll 1
                for (int wi = 0; wi < 4; ++wi) {
                    const uint4 xv0 = *reinterpret_cast<const uint4 *>(xr + 16 * wi);
                    const uint4 xv1 = *reinterpret_cast<const uint4 *>(xr + 16 * wi + 8);
                    const uint32_t xw[8] = {xv0.x, xv0.y, xv0.z, xv0.w, xv1.x, xv1.y, xv1.z, xv1.w};
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const uint16_t hb = (uint16_t)(xw[j >> 1] >> (16 * (j & 1)));
                        float xf = __half2float(__ushort_as_half(hb));
                        if (convert) xf = fq_code(xf, a.inv_scale);
                        const float wv = (float)((int)((w4[wi] >> (2 * j)) & 3u) - 1);
                        part = fmaf(xf, wv, part);
                    }
                }
                acc[m] = fmaf(dv, part, acc[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < kM; ++m) {
            float s = acc[m];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
            if (prologue) s *= a.act_scale;
            s = dev::requant_out(s, a.out_scale, a.inv_out);
            if (lane == 0 && TQ2_IN((int64_t)m * a.N + n < (int64_t)a.M * a.N, a.status)) {
                if (a.y_f16)
                    reinterpret_cast<__half *>(a.y)[(int64_t)m * a.N + n] = __float2half_rn(s);
                else
                    reinterpret_cast<float *>(a.y)[(int64_t)m * a.N + n] = s;
            }
        }
    }
}

template <int kM>
cudaError_t launch_m(const MatvecArgs &a, int device)
{
    const int warps = kSimtThreads / 32;
    int64_t grid = (a.N + warps - 1) / warps;
    const int64_t cap = (int64_t)sm_count(device) * 8;
    if (grid > cap) grid = cap;
    matvec_simt_kernel<kM><<<(unsigned)grid, kSimtThreads, 0, a.stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_matvec_simt(const MatvecArgs &a, int device)
{
    switch (a.M) {
    case 1: return launch_m<1>(a, device);
    case 2: return launch_m<2>(a, device);
    case 3: return launch_m<3>(a, device);
    case 4: return launch_m<4>(a, device);
    case 5: return launch_m<5>(a, device);
    case 6: return launch_m<6>(a, device);
    case 7: return launch_m<7>(a, device);
    case 8: return launch_m<8>(a, device);
    case 9: return launch_m<9>(a, device);
    case 10: return launch_m<10>(a, device);
    case 11: return launch_m<11>(a, device);
    case 12: return launch_m<12>(a, device);
    case 13: return launch_m<13>(a, device);
    case 14: return launch_m<14>(a, device);
    case 15: return launch_m<15>(a, device);
    case 16: return launch_m<16>(a, device);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace tq2
