// tq2_layout.cu -- pack / unpack / from_dense kernels for the TQ2_0-style
// packed ternary layout.
//
// Format (BitCPM ternary page, "TQ2_0 (llama.cpp)" paragraph): a 2-bit code
// q in {0,1,2} stands for q-1; one fp16 scale per 256-element block along K.
// Layout: code k of a row sits at bits 2*(k%4) of byte k/4.
// Recovery (same page, recovery paragraph): d = max|W| over the block,
// code = round(W/d) + 1.
//
// These run once per weight tensor (model load), not per token; they are
// plain memory-bound element-wise kernels.
#include <cuda_fp16.h>

#include "tq2_internal.cuh"

namespace tq2 {
namespace {

constexpr int kLayoutThreads = 256;

__device__ __forceinline__ void or_flags(uint32_t *status, uint32_t bits, bool mine)
{
    // one atomic per warp that saw the condition
    unsigned any = __ballot_sync(0xffffffffu, mine);
    if (status && any && (threadIdx.x & 31) == (__ffs(any) - 1))
        atomicOr(status, bits);
}

// One thread per 16 codes (4 packed bytes).  `vec` selects 16-byte code loads
// and 4-byte stores when both pointers allow them.
template <bool kVec>
__global__ void __launch_bounds__(kLayoutThreads)
pack_kernel(const int8_t *__restrict__ codes, int64_t nwords, uint8_t *__restrict__ qs,
            uint32_t *status)
{
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    bool bad = false;
    if (i < nwords) {
        int8_t c[16];
        if (kVec) {
            int4 v = reinterpret_cast<const int4 *>(codes)[i];
            *reinterpret_cast<int4 *>(c) = v;
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) c[j] = codes[16 * i + j];
        }
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            bad |= (c[j] < 0) | (c[j] > 2);
            word |= ((uint32_t)(uint8_t)c[j] & 3u) << (2 * j);
        }
        if (kVec) {
            reinterpret_cast<uint32_t *>(qs)[i] = word;
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) qs[4 * i + j] = (uint8_t)(word >> (8 * j));
        }
    }
    or_flags(status, TQ2_FLAG_BAD_CODE, bad);
}

template <bool kVec>
__global__ void __launch_bounds__(kLayoutThreads)
unpack_kernel(const uint8_t *__restrict__ qs, int64_t nwords, int8_t *__restrict__ codes)
{
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= nwords) return;
    uint32_t word;
    if (kVec) {
        word = reinterpret_cast<const uint32_t *>(qs)[i];
    } else {
        word = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) word |= (uint32_t)qs[4 * i + j] << (8 * j);
    }
    int8_t c[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) c[j] = (int8_t)((word >> (2 * j)) & 3u);
    if (kVec) {
        reinterpret_cast<int4 *>(codes)[i] = *reinterpret_cast<int4 *>(c);
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) codes[16 * i + j] = c[j];
    }
}

__device__ __forceinline__ float load_w(const void *W, int w_f16, int64_t idx)
{
    if (w_f16) {
        unsigned short h = reinterpret_cast<const unsigned short *>(W)[idx];
        return __half2float(__ushort_as_half(h));
    }
    return reinterpret_cast<const float *>(W)[idx];
}

// One warp per (row, 256-block); lane l owns elements 8l .. 8l+7.
__global__ void __launch_bounds__(kLayoutThreads)
from_dense_kernel(const void *__restrict__ W, int w_f16, int64_t N, int64_t K,
                  uint8_t *__restrict__ qs, uint16_t *__restrict__ d, uint32_t *status)
{
    const int lane = threadIdx.x & 31;
    const int64_t B = K / 256;
    const int64_t unit = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const bool active = unit < N * B;  // warp-uniform
    bool nonfinite = false, inexact = false;
    if (active) {
        const int64_t n = unit / B, b = unit % B;
        const int64_t base = n * K + b * 256 + 8 * lane;
        float v[8];
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            v[j] = load_w(W, w_f16, base + j);
            nonfinite |= !isfinite(v[j]);
            float a = fabsf(v[j]);
            amax = (a > amax) ? a : amax;  // NaN is skipped
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        const __half dh = __float2half_rn(amax);
        const float dv = __half2float(dh);
        nonfinite |= !isfinite(dv);
        uint32_t packed = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            int code;
            if (dv == 0.0f) {
                code = 1;
            } else {
                float r = __fdiv_rn(v[j], dv);
                if (isnan(r)) {
                    code = 1;
                } else {
                    float rr = rintf(r);
                    rr = fminf(fmaxf(rr, -1.0f), 1.0f);
                    code = (int)rr + 1;
                }
            }
            inexact |= !(__fmul_rn(dv, (float)(code - 1)) == v[j]);
            packed |= (uint32_t)code << (2 * j);
        }
        uint8_t *row = qs + n * (K / 4) + b * 64 + 2 * lane;
        row[0] = (uint8_t)(packed & 0xffu);
        row[1] = (uint8_t)(packed >> 8);
        if (lane == 0) d[n * B + b] = __half_as_ushort(dh);
    }
    or_flags(status, TQ2_FLAG_NONFINITE, nonfinite);
    or_flags(status, TQ2_FLAG_INEXACT, inexact);
}

}  // namespace

cudaError_t launch_pack(const int8_t *codes, int64_t N, int64_t K, uint8_t *qs,
                        uint32_t *status, cudaStream_t s)
{
    const int64_t nwords = N * K / 16;
    if (nwords == 0) return cudaSuccess;
    const int64_t grid = (nwords + kLayoutThreads - 1) / kLayoutThreads;
    const bool vec = ((uintptr_t)codes % 16 == 0) && ((uintptr_t)qs % 4 == 0);
    if (vec)
        pack_kernel<true><<<(unsigned)grid, kLayoutThreads, 0, s>>>(codes, nwords, qs, status);
    else
        pack_kernel<false><<<(unsigned)grid, kLayoutThreads, 0, s>>>(codes, nwords, qs, status);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t *qs, int64_t N, int64_t K, int8_t *codes,
                          cudaStream_t s)
{
    const int64_t nwords = N * K / 16;
    if (nwords == 0) return cudaSuccess;
    const int64_t grid = (nwords + kLayoutThreads - 1) / kLayoutThreads;
    const bool vec = ((uintptr_t)codes % 16 == 0) && ((uintptr_t)qs % 4 == 0);
    if (vec)
        unpack_kernel<true><<<(unsigned)grid, kLayoutThreads, 0, s>>>(qs, nwords, codes);
    else
        unpack_kernel<false><<<(unsigned)grid, kLayoutThreads, 0, s>>>(qs, nwords, codes);
    return cudaGetLastError();
}

cudaError_t launch_from_dense(const void *W, int w_f16, int64_t N, int64_t K, uint8_t *qs,
                              uint16_t *d, uint32_t *status, cudaStream_t s)
{
    const int64_t units = N * (K / 256);
    if (units == 0) return cudaSuccess;
    const int64_t warps_per_block = kLayoutThreads / 32;
    const int64_t grid = (units + warps_per_block - 1) / warps_per_block;
    from_dense_kernel<<<(unsigned)grid, kLayoutThreads, 0, s>>>(W, w_f16, N, K, qs, d, status);
    return cudaGetLastError();
}

}  // namespace tq2
