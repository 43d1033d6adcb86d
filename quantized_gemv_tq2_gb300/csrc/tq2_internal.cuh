// tq2_internal.cuh -- declarations shared by the library's own translation
// units (layout kernels, the two matvec kernels, the C-ABI shim).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "../../include/tq2.h"

namespace tq2 {

// Everything a matvec launcher needs, already validated by the ABI shim.
struct MatvecArgs {
    const uint16_t *x;   // [M, K] fp16 bits
    const uint8_t *qs;   // [N, K/4]
    const uint16_t *d;   // [N, K/256] fp16 bits
    void *y;             // [M, N] fp32 or fp16
    uint32_t *status;    // optional device flag word
    int64_t N, K;
    int M;
    int y_f16;           // 0: fp32 y, 1: fp16 y
    float act_scale;     // 0: no prologue
    float inv_scale;     // fp32(1/act_scale), correctly rounded on the host
    float out_scale;     // 0: y stored as computed; else requantised to int8 at store
    float inv_out;       // fp32(1/out_scale), correctly rounded on the host
    cudaStream_t stream;
    // Limit of every bounded device wait of the class-column kernel (0: the
    // default, 200 ms), and a test hook of that kernel: the weight producer
    // skips the copy of this stage (-1: none), so that the consumers' wait
    // for it runs out and the timeout path runs.
    unsigned long long wait_limit_ns = 0;
    int stall_stage = -1;
    // 1: x already holds the prologue's codes (fp16 integers in [-128, 127],
    // written by launch_fq_codes), so the kernel does not convert it again;
    // it still multiplies its sums by act_scale at the store.
    int x_codes = 0;
};

// The prologue as a pass of its own: codes[i] = fp16(clamp(rint(x[i] *
// inv_scale), -128, 127)) for i < n (n a multiple of 8; x and codes 16-byte
// aligned), the same fp32 decision every kernel takes when it converts x
// itself.  Waits for the previous kernel on the stream before reading x and
// lets the next kernel launch (and fetch its weights) as soon as it runs.
cudaError_t launch_fq_codes(const uint16_t *x, int64_t n, float inv_scale, uint16_t *codes, cudaStream_t stream,
                            int device);

// The static scratch of tq2_gemm_static_ws: 16 MiB (the codes of 2^23
// activations), its address taken once per device (cudaGetSymbolAddress).
constexpr size_t kStaticScratchBytes = (size_t)16 << 20;
cudaError_t static_codes_scratch(int device, void **ptr);

// Tensor-core path (mma.sync on masked code words, TMA bulk staging).
// Returns false when the shape is outside what the kernel supports
// (M > 2 or shared memory would not fit); nothing is launched then.
bool mma_matvec_supported(int M, int64_t N, int64_t K, int device);
cudaError_t launch_matvec_mma(const MatvecArgs &a, int device);

// The same kernel over a group of up to 4 weight matrices that share x: one
// launch, CTAs split in proportion to the rows.  qs/d/y/N are host arrays of
// n device pointers / row counts; out_scale/inv_out host arrays of n output
// scales and their fp32 reciprocals (nullptr: none).
bool mma_group_supported(int M, int n, const int64_t *N, int64_t K, int device);
cudaError_t launch_matvec_mma_group(const MatvecArgs &a, int n, const uint8_t *const *qs, const uint16_t *const *d,
                                    void *const *y, const int64_t *N, const float *out_scale,
                                    const float *inv_out, int device);

// The pre-scaled kernel over such a group (M in 1..16).
bool ps_group_supported(int M, int n, const int64_t *N, int64_t K, int device);
cudaError_t launch_matvec_ps_group(const MatvecArgs &a, int n, const uint8_t *const *qs, const uint16_t *const *d,
                                   void *const *y, const int64_t *N, const float *out_scale,
                                   const float *inv_out, int device);

// Ternary GEMM for many activation rows (any M): tcgen05 MMAs over weights
// expanded to (q - 1) * d in tensor memory, x tiles by TMA (fake-quantised in
// shared memory when act_scale != 0).
bool gemm_tc05_supported(int64_t M, int64_t N, int64_t K, int device);
cudaError_t launch_gemm_tc05(const MatvecArgs &a, int device);

// Tensor-core path with pre-scaled x (all four code classes in one
// accumulator, 8 activation rows per n-tile), M in 1..16.  Returns false
// when the shape does not fit.
bool ps_matvec_supported(int M, int64_t N, int64_t K, int device);
cudaError_t launch_matvec_ps(const MatvecArgs &a, int device);

// Affine-int4 matvec (zero point factored out per group of G codes): codes
// [N][K/2] (two per byte, low nibble first), s and z fp16 [N][K/G], G in
// {64, 128, 256}; activation rows two per launch.
struct Affine4Args {
    const uint16_t *x;   // [M, K] fp16 bits
    const uint8_t *qs;   // [N, K/2]
    const uint16_t *s;   // [N, K/G] fp16 bits
    const uint16_t *z;   // [N, K/G] fp16 bits
    void *y;             // [M, N] fp32 or fp16
    uint32_t *status;    // optional device flag word
    int64_t M, N, K, G;
    int y_f16;
    cudaStream_t stream;
};
bool affine4_supported(int64_t M, int64_t N, int64_t K, int64_t G, int device);
cudaError_t launch_affine4(const Affine4Args &a, int device);

// Few-rows-per-CTA path for small N (k/v-sized): M <= 2, K <= 16384, at most
// 4 output rows per CTA with one CTA per SM; codes and scales in registers
// before the PDL wait, CUDA-core sums, one reduction.  Returns false when
// the shape does not fit.
bool smalln_matvec_supported(int M, int64_t N, int64_t K, int device);
bool smalln_matvec_preferred(int M, int64_t N, int64_t K, int device);  // faster than impl 1 here
cudaError_t launch_matvec_smalln(const MatvecArgs &a, int device);

// CUDA-core path (fp32 FMA per code), any M in 1..16.
cudaError_t launch_matvec_simt(const MatvecArgs &a, int device);

// Layout kernels.
cudaError_t launch_pack(const int8_t *codes, int64_t N, int64_t K, uint8_t *qs,
                        uint32_t *status, cudaStream_t s);
cudaError_t launch_unpack(const uint8_t *qs, int64_t N, int64_t K, int8_t *codes,
                          cudaStream_t s);
cudaError_t launch_from_dense(const void *W, int w_f16, int64_t N, int64_t K, uint8_t *qs,
                              uint16_t *d, uint32_t *status, cudaStream_t s);

// The trace build's phase stamps of the class-column kernel (TQ2_TRACE):
// their size in bytes (0 in other builds), and a copy of them to host memory
// (cudaErrorNotSupported in other builds).
size_t trace_bytes();
cudaError_t trace_read(void *dst, size_t bytes);

// Number of SMs of the current device (cached per device).
int sm_count(int device);

// The driver's cuTensorMapEncodeTiled (looked up once), or nullptr.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

}  // namespace tq2
