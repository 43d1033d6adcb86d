// tq2_prologue.cu -- the static int8 fake-quant of x as a pass of its own.
//
// gemma4 wNa8o8 page, "Implemented": at a linear's input x is replaced by
// s * clamp(rint(x / s), -128, 127).  Every kernel of this library can do
// that itself while it stages x, but then each CTA converts the x it reads:
// the GEMM converts the whole of x once per 128-row weight tile, the matvec
// kernels once per CTA.  Given scratch for it, a call converts x once here,
// writes the codes as fp16 integers in [-128, 127] (exact), and the kernel
// reads them like x and multiplies its fp32 sums by s at the store, as it
// does after converting x itself.  The decision rint(fp32(x) * fp32(1/s)) is
// the one every kernel takes (dev::fq_code), so the two plans give the same
// bits.
#include <cuda_fp16.h>

#include <atomic>

#include "tq2_device.cuh"
#include "tq2_internal.cuh"

namespace tq2 {
namespace {

constexpr int kFqThreads = 256;
constexpr int kFqUnroll = 4;  // independent 16-byte loads in flight per thread

__device__ __forceinline__ uint32_t fq_pair(uint32_t w, float inv_s)
{
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w));
    const __half2 h = __floats2half2_rn(dev::fq_code(f.x, inv_s), dev::fq_code(f.y, inv_s));  // exact
    return *reinterpret_cast<const uint32_t *>(&h);
}

__global__ void __launch_bounds__(kFqThreads) fq_codes_kernel(const uint4 *__restrict__ x, uint4 *__restrict__ c,
                                                             int64_t n16, float inv_s)
{
    // The next kernel may launch at once, as it would right behind the
    // previous kernel without this pass: it fetches its weights (which
    // nothing here writes) early and reads the codes only after its own
    // wait, which returns once this grid has completed.  x may come from the
    // previous kernel: read it only after the wait for that one.
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t stride = (int64_t)gridDim.x * kFqThreads;
    for (int64_t i0 = (int64_t)blockIdx.x * kFqThreads + threadIdx.x; i0 < n16; i0 += kFqUnroll * stride) {
        uint4 v[kFqUnroll];
#pragma unroll
        for (int u = 0; u < kFqUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < n16) v[u] = x[i];
        }
#pragma unroll
        for (int u = 0; u < kFqUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            if (i < n16)
                c[i] = make_uint4(fq_pair(v[u].x, inv_s), fq_pair(v[u].y, inv_s), fq_pair(v[u].z, inv_s),
                                  fq_pair(v[u].w, inv_s));
        }
    }
}

// Scratch of the entry point that allocates nothing (tq2_gemm_static_ws):
// one array per device, in the library's own module, for the codes of at
// most kStaticScratchBytes / 2 activations.
static __device__ __align__(256) uint16_t g_static_codes[kStaticScratchBytes / 2];

std::atomic<uintptr_t> g_static_codes_addr[64];

}  // namespace

cudaError_t static_codes_scratch(int device, void **ptr)
{
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    uintptr_t v = g_static_codes_addr[device].load(std::memory_order_acquire);
    if (v == 0) {  // once per device: the array's address in this device's context
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_codes);
        if (e != cudaSuccess) return e;
        v = reinterpret_cast<uintptr_t>(p);
        g_static_codes_addr[device].store(v, std::memory_order_release);
    }
    *ptr = reinterpret_cast<void *>(v);
    return cudaSuccess;
}

cudaError_t launch_fq_codes(const uint16_t *x, int64_t n, float inv_scale, uint16_t *codes, cudaStream_t stream,
                            int device)
{
    const int64_t n16 = n / 8;
    if (n16 <= 0) return cudaSuccess;
    // kFqUnroll 16-byte loads per thread, at most 4 CTAs per SM (each thread
    // loops beyond): small enough that the next kernel's CTAs find room
    // beside the ones still waiting for the previous kernel
    int64_t blocks = (n16 + kFqThreads * kFqUnroll - 1) / (kFqThreads * kFqUnroll);
    const int64_t cap = 4 * (int64_t)sm_count(device);
    if (blocks > cap) blocks = cap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kFqThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fq_codes_kernel, reinterpret_cast<const uint4 *>(x),
                              reinterpret_cast<uint4 *>(codes), n16, inv_scale);
}

}  // namespace tq2
