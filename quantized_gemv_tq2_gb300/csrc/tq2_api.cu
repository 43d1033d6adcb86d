// tq2_api.cu -- the C ABI (include/tq2.h): host-side validation, kernel
// choice and launch on the caller's stream.  Every argument check happens
// before any CUDA call, so invalid arguments return a status without touching
// the device (these checks run even on a machine without a GPU).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdio>

#include "tq2_internal.cuh"

namespace tq2 {

static std::atomic<int> g_sm_count[64];

int sm_count(int device)
{
    if (device < 0 || device >= 64) return 148;
    int v = g_sm_count[device].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || v <= 0)
        v = 148;
    g_sm_count[device].store(v, std::memory_order_relaxed);
    return v;
}

// cuTensorMapEncodeTiled from the driver, looked up once (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static std::atomic<void *> fn{nullptr};
    void *f = fn.load();
    if (f) return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || f == nullptr) {
        cudaGetLastError();
        return nullptr;
    }
    fn.store(f);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

}  // namespace tq2

namespace {

constexpr int64_t kMaxElems = (int64_t)1 << 62;

bool aligned(const void *p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

// N, K >= 0, K % 256 == 0, N*K representable.
tq2_status check_nk(int64_t N, int64_t K)
{
    if (N < 0 || K < 0 || K % 256 != 0) return TQ2_ERR_SHAPE;
    if (K > 0 && N > kMaxElems / K) return TQ2_ERR_SHAPE;
    return TQ2_OK;
}

thread_local cudaError_t t_last_cuda_error = cudaSuccess;

tq2_status from_cuda(cudaError_t e)
{
    if (e == cudaSuccess) return TQ2_OK;
    t_last_cuda_error = e;
    cudaGetLastError();  // the error is returned; do not leave it sticky for the caller
    return TQ2_ERR_CUDA;
}

tq2_status current_device(int *dev)
{
    return from_cuda(cudaGetDevice(dev));
}

// The tcgen05 GEMM beats the pre-scaled kernel (crossovers measured, see
// the dispatch in matvec_common; the same with and without the prologue
// when each kernel converts x itself).  With the prologue run as a pass of
// its own (`pass`: act_scale > 0 and a workspace) the GEMM also wins for
// down-sized K at M = 8: 27.3 against 30.5 us (at M = 6: 27.3 against 24.1).
bool gemm_preferred(int M, int64_t N, int64_t K, bool pass = false)
{
    return (M >= 9 && (K >= 8192 || N <= 512)) || (M >= 12 && N < 8192) || (pass && M >= 8 && K >= 8192 && N > 512);
}

// Scratch for the prologue as a pass of its own (tq2_prologue.cu): the
// M x K codes as fp16.
size_t codes_bytes(int64_t M, int64_t K)
{
    return (M > 0 && K > 0) ? (size_t)(2 * M * K) : 0;
}

// Whether converting x once (a pass of its own) beats each CTA of kernel
// `which` (1, 2, 4, 6 or 7 as in tq2_matvec_impl) converting the x it
// reads.  Measured on GB300, us per call back to back over distinct weights,
// each CTA converting / the pass:
//   GEMM, M = 1..16: gate/up 16384x4096 30.5-30.8 / 24.1-24.7, down
//     4096x16384 33.9-34.0 / 27.1-27.7, q/o 4096x4096 11.3-11.4 /
//     10.6-11.0, k/v 256x4096 7.2-7.3 / 7.6-8.0 (two weight tiles: little
//     to save); prefill gate/up M = 32 / 128 / 512 / 2048: 35.5 / 57.7 /
//     169.0 / 590.3 against 25.4 / 29.4 / 67.9 / 237.0, k/v M = 32 / 128:
//     8.3 / 13.2 against 8.6 / 11.4;
//   pre-scaled kernel, M = 9..16: down 39.5-55.4 / 36.4-50.0; q/o, k/v and
//     gate/up within 0.9 either way;
//   the kernels for M <= 8 lose 1-5 us: their CTAs start behind the pass's
//     instead of beside the previous kernel's.
bool prepass_pays(int which, int M, int64_t N, int64_t K)
{
    if (which == 6) return N > 512 || M > 64;
    if (which == 4) return M >= 9 && K >= 8192;
    return false;
}

// The workspace arguments: 0 bytes is none; otherwise non-NULL, 16-byte aligned.
tq2_status check_workspace(const void *ws, size_t ws_bytes)
{
    if (ws_bytes == 0) return TQ2_OK;
    if (ws == nullptr) return TQ2_ERR_NULL;
    if (!aligned(ws, 16)) return TQ2_ERR_ALIGN;
    return TQ2_OK;
}

// With act_scale > 0 and a workspace, and where it pays for kernel `which`:
// convert x into the workspace (enqueued on a.stream) and point the kernel's
// x at the codes.  TQ2_ERR_ARG (nothing enqueued) when the workspace is too
// small for the pass the call would run.
tq2_status maybe_convert_first(tq2::MatvecArgs &a, int which, void *ws, size_t ws_bytes, int dev)
{
    if (a.act_scale == 0.0f || ws_bytes == 0 || !prepass_pays(which, a.M, a.N, a.K)) return TQ2_OK;
    if (ws_bytes < codes_bytes(a.M, a.K)) return TQ2_ERR_ARG;
    cudaError_t e = tq2::launch_fq_codes(a.x, (int64_t)a.M * a.K, a.inv_scale, static_cast<uint16_t *>(ws), a.stream,
                                         dev);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return from_cuda(e);
    a.x = static_cast<const uint16_t *>(ws);
    a.x_codes = 1;
    return TQ2_OK;
}

tq2_status matvec_common(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d,
                         int64_t N, int64_t K, void *y, tq2_dtype y_dtype, float act_scale,
                         float out_scale, void *ws, size_t ws_bytes, uint32_t *d_status, tq2_stream_t stream,
                         int impl, int stall_stage = -1, unsigned long long wait_limit_ns = 0, bool x_codes = false)
{
    tq2_status st = check_nk(N, K);
    if (st != TQ2_OK) return st;
    if (M < 0 || M > 16) return TQ2_ERR_SHAPE;
    if (y_dtype != TQ2_F32 && y_dtype != TQ2_F16) return TQ2_ERR_DTYPE;
    if (!(act_scale >= 0.0f) || !std::isfinite(act_scale)) return TQ2_ERR_ARG;
    if (!(out_scale >= 0.0f) || !std::isfinite(out_scale)) return TQ2_ERR_ARG;
    if (impl < 0 || impl > 7 || impl == 3 || impl == 5) return TQ2_ERR_ARG;  // 3, 5: retired
    if ((impl == 1 || impl == 7) && M > 2) return TQ2_ERR_ARG;
    if (M == 0 || N == 0) return TQ2_OK;
    if (y == nullptr) return TQ2_ERR_NULL;
    if (K > 0 && (x == nullptr || qs == nullptr || d == nullptr)) return TQ2_ERR_NULL;
    if (!aligned(x, 16) || !aligned(qs, 16) || !aligned(d, 2)) return TQ2_ERR_ALIGN;
    if (!aligned(y, y_dtype == TQ2_F32 ? 4 : 2)) return TQ2_ERR_ALIGN;
    if (d_status && !aligned(d_status, 4)) return TQ2_ERR_ALIGN;
    if ((st = check_workspace(ws, ws_bytes)) != TQ2_OK) return st;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t ybytes = (size_t)(M * N) * (y_dtype == TQ2_F32 ? 4 : 2);
    if (K == 0)  // empty sums: y = 0 (all-zero bits are +0 in fp32 and fp16; requantised, still 0)
        return from_cuda(cudaMemsetAsync(y, 0, ybytes, s));

    int dev = 0;
    if ((st = current_device(&dev)) != TQ2_OK) return st;
    tq2::MatvecArgs a;
    a.x = x;
    a.qs = qs;
    a.d = d;
    a.y = y;
    a.status = d_status;
    a.N = N;
    a.K = K;
    a.M = (int)M;
    a.y_f16 = (y_dtype == TQ2_F16);
    a.act_scale = act_scale;
    a.inv_scale = act_scale != 0.0f ? 1.0f / act_scale : 0.0f;  // IEEE-correct division
    a.out_scale = out_scale;
    a.inv_out = out_scale != 0.0f ? 1.0f / out_scale : 0.0f;
    a.stream = s;
    a.stall_stage = stall_stage;
    a.wait_limit_ns = wait_limit_ns;
    a.x_codes = x_codes ? 1 : 0;  // x holds the prologue's codes already (the grouped call's pass)

    // impl 0: for M <= 2 and a few output rows per CTA (k/v-sized N) the
    // small-N kernel, else for M <= 2 the class-column mma.sync kernel; for more rows the
    // pre-scaled mma.sync kernel, whose time grows with M, until the tcgen05
    // GEMM (whose time is flat up to 16 rows: an MMA of 128 weight rows x up
    // to 64 activation rows costs the same) is faster; CUDA cores as the last
    // resort.  The crossovers, measured on GB300 (us per call, back to back
    // over distinct weights, pre-scaled against GEMM, without / with the int8
    // prologue):
    //   q/o 4096x4096:      M = 10: 9.0 / 9.7, 10.5 / 11.4; M = 12: 10.1 / 9.7, 11.8 / 11.4
    //   k/v 256x4096:       M = 8: 5.2 / 6.5, 6.5 / 7.1; M = 10: 7.5 / 6.5, 9.0 / 7.2
    //   gate/up 16384x4096: M = 16: 20.7 / 23.4, 23.1 / 30.8 (the pre-scaled kernel throughout)
    //   down 4096x16384:    M = 8: 26.0 / 26.1, 31.2 / 34.1; M = 10: 35.7 / 26.1, 41.8 / 34.1
    // (M = 9 starts the pre-scaled kernel's second n-tile of 8 rows).
    int which = impl;
    if (impl == 0) {
        const bool gemm_wins = gemm_preferred(a.M, N, K, act_scale != 0.0f && (ws_bytes != 0 || x_codes));
        if (a.M <= 2 && tq2::smalln_matvec_preferred(a.M, N, K, dev)) which = 7;
        else if (a.M <= 2 && tq2::mma_matvec_supported(a.M, N, K, dev)) which = 1;
        else if (gemm_wins && tq2::gemm_tc05_supported(a.M, N, K, dev)) which = 6;
        else if (tq2::ps_matvec_supported(a.M, N, K, dev)) which = 4;
        else which = 2;
    } else if (impl == 1 && !tq2::mma_matvec_supported(a.M, N, K, dev)) {
        return TQ2_ERR_ARG;
    } else if (impl == 4 && !tq2::ps_matvec_supported(a.M, N, K, dev)) {
        return TQ2_ERR_ARG;
    } else if (impl == 6 && !tq2::gemm_tc05_supported(a.M, N, K, dev)) {
        return TQ2_ERR_ARG;
    } else if (impl == 7 && !tq2::smalln_matvec_supported(a.M, N, K, dev)) {
        return TQ2_ERR_ARG;
    }
    if (!x_codes && (st = maybe_convert_first(a, which, ws, ws_bytes, dev)) != TQ2_OK) return st;
    cudaError_t e = (which == 1)   ? tq2::launch_matvec_mma(a, dev)
                    : (which == 4) ? tq2::launch_matvec_ps(a, dev)
                    : (which == 6) ? tq2::launch_gemm_tc05(a, dev)
                    : (which == 7) ? tq2::launch_matvec_smalln(a, dev)
                                   : tq2::launch_matvec_simt(a, dev);
    if (e == cudaSuccess) e = cudaGetLastError();
    return from_cuda(e);
}

}  // namespace

extern "C" {

tq2_status tq2_pack(const int8_t *codes, int64_t N, int64_t K, uint8_t *qs, uint32_t *d_status,
                    tq2_stream_t stream)
{
    tq2_status st = check_nk(N, K);
    if (st != TQ2_OK) return st;
    if (N == 0 || K == 0) return TQ2_OK;
    if (codes == nullptr || qs == nullptr) return TQ2_ERR_NULL;
    if (d_status && !aligned(d_status, 4)) return TQ2_ERR_ALIGN;
    return from_cuda(tq2::launch_pack(codes, N, K, qs, d_status,
                                      reinterpret_cast<cudaStream_t>(stream)));
}

tq2_status tq2_unpack(const uint8_t *qs, int64_t N, int64_t K, int8_t *codes, tq2_stream_t stream)
{
    tq2_status st = check_nk(N, K);
    if (st != TQ2_OK) return st;
    if (N == 0 || K == 0) return TQ2_OK;
    if (codes == nullptr || qs == nullptr) return TQ2_ERR_NULL;
    return from_cuda(tq2::launch_unpack(qs, N, K, codes, reinterpret_cast<cudaStream_t>(stream)));
}

tq2_status tq2_from_dense(const void *W, tq2_dtype w_dtype, int64_t N, int64_t K, uint8_t *qs,
                          uint16_t *d, uint32_t *d_status, tq2_stream_t stream)
{
    tq2_status st = check_nk(N, K);
    if (st != TQ2_OK) return st;
    if (w_dtype != TQ2_F32 && w_dtype != TQ2_F16) return TQ2_ERR_DTYPE;
    if (N == 0 || K == 0) return TQ2_OK;
    if (W == nullptr || qs == nullptr || d == nullptr) return TQ2_ERR_NULL;
    if (!aligned(W, w_dtype == TQ2_F32 ? 4 : 2) || !aligned(d, 2)) return TQ2_ERR_ALIGN;
    if (d_status && !aligned(d_status, 4)) return TQ2_ERR_ALIGN;
    return from_cuda(tq2::launch_from_dense(W, w_dtype == TQ2_F16, N, K, qs, d, d_status,
                                            reinterpret_cast<cudaStream_t>(stream)));
}

tq2_status tq2_matvec(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d,
                      int64_t N, int64_t K, void *y, tq2_dtype y_dtype, float act_scale,
                      void *workspace, size_t workspace_bytes, uint32_t *d_status,
                      tq2_stream_t stream)
{
    return matvec_common(x, M, qs, d, N, K, y, y_dtype, act_scale, 0.0f, workspace, workspace_bytes, d_status,
                         stream, 0);
}

tq2_status tq2_matvec_impl(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d,
                           int64_t N, int64_t K, void *y, tq2_dtype y_dtype, float act_scale,
                           void *workspace, size_t workspace_bytes, uint32_t *d_status,
                           tq2_stream_t stream, int impl)
{
    return matvec_common(x, M, qs, d, N, K, y, y_dtype, act_scale, 0.0f, workspace, workspace_bytes, d_status,
                         stream, impl);
}

tq2_status tq2_matvec_requant(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d,
                              int64_t N, int64_t K, void *y, tq2_dtype y_dtype, float act_scale,
                              float out_scale, void *workspace, size_t workspace_bytes,
                              uint32_t *d_status, tq2_stream_t stream, int impl)
{
    return matvec_common(x, M, qs, d, N, K, y, y_dtype, act_scale, out_scale, workspace, workspace_bytes, d_status,
                         stream, impl);
}

size_t tq2_trace_size(void) { return tq2::trace_bytes(); }

tq2_status tq2_trace_read(void *host_dst, size_t bytes)
{
    if (tq2::trace_bytes() == 0) return TQ2_ERR_ARG;  // not a trace build
    if (host_dst == nullptr) return TQ2_ERR_NULL;
    if (bytes < tq2::trace_bytes()) return TQ2_ERR_ARG;
    return from_cuda(tq2::trace_read(host_dst, bytes));
}

tq2_status tq2_test_matvec_stall(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d, int64_t N,
                                 int64_t K, float *y, uint32_t *d_status, tq2_stream_t stream, int stall_stage,
                                 int wait_limit_us)
{
    if (stall_stage < 0) return TQ2_ERR_ARG;
    if (wait_limit_us < 1 || wait_limit_us > 200000) return TQ2_ERR_ARG;
    if (d_status == nullptr) return TQ2_ERR_NULL;
    return matvec_common(x, M, qs, d, N, K, y, TQ2_F32, 0.0f, 0.0f, nullptr, 0, d_status, stream, 1, stall_stage,
                         (unsigned long long)wait_limit_us * 1000ull);
}

}  // extern "C"

namespace {

// tq2_matvec_grouped and tq2_matvec_grouped_requant (out_scale: host array of
// n_mats scales, or nullptr for none).
// How a group of n matrices sharing x runs, before the device's own checks
// (`pass`: the prologue is on and a workspace given):
//   0  one launch of the class-column kernel (M <= 2);
//   1  one launch of the pre-scaled kernel;
//   2  consecutive single calls (with `pass`, x converted once for all).
// M = 3..8: one launch unless a matrix's single call would take the GEMM.
// M = 9..16: one launch saves the GEMM's per-call floor on k/v-sized
// matrices and beats separate pre-scaled calls up to M = 11; measured on
// GB300, us per group back to back over distinct weights, consecutive calls
// against one launch: q/k/v 4096x4096 + 2 x 256x4096 M = 9 / 12 / 16: 21.6 /
// 22.8 / 22.8 against 8.8 / 10.2 / 12.1 (with the prologue 24.5 / 25.7 /
// 25.7 against 10.1 / 11.8 / 14.3); gate/up 2 x 16384x4096 M = 9 / 12 / 16:
// 30.0 / 34.4 / 41.0 against 23.8 / 35.5 / 42.4.  At K >= 8192 the GEMM's
// single calls are far ahead of the pre-scaled kernel (down-sized K, M >= 9).
int grouped_plan(int64_t M, int64_t K, int n, const int64_t *N, bool pass)
{
    if (M <= 2) return 0;
    if (M <= 8) {
        for (int j = 0; j < n; ++j)
            if (N[j] > 0 && gemm_preferred((int)M, N[j], K, pass)) return 2;
        return 1;
    }
    if (K >= 8192) return 2;
    if (M <= 11) return 1;
    for (int j = 0; j < n; ++j)
        if (N[j] > 0 && N[j] <= 512) return 1;
    return 2;
}

// Whether a grouped call with the prologue and a workspace converts x once
// for the group: when it runs as consecutive calls.  (In one launch each CTA
// converts the x it reads: the pass measured no faster there, as for single
// calls at M <= 8.)
bool grouped_pass(int64_t M, int64_t K, int n, const int64_t *N)
{
    return M >= 3 && K > 0 && n > 1 && grouped_plan(M, K, n, N, true) == 2;
}

tq2_status matvec_grouped_common(const uint16_t *x, int64_t M, int64_t K, int n_mats, const uint8_t *const *qs,
                                 const uint16_t *const *d, const int64_t *N, void *const *y, tq2_dtype y_dtype,
                                 float act_scale, const float *out_scale, void *ws, size_t ws_bytes,
                                 uint32_t *d_status, tq2_stream_t stream)
{
    if (n_mats < 1 || n_mats > TQ2_MAX_GROUP) return TQ2_ERR_ARG;
    if (qs == nullptr || d == nullptr || N == nullptr || y == nullptr) return TQ2_ERR_NULL;
    // every matrix must pass the checks of a single call (no CUDA call yet)
    int live = 0;
    for (int j = 0; j < n_mats; ++j) {
        tq2_status st = check_nk(N[j], K);
        if (st != TQ2_OK) return st;
        if (M < 0 || M > 16) return TQ2_ERR_SHAPE;
        if (y_dtype != TQ2_F32 && y_dtype != TQ2_F16) return TQ2_ERR_DTYPE;
        if (!(act_scale >= 0.0f) || !std::isfinite(act_scale)) return TQ2_ERR_ARG;
        if (out_scale && (!(out_scale[j] >= 0.0f) || !std::isfinite(out_scale[j]))) return TQ2_ERR_ARG;
        if (M == 0 || N[j] == 0) continue;
        if (y[j] == nullptr) return TQ2_ERR_NULL;
        if (K > 0 && (x == nullptr || qs[j] == nullptr || d[j] == nullptr)) return TQ2_ERR_NULL;
        if (!aligned(x, 16) || !aligned(qs[j], 16) || !aligned(d[j], 2)) return TQ2_ERR_ALIGN;
        if (!aligned(y[j], y_dtype == TQ2_F32 ? 4 : 2)) return TQ2_ERR_ALIGN;
        ++live;
    }
    if (d_status && !aligned(d_status, 4)) return TQ2_ERR_ALIGN;
    tq2_status wst = check_workspace(ws, ws_bytes);
    if (wst != TQ2_OK) return wst;
    if (live == 0) return TQ2_OK;

    const uint8_t *gq[TQ2_MAX_GROUP];
    const uint16_t *gd[TQ2_MAX_GROUP];
    void *gy[TQ2_MAX_GROUP];
    int64_t gn[TQ2_MAX_GROUP];
    float gs[TQ2_MAX_GROUP], gi[TQ2_MAX_GROUP];
    int n = 0;
    for (int j = 0; j < n_mats; ++j) {
        if (M == 0 || N[j] == 0) continue;
        gq[n] = qs[j];
        gd[n] = d[j];
        gy[n] = y[j];
        gn[n] = N[j];
        gs[n] = out_scale ? out_scale[j] : 0.0f;
        gi[n] = gs[n] != 0.0f ? 1.0f / gs[n] : 0.0f;  // IEEE-correct division
        ++n;
    }
    int dev = 0;
    tq2_status st = TQ2_OK;
    if (K > 0 && n > 1) {
        if ((st = current_device(&dev)) != TQ2_OK) return st;
        // the pre-scaled kernel where a single call would run it, up to 8
        // rows (one n-tile): measured back to back over distinct weights,
        // q/k/v grouped against separate calls at M = 4 / 8: 5.0 / 6.4 against
        // 12.9 / 17.1 us, gate/up 16.7 / 19.6 against 20.1 / 25.0 us; at
        // M = 16 gate/up grouped took 42.4 against 41.6 us
        const int plan = grouped_plan(M, K, n, gn, act_scale != 0.0f && ws_bytes != 0);
        const bool mma = plan == 0 && tq2::mma_group_supported((int)M, n, gn, K, dev);
        const bool ps = plan == 1 && tq2::ps_group_supported((int)M, n, gn, K, dev);
        if (mma || ps) {
            tq2::MatvecArgs a;
            a.x = x;
            a.qs = nullptr;
            a.d = nullptr;
            a.y = nullptr;
            a.status = d_status;
            a.N = 0;
            a.K = K;
            a.M = (int)M;
            a.y_f16 = (y_dtype == TQ2_F16);
            a.act_scale = act_scale;
            a.inv_scale = act_scale != 0.0f ? 1.0f / act_scale : 0.0f;
            a.out_scale = 0.0f;  // per matrix: gs, gi
            a.inv_out = 0.0f;
            a.stream = reinterpret_cast<cudaStream_t>(stream);
            cudaError_t e = mma ? tq2::launch_matvec_mma_group(a, n, gq, gd, gy, gn, gs, gi, dev)
                                : tq2::launch_matvec_ps_group(a, n, gq, gd, gy, gn, gs, gi, dev);
            if (e == cudaSuccess) e = cudaGetLastError();
            return from_cuda(e);
        }
    }
    // otherwise one call per matrix, same x, same stream; with the prologue
    // and a workspace, x is converted once for all of them (the pages'
    // recipe: one input quantisation shared by q/k/v, one by gate/up)
    const bool pass = act_scale != 0.0f && ws_bytes >= codes_bytes(M, K) && grouped_pass(M, K, n, gn);
    if (act_scale != 0.0f && ws_bytes != 0 && !pass && grouped_pass(M, K, n, gn)) return TQ2_ERR_ARG;  // too small
    if (pass) {
        if (n == 1 && (st = current_device(&dev)) != TQ2_OK) return st;  // (n > 1 queried it above)
        cudaError_t e = tq2::launch_fq_codes(x, M * K, 1.0f / act_scale, static_cast<uint16_t *>(ws),
                                             reinterpret_cast<cudaStream_t>(stream), dev);
        if (e == cudaSuccess) e = cudaGetLastError();
        if (e != cudaSuccess) return from_cuda(e);
    }
    // without the group's pass (a single matrix, or a group the device
    // could not launch at once) each call may use the workspace by itself
    const uint16_t *xc = pass ? static_cast<const uint16_t *>(ws) : x;
    for (int j = 0; j < n; ++j) {
        st = matvec_common(xc, M, gq[j], gd[j], gn[j], K, gy[j], y_dtype, act_scale, gs[j], pass ? nullptr : ws,
                           pass ? 0 : ws_bytes, d_status, stream, 0, -1, 0, pass);
        if (st != TQ2_OK) return st;
    }
    return TQ2_OK;
}

}  // namespace

extern "C" {

tq2_status tq2_matvec_grouped(const uint16_t *x, int64_t M, int64_t K, int n_mats, const uint8_t *const *qs,
                              const uint16_t *const *d, const int64_t *N, void *const *y, tq2_dtype y_dtype,
                              float act_scale, void *workspace, size_t workspace_bytes, uint32_t *d_status,
                              tq2_stream_t stream)
{
    return matvec_grouped_common(x, M, K, n_mats, qs, d, N, y, y_dtype, act_scale, nullptr, workspace,
                                 workspace_bytes, d_status, stream);
}

tq2_status tq2_matvec_grouped_requant(const uint16_t *x, int64_t M, int64_t K, int n_mats, const uint8_t *const *qs,
                                      const uint16_t *const *d, const int64_t *N, void *const *y, tq2_dtype y_dtype,
                                      float act_scale, const float *out_scale, void *workspace,
                                      size_t workspace_bytes, uint32_t *d_status, tq2_stream_t stream)
{
    if (out_scale == nullptr) return TQ2_ERR_NULL;
    return matvec_grouped_common(x, M, K, n_mats, qs, d, N, y, y_dtype, act_scale, out_scale, workspace,
                                 workspace_bytes, d_status, stream);
}

size_t tq2_matvec_grouped_workspace_size(int64_t M, int64_t K, int n_mats, const int64_t *N)
{
    if (M < 1 || M > 16 || n_mats < 1 || n_mats > TQ2_MAX_GROUP || N == nullptr) return 0;
    for (int j = 0; j < n_mats; ++j)
        if (check_nk(N[j], K) != TQ2_OK) return 0;
    return grouped_pass(M, K, n_mats, N) ? codes_bytes(M, K) : 0;
}

}  // extern "C"

namespace {

// The host-side checks of tq2_gemm (no CUDA call); TQ2_OK with *done set
// when the call has nothing to do.
tq2_status gemm_check(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d, int64_t N, int64_t K,
                      void *y, tq2_dtype y_dtype, float act_scale, float out_scale, void *ws, size_t ws_bytes,
                      uint32_t *d_status, int impl, bool *done)
{
    *done = true;
    tq2_status st = check_nk(N, K);
    if (st != TQ2_OK) return st;
    if (M < 0 || M > ((int64_t)1 << 30)) return TQ2_ERR_SHAPE;
    if (M > 0 && N > 0 && M > kMaxElems / (N > K ? N : (K > 0 ? K : 1))) return TQ2_ERR_SHAPE;
    if (y_dtype != TQ2_F32 && y_dtype != TQ2_F16) return TQ2_ERR_DTYPE;
    if (!(act_scale >= 0.0f) || !std::isfinite(act_scale)) return TQ2_ERR_ARG;
    if (!(out_scale >= 0.0f) || !std::isfinite(out_scale)) return TQ2_ERR_ARG;
    if (impl < 0 || impl > 2) return TQ2_ERR_ARG;
    if (M == 0 || N == 0) return TQ2_OK;
    if (y == nullptr) return TQ2_ERR_NULL;
    if (K > 0 && (x == nullptr || qs == nullptr || d == nullptr)) return TQ2_ERR_NULL;
    if (!aligned(x, 16) || !aligned(qs, 16) || !aligned(d, 2)) return TQ2_ERR_ALIGN;
    if (!aligned(y, y_dtype == TQ2_F32 ? 4 : 2)) return TQ2_ERR_ALIGN;
    if (d_status && !aligned(d_status, 4)) return TQ2_ERR_ALIGN;
    if ((st = check_workspace(ws, ws_bytes)) != TQ2_OK) return st;
    *done = false;
    return TQ2_OK;
}

tq2_status gemm_common(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d, int64_t N, int64_t K,
                       void *y, tq2_dtype y_dtype, float act_scale, float out_scale, void *ws, size_t ws_bytes,
                       uint32_t *d_status, tq2_stream_t stream, int impl, int stall_stage = -1,
                       unsigned long long wait_limit_ns = 0)
{
    bool done = true;
    tq2_status st = gemm_check(x, M, qs, d, N, K, y, y_dtype, act_scale, out_scale, ws, ws_bytes, d_status, impl, &done);
    if (st != TQ2_OK || done) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t ebytes = (y_dtype == TQ2_F32 ? 4 : 2);
    if (K == 0) return from_cuda(cudaMemsetAsync(y, 0, (size_t)(M * N) * ebytes, s));

    int dev = 0;
    if ((st = current_device(&dev)) != TQ2_OK) return st;
    // impl 0: the tcgen05 GEMM for M > 16, else the matvec kernels on 16-row
    // slices of x (the same result contract)
    bool gemm = (impl == 1);
    if (impl == 0) gemm = M > 16 && tq2::gemm_tc05_supported(M, N, K, dev);
    if (gemm) {
        if (!tq2::gemm_tc05_supported(M, N, K, dev)) return TQ2_ERR_ARG;
        tq2::MatvecArgs a;
        a.x = x;
        a.qs = qs;
        a.d = d;
        a.y = y;
        a.status = d_status;
        a.N = N;
        a.K = K;
        a.M = (int)M;
        a.y_f16 = (y_dtype == TQ2_F16);
        a.act_scale = act_scale;
        a.inv_scale = act_scale != 0.0f ? 1.0f / act_scale : 0.0f;
        a.out_scale = out_scale;
        a.inv_out = out_scale != 0.0f ? 1.0f / out_scale : 0.0f;
        a.stream = s;
        a.stall_stage = stall_stage;
        a.wait_limit_ns = wait_limit_ns;
        if ((st = maybe_convert_first(a, 6, ws, ws_bytes, dev)) != TQ2_OK) return st;
        cudaError_t e = tq2::launch_gemm_tc05(a, dev);
        if (e == cudaSuccess) e = cudaGetLastError();
        return from_cuda(e);
    }
    for (int64_t m0 = 0; m0 < M; m0 += 16) {
        const int64_t mc = (M - m0 < 16) ? (M - m0) : 16;
        st = matvec_common(x + m0 * K, mc, qs, d, N, K, static_cast<uint8_t *>(y) + (size_t)(m0 * N) * ebytes,
                           y_dtype, act_scale, out_scale, ws, ws_bytes, d_status, stream, 0);
        if (st != TQ2_OK) return st;
    }
    return TQ2_OK;
}

}  // namespace

extern "C" {

tq2_status tq2_gemm(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d, int64_t N, int64_t K,
                    void *y, tq2_dtype y_dtype, float act_scale, float out_scale, void *workspace,
                    size_t workspace_bytes, uint32_t *d_status, tq2_stream_t stream, int impl)
{
    return gemm_common(x, M, qs, d, N, K, y, y_dtype, act_scale, out_scale, workspace, workspace_bytes, d_status,
                       stream, impl);
}

tq2_status tq2_gemm_static_ws(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d, int64_t N,
                              int64_t K, void *y, tq2_dtype y_dtype, float act_scale, float out_scale,
                              uint32_t *d_status, tq2_stream_t stream, int impl)
{
    void *ws = nullptr;
    size_t ws_bytes = 0;
    bool done = true;
    tq2_status st = gemm_check(x, M, qs, d, N, K, y, y_dtype, act_scale, out_scale, nullptr, 0, d_status, impl, &done);
    if (st != TQ2_OK || done) return st;
    if (act_scale > 0.0f && K > 0) {
        // the codes of M x K activations must fit the static scratch
        if (M > (int64_t)(tq2::kStaticScratchBytes / 2) / K) return TQ2_ERR_SHAPE;
        int dev = 0;
        st = current_device(&dev);
        if (st != TQ2_OK) return st;
        if ((st = from_cuda(tq2::static_codes_scratch(dev, &ws))) != TQ2_OK) return st;
        ws_bytes = tq2::kStaticScratchBytes;
    }
    return gemm_common(x, M, qs, d, N, K, y, y_dtype, act_scale, out_scale, ws, ws_bytes, d_status, stream, impl);
}

tq2_status tq2_test_gemm_stall(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *d, int64_t N,
                               int64_t K, float *y, float act_scale, uint32_t *d_status, tq2_stream_t stream,
                               int stall_stage, int wait_limit_us)
{
    if (stall_stage < 0) return TQ2_ERR_ARG;
    if (wait_limit_us < 1 || wait_limit_us > 200000) return TQ2_ERR_ARG;
    if (d_status == nullptr) return TQ2_ERR_NULL;
    return gemm_common(x, M, qs, d, N, K, y, TQ2_F32, act_scale, 0.0f, nullptr, 0, d_status, stream, 1, stall_stage,
                       (unsigned long long)wait_limit_us * 1000ull);
}

tq2_status tq2_affine4_matvec(const uint16_t *x, int64_t M, const uint8_t *qs, const uint16_t *s,
                              const uint16_t *z, int64_t N, int64_t K, int64_t G, void *y, tq2_dtype y_dtype,
                              uint32_t *d_status, tq2_stream_t stream)
{
    tq2_status st = check_nk(N, K);
    if (st != TQ2_OK) return st;
    if (M < 0 || M > 16) return TQ2_ERR_SHAPE;
    if (y_dtype != TQ2_F32 && y_dtype != TQ2_F16) return TQ2_ERR_DTYPE;
    if (G != 64 && G != 128 && G != 256) return TQ2_ERR_ARG;
    if (M == 0 || N == 0) return TQ2_OK;
    if (y == nullptr) return TQ2_ERR_NULL;
    if (K > 0 && (x == nullptr || qs == nullptr || s == nullptr || z == nullptr)) return TQ2_ERR_NULL;
    if (!aligned(x, 16) || !aligned(qs, 16) || !aligned(s, 16) || !aligned(z, 16)) return TQ2_ERR_ALIGN;
    if (!aligned(y, y_dtype == TQ2_F32 ? 4 : 2)) return TQ2_ERR_ALIGN;
    if (d_status && !aligned(d_status, 4)) return TQ2_ERR_ALIGN;
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) return from_cuda(cudaMemsetAsync(y, 0, (size_t)(M * N) * (y_dtype == TQ2_F32 ? 4 : 2), cs));

    int dev = 0;
    if ((st = current_device(&dev)) != TQ2_OK) return st;
    if (!tq2::affine4_supported(M, N, K, G, dev)) return TQ2_ERR_ARG;
    tq2::Affine4Args a;
    a.x = x;
    a.qs = qs;
    a.s = s;
    a.z = z;
    a.y = y;
    a.status = d_status;
    a.M = M;
    a.N = N;
    a.K = K;
    a.G = G;
    a.y_f16 = (y_dtype == TQ2_F16);
    a.stream = cs;
    cudaError_t e = tq2::launch_affine4(a, dev);
    if (e == cudaSuccess) e = cudaGetLastError();
    return from_cuda(e);
}

size_t tq2_matvec_workspace_size(int64_t M, int64_t N, int64_t K)
{
    if (M < 1 || M > 16 || check_nk(N, K) != TQ2_OK || N == 0 || K == 0) return 0;
    // the automatic plan runs the pass with the GEMM only (the pre-scaled
    // kernel would use it at M >= 9 with K >= 8192, where the GEMM runs)
    return (gemm_preferred((int)M, N, K, true) && prepass_pays(6, (int)M, N, K)) ? codes_bytes(M, K) : 0;
}

size_t tq2_gemm_workspace_size(int64_t M, int64_t N, int64_t K)
{
    if (M < 1 || M > ((int64_t)1 << 30) || check_nk(N, K) != TQ2_OK || N == 0 || K == 0) return 0;
    if (M > kMaxElems / (N > K ? N : K)) return 0;
    return codes_bytes(M, K);
}

const char *tq2_status_string(tq2_status status)
{
    switch (status) {
    case TQ2_OK: return "TQ2_OK";
    case TQ2_ERR_NULL: return "TQ2_ERR_NULL: a required pointer is NULL";
    case TQ2_ERR_SHAPE: return "TQ2_ERR_SHAPE: invalid shape (K % 256, negative size, M > 16, overflow)";
    case TQ2_ERR_ALIGN: return "TQ2_ERR_ALIGN: a pointer is not aligned as required";
    case TQ2_ERR_DTYPE: return "TQ2_ERR_DTYPE: unknown dtype";
    case TQ2_ERR_ARG: return "TQ2_ERR_ARG: invalid argument";
    case TQ2_ERR_CUDA: return "TQ2_ERR_CUDA: a CUDA call or kernel launch failed";
    case TQ2_ERR_TIMEOUT: return "TQ2_ERR_TIMEOUT: a bounded device wait ran out";
    }
    return "unknown tq2_status";
}

int tq2_version(void) { return 100; }

const char *tq2_last_cuda_error(void)
{
    static thread_local char buf[256];
    const cudaError_t e = t_last_cuda_error;
    snprintf(buf, sizeof buf, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return buf;
}

}  // extern "C"
