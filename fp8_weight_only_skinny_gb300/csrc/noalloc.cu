// noalloc.cu -- nvfp4_gemm_noalloc: the NVFP4 linear for callers that cannot
// allocate device memory.
//
// nvfp4_gemm needs the workspace that sk_init() obtains with cudaMalloc.  Some
// callers cannot do that: code that runs where allocation is forbidden or
// unsafe (inside a memory-pool or arena allocator that owns all device memory,
// in a process whose allocator is frozen after start-up, or under a strict
// no-allocation policy on the serving path).  This entry point serves them: its
// scratch memory (the control block and the split-K partial slots)
// is a file-scope static __device__ array of fixed size, created when the
// library is loaded and kept by every GPU that loads it until the process
// exits.  The caller passes only inputs and outputs.
//
// Set-up: the first call on a device (with that device current) resolves the
// array's device address with cudaGetSymbolAddress, the driver's tensor-map
// encoder and the SM count; make that first call before any stream capture.
// Every call shares the one array and leaves its contents behind, so calls
// whose kernels overlap on the GPU (different streams, or different host
// threads) race on it; each call resets the part it uses (the control block
// to zero, the partial slots it needs to empty) before its kernel.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/skinny.h"
#include "internal.h"
#include "kernel.cuh"

namespace {

// 8 MiB: the 4 KiB control block of the workspace layout and 8,384,512 bytes
// of split-K partial slots.
constexpr size_t NOALLOC_SCRATCH_BYTES = size_t(8) << 20;
static_assert(NOALLOC_SCRATCH_BYTES > sk::WS_PARTIAL_OFFSET, "scratch must hold the fixed workspace header");

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;

struct NoAllocDevice {
    unsigned char *scratch = nullptr;   // device address of g_noalloc_scratch on this device
    int num_sms = 0;
};

NoAllocDevice g_na[MAX_DEVICES];
std::mutex g_na_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_na_encode = nullptr;

// One-time set-up for the current device (see the file comment).
sk_status setup_current(NoAllocDevice **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return SK_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_na_mu);
    NoAllocDevice &d = g_na[dev];
    if (!d.scratch) {
        if (!g_na_encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return SK_ERR_CUDA;
            g_na_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        // In host code g_noalloc_scratch names a host-side stand-in, not device
        // memory: the kernel must get the address that this call returns.
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return SK_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SK_ERR_CUDA;
        d.num_sms = sms;
        d.scratch = static_cast<unsigned char *>(ptr);
    }
    *out = &d;
    return SK_OK;
}

bool na_aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" {

sk_status nvfp4_gemm_noalloc(const void *x, const uint8_t *W_codes, const uint8_t *W_scales, float W_gscale,
                             float *y, int M, int N, int K, void *stream) {
    // The same argument rules as nvfp4_gemm.
    if (M < 1 || M > 8 || N < 0 || K < 0) return SK_ERR_INVALID_ARG;
    if (!x || !W_codes || !W_scales || !y) return SK_ERR_INVALID_ARG;
    if (K % 256) return SK_ERR_UNSUPPORTED_SHAPE;
    if (!na_aligned(x, 16) || !na_aligned(W_codes, 16) || !na_aligned(W_scales, 16)) return SK_ERR_MISALIGNED;
    if (!na_aligned(y, 4)) return SK_ERR_MISALIGNED;
    NoAllocDevice *d = nullptr;
    if (sk_status st = setup_current(&d); st != SK_OK) return st;
    const long long G = (N + sk::RG - 1) / sk::RG, C = (K + sk::KC - 1) / sk::KC;
    const long long cap = (long long)(d->num_sms > 0 ? d->num_sms : 1) * 2;
    const int grid = int(G * C < cap ? G * C : cap);
    const int mp = sk::choose_mp(M, true, G * C, grid);
    // The split-K partial sums must fit in the static scratch.
    if (C > 1 && sk::WS_PARTIAL_OFFSET + size_t(G * C) * sk::unit_partial_bytes(mp) > NOALLOC_SCRATCH_BYTES)
        return SK_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (N == 0) return SK_OK;
    if (K == 0) return cudaMemsetAsync(y, 0, size_t(M) * N * 4, s) == cudaSuccess ? SK_OK : SK_ERR_CUDA;

    // The control block must start at zero and the partial slots the kernel
    // uses empty.  A completed call leaves them so, but the array is shared by
    // every call, so reset them here too (an aborted call may have left
    // partial sums behind).
    if (cudaMemsetAsync(d->scratch, 0, sk::WS_CTRL_BYTES, s) != cudaSuccess ||
        (C > 1 && sk::empty_partials(d->scratch, size_t(G * C) * sk::unit_partial_bytes(mp), s) != cudaSuccess))
        return SK_ERR_CUDA;

    sk::Params p = {};
    p.x = reinterpret_cast<const __half *>(x);
    p.fp8_scales = nullptr;
    p.gscale = W_gscale;
    p.y = y;
    p.argmax = nullptr;
    p.ws = d->scratch;
    p.M = M;
    p.N = N;
    p.K = K;
    p.G = int(G);
    p.C = int(C);
    p.KB = (K + 127) / 128;
    p.U = G * C;
    p.stall = sk::take_inject_stall();   // the test hook of sk_inject_wait_timeout()
    CUtensorMap tm_codes, tm_scales;
    if (!sk::encode_weight_maps(g_na_encode, true, W_codes, W_scales, K, N, &tm_codes, &tm_scales))
        return SK_ERR_CUDA;
    sk::take_weights_written(s);   // launched without PDL anyway; clears a quantizer's mark
    if (sk::launch_nvfp4(mp, sk::use_wide_x(x, M), false, false, tm_codes, tm_scales, p, grid, s, false, false) != cudaSuccess)
        return SK_ERR_CUDA;
    return SK_OK;
}

}  // extern "C"
