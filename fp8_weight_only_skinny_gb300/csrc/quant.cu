// quant.cu -- FP16 weights -> NVFP4 (two-level scale) and FP8-E4M3 (128 x 128
// block scales), on the GPU: the conversion step that precedes the skinny
// linear layers (the pages convert an FP16 checkpoint to NVFP4 -- v100-skinny
// ai-manual.ru article, section "Конвертация модели в NVFP4" -- and keep the
// FP8 regions in FP8, page "NVFP4 在 Volta 上！", v1.1 section).
//
// Every step is an IEEE binary32 operation rounded to nearest-even, in the
// order include/skinny.h states, so the result is bit-for-bit reproducible:
// divisions and products use __fdiv_rn / __fmul_rn (no contraction), and the
// final roundings use the hardware's nearest-even, saturating conversions
// cvt.rn.satfinite.{e4m3x2,e2m1x2}.f32.  Both kernels are memory-bound
// streams (read 2 bytes, write 1 or 0.5 byte per weight, 16-byte accesses).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/skinny.h"
#include "internal.h"
#include "kernel.cuh"

namespace {

constexpr int QT = 256;   // threads per CTA

// Two FP32 values -> two E4M3 codes, nearest-even, saturating; lo in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_rn(float lo, float hi) {
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
    return d;
}

// Two FP32 values -> two E2M1 codes, nearest-even, saturating; lo in the low nibble.
__device__ __forceinline__ uint32_t e2m1x2_rn(float lo, float hi) {
    uint32_t d;
    asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// An E4M3 code -> its value (exact in FP16, then FP32).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(uint16_t(code & 0xFFu)));
    return __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFFu)));
}

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 p = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
        f[2 * i] = p.x;
        f[2 * i + 1] = p.y;
    }
}

__device__ __forceinline__ float block_max(float a, float *red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const int wid = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) red[wid] = a;
    __syncthreads();
    if (threadIdx.x < 32) {
        a = threadIdx.x < QT / 32 ? red[threadIdx.x] : 0.f;
#pragma unroll
        for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        if (threadIdx.x == 0) red[0] = a;
    }
    __syncthreads();
    return red[0];
}

// FP8: persistent CTAs, each streaming 128 x 128 blocks (b = blockIdx.x,
// blockIdx.x + gridDim.x, ...) through two shared-memory buffers filled by 2-D
// TMA loads (rows or columns past N or K are zero-filled, which leaves the
// block maximum unchanged).  Each thread keeps its 64 halves of the block in
// registers: their absolute maximum, the block maximum (two barriers), then
// the codes from the same registers.  The block's buffer is refilled with the
// block two ahead as soon as every thread has read it, so each CTA keeps two
// blocks in flight and HBM is read once per weight.
constexpr int FQ_BLK = 128;
constexpr int FQ_BUF = FQ_BLK * FQ_BLK * 2;          // 32 KB of FP16
constexpr size_t FQ_SMEM = 1024 + 2 * FQ_BUF + 16;
constexpr uint64_t FQ_WAIT_NS = 1000000000ull;       // bounded waits: ~1 s

__global__ void __launch_bounds__(QT) fp8_quantize_kernel(const __grid_constant__ CUtensorMap tm_w, int N, int K,
                                                          int nbx, int nblocks, uint8_t *codes, float *scales) {
    extern __shared__ unsigned char fq_smem[];
    __shared__ float red[QT / 32];
    const uint32_t raw = sk::smem_u32(fq_smem);
    const uint32_t buf0 = (raw + 1023u) & ~1023u;
    const uint32_t bar = buf0 + 2 * FQ_BUF;
    const int tid = threadIdx.x;
    if (tid == 0) {
        sk::mbar_init(bar, 1);
        sk::mbar_init(bar + 8, 1);
        sk::fence_barrier_init();
    }
    __syncthreads();
    auto issue = [&](int blk, int b) {
        sk::mbar_arrive_expect_tx(bar + 8 * b, FQ_BUF);
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
            ::"r"(buf0 + b * FQ_BUF), "l"(reinterpret_cast<uint64_t>(&tm_w)), "r"((blk % nbx) * FQ_BLK),
              "r"((blk / nbx) * FQ_BLK), "r"(bar + 8 * b)
            : "memory");
    };
    if (tid == 0) {
        if (int(blockIdx.x) < nblocks) issue(blockIdx.x, 0);
        if (int(blockIdx.x + gridDim.x) < nblocks) issue(blockIdx.x + gridDim.x, 1);
    }
    int it = 0;
    for (int blk = blockIdx.x; blk < nblocks; blk += gridDim.x, ++it) {
        const int b = it & 1;
        const uint64_t t0 = sk::globaltimer_ns();
        while (!sk::mbar_try_wait(bar + 8 * b, (it >> 1) & 1)) {
            if (sk::globaltimer_ns() - t0 > FQ_WAIT_NS) return;   // copy never landed: give up (codes unspecified)
        }
        // Thread tid holds words tid + 256 i of the block: row tid / 16 + 16 i,
        // columns 8 (tid % 16) .. + 8 (a warp reads 512 contiguous bytes).
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = sk::ld_shared_v4(buf0 + b * FQ_BUF + (tid + QT * i) * 16);
        float a = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float f[8];
            unpack8(v[i], f);
#pragma unroll
            for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(f[j]));
        }
        a = block_max(a, red);          // its barriers also order every read of the buffer
        if (tid == 0 && blk + 2 * int(gridDim.x) < nblocks) issue(blk + 2 * gridDim.x, b);
        const float s = a > 0.f ? __fdiv_rn(a, 448.f) : 1.f;
        const int r0 = (blk / nbx) * FQ_BLK, c0 = (blk % nbx) * FQ_BLK;
        if (tid == 0) scales[blk] = s;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = r0 + tid / 16 + 16 * i, cc = c0 + (tid % 16) * 8;
            if (r >= N || cc >= K) continue;
            float f[8];
            unpack8(v[i], f);
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int j = 0; j < 4; j += 2) {
                lo |= e4m3x2_rn(__fdiv_rn(f[j], s), __fdiv_rn(f[j + 1], s)) << (8 * j);
                hi |= e4m3x2_rn(__fdiv_rn(f[j + 4], s), __fdiv_rn(f[j + 5], s)) << (8 * j);
            }
            *reinterpret_cast<uint2 *>(codes + size_t(r) * K + cc) = make_uint2(lo, hi);
        }
    }
}

// max |w| over the whole tensor into *amax (float bits; non-negative floats
// order like their bit patterns, so an integer maximum is exact).
__global__ void __launch_bounds__(QT) tensor_amax_kernel(const __half *w, long long n8, unsigned int *amax) {
    __shared__ float red[QT / 32];
    float a = 0.f;
    for (long long i = blockIdx.x * (long long)QT + threadIdx.x; i < n8; i += (long long)gridDim.x * QT) {
        float f[8];
        unpack8(reinterpret_cast<const uint4 *>(w)[i], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(f[j]));
    }
    a = block_max(a, red);
    if (threadIdx.x == 0) atomicMax(amax, __float_as_uint(a));
}

// One thread per 16-element block of a row (row-major, so block b starts at
// element 16 b): its E4M3 scale and its eight code bytes.
__global__ void __launch_bounds__(QT) nvfp4_quantize_kernel(const __half *w, long long nblocks,
                                                            const unsigned int *amax, uint8_t *codes,
                                                            uint8_t *scales, float *gscale) {
    const float A = __uint_as_float(*amax);
    const float G = A > 0.f ? __fdiv_rn(A, 2688.f) : 1.f;
    if (blockIdx.x == 0 && threadIdx.x == 0) *gscale = G;
    const long long b = blockIdx.x * (long long)QT + threadIdx.x;
    if (b >= nblocks) return;
    float f[16];
    {
        const uint4 *src = reinterpret_cast<const uint4 *>(w + b * 16);
        float t[8];
        unpack8(src[0], t);
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = t[i];
        unpack8(src[1], t);
#pragma unroll
        for (int i = 0; i < 8; ++i) f[8 + i] = t[i];
    }
    float bmax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(f[i]));
    const uint32_t sc = e4m3x2_rn(__fdiv_rn(__fdiv_rn(bmax, 6.f), G), 0.f) & 0xFFu;
    const float S = e4m3_value(sc);
    uint32_t out[2] = {0u, 0u};
    if (S == 0.f) {
        // The scale underflowed: every code is a zero carrying the input's sign.
#pragma unroll
        for (int i = 0; i < 16; ++i)
            if (__float_as_uint(f[i]) >> 31) out[i >> 3] |= 0x8u << (4 * (i & 7));
    } else {
        const float denom = __fmul_rn(S, G);
#pragma unroll
        for (int i = 0; i < 16; i += 2)
            out[i >> 3] |= e2m1x2_rn(__fdiv_rn(f[i], denom), __fdiv_rn(f[i + 1], denom)) << (4 * (i & 7));
    }
    *reinterpret_cast<uint2 *>(codes + b * 8) = make_uint2(out[0], out[1]);
    scales[b] = uint8_t(sc);
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" {

sk_status fp8_quantize(const void *w, uint8_t *codes, float *scales, int N, int K, void *stream) {
    if (N < 0 || K < 0) return SK_ERR_INVALID_ARG;
    if (N == 0 || K == 0) return SK_OK;
    if (!w || !codes || !scales) return SK_ERR_INVALID_ARG;
    if (K % 8) return SK_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(w, 16) || !aligned(codes, 8) || !aligned(scales, 4)) return SK_ERR_MISALIGNED;
    const long long nbx = (K + 127) / 128, nby = (N + 127) / 128;
    if (nbx * nby > 0x7FFFFFFFLL) return SK_ERR_UNSUPPORTED_SHAPE;
    const int nblocks = int(nbx * nby);
    CUtensorMap tm;
    if (!sk::encode_2d_u16(&tm, w, uint64_t(K), uint64_t(N), FQ_BLK, FQ_BLK)) return SK_ERR_CUDA;
    static bool attr_done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SK_ERR_CUDA;
    if (dev < 64 && !attr_done[dev]) {
        if (cudaFuncSetAttribute(fp8_quantize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(FQ_SMEM)) !=
            cudaSuccess)
            return SK_ERR_CUDA;
        attr_done[dev] = true;
    }
    const int sms = sk::device_sm_count();
    const int cap = (sms > 0 ? sms : 1) * 3;                   // three CTAs (2 x 32 KB buffers) per SM
    const int grid = nblocks < cap ? nblocks : cap;
    fp8_quantize_kernel<<<grid, QT, FQ_SMEM, reinterpret_cast<cudaStream_t>(stream)>>>(tm, N, K, int(nbx), nblocks,
                                                                                    codes, scales);
    if (cudaGetLastError() != cudaSuccess) return SK_ERR_CUDA;
    sk::note_weights_written(reinterpret_cast<cudaStream_t>(stream));
    return SK_OK;
}

sk_status nvfp4_quantize(const void *w, uint8_t *codes, uint8_t *scales, float *gscale, int N, int K,
                         void *stream) {
    if (N < 0 || K < 0) return SK_ERR_INVALID_ARG;
    if (!w || !codes || !scales || !gscale) return SK_ERR_INVALID_ARG;
    if (K % 16) return SK_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(w, 16) || !aligned(codes, 8) || !aligned(gscale, 4)) return SK_ERR_MISALIGNED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    unsigned char *ws = sk::workspace_for(s);
    if (!ws) return SK_ERR_NOT_INITIALIZED;
    unsigned int *amax = &reinterpret_cast<sk::Ctrl *>(ws)->qamax;
    const long long n8 = (long long)N * K / 8, nblocks = (long long)N * (K / 16);
    if (cudaMemsetAsync(amax, 0, sizeof(unsigned int), s) != cudaSuccess) return SK_ERR_CUDA;
    if (n8 > 0) {
        const long long want = (n8 + QT - 1) / QT;
        tensor_amax_kernel<<<int(want < 1024 ? want : 1024), QT, 0, s>>>(reinterpret_cast<const __half *>(w), n8,
                                                                         amax);
    }
    const long long grid = nblocks > 0 ? (nblocks + QT - 1) / QT : 1;
    if (grid > 0x7FFFFFFFLL) return SK_ERR_UNSUPPORTED_SHAPE;
    nvfp4_quantize_kernel<<<unsigned(grid), QT, 0, s>>>(reinterpret_cast<const __half *>(w), nblocks, amax, codes,
                                                        scales, gscale);
    if (cudaGetLastError() != cudaSuccess) return SK_ERR_CUDA;
    sk::note_weights_written(s);
    return SK_OK;
}

}  // extern "C"
