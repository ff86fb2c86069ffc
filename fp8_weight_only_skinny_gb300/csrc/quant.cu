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
// cvt.rn.satfinite.{e4m3x2,e2m1x2}.f32.  The per-weight quotients are formed
// by a product with the rounded reciprocal where that provably gives the same
// code (quotient_codes).  Both kernels stream the weight once (read 2 bytes,
// write 1 or 0.5 byte per weight, 16-byte accesses); with ~13 instructions per
// weight they sit between the HBM and the issue limits.
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

// Codes of a quotient pair (x0 / d, x1 / d): each code is defined from the
// binary32 quotient rounded to nearest-even, q = RN(x / d).  The kernels form
// p = RN(x * r) with r = RN(1 / d), which is faster than the division and in
// all but a few cases rounds to the same code.  The two roundings each add a
// relative error of at most 2^-24, so |p - x / d| <= (2^-23 + 2^-48) |x / d|
// and q lies within 3 units in the last place of x / d's binade from p: within
// 6 steps of p's bit pattern (3, or up to twice that where p and q sit in
// neighbouring binades).  Every rounding boundary of the code format (a
// midpoint between neighbouring values) has a binary32 pattern whose low bits
// are zero: 19 bits for E4M3, subnormal midpoints included (MASK = 2^19 - 1),
// 21 for E2M1 (MASK = 2^21 - 1).  Rounding to a code is monotone in the
// magnitude, so p and q can get different codes only when a boundary lies
// between them, hence within 6 steps of p; p's code is taken unless p's pattern
// is within 8 steps of a multiple of MASK + 1, and the pair is divided then.
// A zero p (x = 0) is such a multiple and is divided too.
template <uint32_t MASK, typename Cvt>
__device__ __forceinline__ uint32_t quotient_codes(float x0, float x1, float d, float r, Cvt cvt) {
    const float p0 = __fmul_rn(x0, r), p1 = __fmul_rn(x1, r);
    const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
    if (((b0 + 8u) & MASK) < 16u || ((b1 + 8u) & MASK) < 16u) return cvt(__fdiv_rn(x0, d), __fdiv_rn(x1, d));
    return cvt(p0, p1);
}

// Largest |value| of the eight FP16 values in v, as a bit pattern, folded into
// m: with the sign cleared, FP16 bit patterns order like the magnitudes
// (finite inputs).
__device__ __forceinline__ uint32_t absmax_bits8(const uint4 &v, uint32_t m) {
    m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
    return __vmaxu2(m, v.w & 0x7FFF7FFFu);
}

// The larger of the two FP16 bit patterns held in m2, as its FP32 value.
__device__ __forceinline__ float half_bits_value(uint32_t m2) {
    return __half2float(__ushort_as_half(uint16_t(__vmaxu2(m2, m2 >> 16) & 0xFFFFu)));
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

// FP8: persistent CTAs, four per SM, each streaming 128 x 128 blocks
// (b = blockIdx.x, blockIdx.x + gridDim.x, ...) through one shared-memory
// buffer filled by 2-D TMA loads (rows or columns past N or K are zero-filled,
// which leaves the block maximum unchanged).  Each thread keeps its 64 halves
// of the block in registers: their absolute maximum (on the bit patterns), the
// block maximum (two barriers), then the codes from the same registers.  The
// buffer is refilled with the CTA's next block as soon as every thread has
// read it, so that copy overlaps the codes of this one, and HBM is read once
// per weight.  Measured on the gate_up shape against three CTAs per SM with
// two buffers each: 112 -> 107 us; the CTAs' barriers, not the copies in
// flight, set the pace (two CTAs of three buffers: 127 us; 512 threads: 118
// us).
constexpr int FQ_BLK = 128;
constexpr int FQ_BUF = FQ_BLK * FQ_BLK * 2;          // 32 KB of FP16
constexpr size_t FQ_SMEM = 1024 + FQ_BUF + 8;
constexpr int FQ_CTAS_PER_SM = 4;                    // 64 registers x 256 threads x 4 fill the register file
constexpr uint64_t FQ_WAIT_NS = 1000000000ull;       // bounded waits: ~1 s

__global__ void __launch_bounds__(QT, FQ_CTAS_PER_SM) fp8_quantize_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                                          int N, int K,
                                                          int nbx, int nblocks, uint8_t *codes, float *scales) {
    extern __shared__ unsigned char fq_smem[];
    __shared__ float red[QT / 32];
    const uint32_t raw = sk::smem_u32(fq_smem);
    const uint32_t buf0 = (raw + 1023u) & ~1023u;
    const uint32_t bar = buf0 + FQ_BUF;
    const int tid = threadIdx.x;
    if (tid == 0) {
        sk::mbar_init(bar, 1);
        sk::fence_barrier_init();
    }
    __syncthreads();
    auto issue = [&](int blk) {
        sk::mbar_arrive_expect_tx(bar, FQ_BUF);
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
            ::"r"(buf0), "l"(reinterpret_cast<uint64_t>(&tm_w)), "r"((blk % nbx) * FQ_BLK),
              "r"((blk / nbx) * FQ_BLK), "r"(bar)
            : "memory");
    };
    if (tid == 0 && int(blockIdx.x) < nblocks) issue(blockIdx.x);
    int it = 0;
    for (int blk = blockIdx.x; blk < nblocks; blk += gridDim.x, ++it) {
        const uint64_t t0 = sk::globaltimer_ns();
        while (!sk::mbar_try_wait(bar, it & 1)) {
            if (sk::globaltimer_ns() - t0 > FQ_WAIT_NS) return;   // copy never landed: give up (codes unspecified)
        }
        // Thread tid holds words tid + 256 i of the block: row tid / 16 + 16 i,
        // columns 8 (tid % 16) .. + 8 (a warp reads 512 contiguous bytes).
        uint4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = sk::ld_shared_v4(buf0 + (tid + QT * i) * 16);
        uint32_t m2 = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) m2 = absmax_bits8(v[i], m2);
        const float a = block_max(half_bits_value(m2), red);   // its barriers also order every read of the buffer
        if (tid == 0 && blk + int(gridDim.x) < nblocks) issue(blk + gridDim.x);
        const float s = a > 0.f ? __fdiv_rn(a, 448.f) : 1.f;
        const float rs = __frcp_rn(s);
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
                lo |= quotient_codes<0x7FFFFu>(f[j], f[j + 1], s, rs, e4m3x2_rn) << (8 * j);
                hi |= quotient_codes<0x7FFFFu>(f[j + 4], f[j + 5], s, rs, e4m3x2_rn) << (8 * j);
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
    const uint4 *src = reinterpret_cast<const uint4 *>(w);
    const long long stride = (long long)gridDim.x * QT;
    long long i = blockIdx.x * (long long)QT + threadIdx.x;
    for (; i + 3 * stride < n8; i += 4 * stride) {   // four independent loads in flight per thread
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = src[i + u * stride];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float f[8];
            unpack8(v[u], f);
#pragma unroll
            for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(f[j]));
        }
    }
    for (; i < n8; i += stride) {
        float f[8];
        unpack8(src[i], f);
#pragma unroll
        for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(f[j]));
    }
    a = block_max(a, red);
    if (threadIdx.x == 0) atomicMax(amax, __float_as_uint(a));
}

// One 16-weight block (two 16-byte words of FP16): its E4M3 scale code and
// its eight code bytes.
__device__ __forceinline__ uint32_t encode_block(const uint4 &v0, const uint4 &v1, float G, uint2 &cw) {
    float f[16];
    {
        float t[8];
        unpack8(v0, t);
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = t[i];
        unpack8(v1, t);
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
        const float rd = __frcp_rn(denom);
#pragma unroll
        for (int i = 0; i < 16; i += 2)
            out[i >> 3] |= quotient_codes<0x1FFFFFu>(f[i], f[i + 1], denom, rd, e2m1x2_rn) << (4 * (i & 7));
    }
    cw = make_uint2(out[0], out[1]);
    return sc;
}

// One thread per two consecutive 16-element blocks of a row-major tensor
// (blocks 2j and 2j + 1 start at elements 32 j and 32 j + 16): two blocks'
// loads and arithmetic in flight per thread.  Measured on the gate_up shape
// against one block per thread: 145 -> 139 us (152 -> 147 us on a weight draw
// with more products near the boundary grid); four per thread: 170 us.
__global__ void __launch_bounds__(QT) nvfp4_quantize_kernel(const __half *w, long long nblocks,
                                                            const unsigned int *amax, uint8_t *codes,
                                                            uint8_t *scales, float *gscale) {
    const float A = __uint_as_float(*amax);
    const float G = A > 0.f ? __fdiv_rn(A, 2688.f) : 1.f;
    if (blockIdx.x == 0 && threadIdx.x == 0) *gscale = G;
    // Last pair first: the maximum's pass ends on the tensor's tail, which is
    // still in L2 when this pass starts.
    const long long npairs = (nblocks + 1) / 2;
    const long long pr = npairs - 1 - (blockIdx.x * (long long)QT + threadIdx.x);
    if (pr < 0) return;
    const long long b = 2 * pr;
    const bool two = b + 1 < nblocks;
    const uint4 *src = reinterpret_cast<const uint4 *>(w + b * 16);
    const uint4 v0 = src[0], v1 = src[1];
    uint4 v2 = make_uint4(0, 0, 0, 0), v3 = v2;
    if (two) {
        v2 = src[2];
        v3 = src[3];
    }
    uint2 c0, c1;
    const uint32_t s0 = encode_block(v0, v1, G, c0);
    if (two) {
        const uint32_t s1 = encode_block(v2, v3, G, c1);
        // codes and scales are only 8-byte and 1-byte aligned: 8-byte and byte stores
        *reinterpret_cast<uint2 *>(codes + b * 8) = c0;
        *reinterpret_cast<uint2 *>(codes + b * 8 + 8) = c1;
        scales[b] = uint8_t(s0);
        scales[b + 1] = uint8_t(s1);
    } else {
        *reinterpret_cast<uint2 *>(codes + b * 8) = c0;
        scales[b] = uint8_t(s0);
    }
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
    const int cap = (sms > 0 ? sms : 1) * FQ_CTAS_PER_SM;
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
        const long long cap = 8LL * (sk::device_sm_count() > 0 ? sk::device_sm_count() : 1);
        tensor_amax_kernel<<<int(want < cap ? want : cap), QT, 0, s>>>(reinterpret_cast<const __half *>(w), n8,
                                                                         amax);
    }
    const long long pairs = (nblocks + 1) / 2;
    const long long grid = pairs > 0 ? (pairs + QT - 1) / QT : 1;
    if (grid > 0x7FFFFFFFLL) return SK_ERR_UNSUPPORTED_SHAPE;
    nvfp4_quantize_kernel<<<unsigned(grid), QT, 0, s>>>(reinterpret_cast<const __half *>(w), nblocks, amax, codes,
                                                        scales, gscale);
    if (cudaGetLastError() != cudaSuccess) return SK_ERR_CUDA;
    sk::note_weights_written(s);
    return SK_OK;
}

}  // extern "C"
