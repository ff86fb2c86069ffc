// sample.cu -- the sampled pick of each lm_head row: temperature, top-k and
// top-p, with the random draw passed in (one uniform per row).  The server
// the pages describe samples at a temperature (page "NVFP4 在 Volta 上！", the
// "温度 0.6" run) besides the greedy pick; include/skinny.h states the rule.
//
// One CTA of 1024 threads per row: (1) a radix select over the row's ordered
// FP32 keys finds the top_k-th largest; (2) an index-ordered pass gathers the
// top_k candidates (ties at the threshold taken lowest index first); (3) a
// bitonic sort orders them by value, then index; (4) a block scan of
// exp((z - z_max) / T) gives the running sums that decide the top-p cut and
// the draw.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/skinny.h"

namespace {

constexpr int ST = 1024;   // threads per CTA, and the largest top_k

__device__ __forceinline__ unsigned int key_of(float v) {
    const unsigned int u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float value_of(unsigned int k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Exclusive prefix count of `flag` over the CTA, in thread order; the sum goes
// to *total (shared memory), readable by every thread on return.
__device__ __forceinline__ int block_rank(bool flag, int *warp_tot, int *total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const unsigned int b = __ballot_sync(0xffffffffu, flag);
    const int in_warp = __popc(b & ((1u << lane) - 1u));
    if (lane == 0) warp_tot[wid] = __popc(b);
    __syncthreads();
    if (wid == 0) {
        const int v = warp_tot[lane];
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        warp_tot[lane] = x - v;               // exclusive
        if (lane == 31) *total = x;
    }
    __syncthreads();
    const int r = warp_tot[wid] + in_warp;
    __syncthreads();
    return r;
}

// Inclusive prefix sum of v over the CTA, in thread order.
__device__ __forceinline__ float block_scan(float v, float *warp_sum) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    float x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sum[wid] = x;
    __syncthreads();
    if (wid == 0) {
        float s = warp_sum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_sum[lane] = s;                   // inclusive over warps
    }
    __syncthreads();
    const float r = x + (wid > 0 ? warp_sum[wid - 1] : 0.f);
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(ST) sample_kernel(const float *logits, int N, const float *u, float T, int top_k,
                                                    float top_p, int32_t *token) {
    __shared__ unsigned int hist[256];
    __shared__ unsigned long long cand[ST];
    __shared__ float cum[ST];
    __shared__ int warp_tmp[32];
    __shared__ float warp_f[32];
    __shared__ unsigned int s_prefix, s_k;
    __shared__ int s_total, s_gt, s_eq, s_keep, s_pick;
    const int tid = threadIdx.x;
    const float *z = logits + size_t(blockIdx.x) * N;

    // (1) radix select, 8 bits at a time from the top: the top_k-th largest key
    unsigned int prefix = 0, mask = 0, k = unsigned(top_k);
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += ST) hist[i] = 0u;
        __syncthreads();
        for (int i = tid; i < N; i += ST) {
            const unsigned int key = key_of(z[i]);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (tid == 0) {
            unsigned int acc = 0;
            int d = 255;
            for (; d > 0; --d) {
                if (acc + hist[d] >= k) break;
                acc += hist[d];
            }
            s_prefix = prefix | (unsigned(d) << shift);
            s_k = k - acc;
        }
        __syncthreads();
        prefix = s_prefix;
        k = s_k;
        mask |= 0xFFu << shift;
        __syncthreads();
    }
    const unsigned int thr_key = prefix;           // top_k - k keys are above it; k more equal it
    const int need_eq = int(k), n_gt = top_k - int(k);

    // (2) gather: every key above the threshold, then the first need_eq equal
    // keys in index order.  Sort key: (ordered value << 32) | ~index, so that a
    // descending sort puts larger values first and, among equals, lower indices.
    if (tid == 0) {
        s_gt = 0;
        s_eq = 0;
    }
    __syncthreads();
    for (int base = 0; base < N; base += ST) {
        const int i = base + tid;
        const unsigned int key = i < N ? key_of(z[i]) : 0u;
        const bool gt = i < N && key > thr_key, eq = i < N && key == thr_key;
        const unsigned long long ck = (static_cast<unsigned long long>(key) << 32) | static_cast<unsigned int>(~i);
        if (gt) cand[atomicAdd(&s_gt, 1)] = ck;
        const int r = block_rank(eq, warp_tmp, &s_total);
        const int rank = s_eq + r;
        if (eq && rank < need_eq) cand[n_gt + rank] = ck;
        __syncthreads();
        if (tid == 0) s_eq += s_total;
        __syncthreads();
    }
    if (tid >= top_k) cand[tid] = 0ull;            // padding sorts last
    __syncthreads();

    // (3) bitonic sort, descending
    for (int size = 2; size <= ST; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            const int j = tid ^ stride;
            if (j > tid) {
                const unsigned long long a = cand[tid], b = cand[j];
                const bool desc = (tid & size) == 0;
                if (desc ? (a < b) : (a > b)) {
                    cand[tid] = b;
                    cand[j] = a;
                }
            }
            __syncthreads();
        }
    }

    // (4) weights, running sums, the top-p cut and the draw
    const float z0 = value_of(static_cast<unsigned int>(cand[0] >> 32));
    if (!(T > 0.f)) {
        if (tid == 0) token[blockIdx.x] = int32_t(~static_cast<unsigned int>(cand[0] & 0xFFFFFFFFull));
        return;
    }
    const float zj = value_of(static_cast<unsigned int>(cand[tid] >> 32));
    const float p = tid < top_k ? expf((zj - z0) / T) : 0.f;
    cum[tid] = block_scan(p, warp_f);
    __syncthreads();
    const float total = cum[top_k - 1];
    const float thr = top_p * total;
    if (tid == 0) s_keep = top_k;
    __syncthreads();
    if (tid < top_k && cum[tid] >= thr && (tid == 0 || cum[tid - 1] < thr)) s_keep = tid + 1;
    __syncthreads();
    const int keep = s_keep;
    const float target = u[blockIdx.x] * cum[keep - 1];
    if (tid == 0) s_pick = keep - 1;
    __syncthreads();
    if (tid < keep && cum[tid] > target && (tid == 0 || cum[tid - 1] <= target)) s_pick = tid;
    __syncthreads();
    if (tid == 0) token[blockIdx.x] = int32_t(~static_cast<unsigned int>(cand[s_pick] & 0xFFFFFFFFull));
}

bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" {

sk_status lm_head_sample(const void *x, const uint8_t *W_codes, const uint8_t *W_scales, float W_gscale,
                         float *logits, const float *u, float temperature, int top_k, float top_p, int32_t *token,
                         int M, int N, int K, void *stream) {
    if (!logits || !u || !token) return SK_ERR_INVALID_ARG;
    if (M < 1 || M > 8 || N < 1 || K < 1) return SK_ERR_INVALID_ARG;
    if (top_k < 1 || top_k > N) return SK_ERR_INVALID_ARG;
    if (top_k > ST) return SK_ERR_UNSUPPORTED_SHAPE;
    if (!(top_p > 0.f && top_p <= 1.f)) return SK_ERR_INVALID_ARG;
    if (!aligned4(u) || !aligned4(token)) return SK_ERR_MISALIGNED;
    const sk_status st = nvfp4_gemm(x, W_codes, W_scales, W_gscale, logits, M, N, K, stream);
    if (st != SK_OK) return st;
    sample_kernel<<<M, ST, 0, reinterpret_cast<cudaStream_t>(stream)>>>(logits, N, u, temperature, top_k, top_p,
                                                                       token);
    return cudaGetLastError() == cudaSuccess ? SK_OK : SK_ERR_CUDA;
}

}  // extern "C"
