// sample.cu -- the sampled pick of each lm_head row: temperature, top-k and
// top-p, with the random draw passed in (one uniform per row).  The server
// the pages describe samples at a temperature (page "NVFP4 在 Volta 上！", the
// "温度 0.6" run) besides the greedy pick; include/skinny.h states the rule.
//
// One thread-block cluster of SC CTAs per row (16 for up to seven rows, 12 for
// eight), each CTA holding a contiguous slice of the row (copied into shared
// memory with every copy in flight at once): (1) a radix select, 8 bits at a
// time, finds the top_k-th largest of the row's ordered FP32 keys -- each CTA
// counts its slice into a histogram, and every CTA sums all SC histograms
// through distributed shared memory (SC / 4 remote reads per thread) to take
// the same decision; (2) every CTA writes its
// candidates (keys above that threshold, then keys equal to it, lowest index
// first) straight into the first CTA's shared memory, at offsets from the
// CTAs' published counts, each thread scanning one contiguous run of keys.
// As soon as the keys at or above the digits found so far number at most ST
// (usually after the first or second pass: a top_k of a few dozen sits in a
// sparse tail of the row), all of them become the candidates and the later
// passes are skipped (measured: the sampled pick 7-8 us faster per call);
// (3) that CTA sorts them by value, then index (bitonic: stages within a warp
// through register shuffles, the others through shared memory), and (4) a
// block scan of exp((z - z_max) / T) gives the running sums that decide the
// top-p cut and the draw.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/skinny.h"
#include "internal.h"

namespace {

constexpr int ST = 1024;   // threads per CTA, and the largest top_k

__device__ __forceinline__ unsigned int key_of(float v) {
    const unsigned int u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float value_of(unsigned int k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Exclusive prefix sum of v over the CTA, in thread order; the sum goes to
// *total (shared memory), readable by every thread on return.
__device__ __forceinline__ int block_excl_scan(int v, int *warp_tot, int *total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[wid] = x;
    __syncthreads();
    if (wid == 0) {
        const int w = warp_tot[lane];
        int t = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        warp_tot[lane] = t - w;               // exclusive over warps
        if (lane == 31) *total = t;
    }
    __syncthreads();
    const int r = warp_tot[wid] + x - v;
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

constexpr int CACHE = 49152;   // keys of a slice kept in shared memory (192 KB); the rest re-read from L2
// CTAs per row (non-portable cluster sizes): 16 for up to WIDE_MAX_M rows, 12
// for more.  Measured on the 151936-wide vocabulary against 8 CTAs per row:
// 16 were 3.4-3.9 us faster per call at M = 1 to 7 (half the slice per CTA to
// count and scan) but 4-5.4 us slower at M = 8, also with one CTA per SM
// forced; 12 were 2.2-2.9 us faster at M = 8.
constexpr int WIDE_MAX_M = 7;
constexpr int PDL_MAX_M = 5;

__device__ __forceinline__ unsigned int cluster_rank() {
    unsigned int r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA in the cluster: writes before it (shared or
// distributed shared) are visible to reads after it.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of `p` (a shared variable) in CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_addr(const void *p, unsigned int rank) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}

__device__ __forceinline__ unsigned int ld_dsmem(uint32_t a) {
    unsigned int v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return v;
}

__device__ __forceinline__ void st_dsmem(uint32_t a, unsigned long long v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}

// 4-byte asynchronous copy global -> shared; cp_async_wait_all waits for all
// of the thread's copies.
__device__ __forceinline__ void cp_async4(void *dst_smem, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<uint32_t>(
                     __cvta_generic_to_shared(dst_smem))),
                 "l"(src)
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Candidate sort key: (ordered value << 32) | ~index, so that a descending
// sort puts larger values first and, among equals, lower indices.
__device__ __forceinline__ unsigned long long cand_key(unsigned int key, int index) {
    return (static_cast<unsigned long long>(key) << 32) | static_cast<unsigned int>(~index);
}

// SC CTAs per row, one cluster (a multiple of 4; 12 and 16 are non-portable sizes).
template <int SC>
__global__ void __cluster_dims__(SC, 1, 1) __launch_bounds__(ST)
    sample_kernel(const float *logits, int N, const float *u, float T, int top_k, float top_p, int32_t *token) {
    static_assert(ST == 4 * 256 && SC % 4 == 0, "the histogram merge gives each thread SC / 4 of the ranks");
    extern __shared__ unsigned int skey[];           // this slice's FP32 bits (up to CACHE)
    __shared__ unsigned int hist[2][256];            // per pass, double-buffered across the cluster
    __shared__ unsigned int part[4][256];            // cluster totals of one pass, SC / 4 ranks per row
    __shared__ unsigned long long cand[ST];          // used in the first CTA of the cluster
    __shared__ float cum[ST];
    __shared__ unsigned long long warp_u64[8];
    __shared__ int warp_tmp[32];
    __shared__ float warp_f[32];
    __shared__ int s_cnt[2];                         // this CTA's keys above / equal to the threshold
    __shared__ unsigned int s_prefix, s_k;
    __shared__ int s_above, s_total, s_gt, s_gt_off, s_eq_off, s_keep, s_pick;
    __shared__ unsigned int s_bintot, s_binown;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const unsigned int rank = cluster_rank();
    const int row = blockIdx.x / SC;
    const int slice = (N + SC - 1) / SC;
    const int start = min(N, int(rank) * slice);
    const int len = min(N, start + slice) - start;
    const int ncache = min(len, CACHE);
    const float *z = logits + size_t(row) * N + start;
    // The logits belong to the projection until it has completed (a no-op
    // when this kernel was not launched as its programmatic dependent).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int i = tid; i < ncache; i += ST) cp_async4(skey + i, z + i);
    cp_async_wait_all();
    __syncthreads();
    auto key_at = [&](int i) -> unsigned int { return key_of(i < ncache ? __uint_as_float(skey[i]) : z[i]); };

    // (1) radix select over the cluster, 8 bits at a time from the top
    unsigned int prefix = 0, mask = 0, k = unsigned(top_k);
    int n_early = 0, own_early = 0;                  // early exit: candidates in the cluster / in this CTA
    int above = 0;                                   // this CTA's keys above the prefix found so far
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        unsigned int *h = hist[pass & 1];
        if (tid < 256) h[tid] = 0u;
        __syncthreads();
        for (int i0 = 0; i0 < len; i0 += 4 * ST) {
            unsigned int kk[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int i = i0 + j * ST + tid;
                kk[j] = i < len ? key_at(i) : 0u;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool act = i0 + j * ST + tid < len && (kk[j] & mask) == prefix;
                if (__any_sync(0xffffffffu, act)) {
                    const unsigned int bin = (kk[j] >> shift) & 255u;
                    // lanes with the same bin add once (the first pass's bins are few and crowded)
                    const unsigned int peers = __match_any_sync(0xffffffffu, act ? bin : 0xFFFFFFFFu);
                    if (act && __ffs(peers) - 1 == lane) atomicAdd(&h[bin], unsigned(__popc(peers)));
                }
            }
        }
        cluster_sync();
        {
            // every thread reads one bin of SC / 4 ranks (all loads in flight together)
            const unsigned int b = unsigned(tid) & 255u, r0 = unsigned(tid) >> 8;
            unsigned int v[SC / 4];
#pragma unroll
            for (int j = 0; j < SC / 4; ++j) v[j] = ld_dsmem(dsmem_addr(h + b, r0 + 4u * unsigned(j)));
            unsigned int t = 0u;
#pragma unroll
            for (int j = 0; j < SC / 4; ++j) t += v[j];
            part[r0][b] = t;
        }
        __syncthreads();
        // Thread t < 256 takes bin 255 - t: an inclusive scan over t is the
        // suffix sum over bins, of the cluster's total (high word) and of this
        // CTA's own count (low word).
        unsigned long long v = 0ull, tot = 0ull, own = 0ull;
        if (tid < 256) {
            const unsigned int b = 255u - unsigned(tid);
            tot = (unsigned long long)part[0][b] + part[1][b] + part[2][b] + part[3][b];
            own = h[b];
            v = (tot << 32) | own;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned long long y = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += y;
            }
            if (lane == 31) warp_u64[wid] = v;
        }
        __syncthreads();
        if (tid < 256) {
            for (int w = 0; w < wid; ++w) v += warp_u64[w];
            const unsigned long long s_tot = v >> 32, s_own = v & 0xFFFFFFFFull;
            // the digit: the cluster has >= k keys at or above it, < k above it
            if (s_tot >= k && s_tot - tot < k) {
                s_prefix = prefix | ((255u - unsigned(tid)) << shift);
                s_k = k - unsigned(s_tot - tot);
                s_above = int(s_own - own);
                s_bintot = unsigned(tot);
                s_binown = unsigned(own);
            }
        }
        __syncthreads();
        prefix = s_prefix;
        k = s_k;
        above += s_above;
        mask |= 0xFFu << shift;
        // Early exit: the keys whose top bits reach the prefix found so far
        // number at most ST, so all of them can be the candidates (the sort
        // orders them and the first top_k are the top_k).  The count comes
        // from cluster totals, so every CTA of the cluster decides alike.
        if (pass < 3 && top_k - int(k) + int(s_bintot) <= ST) {
            n_early = top_k - int(k) + int(s_bintot);
            own_early = above + int(s_binown);
            break;
        }
    }
    const uint32_t lead_cand = dsmem_addr(cand, 0);
    if (n_early > 0) {
        // every key whose masked top bits are at or above the prefix, after
        // those of lower ranks
        if (tid == 0) s_cnt[0] = own_early;
        cluster_sync();
        if (tid < 32) {
            int go = 0;
            if (tid < int(rank)) go = int(ld_dsmem(dsmem_addr(&s_cnt[0], unsigned(tid))));
#pragma unroll
            for (int o = 16; o; o >>= 1) go += __shfl_xor_sync(0xffffffffu, go, o);
            if (tid == 0) s_gt_off = go;
        }
        __syncthreads();
        const int per = (len + ST - 1) / ST;
        const int i_lo = min(len, tid * per), i_hi = min(len, i_lo + per);
        int n_mine = 0;
        for (int i = i_lo; i < i_hi; ++i) n_mine += (key_at(i) & mask) >= prefix;
        int pos = s_gt_off + block_excl_scan(n_mine, warp_tmp, &s_total);
        for (int i = i_lo; i < i_hi && n_mine > 0; ++i) {
            const unsigned int key = key_at(i);
            if ((key & mask) >= prefix) {
                st_dsmem(lead_cand + 8u * unsigned(pos), cand_key(key, start + i));
                ++pos;
                --n_mine;
            }
        }
    } else {
    const unsigned int thr_key = prefix;             // top_k - k keys of the row are above it, k more equal it
    const int need_eq = int(k), n_gt = top_k - int(k);

    // (2) publish this CTA's counts; candidates go to the first CTA's array
    if (tid == 0) {
        s_cnt[0] = above;
        s_cnt[1] = int(hist[1][thr_key & 255u]);    // the last pass's count at the final digit
        s_gt = 0;
    }
    cluster_sync();
    if (tid < 32) {                                  // lane r < rank reads rank r's counts
        int go = 0, eo = 0;
        if (tid < int(rank)) {
            go = int(ld_dsmem(dsmem_addr(&s_cnt[0], unsigned(tid))));
            eo = int(ld_dsmem(dsmem_addr(&s_cnt[1], unsigned(tid))));
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            go += __shfl_xor_sync(0xffffffffu, go, o);
            eo += __shfl_xor_sync(0xffffffffu, eo, o);
        }
        if (tid == 0) {
            s_gt_off = go;
            s_eq_off = eo;
        }
    }
    __syncthreads();
    const int gt_off = s_gt_off, eq_off = s_eq_off;
    // Each thread scans one contiguous run of the slice, so that index order
    // within a thread and thread order agree for the tied keys.
    const int per = (len + ST - 1) / ST;
    const int i_lo = min(len, tid * per), i_hi = min(len, i_lo + per);
    int n_eq = 0;
    for (int i = i_lo; i < i_hi; ++i) {
        const unsigned int key = key_at(i);
        if (key > thr_key) st_dsmem(lead_cand + 8u * unsigned(gt_off + atomicAdd(&s_gt, 1)), cand_key(key, start + i));
        n_eq += key == thr_key;
    }
    if (eq_off < need_eq) {                          // the same for every thread of the CTA
        int r = eq_off + block_excl_scan(n_eq, warp_tmp, &s_total);
        for (int i = i_lo; i < i_hi && n_eq > 0 && r < need_eq; ++i) {
            if (key_at(i) == thr_key) {
                st_dsmem(lead_cand + 8u * unsigned(n_gt + r), cand_key(thr_key, start + i));
                ++r;
            }
        }
    }
    }
    cluster_sync();                                  // all candidates are in the first CTA
    if (rank != 0) return;

    // (3) bitonic sort of the first pow2 >= top_k slots, descending; thread t
    // holds slot t, exchanging with slot t ^ stride through a shuffle within a
    // warp and through shared memory across warps
    const int n_cand = n_early > 0 ? n_early : top_k;
    int P2 = 1;
    while (P2 < n_cand) P2 <<= 1;
    unsigned long long v = tid < n_cand ? cand[tid] : 0ull;    // padding sorts last
    for (int size = 2; size <= P2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            unsigned long long w;
            if (stride >= 32) {
                __syncthreads();
                cand[tid] = v;
                __syncthreads();
                w = cand[tid ^ stride];
            } else {
                w = __shfl_xor_sync(0xffffffffu, v, stride);
            }
            const bool desc = (tid & size) == 0, lower = (tid & stride) == 0;
            const unsigned long long hi = v > w ? v : w, lo = v > w ? w : v;
            v = desc == lower ? hi : lo;
        }
    }
    __syncthreads();
    cand[tid] = v;
    __syncthreads();

    // (4) weights, running sums, the top-p cut and the draw
    const float z0 = value_of(static_cast<unsigned int>(cand[0] >> 32));
    if (!(T > 0.f)) {
        if (tid == 0) token[row] = int32_t(~static_cast<unsigned int>(cand[0] & 0xFFFFFFFFull));
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
    const float target = u[row] * cum[keep - 1];
    if (tid == 0) s_pick = keep - 1;
    __syncthreads();
    if (tid < keep && cum[tid] > target && (tid == 0 || cum[tid - 1] <= target)) s_pick = tid;
    __syncthreads();
    if (tid == 0) token[row] = int32_t(~static_cast<unsigned int>(cand[s_pick] & 0xFFFFFFFFull));
}

bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// pdl: launched as the projection's programmatic dependent, so that its CTAs
// are placed and wait on the device instead of after the projection retires.
template <int SC>
sk_status launch_sample(const float *logits, int N, const float *u, float T, int top_k, float top_p,
                        int32_t *token, int M, cudaStream_t s, bool pdl) {
    const int slice = (N + SC - 1) / SC;
    const size_t smem = size_t(slice < CACHE ? slice : CACHE) * sizeof(unsigned int);
    if (cudaFuncSetAttribute(sample_kernel<SC>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) !=
            cudaSuccess ||
        cudaFuncSetAttribute(sample_kernel<SC>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
        return SK_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(M * SC);
    cfg.blockDim = dim3(ST);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, sample_kernel<SC>, logits, N, u, T, top_k, top_p, token) == cudaSuccess
               ? SK_OK
               : SK_ERR_CUDA;
}

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
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Programmatic dependent launch up to PDL_MAX_M rows: measured 2.8 / 1.8 /
    // 1.2 us faster per call at M = 1 / 4 / 5, but 4.4 us slower at M = 7 and
    // 3.9 us at M = 8 (the early clusters then stand in the projection's way).
    const bool pdl = sk::pdl_enabled() && M <= PDL_MAX_M;
    return M <= WIDE_MAX_M ? launch_sample<16>(logits, N, u, temperature, top_k, top_p, token, M, s, pdl)
                           : launch_sample<12>(logits, N, u, temperature, top_k, top_p, token, M, s, pdl);
}

}  // extern "C"
