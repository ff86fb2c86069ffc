// api.cu -- the C ABI of libskinny (see include/skinny.h): argument checks,
// workspace management, TMA descriptor encoding and kernel selection.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>

#include "../../include/skinny.h"
#include "internal.h"
#include "kernel.cuh"

namespace {

constexpr int MAX_DEVICES = 64;
constexpr size_t DEFAULT_WORKSPACE = size_t(64) << 20;

struct DeviceState {
    unsigned char *ws = nullptr;
    size_t bytes = 0;
    int num_sms = 0;
};

DeviceState g_dev[MAX_DEVICES];
std::mutex g_mu;

// Workspaces of individual streams (sk_stream_workspace), guarded by g_mu.
struct StreamWs {
    int dev = -1;
    cudaStream_t stream = nullptr;
    unsigned char *ws = nullptr;
    size_t bytes = 0;
};
constexpr int MAX_STREAM_WS = 64;
StreamWs g_sws[MAX_STREAM_WS];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
int g_pdl = 1;
std::atomic<int> g_variant{SK_VARIANT_AUTO};
std::atomic<int> g_inject_stall{0};

// Streams whose latest launch of this library was a weight quantizer (a short
// list: one entry per stream that quantizes; see internal.h).
std::mutex g_wq_mu;
constexpr int MAX_MARKED_STREAMS = 64;
cudaStream_t g_wq_streams[MAX_MARKED_STREAMS];
int g_wq_n = 0;
bool g_wq_overflow = false;   // more streams than slots: no linear launch uses PDL until one clears

sk_status resolve_encode() {
    if (g_encode) return SK_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return SK_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return SK_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// The workspace a call on `s` uses on the current device: the stream's own if
// it has one (then `own` is set), else the device's; false if neither exists.
struct WsRef {
    unsigned char *ws = nullptr;
    size_t bytes = 0;
    int num_sms = 0;
    bool own = false;
};
bool workspace_ref(cudaStream_t s, WsRef *r) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    for (const StreamWs &e : g_sws)
        if (e.ws && e.dev == dev && e.stream == s) {
            *r = WsRef{e.ws, e.bytes, g_dev[dev].num_sms, true};
            return true;
        }
    if (!g_dev[dev].ws) return false;
    *r = WsRef{g_dev[dev].ws, g_dev[dev].bytes, g_dev[dev].num_sms, false};
    return true;
}

// Persistent grid: CTAS_PER_SM CTAs per SM, never more CTAs than units.
// SK_CTAS_PER_SM (1..4) overrides the CTAs per SM; SK_MAX_CTAS caps the grid,
// which the tests use to give every CTA many units on small shapes (ring
// wrap-around, k-chunk changes and multi-unit fix-ups).
int grid_for(int num_sms, long long units) {
    int per_sm = 2;
    if (const char *e = std::getenv("SK_CTAS_PER_SM")) {
        const int v = std::atoi(e);
        if (v >= 1 && v <= 4) per_sm = v;
    }
    long long g = (long long)(num_sms > 0 ? num_sms : 1) * per_sm;
    if (const char *e = std::getenv("SK_MAX_CTAS")) {
        const long long v = std::atoll(e);
        if (v >= 1 && v < g) g = v;
    }
    return int(units < g ? units : g);
}

enum class Kind { NVFP4, NVFP4_F16, FP8, FP8_F16, LMHEAD };

sk_status zero_outputs(void *y, size_t y_bytes, int32_t *argmax, int M, cudaStream_t s) {
    if (y && y_bytes && cudaMemsetAsync(y, 0, y_bytes, s) != cudaSuccess) return SK_ERR_CUDA;
    if (argmax && cudaMemsetAsync(argmax, 0, size_t(M) * 4, s) != cudaSuccess) return SK_ERR_CUDA;
    return SK_OK;
}

sk_status run(Kind kind, const void *x, const uint8_t *codes, const void *scales, float gscale, void *y,
              int32_t *argmax, int M, int N, int K, void *stream, const int32_t *draft = nullptr,
              int32_t *accept = nullptr) {
    const bool nv = (kind == Kind::NVFP4 || kind == Kind::NVFP4_F16 || kind == Kind::LMHEAD);
    const bool f16 = (kind == Kind::NVFP4_F16 || kind == Kind::FP8_F16);
    const bool am = (kind == Kind::LMHEAD);
    // ---- argument checks (nothing is launched before these pass)
    if (M < 1 || M > 8 || N < 0 || K < 0) return SK_ERR_INVALID_ARG;
    if (am && N < 1) return SK_ERR_INVALID_ARG;
    if (!x || !codes || !scales) return SK_ERR_INVALID_ARG;
    if (am ? !argmax : !y) return SK_ERR_INVALID_ARG;
    if (nv ? (K % 256) : (K % 128)) return SK_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(x, 16) || !aligned(codes, 16)) return SK_ERR_MISALIGNED;
    if (nv ? !aligned(scales, 16) : !aligned(scales, 4)) return SK_ERR_MISALIGNED;
    if (y && !aligned(y, f16 ? 2 : 4)) return SK_ERR_MISALIGNED;
    if (argmax && !aligned(argmax, 4)) return SK_ERR_MISALIGNED;
    if (accept) {
        if (M > 1 && !draft) return SK_ERR_INVALID_ARG;
        if (K == 0) return SK_ERR_UNSUPPORTED_SHAPE;   // no logits to verify against
        if (!aligned(accept, 4) || (draft && !aligned(draft, 4))) return SK_ERR_MISALIGNED;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    WsRef wr;
    if (!workspace_ref(s, &wr)) return SK_ERR_NOT_INITIALIZED;
    if (N == 0) return SK_OK;
    if (K == 0) return zero_outputs(y, size_t(M) * N * (f16 ? 2 : 4), argmax, M, s);

    sk::Params p = {};
    p.x = reinterpret_cast<const __half *>(x);
    p.fp8_scales = nv ? nullptr : reinterpret_cast<const float *>(scales);
    p.gscale = nv ? gscale : 1.0f;
    p.y = y;
    p.argmax = argmax;
    p.draft = draft;
    p.accept = accept;
    p.ws = wr.ws;
    p.M = M;
    p.N = N;
    p.K = K;
    p.G = (N + sk::RG - 1) / sk::RG;
    p.C = (K + sk::KC - 1) / sk::KC;
    p.KB = (K + 127) / 128;
    p.U = (long long)p.G * p.C;
    const int grid = grid_for(wr.num_sms, p.U);
    const int mp = sk::choose_mp(M, nv, p.U, grid);
    const bool xwide = sk::use_wide_x(x, M);
    if (p.C > 1) {
        const size_t need = size_t(p.U) * sk::unit_partial_bytes(mp);
        if (sk::WS_PARTIAL_OFFSET + need > wr.bytes) return SK_ERR_WORKSPACE;
    }
    p.stall = sk::take_inject_stall();
    // No programmatic dependent launch right after a quantizer on this stream:
    // its codes and scales must be complete before this kernel reads weights.
    // A stream with a workspace of its own may run beside other streams: its
    // kernels launch cooperatively, so that the whole grid is resident before
    // any CTA starts (the split-K owners wait on other CTAs of the grid), and
    // without PDL.
    const bool coop = wr.own;
    const bool pdl = !sk::take_weights_written(s) && g_pdl != 0 && !coop;

    CUtensorMap tm_codes, tm_scales;
    if (nv) {
        if (!sk::encode_weight_maps(g_encode, true, codes, scales, K, N, &tm_codes, &tm_scales))
            return SK_ERR_CUDA;
        if (sk::launch_nvfp4(mp, xwide, f16, am, tm_codes, tm_scales, p, grid, s, pdl, coop) != cudaSuccess)
            return SK_ERR_CUDA;
    } else {
        if (!sk::encode_weight_maps(g_encode, false, codes, nullptr, K, N, &tm_codes, nullptr))
            return SK_ERR_CUDA;
        if (sk::launch_fp8(mp, xwide, f16, tm_codes, p, grid, s, pdl, coop) != cudaSuccess) return SK_ERR_CUDA;
    }
    return SK_OK;
}

}  // namespace

namespace sk {

__global__ void fill_u32_kernel(unsigned int *p, size_t n, unsigned int v) {
    for (size_t i = size_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x)
        p[i] = v;
}

cudaError_t empty_partials(unsigned char *ws, size_t bytes, cudaStream_t stream) {
    const size_t n = bytes / 4;
    if (n == 0) return cudaSuccess;
    const size_t blocks = (n + 255) / 256;
    fill_u32_kernel<<<unsigned(blocks < 1024 ? blocks : 1024), 256, 0, stream>>>(
        reinterpret_cast<unsigned int *>(ws + WS_PARTIAL_OFFSET), n, PARTIAL_EMPTY);
    return cudaGetLastError();
}

// Measured on GB300 (cold L2, graphs of back-to-back launches): for M >= 2 the
// tensor-core variant is faster on every decode-layer shape (up to 2x at M = 4);
// for M = 1 the SIMT variant wins only when each CTA streams many units (FP8
// gate_up 5120x34816 at 36 units per CTA, NVFP4 lm_head at 156), because its
// per-unit arithmetic is lighter while its fix-up and start-up are not.
int take_inject_stall() { return g_inject_stall.exchange(0); }

bool encode_weight_maps(PFN_cuTensorMapEncodeTiled_v12000 enc, bool nvfp4, const void *codes,
                        const void *scales, int K, int N, CUtensorMap *tm_codes, CUtensorMap *tm_scales) {
    // Every map views its bytes as u32 words, reads out of bounds as zero and
    // has boxes of one unit's tile (the tile layouts beside Traits, kernel.cuh).
    auto enc3 = [&](CUtensorMap *m, const void *ptr, const cuuint64_t (&dims)[3], const cuuint64_t (&strides)[2],
                    const cuuint32_t (&box)[3]) {
        const cuuint32_t estr[3] = {1, 1, 1};
        return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    };
    const uint64_t rows = uint64_t(N), row_bytes = nvfp4 ? uint64_t(K) / 2 : uint64_t(K);
    if (!nvfp4) {
        // codes {word in a 128-byte segment, row, segment}: box [8 segments][16 rows][128 B]
        return enc3(tm_codes, codes, {32, rows, row_bytes / 128}, {row_bytes, 128},
                    {32, uint32_t(RG), uint32_t(Traits<FP8>::SEGS)});
    }
    // codes {word in a 128-byte segment, segment, row}: box [16 rows][4 segments][128 B]
    if (!enc3(tm_codes, codes, {32, row_bytes / 128, rows}, {128, row_bytes},
              {32, uint32_t(Traits<NVFP4>::SEGS), uint32_t(RG)}))
        return false;
    // scales {word, row}: box [16 rows][64 B], 64-byte swizzle.  L2 promotion
    // to 64 bytes, the box row itself: promoted to 256 bytes, each row fetch
    // also brought in the next three chunks' scales, which the weight stream
    // (evict-first) pushed out of L2 before the units that need them ran, so
    // scale bytes came from DRAM up to four times (ncu on the lm_head at M = 8:
    // DRAM reads 1.145 x the weight bytes; measured with 64-byte promotion:
    // the lm_head 12 % faster, the decode stacks 1.4-1.8 %).
    const uint64_t srow = uint64_t(K) / 16;
    const cuuint64_t dims[2] = {srow / 4, rows};
    const cuuint64_t strides[1] = {srow};
    const cuuint32_t box[2] = {uint32_t(Traits<NVFP4>::SCALE_BOX_X), uint32_t(RG)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(tm_scales, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(scales), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_64B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_2d_u16(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint32_t box_cols,
                   uint32_t box_rows) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (resolve_encode() != SK_OK) return false;
    }
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int device_sm_count() {
    static int cached[MAX_DEVICES] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return 0;
    if (cached[dev] == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = sms;
    }
    return cached[dev];
}

void note_weights_written(cudaStream_t stream) {
    std::lock_guard<std::mutex> lk(g_wq_mu);
    for (int i = 0; i < g_wq_n; ++i)
        if (g_wq_streams[i] == stream) return;
    if (g_wq_n < MAX_MARKED_STREAMS) g_wq_streams[g_wq_n++] = stream;
    else g_wq_overflow = true;
}

bool take_weights_written(cudaStream_t stream) {
    std::lock_guard<std::mutex> lk(g_wq_mu);
    for (int i = 0; i < g_wq_n; ++i)
        if (g_wq_streams[i] == stream) {
            g_wq_streams[i] = g_wq_streams[--g_wq_n];
            return true;
        }
    return g_wq_overflow;
}

unsigned char *workspace_for(cudaStream_t stream) {
    WsRef r;
    return workspace_ref(stream, &r) ? r.ws : nullptr;
}

bool use_wide_x(const void *x, int M) {
    return M >= 4 && reinterpret_cast<uintptr_t>(x) % 32 == 0;
}

int choose_mp(int M, bool nvfp4, long long U, long long P) {
    const int v = g_variant.load(std::memory_order_relaxed);
    if (M > 1 || v == SK_VARIANT_TENSOR) return 8;
    if (v == SK_VARIANT_SIMT) return 1;
    const long long per_cta = U / (P > 0 ? P : 1);
    return per_cta >= (nvfp4 ? 96 : 24) ? 1 : 8;
}

bool pdl_enabled() { return g_pdl != 0; }

}  // namespace sk

extern "C" {

sk_status sk_init(size_t workspace_bytes) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (resolve_encode() != SK_OK) return SK_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return SK_ERR_CUDA;
    size_t bytes = workspace_bytes ? workspace_bytes : DEFAULT_WORKSPACE;
    if (bytes < sk::WS_PARTIAL_OFFSET) bytes = sk::WS_PARTIAL_OFFSET;
    DeviceState &d = g_dev[dev];
    if (d.ws) {
        if (cudaDeviceSynchronize() != cudaSuccess) return SK_ERR_CUDA;
        cudaFree(d.ws);
        d.ws = nullptr;
        d.bytes = 0;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SK_ERR_CUDA;
    void *p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) return SK_ERR_CUDA;
    if (cudaMemset(p, 0, sk::WS_CTRL_BYTES) != cudaSuccess ||
        sk::empty_partials(static_cast<unsigned char *>(p), bytes - sk::WS_PARTIAL_OFFSET, 0) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(p);
        return SK_ERR_CUDA;
    }
    d.ws = static_cast<unsigned char *>(p);
    d.bytes = bytes;
    d.num_sms = sms;
    return SK_OK;
}

sk_status sk_stream_workspace(void *stream, size_t workspace_bytes) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (resolve_encode() != SK_OK) return SK_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return SK_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    StreamWs *slot = nullptr;
    for (StreamWs &e : g_sws)
        if (e.ws && e.dev == dev && e.stream == s) slot = &e;
    if (slot) {
        // Replace or remove: the stream's work must have finished with it.
        if (cudaStreamSynchronize(s) != cudaSuccess) return SK_ERR_CUDA;
        cudaFree(slot->ws);
        *slot = StreamWs{};
    }
    if (workspace_bytes == 0) return SK_OK;
    for (StreamWs &e : g_sws)
        if (!e.ws) {
            slot = &e;
            break;
        }
    if (!slot) return SK_ERR_INVALID_ARG;   // MAX_STREAM_WS workspaces already
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SK_ERR_CUDA;
    const size_t bytes = workspace_bytes < sk::WS_PARTIAL_OFFSET ? sk::WS_PARTIAL_OFFSET : workspace_bytes;
    void *p = nullptr;
    if (cudaMalloc(&p, bytes) != cudaSuccess) return SK_ERR_CUDA;
    if (cudaMemset(p, 0, sk::WS_CTRL_BYTES) != cudaSuccess ||
        sk::empty_partials(static_cast<unsigned char *>(p), bytes - sk::WS_PARTIAL_OFFSET, 0) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(p);
        return SK_ERR_CUDA;
    }
    g_dev[dev].num_sms = sms;
    *slot = StreamWs{dev, s, static_cast<unsigned char *>(p), bytes};
    return SK_OK;
}

sk_status sk_shutdown(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    int prev = 0;
    cudaGetDevice(&prev);
    sk_status st = SK_OK;
    for (StreamWs &e : g_sws) {
        if (!e.ws) continue;
        if (cudaSetDevice(e.dev) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) st = SK_ERR_CUDA;
        cudaFree(e.ws);
        e = StreamWs{};
    }
    for (int i = 0; i < MAX_DEVICES; ++i) {
        if (!g_dev[i].ws) continue;
        if (cudaSetDevice(i) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) st = SK_ERR_CUDA;
        cudaFree(g_dev[i].ws);
        g_dev[i] = DeviceState{};
    }
    cudaSetDevice(prev);
    return st;
}

sk_status nvfp4_gemm(const void *x, const uint8_t *W_codes, const uint8_t *W_scales, float W_gscale, float *y,
                     int M, int N, int K, void *stream) {
    return run(Kind::NVFP4, x, W_codes, W_scales, W_gscale, y, nullptr, M, N, K, stream);
}

sk_status nvfp4_gemm_f16out(const void *x, const uint8_t *W_codes, const uint8_t *W_scales, float W_gscale,
                            void *y, int M, int N, int K, void *stream) {
    return run(Kind::NVFP4_F16, x, W_codes, W_scales, W_gscale, y, nullptr, M, N, K, stream);
}

sk_status fp8_gemm(const void *x, const uint8_t *W_codes, const float *W_scales, float *y, int M, int N, int K,
                   void *stream) {
    return run(Kind::FP8, x, W_codes, W_scales, 1.0f, y, nullptr, M, N, K, stream);
}

sk_status fp8_gemm_f16out(const void *x, const uint8_t *W_codes, const float *W_scales, void *y, int M, int N,
                          int K, void *stream) {
    return run(Kind::FP8_F16, x, W_codes, W_scales, 1.0f, y, nullptr, M, N, K, stream);
}

sk_status lm_head_argmax(const void *x, const uint8_t *W_codes, const uint8_t *W_scales, float W_gscale,
                         float *logits, int32_t *argmax, int M, int N, int K, void *stream) {
    return run(Kind::LMHEAD, x, W_codes, W_scales, W_gscale, logits, argmax, M, N, K, stream);
}

sk_status lm_head_verify(const void *x, const uint8_t *W_codes, const uint8_t *W_scales, float W_gscale,
                         float *logits, int32_t *argmax, const int32_t *draft, int32_t *accept, int M, int N,
                         int K, void *stream) {
    if (!accept) return SK_ERR_INVALID_ARG;
    return run(Kind::LMHEAD, x, W_codes, W_scales, W_gscale, logits, argmax, M, N, K, stream, draft, accept);
}

const char *sk_status_string(sk_status status) {
    switch (status) {
        case SK_OK: return "SK_OK";
        case SK_ERR_INVALID_ARG: return "SK_ERR_INVALID_ARG: invalid argument";
        case SK_ERR_UNSUPPORTED_SHAPE: return "SK_ERR_UNSUPPORTED_SHAPE: unsupported shape";
        case SK_ERR_MISALIGNED: return "SK_ERR_MISALIGNED: misaligned pointer";
        case SK_ERR_NOT_INITIALIZED: return "SK_ERR_NOT_INITIALIZED: sk_init() not called on this device";
        case SK_ERR_CUDA: return "SK_ERR_CUDA: CUDA error";
        case SK_ERR_TIMEOUT: return "SK_ERR_TIMEOUT: a bounded in-kernel wait timed out";
        case SK_ERR_WORKSPACE: return "SK_ERR_WORKSPACE: workspace too small";
    }
    return "unknown sk_status";
}

sk_status sk_last_device_error(void *stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return SK_ERR_CUDA;
    WsRef wr;
    if (!workspace_ref(s, &wr)) return SK_ERR_NOT_INITIALIZED;
    unsigned int err = 0;
    unsigned char *word = wr.ws + offsetof(sk::Ctrl, err);
    if (cudaMemcpy(&err, word, sizeof(err), cudaMemcpyDeviceToHost) != cudaSuccess) return SK_ERR_CUDA;
    if (err) {
        if (cudaMemset(word, 0, sizeof(err)) != cudaSuccess) return SK_ERR_CUDA;
        return SK_ERR_TIMEOUT;
    }
    return SK_OK;
}

int sk_set_variant(int variant) {
    if (variant != SK_VARIANT_AUTO && variant != SK_VARIANT_TENSOR && variant != SK_VARIANT_SIMT) return -1;
    return g_variant.exchange(variant);
}

int sk_set_pdl(int enable) {
    int prev = g_pdl;
    g_pdl = enable ? 1 : 0;
    return prev;
}

void sk_inject_wait_timeout(int enable) { g_inject_stall.store(enable ? 1 : 0); }

int sk_version(void) { return 100; }

}  // extern "C"
