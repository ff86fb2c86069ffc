// kernel.cuh -- the skinny weight-only linear kernel for sm_103a.
//
// One persistent CTA per SM streams compressed weight tiles HBM -> shared
// memory with 2-D TMA into an mbarrier ring, and two consumer groups of four
// warps decode them in registers and multiply-accumulate in FP32:
//
//   * MP = 1 ("SIMT" variant, one token): E2M1 / E4M3 pairs -> f16x2 with
//     cvt.rn.f16x2.*, exact FP16 products accumulated in FP32 with the
//     mixed-precision FMA, the 16-element (NVFP4) or 128x128 (FP8) block scale
//     applied once per block sum.  The template also compiles for MP = 2 and
//     4, but the library instantiates MP = 1 only.
//   * MP = 8 ("MMA" variant, M = 1..8 tokens; the 8-row speculative-verify
//     round fills it): swap-AB mma.sync.m16n8k16 with the 16 weight rows as the
//     16-wide operand and the (zero-padded) 8 tokens as the 8-wide one.  For NVFP4 each decoded pair
//     is multiplied by its E4M3 block scale in FP16 first, which is exact
//     (E2M1 has 2 and E4M3 4 significant bits, and their product stays in the
//     FP16 normal range), so the MMA sees exact weights and accumulates in
//     FP32.  For FP8 the per-block scale multiplies the FP32 accumulators.
//
// This is the decode-time linear layer of the pages' system, where weights are
// read compressed from HBM and each small piece becomes FP16 register
// operands (page "NVFP4 在 Volta 上！", section "我实际构建了什么"), and the
// 8-row tensor-core tile carries the k=7 verify round (same page, the
// paragraph after the kernel table).  The Volta design itself (HMMA.884, the
// SIMT kernel) is not reproduced: the ring, TMA and the block-scale folding are
// this library's.
//
// Work decomposition ("units").  A unit is RG = 16 weight rows x KC = 1024 k.
// Units are numbered chunk-major, u = c * G + g (G row groups, C k-chunks),
// and CTA b takes the contiguous range [b*U/P, (b+1)*U/P), so every CTA
// streams the same number of bytes (+-1 unit) whatever the shape.  Each unit
// yields a 16 x MP partial sum; when C > 1 it goes to a slot of its own in
// the workspace, and the row group's owner CTA waits for its C slots to fill,
// sums them in ascending chunk order and writes y.  The sum order is fixed:
// results are bitwise reproducible.
#pragma once
#include <cuda.h>
#include <cstdint>
#include <cuda_fp16.h>
#include "ptx.cuh"

namespace sk {

enum Fmt : int { NVFP4 = 0, FP8 = 1 };

constexpr int RG = 16;            // weight rows per unit
constexpr int KC = 1024;          // k per unit
constexpr int NGROUPS = 2;        // consumer groups per CTA
constexpr int GROUP_THREADS = 128;
constexpr int CTA_THREADS = NGROUPS * GROUP_THREADS + 32;   // + one producer warp
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;            // bounded waits: ~1 s
// Copies outstanding per CTA during the first pass over the ring: two for
// short ranges (up to START_SHORT units per CTA), three otherwise.
constexpr int START_INFLIGHT = 3;
constexpr int START_INFLIGHT_SHORT = 2;
constexpr int START_SHORT = 12;
// An empty split-K partial slot: a signalling-NaN bit pattern, which FP32
// arithmetic never produces (its NaN results are the canonical quiet NaN), so
// a slot holding anything else holds a partial sum.  Every slot of a workspace
// is empty between launches: the workspace is created filled with it, and an
// owner empties each slot it has summed.
constexpr unsigned int PARTIAL_EMPTY = 0x7FBADBADu;
// flags: [0] abort
constexpr int FLAG_BYTES = 64;

// Workspace layout (bytes): control block, then the split-K partial slots.
constexpr size_t WS_CTRL_BYTES = 4096;
constexpr size_t WS_PARTIAL_OFFSET = WS_CTRL_BYTES;

struct Ctrl {
    unsigned long long argmax_key[8];   // per token: (ordered logit << 32) | ~n
    unsigned int done;                  // CTAs finished (argmax epilogue)
    unsigned int err;                   // device error word (bit 0: a wait timed out)
    unsigned int qamax;                 // quantizer: max |w| over the tensor (float bits)
};

enum : unsigned int { ERR_TIMEOUT = 1u };

// Shared-memory tiles of one unit (16 rows x 1024 k), as TMA writes them.
// The copies use the hardware swizzle, so that a consumer load, which takes
// the same 16 bytes of eight rows at once, is spread over all 32 banks.  In
// 128-byte mode the 16-byte chunk j of the tile's 128-byte line L is stored
// as chunk j ^ (L mod 8); in 64-byte mode chunk j of 64-byte row r is stored
// as chunk j ^ ((r >> 1) mod 4).
//   NVFP4 codes:  [16 rows][4 segments of 128 B], 128-byte mode, L = 4 row + segment;
//   NVFP4 scales: [16 rows][64 B], 64-byte mode;
//   FP8 codes:    [8 segments][16 rows][128 B], 128-byte mode, L = 16 segment + row
//                 (segment-major, so that the rows read together differ in L mod 8).
// Measured against plain row-major tiles, whose loads conflicted 2- to 4-way:
// NVFP4 gate_up and down 0.5 us faster per launch at M = 8, the decode stack
// 2 % faster at M = 8 and 1 % at M = 1.
template <int FMT> struct Traits;
template <> struct Traits<NVFP4> {
    static constexpr int ROW_BYTES = KC / 2;           // codes of one row in a unit
    static constexpr int SEGS = ROW_BYTES / 128;       // 128-byte segments per row: 4
    static constexpr int CODE_TILE = RG * ROW_BYTES;   // 8192
    static constexpr int SCALE_ROW = KC / 16;          // 64 E4M3 scales per row
    static constexpr int SCALE_TILE = RG * SCALE_ROW;  // 1024
    static constexpr int STAGE_BYTES = CODE_TILE + SCALE_TILE;
    static constexpr int STAGES = 8;
    static constexpr int SCALE_BOX_X = SCALE_ROW / 4;  // tensor map element = u32
    static constexpr int L2_AHEAD = 0;
};
template <> struct Traits<FP8> {
    static constexpr int ROW_BYTES = KC;
    static constexpr int SEGS = ROW_BYTES / 128;       // 8
    static constexpr int CODE_TILE = RG * ROW_BYTES;   // 16384
    static constexpr int SCALE_TILE = 0;
    static constexpr int STAGE_BYTES = CODE_TILE;
    static constexpr int STAGES = 6;
    static constexpr int SCALE_BOX_X = 0;
    // Past the first ring pass the producer keeps this many units prefetched
    // into L2 ahead of the ring: six 16 KB stages are all that fit twice per
    // SM, and two more units in flight made every FP8 layer 2-5 % faster
    // (NVFP4, with eight stages, measured slower with any prefetch front).
    static constexpr int L2_AHEAD = 2;
};

// Consecutive uses of a ring stage must go to the same consumer group: stage
// s then always serves units i = s (mod STAGES) of group s % NGROUPS, which that
// group consumes in order, so a waiter can never see a parity left over from
// a stage use two phases back.
static_assert(Traits<NVFP4>::STAGES % NGROUPS == 0, "ring stages must be a multiple of NGROUPS");
static_assert(Traits<FP8>::STAGES % NGROUPS == 0, "ring stages must be a multiple of NGROUPS");
static_assert(START_INFLIGHT >= 1 && START_INFLIGHT <= Traits<FP8>::STAGES &&
                  START_INFLIGHT <= Traits<NVFP4>::STAGES && START_INFLIGHT_SHORT >= 1 &&
                  START_INFLIGHT_SHORT <= START_INFLIGHT,
              "start-up pacing must fit the ring");

struct Params {
    const __half *x;            // [M][K]
    const float *fp8_scales;    // FP8: [ceil(N/128)][KB]
    float gscale;               // NVFP4 tensor scale (1 for FP8)
    void *y;                    // [M][N] f32 or f16; may be null with ARGMAX
    int32_t *argmax;            // [M] (ARGMAX only)
    const int32_t *draft;       // [M - 1] drafted tokens, or null (ARGMAX only)
    int32_t *accept;            // [2] accepted drafts, bonus token; with draft (ARGMAX only)
    unsigned char *ws;          // workspace base
    int M, N, K;
    int G, C, KB;               // row groups, k-chunks, FP8 scale row stride
    long long U;                // units = G * C
    int stall;                  // failure injection: the producer issues no copies
};

// Floats of a group's per-unit reduction buffer: MMA = 4 warps x (16 rows x 8
// tokens), SIMT = 16 rows x MP.
template <int MP>
__host__ __device__ constexpr int red_floats() { return MP == 8 ? 4 * 128 : RG * MP; }

template <int FMT, int MP>
__host__ __device__ constexpr size_t smem_bytes() {
    return 1024 + size_t(Traits<FMT>::STAGES) * Traits<FMT>::STAGE_BYTES + 16 * Traits<FMT>::STAGES +
           NGROUPS * red_floats<MP>() * 4 + FLAG_BYTES + NGROUPS * GROUP_THREADS * 8;
}

// Bounded mbarrier wait.  Gives up when the CTA's abort flag is set or after
// WAIT_LIMIT_NS; on a timeout it raises the abort flag and the device error
// word.  Returns false when it gave up.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort,
                                             unsigned int *err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                *abort = 1;
                atomicOr(err, ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Advance unit (c, g) by `by` units in chunk-major order (u = c * G + g),
// without a division per unit (the loop runs more than once only when G < by).
__device__ __forceinline__ void step_unit(int &c, int &g, int by, int G) {
    g += by;
    while (g >= G) {
        g -= G;
        c += 1;
    }
}

// Order-preserving map of an FP32 value to u32 (larger value -> larger key).
__device__ __forceinline__ unsigned int ordered_bits(float v) {
    unsigned int u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Warp reduction of NV values per lane.  Afterwards lane l holds the full sum
// of value index reduce_index<NV>(l) in v[0].
template <int NV>
__device__ __forceinline__ void warp_reduce_split(float (&v)[NV], int lane) {
    int n = NV;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        if (n > 1) {
            const int h = n / 2;
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int e = 0; e < NV / 2; ++e) {
                if (e < h) {
                    float send = upper ? v[e] : v[e + h];
                    float keep = upper ? v[e + h] : v[e];
                    v[e] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            n = h;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
    }
}

template <int NV>
__device__ __forceinline__ int reduce_index(int lane) {
    int idx = 0, n = NV;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        if (n > 1) {
            const int h = n / 2;
            if (lane & o) idx += h;
            n = h;
        }
    }
    return idx;
}

// ----------------------------------------------------------------------------
// Activation registers for one k-chunk.
//   MMA (MP == 8): lane (j = lane/4, q = lane%4) of warp w holds, for each of
//     the 32 mma k-steps of its k slice, the B fragment of token j.
//   SIMT: lane l holds 32 activations (16 f16x2 words) per token.
// Tokens >= M and k >= K read as zero.
template <int FMT, int MP>
struct XRegs {
    static constexpr int PIECES = (MP == 8) ? (FMT == NVFP4 ? 2 : 4) : 1;
    static constexpr int WORDS = (MP == 8) ? (FMT == NVFP4 ? 16 : 8) : 16;
    static constexpr int TOK = (MP == 8) ? 1 : MP;
    uint32_t w[TOK][PIECES][WORDS];
};

template <int FMT, int MP, bool XWIDE>
__device__ __forceinline__ void load_x(XRegs<FMT, MP> &xr, const Params &p, int c, int warp_in_group,
                                       int lane) {
    const int kbase = c * KC;
    if constexpr (MP == 8) {
        const int j = lane >> 2, q = lane & 3;
#pragma unroll
        for (int t = 0; t < XRegs<FMT, MP>::PIECES; ++t) {
            const int k0 = (FMT == NVFP4) ? kbase + 256 * warp_in_group + 128 * t + 32 * q
                                          : kbase + 256 * warp_in_group + 64 * t + 16 * q;
            if constexpr (XWIDE) {   // x 32-byte aligned; k0 a multiple of 16
#pragma unroll
                for (int v = 0; v < XRegs<FMT, MP>::WORDS / 8; ++v) {
                    const int k = k0 + 16 * v;
                    uint32_t val[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                    if (j < p.M && k < p.K) ld_global_v8(p.x + size_t(j) * p.K + k, val);
#pragma unroll
                    for (int e = 0; e < 8; ++e) xr.w[0][t][8 * v + e] = val[e];
                }
            } else {
#pragma unroll
                for (int v = 0; v < XRegs<FMT, MP>::WORDS / 4; ++v) {
                    const int k = k0 + 8 * v;
                    uint4 val = make_uint4(0, 0, 0, 0);
                    if (j < p.M && k < p.K) val = ld_global_v4(p.x + size_t(j) * p.K + k);
                    xr.w[0][t][4 * v + 0] = val.x;
                    xr.w[0][t][4 * v + 1] = val.y;
                    xr.w[0][t][4 * v + 2] = val.z;
                    xr.w[0][t][4 * v + 3] = val.w;
                }
            }
        }
    } else {
#pragma unroll
        for (int m = 0; m < MP; ++m) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                // NVFP4: k = 32*lane + 8v;  FP8: pieces [16*lane, +16) and [512 + 16*lane, +16)
                const int k = (FMT == NVFP4) ? kbase + 32 * lane + 8 * v
                                             : kbase + (v >> 1) * 512 + 16 * lane + 8 * (v & 1);
                uint4 val = make_uint4(0, 0, 0, 0);
                if (m < p.M && k < p.K) val = ld_global_v4(p.x + size_t(m) * p.K + k);
                xr.w[m][0][4 * v + 0] = val.x;
                xr.w[m][0][4 * v + 1] = val.y;
                xr.w[m][0][4 * v + 2] = val.z;
                xr.w[m][0][4 * v + 3] = val.w;
            }
        }
    }
}

// FP8 tensor-core variant: the tile row that MMA fragment row f (0..15) holds
// (the reduction buffer puts each D row back at its tile row).  The 16-byte
// code loads are served a quarter-warp -- fragment rows 2i and 2i + 1 -- at a
// time; this order gives those two rows tile rows whose swizzles (tile row
// mod 8) differ in bit 2, so the four consecutive chunks each group of four
// lanes reads fall in distinct banks, while the activations of one token's
// four lanes stay in one 128-byte line.  Measured against k pieces taken in
// pairs (also conflict-free, two activation lines per token): the per-rank
// FP8 layers 0.2-0.3 us faster per launch at M = 8, the rest unchanged.
// Rows f and f + 8 stay 8 apart.
__device__ __forceinline__ int fp8_tile_row(int f) { return (f & 8) | ((f & 1) << 2) | ((f >> 1) & 3); }

// ----------------------------------------------------------------------------
// MMA path, one unit, one warp: D (16 rows x 8 tokens) of this warp's k slice.
template <int FMT>
__device__ __forceinline__ void unit_mma(float (&d)[4], const XRegs<FMT, 8> &xr, uint32_t stage,
                                         const Params &p, int g, int c, int w, int lane) {
    const int r = lane >> 2, q = lane & 3;
    if constexpr (FMT == NVFP4) {
        const uint32_t codes = stage, scales = stage + Traits<NVFP4>::CODE_TILE;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        // Per t, lane (r, q) takes code bytes 128w + 64t + 16q of rows r and
        // r + 8 (segment w, chunk 4t + q; the same swizzle for both rows) and
        // scale bytes 16w + 8t + 2q, 2q + 1 (chunk w of the scale row).
        const uint32_t cx = uint32_t((4 * r + w) & 7);
        const uint32_t sx = uint32_t(((r >> 1) & 3) ^ w) << 4;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const uint32_t off = 128 * w + ((uint32_t(4 * t + q) ^ cx) << 4);
            const uint4 A = ld_shared_v4(codes + r * 512 + off);
            const uint4 B = ld_shared_v4(codes + (r + 8) * 512 + off);
            const uint32_t soff = sx + 8 * t + 2 * q;
            const uint32_t sa = e4m3x2_h_to_f16x2(ld_shared_u16(scales + r * 64 + soff));
            const uint32_t sb = e4m3x2_h_to_f16x2(ld_shared_u16(scales + (r + 8) * 64 + soff));
            const uint32_t sa0 = bcast_lo(sa), sa1 = bcast_hi(sa);
            const uint32_t sb0 = bcast_lo(sb), sb1 = bcast_hi(sb);
            const uint32_t Aw[4] = {A.x, A.y, A.z, A.w};
            const uint32_t Bw[4] = {B.x, B.y, B.z, B.w};
#pragma unroll
            for (int wd = 0; wd < 4; ++wd) {
                // word wd = bytes 4wd..4wd+3 = k steps ii = 2wd (bytes 0,1) and 2wd+1 (bytes 2,3)
                uint32_t da[4], db[4];
                e2m1x8_to_f16x2x4(Aw[wd], da);
                e2m1x8_to_f16x2x4(Bw[wd], db);
                const uint32_t s_a = wd < 2 ? sa0 : sa1;
                const uint32_t s_b = wd < 2 ? sb0 : sb1;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int ii = 2 * wd + h;
                    mma_16816(acc[ii & 1], hmul2(da[2 * h], s_a), hmul2(db[2 * h], s_b),
                              hmul2(da[2 * h + 1], s_a), hmul2(db[2 * h + 1], s_b),
                              xr.w[0][t][2 * ii], xr.w[0][t][2 * ii + 1]);
                }
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) d[e] = acc[0][e] + acc[1][e];
    } else {
        const uint32_t codes = stage;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        // Piece t of lane q: code bytes 64t + 16q of the warp's 256-byte slice
        // (segment 2w + t / 2, chunk 4 (t mod 2) + q) of tile rows sr and
        // sr + 8, sr = fp8_tile_row(r).
        const uint32_t sr = uint32_t(fp8_tile_row(r));
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const uint32_t off =
                (2 * w + (t >> 1)) * 2048 + sr * 128 + ((uint32_t(4 * (t & 1) + q) ^ (sr & 7u)) << 4);
            const uint4 A = ld_shared_v4(codes + off);
            const uint4 B = ld_shared_v4(codes + off + 8 * 128);
            const uint32_t Aw[4] = {A.x, A.y, A.z, A.w};
            const uint32_t Bw[4] = {B.x, B.y, B.z, B.w};
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) {
                uint32_t a0, a2, a1, a3;
                e4m3x4_to_f16x2x2(Aw[ii], a0, a2);
                e4m3x4_to_f16x2x2(Bw[ii], a1, a3);
                mma_16816(acc[t >> 1], a0, a1, a2, a3, xr.w[0][t][2 * ii], xr.w[0][t][2 * ii + 1]);
            }
        }
        const int rb = g >> 3;                  // 128-row block of this row group
        const int kb0 = c * (KC / 128) + 2 * w; // 128-k blocks of this warp's slice
        const float *srow = p.fp8_scales + size_t(rb) * p.KB;
        const float s0 = kb0 < p.KB ? __ldg(srow + kb0) : 0.f;
        const float s1 = kb0 + 1 < p.KB ? __ldg(srow + kb0 + 1) : 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) d[e] = acc[0][e] * s0 + acc[1][e] * s1;
    }
}

// SIMT path, one unit, one warp: out[i][m] for rows 4w+i of the unit.
template <int FMT, int MP>
__device__ __forceinline__ void unit_simt(float (&out)[4 * MP], const XRegs<FMT, MP> &xr,
                                          uint32_t stage, const Params &p, int g, int c, int w,
                                          int lane) {
    if constexpr (FMT == NVFP4) {
        const uint32_t codes = stage, scales = stage + Traits<NVFP4>::CODE_TILE;
        // Lane l takes code bytes 16l.. of each row (segment l / 8, chunk
        // l mod 8) and scale bytes 2l, 2l + 1 (chunk l / 8): the swizzle of
        // row 4w + i depends only on i mod 2 (codes) and i / 2 (scales).
        const uint32_t seg = uint32_t(lane >> 3), ch = uint32_t(lane & 7);
        const uint32_t co = seg * 128 + ((ch ^ seg) << 4);                  // rows 4w, 4w + 2
        const uint32_t so = ((seg ^ uint32_t((2 * w) & 3)) << 4) + 2 * ch;  // rows 4w, 4w + 1
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = 4 * w + i;
            const uint4 A = ld_shared_v4(codes + row * 512 + (co ^ ((i & 1) << 6)));
            const float2 sf =
                f16x2_to_f32x2(e4m3x2_h_to_f16x2(ld_shared_u16(scales + row * 64 + (so ^ ((i >> 1) << 4)))));
            const uint32_t Aw[4] = {A.x, A.y, A.z, A.w};
            float b0[MP], b1[MP];
#pragma unroll
            for (int m = 0; m < MP; ++m) { b0[m] = 0.f; b1[m] = 0.f; }
#pragma unroll
            for (int wd = 0; wd < 4; ++wd) {
                uint32_t dw[4];
                e2m1x8_to_f16x2x4(Aw[wd], dw);
#pragma unroll
                for (int bb = 0; bb < 4; ++bb) {
                    const int j = 4 * wd + bb;
#pragma unroll
                    for (int m = 0; m < MP; ++m) {
                        if (j < 8) b0[m] = fma2_f16_f32(dw[bb], xr.w[m][0][j], b0[m]);
                        else       b1[m] = fma2_f16_f32(dw[bb], xr.w[m][0][j], b1[m]);
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < MP; ++m) out[i * MP + m] = b0[m] * sf.x + b1[m] * sf.y;
        }
    } else {
        const uint32_t codes = stage;
        const int rb = g >> 3;
        const int kb0 = c * (KC / 128) + (lane >> 3);
        const float *srow = p.fp8_scales + size_t(rb) * p.KB;
        const float s0 = kb0 < p.KB ? __ldg(srow + kb0) : 0.f;
        const float s1 = kb0 + 4 < p.KB ? __ldg(srow + kb0 + 4) : 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int row = 4 * w + i;
            // code bytes 16 lane.. and 512 + 16 lane.. of the row: segments
            // lane / 8 and 4 + lane / 8, chunk lane mod 8, swizzled by the row
            const uint32_t o = (lane >> 3) * 2048 + row * 128 + (uint32_t((lane & 7) ^ (row & 7)) << 4);
            const uint4 A0 = ld_shared_v4(codes + o);
            const uint4 A1 = ld_shared_v4(codes + o + 4 * 2048);
            const uint32_t Aw[8] = {A0.x, A0.y, A0.z, A0.w, A1.x, A1.y, A1.z, A1.w};
            float p0[MP], p1[MP];
#pragma unroll
            for (int m = 0; m < MP; ++m) { p0[m] = 0.f; p1[m] = 0.f; }
#pragma unroll
            for (int wd = 0; wd < 8; ++wd) {
                uint32_t wlo, whi;
                e4m3x4_to_f16x2x2(Aw[wd], wlo, whi);
#pragma unroll
                for (int m = 0; m < MP; ++m) {
                    if (wd < 4) {
                        p0[m] = fma2_f16_f32(wlo, xr.w[m][0][2 * wd], p0[m]);
                        p0[m] = fma2_f16_f32(whi, xr.w[m][0][2 * wd + 1], p0[m]);
                    } else {
                        p1[m] = fma2_f16_f32(wlo, xr.w[m][0][2 * wd], p1[m]);
                        p1[m] = fma2_f16_f32(whi, xr.w[m][0][2 * wd + 1], p1[m]);
                    }
                }
            }
#pragma unroll
            for (int m = 0; m < MP; ++m) out[i * MP + m] = p0[m] * s0 + p1[m] * s1;
        }
    }
}

// Write output o (row o / MP, token o % MP) of row group g; track the best
// argmax key of this thread's token.
template <int FMT, int MP, bool F16OUT, bool ARGMAX>
__device__ __forceinline__ void finalize(const Params &p, int g, int o, float v, unsigned long long &best) {
    const int row = o / MP, m = o % MP;
    const int n = g * RG + row;
    const float val = (FMT == NVFP4) ? v * p.gscale : v;
    if (n < p.N && m < p.M) {
        if (p.y) {
            if constexpr (F16OUT) reinterpret_cast<__half *>(p.y)[size_t(m) * p.N + n] = __float2half_rn(val);
            else reinterpret_cast<float *>(p.y)[size_t(m) * p.N + n] = val;
        }
        if constexpr (ARGMAX) {
            const unsigned long long key =
                (static_cast<unsigned long long>(ordered_bits(val)) << 32) | static_cast<unsigned int>(~n);
            best = key > best ? key : best;
        }
    }
}

// ----------------------------------------------------------------------------
// CTA roles: warps 0 .. 4*NGROUPS-1 are consumers (unit i goes to group
// i % NGROUPS, whose four warps split its k-chunk or its rows); the last warp
// is the producer, one lane of which issues the TMA loads.  Per unit a group
// reduces its warps' partial sums through shared memory and either writes y
// (one k-chunk) or stores the unit's split-K partial into its slot.  The sums
// of the C partials of each owned row group, in ascending chunk order, run
// once per CTA after its whole range, by all consumer threads in parallel: no
// global round trip sits on the per-unit path.  XWIDE (tensor-core variant,
// x 32-byte aligned): activations loaded 32 bytes per lane and instruction.
template <int FMT, int MP, bool F16OUT, bool ARGMAX, bool XWIDE>
__global__ void __launch_bounds__(CTA_THREADS, 2)
skinny_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_scales,
              const Params p) {
    using T = Traits<FMT>;
    constexpr int RED = red_floats<MP>();
    constexpr int NOUT = RG * MP;                 // outputs per unit
    constexpr int CT = NGROUPS * GROUP_THREADS;   // consumer threads

    extern __shared__ unsigned char smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char *sb = smem_raw + (base - raw);
    const uint32_t bar_full = base + T::STAGES * T::STAGE_BYTES;
    const uint32_t bar_empty = bar_full + 8 * T::STAGES;
    float *red = reinterpret_cast<float *>(sb + T::STAGES * T::STAGE_BYTES + 16 * T::STAGES);
    volatile int *flags = reinterpret_cast<volatile int *>(red + NGROUPS * RED);   // [0] abort
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(
        sb + T::STAGES * T::STAGE_BYTES + 16 * T::STAGES + NGROUPS * RED * 4 + FLAG_BYTES);

    Ctrl *ctrl = reinterpret_cast<Ctrl *>(p.ws);
    float *partials = reinterpret_cast<float *>(p.ws + WS_PARTIAL_OFFSET);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long u_lo = (long long)blockIdx.x * p.U / gridDim.x;
    const long long u_hi = (long long)(blockIdx.x + 1) * p.U / gridDim.x;
    const int n_units = int(u_hi - u_lo);
    const int c_lo = int(u_lo / p.G), g_lo = int(u_lo % p.G);   // first unit of the range

    if (threadIdx.x == 0) {
        for (int s = 0; s < T::STAGES; ++s) {
            mbar_init(bar_full + 8 * s, 1);
            mbar_init(bar_empty + 8 * s, 1);
        }
        flags[0] = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // Let the next kernel on the stream start streaming its own weights now;
    // it touches x / y / the workspace only after this grid has completed.
    pdl_launch_dependents();

    if (warp == NGROUPS * 4) {
        // ------------------------------------------------------ producer ---
        if (lane == 0) {
            const uint64_t pol = l2_evict_first_policy();
            int issued = 0;
            int c = c_lo, g = g_lo;                        // unit u_lo + i, stepped without division
            int pc = c_lo, pg = g_lo, pf = 0;              // next unit to prefetch into L2 (pf = its index)
            for (int i = 0; i < (p.stall ? 0 : n_units); ++i, step_unit(c, g, 1, p.G)) {
                const int s = i % T::STAGES;
                if constexpr (T::L2_AHEAD > 0) {
                    if (i >= T::STAGES) {
                        if (pf == 0) {
                            pf = i;
                            step_unit(pc, pg, i, p.G);
                        }
                        for (; pf < n_units && pf < i + T::L2_AHEAD; ++pf, step_unit(pc, pg, 1, p.G))
                            tma_prefetch_l2_3d(&tm_codes, 0, pg * RG, pc * T::SEGS, pol);
                    }
                }
                // Start-up pacing: during the first pass over the ring copy i
                // waits until copy i - START_INFLIGHT has landed.  When every CTA
                // asks for its whole ring at once, HBM serves the burst in no
                // particular order, some CTAs get their first tile microseconds
                // after the others and finish last; pacing the first pass evens
                // the start (measured on the decode layers at M = 8: two copies
                // in flight suit short ranges -- qkv FP8 8.75 -> 8.49 us per
                // launch against three -- while long ranges do better with three
                // -- NVFP4 gate_up 21.95 -> 21.53 us against two; one is slower).
                const int si = n_units <= START_SHORT ? START_INFLIGHT_SHORT : START_INFLIGHT;
                if (i >= si && i < T::STAGES && !wait_bounded(bar_full + 8 * (i - si), 0, flags, &ctrl->err))
                    break;
                if (i >= T::STAGES &&
                    !wait_bounded(bar_empty + 8 * s, ((i / T::STAGES) & 1) ^ 1, flags, &ctrl->err))
                    break;
                const uint32_t dst = base + s * T::STAGE_BYTES;
                mbar_arrive_expect_tx(bar_full + 8 * s, T::STAGE_BYTES);
                if constexpr (FMT == NVFP4) {   // codes {word, segment, row}, scales {word, row}
                    tma_load_3d(dst, &tm_codes, bar_full + 8 * s, 0, c * T::SEGS, g * RG, pol);
                    tma_load_2d(dst + T::CODE_TILE, &tm_scales, bar_full + 8 * s, c * T::SCALE_BOX_X,
                                g * RG, pol);
                } else {                          // codes {word, row, segment}
                    tma_load_3d(dst, &tm_codes, bar_full + 8 * s, 0, g * RG, c * T::SEGS, pol);
                }
                issued = i + 1;
            }
            if (flags[0]) {
                // Aborted: let the copies still in flight land before exiting.
                for (int i = issued - T::STAGES < 0 ? 0 : issued - T::STAGES; i < issued; ++i) {
                    const int s = i % T::STAGES;
                    const uint64_t t0 = globaltimer_ns();
                    while (!mbar_try_wait(bar_full + 8 * s, (i / T::STAGES) & 1) &&
                           globaltimer_ns() - t0 < WAIT_LIMIT_NS) {
                    }
                }
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumers ---
    const int q = warp >> 2, w = warp & 3;
    const int t = threadIdx.x - q * GROUP_THREADS;     // 0..127 within the group
    const int ct = threadIdx.x;                        // 0..CT-1; token of this thread: ct % MP
    const uint32_t bar_id = 1 + q;
    float *gred = red + q * RED;
    unsigned long long best = 0;                       // ARGMAX: best key of token ct % MP

    // Activations of this CTA's first and last k-chunk into L2 while the
    // previous kernel finishes (one 128-byte line per thread).  L2 is the
    // point of coherence, so a line the previous kernel writes afterwards is
    // still read correctly after the wait below; x that is already in L2 (the
    // usual case when the previous kernel produced it) makes this a no-op.
    // Measured on the decode stack, where every layer's x is cold: 2.5 %
    // faster at M = 8.
    {
        constexpr int LINES = KC * 2 / 128;
        if (ct < p.M * LINES && n_units > 0) {
            const int m = ct / LINES, l = ct % LINES;
            const int k = c_lo * KC + l * 64;
            if (k < p.K) prefetch_l2(p.x + size_t(m) * p.K + k);
            const int c_last = int((u_hi - 1) / p.G);
            const int k2 = c_last * KC + l * 64;
            if (c_last != c_lo && k2 < p.K) prefetch_l2(p.x + size_t(m) * p.K + k2);
        }
    }
    pdl_wait_primary();   // x, y and the workspace belong to the previous kernel until here

    XRegs<FMT, MP> xr;
    int cur_c = -1;
    int c = c_lo, g = g_lo;
    step_unit(c, g, q, p.G);                           // unit u_lo + q
    for (int i = q; i < n_units; i += NGROUPS, step_unit(c, g, NGROUPS, p.G)) {
        if (c != cur_c) {
            load_x<FMT, MP, XWIDE>(xr, p, c, w, lane);
            cur_c = c;
        }
        const int s = i % T::STAGES;
        wait_bounded(bar_full + 8 * s, (i / T::STAGES) & 1, flags, &ctrl->err);
        const uint32_t stage = base + s * T::STAGE_BYTES;

        if constexpr (MP == 8) {
            float d[4];
            unit_mma<FMT>(d, xr, stage, p, g, c, w, lane);
            const int r = (FMT == FP8) ? fp8_tile_row(lane >> 2) : lane >> 2, qq = lane & 3;
            *reinterpret_cast<float2 *>(gred + w * 128 + r * 8 + 2 * qq) = make_float2(d[0], d[1]);
            *reinterpret_cast<float2 *>(gred + w * 128 + (r + 8) * 8 + 2 * qq) = make_float2(d[2], d[3]);
        } else {
            float out[4 * MP];
            unit_simt<FMT, MP>(out, xr, stage, p, g, c, w, lane);
            warp_reduce_split<4 * MP>(out, lane);
            constexpr int NV = 4 * MP;
            const int idx = reduce_index<NV>(lane);    // lanes holding a distinct value
            if ((lane & ((32 / NV) - 1)) == 0) gred[(4 * w) * MP + idx] = out[0];
        }
        named_bar_sync(bar_id, GROUP_THREADS);
        // Release the stage only now.  The MMAs / FMAs that consume the shared
        // loads touch registers only, so an arrive placed right after them in
        // program order may be performed before the last loads of the tile
        // have read it, and the producer's next copy into the stage could
        // then overwrite words not yet read.  The reduction-buffer stores
        // depend on every loaded word, and the group barrier orders them (and
        // so the loads) before this arrive.
        if (t == 0) mbar_arrive(bar_empty + 8 * s);

        // output t of this unit: row t / MP, token t % MP
        if (t < NOUT) {
            float v;
            if constexpr (MP == 8) v = gred[t] + gred[128 + t] + gred[256 + t] + gred[384 + t];
            else v = gred[t];
            if (p.C == 1) finalize<FMT, MP, F16OUT, ARGMAX>(p, g, t, v, best);
            else st_relaxed_f32(partials + ((size_t)g * p.C + c) * NOUT + t, v);
        }
        named_bar_sync(bar_id, GROUP_THREADS);   // gred is reused by the next unit
    }

    if (p.C > 1) {
        // Split-K fix-up.  Row group g belongs to CTA g mod P, P owner CTAs
        // (below) with an even share each.  Thread ct takes output o of owned
        // row groups e0, e0 + ES, ... (up to four at a time): it loads their C
        // partial slots (up to eight chunks each; many chunks -- down: 17 --
        // one row group at a time with up to 24 slots in flight), reloads any
        // slot still empty (bounded), sums them in ascending chunk order,
        // writes y and empties the slots again.  No counter, fence or barrier
        // is involved: a partial is usable as soon as its store reaches L2
        // (measured against a release-increment per unit at the end of each
        // CTA's range, counter polls and then the loads: the decode stack 7 %
        // faster at M = 1 and M = 8, every layer 0.5-2 us faster per launch).
        //
        // Owners: the fewest CTAs, but at least the first half of the grid
        // (about one CTA per SM), that each sum their row groups in one round
        // -- cap row groups: 4 * ES, or ES with more than CB chunks, which go
        // one row group per thread at a time -- or, if even the whole grid
        // needs more rounds, every CTA.  The other CTAs leave right after their
        // main loop and the next kernel's CTAs take their slots and start
        // streaming during this tail (measured: qkv / o_proj / down 6 % faster
        // than every CTA owning).  Counting the one-row-group rounds of the
        // many-chunk path (down: 160 owners of 2 row groups instead of 152, of
        // which 16 held 3 and summed in two rounds) made down 0.2-0.3 us faster.
        constexpr int ES = CT / NOUT;
        constexpr int CB = 8;
        const int cap = p.C > CB ? ES : 4 * ES;
        const int PH = (int(gridDim.x) + 1) / 2;
        const int pmin = (p.G + cap - 1) / cap;
        const int P = pmin <= PH ? PH : (pmin <= int(gridDim.x) ? pmin : int(gridDim.x));
        const int n_own =
            (p.G > int(blockIdx.x) && int(blockIdx.x) < P) ? (p.G - 1 - int(blockIdx.x)) / P + 1 : 0;
        const int o = ct % NOUT;
        if (p.C > CB) {
            constexpr int CL = 24;
            for (int e = ct / NOUT; e < n_own; e += ES) {
                const int gq = int(blockIdx.x) + e * P;
                float acc = 0.f;
                for (int c0 = 0; c0 < p.C; c0 += CL) {
                    float *slot = partials + ((size_t)gq * p.C + c0) * NOUT + o;
                    float v[CL];
                    bool miss = false;
#pragma unroll
                    for (int k = 0; k < CL; ++k) v[k] = c0 + k < p.C ? ld_relaxed_f32(slot + k * NOUT) : 0.f;
#pragma unroll
                    for (int k = 0; k < CL; ++k) miss |= __float_as_uint(v[k]) == PARTIAL_EMPTY;
                    if (miss) {
                        const uint64_t t0 = globaltimer_ns();
                        while (miss) {
                            __nanosleep(32);
                            miss = false;
#pragma unroll
                            for (int k = 0; k < CL; ++k)
                                if (__float_as_uint(v[k]) == PARTIAL_EMPTY) v[k] = ld_relaxed_f32(slot + k * NOUT);
#pragma unroll
                            for (int k = 0; k < CL; ++k) miss |= __float_as_uint(v[k]) == PARTIAL_EMPTY;
                            if (miss && globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                                flags[0] = 1;
                                atomicOr(&ctrl->err, ERR_TIMEOUT);
                                break;
                            }
                        }
                    }
#pragma unroll
                    for (int k = 0; k < CL; ++k)
                        if (c0 + k < p.C) {
                            acc += v[k];
                            st_relaxed_f32(slot + k * NOUT, __uint_as_float(PARTIAL_EMPTY));
                        }
                }
                finalize<FMT, MP, F16OUT, ARGMAX>(p, gq, o, acc, best);
            }
        } else
        for (int e = ct / NOUT; e < n_own; e += 4 * ES) {
            int gg[4];
            float acc[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                gg[j] = e + j * ES < n_own ? int(blockIdx.x) + (e + j * ES) * P : -1;
                acc[j] = 0.f;
            }
            for (int c0 = 0; c0 < p.C; c0 += CB) {
                float v[4][CB];
                bool miss = false;
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int k = 0; k < CB; ++k)
                        v[j][k] = (gg[j] >= 0 && c0 + k < p.C)
                                      ? ld_relaxed_f32(partials + ((size_t)gg[j] * p.C + c0 + k) * NOUT + o)
                                      : 0.f;
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int k = 0; k < CB; ++k) miss |= __float_as_uint(v[j][k]) == PARTIAL_EMPTY;
                if (miss) {
                    const uint64_t t0 = globaltimer_ns();
                    while (miss) {
                        __nanosleep(32);
                        miss = false;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int k = 0; k < CB; ++k)
                                if (__float_as_uint(v[j][k]) == PARTIAL_EMPTY)
                                    v[j][k] = ld_relaxed_f32(partials + ((size_t)gg[j] * p.C + c0 + k) * NOUT + o);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int k = 0; k < CB; ++k) miss |= __float_as_uint(v[j][k]) == PARTIAL_EMPTY;
                        if (miss && globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
                            flags[0] = 1;
                            atomicOr(&ctrl->err, ERR_TIMEOUT);
                            break;
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int k = 0; k < CB; ++k)
                        if (gg[j] >= 0 && c0 + k < p.C) {
                            acc[j] += v[j][k];
                            st_relaxed_f32(partials + ((size_t)gg[j] * p.C + c0 + k) * NOUT + o,
                                           __uint_as_float(PARTIAL_EMPTY));
                        }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (gg[j] >= 0) finalize<FMT, MP, F16OUT, ARGMAX>(p, gg[j], o, acc[j], best);
        }
    }

    if constexpr (ARGMAX) {
        // Per-CTA best per token (warp shuffles over the lanes holding the same
        // token, then one value per warp) -> one 64-bit atomicMax per token; the
        // CTA that increments the done counter last (acquire-release, so it
        // sees every CTA's keys) turns the keys into indices and resets them.
        // Measured against a full fence on either side of the increment, a
        // serial scan of the per-thread keys and the last CTA loading one key
        // per round trip: the fused argmax 3 us faster per call, now ~1 us
        // above the plain projection at M = 8.
        unsigned long long b = best;
#pragma unroll
        for (int o = MP; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_xor_sync(0xffffffffu, b, o);
            b = y > b ? y : b;
        }
        if (lane < MP) keys[(ct >> 5) * MP + lane] = b;
        named_bar_sync(15, CT);
        if (ct < MP) {
            unsigned long long k = 0;
#pragma unroll
            for (int w = 0; w < CT / 32; ++w) k = keys[w * MP + ct] > k ? keys[w * MP + ct] : k;
            if (k != 0 && ct < p.M) atomicMax(&ctrl->argmax_key[ct], k);
        }
        named_bar_sync(15, CT);
        if (ct == 0) {
            const unsigned int old = atom_add_acq_rel_u32(&ctrl->done, 1u);
            if (old == gridDim.x - 1) {
                // every load first (one round trip), then the stores
                unsigned long long kk[8];
                int dr[7];
#pragma unroll
                for (int m = 0; m < 8; ++m) kk[m] = m < p.M ? ld_cg_u64(&ctrl->argmax_key[m]) : 0ull;
#pragma unroll
                for (int m = 0; m < 7; ++m) dr[m] = (p.accept && m < p.M - 1) ? p.draft[m] : 0;
                int pick[8];
#pragma unroll
                for (int m = 0; m < 8; ++m) pick[m] = static_cast<int32_t>(~static_cast<unsigned int>(kk[m] & 0xffffffffull));
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    if (m < p.M) {
                        p.argmax[m] = pick[m];
                        ctrl->argmax_key[m] = 0ull;
                    }
                if (p.accept) {
                    // Greedy verification of the speculative round: draft j is
                    // accepted while all earlier ones were and it equals row j's
                    // pick; the target then commits its own pick after them.
                    int a = 0;
                    bool run = true;
#pragma unroll
                    for (int m = 0; m < 7; ++m) {
                        run = run && m < p.M - 1 && dr[m] == pick[m];
                        a += run ? 1 : 0;
                    }
                    int bonus = pick[0];
#pragma unroll
                    for (int m = 1; m < 8; ++m) bonus = a == m ? pick[m] : bonus;
                    p.accept[0] = a;
                    p.accept[1] = bonus;
                }
                ctrl->done = 0u;
            }
        }
    }
}

}  // namespace sk
