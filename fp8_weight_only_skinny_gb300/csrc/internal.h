// internal.h -- declarations shared by the host translation units of libskinny.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace sk {

struct Params;

// Launch one kernel of the given format.  mp: token slots of the variant
// (1 = single-token SIMT variant; 8 = tensor-core variant); pdl: programmatic
// dependent launch; coop: cooperative launch (the whole grid co-resident).
// xwide: 32-byte activation loads in the tensor-core variant (use_wide_x).
cudaError_t launch_nvfp4(int mp, bool xwide, bool f16out, bool argmax, const CUtensorMap &tm_codes,
                         const CUtensorMap &tm_scales, const Params &p, int grid,
                         cudaStream_t stream, bool pdl, bool coop);
cudaError_t launch_fp8(int mp, bool xwide, bool f16out, const CUtensorMap &tm_codes, const Params &p, int grid,
                       cudaStream_t stream, bool pdl, bool coop);

// The TMA maps of a linear call's weights (K, N as in the call; K a multiple
// of 256 for NVFP4, of 128 for FP8): NVFP4 codes and scales, or FP8 codes
// (tm_scales unused), with the tile layouts and swizzles the kernel reads.
// `enc` is the driver's cuTensorMapEncodeTiled; false if it rejects a map.
bool encode_weight_maps(PFN_cuTensorMapEncodeTiled_v12000 enc, bool nvfp4, const void *codes,
                        const void *scales, int K, int N, CUtensorMap *tm_codes, CUtensorMap *tm_scales);

// 2-D TMA map over a row-major matrix of 16-bit elements [rows][cols]
// (row stride cols * 2 bytes), box {box_cols, box_rows}, out-of-bounds reads
// zero-filled.  Resolves the driver's encoder on first use; false on failure.
bool encode_2d_u16(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t rows, uint32_t box_cols,
                   uint32_t box_rows);

// SM count of the current device (cached per device; 0 on failure).
int device_sm_count();

// Mark the first `bytes` of the split-K partial slots of workspace `ws` empty
// (every slot must be empty before a launch uses the workspace), on `stream`.
cudaError_t empty_partials(unsigned char *ws, size_t bytes, cudaStream_t stream);

// Bytes of workspace-resident partial sums one unit writes (16 rows x mp tokens).
inline size_t unit_partial_bytes(int mp) { return size_t(16) * mp * 4; }

// The failure-injection request of sk_inject_wait_timeout(): returns 1 once
// (and clears it) if the next kernel launch should issue no weight copies.
int take_inject_stall();

// The quantizers write weights.  A linear kernel reads its weights before
// griddepcontrol.wait (its producer streams them while the previous kernel on
// the stream finishes), so the first linear launch on a stream after a
// quantizer launch goes without programmatic dependent launch.  The
// quantizers mark their stream; every linear launch takes (clears) the mark
// and learns whether it was set.
void note_weights_written(cudaStream_t stream);
bool take_weights_written(cudaStream_t stream);

// The workspace a call on `stream` uses on the current device: the stream's
// own (sk_stream_workspace), else the device's (sk_init); null if neither.
unsigned char *workspace_for(cudaStream_t stream);

// Whether the tensor-core variant loads the activations 32 bytes per lane
// and instruction (kernel.cuh, load_x) instead of 16: for M >= 4 and x
// 32-byte aligned.  Half the load instructions and line look-ups before the
// first MMA of each k-chunk; measured on the decode layers (cold L2): 0.25-0.5
// us faster per launch at M = 8 on the small shapes (decode stack 1.4 %), a
// little faster at M = 4, neutral at M = 2, and the same code as before at M
// = 1.  The values loaded, and so the results, do not change.
bool use_wide_x(const void *x, int M);

// Whether launches may use programmatic dependent launch (sk_set_pdl).
bool pdl_enabled();

// Token slots of the kernel variant for an M-token call of U units on a grid
// of P CTAs: 1 (SIMT) or 8 (tensor-core), by the process-wide variant setting.
int choose_mp(int M, bool nvfp4, long long U, long long P);

}  // namespace sk
