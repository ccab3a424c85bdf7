// kda_internal.cuh -- internal declarations shared by libkda's translation
// units: workspace layout, kernel parameter blocks, launchers, small device
// helpers.  Not part of the public ABI (include/kda.h is).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

constexpr int kChunk = 64;     // tokens per chunk (the pages' chunk_size)
constexpr int kSub = 16;       // rows per sub-block of the exponent factors
constexpr int kNumSub = kChunk / kSub;

// ---------------------------------------------------------------------------
// Workspace layout (caller-owned device memory, zero-filled before first use)
//   [0, 256)            WsHeader
//   [256, 256+R)        int32 row_offsets[B+1]  (R = B+1 ints rounded to 256 B)
//   [256+R, ...)        int2 runs[B*T]: {start, end} of run i of row b at
//                       runs[b*T + i]
// ---------------------------------------------------------------------------
struct WsHeader {
  uint32_t status;        // KDA_DEVICE_* bits, sticky until cleared
  uint32_t rows_done;     // run-builder completion counter (returns to 0)
  uint32_t total_runs;    // number of runs over all rows (run-builder output)
  uint32_t total_chunks;  // 64-token chunks over all runs (split path only)
  uint32_t reserved[60];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline size_t ws_row_offsets_bytes(int B) {
  return align_up(sizeof(int32_t) * ((size_t)B + 1), 256);
}
inline size_t ws_bytes(int B, int T, bool has_seg) {
  size_t n = sizeof(WsHeader);
  if (has_seg) n += ws_row_offsets_bytes(B) + sizeof(int2) * (size_t)B * T;
  return n;
}

// The split path with segment ids appends, after ws_bytes(B, T, true):
//   int32 run_chunk_base[B*T] (first chunk of run i of row b, within the row),
//   int32 chunk_row_offsets[B+1] (prefix of chunk counts over rows),
//   int2 chunk_coords[B*T] ({b*T + first token, tokens} of every chunk; row
//   b's chunks in order from b*T on, a row of T tokens having at most T),
// then its per-chunk items.
inline size_t ws_chunk_coords_offset(int B, int T) {
  return ws_bytes(B, T, true) + align_up(sizeof(int32_t) * (size_t)B * T, 256) +
         ws_row_offsets_bytes(B);
}
inline size_t ws_chunk_tables_bytes(int B, int T) {
  return align_up(sizeof(int32_t) * (size_t)B * T, 256) + ws_row_offsets_bytes(B) +
         align_up(sizeof(int2) * (size_t)B * T, 256);
}

// Where one unit of work lives: a run of one row, for one head, for one
// tile of value columns.  With no segment ids, run r is the whole row r.
struct RunTable {
  const int32_t *row_offsets;   // [B+1] prefix of run counts, or nullptr
  const int2 *runs;             // [B*T] {start, end}, or nullptr
  const uint32_t *total_runs;   // device count, or nullptr (then = B)
};

struct FwdParams {
  int B, T, H, K, V;
  int v_tile, n_vtiles;
  const void *q, *k, *v;
  const float *g, *beta;
  float scale;
  const float *initial_state;
  void *o;
  float *final_state;
  RunTable runs;
  uint32_t *status;
  // Fallback gate (AUTO with segment ids): when set, the fused kernel runs
  // only if *gate_chunks > gate_capacity, i.e. when the split path's items
  // could not hold the runs of this call; the split kernels then do nothing.
  const uint32_t *gate_chunks;
  uint32_t gate_capacity;
};

struct ConvParams {
  int B, T, H, K, V;
  const void *x[3];
  void *y[3];
  const float *w;
  const int32_t *segment_ids;
  int l2norm_qk;
};

// ---- launchers (each returns cudaSuccess or the launch error) -------------
cudaError_t launch_segment_runs(int B, int T, int H, int K, int V,
                                const int32_t *segment_ids, void *o,
                                int o_is_bf16, const float *initial_state,
                                float *final_state, void *workspace,
                                cudaStream_t stream, bool with_chunks = false);

cudaError_t launch_fwd_simt(const FwdParams &p, bool bf16, cudaStream_t stream);
// Tensor-core path (bf16, K = V = 128).  Returns cudaErrorNotSupported when
// the shape does not apply.
cudaError_t launch_fwd_tc(const FwdParams &p, cudaStream_t stream);
bool fwd_tc_supported(int K, int V, bool bf16, int v_tile);

// Split tensor-core path (parallel prep kernel + recurrence kernel), bf16,
// K = V = 128, no segment ids; needs split_workspace_bytes() of workspace.
// With segment ids, the items are sized for at most max_runs_per_row runs
// per row; the kernels check the real count and report overflow.
size_t split_workspace_bytes(int B, int T, int H, bool has_seg = false,
                             int max_runs_per_row = 0);
bool fwd_split_supported(int K, int V, bool bf16, bool has_seg, int v_tile);
// with_fallback (AUTO): with segment ids, also enqueue the fused kernel,
// gated to run only when the runs overflow the split items.  scan_segs > 0
// (rows without segment ids only): the recurrence as a chunk-parallel scan
// over that many segments per row (scan_segments() rounds the request; 0 in
// scan_segments picks the count that fills the GPU).
cudaError_t launch_fwd_split(const FwdParams &p, void *workspace, size_t workspace_bytes,
                             cudaStream_t stream, bool with_fallback = false, int scan_segs = 0);
int scan_segments(int B, int T, int H, int n_segs);
size_t scan_workspace_bytes(int B, int T, int H, int n_segs);

// Backward (kda_bwd.cu).  Per-tile partial sums of dq, dk, dg ([n_vtiles]
// x [B*T*H*K]) and dbeta ([n_vtiles] x [B*T*H]) are summed into the outputs
// by a second kernel; dv and d_initial are written directly.
struct BwdParams {
  int B, T, H, K, V, n_vtiles;
  const void *q, *k, *v, *d_o;
  const float *g, *beta, *initial_state, *d_final;
  float scale;
  float *dv, *d_initial;
  float *part_q, *part_k, *part_g, *part_b;
  float *ckpt;              // per-CTA checkpoint scratch
  size_t ckpt_cta_floats;   // floats per CTA
  int grid;                 // CTAs (the scratch is sized for them)
  RunTable runs;
};
constexpr int kBwdMaxCtas = 152;
// Scratch after the run table: checkpoints, then the partial sums.
size_t bwd_scratch_bytes(int B, int T, int H, int K, int V);
bool bwd_supported(int K, int V);
cudaError_t launch_bwd(const BwdParams &p, bool bf16, const int32_t *segment_ids,
                       float *dq, float *dk, float *dg, float *dbeta, cudaStream_t stream);

// Tensor-core backward (kda_bwd_tc.cu): bf16, K = V = 128; its workspace
// holds the forward's per-chunk items and the saved states
// (bwd_tc_workspace_bytes; with segment ids, for at most max_runs_per_row
// runs per row, after the run builder's tables).  With segment ids the run
// builder (launch_segment_runs with chunk tables) must have run on the
// workspace; padding tokens get zero gradients.
bool bwd_tc_supported(int K, int V, bool bf16);
size_t bwd_tc_workspace_bytes(int B, int T, int H, bool has_seg, int max_runs_per_row);
// from_saved: the items and saves come from a preceding launch_fwd_save
// on the same inputs and workspace (the forward passes are skipped).
cudaError_t launch_bwd_tc(const BwdParams &p, const int32_t *segment_ids, void *workspace,
                          size_t workspace_bytes, float *dq, float *dk, float *dg,
                          float *dbeta, uint32_t *status, cudaStream_t stream,
                          bool from_saved = false);
// The forward (o, final state of p) that also leaves in the workspace what
// launch_bwd_tc(from_saved) reads; with segment ids the run builder (with
// chunk tables) must have run on the workspace.
cudaError_t launch_fwd_save(const FwdParams &p, void *workspace, size_t workspace_bytes,
                            cudaStream_t stream);

cudaError_t launch_short_conv(const ConvParams &p, bool bf16,
                              cudaStream_t stream);

int num_sms();

// Shape validation shared by the forward entry points (KDA_OK, or the code
// kda_chunk_fwd returns for that shape).
kda_status check_shape(const kda_shape *s);

// ---- device helpers -------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ void set_status(uint32_t *status, uint32_t bits) {
  if (status) atomicOr(status, bits);
}

// Decode unit index -> (row b, run [start, end), first/last flags, h, vt).
struct Unit {
  int b, start, end, h, vt;
  int run_in_row;  // index of the run within its row
  bool first, last;
};

__device__ __forceinline__ uint32_t total_units(const RunTable &rt, int B,
                                                int H, int n_vtiles) {
  const uint32_t runs = rt.total_runs ? *rt.total_runs : (uint32_t)B;
  return runs * (uint32_t)H * (uint32_t)n_vtiles;
}

__device__ __forceinline__ Unit decode_unit(const RunTable &rt, uint32_t u,
                                            int B, int T, int H,
                                            int n_vtiles) {
  Unit x;
  x.vt = (int)(u % (uint32_t)n_vtiles);
  u /= (uint32_t)n_vtiles;
  x.h = (int)(u % (uint32_t)H);
  const int run = (int)(u / (uint32_t)H);
  if (!rt.runs) {
    x.b = run;
    x.start = 0;
    x.end = T;
    x.run_in_row = 0;
    x.first = x.last = true;
    return x;
  }
  // Largest b with row_offsets[b] <= run (rows with no runs are skipped).
  int lo = 0, hi = B;  // invariant: row_offsets[lo] <= run < row_offsets[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (rt.row_offsets[mid] <= run) lo = mid; else hi = mid;
  }
  x.b = lo;
  const int i = run - rt.row_offsets[lo];
  const int n = rt.row_offsets[lo + 1] - rt.row_offsets[lo];
  const int2 r = rt.runs[(size_t)lo * T + i];
  x.start = r.x;
  x.end = r.y;
  x.run_in_row = i;
  x.first = (i == 0);
  x.last = (i == n - 1);
  return x;
}

}  // namespace kda
