// kda_split.cuh -- what the split tensor-core forward (kda_fwd_split.cu) and
// the tensor-core backward (kda_bwd_tc.cu) share: the per-chunk item layout
// in the workspace, the chunk table, and the launchers that make items and
// saved states for the backward.  Internal to libkda.
#pragma once

#include <cuda.h>

#include "kda_internal.cuh"
#include "kda_tc_common.cuh"

namespace kda {
namespace split {

constexpr int C = kChunk;
constexpr int KD = 128;
constexpr int VD = 128;
constexpr int VT = 32;

// ---- one workspace item (per row, chunk, head) ----------------------------
// Each region is already in the shared-memory operand layout the recurrence
// kernel's MMAs read, so a stage is a plain bulk copy of the item.
// Q e^G and A_qk carry the attention scale (folded in by the prep), so the
// products that read them come out scaled.
constexpr uint32_t I_WQ = 0;          // [w ; scale Q e^G]: MN-major, 128 rows x Kd 128 channels
constexpr uint32_t I_AQK = 32768;     // scale A_qk: K-major, 64 rows, Kd 64
constexpr uint32_t I_KHT = 40960;     // (K e^{G_C-G})^T: K-major, 128 channels x Kd 64 rows
constexpr uint32_t I_U = 57344;       // u bf16, 4 tiles of 32 columns, see u_off
constexpr uint32_t I_GAM = 73728;     // e^{G_C} fp32 [128]
constexpr uint32_t ITEM_BYTES = 74240;     // 72.5 KiB, 256-byte aligned
constexpr size_t WS_ITEMS_OFF = 1024;      // after the workspace header
// The backward's items append what its gradient kernel reads instead of
// recomputing the chunk's solve: T = (I + beta A_kk)^-1 (bf16, K-major
// 64 x Kd 64), A_kk without beta (fp32 row-major [r][j], strict lower) and
// K e^G (bf16, K-major 128 channels x Kd 64 rows).
constexpr uint32_t I_T = ITEM_BYTES;             // 8 KiB
constexpr uint32_t I_AKK = I_T + 8192;           // 16 KiB
constexpr uint32_t I_KT = I_AKK + 16384;         // 16 KiB
constexpr uint32_t ITEM_BYTES_BWD = I_KT + 16384;  // 112.5 KiB
// Per (chunk, head) values the backward saves, indexed like the items:
// the state entering the chunk S (K-major keys x Kd 128 values, bf16), U of
// the chunk (K-major 64 rows x Kd 128), the gradient of the state leaving
// the chunk dS' (like S) and dU (like U).
constexpr uint32_t SV_S = 0, SV_U = 32768, SV_DSP = 49152, SV_DU = 81920;
constexpr uint32_t SV_BYTES = 98304;
static_assert(ITEM_BYTES_BWD % 256 == 0 && SV_BYTES % 256 == 0, "item alignment");

// Byte offset of u's 8 columns c .. c + 7 (c a multiple of 8 within the
// 32-column tile vt) of row r: each tile is [column group of 8][row][8]
// bf16, so the 32 rows a warp reads for one column group are 512
// contiguous bytes (no bank conflicts), and a tile is one 4 KiB block.
__device__ __forceinline__ uint32_t u_off(int vt, int c, int r) {
  return (uint32_t)(vt * 4096 + (c >> 3) * 1024 + r * 16);
}

// Chunk items: with segment ids, chunk k of the concatenated runs of all rows
// (run i of row b owns chunks chunk_row_offsets[b] + run_chunk_base[b*T+i] ..);
// without them, row b owns chunks b*n_chunks ... (b+1)*n_chunks - 1.
struct ChunkTable {
  const int32_t *run_chunk_base;     // [B*T] or nullptr (no segment ids)
  const int32_t *chunk_row_offsets;  // [B+1]
  const int2 *coords;                // [B*T]: {b*T + first token, tokens}, row b's
                                     // chunks from b*T on
  const uint32_t *total_chunks;      // device count
  uint32_t capacity;                 // chunk items the workspace holds
  uint32_t item_stride;              // bytes per item (ITEM_BYTES or ITEM_BYTES_BWD)
  int n_chunks_row;                  // chunks per row without segment ids
  int n_rows;                        // B
  int report_overflow;               // set KDA_DEVICE_WORKSPACE on overflow
};

__device__ __forceinline__ uint32_t total_chunk_count(const ChunkTable &ct, int B) {
  return ct.run_chunk_base ? *ct.total_chunks : (uint32_t)B * ct.n_chunks_row;
}

// First token and end of chunk k, and its row.
__device__ __forceinline__ void chunk_of(const ChunkTable &ct, int T, uint32_t k, int &b,
                                         int &t0, int &end) {
  if (!ct.run_chunk_base) {
    b = (int)(k / (uint32_t)ct.n_chunks_row);
    t0 = (int)(k % (uint32_t)ct.n_chunks_row) * C;
    end = T;
    return;
  }
  int lo = 0, hi = ct.n_rows;  // the row: chunk_row_offsets[lo] <= k < [lo + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((uint32_t)ct.chunk_row_offsets[mid] <= k) lo = mid; else hi = mid;
  }
  const int2 e = ct.coords[(size_t)lo * T + (k - (uint32_t)ct.chunk_row_offsets[lo])];
  b = lo;
  t0 = e.x - b * T;
  end = t0 + e.y;
}

// Global index of the first chunk of a unit's run (row b, run i of the row).
__device__ __forceinline__ uint32_t run_chunk_base(const ChunkTable &ct, int b, int T,
                                                   int run_in_row) {
  return ct.run_chunk_base
             ? (uint32_t)(ct.chunk_row_offsets[b] + ct.run_chunk_base[(size_t)b * T + run_in_row])
             : (uint32_t)b * ct.n_chunks_row;
}

__device__ __forceinline__ void st_g16(unsigned char *g, uint32_t off, const float (&v)[8]) {
  uint4 w;
  w.x = tc::pack_bf16(v[0], v[1]);
  w.y = tc::pack_bf16(v[2], v[3]);
  w.z = tc::pack_bf16(v[4], v[5]);
  w.w = tc::pack_bf16(v[6], v[7]);
  *reinterpret_cast<uint4 *>(g + off) = w;
}

// Where the items start in a workspace (after the header, or after the run
// list and the chunk tables with segment ids).
size_t items_offset(int B, int T, bool has_seg);

// What the backward needs from the forward: items of ITEM_BYTES_BWD and the
// saved S and U of every chunk (launch_fwd_for_bwd), in a workspace laid out
// [items_offset][items][saves] (with segment ids, after the run list and
// chunk tables the run builder wrote); the chunk table of that call.
struct BwdLayout {
  unsigned char *items;
  unsigned char *saves;
  ChunkTable ct;
};
// With segment ids the items and saves are sized for at most
// max_runs_per_row runs per row (each run adds at most one partial chunk).
size_t bwd_tc_workspace_bytes(int B, int T, int H, bool has_seg, int max_runs_per_row);
// The layout of such a workspace (false when it is too small).
bool bwd_layout(const FwdParams &p, void *workspace, size_t workspace_bytes, BwdLayout *out);
// The prep kernel with backward items, then the recurrence saving S and U:
// in its save mode (no o, no final state), or with with_outputs as the
// forward itself (o and the final state of p) that also saves.
cudaError_t launch_fwd_for_bwd(const FwdParams &p, void *workspace, size_t workspace_bytes,
                               BwdLayout *out, cudaStream_t stream, bool with_outputs = false);
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize,
              uint64_t cols, uint64_t rows, uint32_t box_cols, CUtensorMapSwizzle swz);

}  // namespace split
}  // namespace kda
