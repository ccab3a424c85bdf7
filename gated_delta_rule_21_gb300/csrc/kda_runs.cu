// kda_runs.cu -- turns packed segment ids into the run list the forward
// kernels schedule over.
//
// Segment ids [B,T] are 1-based with 0 = padding (page "feat(kda): integrate
// KDA attention with tokamax backend and CP support", section "Public API",
// decoder_segment_ids); the state restarts at every segment boundary.  A run
// is a maximal span of equal non-zero ids:
//     start at t  <=>  seg[t] != 0 and (t == 0 or seg[t-1] != seg[t])
//     end after t <=>  seg[t] != 0 and (t == T-1 or seg[t+1] != seg[t])
// The i-th start and the i-th end of a row belong to the same run.
//
// One CTA per row.  Besides the run list it writes o = 0 for padding tokens
// (the forward kernels never visit them) and, for a row with no run,
// final_state = initial_state (or zeros).  For the split path it also splits
// the row's runs into 64-token chunks: each run's first chunk within the row
// and, per chunk, its first token and length (the row's chunk table).  The
// last CTA to finish turns the per-row counts into prefixes (row_offsets, and
// the chunk counts' prefix) and the totals, and returns the completion
// counter to zero so the workspace stays reusable.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 512;
constexpr int kTokPerThread = 16;
constexpr int kTile = kThreads * kTokPerThread;  // 8192 tokens per pass

// Exclusive block-wide scan of a packed 64-bit counter (three 21-bit fields
// added lane-wise; no field exceeds 2^21 because a tile has 8192 tokens).
__device__ unsigned long long block_excl_scan64(unsigned long long v,
                                                unsigned long long *total,
                                                unsigned long long *sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) sm[warp] = x;
  __syncthreads();
  if (warp == 0) {
    unsigned long long s = lane < nwarps ? sm[lane] : 0ull;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += y;
    }
    if (lane < nwarps) sm[lane] = s;
  }
  __syncthreads();
  const unsigned long long before = warp > 0 ? sm[warp - 1] : 0ull;
  *total = sm[nwarps - 1];
  __syncthreads();  // sm is reused by the next call
  return before + x - v;
}

__device__ __forceinline__ int field(unsigned long long x, int i) {
  return (int)((x >> (21 * i)) & ((1ull << 21) - 1));
}

__global__ void __launch_bounds__(kThreads)
    segment_runs_kernel(int B, int T, int H, int K, int V,
                        const int32_t *__restrict__ seg, char *o,
                        int o_elem_bytes, const float *initial_state,
                        float *final_state, WsHeader *hdr,
                        int32_t *row_offsets, int2 *runs,
                        int32_t *run_chunk_base, int32_t *chunk_row_offsets, int2 *coords) {
  __shared__ unsigned long long sm_scan[32];
  __shared__ int sm_pad[kTile];
  __shared__ int sm_is_last;

  const int b = blockIdx.x;
  const int32_t *srow = seg + (size_t)b * T;
  int2 *rrow = runs + (size_t)b * T;
  const size_t o_row_bytes = (size_t)H * V * o_elem_bytes;  // one token
  const size_t o_row_vec = o_row_bytes / 16;                // multiple of 16
  int n_runs = 0, n_ends = 0;

  for (int base = 0; base < T; base += kTile) {
    const int t0 = base + threadIdx.x * kTokPerThread;
    int cur[kTokPerThread + 2];  // seg[t0-1 .. t0+16]
#pragma unroll
    for (int i = 0; i < kTokPerThread + 2; ++i) {
      const int t = t0 - 1 + i;
      cur[i] = (t >= 0 && t < T) ? srow[t] : 0;
    }
    int ns = 0, ne = 0, np = 0;
#pragma unroll
    for (int i = 1; i <= kTokPerThread; ++i) {
      if (t0 - 1 + i >= T) break;
      const int s = cur[i];
      ns += (s != 0 && s != cur[i - 1]);
      ne += (s != 0 && s != cur[i + 1]);
      np += (s == 0);
    }
    unsigned long long tot;
    const unsigned long long pre = block_excl_scan64(
        (unsigned long long)ns | ((unsigned long long)ne << 21) |
            ((unsigned long long)np << 42),
        &tot, sm_scan);
    int ps = n_runs + field(pre, 0), pe = n_ends + field(pre, 1);
    int pp = field(pre, 2);
#pragma unroll
    for (int i = 1; i <= kTokPerThread; ++i) {
      const int t = t0 - 1 + i;
      if (t >= T) break;
      const int s = cur[i];
      if (s != 0 && s != cur[i - 1]) rrow[ps++].x = t;
      if (s != 0 && s != cur[i + 1]) rrow[pe++].y = t + 1;
      if (s == 0) sm_pad[pp++] = t;
    }
    __syncthreads();
    // o = 0 on this tile's padding tokens, 16 bytes per store.
    const int tot_pad = field(tot, 2);
    const size_t n_vec = (size_t)tot_pad * o_row_vec;
    for (size_t i = threadIdx.x; i < n_vec; i += blockDim.x) {
      const int t = sm_pad[i / o_row_vec];
      uint4 *dst = reinterpret_cast<uint4 *>(
          o + ((size_t)b * T + t) * o_row_bytes);
      dst[i % o_row_vec] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    n_runs += field(tot, 0);
    n_ends += field(tot, 1);
  }

  // A row with no run: its final state is the initial state (or zeros).
  if (n_runs == 0 && final_state) {
    const size_t n4 = (size_t)H * K * V / 4;
    const size_t off = (size_t)b * H * K * V;
    float4 *dst = reinterpret_cast<float4 *>(final_state + off);
    const float4 *src =
        initial_state ? reinterpret_cast<const float4 *>(initial_state + off)
                      : nullptr;
    for (size_t i = threadIdx.x; i < n4; i += blockDim.x)
      dst[i] = src ? src[i] : make_float4(0.f, 0.f, 0.f, 0.f);
  }

  // Chunks of 64 tokens per run and their prefix inside the row (for the
  // split path, whose work items are (run, chunk, head)), and each chunk's
  // tokens {b*T + first token, tokens} at coords[b*T + chunk within the row]
  // (a row has at most T chunks).
  int n_chunks_row = 0;
  if (run_chunk_base) {
    __syncthreads();  // this row's run records are written
    for (int base = 0; base < n_runs; base += blockDim.x) {
      const int i = base + threadIdx.x;
      int cnt = 0;
      int2 r = make_int2(0, 0);
      if (i < n_runs) {
        r = rrow[i];
        cnt = (r.y - r.x + kChunk - 1) / kChunk;
      }
      unsigned long long tot;
      const unsigned long long ex =
          block_excl_scan64((unsigned long long)cnt, &tot, sm_scan);
      if (i < n_runs) {
        const int lb = n_chunks_row + (int)ex;
        run_chunk_base[(size_t)b * T + i] = lb;
        int2 *crow = coords + (size_t)b * T + lb;
        const int y0 = b * T + r.x;
        for (int j = 0; j < cnt; ++j)
          crow[j] = make_int2(y0 + j * kChunk, min(kChunk, r.y - r.x - j * kChunk));
      }
      n_chunks_row += (int)tot;
    }
  }

  if (threadIdx.x == 0) {
    row_offsets[b + 1] = n_runs;
    if (chunk_row_offsets) chunk_row_offsets[b + 1] = n_chunks_row;
    __threadfence();
    const unsigned prev = atomicAdd(&hdr->rows_done, 1u);
    __threadfence();
    sm_is_last = (prev == (unsigned)(B - 1));
  }
  __syncthreads();
  if (!sm_is_last) return;

  // Last CTA: inclusive prefix of the counts in place, then the total.
  int carry = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int i = base + threadIdx.x;
    const int c = i < B ? __ldcg(row_offsets + i + 1) : 0;
    unsigned long long tot;
    const unsigned long long ex =
        block_excl_scan64((unsigned long long)c, &tot, sm_scan);
    if (i < B) row_offsets[i + 1] = carry + (int)ex + c;
    carry += (int)tot;
  }
  int chunk_carry = 0;
  if (chunk_row_offsets) {
    for (int base = 0; base < B; base += blockDim.x) {
      const int i = base + threadIdx.x;
      const int c = i < B ? __ldcg(chunk_row_offsets + i + 1) : 0;
      unsigned long long tot;
      const unsigned long long ex =
          block_excl_scan64((unsigned long long)c, &tot, sm_scan);
      if (i < B) chunk_row_offsets[i + 1] = chunk_carry + (int)ex + c;
      chunk_carry += (int)tot;
    }
  }
  if (threadIdx.x == 0) {
    row_offsets[0] = 0;
    hdr->total_runs = (uint32_t)carry;
    if (chunk_row_offsets) {
      chunk_row_offsets[0] = 0;
      hdr->total_chunks = (uint32_t)chunk_carry;
    }
    hdr->rows_done = 0u;
  }
}

}  // namespace

cudaError_t launch_segment_runs(int B, int T, int H, int K, int V,
                                const int32_t *segment_ids, void *o,
                                int o_is_bf16, const float *initial_state,
                                float *final_state, void *workspace,
                                cudaStream_t stream, bool with_chunks) {
  char *ws = static_cast<char *>(workspace);
  WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
  int32_t *row_offsets = reinterpret_cast<int32_t *>(ws + sizeof(WsHeader));
  int2 *runs =
      reinterpret_cast<int2 *>(ws + sizeof(WsHeader) + ws_row_offsets_bytes(B));
  int32_t *chunk_base = nullptr, *chunk_rows = nullptr;
  int2 *coords = nullptr;
  if (with_chunks) {
    coords = reinterpret_cast<int2 *>(ws + ws_chunk_coords_offset(B, T));
    chunk_base = reinterpret_cast<int32_t *>(ws + ws_bytes(B, T, true));
    chunk_rows = reinterpret_cast<int32_t *>(ws + ws_bytes(B, T, true) +
                                             align_up(sizeof(int32_t) * (size_t)B * T, 256));
  }
  segment_runs_kernel<<<B, kThreads, 0, stream>>>(
      B, T, H, K, V, segment_ids, static_cast<char *>(o), o_is_bf16 ? 2 : 4,
      initial_state, final_state, hdr, row_offsets, runs, chunk_base, chunk_rows, coords);
  return cudaGetLastError();
}

}  // namespace kda
