// kda_fwd_split.cu -- chunked KDA forward as two tensor-core kernels:
//
//   1. fwd_prep_kernel: every (row, chunk, head) item is independent of the
//      recurrent state, so all of them run in parallel over the whole GPU.
//      Per item (64 tokens of one head) it builds the gate cumsum and decay
//      factors, the intra-chunk products A_kk / A_qk on tcgen05 (one MMA per
//      16-row block), the triangular inverse T = (I + beta A_kk)^-1 (fp32,
//      blocked), and [w | u] = T diag(beta) [K e^G | V] on tcgen05, and
//      writes the operands the recurrence needs into the workspace, already
//      in the shared-memory layouts the tensor cores read:
//         [w ; scale Q e^G] (128 x 128 bf16), scale A_qk (64 x 64 bf16),
//         (K e^{G_C - G})^T (128 x 64 bf16), u (64 x 128 bf16), e^{G_C}
//      (the attention scale is folded into the Q e^G and A_qk operands).
//   2. fwd_rec_kernel: one CTA per (row, head, value tile of 32 or 64
//      columns) walks
//      the chunks in order with the fp32 state in registers; per chunk it
//      bulk-copies the item (double-buffered) and runs only the
//      state-dependent MMAs:  D1 = [w ; Q e^G] S,  U = u - w S,
//      D1 += [0 ; A_qk] U,  D2 = (K e^{G_C-G})^T U,  S <- e^{G_C} S + D2,
//      o = D1[64:128] (already scaled).
//
// The arithmetic is the same chunk form, sub-block factors and rounding
// points as the fused kernel (kda_fwd_tc.cu); see there for the algebra.
// This path needs a workspace of split_workspace_bytes() (about 73 KB per
// chunk and head).  With segment ids the chunks are those of each run (a
// run's last chunk may be short), sized for a caller bound on runs per row;
// the kernels check the real chunk count and report KDA_DEVICE_WORKSPACE
// (doing nothing else) when it does not fit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <type_traits>

#include "kda_f32x2.cuh"
#include "kda_internal.cuh"
#include "kda_split.cuh"
#include "kda_tc_common.cuh"

namespace kda {
using namespace split;
namespace {
using namespace tc;

// ---- prep kernel --------------------------------------------------------------
// Two CTAs of 256 threads per SM, each working on its own item, so that one
// CTA's serial phases (the block solve, the MMA round trips) overlap the
// other's.  To fit two CTAs, the intra-chunk operands are built in two
// halves of 64 key channels (the A products accumulate over both halves on
// the tensor cores).
//
// Elementwise work (gate cumsum, decay factors, operand tiles) is done by
// channel owners: thread (c, b) holds key channel c of the half for the 16
// rows of sub-block b, so the cumsum runs down its own registers, every
// per-(block, channel) factor is a per-thread constant, and each operand is
// written in the layout that keeps a channel's 8 consecutive rows in one
// 16-byte chunk: MN-major X, Y (A products) and Q e^G (item), K-major
// (K e^G)^T (the w product) and (K e^{G_C-G})^T (item).  w is produced
// transposed, w^T = (K e^G)^T (T diag(beta))^T, so its TMEM lanes are
// channels too and its rows leave TMEM as MN-major 16-byte chunks.
//
// Shared memory (offsets from a 1 KiB-aligned base):
//   RAW   q, k (64 rows x 64 channels bf16, 128 B per row) and g (two
//         64 x 32 fp32 boxes, 128 B per row) of one channel half, no swizzle:
//         a warp reads 32 consecutive channels of one row;
//   X, Y  [K e1 ; Q e1] (128 rows) and Y_0..Y_3 (160 rows), MN-major, Kd 64;
//   KT    (K e^G)^T, K-major, 128 channels x Kd 64 rows (both halves);
//   TB    T diag(beta), K-major, 64 rows x Kd 64 (the w product's B operand,
//         and the u product's A operand, whose rows 64..127 read V: ignored);
//   V     v, MN-major, 128 columns x Kd 64 rows (TMA);
//   solver fp32 buffers, aliased over RAW + X once the A products are in
//   TMEM.
constexpr int PT = 256;                       // threads
constexpr int KH = 64;                        // key channels per half
constexpr uint32_t P_RAW_Q = 0, P_RAW_K = 8192, P_RAW_G = 16384;
constexpr uint32_t P_RAW_TX = 8192 * 2 + 16384;
constexpr uint32_t P_X = 32768;               // 128 x Kd 64
constexpr uint32_t P_Y = P_X + 16384;         // Y_0..Y_3, 160 rows x Kd 64
constexpr uint32_t P_KT = P_Y + 20480;        // 128 x Kd 64, K-major
constexpr uint32_t P_TB = P_KT + 16384;       // 64 x Kd 64, K-major
constexpr uint32_t P_V = P_TB + 8192;         // 128 x Kd 64, MN-major
constexpr uint32_t P_V_TX = 16384;
constexpr uint32_t P_MISC = P_V + 16384;
constexpr uint32_t P_BETA = P_MISC;           // 64 fp32
constexpr uint32_t P_BSUM = P_BETA + 256;     // 4 x 64 fp32: log2e x block sums of g (one half)
constexpr uint32_t P_BAR = P_BSUM + 1024;     // raw, mma, v
constexpr uint32_t P_SLOT = P_BAR + 24;
constexpr uint32_t P_ABORT = P_SLOT + 4;
constexpr uint32_t P_SMEM = P_ABORT + 12;
constexpr uint32_t P_ALLOC = P_SMEM + 1024;
constexpr int LDF = C + 4;
constexpr uint32_t P_AKK = 0;                      // fp32 64 x 68 (beta A_kk)
constexpr uint32_t P_TF = P_AKK + 64 * LDF * 4;    // fp32 64 x 68 (T)
constexpr uint32_t P_SCR = P_TF + 64 * LDF * 4;    // 10 blocks of 16 x LDS fp32
constexpr int LDS = 20;                            // padded: conflict-free rows
static_assert(P_SCR + 10 * 16 * LDS * 4 <= P_Y, "solver buffers stay in RAW + X");
static_assert(LDF % 4 == 0 && LDS % 4 == 0 && P_TF % 16 == 0 && P_SCR % 16 == 0,
              "16-byte rows for the block products' vector loads");
static_assert(P_TB + 16384 <= P_V + 16384, "the u product's 128-row A operand stays in smem");
static_assert(P_X % 1024 == 0 && P_Y % 1024 == 0 && P_KT % 1024 == 0 && P_V % 1024 == 0,
              "operand alignment");
static_assert(2 * (P_ALLOC + 1024) <= 233472, "two prep CTAs fit one SM");

// Y_0..Y_3 are stored back to back (row groups of 8), so together they form
// one 160-row B operand: a single N = 160 MMA gives X Y_b^T for every b at
// TMEM columns 8 b (b + 1) ... 8 b (b + 1) + 16 (b + 1) - 1.
__device__ __forceinline__ uint32_t p_y_off(int b) {
  return P_Y + 128u * (uint32_t)(8 * b * (b + 1));
}
__device__ __forceinline__ uint32_t tm_a(int b) { return 8u * (uint32_t)(b * (b + 1)); }
// The 16-column TMEM pieces of X Y^T that hold the products of the rows of
// lane quadrant `quad` (blocks 0-1 for even quadrants, 2-3 for odd ones).
__device__ __forceinline__ int piece_count(int quad) { return (quad & 1) ? 7 : 3; }
__device__ __forceinline__ void piece(int quad, int i, int &b, int &pp) {
  if ((quad & 1) == 0) {
    b = i == 0 ? 0 : 1;
    pp = i == 0 ? 0 : i - 1;
  } else {
    b = i < 3 ? 2 : 3;
    pp = i < 3 ? i : i - 3;
  }
}

// One 16 x 16 block product on the CUDA cores by one warp (e = lane: rows
// e / 4 and e / 4 + 8, four columns each): dst = sgn X Y + add_sgn add.
// Column pairs accumulate in packed f32x2 registers (each lane an ordinary
// fp32 FMA, in the same order over t as the scalar loop), and X is read
// four k-steps per 16-byte load (ldx and the row starts are multiples of 4).
__device__ __forceinline__ void blk_prod(float *dst, int ldd, const float *X, int ldx,
                                         const float *Y, int ldy, float sgn, const float *add,
                                         int lda, int e, float add_sgn = -1.f) {
  const int r = e >> 2, c4 = (e & 3) * 4;
  u64 a[2][2] = {{0ull, 0ull}, {0ull, 0ull}};  // [row r | r + 8][columns c4.. | c4 + 2..]
#pragma unroll
  for (int t4 = 0; t4 < 4; ++t4) {
    const float4 x0 = *reinterpret_cast<const float4 *>(X + r * ldx + 4 * t4);
    const float4 x1 = *reinterpret_cast<const float4 *>(X + (r + 8) * ldx + 4 * t4);
    const float xa[4] = {x0.x, x0.y, x0.z, x0.w}, xb[4] = {x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int tt = 0; tt < 4; ++tt) {
      const float4 y = *reinterpret_cast<const float4 *>(Y + (4 * t4 + tt) * ldy + c4);
      const u64 y01 = pk2(y.x, y.y), y23 = pk2(y.z, y.w);
      const u64 xa2 = pk2(xa[tt], xa[tt]), xb2 = pk2(xb[tt], xb[tt]);
      a[0][0] = fma2(xa2, y01, a[0][0]);
      a[0][1] = fma2(xa2, y23, a[0][1]);
      a[1][0] = fma2(xb2, y01, a[1][0]);
      a[1][1] = fma2(xb2, y23, a[1][1]);
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int rr = r + 8 * h;
    float4 o;
    upk2(a[h][0], o.x, o.y);
    upk2(a[h][1], o.z, o.w);
    o = make_float4(sgn * o.x, sgn * o.y, sgn * o.z, sgn * o.w);
    if (add) {
      const float4 z = *reinterpret_cast<const float4 *>(add + rr * lda + c4);
      o.x = fmaf(add_sgn, z.x, o.x);
      o.y = fmaf(add_sgn, z.y, o.y);
      o.z = fmaf(add_sgn, z.z, o.z);
      o.w = fmaf(add_sgn, z.w, o.w);
    }
    *reinterpret_cast<float4 *>(dst + rr * ldd + c4) = o;
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }

// 8 fp32 values (consecutive rows of one channel) as one 16-byte bf16 chunk.
__device__ __forceinline__ uint4 pack8(const float (&v)[8]) {
  return make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                    pack_bf16(v[6], v[7]));
}
__device__ __forceinline__ uint4 pack8s(const float (&v)[8], float s) {
  return make_uint4(pack_bf16(v[0] * s, v[1] * s), pack_bf16(v[2] * s, v[3] * s),
                    pack_bf16(v[4] * s, v[5] * s), pack_bf16(v[6] * s, v[7] * s));
}
// The same from 4 packed f32x2 row pairs (scaled on the FMA pipe two lanes
// at a time: each lane is the scalar fp32 product).
__device__ __forceinline__ uint32_t pack_bf16x2(u64 v) {
  float a, b;
  upk2(v, a, b);
  return pack_bf16(a, b);
}
__device__ __forceinline__ uint4 pack8x2(const u64 (&v)[4]) {
  return make_uint4(pack_bf16x2(v[0]), pack_bf16x2(v[1]), pack_bf16x2(v[2]), pack_bf16x2(v[3]));
}
__device__ __forceinline__ uint4 pack8x2s(const u64 (&v)[4], float s) {
  const u64 s2 = pk2(s, s);
  return make_uint4(pack_bf16x2(mul2(v[0], s2)), pack_bf16x2(mul2(v[1], s2)),
                    pack_bf16x2(mul2(v[2], s2)), pack_bf16x2(mul2(v[3], s2)));
}

__global__ void __launch_bounds__(PT, 2)
    fwd_prep_kernel(const FwdParams p, unsigned char *items, const ChunkTable ct,
                    const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_g,
                    const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  float *sBeta = reinterpret_cast<float *>(smem + P_BETA);
  float *sBsum = reinterpret_cast<float *>(smem + P_BSUM);
  float *sAkk = reinterpret_cast<float *>(smem + P_AKK);
  float *sT = reinterpret_cast<float *>(smem + P_TF);
  float *sScr = reinterpret_cast<float *>(smem + P_SCR);
  volatile uint32_t *sAbort = reinterpret_cast<volatile uint32_t *>(smem + P_ABORT);
  const uint32_t raw_bar = sb + P_BAR, mma_bar = sb + P_BAR + 8, v_bar = sb + P_BAR + 16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, sub = warp >> 2;  // 2 warps per TMEM lane quadrant
  const int L = 32 * quad + lane;
  // Channel owner: channel ec of the half, sub-block eb (rows 16 eb ..).  The
  // two warps on each scheduler get blocks {0, 3} or {1, 2}, which balances
  // the Y versions they write (block b writes 4 - b of them).
  const int ec = 32 * (warp & 1) + lane;
  const int eb = (warp >> 1) ^ ((warp >> 2) & 1);
  const int er0 = kSub * eb;
  // The MMAs are issued by a thread of warp 4 (block 3, the lightest share
  // of the elementwise work): issuing holds a thread for about the MMA's
  // execution time.
  constexpr int kIssuer = 128;
  const int H = p.H, T = p.T;

  if (warp == 0) tmem_alloc(sb + P_SLOT, 256);
  if (tid == 0) {
    mbar_init(raw_bar, 1);
    mbar_init(mma_bar, 1);
    mbar_init(v_bar, 1);
    *sAbort = 0u;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + P_SLOT);
  const uint32_t tq = tmem + ((uint32_t)(32 * quad) << 16);
  uint32_t raw_phase = 0, mma_phase = 0, v_phase = 0;
  uint32_t raw_pending = 0, mma_pending = 0, v_pending = 0;
  bool raw_inflight = false, mma_inflight = false, v_inflight = false;
  auto abort_all = [&]() {
    *sAbort = 1u;
    set_status(p.status, KDA_DEVICE_TIMEOUT);
  };
  auto wait_raw = [&]() {
    if (!mbar_wait(raw_bar, raw_phase)) abort_all();
    else raw_inflight = false;
    raw_phase ^= 1u;
  };
  auto wait_mma = [&]() {
    mma_inflight = true;
    mma_pending = mma_phase;
    if (!mbar_wait(mma_bar, mma_phase)) abort_all();
    else mma_inflight = false;
    mma_phase ^= 1u;
  };

  // Items for the backward also carry T, A_kk and K e^G.
  const bool bwd_items = ct.item_stride == ITEM_BYTES_BWD;
  const uint32_t n_chunk_items = total_chunk_count(ct, p.B);
  if (n_chunk_items > ct.capacity && ct.report_overflow && tid == 0 && blockIdx.x == 0)
    set_status(p.status, KDA_DEVICE_WORKSPACE);  // the items cannot hold every chunk
  const uint32_t n_items = n_chunk_items > ct.capacity ? 0u : n_chunk_items * (uint32_t)H;
  // Where an item's tokens are (with segment ids, two binary searches over
  // global tables): computed once per item and carried to the next iteration.
  struct Coords {
    int b, t0, end, h;
  };
  auto item_coords = [&](uint32_t it) {
    Coords x;
    x.h = (int)(it % (uint32_t)H);
    chunk_of(ct, T, it / (uint32_t)H, x.b, x.t0, x.end);
    return x;
  };
  // Both issue functions are called by all 32 lanes of one warp: lane 0
  // arms the barrier, then one box per lane.
  // Half 0's request also pulls half 1's boxes into L2, so their copy,
  // issued once half 0's tiles are consumed, does not wait on DRAM.
  auto issue_raw = [&](const Coords &xc, int half) {  // q, k, g of one channel half
    const int y = xc.b * T + xc.t0, x = xc.h * KD + KH * half;
    if (lane == 0) mbar_expect_tx(raw_bar, P_RAW_TX);
    __syncwarp();
    if (lane == 0) tma_load_2d(sb + P_RAW_Q, &tm_q, x, y, raw_bar);
    else if (lane == 1) tma_load_2d(sb + P_RAW_K, &tm_k, x, y, raw_bar);
    else if (lane < 4) tma_load_2d(sb + P_RAW_G + 8192 * (lane - 2), &tm_g, x + 32 * (lane - 2), y, raw_bar);
    else if (half == 0 && lane == 4) tma_prefetch_2d(&tm_q, x + KH, y);
    else if (half == 0 && lane == 5) tma_prefetch_2d(&tm_k, x + KH, y);
    else if (half == 0 && lane < 8) tma_prefetch_2d(&tm_g, x + KH + 32 * (lane - 6), y);
  };
  // v as 16 column groups of 8, each 64 rows x 16 bytes: the MN-major layout
  // of V (read by the u product).
  auto issue_v = [&](const Coords &xc) {
    const int y = xc.b * T + xc.t0;
    if (lane == 0) mbar_expect_tx(v_bar, P_V_TX);
    __syncwarp();
    if (lane < VD / 8)
      tma_load_2d(sb + P_V + mn_off(8 * lane, 0, C), &tm_v, xc.h * VD + 8 * lane, y, v_bar);
  };
  auto load_beta = [&](const Coords &xc) -> float {
    const int t = xc.t0 + tid;
    return t < xc.end ? p.beta[((size_t)xc.b * T + t) * H + xc.h] : 0.f;
  };

  uint32_t item = blockIdx.x;
  float beta_next = 0.f;
  Coords cur = {0, 0, 0, 0};
  if (item < n_items) {
    cur = item_coords(item);
    if (warp == 0) issue_raw(cur, 0);
    if (warp == 1) issue_v(cur);
    raw_inflight = v_inflight = true;
    raw_pending = raw_phase;
    v_pending = v_phase;
    if (tid < C) beta_next = load_beta(cur);
  }
  for (; item < n_items; item += gridDim.x) {
    const int n = min(C, cur.end - cur.t0);
    const uint32_t next = item + gridDim.x;
    const bool has_next = next < n_items;
    const Coords nxt = has_next ? item_coords(next) : cur;
    unsigned char *gi = items + (size_t)item * ct.item_stride;
    if (tid < C) sBeta[tid] = beta_next;

    for (int half = 0; half < 2; ++half) {
      const int ch = KH * half + ec;  // this thread's channel (of 128)
      // ---- P17: this half's raw tiles
      wait_raw();

      // ---- P0: gate cumsum down this thread's 16 rows (log2 units; rows
      //      past the chunk's end add nothing), block sums to smem ----
      // A full chunk (every item but a run's last) takes code with no
      // per-row tests: `full` is a compile-time constant in each branch.
      const bool full_chunk = n == C;
      float G[kSub];
      auto cumsum = [&](auto full) {
        const unsigned char *gcol = smem + P_RAW_G + 8192 * (ec >> 5) + 4 * (ec & 31);
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < kSub; ++i) {
          const int r = er0 + i;
          const float gv = (decltype(full)::value || r < n)
                               ? *reinterpret_cast<const float *>(gcol + 128 * r) : 0.f;
          acc = fmaf(gv, kLog2e, acc);
          G[i] = acc;
        }
        sBsum[eb * KH + ec] = acc;
      };
      if (full_chunk) cumsum(std::true_type{});
      else cumsum(std::false_type{});
      __syncthreads();
      // ---- P1: block offsets and factors of (block eb, channel ch), then
      //      this half's operands: X, Y_b, (K e^G)^T (smem, for the MMAs),
      //      Q e^G and (K e^{G_C-G})^T (the item) ----
      float bs[kNumSub];
#pragma unroll
      for (int i = 0; i < kNumSub; ++i) bs[i] = sBsum[i * KH + ec];
      float P2 = 0.f, GC2 = 0.f;  // G before block eb, G at the chunk's end
#pragma unroll
      for (int i = 0; i < kNumSub; ++i) {
        if (i < eb) P2 += bs[i];
        GC2 += bs[i];
      }
      const float E2 = P2 + bs[eb];   // G at block eb's last row
      const float E3 = eb + 1 < kNumSub ? E2 + bs[min(eb + 1, kNumSub - 1)] : E2;
      const float E4 = eb + 2 < kNumSub ? E3 + bs[min(eb + 2, kNumSub - 1)] : E3;
      const float pre = ex2(P2);        // e^{G before the block}
      const float pre_s = pre * p.scale;
      const float suf = ex2(GC2 - E2);  // e^{G_C - E_b}
      const float rD = ex2(P2 - E2);    // 1 / D_b
      const float x2 = ex2(E3 - E2);    // D_{b+1}
      const float x3 = ex2(E4 - E2);    // D_{b+1} D_{b+2}
      if (eb == 0) reinterpret_cast<float *>(gi + I_GAM)[ch] = ex2(GC2);  // e^{G_C}
      if (half == 1) wait_mma();  // the half-0 MMA has read X and Y
      auto operands = [&](auto full) {
#pragma unroll
        for (int o = 0; o < 2; ++o) {
          const int r8 = er0 + 8 * o;  // first of the 8 rows of this chunk
          // pairs of consecutive rows in packed f32x2 registers
          u64 xk[4], xq[4], ke[4];
          const unsigned char *kcol = smem + P_RAW_K + 2 * ec;
          const unsigned char *qcol = smem + P_RAW_Q + 2 * ec;
#pragma unroll
          for (int i = 0; i < 8; i += 2) {
            float kv[2], qv[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int r = r8 + i + e;
              const bool valid = decltype(full)::value || r < n;
              kv[e] = valid ? bf16_lo(*reinterpret_cast<const unsigned short *>(kcol + 128 * r)) : 0.f;
              qv[e] = valid ? bf16_lo(*reinterpret_cast<const unsigned short *>(qcol + 128 * r)) : 0.f;
            }
            const float g0 = G[8 * o + i], g1 = G[8 * o + i + 1];
            const u64 e1 = pk2(ex2(g0), ex2(g1));                  // e^{G_r - P_b} in (0, 1]
            const u64 e2 = pk2(ex2(bs[eb] - g0), ex2(bs[eb] - g1));  // e^{E_b - G_r} in (0, 1]
            const u64 k2 = pk2(kv[0], kv[1]);
            xk[i / 2] = mul2(k2, e1);
            xq[i / 2] = mul2(pk2(qv[0], qv[1]), e1);
            ke[i / 2] = mul2(k2, e2);
          }
          *reinterpret_cast<uint4 *>(smem + P_X + mn_off(r8, ec, KH)) = pack8x2(xk);
          *reinterpret_cast<uint4 *>(smem + P_X + mn_off(64 + r8, ec, KH)) = pack8x2(xq);
          *reinterpret_cast<uint4 *>(smem + p_y_off(eb) + mn_off(r8, ec, KH)) = pack8x2s(ke, rD);
          if (eb + 1 < kNumSub)
            *reinterpret_cast<uint4 *>(smem + p_y_off(eb + 1) + mn_off(r8, ec, KH)) = pack8x2(ke);
          if (eb + 2 < kNumSub)
            *reinterpret_cast<uint4 *>(smem + p_y_off(eb + 2) + mn_off(r8, ec, KH)) = pack8x2s(ke, x2);
          if (eb + 3 < kNumSub)
            *reinterpret_cast<uint4 *>(smem + p_y_off(eb + 3) + mn_off(r8, ec, KH)) = pack8x2s(ke, x3);
          // K e^G (beta goes into T's columns), transposed for the w product
          {
            const uint4 kt = pack8x2s(xk, pre);
            *reinterpret_cast<uint4 *>(smem + P_KT + op_off(ch, r8, C)) = kt;
            if (bwd_items) *reinterpret_cast<uint4 *>(gi + I_KT + op_off(ch, r8, C)) = kt;
          }
          // scale folded in: the o rows of D1 and the o product come out scaled
          *reinterpret_cast<uint4 *>(gi + I_WQ + mn_off(64 + r8, ch, KD)) = pack8x2s(xq, pre_s);
          *reinterpret_cast<uint4 *>(gi + I_KHT + op_off(ch, r8, C)) = pack8x2s(ke, suf);
        }
      };
      if (full_chunk) operands(std::true_type{});
      else operands(std::false_type{});
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();
      if (*sAbort) goto done;

      // ---- P2: this half's share of the A products on the tensor cores;
      //      the next half's tiles (RAW is free once every thread passed) ----
      if (tid == kIssuer) {
        tc_fence_after();
        mma_group(tmem, sb + P_X, sb + P_Y, KH, 160, half > 0, 1, 1);
        mma_commit(mma_bar);
      }
      if (half == 0) {
        if (warp == 1) issue_raw(cur, 1);
        raw_inflight = true;
        raw_pending = raw_phase;
      }
      if (half == 1 && has_next && tid < C) beta_next = load_beta(nxt);
    }
    // ---- P16: the A products of both halves
    wait_mma();
    __syncthreads();
    if (*sAbort) goto done;
    tc_fence_after();
    // ---- P3: beta A_kk (fp32, strict) to smem; A_qk (inclusive) to the item ----
    {
      const int r = L & 63;
      const bool is_q = L >= 64;
      const int bme = r >> 4;
      const int np = piece_count(quad);
      for (int pi = sub; pi < np; pi += 4) {
        float v[2][16];
        int bb[2], pp[2];
        piece(quad, pi, bb[0], pp[0]);
        const bool two = pi + 2 < np;
        if (two) {
          piece(quad, pi + 2, bb[1], pp[1]);
          tmem_ld16x2(tq + tm_a(bb[0]) + 16 * pp[0], tq + tm_a(bb[1]) + 16 * pp[1], v[0], v[1]);
        } else {
          bb[1] = -1;
          pp[1] = 0;
          tmem_ld16(tq + tm_a(bb[0]) + 16 * pp[0], v[0]);
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          if (bb[e] != bme) continue;
          const int j0 = 16 * pp[e];
          if (!is_q) {
            const float br = sBeta[r];
            float4 *dst = reinterpret_cast<float4 *>(sAkk + r * LDF + j0);
            float4 *raw = reinterpret_cast<float4 *>(gi + I_AKK + (r * C + j0) * 4);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              float a[4];
#pragma unroll
              for (int i = 0; i < 4; ++i)
                a[i] = (j0 + 4 * q4 + i < r) ? v[e][4 * q4 + i] : 0.f;
              if (bwd_items) raw[q4] = make_float4(a[0], a[1], a[2], a[3]);
              dst[q4] = make_float4(br * a[0], br * a[1], br * a[2], br * a[3]);
            }
          } else {
            float a0[8], a1[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              a0[i] = (j0 + i <= r) ? p.scale * v[e][i] : 0.f;
              a1[i] = (j0 + 8 + i <= r) ? p.scale * v[e][8 + i] : 0.f;
            }
            st_g16(gi, I_AQK + op_off(r, j0, C), a0);
            st_g16(gi, I_AQK + op_off(r, j0 + 8, C), a1);
          }
        }
      }
      if (is_q && sub == 0) {
        const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int jj = 16 * (bme + 1); jj < C; jj += 8) st_g16(gi, I_AQK + op_off(r, jj, C), z);
      }
    }
    tc_fence_before();
    __syncthreads();

    // ---- P4: T = (I + beta A_kk)^-1, blocked fp32: diagonal blocks ----
    if (tid < 64) {
      const int i = tid >> 4, cc = tid & 15, base = 16 * i;
      float x[16];
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) x[rr] = rr == cc ? 1.f : 0.f;
#pragma unroll
      for (int m = 0; m < 15; ++m) {
        const float xm = x[m];
#pragma unroll
        for (int rr = m + 1; rr < 16; ++rr)
          x[rr] = fmaf(-sAkk[(base + rr) * LDF + base + m], xm, x[rr]);
      }
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) sT[(base + rr) * LDF + base + cc] = x[rr];
    }
    __syncthreads();
    // ---- P7: off-diagonal blocks of T.  With D = blockdiag(I + N_ii) and L
    //      the blocks below it, T = (I + D^-1 L)^-1 D^-1; with Nt = D^-1 L
    //      (Nt_ij = T_ii N_ij) and R = (I + Nt)^-1 (R_ij = -sum_m Nt_im R_mj),
    //      T_ij = R_ij T_jj.  Four steps of independent 16 x 16 products,
    //      one warp each.
    {
      const int pr = warp, e = lane;
      auto Tb = [&](int i, int j) { return sT + 16 * i * LDF + 16 * j; };
      auto Sc = [&](int k) { return sScr + k * 16 * LDS; };
      if (pr < 6) {  // Nt_ij for (1,0) (2,1) (3,2) (2,0) (3,1) (3,0)
        const int i = pr < 3 ? pr + 1 : (pr < 5 ? pr - 1 : 3);
        const int j = pr < 3 ? pr : (pr < 5 ? pr - 3 : 0);
        blk_prod(Sc(pr), LDS, Tb(i, i), LDF, sAkk + 16 * i * LDF + 16 * j, LDF, 1.f, nullptr, 0, e);
      }
      __syncthreads();
      if (pr < 3) {          // T_{i,i-1} = -Nt_{i,i-1} T_{i-1,i-1}
        blk_prod(Tb(pr + 1, pr), LDF, Sc(pr), LDS, Tb(pr, pr), LDF, -1.f, nullptr, 0, e);
      } else if (pr == 3) {  // R_20 = Nt_21 Nt_10 - Nt_20
        blk_prod(Sc(6), LDS, Sc(1), LDS, Sc(0), LDS, 1.f, Sc(3), LDS, e);
      } else if (pr == 4) {  // R_31 = Nt_32 Nt_21 - Nt_31
        blk_prod(Sc(7), LDS, Sc(2), LDS, Sc(1), LDS, 1.f, Sc(4), LDS, e);
      } else if (pr == 5) {  // Nt_31 Nt_10 - Nt_30 (first two terms of R_30)
        blk_prod(Sc(8), LDS, Sc(4), LDS, Sc(0), LDS, 1.f, Sc(5), LDS, e);
      }
      __syncthreads();
      if (pr == 0) {         // T_20 = R_20 T_00
        blk_prod(Tb(2, 0), LDF, Sc(6), LDS, Tb(0, 0), LDF, 1.f, nullptr, 0, e);
      } else if (pr == 1) {  // T_31 = R_31 T_11
        blk_prod(Tb(3, 1), LDF, Sc(7), LDS, Tb(1, 1), LDF, 1.f, nullptr, 0, e);
      } else if (pr == 2) {  // R_30 = (Nt_31 Nt_10 - Nt_30) - Nt_32 R_20
        blk_prod(Sc(9), LDS, Sc(2), LDS, Sc(6), LDS, -1.f, Sc(8), LDS, e, 1.f);
      }
      __syncthreads();
      if (pr == 0)           // T_30 = R_30 T_00
        blk_prod(Tb(3, 0), LDF, Sc(9), LDS, Tb(0, 0), LDF, 1.f, nullptr, 0, e);
      __syncthreads();
    }
    // ---- P8: T diag(beta) to bf16 (beta folds into T's columns, so the
    //      right-hand sides are K e^G and V as loaded) ----
    {
      const int rl8 = tid & 7, jc = (tid >> 3) & 3, r = 8 * (tid >> 5) + rl8;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j8 = 16 * jc + 8 * e;
        const float4 *src = reinterpret_cast<const float4 *>(sT + r * LDF + j8);
        const float4 a = src[0], b4 = src[1];
        float t8[8] = {a.x, a.y, a.z, a.w, b4.x, b4.y, b4.z, b4.w};
        const bool upper = (j8 >> 4) > (r >> 4);
        if (bwd_items) {  // T itself, for the backward
#pragma unroll
          for (int i = 0; i < 8; ++i) t8[i] = upper ? 0.f : t8[i];
          st_g16(gi, I_T + op_off(r, j8, C), t8);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) t8[i] = upper ? 0.f : t8[i] * sBeta[j8 + i];
        st_bf16x8(smem, P_TB + op_off(r, j8, C), t8);
      }
    }
    // v of this item
    v_inflight = true;
    if (!mbar_wait(v_bar, v_phase)) abort_all();
    else v_inflight = false;
    v_phase ^= 1u;
    if (n < C) {  // rows past the chunk's end: zero (they may hold anything)
      const int m = C - n;
      for (int i = tid; i < (VD / 8) * m; i += PT) {
        const int grp = i / m, rr = n + i % m;
        *reinterpret_cast<uint4 *>(smem + P_V + mn_off(8 * grp, rr, C)) =
            make_uint4(0u, 0u, 0u, 0u);
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    if (*sAbort) goto done;

    // ---- P5: w^T = (K e^G)^T (T diag(beta))^T (TMEM columns 0..63, lanes =
    //      channels) and u = T diag(beta) V (columns 64..191, lanes 0..63 =
    //      rows; rows 64..127 of its A operand are ignored) ----
    if (tid == kIssuer) {
      tc_fence_after();
      mma_group(tmem, sb + P_KT, sb + P_TB, C, C, false, 0, 0);
      mma_group(tmem + C, sb + P_TB, sb + P_V, C, VD, false, 0, 1);
      mma_commit(mma_bar);
    }
    if (has_next) {  // RAW and the solver buffers are free: next item's q, k, g
      if (warp == 0) issue_raw(nxt, 0);
      raw_inflight = true;
      raw_pending = raw_phase;
    }
    wait_mma();
    if (has_next) {  // V has been read: next item's v
      if (warp == 1) issue_v(nxt);
      v_inflight = true;
      v_pending = v_phase;
    }
    tc_fence_after();
    // ---- P9: w (rows 0..63 of [w ; Q e^G], MN-major) and u out of TMEM
    {
      const int r0 = 32 * sub;  // rows r0 .. r0 + 31 of channel L
      float v0[16], v1[16];
      tmem_ld16x2(tq + r0, tq + r0 + 16, v0, v1);
#pragma unroll
      for (int o = 0; o < 4; ++o) {
        float a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = (o < 2 ? v0 : v1)[8 * (o & 1) + i];
        st_g16(gi, I_WQ + mn_off(r0 + 8 * o, L, KD), a);
      }
    }
    if (quad < 2) {  // lanes 0..63: chunk rows; 2 warps share the 8 u pieces
      const int r = L;
#pragma unroll
      for (int k2 = 0; k2 < 2; ++k2) {
        const int p0 = sub + 4 * k2, p1 = p0 + 2;  // pieces of 16 columns
        float v0[16], v1[16];
        tmem_ld16x2(tq + C + 16 * p0, tq + C + 16 * p1, v0, v1);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int col = 16 * (e ? p1 : p0), vt = col >> 5, cv = col & 31;
          const float *vv = e ? v1 : v0;
          unsigned char *dst = gi + I_U + u_off(vt, cv, r);
          *reinterpret_cast<uint4 *>(dst) =
              make_uint4(pack_bf16(vv[0], vv[1]), pack_bf16(vv[2], vv[3]),
                         pack_bf16(vv[4], vv[5]), pack_bf16(vv[6], vv[7]));
          *reinterpret_cast<uint4 *>(dst + 1024) =
              make_uint4(pack_bf16(vv[8], vv[9]), pack_bf16(vv[10], vv[11]),
                         pack_bf16(vv[12], vv[13]), pack_bf16(vv[14], vv[15]));
        }
      }
    }
    tc_fence_before();
    __syncthreads();
    cur = nxt;
  }

done:
  if (raw_inflight) mbar_wait(raw_bar, raw_pending);
  if (v_inflight) mbar_wait(v_bar, v_pending);
  if (mma_inflight) mbar_wait(mma_bar, mma_pending);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ---- recurrence kernel --------------------------------------------------------
// One CTA per (run, head, VTR-column value tile), WPQ warps per TMEM lane
// quadrant, each owning VTR / WPQ of the tile's value columns (warp w:
// quadrant w % 4, columns (VTR / WPQ) (w / 4) ..).  VTR is 32, 64 or 128;
// a wider tile pulls each item from L2 fewer times and does more work per
// MMA instruction at the same MMA latency (an M = 128, K = 16 step takes
// about as long for N = 32 as for N = 128), so VTR = 128 (one CTA per run
// and head, 16 warps) reads every item exactly once.
// One stage mirrors the item's start: [w ; Q e^G] | A_qk | (K e^{G_C-G})^T
// (one copy), then this unit's u columns (VTR / 32 tiles of 64 x 32 bf16)
// and e^{G_C}.  A_qk is read as the 128-row A operand starting 64 rows
// before it: those rows (the tail of Q e^G) only feed D1 rows 0..63, which
// are dead once U is formed.
// Chunk-parallel state scan (rows without segment ids): each row's chunks
// are cut into n_segs segments of cps chunks.  The chunk form is affine in
// the state entering a chunk, S' = (diag(e^{G_C}) - (K e^{G_C-G})^T w) S +
// (K e^{G_C-G})^T u, so a segment maps its entering state to
// S_end = M S_start + B.  The map pass (MAP = 1) runs the recurrence of
// segments 0 .. n_segs - 2 on X = [B | M] (K x (V + K)) from [0 | I], with
// u replaced by [u | 0] and no outputs, and writes X to `maps`
// [B][n_segs - 1][H][K][V + K]; scan_combine_kernel chains
// S_start(s + 1) = M_s S_start(s) + B_s into `starts` [B][n_segs][H][K][V];
// the finish pass (MAP = 0) runs every segment from its S_start, writing o
// and, for the last segment, the final state.  n_segs = 0: no scan.
struct ScanParams {
  int n_segs, cps;
  float *maps;
  float *starts;
  // Saves for the backward (MODE = 2, or MODE = 0 when set): per (chunk,
  // head), at the item's index, SV_BYTES holding the state entering the
  // chunk and U (bf16).
  unsigned char *save;
};

constexpr uint32_t S_WQ = I_WQ, S_AQK = I_AQK, S_KHT = I_KHT, S_U = I_U;
static_assert(S_WQ == 0 && S_AQK == 32768 && S_KHT == S_AQK + 8192 && S_U == S_KHT + 16384,
              "stage layout");
template <int VTR, int NST>
struct RecLayout {
  static constexpr int WPQ = VTR == 128 ? 4 : 2;                // warps per lane quadrant
  static constexpr int THREADS = 128 * WPQ;
  static constexpr int CPT = VTR / WPQ;                         // value columns per thread
  static constexpr int NT = VTR / VT;                           // u tiles per unit
  static constexpr uint32_t S_GAM = S_U + 4096u * NT;
  static constexpr uint32_t S_BYTES = S_GAM + 512;               // copied per stage
  static constexpr uint32_t STAGE = (S_BYTES + 1023) / 1024 * 1024;
  static constexpr uint32_t ST = NST * STAGE;                   // S^T MN-major VTR x Kd 128
  static constexpr uint32_t UT = ST + 256u * VTR;               // U^T MN-major VTR x Kd 64
  static constexpr uint32_t BAR = UT + 128u * VTR;              // stages, d1, s, o
  static constexpr uint32_t SLOT = BAR + 8 * (NST + 3);
  static constexpr uint32_t ABORT = SLOT + 4;
  static constexpr uint32_t ALLOC = ABORT + 12 + 1024;
  // TMEM: D1 double-buffered (chunk parity) so the o rows of chunk n are read
  // while the first MMA of chunk n + 1 runs; D2 single.
  static constexpr uint32_t TM_D1 = 0, TM_D2 = 2 * VTR;
  static constexpr uint32_t TM_COLS = 3 * VTR <= 128 ? 128 : (3 * VTR <= 256 ? 256 : 512);
  static_assert(CPT == 16 || CPT == 32, "columns per thread");
  static_assert(ALLOC <= 232448, "rec smem fits");
};

// Per chunk, three MMA groups, each committed to its own mbarrier:
//   D1  = [w ; Q e^G] S          (d1 barrier; U = u - D1[0:64] follows)
//   D2  = (K e^{G_C-G})^T U       (s barrier; the state update follows)
//   D1 += [* ; A_qk] U            (o barrier; only the o rows wait for it)
// D2 is issued before the o product, so the state update, and with it the
// next chunk's first MMA, waits only for the products on the serial chain;
// the o product runs on the tensor pipe while the CUDA cores update S.
// MODE 0: the forward (which also saves like MODE 2 when sc.save is set);
// 1: the scan's map pass (see ScanParams); 2: the backward's save pass (no
// outputs; each chunk's entering state and U are written to sc.save).
template <int VTR, int NST, int MODE>
__global__ void __launch_bounds__(RecLayout<VTR, NST>::THREADS, 1)
    fwd_rec_kernel(const FwdParams p, const unsigned char *items, const ChunkTable ct,
                   const ScanParams sc) {
  using Lay = RecLayout<VTR, NST>;
  constexpr int CPT = Lay::CPT;
  constexpr int NVT_V = VD / VTR;  // tiles of V; map tiles past them are M's columns
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  volatile uint32_t *sAbort = reinterpret_cast<volatile uint32_t *>(smem + Lay::ABORT);
  const uint32_t bar0 = sb + Lay::BAR;
  const uint32_t d1_bar = bar0 + 8 * NST, s_bar = d1_bar + 8, o_bar = d1_bar + 16;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, grp = warp >> 2;
  const int L = 32 * quad + lane;   // TMEM lane: chunk row (0..63) / o row / key row
  const int col0 = CPT * grp;       // this thread's value columns within the tile
  const int H = p.H, T = p.T;
  // The thread that issues the stage refills: lane 0 of the first warp of
  // quadrant 2, which waits for the o product (the last reader of a stage).
  constexpr int kRefillTid = 64;
#ifndef KDA_REC_PREFETCH
#define KDA_REC_PREFETCH 2
#endif
  // Items are also pulled into L2 this many chunks ahead of their stage
  // copy, so the copies hit L2 instead of waiting on DRAM.
  constexpr int kRecPrefetch = KDA_REC_PREFETCH;

  if (warp == 0) tmem_alloc(sb + Lay::SLOT, Lay::TM_COLS);
  if (tid == 0) {
    for (int i = 0; i < NST; ++i) mbar_init(bar0 + 8u * i, 1);
    mbar_init(d1_bar, 1);
    mbar_init(s_bar, 1);
    mbar_init(o_bar, 1);
    *sAbort = 0u;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + Lay::SLOT);
  const uint32_t tq = tmem + ((uint32_t)(32 * quad) << 16);
  uint32_t st_phase[NST] = {};
  uint32_t st_issued = 0;  // per-stage bit: copy issued and not yet waited
  // Completions of each MMA barrier this thread has waited for (the k-th
  // completion has parity k & 1), and, for the issuing thread 0, the
  // barrier and completion index of its last commit (drained on abort).
  uint32_t n_d1 = 0, n_s = 0, n_o = 0;
  uint32_t c_d1 = 0, c_s = 0, c_o = 0;  // commits issued (thread 0)
  uint32_t last_bar = 0, last_k = 0;
  bool committed = false;
  auto abort_all = [&]() {
    *sAbort = 1u;
    set_status(p.status, KDA_DEVICE_TIMEOUT);
  };
  auto issue_stage = [&](int s, const unsigned char *src, int vt) {
    const uint32_t dst = sb + (uint32_t)s * Lay::STAGE;
    const uint32_t bar = bar0 + 8u * (uint32_t)s;
    mbar_expect_tx(bar, Lay::S_BYTES);
    bulk_load(dst, src, S_U, bar);  // [w ; Q e^G] | A_qk | K^T
    bulk_load(dst + S_U, src + I_U + (size_t)vt * (4096u * Lay::NT), 4096u * Lay::NT, bar);
    bulk_load(dst + Lay::S_GAM, src + I_GAM, 512, bar);
  };
  auto wait_stage = [&](int s) {
    if (!mbar_wait(bar0 + 8u * s, st_phase[s])) abort_all();
    else st_issued &= ~(1u << s);
    st_phase[s] ^= 1u;
  };
  auto wait_bar = [&](uint32_t bar, uint32_t &n) {
    if (!mbar_wait(bar, n & 1u)) abort_all();
    ++n;
  };
  auto commit = [&](uint32_t bar, uint32_t &c) {  // thread 0
    mma_commit(bar);
    last_bar = bar;
    last_k = c++;
    committed = true;
  };
  // CPT consecutive fp32 TMEM columns of this thread's lane.
  auto tmem_ld_cpt = [&](uint32_t taddr, float (&v)[CPT]) {
    if constexpr (CPT == 16) {
      tmem_ld16(taddr, v);
    } else {
      float a[16], b[16];
      tmem_ld16x2(taddr, taddr + 16, a, b);
#pragma unroll
      for (int i = 0; i < 16; ++i) { v[i] = a[i]; v[16 + i] = b[i]; }
    }
  };
  auto store_st = [&](const float (&S)[CPT], int key) {  // S^T bf16, MN-major
#pragma unroll
    for (int e = 0; e < CPT / 8; ++e) {
      float t8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) t8[i] = S[8 * e + i];
      st_bf16x8(smem, Lay::ST + mn_off(col0 + 8 * e, key, KD), t8);
    }
  };

  float S[CPT];  // S[key row L][col0 .. col0 + CPT - 1], fp32
  const bool fits = total_chunk_count(ct, p.B) <= ct.capacity;
  constexpr bool MAP = MODE == 1, SAVE = MODE == 2;
  // the forward also saves for the backward when given a save area
  const bool save_on = SAVE || (MODE == 0 && sc.save != nullptr);
  const int seg_units = MAP ? sc.n_segs - 1 : sc.n_segs;
  const uint32_t n_units =
      !fits ? 0u
            : sc.n_segs > 0 ? (uint32_t)seg_units * (uint32_t)p.B * (uint32_t)H * (uint32_t)p.n_vtiles
                            : total_units(p.runs, p.B, H, p.n_vtiles);
  for (uint32_t unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    int vt, h, b, ustart, uend, seg = 0;
    bool ufirst, ulast;
    uint32_t cbase;
    if (sc.n_segs > 0) {  // (segment, row, head, tile), rows without segment ids
      uint32_t x = unit;
      vt = (int)(x % (uint32_t)p.n_vtiles);
      x /= (uint32_t)p.n_vtiles;
      h = (int)(x % (uint32_t)H);
      x /= (uint32_t)H;
      b = (int)(x % (uint32_t)p.B);
      seg = (int)(x / (uint32_t)p.B);
      const int c0 = seg * sc.cps, c1 = min(c0 + sc.cps, ct.n_chunks_row);
      ustart = c0 * C;
      uend = min(c1 * C, T);
      ufirst = seg == 0;
      ulast = seg == sc.n_segs - 1;
      cbase = (uint32_t)b * ct.n_chunks_row + (uint32_t)c0;
    } else {
      const Unit u = decode_unit(p.runs, unit, p.B, T, H, p.n_vtiles);
      vt = u.vt; h = u.h; b = u.b;
      ustart = u.start; uend = u.end;
      ufirst = u.first; ulast = u.last;
      cbase = ct.run_chunk_base
          ? (uint32_t)(ct.chunk_row_offsets[b] + ct.run_chunk_base[(size_t)b * T + u.run_in_row])
          : (uint32_t)b * ct.n_chunks_row;
    }
    const int vc0 = vt * VTR;
    const int n_chunks = uend > ustart ? (uend - ustart + C - 1) / C : 0;
    if (n_chunks == 0) continue;
    // map pass: the tiles of M read no u (its columns of [u | 0] are zero)
    const bool m_tile = MAP && vt >= NVT_V;
    const int vt_u = m_tile ? 0 : vt;
    auto item_ptr = [&](int c) {
      return items + ((size_t)(cbase + c) * H + h) * ct.item_stride;
    };
    // the first stages' copies go out before the entering state's load, so
    // the two latencies overlap (the previous unit's readers of the stages
    // and of S^T finished before its closing barrier)
    if (tid == 0) {
      for (int c = 0; c < NST && c < n_chunks; ++c) issue_stage(c, item_ptr(c), vt_u);
      for (int c = NST; c < NST + kRecPrefetch && c < n_chunks; ++c) prefetch_l2(item_ptr(c), ITEM_BYTES);
    }
    // state entering the run (or segment); S^T operand (MN-major: v contiguous)
    const float *s_src = nullptr;
    if (!MAP) {
      if (ufirst) s_src = p.initial_state
          ? p.initial_state + (((size_t)b * H + h) * KD + L) * p.V + vc0 + col0 : nullptr;
      else if (sc.n_segs > 0)
        s_src = sc.starts + ((((size_t)b * sc.n_segs + seg) * H + h) * KD + L) * p.V + vc0 + col0;
    }
    if (s_src) {
      const float4 *src = reinterpret_cast<const float4 *>(s_src);
#pragma unroll
      for (int q4 = 0; q4 < CPT / 4; ++q4) {
        const float4 x = src[q4];
        S[4 * q4] = x.x; S[4 * q4 + 1] = x.y; S[4 * q4 + 2] = x.z; S[4 * q4 + 3] = x.w;
      }
    } else if (m_tile) {  // identity columns of M
#pragma unroll
      for (int i = 0; i < CPT; ++i) S[i] = (L == (vt - NVT_V) * VTR + col0 + i) ? 1.f : 0.f;
    } else {
#pragma unroll
      for (int i = 0; i < CPT; ++i) S[i] = 0.f;
    }
    store_st(S, L);
    st_issued = (1u << (NST < n_chunks ? NST : n_chunks)) - 1u;
    fence_proxy_async();
    wait_stage(0);
    tc_fence_before();
    __syncthreads();
    if (*sAbort) goto done;
    // ---- P11: D1[0] = [w ; Q e^G] S for chunk 0
    if (tid == 0) {
      tc_fence_after();
      mma_group(tmem + Lay::TM_D1, sb + S_WQ, sb + Lay::ST, KD, VTR, false, 1, 1);
      commit(d1_bar, c_d1);
    }

    int s = 0;  // stage of chunk c
    for (int c = 0; c < n_chunks; ++c) {
      const int s1 = s + 1 == NST ? 0 : s + 1;  // stage of chunk c + 1
      const int t0 = ustart + c * C;
      const int n = min(C, uend - t0);
      const size_t tok0 = (size_t)b * T + t0;
      const unsigned char *stg = smem + (uint32_t)s * Lay::STAGE;
      const uint32_t sstg = sb + (uint32_t)s * Lay::STAGE;
      const uint32_t d1 = Lay::TM_D1 + (uint32_t)VTR * (uint32_t)(c & 1);
      unsigned char *sv = save_on ? sc.save + ((size_t)(cbase + c) * H + h) * SV_BYTES : nullptr;
      if (save_on) {  // the state entering this chunk
#pragma unroll
        for (int e = 0; e < CPT / 8; ++e) {
          float t8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) t8[i] = S[8 * e + i];
          st_g16(sv, SV_S + op_off(L, vc0 + col0 + 8 * e, KD), t8);
        }
      }
      // ---- P10: wait for D1 = [w ; Q e^G] S of this chunk (every thread
      //      waits on the barrier itself; an abort is seen after the next
      //      block barrier, which also keeps the phases in step)
      wait_bar(d1_bar, n_d1);
      tc_fence_after();

      // ---- P12: U = u - w S (lanes 0..63)
      if (quad < 2) {
        const int r = L;
        float v[CPT];
        tmem_ld_cpt(tq + d1 + col0, v);
#pragma unroll
        for (int e = 0; e < CPT / 8; ++e) {
          const int col = col0 + 8 * e;
          float uu[8], a[8];
          if (m_tile) {
#pragma unroll
            for (int i = 0; i < 8; ++i) uu[i] = 0.f;
          } else {
            ld_bf16x8(stg + S_U + u_off(col >> 5, col & 31, r), uu);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) a[i] = uu[i] - v[8 * e + i];
          st_bf16x8(smem, Lay::UT + mn_off(col, r, C), a);
          if (save_on) st_g16(sv, SV_U + op_off(r, vc0 + col, KD), a);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();
      if (*sAbort) goto done;

      // ---- P13: D2 = (K e^{G_C-G})^T U (the chain), then D1 += [* ; A_qk] U
      if (tid == 0) {
        tc_fence_after();
        mma_group(tmem + Lay::TM_D2, sstg + S_KHT, sb + Lay::UT, C, VTR, false, 0, 1);
        commit(s_bar, c_s);
        if (MODE == 0) mma_group(tmem + d1, sstg + S_AQK - 8192, sb + Lay::UT, C, VTR, true, 0, 1);
        commit(o_bar, c_o);  // without the o product this tracks D2
      }
      wait_bar(s_bar, n_s);
      tc_fence_after();

      // ---- P14: state update (all lanes = key rows), next chunk's first MMA
      {
        const float gam = reinterpret_cast<const float *>(stg + Lay::S_GAM)[L];
        float v[CPT];
        tmem_ld_cpt(tq + Lay::TM_D2 + col0, v);
#pragma unroll
        for (int i = 0; i < CPT; ++i) S[i] = fmaf(gam, S[i], v[i]);
        store_st(S, L);
      }
      // Refill stage s as early as possible: when the o product (its last
      // reader) is already done, now; else after the o rows wait for it.
      bool refilled = false;
      if (tid == kRefillTid && c + NST < n_chunks && mbar_try_wait(o_bar, n_o & 1u)) {
        tc_fence_after();
        issue_stage(s, item_ptr(c + NST), vt_u);
        if (c + NST + kRecPrefetch < n_chunks) prefetch_l2(item_ptr(c + NST + kRecPrefetch), ITEM_BYTES);
        refilled = true;
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();
      if (*sAbort) goto done;
      if (c + 1 < n_chunks) {
        wait_stage(s1);
        if (tid == 0) {
          tc_fence_after();
          mma_group(tmem + Lay::TM_D1 + (uint32_t)VTR * (uint32_t)((c + 1) & 1),
                    sb + (uint32_t)s1 * Lay::STAGE + S_WQ, sb + Lay::ST, KD, VTR, false, 1, 1);
          commit(d1_bar, c_d1);
        }
      }
      // o rows of this chunk (lanes 64..127) while the next MMA runs; the o
      // product is the last reader of stage s, so the refill follows it
      if (quad >= 2) {
        wait_bar(o_bar, n_o);
        tc_fence_after();
        if (tid == kRefillTid && !refilled && c + NST < n_chunks) {
          issue_stage(s, item_ptr(c + NST), vt_u);
          if (c + NST + kRecPrefetch < n_chunks) prefetch_l2(item_ptr(c + NST + kRecPrefetch), ITEM_BYTES);
        }
        const int r = L - 64;
        float v[CPT];
        if (MODE == 0) tmem_ld_cpt(tq + d1 + col0, v);
        if (MODE == 0 && r < n) {
          uint4 *dst = reinterpret_cast<uint4 *>(
              static_cast<__nv_bfloat16 *>(p.o) + ((tok0 + r) * H + h) * p.V + vc0 + col0);
#pragma unroll
          for (int e = 0; e < CPT / 8; ++e) {
            uint4 w;
            w.x = pack_bf16(v[8 * e + 0], v[8 * e + 1]);  // D1's o rows carry the scale
            w.y = pack_bf16(v[8 * e + 2], v[8 * e + 3]);
            w.z = pack_bf16(v[8 * e + 4], v[8 * e + 5]);
            w.w = pack_bf16(v[8 * e + 6], v[8 * e + 7]);
            dst[e] = w;
          }
        }
      }
      if (c + NST < n_chunks) st_issued |= 1u << s;
      tc_fence_before();
      s = s1;
    }
    float *s_dst = nullptr;
    if (MAP)
      s_dst = sc.maps + ((((size_t)b * (sc.n_segs - 1) + seg) * H + h) * KD + L) * (VD + KD) +
              vc0 + col0;
    else if (!SAVE && ulast && p.final_state)
      s_dst = p.final_state + (((size_t)b * H + h) * KD + L) * p.V + vc0 + col0;
    if (s_dst) {
      float4 *dst = reinterpret_cast<float4 *>(s_dst);
#pragma unroll
      for (int q4 = 0; q4 < CPT / 4; ++q4)
        dst[q4] = make_float4(S[4 * q4], S[4 * q4 + 1], S[4 * q4 + 2], S[4 * q4 + 3]);
    }
    __syncthreads();
  }

done:
  // Drain this thread's copies and (thread 0) its last MMA commit, each
  // wait bounded, before TMEM is freed.
  for (int s = 0; s < NST; ++s)
    if (st_issued & (1u << s)) mbar_wait(bar0 + 8u * s, st_phase[s]);
  if (tid == 0 && committed) mbar_wait(last_bar, last_k & 1u);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::TM_COLS);
  }
}

// S_start(s + 1) = M_s S_start(s) + B_s for s = 0 .. n_segs - 2, in fp32:
// one CTA per (row, head, 8 columns of S), each thread rows r, r + 64 by two
// columns (r = tid / 4); S_start(0) is the initial state (or zero).  M_s is
// staged in shared memory by 16-byte cp.async copies, the next step's while
// this one computes (two buffers); its rows are padded to 132 floats (16-byte
// rows for the copies; the 8 rows a warp reads per step fall in distinct
// banks).  Each output accumulates B_s, then m = 0 .. K-1 in order.
constexpr int kCombCols = 8;
constexpr int kCombLd = KD + 4;
constexpr uint32_t kCombSmem = (uint32_t)(2 * KD * kCombLd + KD * kCombCols) * 4;
static_assert((kCombLd * 4) % 16 == 0, "16-byte rows for cp.async");

__device__ __forceinline__ void comb_cp16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void comb_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

__global__ void __launch_bounds__(256)
    scan_combine_kernel(const FwdParams p, const ScanParams sc) {
  extern __shared__ __align__(16) float csm[];
  float *sM = csm;                          // M_s, two buffers [2][KD][kCombLd]
  float *sS = csm + 2 * KD * kCombLd;       // S_start(s)[:, tile] [KD][kCombCols]
  const int tile = blockIdx.x % (VD / kCombCols), bh = blockIdx.x / (VD / kCombCols);
  const int h = bh % p.H, b = bh / p.H;
  const int tid = threadIdx.x, r0 = tid >> 2, c0 = 2 * (tid & 3);
  const int col = kCombCols * tile;
  auto map_of = [&](int s) {
    return sc.maps + (((size_t)b * (sc.n_segs - 1) + s) * p.H + h) * KD * (VD + KD);
  };
  auto prefetch = [&](int s, int buf) {  // M_s = map[:, VD:] into buffer buf
    const float *map = map_of(s);
    float *dst = sM + buf * KD * kCombLd;
    for (int i = tid; i < KD * KD / 4; i += 256) {
      const int kk = i / (KD / 4), m4 = i % (KD / 4);
      comb_cp16(smem_u32(dst + kk * kCombLd + 4 * m4), map + (size_t)kk * (VD + KD) + VD + 4 * m4);
    }
    comb_commit();
  };
  for (int i = tid; i < KD * kCombCols; i += 256) {
    const int kk = i / kCombCols, cc = i % kCombCols;
    sS[i] = p.initial_state
                ? p.initial_state[(((size_t)b * p.H + h) * KD + kk) * VD + col + cc]
                : 0.f;
  }
  if (sc.n_segs > 1) prefetch(0, 0);
  for (int s = 0; s + 1 < sc.n_segs; ++s) {
    const int buf = s & 1;
    // the next step's M (its buffer was last read before the previous
    // step's closing barrier); then wait for this step's copies
    if (s + 2 < sc.n_segs) {
      prefetch(s + 1, buf ^ 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    const float *map = map_of(s);
    float acc[2][2];
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {  // B_s
      const float2 x = *reinterpret_cast<const float2 *>(
          map + (size_t)(r0 + 64 * rr) * (VD + KD) + col + c0);
      acc[rr][0] = x.x; acc[rr][1] = x.y;
    }
    __syncthreads();  // every thread's copies of M_s landed; sS of this step written
    const float *M = sM + buf * KD * kCombLd;
#pragma unroll 8
    for (int m = 0; m < KD; ++m) {
      const float2 sv = *reinterpret_cast<const float2 *>(sS + m * kCombCols + c0);
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const float mv = M[(r0 + 64 * rr) * kCombLd + m];
        acc[rr][0] = fmaf(mv, sv.x, acc[rr][0]);
        acc[rr][1] = fmaf(mv, sv.y, acc[rr][1]);
      }
    }
    __syncthreads();  // every thread has read sS and this buffer of M
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const int r = r0 + 64 * rr;
      const float2 x = make_float2(acc[rr][0], acc[rr][1]);
      *reinterpret_cast<float2 *>(sS + r * kCombCols + c0) = x;
      *reinterpret_cast<float2 *>(
          sc.starts + ((((size_t)b * sc.n_segs + s + 1) * p.H + h) * KD + r) * VD + col + c0) = x;
    }
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

}  // namespace

bool split::make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int esize,
                     uint64_t cols, uint64_t rows, uint32_t box_cols, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * (uint64_t)esize};
  const cuuint32_t box[2] = {box_cols, (cuuint32_t)C};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// Byte offset of the first item: after the header (no segment ids) or after
// the run list and the chunk tables (segment ids).
size_t split::items_offset(int B, int T, bool has_seg) {
  return has_seg ? align_up(ws_bytes(B, T, true) + ws_chunk_tables_bytes(B, T), 1024)
                 : WS_ITEMS_OFF;
}

size_t split_workspace_bytes(int B, int T, int H, bool has_seg, int max_runs_per_row) {
  const size_t nc = ((size_t)T + C - 1) / C;
  const size_t chunks = has_seg ? (size_t)B * (nc + (size_t)(max_runs_per_row > 0 ? max_runs_per_row : 0))
                                : (size_t)B * nc;
  return items_offset(B, T, has_seg) + chunks * H * ITEM_BYTES;
}

int scan_segments(int B, int T, int H, int n_segs) {
  const int nc = (T + C - 1) / C;
  if (n_segs == 0) {  // as many as the finish pass's 64-column units fit the SMs
    const long units = (long)B * H * (VD / 64);
    n_segs = (int)(num_sms() / (units > 0 ? units : 1));
  }
  if (n_segs < 2) n_segs = 2;
  if (n_segs > nc) n_segs = nc;
  const int cps = (nc + n_segs - 1) / n_segs;
  return (nc + cps - 1) / cps;  // segments that hold at least one chunk
}

size_t scan_workspace_bytes(int B, int T, int H, int n_segs) {
  const int P = scan_segments(B, T, H, n_segs);
  if (P < 2) return 0;
  const size_t maps = (size_t)(P - 1) * B * H * KD * (VD + KD) * 4;
  const size_t starts = (size_t)P * B * H * KD * VD * 4;
  return align_up(split_workspace_bytes(B, T, H, false, 0), 256) + align_up(maps, 256) + starts;
}

bool fwd_split_supported(int K, int V, bool bf16, bool, int v_tile) {
  return bf16 && K == KD && V == VD &&
         (v_tile == 0 || v_tile == 32 || v_tile == 64 || v_tile == 128);
}

// Two stages in flight: a third only lengthens the copies' latency (more
// bytes queued at the same L2 -> SM throughput) and measured slower.
constexpr int kRecStages = 2;
namespace {
template <int VTR, int NST, int MAP>
cudaError_t launch_rec(const FwdParams &p, const unsigned char *items, const ChunkTable &ct,
                       bool has_seg, const ScanParams &sc, cudaStream_t stream) {
  using Lay = RecLayout<VTR, NST>;
  cudaError_t e = cudaFuncSetAttribute(fwd_rec_kernel<VTR, NST, MAP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Lay::ALLOC);
  if (e != cudaSuccess) return e;
  const long sms = num_sms();
  const long rows = sc.n_segs > 0 ? (long)p.B * (MAP ? sc.n_segs - 1 : sc.n_segs) : (long)p.B;
  const long n_units = has_seg ? (long)p.B * p.T * p.H * p.n_vtiles : rows * p.H * p.n_vtiles;
  const int g2 = (int)(n_units < sms ? n_units : sms);
  fwd_rec_kernel<VTR, NST, MAP><<<g2 > 0 ? g2 : 1, Lay::THREADS, Lay::ALLOC, stream>>>(p, items,
                                                                                         ct, sc);
  return cudaGetLastError();
}

template <int MAP>
cudaError_t launch_rec_tile(const FwdParams &p, const unsigned char *items, const ChunkTable &ct,
                            bool has_seg, const ScanParams &sc, cudaStream_t stream) {
  return p.v_tile == 32   ? launch_rec<32, kRecStages, MAP>(p, items, ct, has_seg, sc, stream)
         : p.v_tile == 64 ? launch_rec<64, kRecStages, MAP>(p, items, ct, has_seg, sc, stream)
                          : launch_rec<128, kRecStages, MAP>(p, items, ct, has_seg, sc, stream);
}

// Narrowest value tile (32, 64 or 128 columns) whose `units` per tile
// count, times the tiles of `cols` columns, fits one CTA per SM.
int fit_tile(long units, int cols) {
  const long sms = num_sms();
  if (units * (cols / 32) <= sms) return 32;
  if (units * (cols / 64) <= sms) return 64;
  return 128;
}

// The prep kernel over every item of `ct` (two CTAs per SM).
cudaError_t launch_prep(const FwdParams &p, unsigned char *items, const ChunkTable &ct,
                        cudaStream_t stream) {
  const uint64_t rows = (uint64_t)p.B * p.T;
  CUtensorMap mq, mk, mg, mv;
  // q, k, g unswizzled: the prep kernel's channel owners read one row's 32
  // consecutive channels per warp (128 contiguous bytes of g, 64 of q or k)
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (!make_map(&mq, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)p.H * KD, rows, 64, sw) ||
      !make_map(&mk, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)p.H * KD, rows, 64, sw) ||
      !make_map(&mg, p.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)p.H * KD, rows, 32, sw) ||
      !make_map(&mv, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)p.H * VD, rows, 8,
                CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  const long sms = num_sms();
  cudaError_t e = cudaFuncSetAttribute(fwd_prep_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)P_ALLOC);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fwd_prep_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  const long n_items = (long)ct.capacity * p.H;  // upper bound of the real count
  const int g1 = (int)(n_items < 2 * sms ? n_items : 2 * sms);  // two CTAs per SM
  fwd_prep_kernel<<<g1 > 0 ? g1 : 1, PT, P_ALLOC, stream>>>(p, items, ct, mq, mk, mg, mv);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return cudaSuccess;
}

// The chunk table of a call: items from `ioff` on, `stride` bytes each.
ChunkTable make_table(const FwdParams &p, unsigned char *ws, size_t ioff, size_t bytes,
                      uint32_t stride, bool has_seg, bool with_fallback) {
  ChunkTable ct;
  ct.report_overflow = with_fallback ? 0 : 1;
  ct.n_chunks_row = (p.T + C - 1) / C;
  ct.n_rows = p.B;
  ct.item_stride = stride;
  ct.capacity = (uint32_t)((bytes - ioff) / ((size_t)p.H * stride));
  if (has_seg) {
    ct.run_chunk_base = reinterpret_cast<const int32_t *>(ws + ws_bytes(p.B, p.T, true));
    ct.chunk_row_offsets = reinterpret_cast<const int32_t *>(
        ws + ws_bytes(p.B, p.T, true) + align_up(sizeof(int32_t) * (size_t)p.B * p.T, 256));
    ct.total_chunks = &reinterpret_cast<const WsHeader *>(ws)->total_chunks;
    ct.coords = reinterpret_cast<const int2 *>(ws + ws_chunk_coords_offset(p.B, p.T));
  } else {
    ct.run_chunk_base = nullptr;
    ct.chunk_row_offsets = nullptr;
    ct.coords = nullptr;
    ct.total_chunks = nullptr;
  }
  return ct;
}
}  // namespace

cudaError_t launch_fwd_split(const FwdParams &p_in, void *workspace, size_t workspace_bytes,
                             cudaStream_t stream, bool with_fallback, int scan_segs) {
  const bool has_seg = p_in.runs.runs != nullptr;
  if (!fwd_split_supported(p_in.K, p_in.V, true, has_seg, p_in.v_tile))
    return cudaErrorNotSupported;
  if (scan_segs < 0 || (scan_segs > 0 && has_seg)) return cudaErrorNotSupported;
  FwdParams p = p_in;
  // Recurrence value tile: without segment ids, the narrowest tile whose
  // (row, head, tile) units all run at once, one CTA each (32 columns give
  // the shortest serial chain: the four CTAs of a head share the per-chunk
  // shared-memory traffic); with segment ids (many short runs) 128 columns,
  // which reads each item once and does the most work per MMA.
  const long bh = (long)p.B * p.H, sms = num_sms();
  if (p_in.v_tile != 0) p.v_tile = p_in.v_tile;
  else if (has_seg) p.v_tile = 128;
  else p.v_tile = bh * 4 <= sms ? 32 : (bh * 2 <= sms ? 64 : 128);
  p.n_vtiles = VD / p.v_tile;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  const size_t ioff = items_offset(p.B, p.T, has_seg);
  if (workspace_bytes < ioff + (size_t)p.H * ITEM_BYTES) return cudaErrorInvalidValue;
  unsigned char *items = ws + ioff;
  const ChunkTable ct = make_table(p, ws, ioff, workspace_bytes, ITEM_BYTES, has_seg, with_fallback);
  cudaError_t e = launch_prep(p, items, ct, stream);
  if (e != cudaSuccess) return e;
  ScanParams sc = {0, 0, nullptr, nullptr, nullptr};
  if (scan_segs > 0) {
    // chunk-parallel scan: map pass, combine, finish pass (see ScanParams)
    const int nc = ct.n_chunks_row;
    sc.n_segs = scan_segments(p.B, p.T, p.H, scan_segs);
    sc.cps = (nc + sc.n_segs - 1) / sc.n_segs;
    const size_t items_end = align_up(split_workspace_bytes(p.B, p.T, p.H, false, 0), 256);
    const size_t maps_bytes = align_up((size_t)(sc.n_segs - 1) * p.B * p.H * KD * (VD + KD) * 4, 256);
    if (workspace_bytes < scan_workspace_bytes(p.B, p.T, p.H, scan_segs)) return cudaErrorInvalidValue;
    sc.maps = reinterpret_cast<float *>(ws + items_end);
    sc.starts = reinterpret_cast<float *>(ws + items_end + maps_bytes);
    FwdParams pm = p;
    pm.v_tile = fit_tile((long)p.B * p.H * (sc.n_segs - 1), VD + KD);
    pm.n_vtiles = (VD + KD) / pm.v_tile;
    e = launch_rec_tile<1>(pm, items, ct, false, sc, stream);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(scan_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kCombSmem);
    if (e != cudaSuccess) return e;
    scan_combine_kernel<<<p.B * p.H * (VD / kCombCols), 256, kCombSmem, stream>>>(p, sc);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (p_in.v_tile == 0) p.v_tile = fit_tile((long)p.B * p.H * sc.n_segs, VD);
    p.n_vtiles = VD / p.v_tile;
  }
  e = launch_rec_tile<0>(p, items, ct, has_seg, sc, stream);
  if (e != cudaSuccess || !with_fallback || !has_seg) return e;
  // The fused kernel covers calls whose runs overflow the items (it exits
  // at once when they fit).
  FwdParams pf = p_in;
  pf.gate_chunks = ct.total_chunks;
  pf.gate_capacity = ct.capacity;
  return launch_fwd_tc(pf, stream);
}

// ---- the forward pass the tensor-core backward starts from ------------------
size_t split::bwd_tc_workspace_bytes(int B, int T, int H, bool has_seg, int max_runs_per_row) {
  const size_t nc = ((size_t)T + C - 1) / C;
  const size_t chunks = (size_t)B * (nc + (has_seg && max_runs_per_row > 0 ? (size_t)max_runs_per_row : 0));
  return items_offset(B, T, has_seg) + chunks * H * ((size_t)ITEM_BYTES_BWD + SV_BYTES);
}

// Items of ITEM_BYTES_BWD (the forward's, plus T, A_kk and K e^G), then the
// recurrence in its save mode: the state entering every chunk and U, no o
// and no final state.
bool split::bwd_layout(const FwdParams &p_in, void *workspace, size_t workspace_bytes,
                       BwdLayout *out) {
  const bool has_seg = p_in.runs.runs != nullptr;
  const size_t ioff = items_offset(p_in.B, p_in.T, has_seg);
  const size_t per_chunk = (size_t)p_in.H * ((size_t)ITEM_BYTES_BWD + SV_BYTES);
  if (workspace_bytes < ioff + per_chunk) return false;
  // every row's chunks without segment ids; with them, the chunks of all
  // runs (counted on the device; an overflow is reported, nothing is done)
  const size_t cap = (workspace_bytes - ioff) / per_chunk;
  if (!has_seg && cap < (size_t)p_in.B * ((p_in.T + C - 1) / C)) return false;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  const size_t items_end = ioff + cap * p_in.H * ITEM_BYTES_BWD;
  out->items = ws + ioff;
  out->saves = ws + items_end;
  out->ct = make_table(p_in, ws, ioff, items_end, ITEM_BYTES_BWD, has_seg, false);
  return true;
}

cudaError_t split::launch_fwd_for_bwd(const FwdParams &p_in, void *workspace,
                                      size_t workspace_bytes, BwdLayout *out,
                                      cudaStream_t stream, bool with_outputs) {
  const bool has_seg = p_in.runs.runs != nullptr;
  if (!fwd_split_supported(p_in.K, p_in.V, true, has_seg, 0)) return cudaErrorNotSupported;
  BwdLayout lay;
  if (!bwd_layout(p_in, workspace, workspace_bytes, &lay)) return cudaErrorInvalidValue;
  FwdParams p = p_in;
  if (with_outputs) {  // the forward's own value tile (as launch_fwd_split)
    const long bh = (long)p.B * p.H, sms = num_sms();
    p.v_tile = has_seg ? 128 : (bh * 4 <= sms ? 32 : (bh * 2 <= sms ? 64 : 128));
  } else {
    p.v_tile = has_seg ? 128 : fit_tile((long)p.B * p.H, VD);
    p.o = nullptr;
    p.final_state = nullptr;
  }
  p.n_vtiles = VD / p.v_tile;
  cudaError_t e = launch_prep(p, lay.items, lay.ct, stream);
  if (e != cudaSuccess) return e;
  const ScanParams sc = {0, 0, nullptr, nullptr, lay.saves};
  e = with_outputs ? launch_rec_tile<0>(p, lay.items, lay.ct, has_seg, sc, stream)
                   : launch_rec_tile<2>(p, lay.items, lay.ct, has_seg, sc, stream);
  if (e == cudaSuccess && out) *out = lay;
  return e;
}

}  // namespace kda
