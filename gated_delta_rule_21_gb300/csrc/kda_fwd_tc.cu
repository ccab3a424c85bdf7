// kda_fwd_tc.cu -- chunked KDA forward on the 5th-generation tensor cores
// (tcgen05 MMAs with TMEM accumulators, TMA tile staging), bf16 q/k/v,
// K = V = 128, chunks of 64 tokens.
//
// The method (page "feat(kda): integrate KDA attention with tokamax backend
// and CP support", section "Delta Rule formulation") in the chunk form the
// SIMT kernel also uses.  Per unit = (run, head, 32-column value tile) and per
// chunk of C = 64 rows entering with state S0 (K x 32, fp32 in registers):
//
//   G      = cumsum of g (per channel); block decays D_b = e^{E_b - P_b}
//   X      = [K e1 ; Q e1]                       (128 x 128, A operand)
//   Y_b    = K_{0..16b+15} * e^{P_b - G}         (B operands, one per block)
//   D      = X [Y_0 ; Y_1 ; Y_2 ; Y_3]^T (one MMA, N = 160) -> rows of block
//            b against Y_b: A_kk (k rows), A_qk (q rows)
//   T      = (I + beta * strict(A_kk))^-1        (fp32, blocked, CUDA cores)
//   [w|u]  = [T ; A_qk] [beta K e^{G} | beta V]  (one MMA, N = 160)
//   D1     = [w ; Q e^{G}] S0                    (M = 128: w S0 and Q e^G S0)
//   U      = u - w S0                            (CUDA cores, bf16 operand)
//   D1    += [T ; A_qk] U                        (rows 64..127: O / scale)
//   D2     = (K e^{G_C - G})^T U ;  S1 = e^{G_C} S0 + D2
//
// with e1 = e^{G - P_b}, P_b = G before 16-row block b, E_b = G at its last
// row.  Every factor stays inside bf16/fp32 range for g in [-5, 0]: the
// same-block factor e^{P_b - G} <= e^80, all others <= 1.
//
// All MMAs are tcgen05.mma.cta_group::1.kind::f16 with M = 128, bf16
// operands in shared memory (K-major, no swizzle, 8x16-byte core matrices:
// row groups of 8 rows are contiguous blocks of Kd*16 bytes, the core
// matrices of a row group follow each other every 128 bytes), fp32
// accumulators in TMEM.  One thread issues the MMAs and commits them to an
// mbarrier; every mbarrier wait is bounded and reports a timeout through
// the workspace status word instead of hanging.
//
// Phases run one after another inside the CTA (no warp specialisation); the
// raw tiles of the next chunk are fetched by TMA while the current chunk
// finishes.  256 threads, one CTA per SM (about 219 KB of shared memory),
// all 512 TMEM columns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_internal.cuh"
#include "kda_tc_common.cuh"

namespace kda {
namespace {
using namespace tc;

constexpr int kThreads = 256;
constexpr int C = kChunk;  // 64
constexpr int KD = 128;    // key dim
constexpr int VT = 32;     // value columns per CTA

// ---- shared memory map (byte offsets from a 1024-aligned base) -----------
constexpr uint32_t RAW_Q = 0;                 // 64 x 128 bf16, 256-byte rows
constexpr uint32_t RAW_K = RAW_Q + 16384;
constexpr uint32_t RAW_G = RAW_K + 16384;     // 64 x 128 fp32, 512-byte rows
constexpr uint32_t RAW_V = RAW_G + 32768;     // 64 x 32 bf16, 64-byte rows
constexpr uint32_t RAW_TX_BYTES = 16384 + 16384 + 32768 + 4096;
constexpr uint32_t X_OFF = RAW_V + 4096;      // X: 128 rows x Kd 128
constexpr uint32_t Y_OFF = X_OFF + 32768;     // Y_0..Y_3: 16/32/48/64 rows x 128
constexpr uint32_t ST_OFF = Y_OFF + 160 * 256;  // S^T: 32 rows x Kd 128
constexpr uint32_t WQ_OFF = ST_OFF + 8192;    // [w ; Q e^G]: 128 x 128
constexpr uint32_t KHT_OFF = WQ_OFF + 32768;  // (K e^{G_C-G})^T: 128 x Kd 64
constexpr uint32_t RHST_OFF = KHT_OFF + 16384;  // [beta K e^G | beta V]^T: 160 x 64
constexpr uint32_t MISC_OFF = RHST_OFF + 20480;
constexpr uint32_t BETA_OFF = MISC_OFF;           // 64 fp32
constexpr uint32_t DBLK_OFF = MISC_OFF + 256;     // 4 x 128 fp32 block decays
constexpr uint32_t BAR_OFF = MISC_OFF + 2304;     // two mbarriers
constexpr uint32_t TMEMSLOT_OFF = BAR_OFF + 16;   // u32 TMEM base
constexpr uint32_t ABORT_OFF = TMEMSLOT_OFF + 4;  // u32 abort flag
constexpr uint32_t SMEM_BYTES = ABORT_OFF + 12;
constexpr uint32_t SMEM_ALLOC = SMEM_BYTES + 1024;  // slack for alignment
// Reused after the intra-chunk MMAs are done with X and Y:
constexpr int LDF = C + 4;                        // padded fp32 row stride
constexpr uint32_t AKK_OFF = X_OFF;               // fp32 64 x 65: beta A_kk
constexpr uint32_t TF_OFF = AKK_OFF + 64 * LDF * 4;  // fp32 64 x 65: T
constexpr uint32_t TAQ_OFF = TF_OFF + 64 * LDF * 4;  // [T ; A_qk]: 128 x Kd 64
constexpr uint32_t UT_OFF = TAQ_OFF + 16384;      // U^T: 32 x Kd 64
constexpr uint32_t SCR_OFF = UT_OFF + 4096;       // 3 x 16 x 16 fp32
static_assert(SCR_OFF + 3072 <= ST_OFF, "aliases stay inside X and Y");
static_assert(TAQ_OFF % 16 == 0 && UT_OFF % 16 == 0, "operands 16-byte aligned");
static_assert(SMEM_ALLOC <= 232448, "fits the 227 KB opt-in limit");

// Rows before Y_b (rows of Y_b = 16 (b + 1)).
__device__ __forceinline__ uint32_t y_off(int b) {
  return Y_OFF + 256u * (uint32_t)(8 * b * (b + 1));
}

// ---- TMEM column map (512 columns allocated) ------------------------------
constexpr uint32_t TM_TX = 192;  // 160 columns: [w | u]
constexpr uint32_t TM_D1 = 352;  // 32 columns
constexpr uint32_t TM_D2 = 384;  // 32 columns
constexpr uint32_t TMEM_COLS = 512;
static_assert(TM_D2 + 32 <= TMEM_COLS, "TMEM map fits");
// Y_0..Y_3 are stored back to back, so together they form one 160-row B
// operand: a single N = 160 MMA gives X Y_b^T for every b, block b at TMEM
// columns 8 b (b + 1) ... 8 b (b + 1) + 16 (b + 1) - 1 (below TM_TX).
__device__ __forceinline__ uint32_t tm_a(int b) { return 8u * (uint32_t)(b * (b + 1)); }

// Which 16-column pieces of the intra-chunk products each TMEM lane quadrant
// reads: quadrants 0/2 hold rows 0..31 (blocks 0, 1), 1/3 rows 32..63.
__device__ __forceinline__ int piece_count(int quad) { return (quad & 1) ? 7 : 3; }
__device__ __forceinline__ void piece(int quad, int i, int &b, int &p) {
  if ((quad & 1) == 0) {
    b = i == 0 ? 0 : 1;
    p = i == 0 ? 0 : i - 1;
  } else {
    b = i < 3 ? 2 : 3;
    p = i < 3 ? i : i - 3;
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    fwd_tc_kernel(const FwdParams p, const __grid_constant__ CUtensorMap tm_q,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_g,
                  const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  float *sBeta = reinterpret_cast<float *>(smem + BETA_OFF);
  float *sDblk = reinterpret_cast<float *>(smem + DBLK_OFF);
  float *sG = reinterpret_cast<float *>(smem + RAW_G);
  float *sAkk = reinterpret_cast<float *>(smem + AKK_OFF);
  float *sT = reinterpret_cast<float *>(smem + TF_OFF);
  float *sScr = reinterpret_cast<float *>(smem + SCR_OFF);
  volatile uint32_t *sAbort = reinterpret_cast<volatile uint32_t *>(smem + ABORT_OFF);
  const uint32_t tma_bar = sb + BAR_OFF, mma_bar = sb + BAR_OFF + 8;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;
  const int L = 32 * quad + lane;  // this thread's TMEM lane
  const int H = p.H, T = p.T;

  // Fallback gate: nothing to do when the split path served this call.
  if (p.gate_chunks && *p.gate_chunks <= p.gate_capacity) return;
  if (warp == 0) tmem_alloc(sb + TMEMSLOT_OFF, TMEM_COLS);
  if (tid == 0) {
    mbar_init(tma_bar, 1);
    mbar_init(mma_bar, 1);
    *sAbort = 0u;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + TMEMSLOT_OFF);
  const uint32_t tq = tmem + ((uint32_t)(32 * quad) << 16);  // lane base of quad
  uint32_t tma_phase = 0, mma_phase = 0;
  // Copies / MMAs issued and not yet seen complete, with the barrier phase
  // parity they will complete (uniform over the CTA).
  bool tma_inflight = false, mma_inflight = false;
  uint32_t tma_pending = 0, mma_pending = 0;

  float S[VT];      // state rows (threads 0..127: key row = tid), fp32
  float u_reg[VT];  // u rows (threads 0..63)
#pragma unroll
  for (int i = 0; i < VT; ++i) S[i] = u_reg[i] = 0.f;

  auto abort_all = [&]() {
    *sAbort = 1u;
    set_status(p.status, KDA_DEVICE_TIMEOUT);
  };

  const uint32_t n_units = total_units(p.runs, p.B, H, p.n_vtiles);
  for (uint32_t unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    const Unit u = decode_unit(p.runs, unit, p.B, T, H, p.n_vtiles);
    const int vc0 = u.vt * VT;  // first value column of this unit

    // ---- state entering the run; S^T operand (MN-major: v contiguous) ----
    if (tid < 128) {
      const int c = tid;
      if (u.first && p.initial_state) {
        const float4 *src = reinterpret_cast<const float4 *>(
            p.initial_state + (((size_t)u.b * H + u.h) * KD + c) * p.V + vc0);
#pragma unroll
        for (int q4 = 0; q4 < VT / 4; ++q4) {
          const float4 x = src[q4];
          S[4 * q4] = x.x; S[4 * q4 + 1] = x.y; S[4 * q4 + 2] = x.z; S[4 * q4 + 3] = x.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < VT; ++i) S[i] = 0.f;
      }
#pragma unroll
      for (int vg = 0; vg < VT / 8; ++vg) {
        float t8[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) t8[i] = S[8 * vg + i];
        st_bf16x8(smem, ST_OFF + mn_off(8 * vg, c, KD), t8);
      }
    }
    float beta_next = 0.f;
    if (tid >= 128 && tid < 192) {
      const int r = tid - 128;
      if (u.start + r < u.end)
        beta_next = p.beta[((size_t)u.b * T + u.start + r) * H + u.h];
    }
    if (tid == 0) {
      const int y = u.b * T + u.start;
      mbar_expect_tx(tma_bar, RAW_TX_BYTES);
      tma_load_2d(sb + RAW_Q, &tm_q, u.h * KD, y, tma_bar);
      tma_load_2d(sb + RAW_K, &tm_k, u.h * KD, y, tma_bar);
      tma_load_2d(sb + RAW_G, &tm_g, u.h * KD, y, tma_bar);
      tma_load_2d(sb + RAW_V, &tm_v, u.h * p.V + vc0, y, tma_bar);
    }
    tma_inflight = true;
    tma_pending = tma_phase;

    for (int c0 = u.start; c0 < u.end; c0 += C) {
      const int n = min(C, u.end - c0);
      const bool has_next = c0 + C < u.end;
      const size_t tok0 = (size_t)u.b * T + c0;

      if (tid >= 128 && tid < 192) sBeta[tid - 128] = beta_next;
      if (!mbar_wait(tma_bar, tma_phase)) abort_all();
      else tma_inflight = false;
      tma_phase ^= 1u;
      __syncthreads();
      if (*sAbort) goto done;

      // ---- P0: gate cumsum per channel (two halves of 32 rows), block decays ----
      {
        const int c = tid & 127, hf = tid >> 7;
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int r = 32 * hf + i;
          v[i] = r < n ? sG[r * KD + c] : 0.f;
        }
#pragma unroll
        for (int i = 1; i < 32; ++i) v[i] += v[i - 1];
        sDblk[(2 * hf) * KD + c] = ex2(v[15] * kLog2e);
        sDblk[(2 * hf + 1) * KD + c] = ex2((v[31] - v[15]) * kLog2e);
        if (hf == 0) {
#pragma unroll
          for (int i = 0; i < 32; ++i) sG[i * KD + c] = v[i];
        }
        __syncthreads();
        if (hf == 1) {
          const float base = sG[31 * KD + c];
#pragma unroll
          for (int i = 0; i < 32; ++i) sG[(32 + i) * KD + c] = v[i] + base;
        }
      }
      __syncthreads();

      // ---- P1: decay factors and bf16 MMA operands ----
      // Thread -> 8 channels (cg) x 4 rows, one row per 16-row block; a warp
      // covers 8 consecutive rows x 4 channel groups (conflict-free stores).
      {
        const int rl = tid & 7, cg = (tid >> 3) & 15, hi = tid >> 7;
        const int cc0 = cg * 8;
#pragma unroll
        for (int b = 0; b < kNumSub; ++b) {  // the thread's row in block b
          const int r = kSub * b + 8 * hi + rl;
          const bool valid = r < n;
          const float br = sBeta[r];
          // block decays of the 8 channels and G at the block boundaries
          float D[kNumSub][8], Pb[8], Eb[8];
#pragma unroll
          for (int i = 0; i < kNumSub; ++i) {
            const float4 *dp = reinterpret_cast<const float4 *>(sDblk + i * KD + cc0);
            const float4 d0 = dp[0], d1 = dp[1];
            D[i][0] = d0.x; D[i][1] = d0.y; D[i][2] = d0.z; D[i][3] = d0.w;
            D[i][4] = d1.x; D[i][5] = d1.y; D[i][6] = d1.z; D[i][7] = d1.w;
          }
          {
            const float4 *ep = reinterpret_cast<const float4 *>(sG + (b * kSub + kSub - 1) * KD + cc0);
            const float4 e0 = ep[0], e1v = ep[1];
            Eb[0] = e0.x; Eb[1] = e0.y; Eb[2] = e0.z; Eb[3] = e0.w;
            Eb[4] = e1v.x; Eb[5] = e1v.y; Eb[6] = e1v.z; Eb[7] = e1v.w;
            if (b > 0) {
              const float4 *pp = reinterpret_cast<const float4 *>(sG + (b * kSub - 1) * KD + cc0);
              const float4 p0 = pp[0], p1 = pp[1];
              Pb[0] = p0.x; Pb[1] = p0.y; Pb[2] = p0.z; Pb[3] = p0.w;
              Pb[4] = p1.x; Pb[5] = p1.y; Pb[6] = p1.z; Pb[7] = p1.w;
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) Pb[j] = 0.f;
            }
          }
          float kk[8], qq[8], G[8];
          ld_bf16x8(smem + RAW_K + r * 256 + cc0 * 2, kk);
          ld_bf16x8(smem + RAW_Q + r * 256 + cc0 * 2, qq);
          {
            const float4 *gp = reinterpret_cast<const float4 *>(sG + r * KD + cc0);
            const float4 g0 = gp[0], g1 = gp[1];
            G[0] = g0.x; G[1] = g0.y; G[2] = g0.z; G[3] = g0.w;
            G[4] = g1.x; G[5] = g1.y; G[6] = g1.z; G[7] = g1.w;
          }
          float xk[8], xq[8], qt[8], kb[8], kh[8], yd[8], y1[8], y2[8], y3[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            float pre = 1.f, suf = 1.f;
#pragma unroll
            for (int i = 0; i < kNumSub; ++i) {
              if (i < b) pre *= D[i][j];
              if (i > b) suf *= D[i][j];
            }
            const float Pl = Pb[j] * kLog2e;
            const float El = Eb[j] * kLog2e;
            const float gl = G[j] * kLog2e;
            const float e1 = ex2(gl - Pl);   // e^{G - P_b}
            const float e2 = ex2(El - gl);   // e^{E_b - G}
            const float kv = valid ? kk[j] : 0.f;
            const float qv = valid ? qq[j] : 0.f;
            xk[j] = kv * e1;
            xq[j] = qv * e1;
            qt[j] = xq[j] * pre;
            kb[j] = xk[j] * (br * pre);
            const float ke2 = kv * e2;
            kh[j] = ke2 * suf;
            yd[j] = ke2 * __frcp_rn(D[b][j]);
            y1[j] = ke2;
            y2[j] = b + 2 < kNumSub ? ke2 * D[b + 2 < kNumSub ? b + 1 : 0][j] : 0.f;
            y3[j] = b + 3 < kNumSub ? y2[j] * D[b + 3 < kNumSub ? b + 2 : 0][j] : 0.f;
          }
          st_bf16x8(smem, X_OFF + op_off(r, cc0, KD), xk);
          st_bf16x8(smem, X_OFF + op_off(64 + r, cc0, KD), xq);
          st_bf16x8(smem, WQ_OFF + op_off(64 + r, cc0, KD), qt);
          st_bf16x8(smem, y_off(b) + op_off(r, cc0, KD), yd);
          if (b + 1 < kNumSub) st_bf16x8(smem, y_off(b + 1) + op_off(r, cc0, KD), y1);
          if (b + 2 < kNumSub) st_bf16x8(smem, y_off(b + 2) + op_off(r, cc0, KD), y2);
          if (b + 3 < kNumSub) st_bf16x8(smem, y_off(b + 3) + op_off(r, cc0, KD), y3);
          st_bf16x8(smem, KHT_OFF + mn_off(cc0, r, C), kh);   // (K e^{G_C-G})^T
          st_bf16x8(smem, RHST_OFF + mn_off(cc0, r, C), kb);  // (beta K e^G)^T
        }
        {  // (beta V)^T: thread -> row r, 8 value columns
          const int r = tid >> 2, vg = tid & 3;
          float vv[8];
          ld_bf16x8(smem + RAW_V + r * 64 + vg * 16, vv);
          const float br = r < n ? sBeta[r] : 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) vv[i] *= br;
          st_bf16x8(smem, RHST_OFF + mn_off(KD + 8 * vg, r, C), vv);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();

      // ---- P2: intra-chunk products on the tensor cores; next TMA ----
      if (tid == 0) {
        tc_fence_after();
        mma_group(tmem, sb + X_OFF, sb + Y_OFF, KD, 160, false, 0, 0);
        mma_commit(mma_bar);
        if (has_next) {
          const int y = (int)(tok0 + C);
          mbar_expect_tx(tma_bar, RAW_TX_BYTES);
          tma_load_2d(sb + RAW_Q, &tm_q, u.h * KD, y, tma_bar);
          tma_load_2d(sb + RAW_K, &tm_k, u.h * KD, y, tma_bar);
          tma_load_2d(sb + RAW_G, &tm_g, u.h * KD, y, tma_bar);
          tma_load_2d(sb + RAW_V, &tm_v, u.h * p.V + vc0, y, tma_bar);
        }
      }
      if (has_next) {
        tma_inflight = true;
        tma_pending = tma_phase;
      }
      if (tid >= 128 && tid < 192) {
        const int r = tid - 128;
        beta_next = (has_next && c0 + C + r < u.end)
                        ? p.beta[(tok0 + C + r) * H + u.h] : 0.f;
      }
      mma_inflight = true;
      mma_pending = mma_phase;
      if (!mbar_wait(mma_bar, mma_phase)) abort_all();
      else mma_inflight = false;
      mma_phase ^= 1u;
      __syncthreads();
      if (*sAbort) goto done;
      tc_fence_after();

      // ---- P3: A_kk (fp32, beta, strict) and A_qk (bf16, inclusive) ----
      {
        const int r = L & 63;
        const bool is_q = L >= 64;
        const int bme = r >> 4;
        const int np = piece_count(quad);
        for (int pi = half; pi < np; pi += 4) {
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
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                float a[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  a[i] = (j0 + 4 * q4 + i < r) ? br * v[e][4 * q4 + i] : 0.f;
                dst[q4] = make_float4(a[0], a[1], a[2], a[3]);
              }
            } else {
              float a0[8], a1[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                a0[i] = (j0 + i <= r) ? v[e][i] : 0.f;
                a1[i] = (j0 + 8 + i <= r) ? v[e][8 + i] : 0.f;
              }
              st_bf16x8(smem, TAQ_OFF + op_off(64 + r, j0, C), a0);
              st_bf16x8(smem, TAQ_OFF + op_off(64 + r, j0 + 8, C), a1);
            }
          }
        }
        if (is_q && half == 0) {
          const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          for (int jj = 16 * (bme + 1); jj < C; jj += 8)
            st_bf16x8(smem, TAQ_OFF + op_off(64 + r, jj, C), z);
        }
      }
      tc_fence_before();
      __syncthreads();

      // ---- P4: T = (I + L)^-1, blocked, fp32 ----
      if (tid < 64) {  // diagonal 16 x 16 blocks: right-looking substitution
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
      for (int d = 1; d < kNumSub; ++d) {
        // Blocks (i, j = i - d): M = sum_{m=j}^{i-1} L_im T_mj, then
        // T_ij = -T_ii M.  64 threads per block, 2 x 2 outputs each.
        const int nblk = kNumSub - d;
        const int blk = tid >> 6, e = tid & 63, ra = 2 * (e >> 3), cb = 2 * (e & 7);
        const bool act = blk < nblk;
        const int i = d + blk, j = blk;
        if (act) {
          float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
          for (int m = j; m < i; ++m) {
#pragma unroll
            for (int t = 0; t < 16; ++t) {
              const float l0 = sAkk[(16 * i + ra) * LDF + 16 * m + t];
              const float l1 = sAkk[(16 * i + ra + 1) * LDF + 16 * m + t];
              const float2 tv = *reinterpret_cast<const float2 *>(
                  sT + (16 * m + t) * LDF + 16 * j + cb);
              a00 = fmaf(l0, tv.x, a00); a01 = fmaf(l0, tv.y, a01);
              a10 = fmaf(l1, tv.x, a10); a11 = fmaf(l1, tv.y, a11);
            }
          }
          float *mm = sScr + blk * 256;
          *reinterpret_cast<float2 *>(mm + ra * 16 + cb) = make_float2(a00, a01);
          *reinterpret_cast<float2 *>(mm + (ra + 1) * 16 + cb) = make_float2(a10, a11);
        }
        __syncthreads();
        if (act) {
          const float *mm = sScr + blk * 256;
          float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
#pragma unroll
          for (int t = 0; t < 16; ++t) {
            const float d0 = sT[(16 * i + ra) * LDF + 16 * i + t];
            const float d1 = sT[(16 * i + ra + 1) * LDF + 16 * i + t];
            const float2 mv = *reinterpret_cast<const float2 *>(mm + t * 16 + cb);
            a00 = fmaf(d0, mv.x, a00); a01 = fmaf(d0, mv.y, a01);
            a10 = fmaf(d1, mv.x, a10); a11 = fmaf(d1, mv.y, a11);
          }
          *reinterpret_cast<float2 *>(sT + (16 * i + ra) * LDF + 16 * j + cb) = make_float2(-a00, -a01);
          *reinterpret_cast<float2 *>(sT + (16 * i + ra + 1) * LDF + 16 * j + cb) = make_float2(-a10, -a11);
        }
        __syncthreads();
      }
      {  // T -> bf16 rows 0..63 of [T ; A_qk]
        const int r = tid >> 2, jq = (tid & 3) * 16;
        const float4 *src = reinterpret_cast<const float4 *>(sT + r * LDF + jq);
        float t0[8], t1[8];
        const bool zero = (jq >> 4) > (r >> 4);
#pragma unroll
        for (int q4 = 0; q4 < 2; ++q4) {
          const float4 a = src[q4], b4 = src[2 + q4];
          t0[4 * q4] = a.x; t0[4 * q4 + 1] = a.y; t0[4 * q4 + 2] = a.z; t0[4 * q4 + 3] = a.w;
          t1[4 * q4] = b4.x; t1[4 * q4 + 1] = b4.y; t1[4 * q4 + 2] = b4.z; t1[4 * q4 + 3] = b4.w;
        }
        if (zero) {
#pragma unroll
          for (int i = 0; i < 8; ++i) t0[i] = t1[i] = 0.f;
        }
        st_bf16x8(smem, TAQ_OFF + op_off(r, jq, C), t0);
        st_bf16x8(smem, TAQ_OFF + op_off(r, jq + 8, C), t1);
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();

      // ---- P5: [w | u] = T [beta K e^G | beta V] ----
      if (tid == 0) {
        tc_fence_after();
        mma_group(tmem + TM_TX, sb + TAQ_OFF, sb + RHST_OFF, C, KD + VT, false, 0, 1);
        mma_commit(mma_bar);
      }
      mma_inflight = true;
      mma_pending = mma_phase;
      if (!mbar_wait(mma_bar, mma_phase)) abort_all();
      else mma_inflight = false;
      mma_phase ^= 1u;
      __syncthreads();
      if (*sAbort) goto done;
      tc_fence_after();
      if (quad < 2) {  // TMEM lanes 0..63 = chunk rows
        const int r = L;
        if (half == 0) {
          float v0[16], v1[16];
          tmem_ld16x2(tq + TM_TX + KD, tq + TM_TX + KD + 16, v0, v1);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            u_reg[i] = v0[i];
            u_reg[16 + i] = v1[i];
          }
        }
#pragma unroll
        for (int pc = 0; pc < 4; pc += 2) {
          const int c16 = half * 4 + pc;
          float v0[16], v1[16];
          tmem_ld16x2(tq + TM_TX + 16 * c16, tq + TM_TX + 16 * (c16 + 1), v0, v1);
          float a[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) a[i] = v0[i];
          st_bf16x8(smem, WQ_OFF + op_off(r, 16 * c16, KD), a);
#pragma unroll
          for (int i = 0; i < 8; ++i) a[i] = v0[8 + i];
          st_bf16x8(smem, WQ_OFF + op_off(r, 16 * c16 + 8, KD), a);
#pragma unroll
          for (int i = 0; i < 8; ++i) a[i] = v1[i];
          st_bf16x8(smem, WQ_OFF + op_off(r, 16 * c16 + 16, KD), a);
#pragma unroll
          for (int i = 0; i < 8; ++i) a[i] = v1[8 + i];
          st_bf16x8(smem, WQ_OFF + op_off(r, 16 * c16 + 24, KD), a);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();

      // ---- P6: D1 = [w ; Q e^G] S0 ----
      if (tid == 0) {
        tc_fence_after();
        mma_group(tmem + TM_D1, sb + WQ_OFF, sb + ST_OFF, KD, VT, false, 0, 1);
        mma_commit(mma_bar);
      }
      mma_inflight = true;
      mma_pending = mma_phase;
      if (!mbar_wait(mma_bar, mma_phase)) abort_all();
      else mma_inflight = false;
      mma_phase ^= 1u;
      __syncthreads();
      if (*sAbort) goto done;
      tc_fence_after();

      // ---- P7: U = u - w S0 -> U^T (bf16, MN-major) ----
      if (quad < 2 && half == 0) {
        const int r = L;
        float v0[16], v1[16];
        tmem_ld16x2(tq + TM_D1, tq + TM_D1 + 16, v0, v1);
#pragma unroll
        for (int vg = 0; vg < VT / 8; ++vg) {
          float a[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int col = 8 * vg + i;
            a[i] = u_reg[col] - (col < 16 ? v0[col & 15] : v1[col & 15]);
          }
          st_bf16x8(smem, UT_OFF + mn_off(8 * vg, r, C), a);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();

      // ---- P8: D1 += [T ; A_qk] U ; D2 = (K e^{G_C-G})^T U ----
      if (tid == 0) {
        tc_fence_after();
        mma_group(tmem + TM_D1, sb + TAQ_OFF, sb + UT_OFF, C, VT, true, 0, 1);
        mma_group(tmem + TM_D2, sb + KHT_OFF, sb + UT_OFF, C, VT, false, 1, 1);
        mma_commit(mma_bar);
      }
      mma_inflight = true;
      mma_pending = mma_phase;
      if (!mbar_wait(mma_bar, mma_phase)) abort_all();
      else mma_inflight = false;
      mma_phase ^= 1u;
      __syncthreads();
      if (*sAbort) goto done;
      tc_fence_after();

      // ---- P9: o rows, state update, S^T for the next chunk ----
      if (half == 0) {
        if (quad >= 2) {
          const int r = L - 64;
          float v0[16], v1[16];
          tmem_ld16x2(tq + TM_D1, tq + TM_D1 + 16, v0, v1);
          if (r < n) {
            uint4 *dst = reinterpret_cast<uint4 *>(
                static_cast<__nv_bfloat16 *>(p.o) + ((tok0 + r) * H + u.h) * p.V + vc0);
#pragma unroll
            for (int q4 = 0; q4 < VT / 8; ++q4) {
              float o[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int col = 8 * q4 + i;
                o[i] = p.scale * (col < 16 ? v0[col & 15] : v1[col & 15]);
              }
              uint4 w;
              w.x = pack_bf16(o[0], o[1]);
              w.y = pack_bf16(o[2], o[3]);
              w.z = pack_bf16(o[4], o[5]);
              w.w = pack_bf16(o[6], o[7]);
              dst[q4] = w;
            }
          }
        }
        {
          const int c = L;  // key row
          float gam = 1.f;
#pragma unroll
          for (int i = 0; i < kNumSub; ++i) gam *= sDblk[i * KD + c];
          float v0[16], v1[16];
          tmem_ld16x2(tq + TM_D2, tq + TM_D2 + 16, v0, v1);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            S[i] = fmaf(gam, S[i], v0[i]);
            S[16 + i] = fmaf(gam, S[16 + i], v1[i]);
          }
#pragma unroll
          for (int vg = 0; vg < VT / 8; ++vg) {
            float t8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) t8[i] = S[8 * vg + i];
            st_bf16x8(smem, ST_OFF + mn_off(8 * vg, c, KD), t8);
          }
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();
    }

    if (u.last && p.final_state && tid < 128) {
      float4 *dst = reinterpret_cast<float4 *>(
          p.final_state + (((size_t)u.b * H + u.h) * KD + tid) * p.V + vc0);
#pragma unroll
      for (int q4 = 0; q4 < VT / 4; ++q4)
        dst[q4] = make_float4(S[4 * q4], S[4 * q4 + 1], S[4 * q4 + 2], S[4 * q4 + 3]);
    }
  }

done:
  // On a timeout, give what is still in flight one more bounded wait before
  // the shared memory and TMEM are released.
  if (tma_inflight) mbar_wait(tma_bar, tma_pending);
  if (mma_inflight) mbar_wait(mma_bar, mma_pending);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ---- host side --------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 2-D view [rows, cols] of a row-major tensor, box [64 rows, box_cols].
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt,
              int esize, uint64_t cols, uint64_t rows, uint32_t box_cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * (uint64_t)esize};
  const cuuint32_t box[2] = {box_cols, (cuuint32_t)C};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool fwd_tc_supported(int K, int V, bool bf16, int v_tile) {
  return bf16 && K == KD && V == 128 && (v_tile == 0 || v_tile == VT);
}

cudaError_t launch_fwd_tc(const FwdParams &p_in, cudaStream_t stream) {
  if (!fwd_tc_supported(p_in.K, p_in.V, true, p_in.v_tile)) return cudaErrorNotSupported;
  FwdParams p = p_in;
  p.v_tile = VT;
  p.n_vtiles = p.V / VT;
  const uint64_t rows = (uint64_t)p.B * p.T;
  CUtensorMap mq, mk, mg, mv;
  if (!make_map(&mq, p.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)p.H * p.K, rows, KD) ||
      !make_map(&mk, p.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)p.H * p.K, rows, KD) ||
      !make_map(&mg, p.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)p.H * p.K, rows, KD) ||
      !make_map(&mv, p.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)p.H * p.V, rows, VT))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(
      fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
  if (e != cudaSuccess) return e;
  const long cap = num_sms();
  long units = p.runs.runs ? (long)p.B * p.T * p.H * p.n_vtiles
                           : (long)p.B * p.H * p.n_vtiles;
  const int grid = (int)(units < cap ? units : cap);
  fwd_tc_kernel<<<grid > 0 ? grid : 1, kThreads, SMEM_ALLOC, stream>>>(p, mq, mk, mg, mv);
  return cudaGetLastError();
}

}  // namespace kda
