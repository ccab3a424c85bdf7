// kda_bwd_tc.cu -- the chunked backward of the KDA forward on the tensor cores
// (bf16 q, k, v, d_o; K = V = 128; with or without segment ids).
//
// Page "feat(kda): integrate KDA attention with tokamax backend and CP
// support", section "Delta Rule formulation", gives the forward; the pages
// print no backward (their roadmap lists it next), so this is reverse-mode
// differentiation of the chunk form the forward kernels evaluate.  Per chunk
// of C = 64 rows with entering state S (rows past the row's end are zero):
//
//   G = cumsum(g), Q~ = Q e^G, K~ = K e^G, K^ = K e^{G_C - G}, gam = e^{G_C}
//   A_kk[r,j] = sum_c k_rc k_jc e^{G_rc-G_jc} (j < r), A_qk likewise (j <= r)
//   T = (I + diag(beta) A_kk)^-1, [u | w] = T [beta V | beta K~]
//   U = u - w S,  O = scale (Q~ S + A_qk U),  S' = gam * S + K^^T U
//
// and with dS' the gradient of the state leaving the chunk:
//
//   dU = scale A_qk^T dO + K^ dS'          (the only serial chain,
//   dS = scale Q~^T dO + gam * dS' - w^T dU  walked from the last chunk)
//   dQ~ = scale dO S^T, dw = -dU S^T, dK^ = U dS'^T, dA_qk = scale dO U^T,
//   dgam = rowsum(S * dS'), dT = [dU | dw] [beta V | beta K~]^T,
//   dY = T^T [dU | dw] (dV = beta dY_v, dK~ = beta dY_k),
//   dL = -(T^T dT T^T) strictly lower, dA_kk = diag(beta) dL,
//   dbeta_j = sum_r T[r,j] dT'[r,j] + sum_i dL[j,i] A_kk[j,i]  (dT' = dT / beta_j),
//
// then through the decayed products A_kk, A_qk and the exponentials to q, k
// and G, and dg is the reverse cumsum of dG within the chunk.
//
// Three passes:
//  1. the forward's prep kernel with larger items (also T, A_kk and K e^G)
//     and its recurrence in save mode (the state entering every chunk, U);
//  2. bwd_chain_kernel: the dS chain, one CTA per (run, head, value tile),
//     chunks from the last; it saves dS' and dU per chunk and writes
//     d_initial (a row's first run; later runs start from a reset state);
//  3. bwd_grad_kernel: every (chunk, head) independently, all gradients of
//     the chunk's tokens from the saved S, U, dS', dU and the inputs: a
//     dozen MMA groups on tcgen05 (TMEM accumulators), the intra-chunk
//     decayed products as per-sub-block products on the tensor cores, the
//     exponentials and the reverse cumsum on the CUDA cores.
#include <cuda.h>

#include "kda_f32x2.cuh"
#include "kda_split.cuh"

namespace kda {
namespace {

using namespace tc;
using namespace split;

struct BwdTcParams {
  int B, T, H;
  float scale;
  const float *g, *beta, *d_final;
  float *dq, *dk, *dv, *dg, *dbeta, *d_initial;
  const unsigned char *items;
  unsigned char *saves;
  ChunkTable ct;
  RunTable runs;  // with segment ids: the run list (units are runs); else none
  int v_tile, n_vtiles;
  uint32_t *status;
};

constexpr uint32_t align1k(uint32_t x) { return (x + 1023u) / 1024u * 1024u; }

// ---- the dS chain ---------------------------------------------------------------
// A stage holds the item's [w ; s Q e^G] | s A_qk | (K e^{G_C-G})^T (one
// copy; the prep folds the attention scale s into Q e^G and A_qk), this
// unit's d_o columns (VTR / 8 boxes of 64 rows x 8, zero past the chunk's
// end) and e^{G_C}.  Per chunk:
//   D_U  = (s A_qk)^T dO + K^ dS'        (u barrier; dU = D_U rows 0..63)
//   D_S  = (s Q~)^T dO + w^T (-dU)       (s barrier; dS = gam dS' + D_S)
// A_qk^T and K^ are read from the stored A_qk and K^^T through the
// transposed view; Q~^T and w^T from [w ; Q e^G] as K-major operands.
template <int VTR>
struct ChainLayout {
  static constexpr int WPQ = VTR == 128 ? 4 : 2;  // warps per TMEM lane quadrant
  static constexpr int THREADS = 128 * WPQ;
  static constexpr int CPT = VTR / WPQ;           // value columns per thread
  static constexpr uint32_t S_ITEM = I_U;         // bytes of the item copied
  static constexpr uint32_t S_DO = S_ITEM;        // d_o: mn_off(v, r, 64)
  static constexpr uint32_t S_GAM = S_DO + 128u * VTR;
  static constexpr uint32_t S_TX = S_GAM + 512;   // bytes per stage copy
  static constexpr uint32_t STAGE = align1k(S_TX);
  static constexpr uint32_t DST = 2 * STAGE;          // dS'^T, MN-major VTR x Kd 128
  static constexpr uint32_t NDU = DST + 256u * VTR;   // -dU^T, MN-major VTR x Kd 64
  static constexpr uint32_t BAR = NDU + 128u * VTR;   // 2 stages, u, s
  static constexpr uint32_t SLOT = BAR + 32;
  static constexpr uint32_t ABORT = SLOT + 4;
  static constexpr uint32_t ALLOC = ABORT + 12 + 1024;
  static constexpr uint32_t TM_U = 0, TM_S = VTR;
  static constexpr uint32_t TM_COLS = 2 * VTR <= 64 ? 64 : (2 * VTR <= 128 ? 128 : 256);
  static_assert(CPT == 16 || CPT == 32, "columns per thread");
  static_assert(ALLOC <= 232448, "chain smem fits");
};

template <int VTR>
__global__ void __launch_bounds__(ChainLayout<VTR>::THREADS, 1)
    bwd_chain_kernel(const BwdTcParams p, const __grid_constant__ CUtensorMap tm_do) {
  using Lay = ChainLayout<VTR>;
  constexpr int CPT = Lay::CPT;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  volatile uint32_t *sAbort = reinterpret_cast<volatile uint32_t *>(smem + Lay::ABORT);
  const uint32_t bar0 = sb + Lay::BAR, u_bar = bar0 + 16, s_bar = bar0 + 24;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, grp = warp >> 2;
  const int L = 32 * quad + lane;  // TMEM lane: chunk row (0..63) / key row
  const int col0 = CPT * grp;
  const int H = p.H, T = p.T;
  const ChunkTable &ct = p.ct;

  if (warp == 0) tmem_alloc(sb + Lay::SLOT, Lay::TM_COLS);
  if (tid == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar0 + 8, 1);
    mbar_init(u_bar, 1);
    mbar_init(s_bar, 1);
    *sAbort = 0u;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + Lay::SLOT);
  const uint32_t tq = tmem + ((uint32_t)(32 * quad) << 16);
  uint32_t st_phase[2] = {0u, 0u};
  uint32_t st_issued = 0;
  uint32_t n_u = 0, n_s = 0, c_u = 0, c_s = 0;
  uint32_t last_bar = 0, last_k = 0;
  bool committed = false;
  auto abort_all = [&]() {
    *sAbort = 1u;
    set_status(p.status, KDA_DEVICE_TIMEOUT);
  };
  auto wait_bar = [&](uint32_t bar, uint32_t &n) {
    if (!mbar_wait(bar, n & 1u)) abort_all();
    ++n;
  };
  auto commit = [&](uint32_t bar, uint32_t &c) {
    mma_commit(bar);
    last_bar = bar;
    last_k = c++;
    committed = true;
  };
  auto tmem_ld_cpt = [&](uint32_t taddr, float (&v)[CPT]) {
    if constexpr (CPT == 16) {
      tmem_ld16(taddr, v);
    } else {
      tmem_ld32(taddr, v);
    }
  };

  const bool fits = total_chunk_count(ct, p.B) <= ct.capacity;
  const uint32_t n_units = fits ? total_units(p.runs, p.B, H, p.n_vtiles) : 0u;
  for (uint32_t unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    // one run (the whole row without segment ids) of one head, VTR columns
    const Unit u = decode_unit(p.runs, unit, p.B, T, H, p.n_vtiles);
    const int vt = u.vt, h = u.h, b = u.b;
    const int vc0 = vt * VTR;
    const uint32_t cbase = run_chunk_base(ct, b, T, u.run_in_row);
    const int nc = u.end > u.start ? (u.end - u.start + C - 1) / C : 0;
    if (nc == 0) continue;
    auto item_ptr = [&](int c) {
      return p.items + ((size_t)(cbase + c) * H + h) * ct.item_stride;
    };
    // the stage of chunk c (processing order i: c = nc - 1 - i)
    auto issue_stage = [&](int s, int c) {
      const uint32_t dst = sb + (uint32_t)s * Lay::STAGE;
      const uint32_t bar = bar0 + 8u * (uint32_t)s;
      const unsigned char *src = item_ptr(c);
      mbar_expect_tx(bar, Lay::S_TX);
      bulk_load(dst, src, Lay::S_ITEM, bar);
      bulk_load(dst + Lay::S_GAM, src + I_GAM, 512, bar);
      for (int j = 0; j < VTR / 8; ++j)
        tma_load_2d(dst + Lay::S_DO + 1024u * j, &tm_do, h * VD + vc0 + 8 * j,
                    b * T + u.start + c * C, bar);
    };
    // the first stages' copies go out before d_final's load, so the two
    // latencies overlap (the previous unit's MMAs finished before its last
    // barrier)
    if (tid == 0)
      for (int i = 0; i < 2 && i < nc; ++i) issue_stage(i, nc - 1 - i);
    float dS[CPT];  // gradient of the state leaving the chunk, [key L][col0 ..]
    if (u.last && p.d_final) {  // the row's last run leaves the final state
      const float4 *src = reinterpret_cast<const float4 *>(
          p.d_final + (((size_t)b * H + h) * KD + L) * VD + vc0 + col0);
#pragma unroll
      for (int q4 = 0; q4 < CPT / 4; ++q4) {
        const float4 x = src[q4];
        dS[4 * q4] = x.x; dS[4 * q4 + 1] = x.y; dS[4 * q4 + 2] = x.z; dS[4 * q4 + 3] = x.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < CPT; ++i) dS[i] = 0.f;
    }
    st_issued = nc >= 2 ? 3u : 1u;

    for (int i = 0; i < nc; ++i) {
      const int c = nc - 1 - i, s = i & 1;
      const int n = min(C, u.end - (u.start + c * C));
      unsigned char *stg = smem + (uint32_t)s * Lay::STAGE;
      const uint32_t sstg = sb + (uint32_t)s * Lay::STAGE;
      unsigned char *sv = p.saves + ((size_t)(cbase + c) * H + h) * SV_BYTES;
      // ---- dS' (the gradient of the state leaving chunk c): B operand and save
#pragma unroll
      for (int e = 0; e < CPT / 8; ++e) {
        float t8[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) t8[k] = dS[8 * e + k];
        st_bf16x8(smem, Lay::DST + mn_off(col0 + 8 * e, L, KD), t8);
        st_g16(sv, SV_DSP + op_off(L, vc0 + col0 + 8 * e, KD), t8);
      }
      if (!mbar_wait(bar0 + 8u * s, st_phase[s])) abort_all();
      else st_issued &= ~(1u << s);
      st_phase[s] ^= 1u;
      // ---- d_o rows past the chunk's end zero (the items' A_qk and Q e^G
      //      carry the scale, so d_o is used as loaded)
      if (n < C) {
        const int m = C - n;
        for (int j = tid; j < (VTR / 8) * m; j += Lay::THREADS) {
          const int r = n + j % m;
          *reinterpret_cast<uint4 *>(stg + Lay::S_DO + 1024u * (j / m) + 16u * r) =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();
      if (*sAbort) goto done;
      if (tid == 0) {
        tc_fence_after();
        // D_U = (s A_qk)^T dO + K^ dS'
        mma_k(tmem + Lay::TM_U, Opnd{sstg + I_AQK, 1024, 128}, 1,
              Opnd{sstg + Lay::S_DO, 128, 1024}, 1, 4, VTR, false);
        mma_k(tmem + Lay::TM_U, Opnd{sstg + I_KHT, 1024, 128}, 1,
              Opnd{sb + Lay::DST, 128, 2048}, 1, 8, VTR, true);
        commit(u_bar, c_u);
        // D_S = (s Q~)^T dO, completed below by w^T (-dU)
        mma_k(tmem + Lay::TM_S, Opnd{sstg + I_WQ + 16384, 2048, 128}, 0,
              Opnd{sstg + Lay::S_DO, 128, 1024}, 1, 4, VTR, false);
      }
      wait_bar(u_bar, n_u);
      tc_fence_after();
      if (quad < 2) {  // lanes 0..63: dU rows
        const int r = L;
        float v[CPT];
        tmem_ld_cpt(tq + Lay::TM_U + col0, v);
#pragma unroll
        for (int e = 0; e < CPT / 8; ++e) {
          float a[8], na[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            a[k] = v[8 * e + k];
            na[k] = -a[k];
          }
          st_g16(sv, SV_DU + op_off(r, vc0 + col0 + 8 * e, KD), a);
          st_bf16x8(smem, Lay::NDU + mn_off(col0 + 8 * e, r, C), na);
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncthreads();
      if (*sAbort) goto done;
      if (tid == 0) {
        tc_fence_after();
        mma_k(tmem + Lay::TM_S, Opnd{sstg + I_WQ, 2048, 128}, 0, Opnd{sb + Lay::NDU, 128, 1024},
              1, 4, VTR, true);
        commit(s_bar, c_s);
      }
      wait_bar(s_bar, n_s);
      tc_fence_after();
      {
        const float gam = reinterpret_cast<const float *>(stg + Lay::S_GAM)[L];
        float v[CPT];
        tmem_ld_cpt(tq + Lay::TM_S + col0, v);
#pragma unroll
        for (int k = 0; k < CPT; ++k) dS[k] = fmaf(gam, dS[k], v[k]);
      }
      tc_fence_before();
      __syncthreads();
      if (*sAbort) goto done;
      // stage s is free: the chunk two places on
      if (i + 2 < nc) {
        if (tid == 0) issue_stage(s, nc - 1 - (i + 2));
        st_issued |= 1u << s;
      }
    }
    if (u.first && p.d_initial) {  // the row's first run starts from the initial state
      float4 *dst = reinterpret_cast<float4 *>(
          p.d_initial + (((size_t)b * H + h) * KD + L) * VD + vc0 + col0);
#pragma unroll
      for (int q4 = 0; q4 < CPT / 4; ++q4)
        dst[q4] = make_float4(dS[4 * q4], dS[4 * q4 + 1], dS[4 * q4 + 2], dS[4 * q4 + 3]);
    }
  }

done:
  // one more commit covers every MMA thread 0 issued (after an abort the
  // (s Q~)^T dO product can follow the last commit)
  if (tid == 0 && committed) commit(u_bar, c_u);
  for (int s = 0; s < 2; ++s)
    if (tid == 0 && (st_issued & (1u << s))) mbar_wait(bar0 + 8u * s, st_phase[s]);
  if (tid == 0 && committed) mbar_wait(last_bar, last_k & 1u);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, Lay::TM_COLS);
  }
}

// ---- per-chunk gradients ----------------------------------------------------------
// Shared memory (bytes).  Loaded per item: the saves S | U | dS' | dU, the
// d_o and v tiles ([8-column group][row][8]: a K-major operand over rows),
// T and K e^G from the item, g (cumsum'd in place to G, log2 units) and the
// raw q, k tiles ([half][row][64]).  Regions are reused once dead: after
// the first products (S, U, dS') the dA tiles, dT, P and dw; after the
// T products the per-sub-block operands of the decayed products.
namespace gl {
constexpr uint32_t SV = 0;
constexpr uint32_t S_S = SV + SV_S, S_U = SV + SV_U, S_DSP = SV + SV_DSP, S_DU = SV + SV_DU;
constexpr uint32_t DO = SV_BYTES;        // 16 KiB
constexpr uint32_t VV = DO + 16384;      // 16 KiB
constexpr uint32_t TT = VV + 16384;      // T, op_off(r, j, 64), 8 KiB
constexpr uint32_t KT = TT + 8192;       // K e^G, op_off(c, j, 64), 16 KiB
constexpr uint32_t GG = KT + 16384;      // G fp32 [quarter][row][32], 32 KiB
constexpr uint32_t QQ = GG + 32768;      // q bf16 [half][row][64]
constexpr uint32_t KK = QQ + 16384;      // k bf16 [half][row][64]
constexpr uint32_t MISC = KK + 16384;
constexpr uint32_t BETA = MISC;          // 64 fp32
constexpr uint32_t DGAM = BETA + 256;    // dgam, 128 fp32
constexpr uint32_t DB = DGAM + 512;      // dbeta parts [3][64] fp32
constexpr uint32_t GP = DB + 768;        // dG half sums [2][128] fp32
constexpr uint32_t GCP = GP + 1024;      // sum_r dK^ K^ halves [2][128] fp32
constexpr uint32_t BAR = GCP + 1024;     // loads A, G, R; mma
constexpr uint32_t SLOT = BAR + 32;
constexpr uint32_t ABORT = SLOT + 4;
constexpr uint32_t ALLOC = ABORT + 12 + 1024;
// three load groups: what the first products read (saves, d_o), issued
// while the previous item's final readout runs (those regions are dead
// then); g for the cumsum; what the later phases read (v, T, K e^G, q, k)
constexpr uint32_t LOADA_TX = SV_BYTES + 16384;
constexpr uint32_t LOADG_TX = 32768;
constexpr uint32_t LOADR_TX = 16384 + 8192 + 16384 + 16384 * 2;
// after the first products
// dA tiles, 16 KiB: per 16-row block b, the block's rows of scale dO U^T
// (j <= r; "q") then of diag(beta) dL ("k"), each K-major over j, so the
// two form one 32-row operand for the block's row sums
constexpr uint32_t DA = 0;
__host__ __device__ constexpr uint32_t da_off(int kq, int r, int j) {
  return 4096u * (uint32_t)(r >> 4) + 2048u * (uint32_t)kq +
         (uint32_t)((r & 7) * 16 + ((r >> 3) & 1) * 1024 + (j >> 3) * 128 + (j & 7) * 2);
}
constexpr uint32_t DTS = 16384;          // dT = dT' diag(beta), op_off(r, j, 64)
constexpr uint32_t DTU = 24576;          // dT', mn_off(j, r, 64)
constexpr uint32_t PP = 32768;           // P = dT T^T, mn_off(b, r, 64)
constexpr uint32_t DW = S_DSP;           // dw, op_off(c, r, 64), 16 KiB
// decayed products, per 16-row block b with P_b = G before the block
// (0 for b = 0): KK_b[c][j] = k_jc 2^{P_b - G_jc} for j < 16 (b + 1), and
// YQ[c][r] = q_rc 2^{G_rc - P_b(r)}, YK likewise with k; K-major over
// channels.  The row sums (over j) and the column sums (over r) are both
// formed from these same bf16 values, so each (r, j) pair enters dG_r and
// dG_j as the same fp32 products and cancels exactly in the reverse cumsum.
constexpr uint32_t OKK = 16384;
constexpr uint32_t OYQ = OKK + 40960;
constexpr uint32_t OYK = OYQ + 16384;
__host__ __device__ constexpr uint32_t kk_off(int b) { return 2048u * b * (b + 1); }
__host__ __device__ constexpr uint32_t w_col(int b) { return 8u * b * (b + 1); }
static_assert(OYK + 16384 <= GG, "decayed-product operands below G");
static_assert(64 * 128 * 4 <= GG - VV, "dG rows fit over v, T and K e^G");
static_assert(DW + 16384 + 1024 <= S_DU, "dw and its transposed view's overrun");
static_assert(ALLOC <= 232448, "grad smem fits");
// TMEM columns
constexpr uint32_t C_DQT = 0;    // dQ~^T / scale   [c][r]
constexpr uint32_t C_DKH = 64;   // dK^^T           [c][r]
constexpr uint32_t C_DYK = 128;  // dY_k^T          [c][j]
constexpr uint32_t C_ROW = 192;  // row sums [c][32 b + (q 0..15 | k 16..31)]; first dY_v [j][v]
constexpr uint32_t C_W = 320;    // column sums W_b [c][j < 16 (b + 1)] at C_W + w_col(b), 160
constexpr uint32_t C_X = 384;    // -dw^T, then dT', then P
constexpr uint32_t C_Y = 448;    // dA_qk / scale, then T^T dT', then -dL
}  // namespace gl

struct GradMaps {
  CUtensorMap q, k, g, v, d_o;
};

__global__ void __launch_bounds__(256, 1)
    bwd_grad_kernel(const BwdTcParams p, const __grid_constant__ GradMaps maps) {
  using namespace gl;
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  volatile uint32_t *sAbort = reinterpret_cast<volatile uint32_t *>(smem + ABORT);
  const uint32_t lda_bar = sb + BAR, ldg_bar = sb + BAR + 8, ldr_bar = sb + BAR + 16;
  const uint32_t mma_bar = sb + BAR + 24;
  float *sBeta = reinterpret_cast<float *>(smem + BETA);
  float *sDgam = reinterpret_cast<float *>(smem + DGAM);
  float *sDb = reinterpret_cast<float *>(smem + DB);
  float *sGp = reinterpret_cast<float *>(smem + GP);
  float *sGcp = reinterpret_cast<float *>(smem + GCP);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int quad = warp & 3, hh = warp >> 2;
  const int L = 32 * quad + lane;  // TMEM lane: channel c, or chunk row r (< 64)
  const int H = p.H, T = p.T;
  const ChunkTable &ct = p.ct;
  const float scale = p.scale;

  if (warp == 0) tmem_alloc(sb + SLOT, 512);
  if (tid == 0) {
    mbar_init(lda_bar, 1);
    mbar_init(ldg_bar, 1);
    mbar_init(ldr_bar, 1);
    mbar_init(mma_bar, 1);
    *sAbort = 0u;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(smem + SLOT);
  const uint32_t tq = tmem + ((uint32_t)(32 * quad) << 16);
  // each load barrier completes once per item: ph_a / ph_g / ph_r are the
  // parities of the next completion to wait for
  uint32_t ph_a = 0, ph_g = 0, ph_r = 0, n_mma = 0;
  bool lda_inflight = false, ldg_inflight = false, ldr_inflight = false, mma_inflight = false;
  auto abort_all = [&]() {
    *sAbort = 1u;
    set_status(p.status, KDA_DEVICE_TIMEOUT);
  };
  // one MMA batch: issued by thread 0 after a block barrier, waited on by all
  auto mma_wait = [&]() {
    mma_inflight = true;
    if (!mbar_wait(mma_bar, n_mma & 1u)) abort_all();
    else mma_inflight = false;
    ++n_mma;
    tc_fence_after();
  };
  auto sync_smem = [&]() {  // generic-proxy writes -> MMA reads
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
  };
  // G (log2 units) of row r, channel c
  auto Gat = [&](int r, int c) -> float {
    return *reinterpret_cast<const float *>(smem + GG + (c >> 5) * 8192 + r * 128 + (c & 31) * 4);
  };
  auto raw_at = [&](uint32_t base, int r, int c) -> float {
    const unsigned short u =
        *reinterpret_cast<const unsigned short *>(smem + base + (c >> 6) * 8192 + r * 128 + (c & 63) * 2);
    return __uint_as_float((uint32_t)u << 16);
  };

  const uint32_t n_items = total_chunk_count(ct, p.B) <= ct.capacity
                               ? total_chunk_count(ct, p.B) * (uint32_t)H : 0u;
  // group A of an item (warp 0): the saves and d_o
  auto issue_a = [&](uint32_t it) {
    const int hx = (int)(it % (uint32_t)H);
    int bx, tx, ex;
    chunk_of(ct, T, it / (uint32_t)H, bx, tx, ex);
    if (lane == 0) {
      mbar_expect_tx(lda_bar, LOADA_TX);
      bulk_load(sb + SV, p.saves + (size_t)it * SV_BYTES, SV_BYTES, lda_bar);
    }
    __syncwarp();
    if (lane < 16) tma_load_2d(sb + DO + 1024u * lane, &maps.d_o, hx * VD + 8 * lane, bx * T + tx, lda_bar);
  };
  if (warp == 0 && blockIdx.x < n_items) issue_a(blockIdx.x);
  lda_inflight = blockIdx.x < n_items;
  // beta of an item's rows (threads < C), loaded one item ahead into a
  // register so the load's latency is spent while the previous item computes
  auto load_beta = [&](uint32_t it) -> float {
    const int hx = (int)(it % (uint32_t)H);
    int bx, tx, ex;
    chunk_of(ct, T, it / (uint32_t)H, bx, tx, ex);
    return tid < min(C, ex - tx) ? p.beta[((size_t)bx * T + tx + tid) * H + hx] : 0.f;
  };
  float beta_next = 0.f;
  if (tid < C && blockIdx.x < n_items) beta_next = load_beta(blockIdx.x);
  for (uint32_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int h = (int)(item % (uint32_t)H);
    int b, t0, end;
    chunk_of(ct, T, item / (uint32_t)H, b, t0, end);
    const int n = min(C, end - t0);
    const size_t tok0 = (size_t)b * T + t0;
    const unsigned char *gi = p.items + (size_t)item * ct.item_stride;

    // ---- loads: g, then v, T, K e^G, q, k (group A was issued earlier)
    if (warp == 0) {
      if (lane == 0) {
        mbar_expect_tx(ldg_bar, LOADG_TX);
        mbar_expect_tx(ldr_bar, LOADR_TX);
      }
      __syncwarp();
      const int y = (int)tok0;
      if (lane < 4) tma_load_2d(sb + GG + 8192u * lane, &maps.g, h * KD + 32 * lane, y, ldg_bar);
      __syncwarp();
      if (lane == 0) {
        bulk_load(sb + TT, gi + I_T, 8192, ldr_bar);
        bulk_load(sb + KT, gi + I_KT, 16384, ldr_bar);
      }
      if (lane < 16) {
        tma_load_2d(sb + VV + 1024u * lane, &maps.v, h * VD + 8 * lane, y, ldr_bar);
      } else if (lane < 18) {
        const int hf = lane - 16;
        tma_load_2d(sb + QQ + 8192u * hf, &maps.q, h * KD + 64 * hf, y, ldr_bar);
        tma_load_2d(sb + KK + 8192u * hf, &maps.k, h * KD + 64 * hf, y, ldr_bar);
      }
    }
    ldg_inflight = ldr_inflight = true;
    if (tid < C) {
      sBeta[tid] = beta_next;
      if (item + gridDim.x < n_items) beta_next = load_beta(item + gridDim.x);
    }
    if (!mbar_wait(lda_bar, ph_a)) abort_all();
    else lda_inflight = false;
    ph_a ^= 1u;
    // the next item's later inputs into L2 while this one computes
    if (warp == 0 && item + gridDim.x < n_items) {
      const uint32_t nx = item + gridDim.x;
      const int hn = (int)(nx % (uint32_t)H);
      int bn, tn, en;
      chunk_of(ct, T, nx / (uint32_t)H, bn, tn, en);
      const int yn = bn * T + tn;
      const unsigned char *gin = p.items + (size_t)nx * ct.item_stride;
      if (lane == 0) prefetch_l2(gin + I_T, 8192);
      else if (lane == 1) prefetch_l2(gin + I_KT, 16384);
      else if (lane == 2) prefetch_l2(gin + I_AKK, 16384);
      else if (lane < 7) tma_prefetch_2d(&maps.g, hn * KD + 32 * (lane - 3), yn);
      else if (lane < 9) tma_prefetch_2d(&maps.q, hn * KD + 64 * (lane - 7), yn);
      else if (lane < 11) tma_prefetch_2d(&maps.k, hn * KD + 64 * (lane - 9), yn);
      if (lane < 16) tma_prefetch_2d(&maps.v, hn * VD + 8 * lane, yn);
    }
    if (n < C) {  // rows past the chunk's end: zero (they may hold the next row)
      const int m = C - n;
      for (int i = tid; i < 16 * m; i += 256) {
        const int grp = i / m, r = n + i % m;
        *reinterpret_cast<uint4 *>(smem + DO + 1024 * grp + 16 * r) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    sync_smem();
    if (*sAbort) goto done;

    // ---- first products (lanes = channels unless noted)
    if (tid == 0) {
      tc_fence_after();
      mma_k(tmem + C_DQT, Opnd{sb + S_S, 128, 2048}, 0, Opnd{sb + DO, 1024, 128}, 0, 8, 64, false);
      mma_k(tmem + C_X, Opnd{sb + S_S, 128, 2048}, 0, Opnd{sb + S_DU, 128, 2048}, 0, 8, 64, false);
      mma_k(tmem + C_DKH, Opnd{sb + S_DSP, 128, 2048}, 0, Opnd{sb + S_U, 128, 2048}, 0, 8, 64, false);
      // lanes = rows: dO U^T
      mma_k(tmem + C_Y, Opnd{sb + DO, 1024, 128}, 0, Opnd{sb + S_U, 128, 2048}, 0, 8, 64, false);
      mma_commit(mma_bar);
    }
    // meanwhile: G = cumsum(g) (log2 units) per channel; dgam = rowsum(S * dS')
    if (!mbar_wait(ldg_bar, ph_g)) abort_all();
    else ldg_inflight = false;
    ph_g ^= 1u;
    if (n < C) {
      const int m = C - n;
      for (int i = tid; i < 4 * 8 * m; i += 256) {  // g: 8 x 16 B per row and quarter
        const int qd = i / (8 * m), rem = i % (8 * m), r = n + rem / 8, part = rem % 8;
        *reinterpret_cast<uint4 *>(smem + GG + 8192 * qd + 128 * r + 16 * part) = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncthreads();
    }
    if (hh == 0) {
      const int ch = L;
      float acc = 0.f;
      float *gcol = reinterpret_cast<float *>(smem + GG + (ch >> 5) * 8192 + (ch & 31) * 4);
      for (int r = 0; r < C; ++r) {
        acc = fmaf(gcol[32 * r], kLog2e, acc);
        gcol[32 * r] = acc;
      }
    } else {  // dgam = rowsum(S * dS')
      const int ch = L;
      float acc = 0.f;
#pragma unroll 4
      for (int v8 = 0; v8 < VD / 8; ++v8) {
        float a[8], d[8];
        ld_bf16x8(smem + S_S + op_off(ch, 8 * v8, KD), a);
        ld_bf16x8(smem + S_DSP + op_off(ch, 8 * v8, KD), d);
#pragma unroll
        for (int k = 0; k < 8; ++k) acc = fmaf(a[k], d[k], acc);
      }
      sDgam[ch] = acc;
    }
    mma_wait();
    __syncthreads();  // G, dgam written; S and dS' are no longer read
    if (*sAbort) goto done;
    // ---- dw (K-major over rows) and dA_qk (rows < 64)
    {
      float v[32];
      tmem_ld32(tq + C_X + 32 * hh, v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float a[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) a[k] = -v[8 * e + k];
        st_bf16x8(smem, DW + op_off(L, 32 * hh + 8 * e, C), a);
      }
      if (quad < 2) {
        const int r = L;
        tmem_ld32(tq + C_Y + 32 * hh, v);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j8 = 32 * hh + 8 * e;
          float a[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) a[k] = j8 + k <= r ? scale * v[8 * e + k] : 0.f;
          st_bf16x8(smem, DA + da_off(0, r, j8), a);
        }
      }
    }
    // the later phases' inputs (issued with the first group)
    if (!mbar_wait(ldr_bar, ph_r)) abort_all();
    else ldr_inflight = false;
    ph_r ^= 1u;
    if (n < C) {
      const int m = C - n;
      for (int i = tid; i < 16 * m; i += 256) {
        const int grp = i / m, r = n + i % m;
        *reinterpret_cast<uint4 *>(smem + VV + 1024 * grp + 16 * r) = make_uint4(0u, 0u, 0u, 0u);
      }
      for (int i = tid; i < 8 * m; i += 256) {  // q, k: 8 x 16 B per row and half
        const int r = n + i / 8, part = i % 8;
        for (int hf = 0; hf < 2; ++hf) {
          *reinterpret_cast<uint4 *>(smem + QQ + 8192 * hf + 128 * r + 16 * part) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4 *>(smem + KK + 8192 * hf + 128 * r + 16 * part) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    sync_smem();
    if (*sAbort) goto done;
    // ---- T products
    if (tid == 0) {
      tc_fence_after();
      // dT' = dU V^T + dw (K e^G)^T              lanes = rows r
      mma_k(tmem + C_X, Opnd{sb + S_DU, 128, 2048}, 0, Opnd{sb + VV, 1024, 128}, 0, 8, 64, false);
      mma_k(tmem + C_X, Opnd{sb + DW, 1024, 128}, 1, Opnd{sb + KT, 1024, 128}, 1, 8, 64, true);
      // dY_k^T = dw^T T                           lanes = channels
      mma_k(tmem + C_DYK, Opnd{sb + DW, 128, 1024}, 0, Opnd{sb + TT, 1024, 128}, 1, 4, 64, false);
      // dY_v^T = dU^T T                            lanes = value columns v
      mma_k(tmem + C_ROW, Opnd{sb + S_DU, 2048, 128}, 1, Opnd{sb + TT, 1024, 128}, 1, 4, 64, false);
      mma_commit(mma_bar);
    }
    mma_wait();
    if (*sAbort) goto done;
    if (quad < 2) {  // lanes = rows (warp-uniform): only rows 0..63 hold results
      float v[32];
      tmem_ld32(tq + C_X + 32 * hh, v);
      {  // dT' row r: dT (beta_j) K-major and dT' MN-major
        const int r = L;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j8 = 32 * hh + 8 * e;
          float a[8], s8[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            a[k] = v[8 * e + k];
            s8[k] = a[k] * sBeta[j8 + k];
          }
          st_bf16x8(smem, DTS + op_off(r, j8, C), s8);
          st_bf16x8(smem, DTU + mn_off(j8, r, C), a);
        }
      }
    }
    {  // dv = beta dY_v: value column L, rows j = 32 hh .. (a warp writes 128
       // contiguous bytes per row)
      float v[32];
      tmem_ld32(tq + C_ROW + 32 * hh, v);
      float *dst = p.dv + tok0 * H * VD + (size_t)h * VD + L;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int j = 32 * hh + k;
        if (j < n) dst[(size_t)j * H * VD] = sBeta[j] * v[k];
      }
    }
    sync_smem();
    if (*sAbort) goto done;
    if (tid == 0) {
      tc_fence_after();
      // T^T dT' (its diagonal: the dT part of dbeta)   lanes = rows j
      mma_k(tmem + C_Y, Opnd{sb + TT, 1024, 128}, 1, Opnd{sb + DTU, 128, 1024}, 1, 4, 64, false);
      // P = dT T^T                                     lanes = rows r
      mma_k(tmem + C_X, Opnd{sb + DTS, 128, 1024}, 0, Opnd{sb + TT, 128, 1024}, 0, 4, 64, false);
      mma_commit(mma_bar);
    }
    mma_wait();
    if (*sAbort) goto done;
    if (quad < 2) {
      float v[32];
      if (hh == 0) {  // diagonal: row j = L reads column j of its quadrant
        tmem_ld32(tq + C_Y + 32 * quad, v);
        float d = 0.f;
#pragma unroll
        for (int k = 0; k < 32; ++k) d = k == lane ? v[k] : d;
        sDb[L] = d;
      }
      tmem_ld32(tq + C_X + 32 * hh, v);
      {
        const int r = L;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float a[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) a[k] = v[8 * e + k];
          st_bf16x8(smem, PP + mn_off(32 * hh + 8 * e, r, C), a);
        }
      }
    }
    sync_smem();
    if (*sAbort) goto done;
    if (tid == 0) {
      tc_fence_after();
      // T^T P = T^T dT T^T = -dL (before the mask)     lanes = rows a
      mma_k(tmem + C_Y, Opnd{sb + TT, 1024, 128}, 1, Opnd{sb + PP, 128, 1024}, 1, 4, 64, false);
      mma_commit(mma_bar);
    }
    float4 akk[8];  // A_kk row a = L, this thread's 32 columns (read while the MMA runs)
    if (quad < 2) {
      const float4 *src = reinterpret_cast<const float4 *>(gi + I_AKK + (L * C + 32 * hh) * 4);
#pragma unroll
      for (int i = 0; i < 8; ++i) akk[i] = src[i];
    }
    mma_wait();
    if (*sAbort) goto done;
    if (quad < 2) {
      float v[32];
      tmem_ld32(tq + C_Y + 32 * hh, v);
      {
        const int a_ = L;
        const float ba = sBeta[a_];
        float db = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int b8 = 32 * hh + 8 * e;
          const float4 x0 = akk[2 * e], x1 = akk[2 * e + 1];
          const float ak[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          float d[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float dl = b8 + k < a_ ? -v[8 * e + k] : 0.f;
            db = fmaf(dl, ak[k], db);
            d[k] = ba * dl;
          }
          st_bf16x8(smem, DA + da_off(1, a_, b8), d);
        }
        sDb[64 * (1 + hh) + a_] = db;
      }
    }
    // ---- operands of the decayed products (channel c = L, this thread's
    //      rows r = 32 hh ..): YQ, YK (row r scaled into its block's frame)
    //      and row r of KK_b for every block b >= b(r)
    {
      const int ch = L;
      float E[kNumSub];
#pragma unroll
      for (int i = 0; i < kNumSub; ++i) E[i] = Gat(16 * i + 15, ch);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r8 = 32 * hh + 8 * e;
        const int br = r8 >> 4;
        const float Pr = br == 0 ? 0.f : E[br - 1];
        float yq[8], yk[8], ik[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float Gr = Gat(r8 + k, ch);
          const float e1 = ex2(Gr - Pr);   // in (0, 1]
          const float kr = raw_at(KK, r8 + k, ch);
          yq[k] = raw_at(QQ, r8 + k, ch) * e1;
          yk[k] = kr * e1;
          ik[k] = kr * ex2(Pr - Gr);       // k_r 2^{P_b(r) - G_r}, at most 2^116 |k|
        }
        st_bf16x8(smem, OYQ + op_off(ch, r8, C), yq);
        st_bf16x8(smem, OYK + op_off(ch, r8, C), yk);
#pragma unroll
        for (int bb = 0; bb < kNumSub; ++bb) {
          if (bb < br) continue;
          const float fac = bb == br ? 1.f : ex2(E[bb - 1] - Pr);  // 2^{P_bb - P_b(r)} <= 1
          float a[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) a[k] = ik[k] * fac;
          st_bf16x8(smem, OKK + kk_off(bb) + op_off(ch, r8, 16 * (bb + 1)), a);
        }
      }
    }
    sync_smem();
    if (*sAbort) goto done;
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int bb = 0; bb < kNumSub; ++bb) {
        const uint32_t sbo = 256u * (bb + 1);
        // row sums of block bb: [c][r in block bb, q rows | k rows] =
        // sum_j KK_bb[c][j] dA[r][j], one N = 32 product over both tiles
        mma_k(tmem + C_ROW + 32 * bb, Opnd{sb + OKK + kk_off(bb), 128, sbo}, 0,
              Opnd{sb + DA + 4096u * bb, 128, 1024}, 0, bb + 1, 32, false);
        // column sums of block bb: W_bb[c][j] = sum_{r in bb} YK[c][r] dA_kk[r][j]
        //   + YQ[c][r] dA_qk[r][j], j < 16 (bb + 1) (dA read transposed)
        mma_k(tmem + C_W + w_col(bb), Opnd{sb + OYK + 256u * bb, 128, 1024}, 0,
              Opnd{sb + DA + 4096u * bb + 2048u, 1024, 128}, 1, 1, 16 * (bb + 1), false);
        mma_k(tmem + C_W + w_col(bb), Opnd{sb + OYQ + 256u * bb, 128, 1024}, 0,
              Opnd{sb + DA + 4096u * bb, 1024, 128}, 1, 1, 16 * (bb + 1), true);
      }
      mma_commit(mma_bar);
    }
    mma_wait();
    if (*sAbort) goto done;
    // every reader of the saves and d_o regions is done: the next item's
    // group A loads while this item's final readout runs
    if (item + gridDim.x < n_items) {
      if (warp == 0) issue_a(item + gridDim.x);
      lda_inflight = true;
    }

    // ---- final: this thread's channel c = L and rows 32 hh .. 32 hh + 31
    {
      const int ch = L;
      float E[kNumSub];
#pragma unroll
      for (int i = 0; i < kNumSub; ++i) E[i] = Gat(16 * i + 15, ch);
      const float GC = E[kNumSub - 1];
      // dG per row into shared memory ([row][channel] fp32, over v, T and
      // K e^G, whose last readers were the T products)
      float *sDG = reinterpret_cast<float *>(smem + VV);
      float gsum = 0.f, gcp = 0.f;
      // the bf16 values the MMAs read, recomputed bit for bit as the operand
      // build formed them (same expressions, round to nearest even)
      auto bfr2 = [](u64 x) {  // both lanes rounded to bf16 (nearest even) and back
        float a, b;
        upk2(x, a, b);
        const uint32_t hw = pack_bf16(a, b);
        return pk2(__uint_as_float(hw << 16), __uint_as_float(hw & 0xffff0000u));
      };
      auto neg2 = [](u64 x) { return x ^ 0x8000000080000000ull; };
#pragma unroll 1
      for (int e = 0; e < 4; ++e) {
        const int r8 = 32 * hh + 8 * e;
        const int br = r8 >> 4;
        // this group's TMEM columns: one batch of loads, one wait
        uint32_t u_[5 + kNumSub][8];
        tmem_ld8_nw(tq + C_DQT + r8, u_[0]);
        tmem_ld8_nw(tq + C_DKH + r8, u_[1]);
        tmem_ld8_nw(tq + C_DYK + r8, u_[2]);
        tmem_ld8_nw(tq + C_ROW + 32 * br + (r8 & 15), u_[3]);
        tmem_ld8_nw(tq + C_ROW + 32 * br + 16 + (r8 & 15), u_[4]);
#pragma unroll
        for (int bb = 0; bb < kNumSub; ++bb)  // W_bb holds row r only for bb >= b(r)
          tmem_ld8_nw(tq + C_W + w_col(bb) + (bb >= br ? r8 : 0), u_[5 + bb]);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 5 + kNumSub; ++i) reg_fence8(u_[i]);
        float dqt[8], dkh[8], dyk[8], rq[8], rk[8], w[kNumSub][8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          dqt[k] = __uint_as_float(u_[0][k]);
          dkh[k] = __uint_as_float(u_[1][k]);
          dyk[k] = __uint_as_float(u_[2][k]);
          rq[k] = __uint_as_float(u_[3][k]);
          rk[k] = __uint_as_float(u_[4][k]);
#pragma unroll
          for (int bb = 0; bb < kNumSub; ++bb) w[bb][k] = __uint_as_float(u_[5 + bb][k]);
        }
        const float Pr = br == 0 ? 0.f : E[br - 1];
        float fac[kNumSub];
#pragma unroll
        for (int bb = 0; bb < kNumSub; ++bb)
          fac[bb] = bb <= br ? 1.f : ex2(E[bb - 1] - Pr);
        // per block: 2^{P_b}, 2^{E_b - P_b}, 2^{G_C - E_b} (all <= 1), so that
        // 2^{G_r} = e1 2^{P_b} and 2^{G_C - G_r} = (ie1 2^{E_b - P_b}) 2^{G_C - E_b}
        // with every partial product <= 1 (no overflow; underflow only where
        // the value itself is below the fp32 range)
        const float ePr = ex2(Pr), fE = ex2(E[br] - Pr), fC = ex2(GC - E[br]);
        // rows in pairs (k, k + 1): packed f32x2 arithmetic, each lane the
        // fp32 operation of its row
        const u64 ePr2 = pk2(ePr, ePr), fE2 = pk2(fE, fE), fC2 = pk2(fC, fC);
        const u64 sc2 = pk2(scale, scale);
#pragma unroll
        for (int k = 0; k < 8; k += 2) {
          const int r = r8 + k;
          const float Ga = Gat(r, ch), Gb = Gat(r + 1, ch);
          const u64 e1 = pk2(ex2(Ga - Pr), ex2(Gb - Pr));
          const u64 ie1 = pk2(ex2(Pr - Ga), ex2(Pr - Gb));
          const u64 eG = mul2(e1, ePr2), eH = mul2(mul2(ie1, fE2), fC2);
          const float kra = raw_at(KK, r, ch), krb = raw_at(KK, r + 1, ch);
          const u64 kr = pk2(kra, krb), qr = pk2(raw_at(QQ, r, ch), raw_at(QQ, r + 1, ch));
          const u64 yq = bfr2(mul2(qr, e1)), yk = bfr2(mul2(kr, e1));
          const u64 ik = mul2(kr, ie1);
          u64 ccol = 0ull, gcol = 0ull;  // column sums: dk (fp32 factors), dG (the KK values)
#pragma unroll
          for (int bb = 0; bb < kNumSub; ++bb) {
            if (bb < br) continue;
            const u64 w2 = pk2(w[bb][k], w[bb][k + 1]), f2 = pk2(fac[bb], fac[bb]);
            ccol = fma2(w2, f2, ccol);
            gcol = fma2(w2, bfr2(mul2(ik, f2)), gcol);
          }
          const u64 rq2 = pk2(rq[k], rq[k + 1]), rk2 = pk2(rk[k], rk[k + 1]);
          const u64 dQt = mul2(mul2(sc2, pk2(dqt[k], dqt[k + 1])), eG);              // dQ~ e^G
          const u64 dKt = mul2(mul2(pk2(sBeta[r], sBeta[r + 1]), pk2(dyk[k], dyk[k + 1])), eG);  // dK~ e^G
          const u64 dKh = mul2(pk2(dkh[k], dkh[k + 1]), eH);                         // dK^ e^{G_C - G}
          const u64 dq = fma2(e1, rq2, dQt);
          const u64 dk = add2(add2(fma2(e1, rk2, mul2(ie1, ccol)), dKt), dKh);
          const u64 dG = fma2(kr, add2(dKt, neg2(dKh)),
                              fma2(qr, dQt, add2(fma2(yq, rq2, mul2(yk, rk2)), neg2(gcol))));
          float dga, dgb, dqa, dqb, dka, dkb, dha, dhb;
          upk2(dG, dga, dgb);
          upk2(dq, dqa, dqb);
          upk2(dk, dka, dkb);
          upk2(dKh, dha, dhb);
          sDG[r * KD + ch] = dga;
          sDG[(r + 1) * KD + ch] = dgb;
          gsum += dga;
          gsum += dgb;
          gcp = fmaf(kra, dha, gcp);
          gcp = fmaf(krb, dhb, gcp);
          if (r < n) {
            p.dq[((tok0 + r) * H + h) * KD + ch] = dqa;
            p.dk[((tok0 + r) * H + h) * KD + ch] = dka;
          }
          if (r + 1 < n) {
            p.dq[((tok0 + r + 1) * H + h) * KD + ch] = dqb;
            p.dk[((tok0 + r + 1) * H + h) * KD + ch] = dkb;
          }
        }
      }
      sGp[128 * hh + ch] = gsum;
      sGcp[128 * hh + ch] = gcp;
      __syncthreads();
      // d/dG_C (through K e^{G_C - G} and e^{G_C}) enters at the chunk's
      // last row.  Summed from the same dK^ the rows use: the two parts
      // cancel where the state update erases the decayed state, and the
      // rounding of dS' then cancels with them.
      const float dGC = sGcp[ch] + sGcp[128 + ch] + sDgam[ch] * ex2(GC);
      float carry = dGC + (hh == 0 ? sGp[128 + ch] : 0.f);
#pragma unroll 8
      for (int k = 31; k >= 0; --k) {
        const int r = 32 * hh + k;
        carry += sDG[r * KD + ch];
        if (r < n) p.dg[((tok0 + r) * H + h) * KD + ch] = carry;
      }
      if (tid < n) p.dbeta[(tok0 + tid) * H + h] = sDb[tid] + sDb[64 + tid] + sDb[128 + tid];
    }
    tc_fence_before();
    __syncthreads();  // TMEM, shared memory and the misc sums free for the next item
  }

done:
  if (tid == 0) {
    if (lda_inflight) mbar_wait(lda_bar, ph_a);
    if (ldg_inflight) mbar_wait(ldg_bar, ph_g);
    if (ldr_inflight) mbar_wait(ldr_bar, ph_r);
    if (mma_inflight) mbar_wait(mma_bar, (n_mma - 1) & 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Zero gradients for padding tokens (segment id 0): one warp per token.
__global__ void __launch_bounds__(256)
    bwd_zero_padding_kernel(const int32_t *segment_ids, int BT, int H, float *dq, float *dk,
                            float *dg, float *dbeta) {
  const int tok = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (tok >= BT || segment_ids[tok] != 0) return;
  const size_t base = (size_t)tok * H * KD;
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i = lane; i < H * KD / 4; i += 32) {
    reinterpret_cast<float4 *>(dq + base)[i] = z;
    reinterpret_cast<float4 *>(dk + base)[i] = z;
    reinterpret_cast<float4 *>(dg + base)[i] = z;
  }
  for (int i = lane; i < H; i += 32) dbeta[(size_t)tok * H + i] = 0.f;
}

template <int VTR>
cudaError_t launch_chain(const BwdTcParams &p, const CUtensorMap &m_do, cudaStream_t stream) {
  using Lay = ChainLayout<VTR>;
  cudaError_t e = cudaFuncSetAttribute(bwd_chain_kernel<VTR>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)Lay::ALLOC);
  if (e != cudaSuccess) return e;
  const long rows = p.runs.runs ? (long)p.B * p.T : (long)p.B;  // an upper bound of the runs
  const long units = rows * p.H * p.n_vtiles, sms = num_sms();
  const int grid = (int)(units < sms ? units : sms);
  bwd_chain_kernel<VTR><<<grid > 0 ? grid : 1, Lay::THREADS, Lay::ALLOC, stream>>>(p, m_do);
  return cudaGetLastError();
}

}  // namespace

bool bwd_tc_supported(int K, int V, bool bf16) { return bf16 && K == KD && V == VD; }

size_t bwd_tc_workspace_bytes(int B, int T, int H, bool has_seg, int max_runs_per_row) {
  return split::bwd_tc_workspace_bytes(B, T, H, has_seg, max_runs_per_row);
}

cudaError_t launch_fwd_save(const FwdParams &p, void *workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  return launch_fwd_for_bwd(p, workspace, workspace_bytes, nullptr, stream, true);
}

cudaError_t launch_bwd_tc(const BwdParams &bp, const int32_t *segment_ids, void *workspace,
                          size_t workspace_bytes, float *dq, float *dk, float *dg, float *dbeta,
                          uint32_t *status, cudaStream_t stream, bool from_saved) {
  if (bp.K != KD || bp.V != VD || (segment_ids != nullptr) != (bp.runs.runs != nullptr))
    return cudaErrorNotSupported;
  FwdParams fp;
  memset(&fp, 0, sizeof(fp));
  fp.B = bp.B; fp.T = bp.T; fp.H = bp.H; fp.K = bp.K; fp.V = bp.V;
  fp.q = bp.q; fp.k = bp.k; fp.v = bp.v; fp.g = bp.g; fp.beta = bp.beta;
  fp.scale = bp.scale;
  fp.initial_state = bp.initial_state;
  fp.status = status;
  fp.runs = bp.runs;
  BwdLayout lay;
  cudaError_t e = cudaSuccess;
  if (from_saved) {  // a saving forward on the same inputs left items and saves
    if (!bwd_layout(fp, workspace, workspace_bytes, &lay)) return cudaErrorInvalidValue;
  } else {
    e = launch_fwd_for_bwd(fp, workspace, workspace_bytes, &lay, stream);
    if (e != cudaSuccess) return e;
  }

  BwdTcParams p;
  memset(&p, 0, sizeof(p));
  p.B = bp.B; p.T = bp.T; p.H = bp.H;
  p.scale = bp.scale;
  p.g = bp.g; p.beta = bp.beta; p.d_final = bp.d_final;
  p.dq = dq; p.dk = dk; p.dv = bp.dv; p.dg = dg; p.dbeta = dbeta; p.d_initial = bp.d_initial;
  p.items = lay.items;
  p.saves = lay.saves;
  p.ct = lay.ct;
  p.runs = bp.runs;
  p.status = status;
  const long bh = (long)p.B * p.H, sms = num_sms();
  // value tile of the chain: as the forward recurrence (many short runs:
  // 128 columns, each item read once)
  p.v_tile = bp.runs.runs ? 128 : (bh * 4 <= sms ? 32 : (bh * 2 <= sms ? 64 : 128));
  p.n_vtiles = VD / p.v_tile;
  const uint64_t rows = (uint64_t)p.B * p.T;
  const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_NONE;
  GradMaps gm;
  if (!make_map(&gm.q, bp.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)p.H * KD, rows, 64, sw) ||
      !make_map(&gm.k, bp.k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)p.H * KD, rows, 64, sw) ||
      !make_map(&gm.g, bp.g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, (uint64_t)p.H * KD, rows, 32, sw) ||
      !make_map(&gm.v, bp.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)p.H * VD, rows, 8, sw) ||
      !make_map(&gm.d_o, bp.d_o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (uint64_t)p.H * VD, rows, 8, sw))
    return cudaErrorInvalidValue;
  e = p.v_tile == 32   ? launch_chain<32>(p, gm.d_o, stream)
      : p.v_tile == 64 ? launch_chain<64>(p, gm.d_o, stream)
                       : launch_chain<128>(p, gm.d_o, stream);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_grad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)gl::ALLOC);
  if (e != cudaSuccess) return e;
  const long items = (long)lay.ct.capacity * p.H;  // an upper bound of the real count
  const int grid = (int)(items < sms ? items : sms);
  bwd_grad_kernel<<<grid > 0 ? grid : 1, 256, gl::ALLOC, stream>>>(p, gm);
  e = cudaGetLastError();
  if (e != cudaSuccess || !segment_ids) return e;
  const int bt = p.B * p.T;
  bwd_zero_padding_kernel<<<(bt + 7) / 8, 256, 0, stream>>>(segment_ids, bt, p.H, dq, dk, dg,
                                                            dbeta);
  return cudaGetLastError();
}

}  // namespace kda
