// kda_fwd_simt.cu -- chunked KDA forward on the CUDA cores, fp32 arithmetic.
//
// Serves every supported shape (K, V in {32, 64, 128}; fp32 or bf16 q/k/v).
// It evaluates the chunk form of the gated delta rule (page "feat(kda):
// integrate KDA attention with tokamax backend and CP support", section
// "Delta Rule formulation"), derived from the token recurrence: per run,
// head and tile of value columns, for each chunk of 64 rows with state S0:
//
//   G      = inclusive cumsum of g over the chunk's rows, per key channel
//   A_kk   = beta_r sum_c k_rc k_jc e^{G_rc - G_jc}   (j <  r)
//   A_qk   =        sum_c q_rc k_jc e^{G_rc - G_jc}   (j <= r)
//   [u|w]  = (I + A_kk)^-1 diag(beta) [V | K e^{G}]   (forward substitution)
//   U      = u - w S0
//   O      = scale (Q e^{G} S0 + A_qk U)
//   S1     = diag(e^{G_C}) S0 + (K e^{G_C - G})^T U
//
// The factors e^{G_r - G_j} are built per 16-row sub-block b from
//   E1_r = e^{G_r - P_b} (P_b = G before the block), E2_r = e^{E_b - G_r}
//   (E_b = G at the block's last row): same block e^{G_r-G_j} = E1_r/E1_j,
//   earlier block b' e^{G_r-G_j} = E1_r * e^{P_b - E_b'} * E2_j,
// which keeps every factor inside fp32 range for g in [-5, 0] (a 16-row span
// is at most 80 < ln FLT_MAX).  Rows past the run end are zero (q = k = v = 0,
// beta = g = 0) so they contribute nothing.
//
// One CTA (256 threads) per unit (run, head, value tile); CTAs stride over
// units.  All intermediates live in shared memory.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int C = kChunk;

template <int K, int VT>
struct SimtSmem {
  static constexpr int LDK = K + 1;   // padded row stride of C x K tiles
  static constexpr int LDA = C + 1;   // padded row stride of C x C tiles
  static constexpr int oQ = 0;                    // C x LDK: q -> X2 -> Q e^G
  static constexpr int oK = oQ + C * LDK;         // k -> X1 -> w
  static constexpr int oG = oK + C * LDK;         // g -> G -> K E2 -> K e^{G_C-G}
  static constexpr int oYd = oG + C * LDK;        // k / E1 (same-block operand)
  static constexpr int oV = oYd + C * LDK;        // C x VT: v -> u
  static constexpr int oU = oV + C * VT;          // C x VT: U
  static constexpr int oS = oU + C * VT;          // K x VT: state
  static constexpr int oAkk = oS + K * VT;        // C x LDA
  static constexpr int oAqk = oAkk + C * LDA;     // C x LDA
  static constexpr int oBeta = oAqk + C * LDA;    // C
  static constexpr int oP = oBeta + C;            // 4 x K: G before block
  static constexpr int oE = oP + kNumSub * K;     // 4 x K: G at block end
  static constexpr int oPre = oE + kNumSub * K;   // 4 x K: e^{P_b}
  static constexpr int oSuf = oPre + kNumSub * K; // 4 x K: e^{G_C - E_b}
  static constexpr int oCross = oSuf + kNumSub * K;  // 6 x K: e^{P_b - E_b'}
  static constexpr int oGam = oCross + 6 * K;     // K: e^{G_C}
  static constexpr int total = oGam + K;
  static constexpr size_t bytes = sizeof(float) * (size_t)total;
};

// Index of the block pair (b, b') with b' < b in the 6-entry cross table.
__device__ __forceinline__ int cross_index(int b, int bp) {
  return b * (b - 1) / 2 + bp;  // (1,0)=0 (2,0)=1 (2,1)=2 (3,0)=3 (3,1)=4 (3,2)=5
}

template <int K, int VT, typename Tin>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_simt_kernel(const FwdParams p) {
  using L = SimtSmem<K, VT>;
  extern __shared__ float smem[];
  float *sQ = smem + L::oQ, *sK = smem + L::oK, *sG = smem + L::oG;
  float *sYd = smem + L::oYd, *sV = smem + L::oV, *sU = smem + L::oU;
  float *sS = smem + L::oS, *sAkk = smem + L::oAkk, *sAqk = smem + L::oAqk;
  float *sBeta = smem + L::oBeta, *sP = smem + L::oP, *sE = smem + L::oE;
  float *sPre = smem + L::oPre, *sSuf = smem + L::oSuf;
  float *sCross = smem + L::oCross, *sGam = smem + L::oGam;
  constexpr int LDK = L::LDK, LDA = L::LDA;
  const int tid = threadIdx.x;

  const Tin *__restrict__ gq = static_cast<const Tin *>(p.q);
  const Tin *__restrict__ gk = static_cast<const Tin *>(p.k);
  const Tin *__restrict__ gv = static_cast<const Tin *>(p.v);
  Tin *__restrict__ go = static_cast<Tin *>(p.o);
  const int H = p.H, T = p.T, V = p.V;

  // The strictly-upper micro tiles of A are never written: zero them once.
  for (int i = tid; i < 2 * C * LDA; i += kThreads) sAkk[i] = 0.f;
  __syncthreads();

  const uint32_t n_units = total_units(p.runs, p.B, H, p.n_vtiles);
  for (uint32_t unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    const Unit u = decode_unit(p.runs, unit, p.B, T, H, p.n_vtiles);
    const int v0 = u.vt * VT;

    // ---- state entering the run ----
    for (int i = tid; i < K * VT; i += kThreads) {
      const int c = i / VT, j = i % VT;
      float s = 0.f;
      if (u.first && p.initial_state)
        s = p.initial_state[(((size_t)u.b * H + u.h) * K + c) * V + v0 + j];
      sS[i] = s;
    }

    for (int c0 = u.start; c0 < u.end; c0 += C) {
      const int n = min(C, u.end - c0);
      const size_t tok0 = (size_t)u.b * T + c0;  // first token of the chunk
      __syncthreads();  // previous chunk done with every buffer

      // ---- 1. stage the chunk (rows >= n are zero) ----
      for (int i = tid; i < C * K; i += kThreads) {
        const int r = i / K, c = i % K;
        float qv = 0.f, kv = 0.f, gvl = 0.f;
        if (r < n) {
          const size_t off = ((tok0 + r) * H + u.h) * K + c;
          qv = to_f32(gq[off]);
          kv = to_f32(gk[off]);
          gvl = p.g[off];
        }
        sQ[r * LDK + c] = qv;
        sK[r * LDK + c] = kv;
        sG[r * LDK + c] = gvl;
      }
      for (int i = tid; i < C * VT; i += kThreads) {
        const int r = i / VT, j = i % VT;
        sV[i] = r < n ? to_f32(gv[((tok0 + r) * H + u.h) * V + v0 + j]) : 0.f;
      }
      if (tid < C) sBeta[tid] = tid < n ? p.beta[(tok0 + tid) * H + u.h] : 0.f;
      __syncthreads();

      // ---- 2. cumsum and per-channel block factors ----
      if (tid < K) {
        const int c = tid;
        float acc = 0.f;
        for (int r = 0; r < C; ++r) {
          acc += sG[r * LDK + c];
          sG[r * LDK + c] = acc;
        }
        float D[kNumSub];
#pragma unroll
        for (int b = 0; b < kNumSub; ++b) {
          const float P = b == 0 ? 0.f : sG[(b * kSub - 1) * LDK + c];
          const float E = sG[(b * kSub + kSub - 1) * LDK + c];
          sP[b * K + c] = P;
          sE[b * K + c] = E;
          D[b] = expf(E - P);
        }
        float pre = 1.f;
#pragma unroll
        for (int b = 0; b < kNumSub; ++b) {
          sPre[b * K + c] = pre;
          pre *= D[b];
        }
        sGam[c] = pre;
        float suf = 1.f;
#pragma unroll
        for (int b = kNumSub - 1; b >= 0; --b) {
          sSuf[b * K + c] = suf;
          suf *= D[b];
        }
#pragma unroll
        for (int b = 1; b < kNumSub; ++b) {
          float f = 1.f;
          for (int bp = b - 1; bp >= 0; --bp) {
            sCross[cross_index(b, bp) * K + c] = f;  // prod_{i=bp+1}^{b-1} D_i
            f *= D[bp];
          }
        }
      }
      __syncthreads();

      // ---- 3. elementwise factors ----
      for (int i = tid; i < C * K; i += kThreads) {
        const int r = i / K, c = i % K, b = r / kSub;
        const float G = sG[r * LDK + c];
        const float e1 = expf(G - sP[b * K + c]);
        const float e2 = expf(sE[b * K + c] - G);
        const float kv = sK[r * LDK + c];
        const float qv = sQ[r * LDK + c];
        sK[r * LDK + c] = kv * e1;   // X1: row operand of A_kk
        sQ[r * LDK + c] = qv * e1;   // X2: row operand of A_qk
        sG[r * LDK + c] = kv * e2;   // column operand, earlier blocks
        sYd[r * LDK + c] = kv / e1;  // column operand, same block
      }
      __syncthreads();

      // ---- 4. A_kk, A_qk: 4x4 micro tiles of the lower triangle ----
      if (tid < 136) {  // 16*17/2 micro tiles with J <= R
        int R = 0, rem = tid;
        while (rem > R) { rem -= R + 1; ++R; }
        const int J = rem;
        const int b = R / 4, bp = J / 4;  // sub-blocks of rows and columns
        const bool same = (b == bp);
        const float *Y = same ? sYd : sG;
        const float *cf = same ? nullptr : sCross + cross_index(b, bp) * K;
        float akk[4][4] = {}, aqk[4][4] = {};
        for (int c = 0; c < K; ++c) {
          float x1[4], x2[4], y[4];
          const float f = same ? 1.f : cf[c];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            x1[i] = sK[(4 * R + i) * LDK + c];
            x2[i] = sQ[(4 * R + i) * LDK + c];
            y[i] = Y[(4 * J + i) * LDK + c] * f;
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              akk[i][j] = fmaf(x1[i], y[j], akk[i][j]);
              aqk[i][j] = fmaf(x2[i], y[j], aqk[i][j]);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int r = 4 * R + i, jj = 4 * J + j;
            sAkk[r * LDA + jj] = jj < r ? sBeta[r] * akk[i][j] : 0.f;
            sAqk[r * LDA + jj] = jj <= r ? aqk[i][j] : 0.f;
          }
      }
      __syncthreads();

      // ---- 5. forward substitution for [u | w]; in-place decay of Q, K ----
      if (tid < VT + K) {
        const int col = tid;
        const bool is_u = col < VT;
        const int c = col - VT;
        float x[C];
#pragma unroll
        for (int r = 0; r < C; ++r) {
          const float rhs =
              is_u ? sV[r * VT + col]
                   : sK[r * LDK + c] * sPre[(r / kSub) * K + c];  // K e^{G}
          float acc = sBeta[r] * rhs;
#pragma unroll
          for (int j = 0; j < r; ++j) acc = fmaf(-sAkk[r * LDA + j], x[j], acc);
          x[r] = acc;
        }
#pragma unroll
        for (int r = 0; r < C; ++r) {
          if (is_u) sV[r * VT + col] = x[r];
          else sK[r * LDK + c] = x[r];
        }
      } else {
        for (int i = tid - (VT + K); i < C * K; i += kThreads - (VT + K)) {
          const int r = i / K, c = i % K, b = r / kSub;
          sQ[r * LDK + c] *= sPre[b * K + c];  // Q e^{G}
          sG[r * LDK + c] *= sSuf[b * K + c];  // K e^{G_C - G}
        }
      }
      __syncthreads();

      // ---- 6. U = u - w S0 (2 rows x 4 columns per item) ----
      for (int it = tid; it < (C / 2) * (VT / 4); it += kThreads) {
        const int r = 2 * (it / (VT / 4)), j = 4 * (it % (VT / 4));
        float a0[4], a1[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          a0[t] = sV[r * VT + j + t];
          a1[t] = sV[(r + 1) * VT + j + t];
        }
        for (int c = 0; c < K; ++c) {
          const float w0 = sK[r * LDK + c], w1 = sK[(r + 1) * LDK + c];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float s = sS[c * VT + j + t];
            a0[t] = fmaf(-w0, s, a0[t]);
            a1[t] = fmaf(-w1, s, a1[t]);
          }
        }
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          sU[r * VT + j + t] = a0[t];
          sU[(r + 1) * VT + j + t] = a1[t];
        }
      }
      __syncthreads();

      // ---- 7a. O = scale (Q e^G S0 + A_qk U), stored for valid rows ----
      for (int it = tid; it < (C / 2) * (VT / 4); it += kThreads) {
        const int r = 2 * (it / (VT / 4)), j = 4 * (it % (VT / 4));
        float a0[4] = {}, a1[4] = {};
        for (int c = 0; c < K; ++c) {
          const float q0 = sQ[r * LDK + c], q1 = sQ[(r + 1) * LDK + c];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float s = sS[c * VT + j + t];
            a0[t] = fmaf(q0, s, a0[t]);
            a1[t] = fmaf(q1, s, a1[t]);
          }
        }
        for (int jj = 0; jj <= r + 1; ++jj) {
          const float m0 = sAqk[r * LDA + jj], m1 = sAqk[(r + 1) * LDA + jj];
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const float uu = sU[jj * VT + j + t];
            a0[t] = fmaf(m0, uu, a0[t]);
            a1[t] = fmaf(m1, uu, a1[t]);
          }
        }
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          if (r + rr < n) {
            Tin *dst = go + ((tok0 + r + rr) * H + u.h) * V + v0 + j;
#pragma unroll
            for (int t = 0; t < 4; ++t)
              dst[t] = from_f32<Tin>(p.scale * (rr ? a1[t] : a0[t]));
          }
        }
      }

      // ---- 7b. S1 = diag(e^{G_C}) S0 + (K e^{G_C-G})^T U (4x4 per item) ----
      constexpr int kItemsS = (K / 4) * (VT / 4);
      static_assert(kItemsS <= kThreads, "one state item per thread");
      float snew[4][4];
      const bool has_s = tid < kItemsS;
      const int sc = 4 * (tid / (VT / 4)), sj = 4 * (tid % (VT / 4));
      if (has_s) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int t = 0; t < 4; ++t)
            snew[i][t] = sGam[sc + i] * sS[(sc + i) * VT + sj + t];
        for (int r = 0; r < C; ++r) {
          float kh[4], uu[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) kh[i] = sG[r * LDK + sc + i];
#pragma unroll
          for (int t = 0; t < 4; ++t) uu[t] = sU[r * VT + sj + t];
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int t = 0; t < 4; ++t) snew[i][t] = fmaf(kh[i], uu[t], snew[i][t]);
        }
      }
      __syncthreads();  // 7a is done reading S0
      if (has_s) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int t = 0; t < 4; ++t) sS[(sc + i) * VT + sj + t] = snew[i][t];
      }
    }
    __syncthreads();

    if (u.last && p.final_state) {
      for (int i = tid; i < K * VT; i += kThreads) {
        const int c = i / VT, j = i % VT;
        p.final_state[(((size_t)u.b * H + u.h) * K + c) * V + v0 + j] = sS[i];
      }
    }
    __syncthreads();  // sS is reinitialised by the next unit
  }
}

template <int K, int VT, typename Tin>
cudaError_t launch_typed(const FwdParams &p, cudaStream_t stream) {
  using L = SimtSmem<K, VT>;
  auto kern = fwd_simt_kernel<K, VT, Tin>;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::bytes);
  if (e != cudaSuccess) return e;
  const long units_upper = (long)p.B * p.T * p.H * p.n_vtiles;  // >= units
  const long grid_cap = (long)num_sms();
  int grid = (int)(units_upper < grid_cap ? units_upper : grid_cap);
  if (!p.runs.runs) {
    const long units = (long)p.B * p.H * p.n_vtiles;
    grid = (int)(units < grid_cap ? units : grid_cap);
  }
  if (grid < 1) grid = 1;
  kern<<<grid, kThreads, L::bytes, stream>>>(p);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_by_shape(const FwdParams &p, cudaStream_t stream) {
  if (p.v_tile != 32) return cudaErrorNotSupported;
  switch (p.K) {
    case 32: return launch_typed<32, 32, Tin>(p, stream);
    case 64: return launch_typed<64, 32, Tin>(p, stream);
    case 128: return launch_typed<128, 32, Tin>(p, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace

cudaError_t launch_fwd_simt(const FwdParams &p, bool bf16,
                            cudaStream_t stream) {
  return bf16 ? launch_by_shape<__nv_bfloat16>(p, stream)
              : launch_by_shape<float>(p, stream);
}

}  // namespace kda
