// kda_bwd.cu -- gradient of the KDA forward (its vector-Jacobian product) on
// the CUDA cores, fp32.
//
// Page "feat(kda): integrate KDA attention with tokamax backend and CP
// support", section "Delta Rule formulation": per (b, h) and token t of a run
//     S' = diag(e^{g_t}) S_{t-1},  r = v_t - S'^T k_t,
//     S_t = S' + beta_t k_t r^T,   o_t = scale * S_t^T q_t,
// with the packed runs of section "Public API".  Given do (the gradient of o)
// and d_final (of the final state), reverse-mode differentiation of that
// recurrence, one token at a time from the last, with dS the gradient of S_t:
//     dS += scale q_t do_t^T;            dq_t = scale S_t do_t
//     a = dS^T k_t;  dr = beta_t a;      dbeta_t = a . r;  dv_t = dr
//     dk_t = beta_t dS r - S' dr;        dS' = dS - k_t dr^T
//     dg_t[i] = sum_j S'[i][j] dS'[i][j]; dS <- diag(e^{g_t}) dS'
// A run's backward stops at its first token; the row's first run hands dS to
// d_initial.  The value columns are independent in S, so one CTA takes one
// (run, head, 32-column value tile) and dq, dk, dg, dbeta (sums over all
// value columns) are written per tile and summed by a second kernel.
//
// The states S_{t-1} are recomputed: a forward pass over the run keeps S at
// every 8th token (global scratch, per CTA); then, block by block from the
// end, the block is replayed from its checkpoint with the states kept in
// shared memory and walked backwards.  256 threads: warp w owns keys
// w K/8 .. (w+1) K/8 - 1, lane = value column; sums over keys go through
// shared memory, sums over value columns are butterfly reductions inside the
// warp.  This is the first correct path (no tensor cores).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kBwdThreads = 256;
constexpr int kWarps = kBwdThreads / 32;
constexpr int kVT = 32;   // value columns per CTA
constexpr int kCKB = 8;   // tokens per checkpoint block

template <int K>
struct BwdSmem {
  // floats, in order
  static constexpr int Q = 0;                       // q       [kCKB][K]
  static constexpr int KK = Q + kCKB * K;           // k       [kCKB][K]
  static constexpr int E = KK + kCKB * K;           // e^g     [kCKB][K]
  static constexpr int VV = E + kCKB * K;           // v tile  [kCKB][kVT]
  static constexpr int DO = VV + kCKB * kVT;        // do tile [kCKB][kVT]
  static constexpr int BETA = DO + kCKB * kVT;      // beta    [kCKB]
  static constexpr int RED = BETA + 32;             // [2 parities][2][kWarps][kVT]
  static constexpr int BLK = RED + 2 * 2 * kWarps * kVT;  // states [kCKB][K][kVT]
  static constexpr int FLOATS = BLK + kCKB * K * kVT;
  static constexpr size_t BYTES = sizeof(float) * (size_t)FLOATS;
};

// N values per lane (N = 4, 8 or 16, one per key of the warp); returns the
// sum over the 32 lanes for key (lane >> (5 - log2 N)) & (N - 1), in every
// lane.  Each step halves the values a lane keeps and adds its partner's.
template <int N>
__device__ __forceinline__ float lane_sum_transposed(const float (&v)[N], int lane) {
  float cur[N];
#pragma unroll
  for (int i = 0; i < N; ++i) cur[i] = v[i];
  int off = 16;
#pragma unroll
  for (int n = N; n > 1; n >>= 1, off >>= 1) {
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = up ? cur[i] : cur[i + n / 2];
      const float keep = up ? cur[i + n / 2] : cur[i];
      cur[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  float d = cur[0];
#pragma unroll
  for (; off >= 1; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
  return d;
}

template <int N>
__host__ __device__ constexpr int log2_of() { return N == 4 ? 2 : N == 8 ? 3 : 4; }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

template <typename TI, int K>
struct BwdCta {
  static constexpr int KPW = K / kWarps;  // keys per warp
  using L = BwdSmem<K>;
  const BwdParams &p;
  float *sm;
  int warp, lane, i0;
  int par = 0;                            // reduction buffer of this token
  float S[KPW], dS[KPW];

  __device__ BwdCta(const BwdParams &p_, float *sm_) : p(p_), sm(sm_) {
    warp = threadIdx.x >> 5;
    lane = threadIdx.x & 31;
    i0 = warp * KPW;
  }
  __device__ float *red(int which, int w) { return sm + L::RED + ((par * 2 + which) * kWarps + w) * kVT; }

  // Tokens t0 .. t0 + n - 1 of row b, head h, into shared memory (q and do
  // only for the backward walk).
  __device__ void stage(int b, int h, int vt, int t0, int n, bool with_bwd) {
    const size_t HK = (size_t)p.H * K, HV = (size_t)p.H * p.V;
    for (int idx = threadIdx.x; idx < kCKB * K; idx += kBwdThreads) {
      const int tau = idx / K, i = idx % K;
      float kv = 0.f, ev = 1.f, qv = 0.f;
      if (tau < n) {
        const size_t off = ((size_t)b * p.T + t0 + tau) * HK + (size_t)h * K + i;
        kv = to_f32(static_cast<const TI *>(p.k)[off]);
        ev = expf(p.g[off]);
        if (with_bwd) qv = to_f32(static_cast<const TI *>(p.q)[off]);
      }
      sm[L::KK + idx] = kv;
      sm[L::E + idx] = ev;
      sm[L::Q + idx] = qv;
    }
    for (int idx = threadIdx.x; idx < kCKB * kVT; idx += kBwdThreads) {
      const int tau = idx / kVT, j = idx % kVT;
      float vv = 0.f, dv = 0.f;
      if (tau < n) {
        const size_t off = ((size_t)b * p.T + t0 + tau) * HV + (size_t)h * p.V + vt * kVT + j;
        vv = to_f32(static_cast<const TI *>(p.v)[off]);
        if (with_bwd) dv = to_f32(static_cast<const TI *>(p.d_o)[off]);
      }
      sm[L::VV + idx] = vv;
      sm[L::DO + idx] = dv;
    }
    if (threadIdx.x < kCKB) {
      const int tau = threadIdx.x;
      sm[L::BETA + tau] =
          tau < n ? p.beta[((size_t)b * p.T + t0 + tau) * p.H + h] : 0.f;
    }
  }

  // One forward token on S (the staged token tau).
  __device__ void fwd_token(int tau) {
    const float *kt = sm + L::KK + tau * K + i0, *et = sm + L::E + tau * K + i0;
    float pr = 0.f;
#pragma unroll
    for (int m = 0; m < KPW; ++m) {
      S[m] *= et[m];
      pr = fmaf(S[m], kt[m], pr);
    }
    red(0, warp)[lane] = pr;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tot += red(0, w)[lane];
    const float r = sm[L::VV + tau * kVT + lane] - tot;
    const float bt = sm[L::BETA + tau];
#pragma unroll
    for (int m = 0; m < KPW; ++m) S[m] = fmaf(bt * kt[m], r, S[m]);
    par ^= 1;
  }


  // One backward token (the staged token tau, its entering state in BLK);
  // th = (b T + t) H + h.
  __device__ void bwd_token(int tau, size_t th, int vt) {
    const float *kt = sm + L::KK + tau * K + i0, *et = sm + L::E + tau * K + i0;
    const float *qt = sm + L::Q + tau * K + i0;
    const float *bk = sm + L::BLK + (size_t)tau * K * kVT;
    const float bt = sm[L::BETA + tau], dov = sm[L::DO + tau * kVT + lane];
    float Sp[KPW];
    float pr = 0.f, pa = 0.f;
#pragma unroll
    for (int m = 0; m < KPW; ++m) {
      Sp[m] = bk[(i0 + m) * kVT + lane] * et[m];
      pr = fmaf(Sp[m], kt[m], pr);
      dS[m] = fmaf(p.scale * qt[m], dov, dS[m]);   // o_t = scale S_t^T q_t
      pa = fmaf(dS[m], kt[m], pa);
    }
    red(0, warp)[lane] = pr;
    red(1, warp)[lane] = pa;
    __syncthreads();
    float rs = 0.f, as = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      rs += red(0, w)[lane];
      as += red(1, w)[lane];
    }
    const float r = sm[L::VV + tau * kVT + lane] - rs;   // r_j
    const float dr = bt * as;                              // dr_j
    float vq[KPW], vk[KPW], vg[KPW];
#pragma unroll
    for (int m = 0; m < KPW; ++m) {
      const float st = fmaf(bt * kt[m], r, Sp[m]);         // S_t[i][j]
      vq[m] = st * dov;
      vk[m] = bt * dS[m] * r - Sp[m] * dr;
      const float dsp = fmaf(-kt[m], dr, dS[m]);          // dS'[i][j]
      vg[m] = Sp[m] * dsp;
      dS[m] = et[m] * dsp;                                 // gradient of S_{t-1}
    }
    const float sq = lane_sum_transposed<KPW>(vq, lane);
    const float sk = lane_sum_transposed<KPW>(vk, lane);
    const float sg = lane_sum_transposed<KPW>(vg, lane);
    const float db = warp_sum(as * r);
    constexpr int SH = 5 - log2_of<KPW>();
    const size_t nK = (size_t)p.B * p.T * p.H * K;
    if ((lane & ((1 << SH) - 1)) == 0) {
      const size_t o = (size_t)vt * nK + th * K + i0 + (lane >> SH);
      p.part_q[o] = p.scale * sq;
      p.part_k[o] = sk;
      p.part_g[o] = sg;
    }
    if (warp == 0) {
      p.dv[th * p.V + vt * kVT + lane] = dr;
      if (lane == 0) p.part_b[(size_t)vt * ((size_t)p.B * p.T * p.H) + th] = db;
    }
    par ^= 1;
  }

  __device__ void run_unit(const Unit &u) {
    const int b = u.b, h = u.h, vt = u.vt;
    const int nck = (u.end - u.start + kCKB - 1) / kCKB;
    float *ck = p.ckpt + (size_t)blockIdx.x * p.ckpt_cta_floats;   // [nck][K][kVT]
    const size_t st0 = ((size_t)b * p.H + h) * K * p.V + (size_t)vt * kVT + lane;
#pragma unroll
    for (int m = 0; m < KPW; ++m)
      S[m] = (u.first && p.initial_state) ? p.initial_state[st0 + (size_t)(i0 + m) * p.V] : 0.f;
    // forward over the run, keeping S at every kCKB-th token
    for (int c = 0; c < nck; ++c) {
      const int t0 = u.start + c * kCKB, n = min(kCKB, u.end - t0);
#pragma unroll
      for (int m = 0; m < KPW; ++m) ck[((size_t)c * K + i0 + m) * kVT + lane] = S[m];
      stage(b, h, vt, t0, n, false);
      __syncthreads();
      for (int tau = 0; tau < n; ++tau) fwd_token(tau);
      __syncthreads();
    }
    // backward, block by block from the end
#pragma unroll
    for (int m = 0; m < KPW; ++m)
      dS[m] = (u.last && p.d_final) ? p.d_final[st0 + (size_t)(i0 + m) * p.V] : 0.f;
    for (int c = nck - 1; c >= 0; --c) {
      const int t0 = u.start + c * kCKB, n = min(kCKB, u.end - t0);
#pragma unroll
      for (int m = 0; m < KPW; ++m) S[m] = ck[((size_t)c * K + i0 + m) * kVT + lane];
      stage(b, h, vt, t0, n, true);
      __syncthreads();
      for (int tau = 0; tau < n; ++tau) {   // replay: the state entering each token
        float *bk = sm + L::BLK + (size_t)tau * K * kVT;
#pragma unroll
        for (int m = 0; m < KPW; ++m) bk[(i0 + m) * kVT + lane] = S[m];
        if (tau + 1 < n) fwd_token(tau);
      }
      for (int tau = n - 1; tau >= 0; --tau)
        bwd_token(tau, ((size_t)b * p.T + t0 + tau) * p.H + h, vt);
      __syncthreads();
    }
    if (u.first && p.d_initial) {
#pragma unroll
      for (int m = 0; m < KPW; ++m) p.d_initial[st0 + (size_t)(i0 + m) * p.V] = dS[m];
    }
  }
};

template <typename TI, int K>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_simt_kernel(const BwdParams p) {
  extern __shared__ float bwd_sm[];
  BwdCta<TI, K> cta(p, bwd_sm);
  const uint32_t n_units = total_units(p.runs, p.B, p.H, p.n_vtiles);
  for (uint32_t unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
    const Unit u = decode_unit(p.runs, unit, p.B, p.T, p.H, p.n_vtiles);
    cta.run_unit(u);
    __syncthreads();
  }
}

// dq, dk, dg, dbeta = the sum of the value tiles' partials; zero on padding.
__global__ void __launch_bounds__(256)
    bwd_reduce_kernel(int K, int H, int n_vt, size_t nK, size_t nB, const float *pq,
                      const float *pk, const float *pg, const float *pb,
                      const int32_t *seg, float *dq, float *dk, float *dg, float *dbeta) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nK; i += stride) {
    const size_t tok = i / ((size_t)K * H);   // b T + t
    float a = 0.f, c = 0.f, d = 0.f;
    if (!seg || seg[tok] != 0) {
      for (int v = 0; v < n_vt; ++v) {
        a += pq[(size_t)v * nK + i];
        c += pk[(size_t)v * nK + i];
        d += pg[(size_t)v * nK + i];
      }
    }
    dq[i] = a;
    dk[i] = c;
    dg[i] = d;
  }
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nB; i += stride) {
    const size_t tok = i / (size_t)H;
    float a = 0.f;
    if (!seg || seg[tok] != 0)
      for (int v = 0; v < n_vt; ++v) a += pb[(size_t)v * nB + i];
    dbeta[i] = a;
  }
}

template <typename TI, int K>
cudaError_t launch_bwd_t(const BwdParams &p, cudaStream_t stream) {
  const size_t bytes = BwdSmem<K>::BYTES;
  cudaError_t e = cudaFuncSetAttribute(bwd_simt_kernel<TI, K>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  bwd_simt_kernel<TI, K><<<p.grid, kBwdThreads, bytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

bool bwd_supported(int K, int V) {
  return (K == 32 || K == 64 || K == 128) && V >= kVT && V % kVT == 0;
}

size_t bwd_scratch_bytes(int B, int T, int H, int K, int V) {
  const size_t nck = ((size_t)T + kCKB - 1) / kCKB;
  const size_t n_vt = (size_t)V / kVT;
  const size_t nK = (size_t)B * T * H * K, nB = (size_t)B * T * H;
  return align_up(sizeof(float) * kBwdMaxCtas * nck * K * kVT, 256) +
         3 * align_up(sizeof(float) * n_vt * nK, 256) + align_up(sizeof(float) * n_vt * nB, 256);
}

cudaError_t launch_bwd(const BwdParams &p, bool bf16, const int32_t *segment_ids, float *dq,
                       float *dk, float *dg, float *dbeta, cudaStream_t stream) {
  cudaError_t e;
  if (bf16) {
    e = p.K == 32 ? launch_bwd_t<__nv_bfloat16, 32>(p, stream)
      : p.K == 64 ? launch_bwd_t<__nv_bfloat16, 64>(p, stream)
                  : launch_bwd_t<__nv_bfloat16, 128>(p, stream);
  } else {
    e = p.K == 32 ? launch_bwd_t<float, 32>(p, stream)
      : p.K == 64 ? launch_bwd_t<float, 64>(p, stream)
                  : launch_bwd_t<float, 128>(p, stream);
  }
  if (e != cudaSuccess) return e;
  const size_t nK = (size_t)p.B * p.T * p.H * p.K, nB = (size_t)p.B * p.T * p.H;
  const size_t want = (nK + 255) / 256;
  const unsigned grid = (unsigned)(want < 4u * kBwdMaxCtas ? (want > 0 ? want : 1) : 4u * kBwdMaxCtas);
  bwd_reduce_kernel<<<grid, 256, 0, stream>>>(p.K, p.H, p.n_vtiles, nK, nB, p.part_q, p.part_k,
                                             p.part_g, p.part_b, segment_ids, dq, dk, dg, dbeta);
  return cudaGetLastError();
}

}  // namespace kda
