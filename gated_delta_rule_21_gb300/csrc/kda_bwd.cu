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
// shared memory and walked backwards.  512 threads: warp w owns the tile's
// value columns 2w, 2w + 1 for all keys (lane l: the K / 32 keys from
// (K / 32) l on).
// The value columns are independent in the recurrence, so each warp's chain
// needs only in-warp sums over keys and no block barrier per token; the
// sums over value columns (dq, dk, dg, dbeta) are per-warp partials in
// shared memory, added up every 2 tokens.  This is the first path on the
// CUDA cores (no tensor cores).
#include "kda_internal.cuh"
#include "kda_f32x2.cuh"

namespace kda {
namespace {

constexpr int kBwdThreads = 512;
constexpr int kWarps = kBwdThreads / 32;
constexpr int kVT = 32;   // value columns per CTA
constexpr int kCKB = 8;   // tokens per checkpoint block

constexpr int kCPW = kVT / kWarps;   // value columns per warp
constexpr int kFlush = 2;             // tokens per reduction of the column sums

template <int K>
struct BwdSmem {
  // floats, in order
  static constexpr int Q = 0;                       // q       [kCKB][K]
  static constexpr int KK = Q + kCKB * K;           // k       [kCKB][K]
  static constexpr int E = KK + kCKB * K;           // e^g     [kCKB][K]
  static constexpr int VV = E + kCKB * K;           // v tile  [kCKB][kVT]
  static constexpr int DO = VV + kCKB * kVT;        // do tile [kCKB][kVT]
  static constexpr int BETA = DO + kCKB * kVT;      // beta    [kCKB]
  static constexpr int PQ = BETA + 32;              // per-warp column sums [kFlush][kWarps][K]
  static constexpr int PK = PQ + kFlush * kWarps * K;
  static constexpr int PG = PK + kFlush * kWarps * K;
  static constexpr int PB = PG + kFlush * kWarps * K;   // [kFlush][kWarps]
  static constexpr int BLK = PB + kFlush * kWarps;      // states [kCKB][kVT][K]
  static constexpr int FLOATS = BLK + kCKB * kVT * K;
  static constexpr size_t BYTES = sizeof(float) * (size_t)FLOATS;
};

// x[m] <- the sum of x[m] over the 32 lanes, for N independent values.
template <int N>
__device__ __forceinline__ void warp_sums(float (&x)[N]) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
#pragma unroll
    for (int m = 0; m < N; ++m) x[m] += __shfl_xor_sync(0xffffffffu, x[m], off);
  }
}

// N consecutive floats (N = 1, 2 or 4; src and dst 4N-byte aligned) in one
// load or store.
template <int N>
__device__ __forceinline__ void ld_vec(const float *src, float (&v)[N]) {
  if constexpr (N == 4) {
    const float4 x = *reinterpret_cast<const float4 *>(src);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  } else if constexpr (N == 2) {
    const float2 x = *reinterpret_cast<const float2 *>(src);
    v[0] = x.x; v[1] = x.y;
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) v[i] = src[i];
  }
}
template <int N>
__device__ __forceinline__ void st_vec(float *dst, const float (&v)[N]) {
  if constexpr (N == 4) {
    *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
  } else if constexpr (N == 2) {
    *reinterpret_cast<float2 *>(dst) = make_float2(v[0], v[1]);
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) dst[i] = v[i];
  }
}

// One CTA's walk of one unit.  Lane l of warp w holds the K / 32 consecutive
// keys KPL l .. KPL l + KPL - 1 (one vector load or store of each per-key
// row) for the warp's kCPW value columns.  The state
// recurrence is independent per value column, so a warp's chain needs only
// in-warp sums over keys; the sums over value columns (dq, dk, dg, dbeta)
// are per-warp partials in shared memory, added up every kFlush tokens.
template <typename TI, int K>
struct BwdCta {
  static constexpr int KPL = K / 32;  // keys per lane
  using L = BwdSmem<K>;
  const BwdParams &p;
  float *sm;
  int warp, lane, c0;
  float S[KPL][kCPW], dS[KPL][kCPW];

  __device__ int key0() const { return lane * KPL; }   // this lane's first key

  __device__ BwdCta(const BwdParams &p_, float *sm_) : p(p_), sm(sm_) {
    warp = threadIdx.x >> 5;
    lane = threadIdx.x & 31;
    c0 = warp * kCPW;
  }

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

  __device__ void load_k_e(int tau, float (&kk)[KPL], float (&ee)[KPL]) const {
    ld_vec(sm + L::KK + tau * K + key0(), kk);
    ld_vec(sm + L::E + tau * K + key0(), ee);
  }

  // One forward token on S (the staged token tau).  With an even number of
  // keys per lane, neighbouring keys go through the packed f32x2 FMA pipe as
  // one pair.
  __device__ void fwd_token(int tau) {
    float kk[KPL], ee[KPL], pr[kCPW];
    load_k_e(tau, kk, ee);
    const float bt = sm[L::BETA + tau];
    if constexpr (KPL % 2 == 0) {
      constexpr int NP = KPL / 2;
      u64 k2[NP], pr2[kCPW];
#pragma unroll
      for (int m = 0; m < kCPW; ++m) pr2[m] = pk2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < NP; ++q) {
        k2[q] = pk2(kk[2 * q], kk[2 * q + 1]);
        const u64 e2 = pk2(ee[2 * q], ee[2 * q + 1]);
#pragma unroll
        for (int m = 0; m < kCPW; ++m) {
          const u64 s2 = mul2(pk2(S[2 * q][m], S[2 * q + 1][m]), e2);
          pr2[m] = fma2(s2, k2[q], pr2[m]);
          upk2(s2, S[2 * q][m], S[2 * q + 1][m]);
        }
      }
#pragma unroll
      for (int m = 0; m < kCPW; ++m) {
        float a, b;
        upk2(pr2[m], a, b);
        pr[m] = a + b;
      }
      warp_sums(pr);
      const u64 bt2 = pk2(bt, bt);
#pragma unroll
      for (int m = 0; m < kCPW; ++m) {
        const float r = sm[L::VV + tau * kVT + c0 + m] - pr[m];
        const u64 r2 = pk2(r, r);
#pragma unroll
        for (int q = 0; q < NP; ++q)
          upk2(fma2(mul2(bt2, k2[q]), r2, pk2(S[2 * q][m], S[2 * q + 1][m])), S[2 * q][m],
               S[2 * q + 1][m]);
      }
    } else {
#pragma unroll
      for (int m = 0; m < kCPW; ++m) pr[m] = 0.f;
#pragma unroll
      for (int n = 0; n < KPL; ++n)
#pragma unroll
        for (int m = 0; m < kCPW; ++m) {
          S[n][m] *= ee[n];
          pr[m] = fmaf(S[n][m], kk[n], pr[m]);
        }
      warp_sums(pr);
#pragma unroll
      for (int m = 0; m < kCPW; ++m) {
        const float r = sm[L::VV + tau * kVT + c0 + m] - pr[m];
#pragma unroll
        for (int n = 0; n < KPL; ++n) S[n][m] = fmaf(bt * kk[n], r, S[n][m]);
      }
    }
  }
  // One backward token with one key per lane (K = 32), scalar fp32.
  __device__ void bwd_token_scalar(int tau, int slot, size_t th, int vt) {
    float kk[KPL], ee[KPL], qq[KPL];
    load_k_e(tau, kk, ee);
#pragma unroll
    for (int n = 0; n < KPL; ++n) qq[n] = sm[L::Q + tau * K + key0() + n];
    const float *bk = sm + L::BLK + (size_t)tau * kVT * K;
    const float bt = sm[L::BETA + tau];
    float dov[kCPW], Sp[KPL][kCPW], pr[kCPW], pa[kCPW];
#pragma unroll
    for (int m = 0; m < kCPW; ++m) {
      dov[m] = sm[L::DO + tau * kVT + c0 + m];
      pr[m] = 0.f;
      pa[m] = 0.f;
    }
#pragma unroll
    for (int n = 0; n < KPL; ++n)
#pragma unroll
      for (int m = 0; m < kCPW; ++m) {
        Sp[n][m] = bk[(c0 + m) * K + key0() + n] * ee[n];
        pr[m] = fmaf(Sp[n][m], kk[n], pr[m]);
        dS[n][m] = fmaf(p.scale * qq[n], dov[m], dS[n][m]);   // o_t = scale S_t^T q_t
        pa[m] = fmaf(dS[n][m], kk[n], pa[m]);
      }
    warp_sums(pr);
    warp_sums(pa);
    float r[kCPW], dr[kCPW], db = 0.f;
#pragma unroll
    for (int m = 0; m < kCPW; ++m) {
      r[m] = sm[L::VV + tau * kVT + c0 + m] - pr[m];
      dr[m] = bt * pa[m];
      db = fmaf(pa[m], r[m], db);
    }
    float* const pq = sm + L::PQ + (slot * kWarps + warp) * K;
    float* const pk = sm + L::PK + (slot * kWarps + warp) * K;
    float* const pg = sm + L::PG + (slot * kWarps + warp) * K;
#pragma unroll
    for (int n = 0; n < KPL; ++n) {
      float aq = 0.f, ak = 0.f, ag = 0.f;
#pragma unroll
      for (int m = 0; m < kCPW; ++m) {
        const float st = fmaf(bt * kk[n], r[m], Sp[n][m]);          // S_t
        aq = fmaf(st, dov[m], aq);
        ak += bt * dS[n][m] * r[m] - Sp[n][m] * dr[m];
        const float dsp = fmaf(-kk[n], dr[m], dS[n][m]);           // dS'
        ag = fmaf(Sp[n][m], dsp, ag);
        dS[n][m] = ee[n] * dsp;                                     // gradient of S_{t-1}
      }
      pq[key0() + n] = p.scale * aq;
      pk[key0() + n] = ak;
      pg[key0() + n] = ag;
    }
    if (lane == 0) sm[L::PB + slot * kWarps + warp] = db;
    float drl = dr[0];
#pragma unroll
    for (int m = 1; m < kCPW; ++m)
      if (lane == m) drl = dr[m];
    if (lane < kCPW) p.dv[th * p.V + vt * kVT + c0 + lane] = drl;
  }

  // One backward token (the staged token tau, its entering state in BLK);
  // the per-warp column sums go to slot `slot` of PQ/PK/PG/PB.  With an even
  // number of keys per lane, neighbouring keys are one f32x2 pair, so the
  // per-key values and the state pairs feed the packed FMA pipe and only the
  // per-column scalars are broadcast.
  __device__ void bwd_token(int tau, int slot, size_t th, int vt) {
    if constexpr (KPL % 2 != 0) {
      bwd_token_scalar(tau, slot, th, vt);
    } else {
      constexpr int NP = KPL / 2;
      const float *bk = sm + L::BLK + (size_t)tau * kVT * K;
      const float bt = sm[L::BETA + tau];
      const u64 bt2 = pk2(bt, bt), sc2 = pk2(p.scale, p.scale);
      u64 k2[NP], e2[NP], Sp2[NP][kCPW], dS2[NP][kCPW], dov2[kCPW], pr2[kCPW], pa2[kCPW];
      float dov[kCPW];
#pragma unroll
      for (int m = 0; m < kCPW; ++m) {
        dov[m] = sm[L::DO + tau * kVT + c0 + m];
        dov2[m] = pk2(dov[m], dov[m]);
        pr2[m] = pk2(0.f, 0.f);
        pa2[m] = pk2(0.f, 0.f);
      }
      float kk[KPL], ee[KPL], qq[KPL], sp[kCPW][KPL];
      ld_vec(sm + L::KK + tau * K + key0(), kk);
      ld_vec(sm + L::E + tau * K + key0(), ee);
      ld_vec(sm + L::Q + tau * K + key0(), qq);
#pragma unroll
      for (int m = 0; m < kCPW; ++m) ld_vec(bk + (c0 + m) * K + key0(), sp[m]);
#pragma unroll
      for (int q = 0; q < NP; ++q) {
        k2[q] = pk2(kk[2 * q], kk[2 * q + 1]);
        e2[q] = pk2(ee[2 * q], ee[2 * q + 1]);
        const u64 sq2 = mul2(sc2, pk2(qq[2 * q], qq[2 * q + 1]));
#pragma unroll
        for (int m = 0; m < kCPW; ++m) {
          Sp2[q][m] = mul2(pk2(sp[m][2 * q], sp[m][2 * q + 1]), e2[q]);
          pr2[m] = fma2(Sp2[q][m], k2[q], pr2[m]);
          // o_t = scale S_t^T q_t
          dS2[q][m] = fma2(sq2, dov2[m], pk2(dS[2 * q][m], dS[2 * q + 1][m]));
          pa2[m] = fma2(dS2[q][m], k2[q], pa2[m]);
        }
      }
      float pr[kCPW], pa[kCPW];
#pragma unroll
      for (int m = 0; m < kCPW; ++m) {
        float a, b;
        upk2(pr2[m], a, b);
        pr[m] = a + b;
        upk2(pa2[m], a, b);
        pa[m] = a + b;
      }
      warp_sums(pr);
      warp_sums(pa);
      float r[kCPW], dr[kCPW], db = 0.f;
      u64 r2[kCPW], ndr2[kCPW], btr2[kCPW];
#pragma unroll
      for (int m = 0; m < kCPW; ++m) {
        r[m] = sm[L::VV + tau * kVT + c0 + m] - pr[m];
        dr[m] = bt * pa[m];
        db = fmaf(pa[m], r[m], db);
        r2[m] = pk2(r[m], r[m]);
        ndr2[m] = pk2(-dr[m], -dr[m]);
        btr2[m] = pk2(bt * r[m], bt * r[m]);
      }
      float aq[KPL], ak[KPL], ag[KPL];
#pragma unroll
      for (int q = 0; q < NP; ++q) {
        const u64 btk2 = mul2(bt2, k2[q]);
        u64 aq2 = pk2(0.f, 0.f), ak2 = pk2(0.f, 0.f), ag2 = pk2(0.f, 0.f);
#pragma unroll
        for (int m = 0; m < kCPW; ++m) {
          const u64 st2 = fma2(btk2, r2[m], Sp2[q][m]);             // S_t
          aq2 = fma2(st2, dov2[m], aq2);
          ak2 = fma2(dS2[q][m], btr2[m], ak2);                       // beta dS r
          ak2 = fma2(Sp2[q][m], ndr2[m], ak2);                       // - S' dr
          const u64 dsp2 = fma2(k2[q], ndr2[m], dS2[q][m]);          // dS'
          ag2 = fma2(Sp2[q][m], dsp2, ag2);
          upk2(mul2(e2[q], dsp2), dS[2 * q][m], dS[2 * q + 1][m]);   // gradient of S_{t-1}
        }
        upk2(mul2(sc2, aq2), aq[2 * q], aq[2 * q + 1]);
        upk2(ak2, ak[2 * q], ak[2 * q + 1]);
        upk2(ag2, ag[2 * q], ag[2 * q + 1]);
      }
      st_vec(sm + L::PQ + (slot * kWarps + warp) * K + key0(), aq);
      st_vec(sm + L::PK + (slot * kWarps + warp) * K + key0(), ak);
      st_vec(sm + L::PG + (slot * kWarps + warp) * K + key0(), ag);
      if (lane == 0) sm[L::PB + slot * kWarps + warp] = db;
      float drl = dr[0];
#pragma unroll
      for (int m = 1; m < kCPW; ++m)
        if (lane == m) drl = dr[m];
      if (lane < kCPW) p.dv[th * p.V + vt * kVT + c0 + lane] = drl;
    }
  }

  // The column sums of `count` tokens (slot s = token t_hi - s), over the
  // warps, into this tile's partials.
  __device__ void flush(size_t th_hi, int count, int vt) {
    __syncthreads();
    const size_t nK = (size_t)p.B * p.T * p.H * K;
    for (int idx = threadIdx.x; idx < count * K; idx += kBwdThreads) {
      const int slot = idx / K, i = idx % K;
      float a = 0.f, c = 0.f, d = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        a += sm[L::PQ + (slot * kWarps + w) * K + i];
        c += sm[L::PK + (slot * kWarps + w) * K + i];
        d += sm[L::PG + (slot * kWarps + w) * K + i];
      }
      const size_t o = (size_t)vt * nK + (th_hi - (size_t)slot * p.H) * K + i;
      p.part_q[o] = a;
      p.part_k[o] = c;
      p.part_g[o] = d;
    }
    if (threadIdx.x < count) {
      const int slot = threadIdx.x;
      float a = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) a += sm[L::PB + slot * kWarps + w];
      p.part_b[(size_t)vt * ((size_t)p.B * p.T * p.H) + th_hi - (size_t)slot * p.H] = a;
    }
    __syncthreads();
  }

  __device__ void run_unit(const Unit &u) {
    const int b = u.b, h = u.h, vt = u.vt;
    const int nck = (u.end - u.start + kCKB - 1) / kCKB;
    float *ck = p.ckpt + (size_t)blockIdx.x * p.ckpt_cta_floats;   // [nck][kVT][K]
    const size_t st0 = ((size_t)b * p.H + h) * K * p.V + (size_t)vt * kVT + c0;
#pragma unroll
    for (int n = 0; n < KPL; ++n)
#pragma unroll
      for (int m = 0; m < kCPW; ++m)
        S[n][m] = (u.first && p.initial_state)
                      ? p.initial_state[st0 + (size_t)(key0() + n) * p.V + m] : 0.f;
    // forward over the run, keeping S at every kCKB-th token
    for (int c = 0; c < nck; ++c) {
      const int t0 = u.start + c * kCKB, n = min(kCKB, u.end - t0);
#pragma unroll
      for (int m = 0; m < kCPW; ++m) {
        float t[KPL];
#pragma unroll
        for (int kn = 0; kn < KPL; ++kn) t[kn] = S[kn][m];
        st_vec(ck + ((size_t)c * kVT + c0 + m) * K + key0(), t);
      }
      stage(b, h, vt, t0, n, false);
      __syncthreads();
      for (int tau = 0; tau < n; ++tau) fwd_token(tau);
      __syncthreads();
    }
    // backward, block by block from the end
#pragma unroll
    for (int n = 0; n < KPL; ++n)
#pragma unroll
      for (int m = 0; m < kCPW; ++m)
        dS[n][m] = (u.last && p.d_final)
                       ? p.d_final[st0 + (size_t)(key0() + n) * p.V + m] : 0.f;
    for (int c = nck - 1; c >= 0; --c) {
      const int t0 = u.start + c * kCKB, n = min(kCKB, u.end - t0);
#pragma unroll
      for (int m = 0; m < kCPW; ++m) {
        float t[KPL];
        ld_vec(ck + ((size_t)c * kVT + c0 + m) * K + key0(), t);
#pragma unroll
        for (int kn = 0; kn < KPL; ++kn) S[kn][m] = t[kn];
      }
      stage(b, h, vt, t0, n, true);
      __syncthreads();
      for (int tau = 0; tau < n; ++tau) {   // replay: the state entering each token
        float *bk = sm + L::BLK + (size_t)tau * kVT * K;
#pragma unroll
        for (int m = 0; m < kCPW; ++m) {
          float t[KPL];
#pragma unroll
          for (int kn = 0; kn < KPL; ++kn) t[kn] = S[kn][m];
          st_vec(bk + (c0 + m) * K + key0(), t);
        }
        if (tau + 1 < n) fwd_token(tau);
      }
      for (int hi = n - 1; hi >= 0; hi -= kFlush) {   // groups of kFlush tokens
        const int count = min(kFlush, hi + 1);
        for (int s = 0; s < count; ++s)
          bwd_token(hi - s, s, ((size_t)b * p.T + t0 + hi - s) * p.H + h, vt);
        flush(((size_t)b * p.T + t0 + hi) * p.H + h, count, vt);
      }
    }
    if (u.first && p.d_initial) {
#pragma unroll
      for (int n = 0; n < KPL; ++n)
#pragma unroll
        for (int m = 0; m < kCPW; ++m)
          p.d_initial[st0 + (size_t)(key0() + n) * p.V + m] = dS[n][m];
    }
  }
};

template <typename TI, int K>
__global__ void __launch_bounds__(kBwdThreads, 1) bwd_simt_kernel(const BwdParams p) {
  extern __shared__ __align__(16) float bwd_sm[];
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
