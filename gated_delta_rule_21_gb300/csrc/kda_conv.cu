// kda_conv.cu -- short-convolution prologue of the KDA layer.
//
// Page "feat(kda): integrate KDA attention with tokamax backend and CP
// support", section "Layer architecture", step 1: Q, K and V each pass
// through a causal depthwise 1-D convolution of width 4 with SiLU; step 5
// (and "Public API", use_qk_l2norm_in_kernel): optional L2 normalisation of
// q and k.  The convolution is segment-aware: a tap counts only when it lies
// in the same run of equal non-zero segment ids as the output token.
//
//     y_t[c] = SiLU( sum_{i=0}^{3} w[c][3-i] x_{t-i}[c] ),  SiLU(z) = z/(1+e^-z)
//     q, k  <- y / sqrt(sum_head y^2 + 1e-6)        (when l2norm_qk)
//
// Padding tokens (id 0) give y = 0.  Every element is read once and written
// once, so the kernel should be bound by HBM bandwidth; its layout serves the
// memory system and keeps the instruction count per element low.
//   * Each thread owns 8 consecutive channels; a CTA of 128 threads covers
//     1024 channels of one tensor for 24 tokens.
//   * The CTA's input rows (its tokens and the 3 before them) are staged in
//     shared memory by 16-byte cp.async copies that each thread issues for
//     its own channels, in two groups: the copies of the second group stay
//     in flight while the first is computed, and no register holds a load.
//   * The window of the 3 previous inputs lives in registers; tokens are
//     processed 6 per loop iteration (a multiple of the window length), so
//     the window rotates without register moves.
//   * Segments: a tile whose rows all lie in one run of ids takes a path
//     with no per-token tests.  Otherwise the window is cleared where a new
//     run starts (so the taps need no per-channel predicates) and a padding
//     token skips the arithmetic.
//   * The taps, SiLU and the sum of squares run on channel pairs with the
//     packed f32x2 instructions of the FMA pipe.  SiLU(z) = z * rcp(1 +
//     2^(-z log2 e)) takes two approximate special-function instructions (a
//     few ulp of relative error); for z < -87 the exponential flushes to
//     +inf or its reciprocal to 0, giving -0 (the exact value is below 1e-36
//     in size).
//   * A head of K channels is K/8 adjacent lanes, so the L2 norm of q and k
//     is a shuffle reduction inside the warp, done for 3 tokens at a time.
#include "kda_internal.cuh"
#include "kda_f32x2.cuh"

namespace kda {
namespace {

constexpr int kThreads = 128;
constexpr int kVec = 8;      // channels per thread
constexpr int kW = 4;        // conv width
constexpr int kTT = 24;      // tokens per CTA
constexpr int kIter = 6;     // tokens per loop iteration (a multiple of kW - 1)
constexpr int kBatch = 3;    // tokens per shuffle batch
constexpr int kHalf = kTT / 2;  // tokens per cp.async group
constexpr int kRows = kTT + kW - 1;
static_assert(kIter % (kW - 1) == 0 && kIter % kBatch == 0 && kHalf % kIter == 0, "tile shape");

// Flags of a staged row: a new run of segment ids starts here (the window
// is cleared), or the row is padding / outside [0, T) (y = 0).
constexpr int kRowReset = 1, kRowPad = 2;

template <typename T>
constexpr size_t conv_smem_bytes() {
  return (size_t)kRows * kThreads * kVec * sizeof(T);
}

// 16-byte global -> shared copy; src_bytes = 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Wait until at most `pending` of this thread's copy groups are in flight.
__device__ __forceinline__ void cp_async_wait(int pending) {
  if (pending == 0) asm volatile("cp.async.wait_group 0;" ::: "memory");
  else asm volatile("cp.async.wait_group 1;" ::: "memory");
}

__device__ __forceinline__ float sfu_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float sfu_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 8 channels of one staged row (shared layout [row][16-byte piece][thread]).
__device__ __forceinline__ void lds8(const unsigned char *row, int tid, const __nv_bfloat16 *,
                                     float (&f)[kVec]) {
  const uint4 a = *reinterpret_cast<const uint4 *>(row + (size_t)tid * 16);
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void lds8(const unsigned char *row, int tid, const float *,
                                     float (&f)[kVec]) {
  const float4 a = *reinterpret_cast<const float4 *>(row + (size_t)tid * 16);
  const float4 b = *reinterpret_cast<const float4 *>(row + (size_t)(kThreads + tid) * 16);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__device__ __forceinline__ void store8(__nv_bfloat16 *p, const float (&f)[kVec]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t *>(&h);
  }
  *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}
__device__ __forceinline__ void store8(float *p, const float (&f)[kVec]) {
  *reinterpret_cast<float4 *>(p) = make_float4(f[0], f[1], f[2], f[3]);
  *reinterpret_cast<float4 *>(p + 4) = make_float4(f[4], f[5], f[6], f[7]);
}

// The register state of one thread and the per-tile loop.  GENERAL tiles
// test every row's flags; plain tiles (one run throughout) do not.
template <typename T, int KL>
struct ConvThread {
  static constexpr int kPieces = kVec * (int)sizeof(T) / 16;   // 16-byte pieces per row
  static constexpr int kRowBytes = kPieces * kThreads * 16;
  const unsigned char *smem;
  const int *flags;
  int tid;
  float wt[kVec][kW];                           // wt[c][3] multiplies x_t
  float win[kW - 1][kVec];                      // x_{t-3}, x_{t-2}, x_{t-1} of t's run

  __device__ __forceinline__ void shift_in(const float (&xt)[kVec]) {
#pragma unroll
    for (int c = 0; c < kVec; ++c) {
      win[0][c] = win[1][c];
      win[1][c] = win[2][c];
      win[2][c] = xt[c];
    }
  }
  __device__ __forceinline__ void clear_window() {
#pragma unroll
    for (int i = 0; i < kW - 1; ++i)
#pragma unroll
      for (int c = 0; c < kVec; ++c) win[i][c] = 0.f;
  }
  __device__ __forceinline__ void load_row(int r, float (&xr)[kVec]) const {
    lds8(smem + (size_t)r * kRowBytes, tid, (const T *)nullptr, xr);
  }

  template <bool GENERAL>
  __device__ __forceinline__ void run(T *y, int t0, int T_len, bool active, bool norm, int C) {
    // The 3 rows before the tile, run by run.
    cp_async_wait(1);
    clear_window();
#pragma unroll
    for (int r = 0; r < kW - 1; ++r) {
      float xr[kVec];
      load_row(r, xr);
      if (GENERAL && (flags[r] & kRowReset)) clear_window();
      shift_in(xr);
    }
#pragma unroll 1
    for (int i0 = 0; i0 < kTT; i0 += kIter) {
      if (i0 == kHalf) cp_async_wait(0);        // the second group's rows
#pragma unroll
      for (int j0 = 0; j0 < kIter; j0 += kBatch) {
        float out[kBatch][kVec], ss[kBatch];
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int r = kW - 1 + i0 + j0 + j;   // staged row of the token
          float xt[kVec];
          load_row(r, xt);
          int fl = 0;
          if (GENERAL) {
            fl = flags[r];
            if (fl & kRowReset) clear_window();
          }
          ss[j] = 0.f;
          if (GENERAL && (fl & kRowPad)) {
#pragma unroll
            for (int c = 0; c < kVec; ++c) out[j][c] = 0.f;
          } else {
            constexpr float kNegLog2e = -1.4426950408889634f;
            u64 ss2 = pk2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < kVec; c += 2) {   // channels c, c + 1
              u64 acc = mul2(pk2(wt[c][kW - 1], wt[c + 1][kW - 1]), pk2(xt[c], xt[c + 1]));
              acc = fma2(pk2(wt[c][kW - 2], wt[c + 1][kW - 2]), pk2(win[2][c], win[2][c + 1]), acc);
              acc = fma2(pk2(wt[c][kW - 3], wt[c + 1][kW - 3]), pk2(win[1][c], win[1][c + 1]), acc);
              acc = fma2(pk2(wt[c][kW - 4], wt[c + 1][kW - 4]), pk2(win[0][c], win[0][c + 1]), acc);
              float e0, e1, d0, d1;
              upk2(mul2(acc, pk2(kNegLog2e, kNegLog2e)), e0, e1);
              upk2(add2(pk2(1.f, 1.f), pk2(sfu_ex2(e0), sfu_ex2(e1))), d0, d1);
              const u64 o = mul2(acc, pk2(sfu_rcp(d0), sfu_rcp(d1)));   // SiLU
              upk2(o, out[j][c], out[j][c + 1]);
              ss2 = fma2(o, o, ss2);
            }
            float s0, s1;
            upk2(ss2, s0, s1);
            ss[j] = s0 + s1;
          }
          shift_in(xt);
        }
        if (norm) {
#pragma unroll
          for (int off = 1; off < KL; off <<= 1) {
#pragma unroll
            for (int j = 0; j < kBatch; ++j) ss[j] += __shfl_xor_sync(0xffffffffu, ss[j], off);
          }
#pragma unroll
          for (int j = 0; j < kBatch; ++j) {
            const float rs = rsqrtf(ss[j] + 1e-6f);
            const u64 rs2 = pk2(rs, rs);
#pragma unroll
            for (int c = 0; c < kVec; c += 2)
              upk2(mul2(pk2(out[j][c], out[j][c + 1]), rs2), out[j][c], out[j][c + 1]);
          }
        }
#pragma unroll
        for (int j = 0; j < kBatch; ++j) {
          const int t = t0 + i0 + j0 + j;
          if (active && (!GENERAL || t < T_len)) store8(y + (size_t)t * C, out[j]);
        }
      }
    }
  }
};

// KL = lanes per q/k head = K / 8.
template <typename T, int KL>
__global__ void __launch_bounds__(kThreads, 4)
    short_conv_kernel(const ConvParams p) {
  extern __shared__ __align__(16) unsigned char conv_smem[];
  __shared__ int s_flags[kRows];
  using Th = ConvThread<T, KL>;

  const int tid = threadIdx.x;
  const int z = blockIdx.z;                    // 0 = q, 1 = k, 2 = v
  const int D = z < 2 ? p.K : p.V;
  const int C = p.H * D;                       // channels of this tensor
  const int ch = (blockIdx.x * kThreads + tid) * kVec;
  const int tiles_per_row = (p.T + kTT - 1) / kTT;
  const int b = blockIdx.y / tiles_per_row;
  const int t0 = (blockIdx.y % tiles_per_row) * kTT;
  if (blockIdx.x * kThreads * kVec >= C) return;  // whole CTA idle (uniform)

  // A head is D/8 adjacent lanes (C and 1024 are multiples of D), so a head
  // is either wholly active or wholly idle; idle lanes stage zeros and still
  // take part in the shuffles.
  const bool active = ch < C;
  // (selected, not indexed by z: a dynamic index would copy the parameter
  // arrays to local memory)
  const void *xz = z == 0 ? p.x[0] : z == 1 ? p.x[1] : p.x[2];
  void *yz = z == 0 ? p.y[0] : z == 1 ? p.y[1] : p.y[2];
  const T *x = static_cast<const T *>(xz) + (size_t)b * p.T * C;
  T *y = static_cast<T *>(yz) + (size_t)b * p.T * C + ch;

  // Stage rows t0-3 .. t0+kTT-1 (row r holds token t0 - 3 + r): group 0 the
  // 3 rows before the tile and its first half, group 1 the second half.
  // Rows outside [0, T) and idle channels are zero-filled.
  const uint32_t sbase = static_cast<uint32_t>(__cvta_generic_to_shared(conv_smem));
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int r0 = g == 0 ? 0 : kW - 1 + kHalf;
    const int r1 = g == 0 ? kW - 1 + kHalf : kRows;
#pragma unroll 1
    for (int r = r0; r < r1; ++r) {
      const int t = t0 - (kW - 1) + r;
      const bool ok = active && t >= 0 && t < p.T;
      const T *src = ok ? x + (size_t)t * C + ch : x;
#pragma unroll
      for (int pc = 0; pc < Th::kPieces; ++pc)
        cp_async16(sbase + (uint32_t)(r * Th::kRowBytes + (pc * kThreads + tid) * 16),
                   src + pc * (16 / (int)sizeof(T)), ok ? 16 : 0);
    }
    cp_async_commit();
  }

  int irregular = 0;
  if (tid < kRows) {
    const int t = t0 - (kW - 1) + tid;
    auto id = [&](int tt) {
      if (tt < 0 || tt >= p.T) return 0;
      return p.segment_ids ? p.segment_ids[(size_t)b * p.T + tt] : 1;
    };
    const int sv = id(t);
    const int fl = (sv == 0 ? kRowPad : 0) | (sv != id(t - 1) ? kRowReset : 0);
    s_flags[tid] = fl;
    irregular = (fl & kRowPad) || (tid > 0 && (fl & kRowReset));
  }
  Th th;
  th.smem = conv_smem;
  th.flags = s_flags;
  th.tid = tid;
  size_t w_off = 0;
  if (z >= 1) w_off += (size_t)p.H * p.K * kW;
  if (z >= 2) w_off += (size_t)p.H * p.K * kW;
#pragma unroll
  for (int c = 0; c < kVec; ++c) {
    float4 wv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active) wv = *reinterpret_cast<const float4 *>(p.w + w_off + (size_t)(ch + c) * kW);
    th.wt[c][0] = wv.x; th.wt[c][1] = wv.y; th.wt[c][2] = wv.z; th.wt[c][3] = wv.w;
  }
  // s_flags visible; the tile is plain when all its rows lie in one run
  const bool general = __syncthreads_or(irregular) != 0;
  const bool norm = z < 2 && p.l2norm_qk;
  if (general) th.template run<true>(y, t0, p.T, active, norm, C);
  else th.template run<false>(y, t0, p.T, active, norm, C);
}

template <typename T>
cudaError_t launch_conv_t(const ConvParams &p, dim3 grid, cudaStream_t stream) {
  auto kern = p.K == 32 ? short_conv_kernel<T, 4>
            : p.K == 64 ? short_conv_kernel<T, 8>
                        : short_conv_kernel<T, 16>;
  // The staged rows exceed the default 48 KB of dynamic shared memory.
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)conv_smem_bytes<T>());
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, conv_smem_bytes<T>(), stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_short_conv(const ConvParams &p, bool bf16,
                              cudaStream_t stream) {
  if (p.K != 32 && p.K != 64 && p.K != 128) return cudaErrorNotSupported;
  const int max_c = p.H * (p.K > p.V ? p.K : p.V);
  const int per_cta = kThreads * kVec;
  const long long tiles = (long long)p.B * ((p.T + kTT - 1) / kTT);
  if (tiles > 65535) return cudaErrorNotSupported;
  dim3 grid((max_c + per_cta - 1) / per_cta, (unsigned)tiles, 3);
  return bf16 ? launch_conv_t<__nv_bfloat16>(p, grid, stream)
              : launch_conv_t<float>(p, grid, stream);
}

}  // namespace kda
