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
// Padding tokens (id 0) give y = 0.  One CTA of 128 threads (one channel
// each) covers 32 tokens of one row for one of the three tensors.
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kThreads = 128;
constexpr int kTT = 32;   // tokens per CTA
constexpr int kW = 4;     // conv width

template <typename T>
__global__ void __launch_bounds__(kThreads)
    short_conv_kernel(const ConvParams p) {
  __shared__ int s_seg[kTT + kW - 1];
  __shared__ float s_part[kThreads / 32][kTT];

  const int z = blockIdx.z;                    // 0 = q, 1 = k, 2 = v
  const int D = z < 2 ? p.K : p.V;
  const int C = p.H * D;                       // channels of this tensor
  const int ch = blockIdx.x * kThreads + threadIdx.x;
  const int tiles_per_row = (p.T + kTT - 1) / kTT;
  const int b = blockIdx.y / tiles_per_row;
  const int t0 = (blockIdx.y % tiles_per_row) * kTT;
  if (blockIdx.x * kThreads >= C) return;      // whole CTA idle (uniform)

  for (int i = threadIdx.x; i < kTT + kW - 1; i += kThreads) {
    const int t = t0 - (kW - 1) + i;
    int s = 0;
    if (t >= 0 && t < p.T) s = p.segment_ids ? p.segment_ids[(size_t)b * p.T + t] : 1;
    s_seg[i] = s;
  }
  __syncthreads();

  const bool active = ch < C;                  // C is a multiple of 32
  const T *x = static_cast<const T *>(p.x[z]);
  T *y = static_cast<T *>(p.y[z]);
  size_t w_off = 0;
  if (z >= 1) w_off += (size_t)p.H * p.K * kW;
  if (z >= 2) w_off += (size_t)p.H * p.K * kW;
  float4 wv = make_float4(0.f, 0.f, 0.f, 0.f);
  if (active) wv = *reinterpret_cast<const float4 *>(p.w + w_off + (size_t)ch * kW);
  const float wt[kW] = {wv.x, wv.y, wv.z, wv.w};  // wt[3] * x_t

  float win[kW - 1] = {0.f, 0.f, 0.f};         // x_{t-3}, x_{t-2}, x_{t-1}
  if (active) {
#pragma unroll
    for (int i = 0; i < kW - 1; ++i) {
      const int t = t0 - (kW - 1) + i;
      win[i] = t >= 0 ? to_f32(x[((size_t)b * p.T + t) * C + ch]) : 0.f;
    }
  }
  float out[kTT];
#pragma unroll
  for (int i = 0; i < kTT; ++i) {
    const int t = t0 + i;
    float xt = 0.f;
    if (active && t < p.T) xt = to_f32(x[((size_t)b * p.T + t) * C + ch]);
    const int s = s_seg[i + kW - 1];
    float acc = 0.f;
    if (s != 0) {
      acc = wt[kW - 1] * xt;
      bool same = true;
#pragma unroll
      for (int j = 1; j < kW; ++j) {           // tap x_{t-j}
        same = same && (s_seg[i + kW - 1 - j] == s);
        if (same) acc = fmaf(wt[kW - 1 - j], win[kW - 1 - j], acc);
      }
      acc = acc / (1.f + expf(-acc));
    }
    out[i] = acc;
    win[0] = win[1];
    win[1] = win[2];
    win[2] = xt;
  }

  if (z < 2 && p.l2norm_qk) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < kTT; ++i) {
      float ss = out[i] * out[i];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      if (lane == 0) s_part[warp][i] = ss;
    }
    __syncthreads();
    // Warps of this thread's head inside the CTA: D/32 warps, head-aligned
    // because 128 % D == 0 and CTAs start on multiples of 128 channels.
    const int wph = D / 32;
    const int w0 = (warp / wph) * wph;
#pragma unroll
    for (int i = 0; i < kTT; ++i) {
      float ss = 0.f;
      for (int j = 0; j < wph; ++j) ss += s_part[w0 + j][i];
      out[i] *= rsqrtf(ss + 1e-6f);
    }
  }

  if (active) {
#pragma unroll
    for (int i = 0; i < kTT; ++i) {
      const int t = t0 + i;
      if (t < p.T) y[((size_t)b * p.T + t) * C + ch] = from_f32<T>(out[i]);
    }
  }
}

}  // namespace

cudaError_t launch_short_conv(const ConvParams &p, bool bf16,
                              cudaStream_t stream) {
  const int max_c = p.H * (p.K > p.V ? p.K : p.V);
  dim3 grid((max_c + kThreads - 1) / kThreads,
            p.B * ((p.T + kTT - 1) / kTT), 3);
  if (bf16)
    short_conv_kernel<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(p);
  else
    short_conv_kernel<float><<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace kda
