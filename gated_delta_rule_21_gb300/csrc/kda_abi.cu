// kda_abi.cu -- the extern "C" boundary of libkda (declared in include/kda.h).
//
// Every entry point validates its arguments on the host before enqueuing
// anything, maps CUDA errors to kda_status, and never throws.  The forward
// call builds the run list (packed segment ids) and then launches the chunk
// kernel: the tcgen05/TMA tensor-core kernel for bf16 K = V = 128, the fp32
// SIMT kernel otherwise.
#include <stdint.h>
#include <string.h>

#include "kda_internal.cuh"

namespace kda {

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
      cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

namespace {

bool aligned(const void *p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

bool supported_dim(int d) { return d == 32 || d == 64 || d == 128; }

}  // namespace

kda_status check_shape(const kda_shape *s) {
  if (!s) return KDA_ERR_INVALID_ARG;
  if (s->B < 1 || s->T < 1 || s->H < 1) return KDA_ERR_INVALID_ARG;
  if (s->qkv_dtype != KDA_DTYPE_F32 && s->qkv_dtype != KDA_DTYPE_BF16)
    return KDA_ERR_INVALID_ARG;
  if (!supported_dim(s->K) || !supported_dim(s->V)) return KDA_ERR_UNSUPPORTED;
  const long long d = s->K > s->V ? s->K : s->V;
  if ((long long)s->B * s->T * s->H * d >= (1ll << 31)) return KDA_ERR_UNSUPPORTED;
  return KDA_OK;
}

namespace {

// Runs per row the default split workspace is sized for (runs of 64 tokens
// on average).
int default_runs_bound(int T) { return (T + kChunk - 1) / kChunk; }

// AUTO takes the chunk-parallel scan (rows without segment ids) when the
// single chains would leave SMs idle and the segments stay long enough to
// pay for the map pass (about twice the per-chunk work): at least 3
// segments, and 8 or more chunks per segment when there are 8 or more
// segments (the chains would then fill at most a quarter of the SMs), else
// 32 or more.  Measured (default segment count; scan against chain, ms):
// B1 H8 T4096 0.099 / 0.113, B1 H8 T8192 0.146 / 0.208, B1 H8 T32768 0.388 /
// 0.758, B1 H4 T65536 0.406 / 1.348, B1 H16 T8192 0.234 / 0.244, B1 H16
// T16384 0.407 / 0.460, but B1 H16 T4096 (16 chunks per segment) 0.146 /
// 0.134 and B1 H32 T8192 (2 segments) 0.377 / 0.315.
bool scan_preferred(const kda_shape *s) {
  const int P = scan_segments(s->B, s->T, s->H, 0);
  const int nc = (s->T + kChunk - 1) / kChunk;
  const int per_segment = P > 0 ? (nc + P - 1) / P : 0;
  return P >= 3 && per_segment >= (P >= 8 ? 8 : 32);
}

kda_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return KDA_OK;
  if (e == cudaErrorNotSupported) return KDA_ERR_UNSUPPORTED;
  return KDA_ERR_CUDA;
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" {

const char *kda_status_string(kda_status st) {
  switch (st) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported shape, dtype or option";
    case KDA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case KDA_ERR_WORKSPACE: return "workspace missing or too small";
    case KDA_ERR_CUDA: return "CUDA runtime error";
    case KDA_ERR_TIMEOUT: return "device: bounded wait timed out";
    case KDA_ERR_DEVICE: return "device: error reported by a kernel";
  }
  return "unknown status";
}

int kda_version(void) { return KDA_VERSION; }

size_t kda_chunk_fwd_workspace_size(const kda_shape *s, int has_segment_ids) {
  // The size AUTO needs for its fastest kernel on this shape.
  return kda_chunk_fwd_workspace_size_for(s, has_segment_ids, KDA_IMPL_AUTO);
}

size_t kda_chunk_fwd_workspace_size_for(const kda_shape *s, int has_segment_ids,
                                        kda_impl impl) {
  if (check_shape(s) != KDA_OK) return 0;
  const bool has_seg = has_segment_ids != 0;
  const bool bf16 = s->qkv_dtype == KDA_DTYPE_BF16;
  const size_t base = ws_bytes(s->B, s->T, has_seg);
  const bool split_ok = fwd_split_supported(s->K, s->V, bf16, has_seg, 0);
  const size_t split = split_ok ? split_workspace_bytes(s->B, s->T, s->H, has_seg,
                                                        default_runs_bound(s->T))
                                : 0;
  switch (impl) {
    case KDA_IMPL_SIMT:
      return base;
    case KDA_IMPL_TC:
      return fwd_tc_supported(s->K, s->V, bf16, 0) ? base : 0;
    case KDA_IMPL_SPLIT:
      return split;
    case KDA_IMPL_AUTO:
      if (split_ok && !has_seg && scan_preferred(s))
        return scan_workspace_bytes(s->B, s->T, s->H, 0);
      return split_ok ? split : base;
  }
  return 0;
}

size_t kda_chunk_fwd_workspace_size_packed(const kda_shape *s, int max_runs_per_row) {
  if (check_shape(s) != KDA_OK || max_runs_per_row < 1) return 0;
  if (!fwd_split_supported(s->K, s->V, s->qkv_dtype == KDA_DTYPE_BF16, true, 0)) return 0;
  return split_workspace_bytes(s->B, s->T, s->H, true, max_runs_per_row);
}

kda_status kda_chunk_fwd_ex(const kda_shape *s, const void *q, const void *k,
                            const void *v, const float *g, const float *beta,
                            float scale, int chunk_size,
                            const float *initial_state,
                            const int32_t *segment_ids, void *o,
                            float *final_state, void *workspace,
                            size_t workspace_bytes, kda_impl impl, int v_tile,
                            kda_stream_t stream) {
  kda_status st = check_shape(s);
  if (st != KDA_OK) return st;
  if (!q || !k || !v || !g || !beta || !o) return KDA_ERR_INVALID_ARG;
  if (chunk_size != kChunk) return KDA_ERR_UNSUPPORTED;
  if (impl != KDA_IMPL_AUTO && impl != KDA_IMPL_SIMT && impl != KDA_IMPL_TC &&
      impl != KDA_IMPL_SPLIT)
    return KDA_ERR_INVALID_ARG;
  if (v_tile < 0) return KDA_ERR_INVALID_ARG;
  if (!(scale == scale)) return KDA_ERR_INVALID_ARG;  // NaN scale
  const void *ptrs[] = {q, k, v, g, beta, o, initial_state, final_state,
                        segment_ids};
  for (const void *ptr : ptrs)
    if (ptr && !aligned(ptr, 16)) return KDA_ERR_ALIGNMENT;
  const bool has_seg = segment_ids != nullptr;
  if (!workspace || workspace_bytes < ws_bytes(s->B, s->T, has_seg))
    return KDA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return KDA_ERR_ALIGNMENT;

  const bool bf16 = s->qkv_dtype == KDA_DTYPE_BF16;
  const bool tc_ok = fwd_tc_supported(s->K, s->V, bf16, v_tile);
  const bool split_ok = fwd_split_supported(s->K, s->V, bf16, has_seg, v_tile);
  // AUTO takes the split path when the workspace has the default room; with
  // segment ids it also enqueues the fused kernel, which runs only when the
  // runs of this call overflow the split items.  An explicit SPLIT needs
  // room for ceil(T/64) chunks per row at least and reports an overflow in
  // the status word.
  const size_t split_need =
      split_ok ? split_workspace_bytes(s->B, s->T, s->H, has_seg, default_runs_bound(s->T)) : 0;
  const size_t split_min = split_ok ? split_workspace_bytes(s->B, s->T, s->H, has_seg, 0) : 0;
  bool use_tc = false, use_split = false;
  int scan_segs = 0;
  if (impl == KDA_IMPL_AUTO && split_ok && !has_seg && scan_preferred(s) &&
      workspace_bytes >= scan_workspace_bytes(s->B, s->T, s->H, 0))
    scan_segs = scan_segments(s->B, s->T, s->H, 0);
  if (impl == KDA_IMPL_SPLIT) {
    if (!split_ok) return KDA_ERR_UNSUPPORTED;
    if (workspace_bytes < split_min) return KDA_ERR_WORKSPACE;
    use_split = true;
  } else if (impl == KDA_IMPL_TC) {
    if (!tc_ok) return KDA_ERR_UNSUPPORTED;
    use_tc = true;
  } else if (impl == KDA_IMPL_AUTO) {
    // Without segment ids every chunk item must fit; with them the fused
    // fallback covers any overflow, so the minimum split workspace suffices.
    use_split = split_ok && workspace_bytes >= (has_seg && tc_ok ? split_min : split_need);
    use_tc = !use_split && tc_ok;
  }
  if (!use_tc && !use_split) {
    if (v_tile == 0) v_tile = 32;
    if (v_tile != 32 || s->V % v_tile) return KDA_ERR_UNSUPPORTED;
  }

  FwdParams p;
  memset(&p, 0, sizeof(p));
  p.B = s->B; p.T = s->T; p.H = s->H; p.K = s->K; p.V = s->V;
  p.v_tile = v_tile;
  p.n_vtiles = v_tile > 0 ? s->V / v_tile : 0;
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
  p.scale = scale;
  p.initial_state = initial_state;
  p.o = o;
  p.final_state = final_state;
  char *ws = static_cast<char *>(workspace);
  p.status = &reinterpret_cast<WsHeader *>(ws)->status;
  if (has_seg) {
    p.runs.row_offsets = reinterpret_cast<const int32_t *>(ws + sizeof(WsHeader));
    p.runs.runs = reinterpret_cast<const int2 *>(ws + sizeof(WsHeader) +
                                                 ws_row_offsets_bytes(s->B));
    p.runs.total_runs = &reinterpret_cast<WsHeader *>(ws)->total_runs;
  }

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (has_seg) {
    e = launch_segment_runs(s->B, s->T, s->H, s->K, s->V, segment_ids, o,
                            bf16 ? 1 : 0, initial_state, final_state,
                            workspace, cs, use_split);
    if (e != cudaSuccess) return from_cuda(e);
  }
  if (use_split) e = launch_fwd_split(p, workspace, workspace_bytes, cs,
                                      impl == KDA_IMPL_AUTO && tc_ok, scan_segs);
  else if (use_tc) e = launch_fwd_tc(p, cs);
  else e = launch_fwd_simt(p, bf16, cs);
  return from_cuda(e);
}

int kda_chunk_fwd_scan_segments(const kda_shape *s, int n_segments) {
  if (kda_chunk_fwd_scan_workspace_size(s, n_segments) == 0) return 0;
  return scan_segments(s->B, s->T, s->H, n_segments);
}

size_t kda_chunk_fwd_scan_workspace_size(const kda_shape *s, int n_segments) {
  if (check_shape(s) != KDA_OK || n_segments < 0 || n_segments == 1) return 0;
  if (!fwd_split_supported(s->K, s->V, s->qkv_dtype == KDA_DTYPE_BF16, false, 0)) return 0;
  if ((s->T + kChunk - 1) / kChunk < 2) return 0;
  return scan_workspace_bytes(s->B, s->T, s->H, n_segments);
}

kda_status kda_chunk_fwd_scan(const kda_shape *s, const void *q, const void *k, const void *v,
                              const float *g, const float *beta, float scale, int chunk_size,
                              const float *initial_state, void *o, float *final_state,
                              int n_segments, void *workspace, size_t workspace_bytes,
                              kda_stream_t stream) {
  kda_status st = check_shape(s);
  if (st != KDA_OK) return st;
  if (!q || !k || !v || !g || !beta || !o) return KDA_ERR_INVALID_ARG;
  if (chunk_size != kChunk) return KDA_ERR_UNSUPPORTED;
  if (n_segments < 0 || n_segments == 1) return KDA_ERR_INVALID_ARG;
  if (!(scale == scale)) return KDA_ERR_INVALID_ARG;
  const void *ptrs[] = {q, k, v, g, beta, o, initial_state, final_state};
  for (const void *ptr : ptrs)
    if (ptr && !aligned(ptr, 16)) return KDA_ERR_ALIGNMENT;
  const size_t need = kda_chunk_fwd_scan_workspace_size(s, n_segments);
  if (need == 0) return KDA_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < need) return KDA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return KDA_ERR_ALIGNMENT;
  FwdParams p;
  memset(&p, 0, sizeof(p));
  p.B = s->B; p.T = s->T; p.H = s->H; p.K = s->K; p.V = s->V;
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
  p.scale = scale;
  p.initial_state = initial_state;
  p.o = o;
  p.final_state = final_state;
  p.status = &reinterpret_cast<WsHeader *>(workspace)->status;
  const int P = scan_segments(s->B, s->T, s->H, n_segments);
  return from_cuda(launch_fwd_split(p, workspace, workspace_bytes,
                                    reinterpret_cast<cudaStream_t>(stream), false, P));
}

int kda_impl_available(kda_impl impl, const kda_shape *s, int v_tile) {
  if (check_shape(s) != KDA_OK || v_tile < 0) return 0;
  const bool bf16 = s->qkv_dtype == KDA_DTYPE_BF16;
  const bool simt_ok = (v_tile == 0 || v_tile == 32) && s->V % 32 == 0;
  switch (impl) {
    case KDA_IMPL_AUTO: return fwd_tc_supported(s->K, s->V, bf16, v_tile) || simt_ok;
    case KDA_IMPL_SIMT: return simt_ok;
    case KDA_IMPL_TC: return fwd_tc_supported(s->K, s->V, bf16, v_tile);
    case KDA_IMPL_SPLIT: return fwd_split_supported(s->K, s->V, bf16, true, v_tile);
  }
  return 0;
}

kda_status kda_chunk_fwd(const kda_shape *s, const void *q, const void *k,
                         const void *v, const float *g, const float *beta,
                         float scale, int chunk_size,
                         const float *initial_state,
                         const int32_t *segment_ids, void *o,
                         float *final_state, void *workspace,
                         size_t workspace_bytes, kda_stream_t stream) {
  return kda_chunk_fwd_ex(s, q, k, v, g, beta, scale, chunk_size,
                          initial_state, segment_ids, o, final_state,
                          workspace, workspace_bytes, KDA_IMPL_AUTO, 0, stream);
}

kda_status kda_short_conv_silu(const kda_shape *s, const void *x_q,
                               const void *x_k, const void *x_v,
                               const float *w, const int32_t *segment_ids,
                               int l2norm_qk, void *q, void *k, void *v,
                               kda_stream_t stream) {
  kda_status st = check_shape(s);
  if (st != KDA_OK) return st;
  if (!x_q || !x_k || !x_v || !w || !q || !k || !v) return KDA_ERR_INVALID_ARG;
  const void *ptrs[] = {x_q, x_k, x_v, w, q, k, v, segment_ids};
  for (const void *ptr : ptrs)
    if (ptr && !aligned(ptr, 16)) return KDA_ERR_ALIGNMENT;
  if (x_q == q || x_k == k || x_v == v) return KDA_ERR_INVALID_ARG;
  // grid.y = B x tiles of 24 tokens
  if ((long long)s->B * ((s->T + 23) / 24) > 65535) return KDA_ERR_UNSUPPORTED;
  ConvParams p;
  memset(&p, 0, sizeof(p));
  p.B = s->B; p.T = s->T; p.H = s->H; p.K = s->K; p.V = s->V;
  p.x[0] = x_q; p.x[1] = x_k; p.x[2] = x_v;
  p.y[0] = q; p.y[1] = k; p.y[2] = v;
  p.w = w;
  p.segment_ids = segment_ids;
  p.l2norm_qk = l2norm_qk != 0;
  return from_cuda(launch_short_conv(p, s->qkv_dtype == KDA_DTYPE_BF16,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

kda_status kda_read_device_status(const void *workspace, kda_stream_t stream,
                                  uint32_t *device_bits) {
  if (!workspace || !device_bits) return KDA_ERR_INVALID_ARG;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint32_t bits = 0;
  if (cudaStreamSynchronize(cs) != cudaSuccess) return KDA_ERR_CUDA;
  if (cudaMemcpy(&bits, workspace, sizeof(bits), cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return KDA_ERR_CUDA;
  *device_bits = bits;
  if (bits & KDA_DEVICE_TIMEOUT) return KDA_ERR_TIMEOUT;
  if (bits & KDA_DEVICE_WORKSPACE) return KDA_ERR_WORKSPACE;
  if (bits) return KDA_ERR_DEVICE;
  return KDA_OK;
}

kda_status kda_clear_device_status(void *workspace, kda_stream_t stream) {
  if (!workspace) return KDA_ERR_INVALID_ARG;
  return from_cuda(cudaMemsetAsync(workspace, 0, sizeof(uint32_t),
                                   reinterpret_cast<cudaStream_t>(stream)));
}

size_t kda_chunk_bwd_workspace_size_for(const kda_shape *s, int has_segment_ids,
                                        kda_impl impl) {
  if (check_shape(s) != KDA_OK || !bwd_supported(s->K, s->V)) return 0;
  const bool has_seg = has_segment_ids != 0;
  const bool tc_ok = bwd_tc_supported(s->K, s->V, s->qkv_dtype == KDA_DTYPE_BF16);
  const size_t simt = align_up(ws_bytes(s->B, s->T, has_seg), 256) +
                      bwd_scratch_bytes(s->B, s->T, s->H, s->K, s->V);
  // with segment ids: room for ceil(T/64) runs per row beyond the chunks of T
  const size_t tc = tc_ok ? bwd_tc_workspace_bytes(s->B, s->T, s->H, has_seg,
                                                   default_runs_bound(s->T))
                          : 0;
  switch (impl) {
    case KDA_IMPL_SIMT: return simt;
    case KDA_IMPL_TC:
    case KDA_IMPL_SPLIT: return tc;
    case KDA_IMPL_AUTO: return tc_ok ? tc : simt;
  }
  return 0;
}

size_t kda_chunk_bwd_workspace_size_packed(const kda_shape *s, int max_runs_per_row) {
  if (check_shape(s) != KDA_OK || max_runs_per_row < 1) return 0;
  if (!bwd_tc_supported(s->K, s->V, s->qkv_dtype == KDA_DTYPE_BF16)) return 0;
  return bwd_tc_workspace_bytes(s->B, s->T, s->H, true, max_runs_per_row);
}

size_t kda_chunk_bwd_workspace_size(const kda_shape *s, int has_segment_ids) {
  return kda_chunk_bwd_workspace_size_for(s, has_segment_ids, KDA_IMPL_AUTO);
}

kda_status kda_chunk_bwd(const kda_shape *s, const void *q, const void *k, const void *v,
                         const float *g, const float *beta, float scale, int chunk_size,
                         const float *initial_state, const int32_t *segment_ids,
                         const void *d_o, const float *d_final, float *dq, float *dk,
                         float *dv, float *dg, float *dbeta, float *d_initial,
                         void *workspace, size_t workspace_bytes, kda_stream_t stream) {
  return kda_chunk_bwd_ex(s, q, k, v, g, beta, scale, chunk_size, initial_state, segment_ids,
                          d_o, d_final, dq, dk, dv, dg, dbeta, d_initial, workspace,
                          workspace_bytes, KDA_IMPL_AUTO, stream);
}

}  // extern "C"

namespace {
// kda_chunk_bwd_ex and kda_chunk_bwd_from_saved (from_saved: the
// tensor-core path on the items and saves a kda_chunk_fwd_save left).
kda_status bwd_entry(const kda_shape *s, const void *q, const void *k, const void *v,
                     const float *g, const float *beta, float scale, int chunk_size,
                     const float *initial_state, const int32_t *segment_ids, const void *d_o,
                     const float *d_final, float *dq, float *dk, float *dv, float *dg,
                     float *dbeta, float *d_initial, void *workspace, size_t workspace_bytes,
                     kda_impl impl, bool from_saved, kda_stream_t stream) {
  kda_status st = check_shape(s);
  if (st != KDA_OK) return st;
  if (!bwd_supported(s->K, s->V)) return KDA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !g || !beta || !d_o || !dq || !dk || !dv || !dg || !dbeta)
    return KDA_ERR_INVALID_ARG;
  if (chunk_size != kChunk) return KDA_ERR_UNSUPPORTED;
  if (!(scale == scale)) return KDA_ERR_INVALID_ARG;
  if (impl != KDA_IMPL_AUTO && impl != KDA_IMPL_SIMT && impl != KDA_IMPL_TC &&
      impl != KDA_IMPL_SPLIT)
    return KDA_ERR_INVALID_ARG;
  const void *ptrs[] = {q, k, v, g, beta, d_o, initial_state, d_final, segment_ids,
                        dq, dk, dv, dg, dbeta, d_initial};
  for (const void *ptr : ptrs)
    if (ptr && !aligned(ptr, 16)) return KDA_ERR_ALIGNMENT;
  const bool has_seg = segment_ids != nullptr;
  const bool tc_ok = bwd_tc_supported(s->K, s->V, s->qkv_dtype == KDA_DTYPE_BF16);
  if ((impl == KDA_IMPL_TC || impl == KDA_IMPL_SPLIT) && !tc_ok) return KDA_ERR_UNSUPPORTED;
  const bool use_tc = impl == KDA_IMPL_TC || impl == KDA_IMPL_SPLIT ||
                      (impl == KDA_IMPL_AUTO && tc_ok);
  // the tensor-core path with segment ids takes any workspace that holds the
  // chunks of T per row (more runs than it has room for: KDA_DEVICE_WORKSPACE)
  const size_t need = use_tc ? bwd_tc_workspace_bytes(s->B, s->T, s->H, has_seg, 0)
                             : kda_chunk_bwd_workspace_size_for(s, has_seg ? 1 : 0,
                                                                KDA_IMPL_SIMT);
  if (!workspace || workspace_bytes < need) return KDA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return KDA_ERR_ALIGNMENT;

  const size_t nck = ((size_t)s->T + 7) / 8;
  const size_t n_vt = (size_t)s->V / 32;
  const size_t nK = (size_t)s->B * s->T * s->H * s->K;
  char *ws = static_cast<char *>(workspace);
  char *scratch = ws + align_up(ws_bytes(s->B, s->T, has_seg), 256);
  BwdParams p;
  memset(&p, 0, sizeof(p));
  p.B = s->B; p.T = s->T; p.H = s->H; p.K = s->K; p.V = s->V;
  p.n_vtiles = (int)n_vt;
  p.q = q; p.k = k; p.v = v; p.d_o = d_o;
  p.g = g; p.beta = beta; p.initial_state = initial_state; p.d_final = d_final;
  p.scale = scale;
  p.dv = dv; p.d_initial = d_initial;
  p.ckpt_cta_floats = nck * (size_t)s->K * 32;
  p.ckpt = reinterpret_cast<float *>(scratch);
  size_t off = align_up(sizeof(float) * kBwdMaxCtas * p.ckpt_cta_floats, 256);
  p.part_q = reinterpret_cast<float *>(scratch + off); off += align_up(sizeof(float) * n_vt * nK, 256);
  p.part_k = reinterpret_cast<float *>(scratch + off); off += align_up(sizeof(float) * n_vt * nK, 256);
  p.part_g = reinterpret_cast<float *>(scratch + off); off += align_up(sizeof(float) * n_vt * nK, 256);
  p.part_b = reinterpret_cast<float *>(scratch + off);
  const long long max_units =
      (long long)s->B * (has_seg ? s->T : 1) * s->H * (long long)n_vt;
  p.grid = (int)(max_units < kBwdMaxCtas ? max_units : kBwdMaxCtas);
  if (has_seg) {
    p.runs.row_offsets = reinterpret_cast<const int32_t *>(ws + sizeof(WsHeader));
    p.runs.runs = reinterpret_cast<const int2 *>(ws + sizeof(WsHeader) +
                                                 ws_row_offsets_bytes(s->B));
    p.runs.total_runs = &reinterpret_cast<WsHeader *>(ws)->total_runs;
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (use_tc) {
    if (has_seg) {
      // runs and chunk tables; dv = 0 on padding; d_initial = d_final (or 0)
      // for rows without a run
      cudaError_t e = launch_segment_runs(s->B, s->T, s->H, s->K, s->V, segment_ids, dv, 0,
                                          d_final, d_initial, workspace, cs, true);
      if (e != cudaSuccess) return from_cuda(e);
    }
    return from_cuda(launch_bwd_tc(p, segment_ids, workspace, workspace_bytes, dq, dk, dg,
                                   dbeta, &reinterpret_cast<WsHeader *>(ws)->status, cs,
                                   from_saved));
  }
  if (has_seg) {
    // Runs; dv = 0 on padding; d_initial = d_final (or 0) for rows without a run.
    cudaError_t e = launch_segment_runs(s->B, s->T, s->H, s->K, s->V, segment_ids, dv, 0,
                                        d_final, d_initial, workspace, cs, false);
    if (e != cudaSuccess) return from_cuda(e);
  }
  return from_cuda(launch_bwd(p, s->qkv_dtype == KDA_DTYPE_BF16, segment_ids, dq, dk, dg,
                              dbeta, cs));
}
}  // namespace

extern "C" {

kda_status kda_chunk_bwd_ex(const kda_shape *s, const void *q, const void *k, const void *v,
                            const float *g, const float *beta, float scale, int chunk_size,
                            const float *initial_state, const int32_t *segment_ids,
                            const void *d_o, const float *d_final, float *dq, float *dk,
                            float *dv, float *dg, float *dbeta, float *d_initial,
                            void *workspace, size_t workspace_bytes, kda_impl impl,
                            kda_stream_t stream) {
  return bwd_entry(s, q, k, v, g, beta, scale, chunk_size, initial_state, segment_ids, d_o,
                   d_final, dq, dk, dv, dg, dbeta, d_initial, workspace, workspace_bytes, impl,
                   false, stream);
}

size_t kda_chunk_fwd_save_workspace_size(const kda_shape *s, int has_segment_ids) {
  return kda_chunk_bwd_workspace_size_for(s, has_segment_ids, KDA_IMPL_TC);
}

kda_status kda_chunk_fwd_save(const kda_shape *s, const void *q, const void *k, const void *v,
                              const float *g, const float *beta, float scale, int chunk_size,
                              const float *initial_state, const int32_t *segment_ids, void *o,
                              float *final_state, void *workspace, size_t workspace_bytes,
                              kda_stream_t stream) {
  kda_status st = check_shape(s);
  if (st != KDA_OK) return st;
  if (!q || !k || !v || !g || !beta || !o) return KDA_ERR_INVALID_ARG;
  if (chunk_size != kChunk) return KDA_ERR_UNSUPPORTED;
  if (!(scale == scale)) return KDA_ERR_INVALID_ARG;
  if (!bwd_tc_supported(s->K, s->V, s->qkv_dtype == KDA_DTYPE_BF16)) return KDA_ERR_UNSUPPORTED;
  const void *ptrs[] = {q, k, v, g, beta, o, initial_state, final_state, segment_ids};
  for (const void *ptr : ptrs)
    if (ptr && !aligned(ptr, 16)) return KDA_ERR_ALIGNMENT;
  const bool has_seg = segment_ids != nullptr;
  if (!workspace || workspace_bytes < bwd_tc_workspace_bytes(s->B, s->T, s->H, has_seg, 0))
    return KDA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return KDA_ERR_ALIGNMENT;
  FwdParams p;
  memset(&p, 0, sizeof(p));
  p.B = s->B; p.T = s->T; p.H = s->H; p.K = s->K; p.V = s->V;
  p.q = q; p.k = k; p.v = v; p.g = g; p.beta = beta;
  p.scale = scale;
  p.initial_state = initial_state;
  p.o = o;
  p.final_state = final_state;
  char *ws = static_cast<char *>(workspace);
  p.status = &reinterpret_cast<WsHeader *>(ws)->status;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (has_seg) {
    p.runs.row_offsets = reinterpret_cast<const int32_t *>(ws + sizeof(WsHeader));
    p.runs.runs = reinterpret_cast<const int2 *>(ws + sizeof(WsHeader) +
                                                 ws_row_offsets_bytes(s->B));
    p.runs.total_runs = &reinterpret_cast<WsHeader *>(ws)->total_runs;
    cudaError_t e = launch_segment_runs(s->B, s->T, s->H, s->K, s->V, segment_ids, o, 1,
                                        initial_state, final_state, workspace, cs, true);
    if (e != cudaSuccess) return from_cuda(e);
  }
  return from_cuda(launch_fwd_save(p, workspace, workspace_bytes, cs));
}

kda_status kda_chunk_bwd_from_saved(const kda_shape *s, const void *q, const void *k,
                                    const void *v, const float *g, const float *beta,
                                    float scale, int chunk_size, const float *initial_state,
                                    const int32_t *segment_ids, const void *d_o,
                                    const float *d_final, float *dq, float *dk, float *dv,
                                    float *dg, float *dbeta, float *d_initial,
                                    void *workspace, size_t workspace_bytes,
                                    kda_stream_t stream) {
  return bwd_entry(s, q, k, v, g, beta, scale, chunk_size, initial_state, segment_ids, d_o,
                   d_final, dq, dk, dv, dg, dbeta, d_initial, workspace, workspace_bytes,
                   KDA_IMPL_TC, true, stream);
}

}  // extern "C"
