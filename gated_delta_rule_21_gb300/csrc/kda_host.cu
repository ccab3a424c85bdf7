// kda_host.cu -- kda_chunk_fwd_host: the chunked forward on HOST buffers,
// pipelined by groups of heads.
//
// Heads are independent problems, so the forward of a group of heads needs
// only that group's slices of q, k, v, g, beta and the states.  The call
// splits the heads into groups; each group copies its slices in (2-D copies
// out of the [B, T, H, .] host layout into contiguous device buffers), runs
// the forward on them and copies its o and final state back, on a stream of
// its own.  The host-to-device copies are chained group after group, so the
// copy engine delivers group 0 first and the compute of group 0 overlaps the
// copies of groups 1, 2, ...; the copies back use the other direction of the
// link.  Every device buffer is carved from the caller's `device_buffer`.
// The library creates (once per device, for the process lifetime) the
// group streams and events it uses; it allocates no device memory.
#include <algorithm>
#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr int kMaxGroups = 2;
constexpr int kMaxDevices = 64;

struct GroupPlan {
  int groups = 1, hg = 1;  // number of head groups, heads per group
};

// Two groups when H is even.  More groups overlap more of the copies, but
// each group's recurrence is a full-length serial chain and the groups'
// kernels then contend for the SMs: on the B1 H32 T8192 shape 2 groups
// measured 2.23 ms end to end, 4 groups 2.37 ms, 8 groups 2.48 ms.
GroupPlan plan_groups(int H) {
  GroupPlan p;
  p.groups = H % 2 == 0 ? 2 : 1;
  p.hg = H / p.groups;
  return p;
}

size_t a256(size_t x) { return (x + 255) / 256 * 256; }

// Per-group device regions, in order: q, k, v, g, beta, S0, o, S_final,
// workspace; then the shared segment ids and the full beta.
struct Layout {
  size_t q, k, v, g, beta, s0, o, fs, ws, ws_bytes, group_bytes;
  size_t seg, beta_full, total;
};

Layout layout(const kda_shape &s, bool has_seg, const GroupPlan &gp) {
  Layout L;
  const size_t e = s.qkv_dtype == KDA_DTYPE_BF16 ? 2 : 4;
  const size_t bt = (size_t)s.B * s.T, hg = (size_t)gp.hg;
  kda_shape sg = s;
  sg.H = gp.hg;
  size_t off = 0;
  L.q = off;    off += a256(bt * hg * s.K * e);
  L.k = off;    off += a256(bt * hg * s.K * e);
  L.v = off;    off += a256(bt * hg * s.V * e);
  L.g = off;    off += a256(bt * hg * s.K * 4);
  L.beta = off; off += a256(bt * hg * 4);
  L.s0 = off;   off += a256((size_t)s.B * hg * s.K * s.V * 4);
  L.o = off;    off += a256(bt * hg * s.V * e);
  L.fs = off;   off += a256((size_t)s.B * hg * s.K * s.V * 4);
  L.ws = off;
  L.ws_bytes = kda_chunk_fwd_workspace_size_for(&sg, has_seg ? 1 : 0, KDA_IMPL_AUTO);
  off += a256(L.ws_bytes);
  L.group_bytes = off;
  L.seg = L.group_bytes * gp.groups;
  L.beta_full = L.seg + a256(has_seg ? bt * 4 : 0);
  L.total = L.beta_full + a256(bt * s.H * 4);
  return L;
}

// Streams and events of the pipeline, created once per device.
struct Pipeline {
  cudaStream_t streams[kMaxGroups] = {};
  cudaEvent_t start = nullptr, copied[kMaxGroups] = {}, done[kMaxGroups] = {};
  bool ready = false;
};
std::mutex g_mutex;
Pipeline g_pipes[kMaxDevices];

kda_status pipeline_for_current_device(Pipeline **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  Pipeline &p = g_pipes[dev];
  if (!p.ready) {
    const unsigned ef = cudaEventDisableTiming;
    if (cudaEventCreateWithFlags(&p.start, ef) != cudaSuccess) return KDA_ERR_CUDA;
    for (int i = 0; i < kMaxGroups; ++i) {
      if (cudaStreamCreateWithFlags(&p.streams[i], cudaStreamNonBlocking) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.copied[i], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.done[i], ef) != cudaSuccess)
        return KDA_ERR_CUDA;
    }
    p.ready = true;
  }
  *out = &p;
  return KDA_OK;
}

}  // namespace

extern "C" size_t kda_chunk_fwd_host_buffer_size(const kda_shape *s, int has_segment_ids) {
  if (!s || kda_chunk_fwd_workspace_size(s, has_segment_ids) == 0) return 0;
  return layout(*s, has_segment_ids != 0, plan_groups(s->H)).total;
}

extern "C" kda_status kda_chunk_fwd_host(const kda_shape *s, const void *q, const void *k,
                                         const void *v, const float *g, const float *beta,
                                         float scale, int chunk_size,
                                         const float *initial_state,
                                         const int32_t *segment_ids, void *o,
                                         float *final_state, void *device_buffer,
                                         size_t device_buffer_bytes, kda_stream_t stream) {
  // Argument checks first, so that nothing is enqueued on error.
  const bool has_seg = segment_ids != nullptr;
  const size_t need = kda_chunk_fwd_host_buffer_size(s, has_seg ? 1 : 0);
  if (need == 0) return s ? KDA_ERR_UNSUPPORTED : KDA_ERR_INVALID_ARG;
  if (!q || !k || !v || !g || !beta || !o || !device_buffer) return KDA_ERR_INVALID_ARG;
  if (chunk_size != kda::kChunk) return KDA_ERR_UNSUPPORTED;
  if (!(scale == scale)) return KDA_ERR_INVALID_ARG;
  if (device_buffer_bytes < need) return KDA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(device_buffer) & 255u) != 0) return KDA_ERR_ALIGNMENT;
  if (!kda_impl_available(KDA_IMPL_AUTO, s, 0)) return KDA_ERR_UNSUPPORTED;

  Pipeline *pl = nullptr;
  kda_status st = pipeline_for_current_device(&pl);
  if (st != KDA_OK) return st;
  // One enqueue at a time: the group streams and events are shared by the
  // calls on this device (the work itself runs asynchronously).
  std::lock_guard<std::mutex> lock(g_mutex);
  const GroupPlan gp = plan_groups(s->H);
  const Layout L = layout(*s, has_seg, gp);
  const size_t e = s->qkv_dtype == KDA_DTYPE_BF16 ? 2 : 4;
  const size_t bt = (size_t)s->B * s->T, hg = (size_t)gp.hg, H = (size_t)s->H;
  const size_t K = (size_t)s->K, V = (size_t)s->V;
  unsigned char *dev = static_cast<unsigned char *>(device_buffer);
  cudaStream_t user = reinterpret_cast<cudaStream_t>(stream);
  auto ok = [](cudaError_t err) { return err == cudaSuccess; };

  // Shared inputs on the caller's stream: segment ids and the whole beta
  // (its per-group slices are gathered on the device: 4-byte host rows
  // would make a slow 2-D copy).
  if (has_seg && !ok(cudaMemcpyAsync(dev + L.seg, segment_ids, bt * 4,
                                     cudaMemcpyHostToDevice, user)))
    return KDA_ERR_CUDA;
  if (!ok(cudaMemcpyAsync(dev + L.beta_full, beta, bt * H * 4, cudaMemcpyHostToDevice, user)))
    return KDA_ERR_CUDA;
  if (!ok(cudaEventRecord(pl->start, user))) return KDA_ERR_CUDA;

  kda_shape sg = *s;
  sg.H = gp.hg;
  for (int gi = 0; gi < gp.groups; ++gi) {
    cudaStream_t cs = pl->streams[gi];
    unsigned char *base = dev + (size_t)gi * L.group_bytes;
    const size_t h0 = (size_t)gi * hg;
    if (!ok(cudaStreamWaitEvent(cs, pl->start, 0))) return KDA_ERR_CUDA;
    // host -> device, after the previous group's copies (in group order)
    if (gi > 0 && !ok(cudaStreamWaitEvent(cs, pl->copied[gi - 1], 0))) return KDA_ERR_CUDA;
    auto in2d = [&](size_t dst, const void *src, size_t row_elems, size_t esz) {
      return ok(cudaMemcpy2DAsync(base + dst, hg * row_elems * esz,
                                  static_cast<const unsigned char *>(src) + h0 * row_elems * esz,
                                  H * row_elems * esz, hg * row_elems * esz, bt,
                                  cudaMemcpyHostToDevice, cs));
    };
    if (!in2d(L.q, q, K, e) || !in2d(L.k, k, K, e) || !in2d(L.v, v, V, e) ||
        !in2d(L.g, g, K, 4))
      return KDA_ERR_CUDA;
    if (!ok(cudaMemcpy2DAsync(base + L.beta, hg * 4, dev + L.beta_full + h0 * 4, H * 4, hg * 4,
                              bt, cudaMemcpyDeviceToDevice, cs)))
      return KDA_ERR_CUDA;
    const size_t state_row = hg * K * V * 4;  // one b's heads of this group
    if (initial_state &&
        !ok(cudaMemcpy2DAsync(base + L.s0, state_row,
                              reinterpret_cast<const unsigned char *>(initial_state) +
                                  h0 * K * V * 4,
                              H * K * V * 4, state_row, (size_t)s->B,
                              cudaMemcpyHostToDevice, cs)))
      return KDA_ERR_CUDA;
    if (!ok(cudaEventRecord(pl->copied[gi], cs))) return KDA_ERR_CUDA;
    // the forward of this group
    st = kda_chunk_fwd(&sg, base + L.q, base + L.k, base + L.v,
                       reinterpret_cast<const float *>(base + L.g),
                       reinterpret_cast<const float *>(base + L.beta), scale, chunk_size,
                       initial_state ? reinterpret_cast<const float *>(base + L.s0) : nullptr,
                       has_seg ? reinterpret_cast<const int32_t *>(dev + L.seg) : nullptr,
                       base + L.o, final_state ? reinterpret_cast<float *>(base + L.fs) : nullptr,
                       base + L.ws, L.ws_bytes, reinterpret_cast<kda_stream_t>(cs));
    if (st != KDA_OK) return st;
    // device -> host
    if (!ok(cudaMemcpy2DAsync(static_cast<unsigned char *>(o) + h0 * V * e, H * V * e,
                              base + L.o, hg * V * e, hg * V * e, bt, cudaMemcpyDeviceToHost,
                              cs)))
      return KDA_ERR_CUDA;
    if (final_state &&
        !ok(cudaMemcpy2DAsync(reinterpret_cast<unsigned char *>(final_state) + h0 * K * V * 4,
                              H * K * V * 4, base + L.fs, state_row, state_row, (size_t)s->B,
                              cudaMemcpyDeviceToHost, cs)))
      return KDA_ERR_CUDA;
    if (!ok(cudaEventRecord(pl->done[gi], cs))) return KDA_ERR_CUDA;
  }
  for (int gi = 0; gi < gp.groups; ++gi)
    if (!ok(cudaStreamWaitEvent(user, pl->done[gi], 0))) return KDA_ERR_CUDA;
  return KDA_OK;
}
