// kda_host.cu -- kda_chunk_fwd_host: the chunked forward on HOST buffers,
// with the copies overlapped with the compute.
//
// Without segment ids the call pipelines over TIME.  The tokens are split
// into ranges of a multiple of 64 tokens; the state leaving one range (the
// forward's final state, exact fp32) enters the next as its initial state,
// and chunk boundaries stay where they are, so the result is bitwise that of
// one forward over all tokens.  Each range's inputs are contiguous in the
// [B, T, H, .] host layout (one run of bytes per row b), so the copies are
// large and run at the host link's full rate: the host-to-device copies of
// all ranges queue back to back on one stream, the forward of range r runs
// on a second stream as soon as its inputs are in, and its o goes back on a
// third (the other direction of the link).  Only the last range's compute
// and copy back are not hidden behind the copies in.
//
// With segment ids (a range boundary may fall inside a run or at its start,
// and rows may end in padding) the call pipelines over HEADS instead: heads
// are independent problems, so each group of heads copies its slices in
// (2-D copies out of the [B, T, H, .] layout), runs the forward on them and
// copies its o and final state back, on a stream of its own; the copies in
// are chained group after group.
//
// Every device buffer is carved from the caller's `device_buffer`.  The
// library creates (once per device, for the process lifetime) the streams
// and events it uses; it allocates no device memory.
#include <algorithm>
#include <mutex>

#include "kda_internal.cuh"

namespace {

constexpr int kMaxGroups = 2;
constexpr int kUniformRanges = 8;
constexpr int kMaxRanges = kUniformRanges + 1;   // the last one may be split in two
constexpr int kTailTokens = 256;
constexpr int kMaxDevices = 64;
static_assert(kMaxGroups <= kMaxRanges, "the head groups use the range events");

// Time ranges: at least 512 tokens each and at most kMaxRanges of them; a
// multiple of 64 tokens, the last one possibly shorter.  Each range's
// forward is well shorter than its copies in (about 50 us of compute
// against 200 us of copies per 1024 tokens of the B1 H32 K=V=128 bf16
// shape), so the compute keeps up.  Smaller ranges shorten the unhidden
// tail (the last range's compute and copy back) but add copies, each with
// a fixed cost of about 2 us: on that shape 4, 8, 16 and 32 ranges measured
// 1.97, 1.95, 2.02 and 2.15 ms end to end.  The last range, whose compute
// and copy back are the unhidden tail, is split off into its own last
// kTailTokens or so tokens (on a chunk boundary) when it is long enough.
struct RangePlan {
  int ranges = 1, R = 1;          // number of ranges, longest range
  int start[kMaxRanges + 1] = {};  // range r is tokens [start[r], start[r + 1])
};
RangePlan plan_ranges(int T) {
  RangePlan rp;
  const int per = ((T + kUniformRanges - 1) / kUniformRanges + kda::kChunk - 1) /
                  kda::kChunk * kda::kChunk;
  rp.R = std::max(512, per);
  rp.ranges = (T + rp.R - 1) / rp.R;
  for (int r = 0; r < rp.ranges; ++r) rp.start[r] = r * rp.R;
  rp.start[rp.ranges] = T;
  // the split point stays on a 64-token chunk boundary of the whole sequence
  const int split = (T - kTailTokens) / kda::kChunk * kda::kChunk;
  if (split - rp.start[rp.ranges - 1] >= kTailTokens) {
    rp.start[rp.ranges + 1] = T;
    rp.start[rp.ranges] = split;
    ++rp.ranges;
  }
  return rp;
}

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

// Time-pipeline device regions: q, k, v, g, beta, o for all tokens in range
// order (range r of [B, T_r, H, .] at the offset of its first token), the
// whole beta as copied in (one small copy instead of one per range), the
// initial state, two state buffers the ranges alternate between, and the
// workspace of one range.
struct TimeLayout {
  size_t q, k, v, g, beta, beta_full, o, s0, st[2], ws, ws_bytes, total;
};

TimeLayout time_layout(const kda_shape &s, const RangePlan &rp) {
  TimeLayout L;
  const size_t e = s.qkv_dtype == KDA_DTYPE_BF16 ? 2 : 4;
  const size_t bth = (size_t)s.B * s.T * s.H, state = (size_t)s.B * s.H * s.K * s.V * 4;
  kda_shape sr = s;
  sr.T = std::min(rp.R, s.T);
  size_t off = 0;
  L.q = off;    off += a256(bth * s.K * e);
  L.k = off;    off += a256(bth * s.K * e);
  L.v = off;    off += a256(bth * s.V * e);
  L.g = off;    off += a256(bth * s.K * 4);
  L.beta = off; off += a256(bth * 4);
  L.beta_full = off; off += a256(bth * 4);
  L.o = off;    off += a256(bth * s.V * e);
  L.s0 = off;   off += a256(state);
  L.st[0] = off; off += a256(state);
  L.st[1] = off; off += a256(state);
  L.ws = off;
  L.ws_bytes = kda_chunk_fwd_workspace_size_for(&sr, 0, KDA_IMPL_AUTO);
  off += a256(L.ws_bytes);
  L.total = off;
  return L;
}

// Streams and events of the pipelines, created once per device.
struct Pipeline {
  cudaStream_t streams[3] = {};
  cudaEvent_t start = nullptr, end = nullptr, ev_a[kMaxRanges] = {}, ev_b[kMaxRanges] = {};
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
    if (cudaEventCreateWithFlags(&p.start, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.end, ef) != cudaSuccess)
      return KDA_ERR_CUDA;
    for (int i = 0; i < 3; ++i)
      if (cudaStreamCreateWithFlags(&p.streams[i], cudaStreamNonBlocking) != cudaSuccess)
        return KDA_ERR_CUDA;
    for (int i = 0; i < kMaxRanges; ++i)
      if (cudaEventCreateWithFlags(&p.ev_a[i], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.ev_b[i], ef) != cudaSuccess)
        return KDA_ERR_CUDA;
    p.ready = true;
  }
  *out = &p;
  return KDA_OK;
}

// The time pipeline (no segment ids).  Arguments are checked by the caller.
kda_status enqueue_time_pipeline(const kda_shape *s, const void *q, const void *k,
                                 const void *v, const float *g, const float *beta, float scale,
                                 int chunk_size, const float *initial_state, void *o,
                                 float *final_state, unsigned char *dev, Pipeline *pl,
                                 cudaStream_t user) {
  const RangePlan rp = plan_ranges(s->T);
  const TimeLayout L = time_layout(*s, rp);
  const size_t e = s->qkv_dtype == KDA_DTYPE_BF16 ? 2 : 4;
  const size_t B = (size_t)s->B, T = (size_t)s->T, H = (size_t)s->H;
  const size_t K = (size_t)s->K, V = (size_t)s->V, state = B * H * K * V * 4;
  cudaStream_t cin = pl->streams[0], cfw = pl->streams[1], cout = pl->streams[2];
  auto ok = [](cudaError_t err) { return err == cudaSuccess; };
  if (!ok(cudaEventRecord(pl->start, user))) return KDA_ERR_CUDA;
  for (cudaStream_t cs : {cin, cfw, cout})
    if (!ok(cudaStreamWaitEvent(cs, pl->start, 0))) return KDA_ERR_CUDA;
  if (initial_state &&
      !ok(cudaMemcpyAsync(dev + L.s0, initial_state, state, cudaMemcpyHostToDevice, cin)))
    return KDA_ERR_CUDA;
  if (!ok(cudaMemcpyAsync(dev + L.beta_full, beta, B * T * H * 4, cudaMemcpyHostToDevice, cin)))
    return KDA_ERR_CUDA;
  for (int r = 0; r < rp.ranges; ++r) {
    const size_t t0 = (size_t)rp.start[r], tr = (size_t)(rp.start[r + 1] - rp.start[r]);
    // device copy of range r: [B, tr, H, d] at the offset of its first token
    auto at = [&](size_t region, size_t d, size_t esz) {
      return dev + region + B * t0 * H * d * esz;
    };
    // host rows b, tokens [t0, t0 + tr) of [B, T, H, d]: one run of bytes each
    auto in = [&](size_t region, const void *src, size_t d, size_t esz) {
      const size_t row = tr * H * d * esz;
      return ok(cudaMemcpy2DAsync(at(region, d, esz), row,
                                  static_cast<const unsigned char *>(src) + t0 * H * d * esz,
                                  T * H * d * esz, row, B, cudaMemcpyHostToDevice, cin));
    };
    if (!in(L.q, q, K, e) || !in(L.k, k, K, e) || !in(L.v, v, V, e) || !in(L.g, g, K, 4))
      return KDA_ERR_CUDA;
    if (!ok(cudaEventRecord(pl->ev_a[r], cin))) return KDA_ERR_CUDA;
    // the forward of this range, entering with the state the previous one left
    if (!ok(cudaStreamWaitEvent(cfw, pl->ev_a[r], 0))) return KDA_ERR_CUDA;
    // beta of the range: the rows of the whole copy (contiguous when B = 1)
    const unsigned char *beta_r = dev + L.beta_full + t0 * H * 4;
    if (B > 1) {
      if (!ok(cudaMemcpy2DAsync(at(L.beta, 1, 4), tr * H * 4, beta_r, T * H * 4, tr * H * 4, B,
                                cudaMemcpyDeviceToDevice, cfw)))
        return KDA_ERR_CUDA;
      beta_r = at(L.beta, 1, 4);
    }
    kda_shape sr = *s;
    sr.T = (int)tr;
    const float *s_in =
        r == 0 ? (initial_state ? reinterpret_cast<const float *>(dev + L.s0) : nullptr)
               : reinterpret_cast<const float *>(dev + L.st[(r - 1) & 1]);
    const kda_status st = kda_chunk_fwd(
        &sr, at(L.q, K, e), at(L.k, K, e), at(L.v, V, e),
        reinterpret_cast<const float *>(at(L.g, K, 4)),
        reinterpret_cast<const float *>(beta_r), scale, chunk_size, s_in, nullptr,
        at(L.o, V, e), reinterpret_cast<float *>(dev + L.st[r & 1]), dev + L.ws, L.ws_bytes,
        reinterpret_cast<kda_stream_t>(cfw));
    if (st != KDA_OK) return st;
    if (!ok(cudaEventRecord(pl->ev_b[r], cfw))) return KDA_ERR_CUDA;
    // o of this range back into the host rows
    if (!ok(cudaStreamWaitEvent(cout, pl->ev_b[r], 0))) return KDA_ERR_CUDA;
    const size_t orow = tr * H * V * e;
    if (!ok(cudaMemcpy2DAsync(static_cast<unsigned char *>(o) + t0 * H * V * e, T * H * V * e,
                              at(L.o, V, e), orow, orow, B, cudaMemcpyDeviceToHost, cout)))
      return KDA_ERR_CUDA;
  }
  if (final_state &&
      !ok(cudaMemcpyAsync(final_state, dev + L.st[(rp.ranges - 1) & 1], state,
                          cudaMemcpyDeviceToHost, cout)))
    return KDA_ERR_CUDA;
  if (!ok(cudaEventRecord(pl->end, cout)) || !ok(cudaStreamWaitEvent(user, pl->end, 0)))
    return KDA_ERR_CUDA;
  return KDA_OK;
}

}  // namespace

extern "C" size_t kda_chunk_fwd_host_buffer_size(const kda_shape *s, int has_segment_ids) {
  if (!s || kda_chunk_fwd_workspace_size(s, has_segment_ids) == 0) return 0;
  if (has_segment_ids == 0) return time_layout(*s, plan_ranges(s->T)).total;
  return layout(*s, true, plan_groups(s->H)).total;
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
  // One enqueue at a time: the streams and events are shared by the calls on
  // this device (the work itself runs asynchronously).
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!has_seg)
    return enqueue_time_pipeline(s, q, k, v, g, beta, scale, chunk_size, initial_state, o,
                                 final_state, static_cast<unsigned char *>(device_buffer), pl,
                                 reinterpret_cast<cudaStream_t>(stream));
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
    if (gi > 0 && !ok(cudaStreamWaitEvent(cs, pl->ev_a[gi - 1], 0))) return KDA_ERR_CUDA;
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
    if (!ok(cudaEventRecord(pl->ev_a[gi], cs))) return KDA_ERR_CUDA;
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
    if (!ok(cudaEventRecord(pl->ev_b[gi], cs))) return KDA_ERR_CUDA;
  }
  for (int gi = 0; gi < gp.groups; ++gi)
    if (!ok(cudaStreamWaitEvent(user, pl->ev_b[gi], 0))) return KDA_ERR_CUDA;
  return KDA_OK;
}
