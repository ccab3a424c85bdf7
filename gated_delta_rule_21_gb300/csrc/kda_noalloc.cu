// kda_noalloc.cu -- kda_chunk_fwd_noalloc: the chunked forward for callers
// that cannot allocate device memory, and kda_chunk_fwd_noalloc_status, its
// device status query.
//
// Some callers cannot call cudaMalloc or hand libkda a workspace: a plugin
// inside a host application that passes it only the tensors it owns, code
// running under a fixed memory budget held by another allocator, or a hot
// path where allocating is not allowed because of its latency and the
// fragmentation it causes.  For them this entry point keeps its scratch (the
// status word, the per-row run counts and the run list built from segment
// ids, and the split path's per-chunk operands when they fit) in a fixed
// array in device memory that the library itself defines.  The caller still
// passes every input and output.
//
// Limits and rules of use:
//   * The array holds KDA_NOALLOC_SCRATCH_BYTES (1 MiB).  Every GPU that
//     loads libkda keeps that much device memory until the process exits.
//     Shapes whose smallest workspace (kda_chunk_fwd_workspace_size_for(s,
//     has_segment_ids, KDA_IMPL_SIMT)) is larger are rejected with
//     KDA_ERR_WORKSPACE; with segment ids that is about B*T > 130000 tokens,
//     without them any shape fits.
//   * All calls share the one array.  Calls whose work overlaps on the GPU
//     (on different streams, or from different host threads without
//     ordering) race on it and give wrong results; order them on one stream.
//   * The array's device address is looked up (cudaGetSymbolAddress, with
//     the device current) on the first call in each CUDA context of a device
//     and kept for that context.  A device reset destroys the context; the
//     next call sees a new context and looks the address up again.  Make the
//     first call on a device before any stream capture begins.
//   * The scratch header is cleared on the caller's stream at the start of
//     each call, so a call never sees the previous call's counters; its
//     status word then holds the bits of the last call until the next one.
#include <cudaTypedefs.h>

#include <mutex>

#include "kda_internal.cuh"

namespace {

// The scratch array.  In host code this name is only a host-side handle:
// its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char
    g_kda_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
struct Entry {
  void *addr;
  unsigned long long ctx_id;  // the context the address belongs to
};
std::mutex g_mutex;
Entry g_scratch[kMaxDevices] = {};

// Unique id of the calling thread's current CUDA context (driver entry
// points reached through the runtime, so the library needs no -lcuda).
// False when no context is current or the driver lacks the query.
bool current_context_id(unsigned long long *id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault,
                                         &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the array in the current device's current context,
// looked up once per context (every call when the context cannot be
// identified).
kda_status scratch_for_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
  unsigned long long id = 0;
  bool have_id = current_context_id(&id);
  std::lock_guard<std::mutex> lock(g_mutex);
  Entry &e = g_scratch[dev];
  if (!have_id || !e.addr || e.ctx_id != id) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kda_noalloc_scratch) != cudaSuccess || !p)
      return KDA_ERR_CUDA;
    // The lookup made the device's primary context current if none was.
    have_id = current_context_id(&id);
    e.addr = have_id ? p : nullptr;  // keep it only when its context is known
    e.ctx_id = id;
    *out = p;
    return KDA_OK;
  }
  *out = e.addr;
  return KDA_OK;
}

bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace

extern "C" kda_status kda_chunk_fwd_noalloc(
    const kda_shape *s, const void *q, const void *k, const void *v,
    const float *g, const float *beta, float scale, int chunk_size,
    const float *initial_state, const int32_t *segment_ids, void *o,
    float *final_state, kda_stream_t stream) {
  // The same checks, in the same order, as kda_chunk_fwd, so that both
  // return the same code for the same bad input; nothing is enqueued on
  // error.
  kda_status st = kda::check_shape(s);
  if (st != KDA_OK) return st;
  if (!q || !k || !v || !g || !beta || !o) return KDA_ERR_INVALID_ARG;
  if (chunk_size != kda::kChunk) return KDA_ERR_UNSUPPORTED;
  if (!(scale == scale)) return KDA_ERR_INVALID_ARG;
  const void *ptrs[] = {q, k, v, g, beta, o, initial_state, final_state,
                        segment_ids};
  for (const void *ptr : ptrs)
    if (ptr && !aligned16(ptr)) return KDA_ERR_ALIGNMENT;
  const size_t need = kda::ws_bytes(s->B, s->T, segment_ids != nullptr);
  if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;

  void *scratch = nullptr;
  st = scratch_for_current_device(&scratch);
  if (st != KDA_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, sizeof(kda::WsHeader), cs) != cudaSuccess)
    return KDA_ERR_CUDA;
  return kda_chunk_fwd(s, q, k, v, g, beta, scale, chunk_size, initial_state,
                       segment_ids, o, final_state, scratch,
                       (size_t)KDA_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" kda_status kda_chunk_fwd_noalloc_status(kda_stream_t stream,
                                                   uint32_t *device_bits) {
  if (!device_bits) return KDA_ERR_INVALID_ARG;
  void *scratch = nullptr;
  const kda_status st = scratch_for_current_device(&scratch);
  if (st != KDA_OK) return st;
  return kda_read_device_status(scratch, stream, device_bits);
}
