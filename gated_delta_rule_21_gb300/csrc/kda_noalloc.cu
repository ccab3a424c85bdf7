// kda_noalloc.cu -- kda_chunk_fwd_noalloc: the chunked forward for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand libkda a workspace: a plugin
// inside a host application that passes it only the tensors it owns, code
// running under a fixed memory budget held by another allocator, or a hot
// path where allocating is not allowed because of its latency and the
// fragmentation it causes.  For them this entry point keeps its scratch (the
// status word, the per-row run counts and the run list built from segment
// ids) in a fixed array in device memory that the library itself defines.
// The caller still passes every input and output.
//
// Limits and rules of use:
//   * The array holds KDA_NOALLOC_SCRATCH_BYTES (1 MiB).  Every GPU that
//     loads libkda keeps that much device memory until the process exits.
//     Shapes whose scratch need (kda_chunk_fwd_workspace_size) is larger are
//     rejected with KDA_ERR_WORKSPACE; with segment ids that is about
//     B*T > 130000 tokens, without them any shape fits.
//   * All calls share the one array.  Calls whose work overlaps on the GPU
//     (on different streams, or from different host threads without
//     ordering) race on it and give wrong results; order them on one stream.
//   * The first call on each device looks up the array's device address
//     (cudaGetSymbolAddress, with that device current) and caches it; make
//     that first call before any stream capture begins.
//   * The scratch header is cleared on the caller's stream at the start of
//     each call, so a call never sees the previous call's counters.
#include <mutex>

#include "kda_internal.cuh"

namespace {

// The scratch array.  In host code this name is only a host-side handle:
// its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char
    g_kda_noalloc_scratch[KDA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once.
kda_status scratch_for_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kda_noalloc_scratch) != cudaSuccess || !p)
      return KDA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
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
  // Argument checks first, so that nothing is enqueued on error.
  const size_t need = kda_chunk_fwd_workspace_size(s, segment_ids != nullptr);
  if (need == 0) return s ? KDA_ERR_UNSUPPORTED : KDA_ERR_INVALID_ARG;
  if (need > (size_t)KDA_NOALLOC_SCRATCH_BYTES) return KDA_ERR_WORKSPACE;
  if (!q || !k || !v || !g || !beta || !o) return KDA_ERR_INVALID_ARG;
  if (chunk_size != kda::kChunk) return KDA_ERR_UNSUPPORTED;
  if (!(scale == scale)) return KDA_ERR_INVALID_ARG;
  const void *ptrs[] = {q, k, v, g, beta, o, initial_state, final_state,
                        segment_ids};
  for (const void *ptr : ptrs)
    if (ptr && !aligned16(ptr)) return KDA_ERR_ALIGNMENT;
  if (!kda_impl_available(KDA_IMPL_AUTO, s, 0)) return KDA_ERR_UNSUPPORTED;

  void *scratch = nullptr;
  kda_status st = scratch_for_current_device(&scratch);
  if (st != KDA_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, sizeof(kda::WsHeader), cs) != cudaSuccess)
    return KDA_ERR_CUDA;
  return kda_chunk_fwd(s, q, k, v, g, beta, scale, chunk_size, initial_state,
                       segment_ids, o, final_state, scratch,
                       (size_t)KDA_NOALLOC_SCRATCH_BYTES, stream);
}
