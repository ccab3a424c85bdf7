// kda_fwd_tc.cu -- tensor-core (tcgen05 / TMEM / TMA) chunked KDA forward.
// Placeholder until the kernel lands: reports "not supported" so the ABI
// falls back to the SIMT kernel under KDA_IMPL_AUTO.
#include "kda_internal.cuh"

namespace kda {

bool fwd_tc_supported(int, int, bool, int) { return false; }

cudaError_t launch_fwd_tc(const FwdParams &, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace kda
