// kda_selftest.cu -- exercises the bounded-wait failure path of the
// tensor-core kernels without a fault: one thread waits on an mbarrier that
// nothing ever arrives at, with a short limit, and reports the timeout in
// the workspace status word exactly as the forward kernels do.
#include "kda_internal.cuh"
#include "kda_tc_common.cuh"

namespace kda {
namespace {

__global__ void wait_timeout_kernel(uint32_t *status, long long limit) {
  __shared__ __align__(8) unsigned long long bar;
  const uint32_t b = tc::smem_u32(&bar);
  tc::mbar_init(b, 1);  // count 1, and no thread arrives
  tc::fence_mbar_init();
  if (!tc::mbar_wait(b, 0u, limit)) set_status(status, KDA_DEVICE_TIMEOUT);
}

}  // namespace
}  // namespace kda

extern "C" KDA_API kda_status kda_selftest_wait_timeout(void *workspace, long long limit_cycles,
                                                        kda_stream_t stream) {
  if (!workspace || limit_cycles < 1 || limit_cycles > kda::tc::kWaitLimit)
    return KDA_ERR_INVALID_ARG;
  uint32_t *status = &reinterpret_cast<kda::WsHeader *>(workspace)->status;
  kda::wait_timeout_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status,
                                                                               limit_cycles);
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
