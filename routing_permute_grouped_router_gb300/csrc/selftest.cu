// Self-test of the bounded pipeline waits.  Every mbarrier wait in the
// tensor-core kernels gives up after a time limit, records DEV_TIMEOUT in the
// device error word and lets the kernel drain and exit, so a stalled pipeline
// is reported instead of hanging the GPU.  This entry point exercises that
// same wait helper on a barrier nothing arrives at (or, as a control, one that
// a second warp arrives at) with a short limit.
#include "../../include/moe.h"
#include "common.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

__global__ void bounded_wait_kernel(uint32_t* err, uint64_t limit_ns, int arrive) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 32 && arrive) mbar_arrive(smem_addr(&bar));
  if (threadIdx.x == 0) mbar_wait(smem_addr(&bar), 0, &abort_flag, err, 700, limit_ns);
  __syncthreads();
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_selftest_bounded_wait(int64_t limit_ns, int arrive, moe_stream_t stream) {
  using namespace moe;
  if (limit_ns < 1000000 || limit_ns > 2000000000 || (arrive != 0 && arrive != 1)) return MOE_ERR_INVALID_ARG;
  uint32_t* err = nullptr;
  const moe_status st = static_cast<moe_status>(current_error_word(&err));
  if (st != MOE_OK) return st;
  LaunchScope ls(KK_SELFTEST, stream);
  bounded_wait_kernel<<<1, 64, 0, stream>>>(err, (uint64_t)limit_ns, arrive);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
