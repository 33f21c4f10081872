// attn_diag.cu -- a self-test of the device-side failure path.
//
// Every pipeline wait in the attention kernels is bounded; when one runs out
// the kernel records ATTN_ERR_TIMEOUT in the sticky status word, stops its
// roles and returns instead of hanging.  attn_debug_wait_timeout runs that
// same bounded wait on an mbarrier that nothing will ever arrive on, so a
// test can check that the wait gives up, the status is reported and cleared
// by attn_sync_status, and the CUDA context stays usable afterwards.
#include <cstdint>

#include "attn.h"
#include "attn_internal.h"
#include "tc_sm103.cuh"

namespace attn {
namespace {

__global__ void __launch_bounds__(32, 1) wait_never_arrives_kernel(uint64_t limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);  // expects one arrival that never comes
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait_limit(smem_addr(&bar), 0, &abort_flag, status, limit_ns);
  __syncwarp();
}

}  // namespace
}  // namespace attn

extern "C" int attn_debug_wait_timeout(int limit_us, void* stream) {
  using namespace attn;
  if (limit_us < 1 || limit_us > 2000000) return kStatusInvalid;
  int* st = status_word_current_device();
  if (!st) return kStatusCuda;
  wait_never_arrives_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint64_t>(limit_us) * 1000ull, st);
  return cudaGetLastError() == cudaSuccess ? kStatusOk : kStatusCuda;
}
