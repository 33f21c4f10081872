// attn_diag.cu -- diagnostics that sit beside the attention kernels (declared
// in include/attn_diag.h, apart from the attention ABI of attn.h).
//
// 1. A self-test of the device-side failure path.  Every pipeline wait in the
//    attention kernels is bounded; when one runs out the kernel records
//    ATTN_ERR_TIMEOUT in the sticky status word, stops its roles and returns
//    instead of hanging.  attn_debug_wait_timeout runs that same bounded wait
//    on an mbarrier that nothing will ever arrive on, so a test can check that
//    the wait gives up, the status is reported and cleared by
//    attn_sync_status, and the CUDA context stays usable afterwards.
// 2. A throughput probe of the exponential unit (attn_probe_ex2): the
//    softmax step needs one exp2 per score, so the unit's measured rate is a
//    second bound on the forward and backward next to the tensor cores.
#include <cstdint>

#include "attn.h"
#include "attn_diag.h"
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

// Each thread keeps kChains independent recurrences x <- 2^x - 1.5 (x stays in
// (-1.25, -1]), so per thread kChains ex2.approx are in flight each round and,
// with several blocks per SM, the exponential unit rather than its latency
// sets the pace.  The sum is stored so that nothing is optimised away.
constexpr int kEx2Chains = 8;
constexpr int kEx2Threads = 256;

__global__ void __launch_bounds__(kEx2Threads) ex2_rate_kernel(float* __restrict__ sink, int iters) {
  float x[kEx2Chains];
#pragma unroll
  for (int i = 0; i < kEx2Chains; ++i) x[i] = -1.0f - 0.01f * static_cast<float>(threadIdx.x & 7) - 0.001f * i;
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < kEx2Chains; ++i) x[i] = ex2_approx(x[i]) - 1.5f;
  }
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kEx2Chains; ++i) acc += x[i];
  sink[static_cast<size_t>(blockIdx.x) * kEx2Threads + threadIdx.x] = acc;
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

extern "C" int attn_probe_ex2(float* sink, int blocks, int iters, void* stream) {
  using namespace attn;
  if (!sink || (reinterpret_cast<uintptr_t>(sink) & 3u) || blocks < 1 || blocks > 65535 || iters < 1 ||
      iters > (1 << 20))
    return kStatusInvalid;
  ex2_rate_kernel<<<blocks, kEx2Threads, 0, static_cast<cudaStream_t>(stream)>>>(sink, iters);
  return cudaGetLastError() == cudaSuccess ? kStatusOk : kStatusCuda;
}
