// attn_noalloc.cu -- a backward entry point that allocates no memory.
//
// attn_bwd takes its fp32 scratch (the dQ accumulator and two per-row
// vectors) from the stream-ordered allocator on every call.  Some callers
// cannot allow that: code running under an allocator that must not be
// re-entered, runtimes that forbid device allocations once they are set up
// (for example while a fixed memory budget is enforced), or embedded hosts
// that hand the library only the tensors themselves.  attn_bwd_noalloc
// serves them: the same kernels, with the scratch taken from one fixed array
// in device memory that the library owns.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes.  A
// GPU that loads it keeps it until the process exits (with the CUDA runtime's
// default lazy module loading that happens at the latest on the first call on
// that device).  Its device address is looked up once per device, by the
// first call made with that device current, and cached for the life of the
// process; a cudaDeviceReset of that device discards the array with the
// context, so the cached address must not be used after one.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn.h"
#include "attn_internal.h"

// 32.5 MiB: the dQ accumulator of 8 Mi elements of B*H*N*d (32 MiB) plus the
// two per-row vectors of such a problem (2 x 256 KiB at N = 8192), so that,
// for example, B=1, H=8, N=8192, d=128 fits exactly.  The rule is in attn.h.
constexpr size_t kNoAllocScratchBytes = (size_t(32) << 20) + (size_t(512) << 10);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace attn {
namespace {

constexpr int kNoAllocMaxDevices = 64;

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device, or nullptr.
// In host code the array's name is only a stand-in; the address the kernels
// need comes from the runtime, per device.
void* noalloc_scratch_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

bool ptr_ok(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool disjoint(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return !(x < y + nb && y < x + na);
}

}  // namespace
}  // namespace attn

extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                const void* dO, const float* lse, void* dq, void* dk, void* dv,
                                int B, int H, int N, int d, float scale, int causal,
                                void* stream) {
  using namespace attn;
  if (!ptr_ok(q) || !ptr_ok(k) || !ptr_ok(v) || !ptr_ok(o) || !ptr_ok(dO) || !ptr_ok(dq) ||
      !ptr_ok(dk) || !ptr_ok(dv) || !lse || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return kStatusInvalid;
  if (B < 1 || H < 1 || N < 1 || !std::isfinite(scale)) return kStatusInvalid;
  if (d != 32 && d != 64 && d != 128) return kStatusUnsupported;
  if (static_cast<int64_t>(B) * H > 65535 || N > (1 << 24)) return kStatusUnsupported;
  const size_t nbytes = static_cast<size_t>(B) * H * N * d * 2;
  const size_t lbytes = static_cast<size_t>(B) * H * N * 4;
  for (const void* out : {static_cast<const void*>(dq), static_cast<const void*>(dk),
                          static_cast<const void*>(dv)}) {
    for (const void* in : {q, k, v, o, dO})
      if (!disjoint(out, nbytes, in, nbytes)) return kStatusInvalid;
    if (!disjoint(out, nbytes, lse, lbytes)) return kStatusInvalid;
  }
  if (!disjoint(dq, nbytes, dk, nbytes) || !disjoint(dq, nbytes, dv, nbytes) ||
      !disjoint(dk, nbytes, dv, nbytes))
    return kStatusInvalid;
  // The whole problem's scratch must fit in the fixed array.
  const BwdScratch lay = bwd_scratch_layout(B * H, N, d);
  if (lay.total > kNoAllocScratchBytes) return kStatusUnsupported;

  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return kStatusCuda;
  if (major != 10 || minor != 3) return kStatusArch;
  char* ws = static_cast<char*>(noalloc_scratch_current_device());
  int* st = status_word_current_device();
  if (!ws || !st) return kStatusCuda;

  BwdArgs a;
  a.q = q; a.k = k; a.v = v; a.o = o; a.dO = dO; a.lse = lse;
  a.dq = dq; a.dk = dk; a.dv = dv;
  a.BH = B * H; a.N = N; a.d = d;
  a.sl2 = std::fabs(scale) * 1.4426950408889634f;
  a.scale = scale;
  a.causal = causal ? 1 : 0;
  a.negate = scale < 0.f ? 1 : 0;
  a.bf16 = true;
  a.stream = static_cast<cudaStream_t>(stream);
  a.status = st;
  // The preprocess launch rewrites every scratch entry this call reads (it
  // zeroes the dQ accumulator and fills both per-row vectors), so whatever an
  // earlier call left in the array does not matter.
  a.ws_dq = reinterpret_cast<float*>(ws + lay.dq_off);
  a.ws_lse2 = reinterpret_cast<float*>(ws + lay.lse2_off);
  a.ws_d = reinterpret_cast<float*>(ws + lay.d_off);
  return launch_bwd(a);
}
