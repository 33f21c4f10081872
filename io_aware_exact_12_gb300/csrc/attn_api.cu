// attn_api.cu -- the C ABI declared in include/attn.h: argument validation,
// tensor-map encoding, backward scratch, launch bookkeeping and the sticky
// device status word.  Every step of the computation runs in the kernels of
// attn_fwd.cu / attn_bwd.cu; this file only checks and marshals.
#include <cmath>
#include <cstdint>
#include <atomic>
#include <cstring>
#include <mutex>

#include "attn.h"
#include "attn_internal.h"

// Sticky device-side status (one copy per device that loads the library).
__device__ int g_attn_status;

namespace attn {
namespace {

constexpr int kMaxDevices = 64;
thread_local int t_last_launches = 0;

std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {};
int g_arch_ok[kMaxDevices] = {};  // 0 unknown, 1 ok, -1 wrong arch
cuuint64_t g_smem_attr_done[kMaxDevices][8] = {};
const void* g_smem_attr_func[kMaxDevices][8] = {};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Current device, checked to be compute capability 10.3; returns a status.
int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) return kStatusCuda;
  if (*dev < 0 || *dev >= kMaxDevices) return kStatusUnsupported;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_arch_ok[*dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess)
      return kStatusCuda;
    g_arch_ok[*dev] = (major == 10 && minor == 3) ? 1 : -1;
  }
  return g_arch_ok[*dev] == 1 ? kStatusOk : kStatusArch;
}

int* status_ptr(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Checks shared by forward and backward.  Pure host logic: no CUDA call.
int validate_common(int B, int H, int N, int d, float scale) {
  if (B < 1 || H < 1 || N < 1) return kStatusInvalid;
  if (!std::isfinite(scale)) return kStatusInvalid;
  if (d != 32 && d != 64 && d != 128) return kStatusUnsupported;
  const int64_t BH = static_cast<int64_t>(B) * H;
  if (BH > 65535) return kStatusUnsupported;           // grid.y limit
  if (N > (1 << 24)) return kStatusUnsupported;         // keeps row indices and TMA coords in range
  return kStatusOk;
}

}  // namespace

bool encode_bhnd_map(CUtensorMap* map, const void* base, int BH, int N, int d, int box_inner,
                     int box_rows, int row_bytes, bool bf16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(d) * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows),
                             1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapSwizzle swz =
      row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_map_u8(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t stride1, uint64_t stride2, uint32_t b0, uint32_t b1) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1, stride2};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool ensure_smem_attr(const void* func, int bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < 8; ++i) {
    if (g_smem_attr_func[dev][i] == func && g_smem_attr_done[dev][i] >= (cuuint64_t)bytes) return true;
  }
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return false;
  for (int i = 0; i < 8; ++i) {
    if (g_smem_attr_func[dev][i] == nullptr || g_smem_attr_func[dev][i] == func) {
      g_smem_attr_func[dev][i] = func;
      g_smem_attr_done[dev][i] = static_cast<cuuint64_t>(bytes);
      break;
    }
  }
  return true;
}

bool check_launch_regs(const void* func, int regs) {
  // The register count is a property of the compiled kernel: look it up once
  // per kernel (cudaFuncGetAttributes costs about a microsecond per call).
  static std::mutex mu;
  static const void* seen_func[64] = {};
  static int seen_regs[64] = {};
  {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < 64 && seen_func[i]; ++i)
      if (seen_func[i] == func) return seen_regs[i] == regs;
  }
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, func) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lk(mu);
  for (int i = 0; i < 64; ++i) {
    if (seen_func[i] == func) break;
    if (!seen_func[i]) {
      seen_func[i] = func;
      seen_regs[i] = fa.numRegs;
      break;
    }
  }
  return fa.numRegs == regs;
}

int device_sm_count() {
  static std::atomic<int> count[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int n = count[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 0;
  count[dev].store(n, std::memory_order_relaxed);
  return n;
}

int bwd_tail_split(int BH, int N, int causal) {
  return bwd_tail_split_items(BH, N, causal, device_sm_count());
}

int* status_word_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  return status_ptr(dev);
}

BwdScratch bwd_scratch_layout(int BH, int N, int d) {
  auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
  const size_t Npad = static_cast<size_t>((N + 127) / 128) * 128;
  BwdScratch s;
  s.dq_off = 0;
  s.lse2_off = up(static_cast<size_t>(BH) * N * d * sizeof(float));
  s.d_off = s.lse2_off + up(static_cast<size_t>(BH) * Npad * sizeof(float));
  s.total = s.d_off + up(static_cast<size_t>(BH) * Npad * sizeof(float));
  return s;
}

namespace {

constexpr DropParams kNoDrop = {0u, 0u, 0u, 0u, 1.f};

// Dropout probability -> keep threshold and Philox key.  t = 256 keeps
// everything, which is no dropout (t = 0 in the result).
int make_drop(float p, unsigned long long seed, unsigned int offset, DropParams* out) {
  if (!std::isfinite(p) || p < 0.f || p >= 1.f) return kStatusInvalid;
  const double t = std::floor((1.0 - static_cast<double>(p)) * 256.0 + 0.5);
  if (t < 1.0) return kStatusInvalid;
  *out = kNoDrop;
  if (t >= 256.0) return kStatusOk;
  out->t = static_cast<uint32_t>(t);
  out->k0 = static_cast<uint32_t>(seed);
  out->k1 = static_cast<uint32_t>(seed >> 32);
  out->offset = offset;
  out->rscale = static_cast<float>(256.0 / t);
  return kStatusOk;
}

int fwd_entry(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
              int N, int d, float scale, int causal, void* stream, bool bf16,
              const DropParams& drop = kNoDrop) {
  if (!q || !k || !v || !o || !lse) return kStatusInvalid;
  int rc = validate_common(B, H, N, d, scale);
  if (rc) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return kStatusInvalid;
  const size_t nbytes = static_cast<size_t>(B) * H * N * d * 2;
  const size_t lbytes = static_cast<size_t>(B) * H * N * 4;
  for (const void* in : {q, k, v})
    if (overlaps(o, nbytes, in, nbytes) || overlaps(lse, lbytes, in, nbytes)) return kStatusInvalid;
  if (overlaps(o, nbytes, lse, lbytes)) return kStatusInvalid;
  int dev = 0;
  if ((rc = current_device(&dev))) return rc;
  int* st = status_ptr(dev);
  if (!st) return kStatusCuda;
  FwdArgs a;
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  a.BH = B * H; a.N = N; a.d = d;
  a.sl2 = std::fabs(scale) * 1.4426950408889634f;
  a.causal = causal ? 1 : 0;
  a.negate = scale < 0.f ? 1 : 0;
  a.bf16 = bf16;
  a.stream = static_cast<cudaStream_t>(stream);
  a.status = st;
  a.drop = drop;
  rc = launch_fwd(a);
  if (rc == kStatusOk) t_last_launches = 1;
  return rc;
}

int bwd_entry(const void* q, const void* k, const void* v, const void* o, const void* dO,
              const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
              float scale, int causal, void* stream, bool bf16, const DropParams& drop = kNoDrop,
              const uint8_t* bmask = nullptr, int mask_heads = 1) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return kStatusInvalid;
  int rc = validate_common(B, H, N, d, scale);
  if (rc) return rc;
  for (const void* p : {q, k, v, o, dO, static_cast<const void*>(dq), static_cast<const void*>(dk),
                        static_cast<const void*>(dv)})
    if (!aligned16(p)) return kStatusInvalid;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return kStatusInvalid;
  const size_t nbytes = static_cast<size_t>(B) * H * N * d * 2;
  const size_t lbytes = static_cast<size_t>(B) * H * N * 4;
  for (const void* out : {static_cast<const void*>(dq), static_cast<const void*>(dk),
                          static_cast<const void*>(dv)}) {
    for (const void* in : {q, k, v, o, dO})
      if (overlaps(out, nbytes, in, nbytes)) return kStatusInvalid;
    if (overlaps(out, nbytes, lse, lbytes)) return kStatusInvalid;
  }
  if (overlaps(dq, nbytes, dk, nbytes) || overlaps(dq, nbytes, dv, nbytes) ||
      overlaps(dk, nbytes, dv, nbytes))
    return kStatusInvalid;
  int dev = 0;
  if ((rc = current_device(&dev))) return rc;
  int* st = status_ptr(dev);
  if (!st) return kStatusCuda;
  const BwdScratch lay = bwd_scratch_layout(B * H, N, d);
  const int tail = bmask ? 0 : bwd_tail_split(B * H, N, causal);
  const size_t part_bytes = static_cast<size_t>(tail) * 4 * 128 * d * sizeof(float);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, lay.total + part_bytes, s) != cudaSuccess) return kStatusCuda;
  BwdArgs a;
  a.q = q; a.k = k; a.v = v; a.o = o; a.dO = dO; a.lse = lse;
  a.dq = dq; a.dk = dk; a.dv = dv;
  a.BH = B * H; a.N = N; a.d = d;
  a.sl2 = std::fabs(scale) * 1.4426950408889634f;
  a.scale = scale;
  a.causal = causal ? 1 : 0;
  a.negate = scale < 0.f ? 1 : 0;
  a.bf16 = bf16;
  a.stream = s;
  a.status = st;
  a.ws_dq = reinterpret_cast<float*>(static_cast<char*>(ws) + lay.dq_off);
  a.ws_lse2 = reinterpret_cast<float*>(static_cast<char*>(ws) + lay.lse2_off);
  a.ws_d = reinterpret_cast<float*>(static_cast<char*>(ws) + lay.d_off);
  a.drop = drop;
  a.bmask = bmask;
  a.H = H;
  a.mask_heads = mask_heads;
  a.tail_split = tail;
  a.ws_part = tail ? reinterpret_cast<float*>(static_cast<char*>(ws) + lay.total) : nullptr;
  rc = launch_bwd(a);
  const cudaError_t fe = cudaFreeAsync(ws, s);
  if (rc == kStatusOk && fe != cudaSuccess) rc = kStatusCuda;
  if (rc == kStatusOk) t_last_launches = 3;
  return rc;
}

int blocksparse_entry(const void* q, const void* k, const void* v, void* o, float* lse,
                      const uint8_t* mask, int mask_heads, int B, int H, int N, int d, float scale,
                      int causal, void* stream, bool bf16, const DropParams& drop = kNoDrop) {
  if (!mask) return kStatusInvalid;
  if (mask_heads != 1 && mask_heads != H) return kStatusInvalid;
  if ((N + 127) / 128 > kMaxSparseTiles) return kStatusUnsupported;
  if (!q || !k || !v || !o || !lse) return kStatusInvalid;
  int rc = validate_common(B, H, N, d, scale);
  if (rc) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return kStatusInvalid;
  const size_t nbytes = static_cast<size_t>(B) * H * N * d * 2;
  const size_t lbytes = static_cast<size_t>(B) * H * N * 4;
  for (const void* in : {q, k, v})
    if (overlaps(o, nbytes, in, nbytes) || overlaps(lse, lbytes, in, nbytes)) return kStatusInvalid;
  if (overlaps(o, nbytes, lse, lbytes)) return kStatusInvalid;
  int dev = 0;
  if ((rc = current_device(&dev))) return rc;
  int* st = status_ptr(dev);
  if (!st) return kStatusCuda;
  FwdArgs a;
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  a.BH = B * H; a.N = N; a.d = d;
  a.sl2 = std::fabs(scale) * 1.4426950408889634f;
  a.causal = causal ? 1 : 0;
  a.negate = scale < 0.f ? 1 : 0;
  a.bf16 = bf16;
  a.stream = static_cast<cudaStream_t>(stream);
  a.status = st;
  a.bmask = mask;
  a.H = H;
  a.mask_heads = mask_heads;
  a.drop = drop;
  rc = launch_fwd(a);
  if (rc == kStatusOk) t_last_launches = 1;
  return rc;
}

int decode_entry(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int L, int d, float scale, void* stream) {
  if (!q || !k || !v || !o || !lse) return kStatusInvalid;
  int rc = validate_common(B, H, L, d, scale);
  if (rc) return rc;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return kStatusInvalid;
  const size_t qbytes = static_cast<size_t>(B) * H * d * 2;
  const size_t kvbytes = qbytes * static_cast<size_t>(L);
  const size_t lbytes = static_cast<size_t>(B) * H * 4;
  for (const void* in : {q, k, v}) {
    const size_t n = in == q ? qbytes : kvbytes;
    if (overlaps(o, qbytes, in, n) || overlaps(lse, lbytes, in, n)) return kStatusInvalid;
  }
  if (overlaps(o, qbytes, lse, lbytes)) return kStatusInvalid;
  int dev = 0;
  if ((rc = current_device(&dev))) return rc;
  DecodeArgs a;
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  a.BH = B * H; a.L = L; a.d = d;
  a.sl2 = scale * 1.4426950408889634f;
  a.splits = decode_splits(a.BH, L);
  a.stream = static_cast<cudaStream_t>(stream);
  const size_t ws_bytes = static_cast<size_t>(a.BH) * a.splits * (d + 2) * sizeof(float);
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, ws_bytes, a.stream) != cudaSuccess) return kStatusCuda;
  a.ws = static_cast<float*>(ws);
  rc = launch_decode(a);
  const cudaError_t fe = cudaFreeAsync(ws, a.stream);
  if (rc == kStatusOk && fe != cudaSuccess) rc = kStatusCuda;
  if (rc == kStatusOk) t_last_launches = 2;
  return rc;
}

int fp8_entry(const void* q, const void* k, const void* v, float dq_s, float dk_s, float dv_s, void* o,
              float* lse, int B, int H, int N, int d, float scale, int causal, void* stream) {
  if (!q || !k || !v || !o || !lse) return kStatusInvalid;
  int rc = validate_common(B, H, N, d, scale);
  if (rc) return rc;
  if (!std::isfinite(dq_s) || !std::isfinite(dk_s) || !std::isfinite(dv_s) || dq_s <= 0.f ||
      dk_s <= 0.f || dv_s <= 0.f)
    return kStatusInvalid;
  if (d != 128 || scale < 0.f) return kStatusUnsupported;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return kStatusInvalid;
  const size_t ibytes = static_cast<size_t>(B) * H * N * d;  // one byte per input element
  const size_t obytes = ibytes * 2, lbytes = static_cast<size_t>(B) * H * N * 4;
  for (const void* in : {q, k, v})
    if (overlaps(o, obytes, in, ibytes) || overlaps(lse, lbytes, in, ibytes)) return kStatusInvalid;
  if (overlaps(o, obytes, lse, lbytes)) return kStatusInvalid;
  int dev = 0;
  if ((rc = current_device(&dev))) return rc;
  int* st = status_ptr(dev);
  if (!st) return kStatusCuda;
  Fp8Args a;
  a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
  a.BH = B * H; a.N = N; a.d = d;
  a.sl2 = scale * dq_s * dk_s * 1.4426950408889634f;
  a.descale_v = dv_s;
  a.causal = causal ? 1 : 0;
  a.stream = static_cast<cudaStream_t>(stream);
  a.status = st;
  const size_t Npad = static_cast<size_t>((N + 127) / 128) * 128;
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, static_cast<size_t>(a.BH) * 128 * Npad, a.stream) != cudaSuccess)
    return kStatusCuda;
  a.ws_vt = static_cast<uint8_t*>(ws);
  rc = launch_fwd_fp8(a);
  const cudaError_t fe = cudaFreeAsync(ws, a.stream);
  if (rc == kStatusOk && fe != cudaSuccess) rc = kStatusCuda;
  if (rc == kStatusOk) t_last_launches = 2;
  return rc;
}

}  // namespace
}  // namespace attn

extern "C" {

int attn_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int N, int d, float scale, int causal, float p_drop,
                     unsigned long long seed, unsigned int offset, void* stream) {
  attn::DropParams dr;
  const int rc = attn::make_drop(p_drop, seed, offset, &dr);
  if (rc) return rc;
  return attn::fwd_entry(q, k, v, o, lse, B, H, N, d, scale, causal, stream, true, dr);
}

int attn_fwd_dropout_f16(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int N, int d, float scale, int causal, float p_drop,
                         unsigned long long seed, unsigned int offset, void* stream) {
  attn::DropParams dr;
  const int rc = attn::make_drop(p_drop, seed, offset, &dr);
  if (rc) return rc;
  return attn::fwd_entry(q, k, v, o, lse, B, H, N, d, scale, causal, stream, false, dr);
}

int attn_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const void* dO,
                     const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                     float scale, int causal, float p_drop, unsigned long long seed,
                     unsigned int offset, void* stream) {
  attn::DropParams dr;
  const int rc = attn::make_drop(p_drop, seed, offset, &dr);
  if (rc) return rc;
  return attn::bwd_entry(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, stream, true, dr);
}

int attn_bwd_dropout_f16(const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                         float scale, int causal, float p_drop, unsigned long long seed,
                         unsigned int offset, void* stream) {
  attn::DropParams dr;
  const int rc = attn::make_drop(p_drop, seed, offset, &dr);
  if (rc) return rc;
  return attn::bwd_entry(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, stream, false, dr);
}

int attn_fwd_fp8(const void* q, const void* k, const void* v, float descale_q, float descale_k,
                 float descale_v, void* o, float* lse, int B, int H, int N, int d, float scale,
                 int causal, void* stream) {
  return attn::fp8_entry(q, k, v, descale_q, descale_k, descale_v, o, lse, B, H, N, d, scale, causal,
                         stream);
}

}  // extern "C"

namespace attn {
namespace {
int blocksparse_bwd_entry(const void* q, const void* k, const void* v, const void* o, const void* dO,
                          const float* lse, void* dq, void* dk, void* dv, const unsigned char* block_mask,
                          int mask_heads, int B, int H, int N, int d, float scale, int causal, void* stream,
                          bool bf16, const DropParams& drop = kNoDrop) {
  if (!block_mask) return kStatusInvalid;
  if (mask_heads != 1 && mask_heads != H) return kStatusInvalid;
  if (N > 0 && (N + 127) / 128 > kMaxSparseTiles) return kStatusUnsupported;
  return bwd_entry(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, stream, bf16, drop,
                   block_mask, mask_heads);
}
}  // namespace
}  // namespace attn

extern "C" {

int attn_bwd_blocksparse(const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, void* dq, void* dk, void* dv,
                         const unsigned char* block_mask, int mask_heads, int B, int H, int N, int d,
                         float scale, int causal, void* stream) {
  return attn::blocksparse_bwd_entry(q, k, v, o, dO, lse, dq, dk, dv, block_mask, mask_heads, B, H, N, d,
                                     scale, causal, stream, true);
}

int attn_bwd_blocksparse_f16(const void* q, const void* k, const void* v, const void* o, const void* dO,
                             const float* lse, void* dq, void* dk, void* dv,
                             const unsigned char* block_mask, int mask_heads, int B, int H, int N, int d,
                             float scale, int causal, void* stream) {
  return attn::blocksparse_bwd_entry(q, k, v, o, dO, lse, dq, dk, dv, block_mask, mask_heads, B, H, N, d,
                                     scale, causal, stream, false);
}

int attn_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse,
                         const unsigned char* block_mask, int mask_heads, int B, int H, int N, int d,
                         float scale, int causal, void* stream) {
  return attn::blocksparse_entry(q, k, v, o, lse, block_mask, mask_heads, B, H, N, d, scale, causal,
                                 stream, true);
}

int attn_fwd_blocksparse_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                             const unsigned char* block_mask, int mask_heads, int B, int H, int N, int d,
                             float scale, int causal, void* stream) {
  return attn::blocksparse_entry(q, k, v, o, lse, block_mask, mask_heads, B, H, N, d, scale, causal,
                                 stream, false);
}

int attn_fwd_blocksparse_dropout(const void* q, const void* k, const void* v, void* o, float* lse,
                                 const unsigned char* block_mask, int mask_heads, int B, int H, int N, int d,
                                 float scale, int causal, float p_drop, unsigned long long seed,
                                 unsigned int offset, void* stream) {
  attn::DropParams dr;
  const int rc = attn::make_drop(p_drop, seed, offset, &dr);
  if (rc) return rc;
  return attn::blocksparse_entry(q, k, v, o, lse, block_mask, mask_heads, B, H, N, d, scale, causal,
                                 stream, true, dr);
}

int attn_fwd_blocksparse_dropout_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                                     const unsigned char* block_mask, int mask_heads, int B, int H, int N,
                                     int d, float scale, int causal, float p_drop, unsigned long long seed,
                                     unsigned int offset, void* stream) {
  attn::DropParams dr;
  const int rc = attn::make_drop(p_drop, seed, offset, &dr);
  if (rc) return rc;
  return attn::blocksparse_entry(q, k, v, o, lse, block_mask, mask_heads, B, H, N, d, scale, causal,
                                 stream, false, dr);
}

int attn_bwd_blocksparse_dropout(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                 const float* lse, void* dq, void* dk, void* dv,
                                 const unsigned char* block_mask, int mask_heads, int B, int H, int N, int d,
                                 float scale, int causal, float p_drop, unsigned long long seed,
                                 unsigned int offset, void* stream) {
  attn::DropParams dr;
  const int rc = attn::make_drop(p_drop, seed, offset, &dr);
  if (rc) return rc;
  return attn::blocksparse_bwd_entry(q, k, v, o, dO, lse, dq, dk, dv, block_mask, mask_heads, B, H, N, d,
                                     scale, causal, stream, true, dr);
}

int attn_bwd_blocksparse_dropout_f16(const void* q, const void* k, const void* v, const void* o,
                                     const void* dO, const float* lse, void* dq, void* dk, void* dv,
                                     const unsigned char* block_mask, int mask_heads, int B, int H, int N,
                                     int d, float scale, int causal, float p_drop, unsigned long long seed,
                                     unsigned int offset, void* stream) {
  attn::DropParams dr;
  const int rc = attn::make_drop(p_drop, seed, offset, &dr);
  if (rc) return rc;
  return attn::blocksparse_bwd_entry(q, k, v, o, dO, lse, dq, dk, dv, block_mask, mask_heads, B, H, N, d,
                                     scale, causal, stream, false, dr);
}

int attn_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int L, int d, float scale, void* stream) {
  return attn::decode_entry(q, k, v, o, lse, B, H, L, d, scale, stream);
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int N, int d, float scale, int causal, void* stream) {
  return attn::fwd_entry(q, k, v, o, lse, B, H, N, d, scale, causal, stream, true);
}

int attn_fwd_f16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, void* stream) {
  return attn::fwd_entry(q, k, v, o, lse, B, H, N, d, scale, causal, stream, false);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
             const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
             float scale, int causal, void* stream) {
  return attn::bwd_entry(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, stream, true);
}

int attn_bwd_f16(const void* q, const void* k, const void* v, const void* o, const void* dO,
                 const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 float scale, int causal, void* stream) {
  return attn::bwd_entry(q, k, v, o, dO, lse, dq, dk, dv, B, H, N, d, scale, causal, stream, false);
}

int attn_sync_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return attn::kStatusCuda;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return attn::kStatusCuda;
  int value = 0;
  const int zero = 0;
  if (cudaMemcpyFromSymbol(&value, g_attn_status, sizeof(int)) != cudaSuccess) return attn::kStatusCuda;
  if (value != 0 && cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(int)) != cudaSuccess)
    return attn::kStatusCuda;
  return value;
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_CUDA: return "CUDA runtime error";
    case ATTN_ERR_TIMEOUT: return "device pipeline wait timed out";
    case ATTN_ERR_ARCH: return "device is not sm_103 (GB300)";
    case ATTN_ERR_DEVICE_CHECK: return "device-side check failed";
    default: return "unknown status";
  }
}

int attn_last_launch_count(void) { return attn::t_last_launches; }

}  // extern "C"
