// attn_decode.cu -- exact attention for one query token per (batch, head)
// against a long key/value cache, split across CTAs ("FlashDecoding").
//
// FlashAttention (PKM page), "注意" section: at decode time each step has a
// single query token, no N x N matrix exists, and the cost is reading the
// KV cache; the decode variant splits the keys.  The split is exact because
// of the same online-softmax algebra as the fused forward (PKM "三招" 2,
// FlashAttention深度攻略 §4): every split returns its running max m_s, sum
// l_s and unnormalised output O_s, and
//     m = max_s m_s,  l = sum_s e^{m_s - m} l_s,  O = sum_s e^{m_s - m} O_s / l.
//
// The work is a stream over K and V (4 B*H*L*d bytes of bf16) with about one
// FLOP per byte, so HBM bandwidth bounds it and no tensor core is involved:
//   attn_decode_split_kernel : grid (splits, B*H), 128 threads.  Each half
//       warp owns one key at a time (16 lanes x d/16 elements), keeps q in
//       registers, loads K and V rows of U keys ahead with 16-byte loads,
//       reduces q.k with 4 shuffles, and runs the online softmax in exp2
//       units.  The 8 half-warps are merged through shared memory and one
//       partial (m, l, O) per split goes to scratch.
//   attn_decode_merge_kernel : one CTA per (b, h) merges the splits, writes
//       O (bf16) and LSE.
#include <cmath>
#include <cstdint>

#include "attn.h"
#include "attn_internal.h"
#include "tc_sm103.cuh"

namespace attn {
namespace {

constexpr int kDecThreads = 128;
constexpr int kDecGroups = kDecThreads / 16;  // half warps per CTA
constexpr int kDecUnroll = 4;                 // keys in flight per half warp

template <int D>
struct DecVec;  // d/16 bf16 per lane
template <>
struct DecVec<128> {
  using T = uint4;
  static constexpr int E = 8;
};
template <>
struct DecVec<64> {
  using T = uint2;
  static constexpr int E = 4;
};
template <>
struct DecVec<32> {
  using T = uint32_t;
  static constexpr int E = 2;
};

template <int E>
__device__ __forceinline__ void unpack_bf16(const uint32_t* w, float* f) {
#pragma unroll
  for (int i = 0; i < E / 2; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <int D>
__global__ void __launch_bounds__(kDecThreads) attn_decode_split_kernel(
    const uint8_t* __restrict__ q, const uint8_t* __restrict__ k, const uint8_t* __restrict__ v,
    float* __restrict__ part, int L, int keys_per_split, float sl2) {
  griddep_wait();  // launched overlapped (launch_serialized)
  griddep_launch_dependents();
  using V = DecVec<D>;
  constexpr int E = V::E;
  const int s = blockIdx.x, bh = blockIdx.y, S = gridDim.x;
  const int g = threadIdx.x >> 4, l16 = threadIdx.x & 15;
  const int k0 = s * keys_per_split, k1 = min(L, k0 + keys_per_split);
  const size_t head = static_cast<size_t>(bh) * L * D;

  float qf[E];
  {
    typename V::T w = reinterpret_cast<const typename V::T*>(q + static_cast<size_t>(bh) * D * 2)[l16];
    unpack_bf16<E>(reinterpret_cast<const uint32_t*>(&w), qf);
  }
  float m = -INFINITY, l = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;

  const typename V::T* kb = reinterpret_cast<const typename V::T*>(k + head * 2);
  const typename V::T* vb = reinterpret_cast<const typename V::T*>(v + head * 2);
  // Every thread runs the same number of iterations (the shuffles below are
  // warp-wide); keys at or past k1 are masked.
  const int n_iter = (k1 - k0 + kDecGroups * kDecUnroll - 1) / (kDecGroups * kDecUnroll);
  for (int it = 0; it < n_iter; ++it) {
    const int j0 = k0 + g + it * kDecGroups * kDecUnroll;
    typename V::T kw[kDecUnroll], vw[kDecUnroll];
#pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      const int j = j0 + u * kDecGroups;
      if (j < k1) {
        kw[u] = __ldg(kb + static_cast<size_t>(j) * 16 + l16);
        vw[u] = __ldg(vb + static_cast<size_t>(j) * 16 + l16);
      } else {  // past the split: zeros, so p = 0 multiplies finite values
        kw[u] = typename V::T{};
        vw[u] = typename V::T{};
      }
    }
    float t[kDecUnroll];
#pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      float kf[E];
      unpack_bf16<E>(reinterpret_cast<const uint32_t*>(&kw[u]), kf);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) dot = fmaf(qf[e], kf[e], dot);
      dot += __shfl_xor_sync(0xffffffffu, dot, 8);
      dot += __shfl_xor_sync(0xffffffffu, dot, 4);
      dot += __shfl_xor_sync(0xffffffffu, dot, 2);
      dot += __shfl_xor_sync(0xffffffffu, dot, 1);
      t[u] = (j0 + u * kDecGroups < k1) ? dot * sl2 : -INFINITY;
    }
    float mx = fmaxf(fmaxf(t[0], t[1]), fmaxf(t[2], t[3]));
    const float m_new = fmaxf(m, mx);
    if (m_new == -INFINITY) continue;            // no valid key seen yet by this half warp
    const float alpha = ex2_approx(m - m_new);  // 0 while m = -inf
    m = m_new;
    l *= alpha;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] *= alpha;
#pragma unroll
    for (int u = 0; u < kDecUnroll; ++u) {
      const float p = ex2_approx(t[u] - m);  // t = -inf gives 0 (m is finite here)
      l += p;
      float vf[E];
      unpack_bf16<E>(reinterpret_cast<const uint32_t*>(&vw[u]), vf);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(p, vf[e], acc[e]);
    }
  }

  // merge the 8 half-warps of the CTA
  __shared__ float sm_m[kDecGroups], sm_l[kDecGroups];
  __shared__ float sm_o[kDecGroups][D];
  if (l16 == 0) {
    sm_m[g] = m;
    sm_l[g] = l;
  }
#pragma unroll
  for (int e = 0; e < E; ++e) sm_o[g][l16 * E + e] = acc[e];
  __syncthreads();
  float mm = -INFINITY;
#pragma unroll
  for (int i = 0; i < kDecGroups; ++i) mm = fmaxf(mm, sm_m[i]);
  float* out = part + (static_cast<size_t>(bh) * S + s) * (D + 2);
  for (int c = threadIdx.x; c < D; c += kDecThreads) {
    float o = 0.f;
#pragma unroll
    for (int i = 0; i < kDecGroups; ++i)
      if (sm_m[i] != -INFINITY) o += ex2_approx(sm_m[i] - mm) * sm_o[i][c];
    out[2 + c] = o;
  }
  if (threadIdx.x == 0) {
    float ll = 0.f;
#pragma unroll
    for (int i = 0; i < kDecGroups; ++i)
      if (sm_m[i] != -INFINITY) ll += ex2_approx(sm_m[i] - mm) * sm_l[i];
    out[0] = mm;
    out[1] = ll;
  }
}

template <int D>
__global__ void __launch_bounds__(128) attn_decode_merge_kernel(const float* __restrict__ part,
                                                                uint8_t* __restrict__ o,
                                                                float* __restrict__ lse, int S) {
  griddep_wait();  // launched overlapped (launch_serialized)
  griddep_launch_dependents();
  const int bh = blockIdx.x;
  const float* p = part + static_cast<size_t>(bh) * S * (D + 2);
  float mm = -INFINITY;
  for (int s = 0; s < S; ++s) mm = fmaxf(mm, p[s * (D + 2)]);
  float l = 0.f;
  for (int s = 0; s < S; ++s) {
    const float ms = p[s * (D + 2)];
    if (ms != -INFINITY) l += ex2_approx(ms - mm) * p[s * (D + 2) + 1];
  }
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < S; ++s) {
      const float ms = p[s * (D + 2)];
      if (ms != -INFINITY) acc += ex2_approx(ms - mm) * p[s * (D + 2) + 2 + c];
    }
    const __nv_bfloat16 b = __float2bfloat16_rn(acc / l);
    reinterpret_cast<__nv_bfloat16*>(o)[static_cast<size_t>(bh) * D + c] = b;
  }
  if (threadIdx.x == 0) lse[bh] = (mm + log2f(l)) * 0.69314718055994531f;
}

template <int D>
int launch_decode_t(const DecodeArgs& a) {
  const int S = a.splits;
  const int kps = (a.L + S - 1) / S;
  // Both launches overlap their predecessor's tail (a decode step is short,
  // so the launch latency is a visible share of it); each kernel waits for
  // its predecessor before reading anything.
  if (launch_serialized(true, attn_decode_split_kernel<D>, dim3(S, a.BH), dim3(kDecThreads), 0, a.stream,
                        static_cast<const uint8_t*>(a.q), static_cast<const uint8_t*>(a.k),
                        static_cast<const uint8_t*>(a.v), a.ws, a.L, kps,
                        a.sl2) != cudaSuccess)  // sl2 = scale*log2(e), signed
    return kStatusCuda;
  return launch_serialized(true, attn_decode_merge_kernel<D>, dim3(a.BH), dim3(128), 0, a.stream, a.ws,
                           static_cast<uint8_t*>(a.o), a.lse, S) == cudaSuccess
             ? kStatusOk
             : kStatusCuda;
}

}  // namespace

int decode_splits(int BH, int L) {
  // Enough CTAs for about 8 per SM on 152 SMs, at least 256 keys per split.
  const int want = (152 * 8 + BH - 1) / BH;
  const int cap = (L + 255) / 256;
  return std::max(1, std::min(std::min(want, cap), 256));
}

int launch_decode(const DecodeArgs& a) {
  switch (a.d) {
    case 32: return launch_decode_t<32>(a);
    case 64: return launch_decode_t<64>(a);
    case 128: return launch_decode_t<128>(a);
    default: return kStatusUnsupported;
  }
}

}  // namespace attn
