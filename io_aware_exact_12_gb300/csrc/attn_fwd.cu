// attn_fwd.cu -- fused exact-attention forward for sm_103a.
//
// Method (FlashAttention (PKM page), "三招" 1 Tiling and 2 Online Softmax;
// FlashAttention深度攻略 §3 tiling, §4 online softmax, §7 fusion): for a block
// of query rows, stream the key/value blocks through on-chip memory, keep per
// row the running max m, running sum l and an unnormalised output O, rescale
// O and l by exp(m_old - m_new) whenever the max grows, and divide by l once
// at the end.  S = Q K^T and P never leave the SM.
//
// GB300 mapping (one CTA per SM, 10 warps):
//   * CTA = 256 query rows of one (batch, head): two 128-row tiles Q0, Q1 that
//     take turns on the tensor core (while one tile's softmax runs, the other
//     tile's MMAs do), sharing every K/V tile loaded.
//   * warp 8  : TMA producer -- Q0/Q1 once, then K_j and V_j into an
//               NST-stage ring (128B-swizzled tiles, 3-D tensor maps so a
//               tile never straddles two heads and rows >= N read as zero).
//   * warp 9  : TMEM owner and single-thread tcgen05.mma issuer.
//               S_q = Q_q K_j^T  (SS: both operands K-major in shared memory)
//               O_q += P_q V_j   (TS: P from TMEM, V MN-major in shared memory)
//   * warps 0-3 / 4-7 : softmax for Q0 / Q1, one thread per query row (TMEM
//               lane).  exp2 with scale*log2(e) folded in; the reference max is
//               only moved when it grows by more than 2^8 (the same stale max
//               is used for l and for P, so the result is unchanged); O is
//               rescaled in TMEM by the same thread; P is written back to TMEM
//               as bf16/fp16 over the first half of its S columns.
//   * TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D,256+2D).
// Causal: key tiles entirely above the diagonal are never loaded or
// multiplied; only the diagonal tile (and the ragged last tile) are masked.
#include "attn_internal.h"
#include "tc_sm103.cuh"

namespace attn {

namespace {

constexpr float kRescaleThresholdLog2 = 8.0f;

template <int D>
struct FwdCfg {
  static constexpr int BM = 128;                     // query rows per tile (MMA M)
  static constexpr int BN = 128;                     // key rows per tile
  static constexpr int ROWB = (D >= 64) ? 128 : 64;  // bytes per swizzled row
  static constexpr int CH = ROWB / 2;                // elements per swizzled row
  static constexpr int NCH = D / CH;                 // column chunks per tile
  static constexpr uint32_t SWZ = (ROWB == 128) ? kSwizzle128B : kSwizzle64B;
  static constexpr int SBO = 8 * ROWB;               // bytes between 8-row groups
  static constexpr int CHUNK_BYTES = 128 * ROWB;     // one column chunk of a 128-row tile
  static constexpr int TILE_BYTES = 128 * D * 2;
  static constexpr int NST = (D == 128) ? 2 : 3;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = 2 * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NST * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_V + NST * TILE_BYTES;
  // barriers: q_full | k_full[NST] | k_empty[NST] | v_full[NST] | v_empty[NST]
  //           | s_full[2] | p_full[2] | o_done[2] | mma_done
  static constexpr int B_QFULL = 0;
  static constexpr int B_KFULL = 1;
  static constexpr int B_KEMPTY = B_KFULL + NST;
  static constexpr int B_VFULL = B_KEMPTY + NST;
  static constexpr int B_VEMPTY = B_VFULL + NST;
  static constexpr int B_SFULL = B_VEMPTY + NST;
  static constexpr int B_PFULL = B_SFULL + 2;
  static constexpr int B_ODONE = B_PFULL + 2;
  static constexpr int B_MMADONE = B_ODONE + 2;
  static constexpr int NBAR = B_MMADONE + 1;
  static constexpr int OFF_TMEMSLOT = OFF_BAR + NBAR * 8;
  static constexpr int OFF_ABORT = OFF_TMEMSLOT + 4;
  static constexpr int SMEM_BYTES = OFF_ABORT + 12;
  static constexpr int THREADS = 320;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(2 * 128 + 2 * D <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// K-major operand tile (rows x D, row-major in global): descriptor for the
// 16-element K slice `kk`.
template <int D>
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile, int kk) {
  using C = FwdCfg<D>;
  const int e = kk * 16;
  return smem_desc(tile + (e / C::CH) * C::CHUNK_BYTES + (e % C::CH) * 2, 16, C::SBO, C::SWZ);
}

// MN-major operand tile (K rows x D columns, D contiguous): descriptor for the
// 16-row K slice `kk`.
template <int D>
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t tile, int kk) {
  using C = FwdCfg<D>;
  return smem_desc(tile + kk * 16 * C::ROWB, C::CHUNK_BYTES, C::SBO, C::SWZ);
}

// Waits that ignore the abort flag: used only to drain work already issued.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(FwdCfg<D>::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, uint8_t* __restrict__ o_out,
                    float* __restrict__ lse_out, int N, float sl2, int causal, int negate,
                    int* status) {
  using C = FwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int qb = causal ? (gridDim.x - 1 - blockIdx.x) : blockIdx.x;  // heavy tiles first
  const int nkv_all = (N + C::BN - 1) / C::BN;
  int nkv[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int row0 = qb * 2 * C::BM + q * C::BM;
    nkv[q] = (row0 >= N) ? 0 : (causal ? min(nkv_all, row0 / C::BN + 1) : nkv_all);
  }
  const int nkv_max = max(nkv[0], nkv[1]);

  const uint32_t sbase = smem_addr(smem);
  if (sbase & 1023u) {  // swizzle atoms need 1024-byte alignment; never expected
    if (threadIdx.x == 0) atomicExch(status, kStatusDeviceCheck);
    return;
  }
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEMSLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);

  if (threadIdx.x == 0) {
    mbar_init(bar(C::B_QFULL), 1);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar(C::B_KFULL + s), 1);
      mbar_init(bar(C::B_KEMPTY + s), 1);
      mbar_init(bar(C::B_VFULL + s), 1);
      mbar_init(bar(C::B_VEMPTY + s), 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(bar(C::B_SFULL + q), 1);
      mbar_init(bar(C::B_PFULL + q), C::BM);
      mbar_init(bar(C::B_ODONE + q), 1);
    }
    mbar_init(bar(C::B_MMADONE), 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(smem_addr(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  const uint32_t sQ = sbase + C::OFF_Q;
  const uint32_t sK = sbase + C::OFF_K;
  const uint32_t sV = sbase + C::OFF_V;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      mbar_arrive_expect_tx(bar(C::B_QFULL), 2 * C::TILE_BYTES);
      for (int q = 0; q < 2; ++q)
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(sQ + q * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_q, bar(C::B_QFULL), c * C::CH,
                      qb * 2 * C::BM + q * C::BM, bh);
      int issued = 0;
      for (int j = 0; j < nkv_max; ++j) {
        const int s = j % C::NST, u = j / C::NST;
        if (u > 0 && !mbar_wait(bar(C::B_KEMPTY + s), (u - 1) & 1, abort_flag, status)) break;
        mbar_arrive_expect_tx(bar(C::B_KFULL + s), C::TILE_BYTES);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(sK + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_k, bar(C::B_KFULL + s),
                      c * C::CH, j * C::BN, bh);
        if (u > 0 && !mbar_wait(bar(C::B_VEMPTY + s), (u - 1) & 1, abort_flag, status)) {
          issued = -(j + 1);  // K_j issued, V_j not
          break;
        }
        mbar_arrive_expect_tx(bar(C::B_VFULL + s), C::TILE_BYTES);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(sV + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_v, bar(C::B_VFULL + s),
                      c * C::CH, j * C::BN, bh);
        issued = j + 1;
      }
      if (*abort_flag) {
        // Let every copy already issued land before the CTA's shared memory goes away.
        drain_wait(bar(C::B_QFULL), 0);
        const int nk = issued >= 0 ? issued : -issued;
        const int nv = issued >= 0 ? issued : -issued - 1;
        for (int s = 0; s < C::NST; ++s) {
          const int ck = nk > s ? (nk - 1 - s) / C::NST + 1 : 0;  // loads issued on stage s
          const int cv = nv > s ? (nv - 1 - s) / C::NST + 1 : 0;
          if (ck) drain_wait(bar(C::B_KFULL + s), (ck - 1) & 1);
          if (cv) drain_wait(bar(C::B_VFULL + s), (cv - 1) & 1);
        }
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = instr_desc_f16(C::BM, C::BN, BF16, false, false, negate != 0);
      const uint32_t idesc_o = instr_desc_f16(C::BM, D, BF16, false, true);
      bool ok = nkv_max == 0 || mbar_wait(bar(C::B_QFULL), 0, abort_flag, status);
      for (int j = 0; ok && j < nkv_max; ++j) {
        const int s = j % C::NST;
        const uint32_t ph = (j / C::NST) & 1;
        if (!(ok = mbar_wait(bar(C::B_KFULL + s), ph, abort_flag, status))) break;
        tc_fence_after_sync();
        for (int q = 0; q < 2 && ok; ++q) {
          if (j >= nkv[q]) continue;
          if (j > 0) {  // P_q of the previous step must be consumed before S_q is overwritten
            if (!(ok = mbar_wait(bar(C::B_ODONE + q), (j - 1) & 1, abort_flag, status))) break;
            tc_fence_after_sync();
          }
          const uint32_t d_s = tmem + q * C::BN;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss(d_s, desc_kmajor<D>(sQ + q * C::TILE_BYTES, kk),
                   desc_kmajor<D>(sK + s * C::TILE_BYTES, kk), idesc_s, kk > 0 ? 1u : 0u);
          tc_commit(bar(C::B_SFULL + q));
        }
        if (!ok) break;
        tc_commit(bar(C::B_KEMPTY + s));
        if (!(ok = mbar_wait(bar(C::B_VFULL + s), ph, abort_flag, status))) break;
        tc_fence_after_sync();
        for (int q = 0; q < 2 && ok; ++q) {
          if (j >= nkv[q]) continue;
          if (!(ok = mbar_wait(bar(C::B_PFULL + q), j & 1, abort_flag, status))) break;
          tc_fence_after_sync();
          const uint32_t d_o = tmem + 2 * C::BN + q * D;
          const uint32_t a_p = tmem + q * C::BN;
#pragma unroll
          for (int kk = 0; kk < C::BN / 16; ++kk)
            mma_ts(d_o, a_p + kk * 8, desc_mnmajor<D>(sV + s * C::TILE_BYTES, kk), idesc_o,
                   (j > 0 || kk > 0) ? 1u : 0u);
          tc_commit(bar(C::B_ODONE + q));
        }
        if (!ok) break;
        tc_commit(bar(C::B_VEMPTY + s));
      }
      // Every MMA issued above must finish before TMEM is released.
      tc_commit(bar(C::B_MMADONE));
      drain_wait(bar(C::B_MMADONE), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    const int q = warp >> 2;
    const int r = threadIdx.x & 127;
    const int row0 = qb * 2 * C::BM + q * C::BM;
    const int row = row0 + r;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + q * C::BN;
    const uint32_t tO = tmem + lane_off + 2 * C::BN + q * D;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    const int nk = nkv[q];
    for (int j = 0; j < nk; ++j) {
      if (!(ok = mbar_wait(bar(C::B_SFULL + q), j & 1, abort_flag, status))) break;
      tc_fence_after_sync();
      float sv[128];
      {
        uint32_t u[64];
        tmem_ld64(tS, u);
#pragma unroll
        for (int c = 0; c < 64; ++c) sv[c] = __uint_as_float(u[c]);
        tmem_ld64(tS + 64, u);
#pragma unroll
        for (int c = 0; c < 64; ++c) sv[64 + c] = __uint_as_float(u[c]);
      }
      const int kv0 = j * C::BN;
      const bool masked = (kv0 + C::BN > N) || (causal && kv0 + C::BN - 1 > row0);
      int lim = C::BN;  // keys kv0 + c with c < lim are visible to this row
      if (masked) {
        lim = min(N - kv0, C::BN);
        if (causal) lim = min(lim, row - kv0 + 1);
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= lim) sv[c] = -INFINITY;
      }
      float mx = sv[0];
#pragma unroll
      for (int c = 1; c < 128; ++c) mx = fmaxf(mx, sv[c]);
      const float m_new = fmaxf(m, mx * sl2);
      float alpha = 1.f;
      if (m_new > m + kRescaleThresholdLog2) {  // also taken on the first tile (m = -inf)
        alpha = ex2_approx(m - m_new);
        m = m_new;
      }
      const float neg_m = (m == -INFINITY) ? 0.f : -m;
      if (masked) {
#pragma unroll
        for (int c = 0; c < 128; ++c) sv[c] = (c < lim) ? ex2_approx(fmaf(sv[c], sl2, neg_m)) : 0.f;
      } else {
#pragma unroll
        for (int c = 0; c < 128; ++c) sv[c] = ex2_approx(fmaf(sv[c], sl2, neg_m));
      }
      // O_q holds the previous steps' sum: rescale it when any row of this warp moved its max.
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int c0 = 0; c0 < D / 32; ++c0) {
          uint32_t ov[32];
          tmem_ld32(tO + c0 * 32, ov);
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tmem_st32(tO + c0 * 32, ov);
        }
      }
      // P is rounded to the input type for the P V product; l sums the rounded
      // values, so the weights that multiply V sum to exactly l.
      float rs = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < 2; ++c0) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          pk[i] = pack2<BF16>(sv[c0 * 64 + 2 * i], sv[c0 * 64 + 2 * i + 1]);
          const float2 r = unpack2<BF16>(pk[i]);
          rs += r.x + r.y;
        }
        tmem_st32(tS + c0 * 32, pk);
      }
      l = l * alpha + rs;
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(C::B_PFULL + q));
    }
    // ------------------------------------------------------------ epilogue
    if (ok && nk > 0 && mbar_wait(bar(C::B_ODONE + q), (nk - 1) & 1, abort_flag, status)) {
      tc_fence_after_sync();
      const float inv_l = 1.0f / l;
      uint8_t* orow = o_out + (static_cast<int64_t>(bh) * N + row) * (D * 2);
#pragma unroll
      for (int c0 = 0; c0 < D / 32; ++c0) {
        uint32_t ov[32];
        tmem_ld32(tO + c0 * 32, ov);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack2<BF16>(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l);
        if (row < N) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c0 * 64);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if (row < N) lse_out[static_cast<int64_t>(bh) * N + row] = (m + log2f(l)) * 0.69314718055994531f;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool BF16>
int launch_fwd_t(const FwdArgs& a) {
  using C = FwdCfg<D>;
  CUtensorMap mq, mk, mv;
  const int rowb = C::ROWB;
  if (!encode_bhnd_map(&mq, a.q, a.BH, a.N, D, C::CH, 128, rowb, BF16) ||
      !encode_bhnd_map(&mk, a.k, a.BH, a.N, D, C::CH, 128, rowb, BF16) ||
      !encode_bhnd_map(&mv, a.v, a.BH, a.N, D, C::CH, 128, rowb, BF16))
    return kStatusCuda;
  auto kern = attn_fwd_kernel<D, BF16>;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), C::SMEM_BYTES)) return kStatusCuda;
  dim3 grid((a.N + 2 * C::BM - 1) / (2 * C::BM), a.BH);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, a.stream>>>(mq, mk, mv, static_cast<uint8_t*>(a.o), a.lse,
                                                      a.N, a.sl2, a.causal, a.negate, a.status);
  return cudaGetLastError() == cudaSuccess ? kStatusOk : kStatusCuda;
}

}  // namespace

int launch_fwd(const FwdArgs& a) {
  switch (a.d) {
    case 32: return a.bf16 ? launch_fwd_t<32, true>(a) : launch_fwd_t<32, false>(a);
    case 64: return a.bf16 ? launch_fwd_t<64, true>(a) : launch_fwd_t<64, false>(a);
    case 128: return a.bf16 ? launch_fwd_t<128, true>(a) : launch_fwd_t<128, false>(a);
    default: return kStatusUnsupported;
  }
}

}  // namespace attn
