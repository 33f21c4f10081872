// attn_fwd_fp8.cu -- fused exact-attention forward with FP8 (e4m3) operands.
//
// FlashAttention (PKM page), 效果 table and the FA2/FA3 note, and
// FlashAttention深度攻略 (前沿研究方向): FP8 is named as the further gain of the
// Hopper-era kernel.  Here Q, K and V are e4m3 with one descale factor per
// tensor (real value = descale * e4m3 value); the method is the one of
// attn_fwd.cu (tiling, online softmax, final division) and O is bf16.
//
// Differences from the bf16 kernel, all forced by the 8-bit operands:
//   * tcgen05.mma kind::f8f6f4 (E4M3 x E4M3 -> F32), K = 32 per instruction;
//     a d = 128 row is one 128-byte swizzle row.
//   * Both MMAs are SS with K-major operands.  P is rounded to e4m3 and
//     written to shared memory (128-byte swizzled, one 16 KB tile per query
//     tile) instead of TMEM; V is used as V^T, K-major, which a small
//     pre-pass (attn_fp8_transpose_kernel) writes to scratch as
//     [B*H][d][ceil(N/128)*128] with zero padding.
//   * P keeps a fixed headroom: p = exp2(t - m + 7) with the reference max
//     moved when the row max grows by more than 1.5 (log2 units), so
//     p <= 2^8.5 < 448 (the e4m3 maximum) and small weights stay in the
//     normal range longer.
//   * l is kept twice (exact fp32 sum for LSE; sum of the e4m3-rounded P,
//     converted back exactly through f16, to normalise O), and the epilogue
//     multiplies by descale_v.
// Roles, TMEM layout (S0 S1 O0 O1), ping-pong of two query tiles and the
// event-driven MMA issuer are those of the bf16 kernel.  As P lives in shared
// memory, S_q(j+1) goes out as soon as the softmax has read S_q(j) into
// registers; the softmax waits for P_q(j) V_j only before it rescales O_q and
// overwrites the P tile (as the bf16 kernel does at d <= 64).
#include "attn_internal.h"
#include "tc_sm103.cuh"

namespace attn {

namespace {

constexpr float kFp8Shift = 7.0f;           // log2 headroom of P below the e4m3 maximum
constexpr float kFp8RescaleThreshold = 1.5f;

struct Fp8Cfg {
  static constexpr int D = 128;
  static constexpr int BM = 128, BN = 128;
  static constexpr int TILE_BYTES = 128 * 128;  // 128 rows x 128 one-byte elements
  static constexpr int NST = 3;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = 2 * TILE_BYTES;
  static constexpr int OFF_V = OFF_K + NST * TILE_BYTES;
  static constexpr int OFF_P = OFF_V + NST * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_P + 2 * TILE_BYTES;
  static constexpr int B_QFULL = 0;
  static constexpr int B_KFULL = 1;
  static constexpr int B_KEMPTY = B_KFULL + NST;
  static constexpr int B_VFULL = B_KEMPTY + NST;
  static constexpr int B_VEMPTY = B_VFULL + NST;
  static constexpr int B_SFULL = B_VEMPTY + NST;
  static constexpr int B_PFULL = B_SFULL + 2;
  static constexpr int B_ODONE = B_PFULL + 2;
  static constexpr int B_MMADONE = B_ODONE + 2;
  static constexpr int B_STAKEN = B_MMADONE + 1;  // [2]: S_q read into registers
  static constexpr int NBAR = B_STAKEN + 2;
  static constexpr int OFF_TMEMSLOT = OFF_BAR + NBAR * 8;
  static constexpr int OFF_ABORT = OFF_TMEMSLOT + 4;
  static constexpr int SMEM_BYTES = OFF_ABORT + 12;
  static constexpr int THREADS = 384;
  static constexpr int REGS_LAUNCH = 168;
  static constexpr int REGS_MATH = 224;
  static constexpr int REGS_CTRL = 56;
  static_assert(2 * 128 * REGS_MATH + 128 * REGS_CTRL <= THREADS * REGS_LAUNCH, "register split");
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// K-major 8-bit operand tiles: 128 rows x 128 bytes, 128-byte swizzle, 8-row
// groups 1024 bytes apart; a 32-element K slice is 32 bytes along the row.

// kind::f8f6f4 instruction descriptor: D = F32, A = B = E4M3 (format 0),
// both K-major, M = 128, N = 128.
constexpr uint32_t kIdescE4m3 = (1u << 4) | (0u << 7) | (0u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

// The same with the descriptors as words (smem_desc_lo/hi): the K slice kk of
// a tile whose low word is lo starts at lo + 2 kk (32 bytes).
constexpr uint32_t kHi8 = smem_desc_hi(1024, kSwizzle128B);
__device__ __forceinline__ void mma_ss_f8_w(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "mov.b64 da, {%1, %3};\n\tmov.b64 db, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], da, db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(kHi8), "r"(kIdescE4m3), "r"(accumulate)
      : "memory");
}

// Two floats -> two e4m3 bytes (lo in the low byte), round to nearest, saturating.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t p;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(p) : "f"(hi), "f"(lo));
  return p;
}

// acc + both e4m3 values of the low 16 bits of w (exact via f16).
__device__ __forceinline__ float add_e4m3x2(float acc, uint32_t w) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<uint16_t>(w)));
  return add_halves<false>(acc, h2);
}

__device__ __forceinline__ void drain_wait8(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

// v [BH][N][128] e4m3 -> vt [BH][128][Npad] (zero for kv >= N).  One CTA per
// (128-key block, head); 16-byte loads and stores through a shared tile.
__global__ void __launch_bounds__(256) attn_fp8_transpose_kernel(const uint8_t* __restrict__ v,
                                                                  uint8_t* __restrict__ vt, int N,
                                                                  int Npad) {
  griddep_wait();  // launched overlapped (launch_serialized)
  griddep_launch_dependents();
  __shared__ uint8_t tile[128][128 + 16];
  const int kb = blockIdx.x, bh = blockIdx.y;
  const uint8_t* src = v + (static_cast<size_t>(bh) * N + static_cast<size_t>(kb) * 128) * 128;
  for (int i = threadIdx.x; i < 128 * 8; i += blockDim.x) {
    const int r = i >> 3, c = (i & 7) * 16;  // key row r, byte column c
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (kb * 128 + r < N) w = *reinterpret_cast<const uint4*>(src + static_cast<size_t>(r) * 128 + c);
    const uint8_t* b = reinterpret_cast<const uint8_t*>(&w);
#pragma unroll
    for (int e = 0; e < 16; ++e) tile[r][c + e] = b[e];
  }
  __syncthreads();
  uint8_t* dst = vt + static_cast<size_t>(bh) * 128 * Npad + static_cast<size_t>(kb) * 128;
  for (int i = threadIdx.x; i < 128 * 8; i += blockDim.x) {
    const int dcol = i >> 3, c = (i & 7) * 16;  // output row = head-dim index, 16 keys
    uint8_t b[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) b[e] = tile[c + e][dcol];
    *reinterpret_cast<uint4*>(dst + static_cast<size_t>(dcol) * Npad + c) = *reinterpret_cast<uint4*>(b);
  }
}

__global__ void __launch_bounds__(Fp8Cfg::THREADS, 1)
    attn_fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_vt, uint8_t* __restrict__ o_out,
                        float* __restrict__ lse_out, int N, float sl2, float descale_v, int causal,
                        int* status, int head_group, int overlap) {
  using C = Fp8Cfg;
  constexpr int D = C::D;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (overlap) {  // launched overlapped (launch_serialized)
    griddep_wait();
    griddep_launch_dependents();
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  int bh = blockIdx.y, qb = blockIdx.x;
  if (causal) {  // heaviest query blocks (of a group of heads) first
    int rank;
    grouped_rank_order(blockIdx.x + blockIdx.y * gridDim.x, gridDim.x, gridDim.y, head_group, rank, bh);
    qb = gridDim.x - 1 - rank;
  }
  const int nkv_all = (N + C::BN - 1) / C::BN;
  int nkv[2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const int row0 = qb * 2 * C::BM + q * C::BM;
    nkv[q] = (row0 >= N) ? 0 : (causal ? min(nkv_all, row0 / C::BN + 1) : nkv_all);
  }
  const int nkv_max = max(nkv[0], nkv[1]);

  const uint32_t sbase = smem_addr(smem);
  if (sbase & 1023u) {
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
      mbar_init(bar(C::B_KEMPTY + s), 2);  // one unit per query tile (see the softmax)
      mbar_init(bar(C::B_VFULL + s), 1);
      mbar_init(bar(C::B_VEMPTY + s), 2);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(bar(C::B_SFULL + q), 1);
      mbar_init(bar(C::B_PFULL + q), C::BM);
      mbar_init(bar(C::B_ODONE + q), 1);
      mbar_init(bar(C::B_STAKEN + q), C::BM);
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

  const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V,
                 sP = sbase + C::OFF_P;

  if (warp >= 8) {
    regs_decrease<C::REGS_CTRL>();
    if (warp == 8 && lane == 0) {
      // ---------------------------------------------------------- producer
      prefetch_tensormap(&tm_q);
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_vt);
      mbar_arrive_expect_tx(bar(C::B_QFULL), 2 * C::TILE_BYTES);
      for (int q = 0; q < 2; ++q)
        tma_load_3d(sQ + q * C::TILE_BYTES, &tm_q, bar(C::B_QFULL), 0, qb * 2 * C::BM + q * C::BM, bh);
      int issued = 0;
      for (int j = 0; j < nkv_max; ++j) {
        const int s = j % C::NST, u = j / C::NST;
        if (u > 0 && !mbar_wait(bar(C::B_KEMPTY + s), (u - 1) & 1, abort_flag, status)) break;
        mbar_arrive_expect_tx(bar(C::B_KFULL + s), C::TILE_BYTES);
        tma_load_3d(sK + s * C::TILE_BYTES, &tm_k, bar(C::B_KFULL + s), 0, j * C::BN, bh);
        if (u > 0 && !mbar_wait(bar(C::B_VEMPTY + s), (u - 1) & 1, abort_flag, status)) {
          issued = -(j + 1);
          break;
        }
        mbar_arrive_expect_tx(bar(C::B_VFULL + s), C::TILE_BYTES);
        tma_load_3d(sV + s * C::TILE_BYTES, &tm_vt, bar(C::B_VFULL + s), j * C::BN, 0, bh);
        issued = j + 1;
      }
      if (*abort_flag) {
        drain_wait8(bar(C::B_QFULL), 0);
        const int nk = issued >= 0 ? issued : -issued;
        const int nv = issued >= 0 ? issued : -issued - 1;
        for (int s = 0; s < C::NST; ++s) {
          const int ck = nk > s ? (nk - 1 - s) / C::NST + 1 : 0;
          const int cv = nv > s ? (nv - 1 - s) / C::NST + 1 : 0;
          if (ck) drain_wait8(bar(C::B_KFULL + s), (ck - 1) & 1);
          if (cv) drain_wait8(bar(C::B_VFULL + s), (cv - 1) & 1);
        }
      }
    } else if (warp == 9 && lane == 0) {
      // -------------------------------------------------------- MMA issuer
      // One S/PV chain per query tile, issued whenever ready (see attn_fwd.cu):
      //   S_q(j) needs K_j and the softmax done reading S_q(j-1);
      //   PV_q(j) needs V_j^T and P_q(j) written to shared memory.
      // The softmax threads release the K/V stages (see there).
      bool ok = nkv_max == 0 || mbar_wait(bar(C::B_QFULL), 0, abort_flag, status);
      tc_fence_after_sync();
      const uint32_t q_lo0 = smem_desc_lo(sQ, 16), q_lo1 = smem_desc_lo(sQ + C::TILE_BYTES, 16);
      int js[2] = {0, 0}, jp[2] = {0, 0};
      IdleWatch watch;
      while (ok && (jp[0] < nkv[0] || jp[1] < nkv[1])) {
        bool progress = false;
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {  // tile 1 (the longer causal chain) first
          const int q = 1 - qq;
          const int jv = jp[q];
          if (jv < nkv[q] && jv < js[q] &&
              mbar_probe(bar(C::B_VFULL + jv % C::NST), (jv / C::NST) & 1) &&
              mbar_probe(bar(C::B_PFULL + q), jv & 1)) {
            tc_fence_after_sync();
            const uint32_t v_lo = smem_desc_lo(sV + (jv % C::NST) * C::TILE_BYTES, 16);
            const uint32_t p_lo = smem_desc_lo(sP + q * C::TILE_BYTES, 16);
#pragma unroll
            for (int kk = 0; kk < C::BN / 32; ++kk)
              mma_ss_f8_w(tmem + 2 * C::BN + q * D, p_lo + 2 * kk, v_lo + 2 * kk, (jv > 0 || kk > 0) ? 1u : 0u);
            tc_commit(bar(C::B_ODONE + q));
            jp[q] = jv + 1;
            progress = true;
          }
          const int jk = js[q];
          if (jk < nkv[q] &&
              mbar_probe(bar(C::B_KFULL + jk % C::NST), (jk / C::NST) & 1) &&
              (jk == 0 || mbar_probe(bar(C::B_STAKEN + q), (jk - 1) & 1))) {
            tc_fence_after_sync();
            const uint32_t k_lo = smem_desc_lo(sK + (jk % C::NST) * C::TILE_BYTES, 16);
            const uint32_t a_lo = q ? q_lo1 : q_lo0;
#pragma unroll
            for (int kk = 0; kk < D / 32; ++kk)
              mma_ss_f8_w(tmem + q * C::BN, a_lo + 2 * kk, k_lo + 2 * kk, kk > 0 ? 1u : 0u);
            tc_commit(bar(C::B_SFULL + q));
            js[q] = jk + 1;
            progress = true;
          }
        }
        if (progress) {
          watch.progress();
        } else {
          ok = watch.idle(abort_flag, status, kWaitLimitNs);
        }
      }
      tc_commit(bar(C::B_MMADONE));
      drain_wait8(bar(C::B_MMADONE), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    regs_increase<C::REGS_MATH>();
    const int q = warp >> 2;
    const int r = threadIdx.x & 127;
    const int row0 = qb * 2 * C::BM + q * C::BM;
    const int row = row0 + r;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + q * C::BN;
    const uint32_t tO = tmem + lane_off + 2 * C::BN + q * D;
    uint8_t* prow = smem + C::OFF_P + q * C::TILE_BYTES + r * 128;
    float m = -INFINITY;  // row max (log2 units) the weights are taken against, moved lazily
    float l_exact = 0.f, l_round = 0.f;
    bool ok = true;
    const int nk = q ? nkv[1] : nkv[0];
    const int nk_other = q ? nkv[0] : nkv[1];
    const float2 sl2x2 = make_float2(sl2, sl2);
    // K/V stage release (as in attn_fwd.cu): each position's empty barrier
    // takes one unit from each tile that uses it, or two from the only one.
    // K_j is free once S_q(j) is complete (this tile's S wait); V_j once P_q(j)
    // V_j is (the O wait of the next step, or the epilogue's).
    auto release = [&](int first_bar, int p) {
      if (r == 0) mbar_arrive_cnt(bar(first_bar + p % C::NST), p < nk_other ? 1u : 2u);
    };
    for (int j = 0; j < nk; ++j) {
      // warp-uniform, as the step votes across the warp (rescale) further on:
      // a lane that left alone would leave the others waiting at the vote
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SFULL + q), j & 1, abort_flag, status)))) break;
      tc_fence_after_sync();
      release(C::B_KEMPTY, j);
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
      tc_fence_before_sync();
      mbar_arrive(bar(C::B_STAKEN + q));  // S_q may be overwritten by the next S now
      const int kv0 = j * C::BN;
      const bool masked = (kv0 + C::BN > N) || (causal && kv0 + C::BN - 1 > row0);
      int lim = C::BN;
      if (masked) {
        lim = min(N - kv0, C::BN);
        if (causal) lim = min(lim, row - kv0 + 1);
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= lim) sv[c] = -INFINITY;
      }
      float mx;
      {
        float a0 = sv[0], a1 = sv[1], a2 = sv[2], a3 = sv[3];
#pragma unroll
        for (int c = 4; c < 128; c += 8) {
          a0 = max3f(a0, sv[c], sv[c + 1]);
          a1 = max3f(a1, sv[c + 2], sv[c + 3]);
          a2 = max3f(a2, sv[c + 4], sv[c + 5]);
          a3 = max3f(a3, sv[c + 6], sv[c + 7]);
        }
        mx = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
      }
      const float m_new = fmaxf(m, mx * sl2);
      float alpha = 1.f;
      if (m_new > m + kFp8RescaleThreshold) {
        alpha = ex2_approx(m - m_new);
        m = m_new;
      }
      // p = exp2(t - m + shift): at most 2^(shift + threshold) = 2^8.5 < 448
      const float neg_ref = (m == -INFINITY) ? 0.f : kFp8Shift - m;
      const float2 nr2 = make_float2(neg_ref, neg_ref);
#pragma unroll
      for (int c = 0; c < 128; c += 2) {
        const float2 t = fma2(make_float2(sv[c], sv[c + 1]), sl2x2, nr2);
        sv[c] = ex2_approx(t.x);
        sv[c + 1] = ex2_approx(t.y);
      }
      if (masked) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= lim) sv[c] = 0.f;
      }
      // P_q(j-1) V_{j-1} may still be running: it must finish before O_q is
      // rescaled and before the P tile is overwritten.
      if (j > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_ODONE + q), (j - 1) & 1, abort_flag, status));
        if (!ok) break;
        tc_fence_after_sync();
        release(C::B_VEMPTY, j - 1);
      }
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
      // P -> e4m3, 16 keys per 16-byte unit, 128-byte-swizzled row of the P
      // tile; the row sums follow the hand-off and overlap the P V product.
      uint32_t pw[32];
#pragma unroll
      for (int uu = 0; uu < 8; ++uu) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = uu * 16 + i * 4;
          pw[4 * uu + i] = e4m3x2(sv[c], sv[c + 1]) | (e4m3x2(sv[c + 2], sv[c + 3]) << 16);
        }
        *reinterpret_cast<uint4*>(prow + ((uu ^ (r & 7)) * 16)) =
            make_uint4(pw[4 * uu], pw[4 * uu + 1], pw[4 * uu + 2], pw[4 * uu + 3]);
      }
      tmem_st_wait();
      fence_proxy_async_smem();  // P (generic-proxy writes) before the MMA reads it
      tc_fence_before_sync();
      mbar_arrive(bar(C::B_PFULL + q));
      float2 se0 = make_float2(0.f, 0.f), se1 = se0;
      float sr0 = 0.f, sr1 = 0.f, sr2 = 0.f, sr3 = 0.f;
#pragma unroll
      for (int c = 0; c < 128; c += 4) {
        se0 = add2(se0, make_float2(sv[c], sv[c + 1]));
        se1 = add2(se1, make_float2(sv[c + 2], sv[c + 3]));
      }
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        sr0 = add_e4m3x2(sr0, pw[i] & 0xffffu);
        sr1 = add_e4m3x2(sr1, pw[i] >> 16);
        sr2 = add_e4m3x2(sr2, pw[i + 1] & 0xffffu);
        sr3 = add_e4m3x2(sr3, pw[i + 1] >> 16);
      }
      l_exact = l_exact * alpha + ((se0.x + se0.y) + (se1.x + se1.y));
      l_round = l_round * alpha + ((sr0 + sr1) + (sr2 + sr3));
    }
    if (ok && nk > 0 && mbar_wait(bar(C::B_ODONE + q), (nk - 1) & 1, abort_flag, status)) {
      tc_fence_after_sync();
      release(C::B_VEMPTY, nk - 1);
      const float mul = descale_v / l_round;
      uint8_t* orow = o_out + (static_cast<int64_t>(bh) * N + row) * (D * 2);
#pragma unroll
      for (int c0 = 0; c0 < D / 32; ++c0) {
        uint32_t ov[32];
        tmem_ld32(tO + c0 * 32, ov);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack2<true>(__uint_as_float(ov[2 * i]) * mul, __uint_as_float(ov[2 * i + 1]) * mul);
        if (row < N) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c0 * 64);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      // LSE = ln sum_j exp(scaled logit): the weights were exp2(t - (m - shift))
      if (row < N)
        lse_out[static_cast<int64_t>(bh) * N + row] = (m - kFp8Shift + log2f(l_exact)) * 0.69314718055994531f;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace

int launch_fwd_fp8(const Fp8Args& a) {
  using C = Fp8Cfg;
  if (a.d != 128) return kStatusUnsupported;
  const int Npad = ((a.N + 127) / 128) * 128;
  // both launches overlap their predecessor's tail on grids of at most 8 waves
  dim3 grid((a.N + 2 * C::BM - 1) / (2 * C::BM), a.BH);
  const bool overlap = overlap_launches(static_cast<int64_t>(grid.x) * grid.y, 1);
  if (launch_serialized(overlap, attn_fp8_transpose_kernel, dim3(Npad / 128, a.BH), dim3(256), 0, a.stream,
                        static_cast<const uint8_t*>(a.v), a.ws_vt, a.N, Npad) != cudaSuccess)
    return kStatusCuda;
  CUtensorMap mq, mk, mvt;
  if (!encode_map_u8(&mq, a.q, 128, a.N, a.BH, 128, static_cast<uint64_t>(a.N) * 128, 128, 128) ||
      !encode_map_u8(&mk, a.k, 128, a.N, a.BH, 128, static_cast<uint64_t>(a.N) * 128, 128, 128) ||
      !encode_map_u8(&mvt, a.ws_vt, Npad, 128, a.BH, Npad, static_cast<uint64_t>(Npad) * 128, 128, 128))
    return kStatusCuda;
  auto kern = attn_fwd_fp8_kernel;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), C::SMEM_BYTES)) return kStatusCuda;
  if (!check_launch_regs(reinterpret_cast<const void*>(kern), C::REGS_LAUNCH)) return kStatusDeviceCheck;
  return launch_serialized(overlap, kern, grid, dim3(C::THREADS), C::SMEM_BYTES, a.stream, mq, mk, mvt,
                           static_cast<uint8_t*>(a.o), a.lse, a.N, a.sl2, a.descale_v, a.causal, a.status,
                           order_head_group(a.BH, int64_t{2} * a.N * C::D, int64_t{128} << 20),
                           overlap ? 1 : 0) == cudaSuccess
             ? kStatusOk
             : kStatusCuda;
}

}  // namespace attn
