// attn_bwd.cu -- recomputation backward of exact attention for sm_103a.
//
// Method (FlashAttention (PKM page), "三招" 3 Recomputation; FlashAttention深度攻略
// §6): the forward keeps only O and one statistic per row (here LSE); the
// backward rebuilds P = exp(scale Q K^T - LSE) tile by tile on chip and forms
//   dV = P^T dO,  dP = dO V^T,  D_i = sum_k dO_ik O_ik,  dS = P o (dP - D),
//   dK = scale dS^T Q,  dQ = scale dS K.
//
// Three launches on the caller's stream:
//   1. attn_bwd_pre_kernel   : -D_i (fp32) and -LSE * log2(e) into padded row
//                              vectors (-inf on padding rows, so their P is 0),
//                              and zeroes the fp32 dQ accumulator.
//   2. attn_bwd_kernel       : one CTA per (128-key tile, head), the key tile
//                              stays in shared memory and dK/dV accumulate in
//                              TMEM over every query tile that can see it
//                              (without the causal mask, a last partial wave of
//                              at most half the SMs runs each of its tiles as
//                              two CTAs over half of the query tiles, writing
//                              fp32 partial dK/dV).
//   3. attn_dq_convert_kernel: fp32 dQ accumulator -> bf16/fp16 dQ, and the
//                              split tiles' dK/dV = sum of their two partials.
//
// attn_bwd_kernel roles (16 warps = 4 warpgroups, one CTA per SM; warpgroup 3
// hands registers to warpgroups 0-2 with setmaxnreg: 152, 152, 144 / 64):
//   * warp 12    : TMA producer: K_j and V_j once; Q_i, dO_i (2-stage ring)
//                  plus the 128 -LSE*log2e and -D values of tile i (bulk copies);
//                  its thread also sets up the barriers and issues K, V and the
//                  first stages before the CTA's set-up barrier.
//   * warp 13    : TMEM owner and single-thread tcgen05.mma issuer, per tile i:
//                    S^T  = K_j Q_i^T          (SS, both K-major)
//                    dP^T = V_j dO_i^T         (SS, both K-major)
//                    dV  += P^T dO_i           (TS, P^T from TMEM, dO MN-major)
//                    dK  += dS^T Q_i           (SS, dS^T K-major, Q MN-major)
//                    dQ_i = dS K_j             (SS, dS MN-major view of the same
//                                               shared tile, K MN-major; at d = 128
//                                               as dQ_i^T = K_j^T dS^T, operands swapped)
//   * warps 0-7  : two threads per key row (warpgroup g takes query columns
//                  64g..64g+63): P^T from S^T and LSE (exp2), P^T to TMEM,
//                  dS^T = P^T o (dP^T - D) to shared memory (bf16/fp16,
//                  128B-swizzled); at the end warpgroup 0 stores dK (x scale)
//                  and warpgroup 1 stores dV.
//   * warps 8-11 : dQ_i from TMEM (released as soon as it is in registers),
//                  x scale, added into the fp32 accumulator with reductions.
//                  At d = 128 the MMA produces dQ_i^T = K_j^T dS^T instead, so a
//                  thread holds one head-dim column and each warp-wide reduction
//                  is 128 contiguous bytes of a dQ row (8x fewer L2 requests
//                  than row-per-thread 16-byte vector reductions); at d <= 64
//                  (dQ_i = dS K_j, a thread per query row) groups of 8 lanes
//                  transpose their 16-byte pieces so that each 16-byte vector
//                  reduction instruction covers 4 whole 128-byte row segments.
//   * warps 14-15: idle (they complete warpgroup 3 for the register split).
//   * TMEM (512 columns): S^T/P^T [0,128) dP^T/dQ [128,256) dK [256,256+D)
//                         dV [256+D,256+2D).
// Causal: key tile j only visits query tiles i >= j; the diagonal tile is
// masked elementwise (P^T[key][query] = 0 when key > query), and the CTAs run
// heaviest first across a group of heads (block_order.h).
// Dropout (DROP): the keep bytes of the forward are drawn again (dropout.cuh),
// one visit ahead while the warps wait for the next S^T: each half warp draws
// 16 query rows for its 16 keys and transposes them so a thread holds its
// key's bytes; dropped P^T entries are cleared before the dV product (dV
// scaled by 256 / t at the end) and dP^T is weighted by keep * 256 / t in
// dS^T = P^T o (w dP^T - D).  Block-sparse (SPARSE): see attn_bwd_kernel.
#include "attn_internal.h"
#include "dropout.cuh"
#include "tc_sm103.cuh"

namespace attn {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int BM = 128;  // query rows per tile
  static constexpr int BN = 128;  // key rows per CTA
  static constexpr int ROWB = (D >= 64) ? 128 : 64;
  static constexpr int CH = ROWB / 2;
  static constexpr int NCH = D / CH;
  static constexpr uint32_t SWZ = (ROWB == 128) ? kSwizzle128B : kSwizzle64B;
  static constexpr int SBO = 8 * ROWB;
  static constexpr int CHUNK_BYTES = 128 * ROWB;
  static constexpr int TILE_BYTES = 128 * D * 2;
  static constexpr int DS_CHUNK = 128 * 128;       // 64 query columns x 128 key rows, bf16
  static constexpr int DS_BYTES = 2 * DS_CHUNK;
  static constexpr int NSTQ = 2;
  static constexpr int VEC_BYTES = BM * 4;         // 128 fp32 per query tile
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = TILE_BYTES;
  static constexpr int OFF_Q = 2 * TILE_BYTES;
  static constexpr int OFF_DO = OFF_Q + NSTQ * TILE_BYTES;
  static constexpr int OFF_DS = OFF_DO + NSTQ * TILE_BYTES;
  static constexpr int OFF_LSE = OFF_DS + DS_BYTES;
  static constexpr int OFF_DD = OFF_LSE + NSTQ * VEC_BYTES;
  static constexpr int OFF_BAR = OFF_DD + NSTQ * VEC_BYTES;
  static constexpr int B_KVFULL = 0;
  static constexpr int B_QFULL = 1;
  static constexpr int B_QEMPTY = B_QFULL + NSTQ;
  static constexpr int B_SFULL = B_QEMPTY + NSTQ;
  static constexpr int B_DPFULL = B_SFULL + 1;
  static constexpr int B_PFULL = B_DPFULL + 1;
  static constexpr int B_DSFULL = B_PFULL + 1;
  static constexpr int B_DQFULL = B_DSFULL + 1;
  static constexpr int B_DQEMPTY = B_DQFULL + 1;
  static constexpr int B_MMADONE = B_DQEMPTY + 1;
  static constexpr int NBAR = B_MMADONE + 1;
  static constexpr int OFF_TMEMSLOT = OFF_BAR + NBAR * 8;
  static constexpr int OFF_ABORT = OFF_TMEMSLOT + 4;
  // block-sparse: bit i of word i / 32 set iff query tile i is visited; then the count
  static constexpr int OFF_QBITS = OFF_ABORT + 12;
  static constexpr int OFF_QCOUNT = OFF_QBITS + kMaxSparseTiles / 8;
  static constexpr int SMEM_BYTES = OFF_QCOUNT + 4;
  static constexpr int THREADS = 512;
  static constexpr int REGS_LAUNCH = 128;
  static constexpr int REGS_MATH = 152;  // the two P / dS warpgroups
  // The dQ warpgroup paces the loop: 136 / 72 (no spills left in the
  // single-thread issuer) measured 3-4 % slower than 144 / 64.
  static constexpr int REGS_DQ = 144;    // the dQ warpgroup
  static constexpr int REGS_CTRL = 64;   // producer / MMA warpgroup
  static_assert(128 * (2 * REGS_MATH + REGS_DQ + REGS_CTRL) <= THREADS * REGS_LAUNCH, "register split");
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t T_S = 0, T_DP = 128, T_DK = 256, T_DV = 256 + D;
  // d = 128: the MMA produces dQ^T = K^T dS^T (TMEM lane = head-dim index), so
  // each warp's reduction into the accumulator covers 128 contiguous bytes of
  // one dQ row.  Smaller d keeps dQ = dS K (lane = query row): an M = d < 128
  // accumulator would use a different TMEM layout.
  static constexpr bool DQ_T = (D == 128);
  static_assert(256 + 2 * D <= 512, "TMEM budget");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// Shared-memory descriptors as words (smem_desc_lo/hi): the issuer forms a
// tile's low word once per MMA group and adds these offsets for the 16-deep K
// slice kk.
// K-major operand: a 128-row tile with head-dim rows (column chunks of one
// swizzle width, CHUNK_BYTES apart).
template <int D>
__host__ __device__ constexpr uint32_t k_tile_step(int kk) {
  using C = BwdCfg<D>;
  return static_cast<uint32_t>(((kk * 16) / C::CH * C::CHUNK_BYTES + (kk * 16) % C::CH * 2) >> 4);
}
// MN-major operand: head dim contiguous, 16 rows per slice.
template <int D>
__host__ __device__ constexpr uint32_t mn_tile_step(int kk) {
  return static_cast<uint32_t>((kk * 16 * BwdCfg<D>::ROWB) >> 4);
}
// The dS^T tile: 128 key rows x 128 query columns, 128B-swizzled in two
// 64-column chunks.  As dS^T (M = key, K = query) it is K-major ...
__host__ __device__ constexpr uint32_t ds_k_step(int kk) {
  return static_cast<uint32_t>(((kk * 16) / 64 * (128 * 128) + (kk * 16) % 64 * 2) >> 4);
}
// ... and as dS (M = query, K = key) it is MN-major (LBO 128 * 128).
__host__ __device__ constexpr uint32_t ds_mn_step(int kk) { return static_cast<uint32_t>((kk * 16 * 128) >> 4); }

// Byte offset of 16-byte unit u of row `row` in the epilogue's staging copy of
// a 128-row dK or dV tile (rows of 2 D = 256 bytes): the unit index is XOR-ed
// with the row's low bits, so the row-per-thread writes and the row-contiguous
// reads of a warp each touch eight bank groups per 8-lane phase.
__device__ __forceinline__ uint32_t row_stage_off256(int row, int u) {
  return static_cast<uint32_t>(row * 256 + ((u ^ (row & 7)) << 4));
}

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

// ------------------------------------------------------------ preprocess
template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_bwd_pre_kernel(
    const uint8_t* __restrict__ o, const uint8_t* __restrict__ dO, const float* __restrict__ lse,
    float* __restrict__ lse2, float* __restrict__ dvec, float* __restrict__ dq_acc, int N, int Npad,
    int64_t rows_total) {
  griddep_wait();  // (launch_serialized)
  griddep_launch_dependents();
  // lse2 receives -LSE * log2(e) and dvec receives -D, the forms the main pass adds.
  constexpr int PER = D / 8;  // elements per lane (8 lanes per row)
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t rid = gid >> 3;
  const int sub = threadIdx.x & 7;
  const bool live = rid < rows_total;
  const int64_t bh = live ? rid / Npad : 0;
  const int i = live ? static_cast<int>(rid % Npad) : 0;
  const bool real = live && i < N;
  float acc = 0.f;
  if (real && D >= 64) {
    // The row's 8 lanes take 16-byte pieces sub, sub + 8, ... so that each warp
    // instruction reads (and zeroes) whole 128-byte runs of 4 rows.
    const int64_t row_el = (bh * N + i) * D;
    const uint4* po = reinterpret_cast<const uint4*>(o + row_el * 2);
    const uint4* pd = reinterpret_cast<const uint4*>(dO + row_el * 2);
#pragma unroll
    for (int k = 0; k < D / 64; ++k) {
      const uint4 a = po[sub + 8 * k], b = pd[sub + 8 * k];
      const uint32_t aw[4] = {a.x, a.y, a.z, a.w}, bw[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = unpack2<BF16>(aw[e]), y = unpack2<BF16>(bw[e]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    }
    float4* z = reinterpret_cast<float4*>(dq_acc + row_el);
#pragma unroll
    for (int k = 0; k < D / 32; ++k) z[sub + 8 * k] = make_float4(0.f, 0.f, 0.f, 0.f);
  } else if (real) {
    const int64_t off = (bh * N + i) * D + sub * PER;
    const uint32_t* po = reinterpret_cast<const uint32_t*>(o + off * 2);
    const uint32_t* pd = reinterpret_cast<const uint32_t*>(dO + off * 2);
#pragma unroll
    for (int e = 0; e < PER / 2; ++e) {
      const float2 a = unpack2<BF16>(po[e]);
      const float2 b = unpack2<BF16>(pd[e]);
      acc = fmaf(a.x, b.x, acc);
      acc = fmaf(a.y, b.y, acc);
    }
    float4* z = reinterpret_cast<float4*>(dq_acc + off);
#pragma unroll
    for (int e = 0; e < PER / 4; ++e) z[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  acc += __shfl_xor_sync(0xffffffffu, acc, 4);
  acc += __shfl_xor_sync(0xffffffffu, acc, 2);
  acc += __shfl_xor_sync(0xffffffffu, acc, 1);
  if (live && sub == 0) {
    dvec[rid] = real ? -acc : 0.f;
    // a row that saw no key (LSE = -inf, possible only under a block mask) and
    // padding rows get -inf here, so their P = exp2(s + lse2) is 0
    const float l = real ? lse[bh * N + i] : -INFINITY;
    lse2[rid] = l == -INFINITY ? -INFINITY : -l * kLog2e;
  }
}

// ---------------------------------------------------------------- convert
// fp32 dQ accumulator -> dQ; then, for the key tiles whose query range was
// split over two CTAs (the grid's last partial wave, see launch_bwd_t), dK and
// dV = the sum of the two CTAs' fp32 partial tiles.  part holds, per split
// tile s, half h and output (0 = dK, 1 = dV), a 128 x D fp32 tile:
// part[((s * 2 + h) * 2 + out) * 128 * D + row * D + col].
template <int D, bool BF16>
__global__ void __launch_bounds__(256) attn_dq_convert_kernel(const float* __restrict__ acc,
                                                              uint8_t* __restrict__ dq,
                                                              int64_t groups,
                                                              const float* __restrict__ part, int nsplit,
                                                              int split_from, int nkt, int N,
                                                              uint8_t* __restrict__ dk,
                                                              uint8_t* __restrict__ dv) {
  griddep_wait();  // (launch_serialized)
  griddep_launch_dependents();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (int64_t g = tid; g < groups; g += stride) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * g];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * g + 1];
    reinterpret_cast<uint4*>(dq)[g] = make_uint4(pack2<BF16>(a.x, a.y), pack2<BF16>(a.z, a.w),
                                                 pack2<BF16>(b.x, b.y), pack2<BF16>(b.z, b.w));
  }
  // combine: 8 consecutive columns of one row of one output per step
  constexpr int G = D / 8;  // 8-column groups per row
  const int64_t cgroups = static_cast<int64_t>(nsplit) * 2 * 128 * G;
  for (int64_t g = tid; g < cgroups; g += stride) {
    const int c8 = static_cast<int>(g % G);
    const int row = static_cast<int>((g / G) % 128);
    const int out = static_cast<int>((g / (G * 128)) % 2);
    const int sidx = static_cast<int>(g / (G * 128 * 2));
    const int item = split_from + sidx;  // the split tile's block index before splitting
    const int jt = item % nkt, bh = item / nkt;
    const int kv_row = jt * 128 + row;
    if (kv_row >= N) continue;
    const float* p0 = part + ((static_cast<int64_t>(sidx) * 2 + 0) * 2 + out) * 128 * D + row * D + c8 * 8;
    const float* p1 = part + ((static_cast<int64_t>(sidx) * 2 + 1) * 2 + out) * 128 * D + row * D + c8 * 8;
    const float4 a0 = reinterpret_cast<const float4*>(p0)[0], a1 = reinterpret_cast<const float4*>(p0)[1];
    const float4 b0 = reinterpret_cast<const float4*>(p1)[0], b1 = reinterpret_cast<const float4*>(p1)[1];
    uint8_t* dst = (out == 0 ? dk : dv) + ((static_cast<int64_t>(bh) * N + kv_row) * D + c8 * 8) * 2;
    *reinterpret_cast<uint4*>(dst) = make_uint4(pack2<BF16>(a0.x + b0.x, a0.y + b0.y), pack2<BF16>(a0.z + b0.z, a0.w + b0.w),
                                                pack2<BF16>(a1.x + b1.x, a1.y + b1.y), pack2<BF16>(a1.z + b1.z, a1.w + b1.w));
  }
}

// First set bit at or after `from` among n bits, or n.
__device__ __forceinline__ int next_set_bit(const uint32_t* bits, int from, int n) {
  for (int w = from >> 5; w * 32 < n; ++w) {
    uint32_t m = bits[w];
    if (w == (from >> 5)) m &= 0xffffffffu << (from & 31);
    if (m) return min(w * 32 + __ffs(m) - 1, n);
  }
  return n;
}

// -------------------------------------------------------------- main pass
// SPARSE: the CTA of key tile jt visits only the query tiles i whose block-mask
// entry mask[i][jt] is set (and i >= jt if causal), in increasing order; the
// producer, the P/dS warpgroups and the dQ warpgroup each walk the same list
// (a bitmask in shared memory).  A key tile no query tile sees writes dK = dV = 0.
template <int D, bool BF16, bool DROP, bool SPARSE>
__global__ void __launch_bounds__(BwdCfg<D>::THREADS, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do, const float* __restrict__ lse2,
                    const float* __restrict__ dvec, float* __restrict__ dq_acc,
                    uint8_t* __restrict__ dk_out, uint8_t* __restrict__ dv_out, int N, int Npad,
                    float sl2, float scale, int causal, int negate, int* status,
                    DropParams drop, const uint8_t* __restrict__ bmask, int H, int mask_heads,
                    int head_group, int BH, int split_from, float* __restrict__ part) {
  // (always launched normally: any overlap code here measured 0.3-1.6 % slower
  // at N = 8192, this kernel being sensitive to its code layout)
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nkt = (N + C::BN - 1) / C::BN;
  const int ntq = (N + C::BM - 1) / C::BM;
  // One-dimensional grid over (key tile, head) items.  Blocks from split_from
  // on come in pairs: the two halves of one item's query range (the grid's
  // last partial wave, split so that it takes half a wave; dK and dV then go
  // out as fp32 partial tiles that attn_dq_convert_kernel adds).
  int item, half, sidx;  // sidx: index of a split item's partial tiles
  split_block_item(static_cast<int>(blockIdx.x), split_from, item, half, sidx);
  int jt, bh;  // key tile, head
  if (causal) {  // key tile 0 sees every query tile: heaviest (of a group of heads) first
    grouped_rank_order(item, nkt, BH, head_group, jt, bh);
  } else {
    bh = item / nkt;
    jt = item - bh * nkt;
  }
  const int kv0 = jt * C::BN;
  // query tiles [i0, i0 + nq_dense): from the diagonal under the causal mask,
  // else all of them, or one half of them for a split item
  int i0 = causal ? jt : 0;
  int nq_dense = ntq - i0;
  if (half >= 0) {
    i0 = half == 0 ? 0 : ntq / 2;
    nq_dense = half == 0 ? ntq / 2 : ntq - ntq / 2;
  }

  const uint32_t sbase = smem_addr(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicExch(status, kStatusDeviceCheck);
    return;
  }
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto bar = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEMSLOT);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_ABORT);

  uint32_t* qbits = reinterpret_cast<uint32_t*>(smem + C::OFF_QBITS);
  int* qcount = reinterpret_cast<int*>(smem + C::OFF_QCOUNT);
  const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
  const uint32_t sQ = sbase + C::OFF_Q, sDO = sbase + C::OFF_DO, sDS = sbase + C::OFF_DS;
  // The producer thread sets up the barriers and issues K, V and the first
  // Q/dO stages before the CTA-wide set-up barrier, so that their load
  // latency overlaps the TMEM allocation and the barrier itself.
  int pre_issued = 0;   // visits whose stage loads went out before the barrier
  int pre_qi = i0 - 1;  // (block-sparse) query-tile cursor after them
  auto load_stage = [&](int s, int q0) {
    mbar_arrive_expect_tx(bar(C::B_QFULL + s), 2 * C::TILE_BYTES + 2 * C::VEC_BYTES);
    for (int c = 0; c < C::NCH; ++c) {
      tma_load_3d(sQ + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_q, bar(C::B_QFULL + s), c * C::CH, q0, bh);
      tma_load_3d(sDO + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_do, bar(C::B_QFULL + s), c * C::CH, q0, bh);
    }
    const int64_t voff = static_cast<int64_t>(bh) * Npad + q0;
    bulk_load(sbase + C::OFF_LSE + s * C::VEC_BYTES, lse2 + voff, C::VEC_BYTES, bar(C::B_QFULL + s));
    bulk_load(sbase + C::OFF_DD + s * C::VEC_BYTES, dvec + voff, C::VEC_BYTES, bar(C::B_QFULL + s));
  };
  if (warp == 12 && lane == 0) {
    if constexpr (SPARSE) {
      const uint8_t* mb = bmask + static_cast<size_t>((bh % H) % mask_heads) * ntq * ntq;
      int n = 0;
      for (int w = 0; w < kMaxSparseTiles / 32; ++w) qbits[w] = 0u;
      for (int i = i0; i < ntq; ++i)
        if (mb[static_cast<size_t>(i) * ntq + jt]) {
          qbits[i >> 5] |= 1u << (i & 31);
          ++n;
        }
      *qcount = n;
    }
    mbar_init(bar(C::B_KVFULL), 1);
    for (int s = 0; s < C::NSTQ; ++s) {
      mbar_init(bar(C::B_QFULL + s), 1);
      mbar_init(bar(C::B_QEMPTY + s), 1);
    }
    mbar_init(bar(C::B_SFULL), 1);
    mbar_init(bar(C::B_DPFULL), 1);
    mbar_init(bar(C::B_PFULL), 256);
    mbar_init(bar(C::B_DSFULL), 256);
    mbar_init(bar(C::B_DQFULL), 1);
    mbar_init(bar(C::B_DQEMPTY), 128);
    mbar_init(bar(C::B_MMADONE), 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_do);
    mbar_arrive_expect_tx(bar(C::B_KVFULL), 2 * C::TILE_BYTES);
    for (int c = 0; c < C::NCH; ++c) {
      tma_load_3d(sK + c * C::CHUNK_BYTES, &tm_k, bar(C::B_KVFULL), c * C::CH, kv0, bh);
      tma_load_3d(sV + c * C::CHUNK_BYTES, &tm_v, bar(C::B_KVFULL), c * C::CH, kv0, bh);
    }
    pre_issued = min(SPARSE ? *qcount : nq_dense, C::NSTQ);
    for (int it = 0; it < pre_issued; ++it) {  // stages still empty: no waits
      const int qt = SPARSE ? (pre_qi = next_set_bit(qbits, pre_qi + 1, ntq)) : i0 + it;
      load_stage(it, qt * C::BM);
    }
  }
  if (warp == 13) {
    tmem_alloc(smem_addr(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const int nq = SPARSE ? *qcount : nq_dense;  // query tiles this key tile visits
  // Query tile of visit `it`: i0 + it, or (SPARSE) the next set bit after the
  // cursor `qi` of the previous visit (start qi = i0 - 1).  The dense form is
  // kept as a plain expression: the cursor form measured 4 % slower there.
#define ATTN_BWD_QTILE(it, qi) (SPARSE ? ((qi) = next_set_bit(qbits, (qi) + 1, ntq)) : i0 + (it))


  if (warp >= 12) {
    regs_decrease<C::REGS_CTRL>();
    if (warp == 12 && lane == 0) {
      // ---------------------------------------------------------- producer
      // (K, V and the first min(NSTQ, nq) stages went out before the set-up
      // barrier, see above.)
      int issued = pre_issued;
      int qi = pre_qi;
      for (int it = pre_issued; it < nq; ++it) {
        const int s = it % C::NSTQ, u = it / C::NSTQ;
        const int q0 = ATTN_BWD_QTILE(it, qi) * C::BM;
        if (u > 0 && !mbar_wait(bar(C::B_QEMPTY + s), (u - 1) & 1, abort_flag, status)) break;
        load_stage(s, q0);
        issued = it + 1;
      }
      if (*abort_flag) {
        drain_wait(bar(C::B_KVFULL), 0);
        for (int s = 0; s < C::NSTQ; ++s) {
          const int cnt = issued > s ? (issued - 1 - s) / C::NSTQ + 1 : 0;
          if (cnt) drain_wait(bar(C::B_QFULL + s), (cnt - 1) & 1);
        }
      }
    } else if (warp == 13 && lane == 0) {
      // -------------------------------------------------------- MMA issuer
      // Four chains over the query tiles i, each group issued as soon as ready
      // (checked in pipeline order: S, dP, dV, then dK/dQ, which measured 0.5-3 %
      // faster than the reverse order):
      //   S(i)  = K Q_i^T   needs Q_i resident and dV(i-1) issued (P^T aliases S^T;
      //                     see below)
      //   dP(i) = V dO_i^T  needs dO_i resident and dQ(i-1) read out (dQ aliases dP^T)
      //   dV(i)             needs P^T(i) in TMEM
      //   dK(i), dQ(i)      need dS^T(i) in shared memory (and dV(i) issued)
      // S(i) overwrites the P^T(i-1) that dV(i-1) reads from TMEM.  It is issued
      // right after dV(i-1), without waiting for dV(i-1) to complete: the tensor
      // pipe executes one thread's MMAs in issue order, so dV(i-1) has read its
      // A operand before S(i) writes.  (The PTX ISA promises this order only
      // for MMAs into the same accumulator; on GB300 the in-order form gave
      // bit-identical dK and dV in every repeated run of every configuration
      // tried, and saves the issuer a commit and the S chain a completion
      // round trip per visit.)
      const uint32_t id_st = instr_desc_f16(128, 128, BF16, false, false, negate != 0);
      const uint32_t id_dpt = instr_desc_f16(128, 128, BF16, false, false);
      const uint32_t id_dv = instr_desc_f16(128, D, BF16, false, true);
      const uint32_t id_dk = instr_desc_f16(128, D, BF16, false, true);
      const uint32_t id_dq = instr_desc_f16(128, C::DQ_T ? 128 : D, BF16, true, true);
      constexpr uint32_t HT = smem_desc_hi(C::SBO, C::SWZ);         // Q, K, V, dO tiles
      constexpr uint32_t HDS = smem_desc_hi(1024, kSwizzle128B);    // the dS^T tile
      const uint32_t k_klo = smem_desc_lo(sK, 16), v_klo = smem_desc_lo(sV, 16);
      const uint32_t k_mnlo = smem_desc_lo(sK, C::CHUNK_BYTES);
      const uint32_t ds_klo = smem_desc_lo(sDS, 16), ds_mnlo = smem_desc_lo(sDS, 128 * 128);
      bool ok = mbar_wait(bar(C::B_KVFULL), 0, abort_flag, status);
      tc_fence_after_sync();
      int is = 0, ip = 0, iv = 0, ik = 0;
      IdleWatch watch;
      while (ok && ik < nq) {
        bool progress = false;
        // (the barrier that usually decides is probed first: Q_i, dO_i have long landed)
        if (is < nq && is == iv &&
            mbar_probe(bar(C::B_QFULL + is % C::NSTQ), (is / C::NSTQ) & 1)) {
          tc_fence_after_sync();
          const uint32_t q_lo = smem_desc_lo(sQ + (is % C::NSTQ) * C::TILE_BYTES, 16);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss_w(tmem + C::T_S, k_klo + k_tile_step<D>(kk), HT, q_lo + k_tile_step<D>(kk), HT, id_st,
                     kk > 0 ? 1u : 0u);
          tc_commit(bar(C::B_SFULL));
          ++is;
          progress = true;
        }
        if (ip < nq && ip == ik && (ip == 0 || mbar_probe(bar(C::B_DQEMPTY), (ip - 1) & 1)) &&
            mbar_probe(bar(C::B_QFULL + ip % C::NSTQ), (ip / C::NSTQ) & 1)) {
          tc_fence_after_sync();
          const uint32_t do_lo = smem_desc_lo(sDO + (ip % C::NSTQ) * C::TILE_BYTES, 16);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_ss_w(tmem + C::T_DP, v_klo + k_tile_step<D>(kk), HT, do_lo + k_tile_step<D>(kk), HT, id_dpt,
                     kk > 0 ? 1u : 0u);
          tc_commit(bar(C::B_DPFULL));
          ++ip;
          progress = true;
        }
        if (iv < is && mbar_probe(bar(C::B_PFULL), iv & 1)) {
          tc_fence_after_sync();
          const uint32_t do_lo = smem_desc_lo(sDO + (iv % C::NSTQ) * C::TILE_BYTES, C::CHUNK_BYTES);
#pragma unroll
          for (int kk = 0; kk < C::BM / 16; ++kk)
            mma_ts_w(tmem + C::T_DV, tmem + C::T_S + (kk >> 2) * 64 + (kk & 3) * 8,
                     do_lo + mn_tile_step<D>(kk), HT, id_dv, (iv > 0 || kk > 0) ? 1u : 0u);
          ++iv;
          progress = true;
        }
        if (ik < iv && ik < ip && mbar_probe(bar(C::B_DSFULL), ik & 1)) {
          tc_fence_after_sync();
          const uint32_t q_mnlo = smem_desc_lo(sQ + (ik % C::NSTQ) * C::TILE_BYTES, C::CHUNK_BYTES);
#pragma unroll
          for (int kk = 0; kk < C::BM / 16; ++kk)
            mma_ss_w(tmem + C::T_DK, ds_klo + ds_k_step(kk), HDS, q_mnlo + mn_tile_step<D>(kk), HT, id_dk,
                     (ik > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < C::BN / 16; ++kk) {
            if constexpr (C::DQ_T)  // dQ^T = K^T dS^T: both operands MN-major
              mma_ss_w(tmem + C::T_DP, k_mnlo + mn_tile_step<D>(kk), HT, ds_mnlo + ds_mn_step(kk), HDS, id_dq,
                       kk > 0 ? 1u : 0u);
            else                    // dQ = dS K
              mma_ss_w(tmem + C::T_DP, ds_mnlo + ds_mn_step(kk), HDS, k_mnlo + mn_tile_step<D>(kk), HT, id_dq,
                       kk > 0 ? 1u : 0u);
          }
          // One commit tells three parties that dK(i) and dQ(i) (and every
          // MMA before them) are complete: the dQ warps (dQ_i is in TMEM),
          // the P/dS warps (the dS^T tile may be overwritten) and, through
          // the arrival of one of them (the P/dS warps at d = 128, the dQ
          // warps at d <= 64), the producer (the Q_i, dO_i stage is free).
          // Two tcgen05.commit fewer per visit for the issuing thread.
          tc_commit(bar(C::B_DQFULL));
          ++ik;
          progress = true;
        }
        if (progress) {
          watch.progress();
        } else {
          ok = watch.idle(abort_flag, status, kWaitLimitNs);
        }
      }
      tc_commit(bar(C::B_MMADONE));
      drain_wait(bar(C::B_MMADONE), 0);
    }
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------- P^T and dS^T, key rows, half a row each
    regs_increase<C::REGS_MATH>();
    const int g = warp >> 2;            // query columns 64g .. 64g+63
    const int t = threadIdx.x & 127;    // key row within the tile, TMEM lane
    const int kv_row = kv0 + t;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float* sLSE = reinterpret_cast<const float*>(smem + C::OFF_LSE);
    const float* sDD = reinterpret_cast<const float*>(smem + C::OFF_DD);
    uint8_t* ds_row = smem + C::OFF_DS + g * C::DS_CHUNK + t * 128;
    const float2 sl2x2 = make_float2(sl2, sl2);
    bool ok = true;
    int qi = i0 - 1;
    // Dropout: kw[w] holds this key's keep bytes for queries q0 + 4w .. q0 + 4w + 3
    // of the visit being processed.  The next visit's are drawn ahead, right
    // after this visit's dS^T is handed over, while the thread would otherwise
    // wait for the next S^T: each half warp draws 16 query rows for its 16 keys
    // and transposes the bytes (shuffles; every wait in the loop is made
    // warp-uniform so that no lane leaves the loop while others shuffle).
    uint32_t kw[DROP ? 16 : 1];
    auto draw_visit = [&](int qa) {  // qa: first query of this thread's half
      if constexpr (DROP) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 r4 = philox4x32_10(
              make_uint4(static_cast<uint32_t>(kv_row >> 4), static_cast<uint32_t>(qa + 16 * u + (lane & 15)),
                         static_cast<uint32_t>(bh), drop.offset),
              drop.k0, drop.k1);
          uint32_t w[4] = {r4.x, r4.y, r4.z, r4.w};
          transpose16x16_bytes(w, lane);
#pragma unroll
          for (int e = 0; e < 4; ++e) kw[4 * u + e] = w[e];
        }
      }
    };
    // the query tile of the first visit: i0, or (SPARSE) the first the mask enables
    if (DROP && nq > 0) draw_visit((SPARSE ? next_set_bit(qbits, i0, ntq) : i0) * C::BM + g * 64);
    for (int it = 0; it < nq; ++it) {
      const int s = it % C::NSTQ;
      const int q0 = ATTN_BWD_QTILE(it, qi) * C::BM + g * 64;  // first query of this thread's half
      ok = mbar_wait(bar(C::B_SFULL), it & 1, abort_flag, status);
      if constexpr (DROP) ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();
      float p[64];
      {
        uint32_t u[64];
        tmem_ld64(tmem + lane_off + C::T_S + g * 64, u);
#pragma unroll
        for (int c = 0; c < 64; ++c) p[c] = __uint_as_float(u[c]);
      }
      const float2* nlse = reinterpret_cast<const float2*>(sLSE + s * C::BM + g * 64);  // -LSE*log2(e)
      // query q0 + c sees this key iff kv_row <= q0 + c (causal); key rows >= N are padding
      int first = 0;
      if (kv_row >= N) first = 64;
      else if (causal && kv_row > q0) first = min(kv_row - q0, 64);
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float2 e = fma2(make_float2(p[c], p[c + 1]), sl2x2, nlse[c / 2]);
        p[c] = ex2_approx(e.x);
        p[c + 1] = ex2_approx(e.y);
      }
      if (first > 0) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < first) p[c] = 0.f;
      }
      const uint32_t t2 = drop.t * 0x00010001u;
      {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          pk[i] = pack2<BF16>(p[2 * i], p[2 * i + 1]);
          if constexpr (DROP)
            pk[i] &= ~drop_mask16(drop_lanes(kw[i >> 1], (i & 1) ? kDropSelHi : kDropSelLo, t2));
        }
        tmem_st32(tmem + lane_off + C::T_S + g * 64, pk);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(C::B_PFULL));

      if constexpr (DROP) {  // warp-uniform: the draws at the end of the visit shuffle
        ok = mbar_wait(bar(C::B_DPFULL), it & 1, abort_flag, status);
        if (ok && it > 0) ok = mbar_wait(bar(C::B_DQFULL), (it - 1) & 1, abort_flag, status);
        // visit it-1's MMAs are all complete: its Q, dO stage may be refilled
        // (at d <= 64 the dQ warps release it, see there)
        if (C::DQ_T && ok && it > 0 && threadIdx.x == 0) mbar_arrive(bar(C::B_QEMPTY + (it - 1) % C::NSTQ));
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      } else {
        if (!(ok = mbar_wait(bar(C::B_DPFULL), it & 1, abort_flag, status))) break;
        if (it > 0 && !(ok = mbar_wait(bar(C::B_DQFULL), (it - 1) & 1, abort_flag, status))) break;
        // visit it-1's MMAs are all complete: its Q, dO stage may be refilled
        // (at d <= 64 the dQ warps release it, see there)
        if (C::DQ_T && it > 0 && threadIdx.x == 0) mbar_arrive(bar(C::B_QEMPTY + (it - 1) % C::NSTQ));
      }
      tc_fence_after_sync();
      const float2* nd = reinterpret_cast<const float2*>(sDD + s * C::BM + g * 64);  // -D
#pragma unroll
      for (int c0 = 0; c0 < 2; ++c0) {
        uint32_t dp[32];
        tmem_ld32(tmem + lane_off + C::T_DP + g * 64 + c0 * 32, dp);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = c0 * 32 + 2 * i;
          float2 gd;
          if constexpr (DROP) {  // w dP - D with w = keep * 256 / t
            const uint32_t ln = drop_lanes(kw[c >> 2], (i & 1) ? kDropSelHi : kDropSelLo, t2);
            const uint32_t rs = __float_as_uint(drop.rscale);
            gd = fma2(make_float2(__uint_as_float(dp[2 * i]), __uint_as_float(dp[2 * i + 1])),
                      make_float2(__uint_as_float(rs & ~drop_mask32_first(ln)),
                                  __uint_as_float(rs & ~drop_mask32_second(ln))),
                      nd[c / 2]);
          } else {
            gd = add2(make_float2(__uint_as_float(dp[2 * i]), __uint_as_float(dp[2 * i + 1])), nd[c / 2]);
          }
          const float2 ds = mul2(make_float2(p[c], p[c + 1]), gd);
          pk[i] = pack2<BF16>(ds.x, ds.y);
        }
        // this chunk's 32 query columns are 16-byte units c0*4 .. c0*4+3 of the row
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
          const int unit = (c0 * 4 + uu) ^ (t & 7);
          *reinterpret_cast<uint4*>(ds_row + unit * 16) =
              make_uint4(pk[4 * uu], pk[4 * uu + 1], pk[4 * uu + 2], pk[4 * uu + 3]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      mbar_arrive(bar(C::B_DSFULL));
      if (DROP && it + 1 < nq)  // the next visit's query tile (qi: this visit's under SPARSE)
        draw_visit(SPARSE ? next_set_bit(qbits, qi + 1, ntq) * C::BM + g * 64 : q0 + C::BM);
    }
    // dK (warpgroup 0) or dV (warpgroup 1) once the last MMAs have completed.
    // At d = 128 the rows leave through the K (dK) or V (dV) tile in shared
    // memory, which no MMA reads any more: each thread writes its row there,
    // then each warp stores its 32 rows with 512 contiguous bytes per
    // instruction (as the forward's O).  The warp takes the branch together.
    constexpr bool STAGE = (D == 128);
    bool ep = ok && nq > 0 && mbar_wait(bar(C::B_DQFULL), (nq - 1) & 1, abort_flag, status);
    if constexpr (STAGE) ep = __all_sync(0xffffffffu, ep);
    if (ep && half >= 0) {
      // a split item: this half's fp32 tile (x scale for dK, x 256/t for dV)
      tc_fence_after_sync();
      const uint32_t tcol = tmem + lane_off + (g == 0 ? C::T_DK : C::T_DV);
      const float mul = g == 0 ? scale : (DROP ? drop.rscale : 1.f);
      float4* prow = reinterpret_cast<float4*>(part + ((static_cast<int64_t>(sidx) * 2 + half) * 2 + g) * 128 * D +
                                               static_cast<int64_t>(t) * D);
#pragma unroll
      for (int c0 = 0; c0 < D / 32; ++c0) {
        uint32_t v[32];
        tmem_ld32(tcol + c0 * 32, v);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          prow[c0 * 8 + i] = make_float4(__uint_as_float(v[4 * i]) * mul, __uint_as_float(v[4 * i + 1]) * mul,
                                         __uint_as_float(v[4 * i + 2]) * mul, __uint_as_float(v[4 * i + 3]) * mul);
      }
    } else if (ep) {
      tc_fence_after_sync();
      const int64_t rbase = (static_cast<int64_t>(bh) * N + kv_row) * (D * 2);
      const uint32_t tcol = tmem + lane_off + (g == 0 ? C::T_DK : C::T_DV);
      const float mul = g == 0 ? scale : (DROP ? drop.rscale : 1.f);
      uint8_t* out = g == 0 ? dk_out : dv_out;
      uint8_t* dst_row = out + rbase;
      uint8_t* stage = smem + (g == 0 ? C::OFF_K : C::OFF_V);
#pragma unroll
      for (int c0 = 0; c0 < D / 32; ++c0) {
        uint32_t v[32];
        tmem_ld32(tcol + c0 * 32, v);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack2<BF16>(__uint_as_float(v[2 * i]) * mul, __uint_as_float(v[2 * i + 1]) * mul);
        if constexpr (STAGE) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(stage + row_stage_off256(t, c0 * 4 + i)) =
                make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        } else if (kv_row < N) {
          uint4* dst = reinterpret_cast<uint4*>(dst_row + c0 * 64);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if constexpr (STAGE) {
        __syncwarp();
        const int wrow = t & ~31;  // this warp's first key row of the tile
        uint8_t* obase = out + static_cast<int64_t>(bh) * N * (D * 2);
#pragma unroll
        for (int it = 0; it < 16; ++it) {
          const int lin = it * 32 + lane;
          const int rr = wrow + (lin >> 4), u = lin & 15;
          const uint4 val = *reinterpret_cast<const uint4*>(stage + row_stage_off256(rr, u));
          if (kv0 + rr < N) *reinterpret_cast<uint4*>(obase + static_cast<int64_t>(kv0 + rr) * (D * 2) + u * 16) = val;
        }
      }
    } else if (SPARSE && ok && nq == 0 && kv_row < N) {
      // no query tile sees this key tile: its dK (warpgroup 0) or dV (warpgroup 1) row is 0
      uint4* dst = reinterpret_cast<uint4*>((g == 0 ? dk_out : dv_out) +
                                            (static_cast<int64_t>(bh) * N + kv_row) * (D * 2));
#pragma unroll
      for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
    }
  } else {
    // ------------------------------------------------------ dQ (warps 8-11)
    // DQ_T: thread t holds head-dim column t of dQ for the tile's 128 query
    // rows; otherwise thread t holds query row t.
    regs_increase<C::REGS_DQ>();
    const int t = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    constexpr int NCOL = C::DQ_T ? C::BM : D;
    int qi = i0 - 1;
    for (int it = 0; it < nq; ++it) {
      const int q0 = ATTN_BWD_QTILE(it, qi) * C::BM;
      // warp-uniform (the d <= 64 reductions below shuffle across the warp)
      if (!__all_sync(0xffffffffu, mbar_wait(bar(C::B_DQFULL), it & 1, abort_flag, status))) break;
      // The DQFULL commit follows every MMA of this visit, so the visit's Q, dO
      // stage is free now.  At d <= 64 this warpgroup, idle until here, hands
      // it back (the P/dS warps, which do at d = 128, would only see DQFULL at
      // the next visit's dP wait: +3-5 % measured); at d = 128 the dQ warps
      // are still reducing the previous visit when DQFULL arrives.
      if (!C::DQ_T && t == 0) mbar_arrive(bar(C::B_QEMPTY + it % C::NSTQ));
      tc_fence_after_sync();
      uint32_t v[NCOL];
#pragma unroll
      for (int c0 = 0; c0 < NCOL / 32; ++c0) {
        uint32_t w[32];
        tmem_ld32(tmem + lane_off + C::T_DP + c0 * 32, w);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[c0 * 32 + i] = w[i];
      }
      tc_fence_before_sync();
      mbar_arrive(bar(C::B_DQEMPTY));  // TMEM columns free for the next dP^T
      if constexpr (C::DQ_T) {
        // one fp32 reduction per query row; the warp's 32 lanes are 32 adjacent
        // head-dim columns, i.e. 128 contiguous bytes
        float* dst = dq_acc + static_cast<int64_t>(bh) * N * D + static_cast<int64_t>(q0) * D + t;
        const int nrow = min(C::BM, N - q0);
#pragma unroll
        for (int c = 0; c < C::BM; ++c)
          if (c < nrow) red_add_f32(dst + static_cast<int64_t>(c) * D, __uint_as_float(v[c]) * scale);
      } else {
        // Thread t holds query row q0 + t (d <= 64: 64 or 32 floats).  Each group
        // of 8 lanes (rows r0..r7) transposes its 16-byte pieces in blocks of
        // 8 x 8 (three shuffle stages, each swapping one bit of the lane index
        // with the same bit of the piece index), so that reduction k of a
        // block writes row r_k's 8 pieces, 128 contiguous bytes, from the 8
        // lanes: each warp instruction covers 4 whole lines instead of 32
        // scattered half-sectors.  Measured at B=2 H=16 N=8192 d=64: 540
        // TFLOP/s with the scattered form, 642 with lane pairs covering
        // 32-byte sectors, 665 with these 128-byte rows: the L2's reduction
        // throughput is counted in sectors.
        const int l8 = t & 7;
        const int row0 = q0 + (t & ~7);
#pragma unroll
        for (int g = 0; g < D / 32; ++g) {  // groups of 8 pieces (32 floats)
          float w[8][4];
#pragma unroll
          for (int p = 0; p < 8; ++p)
#pragma unroll
            for (int e = 0; e < 4; ++e) w[p][e] = __uint_as_float(v[32 * g + 4 * p + e]);
          // stage b: lanes differing in bit b exchange pieces whose index bit b differs from their lane bit b
#pragma unroll
          for (int b = 0; b < 3; ++b) {
            const int m = 1 << b;
            const bool hi = (l8 & m) != 0;
#pragma unroll
            for (int p = 0; p < 8; ++p) {
              if (p & m) continue;  // handle pairs (p, p | m)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                // lane with bit clear keeps piece p, sends p|m; lane with bit set keeps p|m, sends p
                const float send = hi ? w[p][e] : w[p | m][e];
                const float got = __shfl_xor_sync(0xffffffffu, send, m);
                if (hi) w[p][e] = got; else w[p | m][e] = got;
              }
            }
          }
          // now lane l8 holds piece l8 of rows row0 + k in w[k]
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (row0 + k < N)
              red_add_v4(dq_acc + (static_cast<int64_t>(bh) * N + row0 + k) * D + 32 * g + 4 * l8,
                         w[k][0] * scale, w[k][1] * scale, w[k][2] * scale, w[k][3] * scale);
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 13) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
#undef ATTN_BWD_QTILE
}

template <int D, bool BF16, bool DROP = false, bool SPARSE = false>
int launch_bwd_t(const BwdArgs& a) {
  using C = BwdCfg<D>;
  const int Npad = ((a.N + 127) / 128) * 128;
  const int64_t rows_total = static_cast<int64_t>(a.BH) * Npad;
  CUtensorMap mq, mk, mv, mdo;
  if (!encode_bhnd_map(&mq, a.q, a.BH, a.N, D, C::CH, 128, C::ROWB, BF16) ||
      !encode_bhnd_map(&mk, a.k, a.BH, a.N, D, C::CH, 128, C::ROWB, BF16) ||
      !encode_bhnd_map(&mv, a.v, a.BH, a.N, D, C::CH, 128, C::ROWB, BF16) ||
      !encode_bhnd_map(&mdo, a.dO, a.BH, a.N, D, C::CH, 128, C::ROWB, BF16))
    return kStatusCuda;
  auto kern = attn_bwd_kernel<D, BF16, DROP, SPARSE>;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), C::SMEM_BYTES)) return kStatusCuda;
  if (!check_launch_regs(reinterpret_cast<const void*>(kern), C::REGS_LAUNCH)) return kStatusDeviceCheck;
  // the preprocess and the dQ conversion overlap their neighbours' tails when
  // the main grid is short (one CTA per SM)
  const bool overlap = overlap_launches(static_cast<int64_t>((a.N + C::BN - 1) / C::BN) * a.BH, 1);
  {
    const int64_t threads = rows_total * 8;
    const int blocks = static_cast<int>((threads + 255) / 256);
    if (launch_serialized(overlap, attn_bwd_pre_kernel<D, BF16>, dim3(blocks), dim3(256), 0, a.stream,
                          static_cast<const uint8_t*>(a.o), static_cast<const uint8_t*>(a.dO), a.lse, a.ws_lse2,
                          a.ws_d, a.ws_dq, a.N, Npad, rows_total) != cudaSuccess)
      return kStatusCuda;
  }
  // One block per (key tile, head) item, head after head; the last tail_split
  // items (no causal mask, no block mask) as two half-range blocks each.
  const int nkt = (a.N + C::BN - 1) / C::BN;
  const int64_t items = static_cast<int64_t>(nkt) * a.BH;
  const int tail = (SPARSE || a.causal || !a.ws_part) ? 0 : a.tail_split;
  if (items + tail > 0x7fffffff) return kStatusUnsupported;
  const int split_from = static_cast<int>(items - tail);
  if (launch_serialized(false, kern, dim3(static_cast<unsigned>(items + tail)), dim3(C::THREADS), C::SMEM_BYTES,
                        a.stream,
                        mq, mk, mv, mdo, a.ws_lse2, a.ws_d, a.ws_dq, static_cast<uint8_t*>(a.dk),
                        static_cast<uint8_t*>(a.dv), a.N, Npad, a.sl2, a.scale, a.causal, a.negate, a.status,
                        a.drop, a.bmask, a.H, a.mask_heads,
                        order_head_group(a.BH, int64_t{8} * a.N * D, int64_t{32} << 20), a.BH, split_from,
                        a.ws_part) != cudaSuccess)
    return kStatusCuda;
  {
    const int64_t groups = static_cast<int64_t>(a.BH) * a.N * D / 8;
    const int blocks = static_cast<int>(std::min<int64_t>((groups + 255) / 256, 152 * 16));
    if (launch_serialized(overlap, attn_dq_convert_kernel<D, BF16>, dim3(blocks), dim3(256), 0, a.stream, a.ws_dq,
                          static_cast<uint8_t*>(a.dq), groups, a.ws_part, tail, split_from, nkt, a.N,
                          static_cast<uint8_t*>(a.dk), static_cast<uint8_t*>(a.dv)) != cudaSuccess)
      return kStatusCuda;
  }
  return cudaGetLastError() == cudaSuccess ? kStatusOk : kStatusCuda;
}

}  // namespace

int launch_bwd(const BwdArgs& a) {
  if (a.bmask && a.drop.t != 0) {  // block-sparse with dropout
    if ((a.N + 127) / 128 > kMaxSparseTiles) return kStatusUnsupported;
    switch (a.d) {
      case 32: return a.bf16 ? launch_bwd_t<32, true, true, true>(a) : launch_bwd_t<32, false, true, true>(a);
      case 64: return a.bf16 ? launch_bwd_t<64, true, true, true>(a) : launch_bwd_t<64, false, true, true>(a);
      case 128: return a.bf16 ? launch_bwd_t<128, true, true, true>(a) : launch_bwd_t<128, false, true, true>(a);
      default: return kStatusUnsupported;
    }
  }
  if (a.bmask) {  // block-sparse: at most kMaxSparseTiles query tiles
    if ((a.N + 127) / 128 > kMaxSparseTiles) return kStatusUnsupported;
    switch (a.d) {
      case 32: return a.bf16 ? launch_bwd_t<32, true, false, true>(a) : launch_bwd_t<32, false, false, true>(a);
      case 64: return a.bf16 ? launch_bwd_t<64, true, false, true>(a) : launch_bwd_t<64, false, false, true>(a);
      case 128: return a.bf16 ? launch_bwd_t<128, true, false, true>(a) : launch_bwd_t<128, false, false, true>(a);
      default: return kStatusUnsupported;
    }
  }
  if (a.drop.t != 0) {  // dropout
    switch (a.d) {
      case 32: return a.bf16 ? launch_bwd_t<32, true, true>(a) : launch_bwd_t<32, false, true>(a);
      case 64: return a.bf16 ? launch_bwd_t<64, true, true>(a) : launch_bwd_t<64, false, true>(a);
      case 128: return a.bf16 ? launch_bwd_t<128, true, true>(a) : launch_bwd_t<128, false, true>(a);
      default: return kStatusUnsupported;
    }
  }
  switch (a.d) {
    case 32: return a.bf16 ? launch_bwd_t<32, true>(a) : launch_bwd_t<32, false>(a);
    case 64: return a.bf16 ? launch_bwd_t<64, true>(a) : launch_bwd_t<64, false>(a);
    case 128: return a.bf16 ? launch_bwd_t<128, true>(a) : launch_bwd_t<128, false>(a);
    default: return kStatusUnsupported;
  }
}

}  // namespace attn
