// attn_fwd.cu -- fused exact-attention forward for sm_103a.
//
// Method (FlashAttention (PKM page), "三招" 1 Tiling and 2 Online Softmax;
// FlashAttention深度攻略 §3 tiling, §4 online softmax, §7 fusion): for a block
// of query rows, stream the key/value blocks through on-chip memory, keep per
// row the running max m, running sum l and an unnormalised output O, rescale
// O and l by exp(m_old - m_new) whenever the max grows, and divide by l once
// at the end.  S = Q K^T and P never leave the SM.
//
// GB300 mapping at d = 128 (one CTA per SM, 12 warps = 3 warpgroups):
//   * CTA = 256 query rows of one (batch, head): two 128-row tiles Q0, Q1 that
//     take turns on the tensor core (while one tile's softmax runs, the other
//     tile's MMAs do), sharing every K/V tile loaded.
//   * warpgroup 2 (warps 8-11) gives most of its registers to the two
//     softmax warpgroups (setmaxnreg 56 / 224), then:
//   * warp 8  : TMA producer -- Q0/Q1 once, then K_j and V_j into an
//               NST-stage ring (128B-swizzled tiles, 3-D tensor maps so a
//               tile never straddles two heads and rows >= N read as zero);
//               its thread also sets up the barriers and issues Q and the
//               first stages before the CTA's set-up barrier.
//   * warp 9  : TMEM owner and single-thread tcgen05.mma issuer.
//               S_q = Q_q K_j^T  (SS: both operands K-major in shared memory)
//               O_q += P_q V_j   (TS: P from TMEM, V MN-major in shared memory)
//   * warps 0-3 / 4-7 : softmax for Q0 / Q1, one thread per query row (TMEM
//               lane), 224 registers each so a whole 128-wide row of S stays in
//               registers.  exp2 with scale*log2(e) folded in (packed f32x2
//               FMAs, three-input max, split accumulators); the reference max is
//               only moved when it grows by more than 2^8 (the same stale max
//               is used for l and for P, so the result is unchanged); O is
//               rescaled in TMEM by the same thread; P is written back to TMEM
//               as bf16/fp16 over the first half of its S columns.  l is kept
//               twice: the exact sum for LSE, and the sum of the rounded P
//               values (the weights actually applied to V) to normalise O.
//   * TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+D) O1 [256+D,256+2D);
//     P_q overwrites half of S_q, and the tile's next S goes out right after
//     the current P V (the tensor pipe runs one thread's MMAs in issue order).
// At d <= 64, and for block-sparse masks at d = 128, a CTA holds ONE query
// tile (NQ = 1: warps 0-3 softmax, 4 the producer, 5 the issuer; 256 TMEM
// columns; a 2-stage ring at d <= 64, 1 stage at d = 128) and two CTAs share
// each SM, so the tile-to-tile overlap comes from the other CTA, which also
// hides this CTA's set-up, first loads, drain and epilogue, and a
// block-sparse CTA walks its own tile's list, not the union of two.  At
// d <= 64 P has TMEM columns of its own, so a tile's next S goes out once its
// softmax has read the current S.
// Causal: key tiles entirely above the diagonal are never loaded or
// multiplied; only the diagonal tile (and the ragged last tile) are masked;
// the CTAs run heaviest first across a group of heads (block_order.h).
// Dropout (DROP): after P is rounded and summed into l, each thread clears
// the dropped halves of its packed P before it goes to TMEM, from keep bytes
// drawn for its row (one Philox call per 16 keys, dropout.cuh) while it was
// waiting for this tile's S; the P V product starts on keys 0-63 while the
// second half is masked, and the epilogue folds 256 / t into 1 / l.  m, l and
// LSE stay those of the undropped softmax.
#include <type_traits>

#include "attn_internal.h"
#include "dropout.cuh"
#include "tc_sm103.cuh"

namespace attn {

namespace {

constexpr float kRescaleThresholdLog2 = 8.0f;

// NQ: query tiles per CTA.  2 everywhere except short sequences at d <= 64,
// where CTAs of one query tile use half the TMEM, a third less shared memory
// and half the softmax warps, so that two of them share an SM and one's
// set-up, first loads, drain and epilogue overlap the other's steps.
template <int D, int NQ = 2, bool DROP = false, bool SPARSE = false>
struct FwdCfg {
  static_assert(NQ == 1 || NQ == 2, "one or two query tiles per CTA");
  static constexpr int BM = 128;                     // query rows per tile (MMA M)
  static constexpr int BN = 128;                     // key rows per tile
  static constexpr int ROWB = (D >= 64) ? 128 : 64;  // bytes per swizzled row
  static constexpr int CH = ROWB / 2;                // elements per swizzled row
  static constexpr int NCH = D / CH;                 // column chunks per tile
  static constexpr uint32_t SWZ = (ROWB == 128) ? kSwizzle128B : kSwizzle64B;
  static constexpr int SBO = 8 * ROWB;               // bytes between 8-row groups
  static constexpr int CHUNK_BYTES = 128 * ROWB;     // one column chunk of a 128-row tile
  static constexpr int TILE_BYTES = 128 * D * 2;
  // (one-tile CTAs at d = 128: a single stage, so that two CTAs fit an SM)
  static constexpr int NST = (NQ == 1 && D == 128) ? 1 : (D == 128 || NQ == 1) ? 2 : 3;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = NQ * TILE_BYTES;
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
  static constexpr int B_PHALF = B_MMADONE + 1;  // dropout: first 64 keys of P_q written
  static constexpr int B_STAKEN = B_PHALF + 2;   // SEPP: S_q read into registers
  static constexpr int NBAR = B_STAKEN + 2;
  static constexpr int OFF_TMEMSLOT = OFF_BAR + NBAR * 8;
  static constexpr int OFF_ABORT = OFF_TMEMSLOT + 4;
  static constexpr int OFF_NPOS = OFF_ABORT + 4;                   // int[3]: positions, per-tile counts
  static constexpr int OFF_LIST = OFF_NPOS + 16;                   // uint16 key tile of each position
  static constexpr int OFF_FLAGS = OFF_LIST + 2 * kMaxSparseTiles;  // uint8 bit q: tile q uses it
  static constexpr int SMEM_BYTES = OFF_FLAGS + kMaxSparseTiles;
  static constexpr int THREADS = 128 * NQ + 128;  // NQ softmax warpgroups, one control warpgroup
  static constexpr int W_PROD = 4 * NQ;           // producer warp (lane 0)
  static constexpr int W_MMA = 4 * NQ + 1;        // MMA issuer warp (lane 0); TMEM owner
  static constexpr int MIN_BLOCKS = 3 - NQ;       // CTAs per SM
  // 65536 / (THREADS * MIN_BLOCKS), rounded down to a multiple of 8: 168, or 128 for one-tile CTAs
  static constexpr int REGS_LAUNCH = (65536 / (THREADS * MIN_BLOCKS)) & ~7;
  // softmax warpgroups / producer and MMA warpgroup.  One-tile CTAs split
  // 256 a thread: 208 / 48; with dropout (a tile of draws carried by the
  // softmax) 224 / 32; block-sparse at d = 128 (the list-walking issuer)
  // 200 / 56 -- each the fastest of the splits measured for its variant
  // (224 / 32 and 208 / 48 measured 14 % and 6 % slower than 200 / 56 there).
  static constexpr int REGS_MATH = NQ == 2 ? 224 : DROP ? 224 : (SPARSE && D == 128) ? 200 : 208;
  static constexpr int REGS_CTRL = NQ == 2 ? 56 : DROP ? 32 : (SPARSE && D == 128) ? 56 : 48;
  static_assert(NQ * 128 * REGS_MATH + 128 * REGS_CTRL <= THREADS * REGS_LAUNCH, "register split");
  static constexpr uint32_t TMEM_COLS = NQ == 2 ? 512 : 256;
  // At d <= 64, P_q has TMEM columns of its own after O0, O1 (64 columns of
  // packed 16-bit values each), so S_q(j+1) can be computed as soon as the
  // softmax has read S_q(j), while P_q(j) V_j is still pending.  At d = 128
  // the 512 columns are full and P_q overwrites the first half of S_q, so
  // S_q(j+1) follows P_q(j) V_j in the tensor pipe's issue order.
  static constexpr bool SEPP = (D <= 64);
  static constexpr uint32_t TM_S = 0;                              // + 128 q
  static constexpr uint32_t TM_O = NQ * BN;                        // + D q
  static constexpr uint32_t TM_P = SEPP ? NQ * BN + NQ * D : 0;    // + (SEPP ? 64 : 128) q
  static constexpr uint32_t TM_PSTRIDE = SEPP ? BN / 2 : BN;
  static_assert(NQ * 128 + NQ * D + (SEPP ? NQ * 64 : 0) <= TMEM_COLS, "TMEM budget");
  static_assert(MIN_BLOCKS * (SMEM_BYTES + 1024) <= 233472, "shared memory budget");
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

// The same two descriptors as words (smem_desc_lo/hi): the issuers form the
// low word of a tile once per MMA group and add these per-slice offsets, so
// each MMA costs one add per operand.
template <int D>
__host__ __device__ constexpr uint32_t kmajor_lo_step(int kk) {
  using C = FwdCfg<D>;
  return static_cast<uint32_t>(((kk * 16) / C::CH * C::CHUNK_BYTES + (kk * 16) % C::CH * 2) >> 4);
}
template <int D>
__host__ __device__ constexpr uint32_t mnmajor_lo_step(int kk) {
  return static_cast<uint32_t>((kk * 16 * FwdCfg<D>::ROWB) >> 4);
}

// Byte offset of 16-byte unit u of row `row` in the epilogue's staging copy of
// an O tile (rows of 2 D bytes).  The unit index is XOR-ed with bits of the row
// so that both the row-per-thread writes and the row-contiguous reads of a
// warp touch eight different bank groups in each 8-lane phase.
template <int D>
__device__ __forceinline__ uint32_t ostage_off(int row, int u) {
  if constexpr (D >= 64) return static_cast<uint32_t>(row * (2 * D) + ((u ^ (row & 7)) << 4));
  else return static_cast<uint32_t>(row * (2 * D) + ((u ^ ((row >> 1) & 3)) << 4));
}

// Waits that ignore the abort flag: used only to drain work already issued.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_test(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
  }
}

// The key/value tiles a CTA visits are "positions" 0..npos-1: dense, position
// p is key tile p and query tile q uses positions p < nkv[q]; block-sparse
// (SPARSE), the positions are the union of the key tiles either query tile's
// mask row enables (after the causal limit), listed in shared memory with a
// per-position bit for each query tile.  Producer, MMA issuer and softmax all
// walk positions, so a K/V tile is loaded once per CTA and each query tile
// runs its S/PV chain over its own positions only.
template <int D, bool BF16, bool SPARSE, bool DROP, int NQ>
__global__ void __launch_bounds__(FwdCfg<D, NQ, DROP, SPARSE>::THREADS, FwdCfg<D, NQ, DROP, SPARSE>::MIN_BLOCKS)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, uint8_t* __restrict__ o_out,
                    float* __restrict__ lse_out, int N, float sl2, int causal, int negate,
                    const uint8_t* __restrict__ bmask, int H, int mask_heads, int* status,
                    DropParams drop, int head_group, int overlap) {
  using C = FwdCfg<D, NQ, DROP, SPARSE>;
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
  for (int q = 0; q < 2; ++q) {  // (a one-tile CTA's tile 1 is empty)
    const int row0 = qb * NQ * C::BM + q * C::BM;
    nkv[q] = (q >= NQ || row0 >= N) ? 0 : (causal ? min(nkv_all, row0 / C::BN + 1) : nkv_all);
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

  uint16_t* pos_tile = reinterpret_cast<uint16_t*>(smem + C::OFF_LIST);
  uint8_t* pos_flags = smem + C::OFF_FLAGS;
  int* npos_slot = reinterpret_cast<int*>(smem + C::OFF_NPOS);
  const uint32_t sQ = sbase + C::OFF_Q;
  const uint32_t sK = sbase + C::OFF_K;
  const uint32_t sV = sbase + C::OFF_V;
  // The producer thread sets up the barriers and issues the Q tiles and the
  // first ring stages before the CTA-wide set-up barrier, so that their load
  // latency overlaps the TMEM allocation and the barrier itself.
  int pre_issued = 0;  // positions whose K and V loads went out before the barrier
  if (warp == C::W_PROD && lane == 0) {
    if constexpr (SPARSE) {
      const uint8_t* mb = bmask + static_cast<size_t>((bh % H) % mask_heads) * nkv_all * nkv_all;
      int n = 0, c0 = 0, c1 = 0;
      for (int j = 0; j < nkv_all; ++j) {
        int f = 0;
        if (j < nkv[0] && mb[static_cast<size_t>(NQ * qb) * nkv_all + j]) f |= 1;
        if (j < nkv[1] && mb[static_cast<size_t>(NQ * qb + 1) * nkv_all + j]) f |= 2;
        if (f) {
          pos_tile[n] = static_cast<uint16_t>(j);
          pos_flags[n] = static_cast<uint8_t>(f);
          c0 += f & 1;
          c1 += f >> 1;
          ++n;
        }
      }
      npos_slot[0] = n;
      npos_slot[1] = c0;
      npos_slot[2] = c1;
    }
    mbar_init(bar(C::B_QFULL), 1);
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar(C::B_KFULL + s), 1);
      // dense: one unit per query tile (the softmax releases); block-sparse:
      // the issuer releases
      mbar_init(bar(C::B_KEMPTY + s), SPARSE ? 1 : 2);
      mbar_init(bar(C::B_VFULL + s), 1);
      mbar_init(bar(C::B_VEMPTY + s), SPARSE ? 1 : 2);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(bar(C::B_SFULL + q), 1);
      mbar_init(bar(C::B_PFULL + q), C::BM);
      mbar_init(bar(C::B_PHALF + q), C::BM);
      mbar_init(bar(C::B_ODONE + q), 1);
      mbar_init(bar(C::B_STAKEN + q), C::BM);
    }
    mbar_init(bar(C::B_MMADONE), 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    const int np = SPARSE ? npos_slot[0] : nkv_max;
    if (np > 0) {  // a CTA with nothing to visit loads nothing
      mbar_arrive_expect_tx(bar(C::B_QFULL), NQ * C::TILE_BYTES);
      for (int q = 0; q < NQ; ++q)
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(sQ + q * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_q, bar(C::B_QFULL), c * C::CH,
                      qb * NQ * C::BM + q * C::BM, bh);
    }
    pre_issued = min(np, C::NST);
    for (int j = 0; j < pre_issued; ++j) {  // stages still empty: no waits
      const int kv_row0 = (SPARSE ? static_cast<int>(pos_tile[j]) : j) * C::BN;
      mbar_arrive_expect_tx(bar(C::B_KFULL + j), C::TILE_BYTES);
      for (int c = 0; c < C::NCH; ++c)
        tma_load_3d(sK + j * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_k, bar(C::B_KFULL + j), c * C::CH, kv_row0,
                    bh);
      mbar_arrive_expect_tx(bar(C::B_VFULL + j), C::TILE_BYTES);
      for (int c = 0; c < C::NCH; ++c)
        tma_load_3d(sV + j * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_v, bar(C::B_VFULL + j), c * C::CH, kv_row0,
                    bh);
    }
  }
  if (warp == C::W_MMA) {
    tmem_alloc(smem_addr(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  const int npos = SPARSE ? npos_slot[0] : nkv_max;
  int cnt[2];
  cnt[0] = SPARSE ? npos_slot[1] : nkv[0];
  cnt[1] = SPARSE ? npos_slot[2] : nkv[1];
  auto kv_tile = [&](int p) -> int { return SPARSE ? static_cast<int>(pos_tile[p]) : p; };
  auto uses = [&](int q, int p) -> bool { return SPARSE ? ((pos_flags[p] >> q) & 1) != 0 : p < nkv[q]; };

  if (warp >= C::W_PROD) {
    regs_decrease<C::REGS_CTRL>();
    if (warp == C::W_PROD && lane == 0) {
      // ---------------------------------------------------------- producer
      // (Q and the first min(NST, npos) positions went out before the set-up
      // barrier, see above.)
      int issued = pre_issued;
      for (int j = pre_issued; j < npos; ++j) {
        const int s = j % C::NST, u = j / C::NST;
        const int kv_row0 = kv_tile(j) * C::BN;
        if (u > 0 && !mbar_wait(bar(C::B_KEMPTY + s), (u - 1) & 1, abort_flag, status)) break;
        mbar_arrive_expect_tx(bar(C::B_KFULL + s), C::TILE_BYTES);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(sK + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_k, bar(C::B_KFULL + s),
                      c * C::CH, kv_row0, bh);
        if (u > 0 && !mbar_wait(bar(C::B_VEMPTY + s), (u - 1) & 1, abort_flag, status)) {
          issued = -(j + 1);  // K_j issued, V_j not
          break;
        }
        mbar_arrive_expect_tx(bar(C::B_VFULL + s), C::TILE_BYTES);
        for (int c = 0; c < C::NCH; ++c)
          tma_load_3d(sV + s * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_v, bar(C::B_VFULL + s),
                      c * C::CH, kv_row0, bh);
        issued = j + 1;
      }
      if (*abort_flag) {
        // Let every copy already issued land before the CTA's shared memory goes away.
        if (npos > 0) drain_wait(bar(C::B_QFULL), 0);
        const int nk = issued >= 0 ? issued : -issued;
        const int nv = issued >= 0 ? issued : -issued - 1;
        for (int s = 0; s < C::NST; ++s) {
          const int ck = nk > s ? (nk - 1 - s) / C::NST + 1 : 0;  // loads issued on stage s
          const int cv = nv > s ? (nv - 1 - s) / C::NST + 1 : 0;
          if (ck) drain_wait(bar(C::B_KFULL + s), (ck - 1) & 1);
          if (cv) drain_wait(bar(C::B_VFULL + s), (cv - 1) & 1);
        }
      }
    } else if (warp == C::W_MMA && lane == 0) {
      // -------------------------------------------------------- MMA issuer
      // Each query tile runs its own chain S, PV, S, PV, ... over the positions
      // it uses; the issuer polls both chains and issues whichever next MMA
      // group is ready, so one tile's softmax never holds up the other's MMAs.
      //   S_q at position p  needs K_p resident and, with P in S's columns
      //                      (d = 128), the tile's previous PV issued;
      //   PV_q at position p needs V_p resident and P_q written by the softmax.
      // The K and V stages are released by the softmax threads (below), which
      // learn from their own waits when the MMAs reading a stage have
      // completed: the issuer's only tcgen05 operations are the MMAs and one
      // commit per group.  (The issuing thread shares its SM sub-partition with
      // two softmax warps, so each instruction it saves shortens the chain.)
      constexpr uint32_t HI = smem_desc_hi(C::SBO, C::SWZ);
      const uint32_t q_lo0 = smem_desc_lo(sQ, 16), q_lo1 = smem_desc_lo(sQ + C::TILE_BYTES, 16);
      if constexpr (!SPARSE) {
        const uint32_t idesc_s = instr_desc_f16(C::BM, C::BN, BF16, false, false, negate != 0);
        const uint32_t idesc_o = instr_desc_f16(C::BM, D, BF16, false, true);
        bool ok = nkv_max == 0 || mbar_wait(bar(C::B_QFULL), 0, abort_flag, status);
        tc_fence_after_sync();
        int js[2] = {0, 0};  // next S index per tile
        int jp[2] = {0, 0};  // next PV index per tile
        bool half[2] = {false, false};  // first half of PV_q(jp) issued
        // d = 128: positions below k_seen / v_seen have had their K / V load
        // seen to land (each tile issues its MMAs in position order, so every
        // lower position was seen first), and a stage is refilled only after
        // both tiles have used it, so such a position stays resident until
        // this tile's MMA on it is issued: the pass probes the P barrier only
        // (each probe is a shared-memory round trip on a sub-partition shared
        // with two softmax warps; +3 % at d = 128, about -1 % at d <= 64,
        // which keeps probing every barrier).
        int k_seen = 0, v_seen = 0;
        IdleWatch watch;
        while (ok && (jp[0] < nkv[0] || jp[1] < nkv[1])) {
          bool progress = false;
          // Tile 1 is checked first: under the causal mask its chain is one key
          // tile longer, and serving it first measured 1-5 % faster causal
          // (no change without the mask).  Within a tile P V comes before S.
  #pragma unroll
          for (int qq = 2 - NQ; qq < 2; ++qq) {
            const int q = 1 - qq;
            // PV_q(jp).  With dropout it goes in two halves: keys 0-63 as soon
            // as the softmax has written that half of P (it draws and writes the
            // second half meanwhile), keys 64-127 once all of P_q is written.
            // Without dropout the second half is too short to hide the extra
            // hand-off, and PV waits for all of P.
            const int jv = jp[q];
            if (jv < nkv[q] && jv < js[q] && !half[q] &&
                (C::SEPP ? mbar_probe(bar(C::B_VFULL + jv % C::NST), (jv / C::NST) & 1) &&
                               mbar_probe(bar((DROP ? C::B_PHALF : C::B_PFULL) + q), jv & 1)
                         : mbar_probe(bar((DROP ? C::B_PHALF : C::B_PFULL) + q), jv & 1) &&
                               (jv < v_seen || mbar_probe(bar(C::B_VFULL + jv % C::NST), (jv / C::NST) & 1)))) {
              v_seen = max(v_seen, jv + 1);
              tc_fence_after_sync();
              const uint32_t d_o = tmem + C::TM_O + q * D;
              const uint32_t a_p = tmem + C::TM_P + q * C::TM_PSTRIDE;
              const uint32_t v_lo = smem_desc_lo(sV + (jv % C::NST) * C::TILE_BYTES, C::CHUNK_BYTES);
              constexpr int KK_FIRST = DROP ? C::BN / 32 : C::BN / 16;
  #pragma unroll
              for (int kk = 0; kk < KK_FIRST; ++kk)
                mma_ts_w(d_o, a_p + kk * 8, v_lo + mnmajor_lo_step<D>(kk), HI, idesc_o, (jv > 0 || kk > 0) ? 1u : 0u);
              if constexpr (DROP) {
                half[q] = true;
              } else {
                tc_commit(bar(C::B_ODONE + q));
                jp[q] = jv + 1;
              }
              progress = true;
            }
            if (DROP && half[q] && mbar_probe(bar(C::B_PFULL + q), jv & 1)) {
              tc_fence_after_sync();
              const uint32_t d_o = tmem + C::TM_O + q * D;
              const uint32_t a_p = tmem + C::TM_P + q * C::TM_PSTRIDE;
              const uint32_t v_lo = smem_desc_lo(sV + (jv % C::NST) * C::TILE_BYTES, C::CHUNK_BYTES);
  #pragma unroll
              for (int kk = C::BN / 32; kk < C::BN / 16; ++kk)
                mma_ts_w(d_o, a_p + kk * 8, v_lo + mnmajor_lo_step<D>(kk), HI, idesc_o, 1u);
              tc_commit(bar(C::B_ODONE + q));
              jp[q] = jv + 1;
              half[q] = false;
              progress = true;
            }
            // S_q(js).  With P apart (SEPP) it needs the previous S read out
            // by the softmax.  With P in S's columns (d = 128) it needs the
            // tile's previous P V issued, not complete: S_q(j+1) overwrites the
            // P_q(j) that P_q(j) V reads from TMEM, and the tensor pipe executes
            // one thread's MMAs in issue order, so that read happens first.
            // (The PTX ISA promises this order only for MMAs into the same
            // accumulator; on GB300 the in-order form gave bit-identical
            // results in every repeated run of every configuration tried, and
            // saves the chain a completion round trip per step: +4 % at d = 128.)
            // The softmax's own waits are unaffected: the commit that signals
            // S_q(j+1) tracks every MMA issued before it, P_q(j) V included.
            const int jk = js[q];
            if (jk < nkv[q] && (C::SEPP || jk == jp[q]) &&
                (C::SEPP ? mbar_probe(bar(C::B_KFULL + jk % C::NST), (jk / C::NST) & 1) &&
                               (jk == 0 || mbar_probe(bar(C::B_STAKEN + q), (jk - 1) & 1))
                         : (jk < k_seen || mbar_probe(bar(C::B_KFULL + jk % C::NST), (jk / C::NST) & 1)))) {
              k_seen = max(k_seen, jk + 1);
              tc_fence_after_sync();
              const uint32_t d_s = tmem + C::TM_S + q * C::BN;
              const uint32_t a_lo = q ? q_lo1 : q_lo0;
              const uint32_t k_lo = smem_desc_lo(sK + (jk % C::NST) * C::TILE_BYTES, 16);
  #pragma unroll
              for (int kk = 0; kk < D / 16; ++kk)
                mma_ss_w(d_s, a_lo + kmajor_lo_step<D>(kk), HI, k_lo + kmajor_lo_step<D>(kk), HI, idesc_s,
                         kk > 0 ? 1u : 0u);
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
      } else {
        const uint32_t idesc_s = instr_desc_f16(C::BM, C::BN, BF16, false, false, negate != 0);
        const uint32_t idesc_o = instr_desc_f16(C::BM, D, BF16, false, true);
        bool ok = npos == 0 || mbar_wait(bar(C::B_QFULL), 0, abort_flag, status);
        tc_fence_after_sync();
        int sp[2] = {0, 0};  // next position to consider for S, per tile
        int pp[2] = {0, 0};  // next position to consider for PV, per tile
        int ns[2] = {0, 0}, np[2] = {0, 0};  // S / PV groups issued per tile
        bool half[2] = {false, false};       // dropout: keys 0-63 of PV_q issued, 64-127 not yet
        int k_ready = 0, v_ready = 0;  // positions whose K / V load has been seen to land
        int k_rel = 0, v_rel = 0;      // next position whose K / V stage is still held
        IdleWatch watch;
        while (ok && (k_rel < npos || v_rel < npos)) {
          bool progress = false;
          // Loads are observed strictly in position order: when position p is
          // probed, every earlier load on its stage has been seen, so the stage
          // barrier is at most one phase ahead and the parity test is exact.  (A
          // tile that skips positions must not probe a later phase directly.)
          while (k_ready < npos && mbar_probe(bar(C::B_KFULL + k_ready % C::NST), (k_ready / C::NST) & 1))
            ++k_ready;
          while (v_ready < npos && mbar_probe(bar(C::B_VFULL + v_ready % C::NST), (v_ready / C::NST) & 1))
            ++v_ready;
  #pragma unroll
          for (int q = 0; q < NQ; ++q) {
            while (sp[q] < npos && !uses(q, sp[q])) ++sp[q];
            while (pp[q] < sp[q] && !uses(q, pp[q])) ++pp[q];
            // PV_q at pp (its S was issued: every used position below sp has one)
            // (with dropout in two halves, as in the dense issuer: keys 0-63
            // once that half of P is written, keys 64-127 once all of it is)
            const int jv = pp[q];
            using KK_FIRST = std::integral_constant<int, DROP ? C::BN / 32 : C::BN / 16>;
            using KK_ALL = std::integral_constant<int, C::BN / 16>;
            auto issue_pv = [&](auto kk0c, auto kk1c) {  // MMA groups [kk0, kk1) of 16 keys
              constexpr int kk0 = decltype(kk0c)::value, kk1 = decltype(kk1c)::value;
              const uint32_t d_o = tmem + C::TM_O + q * D;
              const uint32_t a_p = tmem + C::TM_P + q * C::TM_PSTRIDE;
              // (descriptor words at d <= 64; at d = 128 this issuer measured 9 %
              // faster with the 64-bit descriptors formed per MMA)
              if constexpr (C::SEPP) {
                const uint32_t v_lo = smem_desc_lo(sV + (jv % C::NST) * C::TILE_BYTES, C::CHUNK_BYTES);
  #pragma unroll
                for (int kk = kk0; kk < kk1; ++kk)
                  mma_ts_w(d_o, a_p + kk * 8, v_lo + mnmajor_lo_step<D>(kk), HI, idesc_o,
                           (np[q] > 0 || kk > 0) ? 1u : 0u);
              } else {
                const uint32_t v_s = sV + (jv % C::NST) * C::TILE_BYTES;
  #pragma unroll
                for (int kk = kk0; kk < kk1; ++kk)
                  mma_ts(d_o, a_p + kk * 8, desc_mnmajor<D>(v_s, kk), idesc_o, (np[q] > 0 || kk > 0) ? 1u : 0u);
              }
            };
            if (jv < sp[q] && jv < v_ready && !half[q] &&
                mbar_probe(bar((DROP ? C::B_PHALF : C::B_PFULL) + q), np[q] & 1)) {
              tc_fence_after_sync();
              issue_pv(std::integral_constant<int, 0>{}, KK_FIRST{});
              if constexpr (DROP) {
                half[q] = true;
              } else {
                tc_commit(bar(C::B_ODONE + q));
                pp[q] = jv + 1;
                ++np[q];
              }
              progress = true;
            }
            if (DROP && half[q] && mbar_probe(bar(C::B_PFULL + q), np[q] & 1)) {
              tc_fence_after_sync();
              issue_pv(std::integral_constant<int, C::BN / 32>{}, KK_ALL{});
              tc_commit(bar(C::B_ODONE + q));
              pp[q] = jv + 1;
              ++np[q];
              half[q] = false;
              progress = true;
            }
            // S_q at sp
            const int jk = sp[q];
            if (jk < npos && (C::SEPP || ns[q] == np[q]) && jk < k_ready &&
                (ns[q] == 0 || !C::SEPP || mbar_probe(bar(C::B_STAKEN + q), (ns[q] - 1) & 1))) {
              tc_fence_after_sync();
              const uint32_t d_s = tmem + C::TM_S + q * C::BN;
              if constexpr (C::SEPP) {
                const uint32_t a_lo = q ? q_lo1 : q_lo0;
                const uint32_t k_lo = smem_desc_lo(sK + (jk % C::NST) * C::TILE_BYTES, 16);
  #pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                  mma_ss_w(d_s, a_lo + kmajor_lo_step<D>(kk), HI, k_lo + kmajor_lo_step<D>(kk), HI, idesc_s,
                           kk > 0 ? 1u : 0u);
              } else {
                const uint32_t k_s = sK + (jk % C::NST) * C::TILE_BYTES;
  #pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)
                  mma_ss(d_s, desc_kmajor<D>(sQ + q * C::TILE_BYTES, kk), desc_kmajor<D>(k_s, kk), idesc_s,
                         kk > 0 ? 1u : 0u);
              }
              tc_commit(bar(C::B_SFULL + q));
              sp[q] = jk + 1;
              ++ns[q];
              progress = true;
            }
          }
          // Under a block mask the stages are released here, once both tiles
          // are past a position: a tile's next position may lie beyond the
          // ring, so the softmax could not release V from its next step's wait
          // (the load it needs could be queued behind this very stage); K is
          // released here too, which keeps this loop as it measured fastest.
          while (k_rel < npos && sp[0] > k_rel && (NQ < 2 || sp[1] > k_rel)) {
            tc_commit(bar(C::B_KEMPTY + k_rel % C::NST));
            ++k_rel;
          }
          while (v_rel < npos && pp[0] > v_rel && (NQ < 2 || pp[1] > v_rel)) {
            tc_commit(bar(C::B_VEMPTY + v_rel % C::NST));
            ++v_rel;
          }
          if (progress) {
            watch.progress();
          } else {
            ok = watch.idle(abort_flag, status, kWaitLimitNs);
          }
        }
      }
      // Every MMA issued above must finish before TMEM is released.
      tc_commit(bar(C::B_MMADONE));
      drain_wait(bar(C::B_MMADONE), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    regs_increase<C::REGS_MATH>();
    const int q = warp >> 2;
    const int r = threadIdx.x & 127;
    const int row0 = qb * NQ * C::BM + q * C::BM;
    const int row = row0 + r;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::TM_S + q * C::BN;
    const uint32_t tO = tmem + lane_off + C::TM_O + q * D;
    const uint32_t tP = tmem + lane_off + C::TM_P + q * C::TM_PSTRIDE;
    float m = -INFINITY;   // reference max (log2 units), moved lazily
    float l_exact = 0.f;   // sum of exp2(t - m) in fp32: gives LSE
    float l_round = 0.f;   // sum of the rounded P values: normalises O
    bool ok = true;
    const int nk = cnt[q];
    int pos = 0;  // position of this tile's next key tile
    const float2 sl2x2 = make_float2(sl2, sl2);
    // Dropout: the keep bytes of the next key tile are drawn ahead, right after
    // this tile's P is handed over, while the thread would otherwise wait for
    // the next S; kb[4 g + w] = word w of the draw for keys 16 g .. 16 g + 15.
    uint32_t kb[DROP ? 32 : 1];
    auto draw_tile = [&](int key0) {
      if constexpr (DROP) {
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint4 r4 = philox4x32_10(make_uint4(static_cast<uint32_t>(key0 >> 4) + g, static_cast<uint32_t>(row),
                                                    static_cast<uint32_t>(bh), drop.offset),
                                         drop.k0, drop.k1);
          kb[4 * g] = r4.x;
          kb[4 * g + 1] = r4.y;
          kb[4 * g + 2] = r4.z;
          kb[4 * g + 3] = r4.w;
        }
      }
    };
    // The key tile of this tile's first position (block-sparse: the first it uses).
    if (DROP && nk > 0) {
      int p0 = 0;
      if constexpr (SPARSE)
        while (!uses(q, p0)) ++p0;
      draw_tile(kv_tile(p0) * C::BN);
    }
    // K/V stage release: stage p % NST of position p may be refilled once the
    // MMAs of both tiles that read it have completed.  Each position's empty
    // barrier takes two arrival units: one from each tile that uses it, or
    // both from the only tile that does (thread 0 of the tile arrives).
    //   K_p: S_q(p) is complete once this tile's S wait for p has returned;
    //   V_p: P_q(p) V_p is complete once this tile has waited for it (SEPP:
    //        the O wait of the next step; otherwise the next S wait, whose
    //        commit tracks every MMA issued before that S, P V included), or
    //        in the epilogue for the tile's last position.
    // Dense only: a tile's positions are consecutive there, so that next step
    // never needs a load queued behind the stage it holds (block-sparse, the
    // issuer releases both).
    const int nkv_other = q ? nkv[0] : nkv[1];  // dense: positions the other tile uses
    auto release = [&](int first_bar, int p) {
      if (SPARSE) return;
      if (r == 0) mbar_arrive_cnt(bar(first_bar + p % C::NST), p < nkv_other ? 1u : 2u);
    };
    int prev_p = -1;  // position of this tile's previous step
    for (int j = 0; j < nk; ++j) {
      // warp-uniform, as the step votes across the warp (rescale) further on:
      // a lane that left alone would leave the others waiting at the vote
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SFULL + q), j & 1, abort_flag, status)))) break;
      tc_fence_after_sync();
      int pj = j;  // this step's position
      if constexpr (SPARSE) {
        while (!uses(q, pos)) ++pos;
        pj = pos++;
      }
      release(C::B_KEMPTY, pj);
      if (!C::SEPP && prev_p >= 0) release(C::B_VEMPTY, prev_p);
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
      if constexpr (C::SEPP) {  // S_q may be overwritten by the next S now
        tc_fence_before_sync();
        mbar_arrive(bar(C::B_STAKEN + q));
      }
      const int kv0 = kv_tile(pj) * C::BN;
      const bool masked = (kv0 + C::BN > N) || (causal && kv0 + C::BN - 1 > row0);
      int lim = C::BN;  // keys kv0 + c with c < lim are visible to this row
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
      if (m_new > m + kRescaleThresholdLog2) {  // also taken on the first tile (m = -inf)
        alpha = ex2_approx(m - m_new);
        m = m_new;
      }
      const float neg_m = (m == -INFINITY) ? 0.f : -m;
      const float2 nm2 = make_float2(neg_m, neg_m);
#pragma unroll
      for (int c = 0; c < 128; c += 2) {
        const float2 t = fma2(make_float2(sv[c], sv[c + 1]), sl2x2, nm2);
        sv[c] = ex2_approx(t.x);
        sv[c + 1] = ex2_approx(t.y);
      }
      if (masked) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c >= lim) sv[c] = 0.f;
      }
      // With P apart (SEPP), P_q(j-1) V may still be running: its completion
      // frees P_q and makes O_q final for the rescale below.  (At d = 128 it
      // was issued before S_q(j), so the S wait above covers it.)
      if (C::SEPP && j > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_ODONE + q), (j - 1) & 1, abort_flag, status));
        if (!ok) break;
        tc_fence_after_sync();
        release(C::B_VEMPTY, prev_p);
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
      // P is rounded to the input type for the P V product.
      if constexpr (!DROP && !C::SEPP) {
        // d = 128 without dropout: P goes out first and the two row sums
        // follow, overlapping the P V product instead of delaying it (+2 %;
        // at d = 32 the same order measured 7 % slower, at d = 64 no change).
        uint32_t pk0[32], pk1[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) pk0[i] = pack2<BF16>(sv[2 * i], sv[2 * i + 1]);
        tmem_st32(tP, pk0);
#pragma unroll
        for (int i = 0; i < 32; ++i) pk1[i] = pack2<BF16>(sv[64 + 2 * i], sv[64 + 2 * i + 1]);
        tmem_st32(tP + 32, pk1);
        tmem_st_wait();
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
          sr0 = add_halves<BF16>(sr0, pk0[i]);
          sr1 = add_halves<BF16>(sr1, pk0[i + 1]);
          sr2 = add_halves<BF16>(sr2, pk1[i]);
          sr3 = add_halves<BF16>(sr3, pk1[i + 1]);
        }
        l_exact = l_exact * alpha + ((se0.x + se0.y) + (se1.x + se1.y));
        l_round = l_round * alpha + ((sr0 + sr1) + (sr2 + sr3));
        prev_p = pj;
        continue;
      }
      float2 se0 = make_float2(0.f, 0.f), se1 = se0;
      float sr0 = 0.f, sr1 = 0.f, sr2 = 0.f, sr3 = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < 2; ++c0) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 p0 = make_float2(sv[c0 * 64 + 2 * i], sv[c0 * 64 + 2 * i + 1]);
          const float2 p1 = make_float2(sv[c0 * 64 + 2 * i + 2], sv[c0 * 64 + 2 * i + 3]);
          pk[i] = pack2<BF16>(p0.x, p0.y);
          pk[i + 1] = pack2<BF16>(p1.x, p1.y);
          se0 = add2(se0, p0);
          se1 = add2(se1, p1);
          if (i & 2) {
            sr2 = add_halves<BF16>(sr2, pk[i]);
            sr3 = add_halves<BF16>(sr3, pk[i + 1]);
          } else {
            sr0 = add_halves<BF16>(sr0, pk[i]);
            sr1 = add_halves<BF16>(sr1, pk[i + 1]);
          }
        }
        if constexpr (DROP) {
          // keys kv0 + 64 c0 + 16 g + (0..15): word w of their draw covers keys 4w..4w+3
          const uint32_t t2 = drop.t * 0x00010001u;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              const uint32_t rw = kb[4 * (4 * c0 + g) + w];
              pk[8 * g + 2 * w] &= ~drop_mask16(drop_lanes(rw, kDropSelLo, t2));
              pk[8 * g + 2 * w + 1] &= ~drop_mask16(drop_lanes(rw, kDropSelHi, t2));
            }
          }
        }
        tmem_st32(tP + c0 * 32, pk);
        if (DROP && c0 == 0) {  // keys 0-63 of P (and any O correction) are in TMEM
          tmem_st_wait();
          tc_fence_before_sync();
          mbar_arrive(bar(C::B_PHALF + q));
        }
      }
      l_exact = l_exact * alpha + ((se0.x + se0.y) + (se1.x + se1.y));
      l_round = l_round * alpha + ((sr0 + sr1) + (sr2 + sr3));
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(C::B_PFULL + q));
      if (DROP && j + 1 < nk) {  // the key tile of this tile's next position
        int pn = pj + 1;
        if constexpr (SPARSE)
          while (!uses(q, pn)) ++pn;
        draw_tile(kv_tile(pn) * C::BN);
      }
      prev_p = pj;
    }
    // ------------------------------------------------------------ epilogue
    // At d = 128, O leaves through the tile's Q buffer in shared memory, which
    // no MMA reads once the tile's last P V has completed: each thread writes
    // its row there, then each warp stores its 32 rows with 512 contiguous
    // bytes per instruction instead of 32 scattered 16-byte pieces (+0.6 to
    // +1.7 % measured; at d <= 64, with half as many bytes a row, the direct
    // row stores measured faster and are kept).  The warp takes the branch
    // together (the staging is per warp, joined by __syncwarp).
    constexpr bool STAGE_O = (D == 128);
    bool ep = ok && nk > 0 && mbar_wait(bar(C::B_ODONE + q), (nk - 1) & 1, abort_flag, status);
    if constexpr (STAGE_O) ep = __all_sync(0xffffffffu, ep);
    if (ep) {
      tc_fence_after_sync();
      release(C::B_VEMPTY, prev_p);
      const float inv_l = (DROP ? drop.rscale : 1.0f) / l_round;
      uint8_t* stage = smem + C::OFF_Q + q * C::TILE_BYTES;
      uint8_t* orow = o_out + (static_cast<int64_t>(bh) * N + row) * (D * 2);
#pragma unroll
      for (int c0 = 0; c0 < D / 32; ++c0) {
        uint32_t ov[32];
        tmem_ld32(tO + c0 * 32, ov);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack2<BF16>(__uint_as_float(ov[2 * i]) * inv_l, __uint_as_float(ov[2 * i + 1]) * inv_l);
        if constexpr (STAGE_O) {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(stage + ostage_off<D>(r, c0 * 4 + i)) =
                make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        } else if (row < N) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c0 * 64);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if constexpr (STAGE_O) {
        __syncwarp();
        constexpr int U = D / 8;  // 16-byte units per row
        const int wrow = r & ~31;  // this warp's first row of the tile
        uint8_t* obase = o_out + static_cast<int64_t>(bh) * N * (D * 2);
#pragma unroll
        for (int it = 0; it < U; ++it) {
          const int lin = it * 32 + lane;
          const int rr = wrow + lin / U, u = lin % U;
          const uint4 val = *reinterpret_cast<const uint4*>(stage + ostage_off<D>(rr, u));
          if (row0 + rr < N) *reinterpret_cast<uint4*>(obase + static_cast<int64_t>(row0 + rr) * (D * 2) + u * 16) = val;
        }
      }
      if (row < N) lse_out[static_cast<int64_t>(bh) * N + row] = (m + log2f(l_exact)) * 0.69314718055994531f;
    } else if (SPARSE && ok && nk == 0 && row < N) {
      // the mask hides every key from this row: O = 0, LSE = -inf
      uint4* dst = reinterpret_cast<uint4*>(o_out + (static_cast<int64_t>(bh) * N + row) * (D * 2));
#pragma unroll
      for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
      lse_out[static_cast<int64_t>(bh) * N + row] = -INFINITY;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == C::W_MMA) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool BF16, bool SPARSE, bool DROP = false, int NQ = 2>
int launch_fwd_t(const FwdArgs& a) {
  using C = FwdCfg<D, NQ, DROP, SPARSE>;
  CUtensorMap mq, mk, mv;
  const int rowb = C::ROWB;
  if (!encode_bhnd_map(&mq, a.q, a.BH, a.N, D, C::CH, 128, rowb, BF16) ||
      !encode_bhnd_map(&mk, a.k, a.BH, a.N, D, C::CH, 128, rowb, BF16) ||
      !encode_bhnd_map(&mv, a.v, a.BH, a.N, D, C::CH, 128, rowb, BF16))
    return kStatusCuda;
  auto kern = attn_fwd_kernel<D, BF16, SPARSE, DROP, NQ>;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), C::SMEM_BYTES)) return kStatusCuda;
  // The warpgroup register split adds up only at this launch allocation.
  if (!check_launch_regs(reinterpret_cast<const void*>(kern), C::REGS_LAUNCH)) return kStatusDeviceCheck;
  dim3 grid((a.N + NQ * C::BM - 1) / (NQ * C::BM), a.BH);
  const bool overlap = overlap_launches(static_cast<int64_t>(grid.x) * grid.y, C::MIN_BLOCKS);
  const cudaError_t e = launch_serialized(overlap, kern, grid, dim3(C::THREADS), C::SMEM_BYTES, a.stream, mq, mk, mv,
                                          static_cast<uint8_t*>(a.o), a.lse, a.N, a.sl2, a.causal, a.negate,
                                          a.bmask, a.H, a.mask_heads, a.status, a.drop,
                                          order_head_group(a.BH, int64_t{4} * a.N * D, int64_t{128} << 20),
                                          overlap ? 1 : 0);
  return e == cudaSuccess ? kStatusOk : kStatusCuda;
}

// Query tiles per CTA: one (two CTAs per SM) at d <= 64 and for block-sparse
// masks at d = 128, where a CTA then walks its own tile's key list; two for
// the plain and dropout forward at d = 128 (one-tile CTAs measured mixed
// there, and the dropout softmax needs the two-tile CTA's registers).
template <int D>
int launch_fwd_d(const FwdArgs& a) {
  const bool sparse = a.bmask != nullptr, drop = a.drop.t != 0;
  constexpr int NQ = D == 128 ? 2 : 1;
  if (sparse && drop)
    return a.bf16 ? launch_fwd_t<D, true, true, true, NQ>(a) : launch_fwd_t<D, false, true, true, NQ>(a);
  if (drop) return a.bf16 ? launch_fwd_t<D, true, false, true, NQ>(a) : launch_fwd_t<D, false, false, true, NQ>(a);
  if (sparse) return a.bf16 ? launch_fwd_t<D, true, true, false, 1>(a) : launch_fwd_t<D, false, true, false, 1>(a);
  return a.bf16 ? launch_fwd_t<D, true, false, false, NQ>(a) : launch_fwd_t<D, false, false, false, NQ>(a);
}

}  // namespace

int launch_fwd(const FwdArgs& a) {
  if (a.bmask && (a.N + 127) / 128 > kMaxSparseTiles) return kStatusUnsupported;
  switch (a.d) {
    case 32: return launch_fwd_d<32>(a);
    case 64: return launch_fwd_d<64>(a);
    case 128: return launch_fwd_d<128>(a);
    default: return kStatusUnsupported;
  }
}

}  // namespace attn
