// dropout.cuh -- device side of the dropout fused into the softmax step
// (FlashAttention深度攻略 §7, operator fusion: the softmax step applies the
// mask and dropout in the same kernel).
//
// Keep decisions are regenerated wherever they are needed, never stored:
// element (query i, key j) of head bh is kept iff the byte
//     u_ij = byte (j mod 4) of word (j mod 16) / 4 of
//            Philox4x32-10(counter = (j / 16, i, bh, offset), key = (k0, k1))
// is below t (1 <= t <= 256); kept probabilities are scaled by 256 / t.
// Philox4x32-10 is the counter-based generator of Salmon, Moraes, Dror and
// Shaw (SC'11): ten rounds, each two 32x32->64-bit products of words 0 and 2
// with fixed multipliers, the high halves XORed with words 1 and 3 and the
// round key, the key advanced by two Weyl constants per round.
//
// One Philox call gives the bytes of 16 consecutive keys of one query row.
// The forward owns query rows (one thread per row), so its draws are local.
// The backward owns key rows, so a half warp (16 consecutive keys) computes
// the draws of 16 query rows and transposes the 16 x 16 bytes with shuffles.
#pragma once

#include <stdint.h>

namespace attn {

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * c.x;
    const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * c.z;
    c = make_uint4(static_cast<uint32_t>(p1 >> 32) ^ c.y ^ k0, static_cast<uint32_t>(p1),
                   static_cast<uint32_t>(p0 >> 32) ^ c.w ^ k1, static_cast<uint32_t>(p0));
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// Selectors placing bytes (0, 1) or (2, 3) of a word into the low bytes of
// two 16-bit lanes, with 0x80 above each (operand b = 0x80808080).
constexpr uint32_t kDropSelLo = 0x4140u;
constexpr uint32_t kDropSelHi = 0x4342u;

// 16-bit lanes 0x8000 + u - t for two draws u: bit 15 (31) is set iff the
// first (second) element is dropped.  t2 = t * 0x00010001.
__device__ __forceinline__ uint32_t drop_lanes(uint32_t word, uint32_t sel, uint32_t t2) {
  return prmt(word, 0x80808080u, sel) - t2;
}

// 0xffff in each 16-bit lane whose element is dropped: AND-NOT it into a
// packed pair of 16-bit probabilities.
__device__ __forceinline__ uint32_t drop_mask16(uint32_t lanes) {
  return prmt(lanes, 0u, 0xBB99u);  // sign of byte 1 into bytes 0-1, of byte 3 into bytes 2-3
}

// All-ones 32-bit masks of the first / second element of a lane pair when dropped.
__device__ __forceinline__ uint32_t drop_mask32_first(uint32_t lanes) { return prmt(lanes, 0u, 0x9999u); }
__device__ __forceinline__ uint32_t drop_mask32_second(uint32_t lanes) { return prmt(lanes, 0u, 0xBBBBu); }

// Transposes a 16 x 16 byte matrix held by each half warp: on entry lane l
// holds row l (byte k of its 16 = byte k % 4 of w[k / 4]); on exit it holds
// column l.  Each of the four steps swaps one bit of the lane index with the
// same bit of the byte index, exchanging half the bytes with lane ^ (1 << b).
// Every lane of the warp must call it (full-warp shuffles).
__device__ __forceinline__ void transpose16x16_bytes(uint32_t w[4], int lane) {
  constexpr uint32_t FULL = 0xffffffffu;
  {  // byte bit 3 (word bit 1) <-> lane bit 3
    const bool b = lane & 8;
    uint32_t s0 = b ? w[0] : w[2], s1 = b ? w[1] : w[3];
    s0 = __shfl_xor_sync(FULL, s0, 8);
    s1 = __shfl_xor_sync(FULL, s1, 8);
    if (b) { w[0] = s0; w[1] = s1; } else { w[2] = s0; w[3] = s1; }
  }
  {  // byte bit 2 (word bit 0) <-> lane bit 2
    const bool b = lane & 4;
    uint32_t s0 = b ? w[0] : w[1], s1 = b ? w[2] : w[3];
    s0 = __shfl_xor_sync(FULL, s0, 4);
    s1 = __shfl_xor_sync(FULL, s1, 4);
    if (b) { w[0] = s0; w[2] = s1; } else { w[1] = s0; w[3] = s1; }
  }
  {  // byte bit 1 (16-bit half) <-> lane bit 1
    const bool b = lane & 2;
    const uint32_t gather = b ? 0x5410u : 0x7632u;  // send low halves / high halves
    const uint32_t put0 = b ? 0x3254u : 0x5410u, put1 = b ? 0x3276u : 0x7610u;
    uint32_t s0 = prmt(w[0], w[1], gather), s1 = prmt(w[2], w[3], gather);
    s0 = __shfl_xor_sync(FULL, s0, 2);
    s1 = __shfl_xor_sync(FULL, s1, 2);
    w[0] = prmt(w[0], s0, put0);
    w[1] = prmt(w[1], s0, put1);
    w[2] = prmt(w[2], s1, put0);
    w[3] = prmt(w[3], s1, put1);
  }
  {  // byte bit 0 <-> lane bit 0
    const bool b = lane & 1;
    const uint32_t gather = b ? 0x6420u : 0x7531u;  // send even bytes / odd bytes
    const uint32_t put0 = b ? 0x3514u : 0x5240u, put1 = b ? 0x3716u : 0x7260u;
    uint32_t s0 = prmt(w[0], w[1], gather), s1 = prmt(w[2], w[3], gather);
    s0 = __shfl_xor_sync(FULL, s0, 1);
    s1 = __shfl_xor_sync(FULL, s1, 1);
    w[0] = prmt(w[0], s0, put0);
    w[1] = prmt(w[1], s0, put1);
    w[2] = prmt(w[2], s1, put0);
    w[3] = prmt(w[3], s1, put1);
  }
}

}  // namespace attn
