// attn_internal.h -- declarations shared by the library's translation units
// (host launchers, argument bundles, status codes).  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "block_order.h"

namespace attn {

// Status codes; the public values are those of attn_status_t in attn.h.
constexpr int kStatusOk = 0;
constexpr int kStatusInvalid = 1;
constexpr int kStatusUnsupported = 2;
constexpr int kStatusCuda = 3;
constexpr int kStatusTimeout = 4;
constexpr int kStatusArch = 5;
constexpr int kStatusDeviceCheck = 6;

// Block-sparse: at most this many 128-row tiles (N <= 262144); the forward
// keeps a 3-byte entry per key tile and the backward a bit per query tile in
// shared memory.
constexpr int kMaxSparseTiles = 2048;

// Dropout fused into the softmax step (t == 0: off).  Element (i, j) of head
// bh is kept iff a Philox byte drawn for it is below t; kept probabilities
// are scaled by rscale = 256 / t.
struct DropParams {
  uint32_t t;          // keep threshold, 1..256
  uint32_t k0, k1;     // Philox key: seed low / high words
  uint32_t offset;     // fourth counter word
  float rscale;
};

struct FwdArgs {
  const void *q, *k, *v;
  void* o;
  float* lse;
  int BH, N, d;
  float sl2;  // |scale| * log2(e)
  int causal;
  int negate;  // scale < 0: the S MMA negates its A operand
  bool bf16;
  cudaStream_t stream;
  int* status;
  // block-sparse only (nullptr otherwise): [mask_heads][nb][nb] bytes, nb = ceil(N/128)
  const uint8_t* bmask = nullptr;
  int H = 1;
  int mask_heads = 1;
  DropParams drop = {0u, 0u, 0u, 0u, 1.f};
};

struct BwdArgs {
  const void *q, *k, *v, *o, *dO;
  const float* lse;
  void *dq, *dk, *dv;
  int BH, N, d;
  float sl2;    // |scale| * log2(e)
  float scale;  // signed, applied to dQ and dK
  int causal;
  int negate;
  bool bf16;
  cudaStream_t stream;
  int* status;
  // scratch (device): fp32 dQ accumulator [BH][N][d]; LSE*log2e and D, [BH][Npad]
  float* ws_dq;
  float* ws_lse2;
  float* ws_d;
  DropParams drop = {0u, 0u, 0u, 0u, 1.f};
  // block-sparse only (nullptr otherwise): [mask_heads][nb][nb] bytes, nb = ceil(N/128)
  const uint8_t* bmask = nullptr;
  int H = 1;
  int mask_heads = 1;
  // Split of the grid's last partial wave (0 = none; see bwd_tail_split): the
  // last tail_split (key tile, head) items each run as two CTAs over half of
  // the query tiles, writing fp32 partial dK/dV tiles to ws_part
  // (tail_split * 2 halves * 2 outputs * 128 * d floats).
  int tail_split = 0;
  float* ws_part = nullptr;
};

// Items of the backward's last partial wave to split in two, or 0: without
// the causal mask every (key tile, head) item costs the same, so
// tail_split_items(ceil(N/128) * BH, SMs) of block_order.h applies.
int bwd_tail_split(int BH, int N, int causal);

// Bytes of backward scratch for a problem, and its carve-up.
struct BwdScratch {
  size_t dq_off, lse2_off, d_off, total;
};
BwdScratch bwd_scratch_layout(int BH, int N, int d);

// 3-D tiled tensor map over a [BH][N][d] tensor: dims (d, N, BH), box
// (box_inner, box_rows, 1), 128- or 64-byte swizzle by row_bytes, zero fill.
bool encode_bhnd_map(CUtensorMap* map, const void* base, int BH, int N, int d, int box_inner,
                     int box_rows, int row_bytes, bool bf16);

// Raises the kernel's dynamic shared-memory limit once per device.
bool ensure_smem_attr(const void* func, int bytes);

// True iff the kernel was built with exactly `regs` registers per thread (a
// warpgroup register split that does not add up would wait forever).
bool check_launch_regs(const void* func, int regs);

// Streaming multiprocessors of the current device (looked up once per device);
// 0 on error.
int device_sm_count();

// Launches a kernel, with programmatic stream serialization when `overlap`:
// its blocks may then become resident while the previous kernel in the stream
// (if it is one of this library's, which signal
// griddepcontrol.launch_dependents) finishes its last wave, so the launch
// latency between the passes' kernels overlaps work.  A kernel launched
// overlapped executes griddepcontrol.wait before any other instruction, which
// returns once the previous grid has completed and its memory operations are
// visible: no kernel reads early.  (The small preprocess and dQ conversion
// kernels always execute it -- at once after a normal launch; the forward
// kernel when told; the backward main kernel is always launched normally.)
template <typename... KArgs, typename... Args>
cudaError_t launch_serialized(bool overlap, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Overlapped launches pay where the launch latency is a visible share of a
// pass: grids of at most 8 waves (at B=2 H=16 N=8192 they measured 0.6 %
// slower in the backward, at B=8 H=12 N=1024 3-6 % faster, at N=512 22-38 %).
inline bool overlap_launches(int64_t ctas, int ctas_per_sm) {
  return ctas <= int64_t{8} * ctas_per_sm * std::max(1, device_sm_count());
}

struct DecodeArgs {
  const void *q, *k, *v;  // q [BH][d], k/v [BH][L][d] bf16
  void* o;                // [BH][d] bf16
  float* lse;             // [BH]
  int BH, L, d;
  float sl2;              // scale * log2(e) (signed)
  int splits;
  cudaStream_t stream;
  float* ws;              // [BH][splits][d + 2] fp32 partials
};

struct Fp8Args {
  const void *q, *k, *v;  // e4m3 [BH][N][128]
  void* o;                // bf16 [BH][N][128]
  float* lse;             // [BH][N]
  int BH, N, d;
  float sl2;              // scale * descale_q * descale_k * log2(e), >= 0
  float descale_v;
  int causal;
  cudaStream_t stream;
  int* status;
  uint8_t* ws_vt;         // scratch V^T [BH][128][ceil(N/128)*128]
};
int launch_fwd_fp8(const Fp8Args& a);

// 3-D tiled map over one-byte elements: dims (d0, d1, d2), byte strides of
// dims 1 and 2, box (b0, b1, 1), 128-byte swizzle, zero fill.
bool encode_map_u8(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                   uint64_t stride1, uint64_t stride2, uint32_t b0, uint32_t b1);

// Number of key splits per (batch, head) for a decode problem.
int decode_splits(int BH, int L);

int launch_fwd(const FwdArgs& a);
int launch_decode(const DecodeArgs& a);
int launch_bwd(const BwdArgs& a);

// Device address of the sticky status word on the current device (nullptr on
// failure).  Defined next to the word itself.
int* status_word_current_device();

}  // namespace attn
