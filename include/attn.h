/*
 * attn.h -- C ABI of the GB300 (sm_103a) fused exact-attention library.
 *
 * Exact scaled-dot-product attention, O = softmax(scale * Q K^T [+ causal
 * mask]) V, computed as one fused tiled kernel that keeps the running row
 * max m, running row sum l and an unnormalised O accumulator on chip, so the
 * N x N score and probability matrices never reach HBM.  The forward stores
 * O and the per-row log-sum-exp; the backward recomputes P from that LSE.
 *
 * Sources (web pages on FlashAttention):
 *   - FlashAttention (PKM page), "三招": 1 Tiling, 2 Online Softmax (the m / l /
 *     unnormalised-O recurrence and the final division by l), 3 Recomputation
 *     (store O and the softmax statistics, rebuild P in the backward).
 *   - FlashAttention深度攻略 (xiaohack page) §3 tiling into B_r query rows and
 *     B_c key/value rows, §4 online-softmax derivation, §6 recomputation
 *     backward, §7 kernel fusion, and the live-coding section whose module
 *     works on a (B*H, N, d) view after transposing (B, N, H, d) inputs.
 *   - "Flash Attention 到底做了什么？" (guanweilu page): exactness (differs from
 *     the plain computation only in floating-point rounding order).
 *
 * Conventions shared by every call
 *   - Tensors q, k, v, o, dO, dq, dk, dv are DEVICE pointers to contiguous
 *     row-major [B, H, N, d] arrays of the call's element type (bf16 for the
 *     unsuffixed calls, fp16 for the _f16 twins), 16-byte aligned.  This is
 *     the (B*H, N, d) view of the pages' module; a caller holding (B, N, H, d)
 *     tensors transposes first.
 *   - lse is a DEVICE pointer to fp32 [B, H, N]: LSE_i = ln sum_j
 *     exp(scale * q_i . k_j) over the keys visible to query i (natural log,
 *     in the same units as the scaled logits).
 *   - causal != 0 hides key j from query i iff j > i (square problem: query
 *     and key positions share one index).  scale multiplies Q K^T as given.
 *   - Supported: B, H, N >= 1; N <= 2^24; d in {32, 64, 128}; B*H <= 65535.
 *   - stream is a cudaStream_t (NULL = legacy default stream).  Every call
 *     only enqueues work on it and returns; results are ready when the
 *     stream is.  Calls on different streams that share outputs race.
 *   - All memory passed in is owned by the caller.  The library keeps no
 *     tensor between calls.  Outputs must not alias inputs.
 *   - Errors: argument errors are returned synchronously (nothing is
 *     enqueued).  A kernel that detects a problem on the device (a pipeline
 *     wait that exceeded its time limit) records a sticky status that
 *     attn_sync_status() returns; the kernel itself returns early instead of
 *     hanging, and its outputs are then unspecified.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null/misaligned pointer, non-positive size, non-finite scale */
  ATTN_ERR_UNSUPPORTED = 2, /* head dim not in {32, 64, 128}, or sizes beyond the limits */
  ATTN_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed (launch, allocation, ...) */
  ATTN_ERR_TIMEOUT = 4,     /* a device-side pipeline wait gave up (sticky, see attn_sync_status) */
  ATTN_ERR_ARCH = 5,        /* current device is not compute capability 10.3 (sm_103) */
  ATTN_ERR_DEVICE_CHECK = 6 /* a kernel's own device-side check failed (sticky) */
} attn_status_t;

/*
 * Forward pass, bf16 inputs/outputs, fp32 accumulation.
 *   q, k, v : in,  [B, H, N, d] bf16
 *   o       : out, [B, H, N, d] bf16, O = softmax(scale Q K^T [+mask]) V
 *   lse     : out, [B, H, N] fp32, per-row log-sum-exp of the scaled logits
 * Tiling / online softmax / final 1/l division: FlashAttention (PKM page)
 * "三招" 1 and 2; FlashAttention深度攻略 §3-§4.
 * Returns an attn_status_t.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
             int N, int d, float scale, int causal, void* stream);

/*
 * Backward pass (recomputation), bf16.
 *   q, k, v, o, dO : in, [B, H, N, d] bf16 (o is attn_fwd's output for q, k, v)
 *   lse            : in, [B, H, N] fp32 from attn_fwd
 *   dq, dk, dv     : out, [B, H, N, d] bf16 gradients of L = <O, dO>:
 *                    P = exp(scale Q K^T - LSE) (rebuilt, never stored),
 *                    D_i = sum_k dO_ik O_ik, dS = P o (dO V^T - D),
 *                    dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO.
 * Recomputation: FlashAttention (PKM page) "三招" 3; FlashAttention深度攻略 §6.
 * Scratch: an fp32 dQ accumulator [B, H, N, d] and D [B, H, N] (plus, when
 * a non-causal grid's last partial wave is split over query halves, at most
 * (SMs / 2) x 4 fp32 128 x d tiles of partial dK/dV) are taken from the
 * stream-ordered allocator (cudaMallocAsync on `stream`) and freed on the
 * same stream before the call returns (the memory is released when the
 * stream reaches that point).
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
             const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
             float scale, int causal, void* stream);

/* fp16 twins: identical parameters and semantics with fp16 tensors. */
int attn_fwd_f16(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int N, int d, float scale, int causal, void* stream);
int attn_bwd_f16(const void* q, const void* k, const void* v, const void* o, const void* dO,
                 const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                 float scale, int causal, void* stream);

/*
 * Forward and backward with dropout fused into the softmax step (bf16, and
 * fp16 through the _f16 twins below;
 * FlashAttention深度攻略 §7, operator fusion: the softmax step of the fused
 * kernel also applies dropout).  Inverted dropout on P:
 *   t = floor((1 - p_drop) * 256 + 0.5) (in double), the keep probability
 *   rounded to a multiple of 1/256;
 *   keep_ij = [u_ij < t], u_ij = byte (j mod 4) of word (j mod 16) / 4 of
 *     Philox4x32-10(counter = (j / 16, i, b * H + h, offset),
 *                   key = (seed & 0xffffffff, seed >> 32))
 *     (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *     1, 2, 3", SC'11);
 *   O_i = (256 / t) sum_j keep_ij P_ij V_j; LSE is that of the undropped P.
 * The backward draws the same bytes again (nothing is stored) and returns the
 * gradients of L = <O, dO>: dV = (256/t) (keep o P)^T dO,
 * dS = P o ((256/t) keep o (dO V^T) - D), D_i = sum_k dO_ik O_ik,
 * dQ = scale dS K, dK = scale dS^T Q.  Pass the forward's p_drop, seed and
 * offset.  Other arguments, layouts, scratch and errors are those of
 * attn_fwd / attn_bwd; in addition ATTN_ERR_INVALID_ARG when p_drop is not in
 * [0, 1) or t would be 0 (p_drop > 1 - 1/512).  t = 256 (p_drop < 1/512) is
 * no dropout and runs attn_fwd / attn_bwd.
 */
int attn_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int H, int N, int d, float scale, int causal, float p_drop,
                     unsigned long long seed, unsigned int offset, void* stream);
int attn_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const void* dO,
                     const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                     float scale, int causal, float p_drop, unsigned long long seed,
                     unsigned int offset, void* stream);
/* The same for fp16 q, k, v, o, dO, dq, dk, dv (the keep bytes are identical). */
int attn_fwd_dropout_f16(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                         int H, int N, int d, float scale, int causal, float p_drop,
                         unsigned long long seed, unsigned int offset, void* stream);
int attn_bwd_dropout_f16(const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                         float scale, int causal, float p_drop, unsigned long long seed,
                         unsigned int offset, void* stream);

/*
 * Block-sparse forward (bf16; fp16 through attn_fwd_blocksparse_f16): attn_fwd
 * where whole 128 x 128 tiles of the
 * score matrix are enabled or skipped by a block mask (FlashAttention深度攻略,
 * 进阶追问 "Sparse FlashAttention"; the tiles skipped are never loaded or
 * multiplied, generalising the causal tile skipping).
 *   block_mask : DEVICE pointer, [mask_heads][nb][nb] bytes, nb = ceil(N/128);
 *                head h uses mask (h % H) % mask_heads, mask_heads in {1, H}.
 *                Key j is visible to query i iff
 *                block_mask[..][i / 128][j / 128] != 0 (and j <= i if causal).
 *   A row that sees no key gets O = 0 and LSE = -inf.  N <= 262144 (else
 *   ATTN_ERR_UNSUPPORTED).
 */
int attn_fwd_blocksparse(const void* q, const void* k, const void* v, void* o, float* lse,
                         const unsigned char* block_mask, int mask_heads, int B, int H, int N, int d,
                         float scale, int causal, void* stream);
int attn_fwd_blocksparse_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                             const unsigned char* block_mask, int mask_heads, int B, int H, int N,
                             int d, float scale, int causal, void* stream);

/*
 * Block-sparse backward (bf16; fp16 through attn_bwd_blocksparse_f16): the
 * gradients of attn_fwd_blocksparse's output
 * for the same block_mask, mask_heads and causal flag (o and lse from that
 * call).  The CTA of each 128-key tile visits only the query tiles whose mask
 * entry enables it; a key tile no query tile sees gets dK = dV = 0, and dQ
 * rows of a query block that sees no key are 0.  Scratch and errors as for
 * attn_bwd; the mask constraints as for attn_fwd_blocksparse.
 */
int attn_bwd_blocksparse(const void* q, const void* k, const void* v, const void* o, const void* dO,
                         const float* lse, void* dq, void* dk, void* dv,
                         const unsigned char* block_mask, int mask_heads, int B, int H, int N, int d,
                         float scale, int causal, void* stream);
int attn_bwd_blocksparse_f16(const void* q, const void* k, const void* v, const void* o,
                             const void* dO, const float* lse, void* dq, void* dk, void* dv,
                             const unsigned char* block_mask, int mask_heads, int B, int H, int N,
                             int d, float scale, int causal, void* stream);

/*
 * Block-sparse attention with dropout (both passes; bf16, fp16 through the
 * _f16 twins): the block mask of attn_fwd_blocksparse decides which keys a
 * query sees, and among those the keep rule of attn_fwd_dropout applies
 * unchanged -- keep_ij depends only on (i, j, b * H + h, seed, offset), not on
 * the mask (FlashAttention深度攻略 §7 fuses mask and dropout into the one
 * softmax step; 进阶追问 "Sparse FlashAttention" skips the masked tiles).
 * Arguments are those of attn_fwd_blocksparse / attn_bwd_blocksparse followed
 * by p_drop, seed and offset as for attn_fwd_dropout; the errors are the
 * union of both.  t = 256 runs the block-sparse kernels without dropout.
 */
int attn_fwd_blocksparse_dropout(const void* q, const void* k, const void* v, void* o, float* lse,
                                 const unsigned char* block_mask, int mask_heads, int B, int H, int N, int d,
                                 float scale, int causal, float p_drop, unsigned long long seed,
                                 unsigned int offset, void* stream);
int attn_fwd_blocksparse_dropout_f16(const void* q, const void* k, const void* v, void* o, float* lse,
                                     const unsigned char* block_mask, int mask_heads, int B, int H, int N,
                                     int d, float scale, int causal, float p_drop, unsigned long long seed,
                                     unsigned int offset, void* stream);
int attn_bwd_blocksparse_dropout(const void* q, const void* k, const void* v, const void* o, const void* dO,
                                 const float* lse, void* dq, void* dk, void* dv,
                                 const unsigned char* block_mask, int mask_heads, int B, int H, int N, int d,
                                 float scale, int causal, float p_drop, unsigned long long seed,
                                 unsigned int offset, void* stream);
int attn_bwd_blocksparse_dropout_f16(const void* q, const void* k, const void* v, const void* o,
                                     const void* dO, const float* lse, void* dq, void* dk, void* dv,
                                     const unsigned char* block_mask, int mask_heads, int B, int H, int N,
                                     int d, float scale, int causal, float p_drop, unsigned long long seed,
                                     unsigned int offset, void* stream);

/*
 * Forward with FP8 (e4m3) inputs: q, k, v are [B, H, N, 128] e4m3 bytes whose
 * real values are descale_q*q, descale_k*k, descale_v*v (per-tensor factors,
 * finite and > 0); o is bf16 [B, H, N, 128], lse fp32 [B, H, N] in the units
 * of scale * Q_real K_real^T.  Same method as attn_fwd with 8-bit tensor-core
 * MMAs (FlashAttention (PKM page) 效果 table / FA3 note: FP8 as the further
 * gain); P is rounded to e4m3 for the P V product.  d must be 128 and
 * scale >= 0 (else ATTN_ERR_UNSUPPORTED).  Scratch: a transposed copy of V,
 * B*H*128*ceil(N/128)*128 bytes, from cudaMallocAsync on `stream` (freed on
 * it); launches 2 kernels.
 */
int attn_fwd_fp8(const void* q, const void* k, const void* v, float descale_q, float descale_k,
                 float descale_v, void* o, float* lse, int B, int H, int N, int d, float scale,
                 int causal, void* stream);

/*
 * Decode: exact attention of ONE query token per (batch, head) against a
 * key/value cache of L tokens (bf16), all L keys visible.
 *   q    : in,  [B, H, d] bf16 (the [B, H, 1, d] query of one decode step)
 *   k, v : in,  [B, H, L, d] bf16 cache
 *   o    : out, [B, H, d] bf16;  lse : out, [B, H] fp32
 * The keys of each (b, h) are split across CTAs and the partial results
 * (running max, sum, unnormalised output) merged exactly -- the decode
 * variant named in FlashAttention (PKM page), "注意" section, with the
 * online-softmax merge of "三招" 2.  Bound by reading the cache from HBM.
 * Scratch: B*H*splits*(d+2) floats from cudaMallocAsync on `stream`, freed
 * on it; launches 2 kernels.  Same conventions and errors as attn_fwd.
 */
int attn_decode(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int L, int d, float scale, void* stream);

/*
 * attn_bwd without any memory allocation (bf16).  The pages have no
 * counterpart: this is a deployment variant of attn_bwd.
 *
 * For callers that may not allocate device memory inside the call: code that
 * runs while an allocator must not be re-entered, runtimes that freeze device
 * allocations once a fixed memory budget is set up, or hosts that give the
 * library only the tensors.  Parameters, layouts, ownership and results are
 * those of attn_bwd; the difference is where the scratch lives.  Instead of
 * the stream-ordered allocator it uses one fixed array of 34,078,720 bytes
 * (32.5 MiB) in device memory owned by the library (a GPU that loads the
 * array keeps it until the process exits).  The scratch a problem needs is
 *     align256(4*B*H*N*d) + 2 * align256(4*B*H*ceil(N/128)*128)   bytes;
 * B=1, H=8, N=8192, d=128 needs exactly the whole array.  A problem needing
 * more is rejected with ATTN_ERR_UNSUPPORTED before anything is enqueued
 * (use attn_bwd for it).
 *   - The first call on each device looks up the array's device address on
 *     that device and caches it for the life of the process; make that first
 *     call before any stream capture.  cudaDeviceReset discards the array
 *     together with the context: do not call attn_bwd_noalloc on a device
 *     after resetting it in the same process.
 *   - Every call on a device shares the one array.  A call rewrites all of
 *     the scratch it reads, so it does not depend on what an earlier call
 *     left there, but two calls that can run at the same time on the GPU
 *     (different streams, or different host threads) race on it and give
 *     wrong gradients: order them on one stream or synchronise in between.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dO,
                     const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                     float scale, int causal, void* stream);

/*
 * Synchronises `stream`, then returns and clears the sticky device status of
 * the current device (ATTN_OK, ATTN_ERR_TIMEOUT or ATTN_ERR_DEVICE_CHECK), or
 * ATTN_ERR_CUDA if the synchronisation itself failed.
 */
int attn_sync_status(void* stream);

/* Static, human-readable name of a status code (never NULL). */
const char* attn_status_string(int status);

/* Number of kernel launches the most recent successful attn_fwd* / attn_bwd* /
 * attn_decode call on this thread enqueued (forward 1, backward 3, decode 2). */
int attn_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
