/*
 * attn_diag.h -- diagnostics exported by the same library as attn.h
 * (libattn.so): a self-test of the device failure path and a throughput probe
 * of the exponential unit.  Neither computes attention and the pages have no
 * counterpart to either; they are declared apart from the attention ABI so
 * that a caller of attn.h sees only the method's entry points.  Status codes
 * are attn.h's attn_status_t.
 */
#ifndef ATTN_GB300_DIAG_H
#define ATTN_GB300_DIAG_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Self-test of the device failure path.  Enqueues one tiny kernel that runs
 * the library's bounded pipeline wait on a barrier nothing arrives on, with a
 * limit of `limit_us` microseconds (1 .. 2,000,000).  The wait gives up, the
 * kernel records
 * ATTN_ERR_TIMEOUT in the sticky status and returns; a following
 * attn_sync_status(stream) returns ATTN_ERR_TIMEOUT and clears it.  Nothing
 * hangs or faults; the context stays usable.  Returns ATTN_OK if the kernel
 * was enqueued, ATTN_ERR_INVALID_ARG (nothing enqueued) for a limit out of
 * range.
 */
int attn_debug_wait_timeout(int limit_us, void* stream);

/*
 * Throughput probe of the exponential unit (a measurement aid).  The softmax
 * step needs one exp2 per score (B*H*N^2 per forward, as many again in the
 * backward's recomputation of P), so the unit's rate bounds both passes next
 * to the tensor cores.  Enqueues one kernel of `blocks` x 256 threads; each
 * thread runs `iters` rounds of 8 independent ex2.approx.f32 (the instruction
 * the attention kernels use) and writes one float to `sink`: caller-owned
 * device memory of blocks * 256 floats, 4-byte aligned, overwritten.
 * Exponentials per launch = blocks * 256 * iters * 8; time the launch with
 * events on `stream`.  blocks 1 .. 65535, iters 1 .. 2^20, else
 * ATTN_ERR_INVALID_ARG (nothing enqueued).  Returns ATTN_OK once the kernel
 * is enqueued.
 */
int attn_probe_ex2(float* sink, int blocks, int iters, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_DIAG_H */
