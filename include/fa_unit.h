/*
 * fa_unit.h -- test-only entry points of libfa.so.
 *
 * Each runs one building block of the bf16 attention kernel in isolation on a
 * single 128-row tile, so that a fault in a hand-written PTX primitive
 * (tensor-map load and swizzle, shared-memory matrix descriptors, the MMA
 * instruction descriptor, tensor-memory loads and stores) is found before it
 * is buried inside the full pipeline.  They are not part of the product API.
 *
 * All pointers are DEVICE pointers owned by the caller; every call enqueues
 * one kernel on `stream` (cudaStream_t) and returns without synchronising.
 * d must be 16, 32, 64 or 128.  Errors: FA_ERR_INVALID_ARG for null pointers
 * or a bad flag, FA_ERR_UNSUPPORTED for another d, FA_ERR_MISALIGNED for
 * pointers that are not 16-byte aligned, FA_ERR_CUDA for a failed call.
 *
 * The last one, fa_fwd_simt, runs the true-fp32 CUDA-core kernel on bf16
 * inputs as well, as an independent cross-check of the tensor-core kernel.
 */
#ifndef FA_UNIT_H_
#define FA_UNIT_H_

#include "fa.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Load a [128][d] bf16 tile x (row-major) with the attention kernel's tensor
 * map (3-D, swizzled boxes of at most 64 columns) and copy the raw shared
 * memory image (128 * d * 2 bytes, boxes back to back) to `out`. */
fa_status fa_unit_tma(const void* x, void* out, int d, void* stream);

/* s[128][128] (fp32, row-major) = q[128][d] . k[128][d]^T for bf16 q, k,
 * through TMA loads, one K-major x K-major tcgen05 MMA chain into tensor
 * memory and tcgen05.ld. */
fa_status fa_unit_qk(const void* q, const void* k, float* s, int d, void* stream);

/* o[128][d] (fp32) = bf16(P)[128][128] . v[128][d], with v loaded by TMA as
 * the MN-major B operand of the MMA.  mode selects where P comes from:
 *   0: p (fp32, row-major) rounded to bf16 and written to tensor memory with
 *      tcgen05.st, used as the A operand from tensor memory;
 *   1: as 0, then, right after the P.V chain and without waiting for it, a
 *      second MMA whose accumulator overwrites the tensor-memory columns
 *      holding P (the reuse pattern of the attention kernel); the result must
 *      not change;
 *   2: pb (bf16 [128][128], row-major) loaded by TMA as a K-major shared-memory
 *      A operand (isolates the B operand's descriptor);
 *   3: no MMA: P is written to tensor memory as in mode 0 and its 64 packed
 *      columns are read back into o ([128][64] raw 32-bit words).
 * lbo, sbo: byte strides of the V descriptor (0 = the kernel's own values;
 * otherwise multiples of 16 below 2^18), for layout experiments.  Shared and
 * tensor memory are zeroed first, so a stride that points past the tile reads
 * zeros. */
fa_status fa_unit_pv(const float* p, const void* pb, const void* v, float* o, int d, int mode,
                     unsigned lbo, unsigned sbo, void* stream);

/* Failure-detection check: one CTA of 128 threads waits on an mbarrier that
 * nothing ever arrives on, bounded by budget_cycles SM clocks (1 .. 2^31).
 * Every thread must give up, set the device error word (so that
 * fa_debug_sync_check then returns FA_ERR_TIMEOUT) and see its second wait
 * return at once through the CTA's abort flag; each such thread adds 1 to
 * *gave_up (a device int, 4-byte aligned).  The context stays usable. */
fa_status fa_unit_timeout(long long budget_cycles, int* gave_up, void* stream);

/* Pipe-rate probe, the measured denominator of the softmax rooflines: each
 * of `blocks` CTAs (one per SM: the launch reserves 160 KB of shared memory)
 * runs 512 threads x 8 independent chains x `iters` rounds of one
 * instruction kind -- 0: ex2.approx.ftz.f32 (special-function unit), 1:
 * scalar fp32 FMA, 2: paired fp32 FMA (fma.rn.f32x2) -- and writes its
 * clock64 span to cycles[blockIdx] (device, blocks entries, 8-byte aligned).
 * Instructions per CTA = 512 * 8 * iters for kinds 0 and 1, 512 * 4 * iters
 * for kind 2 (two FMAs each).  sink: device float[512], written only if the
 * chains reach an impossible value (keeps them live).  iters 1 .. 2^24,
 * blocks 1 .. 4096; FA_ERR_INVALID_ARG otherwise. */
fa_status fa_unit_pipe_rate(int kind, int iters, int blocks, float* sink, long long* cycles,
                            void* stream);

/* The fp32 CUDA-core attention kernel for fp32 or bf16 inputs (same
 * arguments and semantics as fa_fwd). */
fa_status fa_fwd_simt(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int Hq, int Hkv, int T, int d, float scale, int causal,
                      fa_dtype dtype, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_UNIT_H_ */
