/* Throughput loops behind the roofline denominators of libqattn's kernels.
 *
 * The pages treat execution rates as something to measure, not to read off a
 * data sheet: the ZINC post's "fp8 is not faster, it is shaped correctly"
 * times its fp8 and int8 tiles against each other, and QFlash reports
 * tensor-core utilisation per workload (Table 2).  These loops measure, on
 * the GPU at hand, the rate of each unit the attention kernels use:
 *   QATTN_PEAK_TC_F16    tcgen05.mma kind::f16 (M = 128, N = n, K = 16):
 *                        the QK^T product on exact fp16 carriers of int8 codes
 *   QATTN_PEAK_TC_F8     tcgen05.mma kind::f8f6f4 e4m3 (M = 128, N = n,
 *                        K = 32): the e4m3 P . V product
 *   QATTN_PEAK_MMA_S8    mma.sync m16n8k32 s8 (the legacy int8 tensor path)
 *   QATTN_PEAK_MMA_F16   mma.sync m16n8k16 f16 -> f32
 *   QATTN_PEAK_MMA_E4M3  mma.sync m16n8k32 e4m3 -> f32
 *   QATTN_PEAK_EX2       ex2.approx.ftz.f32 on the MUFU unit (one per score)
 *   QATTN_PEAK_TC_ATTN_MIX  the fused attention's MMA sequence per key block
 *                        and query tile: 8 kind::f16 MMAs (N = 128, K = 16)
 *                        into one accumulator, then 4 kind::f8f6f4 MMAs
 *                        (N = 128, K = 32) into another
 * Operands are resident in shared memory (tcgen05: one CTA per SM, one
 * issuing thread, 4 MMAs per round over 128-byte K slices, 128B swizzle) or
 * in registers (mma.sync: 8 independent accumulator chains per warp; ex2: 8
 * chains per thread), so only the unit itself is timed.
 */
#ifndef QATTN_PEAKS_H_
#define QATTN_PEAKS_H_

#ifdef __cplusplus
extern "C" {
#endif

enum {
  QATTN_PEAK_TC_F16 = 0,
  QATTN_PEAK_TC_F8 = 1,
  QATTN_PEAK_MMA_S8 = 2,
  QATTN_PEAK_MMA_F16 = 3,
  QATTN_PEAK_MMA_E4M3 = 4,
  QATTN_PEAK_EX2 = 5,
  QATTN_PEAK_TC_ATTN_MIX = 6
};

/* Error bit set in *err when a tcgen05 loop's completion wait ran out
 * (bounded at about 2 s of SM clock); the loop then returns. */
#define kQattnPeakErrTimeout 1u

/* Launches one loop asynchronously on `stream` (a cudaStream_t):
 *   kind    one of the QATTN_PEAK_* values
 *   n       tcgen05 kinds: the MMA's N (64, 128 or 256); ignored otherwise
 *   iters   loop rounds per CTA (tcgen05: 4 MMAs; the attention mix: 8 + 4;
 *           mma.sync: 8 per warp; ex2: 8 per thread)
 *   blocks  CTAs (tcgen05: one per SM, 128 threads; others: 256 threads)
 *   clocks  device buffer of 4 * blocks uint64: per CTA the SM clock
 *           (clock64) at the start and the end of its loop, then the global
 *           timer (nanoseconds) at the same two points
 *   err     device uint32 error word (see kQattnPeakErrTimeout)
 *   sink    device uint32 the loops may increment (keeps them live)
 * Device buffers are owned by the caller; the operation count of a launch
 * is the caller's to compute from kind, n, iters and blocks.
 * Returns 0 on launch, 1 for an invalid argument, 3 for a CUDA error. */
int qattn_peak_loop(int kind, int n, int iters, int blocks, unsigned long long* clocks,
                    unsigned int* err, unsigned int* sink, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* QATTN_PEAKS_H_ */
