/*
 * pipe_peaks.h -- measurement support for the compute side of the roofline.
 *
 * The selective-scan forward does one exponential (MUFU ex2) and four FP32
 * multiply/fused-multiply-add lane operations per (batch, step, channel,
 * state) element, so its compute roofline is set by the MUFU ex2 rate and the
 * FP32 lane rate of the GPU at the clock it runs.  These microbenchmarks
 * measure both on the running device.  They are not part of the scan's path.
 *
 * ssm_pipe_peaks: runs three throughput kernels on `stream`, times each with
 * CUDA events (after one warm-up launch) and writes
 *   out[0] = ex2 results per second        (ex2.approx.ftz.f32)
 *   out[1] = FP32 FMA lane-ops per second  (scalar fma.rn.f32)
 *   out[2] = FP32 FMA lane-ops per second  (packed fma.rn.f32x2, 2 per instruction)
 *   out[3] = SM count used for the grid
 * Synchronises `stream`.  Returns 0, or a nonzero CUDA error code.
 */
#ifndef PIPE_PEAKS_H
#define PIPE_PEAKS_H
#ifdef __cplusplus
extern "C" {
#endif
typedef struct CUstream_st *cudaStream_t;
__attribute__((visibility("default"))) int ssm_pipe_peaks(double out[4], cudaStream_t stream);
#ifdef __cplusplus
}
#endif
#endif
