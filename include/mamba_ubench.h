/*
 * mamba_ubench.h -- throughput micro-benchmarks used to set the roofline
 * denominators of the selective scan (libmamba_ubench.so).  Not part of the
 * scan's ABI; the pages have no counterpart.
 *
 * Each entry point launches `blocks` x `threads` threads on `stream`, each
 * thread running `iters` iterations of 8 independent dependency chains of one
 * instruction kind, and writes one float per thread to `out` (device memory,
 * blocks*threads floats) so the work cannot be removed.  The caller times the
 * launch; operations = blocks * threads * iters * 8 (ex2: exponentials;
 * ffma: fp32 FMAs; ffma2: packed f32x2 FMAs, i.e. two FMAs each; sincos: one
 * sine and one cosine each, i.e. two SFU operations).
 * Returns 0, or 6 (launch failure), or 2 for non-positive sizes.
 */
#ifndef MAMBA_UBENCH_H
#define MAMBA_UBENCH_H

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;

int mamba_ubench_ex2(float *out, int blocks, int threads, int iters, struct CUstream_st *stream);
int mamba_ubench_ffma(float *out, int blocks, int threads, int iters, struct CUstream_st *stream);
int mamba_ubench_ffma2(float *out, int blocks, int threads, int iters, struct CUstream_st *stream);
int mamba_ubench_sincos(float *out, int blocks, int threads, int iters, struct CUstream_st *stream);

#ifdef __cplusplus
}
#endif

#endif
